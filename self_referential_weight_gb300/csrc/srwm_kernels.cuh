// srwm_kernels.cuh -- sm_103a kernels of the SRWM forward recurrence.
//
// The recurrence (per sequence b, head h; "Metalearning Continual Learning
// Algorithms", section 2.3, Eqs. (1)-(3), four-rate version Eqs. (4)-(5)):
//   z_t = [y_t, k_t, q_t, beta_t] = W_{t-1} x~_t
//   W_t = W_{t-1} + diag(g_t) (W_{t-1} (phi(q_t) - phi(k_t))) (outer) phi(k_t)
// with g_t = sigmoid(beta_t) of the row's block and phi = softmax.
//
// GPU formulation.  Each stream's W (m x d fp32) lives in registers for all T
// steps.  One pass over W per step does all three products at once:
//   delta_r  = W[r,:] . u_t          (u_t = phi(q_t) - phi(k_t); Eq. (2) fused)
//   b_r      = W[r,:] . x~_{t+1}     (next step's Eq. (1) on the old matrix)
//   W[r,:]  += g_r delta_r phi(k_t)  (Eq. (3))
//   z_{t+1,r} = b_r + g_r delta_r (phi(k_t) . x~_{t+1})
// The last line is W_t x~_{t+1} written with the rank-one structure of the
// update, so Eq. (1) of step t+1 needs no second sweep over W.  y_{t+1} is
// still the product with the pre-update matrix of step t+1, i.e. W_t.
//
// A thread holds a tile of R rows x 16 (or D/4) columns; the 4 threads of a
// row group finish each dot product with two xor shuffles.  Phase A of a step
// (softmaxes, gates, the scalar phi(k).x~) is O(d) work done by a few warps
// between two barriers.  Inputs stream in by TMA (chunks of TAU steps,
// double-buffered, mbarrier completion with bounded waits); outputs go out by
// TMA from a double-buffered staging area.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "srwm_common.h"
#include "srwm_ptx.cuh"

namespace srwm {

__device__ __forceinline__ float sigmoid_f(float v) { return 1.0f / (1.0f + expf(-v)); }

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// ============================================================================
// d = 64: one CTA per (sequence, head) stream.
// ============================================================================
template <int D_, int NLR_, bool SMX_, int R_>
struct CtaCfg {
    static constexpr int D = D_, NLR = NLR_, R = R_;
    static constexpr bool SMX = SMX_;
    static constexpr int M = 3 * D + NLR;              // rows of W
    static constexpr int CG = 4;                       // column groups (threads per row)
    static constexpr int CPT = D / CG;                 // columns per thread
    static constexpr int NCH = CPT / 4;                // float4 chunks per thread
    static constexpr int RG = rup(cdiv(M, R), 8);      // row groups (threads = RG*CG, whole warps)
    static constexpr int MP = RG * R;                  // padded rows
    static constexpr int NT = RG * CG;                 // threads per CTA
    static constexpr int NW = NT / 32;
    static constexpr int TAU = 32;                     // steps per TMA chunk
    static constexpr int YW = NW - 2;                  // warp issuing y stores
    static constexpr int XW = NW - 1;                  // warp staging x~
    static_assert(D == 64, "the CTA kernel is the d = 64 path");
    static_assert(NW >= 5, "phase A uses five warp roles");
};

template <class C>
struct __align__(128) CtaSmem {
    float xring[2][C::TAU][C::D];   // TMA destination: raw x, two chunks
    float ystage[2][C::TAU][C::D];  // TMA source: y, two chunks
    float z[C::MP];                 // k, q, beta rows of z_t (y rows go to ystage)
    float pk[C::D];                 // phi(k_t)
    float pq[C::D];                 // phi(q_t)
    float xs[2][C::D];              // x~_{t+1}, x~_{t+2}
    float gate[4];                  // sigmoid(beta_t) per block
    float s;                        // phi(k_t) . x~_{t+1}
    int pad[3];
    uint64_t xbar[2];               // "chunk landed" barriers of the x ring
};

template <int D, int NLR, bool SMX, int R>
__global__ void __launch_bounds__(CtaCfg<D, NLR, SMX, R>::NT, 2)
    srwm_cta_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                    const KParams kp)
{
    using C = CtaCfg<D, NLR, SMX, R>;
    constexpr int TAU = C::TAU;
    extern __shared__ unsigned char smem_raw[];
    CtaSmem<C>& sm = *reinterpret_cast<CtaSmem<C>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = tid >> 2, cg = tid & 3;
    const int p = blockIdx.x;
    const int b = p / kp.H, h = p - b * kp.H;
    const int T = kp.T;
    const int nchunks = cdiv(T, TAU);

    // ---- W tile -> registers: rows rg*R + i, columns of chunks cg + 4j.
    float w[R][C::CPT];
    int gsel[R];
    {
        const float* Ws = kp.W_init + static_cast<size_t>(kp.w_per_seq ? p : h) * C::M * D;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = rg * R + i;
            gsel[i] = (NLR == 1) ? 0 : (r < 3 * D ? r / D : 3);
#pragma unroll
            for (int j = 0; j < C::NCH; ++j) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < C::M) v = __ldg(reinterpret_cast<const float4*>(Ws + static_cast<size_t>(r) * D + 4 * (cg + 4 * j)));
                w[i][4 * j + 0] = v.x;
                w[i][4 * j + 1] = v.y;
                w[i][4 * j + 2] = v.z;
                w[i][4 * j + 3] = v.w;
            }
        }
    }

    if (tid == 0) {
        mbar_init(&sm.xbar[0], 1);
        mbar_init(&sm.xbar[1], 1);
        fence_mbar_init();
        if (T > 0) {
            prefetch_tensormap(&tmx);
            prefetch_tensormap(&tmy);
        }
    }
    __syncthreads();

    // ---- x helper state (meaningful in warp XW only)
    int issued = -1;   // highest chunk whose load was issued (or skipped)
    int landed = -1;   // highest chunk seen complete
    constexpr uint32_t kChunkBytes = TAU * D * sizeof(float);

    auto issue_chunk = [&](int c) {
        if (lane == 0 && c != kp.skip_chunk) {
            mbar_arrive_expect_tx(&sm.xbar[c & 1], kChunkBytes);
            tma_load_4d(&sm.xring[c & 1][0][0], &tmx, &sm.xbar[c & 1], 0, h, c * TAU, b);
        }
        issued = c;
    };
    // x~ of step tn into dst (two values per lane: d = 64).
    auto stage_x = [&](int tn, float* dst) {
        if (tn < T) {
            const float* src = sm.xring[(tn / TAU) & 1][tn % TAU];
            float v0 = src[lane], v1 = src[lane + 32];
            if constexpr (SMX) {
                const float mx = group_max<32>(fmaxf(v0, v1));
                v0 = expf(v0 - mx);
                v1 = expf(v1 - mx);
                const float inv = 1.0f / group_sum<32>(v0 + v1);
                v0 *= inv;
                v1 *= inv;
            }
            dst[lane] = v0;
            dst[lane + 32] = v1;
        } else {
            dst[lane] = 0.f;
            dst[lane + 32] = 0.f;
        }
    };

    int fail = 0;
    if (warp == C::XW && T > 0) {
        issue_chunk(0);
        if (nchunks > 1) issue_chunk(1);
        if (__all_sync(0xffffffffu, mbar_wait_bounded(&sm.xbar[0], 0, kp.wait_limit_ns))) {
            landed = 0;
            stage_x(0, sm.xs[0]);
            stage_x(1, sm.xs[1]);
        } else {
            fail = 1;
        }
    }
    int abort = __syncthreads_or(fail);

    // ---- prologue: z_0 = W_0 x~_0
    if (!abort && T > 0) {
        float bb[R];
#pragma unroll
        for (int i = 0; i < R; ++i) bb[i] = 0.f;
#pragma unroll
        for (int j = 0; j < C::NCH; ++j) {
            const float4 xv = ld4(&sm.xs[0][4 * (cg + 4 * j)]);
#pragma unroll
            for (int i = 0; i < R; ++i) {
                bb[i] = fmaf(w[i][4 * j + 0], xv.x, bb[i]);
                bb[i] = fmaf(w[i][4 * j + 1], xv.y, bb[i]);
                bb[i] = fmaf(w[i][4 * j + 2], xv.z, bb[i]);
                bb[i] = fmaf(w[i][4 * j + 3], xv.w, bb[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], 1);
            bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], 2);
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            if ((i & 3) == cg) {
                const int r = rg * R + i;
                if (r < D) sm.ystage[0][0][r] = bb[i];
                else sm.z[r] = bb[i];
            }
        }
        fence_proxy_async_smem();
    }
    __syncthreads();

    // ---- the T steps
    for (int t = 0; t < T && !abort; ++t) {
        // ---------------- phase A: O(d) work on z_t
        fail = 0;
        if (warp == 0) {
            // phi(k_t) and s = phi(k_t) . x~_{t+1}
            const float k0 = sm.z[D + lane], k1 = sm.z[D + 32 + lane];
            const float mx = group_max<32>(fmaxf(k0, k1));
            const float e0 = expf(k0 - mx), e1 = expf(k1 - mx);
            const float* xn = sm.xs[(t + 1) & 1];
            float se = e0 + e1;
            float sx = fmaf(e0, xn[lane], e1 * xn[lane + 32]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                se += __shfl_xor_sync(0xffffffffu, se, o);
                sx += __shfl_xor_sync(0xffffffffu, sx, o);
            }
            const float inv = 1.0f / se;
            sm.pk[lane] = e0 * inv;
            sm.pk[lane + 32] = e1 * inv;
            if (lane == 0) sm.s = sx * inv;
        } else if (warp == 1) {
            // phi(q_t)
            const float q0 = sm.z[2 * D + lane], q1 = sm.z[2 * D + 32 + lane];
            const float mx = group_max<32>(fmaxf(q0, q1));
            const float e0 = expf(q0 - mx), e1 = expf(q1 - mx);
            const float inv = 1.0f / group_sum<32>(e0 + e1);
            sm.pq[lane] = e0 * inv;
            sm.pq[lane + 32] = e1 * inv;
        } else if (warp == 2) {
            // learning rates sigma(beta_t): per block (n_lr = 4) or one for all
            if (lane < 4) sm.gate[lane] = sigmoid_f(sm.z[3 * D + (NLR == 4 ? lane : 0)]);
        } else if (warp == C::YW) {
            // y chunk holding y_t complete -> store it
            if (lane == 0 && (t + 1) % TAU == 0) {
                const int c = t / TAU;
                tma_store_4d(&tmy, &sm.ystage[c & 1][0][0], 0, h, c * TAU, b);
                bulk_commit();
                bulk_wait_read<1>();
            }
        } else if (warp == C::XW) {
            // x~_{t+2} -> xs[t & 1]; a new chunk may have to land first
            const int tn = t + 2;
            if (tn < T && tn % TAU == 0) {
                const int c = tn / TAU;
                const bool ok = mbar_wait_bounded(&sm.xbar[c & 1], (c >> 1) & 1, kp.wait_limit_ns);
                if (__all_sync(0xffffffffu, ok)) {
                    landed = c;
                    if (c + 1 < nchunks) issue_chunk(c + 1);
                } else {
                    fail = 1;
                }
            }
            if (!fail) stage_x(tn, sm.xs[t & 1]);
        }
        abort = __syncthreads_or(fail);
        if (abort) break;

        // ---------------- phase B: one pass over W
        {
            const float* xn = sm.xs[(t + 1) & 1];
            float a[R], bb[R];
#pragma unroll
            for (int i = 0; i < R; ++i) a[i] = bb[i] = 0.f;
            float4 pkv[C::NCH];
#pragma unroll
            for (int j = 0; j < C::NCH; ++j) {
                const int col = 4 * (cg + 4 * j);
                const float4 xv = ld4(xn + col);
                const float4 qv = ld4(sm.pq + col);
                pkv[j] = ld4(sm.pk + col);
                const float u0 = qv.x - pkv[j].x, u1 = qv.y - pkv[j].y;
                const float u2 = qv.z - pkv[j].z, u3 = qv.w - pkv[j].w;
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    a[i] = fmaf(w[i][4 * j + 0], u0, a[i]);
                    bb[i] = fmaf(w[i][4 * j + 0], xv.x, bb[i]);
                    a[i] = fmaf(w[i][4 * j + 1], u1, a[i]);
                    bb[i] = fmaf(w[i][4 * j + 1], xv.y, bb[i]);
                    a[i] = fmaf(w[i][4 * j + 2], u2, a[i]);
                    bb[i] = fmaf(w[i][4 * j + 2], xv.z, bb[i]);
                    a[i] = fmaf(w[i][4 * j + 3], u3, a[i]);
                    bb[i] = fmaf(w[i][4 * j + 3], xv.w, bb[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < R; ++i) {
                a[i] += __shfl_xor_sync(0xffffffffu, a[i], 1);
                bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], 1);
            }
#pragma unroll
            for (int i = 0; i < R; ++i) {
                a[i] += __shfl_xor_sync(0xffffffffu, a[i], 2);
                bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], 2);
            }
            const float4 g4 = ld4(sm.gate);
            const float s = sm.s;
            const bool write_y = (t + 1 < T);
            const int yb = ((t + 1) / TAU) & 1, yr = (t + 1) % TAU;
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const float g = gsel[i] == 0 ? g4.x : gsel[i] == 1 ? g4.y : gsel[i] == 2 ? g4.z : g4.w;
                const float coef = g * a[i];
#pragma unroll
                for (int j = 0; j < C::NCH; ++j) {
                    w[i][4 * j + 0] = fmaf(coef, pkv[j].x, w[i][4 * j + 0]);
                    w[i][4 * j + 1] = fmaf(coef, pkv[j].y, w[i][4 * j + 1]);
                    w[i][4 * j + 2] = fmaf(coef, pkv[j].z, w[i][4 * j + 2]);
                    w[i][4 * j + 3] = fmaf(coef, pkv[j].w, w[i][4 * j + 3]);
                }
                const float zr = fmaf(coef, s, bb[i]);
                if ((i & 3) == cg) {
                    const int r = rg * R + i;
                    if (r < D) {
                        if (write_y) sm.ystage[yb][yr][r] = zr;
                    } else {
                        sm.z[r] = zr;
                    }
                }
            }
            if (write_y && ((t + 2) % TAU == 0 || t + 2 == T)) fence_proxy_async_smem();
        }
        __syncthreads();
    }

    // ---- drain
    if (warp == C::YW && lane == 0) {
        if (!abort && T > 0 && T % TAU != 0) {
            const int c = (T - 1) / TAU;
            tma_store_4d(&tmy, &sm.ystage[c & 1][0][0], 0, h, c * TAU, b);
            bulk_commit();
        }
        bulk_wait_all<0>();
    }
    if (warp == C::XW && abort) {
        // Let every load still in flight land before the CTA gives up its
        // shared memory; report the timeout.
        for (int c = landed + 1; c <= issued; ++c) {
            if (c == kp.skip_chunk) continue;
            mbar_wait_bounded(&sm.xbar[c & 1], (c >> 1) & 1, kp.wait_limit_ns);
        }
        if (lane == 0) atomicOr(kp.status, kStatusTimeout);
    }
    if (abort) return;

    // ---- W_T -> W_out[b, h]
    float* Wd = kp.W_out + static_cast<size_t>(p) * C::M * D;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int r = rg * R + i;
        if (r < C::M) {
#pragma unroll
            for (int j = 0; j < C::NCH; ++j) {
                *reinterpret_cast<float4*>(Wd + static_cast<size_t>(r) * D + 4 * (cg + 4 * j)) =
                    make_float4(w[i][4 * j + 0], w[i][4 * j + 1], w[i][4 * j + 2], w[i][4 * j + 3]);
            }
        }
    }
}

// ============================================================================
// d = 16 and d = 32: one warp per (sequence, head) stream, PPC streams per CTA.
// Lane = (row group rg = lane/4, column group cg = lane%4); rows rg + 8 i.
// ============================================================================
template <int D_, int NLR_, bool SMX_>
struct WarpCfg {
    static constexpr int D = D_, NLR = NLR_;
    static constexpr bool SMX = SMX_;
    static constexpr int M = 3 * D + NLR;
    static constexpr int CG = 4;
    static constexpr int RPT = cdiv(M, 8);   // rows per lane
    static constexpr int MP = 8 * RPT;
    static constexpr int CPT = D / CG;
    static constexpr int NCH = CPT / 4;
    static constexpr int TAU = 16;
    static constexpr int PPC = (D == 16) ? 8 : 6;   // streams (warps) per CTA
    static constexpr int NT = 32 * PPC;
    static_assert(D == 16 || D == 32, "the warp kernel is the d = 16 / 32 path");
    // gate index of row slot i (rows rg + 8i never cross a block boundary)
    SRWM_HD static constexpr int gidx(int i) { return NLR == 1 ? 0 : (8 * i < 3 * D ? (8 * i) / D : 3); }
};

template <class C>
struct __align__(128) WarpSmem {
    float xring[2][C::TAU][C::D];
    float ystage[2][C::TAU][C::D];
    float z[C::MP];
    float pk[C::D];
    float pq[C::D];
    float xs[2][C::D];
    float gate[4];
    float s;
    int pad[3];
    uint64_t xbar[2];
};

template <int D, int NLR, bool SMX>
__global__ void __launch_bounds__(WarpCfg<D, NLR, SMX>::NT, 2)
    srwm_warp_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                     const KParams kp)
{
    using C = WarpCfg<D, NLR, SMX>;
    constexpr int TAU = C::TAU;
    constexpr int RPT = C::RPT;
    extern __shared__ unsigned char smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    WarpSmem<C>& sm = reinterpret_cast<WarpSmem<C>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127))[warp];

    const int p = blockIdx.x * C::PPC + warp;
    if (p >= kp.B * kp.H) return;  // whole warp leaves; no CTA-wide barrier below
    const int b = p / kp.H, h = p - b * kp.H;
    const int rg = lane >> 2, cg = lane & 3;
    const int T = kp.T;
    const int nchunks = cdiv(T, TAU);

    float w[RPT][C::CPT];
    {
        const float* Ws = kp.W_init + static_cast<size_t>(kp.w_per_seq ? p : h) * C::M * D;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int r = rg + 8 * i;
#pragma unroll
            for (int j = 0; j < C::NCH; ++j) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < C::M) v = __ldg(reinterpret_cast<const float4*>(Ws + static_cast<size_t>(r) * D + 4 * (cg + 4 * j)));
                w[i][4 * j + 0] = v.x;
                w[i][4 * j + 1] = v.y;
                w[i][4 * j + 2] = v.z;
                w[i][4 * j + 3] = v.w;
            }
        }
    }

    if (lane == 0) {
        mbar_init(&sm.xbar[0], 1);
        mbar_init(&sm.xbar[1], 1);
        fence_mbar_init();
    }
    __syncwarp();

    int issued = -1, landed = -1;
    constexpr uint32_t kChunkBytes = TAU * D * sizeof(float);
    auto issue_chunk = [&](int c) {
        if (lane == 0 && c != kp.skip_chunk) {
            mbar_arrive_expect_tx(&sm.xbar[c & 1], kChunkBytes);
            tma_load_4d(&sm.xring[c & 1][0][0], &tmx, &sm.xbar[c & 1], 0, h, c * TAU, b);
        }
        issued = c;
    };
    // x~ of step tn into dst.  Lane l handles column l % D (d = 16: both halves
    // compute the same values, the lower half writes).
    auto stage_x = [&](int tn, float* dst) {
        const int col = lane & (D - 1);
        float v = 0.f;
        if (tn < T) {
            v = sm.xring[(tn / TAU) & 1][tn % TAU][col];
            if constexpr (SMX) {
                const float mx = group_max<D>(v);
                v = expf(v - mx);
                v = v / group_sum<D>(v);
            }
        }
        if (lane < D) dst[col] = v;
    };

    int abort = 0;
    if (T > 0) {
        issue_chunk(0);
        if (nchunks > 1) issue_chunk(1);
        const bool ok = mbar_wait_bounded(&sm.xbar[0], 0, kp.wait_limit_ns);
        abort = __any_sync(0xffffffffu, !ok);
        if (!abort) {
            landed = 0;
            stage_x(0, sm.xs[0]);
            stage_x(1, sm.xs[1]);
        }
        __syncwarp();
    }

    // ---- prologue: z_0 = W_0 x~_0
    if (!abort && T > 0) {
        float bb[RPT];
#pragma unroll
        for (int i = 0; i < RPT; ++i) bb[i] = 0.f;
#pragma unroll
        for (int j = 0; j < C::NCH; ++j) {
            const float4 xv = ld4(&sm.xs[0][4 * (cg + 4 * j)]);
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                bb[i] = fmaf(w[i][4 * j + 0], xv.x, bb[i]);
                bb[i] = fmaf(w[i][4 * j + 1], xv.y, bb[i]);
                bb[i] = fmaf(w[i][4 * j + 2], xv.z, bb[i]);
                bb[i] = fmaf(w[i][4 * j + 3], xv.w, bb[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], 1);
            bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], 2);
        }
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            if ((i & 3) == cg) {
                const int r = rg + 8 * i;
                if (r < D) sm.ystage[0][0][r] = bb[i];
                else sm.z[r] = bb[i];
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
    }

    for (int t = 0; t < T && !abort; ++t) {
        // ---------------- phase A (the whole warp)
        if (lane == 0 && (t + 1) % TAU == 0) {
            const int c = t / TAU;
            tma_store_4d(&tmy, &sm.ystage[c & 1][0][0], 0, h, c * TAU, b);
            bulk_commit();
            bulk_wait_read<1>();
        }
        {
            const float* xn = sm.xs[(t + 1) & 1];
            if constexpr (D == 32) {
                const float kv = sm.z[D + lane], qv = sm.z[2 * D + lane];
                float mk = kv, mq = qv;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
                    mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
                }
                const float ek = expf(kv - mk), eq = expf(qv - mq);
                float sk = ek, sq = eq, sx = ek * xn[lane];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    sk += __shfl_xor_sync(0xffffffffu, sk, o);
                    sq += __shfl_xor_sync(0xffffffffu, sq, o);
                    sx += __shfl_xor_sync(0xffffffffu, sx, o);
                }
                const float ik = 1.0f / sk;
                sm.pk[lane] = ek * ik;
                sm.pq[lane] = eq * (1.0f / sq);
                if (lane == 0) sm.s = sx * ik;
            } else {
                // rows D..3D-1 are contiguous: lanes 0-15 take k, lanes 16-31 take q
                const float v = sm.z[D + lane];
                const float mx = group_max<16>(v);
                const float e = expf(v - mx);
                float se = e, sx = (lane < 16) ? e * xn[lane] : 0.f;
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) {
                    se += __shfl_xor_sync(0xffffffffu, se, o);
                    sx += __shfl_xor_sync(0xffffffffu, sx, o);
                }
                const float inv = 1.0f / se;
                if (lane < 16) sm.pk[lane] = e * inv;
                else sm.pq[lane - 16] = e * inv;
                if (lane == 0) sm.s = sx * inv;
            }
            if (lane < 4) sm.gate[lane] = sigmoid_f(sm.z[3 * D + (NLR == 4 ? lane : 0)]);
        }
        {
            const int tn = t + 2;
            bool ok = true;
            if (tn < T && tn % TAU == 0) {
                const int c = tn / TAU;
                ok = mbar_wait_bounded(&sm.xbar[c & 1], (c >> 1) & 1, kp.wait_limit_ns);
                if (__all_sync(0xffffffffu, ok)) {
                    landed = c;
                    if (c + 1 < nchunks) issue_chunk(c + 1);
                } else {
                    ok = false;
                }
            }
            abort = __any_sync(0xffffffffu, !ok);
            if (abort) break;
            stage_x(tn, sm.xs[t & 1]);
        }
        __syncwarp();

        // ---------------- phase B: one pass over W
        {
            const float* xn = sm.xs[(t + 1) & 1];
            float a[RPT], bb[RPT];
#pragma unroll
            for (int i = 0; i < RPT; ++i) a[i] = bb[i] = 0.f;
            float4 pkv[C::NCH];
#pragma unroll
            for (int j = 0; j < C::NCH; ++j) {
                const int col = 4 * (cg + 4 * j);
                const float4 xv = ld4(xn + col);
                const float4 qv = ld4(sm.pq + col);
                pkv[j] = ld4(sm.pk + col);
                const float u0 = qv.x - pkv[j].x, u1 = qv.y - pkv[j].y;
                const float u2 = qv.z - pkv[j].z, u3 = qv.w - pkv[j].w;
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    a[i] = fmaf(w[i][4 * j + 0], u0, a[i]);
                    bb[i] = fmaf(w[i][4 * j + 0], xv.x, bb[i]);
                    a[i] = fmaf(w[i][4 * j + 1], u1, a[i]);
                    bb[i] = fmaf(w[i][4 * j + 1], xv.y, bb[i]);
                    a[i] = fmaf(w[i][4 * j + 2], u2, a[i]);
                    bb[i] = fmaf(w[i][4 * j + 2], xv.z, bb[i]);
                    a[i] = fmaf(w[i][4 * j + 3], u3, a[i]);
                    bb[i] = fmaf(w[i][4 * j + 3], xv.w, bb[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                a[i] += __shfl_xor_sync(0xffffffffu, a[i], 1);
                bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], 1);
            }
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                a[i] += __shfl_xor_sync(0xffffffffu, a[i], 2);
                bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], 2);
            }
            const float4 g4 = ld4(sm.gate);
            const float s = sm.s;
            const bool write_y = (t + 1 < T);
            const int yb = ((t + 1) / TAU) & 1, yr = (t + 1) % TAU;
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int gi = C::gidx(i);
                const float g = gi == 0 ? g4.x : gi == 1 ? g4.y : gi == 2 ? g4.z : g4.w;
                const float coef = g * a[i];
#pragma unroll
                for (int j = 0; j < C::NCH; ++j) {
                    w[i][4 * j + 0] = fmaf(coef, pkv[j].x, w[i][4 * j + 0]);
                    w[i][4 * j + 1] = fmaf(coef, pkv[j].y, w[i][4 * j + 1]);
                    w[i][4 * j + 2] = fmaf(coef, pkv[j].z, w[i][4 * j + 2]);
                    w[i][4 * j + 3] = fmaf(coef, pkv[j].w, w[i][4 * j + 3]);
                }
                const float zr = fmaf(coef, s, bb[i]);
                if ((i & 3) == cg) {
                    const int r = rg + 8 * i;
                    if (r < D) {
                        if (write_y) sm.ystage[yb][yr][r] = zr;
                    } else {
                        sm.z[r] = zr;
                    }
                }
            }
            if (write_y && ((t + 2) % TAU == 0 || t + 2 == T)) fence_proxy_async_smem();
        }
        __syncwarp();
    }

    // ---- drain
    if (lane == 0) {
        if (!abort && T > 0 && T % TAU != 0) {
            const int c = (T - 1) / TAU;
            tma_store_4d(&tmy, &sm.ystage[c & 1][0][0], 0, h, c * TAU, b);
            bulk_commit();
        }
        bulk_wait_all<0>();
    }
    if (abort) {
        for (int c = landed + 1; c <= issued; ++c) {
            if (c == kp.skip_chunk) continue;
            mbar_wait_bounded(&sm.xbar[c & 1], (c >> 1) & 1, kp.wait_limit_ns);
        }
        if (lane == 0) atomicOr(kp.status, kStatusTimeout);
        return;
    }

    float* Wd = kp.W_out + static_cast<size_t>(p) * C::M * D;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int r = rg + 8 * i;
        if (r < C::M) {
#pragma unroll
            for (int j = 0; j < C::NCH; ++j) {
                *reinterpret_cast<float4*>(Wd + static_cast<size_t>(r) * D + 4 * (cg + 4 * j)) =
                    make_float4(w[i][4 * j + 0], w[i][4 * j + 1], w[i][4 * j + 2], w[i][4 * j + 3]);
            }
        }
    }
}

// ============================================================================
// Launch description of one instantiation.
// ============================================================================
template <int D, int NLR, bool SMX>
LaunchInfo launch_info()
{
    if constexpr (D == 64) {
        using C = CtaCfg<D, NLR, SMX, 5>;
        return LaunchInfo{reinterpret_cast<const void*>(&srwm_cta_kernel<D, NLR, SMX, 5>), C::NT, 1,
                          static_cast<int>(sizeof(CtaSmem<C>)) + 128, C::TAU};
    } else {
        using C = WarpCfg<D, NLR, SMX>;
        return LaunchInfo{reinterpret_cast<const void*>(&srwm_warp_kernel<D, NLR, SMX>), C::NT, C::PPC,
                          static_cast<int>(C::PPC * sizeof(WarpSmem<C>)) + 128, C::TAU};
    }
}

}  // namespace srwm
