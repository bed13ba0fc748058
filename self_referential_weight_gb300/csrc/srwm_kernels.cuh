// srwm_kernels.cuh -- the d = 16 / d = 32 kernel of the SRWM forward
// recurrence: one warp per (sequence, head) stream, several streams per CTA.
//
// The recurrence (per sequence b, head h; "Metalearning Continual Learning
// Algorithms", section 2.3, Eqs. (1)-(3), four-rate version Eqs. (4)-(5)):
//   z_t = [y_t, k_t, q_t, beta_t] = W_{t-1} x~_t
//   W_t = W_{t-1} + diag(g_t) (W_{t-1} (phi(q_t) - phi(k_t))) (outer) phi(k_t)
// with g_t = sigmoid(beta_t) of the row's block and phi = softmax.
//
// GPU formulation.  Each stream's W (m x d fp32) lives in the registers of its
// warp for all T steps.  One pass over W per step does all three products:
//   a_r       = W[r,:] . u_t              (u_t = phi(q_t) - phi(k_t); Eq. (2) fused)
//   b_r       = W[r,:] . x~_{t+1}         (next step's Eq. (1) on the old matrix)
//   W[r,:]   += g_r a_r phi(k_t)           (Eq. (3))
//   z_{t+1,r} = b_r + g_r a_r (phi(k_t) . x~_{t+1})
// The last line is W_t x~_{t+1} written with the rank-one structure of the
// update, so Eq. (1) of step t+1 needs no second sweep over W, and y_{t+1} is
// still the product with the pre-update matrix of step t+1, i.e. W_t.
//
// Lane = (row group rg = lane/4, column group cg = lane%4): rows rg + 8 i,
// columns of float4 chunks cg + 4 j.  Phase A of a step (both softmaxes and
// the gates) runs on the whole warp with warp-wide reductions (redux max and a
// fixed-point redux sum); phase B is the row pass, finished by two xor
// shuffles over the four column groups.  No CTA-wide barrier is needed: only
// __syncwarp.  Inputs stream in by TMA (chunks of TAU steps, double-buffered,
// mbarrier completion with bounded waits); outputs go out by TMA from a
// double-buffered staging area.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "srwm_common.h"
#include "srwm_ptx.cuh"

namespace srwm {

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// softmax over D in {16, 32} values, lane l holding entry l % D (for D = 16
// both half-warps hold the same 16 values, so the warp sum counts each twice).
template <int D>
__device__ __forceinline__ float softmax_lane(float v)
{
    const float mx = redux_max(v);
    const float e = __expf(v - mx);
    float sum = warp_sum_unit1(e);
    if constexpr (D == 16) sum *= 0.5f;
    return e * rcp_approx(sum);
}

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
    // Streams (warps) per CTA.  d = 32 holds 104 W registers per lane; six
    // warps per CTA and two CTAs per SM (three warps per scheduler) keep it
    // under the per-scheduler register budget without spills.
    static constexpr int PPC = (D == 16) ? 8 : 6;
    static constexpr int NT = 32 * PPC;
    static_assert(D == 16 || D == 32, "the warp kernel is the d = 16 / 32 path");
    // gate index of row slot i (rows rg + 8i never cross a block boundary)
    SRWM_HD static constexpr int gidx(int i) { return NLR == 1 ? 0 : (8 * i < 3 * D ? (8 * i) / D : 3); }
};

template <class C>
struct __align__(128) WarpSmem {
    float xring[2][C::TAU][C::D];   // TMA destination: raw x, two chunks
    float ystage[2][C::TAU][C::D];  // TMA source: y, two chunks
    float z[C::MP];                 // k, q, beta rows of z_t (y rows go to ystage)
    float pk[C::D];                 // phi(k_t)
    float pq[C::D];                 // phi(q_t)
    float xs[2][C::D];              // x~_{t+1}, x~_{t+2}
    uint64_t xbar[2];               // "chunk landed" barriers of the x ring
};

template <int D, int NLR, bool SMX, bool EMIT = false>
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

    const int rg = lane >> 2, cg = lane & 3;
    const int col = lane & (D - 1);   // column of this lane in the softmax layout
    constexpr uint32_t kChunkBytes = TAU * D * sizeof(float);

    if (lane == 0) {
        mbar_init(&sm.xbar[0], 1);
        mbar_init(&sm.xbar[1], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // completed phases of the two x buffers over all items of this warp
    uint32_t used0 = 0, used1 = 0;
    int abort = 0;
    int issued = -1, landed = -1;   // chunks of the current item

    const int slot = blockIdx.x * C::PPC + warp;
    const int n_slots = gridDim.x * C::PPC;
    for (int item = slot; item < kp.n_items; item += n_slots) {
        const int p = item % kp.n_streams, seg = item / kp.n_streams;
        const int b = p / kp.H, h = p - b * kp.H;
        const int t0 = seg * kp.seg_len;
        const int T = min(kp.seg_len, kp.T - t0);   // steps of this item
        const int nchunks = cdiv(T, TAU);
        issued = -1;
        landed = -1;

        // ---- the previous segment of this stream has to be finished
        if (seg > 0) {
            int ok = 1;
            if (lane == 0) ok = wait_counter_bounded(kp.seg_done + p, seg, kp.wait_limit_ns);
            abort = !__shfl_sync(0xffffffffu, ok, 0);
            if (abort) break;
        }

        // ---- W -> registers (W_init for a first segment, else the state the
        // previous segment left in W_out; read through L2)
        float w[RPT][C::CPT];
        {
            const float* Ws = (seg == 0) ? kp.W_init + static_cast<size_t>(kp.w_per_seq ? p : h) * C::M * D
                                         : kp.W_out + static_cast<size_t>(p) * C::M * D;
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int r = rg + 8 * i;
#pragma unroll
                for (int j = 0; j < C::NCH; ++j) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (r < C::M) v = __ldcg(reinterpret_cast<const float4*>(Ws + static_cast<size_t>(r) * D + 4 * (cg + 4 * j)));
                    w[i][4 * j + 0] = v.x;
                    w[i][4 * j + 1] = v.y;
                    w[i][4 * j + 2] = v.z;
                    w[i][4 * j + 3] = v.w;
                }
            }
        }

        // chunk c of this item is steps t0 + c*TAU .. and lands in buffer c & 1
        auto parity = [&](int c) -> uint32_t { return (((c & 1) ? used1 : used0) + (c >> 1)) & 1; };
        auto issue_chunk = [&](int c) {
            if (lane == 0 && c != kp.skip_chunk) {
                mbar_arrive_expect_tx(&sm.xbar[c & 1], kChunkBytes);
                tma_load_4d(&sm.xring[c & 1][0][0], &tmx, &sm.xbar[c & 1], 0, h, t0 + c * TAU, b);
            }
            issued = c;
        };
        // x~ of step tn into dst (d = 16: both halves compute, the lower one writes).
        auto stage_x = [&](int tn, float* dst) {
            float v = 0.f;
            if (tn < T) {
                v = sm.xring[(tn / TAU) & 1][tn % TAU][col];
                if constexpr (SMX) v = softmax_lane<D>(v);
            }
            if (lane < D) dst[col] = v;
        };

        if (T > 0) {
            issue_chunk(0);
            if (nchunks > 1) issue_chunk(1);
            const bool ok = mbar_wait_bounded(&sm.xbar[0], parity(0), kp.wait_limit_ns);
            abort = __any_sync(0xffffffffu, !ok);
            if (!abort) {
                landed = 0;
                stage_x(0, sm.xs[0]);
                stage_x(1, sm.xs[1]);
            }
            __syncwarp();
        }

        // ---- prologue: z_0 = W x~_0 (y of the item's first step)
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
                tma_store_4d(&tmy, &sm.ystage[c & 1][0][0], 0, h, t0 + c * TAU, b);
                bulk_commit();
                bulk_wait_read<1>();
            }
            const float pk = softmax_lane<D>(sm.z[D + col]);
            const float pq = softmax_lane<D>(sm.z[2 * D + col]);
            float g[4];
            {
                const float4 beta = ld4(&sm.z[3 * D]);
                if constexpr (NLR == 4) {
                    g[0] = sigmoid_fast(beta.x);
                    g[1] = sigmoid_fast(beta.y);
                    g[2] = sigmoid_fast(beta.z);
                    g[3] = sigmoid_fast(beta.w);
                } else {
                    g[0] = g[1] = g[2] = g[3] = sigmoid_fast(beta.x);
                }
            }
            if (lane < D) {
                sm.pk[col] = pk;
                sm.pq[col] = pq;
            }
            // backward record of step t: phi(k), u = pq - pk, gates (a follows below)
            float* em = nullptr;
            if constexpr (EMIT) {
                em = kp.emit + (static_cast<size_t>(p) * kp.T + t0 + t) * kp.emit_stride;
                if (lane < D) {
                    em[col] = pk;
                    em[D + col] = __fsub_rn(pq, pk);   // as the row pass forms it (no contraction)
                }
                if (lane < 4) em[2 * D + lane] = lane == 0 ? g[0] : lane == 1 ? g[1] : lane == 2 ? g[2] : g[3];
            }
            {
                const int tn = t + 2;
                bool ok = true;
                if (tn < T && tn % TAU == 0) {
                    const int c = tn / TAU;
                    ok = mbar_wait_bounded(&sm.xbar[c & 1], parity(c), kp.wait_limit_ns);
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
                float s = 0.f;   // partial phi(k_t) . x~_{t+1} over this lane's columns
                float4 pkv[C::NCH];
#pragma unroll
                for (int j = 0; j < C::NCH; ++j) {
                    const int c4 = 4 * (cg + 4 * j);
                    const float4 xv = ld4(xn + c4);
                    const float4 qv = ld4(sm.pq + c4);
                    pkv[j] = ld4(sm.pk + c4);
                    const float u0 = qv.x - pkv[j].x, u1 = qv.y - pkv[j].y;
                    const float u2 = qv.z - pkv[j].z, u3 = qv.w - pkv[j].w;
                    s = fmaf(pkv[j].x, xv.x, s);
                    s = fmaf(pkv[j].y, xv.y, s);
                    s = fmaf(pkv[j].z, xv.z, s);
                    s = fmaf(pkv[j].w, xv.w, s);
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
                for (int o = 1; o <= 2; o <<= 1) {
#pragma unroll
                    for (int i = 0; i < RPT; ++i) {
                        a[i] += __shfl_xor_sync(0xffffffffu, a[i], o);
                        bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], o);
                    }
                    s += __shfl_xor_sync(0xffffffffu, s, o);
                }
                const bool write_y = (t + 1 < T);
                const int yb = ((t + 1) / TAU) & 1, yr = (t + 1) % TAU;
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const float coef = g[C::gidx(i)] * a[i];
#pragma unroll
                    for (int j = 0; j < C::NCH; ++j) {
                        w[i][4 * j + 0] = fmaf(coef, pkv[j].x, w[i][4 * j + 0]);
                        w[i][4 * j + 1] = fmaf(coef, pkv[j].y, w[i][4 * j + 1]);
                        w[i][4 * j + 2] = fmaf(coef, pkv[j].z, w[i][4 * j + 2]);
                        w[i][4 * j + 3] = fmaf(coef, pkv[j].w, w[i][4 * j + 3]);
                    }
                    const float zr = fmaf(coef, s, bb[i]);
                    if constexpr (EMIT) {
                        if ((i & 3) == cg && rg + 8 * i < C::M) em[2 * D + 4 + rg + 8 * i] = a[i];
                    }
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

        // ---- drain this item's y stores
        if (lane == 0) {
            if (!abort && T > 0 && T % TAU != 0) {
                const int c = (T - 1) / TAU;
                tma_store_4d(&tmy, &sm.ystage[c & 1][0][0], 0, h, t0 + c * TAU, b);
                bulk_commit();
            }
            bulk_wait_all<0>();
        }
        __syncwarp();
        if (abort) break;
        used0 += (nchunks + 1) / 2;
        used1 += nchunks / 2;

        // ---- the state -> W_out[b, h]
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
        __syncwarp();
        if (kp.seg_done != nullptr && lane == 0) {
            __threadfence();
            st_release_gpu(kp.seg_done + p, seg + 1);
        }
    }

    if (abort) {
        // every load still in flight lands before the warp gives up its buffers
        for (int c = landed + 1; c <= issued; ++c) {
            if (c == kp.skip_chunk) continue;
            mbar_wait_bounded(&sm.xbar[c & 1], (((c & 1) ? used1 : used0) + (c >> 1)) & 1, kp.wait_limit_ns);
        }
        if (lane == 0) atomicOr(kp.status, kStatusTimeout);
    }
}

template <int D, int NLR, bool SMX, bool EMIT = false>
LaunchInfo launch_info()
{
    using C = WarpCfg<D, NLR, SMX>;
    return LaunchInfo{reinterpret_cast<const void*>(&srwm_warp_kernel<D, NLR, SMX, EMIT>), C::NT, C::PPC,
                      static_cast<int>(C::PPC * sizeof(WarpSmem<C>)) + 128, C::TAU};
}

}  // namespace srwm
