// srwm_d64r.cuh -- the d = 64 kernel for many streams: one (sequence, head)
// stream per CTA of two warps, four CTAs per SM, whole rows of W per thread.
//
// Math (per step t; "Metalearning Continual Learning Algorithms", section 2.3,
// Eqs. (1)-(3), four-rate version Eqs. (4)-(5)):
//   phi_k = softmax(k_t), phi_q = softmax(q_t), g = sigmoid(beta_t) per block
//   a_r   = W_{t-1}[r,:] . (phi_q - phi_k)
//   W_t[r,:] = W_{t-1}[r,:] + g_r a_r phi_k
//   z_{t+1,r} = b_r + g_r a_r (phi_k . x~_{t+1}),  b_r = W_{t-1}[r,:] . x~_{t+1}
// (the last line is W_t x~_{t+1} through the rank-one structure of the update).
//
// Layout.  Thread t of the 64 holds rows t, 64 + t and 128 + t (its y, k and
// q rows) whole, as 32 column pairs each: 192 registers of W, and a row's dot
// products finish inside the thread.  The n_lr beta rows are spread four
// columns per thread (thread t: beta row t / 16, columns 4 (t % 16) .. + 3;
// threads whose row is >= n_lr hold zeros) and their dots finish over 16
// lanes.  Operand vectors (phi_k, u, x~) are read from shared memory as
// broadcast float4 loads, and the item's bookkeeping lives in shared memory,
// so that W and little else stays in the 255 registers.
//
// One step:
//   1. each warp reads k_t, q_t (exchanged through shared memory at the
//      previous barrier) and computes phi_k, phi_q over all 64 entries (two
//      per lane), so both warps hold the same values without a second
//      barrier.  Beside these softmaxes, which are the step's chain, the
//      thread applies the pending update of step t - 1 to its rows and forms
//      b = W_{t-1} x~_{t+1} (both independent of the softmaxes), per float4
//      column chunk with two-wide FMAs; the beta rows likewise;
//   2. phi_k and u = phi_q - phi_k go to the warp's own buffers (__syncwarp);
//   3. a = W_{t-1} u for the thread's rows (two accumulators per row), with
//      s = phi_k . x~_{t+1} (a warp sum) and the beta rows' sums over 16 lanes
//      beside it;
//   4. gates, the rows' z_{t+1} into shared memory (y rows into the TMA
//      staging ring), barrier.
// Steps run chunk by chunk: waits, TMA loads and stores sit at chunk
// boundaries, and with the input softmax the two warps replace a landed
// chunk's rows by x~ in place there, so a step reads x~ straight from the
// three-chunk x ring.  With records on (the forward of the
// backward pass), step t also writes phi_k, u, the gates and the rows' a.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "srwm_common.h"
#include "srwm_ptx.cuh"

namespace srwm {

namespace d64r {

constexpr int D = 64;
constexpr int TAU = 32;     // steps per TMA chunk
constexpr int NW = 2;       // warps per stream
constexpr int NT = 32 * NW;
constexpr int NP = D / 2;   // column pairs per row

struct __align__(128) Smem {
    float xring[3 * TAU][D];   // x by TMA, three chunks (row = step mod 3 TAU); x~ in place
    float yring[3 * TAU][D];   // y for TMA, three chunks (row = step mod 3 TAU)
    float z[2][3 * D + 8];     // k, q, beta rows of z_t by step parity (index = row)
    float pk[NW][2][D];        // per warp, by step parity: phi_k
    float u[NW][D];            // per warp: u of the current step
    uint64_t xbar[3];          // "chunk landed" barriers of the x ring
    // the current piece and the x ring's bookkeeping (kept here, not in
    // registers, which W fills)
    int b, h, t0, T;
    uint32_t phase;            // bit i: parity of the next completion awaited on x buffer i
    int issued, landed;        // chunks of the current piece
};

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float2 pair_lo(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 pair_hi(float4 v) { return make_float2(v.z, v.w); }

// Sum over the 32 lanes; every lane gets the same bits.
__device__ __forceinline__ float warp_allsum(float v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace d64r

// One step (see the file comment).  coef/coefb and the phi_k buffer of the
// previous step hold the pending update; on return they hold this step's.
template <int NLR, bool EMIT>
__device__ __forceinline__ void d64r_step(d64r::Smem& sm, const KParams& kp, int p, int t, int T, int tid, int lane,
                                          int warp, float2 (&w)[3][d64r::NP], float4& wb, float (&coef)[3],
                                          float& coefb)
{
    using namespace d64r;
    const float* zt = sm.z[t & 1];
    float* zn = sm.z[(t + 1) & 1];
    const float* xn = sm.xring[(t + 1) % (3 * TAU)];   // x~_{t+1} (unused past the piece's end)
    const float* pk_prev = sm.pk[warp][(t + 1) & 1];
    float* pk_cur = sm.pk[warp][t & 1];
    float* u_cur = sm.u[warp];
    const int bc = 4 * (tid & 15);   // beta columns of this thread

    // ---- 1. the softmaxes (every warp, all 64 entries: the step's chain)
    // beside the pending update of step t - 1 and b = W_{t-1} x~_{t+1}, which
    // do not depend on them
    float pk0, pk1, pq0, pq1;
    softmax64(zt[D + lane], zt[D + 32 + lane], pk0, pk1);
    softmax64(zt[2 * D + lane], zt[2 * D + 32 + lane], pq0, pq1);

    float2 bb[3];
    {
        float2 cc[3];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            cc[i] = make_float2(coef[i], coef[i]);
            bb[i] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < NP / 2; ++j) {
            const float4 p4 = lds4(pk_prev + 4 * j);
            const float4 x4 = lds4(xn + 4 * j);
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                w[i][2 * j] = __ffma2_rn(cc[i], pair_lo(p4), w[i][2 * j]);
                w[i][2 * j + 1] = __ffma2_rn(cc[i], pair_hi(p4), w[i][2 * j + 1]);
                bb[i] = __ffma2_rn(w[i][2 * j], pair_lo(x4), bb[i]);
                bb[i] = __ffma2_rn(w[i][2 * j + 1], pair_hi(x4), bb[i]);
            }
        }
    }
    float bbb;
    {
        const float4 p4 = lds4(pk_prev + bc);
        wb.x = fmaf(coefb, p4.x, wb.x);
        wb.y = fmaf(coefb, p4.y, wb.y);
        wb.z = fmaf(coefb, p4.z, wb.z);
        wb.w = fmaf(coefb, p4.w, wb.w);
        const float4 x4 = lds4(xn + bc);
        bbb = fmaf(wb.x, x4.x, fmaf(wb.y, x4.y, fmaf(wb.z, x4.z, wb.w * x4.w)));
    }

    // ---- 2. phi_k and u = phi(q) - phi(k) to the warp's buffers.  u takes an
    // explicit rounded subtraction: a contracted fma(e_q, 1/sum_q, -phi(k))
    // would skip phi(q)'s rounding, so equal k and q rows would no longer give
    // u = 0 exactly
    pk_cur[lane] = pk0;
    pk_cur[lane + 32] = pk1;
    u_cur[lane] = __fsub_rn(pq0, pk0);
    u_cur[lane + 32] = __fsub_rn(pq1, pk1);
    // backward record of step t: phi(k), u, gates, a (the rows' a follow below)
    float* em = nullptr;
    if constexpr (EMIT) {
        em = kp.emit + (static_cast<size_t>(p) * kp.T + sm.t0 + t) * kp.emit_stride;
        if (warp == 0) {
            em[lane] = pk0;
            em[lane + 32] = pk1;
            em[D + lane] = __fsub_rn(pq0, pk0);
            em[D + lane + 32] = __fsub_rn(pq1, pk1);
        }
    }
    const float sp = fmaf(pk0, xn[lane], pk1 * xn[lane + 32]);
    __syncwarp();

    // ---- 3. a = W_{t-1} u (the chain), s and the beta rows' sums beside it
    const float s = warp_allsum(sp);
    float abb;
    {
        const float4 u4 = lds4(u_cur + bc);
        abb = fmaf(wb.x, u4.x, fmaf(wb.y, u4.y, fmaf(wb.z, u4.z, wb.w * u4.w)));
    }
#pragma unroll
    for (int o = 1; o <= 8; o <<= 1) {
        abb += __shfl_xor_sync(0xffffffffu, abb, o);
        bbb += __shfl_xor_sync(0xffffffffu, bbb, o);
    }
    // two accumulators per row (even and odd column chunks): six independent
    // FMA chains instead of three
    float2 aa[3], ao[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) aa[i] = ao[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NP / 2; ++j) {
        const float4 u4 = lds4(u_cur + 4 * j);
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            float2& acc = (j & 1) ? ao[i] : aa[i];
            acc = __ffma2_rn(w[i][2 * j], pair_lo(u4), acc);
            acc = __ffma2_rn(w[i][2 * j + 1], pair_hi(u4), acc);
        }
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) aa[i] = make_float2(aa[i].x + ao[i].x, aa[i].y + ao[i].y);
    // ---- 4. gates and z_{t+1}
    const float4 beta = *reinterpret_cast<const float4*>(&zt[3 * D]);
    float g[4];
    if constexpr (NLR == 4) {
        g[0] = sigmoid_fast(beta.x);
        g[1] = sigmoid_fast(beta.y);
        g[2] = sigmoid_fast(beta.z);
        g[3] = sigmoid_fast(beta.w);
    } else {
        g[0] = g[1] = g[2] = g[3] = sigmoid_fast(beta.x);
    }
    float zr[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        coef[i] = g[NLR == 1 ? 0 : i] * (aa[i].x + aa[i].y);
        zr[i] = fmaf(coef[i], s, bb[i].x + bb[i].y);
    }
    if constexpr (EMIT) {
        float* ea = em + 2 * D + 4;
#pragma unroll
        for (int i = 0; i < 3; ++i) ea[D * i + tid] = aa[i].x + aa[i].y;
        if ((tid & 15) == 0 && (tid >> 4) < NLR) ea[3 * D + (tid >> 4)] = abb;
        if (tid < 4) em[2 * D + tid] = tid == 0 ? g[0] : tid == 1 ? g[1] : tid == 2 ? g[2] : g[3];
    }
    if (t + 1 < T) sm.yring[(t + 1) % (3 * TAU)][tid] = zr[0];
    zn[D + tid] = zr[1];
    zn[2 * D + tid] = zr[2];
    coefb = g[3] * abb;
    if ((tid & 15) == 0 && (tid >> 4) < NLR) zn[3 * D + (tid >> 4)] = fmaf(coefb, s, bbb);
}

template <int NLR, bool SMX, bool EMIT>
__global__ void __launch_bounds__(d64r::NT, 4)
    srwm_d64r_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                     const KParams kp)
{
    using namespace d64r;
    constexpr int M = 3 * D + NLR;
    constexpr uint32_t kChunkBytes = TAU * D * sizeof(float);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    if (!smem_base_ok(smem_raw, kp.status)) return;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int br = tid >> 4, bc = 4 * (tid & 15);   // this thread's beta row and columns
    const bool has_b = br < NLR;

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 3; ++i) mbar_init(&sm.xbar[i], 1);
        fence_mbar_init();
        if (kp.T > 0) {
            prefetch_tensormap(&tmx);
            prefetch_tensormap(&tmy);
        }
        sm.phase = 0;
        sm.issued = sm.landed = -1;
    }
    __syncthreads();

    // chunk c of the current piece (steps t0 + c*TAU ..) into x buffer c % 3 (one thread)
    auto issue = [&](int c) {
        if (c != kp.skip_chunk) {
            const int bi = c % 3;
            mbar_arrive_expect_tx(&sm.xbar[bi], kChunkBytes);
            tma_load_4d(&sm.xring[bi * TAU][0], &tmx, &sm.xbar[bi], 0, sm.h, sm.t0 + c * TAU, sm.b);
        }
        sm.issued = c;
    };
    // every thread waits for chunk c and the CTA agrees on the outcome; with
    // the input softmax, each warp then replaces half of its rows by x~
    auto land = [&](int c) -> bool {
        const int bi = c % 3;
        const bool ok = mbar_wait_bounded(&sm.xbar[bi], (sm.phase >> bi) & 1u, kp.wait_limit_ns);
        if (__syncthreads_or(!ok)) return false;
        if constexpr (SMX) {
#pragma unroll 4
            for (int r = warp; r < TAU; r += NW) {
                float* row = sm.xring[bi * TAU + r];
                float v0 = row[lane], v1 = row[lane + 32];
                softmax64(v0, v1, v0, v1);
                row[lane] = v0;
                row[lane + 32] = v1;
            }
            // the buffer is refilled by TMA later: order these writes first
            fence_proxy_async_smem();
        }
        __syncthreads();
        if (tid == 0) {
            sm.phase ^= 1u << bi;
            sm.landed = c;
        }
        return true;
    };

    int abort = 0;
    for (int item = blockIdx.x; item < kp.n_items; item += gridDim.x) {
        const int p = item % kp.n_streams, seg = item / kp.n_streams;
        // ---- the previous segment of this stream has to be finished
        if (seg > 0) {
            int fail = 0;
            if (tid == 0) fail = !wait_counter_bounded(kp.seg_done + p, seg, kp.wait_limit_ns);
            abort = __syncthreads_or(fail);
            if (abort) break;
        }
        if (tid == 0) {
            const int bb = p / kp.H;
            sm.b = bb;
            sm.h = p - bb * kp.H;
            sm.t0 = seg * kp.seg_len;
            sm.T = min(kp.seg_len, kp.T - seg * kp.seg_len);
            sm.issued = sm.landed = -1;
        }
        // no pending update before the first step: coef = 0 against a zero phi_k
        sm.pk[warp][1][lane] = 0.f;
        sm.pk[warp][1][lane + 32] = 0.f;
        __syncthreads();
        const int T = sm.T;
        const int nchunks = cdiv(T, TAU);

        // ---- W -> registers (W_init for a first segment, else the state the
        // previous segment left in W_out; read through L2)
        float2 w[3][NP];
        float4 wb = make_float4(0.f, 0.f, 0.f, 0.f);
        {
            const float* Ws = (seg == 0) ? kp.W_init + static_cast<size_t>(kp.w_per_seq ? p : sm.h) * M * D
                                         : kp.W_out + static_cast<size_t>(p) * M * D;
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const float4* row = reinterpret_cast<const float4*>(Ws + static_cast<size_t>(D * i + tid) * D);
#pragma unroll
                for (int j = 0; j < NP / 2; ++j) {
                    const float4 v = __ldcg(row + j);
                    w[i][2 * j] = pair_lo(v);
                    w[i][2 * j + 1] = pair_hi(v);
                }
            }
            if (has_b) wb = __ldcg(reinterpret_cast<const float4*>(Ws + static_cast<size_t>(3 * D + br) * D + bc));
        }

        if (T > 0) {
            if (tid == 0) {
                issue(0);
                if (nchunks > 1) issue(1);
            }
            abort = !land(0);
        }

        // ---- prologue: z_0 = W x~_0 (y of the piece's first step)
        if (!abort && T > 0) {
            const float* x0 = sm.xring[0];
            float2 acc[3];
#pragma unroll
            for (int i = 0; i < 3; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < NP / 2; ++j) {
                const float4 x4 = lds4(x0 + 4 * j);
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    acc[i] = __ffma2_rn(w[i][2 * j], pair_lo(x4), acc[i]);
                    acc[i] = __ffma2_rn(w[i][2 * j + 1], pair_hi(x4), acc[i]);
                }
            }
            const float4 x4 = lds4(x0 + bc);
            float zb = fmaf(wb.x, x4.x, fmaf(wb.y, x4.y, fmaf(wb.z, x4.z, wb.w * x4.w)));
#pragma unroll
            for (int o = 1; o <= 8; o <<= 1) zb += __shfl_xor_sync(0xffffffffu, zb, o);
            sm.yring[0][tid] = acc[0].x + acc[0].y;
            sm.z[0][D + tid] = acc[1].x + acc[1].y;
            sm.z[0][2 * D + tid] = acc[2].x + acc[2].y;
            if ((tid & 15) == 0 && has_b) sm.z[0][3 * D + br] = zb;
        }
        __syncthreads();

        // the pending rank-one update (applied in the next step's pass)
        float coef[3] = {0.f, 0.f, 0.f};
        float coefb = 0.f;

        for (int c = 0; c < nchunks && !abort; ++c) {
            // ---- chunk boundary.  The last step of chunk c reads x~ of the
            // first step of chunk c + 1 (issued a chunk ago); chunk c + 2 goes
            // into the buffer of chunk c - 1, whose last row was read before
            // here.  y of chunk c - 1 is complete: out by TMA.
            if (c + 1 < nchunks && !land(c + 1)) {
                abort = 1;
                break;
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                if (c + 2 < nchunks) issue(c + 2);
                if (c > 0) {
                    tma_store_4d(&tmy, &sm.yring[((c - 1) % 3) * TAU][0], 0, sm.h, sm.t0 + (c - 1) * TAU, sm.b);
                    bulk_commit();
                    // the store before it has finished reading the buffer that
                    // steps of chunk c + 1 write
                    bulk_wait_read<1>();
                }
            }
            // the chunk's last step stands apart from the loop over the others:
            // measured 1.07 -> 1.03 ms on mid against one loop over all steps
            // (same results bit for bit; only the compiled schedule differs)
            const int t_end = min(T, (c + 1) * TAU);
            for (int t = c * TAU; t < t_end - 1; ++t) {
                d64r_step<NLR, EMIT>(sm, kp, p, t, T, tid, lane, warp, w, wb, coef, coefb);
                __syncthreads();
            }
            d64r_step<NLR, EMIT>(sm, kp, p, t_end - 1, T, tid, lane, warp, w, wb, coef, coefb);
            __syncthreads();
        }

        // ---- the last chunk's y, then drain this piece's stores
        if (!abort && T > 0) {
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                const int c = nchunks - 1;
                tma_store_4d(&tmy, &sm.yring[(c % 3) * TAU][0], 0, sm.h, sm.t0 + c * TAU, sm.b);
                bulk_commit();
            }
        }
        if (tid == 0) bulk_wait_all<0>();
        if (abort) break;

        // ---- the last pending update, then the state -> W_out[b, h]
        float* Wd = kp.W_out + static_cast<size_t>(p) * M * D;
        const float* pk_last = sm.pk[warp][(T + 1) & 1];   // phi_k of step T-1 (zero when T = 0)
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            float4* row = reinterpret_cast<float4*>(Wd + static_cast<size_t>(D * i + tid) * D);
            const float2 cc = make_float2(coef[i], coef[i]);
#pragma unroll
            for (int j = 0; j < NP / 2; ++j) {
                const float4 p4 = lds4(pk_last + 4 * j);
                const float2 lo = __ffma2_rn(cc, pair_lo(p4), w[i][2 * j]);
                const float2 hi = __ffma2_rn(cc, pair_hi(p4), w[i][2 * j + 1]);
                row[j] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
        if (has_b) {
            const float4 p4 = lds4(pk_last + bc);
            *reinterpret_cast<float4*>(Wd + static_cast<size_t>(3 * D + br) * D + bc) =
                make_float4(fmaf(coefb, p4.x, wb.x), fmaf(coefb, p4.y, wb.y), fmaf(coefb, p4.z, wb.z),
                            fmaf(coefb, p4.w, wb.w));
        }
        __syncthreads();   // the state is stored; shared memory is free for the next item
        if (kp.seg_done != nullptr && tid == 0) {
            __threadfence();
            st_release_gpu(kp.seg_done + p, seg + 1);
        }
    }

    if (abort) {
        if (tid == 0) {
            // every load still in flight lands before the CTA gives up its shared memory
            for (int c = sm.landed + 1; c <= sm.issued; ++c) {
                if (c == kp.skip_chunk) continue;
                const int bi = c % 3;
                mbar_wait_bounded(&sm.xbar[bi], (sm.phase >> bi) & 1u, kp.wait_limit_ns);
                sm.phase ^= 1u << bi;
            }
            atomicOr(kp.status, kStatusTimeout);
        }
    }
}

template <int NLR, bool SMX, bool EMIT = false>
LaunchInfo launch_info_d64r_impl()
{
    return LaunchInfo{reinterpret_cast<const void*>(&srwm_d64r_kernel<NLR, SMX, EMIT>), d64r::NT, 1,
                      static_cast<int>(sizeof(d64r::Smem)) + 128, d64r::TAU};
}

}  // namespace srwm
