// srwm_d64w2.cuh -- the d = 64 kernel for many streams: one (sequence, head)
// stream per CTA of two warps, four CTAs per SM.
//
// Math (per step t; "Metalearning Continual Learning Algorithms", section 2.3,
// Eqs. (1)-(3), four-rate version Eqs. (4)-(5)), as in the four-warp kernel:
//   phi_k = softmax(k_t), phi_q = softmax(q_t), g = sigmoid(beta_t) per block
//   a_r   = W_{t-1}[r,:] . (phi_q - phi_k)
//   W_t[r,:] = W_{t-1}[r,:] + g_r a_r phi_k
//   z_{t+1,r} = b_r + g_r a_r (phi_k . x~_{t+1}),  b_r = W_{t-1}[r,:] . x~_{t+1}
//
// Why two warps: the per-step work that does not scale with the rows a warp
// holds (the softmaxes, the exchange of z through shared memory, the barrier)
// is paid once per warp.  Two warps per stream, each thread holding 6 rows of
// 32 columns (192 registers of W), halve that overhead per stream-step and fit
// four streams' states into one SM's register file.
//
// Layout.  Thread (rg = tid/2, cg = tid%2) holds rows rg + 32 i (i < 6: slots
// 0-1 y, 2-3 k, 4-5 q) over the columns of float4 chunks cg + 2 j (j < 8),
// kept as float2 pairs for the two-wide FMA; a row's dot product finishes
// with one xor shuffle.  The n_lr beta rows are spread four columns per
// thread: thread tid holds beta row tid/16, columns 4 (tid%16) .. +3 (threads
// whose row is >= n_lr hold zeros), and their dots finish over 16 lanes.
// Operand vectors (x~, phi_k, u) are read from shared memory one float4 chunk
// at a time, and the loop state of the item lives in shared memory, so that
// W and little else stays resident in the 255 registers.
//
// One step:
//   1. the pending rank-one update of the previous step (two-wide FMAs with
//      the coefficient duplicated into a pair); meanwhile phi_k, phi_q of z_t
//      in the lane layout (entries lane, lane + 32);
//   2. phi_k and u = phi_q - phi_k go to the warp's own buffer (by step
//      parity); s = phi_k . x~_{t+1} as a warp sum;
//   3. a-dots against u and b-dots against x~_{t+1}, reductions, gates;
//      z_{t+1} to shared memory (y rows to the TMA staging buffer);
//   4. barrier.
// Without the input softmax, x~ = x is read straight from the TMA ring, so no
// warp stages it on the way to the barrier, and the steps run chunk by chunk:
// the tight inner loop holds only the step and its barrier, while the chunk
// boundary (bounded wait for the next chunk, agreed on by the CTA through
// __syncthreads_or, the next TMA load, the y store) runs between chunks.
// Keeping loop state out of the inner loop matters here: W fills 192 of the
// 255 registers, and every value live across the loop competes with the
// step's temporaries (measured: 1.64 -> 1.43 ms on the mid workload).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "srwm_common.h"
#include "srwm_ptx.cuh"

namespace srwm {

namespace d64w2 {

constexpr int D = 64;
constexpr int TAU = 32;     // steps per TMA chunk
constexpr int NW = 2;       // warps per stream
constexpr int NT = 32 * NW;
constexpr int SL = 6;       // row slots per thread
constexpr int NCH = 8;      // float4 column chunks per thread
constexpr int XW = NW - 1;  // warp staging x~ and driving the x TMA ring

struct __align__(128) Smem {
    float xring[2][TAU][D];    // TMA destination: raw x, two chunks
    float ystage[3][TAU][D];   // TMA source: y, three chunks
    float z[2][D * 3 + 8];     // k, q, beta rows of z_t by step parity (index = row)
    float xs[2][D];            // x~_{t+1}, x~_{t+2}
    float pu[NW][2][2][D];     // per warp, by step parity: phi_k, u
    uint64_t xbar[2];          // "chunk landed" barriers of the x ring
    // the current item and the x ring's bookkeeping (kept here, not in
    // registers, which W fills)
    int b, h, t0, T;
    uint32_t used[2];          // completed phases of the two x buffers
    int issued, landed;        // chunks of the current item
};

__device__ __forceinline__ float4 ld4s(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }

// Sum over the 32 lanes; every lane gets the same bits.
__device__ __forceinline__ float warp_allsum(float v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace d64w2

// One step (see the file comment).  coef/coefb and the phi_k buffer of the
// previous step hold the pending update; on return they hold this step's.
template <int NLR>
__device__ __forceinline__ void d64w2_step(d64w2::Smem& sm, int t, int T, int lane, int warp, int tid, int rg,
                                           int cg, float2 (&w)[d64w2::SL][2 * d64w2::NCH], float4& wb,
                                           float (&coef)[d64w2::SL], float& coefb, const float* xn)
{
    using namespace d64w2;
    const float* zt = sm.z[t & 1];
    float* zn = sm.z[(t + 1) & 1];
    const float* pk_prev = sm.pu[warp][(t + 1) & 1][0];
    float* pk_cur = sm.pu[warp][t & 1][0];
    float* u_cur = sm.pu[warp][t & 1][1];
    const int bc = 4 * (tid & 15);   // beta columns of this thread

    // ---- 1. pending update || softmax
    const float k0 = zt[D + lane], k1 = zt[D + 32 + lane];
    const float q0 = zt[2 * D + lane], q1 = zt[2 * D + 32 + lane];

#pragma unroll
    for (int j = 0; j < NCH; ++j) {
        const float4 p4 = ld4s(pk_prev + 4 * (cg + 2 * j));
#pragma unroll
        for (int i = 0; i < SL; ++i) {
            const float2 cc = make_float2(coef[i], coef[i]);
            w[i][2 * j] = __ffma2_rn(cc, lo2(p4), w[i][2 * j]);
            w[i][2 * j + 1] = __ffma2_rn(cc, hi2(p4), w[i][2 * j + 1]);
        }
    }
    {
        const float4 p4 = ld4s(pk_prev + bc);
        wb.x = fmaf(coefb, p4.x, wb.x);
        wb.y = fmaf(coefb, p4.y, wb.y);
        wb.z = fmaf(coefb, p4.z, wb.z);
        wb.w = fmaf(coefb, p4.w, wb.w);
    }

    float pk0, pk1, pq0, pq1;
    softmax64(k0, k1, pk0, pk1);
    softmax64(q0, q1, pq0, pq1);
    // ---- 2. phi_k, u -> the warp's buffer; s = phi_k . x~_{t+1}
    pk_cur[lane] = pk0;
    pk_cur[lane + 32] = pk1;
    // u = phi(q) - phi(k) with an explicit rounded subtraction: a contracted
    // fma(e_q, 1/sum_q, -phi(k)) would skip phi(q)'s rounding, so equal k and
    // q rows would no longer give u = 0 exactly
    u_cur[lane] = __fsub_rn(pq0, pk0);
    u_cur[lane + 32] = __fsub_rn(pq1, pk1);
    const float s = warp_allsum(fmaf(pk0, xn[lane], pk1 * xn[lane + 32]));
    __syncwarp();

    // ---- 3. a-dots, b-dots
    float2 acca[SL], accb[SL];
#pragma unroll
    for (int i = 0; i < SL; ++i) acca[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
        const float4 u4 = ld4s(u_cur + 4 * (cg + 2 * j));
#pragma unroll
        for (int i = 0; i < SL; ++i) {
            acca[i] = __ffma2_rn(w[i][2 * j], lo2(u4), acca[i]);
            acca[i] = __ffma2_rn(w[i][2 * j + 1], hi2(u4), acca[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < SL; ++i) accb[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
        const float4 x4 = ld4s(xn + 4 * (cg + 2 * j));
#pragma unroll
        for (int i = 0; i < SL; ++i) {
            accb[i] = __ffma2_rn(w[i][2 * j], lo2(x4), accb[i]);
            accb[i] = __ffma2_rn(w[i][2 * j + 1], hi2(x4), accb[i]);
        }
    }
    float abb, bbb;
    {
        const float4 u4 = ld4s(u_cur + bc);
        const float4 x4 = ld4s(xn + bc);
        abb = fmaf(wb.x, u4.x, fmaf(wb.y, u4.y, fmaf(wb.z, u4.z, wb.w * u4.w)));
        bbb = fmaf(wb.x, x4.x, fmaf(wb.y, x4.y, fmaf(wb.z, x4.z, wb.w * x4.w)));
    }
    float a[SL], bb[SL];
#pragma unroll
    for (int i = 0; i < SL; ++i) {
        a[i] = acca[i].x + acca[i].y;
        bb[i] = accb[i].x + accb[i].y;
    }
#pragma unroll
    for (int i = 0; i < SL; ++i) {
        a[i] += __shfl_xor_sync(0xffffffffu, a[i], 1);
        bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], 1);
    }
#pragma unroll
    for (int o = 1; o <= 8; o <<= 1) {
        abb += __shfl_xor_sync(0xffffffffu, abb, o);
        bbb += __shfl_xor_sync(0xffffffffu, bbb, o);
    }

    // gates, needed only from here on
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

    // ---- z_{t+1}: slot i is stored by the lane with cg == i % 2
    const bool write_y = (t + 1 < T);
    float* yrow = sm.ystage[((t + 1) / TAU) % 3][(t + 1) % TAU];
#pragma unroll
    for (int i = 0; i < SL; ++i) {
        const int blk = (NLR == 1) ? 0 : i / 2;
        coef[i] = g[blk] * a[i];
        const float zr = fmaf(coef[i], s, bb[i]);
        if ((i & 1) == cg) {
            if (i < 2) {
                if (write_y) yrow[rg + 32 * i] = zr;
            } else {
                zn[rg + 32 * i] = zr;
            }
        }
    }
    coefb = g[3] * abb;
    if ((tid & 15) == 0 && (tid >> 4) < NLR) zn[3 * D + (tid >> 4)] = fmaf(coefb, s, bbb);
    if (write_y && ((t + 2) % TAU == 0 || t + 2 == T)) fence_proxy_async_smem();
}

// Issues the TMA load of chunk c of the current item into buffer c & 1 (one warp).
__device__ __forceinline__ void srwm_d64w2_issue(d64w2::Smem& sm, const CUtensorMap& tmx, const KParams& kp,
                                                 int lane, int c)
{
    using namespace d64w2;
    if (lane == 0) {
        if (c != kp.skip_chunk) {
            mbar_arrive_expect_tx(&sm.xbar[c & 1], TAU * D * sizeof(float));
            tma_load_4d(&sm.xring[c & 1][0][0], &tmx, &sm.xbar[c & 1], 0, sm.h, sm.t0 + c * TAU, sm.b);
        }
        sm.issued = c;
    }
}

// x~ of item step tn (zero past the end) -> dst, one warp.
template <bool SMX>
__device__ __forceinline__ void srwm_d64w2_stage(d64w2::Smem& sm, int tn, int T, int lane, float* dst)
{
    using namespace d64w2;
    float v0 = 0.f, v1 = 0.f;
    if (tn < T) {
        const float* src = sm.xring[(tn / TAU) & 1][tn % TAU];
        v0 = src[lane];
        v1 = src[lane + 32];
        if constexpr (SMX) softmax64(v0, v1, v0, v1);
    }
    dst[lane] = v0;
    dst[lane + 32] = v1;
}

// x~_{tn} -> xs[tn & 1] for the step after next; at a chunk boundary waits
// (bounded) for the chunk and issues the one after it.  Returns 1 when the
// wait ran out.  One warp.
template <bool SMX>
__device__ __forceinline__ int srwm_d64w2_next_x(d64w2::Smem& sm, const CUtensorMap& tmx, const KParams& kp,
                                                int lane, int tn, int T)
{
    using namespace d64w2;
    if (tn < T && tn % TAU == 0) {
        const int c = tn / TAU;
        const bool ok = mbar_wait_bounded(&sm.xbar[c & 1], (sm.used[c & 1] + (c >> 1)) & 1, kp.wait_limit_ns);
        if (!__all_sync(0xffffffffu, ok)) return 1;
        __syncwarp();
        if (lane == 0) sm.landed = c;
        if (c + 1 < cdiv(T, TAU)) srwm_d64w2_issue(sm, tmx, kp, lane, c + 1);
    }
    srwm_d64w2_stage<SMX>(sm, tn, T, lane, sm.xs[tn & 1]);
    return 0;
}

template <int NLR, bool SMX>
__global__ void __launch_bounds__(d64w2::NT, 4)
    srwm_d64w2_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                      const KParams kp)
{
    using namespace d64w2;
    constexpr int M = 3 * D + NLR;
    constexpr uint32_t kChunkBytes = TAU * D * sizeof(float);
    extern __shared__ unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = tid >> 1, cg = tid & 1;
    const int br = tid >> 4, bc = 4 * (tid & 15);   // this thread's beta row and columns
    const bool has_b = br < NLR;

    if (tid == 0) {
        mbar_init(&sm.xbar[0], 1);
        mbar_init(&sm.xbar[1], 1);
        fence_mbar_init();
        if (kp.T > 0) {
            prefetch_tensormap(&tmx);
            prefetch_tensormap(&tmy);
        }
    }
    __syncthreads();

    if (tid == 0) {
        sm.used[0] = sm.used[1] = 0;
        sm.issued = sm.landed = -1;
    }
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
        sm.pu[warp][1][0][lane] = 0.f;
        sm.pu[warp][1][0][lane + 32] = 0.f;
        __syncthreads();
        const int T = sm.T;

        // ---- W -> registers (W_init for a first segment, else the state the
        // previous segment left in W_out; read through L2)
        float2 w[SL][2 * NCH];
        float4 wb = make_float4(0.f, 0.f, 0.f, 0.f);
        {
            const float* Ws = (seg == 0) ? kp.W_init + static_cast<size_t>(kp.w_per_seq ? p : sm.h) * M * D
                                         : kp.W_out + static_cast<size_t>(p) * M * D;
#pragma unroll
            for (int i = 0; i < SL; ++i) {
                const float* row = Ws + static_cast<size_t>(rg + 32 * i) * D;
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(row + 4 * (cg + 2 * j)));
                    w[i][2 * j] = lo2(v);
                    w[i][2 * j + 1] = hi2(v);
                }
            }
            if (has_b) wb = __ldcg(reinterpret_cast<const float4*>(Ws + static_cast<size_t>(3 * D + br) * D + bc));
        }

        int fail = 0;
        if (warp == XW && T > 0) {
            srwm_d64w2_issue(sm, tmx, kp, lane, 0);
            if (T > TAU) srwm_d64w2_issue(sm, tmx, kp, lane, 1);
            if (__all_sync(0xffffffffu, mbar_wait_bounded(&sm.xbar[0], sm.used[0] & 1, kp.wait_limit_ns))) {
                if (lane == 0) sm.landed = 0;
                if constexpr (SMX) {
                    srwm_d64w2_stage<SMX>(sm, 0, T, lane, sm.xs[0]);
                    srwm_d64w2_stage<SMX>(sm, 1, T, lane, sm.xs[1]);
                }
            } else {
                fail = 1;
            }
            __syncwarp();
        }
        abort = __syncthreads_or(fail);

        // ---- prologue: z_0 = W x~_0 (y of the item's first step)
        if (!abort && T > 0) {
            const float* x0 = SMX ? sm.xs[0] : sm.xring[0][0];
            float2 acc[SL];
#pragma unroll
            for (int i = 0; i < SL; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
                const float4 x4 = ld4s(x0 + 4 * (cg + 2 * j));
#pragma unroll
                for (int i = 0; i < SL; ++i) {
                    acc[i] = __ffma2_rn(w[i][2 * j], lo2(x4), acc[i]);
                    acc[i] = __ffma2_rn(w[i][2 * j + 1], hi2(x4), acc[i]);
                }
            }
            const float4 x4 = ld4s(x0 + bc);
            float zb = fmaf(wb.x, x4.x, fmaf(wb.y, x4.y, fmaf(wb.z, x4.z, wb.w * x4.w)));
            float bb[SL];
#pragma unroll
            for (int i = 0; i < SL; ++i) {
                bb[i] = acc[i].x + acc[i].y;
                bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], 1);
            }
#pragma unroll
            for (int o = 1; o <= 8; o <<= 1) zb += __shfl_xor_sync(0xffffffffu, zb, o);
#pragma unroll
            for (int i = 0; i < SL; ++i) {
                if ((i & 1) != cg) continue;
                if (i < 2) sm.ystage[0][0][rg + 32 * i] = bb[i];
                else sm.z[0][rg + 32 * i] = bb[i];
            }
            if ((tid & 15) == 0 && has_b) sm.z[0][3 * D + br] = zb;
            fence_proxy_async_smem();
        }
        __syncthreads();

        // the pending rank-one update (applied at the start of the next step)
        float coef[SL];
#pragma unroll
        for (int i = 0; i < SL; ++i) coef[i] = 0.f;
        float coefb = 0.f;

        if constexpr (!SMX) {
            // x~ = x is read straight from the ring.  Steps go chunk by chunk:
            // the inner loop runs the steps whose x~_{t+1} lies in the
            // current chunk, and the chunk-boundary work (the y store, the
            // wait for the next chunk, the next TMA load) sits between
            // chunks, outside the tight loop.
            for (int c0 = 0; c0 < T && !abort; c0 += TAU) {
                const int tend = min(c0 + TAU, T);
                for (int t = c0; t < tend - 1; ++t) {
                    d64w2_step<NLR>(sm, t, T, lane, warp, tid, rg, cg, w, wb, coef, coefb,
                                    sm.xring[(c0 / TAU) & 1][t + 1 - c0]);
                    __syncthreads();
                }
                const int t = tend - 1;
                const float* xn = sm.xring[(c0 / TAU) & 1][0];   // unused past the end of the item
                if (tend < T) {
                    // chunk c = tend / TAU is needed from the next step on: every
                    // warp waits for it and the CTA agrees on the outcome; then
                    // warp XW refills the other buffer (its chunk c-1 was last
                    // read in the step before this one, before the barrier)
                    const int c = tend / TAU;
                    const bool ok =
                        mbar_wait_bounded(&sm.xbar[c & 1], (sm.used[c & 1] + (c >> 1)) & 1, kp.wait_limit_ns);
                    if (__syncthreads_or(!ok)) {
                        abort = 1;
                        break;
                    }
                    if (warp == XW) {
                        if (lane == 0) sm.landed = c;
                        if (c + 1 < cdiv(T, TAU)) srwm_d64w2_issue(sm, tmx, kp, lane, c + 1);
                    }
                    xn = sm.xring[c & 1][0];
                }
                d64w2_step<NLR>(sm, t, T, lane, warp, tid, rg, cg, w, wb, coef, coefb, xn);
                __syncthreads();
                // y of the chunk's steps complete -> TMA store
                if (warp == 0 && lane == 0 && tend % TAU == 0) {
                    const int cs = c0 / TAU;
                    tma_store_4d(&tmy, &sm.ystage[cs % 3][0][0], 0, sm.h, sm.t0 + c0, sm.b);
                    bulk_commit();
                    bulk_wait_read<1>();
                }
            }
        } else {
            for (int t = 0; t < T && !abort; ++t) {   // abort is uniform: set by __syncthreads_or
                // y chunk holding y_t complete -> TMA store
                if (warp == 0 && lane == 0 && (t + 1) % TAU == 0) {
                    const int c = t / TAU;
                    tma_store_4d(&tmy, &sm.ystage[c % 3][0][0], 0, sm.h, sm.t0 + c * TAU, sm.b);
                    bulk_commit();
                    bulk_wait_read<1>();
                }
                d64w2_step<NLR>(sm, t, T, lane, warp, tid, rg, cg, w, wb, coef, coefb, sm.xs[(t + 1) & 1]);
                // x~_{t+2} -> xs[t & 1]; at a chunk boundary the chunk has to
                // land first, and the CTA agrees on whether it did
                fail = 0;
                if (warp == XW) fail = srwm_d64w2_next_x<SMX>(sm, tmx, kp, lane, t + 2, T);
                if ((t + 2) % TAU == 0) {
                    if (__syncthreads_or(fail)) {
                        abort = 1;
                        break;
                    }
                } else {
                    __syncthreads();
                }
            }
        }
        // ---- drain this item's y stores
        if (warp == 0 && lane == 0) {
            if (!abort && T > 0 && T % TAU != 0) {
                const int c = (T - 1) / TAU;
                tma_store_4d(&tmy, &sm.ystage[c % 3][0][0], 0, sm.h, sm.t0 + c * TAU, sm.b);
                bulk_commit();
            }
            bulk_wait_all<0>();
        }
        if (abort) break;

        // ---- the last pending update, then the state -> W_out[b, h]
        float* Wd = kp.W_out + static_cast<size_t>(p) * M * D;
        const float* pk_last = sm.pu[warp][(T + 1) & 1][0];   // phi_k of step T-1 (zero when T = 0)
#pragma unroll
        for (int i = 0; i < SL; ++i) {
            float* row = Wd + static_cast<size_t>(rg + 32 * i) * D;
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
                const float4 p4 = ld4s(pk_last + 4 * (cg + 2 * j));
                const float2 cc = make_float2(coef[i], coef[i]);
                const float2 lo = __ffma2_rn(cc, lo2(p4), w[i][2 * j]);
                const float2 hi = __ffma2_rn(cc, hi2(p4), w[i][2 * j + 1]);
                *reinterpret_cast<float4*>(row + 4 * (cg + 2 * j)) = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
        if (has_b) {
            const float4 p4 = ld4s(pk_last + bc);
            *reinterpret_cast<float4*>(Wd + static_cast<size_t>(3 * D + br) * D + bc) =
                make_float4(fmaf(coefb, p4.x, wb.x), fmaf(coefb, p4.y, wb.y), fmaf(coefb, p4.z, wb.z),
                            fmaf(coefb, p4.w, wb.w));
        }
        if (tid == 0) {
            const int nchunks = cdiv(T, TAU);
            sm.used[0] += (nchunks + 1) / 2;
            sm.used[1] += nchunks / 2;
        }
        __syncthreads();   // the state is stored; shared memory is free for the next item
        if (kp.seg_done != nullptr && tid == 0) {
            __threadfence();
            st_release_gpu(kp.seg_done + p, seg + 1);
        }
    }

    if (abort) {
        if (warp == XW) {
            // every load still in flight lands before the CTA gives up its shared memory
            for (int c = sm.landed + 1; c <= sm.issued; ++c) {
                if (c == kp.skip_chunk) continue;
                mbar_wait_bounded(&sm.xbar[c & 1], (sm.used[c & 1] + (c >> 1)) & 1, kp.wait_limit_ns);
            }
        }
        if (tid == 0) atomicOr(kp.status, kStatusTimeout);
    }
}

template <int NLR, bool SMX>
LaunchInfo launch_info_d64w2_impl()
{
    return LaunchInfo{reinterpret_cast<const void*>(&srwm_d64w2_kernel<NLR, SMX>), d64w2::NT, 1,
                      static_cast<int>(sizeof(d64w2::Smem)) + 128, d64w2::TAU};
}

}  // namespace srwm
