// srwm_d64.cuh -- the d = 64 kernel: one (sequence, head) stream per CTA of
// four warps, two CTAs per SM.
//
// Math (per step t; "Metalearning Continual Learning Algorithms", section 2.3,
// Eqs. (1)-(3), four-rate version Eqs. (4)-(5)):
//   phi_k = softmax(k_t), phi_q = softmax(q_t), g = sigmoid(beta_t) per block
//   a_r   = W_{t-1}[r,:] . (phi_q - phi_k)                 (Eq. (2), both reads fused)
//   W_t[r,:] = W_{t-1}[r,:] + g_r a_r phi_k                 (Eq. (3) / (5))
//   z_{t+1,r} = W_t[r,:] . x~_{t+1} = b_r + g_r a_r (phi_k . x~_{t+1}),
//               b_r = W_{t-1}[r,:] . x~_{t+1}               (Eq. (1) of step t+1)
// so y_{t+1} = z_{t+1}[0:64] is still read from the pre-update matrix of its
// own step (W_t).
//
// Layout.  A stream has NW warps (4, or 8 when there are fewer streams than
// SMs and a stream should use a whole SM), i.e. RG = 8 NW row groups.  Thread
// (rg = tid/4, cg = tid%4) holds rows rg + RG i (i < 192/RG: blocks y, k, q in
// order) and, in warp 0, row 192 + rg (beta rows, valid for rg < n_lr), over
// the 16 columns of float4 chunks cg, cg+4, cg+8, cg+12, kept as float2 pairs
// for the two-wide FMA.  W never leaves registers.
//
// One step, one CTA barrier:
//   1. every warp computes phi_k, phi_q and the gates from z_t in shared
//      memory (redux max, exp, fixed-point redux sum, approximate reciprocal);
//      beside them, the work that does not depend on them: the y rows' a of
//      step t-1, their gate product and y_t (the y rows never feed the
//      recurrence, so they run one step behind), the previous step's rank-one
//      update of every row, b_r = W_{t-1}[r,:] . x~_{t+1} and its sum over the
//      four column groups;
//   2. phi_k and u = phi_q - phi_k go through a warp-private shared buffer
//      into the thread's column layout;
//   3. a_r of the k, q and beta rows and the partial phi_k . x~_{t+1}; two
//      xor-shuffle levels finish them; owner lanes store z_{t+1} of those rows;
//   4. barrier.
// So the step's chain is z_t -> softmaxes -> u -> a of the k, q and beta rows
// -> z_{t+1} -> barrier.
// z is double-buffered by step parity (a fast warp writes z_{t+1} while a slow
// one still reads z_t); y staging is triple-buffered (one chunk being written,
// up to two still read by bulk stores).
// Without the input softmax x~ = x is read straight from a three-chunk TMA
// ring, and the steps run chunk by chunk: the chunk boundary (wait for the
// next chunk, issue the one after, store the previous chunk's y) sits at the
// start of each chunk, outside the step loop.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "srwm_common.h"
#include "srwm_ptx.cuh"

namespace srwm {

namespace d64 {

constexpr int D = 64;
constexpr int TAU = 32;     // steps per TMA chunk
constexpr int NP = 8;       // float2 column pairs per thread

// NW warps per stream: RG row groups, SLOTS row slots of every thread (rows
// 0..191), one more slot in warp 0 for the beta rows.
template <int NW_>
struct Cfg {
    static constexpr int NW = NW_;
    static constexpr int NT = 32 * NW;
    static constexpr int RG = 8 * NW;
    static constexpr int SLOTS = 3 * D / RG;
    static constexpr int XW = NW - 1;   // warp staging x~ and driving the x TMA ring
    static_assert(NW == 4 || NW == 8, "4 or 8 warps per stream");
    // row block (0 y, 1 k, 2 q) of slot i
    SRWM_HD static constexpr int block_of_slot(int i) { return (RG * i) / D; }
};

template <int NW>
struct __align__(128) Smem {
    float xring[3][TAU][D];    // TMA destination: raw x, three chunks
    float ystage[3][TAU][D];   // TMA source: y, three chunks
    float z[2][D * 3 + 8];     // k, q, beta rows of z_t by step parity (index = row)
    float xs[2][D];            // x~_{t+1}, x~_{t+2}
    float pkq[NW][2][D];       // per warp: phi_k, phi_q in plain column order
    uint64_t xbar[3];          // "chunk landed" barriers of the x ring
};

__device__ __forceinline__ void load_pairs(const float* base, int cg, float2 (&out)[NP])
{
#pragma unroll
    for (int j = 0; j < NP / 2; ++j) {
        const float4 v = *reinterpret_cast<const float4*>(base + 4 * (cg + 4 * j));
        out[2 * j] = make_float2(v.x, v.y);
        out[2 * j + 1] = make_float2(v.z, v.w);
    }
}

}  // namespace d64

// The thread's state between steps, besides its W tile:
//   coef[i]  g a of the pending update of step t-1 for slot i (the y slots'
//            values are formed at the start of step t, see below);
//   pkc      phi_k of step t-1 in the thread's column layout;
//   u2       u of step t-1 in the column layout (for the y slots' a);
//   yb       b of the two y slots for y_t (summed over the four column groups);
//   ys, gy   s = phi_k . x~_t and the y block's gate, both of step t-1.
template <int NW>
struct D64Carry {
    float2 pkc[d64::NP];
    float2 u2[d64::NP];
    float yb[2];
    float ys, gy;
};

// One step of the recurrence for a warp whose threads carry NS row slots
// (slots i < SLOTS: rows rg + RG i; slot SLOTS: beta row 192 + rg).  The y
// rows (slots 0 and 1) never feed the recurrence, so their work runs one step
// behind, off the step's chain: at step t the thread forms a^y of step t-1,
// writes y_t, applies the y rows' update of step t-1 and forms their b for
// y_{t+1}.  The chain itself is: z_t -> softmaxes -> u -> a of the k, q and
// beta rows -> z_{t+1} -> barrier.
template <int NW, int NS, int NLR, bool EMIT = false>
__device__ __forceinline__ void d64_step(d64::Smem<NW>& sm, int t, int T, int lane, int warp, int rg, int cg,
                                         float2 (&w)[d64::Cfg<NW>::SLOTS + 1][d64::NP],
                                         float (&coef)[d64::Cfg<NW>::SLOTS + 1], D64Carry<NW>& cy,
                                         const float* xn, float* em = nullptr, float* em_prev = nullptr)
{
    using namespace d64;
    using C = Cfg<NW>;
    constexpr int SLOTS = C::SLOTS, RG = C::RG;
    constexpr int M = 3 * D + NLR;
    static_assert(C::block_of_slot(0) == 0 && C::block_of_slot(1) == 0 && C::block_of_slot(2) != 0,
                  "slots 0 and 1 are the y rows");
    const float* zt = sm.z[t & 1];
    float* zn = sm.z[(t + 1) & 1];

    // ---- 1. the softmaxes and gates (the chain), and beside them the work
    // that does not depend on them
    const float k0 = zt[D + lane], k1 = zt[D + 32 + lane];
    const float q0 = zt[2 * D + lane], q1 = zt[2 * D + 32 + lane];
    const float4 beta = *reinterpret_cast<const float4*>(&zt[3 * D]);
    float pk0, pk1, pq0, pq1;
    softmax64(k0, k1, pk0, pk1);
    softmax64(q0, q1, pq0, pq1);
    float g[4];
    if constexpr (NLR == 4) {
        g[0] = sigmoid_fast(beta.x);
        g[1] = sigmoid_fast(beta.y);
        g[2] = sigmoid_fast(beta.z);
        g[3] = sigmoid_fast(beta.w);
    } else {
        g[0] = g[1] = g[2] = g[3] = sigmoid_fast(beta.x);
    }

    // the y rows, one step behind: a^y of step t-1 on W^y_{t-2} (which has not
    // yet taken step t-1's update), its gate product, and y_t.  At t = 0 the
    // carried u and gate are zero, so coef stays 0, and y_0 came from the
    // prologue: only the stores are predicated, the rest runs branch-free.
    {
        float ay[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NP; ++q) acc = __ffma2_rn(w[i][q], cy.u2[q], acc);
            ay[i] = acc.x + acc.y;
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
#pragma unroll
            for (int i = 0; i < 2; ++i) ay[i] += __shfl_xor_sync(0xffffffffu, ay[i], o);
        }
        float* yrow = sm.ystage[(t / TAU) % 3][t % TAU];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            coef[i] = cy.gy * ay[i];
            if (i == cg && t > 0) yrow[rg + RG * i] = fmaf(coef[i], cy.ys, cy.yb[i]);
            if constexpr (EMIT) {
                if (i == cg && t > 0) em_prev[2 * D + 4 + rg + RG * i] = ay[i];
            }
        }
    }

    // the pending update of step t-1 (all slots) and b = W_{t-1} x~_{t+1}
    float2 x2[NP];
    load_pairs(xn, cg, x2);
    float b[NS];
    {
        float2 accb[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) accb[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
#pragma unroll
            for (int i = 2; i < NS; ++i) {
                w[i][q] = __ffma2_rn(make_float2(coef[i], coef[i]), cy.pkc[q], w[i][q]);
                accb[i] = __ffma2_rn(w[i][q], x2[q], accb[i]);
            }
        }
#pragma unroll
        for (int q = 0; q < NP; ++q) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                w[i][q] = __ffma2_rn(make_float2(coef[i], coef[i]), cy.pkc[q], w[i][q]);
                accb[i] = __ffma2_rn(w[i][q], x2[q], accb[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < NS; ++i) b[i] = accb[i].x + accb[i].y;
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
#pragma unroll
            for (int i = 0; i < NS; ++i) b[i] += __shfl_xor_sync(0xffffffffu, b[i], o);
        }
    }

    // ---- 2. phi_k and u into the thread's column layout.  u takes an explicit
    // rounded subtraction, so equal k and q rows give u = 0 exactly.
    float* pkq = &sm.pkq[warp][0][0];
    const float u0 = __fsub_rn(pq0, pk0), u1 = __fsub_rn(pq1, pk1);
    pkq[lane] = pk0;
    pkq[lane + 32] = pk1;
    pkq[D + lane] = u0;
    pkq[D + lane + 32] = u1;
    if constexpr (EMIT) {
        // backward record of step t: phi(k), u, gates (the rows' a follow)
        if (warp == 0) {
            em[lane] = pk0;
            em[lane + 32] = pk1;
            em[D + lane] = u0;
            em[D + lane + 32] = u1;
            if (lane < 4) em[2 * D + lane] = lane == 0 ? g[0] : lane == 1 ? g[1] : lane == 2 ? g[2] : g[3];
        }
    }
    __syncwarp();
    load_pairs(pkq, cg, cy.pkc);
    load_pairs(pkq + D, cg, cy.u2);

    // ---- 3. a of the k, q and beta rows (the chain) and s = phi_k . x~_{t+1}
    float a[NS];
    float s;
    {
        float2 acca[NS];
#pragma unroll
        for (int i = 2; i < NS; ++i) acca[i] = make_float2(0.f, 0.f);
        float2 accs = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
#pragma unroll
            for (int i = 2; i < NS; ++i) acca[i] = __ffma2_rn(w[i][q], cy.u2[q], acca[i]);
            accs = __ffma2_rn(cy.pkc[q], x2[q], accs);
        }
#pragma unroll
        for (int i = 2; i < NS; ++i) a[i] = acca[i].x + acca[i].y;
        s = accs.x + accs.y;
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
#pragma unroll
        for (int i = 2; i < NS; ++i) a[i] += __shfl_xor_sync(0xffffffffu, a[i], o);
        s += __shfl_xor_sync(0xffffffffu, s, o);
    }

    // ---- 4. z_{t+1} of the k, q and beta rows; the y rows' values for the
    // next step
#pragma unroll
    for (int i = 2; i < NS; ++i) {
        const int blk = (NLR == 1) ? 0 : (i < SLOTS ? C::block_of_slot(i) : 3);
        coef[i] = g[blk] * a[i];
        const float zr = fmaf(coef[i], s, b[i]);
        if constexpr (EMIT) {
            if ((i & 3) == cg) {
                if (i < SLOTS) em[2 * D + 4 + rg + RG * i] = a[i];
                else if (3 * D + rg < M) em[2 * D + 4 + 3 * D + rg] = a[i];
            }
        }
        if ((i & 3) == cg) {
            if (i < SLOTS) zn[rg + RG * i] = zr;
            else if (3 * D + rg < M) zn[3 * D + rg] = zr;
        }
    }
    cy.yb[0] = b[0];
    cy.yb[1] = b[1];
    cy.ys = s;
    cy.gy = g[0];
    // y_t was the last row of its chunk: order the chunk's writes before the
    // TMA store that reads it (issued after the next barrier).  At the end of
    // the step, where it holds up no other work.
    if (t > 0 && ((t + 1) % TAU == 0 || t + 1 == T)) fence_proxy_async_smem();
}

template <int NW, int NLR, bool SMX, bool EMIT = false>
__global__ void __launch_bounds__(d64::Cfg<NW>::NT, 8 / NW)
    srwm_d64_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                    const KParams kp)
{
    using namespace d64;
    using C = Cfg<NW>;
    constexpr int SLOTS = C::SLOTS, RG = C::RG, XW = C::XW;
    constexpr int M = 3 * D + NLR;
    constexpr int S1 = SLOTS + 1;
    constexpr uint32_t kChunkBytes = TAU * D * sizeof(float);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<NW>& sm = *reinterpret_cast<Smem<NW>*>(smem_raw);
    if (!smem_base_ok(smem_raw, kp.status)) return;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = tid >> 2, cg = tid & 3;
    const bool has_beta = (warp == 0);   // warp-uniform: slot SLOTS = row 192 + rg

    if (tid == 0) {
        mbar_init(&sm.xbar[0], 1);
        mbar_init(&sm.xbar[1], 1);
        mbar_init(&sm.xbar[2], 1);
        fence_mbar_init();
        if (kp.T > 0) {
            prefetch_tensormap(&tmx);
            prefetch_tensormap(&tmy);
        }
    }
    __syncthreads();

    // bit i: parity of the phases x buffer i completed over earlier items
    uint32_t used = 0;
    int abort = 0;
    int issued = -1, landed = -1;   // chunks of the current item (warp XW)

    for (int item = blockIdx.x; item < kp.n_items; item += gridDim.x) {
        const int p = item % kp.n_streams, seg = item / kp.n_streams;
        const int b = p / kp.H, h = p - b * kp.H;
        const int t0 = seg * kp.seg_len;
        const int T = min(kp.seg_len, kp.T - t0);   // steps of this item
        const int nchunks = cdiv(T, TAU);
        issued = -1;
        landed = -1;

        // ---- the previous segment of this stream has to be finished
        if (seg > 0) {
            int fail = 0;
            if (tid == 0) fail = !wait_counter_bounded(kp.seg_done + p, seg, kp.wait_limit_ns);
            abort = __syncthreads_or(fail);
            if (abort) break;
        }

        // ---- W -> registers (W_init for a first segment, else the state that
        // the previous segment left in W_out; read through L2)
        float2 w[S1][NP];
        {
            const float* Ws = (seg == 0) ? kp.W_init + static_cast<size_t>(kp.w_per_seq ? p : h) * M * D
                                         : kp.W_out + static_cast<size_t>(p) * M * D;
#pragma unroll
            for (int i = 0; i < S1; ++i) {
                const int r = (i < SLOTS) ? rg + RG * i : 3 * D + rg;
                const bool ok = (i < SLOTS) || (has_beta && r < M);
#pragma unroll
                for (int j = 0; j < NP / 2; ++j) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (ok) v = __ldcg(reinterpret_cast<const float4*>(Ws + static_cast<size_t>(r) * D + 4 * (cg + 4 * j)));
                    w[i][2 * j] = make_float2(v.x, v.y);
                    w[i][2 * j + 1] = make_float2(v.z, v.w);
                }
            }
        }

        // ---- x staging (warp XW) and its TMA bookkeeping; chunk c of this
        // item is steps t0 + c*TAU .. and lands in buffer c % 3, as that
        // buffer's (c / 3)-th load of the item
        auto parity = [&](int c) -> uint32_t { return ((used >> (c % 3)) + static_cast<uint32_t>(c / 3)) & 1u; };
        auto issue_chunk = [&](int c) {
            if (lane == 0 && c != kp.skip_chunk) {
                mbar_arrive_expect_tx(&sm.xbar[c % 3], kChunkBytes);
                tma_load_4d(&sm.xring[c % 3][0][0], &tmx, &sm.xbar[c % 3], 0, h, t0 + c * TAU, b);
            }
            issued = c;
        };
        auto stage_x = [&](int tn, float* dst) {
            float v0 = 0.f, v1 = 0.f;
            if (tn < T) {
                const float* src = sm.xring[(tn / TAU) % 3][tn % TAU];
                v0 = src[lane];
                v1 = src[lane + 32];
                if constexpr (SMX) softmax64(v0, v1, v0, v1);
            }
            dst[lane] = v0;
            dst[lane + 32] = v1;
        };

        int fail = 0;
        if (warp == XW && T > 0) {
            issue_chunk(0);
            if (nchunks > 1) issue_chunk(1);
            if (__all_sync(0xffffffffu, mbar_wait_bounded(&sm.xbar[0], parity(0), kp.wait_limit_ns))) {
                landed = 0;
                if constexpr (SMX) {
                    stage_x(0, sm.xs[0]);
                    stage_x(1, sm.xs[1]);
                }
            } else {
                fail = 1;
            }
        }
        abort = __syncthreads_or(fail);

        // ---- prologue: z_0 = W x~_0 (y of the item's first step)
        if (!abort && T > 0) {
            float2 x2[NP];
            load_pairs(SMX ? sm.xs[0] : sm.xring[0][0], cg, x2);
            float2 acc[S1];
#pragma unroll
            for (int i = 0; i < S1; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
#pragma unroll
                for (int i = 0; i < S1; ++i) {
                    if (i == SLOTS && !has_beta) continue;
                    acc[i] = __ffma2_rn(w[i][q], x2[q], acc[i]);
                }
            }
            float bb[S1];
#pragma unroll
            for (int i = 0; i < S1; ++i) bb[i] = acc[i].x + acc[i].y;
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
#pragma unroll
                for (int i = 0; i < S1; ++i) bb[i] += __shfl_xor_sync(0xffffffffu, bb[i], o);
            }
#pragma unroll
            for (int i = 0; i < S1; ++i) {
                if ((i & 3) != cg) continue;
                if (i < SLOTS && C::block_of_slot(i) == 0) sm.ystage[0][0][rg + RG * i] = bb[i];
                else if (i < SLOTS) sm.z[0][rg + RG * i] = bb[i];
                else if (has_beta && 3 * D + rg < M) sm.z[0][3 * D + rg] = bb[i];
            }
            fence_proxy_async_smem();
        }
        __syncthreads();

        // the pending rank-one update (applied at the start of the next step)
        // and the y rows' values carried one step
        float coef[S1];
#pragma unroll
        for (int i = 0; i < S1; ++i) coef[i] = 0.f;
        D64Carry<NW> cy;
#pragma unroll
        for (int q = 0; q < NP; ++q) cy.pkc[q] = cy.u2[q] = make_float2(0.f, 0.f);
        cy.yb[0] = cy.yb[1] = cy.ys = cy.gy = 0.f;

        // Warp 0 also carries the beta rows; a compile-time slot count keeps
        // each role's step free of branches.
        auto step = [&](int t, const float* xn) {
            float* em = nullptr;
            if constexpr (EMIT) em = kp.emit + (static_cast<size_t>(p) * kp.T + t0 + t) * kp.emit_stride;
            float* em_prev = EMIT ? em - kp.emit_stride : nullptr;
            if (has_beta) d64_step<NW, S1, NLR, EMIT>(sm, t, T, lane, warp, rg, cg, w, coef, cy, xn, em, em_prev);
            else d64_step<NW, SLOTS, NLR, EMIT>(sm, t, T, lane, warp, rg, cg, w, coef, cy, xn, em, em_prev);
        };
        if constexpr (!SMX) {
            // x~ = x is read straight from the ring, chunk by chunk: the inner
            // loop holds only the step and its barrier; the chunk boundary
            // (bounded wait for the next chunk, agreed on by the CTA, the next
            // TMA load, the y store) runs between chunks.
            for (int c = 0; c < nchunks && !abort; ++c) {
                // The last step of chunk c reads the first row of chunk c + 1,
                // issued a chunk ago; chunk c + 2 goes into the buffer of chunk
                // c - 1, whose last row was read before here.
                if (c + 1 < nchunks) {
                    const bool ok = mbar_wait_bounded(&sm.xbar[(c + 1) % 3], parity(c + 1), kp.wait_limit_ns);
                    if (__syncthreads_or(!ok)) {
                        abort = 1;
                        break;
                    }
                    if (warp == XW) {
                        landed = c + 1;
                        if (c + 2 < nchunks) issue_chunk(c + 2);
                    }
                }
                // y of chunk c - 1 is complete (its last row was written, and
                // fenced, in the chunk's last step) -> TMA store; the store
                // before it has finished reading the buffer this chunk writes
                if (c > 0 && warp == 0 && lane == 0) {
                    tma_store_4d(&tmy, &sm.ystage[(c - 1) % 3][0][0], 0, h, t0 + (c - 1) * TAU, b);
                    bulk_commit();
                    bulk_wait_read<1>();
                }
                const int tend = min(T, (c + 1) * TAU);
                // the chunk's last step (the one that reads the next chunk)
                // stands apart from the loop over the others: measured 5.2 ->
                // 4.2 ms on long against one loop over all steps (same results
                // bit for bit; only the compiled schedule differs)
                const float* ring = sm.xring[c % 3][0];
                for (int t = c * TAU; t < tend - 1; ++t) {
                    step(t, ring + (t + 1 - c * TAU) * D);
                    __syncthreads();
                }
                step(tend - 1, sm.xring[(c + 1) % 3][0]);
                __syncthreads();
            }
        } else {
            for (int t = 0; t < T && !abort; ++t) {
                // y_{t-1} (written during step t - 1, the y rows running one
                // step behind) completed its chunk -> TMA store
                if (warp == 0 && lane == 0 && t > 0 && t % TAU == 0) {
                    const int c = (t - 1) / TAU;
                    tma_store_4d(&tmy, &sm.ystage[c % 3][0][0], 0, h, t0 + c * TAU, b);
                    bulk_commit();
                    bulk_wait_read<1>();
                }
                step(t, sm.xs[(t + 1) & 1]);

                // ---- x~_{t+2} -> xs[t & 1] (a new chunk may have to land first)
                fail = 0;
                if (warp == XW) {
                    const int tn = t + 2;
                    if (tn < T && tn % TAU == 0) {
                        const int c = tn / TAU;
                        const bool ok = mbar_wait_bounded(&sm.xbar[c % 3], parity(c), kp.wait_limit_ns);
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
            }
        }

        // ---- drain this item's y stores (the last chunk's store trails its
        // steps, as every chunk's does)
        if (warp == 0 && lane == 0) {
            if (!abort && T > 0) {
                const int c = (T - 1) / TAU;
                tma_store_4d(&tmy, &sm.ystage[c % 3][0][0], 0, h, t0 + c * TAU, b);
                bulk_commit();
            }
            bulk_wait_all<0>();
        }
        if (abort) break;
#pragma unroll
        for (int i = 0; i < 3; ++i) used ^= (static_cast<uint32_t>(nchunks > i ? (nchunks - 1 - i) / 3 + 1 : 0) & 1u) << i;

        // ---- the y rows' a of the last step (they run one step behind), the
        // last pending update, then the state -> W_out[b, h]
        if (T > 0) {
            float ay[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < NP; ++q) acc = __ffma2_rn(w[i][q], cy.u2[q], acc);
                ay[i] = acc.x + acc.y;
            }
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
#pragma unroll
                for (int i = 0; i < 2; ++i) ay[i] += __shfl_xor_sync(0xffffffffu, ay[i], o);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                coef[i] = cy.gy * ay[i];
                if constexpr (EMIT) {
                    if (i == cg)
                        kp.emit[(static_cast<size_t>(p) * kp.T + t0 + T - 1) * kp.emit_stride + 2 * D + 4 + rg +
                                RG * i] = ay[i];
                }
            }
        }
        float* Wd = kp.W_out + static_cast<size_t>(p) * M * D;
#pragma unroll
        for (int i = 0; i < S1; ++i) {
            const int r = (i < SLOTS) ? rg + RG * i : 3 * D + rg;
            if (i == SLOTS && !(has_beta && r < M)) continue;
#pragma unroll
            for (int q = 0; q < NP; ++q) w[i][q] = __ffma2_rn(make_float2(coef[i], coef[i]), cy.pkc[q], w[i][q]);
#pragma unroll
            for (int j = 0; j < NP / 2; ++j) {
                *reinterpret_cast<float4*>(Wd + static_cast<size_t>(r) * D + 4 * (cg + 4 * j)) =
                    make_float4(w[i][2 * j].x, w[i][2 * j].y, w[i][2 * j + 1].x, w[i][2 * j + 1].y);
            }
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
            for (int c = landed + 1; c <= issued; ++c) {
                if (c == kp.skip_chunk) continue;
                mbar_wait_bounded(&sm.xbar[c % 3], ((used >> (c % 3)) + static_cast<uint32_t>(c / 3)) & 1u,
                                  kp.wait_limit_ns);
            }
        }
        if (tid == 0) atomicOr(kp.status, kStatusTimeout);
    }
}

template <int NW, int NLR, bool SMX, bool EMIT = false>
LaunchInfo launch_info_d64_impl()
{
    return LaunchInfo{reinterpret_cast<const void*>(&srwm_d64_kernel<NW, NLR, SMX, EMIT>), d64::Cfg<NW>::NT, 1,
                      static_cast<int>(sizeof(d64::Smem<NW>)) + 128, d64::TAU};
}

}  // namespace srwm
