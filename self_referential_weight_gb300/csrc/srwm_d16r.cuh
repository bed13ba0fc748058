// srwm_d16r.cuh -- the d = 16 kernel of the SRWM forward recurrence: one warp
// per (sequence, head) stream, each lane holding whole rows of W.
//
// The recurrence (per sequence b, head h; "Metalearning Continual Learning
// Algorithms", section 2.3, Eqs. (1)-(3), four-rate version Eqs. (4)-(5)):
//   z_t = [y_t, k_t, q_t, beta_t] = W_{t-1} x~_t
//   W_t = W_{t-1} + diag(g_t) (W_{t-1} (phi(q_t) - phi(k_t))) (outer) phi(k_t)
// with g_t = sigmoid(beta_t) of the row's block and phi = softmax.
//
// Layout.  W is m x 16 with m = 48 + n_lr.  Lane l holds two rows whole, as
// 8 column pairs each: row l (a y row for l < 16, a k row for l >= 16) and
// row 32 + l (a q row for l < 16, beta row l - 16 for 16 <= l < 16 + n_lr,
// nothing above).  So the dot products of every row finish inside its lane,
// the k entries of z sit in the upper half-warp and the q entries in the
// lower half, and both softmaxes take whole-warp redux.sync reductions with
// the other half masked out.
// u = phi(q) - phi(k) takes one cross-half shuffle; u, phi(k) and x~ reach
// every lane as broadcast shared-memory reads, and every lane forms
// s = phi(k_t) . x~_{t+1} itself in the pass over W, so no sum over the warp
// is left in the step.
//
// One step t, on W_{t-1} in registers:
//   a_r       = W[r,:] . u_t                  (Eq. (2))
//   b_r       = W[r,:] . x~_{t+1}             (Eq. (1) of step t+1 on the old matrix)
//   z_{t+1,r} = b_r + g_r a_r (phi(k_t) . x~_{t+1})
// and the rank-one update W[r,:] += g_r a_r phi(k_t) (Eq. (3)) is applied in
// the next step's pass over W, before that step's products.  The z line is
// W_t x~_{t+1} through the rank-one structure of the update.  Inputs stream in
// by TMA (chunks of TAU steps, three buffers, mbarrier completion with bounded
// waits); with the input softmax, x~ replaces a landed chunk's rows in place.
// Outputs leave by TMA from a two-chunk ring.  Only __syncwarp orders a warp's
// steps; waits, TMA issues and the y stores sit at chunk boundaries.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "srwm_common.h"
#include "srwm_ptx.cuh"

namespace srwm {

namespace d16 {

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float2 pair_lo(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 pair_hi(float4 v) { return make_float2(v.z, v.w); }

// softmax over the 16 values of each half-warp (lane l holds entry l % 16 of
// its half).  Whole-warp reductions with the other half masked out: the
// maximum by redux.sync.max, the sum of the exponentials exactly in fixed
// point (2^-27 steps, so sixteen values in [0, 1] fit 32 bits) by
// redux.sync.add.  Every lane of a half ends with the same shift and sum bits.
__device__ __forceinline__ float softmax16(float v)
{
    const bool lo = (threadIdx.x & 16) == 0;
    const float ninf = __int_as_float(0xff800000);
    const float m_lo = redux_max(lo ? v : ninf);
    const float m_hi = redux_max(lo ? ninf : v);
    const float e = __expf(v - (lo ? m_lo : m_hi));
    const uint32_t q = __float2uint_rn(e * 134217728.0f);
    const uint32_t s_lo = redux_add(lo ? q : 0u);
    const uint32_t s_hi = redux_add(lo ? 0u : q);
    const float sum = static_cast<float>(lo ? s_lo : s_hi) * 7.450580596923828125e-09f;
    return e * rcp_approx(sum);
}

template <int NLR_, bool SMX_>
struct Cfg {
    static constexpr int D = 16, NLR = NLR_;
    static constexpr bool SMX = SMX_;
    static constexpr int M = 3 * D + NLR;
    static constexpr int NP = D / 2;   // column pairs per row
    static constexpr int TAU = 16;     // steps per TMA chunk
    static constexpr int PPC = 8;      // streams (warps) per CTA
    static constexpr int NT = 32 * PPC;
};

template <class C>
struct __align__(128) Smem {
    float xring[3 * C::TAU][C::D];  // x by TMA, three chunks (row = step mod 3 TAU); x~ in place
    float yring[2 * C::TAU][C::D];  // y for TMA, two chunks (row = step mod 2 TAU)
    float pk[3][C::D];              // phi(k) of the last three steps
    float u[2][C::D];               // u of the last two steps
    uint64_t xbar[3];               // "chunk landed" barriers of the x ring
};

}  // namespace d16

template <int NLR, bool SMX, bool EMIT = false>
__global__ void __launch_bounds__(d16::Cfg<NLR, SMX>::NT, 2)
    srwm_d16_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                    const KParams kp)
{
    using C = d16::Cfg<NLR, SMX>;
    using d16::lds4;
    using d16::pair_hi;
    using d16::pair_lo;
    constexpr int D = C::D, TAU = C::TAU, NP = C::NP;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    d16::Smem<C>& sm = reinterpret_cast<d16::Smem<C>*>(smem_raw)[warp];
    if (!smem_base_ok(smem_raw, kp.status)) return;
    constexpr uint32_t kChunkBytes = TAU * D * sizeof(float);

    const bool lo_half = lane < 16;               // rows y (A) and q (B); else k (A) and beta (B)
    const int col = lane & 15;                    // softmax entry of this lane
    const bool has_b = lane < 16 + NLR;           // row B exists
    // gates of the two rows: blocks y / k for row A, q / beta for row B
    const int blk_a = NLR == 1 ? 0 : (lo_half ? 0 : 1);
    const int blk_b = NLR == 1 ? 0 : (lo_half ? 2 : 3);

    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < 3; ++i) mbar_init(&sm.xbar[i], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // bit i: parity of the next completion awaited on x buffer i (every
    // issued chunk is awaited exactly once, in issue order)
    uint32_t phase = 0;
    int abort = 0;
    int issued = -1, landed = -1;   // chunks of the current piece

    // this slot's pieces: the wrap-around schedule, or items slot, slot +
    // n_slots, ... of the segment schedule
    const int slot = blockIdx.x * C::PPC + warp;
    const int n_slots = gridDim.x * C::PPC;
    long long lo = 0, hi = 0;
    if (kp.wrap_len > 0) {
        lo = static_cast<long long>(slot) * kp.wrap_len;
        hi = min(lo + kp.wrap_len, static_cast<long long>(kp.n_streams) * kp.T);
    }
    int item = slot;
    auto next_piece = [&](Piece& pc) -> bool {
        if (kp.wrap_len > 0) return wrap_next(lo, hi, kp.T, pc);
        if (item >= kp.n_items) return false;
        pc.p = item % kp.n_streams;
        pc.seg = item / kp.n_streams;
        pc.t0 = pc.seg * kp.seg_len;
        pc.len = min(kp.seg_len, kp.T - pc.t0);
        item += n_slots;
        return true;
    };
    // x chunk c (steps t0 + c*TAU ..) of stream p into x buffer c % 3
    auto load_x = [&](int p, int t0, int c) {
        if (lane == 0 && c != kp.skip_chunk) {
            const int bi = c % 3, b = p / kp.H, h = p - (p / kp.H) * kp.H;
            mbar_arrive_expect_tx(&sm.xbar[bi], kChunkBytes);
            tma_load_4d(&sm.xring[bi * TAU][0], &tmx, &sm.xbar[bi], 0, h, t0 + c * TAU, b);
        }
    };

    Piece cur;
    bool have = next_piece(cur);
    int pre = 0;   // chunks of `cur` that the previous piece already issued
    while (have) {
        Piece nxt;
        const bool have_next = next_piece(nxt);
        const int p = cur.p, seg = cur.seg, t0 = cur.t0;
        const int b = p / kp.H, h = p - b * kp.H;
        const int T = cur.len;   // steps of this piece
        const int nchunks = cdiv(T, TAU);
        issued = pre - 1;
        landed = -1;

        // ---- the previous segment of this stream has to be finished
        if (seg > 0) {
            int ok = 1;
            if (lane == 0) ok = wait_counter_bounded(kp.seg_done + p, seg, kp.wait_limit_ns);
            abort = !__shfl_sync(0xffffffffu, ok, 0);
            if (abort) break;
        }

        // ---- W -> registers (W_init for a first segment, else the state the
        // previous segment left in W_out; read through L2).  Row A = lane,
        // row B = 32 + lane (zero where there is none).
        float2 w[2][NP];
        {
            const float* Ws = (seg == 0) ? kp.W_init + static_cast<size_t>(kp.w_per_seq ? p : h) * C::M * D
                                         : kp.W_out + static_cast<size_t>(p) * C::M * D;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const bool ok = i == 0 || has_b;
                const float4* row = reinterpret_cast<const float4*>(Ws + static_cast<size_t>(32 * i + lane) * D);
#pragma unroll
                for (int j = 0; j < NP / 2; ++j) {
                    const float4 v = ok ? __ldcg(row + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                    w[i][2 * j] = pair_lo(v);
                    w[i][2 * j + 1] = pair_hi(v);
                }
            }
        }

        auto issue_chunk = [&](int c) {
            load_x(p, t0, c);
            issued = c;
        };
        // waits for chunk c; with softmax_input, replaces its rows by x~ in
        // place (two rows per pass, one per half-warp)
        auto land_chunk = [&](int c) -> bool {
            const int bi = c % 3;
            const bool ok = mbar_wait_bounded(&sm.xbar[bi], (phase >> bi) & 1u, kp.wait_limit_ns);
            if (!__all_sync(0xffffffffu, ok)) return false;
            phase ^= 1u << bi;
            landed = c;
            if constexpr (SMX) {
                float v[TAU / 2];
#pragma unroll
                for (int r = 0; r < TAU / 2; ++r) v[r] = sm.xring[bi * TAU + 2 * r + (lane >> 4)][col];
#pragma unroll
                for (int r = 0; r < TAU / 2; ++r) v[r] = d16::softmax16(v[r]);
#pragma unroll
                for (int r = 0; r < TAU / 2; ++r) sm.xring[bi * TAU + 2 * r + (lane >> 4)][col] = v[r];
                // the buffer is refilled by TMA later: order these writes first
                fence_proxy_async_smem();
            }
            return true;
        };

        // recurrent state between steps: z_t of this lane's two rows (row A: y
        // or k; row B: q or beta) and the pending rank-one update
        float za = 0.f, zb = 0.f;
        float coef[2] = {0.f, 0.f};

        if (T > 0) {
            if (pre < 1) issue_chunk(0);
            if (nchunks > 1 && pre < 2) issue_chunk(1);
            abort = !land_chunk(0);
            if (!abort) {
                // ---- prologue: z_0 = W x~_0; the pending update starts empty
                if (lane < D) sm.pk[2][lane] = 0.f;
                __syncwarp();
                float2 acc[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < NP / 2; ++j) {
                    const float4 x4 = lds4(&sm.xring[0][4 * j]);
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        acc[i] = __ffma2_rn(w[i][2 * j], pair_lo(x4), acc[i]);
                        acc[i] = __ffma2_rn(w[i][2 * j + 1], pair_hi(x4), acc[i]);
                    }
                }
                za = acc[0].x + acc[0].y;
                zb = acc[1].x + acc[1].y;
            }
        }

        int xr = 1;   // x ring row of step t + 1
        int ps = 0;   // phi(k) slot of step t (step t - 1 used ps + 2 mod 3)
        for (int c = 0; c < nchunks && !abort; ++c) {
            // ---- chunk boundary.  Step c*TAU + TAU - 1 reads x~ of the first
            // step of chunk c + 1 (issued a chunk ago); chunk c + 2 goes into
            // the buffer of chunk c - 1, whose last row was read before here.
            if (c + 1 < nchunks) {
                if (!land_chunk(c + 1)) {
                    abort = 1;
                    break;
                }
            }
            // orders this chunk's in-place x~ writes and the last chunk's y
            // writes before the TMA operations below
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (c + 2 < nchunks) issue_chunk(c + 2);
                if (c > 0) {
                    // y of chunk c - 1 is complete; the store before it has then
                    // finished reading the buffer chunk c writes
                    tma_store_4d(&tmy, &sm.yring[((c - 1) & 1) * TAU][0], 0, h, t0 + (c - 1) * TAU, b);
                    bulk_commit();
                    bulk_wait_read<1>();
                }
            }
            if (c + 2 < nchunks) issued = c + 2;
            __syncwarp();
            const int t_end = min(T, (c + 1) * TAU);
            for (int t = c * TAU; t < t_end; ++t) {
                if (lo_half) sm.yring[t & (2 * TAU - 1)][lane] = za;   // y_t
                const float* xrow = sm.xring[xr];                      // x~_{t+1}
                xr = xr == 3 * TAU - 1 ? 0 : xr + 1;
                const int pp = ps == 0 ? 2 : ps - 1;                   // slot of step t - 1
                // softmaxes: phi(k) in the upper half, phi(q) in the lower
                const float ph = d16::softmax16(lo_half ? zb : za);
                const float other = __shfl_xor_sync(0xffffffffu, ph, 16);   // the other half's entry
                const float pk = lo_half ? other : ph;                      // phi(k)[col] on every lane
                // u = phi(q) - phi(k), rounded as such (no contraction)
                const float u = __fsub_rn(lo_half ? ph : other, pk);
                // gates: sigmoid of the beta entries, held by lanes 16 .. 16 + n_lr - 1
                const float sg = sigmoid_fast(zb);
                float g[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) g[r] = __shfl_sync(0xffffffffu, sg, 16 + (NLR == 1 ? 0 : r));
                // both halves hold phi(k)[col] and u[col]: every lane stores (the
                // upper half repeats the lower half's values), no divergence
                sm.pk[ps][col] = pk;
                sm.u[t & 1][col] = u;
                __syncwarp();
                // one pass over W: the pending update of step t - 1 (Eq. (3)),
                // then a = W u_t and b = W x~_{t+1} on the updated columns, and
                // s = phi(k_t) . x~_{t+1} beside them (every lane, the same bits)
                const float* pkp = sm.pk[pp];
                const float* un = sm.u[t & 1];
                const float* pkc = sm.pk[ps];
                float2 cc[2], aa[2], bb[2], ss = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    cc[i] = make_float2(coef[i], coef[i]);
                    aa[i] = bb[i] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < NP / 2; ++j) {
                    const float4 p4 = lds4(pkp + 4 * j);
                    const float4 u4 = lds4(un + 4 * j);
                    const float4 x4 = lds4(xrow + 4 * j);
                    const float4 k4 = lds4(pkc + 4 * j);
                    ss = __ffma2_rn(pair_lo(k4), pair_lo(x4), ss);
                    ss = __ffma2_rn(pair_hi(k4), pair_hi(x4), ss);
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        w[i][2 * j] = __ffma2_rn(cc[i], pair_lo(p4), w[i][2 * j]);
                        w[i][2 * j + 1] = __ffma2_rn(cc[i], pair_hi(p4), w[i][2 * j + 1]);
                        aa[i] = __ffma2_rn(w[i][2 * j], pair_lo(u4), aa[i]);
                        bb[i] = __ffma2_rn(w[i][2 * j], pair_lo(x4), bb[i]);
                        aa[i] = __ffma2_rn(w[i][2 * j + 1], pair_hi(u4), aa[i]);
                        bb[i] = __ffma2_rn(w[i][2 * j + 1], pair_hi(x4), bb[i]);
                    }
                }
                const float s = ss.x + ss.y;
                const float a0 = aa[0].x + aa[0].y, a1 = aa[1].x + aa[1].y;
                const float ga = blk_a == 0 ? g[0] : g[1];
                const float gb = blk_b == 0 ? g[0] : (blk_b == 2 ? g[2] : g[3]);
                coef[0] = ga * a0;
                coef[1] = gb * a1;
                za = fmaf(coef[0], s, bb[0].x + bb[0].y);
                zb = fmaf(coef[1], s, bb[1].x + bb[1].y);
                if constexpr (EMIT) {
                    // backward record of step t: phi(k), u, gates, a
                    float* em = kp.emit + (static_cast<size_t>(p) * kp.T + t0 + t) * kp.emit_stride;
                    if (lo_half) {
                        em[lane] = pk;
                        em[D + lane] = u;
                    }
                    if (lane < 4) em[2 * D + lane] = lane == 0 ? g[0] : lane == 1 ? g[1] : lane == 2 ? g[2] : g[3];
                    float* ea = em + 2 * D + 4;
                    ea[lane] = a0;
                    if (has_b) ea[32 + lane] = a1;
                }
                ps = ps == 2 ? 0 : ps + 1;
            }
        }

        // ---- end of the piece: the last chunk's y goes out, and the next
        // piece's first x chunks (every x buffer is free now)
        pre = 0;
        if (!abort) {
            fence_proxy_async_smem();
            __syncwarp();
            if (T > 0 && lane == 0) {
                const int c = nchunks - 1;
                tma_store_4d(&tmy, &sm.yring[(c & 1) * TAU][0], 0, h, t0 + c * TAU, b);
                bulk_commit();
            }
            if (have_next && nxt.len > 0) {
                load_x(nxt.p, nxt.t0, 0);
                pre = 1;
                if (nxt.len > TAU) {
                    load_x(nxt.p, nxt.t0, 1);
                    pre = 2;
                }
            }
        }
        if (abort) {
            if (lane == 0) bulk_wait_all<0>();
            __syncwarp();
            break;
        }

        // ---- the last step's update, then the state -> W_out[b, h]
        if (T > 0) {
            const float* pkp = sm.pk[ps == 0 ? 2 : ps - 1];
#pragma unroll
            for (int j = 0; j < NP / 2; ++j) {
                const float4 p4 = lds4(pkp + 4 * j);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float2 cc = make_float2(coef[i], coef[i]);
                    w[i][2 * j] = __ffma2_rn(cc, pair_lo(p4), w[i][2 * j]);
                    w[i][2 * j + 1] = __ffma2_rn(cc, pair_hi(p4), w[i][2 * j + 1]);
                }
            }
        }
        float* Wd = kp.W_out + static_cast<size_t>(p) * C::M * D;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (i == 1 && !has_b) continue;
            float4* row = reinterpret_cast<float4*>(Wd + static_cast<size_t>(32 * i + lane) * D);
#pragma unroll
            for (int j = 0; j < NP / 2; ++j)
                row[j] = make_float4(w[i][2 * j].x, w[i][2 * j].y, w[i][2 * j + 1].x, w[i][2 * j + 1].y);
        }
        __syncwarp();
        if (lane == 0) {
            // y written (a later segment may start with rows this store covers)
            // and W_out visible before the next segment may start
            bulk_wait_all<0>();
            if (kp.seg_done != nullptr) {
                __threadfence();
                st_release_gpu(kp.seg_done + p, seg + 1);
            }
        }
        __syncwarp();
        cur = nxt;
        have = have_next;
    }

    if (abort) {
        // every load still in flight lands before the warp gives up its buffers
        for (int c = landed + 1; c <= issued; ++c) {
            if (c == kp.skip_chunk) continue;
            const int bi = c % 3;
            mbar_wait_bounded(&sm.xbar[bi], (phase >> bi) & 1u, kp.wait_limit_ns);
            phase ^= 1u << bi;
        }
        if (lane == 0) atomicOr(kp.status, kStatusTimeout);
    }
}

template <int NLR, bool SMX, bool EMIT = false>
LaunchInfo launch_info_d16_impl()
{
    using C = d16::Cfg<NLR, SMX>;
    return LaunchInfo{reinterpret_cast<const void*>(&srwm_d16_kernel<NLR, SMX, EMIT>), C::NT, C::PPC,
                      static_cast<int>(C::PPC * sizeof(d16::Smem<C>)) + 128, C::TAU, true};
}

}  // namespace srwm
