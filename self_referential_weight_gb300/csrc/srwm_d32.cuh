// srwm_d32.cuh -- the d = 32 kernel of the SRWM forward recurrence: one warp
// per (sequence, head) stream, each lane holding whole rows of W.
//
// The recurrence (per sequence b, head h; "Metalearning Continual Learning
// Algorithms", section 2.3, Eqs. (1)-(3), four-rate version Eqs. (4)-(5)):
//   z_t = [y_t, k_t, q_t, beta_t] = W_{t-1} x~_t
//   W_t = W_{t-1} + diag(g_t) (W_{t-1} (phi(q_t) - phi(k_t))) (outer) phi(k_t)
// with g_t = sigmoid(beta_t) of the row's block and phi = softmax.
//
// Layout.  W is m x 32 with m = 96 + n_lr.  Lane l holds rows l, 32 + l and
// 64 + l (its y, k and q rows) whole, as 16 column pairs each, and column l of
// the n_lr beta rows.  A lane therefore finishes the dot products of its three
// rows without any cross-lane reduction; u = phi(q) - phi(k), phi(k) and x~
// reach every lane as broadcast shared-memory reads, and k_t, q_t stay in the
// registers of the lane that produced them until the next step's softmax.
// Only the beta rows (one column per lane) and s = phi(k_t) . x~_{t+1} are
// summed over the warp (with four beta rows, their eight sums by a
// reduce-scatter butterfly).
//
// One step t, on W_{t-1} in registers:
//   a_r       = W[r,:] . u_t                  (Eq. (2))
//   b_r       = W[r,:] . x~_{t+1}             (Eq. (1) of step t+1 on the old matrix)
//   z_{t+1,r} = b_r + g_r a_r (phi(k_t) . x~_{t+1})
// and the rank-one update W[r,:] += g_r a_r phi(k_t) (Eq. (3)) is applied at
// the start of step t+1, beside that step's softmaxes.  The z line is
// W_t x~_{t+1} through the rank-one structure of the update, so Eq. (1) needs
// no second sweep over W.  All products over W use two-wide FMAs on column
// pairs.  Inputs stream in by TMA (chunks of TAU steps, double-buffered,
// mbarrier completion with bounded waits); outputs leave by TMA from a
// double-buffered staging area.  Only __syncwarp orders a warp's steps.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "srwm_common.h"
#include "srwm_ptx.cuh"

namespace srwm {

namespace d32 {

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float2 pair_lo(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 pair_hi(float4 v) { return make_float2(v.z, v.w); }

// softmax over the 32 values of a warp, lane l holding entry l.
__device__ __forceinline__ float softmax32(float v)
{
    const float mx = redux_max(v);
    const float e = __expf(v - mx);
    return e * rcp_approx(warp_sum_unit1(e));
}

// Sums each of K values over the 32 lanes; every lane ends with the same bits.
template <int K>
__device__ __forceinline__ void allsum(float (&v)[K])
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int k = 0; k < K; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
    }
}

// Sums eight values over the 32 lanes by a reduce-scatter butterfly (each
// level halves the values a lane carries), then broadcasts: value i ends fully
// summed in lanes 4i..4i+3 and reaches every lane from lane 4i, so all lanes
// get the same bits.  17 shuffles instead of 40.
__device__ __forceinline__ void allsum8(float (&v)[8], int lane)
{
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float w[4], x[2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float send = b4 ? v[j] : v[4 + j];
        const float keep = b4 ? v[4 + j] : v[j];
        w[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float send = b3 ? w[j] : w[2 + j];
        const float keep = b3 ? w[2 + j] : w[j];
        x[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float y = (b2 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, b2 ? x[0] : x[1], 4);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    y += __shfl_xor_sync(0xffffffffu, y, 1);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __shfl_sync(0xffffffffu, y, 4 * i);
}

template <int NLR_, bool SMX_>
struct Cfg {
    static constexpr int D = 32, NLR = NLR_;
    static constexpr bool SMX = SMX_;
    static constexpr int M = 3 * D + NLR;
    static constexpr int NP = D / 2;   // column pairs per row
    static constexpr int TAU = 16;     // steps per TMA chunk
    // Streams (warps) per CTA.  Two CTAs per SM give three warps per scheduler
    // at the 168-register cap that holds W (96 + n_lr values per lane).
    static constexpr int PPC = 6;
    static constexpr int NT = 32 * PPC;
    // block (y, k, q, beta) of row slot i for the gate
    SRWM_HD static constexpr int gate(int i) { return NLR == 1 ? 0 : i; }
};

template <class C>
struct __align__(128) Smem {
    float xring[3 * C::TAU][C::D];  // x by TMA, three chunks (row = step mod 3 TAU); x~ in place
    float yring[2 * C::TAU][C::D];  // y for TMA, two chunks (row = step mod 2 TAU)
    float pk[3][C::D];              // phi(k) of the last three steps
    float u[2][C::D];               // u_t = phi(q_t) - phi(k_t) of the last two steps
    uint64_t xbar[3];               // "chunk landed" barriers of the x ring
};

}  // namespace d32

template <int NLR, bool SMX, bool EMIT = false>
__global__ void __launch_bounds__(d32::Cfg<NLR, SMX>::NT, 2)
    srwm_d32_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmy,
                    const KParams kp)
{
    using C = d32::Cfg<NLR, SMX>;
    using d32::lds4;
    using d32::pair_hi;
    using d32::pair_lo;
    constexpr int D = C::D, TAU = C::TAU, NP = C::NP;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    d32::Smem<C>& sm = reinterpret_cast<d32::Smem<C>*>(smem_raw)[warp];
    if (!smem_base_ok(smem_raw, kp.status)) return;
    constexpr uint32_t kChunkBytes = TAU * D * sizeof(float);

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
        // previous segment left in W_out; read through L2)
        float2 w[3][NP];
        float wb[NLR];
        {
            const float* Ws = (seg == 0) ? kp.W_init + static_cast<size_t>(kp.w_per_seq ? p : h) * C::M * D
                                         : kp.W_out + static_cast<size_t>(p) * C::M * D;
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const float4* row = reinterpret_cast<const float4*>(Ws + static_cast<size_t>(32 * i + lane) * D);
#pragma unroll
                for (int j = 0; j < NP / 2; ++j) {
                    const float4 v = __ldcg(row + j);
                    w[i][2 * j] = pair_lo(v);
                    w[i][2 * j + 1] = pair_hi(v);
                }
            }
#pragma unroll
            for (int r = 0; r < NLR; ++r) wb[r] = __ldcg(Ws + static_cast<size_t>(3 * D + r) * D + lane);
        }

        auto issue_chunk = [&](int c) {
            load_x(p, t0, c);
            issued = c;
        };
        // waits for chunk c; with softmax_input, replaces its rows by x~ in
        // place (sixteen independent softmaxes)
        auto land_chunk = [&](int c) -> bool {
            const int bi = c % 3;
            const bool ok = mbar_wait_bounded(&sm.xbar[bi], (phase >> bi) & 1u, kp.wait_limit_ns);
            if (!__all_sync(0xffffffffu, ok)) return false;
            phase ^= 1u << bi;
            landed = c;
            if constexpr (SMX) {
                float v[TAU];
#pragma unroll
                for (int r = 0; r < TAU; ++r) v[r] = sm.xring[bi * TAU + r][lane];
#pragma unroll
                for (int r = 0; r < TAU; ++r) v[r] = d32::softmax32(v[r]);
#pragma unroll
                for (int r = 0; r < TAU; ++r) sm.xring[bi * TAU + r][lane] = v[r];
                // the buffer is refilled by TMA later: order these writes first
                fence_proxy_async_smem();
            }
            return true;
        };

        // recurrent state between steps: y_t, k_t, q_t of this lane's rows,
        // beta_t and the pending rank-one update
        float zy = 0.f, zk = 0.f, zq = 0.f, zb[NLR];
        float coef[3] = {0.f, 0.f, 0.f}, coefb[NLR], pk_last = 0.f;
#pragma unroll
        for (int r = 0; r < NLR; ++r) zb[r] = coefb[r] = 0.f;

        if (T > 0) {
            if (pre < 1) issue_chunk(0);
            if (nchunks > 1 && pre < 2) issue_chunk(1);
            abort = !land_chunk(0);
            if (!abort) {
                // ---- prologue: z_0 = W x~_0; the pending update starts empty
                sm.pk[2][lane] = 0.f;
                __syncwarp();
                const float x0 = sm.xring[0][lane];
                float2 acc[3];
#pragma unroll
                for (int i = 0; i < 3; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < NP / 2; ++j) {
                    const float4 x4 = lds4(&sm.xring[0][4 * j]);
#pragma unroll
                    for (int i = 0; i < 3; ++i) {
                        acc[i] = __ffma2_rn(w[i][2 * j], pair_lo(x4), acc[i]);
                        acc[i] = __ffma2_rn(w[i][2 * j + 1], pair_hi(x4), acc[i]);
                    }
                }
                zy = acc[0].x + acc[0].y;
                zk = acc[1].x + acc[1].y;
                zq = acc[2].x + acc[2].y;
#pragma unroll
                for (int r = 0; r < NLR; ++r) zb[r] = wb[r] * x0;
                d32::allsum(zb);
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
                sm.yring[t & (2 * TAU - 1)][lane] = zy;
                const float* xrow = sm.xring[xr];   // x~_{t+1}
                xr = xr == 3 * TAU - 1 ? 0 : xr + 1;
                const float xc = xrow[lane];
                const int pp = ps == 0 ? 2 : ps - 1;   // slot of step t - 1
#pragma unroll
                for (int r = 0; r < NLR; ++r) wb[r] = fmaf(coefb[r], pk_last, wb[r]);
                const float pk = d32::softmax32(zk);
                const float pq = d32::softmax32(zq);
                const float u = __fsub_rn(pq, pk);   // no contraction into the softmax's last product
                float g[4];
                if constexpr (NLR == 4) {
#pragma unroll
                    for (int r = 0; r < 4; ++r) g[r] = sigmoid_fast(zb[r]);
                } else {
                    g[0] = g[1] = g[2] = g[3] = sigmoid_fast(zb[0]);
                }
                sm.pk[ps][lane] = pk;
                sm.u[t & 1][lane] = u;
                // s = phi(k_t) . x~_{t+1} and the beta rows' a and b, over the warp
                float red[1 + 2 * NLR];
                red[0] = pk * xc;
#pragma unroll
                for (int r = 0; r < NLR; ++r) {
                    red[1 + r] = wb[r] * u;
                    red[1 + NLR + r] = wb[r] * xc;
                }
                __syncwarp();
                if constexpr (NLR == 4) {
                    float sv[1] = {red[0]};
                    float bv[8];
#pragma unroll
                    for (int r = 0; r < 8; ++r) bv[r] = red[1 + r];
                    d32::allsum(sv);
                    d32::allsum8(bv, lane);
                    red[0] = sv[0];
#pragma unroll
                    for (int r = 0; r < 8; ++r) red[1 + r] = bv[r];
                } else {
                    d32::allsum(red);
                }
                // one pass over W: the pending update of step t - 1 (Eq. (3)),
                // then a = W u_t and b = W x~_{t+1} on the updated columns
                const float* pkp = sm.pk[pp];
                const float* un = sm.u[t & 1];
                float2 cc[3], aa[3], bb[3];
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    cc[i] = make_float2(coef[i], coef[i]);
                    aa[i] = bb[i] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < NP / 2; ++j) {
                    const float4 p4 = lds4(pkp + 4 * j);
                    const float4 u4 = lds4(un + 4 * j);
                    const float4 x4 = lds4(xrow + 4 * j);
#pragma unroll
                    for (int i = 0; i < 3; ++i) {
                        w[i][2 * j] = __ffma2_rn(cc[i], pair_lo(p4), w[i][2 * j]);
                        w[i][2 * j + 1] = __ffma2_rn(cc[i], pair_hi(p4), w[i][2 * j + 1]);
                        aa[i] = __ffma2_rn(w[i][2 * j], pair_lo(u4), aa[i]);
                        bb[i] = __ffma2_rn(w[i][2 * j], pair_lo(x4), bb[i]);
                        aa[i] = __ffma2_rn(w[i][2 * j + 1], pair_hi(u4), aa[i]);
                        bb[i] = __ffma2_rn(w[i][2 * j + 1], pair_hi(x4), bb[i]);
                    }
                }
                const float s = red[0];
                float a[3];
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    a[i] = aa[i].x + aa[i].y;
                    coef[i] = g[C::gate(i)] * a[i];
                }
                zy = fmaf(coef[0], s, bb[0].x + bb[0].y);
                zk = fmaf(coef[1], s, bb[1].x + bb[1].y);
                zq = fmaf(coef[2], s, bb[2].x + bb[2].y);
#pragma unroll
                for (int r = 0; r < NLR; ++r) {
                    coefb[r] = g[3] * red[1 + r];
                    zb[r] = fmaf(coefb[r], s, red[1 + NLR + r]);
                }
                if constexpr (EMIT) {
                    // backward record of step t: phi(k), u, gates, a
                    float* em = kp.emit + (static_cast<size_t>(p) * kp.T + t0 + t) * kp.emit_stride;
                    em[lane] = pk;
                    em[D + lane] = u;
                    if (lane < 4) em[2 * D + lane] = lane == 0 ? g[0] : lane == 1 ? g[1] : lane == 2 ? g[2] : g[3];
                    float* ea = em + 2 * D + 4;
                    ea[lane] = a[0];
                    ea[D + lane] = a[1];
                    ea[2 * D + lane] = a[2];
#pragma unroll
                    for (int r = 0; r < NLR; ++r) {
                        if (lane == r) ea[3 * D + r] = red[1 + r];
                    }
                }
                pk_last = pk;
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
                for (int i = 0; i < 3; ++i) {
                    const float2 cc = make_float2(coef[i], coef[i]);
                    w[i][2 * j] = __ffma2_rn(cc, pair_lo(p4), w[i][2 * j]);
                    w[i][2 * j + 1] = __ffma2_rn(cc, pair_hi(p4), w[i][2 * j + 1]);
                }
            }
#pragma unroll
            for (int r = 0; r < NLR; ++r) wb[r] = fmaf(coefb[r], pk_last, wb[r]);
        }
        float* Wd = kp.W_out + static_cast<size_t>(p) * C::M * D;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            float4* row = reinterpret_cast<float4*>(Wd + static_cast<size_t>(32 * i + lane) * D);
#pragma unroll
            for (int j = 0; j < NP / 2; ++j)
                row[j] = make_float4(w[i][2 * j].x, w[i][2 * j].y, w[i][2 * j + 1].x, w[i][2 * j + 1].y);
        }
#pragma unroll
        for (int r = 0; r < NLR; ++r) Wd[static_cast<size_t>(3 * D + r) * D + lane] = wb[r];
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
LaunchInfo launch_info_d32_impl()
{
    using C = d32::Cfg<NLR, SMX>;
    return LaunchInfo{reinterpret_cast<const void*>(&srwm_d32_kernel<NLR, SMX, EMIT>), C::NT, C::PPC,
                      static_cast<int>(C::PPC * sizeof(d32::Smem<C>)) + 128, C::TAU, true};
}

}  // namespace srwm
