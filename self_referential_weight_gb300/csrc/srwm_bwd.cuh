// srwm_bwd.cuh -- backward pass of the SRWM recurrence (gradients of a loss
// L(y, W_final) with respect to x and W0), one CTA per (sequence, head)
// stream, W and dL/dW both held in registers.
//
// Forward ("Metalearning Continual Learning Algorithms", section 2.3,
// Eqs. (1)-(5)), per step t with x~ = x or softmax(x):
//   z = W x~;  y = z[0:d];  pk = phi(z[d:2d]);  pq = phi(z[2d:3d]);  g = sigmoid(beta)
//   u = pq - pk;  a = W u;  coef_r = g_blk(r) a_r;  W' = W + coef (outer) pk
// Backward through one step, from dW' = dL/dW' and dy:
//   W      = W' - coef (outer) pk                  (the recorded update, subtracted)
//   dcoef  = dW' pk;   da = g dcoef;   dg_blk = sum_{r in blk} dcoef_r a_r
//   dpk    = dW'^T coef - W^T da;   dpq = W^T da
//   dk     = pk (dpk - <pk, dpk>);  dq = pq (dpq - <pq, dpq>);  dbeta = dg g (1 - g)
//   dz     = [dy, dk, dq, dbeta];   dx~ = W^T dz
//   dW     = dW' + da (outer) u + dz (outer) x~
// (and dx = x~ (dx~ - <x~, dx~>) when the input goes through softmax).
//
// Memory: the pages name "memory-efficient" backpropagation through time
// without details.  Here the forward pass (the fast forward kernels, with
// their record output on) writes per step the quantities the backward needs:
// phi(k), u, the gates and a (about 1.3 KB per step and stream at d = 64).
// This kernel starts from W_T and walks the steps backwards: each step
// subtracts from W exactly the recorded rank-one update the forward added
// (no matrix inversion, which would amplify rounding wherever the update
// contracts W), so W_{t-1} is recovered to within a few ulps that grow like
// sqrt(T).  x~, dy and the forward's records are staged per KSEG-step
// segment by bulk asynchronous copies into one of two buffers, the next
// segment's while the current one's steps run.
// Layout: thread (rg = tid/4, cg = tid%4) holds rows rg + RG i (i < S) and the
// D/4 columns of float4 chunks cg + 4 j.  Row dot products finish with two xor
// shuffles over the four column groups; column sums over rows finish with a
// transposed butterfly over the eight row groups of a warp and a fixed-order
// sum over warps in shared memory, so the result is deterministic.  A step's
// W^T dz (its dL/dx~) is summed inside the next step's column sum, with that
// step's two vectors, so a step takes two CTA barriers; the last step of a
// segment sums its own.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "srwm_common.h"
#include "srwm_ptx.cuh"

namespace srwm {

struct BwdParams {
    const float* x;        // [B, T, H, D]
    float* WT;             // [B, H, M, D]: W_T of every stream, from the forward pass (and a
                           // split stream's hand-off of W, see wrap_len)
    const float* rec;      // the forward's per-step records (KParams::emit layout)
    int rec_stride;        // floats per record
    const float* dy;       // [B, T, H, D]
    const float* dWf;      // [B, H, M, D] or nullptr (zero)
    float* dx;             // [B, T, H, D]
    float* dW_seq;         // [B, H, M, D]: dL/dW0 of every stream (summed over b later)
    int B, T, H;
    // > 0: the wrap-around schedule over the streams' steps taken backwards
    // (position r of stream p is step T - 1 - r; see wrap_next).  A stream
    // split in two hands W (through WT) and dL/dW (through dW_seq) from its
    // later part to its earlier part, which waits on the stream's counter.
    long long wrap_len;
    int* seg_done;                     // per-stream counters (wrap schedule only)
    unsigned* status;                  // device status word
    unsigned long long wait_limit_ns;  // bounded-wait limit
};

// Bulk copy of `bytes` global -> shared, completing `bytes` on bar (both
// addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

template <int D_, int NLR_>
struct BwdCfg {
    static constexpr int D = D_, NLR = NLR_;
    static constexpr int M = 3 * D + NLR;
    static constexpr int NW = D == 64 ? 8 : (D == 32 ? 4 : 2);
    static constexpr int NT = 32 * NW;
    static constexpr int RG = 8 * NW;            // row groups
    static constexpr int S = cdiv(M, RG);        // row slots per thread
    static constexpr int MP = S * RG;            // padded rows
    static constexpr int CPT = D / 4;            // columns per thread
    static constexpr int NCH = CPT / 4;          // float4 chunks per thread
    static constexpr int KSEG = D == 16 ? 16 : 32;   // steps per segment (two buffers of them)
    static constexpr int RS = emit_record_floats(D, NLR);   // floats per record
    static constexpr int NV2 = 2 * CPT;          // values of a two-vector column reduction
    static constexpr int NV1 = CPT < 8 ? 8 : CPT;  // one-vector reduction (padded to 8)
    static constexpr int NV3 = NV2 + NV1;        // two vectors and one carried (padded)
};

template <class C>
struct __align__(128) BwdSmem {
    // a segment's steps, by buffer: the forward's records as written
    // ([phi(k) | u | gates | a], KParams::emit layout), x~ and dy
    float rec[2][C::KSEG][C::RS];
    float xs[2][C::KSEG][C::D];
    float dyv[2][C::KSEG][C::D];
    uint64_t bar[2];             // "segment landed", by buffer
    float red[C::NW][3][C::D];   // per-warp column partials
    float vec[3][C::D];          // column sums
    float bred[C::NW][4];        // per-warp block sums of dcoef a
    float bsum[4];               // their sums over warps
};

template <class C>
__device__ __forceinline__ int bcol(int cg, int q) { return 4 * (cg + 4 * (q >> 2)) + (q & 3); }

// Transposed butterfly over the 8 row groups of a warp (lanes with equal
// lane%4): afterwards lane holds in v[0 .. N/8) the sums of the entries
// rg_lo*N/8 .. rg_lo*N/8 + N/8 - 1, where rg_lo = (lane / 4) % 8.
template <int N>
__device__ __forceinline__ void rowgroup_reduce(float (&v)[N], int lane)
{
    static_assert(N % 8 == 0, "N must be a multiple of 8");
#pragma unroll
    for (int lvl = 0; lvl < 3; ++lvl) {
        const int mask = 16 >> lvl;
        const int half = N >> (lvl + 1);
        const bool hi = (lane & mask) != 0;
#pragma unroll
        for (int e = 0; e < half; ++e) {
            const float send = hi ? v[e] : v[e + half];
            const float keep = hi ? v[e + half] : v[e];
            v[e] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
    }
}

// softmax over the D values in[0..D) by one warp; writes out[0..D).
template <int D>
__device__ __forceinline__ void warp_softmax(const float* in, float* out, int lane)
{
    if constexpr (D == 64) {
        float p0, p1;
        softmax64(in[lane], in[lane + 32], p0, p1);
        out[lane] = p0;
        out[lane + 32] = p1;
    } else {
        const int c = lane & (D - 1);
        const float mx = redux_max(in[c]);
        const float e = __expf(in[c] - mx);
        float sum = warp_sum_unit1(e);
        if constexpr (D == 16) sum *= 0.5f;
        if (lane < D) out[c] = e * rcp_approx(sum);
    }
}

// softmax backward over D values by one warp: out = s (gin - <s, gin>).
template <int D>
__device__ __forceinline__ void warp_softmax_bwd(const float* s, const float* gin, float* out, int lane)
{
    float dot = 0.f;
    for (int c = lane; c < D; c += 32) dot = fmaf(s[c], gin[c], dot);
    dot = group_sum<32>(dot);
    for (int c = lane; c < D; c += 32) out[c] = s[c] * (gin[c] - dot);
}

// Co-resident CTAs per SM the register budget is sized for: one at d = 64
// (W and dL/dW fill the registers), three at d = 32 and eight at d = 16, which
// fit without spills and hide more latency than the unconstrained allocation
// (measured on rl: 4.28 -> 3.59 ms for the whole backward call).
template <int D>
constexpr int bwd_ctas_per_sm() { return D == 32 ? 3 : (D == 16 ? 8 : 1); }

template <int D, int NLR>
__global__ void __launch_bounds__(BwdCfg<D, NLR>::NT, bwd_ctas_per_sm<D>())
    srwm_bwd_kernel(const BwdParams bp, int softmax_input)
{
    using C = BwdCfg<D, NLR>;
    constexpr int M = C::M, S = C::S, RG = C::RG, CPT = C::CPT, KSEG = C::KSEG;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<C>& sm = *reinterpret_cast<BwdSmem<C>*>(smem_raw);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = tid >> 2, cg = tid & 3;
    int p = blockIdx.x, b = 0, h = 0;   // the current piece's stream
    const int T = bp.T;
    const size_t MD = static_cast<size_t>(M) * D;
    auto blk = [](int r) { return NLR == 1 ? 0 : (r < 3 * D ? r / D : 3); };
    auto gidx = [&](int r) { return blk(r); };

    // W and dL/dW as pairs of adjacent columns (2q, 2q+1 of the thread's
    // columns) for the two-wide FMA
    constexpr int CP = CPT / 2;
    float2 w[S][CP], dw[S][CP];

    auto load_state = [&](const float* src) {
#pragma unroll
        for (int i = 0; i < S; ++i) {
            const int r = rg + RG * i;
#pragma unroll
            for (int j = 0; j < C::NCH; ++j) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < M) v = __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(r) * D + 4 * (cg + 4 * j)));
                w[i][2 * j] = make_float2(v.x, v.y);
                w[i][2 * j + 1] = make_float2(v.z, v.w);
            }
        }
    };
    auto store_tile = [&](float2 (&m)[S][CP], float* dst) {
#pragma unroll
        for (int i = 0; i < S; ++i) {
            const int r = rg + RG * i;
            if (r >= M) continue;
#pragma unroll
            for (int j = 0; j < C::NCH; ++j)
                *reinterpret_cast<float4*>(dst + static_cast<size_t>(r) * D + 4 * (cg + 4 * j)) =
                    make_float4(m[i][2 * j].x, m[i][2 * j].y, m[i][2 * j + 1].x, m[i][2 * j + 1].y);
        }
    };
    // ---- segment staging: one thread per row issues bulk copies of x and dy
    // rows, lane 0 of warp 0 the segment's records (contiguous per stream) and
    // the expected byte count; completion on sm.bar[buffer]
    if (tid == 0) {
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    int n_issued = 0, n_used = 0;   // segments issued / consumed by this CTA (buffer = count % 2)
    bool in_flight[2] = {false, false};
    auto issue = [&](int t0, int len) {
        const int buf = n_issued & 1;
        ++n_issued;
        in_flight[buf] = true;
        if (warp != 0) return;
        const uint32_t row_bytes = D * 4, rec_bytes = static_cast<uint32_t>(len) * C::RS * 4;
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.bar[buf], 2 * len * row_bytes + rec_bytes);
            bulk_load(&sm.rec[buf][0][0], bp.rec + (static_cast<size_t>(p) * T + t0) * C::RS, rec_bytes, &sm.bar[buf]);
        }
        for (int s = lane; s < len; s += 32) {
            const size_t g = ((static_cast<size_t>(b) * T + t0 + s) * bp.H + h) * D;
            bulk_load(&sm.xs[buf][s][0], bp.x + g, row_bytes, &sm.bar[buf]);
            bulk_load(&sm.dyv[buf][s][0], bp.dy + g, row_bytes, &sm.bar[buf]);
        }
    };
    // waits (bounded) for the next issued segment; false on a timeout (every
    // thread agrees)
    auto land = [&]() -> bool {
        const int buf = n_used & 1;
        const uint32_t par = (n_used >> 1) & 1;
        const bool ok = mbar_wait_bounded(&sm.bar[buf], par, bp.wait_limit_ns);
        if (__syncthreads_or(!ok)) return false;
        in_flight[buf] = false;
        ++n_used;
        return true;
    };
    // before giving up the shared memory: the copies still in flight land
    auto drain = [&]() {
        for (int k = n_used; k < n_issued; ++k) {
            const int buf = k & 1;
            if (in_flight[buf]) mbar_wait_bounded(&sm.bar[buf], (k >> 1) & 1, bp.wait_limit_ns);
        }
    };
    // column sums over all rows of per-thread partials v[N] (N/CPT vectors):
    // afterwards sm.vec[vv][c] holds vector vv at column c
    auto colsum = [&](auto& v, int nvec) {
        constexpr int N = sizeof(v) / sizeof(float);
        rowgroup_reduce<N>(v, lane);
        const int rg_lo = (lane >> 2) & 7;
#pragma unroll
        for (int e = 0; e < N / 8; ++e) {
            const int idx = rg_lo * (N / 8) + e;
            const int vv = idx / CPT, q = idx - vv * CPT;
            if (vv < nvec) sm.red[warp][vv][bcol<C>(cg, q)] = v[e];
        }
        __syncthreads();
        for (int idx = tid; idx < nvec * D; idx += C::NT) {
            const int vv = idx / D, c = idx - vv * D;
            float acc = 0.f;
            for (int ww = 0; ww < C::NW; ++ww) acc += sm.red[ww][vv][c];
            sm.vec[vv][c] = acc;
        }
        __syncthreads();
    };

    // colsum with two vectors, plus four block sums (bs: per-thread partials):
    // afterwards sm.vec[0..1] hold the column sums and sm.bsum[0..3] the
    // block sums, all in a fixed order of warps (deterministic)
    auto colsum_gate = [&](float (&v)[C::NV3], float (&bsum4)[4]) {
        constexpr int N = C::NV3;
        rowgroup_reduce<N>(v, lane);
        const int rg_lo = (lane >> 2) & 7;
#pragma unroll
        for (int e = 0; e < N / 8; ++e) {
            const int idx = rg_lo * (N / 8) + e;
            const int vv = idx / CPT, q = idx - vv * CPT;
            if (vv < 3) sm.red[warp][vv][bcol<C>(cg, q)] = v[e];
        }
        // the block sums over the warp's 32 lanes: two transposed levels,
        // then three plain ones; lane bits (4, 3) select the block
        {
            const bool hi16 = (lane & 16) != 0;
            float k0 = hi16 ? bsum4[2] : bsum4[0], k1 = hi16 ? bsum4[3] : bsum4[1];
            const float s0 = hi16 ? bsum4[0] : bsum4[2], s1 = hi16 ? bsum4[1] : bsum4[3];
            k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
            k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
            const bool hi8 = (lane & 8) != 0;
            float k = hi8 ? k1 : k0;
            k += __shfl_xor_sync(0xffffffffu, hi8 ? k0 : k1, 8);
            k += __shfl_xor_sync(0xffffffffu, k, 4);
            k += __shfl_xor_sync(0xffffffffu, k, 2);
            k += __shfl_xor_sync(0xffffffffu, k, 1);
            if ((lane & 7) == 0) sm.bred[warp][lane >> 3] = k;
        }
        __syncthreads();
        for (int idx = tid; idx < 3 * D + 4; idx += C::NT) {
            float acc = 0.f;
            if (idx < 3 * D) {
                const int vv = idx / D, c = idx - vv * D;
                for (int ww = 0; ww < C::NW; ++ww) acc += sm.red[ww][vv][c];
                sm.vec[vv][c] = acc;
            } else {
                for (int ww = 0; ww < C::NW; ++ww) acc += sm.bred[ww][idx - 3 * D];
                sm.bsum[idx - 3 * D] = acc;
            }
        }
        __syncthreads();
    };

    // ---- this CTA's pieces: one whole stream (plain launch), or the
    // wrap-around schedule's pieces taken backwards in time
    long long lo = 0, hi = 0;
    if (bp.wrap_len > 0) {
        lo = static_cast<long long>(blockIdx.x) * bp.wrap_len;
        hi = min(lo + bp.wrap_len, static_cast<long long>(bp.B) * bp.H * T);
    }
    bool first = true;
    for (;;) {
        int t_lo = 0, t_hi = T, seg = 0;   // steps t_lo .. t_hi - 1 of stream p
        if (bp.wrap_len > 0) {
            Piece pc;
            if (!wrap_next(lo, hi, T, pc)) break;
            p = pc.p;
            t_hi = T - pc.t0;
            t_lo = t_hi - pc.len;
            seg = pc.seg;
        } else if (!first) {
            break;
        }
        first = false;
        b = p / bp.H;
        h = p - b * bp.H;
        if (seg > 0) {
            int fail = 0;
            if (tid == 0) fail = !wait_counter_bounded(bp.seg_done + p, seg, bp.wait_limit_ns);
            if (__syncthreads_or(fail)) {
                if (tid == 0) atomicOr(bp.status, kStatusTimeout);
                drain();
                return;
            }
        }

    // ---- W at step t_hi (W_T from the forward pass, or where the later part
    // of the stream left it) and dL/dW there
    load_state(bp.WT + static_cast<size_t>(p) * MD);
    {
        const float* dsrc = seg > 0 ? bp.dW_seq + static_cast<size_t>(p) * MD
                                    : (bp.dWf != nullptr ? bp.dWf + static_cast<size_t>(p) * MD : nullptr);
#pragma unroll
        for (int i = 0; i < S; ++i) {
            const int r = rg + RG * i;
#pragma unroll
            for (int j = 0; j < C::NCH; ++j) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (dsrc != nullptr && r < M)
                    v = __ldcg(reinterpret_cast<const float4*>(dsrc + static_cast<size_t>(r) * D + 4 * (cg + 4 * j)));
                dw[i][2 * j] = make_float2(v.x, v.y);
                dw[i][2 * j + 1] = make_float2(v.z, v.w);
            }
        }
    }
    // ---- segments backwards; each step subtracts its recorded update from W.
    // The copies into a buffer follow the reads of the segment before last
    // (the barrier ending a segment) and the proxy fence of every thread.
    fence_proxy_async_smem();
    __syncthreads();
    if (t_hi > t_lo) issue(max(t_lo, t_hi - KSEG), min(KSEG, t_hi - t_lo));
    for (int top = t_hi; top > t_lo; top -= KSEG) {
        const int t0 = max(t_lo, top - KSEG);
        const int len = top - t0;
        const int buf = n_used & 1;
        if (!land()) {
            if (tid == 0) atomicOr(bp.status, kStatusTimeout);
            drain();
            return;
        }
        if (softmax_input) {
            for (int s = warp; s < len; s += C::NW) warp_softmax<D>(sm.xs[buf][s], sm.xs[buf][s], lane);
            fence_proxy_async_smem();
            __syncthreads();
        }
        // the next segment (earlier steps) into the other buffer
        if (t0 > t_lo) issue(max(t_lo, t0 - KSEG), min(KSEG, t0 - t_lo));
        const float* rec = &sm.rec[buf][0][0];
        // dL/dx of step s of this segment from the column sums in sm.vec[vv]
        // (through the input softmax when present)
        auto write_dx = [&](int s, int vv) {
            const size_t gx = ((static_cast<size_t>(b) * T + t0 + s) * bp.H + h) * D;
            if (softmax_input) {
                if (warp == 0) {
                    const float* dxv = sm.vec[vv];
                    float dot = 0.f;
                    for (int c = lane; c < D; c += 32) dot = fmaf(sm.xs[buf][s][c], dxv[c], dot);
                    dot = group_sum<32>(dot);
                    for (int c = lane; c < D; c += 32) bp.dx[gx + c] = sm.xs[buf][s][c] * (dxv[c] - dot);
                }
            } else if (tid < D) {
                bp.dx[gx + tid] = sm.vec[vv][tid];
            }
        };
        // W^T dz partials of the step before (summed in this step's column sum)
        float cxp[C::NV1];
#pragma unroll
        for (int q = 0; q < C::NV1; ++q) cxp[q] = 0.f;
        auto pk_of = [&](int s) { return rec + s * C::RS; };
        auto u_of = [&](int s) { return rec + s * C::RS + D; };
        auto g_of = [&](int s, int blkidx) { return rec[s * C::RS + 2 * D + blkidx]; };
        auto a_of = [&](int s, int r) { return r < M ? rec[s * C::RS + 2 * D + 4 + r] : 0.f; };
        for (int s = len - 1; s >= 0; --s) {
            // 1. step back: W_{t-1} = W_t - coef (outer) pk; dcoef = dW pk
            float av[S], dco[S];
#pragma unroll
            for (int i = 0; i < S; ++i) {
                const int r = rg + RG * i;
                av[i] = a_of(s, r);
                const float coef = g_of(s, gidx(r)) * av[i];
                const float2 nc = make_float2(-coef, -coef);
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < CP; ++q) {
                    const float2 pk2 = *reinterpret_cast<const float2*>(pk_of(s) + bcol<C>(cg, 2 * q));
                    w[i][q] = __ffma2_rn(nc, pk2, w[i][q]);
                    acc = __ffma2_rn(dw[i][q], pk2, acc);
                }
                dco[i] = acc.x + acc.y;
            }
#pragma unroll
            for (int i = 0; i < S; ++i) {
                dco[i] += __shfl_xor_sync(0xffffffffu, dco[i], 1);
                dco[i] += __shfl_xor_sync(0xffffffffu, dco[i], 2);
            }
            // 2. column sums v1 = dW'^T coef, v2 = W^T da, and the gate
            // gradients' block sums of dcoef a (slot i is block i here)
            float da[S];
            float cv[C::NV3];
            float bs[4];
            {
                float2 c1[CP], c2[CP];
#pragma unroll
                for (int q = 0; q < CP; ++q) c1[q] = c2[q] = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < S; ++i) {
                    const int r = rg + RG * i;
                    const float g = g_of(s, gidx(r));
                    const float coef = g * av[i];
                    da[i] = g * dco[i];
                    bs[i] = cg == 0 ? dco[i] * av[i] : 0.f;
                    const float2 cc = make_float2(coef, coef), dd = make_float2(da[i], da[i]);
#pragma unroll
                    for (int q = 0; q < CP; ++q) {
                        c1[q] = __ffma2_rn(dw[i][q], cc, c1[q]);
                        c2[q] = __ffma2_rn(w[i][q], dd, c2[q]);
                    }
                }
#pragma unroll
                for (int q = 0; q < CP; ++q) {
                    cv[2 * q] = c1[q].x;
                    cv[2 * q + 1] = c1[q].y;
                    cv[CPT + 2 * q] = c2[q].x;
                    cv[CPT + 2 * q + 1] = c2[q].y;
                }
#pragma unroll
                for (int q = 0; q < C::NV1; ++q) cv[C::NV2 + q] = cxp[q];
            }
            if constexpr (NLR == 1) {
                bs[0] = (bs[0] + bs[1]) + (bs[2] + bs[3]);
                bs[1] = bs[2] = bs[3] = 0.f;
            }
            // sm.vec[0] = v1, sm.vec[1] = v2, sm.vec[2] = dx~ of step s + 1, sm.bsum[j] = block j's sum
            colsum_gate(cv, bs);
            if (s + 1 < len) write_dx(s + 1, 2);
            // 3. dz for this thread's rows: y row dy; k, q rows through the
            // softmax backward; beta row through the sigmoid
            float dz[S];
            {
                const float* v1 = sm.vec[0];
                const float* v2 = sm.vec[1];
                float dk = 0.f, dq = 0.f;   // <phi(k), dphi(k)>, <phi(q), dphi(q)>
                for (int c = lane; c < D; c += 32) {
                    const float pkc = pk_of(s)[c], pqc = u_of(s)[c] + pkc;
                    dk = fmaf(pkc, v1[c] - v2[c], dk);
                    dq = fmaf(pqc, v2[c], dq);
                }
                dk = group_sum<32>(dk);
                dq = group_sum<32>(dq);
                const float pkr = pk_of(s)[rg], pqr = u_of(s)[rg] + pkr;
                dz[0] = sm.dyv[buf][s][rg];
                dz[1] = pkr * ((v1[rg] - v2[rg]) - dk);
                dz[2] = pqr * (v2[rg] - dq);
                dz[3] = 0.f;
                if (rg < NLR) {
                    const float g = g_of(s, rg);
                    dz[3] = sm.bsum[rg] * g * (1.f - g);
                }
            }
            // 4. dW += da (outer) u + dz (outer) x~ ; column partials of W^T dz
            {
                float2 c3[CP];
#pragma unroll
                for (int q = 0; q < CP; ++q) c3[q] = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < S; ++i) {
                    const float2 dd = make_float2(da[i], da[i]), zz = make_float2(dz[i], dz[i]);
#pragma unroll
                    for (int q = 0; q < CP; ++q) {
                        const int c = bcol<C>(cg, 2 * q);
                        dw[i][q] = __ffma2_rn(dd, *reinterpret_cast<const float2*>(u_of(s) + c), dw[i][q]);
                        dw[i][q] = __ffma2_rn(zz, *reinterpret_cast<const float2*>(&sm.xs[buf][s][c]), dw[i][q]);
                        c3[q] = __ffma2_rn(w[i][q], zz, c3[q]);
                    }
                }
#pragma unroll
                for (int q = 0; q < CP; ++q) {
                    cxp[2 * q] = c3[q].x;
                    cxp[2 * q + 1] = c3[q].y;
                }
            }
        }
        // the segment's last step (its earliest): its own column sum
        colsum(cxp, 1);   // sm.vec[0] = dx~ of step 0
        write_dx(0, 0);
        // the segment's buffer is read before copies into it (two segments on)
        fence_proxy_async_smem();
        __syncthreads();
    }
    store_tile(dw, bp.dW_seq + static_cast<size_t>(p) * MD);
    if (t_lo > 0) {
        // the earlier part of the stream continues from here
        store_tile(w, bp.WT + static_cast<size_t>(p) * MD);
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            st_release_gpu(bp.seg_done + p, seg + 1);
        }
    }
    }
}

struct BwdLaunch {
    const void* kernel;
    int threads;
    int smem_bytes;
    int kseg;
};

template <int D, int NLR>
BwdLaunch bwd_launch_info()
{
    using C = BwdCfg<D, NLR>;
    return BwdLaunch{reinterpret_cast<const void*>(&srwm_bwd_kernel<D, NLR>), C::NT,
                     static_cast<int>(sizeof(BwdSmem<C>)), C::KSEG};
}

BwdLaunch bwd_info(int d, int n_lr);
int launch_sum_over_batch(const float* dW_seq, float* dW0, int B, size_t per_batch, cudaStream_t stream);

}  // namespace srwm
