// srwm_ffgemm.cu -- the feed-forward products of the Recursive Self-Transformer
// layer on the 5th-generation tensor cores: TMA tile loads, tcgen05.mma with
// the accumulator in tensor memory, tcgen05.ld for the epilogue.
//
// fp32-level accuracy from BF16 tensor cores by a three-term split: every
// fp32 operand x is held as hi = bf16(x) and lo = bf16(x - hi), and
//   X W^T  ~  X_hi W_hi^T + X_hi W_lo^T + X_lo W_hi^T
// accumulated in fp32 (the dropped X_lo W_lo^T term and lo's own rounding are
// ~2^-16 of each product: ~1e-5 relative on the layer's output).
//
// Out[N, Mo] = epilogue(A[N, K] B[Mo, K]^T): A and B row-major, K contiguous
// ("K-major" for both tensor-core operands), as X and a PyTorch Linear weight.
// Epilogues: (1) f = ReLU(acc + bias) written as a bf16 (hi, lo) pair, the
// next product's A operand; (2) out = out + acc + bias in fp32 (out holds the
// residual).
//
// Persistent, warp-specialised CTA (one per SM): warp 0 issues the TMA loads,
// warp 1 the MMAs (one thread each), warps 2-5 run the epilogue, each on the
// 32 tensor-memory lanes (= tile rows) its warp may access.  Tiles of 128 x 256
// outputs; K in steps of 32 (a 64-byte swizzle row of bf16) over four shared-
// memory stages (A_hi, A_lo, B_hi, B_lo: 48 KB each), or for K <= 1024 in
// steps of 64 (128-byte swizzle) over two 96 KB stages; two accumulators in
// tensor memory (2 x 256 columns), so one tile's epilogue overlaps the next
// tile's products.  The epilogue stages each warp's 32 x 32 blocks in shared
// memory (two buffers per warp) and writes them with TMA: a store of the bf16
// pair (1), a reduce-add onto out (2).  Tensor memory holds one tile row per
// lane, so direct stores from registers would scatter every instruction over
// 32 rows; they made the epilogue the products' limit.  Every wait is
// bounded; a timeout sets the status word, stops new work, waits (bounded)
// for work in flight and frees the tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "srwm.h"
#include "srwm_common.h"
#include "srwm_ffgemm.h"
#include "srwm_ptx.cuh"

namespace srwm {
namespace ff {

constexpr int BM = 128, BN = 256, NACC = 2;
constexpr int NTHREADS = 192;

// K step (bf16 elements per swizzled tile row) and shared-memory stages.  The
// products of the layer: K = 512 (eight K steps per tile at BK = 64) is ~4 %
// faster with two 96 KB stages; K = 2048 ~14 % faster with four 48 KB stages
// (its 64 K steps per tile gain from the deeper pipeline).
template <int BK_>
struct Pipe {
    static constexpr int BK = BK_;
    static constexpr int STAGES = BK == 64 ? 2 : 4;
    static constexpr int TILE_A = BM * BK * 2;                    // bytes of one bf16 A tile
    static constexpr int TILE_B = BN * BK * 2;
    static constexpr int STAGE_BYTES = 2 * TILE_A + 2 * TILE_B;   // A_hi | A_lo | B_hi | B_lo
    static constexpr int SBO = BK * 2 * 8;                        // bytes between 8-row atoms
    static constexpr uint64_t SWZ = BK == 64 ? 2 : 4;             // descriptor swizzle mode: 128 / 64 bytes
    static_assert(BK == 32 || BK == 64, "K steps of 32 or 64");
    static_assert(STAGE_BYTES % 1024 == 0 && TILE_A % 1024 == 0 && TILE_B % 1024 == 0,
                  "swizzled tiles start on 1024-byte boundaries");
};
constexpr uint32_t TMEM_COLS = NACC * BN;              // 512: the whole tensor memory of the SM
constexpr int OBUF = 32 * 32 * 4;                      // one 32 x 32 output block: fp32, or the bf16 pair

template <class P>
struct __align__(1024) Smem {
    uint8_t stage[P::STAGES][P::STAGE_BYTES];
    uint8_t ostage[4][2][OBUF];                        // per epilogue warp, two blocks in flight
    uint64_t full[P::STAGES], empty[P::STAGES], acc_full[NACC], acc_empty[NACC];
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// TMA store of a 2-D box shared -> global (bulk group), and the reduce-add form
// (global += box, element type from the map)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}

__device__ __forceinline__ void tma_add_2d(const CUtensorMap* map, const void* src, int c0, int c1)
{
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// the swizzle of its row width (BK bf16 = 64 or 128 bytes): atoms of 8 rows,
// SBO bytes apart; the leading-dimension offset is not used by these layouts.
// Bits: start address >> 4 [0, 14), leading byte offset >> 4 [16, 30), stride
// byte offset >> 4 [32, 46), descriptor version 1 [46, 48), swizzle mode
// [61, 64) (2: 128-byte, 4: 64-byte).
template <class P>
__device__ __forceinline__ uint64_t tile_desc(uint32_t saddr)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(P::SBO >> 4) << 32) | (static_cast<uint64_t>(1) << 46) | (P::SWZ << 61);
}

// Instruction descriptor of tcgen05.mma.kind::f16: fp32 accumulator (bits
// [4, 6) = 1), bf16 A and B ([7, 10) = 1, [10, 13) = 1), both K-major (bits 15,
// 16 = 0), N >> 3 in [17, 23), M >> 4 in [24, 29).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on `bar` once every MMA this thread issued before it has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 columns of the warp's 32 tensor-memory lanes (one row per thread), then
// the wait for the load, in one statement so no use can move ahead of it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// x -> (hi, lo) with hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_bf16(float x, float& hi, float& lo)
{
    hi = __bfloat162float(__float2bfloat16_rn(x));
    lo = x - hi;
}

template <int EPI, class P>
__global__ void __launch_bounds__(NTHREADS, 1)
    ffgemm_kernel(const __grid_constant__ CUtensorMap ta_hi, const __grid_constant__ CUtensorMap ta_lo,
                  const __grid_constant__ CUtensorMap tb_hi, const __grid_constant__ CUtensorMap tb_lo,
                  const __grid_constant__ CUtensorMap to0, const __grid_constant__ CUtensorMap to1,
                  const GemmArgs ga)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    constexpr int BK = P::BK, STAGES = P::STAGES, TILE_A = P::TILE_A, TILE_B = P::TILE_B;
    constexpr int STAGE_BYTES = P::STAGE_BYTES;
    Smem<P>& sm = *reinterpret_cast<Smem<P>*>(smem_raw);
    if ((smem_u32(smem_raw) & 1023u) != 0) {   // the swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicOr(ga.status, kStatusSmemBase);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (ga.N + BM - 1) / BM, n_tiles = (ga.Mo + BN - 1) / BN;
    const int ntiles = m_tiles * n_tiles;
    const int kblocks = (ga.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(&sm.acc_full[a], 1);
            mbar_init(&sm.acc_empty[a], 4);
        }
        sm.abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&ta_hi);
        prefetch_tensormap(&ta_lo);
        prefetch_tensormap(&tb_hi);
        prefetch_tensormap(&tb_lo);
        prefetch_tensormap(&to0);
        if (EPI == 1) prefetch_tensormap(&to1);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sm.tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int* abort = &sm.abort;
    auto fail = [&]() {
        *abort = 1;
        atomicOr(ga.status, kStatusTimeout);
    };

    if (warp == 0) {
        // ---- TMA producer (one thread; the warp's other lanes wait at the end)
        if (lane == 0) {
        int it = 0, last_stage = -1;
        uint32_t last_parity = 0;
        for (int tile = blockIdx.x; tile < ntiles && !*abort; tile += gridDim.x) {
            const int m0 = (tile / n_tiles) * BM, n0 = (tile % n_tiles) * BN;
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                if (!mbar_wait_bounded(&sm.empty[s], ph ^ 1u, ga.wait_limit_ns)) {
                    fail();
                    break;
                }
                if (*abort) break;
                uint8_t* st = sm.stage[s];
                mbar_arrive_expect_tx(&sm.full[s], STAGE_BYTES);
                tma_load_2d(st, &ta_hi, &sm.full[s], kb * BK, m0);
                tma_load_2d(st + TILE_A, &ta_lo, &sm.full[s], kb * BK, m0);
                tma_load_2d(st + 2 * TILE_A, &tb_hi, &sm.full[s], kb * BK, n0);
                tma_load_2d(st + 2 * TILE_A + TILE_B, &tb_lo, &sm.full[s], kb * BK, n0);
                last_stage = s;
                last_parity = ph;
            }
        }
        // the shared memory may only be given up once the last loads landed
        if (last_stage >= 0) mbar_wait_bounded(&sm.full[last_stage], last_parity, ga.wait_limit_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer (one thread; the warp's other lanes wait at the end)
        if (lane == 0) {
        constexpr uint32_t idesc = idesc_bf16(BM, BN);
        int it = 0, li = 0;
        uint64_t* last_commit = nullptr;
        uint32_t last_commit_parity = 0;
        for (int tile = blockIdx.x; tile < ntiles && !*abort; tile += gridDim.x, ++li) {
            const int ab = li & 1;
            const uint32_t aph = (li >> 1) & 1;
            if (!mbar_wait_bounded(&sm.acc_empty[ab], aph ^ 1u, ga.wait_limit_ns)) {
                fail();
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + static_cast<uint32_t>(ab * BN);
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                if (!mbar_wait_bounded(&sm.full[s], ph, ga.wait_limit_ns) || *abort) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t base = smem_u32(sm.stage[s]);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    const uint32_t ko = static_cast<uint32_t>(k * 32);   // 16 bf16 along K
                    const uint64_t a_hi = tile_desc<P>(base + ko), a_lo = tile_desc<P>(base + TILE_A + ko);
                    const uint64_t b_hi = tile_desc<P>(base + 2 * TILE_A + ko);
                    const uint64_t b_lo = tile_desc<P>(base + 2 * TILE_A + TILE_B + ko);
                    umma(d, a_hi, b_hi, idesc, (kb | k) != 0 ? 1u : 0u);
                    umma(d, a_hi, b_lo, idesc, 1u);
                    umma(d, a_lo, b_hi, idesc, 1u);
                }
                umma_commit(&sm.empty[s]);   // the stage is free once these products have read it
                last_commit = &sm.empty[s];
                last_commit_parity = ph;
            }
            if (!ok) {
                fail();
                break;
            }
            umma_commit(&sm.acc_full[ab]);
            last_commit = &sm.acc_full[ab];
            last_commit_parity = aph;
        }
        // tensor memory may only be freed once the products issued completed
        if (last_commit) mbar_wait_bounded(last_commit, last_commit_parity, ga.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ---- epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31,
        // i.e. tile rows 32 (w % 4) .., 32 columns at a time; each 32 x 32
        // block goes through the warp's staging buffers to a TMA store
        const int q = warp & 3;
        int li = 0, nb = 0;   // tiles, blocks staged so far
        for (int tile = blockIdx.x; tile < ntiles && !*abort; tile += gridDim.x, ++li) {
            const int m0 = (tile / n_tiles) * BM, n0 = (tile % n_tiles) * BN;
            const int ab = li & 1;
            const uint32_t aph = (li >> 1) & 1;
            if (!mbar_wait_bounded(&sm.acc_full[ab], aph, ga.wait_limit_ns)) {
                if (lane == 0) fail();
                break;
            }
            tc_fence_after();
            const int r0 = m0 + 32 * q;   // first row of this warp's blocks
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                const int col0 = n0 + 32 * c;
                uint32_t r[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(ab * BN + 32 * c), r);
                if (c == BN / 32 - 1) {
                    // the accumulator may take the next tile
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.acc_empty[ab]);
                }
                if (col0 >= ga.Mo || r0 >= ga.N) continue;
                float v[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {   // bias of columns col0 + 4k .. (zero past the output's width)
                    const float4 b4 = col0 + 4 * k < ga.Mo ? __ldg(reinterpret_cast<const float4*>(ga.bias + col0 + 4 * k))
                                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[4 * k] = __uint_as_float(r[4 * k]) + b4.x;
                    v[4 * k + 1] = __uint_as_float(r[4 * k + 1]) + b4.y;
                    v[4 * k + 2] = __uint_as_float(r[4 * k + 2]) + b4.z;
                    v[4 * k + 3] = __uint_as_float(r[4 * k + 3]) + b4.w;
                }
                uint8_t* buf = sm.ostage[q][nb & 1];
                // the store that read this buffer two blocks ago is done with it
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();
                if constexpr (EPI == 1) {
                    // row `lane` of the hi block (64 bytes) and of the lo block
                    uint4* hrow = reinterpret_cast<uint4*>(buf + 64 * lane);
                    uint4* lrow = reinterpret_cast<uint4*>(buf + 2048 + 64 * lane);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float hi[8], lo[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) split_bf16(fmaxf(v[8 * k + j], 0.f), hi[j], lo[j]);
                        hrow[k] = make_uint4(pack_bf16(hi[0], hi[1]), pack_bf16(hi[2], hi[3]), pack_bf16(hi[4], hi[5]),
                                             pack_bf16(hi[6], hi[7]));
                        lrow[k] = make_uint4(pack_bf16(lo[0], lo[1]), pack_bf16(lo[2], lo[3]), pack_bf16(lo[4], lo[5]),
                                             pack_bf16(lo[6], lo[7]));
                    }
                } else {
                    // row `lane` (128 bytes) in the map's 128-byte swizzle: 16-byte chunk
                    // k sits at chunk k ^ (row % 8), so the eight lanes of a phase hit
                    // eight different bank groups
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<float4*>(buf + 128 * lane + 16 * (k ^ (lane & 7))) =
                            make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (EPI == 1) {
                        tma_store_2d(&to0, buf, col0, r0);
                        tma_store_2d(&to1, buf + 2048, col0, r0);
                    } else {
                        tma_add_2d(&to0, buf, col0, r0);
                    }
                    bulk_commit();
                }
                ++nb;
            }
        }
        // the blocks in flight are written before the CTA ends
        if (lane == 0) bulk_wait_all<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

// fp32 -> (bf16 hi, bf16 lo), elementwise
__global__ void split_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ hi,
                             __nv_bfloat16* __restrict__ lo, long long n)
{
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float x = src[i];
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        hi[i] = h;
        lo[i] = __float2bfloat16_rn(x - __bfloat162float(h));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// 2-D map over a row-major bf16 [rows, K] matrix: boxes of `box_rows` rows x
// bk columns, the swizzle of the box row (64 or 128 bytes), zero fill outside
// the matrix.
int make_map(CUtensorMap* map, const void* base, long long rows, int K, int box_rows, int bk)
{
    auto enc = encoder();
    if (!enc) return SRWM_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(bk), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SRWM_OK : SRWM_ERR_CUDA;
}

// 2-D map over a row-major [rows, cols] output (bf16 or fp32) in boxes of 32 x 32,
// the 128-byte swizzle for fp32 (a box row is 128 bytes), none for bf16.
int make_out_map(CUtensorMap* map, void* base, long long rows, int cols, bool fp32)
{
    auto enc = encoder();
    if (!enc) return SRWM_ERR_CUDA;
    const int es = fp32 ? 4 : 2;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * es};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base,
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           fp32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SRWM_OK : SRWM_ERR_CUDA;
}

}  // namespace ff

int ff_split(const float* src, void* hi, void* lo, long long n, cudaStream_t st)
{
    if (n <= 0) return SRWM_OK;
    const long long blocks = (n + 255) / 256;
    ff::split_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(
        src, static_cast<__nv_bfloat16*>(hi), static_cast<__nv_bfloat16*>(lo), n);
    return cudaGetLastError() == cudaSuccess ? SRWM_OK : SRWM_ERR_CUDA;
}

int ff_gemm(int epi, const void* a_hi, const void* a_lo, const void* b_hi, const void* b_lo, const GemmArgs& args,
            cudaStream_t st)
{
    using namespace ff;
    if (args.N <= 0 || args.Mo <= 0) return SRWM_OK;
    if (args.K <= 0 || args.K % 8 != 0 || args.Mo % 8 != 0) return SRWM_ERR_UNSUPPORTED;
    const int bk = args.K <= 1024 ? 64 : 32;
    CUtensorMap m[6];
    int rc;
    if ((rc = make_map(&m[0], a_hi, args.N, args.K, BM, bk)) != SRWM_OK ||
        (rc = make_map(&m[1], a_lo, args.N, args.K, BM, bk)) != SRWM_OK ||
        (rc = make_map(&m[2], b_hi, args.Mo, args.K, BN, bk)) != SRWM_OK ||
        (rc = make_map(&m[3], b_lo, args.Mo, args.K, BN, bk)) != SRWM_OK)
        return rc;
    if (epi == 1) {
        if ((rc = make_out_map(&m[4], args.out_hi, args.N, args.Mo, false)) != SRWM_OK ||
            (rc = make_out_map(&m[5], args.out_lo, args.N, args.Mo, false)) != SRWM_OK)
            return rc;
    } else {
        if ((rc = make_out_map(&m[4], args.out, args.N, args.Mo, true)) != SRWM_OK) return rc;
        m[5] = m[4];
    }
    const void* kern = bk == 64 ? (epi == 1 ? reinterpret_cast<const void*>(&ffgemm_kernel<1, Pipe<64>>)
                                            : reinterpret_cast<const void*>(&ffgemm_kernel<2, Pipe<64>>))
                                : (epi == 1 ? reinterpret_cast<const void*>(&ffgemm_kernel<1, Pipe<32>>)
                                            : reinterpret_cast<const void*>(&ffgemm_kernel<2, Pipe<32>>));
    const int smem = static_cast<int>(bk == 64 ? sizeof(Smem<Pipe<64>>) : sizeof(Smem<Pipe<32>>)) + 1024;
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    const long long ntiles = static_cast<long long>((args.N + BM - 1) / BM) * ((args.Mo + BN - 1) / BN);
    const unsigned grid = static_cast<unsigned>(ntiles < n_sm ? ntiles : n_sm);
    void* kargs[] = {&m[0], &m[1], &m[2], &m[3], &m[4], &m[5], const_cast<GemmArgs*>(&args)};
    if (cudaLaunchKernel(kern, dim3(grid), dim3(NTHREADS), kargs, static_cast<size_t>(smem), st) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    return SRWM_OK;
}

}  // namespace srwm
