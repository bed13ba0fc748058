// srwm_ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers with bounded
// waits, TMA tiled loads/stores (cp.async.bulk.tensor) and warp reductions.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "srwm_common.h"

namespace srwm {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The kernels lay their shared-memory structures out from the dynamic shared
// memory base, which they take to be 128-byte aligned (TMA buffers sit at
// 128-byte offsets from it).  Checked once at entry: on a misaligned base the
// CTA reports it in the status word and returns before touching anything.
__device__ __forceinline__ bool smem_base_ok(const void* base, unsigned* status)
{
    if ((smem_u32(base) & 127u) == 0) return true;
    if (threadIdx.x == 0) atomicOr(status, kStatusSmemBase);
    return false;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, for at most limit_ns of
// wall time.  Returns false when the limit ran out (the caller reports it).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- TMA
// Tiled 4-D load global -> shared, completing `bytes` on `bar`.  The innermost
// coordinate is always 0 here, so the 16-byte rule on it holds trivially.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar))
        : "memory");
}

// Tiled 4-D store shared -> global; rows outside the tensor are not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group"
        " [%0, {%1, %2, %3, %4}], [%5];" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed bulk groups are still in flight at all.
template <int N>
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- cross-CTA counters
__device__ __forceinline__ int ld_acquire_gpu(const int* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits until *p >= target (another CTA or warp of the same cooperative grid
// publishes it), for at most limit_ns.  Returns false when the limit ran out.
__device__ __forceinline__ bool wait_counter_bounded(const int* p, int target, uint64_t limit_ns)
{
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(100);
        if (ld_acquire_gpu(p) >= target) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- reductions
// Butterfly reductions over aligned groups of W lanes (W a power of two).
// Every lane of a group ends with the same bits: each level adds the same two
// operands on both sides, and float addition is commutative.
template <int W>
__device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int W>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------- fast softmax pieces
// (shared by the kernels; results are identical on every lane of the warp)
__device__ __forceinline__ float redux_max(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ uint32_t redux_add(uint32_t v)
{
    uint32_t r;
    asm volatile("redux.sync.add.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
    return r;
}

__device__ __forceinline__ float rcp_approx(float v)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// Warp sum of one value in [0, 1] per lane, exact in fixed point (2^-31 steps).
__device__ __forceinline__ float warp_sum_unit1(float e)
{
    const uint32_t q = __float2uint_rn(e * 2147483648.0f);
    const uint32_t hi = redux_add(q >> 16);
    const uint32_t lo = redux_add(q & 0xffffu);
    return fmaf(static_cast<float>(hi), 3.0517578125e-05f, static_cast<float>(lo) * 4.656612873077393e-10f);
}

// Warp sum of two values in [0, 1] per lane, exact in fixed point with 2^-31
// resolution (16-bit halves keep the u32 sums from overflowing).  Every lane
// gets the same bits whatever the order of lanes.
__device__ __forceinline__ float warp_sum_unit(float e0, float e1)
{
    const uint32_t q0 = __float2uint_rn(e0 * 2147483648.0f);
    const uint32_t q1 = __float2uint_rn(e1 * 2147483648.0f);
    const uint32_t hi = redux_add((q0 >> 16) + (q1 >> 16));
    const uint32_t lo = redux_add((q0 & 0xffffu) + (q1 & 0xffffu));
    return fmaf(static_cast<float>(hi), 3.0517578125e-05f, static_cast<float>(lo) * 4.656612873077393e-10f);
}

// softmax over 64 values held as (v0, v1) = entries (lane, lane + 32).
__device__ __forceinline__ void softmax64(float v0, float v1, float& p0, float& p1)
{
    const float mx = redux_max(fmaxf(v0, v1));
    const float e0 = __expf(v0 - mx), e1 = __expf(v1 - mx);
    const float inv = rcp_approx(warp_sum_unit(e0, e1));
    p0 = e0 * inv;
    p1 = e1 * inv;
}

__device__ __forceinline__ float sigmoid_fast(float v) { return rcp_approx(1.0f + __expf(-v)); }


}  // namespace srwm
