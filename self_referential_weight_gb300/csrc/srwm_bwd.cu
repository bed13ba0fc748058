// srwm_bwd.cu -- instantiations of the backward kernel.
#include "srwm_bwd.cuh"

namespace srwm {

// dW0[h] = sum over b of dW_seq[b, h], in order of b (deterministic).
__global__ void srwm_sum_over_batch_kernel(const float* __restrict__ dW_seq, float* __restrict__ dW0, int B,
                                           size_t per_batch)
{
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < per_batch;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float acc = 0.f;
        for (int b = 0; b < B; ++b) acc += dW_seq[static_cast<size_t>(b) * per_batch + i];
        dW0[i] = acc;
    }
}

BwdLaunch bwd_info(int d, int n_lr)
{
    if (d == 16) return n_lr == 1 ? bwd_launch_info<16, 1>() : bwd_launch_info<16, 4>();
    if (d == 32) return n_lr == 1 ? bwd_launch_info<32, 1>() : bwd_launch_info<32, 4>();
    return n_lr == 1 ? bwd_launch_info<64, 1>() : bwd_launch_info<64, 4>();
}

int launch_sum_over_batch(const float* dW_seq, float* dW0, int B, size_t per_batch, cudaStream_t stream)
{
    const int threads = 256;
    size_t blocks = (per_batch + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    if (blocks == 0) blocks = 1;
    srwm_sum_over_batch_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(dW_seq, dW0, B, per_batch);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace srwm
