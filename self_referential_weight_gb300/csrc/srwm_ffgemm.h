// srwm_ffgemm.h -- host interface of the tensor-core feed-forward products
// (srwm_ffgemm.cu), used by the layer (srwm_layer.cu).
#pragma once

#include <cuda_runtime.h>

namespace srwm {

struct GemmArgs {
    long long N;                 // rows of A and of the output (tokens)
    int K;                       // inner dimension (a multiple of 8)
    int Mo;                      // rows of B = output columns (a multiple of 8)
    const float* bias;           // [Mo]
    float* out;                  // epilogue 2: [N, Mo] fp32, accumulated onto
    void* out_hi;                // epilogue 1: [N, Mo] bf16 (hi, lo) of ReLU(A B^T + bias)
    void* out_lo;
    unsigned* status;            // device status word
    unsigned long long wait_limit_ns;
};

// The library's device status word and bounded-wait limit (srwm_api.cu).
int device_status_ptr(unsigned** out);
unsigned long long device_wait_limit_ns();

// fp32 [n] -> bf16 hi and lo parts (x ~ hi + lo)
int ff_split(const float* src, void* hi, void* lo, long long n, cudaStream_t st);

// Out = epilogue(A B^T) with A = A_hi + A_lo [N, K] and B = B_hi + B_lo [Mo, K]
// as bf16 pairs (row-major): epi 1 writes ReLU(. + bias) as a bf16 pair, epi 2
// adds . + bias onto the fp32 out.
int ff_gemm(int epi, const void* a_hi, const void* a_lo, const void* b_hi, const void* b_lo, const GemmArgs& args,
            cudaStream_t st);

}  // namespace srwm
