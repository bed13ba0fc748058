// srwm_common.h -- definitions shared by the kernels and the host-side C ABI.
#pragma once

#if defined(__CUDACC__)
#define SRWM_HD __host__ __device__
#else
#define SRWM_HD
#endif

namespace srwm {

SRWM_HD constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }
SRWM_HD constexpr int rup(int a, int b) { return cdiv(a, b) * b; }

// Bits of the device status word.
constexpr unsigned kStatusTimeout = 1u;

// Kernel arguments besides the two tensor maps.
struct KParams {
    const float* W_init;               // [H,m,d] shared, or [B,H,m,d] per sequence
    float* W_out;                      // [B,H,m,d]
    unsigned* status;                  // device status word
    unsigned long long wait_limit_ns;  // bounded-wait limit
    int B, T, H;
    int w_per_seq;                     // 1: W_init is per sequence
    int skip_chunk;                    // fault injection: x chunk not loaded (-1: none)
    // Work items: every stream's T steps are cut into segments of seg_len
    // steps (a multiple of each kernel's TMA chunk; seg_len >= T means one
    // segment).  Item j is segment j / n_streams of stream j % n_streams, and a
    // CTA (d = 64) or warp (d = 16, 32) takes items slot, slot + n_slots, ...
    int n_streams;                     // B * H
    int seg_len;                       // steps per item
    int n_items;                       // n_streams * segments
    // Per-stream count of finished segments (only when streams span several
    // segments; NULL otherwise).  Segment s of a stream waits until its count
    // reaches s; its state comes from W_out, where segment s - 1 left it.
    int* seg_done;
    // Per-step records for the backward pass (NULL: none).  Record of stream p,
    // step t (of the whole sequence) at emit + (p * T + t) * emit_stride:
    //   [phi(k_t) (d) | u_t = phi(q_t) - phi(k_t) (d) | gates (4) | a_t = W_{t-1} u_t (m)]
    float* emit;
    int emit_stride;   // floats per record, a multiple of 4
};

// Floats per backward record (see KParams::emit), rounded up to 16 bytes.
SRWM_HD constexpr int emit_record_floats(int d, int n_lr) { return (2 * d + 4 + 3 * d + n_lr + 3) / 4 * 4; }

// What the host needs to launch one template instantiation.
struct LaunchInfo {
    const void* kernel;   // __global__ function
    int threads;          // per CTA
    int streams_per_cta;  // (sequence, head) streams per CTA
    int smem_bytes;       // dynamic shared memory
    int tau;              // steps per TMA chunk (box height of the x / y tensor maps)
};

// emit: the instantiation that also writes the backward records (KParams::emit).
LaunchInfo launch_info_d16(int n_lr, int softmax_input, bool emit = false);
LaunchInfo launch_info_d32(int n_lr, int softmax_input, bool emit = false);
LaunchInfo launch_info_d64(int n_lr, int softmax_input, long long n_streams, int n_sm, bool emit = false);

}  // namespace srwm
