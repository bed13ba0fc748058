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
// The dynamic shared memory base was not 128-byte aligned (the kernels place
// TMA buffers at 128-byte offsets from it); the kernel did nothing.
constexpr unsigned kStatusSmemBase = 2u;

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
    // > 0: the wrap-around schedule instead of segments (kernels whose
    // LaunchInfo::wraps is set): slot k takes the positions
    // [k * wrap_len, (k + 1) * wrap_len) of all streams' steps laid end to end
    // (see wrap_next).
    long long wrap_len;
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

// One piece of a slot's work: steps t0 .. t0 + len - 1 of stream p, the
// stream's segment number seg (its state comes from segment seg - 1).
struct Piece {
    int p, seg, t0, len;
};

// Wrap-around schedule.  Stream p's steps are the positions p*T .. p*T + T - 1
// of one line; a slot owns the range [lo, hi) of that line and takes it in
// pieces, last piece first: each call returns the piece that ends at hi and
// moves hi to its start.  With ranges of at least T positions a stream falls
// into at most two ranges.  Its first steps end one range and so run first on
// that slot; its last steps begin the next range and so run last on the next
// slot, and as the two parts add up to T <= range length, the second never
// has to wait long for the first (segment 1 waits on segment 0's counter).
SRWM_HD inline bool wrap_next(long long lo, long long& hi, int T, Piece& pc)
{
    if (hi <= lo || T <= 0) return false;
    const long long p = (hi - 1) / T;
    const long long start = lo > p * T ? lo : p * T;
    pc.p = static_cast<int>(p);
    pc.t0 = static_cast<int>(start - p * T);
    pc.len = static_cast<int>(hi - start);
    pc.seg = pc.t0 > 0 ? 1 : 0;
    hi = start;
    return true;
}

// Floats per backward record (see KParams::emit), rounded up to 16 bytes.
SRWM_HD constexpr int emit_record_floats(int d, int n_lr) { return (2 * d + 4 + 3 * d + n_lr + 3) / 4 * 4; }

// What the host needs to launch one template instantiation.
struct LaunchInfo {
    const void* kernel;   // __global__ function
    int threads;          // per CTA
    int streams_per_cta;  // (sequence, head) streams per CTA
    int smem_bytes;       // dynamic shared memory
    int tau;              // steps per TMA chunk (box height of the x / y tensor maps)
    bool wraps;           // takes the wrap-around schedule (KParams::wrap_len)
};

// emit: the instantiation that also writes the backward records (KParams::emit).
LaunchInfo launch_info_d16(int n_lr, int softmax_input, bool emit = false);
LaunchInfo launch_info_d32(int n_lr, int softmax_input, bool emit = false);
LaunchInfo launch_info_d64(int n_lr, int softmax_input, long long n_streams, int n_sm, bool emit = false);

}  // namespace srwm
