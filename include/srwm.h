/*
 * srwm.h -- C ABI of libsrwm.so: the forward recurrence of the multi-head
 * Self-Referential Weight Matrix (SRWM), hand-written for NVIDIA GB300 (sm_103a).
 *
 * The operation (per sequence b and head h, steps t = 0 .. T-1) is the SRWM of
 * "Metalearning Continual Learning Algorithms", section 2.3:
 *   Eq. (1)  [y_t, k_t, q_t, beta_t] = W_{t-1} x~_t
 *   Eq. (2)  v_t = W_{t-1} phi(q_t),   vbar_t = W_{t-1} phi(k_t)
 *   Eq. (3)  W_t = W_{t-1} + sigma(beta_t) (v_t - vbar_t) (outer) phi(k_t)
 * with phi = softmax, sigma = sigmoid, and x~_t = x_t (supervised variant) or
 * softmax(x_t) over the head's d inputs (RL variant).  In the four-learning-rate
 * version (same page, Eqs. (4)-(5)) W has row blocks [W^y; W^k; W^q; W^b] and
 * beta_t = [b^y, b^k, b^q, b^b]; rows of block X use sigma(b^X), the four beta
 * rows use sigma(b^b).  y_t comes from the pre-update matrix W_{t-1} (review of
 * "A Modern Self-Referential Weight Matrix That Learns to Modify Itself",
 * section 2.2).  Heads are independent, each on its own d coordinates of the
 * D = H*d wide input (same review, section 2.4); W_0 is shared by all sequences.
 *
 * Shapes: per head d_in = d_out = d, W has m = 3*d + n_lr rows and d columns,
 * stored row-major (row = output index), blocks in the order y, k, q, beta.
 *
 * Common rules for every entry point below:
 *   - Pointers are DEVICE memory (cudaMalloc'd or managed) of fp32, contiguous,
 *     16-byte aligned.  The caller owns all buffers.  srwm_forward,
 *     srwm_forward_balanced, srwm_forward_balanced_noalloc, srwm_forward_from,
 *     srwm_step and srwm_backward make no device allocation.
 *   - State the library keeps, per device, for the life of the process:
 *       * the device status word (srwm_last_device_status), a file-scope
 *         __device__ variable, present once the library is loaded; its device
 *         address is looked up on the first call on each device;
 *       * srwm_forward_balanced_noalloc's counter array (256 KiB), a
 *         file-scope __device__ array, present once the library is loaded;
 *         its address is looked up on that entry point's first call on each
 *         device;
 *       * srwm_forward_host's two copy streams and twelve events, created on
 *         its first call on each device;
 *       * srwm_layer_forward's cuBLASLt handle, created by cublasLtCreate
 *         (which allocates) on the first call on a device that takes the
 *         cuBLASLt comparison path (srwm_debug_set_layer_gemm 1 or 2); the
 *         default path does not use cuBLASLt.
 *     The cached addresses and handles belong to the device's primary context:
 *     after cudaDeviceReset on a device, do not call the library on that
 *     device again in the same process.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without waiting.  Argument errors are
 *     returned before anything is enqueued; nothing is written then.
 *   - Supported: d in {16, 32, 64}, n_lr in {1, 4}, softmax_input in {0, 1}.
 *   - Outputs must not overlap inputs or each other (srwm_step alone allows
 *     W_out == W_in exactly, for an in-place update).
 *   - Results are deterministic: the same inputs give the same bits.
 */
#ifndef SRWM_H
#define SRWM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum srwm_status {
    SRWM_OK = 0,
    SRWM_ERR_NULL = 1,        /* a required pointer is NULL                               */
    SRWM_ERR_SHAPE = 2,       /* B, H or d <= 0, T < 0, or a size overflows the layout    */
    SRWM_ERR_UNSUPPORTED = 3, /* d not in {16,32,64}, n_lr not in {1,4}, bad flag value   */
    SRWM_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned                         */
    SRWM_ERR_ALIAS = 5,       /* an output overlaps an input or another output            */
    SRWM_ERR_CUDA = 6,        /* a CUDA runtime call failed (launch, attribute, ...)      */
    SRWM_ERR_TIMEOUT = 7,     /* a kernel gave up a bounded wait (see srwm_last_device_status) */
    SRWM_ERR_NOT_DEVICE = 8   /* a pointer is not device-accessible CUDA memory           */
};

/*
 * srwm_forward -- run T steps of Eqs. (1)-(3) (n_lr = 1) or Eqs. (4)-(5)
 * (n_lr = 4) for every (sequence, head) stream, starting from the shared W0.
 *
 *   x        [B, T, H, d]  inputs; step t of stream (b, h) is x[b, t, h, :]
 *   W0       [H, m, d]     initial matrix of each head, shared over b (read only)
 *   B, T, H  batch, steps, heads; T == 0 is valid and copies W0 into W_final
 *   d        per-head width (16, 32 or 64)
 *   n_lr     1 (one learning rate, m = 3d+1) or 4 (four learning rates, m = 3d+4)
 *   softmax_input  0: x~_t = x_t;  1: x~_t = softmax(x_t) over the head's d inputs
 *   y_out    [B, T, H, d]  written: y_t of every stream
 *   W_final  [B, H, m, d]  written: W_T of every stream
 *   stream   cudaStream_t or NULL
 * Returns SRWM_OK or an error code; x and y_out may be NULL only when T == 0.
 */
int srwm_forward(const float* x, const float* W0, int B, int T, int H, int d, int n_lr,
                 int softmax_input, float* y_out, float* W_final, void* stream);

/*
 * srwm_forward_balanced -- srwm_forward (same arguments, same results within
 * fp32 rounding) on a load-balanced schedule, for workloads with more
 * (sequence, head) streams than the GPU holds at once.  A persistent
 * cooperative grid splits streams into segments and hands each stream's state
 * from one segment to the next through W_final, replacing a mostly empty last
 * wave of whole streams.  The d = 32 kernel takes a wrap-around schedule: all
 * streams' steps are laid end to end and every warp slot takes an equal range
 * of them, so a stream is split at most once, its first part running at the
 * start of one slot and its last part at the end of the next.  The other
 * kernels cut every stream into segments of a multiple of 32 steps and
 * process (stream, segment) items in segment-major order.  The recurrence
 * itself is unchanged: the pages' Eqs. (1)-(5) are sequential in t within a
 * stream, and the segments of one stream run strictly in order.
 *
 *   workspace        device memory the call uses for per-stream progress
 *                    counters (zeroed by the call on `stream`); at least
 *                    srwm_forward_workspace_bytes(B, H) bytes, 16-byte aligned,
 *                    owned by the caller, not overlapping any other argument.
 *   workspace_bytes  its size.
 * Calls that share a workspace must not overlap in time on the GPU.
 * Other arguments, rules and return values as srwm_forward; additionally
 * SRWM_ERR_SHAPE if the workspace is too small.
 */
size_t srwm_forward_workspace_bytes(int B, int H);
int srwm_forward_balanced(const float* x, const float* W0, int B, int T, int H, int d, int n_lr,
                          int softmax_input, float* y_out, float* W_final, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * srwm_forward_balanced_noalloc -- srwm_forward_balanced without the
 * workspace argument, for callers that cannot allocate device memory (a host
 * framework that owns every allocation and gives plugins no allocator, or a
 * path that must not call cudaMalloc and accept its implicit synchronisation).
 * The pages have no counterpart to this entry point: it only changes where the
 * schedule's scratch lives.
 *
 * The per-stream progress counters live in a fixed array inside the library
 * (256 KiB on every GPU that loads it, held until the process exits), so at
 * most 65536 streams: B * H above that returns SRWM_ERR_SHAPE before anything
 * is enqueued.  The first call on a device looks up the array's device
 * address; make that first call before any stream capture on that device.
 * All calls share the one array: each call clears the counters it needs
 * before its kernel runs, and calls that overlap in time on the GPU (on
 * different streams, or from different host threads) race on it.
 * Arguments and results otherwise as srwm_forward_balanced.  Nothing is
 * allocated: no cudaMalloc, cudaFree or allocating library call.
 */
int srwm_forward_balanced_noalloc(const float* x, const float* W0, int B, int T, int H, int d,
                                  int n_lr, int softmax_input, float* y_out, float* W_final,
                                  void* stream);

/*
 * srwm_forward_from -- srwm_forward from a per-sequence state instead of the
 * shared W0: the state carried across truncation windows, e.g. RL rollouts
 * that keep W_t until the episode ends (review of "A Modern Self-Referential
 * Weight Matrix That Learns to Modify Itself", section 4.5, on keeping the
 * self-modified state across 50-step windows).  Running T1 steps with
 * srwm_forward and the remaining T - T1 steps with srwm_forward_from on the
 * returned W_final reproduces one srwm_forward over all T steps.
 *
 *   x        [B, T, H, d]   this window's inputs
 *   W_init   [B, H, m, d]   state of every stream at the start of the window (read)
 *   y_out    [B, T, H, d]   written
 *   W_final  [B, H, m, d]   written; may be the same pointer as W_init (in
 *                           place) but must not partially overlap it
 * Other arguments, rules and return values as srwm_forward.
 */
int srwm_forward_from(const float* x, const float* W_init, int B, int T, int H, int d, int n_lr,
                      int softmax_input, float* y_out, float* W_final, void* stream);

/*
 * srwm_forward_host -- srwm_forward with HOST buffers: x, W0 in host memory,
 * y and W_final written to host memory.  The copies overlap the recurrence:
 * the sequence is cut into chunks of chunk_steps steps, or, for chunk_steps
 * <= 0, into chunks that double from 32 steps and halve again at the end,
 * with the middle split evenly into chunks of at most max(256, T / 8) steps
 * at d = 64 and 64 steps at d <= 32, where the copies rather than the
 * recurrence set the pace (a ramp chunk is added on both ends while at least
 * as many steps remain between them, up to half that size), so that the first
 * H2D and the last D2H copy, which nothing overlaps, stay short.  T < 96 is a
 * single chunk.  The H2D copy of chunk k+1 and the D2H
 * copy of chunk k-1 run on the library's own copy streams while chunk k runs
 * on `stream`, the state passing between chunks as in srwm_forward_from.  Results equal srwm_forward's within fp32 rounding (a
 * chunk restarts its first read-out from the stored state).
 *
 *   x_host        [B, T, H, d]  host memory, page-locked (cudaHostAlloc /
 *                 cudaHostRegister) for the copies to overlap; pageable works
 *                 but copies synchronously
 *   W0_host       [H, m, d]     host memory
 *   y_host        [B, T, H, d]  host memory, written
 *   W_final_host  [B, H, m, d]  host memory, written
 *   chunk_steps   steps per chunk; <= 0: the doubling plan above
 *   workspace     DEVICE scratch of srwm_forward_host_workspace_bytes(...)
 *                 bytes, 16-byte aligned
 *
 * Everything is enqueued on `stream`: once it has completed (e.g. after
 * cudaStreamSynchronize), the host outputs are written.  Host buffers and the
 * workspace must stay valid and untouched until then.  The copy streams and
 * events are created on a device's first call and kept until the process
 * exits; calls on one device are enqueued one at a time.  Returns
 * SRWM_ERR_UNSUPPORTED when a "host" pointer is device or managed memory.
 */
size_t srwm_forward_host_workspace_bytes(int B, int T, int H, int d, int n_lr, int chunk_steps);
int srwm_forward_host(const float* x_host, const float* W0_host, int B, int T, int H, int d, int n_lr,
                      int softmax_input, float* y_host, float* W_final_host, int chunk_steps,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * srwm_step -- one step of the same recurrence from a per-sequence state:
 * W_out[b,h] = W_in[b,h] + update, y_t[b,h] = y from W_in[b,h].  Calling it T
 * times, feeding W_out back as W_in, reproduces srwm_forward.
 *
 *   x_t    [B, H, d]      this step's inputs
 *   W_in   [B, H, m, d]   current state of every stream (read)
 *   y_t    [B, H, d]      written
 *   W_out  [B, H, m, d]   written; may be the same pointer as W_in (in place)
 *                         but must not partially overlap it
 */
int srwm_step(const float* x_t, const float* W_in, int B, int H, int d, int n_lr,
              int softmax_input, float* y_t, float* W_out, void* stream);

/*
 * srwm_backward -- gradients of a loss through srwm_forward: given the
 * cotangents dy = dL/dy and (optionally) dW_final = dL/dW_final of one
 * srwm_forward(x, W0, ...) call, writes dx = dL/dx and dW0 = dL/dW0.  The
 * training of these models backpropagates through the whole sequence
 * ("Metalearning Continual Learning Algorithms", section 2.3, which trains
 * the SRWM by gradient descent through its own updates).  The derivative is
 * taken of the exact recurrence above, including the softmaxes, the sigmoid
 * gates and x~ = softmax(x) when softmax_input = 1.
 *
 *   x         [B, T, H, d]    the forward's inputs
 *   W0        [H, m, d]       the forward's shared initial state
 *   dy        [B, T, H, d]    dL/dy
 *   dW_final  [B, H, m, d]    dL/dW_final, or NULL for zero
 *   dx        [B, T, H, d]    written
 *   dW0       [H, m, d]       written: the sum over sequences b of each
 *                             stream's dL/dW0, summed in order of b
 *   workspace device scratch of at least srwm_backward_workspace_bytes(...)
 *             bytes, 16-byte aligned, contents irrelevant on entry.  It holds
 *             the forward's per-step records (phi(k), u, gates, a: about
 *             4 * (5d + 4 + n_lr) bytes per step and stream), W_T, the
 *             forward's y and the per-stream dL/dW0.  It must stay untouched
 *             until the work on `stream` has finished.
 *
 * The call runs the forward pass itself (with the records), then the steps
 * backwards from W_T.  Each step recovers W_{t-1} by subtracting the recorded
 * rank-one update.  y and W_final need not be passed in.  T = 0 writes
 * dW0 = sum_b dW_final (or zero).  The same pointer rules as above apply; the
 * workspace must not overlap anything else.  Returns SRWM_ERR_SHAPE when
 * workspace_bytes is too small.
 */
int srwm_backward(const float* x, const float* W0, int B, int T, int H, int d, int n_lr,
                  int softmax_input, const float* dy, const float* dW_final, float* dx, float* dW0,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * srwm_backward_workspace_bytes -- scratch size srwm_backward needs for these
 * sizes, the sum of 256-byte aligned regions: 2 x 4 B*H*m*d (dL/dW0 per
 * stream, W_T), 4 B*T*H*d (y), 4 B*H*T*ceil4(5d + 4 + n_lr) (records),
 * 4 B*H (counters).  Returns 0 for unsupported or invalid sizes.
 */
size_t srwm_backward_workspace_bytes(int B, int T, int H, int d, int n_lr);

/*
 * srwm_layer_forward -- one Recursive Self-Transformer layer, forward: the
 * multi-head SRWM in place of multi-head self-attention, with the
 * Transformer's layer norms, feed-forward block and residual connections
 * around it ("Metalearning Continual Learning Algorithms", section 2.3; the
 * review "SRWM:让权重矩阵学习修改自身", section 2.4).  Pre-LN block over the
 * N = B*T tokens of width D = H*d:
 *   a = LN1(u);  y = SRWM(a) (as srwm_forward, heads = d-wide slices);
 *   h = u + y;   out = h + W2 ReLU(W1 LN2(h) + b1) + b2
 * LN(v) = (v - mean(v)) / sqrt(var(v) + 1e-5) * gamma + beta over the D
 * entries of a token (biased variance).  Inputs, outputs and every stored
 * value are fp32.  The two feed-forward products run on the tensor cores in
 * this library's tcgen05 kernel with fp32 operands split into bf16 (hi, lo)
 * pairs: X W^T ~ X_hi W_hi^T + X_hi W_lo^T + X_lo W_hi^T accumulated in fp32
 * (about 1e-5 relative error on the products); everything else runs in fp32.
 * d_ff must be a multiple of 8.
 *
 *   u          [B, T, D]      input tokens
 *   ln*_gamma, ln*_beta [D]   layer-norm scale and shift
 *   W0         [H, m, d]      SRWM initial state (as srwm_forward)
 *   W1 [d_ff, D], b1 [d_ff], W2 [D, d_ff], b2 [D]   feed-forward (row-major,
 *              output index first, as a PyTorch Linear weight)
 *   out        [B, T, D]      written
 *   W_final    [B, H, m, d]   the SRWM's final state, written; or NULL
 *   workspace  device scratch of srwm_layer_workspace_bytes(...) bytes,
 *              16-byte aligned, untouched until the work on `stream` ends
 *
 * Supported: D = H*d <= 1024, d_ff a positive multiple of 8, and the
 * srwm_forward limits.  The same pointer rules apply: outputs and workspace
 * overlap nothing else.
 */
int srwm_layer_forward(const float* u, int B, int T, int H, int d, int n_lr, int softmax_input,
                       const float* ln1_gamma, const float* ln1_beta, const float* W0,
                       const float* ln2_gamma, const float* ln2_beta, const float* W1,
                       const float* b1, int d_ff, const float* W2, const float* b2, float* out,
                       float* W_final, void* workspace, size_t workspace_bytes, void* stream);

/* Scratch bytes srwm_layer_forward needs for these sizes; 0 when unsupported. */
size_t srwm_layer_workspace_bytes(int B, int T, int H, int d, int n_lr, int d_ff);

/*
 * srwm_debug_set_layer_gemm -- how srwm_layer_forward's feed-forward products
 * compute: 0 (default) this library's tensor-core kernel; 1 cuBLASLt plain
 * FP32; 2 cuBLASLt FP32 emulated on the BF16 tensor cores where it offers
 * that (else plain FP32).  Modes 1 and 2 exist for comparison; applies to
 * calls made afterwards.  SRWM_ERR_UNSUPPORTED for any other mode.
 */
int srwm_debug_set_layer_gemm(int mode);

/* Human-readable name of a status code (static string, never NULL). */
const char* srwm_status_string(int status);

/*
 * srwm_last_device_status -- synchronise `stream`, then read and clear the
 * device status word that kernels set when a bounded wait gives up (a TMA
 * transfer that never arrived).  Returns SRWM_OK, SRWM_ERR_TIMEOUT, or
 * SRWM_ERR_CUDA if the synchronisation itself failed.
 */
int srwm_last_device_status(void* stream);

/*
 * srwm_set_wait_limit_ns -- the time after which a kernel's wait on an
 * asynchronous copy gives up (default 1 s).  Values < 1000 are clamped to
 * 1000.  Applies to launches made after the call, from any thread.
 */
int srwm_set_wait_limit_ns(long long limit_ns);

/*
 * srwm_debug_skip_x_chunk -- fault injection for tests: the next launches do
 * not issue the TMA load of input chunk `chunk` (a chunk is a fixed number of
 * consecutive steps) so the kernel's bounded wait on it runs out; -1 turns
 * injection off.  The kernel then stops early, waits for its other copies,
 * writes no further outputs, and sets the status word read by
 * srwm_last_device_status.  Not for production use.
 */
int srwm_debug_skip_x_chunk(int chunk);

/*
 * srwm_debug_wrap_len, srwm_debug_wrap_pieces -- tests only: the wrap-around
 * schedule of srwm_forward_balanced (d = 32) without a GPU.
 * srwm_debug_wrap_len returns the steps per warp slot the library chooses for
 * n_streams streams of T steps on `slots` slots with TMA chunks of tau steps
 * (0 when the schedule does not apply: n_streams <= slots, or a size <= 0).
 * srwm_debug_wrap_pieces lists, in the order the slot runs them, the pieces
 * of slot `slot` under range length wrap_len: four ints per piece (stream,
 * segment number 0 or 1, first step, number of steps) into out (room for
 * max_pieces pieces, caller-owned).  It returns the number of pieces (which
 * may exceed max_pieces; only the first max_pieces are written), or -1 for
 * invalid arguments (n_streams or T <= 0, wrap_len < T, slot < 0).
 */
long long srwm_debug_wrap_len(long long n_streams, int T, long long slots, int tau);
int srwm_debug_wrap_pieces(long long n_streams, int T, long long wrap_len, long long slot, int* out,
                           int max_pieces);

/*
 * srwm_debug_chunk_plan -- tests only: the chunk lengths srwm_forward_host
 * uses for T steps of width d and the given chunk_steps, in order, into out (room for
 * max_chunks, caller-owned).  Returns the number of chunks (which may exceed
 * max_chunks; only the first max_chunks are written), or -1 for T < 0,
 * max_chunks < 0, or out NULL with max_chunks > 0.
 */
int srwm_debug_chunk_plan(int T, int d, int chunk_steps, int* out, int max_chunks);

/*
 * srwm_debug_set_segment_len -- tests only: force the segment length (a
 * positive multiple of 32 steps) that srwm_forward_balanced uses, on the
 * segment schedule for every kernel; 0 restores the automatic choice.
 * Returns SRWM_ERR_SHAPE for other values.
 */
int srwm_debug_set_segment_len(int steps);

/*
 * srwm_probe_fma -- calibration kernel for the FP32 FMA roofline: `blocks` CTAs
 * of `threads` threads each run `iters` iterations of 8 independent FMA chains
 * (packed two-wide when `packed` is 1).  out[blocks*threads] receives the
 * chains' sums (device memory).  One launch does blocks*threads*iters*8*(1+packed)
 * FMAs; time it with CUDA events on `stream`.
 */
int srwm_probe_fma(int blocks, int threads, int iters, int packed, float* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SRWM_H */
