// srwm_api.cu -- the C ABI declared in include/srwm.h: argument checks, TMA
// tensor maps, dispatch to the kernel instantiations, device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "srwm.h"
#include "srwm_common.h"
#include "srwm_bwd.cuh"

namespace {

// Set by a kernel whose bounded wait ran out; read by srwm_last_device_status.
__device__ unsigned int g_status_word;

std::atomic<long long> g_wait_limit_ns{1000000000LL};
std::atomic<int> g_skip_chunk{-1};
std::atomic<int> g_force_seg_len{0};

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices];
std::mutex g_status_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_encode;
}

int status_ptr(unsigned** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
            cudaGetLastError();
            return SRWM_ERR_CUDA;
        }
        g_status_ptr[dev] = static_cast<unsigned*>(p);
    }
    *out = g_status_ptr[dev];
    return SRWM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

// Device memory of the current device (or managed memory)?
int check_device_ptr(const void* p)
{
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_NOT_DEVICE;
    }
    if (attr.type == cudaMemoryTypeManaged) return SRWM_OK;
    if (attr.type != cudaMemoryTypeDevice) return SRWM_ERR_NOT_DEVICE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    return attr.device == dev ? SRWM_OK : SRWM_ERR_NOT_DEVICE;
}

// 4-D map over a [B, T, H, d] fp32 tensor, dims innermost first {d, H, T, B};
// one box is `tau` consecutive steps of one (b, h) stream: {d, 1, tau, 1}.
int make_stream_map(CUtensorMap* map, const float* base, int B, int T, int H, int d, int tau)
{
    auto enc = encoder();
    if (!enc) return SRWM_ERR_CUDA;
    const cuuint64_t e = sizeof(float);
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {e * d, e * d * H, e * d * H * static_cast<cuuint64_t>(T)};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(d), 1u, static_cast<cuuint32_t>(tau), 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SRWM_OK : SRWM_ERR_CUDA;
}

// The kernel for a call; at d = 64 it depends on the streams per SM.
int info_for(int d, int n_lr, int smx, long long n_streams, srwm::LaunchInfo* li, bool emit = false)
{
    if (d == 16) {
        *li = srwm::launch_info_d16(n_lr, smx, emit);
        return SRWM_OK;
    }
    if (d == 32) {
        *li = srwm::launch_info_d32(n_lr, smx, emit);
        return SRWM_OK;
    }
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    *li = srwm::launch_info_d64(n_lr, smx, n_streams, n_sm, emit);
    return SRWM_OK;
}

int check_params(int B, int T, int H, int d, int n_lr, int softmax_input)
{
    if (B <= 0 || H <= 0 || d <= 0 || T < 0) return SRWM_ERR_SHAPE;
    if (d != 16 && d != 32 && d != 64) return SRWM_ERR_UNSUPPORTED;
    if (n_lr != 1 && n_lr != 4) return SRWM_ERR_UNSUPPORTED;
    if (softmax_input != 0 && softmax_input != 1) return SRWM_ERR_UNSUPPORTED;
    // Every element count must fit the int64 byte arithmetic below and every
    // TMA stride must stay below 2^40 bytes.
    const long long m = 3LL * d + n_lr;
    const long long pairs = static_cast<long long>(B) * H;
    if (pairs > (1LL << 31) - 1) return SRWM_ERR_SHAPE;
    const long long step_bytes = static_cast<long long>(H) * d * 4;
    if (step_bytes * static_cast<long long>(T > 0 ? T : 1) >= (1LL << 40)) return SRWM_ERR_SHAPE;
    if (pairs * m * d > (1LL << 60) / 4) return SRWM_ERR_SHAPE;
    return SRWM_OK;
}

int set_smem_attr(const srwm::LaunchInfo& li)
{
    if (li.smem_bytes > 48 * 1024 &&
        cudaFuncSetAttribute(li.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, li.smem_bytes) !=
            cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    return SRWM_OK;
}

// grid_ctas <= 0: one CTA per group of streams_per_cta streams (plain launch);
// else a cooperative launch of exactly grid_ctas CTAs.
int launch(const srwm::LaunchInfo& li, const CUtensorMap& tx, const CUtensorMap& ty,
           const srwm::KParams& kp, long long pairs, int grid_ctas, cudaStream_t stream)
{
    int rc = set_smem_attr(li);
    if (rc != SRWM_OK) return rc;
    const bool coop = grid_ctas > 0;
    const dim3 grid(static_cast<unsigned>(
        coop ? grid_ctas : srwm::cdiv(static_cast<int>(pairs), li.streams_per_cta)));
    const dim3 block(static_cast<unsigned>(li.threads));
    void* args[] = {const_cast<CUtensorMap*>(&tx), const_cast<CUtensorMap*>(&ty),
                    const_cast<srwm::KParams*>(&kp)};
    const cudaError_t e =
        coop ? cudaLaunchCooperativeKernel(li.kernel, grid, block, args, static_cast<size_t>(li.smem_bytes), stream)
             : cudaLaunchKernel(li.kernel, grid, block, args, static_cast<size_t>(li.smem_bytes), stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    return SRWM_OK;
}

// Co-resident CTAs of this kernel on the current device (0 on failure).
int resident_ctas(const srwm::LaunchInfo& li)
{
    int dev = 0, n_sm = 0, per_sm = 0;
    if (set_smem_attr(li) != SRWM_OK || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, li.kernel, li.threads,
                                                      static_cast<size_t>(li.smem_bytes)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n_sm * per_sm;
}

// Segment length for the balanced schedule: a multiple of 32 steps (every
// kernel's TMA chunk divides it) minimising rounds * (steps + reload cost),
// where a round is one item on every slot.
int choose_seg_len(long long n_streams, int T, long long slots)
{
    constexpr int kReloadSteps = 8;   // state reload, TMA refill, first read-out
    int best_len = T;
    double best = static_cast<double>((n_streams + slots - 1) / slots) * (T + kReloadSteps);
    for (int len = 32; len < T; len += 32) {
        const long long segs = (T + len - 1) / len;
        const long long rounds = (n_streams * segs + slots - 1) / slots;
        const double cost = static_cast<double>(rounds) * (len + kReloadSteps);
        if (cost < best) {
            best = cost;
            best_len = len;
        }
    }
    return best_len;
}

// Range length of the wrap-around schedule: ceil(total / slots) steps rounded
// up to whole TMA chunks.  With more streams than slots it is at least T.
long long wrap_len_for(long long n_streams, int T, long long slots, int tau)
{
    const long long total = n_streams * T;
    const long long per = (total + slots - 1) / slots;
    return (per + tau - 1) / tau * tau;
}

// Shared body of srwm_forward (per_seq = 0) and srwm_step (per_seq = 1, T = 1).
int run(const float* x, const float* W_init, int per_seq, int B, int T, int H, int d, int n_lr,
        int smx, float* y, float* W_out, cudaStream_t stream, int* seg_done = nullptr,
        size_t seg_done_bytes = 0, float* emit = nullptr, int emit_stride = 0)
{
    const long long m = 3LL * d + n_lr;
    const size_t nx = static_cast<size_t>(B) * T * H * d * sizeof(float);
    const size_t nw_in = static_cast<size_t>(per_seq ? B : 1) * H * m * d * sizeof(float);
    const size_t nw_out = static_cast<size_t>(B) * H * m * d * sizeof(float);

    if (!aligned16(W_init) || !aligned16(W_out) || (T > 0 && (!aligned16(x) || !aligned16(y))))
        return SRWM_ERR_ALIGN;
    if (T > 0) {
        if (overlaps(y, nx, x, nx) || overlaps(y, nx, W_init, nw_in) || overlaps(y, nx, W_out, nw_out))
            return SRWM_ERR_ALIAS;
        if (overlaps(W_out, nw_out, x, nx)) return SRWM_ERR_ALIAS;
    }
    if (overlaps(W_out, nw_out, W_init, nw_in) && !(per_seq && W_out == W_init)) return SRWM_ERR_ALIAS;

    int rc;
    if ((rc = check_device_ptr(W_init)) != SRWM_OK) return rc;
    if ((rc = check_device_ptr(W_out)) != SRWM_OK) return rc;
    if (T > 0) {
        if ((rc = check_device_ptr(x)) != SRWM_OK) return rc;
        if ((rc = check_device_ptr(y)) != SRWM_OK) return rc;
    }

    srwm::LaunchInfo li;
    if ((rc = info_for(d, n_lr, smx, static_cast<long long>(B) * H, &li, emit != nullptr)) != SRWM_OK) return rc;
    CUtensorMap tx, ty;
    std::memset(&tx, 0, sizeof(tx));
    std::memset(&ty, 0, sizeof(ty));
    if (T > 0) {
        if ((rc = make_stream_map(&tx, x, B, T, H, d, li.tau)) != SRWM_OK) return rc;
        if ((rc = make_stream_map(&ty, y, B, T, H, d, li.tau)) != SRWM_OK) return rc;
    }
    srwm::KParams kp;
    kp.W_init = W_init;
    kp.W_out = W_out;
    if ((rc = status_ptr(&kp.status)) != SRWM_OK) return rc;
    kp.wait_limit_ns = static_cast<unsigned long long>(g_wait_limit_ns.load());
    kp.B = B;
    kp.T = T;
    kp.H = H;
    kp.w_per_seq = per_seq;
    kp.skip_chunk = g_skip_chunk.load();
    const long long pairs = static_cast<long long>(B) * H;
    kp.n_streams = static_cast<int>(pairs);
    kp.seg_len = T > 0 ? T : 1;
    kp.n_items = kp.n_streams;
    kp.seg_done = nullptr;
    kp.wrap_len = 0;
    kp.emit = emit;
    kp.emit_stride = emit_stride;
    if (!seg_done) return launch(li, tx, ty, kp, pairs, 0, stream);

    // Balanced schedule: streams cut into segments, a persistent cooperative
    // grid takes (stream, segment) items in segment-major order.
    const int ctas = resident_ctas(li);
    if (ctas <= 0) return SRWM_ERR_CUDA;
    const long long slots = static_cast<long long>(ctas) * li.streams_per_cta;
    int len = g_force_seg_len.load();
    if (len <= 0) {
        // Nothing to balance when every stream has a slot of its own: the plain
        // launch (one stream per slot, spread over the SMs) is the fast one.
        if (pairs <= slots) return launch(li, tx, ty, kp, pairs, 0, stream);
        if (li.wraps && T > 0) {
            // wrap-around: every slot gets ceil(total / slots) steps, rounded up
            // to whole TMA chunks (>= T, as there are more streams than slots)
            const long long wrap = wrap_len_for(pairs, T, slots, li.tau);
            const long long used = (pairs * T + wrap - 1) / wrap;
            if (cudaMemsetAsync(seg_done, 0, seg_done_bytes, stream) != cudaSuccess) {
                cudaGetLastError();
                return SRWM_ERR_CUDA;
            }
            kp.seg_done = seg_done;
            kp.wrap_len = wrap;
            kp.n_items = 0;
            const long long need = (used + li.streams_per_cta - 1) / li.streams_per_cta;
            return launch(li, tx, ty, kp, pairs, static_cast<int>(need < ctas ? need : ctas), stream);
        }
        len = choose_seg_len(pairs, T, slots);
    }
    if (T <= 0 || len >= T) len = T > 0 ? T : 1;
    const long long segs = T > 0 ? (T + len - 1) / len : 1;
    if (pairs * segs > (1LL << 31) - 1) return SRWM_ERR_SHAPE;
    kp.seg_len = len;
    kp.n_items = static_cast<int>(pairs * segs);
    if (cudaMemsetAsync(seg_done, 0, seg_done_bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    kp.seg_done = seg_done;
    const long long need = (kp.n_items + li.streams_per_cta - 1) / li.streams_per_cta;
    return launch(li, tx, ty, kp, pairs, static_cast<int>(need < ctas ? need : ctas), stream);
}


// ---------------------------------------------------------------- host pipeline
// Copy streams and events of srwm_forward_host, created once per device and
// reused; a mutex serialises the enqueueing of concurrent calls on a device.
constexpr int kPipeSlots = 3;
struct Pipe {
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t start, w0, end, in[kPipeSlots], comp[kPipeSlots], out[kPipeSlots];
    std::mutex mu;
};
constexpr int kPipeDevices = 64;
Pipe g_pipe[kPipeDevices];
std::mutex g_pipe_init_mu;

int pipe_for_device(Pipe** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kPipeDevices) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_pipe_init_mu);
    Pipe& p = g_pipe[dev];
    if (!p.ready) {
        bool ok = cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking) == cudaSuccess;
        cudaEvent_t* evs[] = {&p.start, &p.w0, &p.end};
        for (cudaEvent_t* e : evs) ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; i < kPipeSlots; ++i) {
            ok = ok && cudaEventCreateWithFlags(&p.in[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.comp[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.out[i], cudaEventDisableTiming) == cudaSuccess;
        }
        if (!ok) {
            cudaGetLastError();
            return SRWM_ERR_CUDA;
        }
        p.ready = true;
    }
    *out = &p;
    return SRWM_OK;
}

// Host memory (pinned or pageable), not device or managed memory.
int check_host_ptr(const void* ptr)
{
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_UNSUPPORTED;
    }
    return (attr.type == cudaMemoryTypeHost || attr.type == cudaMemoryTypeUnregistered) ? SRWM_OK
                                                                                        : SRWM_ERR_UNSUPPORTED;
}

struct HostWs {
    size_t w0, state, cnt, x[kPipeSlots], y[kPipeSlots], total;
};

bool host_ws(long long B, long long T, long long H, long long d, long long n_lr, long long C, HostWs* w)
{
    const long long m = 3 * d + n_lr;
    auto a256 = [](size_t n) { return (n + 255) / 256 * 256; };
    const size_t chunk = a256(static_cast<size_t>(B * C * H * d) * 4);
    size_t off = 0;
    w->w0 = off;
    off += a256(static_cast<size_t>(H * m * d) * 4);
    w->state = off;
    off += a256(static_cast<size_t>(B * H * m * d) * 4);
    w->cnt = off;
    off += a256(static_cast<size_t>(B * H) * 4);
    for (int i = 0; i < kPipeSlots; ++i) {
        w->x[i] = off;
        off += chunk;
        w->y[i] = off;
        off += chunk;
    }
    w->total = off;
    (void)T;
    return true;
}

// Chunk plan of srwm_forward_host.  chunk_steps > 0: chunks of that many steps
// (the last one ragged).  0: chunks that double from 32 steps and halve again
// at the end, the middle split evenly, so that the first input copy and the
// last output copy (which nothing overlaps) stay short.  The longest chunk
// depends on which side sets the pace.  A step copies 8 d bytes per stream
// each way and does 3 m d FMAs, i.e. 3 m / 8 FMAs per copied byte: ~37 at
// d = 32, ~20 at d = 16, 73.5 at d = 64.  At d <= 32 the host link (~0.3 TB/s
// both ways) is slower than the recurrence, and short chunks (at most 64
// steps) keep the copies flowing from the start (rl: 1.24 ms per call against
// 1.35 ms with 160-step chunks); at d = 64 the recurrence is the slower side,
// and chunks of up to 256 steps, or T / 8 for longer sequences, save launches
// and state reloads.
std::vector<int> chunk_plan(int T, int d, int chunk_steps)
{
    std::vector<int> plan;
    if (T <= 0) return plan;
    if (chunk_steps > 0) {
        for (int t = 0; t < T; t += chunk_steps) plan.push_back(T - t < chunk_steps ? T - t : chunk_steps);
        return plan;
    }
    constexpr int kMin = 32;
    const int kMax = d <= 32 ? 64 : (T / 8 > 256 ? T / 8 : 256);
    std::vector<int> tail;
    int rem = T;
    // A ramp chunk goes on both ends while at least as much is left between
    // them, and only up to half the largest chunk: the middle, split evenly into
    // chunks of at most kMax, then never falls below the last ramp chunk, so the
    // chunk sizes rise and then fall.
    for (int c = kMin; 2 * c <= kMax && rem >= 3 * c; c *= 2) {
        plan.push_back(c);
        tail.push_back(c);
        rem -= 2 * c;
    }
    if (rem > 0) {
        const int n = (rem + kMax - 1) / kMax;
        for (int i = 0; i < n; ++i) plan.push_back(rem / n + (i < rem % n ? 1 : 0));
    }
    plan.insert(plan.end(), tail.rbegin(), tail.rend());
    return plan;
}

int effective_chunk(int T, int d, int chunk_steps)
{
    int c = 1;
    for (int v : chunk_plan(T, d, chunk_steps)) c = v > c ? v : c;
    return c;
}

}  // namespace

namespace srwm {

// For the layer's tensor-core products (srwm_ffgemm.cu): the device status
// word and the bounded-wait limit the kernels of this library share.
int device_status_ptr(unsigned** out) { return status_ptr(out); }
unsigned long long device_wait_limit_ns() { return static_cast<unsigned long long>(g_wait_limit_ns.load()); }

}  // namespace srwm

extern "C" {

int srwm_forward(const float* x, const float* W0, int B, int T, int H, int d, int n_lr,
                 int softmax_input, float* y_out, float* W_final, void* stream)
{
    if (!W0 || !W_final || (T > 0 && (!x || !y_out))) return SRWM_ERR_NULL;
    const int rc = check_params(B, T, H, d, n_lr, softmax_input);
    if (rc != SRWM_OK) return rc;
    return run(x, W0, 0, B, T, H, d, n_lr, softmax_input, y_out, W_final,
               static_cast<cudaStream_t>(stream));
}

size_t srwm_forward_workspace_bytes(int B, int H)
{
    if (B <= 0 || H <= 0) return 0;
    const size_t n = static_cast<size_t>(B) * static_cast<size_t>(H) * sizeof(int);
    return (n + 255) / 256 * 256;
}

int srwm_forward_balanced(const float* x, const float* W0, int B, int T, int H, int d, int n_lr,
                          int softmax_input, float* y_out, float* W_final, void* workspace,
                          size_t workspace_bytes, void* stream)
{
    if (!W0 || !W_final || !workspace || (T > 0 && (!x || !y_out))) return SRWM_ERR_NULL;
    const int rc = check_params(B, T, H, d, n_lr, softmax_input);
    if (rc != SRWM_OK) return rc;
    const size_t need = static_cast<size_t>(B) * H * sizeof(int);
    if (workspace_bytes < need) return SRWM_ERR_SHAPE;
    if (!aligned16(workspace)) return SRWM_ERR_ALIGN;
    const long long m = 3LL * d + n_lr;
    const size_t nx = static_cast<size_t>(B) * T * H * d * sizeof(float);
    const size_t nw0 = static_cast<size_t>(H) * m * d * sizeof(float);
    const size_t nwf = static_cast<size_t>(B) * H * m * d * sizeof(float);
    if (overlaps(workspace, need, x, nx) || overlaps(workspace, need, W0, nw0) ||
        overlaps(workspace, need, y_out, nx) || overlaps(workspace, need, W_final, nwf))
        return SRWM_ERR_ALIAS;
    const int prc = check_device_ptr(workspace);
    if (prc != SRWM_OK) return prc;
    return run(x, W0, 0, B, T, H, d, n_lr, softmax_input, y_out, W_final,
               static_cast<cudaStream_t>(stream), static_cast<int*>(workspace), need);
}

long long srwm_debug_wrap_len(long long n_streams, int T, long long slots, int tau)
{
    if (n_streams <= slots || T <= 0 || slots <= 0 || tau <= 0) return 0;
    return wrap_len_for(n_streams, T, slots, tau);
}

int srwm_debug_wrap_pieces(long long n_streams, int T, long long wrap_len, long long slot, int* out, int max_pieces)
{
    if (n_streams <= 0 || T <= 0 || wrap_len < T || slot < 0 || max_pieces < 0 || (max_pieces > 0 && !out))
        return -1;
    const long long lo = slot * wrap_len;
    long long hi = lo + wrap_len < n_streams * T ? lo + wrap_len : n_streams * T;
    srwm::Piece pc;
    int n = 0;
    while (srwm::wrap_next(lo, hi, T, pc)) {
        if (n < max_pieces) {
            out[4 * n + 0] = pc.p;
            out[4 * n + 1] = pc.seg;
            out[4 * n + 2] = pc.t0;
            out[4 * n + 3] = pc.len;
        }
        ++n;
    }
    return n;
}

int srwm_debug_chunk_plan(int T, int d, int chunk_steps, int* out, int max_chunks)
{
    if (T < 0 || max_chunks < 0 || (max_chunks > 0 && !out)) return -1;
    const std::vector<int> plan = chunk_plan(T, d, chunk_steps);
    for (int i = 0; i < static_cast<int>(plan.size()) && i < max_chunks; ++i) out[i] = plan[i];
    return static_cast<int>(plan.size());
}

int srwm_debug_set_segment_len(int steps)
{
    if (steps != 0 && (steps < 0 || steps % 32 != 0)) return SRWM_ERR_SHAPE;
    g_force_seg_len.store(steps);
    return SRWM_OK;
}

namespace {

// srwm_backward's workspace, each region 256-byte aligned: dL/dW0 per stream,
// W_T, the forward's y (not needed, but the forward kernels write it), the
// per-step records, the schedule counters.
struct BwdWs {
    size_t dws, wt, y, rec, cnt, total;
};

bool bwd_ws(long long B, long long T, long long H, long long d, long long n_lr, BwdWs* w)
{
    const long long m = 3 * d + n_lr, streams = B * H;
    auto a256 = [](size_t n) { return (n + 255) / 256 * 256; };
    const size_t md = static_cast<size_t>(m * d) * 4;
    size_t off = 0;
    w->dws = off;
    off += a256(static_cast<size_t>(streams) * md);
    w->wt = off;
    off += a256(static_cast<size_t>(streams) * md);
    w->y = off;
    off += a256(static_cast<size_t>(B * T * H * d) * 4);
    w->rec = off;
    off += a256(static_cast<size_t>(streams * T) * srwm::emit_record_floats(static_cast<int>(d), static_cast<int>(n_lr)) * 4);
    w->cnt = off;
    off += a256(static_cast<size_t>(streams) * 4);
    w->total = off;
    return true;
}

}  // namespace

size_t srwm_backward_workspace_bytes(int B, int T, int H, int d, int n_lr)
{
    if (B <= 0 || H <= 0 || T < 0 || (d != 16 && d != 32 && d != 64) || (n_lr != 1 && n_lr != 4)) return 0;
    if (check_params(B, T, H, d, n_lr, 0) != SRWM_OK) return 0;
    BwdWs w;
    bwd_ws(B, T, H, d, n_lr, &w);
    return w.total;
}

int srwm_backward(const float* x, const float* W0, int B, int T, int H, int d, int n_lr, int softmax_input,
                  const float* dy, const float* dW_final, float* dx, float* dW0, void* workspace,
                  size_t workspace_bytes, void* stream)
{
    if (!W0 || !dW0 || !workspace || (T > 0 && (!x || !dy || !dx))) return SRWM_ERR_NULL;
    int rc = check_params(B, T, H, d, n_lr, softmax_input);
    if (rc != SRWM_OK) return rc;
    if (static_cast<long long>(B) * H > 0x7fffffffLL) return SRWM_ERR_SHAPE;   // one CTA per stream
    const size_t need = srwm_backward_workspace_bytes(B, T, H, d, n_lr);
    if (workspace_bytes < need) return SRWM_ERR_SHAPE;
    const long long m = 3LL * d + n_lr;
    const size_t nx = static_cast<size_t>(B) * T * H * d * sizeof(float);
    const size_t nw0 = static_cast<size_t>(H) * m * d * sizeof(float);
    const size_t nwf = static_cast<size_t>(B) * H * m * d * sizeof(float);
    if (!aligned16(W0) || !aligned16(dW0) || !aligned16(workspace) || (dW_final && !aligned16(dW_final)) ||
        (T > 0 && (!aligned16(x) || !aligned16(dy) || !aligned16(dx))))
        return SRWM_ERR_ALIGN;
    const void* ins[4] = {x, W0, dy, dW_final};
    const size_t in_bytes[4] = {nx, nw0, nx, nwf};
    for (int i = 0; i < 4; ++i) {
        if (overlaps(dx, nx, ins[i], in_bytes[i]) || overlaps(dW0, nw0, ins[i], in_bytes[i]) ||
            overlaps(workspace, need, ins[i], in_bytes[i]))
            return SRWM_ERR_ALIAS;
    }
    if (overlaps(dx, nx, dW0, nw0) || overlaps(dx, nx, workspace, need) || overlaps(dW0, nw0, workspace, need))
        return SRWM_ERR_ALIAS;
    const void* devs[8] = {W0, dW0, workspace, dW_final, x, dy, dx, nullptr};
    for (int i = 0; i < 7; ++i) {
        if (!devs[i] || (i >= 4 && T == 0)) continue;
        if ((rc = check_device_ptr(devs[i])) != SRWM_OK) return rc;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    BwdWs w;
    bwd_ws(B, T, H, d, n_lr, &w);
    char* base = static_cast<char*>(workspace);
    float* dW_seq = reinterpret_cast<float*>(base + w.dws);
    const size_t per_batch = static_cast<size_t>(H) * m * d;
    if (T == 0) {
        // dL/dW0 = sum over b of dL/dW_final (W_final = W0 for every b)
        if (!dW_final) {
            if (cudaMemsetAsync(dW0, 0, nw0, st) != cudaSuccess) {
                cudaGetLastError();
                return SRWM_ERR_CUDA;
            }
            return SRWM_OK;
        }
        return srwm::launch_sum_over_batch(dW_final, dW0, B, per_batch, st) == 0 ? SRWM_OK : SRWM_ERR_CUDA;
    }
    // 1. the forward pass with its per-step records and W_T
    float* WT = reinterpret_cast<float*>(base + w.wt);
    float* rec = reinterpret_cast<float*>(base + w.rec);
    const int stride = srwm::emit_record_floats(d, n_lr);
    if ((rc = run(x, W0, 0, B, T, H, d, n_lr, softmax_input, reinterpret_cast<float*>(base + w.y), WT, st,
                  reinterpret_cast<int*>(base + w.cnt), static_cast<size_t>(B) * H * 4, rec, stride)) != SRWM_OK)
        return rc;
    // 2. the steps backwards, one CTA per stream or per wrap-around range
    const srwm::BwdLaunch li = srwm::bwd_info(d, n_lr);
    if (cudaFuncSetAttribute(li.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, li.smem_bytes) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    srwm::BwdParams bp;
    bp.x = x;
    bp.WT = WT;
    bp.rec = rec;
    bp.rec_stride = stride;
    bp.dy = dy;
    bp.dWf = dW_final;
    bp.dx = dx;
    bp.dW_seq = dW_seq;
    bp.B = B;
    bp.T = T;
    bp.H = H;
    bp.wrap_len = 0;
    bp.seg_done = nullptr;
    if ((rc = status_ptr(&bp.status)) != SRWM_OK) return rc;
    bp.wait_limit_ns = static_cast<unsigned long long>(g_wait_limit_ns.load());
    int smx = softmax_input;
    void* args[] = {&bp, &smx};
    // More streams than co-resident CTAs: the wrap-around schedule, so that the
    // last wave is not mostly empty (each stream is split at most once).
    const long long pairs = static_cast<long long>(B) * H;
    int dev = 0, n_sm = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, li.kernel, li.threads,
                                                      static_cast<size_t>(li.smem_bytes)) != cudaSuccess ||
        per_sm <= 0) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    const long long slots = static_cast<long long>(n_sm) * per_sm;
    cudaError_t e;
    if (T > 0 && pairs > slots) {
        bp.wrap_len = wrap_len_for(pairs, T, slots, li.kseg);
        bp.seg_done = reinterpret_cast<int*>(base + w.cnt);
        if (cudaMemsetAsync(bp.seg_done, 0, static_cast<size_t>(pairs) * 4, st) != cudaSuccess) {
            cudaGetLastError();
            return SRWM_ERR_CUDA;
        }
        const long long grid = (pairs * T + bp.wrap_len - 1) / bp.wrap_len;
        e = cudaLaunchCooperativeKernel(li.kernel, dim3(static_cast<unsigned>(grid)),
                                        dim3(static_cast<unsigned>(li.threads)), args,
                                        static_cast<size_t>(li.smem_bytes), st);
    } else {
        e = cudaLaunchKernel(li.kernel, dim3(static_cast<unsigned>(pairs)), dim3(static_cast<unsigned>(li.threads)),
                             args, static_cast<size_t>(li.smem_bytes), st);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    // 3. dL/dW0 = sum over sequences, in order of b
    return srwm::launch_sum_over_batch(dW_seq, dW0, B, per_batch, st) == 0 ? SRWM_OK : SRWM_ERR_CUDA;
}

size_t srwm_forward_host_workspace_bytes(int B, int T, int H, int d, int n_lr, int chunk_steps)
{
    if (check_params(B, T, H, d, n_lr, 0) != SRWM_OK) return 0;
    HostWs w;
    host_ws(B, T, H, d, n_lr, effective_chunk(T, d, chunk_steps), &w);
    return w.total;
}

int srwm_forward_host(const float* x_host, const float* W0_host, int B, int T, int H, int d, int n_lr,
                      int softmax_input, float* y_host, float* W_final_host, int chunk_steps, void* workspace,
                      size_t workspace_bytes, void* stream)
{
    if (!W0_host || !W_final_host || !workspace || (T > 0 && (!x_host || !y_host))) return SRWM_ERR_NULL;
    int rc = check_params(B, T, H, d, n_lr, softmax_input);
    if (rc != SRWM_OK) return rc;
    const int C = effective_chunk(T, d, chunk_steps);
    HostWs w;
    host_ws(B, T, H, d, n_lr, C, &w);
    if (workspace_bytes < w.total) return SRWM_ERR_SHAPE;
    if (!aligned16(workspace)) return SRWM_ERR_ALIGN;
    if ((rc = check_device_ptr(workspace)) != SRWM_OK) return rc;
    const long long m = 3LL * d + n_lr;
    const size_t nx = static_cast<size_t>(B) * T * H * d * 4, nwf = static_cast<size_t>(B) * H * m * d * 4;
    if (T > 0 && (overlaps(y_host, nx, x_host, nx) || overlaps(y_host, nx, W0_host, static_cast<size_t>(H * m * d) * 4) ||
                  overlaps(y_host, nx, W_final_host, nwf) || overlaps(W_final_host, nwf, x_host, nx)))
        return SRWM_ERR_ALIAS;
    const void* hosts[] = {x_host, W0_host, y_host, W_final_host};
    for (const void* hp : hosts) {
        if (!hp) continue;
        if ((rc = check_host_ptr(hp)) != SRWM_OK) return rc;
    }
    cudaStream_t sc = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(workspace);
    float* W0d = reinterpret_cast<float*>(base + w.w0);
    float* S = reinterpret_cast<float*>(base + w.state);
    int* cnt = reinterpret_cast<int*>(base + w.cnt);
    const size_t row = static_cast<size_t>(H) * d * 4;   // one step of one sequence
    auto fail = [](cudaError_t e) { return e != cudaSuccess; };
    const std::vector<int> plan = chunk_plan(T, d, chunk_steps);
    const int K = static_cast<int>(plan.size());

    if (K <= 1) {
        // One chunk (or none): there is nothing for the copies to overlap, so
        // they run in order on the caller's stream, without the copy streams
        // and the events that order them.
        float* xb = reinterpret_cast<float*>(base + w.x[0]);
        float* yb = reinterpret_cast<float*>(base + w.y[0]);
        if (fail(cudaMemcpyAsync(W0d, W0_host, static_cast<size_t>(H * m * d) * 4, cudaMemcpyHostToDevice, sc)) ||
            (T > 0 && fail(cudaMemcpyAsync(xb, x_host, nx, cudaMemcpyHostToDevice, sc)))) {
            cudaGetLastError();
            return SRWM_ERR_CUDA;
        }
        if (T == 0) {
            if ((rc = run(nullptr, W0d, 0, B, 0, H, d, n_lr, softmax_input, nullptr, S, sc)) != SRWM_OK) return rc;
        } else if ((rc = run(xb, W0d, 0, B, T, H, d, n_lr, softmax_input, yb, S, sc, cnt,
                             static_cast<size_t>(B) * H * 4)) != SRWM_OK) {
            return rc;
        }
        if ((T > 0 && fail(cudaMemcpyAsync(y_host, yb, nx, cudaMemcpyDeviceToHost, sc))) ||
            fail(cudaMemcpyAsync(W_final_host, S, nwf, cudaMemcpyDeviceToHost, sc))) {
            cudaGetLastError();
            return SRWM_ERR_CUDA;
        }
        return SRWM_OK;
    }

    Pipe* pp = nullptr;
    if ((rc = pipe_for_device(&pp)) != SRWM_OK) return rc;
    Pipe& P = *pp;
    std::lock_guard<std::mutex> lk(P.mu);

    // the copy streams start after the work already on the caller's stream
    if (fail(cudaEventRecord(P.start, sc)) || fail(cudaStreamWaitEvent(P.s_in, P.start, 0)) ||
        fail(cudaStreamWaitEvent(P.s_out, P.start, 0)) ||
        fail(cudaMemcpyAsync(W0d, W0_host, static_cast<size_t>(H * m * d) * 4, cudaMemcpyHostToDevice, P.s_in)) ||
        fail(cudaEventRecord(P.w0, P.s_in)) || fail(cudaStreamWaitEvent(sc, P.w0, 0))) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    for (int k = 0, t0 = 0; k < K; t0 += plan[k], ++k) {
        const int slot = k % kPipeSlots, Ck = plan[k];
        float* xb = reinterpret_cast<float*>(base + w.x[slot]);
        float* yb = reinterpret_cast<float*>(base + w.y[slot]);
        // x chunk k: host [B, T, H, d] rows t0 .. t0+Ck-1 -> contiguous [B, Ck, H, d]
        if ((k >= kPipeSlots && fail(cudaStreamWaitEvent(P.s_in, P.comp[slot], 0))) ||
            fail(cudaMemcpy2DAsync(xb, Ck * row, reinterpret_cast<const char*>(x_host) + t0 * row, T * row, Ck * row,
                                   B, cudaMemcpyHostToDevice, P.s_in)) ||
            fail(cudaEventRecord(P.in[slot], P.s_in)) || fail(cudaStreamWaitEvent(sc, P.in[slot], 0)) ||
            (k >= kPipeSlots && fail(cudaStreamWaitEvent(sc, P.out[slot], 0)))) {
            cudaGetLastError();
            return SRWM_ERR_CUDA;
        }
        // the recurrence on chunk k, carrying the state in S (in place after the first chunk)
        if ((rc = run(xb, k == 0 ? W0d : S, k == 0 ? 0 : 1, B, Ck, H, d, n_lr, softmax_input, yb, S, sc, cnt,
                      static_cast<size_t>(B) * H * 4)) != SRWM_OK)
            return rc;
        // y chunk k back to host rows t0 .. t0+Ck-1
        if (fail(cudaEventRecord(P.comp[slot], sc)) || fail(cudaStreamWaitEvent(P.s_out, P.comp[slot], 0)) ||
            fail(cudaMemcpy2DAsync(reinterpret_cast<char*>(y_host) + t0 * row, T * row, yb, Ck * row, Ck * row, B,
                                   cudaMemcpyDeviceToHost, P.s_out)) ||
            fail(cudaEventRecord(P.out[slot], P.s_out))) {
            cudaGetLastError();
            return SRWM_ERR_CUDA;
        }
    }
    // the final state, then the caller's stream waits for every copy
    if (fail(cudaEventRecord(P.end, sc)) || fail(cudaStreamWaitEvent(P.s_out, P.end, 0)) ||
        fail(cudaMemcpyAsync(W_final_host, S, nwf, cudaMemcpyDeviceToHost, P.s_out)) ||
        fail(cudaEventRecord(P.end, P.s_out)) || fail(cudaStreamWaitEvent(sc, P.end, 0))) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    return SRWM_OK;
}

int srwm_forward_from(const float* x, const float* W_init, int B, int T, int H, int d, int n_lr,
                      int softmax_input, float* y_out, float* W_final, void* stream)
{
    if (!W_init || !W_final || (T > 0 && (!x || !y_out))) return SRWM_ERR_NULL;
    const int rc = check_params(B, T, H, d, n_lr, softmax_input);
    if (rc != SRWM_OK) return rc;
    return run(x, W_init, 1, B, T, H, d, n_lr, softmax_input, y_out, W_final,
               static_cast<cudaStream_t>(stream));
}

int srwm_step(const float* x_t, const float* W_in, int B, int H, int d, int n_lr,
              int softmax_input, float* y_t, float* W_out, void* stream)
{
    if (!x_t || !W_in || !y_t || !W_out) return SRWM_ERR_NULL;
    const int rc = check_params(B, 1, H, d, n_lr, softmax_input);
    if (rc != SRWM_OK) return rc;
    return run(x_t, W_in, 1, B, 1, H, d, n_lr, softmax_input, y_t, W_out,
               static_cast<cudaStream_t>(stream));
}

const char* srwm_status_string(int status)
{
    switch (status) {
        case SRWM_OK: return "SRWM_OK";
        case SRWM_ERR_NULL: return "SRWM_ERR_NULL: a required pointer is NULL";
        case SRWM_ERR_SHAPE: return "SRWM_ERR_SHAPE: invalid or too large B/T/H/d";
        case SRWM_ERR_UNSUPPORTED: return "SRWM_ERR_UNSUPPORTED: d must be 16/32/64, n_lr 1/4, softmax_input 0/1";
        case SRWM_ERR_ALIGN: return "SRWM_ERR_ALIGN: pointers must be 16-byte aligned";
        case SRWM_ERR_ALIAS: return "SRWM_ERR_ALIAS: an output overlaps an input or another output";
        case SRWM_ERR_CUDA: return "SRWM_ERR_CUDA: a CUDA runtime call failed";
        case SRWM_ERR_TIMEOUT: return "SRWM_ERR_TIMEOUT: a kernel gave up a bounded wait";
        case SRWM_ERR_NOT_DEVICE: return "SRWM_ERR_NOT_DEVICE: pointer is not device memory of the current device";
        default: return "SRWM: unknown status";
    }
}

int srwm_last_device_status(void* stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    unsigned* dptr = nullptr;
    int rc = status_ptr(&dptr);
    if (rc != SRWM_OK) return rc;
    unsigned v = 0;
    if (cudaMemcpy(&v, dptr, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    if (v == 0) return SRWM_OK;
    const unsigned zero = 0;
    if (cudaMemcpy(dptr, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    return (v & srwm::kStatusTimeout) ? SRWM_ERR_TIMEOUT : SRWM_ERR_CUDA;
}

int srwm_set_wait_limit_ns(long long limit_ns)
{
    g_wait_limit_ns.store(limit_ns < 1000 ? 1000 : limit_ns);
    return SRWM_OK;
}

int srwm_debug_skip_x_chunk(int chunk)
{
    g_skip_chunk.store(chunk < 0 ? -1 : chunk);
    return SRWM_OK;
}

}  // extern "C"
