// srwm_d64.cu -- instantiations of the d = 64 kernels (one translation unit
// per width so the library builds in parallel).
#include "srwm_d64.cuh"
#include "srwm_d64r.cuh"

namespace srwm {

namespace {

template <bool EMIT>
LaunchInfo pick(int n_lr, int softmax_input, bool two_warps)
{
    if (two_warps) {
        if (n_lr == 1)
            return softmax_input ? launch_info_d64r_impl<1, true, EMIT>() : launch_info_d64r_impl<1, false, EMIT>();
        return softmax_input ? launch_info_d64r_impl<4, true, EMIT>() : launch_info_d64r_impl<4, false, EMIT>();
    }
    if (n_lr == 1)
        return softmax_input ? launch_info_d64_impl<4, 1, true, EMIT>() : launch_info_d64_impl<4, 1, false, EMIT>();
    return softmax_input ? launch_info_d64_impl<4, 4, true, EMIT>() : launch_info_d64_impl<4, 4, false, EMIT>();
}

}  // namespace

// Two kernels, chosen by the number of (sequence, head) streams per SM:
//   * up to two per SM: four warps per stream (two CTAs per SM).  Each stream
//     then has a slot of its own, and four warps give the shortest step.
//     (Eight warps per stream, one stream per SM, was measured slower on the
//     long workload: each warp reloads the step's vectors from shared memory,
//     and that traffic grows with the warp count.)
//   * more: two warps per stream with whole rows of W per thread, four CTAs
//     per SM, so twice as many streams advance at once.
// emit selects the instantiations that also write the backward records.
LaunchInfo launch_info_d64(int n_lr, int softmax_input, long long n_streams, int n_sm, bool emit)
{
    const bool two_warps = n_streams > 2LL * n_sm;
    return emit ? pick<true>(n_lr, softmax_input, two_warps) : pick<false>(n_lr, softmax_input, two_warps);
}

}  // namespace srwm
