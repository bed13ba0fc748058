// srwm_d64.cu -- instantiations of the d = 64 kernel (one translation unit
// per width so the library builds in parallel).
#include "srwm_d64.cuh"

namespace srwm {

// Four warps per stream.  (Eight warps per stream, one stream per SM, was
// measured slower on the long workload: each warp reloads the step's vectors
// from shared memory, and that traffic grows with the warp count.)
LaunchInfo launch_info_d64(int n_lr, int softmax_input)
{
    if (n_lr == 1) return softmax_input ? launch_info_d64_impl<4, 1, true>() : launch_info_d64_impl<4, 1, false>();
    return softmax_input ? launch_info_d64_impl<4, 4, true>() : launch_info_d64_impl<4, 4, false>();
}

}  // namespace srwm
