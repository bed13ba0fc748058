// srwm_d64.cu -- instantiations of the d = 64 kernel (one translation unit
// per width so the library builds in parallel).
#include "srwm_d64.cuh"

namespace srwm {

LaunchInfo launch_info_d64(int n_lr, int softmax_input)
{
    if (n_lr == 1) return softmax_input ? launch_info_d64_impl<1, true>() : launch_info_d64_impl<1, false>();
    return softmax_input ? launch_info_d64_impl<4, true>() : launch_info_d64_impl<4, false>();
}

}  // namespace srwm
