// srwm_d16.cu -- instantiations of the d = 16 kernels (one translation unit
// per width so the library builds in parallel).
#include "srwm_d16r.cuh"

namespace srwm {

LaunchInfo launch_info_d16(int n_lr, int softmax_input, bool emit)
{
    if (emit) {
        if (n_lr == 1) return softmax_input ? launch_info_d16_impl<1, true, true>() : launch_info_d16_impl<1, false, true>();
        return softmax_input ? launch_info_d16_impl<4, true, true>() : launch_info_d16_impl<4, false, true>();
    }
    if (n_lr == 1) return softmax_input ? launch_info_d16_impl<1, true>() : launch_info_d16_impl<1, false>();
    return softmax_input ? launch_info_d16_impl<4, true>() : launch_info_d16_impl<4, false>();
}

}  // namespace srwm
