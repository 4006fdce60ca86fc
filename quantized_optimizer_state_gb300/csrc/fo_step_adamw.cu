// fo_step_adamw.cu -- FlashAdamW launches with the step counter from the host
// (the kernels are in fo_step.cuh; this translation unit instantiates them).
#include "fo_step.cuh"

namespace fo {

cudaError_t launch_step_adamw(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream)
{
    return p.s.v_nonzero ? launch_widths<Opt::kAdamW, true, false>(rho_bits, grad_bits, p, stream)
                         : launch_widths<Opt::kAdamW, false, false>(rho_bits, grad_bits, p, stream);
}

}  // namespace fo
