// fo_step_adamw_dev.cu -- FlashAdamW launches with the step counter read from
// device memory by the kernel (fo_adamw_step_dev; kernels in fo_step.cuh).
#include "fo_step.cuh"

namespace fo {

cudaError_t launch_step_adamw_dev(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream)
{
    return p.s.v_nonzero ? launch_widths<Opt::kAdamW, true, true>(rho_bits, grad_bits, p, stream)
                         : launch_widths<Opt::kAdamW, false, true>(rho_bits, grad_bits, p, stream);
}

}  // namespace fo
