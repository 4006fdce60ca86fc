// fo_step_sgd.cu -- FlashSGD launches (kernels in fo_step.cuh).
#include "fo_step.cuh"

namespace fo {

cudaError_t launch_step_sgd(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream)
{
    return launch_widths<Opt::kSgd, false, false>(rho_bits, grad_bits, p, stream);
}

}  // namespace fo
