// fo_step_lion.cu -- FlashLion launches (kernels in fo_step.cuh).
#include "fo_step.cuh"

namespace fo {

cudaError_t launch_step_lion(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream)
{
    return launch_widths<Opt::kLion, false, false>(rho_bits, grad_bits, p, stream);
}

}  // namespace fo
