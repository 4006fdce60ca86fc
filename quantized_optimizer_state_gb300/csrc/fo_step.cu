// fo_step.cu -- dispatch of a fused-step launch to the translation unit that
// instantiates its kernel (fo_step_adamw.cu, fo_step_adamw_dev.cu,
// fo_step_sgd.cu, fo_step_lion.cu; the kernels are in fo_step.cuh).
#include "fo_internal.h"

namespace fo {

cudaError_t launch_step_adamw(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream);
cudaError_t launch_step_adamw_dev(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream);
cudaError_t launch_step_sgd(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream);
cudaError_t launch_step_lion(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream);

cudaError_t launch_step(Opt opt, int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream)
{
    switch (opt) {
    case Opt::kAdamW:
        return p.s.step_dev ? launch_step_adamw_dev(rho_bits, grad_bits, p, stream)
                            : launch_step_adamw(rho_bits, grad_bits, p, stream);
    case Opt::kSgd: return launch_step_sgd(rho_bits, grad_bits, p, stream);
    default: return launch_step_lion(rho_bits, grad_bits, p, stream);
    }
}

}  // namespace fo
