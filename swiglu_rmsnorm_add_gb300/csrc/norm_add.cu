// Residual-add + RMSNorm launchers (the ADD = true half of the family in norm_impl.cuh).
#include "norm_impl.cuh"

namespace sra {

cudaError_t launch_add_rmsnorm(const NormArgs& a, const NormPlan& p, int dtype, cudaStream_t s) {
    return norm::launch<true>(a, p, dtype, s);
}

}  // namespace sra
