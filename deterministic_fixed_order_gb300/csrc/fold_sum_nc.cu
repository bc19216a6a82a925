// Kernel instantiations and launcher for mode kSumNC (see detfold_kernels.cuh).
#include "detfold_launch.cuh"

namespace detfold {

cudaError_t launch_sum_nc(const LaunchSpec &s, cudaStream_t stream)
{
    return launch_mode<kSumNC>(s, stream);
}

}  // namespace detfold
