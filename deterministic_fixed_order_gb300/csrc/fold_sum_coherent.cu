// Kernel instantiations and launcher for mode kSumCoherent (see detfold_kernels.cuh).
#include "detfold_launch.cuh"

namespace detfold {

cudaError_t launch_sum_coherent(const LaunchSpec &s, cudaStream_t stream)
{
    return launch_mode<kSumCoherent>(s, stream);
}

}  // namespace detfold
