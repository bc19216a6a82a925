// Kernel instantiations and launcher for mode kAllReduce (see detfold_kernels.cuh).
#include "detfold_launch.cuh"

namespace detfold {

cudaError_t launch_allreduce(const LaunchSpec &s, cudaStream_t stream)
{
    return launch_mode<kAllReduce>(s, stream);
}

}  // namespace detfold
