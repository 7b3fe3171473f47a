// reduce_depth.cu -- the fused reduction with the depth-spread weights (a
// translation unit of its own so that the library's sources compile in
// parallel; the kernel template is reduce_kernel.cuh).
#include "reduce_kernel.cuh"

namespace ssb {

cudaError_t launch_reduce_depth(const RedLaunch& P, const SetBatch& sb, cudaStream_t st) {
    return launch_reduce_t<true>(P, sb, st);
}

}  // namespace ssb
