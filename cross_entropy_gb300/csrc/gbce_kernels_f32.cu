// fp32-logit instantiations of the row kernels.
#include "gbce_dispatch.cuh"

namespace gbce {
template cudaError_t launch_rows<float>(const RowParams &, int, cudaStream_t);
}  // namespace gbce
