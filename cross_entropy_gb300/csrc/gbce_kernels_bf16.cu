// bf16-logit instantiations of the row kernels.
#include "gbce_dispatch.cuh"

namespace gbce {
template cudaError_t launch_rows<__nv_bfloat16>(const RowParams &, int, cudaStream_t);
}  // namespace gbce
