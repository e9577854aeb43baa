// InstanceNorm kernels with float input (both output types).
#include "in_kernels.cuh"

namespace fnorm {
template cudaError_t in_launch_t<float, float>(const InParams&, const InPlan&, cudaStream_t);
template int in_max_active_clusters_t<float, float>(const InPlan&);
template cudaError_t in_launch_t<float, __nv_bfloat16>(const InParams&, const InPlan&, cudaStream_t);
template int in_max_active_clusters_t<float, __nv_bfloat16>(const InPlan&);
}  // namespace fnorm
