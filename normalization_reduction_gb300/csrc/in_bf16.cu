// InstanceNorm kernels with __nv_bfloat16 input (both output types).
#include "in_kernels.cuh"

namespace fnorm {
template cudaError_t in_launch_t<__nv_bfloat16, __nv_bfloat16>(const InParams&, const InPlan&, cudaStream_t);
template int in_max_active_clusters_t<__nv_bfloat16, __nv_bfloat16>(const InPlan&);
template cudaError_t in_launch_t<__nv_bfloat16, float>(const InParams&, const InPlan&, cudaStream_t);
template int in_max_active_clusters_t<__nv_bfloat16, float>(const InPlan&);
}  // namespace fnorm
