// SkipGroupNorm kernels for bfloat16 X, S and Y (gamma / beta float32 or
// bfloat16).
#include "group_kernels.cuh"

namespace b200norm {

void* group_coop_kernel_bf16(DType m, int ve, int nv) {
  if (m == DType::F32) return pick_coop<__nv_bfloat16, float>(ve, nv);
  if (m == DType::BF16) return pick_coop<__nv_bfloat16, __nv_bfloat16>(ve, nv);
  return nullptr;
}

void* group_resident_kernel_bf16(DType m, int ve) {
  if (m == DType::F32) return pick_resident<__nv_bfloat16, float>(ve);
  if (m == DType::BF16) return pick_resident<__nv_bfloat16, __nv_bfloat16>(ve);
  return nullptr;
}

void* group_slab_kernel_bf16(DType m, int ve) {
  if (m == DType::F32) return pick_slab<__nv_bfloat16, float>(ve);
  if (m == DType::BF16) return pick_slab<__nv_bfloat16, __nv_bfloat16>(ve);
  return nullptr;
}

void* group_coop_l2_kernel_bf16(DType m, int ve, bool bcast) {
  if (m == DType::F32) return pick_coop_l2<__nv_bfloat16, float>(ve, bcast);
  if (m == DType::BF16) return pick_coop_l2<__nv_bfloat16, __nv_bfloat16>(ve, bcast);
  return nullptr;
}

cudaError_t launch_group_bf16(const SkipGroupCall& c, const GroupPlan& p, cudaStream_t stream) {
  if (c.m == DType::F32) return launch_group_typed<__nv_bfloat16, float>(c, p, stream);
  if (c.m == DType::BF16) return launch_group_typed<__nv_bfloat16, __nv_bfloat16>(c, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace b200norm
