// SkipGroupNorm kernels for float32 X, S and Y (gamma / beta float32 or
// float16).
#include "group_kernels.cuh"

namespace b200norm {

void* group_coop_kernel_f32(DType m, int ve, int nv) {
  if (m == DType::F32) return pick_coop<float, float>(ve, nv);
  if (m == DType::F16) return pick_coop<float, __half>(ve, nv);
  return nullptr;
}

void* group_resident_kernel_f32(DType m, int ve) {
  if (m == DType::F32) return pick_resident<float, float>(ve);
  if (m == DType::F16) return pick_resident<float, __half>(ve);
  return nullptr;
}

void* group_slab_kernel_f32(DType m, int ve) {
  if (m == DType::F32) return pick_slab<float, float>(ve);
  if (m == DType::F16) return pick_slab<float, __half>(ve);
  return nullptr;
}

void* group_coop_l2_kernel_f32(DType m, int ve, bool bcast) {
  if (m == DType::F32) return pick_coop_l2<float, float>(ve, bcast);
  if (m == DType::F16) return pick_coop_l2<float, __half>(ve, bcast);
  return nullptr;
}

cudaError_t launch_group_f32(const SkipGroupCall& c, const GroupPlan& p, cudaStream_t stream) {
  if (c.m == DType::F32) return launch_group_typed<float, float>(c, p, stream);
  if (c.m == DType::F16) return launch_group_typed<float, __half>(c, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace b200norm
