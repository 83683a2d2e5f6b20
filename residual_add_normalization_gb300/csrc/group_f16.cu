// SkipGroupNorm kernels for float16 X, S and Y (gamma / beta float32 or
// float16).
#include "group_kernels.cuh"

namespace b200norm {

void* group_coop_kernel_f16(DType m, int ve, int nv) {
  if (m == DType::F32) return pick_coop<__half, float>(ve, nv);
  if (m == DType::F16) return pick_coop<__half, __half>(ve, nv);
  return nullptr;
}

void* group_resident_kernel_f16(DType m, int ve) {
  if (m == DType::F32) return pick_resident<__half, float>(ve);
  if (m == DType::F16) return pick_resident<__half, __half>(ve);
  return nullptr;
}

void* group_slab_kernel_f16(DType m, int ve) {
  if (m == DType::F32) return pick_slab<__half, float>(ve);
  if (m == DType::F16) return pick_slab<__half, __half>(ve);
  return nullptr;
}

void* group_coop_l2_kernel_f16(DType m, int ve, bool bcast) {
  if (m == DType::F32) return pick_coop_l2<__half, float>(ve, bcast);
  if (m == DType::F16) return pick_coop_l2<__half, __half>(ve, bcast);
  return nullptr;
}

cudaError_t launch_group_f16(const SkipGroupCall& c, const GroupPlan& p, cudaStream_t stream) {
  if (c.m == DType::F32) return launch_group_typed<__half, float>(c, p, stream);
  if (c.m == DType::F16) return launch_group_typed<__half, __half>(c, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace b200norm
