// SkipSimplifiedLayerNormalization row kernels, float16.
#include "rows_ops.cuh"

namespace b200norm {
cudaError_t skip_rms_f16(const SkipRmsCall& c, const RowPlan& p, cudaStream_t st) {
  return p.ve == 8 ? skip_rms_flags<__half, 8>(c, p, st) : skip_rms_flags<__half, 1>(c, p, st);
}
}  // namespace b200norm
