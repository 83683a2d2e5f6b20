// SkipSimplifiedLayerNormalization row kernels, float32.
#include "rows_ops.cuh"

namespace b200norm {
cudaError_t skip_rms_f32(const SkipRmsCall& c, const RowPlan& p, cudaStream_t st) {
  return p.ve == 4 ? skip_rms_flags<float, 4>(c, p, st) : skip_rms_flags<float, 1>(c, p, st);
}
}  // namespace b200norm
