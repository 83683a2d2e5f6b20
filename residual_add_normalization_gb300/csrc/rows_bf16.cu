// SkipSimplifiedLayerNormalization and GatedRMSNorm row kernels, bfloat16.
#include "rows_ops.cuh"

namespace b200norm {

cudaError_t skip_rms_bf16(const SkipRmsCall& c, const RowPlan& p, cudaStream_t st) {
  return p.ve == 8 ? skip_rms_flags<__nv_bfloat16, 8>(c, p, st)
                   : skip_rms_flags<__nv_bfloat16, 1>(c, p, st);
}

cudaError_t gated_bf16(const GatedCall& c, const RowPlan& p, cudaStream_t st) {
  return p.ve == 8 ? gated_go<__nv_bfloat16, 8>(c, p, st) : gated_go<__nv_bfloat16, 1>(c, p, st);
}

}  // namespace b200norm
