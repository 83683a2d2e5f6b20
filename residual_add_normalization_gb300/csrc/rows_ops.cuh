// rows_ops.cuh -- typed entry points of the row kernels, instantiated per
// element type in rows_ssln_f32.cu / rows_ssln_f16.cu / rows_gated.cu.
#pragma once

#include "rows_launch.cuh"

namespace b200norm {

// Row plans that need a cluster the device cannot co-schedule fall back to
// the walking schedule.
template <class Op>
RowPlan settle_plan(RowPlan p, int64_t rows) {
  if (p.mode == 1 && p.csize > 1 && !cluster_fits<Op>(p.nv, p.block, p.csize)) {
    p.mode = 2;
    p.block = kRowsMaxThreads;
    p.tpr = kRowsMaxThreads;
    p.csize = 1;
    p.grid = rows;
  }
  return p;
}

template <typename T, int VE, bool HAS_BIAS, bool WANT_S>
cudaError_t skip_rms_go(const SkipRmsCall& c, const RowPlan& plan, cudaStream_t st) {
  using Op = SkipRmsOp<T, VE, HAS_BIAS, WANT_S>;
  SkipRmsArgs<T> a;
  a.x = static_cast<const T*>(c.x);
  a.skip = static_cast<const T*>(c.skip);
  a.gamma = static_cast<const T*>(c.gamma);
  a.bias = static_cast<const T*>(c.bias);
  a.y = static_cast<T*>(c.y);
  a.s = static_cast<T*>(c.s);
  a.mean = c.mean;
  a.inv_std = c.inv_std;
  a.rows = c.rows;
  a.n = static_cast<int>(c.hidden);
  a.inv_n = 1.0f / static_cast<float>(c.hidden);
  a.eps = c.eps;
  return launch_rows_op<Op>(a, settle_plan<Op>(plan, c.rows), st);
}

template <typename T, int VE>
cudaError_t skip_rms_flags(const SkipRmsCall& c, const RowPlan& p, cudaStream_t st) {
  if (c.bias) {
    return c.s ? skip_rms_go<T, VE, true, true>(c, p, st) : skip_rms_go<T, VE, true, false>(c, p, st);
  }
  return c.s ? skip_rms_go<T, VE, false, true>(c, p, st) : skip_rms_go<T, VE, false, false>(c, p, st);
}

template <typename T, int VE>
cudaError_t gated_go(const GatedCall& c, const RowPlan& plan, cudaStream_t st) {
  using Op = GatedOp<T, VE>;
  GatedArgs<T> a;
  a.x = static_cast<const T*>(c.x);
  a.gate = static_cast<const T*>(c.gate);
  a.scale = static_cast<const T*>(c.scale);
  a.y = static_cast<T*>(c.y);
  a.rows = c.rows;
  a.n = static_cast<int>(c.C);
  a.inv_n = 1.0f / static_cast<float>(c.C);
  a.eps = c.eps;
  return launch_rows_op<Op>(a, settle_plan<Op>(plan, c.rows), st);
}

cudaError_t skip_rms_f32(const SkipRmsCall& c, const RowPlan& p, cudaStream_t st);
cudaError_t skip_rms_f16(const SkipRmsCall& c, const RowPlan& p, cudaStream_t st);
cudaError_t skip_rms_bf16(const SkipRmsCall& c, const RowPlan& p, cudaStream_t st);
cudaError_t gated_bf16(const GatedCall& c, const RowPlan& p, cudaStream_t st);

}  // namespace b200norm
