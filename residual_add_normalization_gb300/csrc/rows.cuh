// rows.cuh -- row-normalization kernels shared by SkipSimplifiedLayerNormalization
// and GatedRMSNorm (sm_103a).
//
// A "row" is one normalization span: the hidden axis of SSLN, or one C-span of
// GatedRMSNorm.  Each row is read once from HBM with 16-byte vector loads, kept
// in registers while its sum of squares is reduced, then normalized and
// written.  Three schedules:
//
//   rows_kernel, tpr <= 32   lane groups of `tpr` threads (a power of two) per
//                            row, several rows per warp, RPG rows per lane group
//                            in flight; the reduction is a segmented butterfly
//                            over the low lane bits (no shared memory, no
//                            barrier).
//   rows_kernel, tpr  > 32   one row per CTA, or per thread-block cluster for
//                            long rows: warp butterflies, a shared-memory
//                            combine, then a DSMEM combine across the cluster.
//   rows_walk_kernel         rows longer than a cluster holds: one CTA walks
//                            the row twice (the second pass is served by L2).
//
// Op policies (SkipRmsOp, GatedOp) supply the per-vector load / combine /
// finish steps; the schedule code is shared.
#pragma once

#include "common.cuh"

namespace b200norm {

// ---------------------------------------------------------------------------
// Arguments
// ---------------------------------------------------------------------------
template <typename T>
struct SkipRmsArgs {
  const T* __restrict__ x;
  const T* __restrict__ skip;
  const T* __restrict__ gamma;
  const T* __restrict__ bias;  // may be null (then HAS_BIAS is false)
  T* __restrict__ y;
  T* __restrict__ s;           // may be null (then WANT_S is false)
  float* __restrict__ mean;    // may be null
  float* __restrict__ inv_std; // may be null
  int64_t rows;
  int n;                       // hidden
  float eps;
};

template <typename T>
struct GatedArgs {
  const T* __restrict__ x;
  const T* __restrict__ gate;
  const T* __restrict__ scale;
  T* __restrict__ y;
  int64_t rows;
  int n;                       // C
  float eps;
};

// ---------------------------------------------------------------------------
// SkipSimplifiedLayerNormalization
//   S = round_T((x + skip) + bias); y = round_T(S * rstd * gamma),
//   rstd = 1 / sqrt(sum(S^2) / n + eps)
// ---------------------------------------------------------------------------
template <typename T, int VE, bool HAS_BIAS, bool WANT_S>
struct SkipRmsOp {
  using Args = SkipRmsArgs<T>;
  using P = Pack<T, VE>;
  static constexpr int kVE = VE;
  struct In {
    P x, k;
  };
  using Hold = P;

  __device__ static __forceinline__ void load(const Args& a, int64_t row, int v, In& in) {
    const int64_t off = row * a.n + static_cast<int64_t>(v) * VE;
    in.x = ld_stream<T, VE>(a.x + off);
    in.k = ld_stream<T, VE>(a.skip + off);
  }

  template <bool STORE_S = WANT_S>
  __device__ static __forceinline__ float combine(const Args& a, int64_t row, int v,
                                                  const In& in, Hold& h) {
    P b;
    if constexpr (HAS_BIAS) b = ld_reuse<T, VE>(a.bias + v * VE);
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      h.v[e] = residual_sum<T, HAS_BIAS>(in.x.v[e], in.k.v[e], HAS_BIAS ? b.v[e] : T());
      const float f = to_f32(h.v[e]);
      ss = fmaf(f, f, ss);
    }
    if constexpr (STORE_S) st_stream<T, VE>(a.s + row * a.n + static_cast<int64_t>(v) * VE, h);
    return ss;
  }

  __device__ static __forceinline__ float rstd(const Args& a, float sumsq) {
    return 1.0f / sqrtf(sumsq / static_cast<float>(a.n) + a.eps);
  }

  __device__ static __forceinline__ void finish(const Args& a, int64_t row, int v,
                                                const Hold& h, float r) {
    const P g = ld_reuse<T, VE>(a.gamma + v * VE);
    P out;
#pragma unroll
    for (int e = 0; e < VE; ++e) out.v[e] = from_f32<T>(to_f32(h.v[e]) * r * to_f32(g.v[e]));
    st_stream<T, VE>(a.y + row * a.n + static_cast<int64_t>(v) * VE, out);
  }

  __device__ static __forceinline__ void row_stats(const Args& a, int64_t row, float r) {
    if (a.mean) a.mean[row] = 0.0f;
    if (a.inv_std) a.inv_std[row] = r;
  }
};

// ---------------------------------------------------------------------------
// GatedRMSNorm
//   y = round_T(x * rstd * scale * SiLU(gate)), rstd = 1 / sqrt(sum(x^2) / C + eps)
// ---------------------------------------------------------------------------
template <typename T, int VE>
struct GatedOp {
  using Args = GatedArgs<T>;
  using P = Pack<T, VE>;
  static constexpr int kVE = VE;
  struct In {
    P x, g;
  };
  using Hold = In;

  __device__ static __forceinline__ void load(const Args& a, int64_t row, int v, In& in) {
    const int64_t off = row * a.n + static_cast<int64_t>(v) * VE;
    in.x = ld_stream<T, VE>(a.x + off);
    in.g = ld_stream<T, VE>(a.gate + off);
  }

  template <bool STORE_S = false>
  __device__ static __forceinline__ float combine(const Args&, int64_t, int, const In& in,
                                                  Hold& h) {
    h = in;
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      const float f = to_f32(in.x.v[e]);
      ss = fmaf(f, f, ss);
    }
    return ss;
  }

  __device__ static __forceinline__ float rstd(const Args& a, float sumsq) {
    return 1.0f / sqrtf(sumsq / static_cast<float>(a.n) + a.eps);
  }

  __device__ static __forceinline__ void finish(const Args& a, int64_t row, int v,
                                                const Hold& h, float r) {
    const P sc = ld_reuse<T, VE>(a.scale + v * VE);
    P out;
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      const float z = to_f32(h.x.v[e]) * r * to_f32(sc.v[e]);
      out.v[e] = from_f32<T>(z * silu_f32(to_f32(h.g.v[e])));
    }
    st_stream<T, VE>(a.y + row * a.n + static_cast<int64_t>(v) * VE, out);
  }

  __device__ static __forceinline__ void row_stats(const Args&, int64_t, float) {}
};

// ---------------------------------------------------------------------------
// Register-resident schedules
// ---------------------------------------------------------------------------
constexpr int kRowsMaxThreads = 512;

// tpr <= 32: lane groups of tpr threads, RPG rows per lane group per CTA.
// tpr  > 32: tpr == blockDim.x * cluster size, one row per CTA / cluster, RPG == 1.
// nvec: vectors of Op::kVE elements per row.  Each thread holds up to NV
// vectors per row (nvec <= NV * tpr).
template <class Op, int NV, int RPG>
__global__ void __launch_bounds__(kRowsMaxThreads)
rows_kernel(const typename Op::Args a, int tpr, int nvec) {
  __shared__ float red[33];
  __shared__ float cl_slot;
  typename Op::In in[RPG][NV];
  typename Op::Hold h[RPG][NV];
  float part[RPG];

  if (tpr <= 32) {
    const int lane = threadIdx.x & (tpr - 1);
    const int group = threadIdx.x / tpr;
    const int groups_per_cta = blockDim.x / tpr;
    const int64_t base = static_cast<int64_t>(blockIdx.x) * groups_per_cta * RPG + group;
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
      const int64_t row = base + static_cast<int64_t>(i) * groups_per_cta;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int v = lane + k * tpr;
        if (row < a.rows && v < nvec) Op::load(a, row, v, in[i][k]);
      }
    }
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
      const int64_t row = base + static_cast<int64_t>(i) * groups_per_cta;
      part[i] = 0.0f;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int v = lane + k * tpr;
        if (row < a.rows && v < nvec) part[i] += Op::combine(a, row, v, in[i][k], h[i][k]);
      }
    }
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
      const int64_t row = base + static_cast<int64_t>(i) * groups_per_cta;
      const float r = Op::rstd(a, seg_sum(part[i], tpr));
      if (row >= a.rows) continue;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int v = lane + k * tpr;
        if (v < nvec) Op::finish(a, row, v, h[i][k], r);
      }
      if (lane == 0) Op::row_stats(a, row, r);
    }
    return;
  }

  // One row per CTA or per cluster.
  const unsigned csize = cluster_size();
  const unsigned rank = csize > 1 ? cluster_rank() : 0u;
  const int64_t row = blockIdx.x / csize;
  const int first = threadIdx.x + static_cast<int>(rank) * blockDim.x;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = first + k * tpr;
    if (v < nvec) Op::load(a, row, v, in[0][k]);
  }
  float acc = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = first + k * tpr;
    if (v < nvec) acc += Op::combine(a, row, v, in[0][k], h[0][k]);
  }
  float total = cta_sum(acc, red);
  if (csize > 1) total = cluster_sum(total, &cl_slot, csize);
  const float r = Op::rstd(a, total);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = first + k * tpr;
    if (v < nvec) Op::finish(a, row, v, h[0][k], r);
  }
  if (first == 0) Op::row_stats(a, row, r);
  if (csize > 1) cluster_sync();  // peers may still read cl_slot
}

// Rows longer than a cluster can hold: one CTA per row walks it twice.  The
// first pass forms S (and stores it), the second re-forms it from the inputs
// (re-reads are served by L2 for any row that fits there).
template <class Op>
__global__ void __launch_bounds__(kRowsMaxThreads)
rows_walk_kernel(const typename Op::Args a, int nvec) {
  __shared__ float red[33];
  const int64_t row = blockIdx.x;
  float acc = 0.0f;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    typename Op::In in;
    typename Op::Hold h;
    Op::load(a, row, v, in);
    acc += Op::combine(a, row, v, in, h);
  }
  const float r = Op::rstd(a, cta_sum(acc, red));
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    typename Op::In in;
    typename Op::Hold h;
    Op::load(a, row, v, in);
    Op::template combine<false>(a, row, v, in, h);
    Op::finish(a, row, v, h, r);
  }
  if (threadIdx.x == 0) Op::row_stats(a, row, r);
}

}  // namespace b200norm
