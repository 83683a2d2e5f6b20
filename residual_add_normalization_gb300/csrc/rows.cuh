// rows.cuh -- row-normalization kernels shared by SkipSimplifiedLayerNormalization
// and GatedRMSNorm (sm_103a).
//
// A "row" is one normalization span: the hidden axis of SSLN, or one C-span of
// GatedRMSNorm.  Each row is read once from HBM with 16-byte vector loads, kept
// in registers while its sum of squares is reduced, then normalized and
// written.  Three schedules:
//
//   rows_lane_kernel         lane groups of `tpr` <= 32 threads (a power of two)
//                            per row, several rows per warp, RPG rows per lane
//                            group in flight, persistent grid; the reduction is
//                            a segmented butterfly over the low lane bits (no
//                            shared memory, no barrier).
//   rows_cta_kernel          one row per CTA, or per thread-block cluster for
//                            long rows: warp butterflies, a shared-memory
//                            combine, then a DSMEM combine across the cluster.
//   rows_walk_kernel         rows longer than a cluster holds: one CTA walks
//                            the row twice (the second pass is served by L2).
//
// Op policies (SkipRmsOp, GatedOp) supply the per-vector load / combine /
// finish steps; the schedule code is shared.  rows_pipe.cuh adds a fourth
// schedule for short spans that streams both inputs through shared memory.
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
  float inv_n;                 // 1 / hidden
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
  float inv_n;                 // 1 / C
  float eps;
};

// 1 / sqrt(mean square + eps) from a row's sum of squares.
__device__ __forceinline__ float row_rstd(float sumsq, float inv_n, float eps) {
  return rsqrtf(fmaf(sumsq, inv_n, eps));
}

// ---------------------------------------------------------------------------
// SkipSimplifiedLayerNormalization
//   S = round_T((x + skip) + bias); y = round_T(S * rstd * gamma),
//   rstd = 1 / sqrt(sum(S^2) / n + eps)
// Per-vector weights (gamma, bias) are loaded once per thread and reused for
// every row the thread handles.
// ---------------------------------------------------------------------------
template <typename T, int VE, bool HAS_BIAS, bool WANT_S>
struct SkipRmsOp {
  using Args = SkipRmsArgs<T>;
  using Elem = T;
  using P = Pack<T, VE>;
  static constexpr int kVE = VE;
  struct In {
    P x, k;
  };
  struct Wt {
    P gamma, bias;
  };
  using Hold = P;

  // the two streamed inputs, for the pipelined schedule
  __device__ static __forceinline__ const T* src0(const Args& a) { return a.x; }
  __device__ static __forceinline__ const T* src1(const Args& a) { return a.skip; }
  __device__ static __forceinline__ void load_pair(const P& p0, const P& p1, In& in) {
    in.x = p0;
    in.k = p1;
  }

  __device__ static __forceinline__ void load_wt(const Args& a, int v, Wt& w) {
    w.gamma = ld_reuse<T, VE>(a.gamma + v * VE);
    if constexpr (HAS_BIAS) w.bias = ld_reuse<T, VE>(a.bias + v * VE);
  }

  __device__ static __forceinline__ void load(const Args& a, int64_t row, int v, In& in) {
    const int64_t off = row * a.n + static_cast<int64_t>(v) * VE;
    in.x = ld_stream<T, VE>(a.x + off);
    in.k = ld_stream<T, VE>(a.skip + off);
  }

  template <bool STORE_S = WANT_S>
  __device__ static __forceinline__ float combine(const Args& a, int64_t row, int v,
                                                  const In& in, const Wt& w, Hold& h) {
    float ss = 0.0f;
    if constexpr (VE % 2 == 0) {
#pragma unroll
      for (int i = 0; i < VE / 2; ++i) {
        const float2 xf = get2(in.x, i), kf = get2(in.k, i);
        float t0 = __fadd_rn(xf.x, kf.x), t1 = __fadd_rn(xf.y, kf.y);
        if constexpr (HAS_BIAS) {
          const float2 bf = get2(w.bias, i);
          t0 = __fadd_rn(t0, bf.x);
          t1 = __fadd_rn(t1, bf.y);
        }
        set2(h, i, t0, t1);  // one rounding to T
        const float2 sf = get2(h, i);
        ss = fmaf(sf.x, sf.x, ss);
        ss = fmaf(sf.y, sf.y, ss);
      }
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        h.v[e] = residual_sum<T, HAS_BIAS>(in.x.v[e], in.k.v[e], HAS_BIAS ? w.bias.v[e] : T());
        const float f = to_f32(h.v[e]);
        ss = fmaf(f, f, ss);
      }
    }
    if constexpr (STORE_S) st_stream<T, VE>(a.s + row * a.n + static_cast<int64_t>(v) * VE, h);
    return ss;
  }

  __device__ static __forceinline__ float rstd(const Args& a, float sumsq) {
    return row_rstd(sumsq, a.inv_n, a.eps);
  }

  __device__ static __forceinline__ void finish(const Args& a, int64_t row, int v,
                                                const Hold& h, const Wt& w, float r) {
    P out;
    if constexpr (VE % 2 == 0) {
#pragma unroll
      for (int i = 0; i < VE / 2; ++i) {
        const float2 sf = get2(h, i), gf = get2(w.gamma, i);
        set2(out, i, sf.x * r * gf.x, sf.y * r * gf.y);
      }
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e)
        out.v[e] = from_f32<T>(to_f32(h.v[e]) * r * to_f32(w.gamma.v[e]));
    }
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
  using Elem = T;
  using P = Pack<T, VE>;
  static constexpr int kVE = VE;
  struct In {
    P x, g;
  };
  struct Wt {
    P scale;
  };
  using Hold = In;

  // the two streamed inputs, for the pipelined schedule
  __device__ static __forceinline__ const T* src0(const Args& a) { return a.x; }
  __device__ static __forceinline__ const T* src1(const Args& a) { return a.gate; }
  __device__ static __forceinline__ void load_pair(const P& p0, const P& p1, In& in) {
    in.x = p0;
    in.g = p1;
  }

  __device__ static __forceinline__ void load_wt(const Args& a, int v, Wt& w) {
    w.scale = ld_reuse<T, VE>(a.scale + v * VE);
  }

  __device__ static __forceinline__ void load(const Args& a, int64_t row, int v, In& in) {
    const int64_t off = row * a.n + static_cast<int64_t>(v) * VE;
    in.x = ld_stream<T, VE>(a.x + off);
    in.g = ld_stream<T, VE>(a.gate + off);
  }

  template <bool STORE_S = false>
  __device__ static __forceinline__ float combine(const Args&, int64_t, int, const In& in,
                                                  const Wt&, Hold& h) {
    h = in;
    float ss = 0.0f;
    if constexpr (VE % 2 == 0) {
#pragma unroll
      for (int i = 0; i < VE / 2; ++i) {
        const float2 xf = get2(in.x, i);
        ss = fmaf(xf.x, xf.x, ss);
        ss = fmaf(xf.y, xf.y, ss);
      }
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e) ss = fmaf(to_f32(in.x.v[e]), to_f32(in.x.v[e]), ss);
    }
    return ss;
  }

  __device__ static __forceinline__ float rstd(const Args& a, float sumsq) {
    return row_rstd(sumsq, a.inv_n, a.eps);
  }

  __device__ static __forceinline__ void finish(const Args& a, int64_t row, int v,
                                                const Hold& h, const Wt& w, float r) {
    P out;
    if constexpr (VE % 2 == 0) {
#pragma unroll
      for (int i = 0; i < VE / 2; ++i) {
        const float2 xf = get2(h.x, i), gf = get2(h.g, i), sc = get2(w.scale, i);
        set2(out, i, xf.x * r * sc.x * silu_f32(gf.x), xf.y * r * sc.y * silu_f32(gf.y));
      }
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e)
        out.v[e] = from_f32<T>(to_f32(h.x.v[e]) * r * to_f32(w.scale.v[e]) *
                               silu_f32(to_f32(h.g.v[e])));
    }
    st_stream<T, VE>(a.y + row * a.n + static_cast<int64_t>(v) * VE, out);
  }

  __device__ static __forceinline__ void row_stats(const Args&, int64_t, float) {}
};

// ---------------------------------------------------------------------------
// Register-resident schedules
// ---------------------------------------------------------------------------
constexpr int kRowsMaxThreads = 512;

// Threads per CTA of the lane-group schedule, by the vectors each thread
// holds in flight (NV * RPG): 1024 with one (measured about 1% faster than
// 256 on C = 128 spans), 256 with more, so those keep their registers.
#ifndef B200NORM_LANE_BLOCK
#define B200NORM_LANE_BLOCK 1024
#endif
__host__ __device__ constexpr int lane_block(int held) {
  return held == 1 ? B200NORM_LANE_BLOCK : 256;
}
// Resident CTAs per SM the lane-group kernel is compiled for: a full SM of
// 2048 threads at one vector per thread, fewer with more vectors in flight.
__host__ __device__ constexpr int lane_min_blocks(int held) {
  return 2048 / lane_block(held) / held > 0 ? 2048 / lane_block(held) / held : 1;
}

// Lane-group schedule (tpr <= 32 threads per row, a power of two).  The grid
// is persistent: CTA b takes row blocks b, b + gridDim.x, ... of
// (blockDim.x / tpr) * RPG rows each; lane group g of the CTA takes rows
// g + i * (blockDim.x / tpr), i < RPG, of a block, so each step covers
// consecutive rows.  Per-vector weights stay in registers across blocks.
// nvec: vectors of Op::kVE elements per row, nvec <= NV * tpr.
template <class Op, int NV, int RPG>
__global__ void __launch_bounds__(lane_block(NV * RPG), lane_min_blocks(NV * RPG))
rows_lane_kernel(const typename Op::Args a, int tpr, int nvec) {
  pdl_wait();
  pdl_trigger();
  typename Op::Wt w[NV];
  const int lane = threadIdx.x & (tpr - 1);
  const int group = threadIdx.x / tpr;
  const int groups_per_cta = lane_block(NV * RPG) / tpr;
  const int64_t rows_per_block = static_cast<int64_t>(groups_per_cta) * RPG;
  const int64_t nblocks = (a.rows + rows_per_block - 1) / rows_per_block;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = lane + k * tpr;
    if (v < nvec) Op::load_wt(a, v, w[k]);
  }
  for (int64_t blk = blockIdx.x; blk < nblocks; blk += gridDim.x) {
    typename Op::In in[RPG][NV];
    typename Op::Hold h[RPG][NV];
    float part[RPG];
    const int64_t base = blk * rows_per_block + group;
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
        if (row < a.rows && v < nvec) part[i] += Op::combine(a, row, v, in[i][k], w[k], h[i][k]);
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
        if (v < nvec) Op::finish(a, row, v, h[i][k], w[k], r);
      }
      if (lane == 0) Op::row_stats(a, row, r);
    }
  }
}

// One row per CTA, or per cluster of CTAs (tpr == blockDim.x * cluster size).
// Weights are loaded where they are used (they are L1/L2 hits).
template <class Op, int NV>
__global__ void __launch_bounds__(kRowsMaxThreads)
rows_cta_kernel(const typename Op::Args a, int tpr, int nvec) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[33];
  __shared__ float cl_slot;
  typename Op::In in[NV];
  typename Op::Hold h[NV];
  const unsigned csize = cluster_size();
  const unsigned rank = csize > 1 ? cluster_rank() : 0u;
  const int64_t row = blockIdx.x / csize;
  const int first = threadIdx.x + static_cast<int>(rank) * blockDim.x;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = first + k * tpr;
    if (v < nvec) Op::load(a, row, v, in[k]);
  }
  float acc = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = first + k * tpr;
    if (v < nvec) {
      typename Op::Wt w;
      Op::load_wt(a, v, w);
      acc += Op::combine(a, row, v, in[k], w, h[k]);
    }
  }
  float total = cta_sum(acc, red);
  if (csize > 1) total = cluster_sum(total, &cl_slot, csize);
  const float r = Op::rstd(a, total);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = first + k * tpr;
    if (v < nvec) {
      typename Op::Wt w;
      Op::load_wt(a, v, w);
      Op::finish(a, row, v, h[k], w, r);
    }
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
  pdl_wait();
  pdl_trigger();
  __shared__ float red[33];
  const int64_t row = blockIdx.x;
  float acc = 0.0f;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    typename Op::In in;
    typename Op::Hold h;
    typename Op::Wt w;
    Op::load_wt(a, v, w);
    Op::load(a, row, v, in);
    acc += Op::combine(a, row, v, in, w, h);
  }
  const float r = Op::rstd(a, cta_sum(acc, red));
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    typename Op::In in;
    typename Op::Hold h;
    typename Op::Wt w;
    Op::load_wt(a, v, w);
    Op::load(a, row, v, in);
    Op::template combine<false>(a, row, v, in, w, h);
    Op::finish(a, row, v, h, w, r);
  }
  if (threadIdx.x == 0) Op::row_stats(a, row, r);
}

}  // namespace b200norm
