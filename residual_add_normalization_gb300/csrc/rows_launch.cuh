// rows_launch.cuh -- host-side launch of the row kernels for one Op policy.
#pragma once

#include <atomic>

#include "launch.h"
#include "rows.cuh"
#include "rows_pipe.cuh"

namespace b200norm {

template <class Op>
using RowsKernelFn = void (*)(const typename Op::Args, int, int);

// CTAs of `block` threads of kernel `fn` that the current device holds at
// once (cached per device and kernel).
inline cudaError_t resident_ctas(const void* fn, int block, int64_t* out) {
  struct Key {
    int dev, block;
    const void* fn;
  };
  static PlanCache<Key, int64_t> cache;
  Key k;
  memset(&k, 0, sizeof(k));
  cudaError_t e = cudaGetDevice(&k.dev);
  if (e != cudaSuccess) return e;
  k.block = block;
  k.fn = fn;
  if (cache.get(k, out)) return cudaSuccess;
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, k.dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, block, 0);
  if (e != cudaSuccess) return e;
  *out = static_cast<int64_t>(per_sm > 0 ? per_sm : 1) * sms;
  cache.put(k, *out);
  return cudaSuccess;
}

// Lane-group instantiations: (NV, RPG) in {(1,1), (1,2), (1,4), (2,1), (4,1)}.
template <class Op>
RowsKernelFn<Op> pick_lane_kernel(int nv, int rpg) {
  if (nv == 1) {
    switch (rpg) {
      case 1: return rows_lane_kernel<Op, 1, 1>;
      case 2: return rows_lane_kernel<Op, 1, 2>;
      case 4: return rows_lane_kernel<Op, 1, 4>;
      default: return nullptr;
    }
  }
  if (rpg != 1) return nullptr;
  switch (nv) {
    case 2: return rows_lane_kernel<Op, 2, 1>;
    case 4: return rows_lane_kernel<Op, 4, 1>;
    default: return nullptr;
  }
}

// CTA / cluster instantiations: NV in {1, 2, 4, 8}.
template <class Op>
RowsKernelFn<Op> pick_cta_kernel(int nv) {
  switch (nv) {
    case 1: return rows_cta_kernel<Op, 1>;
    case 2: return rows_cta_kernel<Op, 2>;
    case 4: return rows_cta_kernel<Op, 4>;
    case 8: return rows_cta_kernel<Op, 8>;
    default: return nullptr;
  }
}

// The pipelined schedule: one CTA per SM, at most one per tile.
template <class Op>
cudaError_t launch_pipe(const typename Op::Args& a, const RowPlan& p, int nvec,
                        cudaStream_t stream) {
  void (*fn)(const typename Op::Args, int, int, unsigned long long, unsigned*, int) =
      rows_pipe_kernel<Op>;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // the ring is larger than the default dynamic shared-memory limit: raise
  // it once per device (every time on devices past the first 64)
  static std::atomic<unsigned long long> raised{0};
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (!bit || !(raised.load() & bit)) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPipeSmemBytes));
    if (e != cudaSuccess) return e;
    raised.fetch_or(bit);
  }
  unsigned* status = pipe_status_word();
  if (!status) return cudaErrorSymbolNotFound;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.stream = stream;
  const int64_t resident = static_cast<int64_t>(sms) * kPipeMinBlocks;
  cfg.gridDim = dim3(static_cast<unsigned>(p.grid < resident ? p.grid : resident));
  cfg.blockDim = dim3(kPipeThreads);
  cfg.dynamicSmemBytes = kPipeSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = add_pdl_attr(attr, 0);
  const bool stall = pipe_stalled();
  return cudaLaunchKernelEx(&cfg, fn, a, p.tpr, nvec, stall ? pipe_stall_limit_ns() : kPipeLimitNs,
                            status, stall ? 1 : 0);
}

template <class Op>
cudaError_t launch_rows_op(const typename Op::Args& a, const RowPlan& p, cudaStream_t stream) {
  const int nvec = static_cast<int>(a.n / p.ve);
  if (p.mode == 3) {
    if constexpr (sizeof(typename Op::P) == 16) return launch_pipe<Op>(a, p, nvec, stream);
    return cudaErrorInvalidConfiguration;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.stream = stream;
  if (p.mode == 2) {
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.blockDim = dim3(p.block);
    cfg.attrs = attr;
    cfg.numAttrs = add_pdl_attr(attr, 0);
    return cudaLaunchKernelEx(&cfg, rows_walk_kernel<Op>, a, nvec);
  }
  RowsKernelFn<Op> fn = p.mode == 0 ? pick_lane_kernel<Op>(p.nv, p.rpg) : pick_cta_kernel<Op>(p.nv);
  if (!fn) return cudaErrorInvalidConfiguration;
  int64_t grid = p.grid;
  if (p.mode == 0) {
    // persistent lane-group schedule: as many CTAs as can be resident
    int64_t resident = 0;
    cudaError_t e = resident_ctas(reinterpret_cast<const void*>(fn), p.block, &resident);
    if (e != cudaSuccess) return e;
    if (grid > resident) grid = resident;
  }
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(p.block);
  cfg.dynamicSmemBytes = 0;
  unsigned nattr = 0;
  if (p.mode == 1 && p.csize > 1) {
    if (p.csize > 8) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    nattr = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = add_pdl_attr(attr, nattr);
  return cudaLaunchKernelEx(&cfg, fn, a, p.tpr, nvec);
}

template <class Op>
bool cluster_fits_query(RowsKernelFn<Op> fn, int block, int csize) {
  if (csize > 8 &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize);
  cfg.blockDim = dim3(block);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return clusters > 0;
}

// Can a cluster of `csize` CTAs of `block` threads of this kernel be resident?
// (cached per device and configuration)
template <class Op>
bool cluster_fits(int nv, int block, int csize) {
  RowsKernelFn<Op> fn = pick_cta_kernel<Op>(nv);
  if (!fn) return false;
  struct Key {
    int dev, block, csize;
    const void* fn;
  };
  static PlanCache<Key, bool> cache;
  Key k;
  memset(&k, 0, sizeof(k));
  if (cudaGetDevice(&k.dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  k.block = block;
  k.csize = csize;
  k.fn = reinterpret_cast<const void*>(fn);
  bool fits = false;
  if (cache.get(k, &fits)) return fits;
  fits = cluster_fits_query<Op>(fn, block, csize);
  cache.put(k, fits);
  return fits;
}


}  // namespace b200norm
