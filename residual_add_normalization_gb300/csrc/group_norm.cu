// group_norm.cu -- SkipGroupNorm planning and dispatch (host side), and the
// grid-barrier timeout probe.  The kernels are in group_kernels.cuh,
// instantiated per element type in group_f32.cu / group_f16.cu /
// group_bf16.cu.
#include <algorithm>

#include "group_kernels.cuh"

namespace b200norm {

// ---------------------------------------------------------------------------
// Test hook: a barrier that can never complete (expects one CTA more than
// the grid has).  Every CTA gives up after limit_ns and records a timeout.
// ---------------------------------------------------------------------------
__global__ void barrier_timeout_probe(Control* ctl, unsigned long long limit_ns) {
  unsigned departure = 0u;
  grid_arrive(ctl);
  grid_wait(ctl, gridDim.x + 1, limit_ns, 99u, departure);
  grid_depart(ctl, departure);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Does route 4 take vectors of `ve` elements here?  (batch items the control
// block counts, channels per CTA row, shared-memory tables, and what the
// second kernel re-reads through L2: `in_bytes`.)
static bool l2_route_ok(int64_t N, int64_t C, int ve, int64_t in_bytes) {
  return N <= kL2MaxItems && C % ve == 0 && C <= 1024 && C / ve <= kL2MaxThreads &&
         in_bytes <= kL2RouteMaxBytes;
}

size_t group_workspace_bytes(int64_t N, int64_t C, int64_t H, int64_t W, int groups, DType t,
                             bool channels_last) {
  if (N <= 0 || C <= 0 || H <= 0 || W <= 0 || groups <= 0) return kControlBytes;
  const int64_t L = (C / groups) * H * W;
  // route 3 (either layout): one piece per chunk of every group instance;
  // route 1 (NCHW) needs no slots
  int64_t slots = N * groups * cdiv(L, kTwoPhaseChunk);
  if (channels_last) {
    // routes 2 and 5: one piece per CTA and group, at most kMaxCoopCtas CTAs
    slots = std::max<int64_t>(slots, static_cast<int64_t>(kMaxCoopCtas) * groups);
    const int64_t es = static_cast<int64_t>(dtype_size(t));
    for (int ve : {1, static_cast<int>(16 / es)}) {
      // route 4: the pieces, then the statistics of every instance
      if (l2_route_ok(N, C, ve, N * H * W * C * es)) {
        const int64_t r4 = static_cast<int64_t>(kMaxCoopCtas) * groups + N * groups;
        if (r4 > slots) slots = r4;
      }
    }
  }
  return kControlBytes + static_cast<size_t>(slots) * sizeof(float4);
}

static void* pick_coop_any(DType t, DType m, int ve, int nv) {
  switch (t) {
    case DType::F32: return group_coop_kernel_f32(m, ve, nv);
    case DType::F16: return group_coop_kernel_f16(m, ve, nv);
    case DType::BF16: return group_coop_kernel_bf16(m, ve, nv);
  }
  return nullptr;
}

static void* pick_resident_any(DType t, DType m, int ve) {
  switch (t) {
    case DType::F32: return group_resident_kernel_f32(m, ve);
    case DType::F16: return group_resident_kernel_f16(m, ve);
    case DType::BF16: return group_resident_kernel_bf16(m, ve);
  }
  return nullptr;
}

static void* pick_coop_l2_any(DType t, DType m, int ve, bool bcast) {
  switch (t) {
    case DType::F32: return group_coop_l2_kernel_f32(m, ve, bcast);
    case DType::F16: return group_coop_l2_kernel_f16(m, ve, bcast);
    case DType::BF16: return group_coop_l2_kernel_bf16(m, ve, bcast);
  }
  return nullptr;
}

static void* pick_slab_any(DType t, DType m, int ve) {
  switch (t) {
    case DType::F32: return group_slab_kernel_f32(m, ve);
    case DType::F16: return group_slab_kernel_f16(m, ve);
    case DType::BF16: return group_slab_kernel_bf16(m, ve);
  }
  return nullptr;
}

static bool resident_cluster_fits(void* fn, int block, int csize, size_t smem) {
  if (csize > 8 &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
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

// Can kernel `fn` take `smem` bytes of dynamic shared memory on device `dev`?
// The kernel's limit is raised to everything the device allows next to its
// static shared memory (never lowered), so that plans cached for this kernel
// with different sizes all stay launchable.
static bool allow_smem(void* fn, size_t smem, int dev) {
  cudaFuncAttributes fa;
  int optin = 0;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const size_t cap = static_cast<size_t>(optin) - fa.sharedSizeBytes;
  if (smem > cap) return false;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(cap)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

// Dynamic shared memory of route 2: the phase area up to coop_k_offset, then
// R[groups] and the second-round R[groups] (padded to 16 bytes), gamma[C]
// and beta[C]; for route 6 (`slab` > 0) then its slab area (coop_slab_bytes).
static size_t coop_smem_bytes(int PL, int C, int B, int groups, size_t slab = 0) {
  return (coop_k_offset(PL, C, B, groups) + coop_tail_floats(groups) + 2ull * C) * sizeof(float) +
         slab;
}

GroupPlan two_phase_plan(const SkipGroupCall& c) {
  const int64_t L = (c.C / c.groups) * c.H * c.W;
  GroupPlan p = {};
  p.route = 3;
  p.ve = 1;
  p.nv = kTwoPhaseEpt;
  p.block = kTwoPhaseThreads;
  p.csize = 1;
  p.chunks = static_cast<int>(cdiv(L, kTwoPhaseChunk));
  p.grid = c.N * c.groups * p.chunks;
  p.smem = 0;
  return p;
}

// Route 4 for an NHWC call, if it applies (the tensors it re-reads stay in
// L2 between its two kernels).
static bool plan_l2_route(const SkipGroupCall& c, bool vector_ok, GroupPlan* p) {
  if (!c.channels_last) return false;
  const int64_t es = static_cast<int64_t>(dtype_size(c.t));
  const int vec = static_cast<int>(16 / es);
  const int ve = (vector_ok && c.C % vec == 0) ? vec : 1;
  const int64_t numel = c.N * c.H * c.W * c.C;
  if (!l2_route_ok(c.N, c.C, ve, numel * es * (c.bcast ? 1 : 2))) return false;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  // about two CTAs per SM over the whole grid, each walking its pixel range
  const int64_t HW = c.H * c.W;
  const int PL = static_cast<int>(kL2MaxThreads / (c.C / ve));
  const int64_t target = std::min<int64_t>(2LL * sms, kMaxCoopCtas);
  int64_t B = std::min<int64_t>(cdiv(HW, PL), std::max<int64_t>(1, target / c.N));
  const int64_t ppc = cdiv(HW, B);
  B = cdiv(HW, ppc);
  *p = GroupPlan{};
  p->route = 4;
  p->ve = ve;
  p->nv = kL2Passes;
  p->block = static_cast<int>(PL * (c.C / ve));
  p->csize = 1;
  p->grid = c.N * B;
  p->ctas_per_item = static_cast<int>(B);
  p->pix_per_cta = static_cast<int>(ppc);
  p->smem = static_cast<size_t>(c.C) * sizeof(float4);
  return true;
}

// Route 5: route 4's passes in one cooperative grid.  Same shape limits as
// route 4 except the batch-item count (it keeps no per-item counters): every
// CTA must be resident at once, at most kMaxCoopCtas of them.
static bool plan_coop_l2_route(const SkipGroupCall& c, bool vector_ok, GroupPlan* p) {
  if (!c.channels_last) return false;
  const int64_t es = static_cast<int64_t>(dtype_size(c.t));
  const int vec = static_cast<int>(16 / es);
  const int ve = (vector_ok && c.C % vec == 0) ? vec : 1;
  const int64_t numel = c.N * c.H * c.W * c.C;
  if (!l2_route_ok(1, c.C, ve, numel * es * (c.bcast ? 1 : 2))) return false;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  void* fn = pick_coop_l2_any(c.t, c.m, ve, c.bcast);
  const int64_t HW = c.H * c.W;
  const int PL = static_cast<int>(kL2MaxThreads / (c.C / ve));
  const int block = static_cast<int>(PL * (c.C / ve));
  const size_t smem = static_cast<size_t>(c.C) * sizeof(float4) +
                      static_cast<size_t>(2 * c.groups) * sizeof(float);
  int per_sm = 0;
  if (!fn || !allow_smem(fn, smem, dev) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, block, smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const int64_t cap = std::min<int64_t>(static_cast<int64_t>(per_sm) * sms, kMaxCoopCtas);
  if (c.N > cap) return false;
  int64_t B = std::min<int64_t>(cdiv(HW, PL), cap / c.N);
  const int64_t ppc = cdiv(HW, B);
  B = cdiv(HW, ppc);
  *p = GroupPlan{};
  p->route = 5;
  p->ve = ve;
  p->nv = kL2Passes;
  p->block = block;
  p->csize = 1;
  p->grid = c.N * B;
  p->ctas_per_item = static_cast<int>(B);
  p->pix_per_cta = static_cast<int>(ppc);
  p->smem = smem;
  return true;
}

// Route 6: route 2 with the slab resident in shared memory.  One CTA per SM
// share of the batch items (at least one CTA per item), as long as the slab
// of X (and of a full-shape skip) fits next to route 2's other shared memory
// and every CTA can be resident at once.
static bool plan_slab_route(const SkipGroupCall& c, bool vector_ok, GroupPlan* p) {
  if (!c.channels_last) return false;
  const int64_t es = static_cast<int64_t>(dtype_size(c.t));
  const int vec = static_cast<int>(16 / es);
  const int ve = (vector_ok && c.C % vec == 0) ? vec : 1;
  const int64_t CV = c.C / ve;
  const int64_t HW = c.H * c.W;
  if (CV > kCoopMaxThreads || HW > 0x7fffffffLL) return false;
  int dev = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  void* fn = pick_slab_any(c.t, c.m, ve);
  cudaFuncAttributes fa;
  if (!fn || cudaFuncGetAttributes(&fa, fn) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const size_t cap = static_cast<size_t>(optin) - fa.sharedSizeBytes;
  const int PL = static_cast<int>(kCoopMaxThreads / CV);
  const int block = static_cast<int>(PL * CV);
  int64_t B = std::max<int64_t>(1, sms / c.N);
  const int64_t ppc = cdiv(HW, B);
  B = cdiv(HW, ppc);
  if (B * c.N > kMaxCoopCtas || ppc * c.C > 0x7fffffffLL) return false;
  const size_t slab = coop_slab_bytes(static_cast<int>(ppc), static_cast<int>(c.C), es, c.bcast);
  const size_t smem = coop_smem_bytes(PL, static_cast<int>(c.C), static_cast<int>(B), c.groups, slab);
  int per_sm = 0;
  if (smem > cap || !allow_smem(fn, smem, dev) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, block, smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (static_cast<int64_t>(per_sm) * sms < B * c.N) return false;
  *p = GroupPlan{};
  p->route = 6;
  p->ve = ve;
  p->nv = static_cast<int>(cdiv(ppc, PL));
  p->block = block;
  p->csize = 1;
  p->grid = B * c.N;
  p->ctas_per_item = static_cast<int>(B);
  p->pix_per_cta = static_cast<int>(ppc);
  p->smem = smem;
  return true;
}

static cudaError_t plan_group_uncached(const SkipGroupCall& c, bool vector_ok, int force,
                                       GroupPlan* p);


#ifndef B200NORM_NCHW_TARGET_KB
#define B200NORM_NCHW_TARGET_KB 40  // S staged per CTA in route 1
#endif

// Plans depend on the device, the shape, the types, the alignment and a
// forced route only; the occupancy queries behind them are costly, so they
// are cached.
struct GroupPlanKey {
  int dev;
  int64_t N, C, H, W;
  int groups, t, m, cl, vec, bcast, force;
};

cudaError_t plan_group(const SkipGroupCall& c, bool vector_ok, int force_route, GroupPlan* p) {
  static PlanCache<GroupPlanKey, GroupPlan> cache;
  GroupPlanKey k;
  memset(&k, 0, sizeof(k));
  cudaError_t e = cudaGetDevice(&k.dev);
  if (e != cudaSuccess) return e;
  k.N = c.N;
  k.C = c.C;
  k.H = c.H;
  k.W = c.W;
  k.groups = c.groups;
  k.t = static_cast<int>(c.t);
  k.m = static_cast<int>(c.m);
  k.cl = c.channels_last ? 1 : 0;
  k.vec = vector_ok ? 1 : 0;
  k.bcast = c.bcast ? 1 : 0;
  k.force = force_route;
  if (cache.get(k, p)) return cudaSuccess;
  e = plan_group_uncached(c, vector_ok, force_route, p);
  if (e == cudaSuccess) cache.put(k, *p);
  return e;
}

static cudaError_t plan_group_uncached(const SkipGroupCall& c, bool vector_ok, int force,
                                       GroupPlan* p) {
  *p = GroupPlan{};
  if (force == 3) {
    *p = two_phase_plan(c);
    return cudaSuccess;
  }
  if (force == 4) return plan_l2_route(c, vector_ok, p) ? cudaSuccess : cudaErrorNotSupported;
  if (force == 5) return plan_coop_l2_route(c, vector_ok, p) ? cudaSuccess : cudaErrorNotSupported;
  if (force == 6) return plan_slab_route(c, vector_ok, p) ? cudaSuccess : cudaErrorNotSupported;
  if (force == 0 && c.channels_last) {
    // NHWC: the cooperative route whenever its grid can hold the pixels in
    // registers, else the cooperative route with the slabs in shared memory,
    // else one cooperative grid re-reading through L2, else the two-kernel
    // L2 route, else two-phase.  (Measured on GB300, graph-timed with the
    // inputs in HBM: (2, 64, 64, 320) fp16 9.9 us in registers vs 10.6 in
    // shared memory and 13.3 / 13.5 through L2 in one grid / two kernels;
    // slabs in shared memory
    // against one grid through L2: (4, 64, 64, 320) fp16 13.7 vs 16.5 us,
    // (2, 64, 64, 640) fp16 14.2 vs 18.3, (2, 64, 64, 320) fp32 11.3 vs
    // 14.8, (8, 64, 64, 320) fp16 20.4 vs 22.8.)
    if (plan_group_uncached(c, vector_ok, 2, p) == cudaSuccess) return cudaSuccess;
    if (plan_slab_route(c, vector_ok, p)) return cudaSuccess;
    if (plan_coop_l2_route(c, vector_ok, p)) return cudaSuccess;
    if (plan_l2_route(c, vector_ok, p)) return cudaSuccess;
    *p = two_phase_plan(c);
    return cudaSuccess;
  }
  if (force == 2 && !c.channels_last) return cudaErrorNotSupported;
  const int64_t HW = c.H * c.W;
  const int64_t cpg = c.C / c.groups;
  const int64_t L = cpg * HW;
  const int vec_elems = static_cast<int>(16 / dtype_size(c.t));
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;

  if (!c.channels_last) {
    // Route 1: each CTA stages at most ~40 KB of S in shared memory (five
    // such CTAs fit an SM), so an instance takes ceil(bytes / 40 KB) CTAs of
    // a cluster (at most 16); small instances under-filling the GPU are split
    // further while each CTA keeps at least two vectors per thread, or one
    // while the cluster stays at most 4 and the grid within 2 x SMs.
    // (Measured on GB300, fp16, SiLU, inputs from HBM: (2, 1280, 16, 16)
    // 4.72 us with clusters of 4 vs 5.30 with 2; (1, 1280, 16, 16) 4.23 vs
    // 5.07; (2, 320, 32, 32) 4.72 vs 5.29; but (2, 640, 32, 32) 6.84 with 8
    // vs 6.15 with 4, and (4, 1280, 16, 16) 6.59 with 512 CTAs vs 6.08.)
    const int ve = (vector_ok && HW % vec_elems == 0) ? vec_elems : 1;
    const int64_t nvec = L / ve;
    const int64_t vbytes = static_cast<int64_t>(ve) * static_cast<int64_t>(dtype_size(c.t));
    const int64_t insts = c.N * c.groups;
    const int64_t target = B200NORM_NCHW_TARGET_KB * 1024;
    int64_t cs = cdiv(nvec * vbytes, target);
    while (cs < 16 && insts * cs < 2LL * sms &&
           (cdiv(nvec, cs * 2) >= 2LL * kNchwThreads ||
            (cs < 4 && insts * cs * 2 <= 2LL * sms && cdiv(nvec, cs * 2) >= kNchwThreads)))
      cs *= 2;
    if (cs > 16 || L > 0x7fffffffLL) {
      *p = two_phase_plan(c);
      return cudaSuccess;
    }
    const int span = static_cast<int>(cdiv(nvec, cs));
    // S, then gamma / beta of the channels a CTA touches (a run of `span`
    // vectors covers at most span / (H*W / ve) + 2 channels)
    const size_t smem = nchw_gb_offset(span, static_cast<size_t>(vbytes)) +
                        static_cast<size_t>(span / (HW / ve) + 2) * sizeof(float2);
    void* fn = pick_resident_any(c.t, c.m, ve);
    if (fn && allow_smem(fn, smem, dev) &&
        (cs == 1 || resident_cluster_fits(fn, kNchwThreads, static_cast<int>(cs), smem)) &&
        insts * cs <= 0x7fffffffLL) {
      p->route = 1;
      p->ve = ve;
      p->nv = span;  // vectors per CTA
      p->block = kNchwThreads;
      p->csize = static_cast<int>(cs);
      p->grid = insts * cs;
      p->smem = smem;
      return cudaSuccess;
    }
    *p = two_phase_plan(c);
    return cudaSuccess;
  }

  // Route 2: NHWC cooperative.  Every CTA must be resident at once, so the
  // grid is at most (CTAs per SM) x (SMs); each CTA's pixel slab must fit in
  // its threads' registers (nv vectors per thread).
  const int ve = (vector_ok && c.C % vec_elems == 0) ? vec_elems : 1;
  const int64_t CV = c.C / ve;
  if (CV <= kCoopMaxThreads && HW <= 0x7fffffffLL) {
    const int PL = static_cast<int>(kCoopMaxThreads / CV);
    const int block = static_cast<int>(PL * CV);
    const size_t smem1 = coop_smem_bytes(PL, static_cast<int>(c.C), 0, c.groups);
    for (int nv : {1, 2, 3, 4, 5, 6, 8}) {
      void* fn = pick_coop_any(c.t, c.m, ve, nv);
      if (!fn) continue;
      // dynamic + static shared memory must fit the per-block opt-in limit
      cudaFuncAttributes fa;
      int optin = 0;
      if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess ||
          cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
              cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      const size_t smem_cap = static_cast<size_t>(optin) - fa.sharedSizeBytes;
      if (smem1 > smem_cap ||
          cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_cap)) != cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, block, smem1) != cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      int64_t cap = static_cast<int64_t>(per_sm) * sms;
      if (cap > kMaxCoopCtas) cap = kMaxCoopCtas;
      const int64_t B = cap / c.N;
      if (B < 1) break;  // more batch items than resident CTAs
      const int64_t ppc = cdiv(HW, B);
      if (ppc > static_cast<int64_t>(nv) * PL) continue;  // slab too big for nv
      const int64_t Bn = cdiv(HW, ppc);  // CTAs actually needed per item
      const size_t smem = coop_smem_bytes(PL, static_cast<int>(c.C), static_cast<int>(Bn), c.groups);
      if (smem > smem_cap) continue;
      if (smem > smem1) {
        int again = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&again, fn, block, smem) != cudaSuccess) {
          cudaGetLastError();
          continue;
        }
        if (static_cast<int64_t>(again) * sms < Bn * c.N) continue;
      }
      p->route = 2;
      p->ve = ve;
      p->nv = nv;
      p->block = block;
      p->csize = 1;
      p->ctas_per_item = static_cast<int>(Bn);
      p->pix_per_cta = static_cast<int>(ppc);
      p->grid = Bn * c.N;
      p->smem = smem;
      return cudaSuccess;
    }
  }
  if (force == 2) return cudaErrorNotSupported;
  *p = two_phase_plan(c);
  return cudaSuccess;
}

cudaError_t launch_group(const SkipGroupCall& c, const GroupPlan& p, cudaStream_t stream) {
  switch (c.t) {
    case DType::F32: return launch_group_f32(c, p, stream);
    case DType::F16: return launch_group_f16(c, p, stream);
    case DType::BF16: return launch_group_bf16(c, p, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_barrier_timeout_probe(void* workspace, unsigned long long limit_ns,
                                         cudaStream_t stream) {
  Control* ctl = static_cast<Control*>(workspace);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, barrier_timeout_probe, ctl, limit_ns);
}

}  // namespace b200norm
