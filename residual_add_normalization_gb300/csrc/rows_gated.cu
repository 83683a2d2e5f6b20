// GatedRMSNorm row kernels (float32 and float16), the row planner, and the
// element-type switches of both row operators.
#include "rows_ops.cuh"

#ifndef B200NORM_SHORT_RPG
#define B200NORM_SHORT_RPG 1   // rows per lane group for spans of <= 32 vectors
#endif
#ifndef B200NORM_SHORT_NV
#define B200NORM_SHORT_NV 1    // vectors per thread for spans of <= 32 vectors
#endif
// CTA-per-row schedules.  Measured on GB300 (fp16 / fp32 rows of 4096 and
// 8192 elements, CUDA-graph replay): with up to kFewRows rows the call is
// latency-bound and the widest CTA (fewest vectors per thread, up to 512
// threads) is fastest -- 1.7 us instead of 2.8 us for one fp16 row of 4096;
// with more rows CTAs of about 256 threads are (nv capped at 4; rows of more
// than 1024 vectors take 512 threads).  Splitting a row over a cluster only
// pays once one CTA cannot hold it.
constexpr int64_t kFewRows = 256;
// Past kFewRows rows (measured on GB300 over widths of 512-16384 elements,
// rows enough for two 512 MB buffer sets, CUDA-graph replay):
//  - SkipSimplifiedLayerNormalization rows of 97-159 vectors go to one CTA
//    per row rather than a warp per row: a warp holding four vectors of two
//    inputs per lane runs at 125 registers, two 256-thread CTAs per SM, too
//    few warps to hide its epilogue (hidden 1024 fp16: 77.2 us vs 87.7; 896:
//    78.5 vs 83.0; at 96 vectors and fewer the warp stays ahead, 84.4 vs
//    89.6 at 768);
//  - a CTA row that is not a whole number of warps takes two vectors per
//    thread (hidden 896: 78.5 vs 81.2 us; 1152: 77.9 vs 81.7);
//  - GatedRMSNorm CTA rows take at least two vectors per thread (C = 1536 /
//    2048 fp16: 78.2 / 78.2 us vs 87.9 / 87.1 with one; bf16 C = 2048 78.5 vs
//    87.8; float32 C = 1024 76.5 vs 77.3); its rows of up to 128 vectors
//    stay on a warp each (C = 1024 fp16: 86.1 us vs 90.1 for a CTA).
constexpr int kSslnCtaFromVec = 97;
constexpr int kSslnPairBelowVec = 160;

namespace b200norm {

static int pow2_ceil(int64_t v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

static int round32(int64_t v) { return static_cast<int>(ceil_div(v, 32) * 32); }

RowPlan plan_rows(int64_t rows, int64_t n, DType t, bool vector_ok, RowOp op) {
  RowPlan p = {};
  p.ve = vector_ok ? static_cast<int>(16 / dtype_size(t)) : 1;
  const int64_t nvec = n / p.ve;
  p.csize = 1;
  p.rpg = 1;
  if (nvec <= 32) {
    // Short spans: a power-of-two lane group per row, several rows per warp.
    p.mode = 0;
    p.nv = nvec >= B200NORM_SHORT_NV ? B200NORM_SHORT_NV : 1;
    p.tpr = pow2_ceil(ceil_div(nvec, p.nv));
    p.rpg = p.nv == 1 && p.tpr <= 16 ? B200NORM_SHORT_RPG : 1;
    p.block = lane_block(p.nv * p.rpg);
    p.grid = ceil_div(rows, static_cast<int64_t>(p.block / p.tpr) * p.rpg);
  } else if (nvec <= 128 &&
             !(op == RowOp::SkipRms && rows > kFewRows && nvec >= kSslnCtaFromVec)) {
    // Warp per row, up to four vectors per lane.
    p.mode = 0;
    p.tpr = 32;
    p.nv = pow2_ceil(ceil_div(nvec, 32));
    p.block = lane_block(p.nv);
    p.grid = ceil_div(rows, p.block / 32);
  } else {
    // CTA per row; a cluster per row once one CTA cannot hold it.
    p.mode = 1;
    const bool many = rows > kFewRows;
    int nv = 1;
    if (many && op == RowOp::Gated) nv = 2;
    if (many && op == RowOp::SkipRms && nvec < kSslnPairBelowVec && nvec % 32 != 0) nv = 2;
    int cta = round32(ceil_div(nvec, nv));
    const int target = many ? 256 : kRowsMaxThreads;
    while (cta > target && nv < 4) {
      nv *= 2;
      cta = round32(ceil_div(nvec, nv));
    }
    while (cta > kRowsMaxThreads && nv < 8) {
      nv *= 2;
      cta = round32(ceil_div(nvec, nv));
    }
    int csize = 1;
    if (cta > kRowsMaxThreads) {
      csize = static_cast<int>(ceil_div(nvec, static_cast<int64_t>(nv) * kRowsMaxThreads));
      cta = round32(ceil_div(nvec, static_cast<int64_t>(nv) * csize));
    }
    if (csize > 16) {
      p.mode = 2;
      p.tpr = kRowsMaxThreads;
      p.block = kRowsMaxThreads;
      p.nv = 1;
      p.grid = rows;
      return p;
    }
    p.nv = nv;
    p.csize = csize;
    p.block = cta;
    p.tpr = cta * csize;
    p.grid = rows * csize;
  }
  return p;
}

bool pipe_plan(int64_t rows, int64_t n, DType t, bool vector_ok, RowPlan* p) {
  const int ve = static_cast<int>(16 / dtype_size(t));
  if (!vector_ok || n % ve != 0 || n / ve > 32 || rows <= 0) return false;
  *p = RowPlan{};
  p->mode = 3;
  p->ve = ve;
  p->tpr = pow2_ceil(n / ve);
  p->nv = 1;
  p->rpg = 1;
  p->block = kPipeThreads;
  p->csize = 1;
  p->grid = ceil_div(rows, static_cast<int64_t>(kPipeWarps) * (32 / p->tpr));  // tiles
  return true;
}

bool prefer_pipe_skip_rms(int64_t rows, int64_t n, DType t, bool vector_ok, RowPlan* p) {
  RowPlan q;
  if (!pipe_plan(rows, n, t, vector_ok, &q) ||
      q.grid < (t == DType::F16 ? kPipeMinTilesF16 : kPipeMinTiles))
    return false;
  *p = q;
  return true;
}

// The pipelined schedule's status word (one per device) and testing stall.
__device__ unsigned g_pipe_status;
static std::atomic<bool> g_pipe_stall{false};
static std::atomic<unsigned long long> g_pipe_stall_limit_ns{kPipeLimitNs};

unsigned* pipe_status_word() {
  constexpr int kCachedDevices = 64;  // devices past these are looked up every time
  static std::atomic<unsigned*> cache[kCachedDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return nullptr;
  }
  unsigned* p = dev < kCachedDevices ? cache[dev].load() : nullptr;
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_pipe_status) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  p = static_cast<unsigned*>(addr);
  if (dev < kCachedDevices) cache[dev].store(p);
  return p;
}

bool pipe_stalled() { return g_pipe_stall.load(); }
unsigned long long pipe_stall_limit_ns() { return g_pipe_stall_limit_ns.load(); }
void set_pipe_stall(bool on, unsigned long long limit_ns) {
  g_pipe_stall_limit_ns.store(limit_ns);
  g_pipe_stall.store(on);
}

cudaError_t launch_skip_rms(const SkipRmsCall& c, const RowPlan& p, cudaStream_t st) {
  switch (c.t) {
    case DType::F32: return skip_rms_f32(c, p, st);
    case DType::F16: return skip_rms_f16(c, p, st);
    case DType::BF16: return skip_rms_bf16(c, p, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gated(const GatedCall& c, const RowPlan& p, cudaStream_t st) {
  switch (c.t) {
    case DType::F32:
      return p.ve == 4 ? gated_go<float, 4>(c, p, st) : gated_go<float, 1>(c, p, st);
    case DType::F16:
      return p.ve == 8 ? gated_go<__half, 8>(c, p, st) : gated_go<__half, 1>(c, p, st);
    case DType::BF16: return gated_bf16(c, p, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace b200norm
