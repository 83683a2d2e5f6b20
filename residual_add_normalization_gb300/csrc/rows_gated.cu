// GatedRMSNorm row kernels (float32 and float16), the row planner, and the
// element-type switches of both row operators.
#include "rows_ops.cuh"

#ifndef B200NORM_SHORT_RPG
#define B200NORM_SHORT_RPG 1   // rows per lane group for spans of <= 32 vectors
#endif
#ifndef B200NORM_SHORT_NV
#define B200NORM_SHORT_NV 1    // vectors per thread for spans of <= 32 vectors
#endif
// CTA-per-row schedules, measured on GB300 (CUDA-graph replay, inputs from
// HBM; widths of 512-16384 elements, 128 rows to 512 MB per call):
//  - up to kFewRows rows the call is latency-bound and the widest CTA (fewest
//    vectors per thread, up to 512 threads) is fastest or within 2% -- 1.7 us
//    instead of 2.8 for one fp16 row of 4096; at 512 rows of 4096 GatedRMSNorm
//    4.21 us vs 4.44 with 256 threads;
//  - with more rows, CTAs of about 256 threads (nv capped at 4; rows of more
//    than 1024 vectors take 512 threads), except that 16-bit SkipSimplified-
//    LayerNormalization rows of 1024 vectors and more take up to 512 threads
//    with two vectors each (hidden 8192 fp16: 12.5 us vs 13.7 at 1024 rows,
//    78.3 vs 78.8 at 8192; bf16 78.4 vs 78.9 at 8192), while float32 rows of
//    1024 vectors keep 256 threads of four (hidden 4096: 41.1 us vs 48.1 at
//    4096 rows);
//  - SkipSimplifiedLayerNormalization rows of 97-128 vectors go to a CTA, not
//    a warp, past kSslnCtaRows rows: the warp, holding four vectors of two
//    inputs per lane, runs at 125 registers, two 256-thread CTAs per SM, too
//    few warps to hide its epilogue (hidden 1024 fp16: 2.49 us vs 3.04 at 512
//    rows, 20.9 vs 22.6 at 16 K rows, 77.1 vs 87.7 at 64 K); at 96 vectors and
//    fewer the warp stays ahead (84.4 vs 89.6 us at 768, 64 K rows);
//  - from kPairRows rows, GatedRMSNorm CTA rows and 16-bit SkipSimplified-
//    LayerNormalization CTA rows of fewer than 160 vectors that are not a
//    whole number of warps take two vectors per thread (GatedRMSNorm C = 2048
//    fp16: 59.8 us vs 65.3 at 32 K rows, 78.2 vs 87.1 at 43 K; hidden 1152
//    fp16: 23.8 vs 24.6 at 16 K); below it one vector per thread is faster
//    (C = 2048: 4.0 us vs 4.2 at 1 K rows; hidden 1152: 2.6 vs 2.9 at 512),
//    and so it is for float32 SkipSimplifiedLayerNormalization rows at any
//    count (hidden 448: 68.3 us vs 71.6, 576: 85.8 vs 97.0 at 64 K rows).
// Splitting a row over a cluster only pays once one CTA cannot hold it.
constexpr int64_t kFewRows = 512;
constexpr int64_t kSslnCtaRows = 256;
constexpr int64_t kPairRows = 8192;
constexpr int kSslnCtaFromVec = 97;
constexpr int kSslnPairBelowVec = 160;
constexpr int kSslnWideFromVec = 1024;

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
             !(op == RowOp::SkipRms && rows > kSslnCtaRows && nvec >= kSslnCtaFromVec)) {
    // Warp per row, up to four vectors per lane.
    p.mode = 0;
    p.tpr = 32;
    p.nv = pow2_ceil(ceil_div(nvec, 32));
    p.block = lane_block(p.nv);
    p.grid = ceil_div(rows, p.block / 32);
  } else {
    // CTA per row; a cluster per row once one CTA cannot hold it.
    p.mode = 1;
    int nv = 1;
    if (rows >= kPairRows &&
        (op == RowOp::Gated ||
         (t != DType::F32 && nvec < kSslnPairBelowVec && nvec % 32 != 0)))
      nv = 2;
    int cta = round32(ceil_div(nvec, nv));
    const int target = rows <= kFewRows ? kRowsMaxThreads
                       : (op == RowOp::SkipRms && t != DType::F32 && nvec >= kSslnWideFromVec)
                           ? kRowsMaxThreads
                           : 256;
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
