// rows_pipe.cuh -- the pipelined lane-group schedule for short spans (sm_103a).
//
// For spans of at most 32 16-byte vectors whose two streamed inputs are plain
// row-major arrays (GatedRMSNorm: X and gate; SkipSimplifiedLayerNormalization:
// input and skip).  The register-resident lane kernel can keep only one
// vector per input per thread in flight at full occupancy (32 registers a
// thread); here the loads go to shared memory instead:
//
//   one producer thread   copies tile after tile of both inputs into a ring
//                         of kPipeStages shared-memory stages with bulk
//                         asynchronous copies (cp.async.bulk); each stage's
//                         "full" mbarrier counts the bytes that landed;
//   kPipeWarps warps      wait for a stage, read their rows' vectors from it,
//                         reduce with the segmented butterfly, write Y (and
//                         S) straight to global memory, then release the
//                         stage on its "empty" mbarrier.
//
// A tile is one step of every consumer warp: kPipeWarps * (32 / tpr) rows.
// Tiles go to CTAs round-robin; one CTA per SM (the ring takes ~192 KB).
// Every wait is bounded: after `limit_ns` the thread records
// B200NORM_ERR_DEVICE_TIMEOUT in `status` and leaves; the producer first
// waits (again bounded) for the copies it has in flight, so no copy lands in
// shared memory after the CTA has left.  `stall` (testing only) makes the
// producer issue nothing, so the consumers' waits run out.
#pragma once

#include "bulk.cuh"
#include "rows.cuh"

namespace b200norm {

#ifndef B200NORM_PIPE_STAGES
#define B200NORM_PIPE_STAGES 6
#endif
#ifndef B200NORM_PIPE_MINB
#define B200NORM_PIPE_MINB 1   // CTAs per SM
#endif
constexpr int kPipeStages = B200NORM_PIPE_STAGES;
constexpr int kPipeMinBlocks = B200NORM_PIPE_MINB;
constexpr int kPipeWarps = 31;                        // consumer warps (+ 1 = 1024 threads)
constexpr int kPipeThreads = (kPipeWarps + 1) * 32;   // + one producer warp
constexpr int kPipeTileBytes = 16384;                 // per input and stage
constexpr size_t kPipeSmemBytes =
    2u * kPipeStages * kPipeTileBytes + 2u * kPipeStages * sizeof(unsigned long long);
constexpr unsigned long long kPipeLimitNs = 1000000000ull;   // waits for copies / consumers
constexpr unsigned long long kPipeDrainNs = 1000000000ull;   // the producer's final waits

// Op must provide Elem, P (its 16-byte pack), src0 / src1 (the two streamed
// inputs, rows * n elements each), load_pair, and the lane kernel's
// load_wt / combine / rstd / finish / row_stats.  tpr: power of two <= 32;
// nvec <= tpr vectors per row.
template <class Op>
__global__ void __launch_bounds__(kPipeThreads, kPipeMinBlocks)
rows_pipe_kernel(const typename Op::Args a, int tpr, int nvec, unsigned long long limit_ns,
                 unsigned* status, int stall) {
  using T = typename Op::Elem;
  using P = typename Op::P;
  static_assert(sizeof(P) == 16, "the pipelined schedule moves 16-byte vectors");
  pdl_wait();
  pdl_trigger();
  extern __shared__ float4 smem4[];
  char* ring = reinterpret_cast<char*>(smem4);
  unsigned long long* full =
      reinterpret_cast<unsigned long long*>(ring + 2 * kPipeStages * kPipeTileBytes);
  unsigned long long* empty = full + kPipeStages;
  const int rows_per_tile = kPipeWarps * (32 / tpr);
  const int64_t row_bytes = static_cast<int64_t>(a.n) * sizeof(T);
  const int64_t ntiles = (a.rows + rows_per_tile - 1) / rows_per_tile;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPipeStages; ++s) {
      mbar_init(full + s, 1u);
      mbar_init(empty + s, static_cast<unsigned>(kPipeWarps));
    }
    mbar_init_fence();
  }
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (warp == kPipeWarps) {
    // ---- producer -------------------------------------------------------
    // stall (a testing mode): issue nothing, so that every consumer wait runs
    // out with no copy in flight
    if (lane != 0 || stall) return;
    const char* src0 = reinterpret_cast<const char*>(Op::src0(a));
    const char* src1 = reinterpret_cast<const char*>(Op::src1(a));
    int issued = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++issued) {
      const int s = issued % kPipeStages;
      // a stage's previous tile must have been read by every consumer warp
      if (issued >= kPipeStages &&
          !mbar_wait(empty + s, ((issued / kPipeStages) & 1) ^ 1, limit_ns)) {
        atomicExch(status, kStatusDeviceTimeout);
        break;
      }
      const int64_t r0 = t * rows_per_tile;
      const int64_t nrows = min(static_cast<int64_t>(rows_per_tile), a.rows - r0);
      const unsigned bytes = static_cast<unsigned>(nrows * row_bytes);
      char* dst = ring + static_cast<size_t>(s) * 2 * kPipeTileBytes;
      mbar_arrive_expect_tx(full + s, 2 * bytes);
      bulk_load(dst, src0 + r0 * row_bytes, bytes, full + s);
      bulk_load(dst + kPipeTileBytes, src1 + r0 * row_bytes, bytes, full + s);
    }
    // the CTA may leave only once its copies have landed
    for (int i = issued > kPipeStages ? issued - kPipeStages : 0; i < issued; ++i)
      if (!mbar_wait(full + i % kPipeStages, (i / kPipeStages) & 1, kPipeDrainNs))
        atomicExch(status, kStatusDeviceTimeout);
    return;
  }

  // ---- consumers ----------------------------------------------------------
  const int li = lane & (tpr - 1);
  const int row_in_tile = warp * (32 / tpr) + lane / tpr;
  typename Op::Wt w;
  if (li < nvec) Op::load_wt(a, li, w);
  int j = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++j) {
    const int s = j % kPipeStages;
    // the warp leaves together (its lanes meet again in __syncwarp and the
    // butterfly), so the give-up decision is the warp's
    const bool landed = mbar_wait(full + s, (j / kPipeStages) & 1, limit_ns);
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) atomicExch(status, kStatusDeviceTimeout);
      return;
    }
    const int64_t row = t * rows_per_tile + row_in_tile;
    const bool live = row < a.rows && li < nvec;
    typename Op::In in;
    typename Op::Hold h;
    float part = 0.0f;
    if (live) {
      const P* s0 = reinterpret_cast<const P*>(ring + static_cast<size_t>(s) * 2 * kPipeTileBytes);
      const P* s1 = reinterpret_cast<const P*>(ring + static_cast<size_t>(s) * 2 * kPipeTileBytes +
                                               kPipeTileBytes);
      const int idx = row_in_tile * nvec + li;
      Op::load_pair(s0[idx], s1[idx], in);
      part = Op::combine(a, row, li, in, w, h);
    }
    const float r = Op::rstd(a, seg_sum(part, tpr));
    if (live) {
      Op::finish(a, row, li, h, w, r);
      if (li == 0) Op::row_stats(a, row, r);
    }
    // Hand the stage back only now.  The Y stores above depend on every value
    // this warp read from the stage, so those reads have completed; releasing
    // right after issuing the shared-memory loads let the next tile's copy
    // land before a load had read (measured: 2 rows in 1 M read the next
    // tile's X).
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
}

}  // namespace b200norm
