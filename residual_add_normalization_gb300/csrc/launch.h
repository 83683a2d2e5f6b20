// launch.h -- host-side interface between the C ABI (api.cu) and the kernel
// translation units.  Every function enqueues work on `stream` and returns the
// CUDA error of the launch (cudaSuccess when nothing needed launching).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "b200norm.h"

namespace b200norm {

// A small thread-safe cache of launch decisions keyed by a plain struct
// (compared bytewise: callers zero the key before filling it).  Oldest
// entries are overwritten once it is full.
template <class Key, class Val, int N = 64>
class PlanCache {
 public:
  bool get(const Key& k, Val* v) {
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < N; ++i)
      if (used_[i] && memcmp(&keys_[i], &k, sizeof(Key)) == 0) {
        *v = vals_[i];
        return true;
      }
    return false;
  }
  void put(const Key& k, const Val& v) {
    std::lock_guard<std::mutex> lock(mu_);
    keys_[next_] = k;
    vals_[next_] = v;
    used_[next_] = true;
    next_ = (next_ + 1) % N;
  }

 private:
  std::mutex mu_;
  Key keys_[N];
  Val vals_[N];
  bool used_[N] = {};
  int next_ = 0;
};

enum class DType { F32 = 0, F16 = 1, BF16 = 2 };

inline size_t dtype_size(DType t) { return t == DType::F32 ? 4 : 2; }

// Schedule chosen for a row-normalization call (see rows.cuh).
struct RowPlan {
  int mode;       // 0: lane groups (tpr <= 32); 1: CTA / cluster per row; 2: walk;
                  // 3: pipelined lane groups (tpr <= 32, inputs through shared memory)
  int ve;         // elements per vector access (16 / sizeof(T)), or 1 (scalar path)
  int tpr;        // threads per row (mode 0/1), CTA threads (mode 2)
  int nv;         // vectors held per thread per row
  int rpg;        // rows per lane group (mode 0)
  int block;      // threads per CTA
  int csize;      // CTAs per cluster (mode 1)
  int64_t grid;   // CTAs
};

struct SkipRmsCall {
  const void* x;
  const void* skip;
  const void* gamma;
  const void* bias;
  void* y;
  void* s;
  float* mean;
  float* inv_std;
  int64_t rows;
  int64_t hidden;
  DType t;
  float eps;
};

struct GatedCall {
  const void* x;
  const void* gate;
  const void* scale;
  void* y;
  int64_t rows;
  int64_t C;
  DType t;
  float eps;
};

// Launches allow programmatic dependent launch (the kernel may be scheduled
// while the preceding grid on the stream drains; it waits for that grid
// before touching memory) unless switched off.  On by default.
bool pdl_enabled();
void set_pdl_enabled(bool on);

// Appends the programmatic-serialization launch attribute to attrs[n] when
// it is enabled; returns the new attribute count.
inline unsigned add_pdl_attr(cudaLaunchAttribute* attrs, unsigned n) {
  if (!pdl_enabled()) return n;
  attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[n].val.programmaticStreamSerializationAllowed = 1;
  return n + 1;
}

// Row plans depend on the operator, the shape, the element type and the
// pointer alignment.
enum class RowOp { SkipRms, Gated };
RowPlan plan_rows(int64_t rows, int64_t n, DType t, bool vector_ok, RowOp op);

// The pipelined lane-group plan for spans of n elements, if the span takes
// it (16-byte vectors, at most 32 of them); false otherwise.
bool pipe_plan(int64_t rows, int64_t n, DType t, bool vector_ok, RowPlan* p);

// SkipSimplifiedLayerNormalization takes the pipelined plan for short rows
// from kPipeMinTiles tiles on (float16: kPipeMinTilesF16).  Measured on GB300
// (rows of 64-256 elements, 16 K-512 K rows, CUDA-graph replay): 3-17% faster
// than the lane-group kernel for float32 and 9-28% for bfloat16 at every size
// measured; for float16 2-4% faster from about 8 K tiles (0.5 M rows of 128),
// up to 3% slower below.  GatedRMSNorm keeps the lane-group kernel, 10-12%
// faster there for 16-bit types and as fast for float32.
constexpr int64_t kPipeMinTiles = 256;
constexpr int64_t kPipeMinTilesF16 = 8192;
bool prefer_pipe_skip_rms(int64_t rows, int64_t n, DType t, bool vector_ok, RowPlan* p);

// The pipelined schedule's bounded waits record B200NORM_ERR_DEVICE_TIMEOUT
// in one device word per device (nullptr if it cannot be resolved).  A test
// can stall it (its producer then issues nothing and the waits give up after
// the given limit).
unsigned* pipe_status_word();
bool pipe_stalled();
unsigned long long pipe_stall_limit_ns();
void set_pipe_stall(bool on, unsigned long long limit_ns);

cudaError_t launch_skip_rms(const SkipRmsCall& c, const RowPlan& p, cudaStream_t stream);
cudaError_t launch_gated(const GatedCall& c, const RowPlan& p, cudaStream_t stream);

// SkipGroupNorm ------------------------------------------------------------
struct SkipGroupCall {
  const void* x;
  const void* skip;
  const void* bias;
  const void* gamma;
  const void* beta;
  void* y;
  void* s;
  int64_t N, C, H, W;
  int groups;
  DType t, m;
  bool bcast;          // skip holds one value per (n, c)
  int activation;
  bool channels_last;
  float eps;
  void* workspace;
  size_t workspace_bytes;
};

// Route chosen for a SkipGroupNorm call.
struct GroupPlan {
  int route;      // 1: NCHW resident (CTA / cluster per group instance)
                  // 2: NHWC cooperative (grid barrier)
                  // 3: two-phase partials -> normalize (any shape)
                  // 4: NHWC through L2 (statistics kernel, then apply kernel)
                  // 5: NHWC through L2 in one cooperative grid (grid barrier)
                  // 6: NHWC cooperative, slab resident in shared memory
  int ve;         // elements per vector access, or 1
  int nv;         // vectors held per thread
  int block;      // threads per CTA
  int csize;      // CTAs per cluster (route 1)
  int64_t grid;   // CTAs
  int ctas_per_item;   // routes 2, 4, 5: CTAs per batch item
  int pix_per_cta;     // routes 2, 4, 5: pixels per CTA
  int chunks;          // route 3: chunks per group instance
  size_t smem;         // dynamic shared memory bytes
};

constexpr size_t kControlBytes = 256;
constexpr int kTwoPhaseChunk = 4096;   // elements per CTA in route 3
constexpr int kMaxCoopCtas = 2048;     // upper bound of route-2 grids

// Workspace a SkipGroupNorm call needs: the control block, then the slots of
// every route that can take the shape in its layout (NCHW: the two-phase
// route's chunks; NHWC also the cooperative and L2 routes' pieces).
size_t group_workspace_bytes(int64_t N, int64_t C, int64_t H, int64_t W, int groups, DType t,
                             bool channels_last);
// Every argument check of b200norm_skip_group except those of the workspace,
// made before anything is enqueued (the message goes to b200norm_last_error);
// B200NORM_OK with *nothing_to_do set when N, H or W is zero.
b200norm_status skip_group_check(const void* x, const void* skip, int skip_rank,
                                 const int64_t* skip_dims, const void* bias, const void* gamma,
                                 const void* beta, const void* y, const void* s, int64_t N,
                                 int64_t C, int64_t H, int64_t W, b200norm_dtype T,
                                 b200norm_dtype M, int groups, float epsilon, int activation,
                                 int channels_last, bool* nothing_to_do);
// force_route 0 picks the route; 2, 3 or 4 asks for that route and returns
// cudaErrorNotSupported when it cannot take the call.
cudaError_t plan_group(const SkipGroupCall& c, bool vector_ok, int force_route, GroupPlan* plan);
GroupPlan two_phase_plan(const SkipGroupCall& c);
cudaError_t launch_group(const SkipGroupCall& c, const GroupPlan& p, cudaStream_t stream);

// Set the thread-local message that b200norm_last_error() returns.
void set_error_message(const char* msg);

// Test hook: a cooperative grid whose barrier can never complete; the waits
// give up after `limit_ns` and record a timeout in the workspace.
cudaError_t launch_barrier_timeout_probe(void* workspace, unsigned long long limit_ns,
                                         cudaStream_t stream);

}  // namespace b200norm
