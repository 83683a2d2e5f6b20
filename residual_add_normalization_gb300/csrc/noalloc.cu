// noalloc.cu -- SkipGroupNorm for callers that cannot allocate device memory.
//
// b200norm_skip_group needs a caller-provided workspace.  Some callers have no
// way to get one: a plugin whose host hands it only the input and output
// buffers and offers no allocator, or a service that reserved all of its
// device memory up front and must not risk an allocation failing (or
// synchronising the device) in the middle of a request.  For them this file
// keeps the workspace in a fixed, file-scope device array that every GPU
// loading the library holds until the process exits, and exposes one more
// entry point that allocates nothing, with a query of the array's
// device-side timeout record.
#include <cstdio>
#include <mutex>

#include "b200norm.h"
#include "b200norm_testing.h"
#include "launch.h"

namespace {

// Largest workspace this entry point can serve: the 256-byte control block
// plus 2 MiB of slots (131,072 slots of 16 bytes).  A call fits exactly when
// b200norm_skip_group_workspace_size() of its shape is at most this.  With
// L = C / groups * H * W: NHWC shapes with at most 32 groups and
// N * ceil(L / 4096) <= 4,096 fit; NCHW shapes fit when
// N * groups * ceil(L / 4096) <= 131,072.
constexpr size_t kScratchBytes = 256 + (2u << 20);

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Control-block words (see Control in common.cuh): the barrier counts
// (bytes 0-7) and the per-item counters (bytes 16-255) must start at zero;
// the error record (bytes 8-15) is left for b200norm_skip_group_noalloc_status.
constexpr size_t kErrorOffset = 8, kErrorBytes = 8;

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// The array's name is only a host-side stand-in; the device address is taken
// once per device, with that device current.
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

b200norm_status cuda_error(cudaError_t e, const char* what) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  b200norm::set_error_message(msg);
  return B200NORM_ERR_CUDA;
}

}  // namespace

extern "C" B200NORM_API b200norm_status b200norm_skip_group_noalloc(
    const void* x, const void* skip, int skip_rank, const int64_t* skip_dims, const void* bias,
    const void* gamma, const void* beta, void* y, void* s, int64_t N, int64_t C, int64_t H,
    int64_t W, b200norm_dtype T, b200norm_dtype M, int groups, float epsilon, int activation,
    int channels_last, b200norm_stream_t stream) {
  // Every argument check first, so an invalid call enqueues nothing.
  bool nothing_to_do = false;
  if (b200norm_status st = b200norm::skip_group_check(
          x, skip, skip_rank, skip_dims, bias, gamma, beta, y, s, N, C, H, W, T, M, groups,
          epsilon, activation, channels_last, &nothing_to_do))
    return st;
  if (nothing_to_do) {
    b200norm::set_error_message("");
    return B200NORM_OK;
  }
  const b200norm::DType t = T == B200NORM_F32   ? b200norm::DType::F32
                            : T == B200NORM_F16 ? b200norm::DType::F16
                                                : b200norm::DType::BF16;
  const size_t need = b200norm::group_workspace_bytes(N, C, H, W, groups, t, channels_last != 0);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "this shape needs %zu bytes of scratch, more than the %zu-byte static scratch "
             "of b200norm_skip_group_noalloc; call b200norm_skip_group with a workspace",
             need, kScratchBytes);
    b200norm::set_error_message(msg);
    return B200NORM_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  // The counters must start at zero (every kernel that uses one returns it to
  // zero, so this only matters after an interrupted launch); the slots are
  // written before they are read.
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* ctl = static_cast<unsigned char*>(scratch);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctl, 0, kErrorOffset, st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(ctl + kErrorOffset + kErrorBytes, 0,
                        b200norm::kControlBytes - kErrorOffset - kErrorBytes, st);
  if (e != cudaSuccess) return cuda_error(e, "static scratch set-up");
  return b200norm_skip_group(x, skip, skip_rank, skip_dims, bias, gamma, beta, y, s, N, C, H, W,
                             T, M, groups, epsilon, activation, channels_last, scratch,
                             kScratchBytes, stream);
}

extern "C" B200NORM_API b200norm_status b200norm_skip_group_noalloc_status(
    b200norm_stream_t stream) {
  void* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) return cuda_error(e, "static scratch set-up");
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned int rec[2] = {0, 0};  // error, error site
  unsigned char* ctl = static_cast<unsigned char*>(scratch);
  e = cudaStreamSynchronize(st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(rec, ctl + kErrorOffset, sizeof(rec), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && rec[0] != 0)
    e = cudaMemsetAsync(ctl + kErrorOffset, 0, kErrorBytes, st);
  if (e == cudaSuccess && rec[0] != 0) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_error(e, "static scratch status read");
  if (rec[0] != 0) {
    char msg[128];
    snprintf(msg, sizeof(msg), "device wait %u gave up", rec[1]);
    b200norm::set_error_message(msg);
    return static_cast<b200norm_status>(rec[0]);
  }
  b200norm::set_error_message("");
  return B200NORM_OK;
}

extern "C" B200NORM_API b200norm_status b200norm_testing_noalloc_barrier_timeout(
    uint64_t limit_ns, b200norm_stream_t stream) {
  if (limit_ns == 0 || limit_ns > 5000000000ull) {
    b200norm::set_error_message("limit_ns must be in (0, 5 s]");
    return B200NORM_ERR_INVALID_ARGUMENT;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e == cudaSuccess)
    e = b200norm::launch_barrier_timeout_probe(scratch, limit_ns,
                                               reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "timeout probe launch");
  b200norm::set_error_message("");
  return B200NORM_OK;
}
