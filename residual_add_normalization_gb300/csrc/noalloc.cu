// noalloc.cu -- SkipGroupNorm for callers that cannot allocate device memory.
//
// b200norm_skip_group needs a caller-provided workspace.  Some callers have no
// way to get one: a plugin whose host hands it only the input and output
// buffers and offers no allocator, or a service that reserved all of its
// device memory up front and must not risk an allocation failing (or
// synchronising the device) in the middle of a request.  For them this file
// keeps the workspace in a fixed, file-scope device array that every GPU
// loading the library holds until the process exits, and exposes one more
// entry point that allocates nothing.
#include <cstdio>
#include <mutex>

#include "b200norm.h"
#include "launch.h"

namespace {

// Largest workspace this entry point can serve: the 256-byte control block
// plus 2 MiB of moment slots (131,072 slots of 16 bytes).  Enough for up to
// 64 groups on every route.
constexpr size_t kScratchBytes = 256 + (2u << 20);

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

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

}  // namespace

extern "C" B200NORM_API b200norm_status b200norm_skip_group_noalloc(
    const void* x, const void* skip, int skip_rank, const int64_t* skip_dims, const void* bias,
    const void* gamma, const void* beta, void* y, void* s, int64_t N, int64_t C, int64_t H,
    int64_t W, b200norm_dtype T, b200norm_dtype M, int groups, float epsilon, int activation,
    int channels_last, b200norm_stream_t stream) {
  // Size check first, so an oversized request is refused with a clear
  // message before anything touches the device.
  char msg[256];
  if (N > 0 && C > 0 && H > 0 && W > 0 && groups > 0 && C % groups == 0) {
    // (the size depends on the element size only)
    const size_t need = b200norm::group_workspace_bytes(
        N, C, H, W, groups, T == B200NORM_F32 ? b200norm::DType::F32 : b200norm::DType::F16);
    if (need > kScratchBytes) {
      snprintf(msg, sizeof(msg),
               "this shape needs %zu bytes of scratch, more than the %zu-byte static scratch "
               "of b200norm_skip_group_noalloc; call b200norm_skip_group with a workspace",
               need, kScratchBytes);
      b200norm::set_error_message(msg);
      return B200NORM_ERR_UNSUPPORTED;
    }
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  // The barrier counters and the error record must start at zero; the moment
  // slots are written before they are read.
  if (e == cudaSuccess)
    e = cudaMemsetAsync(scratch, 0, b200norm::kControlBytes,
                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "static scratch set-up: %s", cudaGetErrorString(e));
    b200norm::set_error_message(msg);
    return B200NORM_ERR_CUDA;
  }
  return b200norm_skip_group(x, skip, skip_rank, skip_dims, bias, gamma, beta, y, s, N, C, H, W,
                             T, M, groups, epsilon, activation, channels_last, scratch,
                             kScratchBytes, stream);
}
