// api.cu -- the C ABI: argument validation, schedule selection and launch.
//
// Every entry point validates its arguments completely before enqueueing
// anything, picks a schedule from the shape, element type and pointer
// alignment (the GB300 counterpart of the pages' per-call choice among
// implementation variants), and launches on the caller's stream.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "b200norm.h"
#include "b200norm_testing.h"
#include "launch.h"

using namespace b200norm;

namespace {

thread_local std::string g_error;
thread_local int g_force_row_mode = 0;
thread_local int g_force_group_route = 0;
thread_local int g_force_csize = 0;  // forced CTA / cluster row split (0: automatic)
thread_local int g_force_nv = 0;

b200norm_status fail(b200norm_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_error = buf;
  return st;
}

b200norm_status ok() {
  g_error.clear();
  return B200NORM_OK;
}

b200norm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(B200NORM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool dtype_ok(b200norm_dtype t) {
  return t == B200NORM_F32 || t == B200NORM_F16 || t == B200NORM_BF16;
}

DType to_dtype(b200norm_dtype t) {
  return t == B200NORM_F32 ? DType::F32 : t == B200NORM_F16 ? DType::F16 : DType::BF16;
}

// SkipGroupNorm (T, M) pairs with kernels: M = float32 or T, and float16
// gamma/beta under float32 X.
bool group_types_ok(b200norm_dtype t, b200norm_dtype m) {
  return dtype_ok(t) && (m == B200NORM_F32 || m == t || (t == B200NORM_F32 && m == B200NORM_F16));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
  const void* p;
  size_t bytes;
  const char* name;
};

bool overlaps(const Range& a, const Range& b) {
  if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Outputs may not overlap inputs or each other.
b200norm_status check_overlaps(const Range* in, int nin, const Range* out, int nout) {
  for (int i = 0; i < nout; ++i) {
    for (int j = 0; j < nin; ++j)
      if (overlaps(out[i], in[j]))
        return fail(B200NORM_ERR_INVALID_ARGUMENT, "output %s overlaps input %s", out[i].name,
                    in[j].name);
    for (int j = i + 1; j < nout; ++j)
      if (overlaps(out[i], out[j]))
        return fail(B200NORM_ERR_INVALID_ARGUMENT, "outputs %s and %s overlap", out[i].name,
                    out[j].name);
  }
  return B200NORM_OK;
}

b200norm_status check_eps(float eps) {
  if (std::isnan(eps) || eps < 0.0f)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "epsilon must be >= 0 and not NaN (got %g)",
                static_cast<double>(eps));
  return B200NORM_OK;
}

constexpr int64_t kMaxGrid = 0x7fffffffLL;

// The forced CTA / cluster split of b200norm_testing_force_split.
b200norm_status forced_split(int64_t rows, int64_t n, RowPlan* p) {
  const int64_t nvec = n / p->ve;
  const int64_t per = static_cast<int64_t>(g_force_nv) * g_force_csize;
  const int64_t block = ((nvec + per - 1) / per + 31) / 32 * 32;
  if (block > 512)
    return fail(B200NORM_ERR_UNSUPPORTED, "forced split needs %lld threads per CTA (max 512)",
                static_cast<long long>(block));
  p->mode = 1;
  p->nv = g_force_nv;
  p->rpg = 1;
  p->csize = g_force_csize;
  p->block = static_cast<int>(block);
  p->tpr = p->block * p->csize;
  p->grid = rows * p->csize;
  return B200NORM_OK;
}

RowPlan forced_walk(int64_t rows, RowPlan p) {
  p.mode = 2;
  p.block = p.tpr = 512;
  p.csize = 1;
  p.nv = p.rpg = 1;
  p.grid = rows;
  return p;
}

b200norm_status skip_rms_impl(const void* input, const void* skip, const void* gamma,
                              const void* bias, void* output, void* sum, float* mean,
                              float* inv_std, int64_t rows, int64_t hidden, b200norm_dtype T,
                              float epsilon, b200norm_stream_t stream) {
  if (!dtype_ok(T)) return fail(B200NORM_ERR_UNSUPPORTED, "element type %d not supported", T);
  if (rows < 0) return fail(B200NORM_ERR_INVALID_ARGUMENT, "rows must be >= 0");
  if (hidden <= 0) return fail(B200NORM_ERR_INVALID_ARGUMENT, "hidden must be > 0");
  if (hidden > 0x7fffffffLL) return fail(B200NORM_ERR_UNSUPPORTED, "hidden exceeds 2^31-1");
  if (b200norm_status st = check_eps(epsilon)) return st;
  if (rows == 0) return ok();
  if (!input || !skip || !gamma || !output)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "input, skip, gamma and output are required");
  const size_t es = dtype_size(to_dtype(T));
  const void* ptrs[] = {input, skip, gamma, bias, output, sum};
  for (const void* p : ptrs)
    if (p && !aligned(p, es))
      return fail(B200NORM_ERR_INVALID_ARGUMENT, "tensor pointer not aligned to its element size");
  if ((mean && !aligned(mean, 4)) || (inv_std && !aligned(inv_std, 4)))
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "statistics pointers must be 4-byte aligned");
  const size_t tb = static_cast<size_t>(rows) * hidden * es, vb = hidden * es;
  const Range in[] = {{input, tb, "input"}, {skip, tb, "skip"}, {gamma, vb, "gamma"},
                      {bias, vb, "bias"}};
  const Range out[] = {{output, tb, "output"}, {sum, tb, "input_skip_bias_sum"},
                       {mean, static_cast<size_t>(rows) * 4, "mean"},
                       {inv_std, static_cast<size_t>(rows) * 4, "inv_std_var"}};
  if (b200norm_status st = check_overlaps(in, 4, out, 4)) return st;

  const int ve = static_cast<int>(16 / es);
  bool vec = hidden % ve == 0;
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) vec = false;
  RowPlan plan = plan_rows(rows, hidden, to_dtype(T), vec, RowOp::SkipRms);
  if (g_force_csize)
    if (b200norm_status st = forced_split(rows, hidden, &plan)) return st;
  if (g_force_row_mode == 0 && !g_force_csize)
    prefer_pipe_skip_rms(rows, hidden, to_dtype(T), vec, &plan);
  if (g_force_row_mode == 2) plan = forced_walk(rows, plan);
  if (g_force_row_mode == 3 && !pipe_plan(rows, hidden, to_dtype(T), vec, &plan))
    return fail(B200NORM_ERR_UNSUPPORTED, "forced pipelined schedule cannot take this call");
  if (plan.grid > kMaxGrid) return fail(B200NORM_ERR_UNSUPPORTED, "too many rows for one launch");
  SkipRmsCall c{input, skip, gamma, bias, output, sum, mean, inv_std, rows, hidden, to_dtype(T),
                epsilon};
  cudaError_t e = launch_skip_rms(c, plan, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "skip_rms launch");
  return ok();
}

// Skip shape classification (SkipGroupNorm README, Inputs, skip):
// returns 0 full, 1 broadcast per (n, c), -1 unrecognised.
int classify_skip(int rank, const int64_t* d, int64_t N, int64_t C, int64_t H, int64_t W,
                  bool cl) {
  if (rank == 4 && d) {
    const int64_t full_cl[4] = {N, H, W, C}, full_cf[4] = {N, C, H, W};
    const int64_t* f = cl ? full_cl : full_cf;
    if (d[0] == f[0] && d[1] == f[1] && d[2] == f[2] && d[3] == f[3]) return 0;
    if (d[0] == N && d[1] == 1 && d[2] == 1 && d[3] == C) return (H == 1 && W == 1) ? 0 : 1;
    return -1;
  }
  if (rank == 2 && d && d[0] == N && d[1] == C) return 1;
  return -1;
}

}  // namespace

namespace b200norm {

namespace {
std::atomic<bool> g_pdl{true};
}

bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed); }

void set_pdl_enabled(bool on) { g_pdl.store(on, std::memory_order_relaxed); }

}  // namespace b200norm

void b200norm::set_error_message(const char* msg) { g_error = msg; }

b200norm_status b200norm::skip_group_check(const void* x, const void* skip, int skip_rank,
                                           const int64_t* skip_dims, const void* bias,
                                           const void* gamma, const void* beta, const void* y,
                                           const void* s, int64_t N, int64_t C, int64_t H,
                                           int64_t W, b200norm_dtype T, b200norm_dtype M,
                                           int groups, float epsilon, int activation,
                                           int channels_last, bool* nothing_to_do) {
  *nothing_to_do = false;
  if (!group_types_ok(T, M))
    return fail(B200NORM_ERR_UNSUPPORTED, "element types T=%d M=%d not supported", T, M);
  if (N < 0 || C <= 0 || H < 0 || W < 0)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "need N >= 0, C > 0, H >= 0, W >= 0");
  if (groups <= 0 || C % groups != 0)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "groups (%d) must be > 0 and divide C (%lld)",
                groups, static_cast<long long>(C));
  if (activation != 0 && activation != 1)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "activation must be 0 (none) or 1 (SiLU)");
  if (b200norm_status st = check_eps(epsilon)) return st;
  const bool cl = channels_last != 0;
  const int bc = classify_skip(skip_rank, skip_dims, N, C, H, W, cl);
  if (bc < 0)
    return fail(B200NORM_ERR_INVALID_ARGUMENT,
                "skip must have X's shape, (N, C) or (N, 1, 1, C)");
  if (N == 0 || H == 0 || W == 0) {
    *nothing_to_do = true;
    return B200NORM_OK;
  }
  if (C > 0x7fffffffLL || H * W > 0x7fffffffLL || N > 0x7fffffffLL)
    return fail(B200NORM_ERR_UNSUPPORTED, "C, H*W or N exceeds 2^31-1");
  if (!x || !skip || !gamma || !beta || !y)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "x, skip, gamma, beta and y are required");
  const size_t es = dtype_size(to_dtype(T)), ms = dtype_size(to_dtype(M));
  const void* tptrs[] = {x, skip, bias, y, s};
  for (const void* p : tptrs)
    if (p && !aligned(p, es))
      return fail(B200NORM_ERR_INVALID_ARGUMENT, "tensor pointer not aligned to its element size");
  if (!aligned(gamma, ms) || !aligned(beta, ms))
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "gamma/beta not aligned to their element size");
  const size_t tb = static_cast<size_t>(N * C * H * W) * es;
  const size_t sb = bc ? static_cast<size_t>(N * C) * es : tb;
  const Range in[] = {{x, tb, "X"}, {skip, sb, "skip"}, {bias, C * es, "bias"},
                      {gamma, C * ms, "gamma"}, {beta, C * ms, "beta"}};
  const Range out[] = {{y, tb, "Y"}, {s, tb, "S"}};
  return check_overlaps(in, 5, out, 2);
}

extern "C" {

int b200norm_version(void) { return 1; }

const char* b200norm_status_string(b200norm_status s) {
  switch (s) {
    case B200NORM_OK: return "B200NORM_OK";
    case B200NORM_ERR_INVALID_ARGUMENT: return "B200NORM_ERR_INVALID_ARGUMENT";
    case B200NORM_ERR_UNSUPPORTED: return "B200NORM_ERR_UNSUPPORTED";
    case B200NORM_ERR_CUDA: return "B200NORM_ERR_CUDA";
    case B200NORM_ERR_WORKSPACE: return "B200NORM_ERR_WORKSPACE";
    case B200NORM_ERR_DEVICE_TIMEOUT: return "B200NORM_ERR_DEVICE_TIMEOUT";
  }
  return "B200NORM_UNKNOWN_STATUS";
}

const char* b200norm_last_error(void) { return g_error.c_str(); }

b200norm_status b200norm_skip_rms(const void* input, const void* skip, const void* gamma,
                                  const void* bias, void* output, void* input_skip_bias_sum,
                                  int64_t rows, int64_t hidden, b200norm_dtype T, float epsilon,
                                  b200norm_stream_t stream) {
  return skip_rms_impl(input, skip, gamma, bias, output, input_skip_bias_sum, nullptr, nullptr,
                       rows, hidden, T, epsilon, stream);
}

b200norm_status b200norm_skip_rms_stats(const void* input, const void* skip, const void* gamma,
                                        const void* bias, void* output,
                                        void* input_skip_bias_sum, float* mean,
                                        float* inv_std_var, int64_t rows, int64_t hidden,
                                        b200norm_dtype T, float epsilon,
                                        b200norm_stream_t stream) {
  return skip_rms_impl(input, skip, gamma, bias, output, input_skip_bias_sum, mean, inv_std_var,
                       rows, hidden, T, epsilon, stream);
}

b200norm_status b200norm_gated_rms(const void* x, const void* gate, const void* scale, void* y,
                                   int64_t numel, int64_t C, b200norm_dtype T, float epsilon,
                                   b200norm_stream_t stream) {
  if (!dtype_ok(T)) return fail(B200NORM_ERR_UNSUPPORTED, "element type %d not supported", T);
  if (C <= 0) return fail(B200NORM_ERR_INVALID_ARGUMENT, "C (numel of scale) must be > 0");
  if (numel < 0) return fail(B200NORM_ERR_INVALID_ARGUMENT, "numel must be >= 0");
  if (numel % C != 0)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "numel (%lld) is not a multiple of C (%lld)",
                static_cast<long long>(numel), static_cast<long long>(C));
  if (C > 0x7fffffffLL) return fail(B200NORM_ERR_UNSUPPORTED, "C exceeds 2^31-1");
  if (b200norm_status st = check_eps(epsilon)) return st;
  if (numel == 0) return ok();
  if (!x || !gate || !scale || !y)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "x, gate, scale and y are required");
  const size_t es = dtype_size(to_dtype(T));
  const void* ptrs[] = {x, gate, scale, y};
  for (const void* p : ptrs)
    if (!aligned(p, es))
      return fail(B200NORM_ERR_INVALID_ARGUMENT, "tensor pointer not aligned to its element size");
  const size_t tb = static_cast<size_t>(numel) * es;
  const Range in[] = {{x, tb, "x"}, {gate, tb, "gate"}, {scale, C * es, "scale"}};
  const Range out[] = {{y, tb, "y"}};
  if (b200norm_status st = check_overlaps(in, 3, out, 1)) return st;
  const int64_t rows = numel / C;
  const int ve = static_cast<int>(16 / es);
  bool vec = C % ve == 0;
  for (const void* p : ptrs)
    if (!aligned(p, 16)) vec = false;
  RowPlan plan = plan_rows(rows, C, to_dtype(T), vec, RowOp::Gated);
  if (g_force_csize)
    if (b200norm_status st = forced_split(rows, C, &plan)) return st;
  if (g_force_row_mode == 2) plan = forced_walk(rows, plan);
  if (g_force_row_mode == 3 && !pipe_plan(rows, C, to_dtype(T), vec, &plan))
    return fail(B200NORM_ERR_UNSUPPORTED, "forced pipelined schedule cannot take this call");
  if (plan.grid > kMaxGrid) return fail(B200NORM_ERR_UNSUPPORTED, "too many rows for one launch");
  GatedCall c{x, gate, scale, y, rows, C, to_dtype(T), epsilon};
  cudaError_t e = launch_gated(c, plan, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gated_rms launch");
  return ok();
}

size_t b200norm_skip_group_workspace_size(int64_t N, int64_t C, int64_t H, int64_t W, int groups,
                                          b200norm_dtype T, int channels_last) {
  if (!dtype_ok(T)) return kControlBytes;
  return group_workspace_bytes(N, C, H, W, groups, to_dtype(T), channels_last != 0);
}

b200norm_status b200norm_skip_group(const void* x, const void* skip, int skip_rank,
                                    const int64_t* skip_dims, const void* bias,
                                    const void* gamma, const void* beta, void* y, void* s,
                                    int64_t N, int64_t C, int64_t H, int64_t W,
                                    b200norm_dtype T, b200norm_dtype M, int groups,
                                    float epsilon, int activation, int channels_last,
                                    void* workspace, size_t workspace_bytes,
                                    b200norm_stream_t stream) {
  bool nothing_to_do = false;
  if (b200norm_status st = skip_group_check(x, skip, skip_rank, skip_dims, bias, gamma, beta, y,
                                            s, N, C, H, W, T, M, groups, epsilon, activation,
                                            channels_last, &nothing_to_do))
    return st;
  if (nothing_to_do) return ok();
  const bool cl = channels_last != 0;
  const size_t need = group_workspace_bytes(N, C, H, W, groups, to_dtype(T), cl);
  if (!workspace || workspace_bytes < need)
    return fail(B200NORM_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu at %p)", need,
                workspace_bytes, workspace);
  if (!aligned(workspace, 256))
    return fail(B200NORM_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  const size_t es = dtype_size(to_dtype(T)), ms = dtype_size(to_dtype(M));
  const int bc = classify_skip(skip_rank, skip_dims, N, C, H, W, cl);
  const size_t tb = static_cast<size_t>(N * C * H * W) * es;
  const size_t sb = bc ? static_cast<size_t>(N * C) * es : tb;
  const Range ws = {workspace, workspace_bytes, "workspace"};
  const Range others[] = {{x, tb, "X"}, {skip, sb, "skip"}, {bias, C * es, "bias"},
                          {gamma, C * ms, "gamma"}, {beta, C * ms, "beta"}, {y, tb, "Y"},
                          {s, tb, "S"}};
  for (const Range& r : others)
    if (overlaps(ws, r))
      return fail(B200NORM_ERR_WORKSPACE, "workspace overlaps %s", r.name);

  SkipGroupCall c{x, skip, bias, gamma, beta, y, s, N, C, H, W, groups, to_dtype(T), to_dtype(M),
                  bc == 1, activation, cl, epsilon, workspace, workspace_bytes};
  bool vec = true;
  const void* tptrs[] = {x, skip, bias, y, s};
  for (const void* p : tptrs)
    if (p && !aligned(p, 16)) vec = false;
  GroupPlan plan;
  cudaError_t e = plan_group(c, vec, g_force_group_route, &plan);
  if (e == cudaErrorNotSupported && g_force_group_route)
    return fail(B200NORM_ERR_UNSUPPORTED, "forced route %d cannot take this call",
                g_force_group_route);
  if (e != cudaSuccess) return cuda_fail(e, "skip_group planning");
  if (plan.grid > kMaxGrid) return fail(B200NORM_ERR_UNSUPPORTED, "problem too large for one launch");
  e = launch_group(c, plan, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(B200NORM_ERR_CUDA,
                "skip_group launch (route %d, grid %lld, block %d, cluster %d, smem %zu): %s",
                plan.route, static_cast<long long>(plan.grid), plan.block, plan.csize, plan.smem,
                cudaGetErrorString(e));
  return ok();
}

b200norm_status b200norm_workspace_init(void* workspace, size_t workspace_bytes,
                                        b200norm_stream_t stream) {
  if (!workspace || workspace_bytes < kControlBytes)
    return fail(B200NORM_ERR_WORKSPACE, "workspace missing or smaller than %zu bytes",
                kControlBytes);
  cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace init");
  return ok();
}

b200norm_status b200norm_workspace_status(const void* workspace, b200norm_stream_t stream) {
  if (!workspace) return fail(B200NORM_ERR_WORKSPACE, "workspace is NULL");
  unsigned int ctl[4] = {0, 0, 0, 0};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctl, workspace, sizeof(ctl), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "workspace status read");
  if (ctl[2] != 0)
    return fail(static_cast<b200norm_status>(ctl[2]), "device wait %u gave up", ctl[3]);
  return ok();
}

b200norm_status b200norm_rows_status(b200norm_stream_t stream) {
  unsigned* word = pipe_status_word();
  if (!word) return fail(B200NORM_ERR_CUDA, "row status word not available on this device");
  unsigned v = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v != 0) e = cudaMemsetAsync(word, 0, sizeof(v), st);
  if (e == cudaSuccess && v != 0) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "row status read");
  if (v != 0) return fail(static_cast<b200norm_status>(v), "a pipelined row wait gave up");
  return ok();
}

// ---- testing hooks ---------------------------------------------------------

b200norm_status b200norm_testing_barrier_timeout(void* workspace, size_t workspace_bytes,
                                                 uint64_t limit_ns, b200norm_stream_t stream) {
  if (!workspace || workspace_bytes < kControlBytes || !aligned(workspace, 256))
    return fail(B200NORM_ERR_WORKSPACE, "workspace missing, small or misaligned");
  if (limit_ns == 0 || limit_ns > 5000000000ull)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "limit_ns must be in (0, 5 s]");
  cudaError_t e = launch_barrier_timeout_probe(workspace, limit_ns,
                                               reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "timeout probe launch");
  return ok();
}

b200norm_status b200norm_testing_force(int row_mode, int group_route) {
  if (row_mode < 0 || row_mode > 3 || group_route < 0 || group_route == 1 || group_route > 6)
    return fail(B200NORM_ERR_INVALID_ARGUMENT,
                "row_mode in {0, 1, 2, 3}, group_route in {0, 2, 3, 4, 5, 6}");
  g_force_row_mode = row_mode;
  g_force_group_route = group_route;
  return ok();
}

b200norm_status b200norm_testing_force_split(int csize, int nv) {
  const bool off = csize == 0 && nv == 0;
  const bool pow2_c = csize == 1 || csize == 2 || csize == 4 || csize == 8 || csize == 16;
  const bool pow2_v = nv == 1 || nv == 2 || nv == 4 || nv == 8;
  if (!off && !(pow2_c && pow2_v))
    return fail(B200NORM_ERR_INVALID_ARGUMENT,
                "csize in {1, 2, 4, 8, 16} and nv in {1, 2, 4, 8}, or both 0");
  g_force_csize = csize;
  g_force_nv = nv;
  return ok();
}

b200norm_status b200norm_testing_pipe_stall(int on, uint64_t limit_ns) {
  if ((on != 0 && on != 1) || (on && (limit_ns == 0 || limit_ns > 5000000000ull)))
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "on in {0, 1}; with on, limit_ns in (0, 5 s]");
  set_pipe_stall(on != 0, on ? limit_ns : 0);
  return ok();
}

b200norm_status b200norm_testing_set_pdl(int on) {
  if (on != 0 && on != 1) return fail(B200NORM_ERR_INVALID_ARGUMENT, "on must be 0 or 1");
  set_pdl_enabled(on != 0);
  return ok();
}

static b200norm_status plan_rows_query(int64_t rows, int64_t n, b200norm_dtype T, int aligned16,
                                       RowOp op, int64_t out[8]) {
  if (!dtype_ok(T) || n <= 0 || rows < 0 || !out)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "bad plan query");
  const int ve = static_cast<int>(16 / dtype_size(to_dtype(T)));
  const RowPlan p = plan_rows(rows, n, to_dtype(T), aligned16 && n % ve == 0, op);
  const int64_t v[8] = {p.mode, p.ve, p.tpr, p.nv, p.rpg, p.block, p.csize, p.grid};
  for (int i = 0; i < 8; ++i) out[i] = v[i];
  return ok();
}

b200norm_status b200norm_testing_plan_rows(int64_t rows, int64_t n, b200norm_dtype T,
                                           int aligned16, int64_t out[8]) {
  return plan_rows_query(rows, n, T, aligned16, RowOp::SkipRms, out);
}

b200norm_status b200norm_testing_plan_gated(int64_t rows, int64_t C, b200norm_dtype T,
                                            int aligned16, int64_t out[8]) {
  return plan_rows_query(rows, C, T, aligned16, RowOp::Gated, out);
}

b200norm_status b200norm_testing_plan_group(int64_t N, int64_t C, int64_t H, int64_t W, int groups,
                                            b200norm_dtype T, b200norm_dtype M, int channels_last,
                                            int aligned16, int64_t out[8]) {
  if (!group_types_ok(T, M) || N <= 0 || C <= 0 || H <= 0 || W <= 0 || groups <= 0 ||
      C % groups != 0 || !out)
    return fail(B200NORM_ERR_INVALID_ARGUMENT, "bad plan query");
  SkipGroupCall c{};
  c.N = N;
  c.C = C;
  c.H = H;
  c.W = W;
  c.groups = groups;
  c.t = to_dtype(T);
  c.m = to_dtype(M);
  c.channels_last = channels_last != 0;
  GroupPlan p;
  cudaError_t e = plan_group(c, aligned16 != 0, 0, &p);
  if (e != cudaSuccess) return cuda_fail(e, "plan_group");
  const int64_t v[8] = {p.route, p.ve, p.nv, p.block, p.csize, p.grid, p.ctas_per_item,
                        p.pix_per_cta};
  for (int i = 0; i < 8; ++i) out[i] = v[i];
  return ok();
}

}  // extern "C"
