// common.cuh -- device helpers shared by the b200norm kernels (sm_103a).
//
// Vector I/O with cache hints, element conversions, warp / CTA / cluster
// reductions (cluster partials exchanged through distributed shared memory),
// Chan's pairwise merge of (count, mean, M2) moments, and a bounded
// grid-wide barrier for cooperative launches.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace b200norm {

// ---------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
// A bfloat16 is the upper half of a binary32: widening is a 16-bit shift.
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) {
  return __uint_as_float(static_cast<unsigned>(__bfloat16_as_ushort(v)) << 16);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) {
  return __float2half_rn(v);  // round to nearest-even, subnormals kept
}
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);  // round to nearest-even, subnormals kept
}

// The 16-bit types convert two elements at a time (one instruction each way).
template <typename T> struct Pair2 { static constexpr bool kPacked = false; };
template <> struct Pair2<__half> {
  static constexpr bool kPacked = true;
  using type = __half2;
  __device__ __forceinline__ static float2 widen(type v) { return __half22float2(v); }
  __device__ __forceinline__ static type narrow(float a, float b) {
    return __floats2half2_rn(a, b);
  }
};
template <> struct Pair2<__nv_bfloat16> {
  static constexpr bool kPacked = true;
  using type = __nv_bfloat162;
  __device__ __forceinline__ static float2 widen(type v) {
    unsigned w;
    memcpy(&w, &v, sizeof(w));
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  __device__ __forceinline__ static type narrow(float a, float b) {
    return __floats2bfloat162_rn(a, b);
  }
};

// A pack of N elements of T moved as one access of sizeof(T) * N bytes.
template <typename T, int N>
struct alignas(sizeof(T) * N) Pack {
  T v[N];
};

template <int BYTES> struct RawOf;
template <> struct RawOf<16> { using type = uint4; };
template <> struct RawOf<8> { using type = uint2; };
template <> struct RawOf<4> { using type = unsigned int; };
template <> struct RawOf<2> { using type = unsigned short; };

// Streaming load: data read exactly once (evict-first in L1 and L2).
template <typename T, int N>
__device__ __forceinline__ Pack<T, N> ld_stream(const T* p) {
  using R = typename RawOf<sizeof(T) * N>::type;
  R r = __ldcs(reinterpret_cast<const R*>(p));
  Pack<T, N> out;
  memcpy(&out, &r, sizeof(R));
  return out;
}

// Read-only load of data reused by many CTAs (weights, biases).
template <typename T, int N>
__device__ __forceinline__ Pack<T, N> ld_reuse(const T* p) {
  using R = typename RawOf<sizeof(T) * N>::type;
  R r = __ldg(reinterpret_cast<const R*>(p));
  Pack<T, N> out;
  memcpy(&out, &r, sizeof(R));
  return out;
}

// Streaming store (evict-first).
template <typename T, int N>
__device__ __forceinline__ void st_stream(T* p, const Pack<T, N>& v) {
  using R = typename RawOf<sizeof(T) * N>::type;
  R r;
  memcpy(&r, &v, sizeof(R));
  __stcs(reinterpret_cast<R*>(p), r);
}

// Widen a pack to binary32 (pairs of halves convert with one instruction).
template <typename T, int N>
__device__ __forceinline__ void unpack(const Pack<T, N>& p, float (&f)[N]) {
  if constexpr (Pair2<T>::kPacked && N % 2 == 0) {
    using P2 = Pair2<T>;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float2 t = P2::widen(reinterpret_cast<const typename P2::type*>(p.v)[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) f[i] = to_f32(p.v[i]);
  }
}

// Narrow binary32 values to a pack, each rounded to nearest-even.
template <typename T, int N>
__device__ __forceinline__ Pack<T, N> pack_from(const float (&f)[N]) {
  Pack<T, N> p;
  if constexpr (Pair2<T>::kPacked && N % 2 == 0) {
    using P2 = Pair2<T>;
#pragma unroll
    for (int i = 0; i < N / 2; ++i)
      reinterpret_cast<typename P2::type*>(p.v)[i] = P2::narrow(f[2 * i], f[2 * i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) p.v[i] = from_f32<T>(f[i]);
  }
  return p;
}

// Element pair (2i, 2i+1) of a pack as binary32, and the reverse (each value
// rounded to nearest-even).  For 16-bit types one instruction converts both.
template <typename T, int N>
__device__ __forceinline__ float2 get2(const Pack<T, N>& p, int i) {
  if constexpr (Pair2<T>::kPacked)
    return Pair2<T>::widen(reinterpret_cast<const typename Pair2<T>::type*>(p.v)[i]);
  else
    return make_float2(to_f32(p.v[2 * i]), to_f32(p.v[2 * i + 1]));
}

template <typename T, int N>
__device__ __forceinline__ void set2(Pack<T, N>& p, int i, float a, float b) {
  if constexpr (Pair2<T>::kPacked)
    reinterpret_cast<typename Pair2<T>::type*>(p.v)[i] = Pair2<T>::narrow(a, b);
  else {
    p.v[2 * i] = from_f32<T>(a);
    p.v[2 * i + 1] = from_f32<T>(b);
  }
}

// The residual sum at type T: binary32 (x + skip), then + bias when present,
// then one rounding to T.
template <typename T, bool HAS_BIAS>
__device__ __forceinline__ T residual_sum(T x, T skip, T bias) {
  float t = __fadd_rn(to_f32(x), to_f32(skip));
  if constexpr (HAS_BIAS) t = __fadd_rn(t, to_f32(bias));
  return from_f32<T>(t);
}

// SiLU in binary32: z * sigmoid(z) = z / (1 + e^-z), with e^-z written as
// 2^(-z * log2(e)) and evaluated by the hardware base-2 exponential, and the
// division by the hardware reciprocal (each a few ulp of binary32, far inside
// the output tolerance).  Flushing subnormals here is harmless: 2^(-z log2 e)
// is subnormal only for z > 87, where 1 + e^-z rounds to 1 anyway, and the
// reciprocal's argument is >= 1.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float silu_f32(float z) {
  constexpr float kLog2e = 1.4426950408889634f;
  return z * rcp_approx(1.0f + ex2_approx(-z * kLog2e));
}

// ---------------------------------------------------------------------------
// Reductions
// ---------------------------------------------------------------------------
// Butterfly sum over aligned segments of `width` lanes (width a power of two
// <= 32).  Every lane of a segment ends with the bitwise-identical total
// (each step adds the same two operands on both partners).
__device__ __forceinline__ float seg_sum(float v, int width) {
  for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the whole CTA; every thread returns the same value.  `red` is a
// shared array of at least 33 floats.  Fixed association order.
__device__ __forceinline__ float cta_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = (blockDim.x + 31) >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float t = lane < nwarps ? red[lane] : 0.0f;
    t = warp_sum(t);
    if (lane == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

// Two CTA-wide sums at once (one pair of barriers); `red` holds 33 float2.
__device__ __forceinline__ float2 cta_sum2(float2 v, float2* red) {
  v.x = warp_sum(v.x);
  v.y = warp_sum(v.y);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = (blockDim.x + 31) >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float2 t = lane < nwarps ? red[lane] : make_float2(0.0f, 0.0f);
    t.x = warp_sum(t.x);
    t.y = warp_sum(t.y);
    if (lane == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

// The same with one barrier: every thread adds the warps' partials itself, in
// warp order (the same bits in every thread).  `red` holds one float2 per
// warp; a later call on the same `red` needs a barrier between the two.
__device__ __forceinline__ float2 cta_sum2_1b(float2 v, float2* red) {
  v.x = warp_sum(v.x);
  v.y = warp_sum(v.y);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = (blockDim.x + 31) >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float2 t = make_float2(0.0f, 0.0f);
  for (int w = 0; w < nwarps; ++w) {
    const float2 u = red[w];
    t.x += u.x;
    t.y += u.y;
  }
  return t;
}

// ---------------------------------------------------------------------------
// Thread-block clusters (distributed shared memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ unsigned cluster_size() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Hardware cluster barrier: every thread of every CTA of the cluster arrives;
// release/acquire make shared (and global) writes before it visible after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Load a float that CTA `rank` of this cluster holds at the same shared
// address as `local` does here.
__device__ __forceinline__ float ld_cluster_f32(const float* local, unsigned rank) {
  unsigned addr = static_cast<unsigned>(__cvta_generic_to_shared(local));
  unsigned remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Load a float4 that CTA `rank` of this cluster holds at the same (16-byte
// aligned) shared address as `local` does here.
__device__ __forceinline__ float4 ld_cluster_f32x4(const float4* local, unsigned rank) {
  unsigned addr = static_cast<unsigned>(__cvta_generic_to_shared(local));
  unsigned remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote) : "memory");
  return v;
}

// Sum of one value per CTA over the cluster, in rank order (identical in every
// CTA).  `slot` is a shared float reserved for this call; the caller must
// cluster_sync() once more before any CTA of the cluster exits.
__device__ __forceinline__ float cluster_sum(float cta_value, float* slot, unsigned csize) {
  if (threadIdx.x == 0) *slot = cta_value;
  cluster_sync();
  float t = 0.0f;
  for (unsigned r = 0; r < csize; ++r) t += ld_cluster_f32(slot, r);
  return t;
}

// Two values per CTA summed over the cluster at once (one cluster barrier).
__device__ __forceinline__ float2 cluster_sum2(float2 cta_value, float* slot_x, float* slot_y,
                                               unsigned csize) {
  if (threadIdx.x == 0) {
    *slot_x = cta_value.x;
    *slot_y = cta_value.y;
  }
  cluster_sync();
  float2 t = make_float2(0.0f, 0.0f);
  for (unsigned r = 0; r < csize; ++r) {
    t.x += ld_cluster_f32(slot_x, r);
    t.y += ld_cluster_f32(slot_y, r);
  }
  return t;
}

// ---------------------------------------------------------------------------
// Moments: Chan et al.'s pairwise update of (count, mean, M2), M2 = sum of
// squared deviations from the mean.
// ---------------------------------------------------------------------------
struct Moments {
  float n, mean, m2;
};

__device__ __forceinline__ Moments merge(Moments a, Moments b) {
  if (b.n == 0.0f) return a;
  if (a.n == 0.0f) return b;
  const float n = a.n + b.n;
  const float d = b.mean - a.mean;
  const float fb = b.n / n;
  Moments r;
  r.n = n;
  r.mean = a.mean + d * fb;
  r.m2 = a.m2 + b.m2 + d * d * a.n * fb;
  return r;
}

// ---------------------------------------------------------------------------
// Bounded grid barrier (cooperative launches only: every CTA is resident).
// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel starts with pdl_wait(): when it
// was launched with programmatic stream serialization it may have been
// scheduled before the preceding grid on the stream finished, and the wait
// holds it (before any global load or store) until that grid has completed
// and its writes are visible.  Without that launch attribute the wait returns
// at once.  pdl_trigger() lets the next grid on the stream be scheduled once
// every CTA of this one has started (or exited); it does not release that
// grid's own pdl_wait() early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Control block at the start of a SkipGroupNorm workspace.
// Every counter is zero between calls (each call that uses one returns it to
// zero), so one workspace serves calls of any shape in turn.
constexpr int kL2MaxItems = 56;  // batch items of the NHWC L2 route
struct Control {
  unsigned int bar_count;  // CTAs arrived at the grid barrier (0 between launches)
  unsigned int bar_gen;    // CTAs that have left the grid barrier (0 between launches)
  unsigned int error;      // 0, or a b200norm_status recorded by a kernel
  unsigned int error_site; // which wait gave up
  unsigned int item_done[kL2MaxItems];  // NHWC L2 route: CTAs of item n done
};
static_assert(sizeof(Control) <= 256, "the control block is 256 bytes");

constexpr unsigned kStatusDeviceTimeout = 5;  // B200NORM_ERR_DEVICE_TIMEOUT

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void red_add_release_gpu(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// A grid barrier used once per launch, in three parts, so that a CTA can do
// work that no other CTA needs (stores of results only it reads) between its
// arrival and its wait.  Control::bar_count counts arrivals and
// Control::bar_gen departures; both are 0 before the launch, and the CTA that
// departs last puts them back to 0 at its end (every CTA has then left its
// wait), so the next launch finds them ready.
//
// grid_arrive publishes every thread's earlier writes to the CTAs that return
// from grid_wait (a release add; the waiters' acquire load reads the count the
// chain of adds produced).  grid_wait waits for `expected` arrivals; after
// `limit_ns` it records a timeout and returns false, and the caller must stop
// after calling grid_depart.  Every CTA of the grid takes a departure ticket
// in grid_wait, whether it timed out or not, and passes it (meaningful in
// thread 0) to grid_depart once it has finished, so that it does not wait for
// that atomic in between; the counts are reset even after a timeout, and the
// error stays recorded until the workspace is initialised again.
__device__ __forceinline__ void grid_arrive(Control* ctl) {
  __syncthreads();  // every thread's earlier writes are ordered before thread 0's release
  if (threadIdx.x == 0) red_add_release_gpu(&ctl->bar_count, 1u);
}

__device__ __forceinline__ bool grid_wait(Control* ctl, unsigned expected,
                                          unsigned long long limit_ns, unsigned site,
                                          unsigned& departure) {
  __shared__ int ok;
  if (threadIdx.x == 0) {
    ok = 1;
    const unsigned long long t0 = global_ns();
    while (ld_acquire_gpu(&ctl->bar_count) < expected) {
      if (global_ns() - t0 > limit_ns) {
        atomicExch(&ctl->error, kStatusDeviceTimeout);
        atomicExch(&ctl->error_site, site);
        ok = 0;
        break;
      }
    }
    departure = atomicAdd(&ctl->bar_gen, 1u);
  }
  __syncthreads();
  return ok != 0;
}

__device__ __forceinline__ void grid_depart(Control* ctl, unsigned departure) {
  if (threadIdx.x == 0 && departure == gridDim.x - 1u) {
    ctl->bar_count = 0u;
    ctl->bar_gen = 0u;
  }
}

}  // namespace b200norm
