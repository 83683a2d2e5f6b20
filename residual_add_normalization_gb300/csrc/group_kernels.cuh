// group_kernels.cuh -- SkipGroupNorm kernels (sm_103a), included by the
// per-element-type translation units group_f32.cu, group_f16.cu and
// group_bf16.cu, and by the planner in group_norm.cu.
//
// S = round_T((X + skip) + bias); Y = round_T(act((S - mean) * rstd * gamma[c] + beta[c]))
// with mean / population variance per (batch item n, group g) over the C/groups
// channels of g and every spatial position (com.microsoft.SkipGroupNorm README,
// Description).  Six routes:
//
//   1. NCHW resident.  A group instance (n, g) is one contiguous run of
//      cpg * H * W elements.  One CTA -- or a cluster of up to 16 CTAs for
//      long runs -- stages its share of S in shared memory: one HBM read,
//      statistics from sums taken while loading, one write.  Cluster pieces
//      are exchanged through distributed shared memory.
//   2. NHWC cooperative.  A group's elements are strided through the tensor
//      (cpg channels of every pixel), so statistics need every CTA that holds
//      a piece of the batch item.  One cooperative grid: each CTA holds a
//      slab of whole pixels in registers, takes its slab's per-group pieces,
//      publishes them, meets the other CTAs at one bounded grid barrier,
//      merges its batch item's pieces and normalizes what it holds.
//   3. Two-phase, any shape or layout.  Kernel A forms S over fixed chunks of
//      each group instance and writes per-chunk pieces; kernel B merges them
//      and re-forms S from the inputs to normalize (the re-read is an L2 hit
//      for anything that fits in L2).
//   4. NHWC through L2, two kernels: per-CTA pieces over pixel ranges, merged
//      by the last CTA of each batch item; then an apply kernel that re-forms
//      S from inputs still in L2.
//   5. Route 4's two passes in one cooperative grid with one grid barrier.
//   6. Route 2 with each CTA's slab in shared memory instead of registers,
//      for slabs larger than registers hold: bulk copies bring X (and a
//      full-shape skip) in, S is formed in place and one bulk store sends it
//      out while the grid barrier is pending.
//
// Statistics.  Every piece of a group instance that one CTA (or one cluster
// rank, or one chunk) sees is summarised as (n, R, mu, m2): n elements, a
// reference R near them (the mean of four of the piece's residual sums; the
// chunk's first residual sum in route 3, whose threads sum twice from
// registers anyway),
// mu = mean - R and m2 = the sum of squared deviations from the mean.  The
// sums of S - R and (S - R)^2 are taken while loading; if R turns out to be
// far from the piece's mean against its spread (an outlier among the four
// samples), the piece is summed again around R + mu from what the CTA holds
// (shared memory, registers, or L2).  Pieces then merge around a common centre
// Kc near the group mean, and every route carries the mean as Kc + d, so that
// (S - Kc) - d stays accurate in binary32 even when |mean| is large against
// the group's spread.
#pragma once

#include <cstring>

#include "bulk.cuh"
#include "common.cuh"
#include "launch.h"

namespace b200norm {

// Division by an invariant divisor as a multiply and a shift (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994):
// for 0 <= n < 2^31, n / d = (umulhi(n, m) + n) >> l with l = ceil(log2 d) and
// m = floor(2^32 * (2^l - d) / d) + 1.
struct FastDiv {
  unsigned m, l;
};

inline FastDiv make_fastdiv(unsigned d) {
  unsigned l = 0;
  while ((1ull << l) < d) ++l;
  FastDiv f;
  f.m = static_cast<unsigned>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
  f.l = l;
  return f;
}

__device__ __forceinline__ unsigned fdiv(unsigned n, FastDiv f) {
  return (__umulhi(n, f.m) + n) >> f.l;
}

template <typename T, typename M>
struct SgnArgs {
  const T* __restrict__ x;
  const T* __restrict__ skip;
  const T* __restrict__ bias;   // may be null
  const M* __restrict__ gamma;
  const M* __restrict__ beta;
  T* __restrict__ y;
  T* __restrict__ s;            // may be null
  int64_t N;
  int C, HW, cpg, groups;
  FastDiv cpg_div;              // division by cpg (channel -> group)
  int bcast;                    // skip holds one value per (n, c)
  int act;                      // 1: SiLU after the affine transform
  float eps;
  Control* ctl;                 // workspace control block
  float4* part;                 // workspace moment slots (n, mean, M2, -)
  unsigned long long limit_ns;  // bound of every cross-CTA wait
};

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s
constexpr int kCoopMaxThreads = 512;
constexpr int kTwoPhaseThreads = 256;
constexpr int kTwoPhaseEpt = kTwoPhaseChunk / kTwoPhaseThreads;

// S element at type T from binary32 x and skip, plus bias when present.
template <typename T>
__device__ __forceinline__ T sgn_sum(float x, float sk, const T* __restrict__ bias, int c) {
  float t = __fadd_rn(x, sk);
  if (bias) t = __fadd_rn(t, to_f32(bias[c]));
  return from_f32<T>(t);
}

// The same with the bias value already loaded (ignored when has_bias is
// false: then there is no add at all).
template <typename T>
__device__ __forceinline__ T sgn_sum_b(float x, float sk, float b, bool has_bias) {
  float t = __fadd_rn(x, sk);
  if (has_bias) t = __fadd_rn(t, b);
  return from_f32<T>(t);
}

// VE consecutive floats of shared memory at a 16-byte aligned address, read
// as 16-byte vectors where VE allows: threads that read VE floats apart meet
// far fewer bank conflicts than with VE scalar reads.
template <int VE>
__device__ __forceinline__ void lds_vec(const float* p, float (&out)[VE]) {
  if constexpr (VE % 4 == 0) {
#pragma unroll
    for (int i = 0; i < VE / 4; ++i) {
      const float4 v = reinterpret_cast<const float4*>(p)[i];
      out[4 * i] = v.x;
      out[4 * i + 1] = v.y;
      out[4 * i + 2] = v.z;
      out[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < VE; ++e) out[e] = p[e];
  }
}

// ((S - K) - d) * rstd * gamma + beta, then SiLU when requested.
__device__ __forceinline__ float sgn_out(float s, float K, float d, float rstd, float ga,
                                         float be, int act) {
  float z = ((s - K) - d) * rstd * ga + be;
  if (act) z = silu_f32(z);
  return z;
}

// Residual sum at (batch item n, channel c, pixel p), as binary32.
template <typename T, typename M>
__device__ __forceinline__ float sgn_at(const SgnArgs<T, M>& a, int64_t n, int c, int64_t p,
                                        bool cl) {
  const int64_t off = cl ? (n * a.HW + p) * a.C + c : (n * a.C + c) * a.HW + p;
  const float sk = a.bcast ? to_f32(a.skip[n * a.C + c]) : to_f32(a.skip[off]);
  return to_f32(sgn_sum<T>(to_f32(a.x[off]), sk, a.bias, c));
}

// ---------------------------------------------------------------------------
// Group statistics from pieces
// ---------------------------------------------------------------------------
// A piece is a float4 (n, R, mu, m2): n elements, reference R, mu = mean - R,
// m2 = sum of squared deviations from the mean.
//
// The one-pass variance s2/n - mu^2 (s1, s2 the sums of S - R and its square)
// carries a relative error of about eps * (1 + mu^2 / var); a piece with
// mu^2 > kIllCond * var is summed again around R + mu, so the variance keeps
// a relative error within ~16 binary32 accumulation errors.
constexpr float kIllCond = 15.0f;

// Reference of a piece: the mean of four of its residual sums (each scaled
// first, so the sum cannot overflow).  Data drawn from one distribution puts
// it within about half a standard deviation of the piece's mean.
__device__ __forceinline__ float ref4(float s0, float s1, float s2, float s3) {
  return (0.25f * s0 + 0.25f * s1) + (0.25f * s2 + 0.25f * s3);
}

// (Counts are whole numbers, so 1 / n from the hardware reciprocal is within
// an ulp; the statistics need nothing closer.)
__device__ __forceinline__ float4 piece_from_sums(float n, float R, float s1, float s2) {
  if (n == 0.0f) return make_float4(0.0f, R, 0.0f, 0.0f);
  const float mu = s1 * rcp_approx(n);
  return make_float4(n, R, mu, fmaxf(fmaf(-s1, mu, s2), 0.0f));
}

// Is the piece's one-pass variance too close to cancellation?  (False for
// NaN statistics: those propagate as they are.)
__device__ __forceinline__ bool piece_ill(float4 p) {
  return p.z * p.z * p.x > kIllCond * p.w;
}

// Pieces merged around a centre Kc: o = (R - Kc) + mu,
// N = sum n, s1 = sum n o, s2 = sum (m2 + n o^2); then d = s1 / N and
// var = (s2 - s1 d) / N.  With Kc within a few standard deviations of the
// mean (the first piece's mean, checked by merge_ill), nothing cancels.
struct MergeAcc {
  float n, s1, s2;
};

__device__ __forceinline__ void merge_add(MergeAcc& m, float4 p, float Kc) {
  const float o = (p.y - Kc) + p.z;
  const float no = p.x * o;
  m.n += p.x;
  m.s1 += no;
  m.s2 += fmaf(no, o, p.w);
}

__device__ __forceinline__ void merge_add(MergeAcc& m, MergeAcc b) {
  m.n += b.n;
  m.s1 += b.s1;
  m.s2 += b.s2;
}

// An accumulation around Kq, given as (Kq, n, s1, s2), moved to the centre
// Kc and added: with dl = Kq - Kc, s1 + n dl and s2 + dl (2 s1 + n dl)
// (exact algebra; nothing cancels while Kq is within the spread of the data
// it summarises).
__device__ __forceinline__ void merge_add_moved(MergeAcc& m, float4 q, float Kc) {
  const float dl = q.x - Kc;
  m.n += q.y;
  m.s1 += fmaf(q.y, dl, q.z);
  m.s2 += fmaf(dl, fmaf(q.y, dl, 2.0f * q.z), q.w);
}

// Group statistics: mean = K + d, population variance var.
struct GStats {
  float K, d, var;
};

__device__ __forceinline__ GStats merge_finish(MergeAcc m, float Kc) {
  const float r = rcp_approx(m.n);
  const float d = m.s1 * r;
  return GStats{Kc, d, fmaxf(fmaf(-m.s1, d, m.s2), 0.0f) * r};
}

__device__ __forceinline__ bool merge_ill(GStats s) { return s.d * s.d > kIllCond * s.var; }


// Statistics of a single piece.
__device__ __forceinline__ GStats piece_stats(float4 p) {
  return GStats{p.y, p.z, p.w * rcp_approx(p.x)};
}

__device__ __forceinline__ float piece_mean(float4 p) { return p.y + p.z; }

// Group g's statistics from B pieces in global memory (piece b at
// part[b * stride + g]), merged afresh: the rare path of the chunked merges,
// kept out of line so that it costs the common path no registers.
static __device__ __noinline__ GStats merge_pieces_global(const float4* part, int64_t stride, int g,
                                                          int B);

// B pieces get(0..B-1), merged in that order around the first piece's mean;
// merged again around the new mean while that is far from the result (at most
// twice more).
template <class Get>
__device__ __forceinline__ GStats merge_pieces(int B, Get get) {
  float Kc = piece_mean(get(0));
  GStats s{};
  for (int round = 0; round < 3; ++round) {
    MergeAcc m{0.0f, 0.0f, 0.0f};
    for (int b = 0; b < B; ++b) merge_add(m, get(b), Kc);
    s = merge_finish(m, Kc);
    if (!merge_ill(s)) break;
    Kc = Kc + s.d;
  }
  return s;
}

static __device__ __noinline__ GStats merge_pieces_global(const float4* part, int64_t stride, int g,
                                                          int B) {
  return merge_pieces(B, [&](int b) { return __ldcg(part + static_cast<int64_t>(b) * stride + g); });
}

// ---------------------------------------------------------------------------
// Route 1: NCHW, one CTA or cluster per group instance, S staged in shared
// memory
// ---------------------------------------------------------------------------
// A group instance (n, g) is the contiguous run of L = cpg * H * W elements at
// (n*C + g*cpg) * H*W.  CTA rank r of the instance's cluster takes vectors
// [r * span, (r + 1) * span) of it: it loads X (+ skip), forms S, keeps S in
// shared memory (span vectors of dynamic shared memory) and accumulates the
// sums of S - R and (S - R)^2 on the way (R the mean of four residual sums of
// its range); its piece (n, R, mu, m2) is summed again from shared memory
// when R was far from the range's mean.  A cluster's pieces meet through
// DSMEM and every CTA merges them in rank order.
// VE > 1 needs H*W % VE == 0 so that a vector never straddles two channels;
// vpc = H*W / VE vectors per channel.
#ifndef B200NORM_NCHW_UNROLL
#define B200NORM_NCHW_UNROLL 2   // vectors per thread in flight while loading (measured)
#endif
#ifndef B200NORM_NCHW_MINB
#define B200NORM_NCHW_MINB 4     // resident CTAs per SM the registers allow
#endif
#ifndef B200NORM_NCHW_THREADS
#define B200NORM_NCHW_THREADS 256
#endif
constexpr int kNchwThreads = B200NORM_NCHW_THREADS;
constexpr int kNchwUnroll = B200NORM_NCHW_UNROLL;

// Byte offset of route 1's gamma / beta table in dynamic shared memory: past
// `span` vectors of S, rounded up to 16 bytes.
__host__ __device__ constexpr size_t nchw_gb_offset(int span, size_t vbytes) {
  return (static_cast<size_t>(span) * vbytes + 15) & ~static_cast<size_t>(15);
}

template <typename T, typename M, int VE>
__global__ void __launch_bounds__(kNchwThreads, B200NORM_NCHW_MINB)
sgn_nchw_smem(const SgnArgs<T, M> a, int span, FastDiv vpc) {
  pdl_wait();
  pdl_trigger();
  using P = Pack<T, VE>;
  extern __shared__ float4 smem4[];
  P* sb = reinterpret_cast<P*>(smem4);
  __shared__ float2 red2[kNchwThreads / 32];
  __shared__ float4 slot_piece;  // this CTA's piece, read by the cluster's CTAs
  const unsigned csize = cluster_size();
  const unsigned rank = csize > 1 ? cluster_rank() : 0u;
  const int64_t inst = blockIdx.x / csize;
  const int64_t n = inst / a.groups;
  const int g = static_cast<int>(inst % a.groups);
  const int L = a.cpg * a.HW;
  const int v0 = static_cast<int>(rank) * span;
  const int cnt = min(span, L / VE - v0);  // may be <= 0 for trailing ranks
  const int64_t base = (n * a.C + static_cast<int64_t>(g) * a.cpg) * a.HW + static_cast<int64_t>(v0) * VE;
  const int cbase = g * a.cpg;
  // gamma and beta of the channels this CTA touches, loaded now and staged in
  // shared memory (after S, at the next 16-byte boundary: a scalar-path S
  // can end anywhere) before the reduction's barrier, so that the output
  // loop does not wait for them
  float2* s_gb = reinterpret_cast<float2*>(reinterpret_cast<char*>(smem4) +
                                           nchw_gb_offset(span, sizeof(P)));
  const int c_lo = cnt > 0 ? cbase + static_cast<int>(fdiv(static_cast<unsigned>(v0), vpc)) : 0;
  const int nch = cnt > 0 ? cbase + static_cast<int>(fdiv(static_cast<unsigned>(v0 + cnt - 1), vpc)) - c_lo + 1 : 0;
  float2 gb = make_float2(0.0f, 0.0f);
  if (static_cast<int>(threadIdx.x) < nch)
    gb = make_float2(to_f32(a.gamma[c_lo + threadIdx.x]), to_f32(a.beta[c_lo + threadIdx.x]));

  // reference R: four residual sums spread over this CTA's range; threads
  // that hold vectors take it right behind their first loads
  auto range_ref = [&]() {
    const int len = cnt * VE;
    float smp[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = v0 * VE + q * (len / 4);  // element of the instance
      smp[q] = sgn_at(a, n, cbase + j / a.HW, j % a.HW, false);
    }
    return ref4(smp[0], smp[1], smp[2], smp[3]);
  };
  float sum = 0.0f, sq = 0.0f;
  float R = 0.0f;
  if (static_cast<int>(threadIdx.x) >= cnt && cnt > 0) R = range_ref();
  for (int i0 = threadIdx.x; i0 < cnt; i0 += kNchwThreads * kNchwUnroll) {
    P xv[kNchwUnroll], kv[kNchwUnroll];
#pragma unroll
    for (int u = 0; u < kNchwUnroll; ++u) {
      const int i = i0 + u * kNchwThreads;
      if (i < cnt) {
        xv[u] = ld_stream<T, VE>(a.x + base + static_cast<int64_t>(i) * VE);
        if (!a.bcast) kv[u] = ld_stream<T, VE>(a.skip + base + static_cast<int64_t>(i) * VE);
      }
    }
    if (i0 == static_cast<int>(threadIdx.x)) R = range_ref();
#pragma unroll
    for (int u = 0; u < kNchwUnroll; ++u) {
      const int i = i0 + u * kNchwThreads;
      if (i < cnt) {
        const int c = cbase + static_cast<int>(fdiv(static_cast<unsigned>(v0 + i), vpc));
        const float skb = a.bcast ? to_f32(a.skip[n * a.C + c]) : 0.0f;
        P sv;
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float sk = a.bcast ? skb : to_f32(kv[u].v[e]);
          sv.v[e] = sgn_sum<T>(to_f32(xv[u].v[e]), sk, a.bias, c);
          const float d = to_f32(sv.v[e]) - R;
          sum += d;
          sq = fmaf(d, d, sq);
        }
        sb[i] = sv;
        if (a.s) st_stream<T, VE>(a.s + base + static_cast<int64_t>(i) * VE, sv);
      }
    }
  }
  // this CTA's piece; summed again from shared memory around R + mu when R
  // was far from the piece's mean (every thread holds the same sums, so the
  // branch is uniform)
  const float n_cta = static_cast<float>(max(cnt, 0) * VE);
  if (static_cast<int>(threadIdx.x) < nch) s_gb[threadIdx.x] = gb;  // published by the barrier below
  float2 t2 = cta_sum2_1b(make_float2(sum, sq), red2);
  float4 piece = piece_from_sums(n_cta, R, t2.x, t2.y);
  if (piece_ill(piece)) {
    const float R2 = R + piece.z;
    float s1 = 0.0f, s2 = 0.0f;
    for (int i = threadIdx.x; i < cnt; i += kNchwThreads) {
      const P sv = sb[i];
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        const float d = to_f32(sv.v[e]) - R2;
        s1 += d;
        s2 = fmaf(d, d, s2);
      }
    }
    __syncthreads();  // every thread has read red2 (one-barrier sums)
    t2 = cta_sum2_1b(make_float2(s1, s2), red2);
    piece = piece_from_sums(n_cta, R2, t2.x, t2.y);
  }
  GStats st;
  if (csize > 1) {
    // the cluster's pieces, merged in rank order by every CTA (same bits)
    if (threadIdx.x == 0) slot_piece = piece;
    cluster_sync();
    st = merge_pieces(static_cast<int>(csize),
                      [&](int r) { return ld_cluster_f32x4(&slot_piece, static_cast<unsigned>(r)); });
  } else {
    st = piece_stats(piece);
  }
  const float rstd = rsqrtf(st.var + a.eps);
  for (int i = threadIdx.x; i < cnt; i += kNchwThreads) {
    const int c = cbase + static_cast<int>(fdiv(static_cast<unsigned>(v0 + i), vpc));
    const float2 gbc = s_gb[c - c_lo];
    const float ga = gbc.x, be = gbc.y;
    const P sv = sb[i];
    P out;
#pragma unroll
    for (int e = 0; e < VE; ++e)
      out.v[e] = from_f32<T>(sgn_out(to_f32(sv.v[e]), st.K, st.d, rstd, ga, be, a.act));
    st_stream<T, VE>(a.y + base + static_cast<int64_t>(i) * VE, out);
  }
  if (csize > 1) cluster_sync();  // peers may still read slot_piece
}

// ---------------------------------------------------------------------------
// Route 2: NHWC, cooperative grid with one bounded grid barrier
// ---------------------------------------------------------------------------
// blockDim.x = CV * PL with CV = C / VE vectors per pixel: thread t covers the
// VE channels (t % CV) * VE .. +VE of pixels p0 + t / CV + k * PL, k < NV.
// CTA b handles batch item b / B, pixels [(b % B) * ppc, +ppc).
// Every CTA takes, per group, the piece (count, R, mu, m2) of the S it holds:
// sums of S - R[g] and (S - R[g])^2 per thread, pixel lane and channel, then
// per group (R[g] the mean of four residual sums of the CTA's pixels in group
// g); groups whose R was far from their mean are summed again from the
// registers.  It stores S between its arrival at the grid barrier and its
// wait.  After the barrier each CTA merges its batch item's B pieces per
// group in a fixed order (chunks of pieces, then the chunks), and stores Y.
// Dynamic shared memory (floats), layout given by k_offset:
//   pieces:  acc[2][PL*C] | col[2][C]
//   merge:   chunk pieces[nchunk*groups] (float4) | centre K[groups] |
//            offset d[groups] | rstd[groups]
//   tail at k_offset, kept throughout: R[groups] | second-round R[groups]
//            (padded to 16 bytes) | gamma[C] | beta[C]
// Each thread loads its own NV vectors of X (and skip) with streaming 16-byte
// loads, all issued before the first is used.  (A bulk copy of the CTA's slab
// into shared memory, which route 6 uses, was slower here with the inputs in
// HBM: 10.1 against 9.9 us per call on the NHWC fp16 workload, and no faster
// when issued earlier or split into 4 or 8 copies; it wins only when the
// inputs are already in L2.)
constexpr int kCoopMergeChunk = 8;

// Bytes of route 6's slab area: the mbarrier, then the S slab and (full skip)
// the skip slab of ppc pixels of C elements of `es` bytes.
__host__ __device__ constexpr size_t coop_slab_bytes(int ppc, int C, size_t es, bool bcast) {
  return 16 + static_cast<size_t>(ppc) * C * es * (bcast ? 1 : 2);
}

// Floats of route 2's shared-memory tail before gamma (16-byte aligned).
__host__ __device__ constexpr int coop_tail_floats(int groups) { return (2 * groups + 3) & ~3; }

// Element q of the four residual sums that give group g's reference over
// pixels [p0, p1) of batch item n (NHWC): pixel p0 + q * (p1 - p0) / 4,
// channel g * cpg + q * cpg / 4.
template <typename T, typename M>
__device__ __forceinline__ float nhwc_sample(const SgnArgs<T, M>& a, int n, int g, int q, int p0,
                                             int p1) {
  const int p = p0 + q * ((p1 - p0) / 4);
  const int c = g * a.cpg + (q * a.cpg) / 4;
  return sgn_at(a, n, c, p, true);
}

// Group g's reference over pixels [p0, p1) of batch item n (NHWC).
template <typename T, typename M>
__device__ __forceinline__ float nhwc_ref(const SgnArgs<T, M>& a, int n, int g, int p0, int p1) {
  return ref4(nhwc_sample(a, n, g, 0, p0, p1), nhwc_sample(a, n, g, 1, p0, p1),
              nhwc_sample(a, n, g, 2, p0, p1), nhwc_sample(a, n, g, 3, p0, p1));
}

template <typename T, typename M, int VE, int NV>
__global__ void __launch_bounds__(kCoopMaxThreads, 1)
sgn_nhwc_coop(const SgnArgs<T, M> a, int B, int ppc, int k_offset) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  float* s_R0 = smem + k_offset;
  float* s_R = s_R0 + a.groups;
  __shared__ int s_again;
  const int C = a.C;
  const int CV = C / VE;
  const int PL = blockDim.x / CV;
  const int tc = threadIdx.x % CV;
  const int tp = threadIdx.x / CV;
  const int n = blockIdx.x / B;
  const int p0 = (blockIdx.x % B) * ppc;
  const int p1 = min(p0 + ppc, a.HW);
  const int64_t nbase = static_cast<int64_t>(n) * a.HW * C;
  const int c0 = tc * VE;

  // --- load and form S (stored while the grid barrier is pending) ----------
  Pack<T, VE> xv[NV], kv[NV], sv[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int p = p0 + tp + k * PL;
    if (p < p1) {
      const int64_t off = nbase + static_cast<int64_t>(p) * C + c0;
      xv[k] = ld_stream<T, VE>(a.x + off);
      if (!a.bcast) kv[k] = ld_stream<T, VE>(a.skip + off);
    }
  }
  Pack<T, VE> skb, bv;
  if (a.bcast) skb = ld_reuse<T, VE>(a.skip + static_cast<int64_t>(n) * C + c0);
  if (a.bias) bv = ld_reuse<T, VE>(a.bias + c0);
  // the affine weights are needed only at the end: stage them now
  float* s_ga = s_R0 + coop_tail_floats(a.groups);  // 16-byte aligned
  float* s_be = s_ga + C;
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    s_ga[c] = to_f32(__ldg(a.gamma + c));
    s_be[c] = to_f32(__ldg(a.beta + c));
  }
  for (int gg = threadIdx.x; gg < a.groups; gg += blockDim.x) s_R0[gg] = nhwc_ref(a, n, gg, p0, p1);
  if (threadIdx.x == 0) s_again = 0;
  __syncthreads();
  float Kl[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) Kl[e] = s_R0[fdiv(c0 + e, a.cpg_div)];
  float lsum[VE], lsq[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) lsum[e] = lsq[e] = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int p = p0 + tp + k * PL;
    if (p < p1) {
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        const float sk = a.bcast ? to_f32(skb.v[e]) : to_f32(kv[k].v[e]);
        sv[k].v[e] = sgn_sum_b<T>(to_f32(xv[k].v[e]), sk, to_f32(bv.v[e]), a.bias != nullptr);
        const float d = to_f32(sv[k].v[e]) - Kl[e];
        lsum[e] += d;
        lsq[e] = fmaf(d, d, lsq[e]);
      }
    }
  }
  // --- this CTA's pieces, per group ----------------------------------------
  // acc is laid out [q][e][tp][tc] so that the stores of a warp hit distinct
  // banks; col is [q][C].  A second round (from the registers, around
  // R + mu) runs only when some group's R was far from its mean.
  float* s_acc = smem;
  float* s_col = smem + 2 * PL * C;
  const int nthr = PL * CV;
  const float n_cta = static_cast<float>(p1 - p0) * static_cast<float>(a.cpg);
  for (int round = 0; round < 2; ++round) {
    if (round == 1) {
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        Kl[e] = s_R[fdiv(c0 + e, a.cpg_div)];
        lsum[e] = lsq[e] = 0.0f;
      }
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (p0 + tp + k * PL < p1) {
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            const float d = to_f32(sv[k].v[e]) - Kl[e];
            lsum[e] += d;
            lsq[e] = fmaf(d, d, lsq[e]);
          }
        }
      }
    }
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      s_acc[(e * PL + tp) * CV + tc] = lsum[e];
      s_acc[nthr * VE + (e * PL + tp) * CV + tc] = lsq[e];
    }
    __syncthreads();
    for (int j = threadIdx.x; j < C; j += blockDim.x) {
      const int e = j / CV, q0 = j % CV;
      float t1 = 0.0f, t2 = 0.0f;
      for (int q = 0; q < PL; ++q) {
        t1 += s_acc[(e * PL + q) * CV + q0];
        t2 += s_acc[nthr * VE + (e * PL + q) * CV + q0];
      }
      s_col[q0 * VE + e] = t1;
      s_col[C + q0 * VE + e] = t2;
    }
    __syncthreads();
    for (int gg = threadIdx.x; gg < a.groups; gg += blockDim.x) {
      float t1 = 0.0f, t2 = 0.0f;
      for (int cc = 0; cc < a.cpg; ++cc) {
        t1 += s_col[gg * a.cpg + cc];
        t2 += s_col[C + gg * a.cpg + cc];
      }
      const float R = round == 0 ? s_R0[gg] : s_R[gg];
      const float4 piece = piece_from_sums(n_cta, R, t1, t2);
      a.part[static_cast<int64_t>(blockIdx.x) * a.groups + gg] = piece;
      if (round == 0) {
        s_R[gg] = R + piece.z;
        if (piece_ill(piece)) s_again = 1;
      }
    }
    __syncthreads();
    if (!s_again) break;
  }
  // the arrival's release (after a CTA barrier) publishes these pieces; S,
  // which no other CTA reads, is stored while the other CTAs arrive
  grid_arrive(a.ctl);
  if (a.s) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int p = p0 + tp + k * PL;
      if (p < p1) st_stream<T, VE>(a.s + nbase + static_cast<int64_t>(p) * C + c0, sv[k]);
    }
  }
  unsigned departure = 0u;
  if (!grid_wait(a.ctl, gridDim.x, a.limit_ns, 1u, departure)) {
    grid_depart(a.ctl, departure);
    return;
  }

  // --- merge the batch item's B pieces per group in a fixed order (every CTA
  // of the item gets the same bits): chunks of kCoopMergeChunk pieces, each
  // summed around its first piece's mean Kq (all loads of a chunk issued
  // before they are added) and kept as (Kq, n, s1, s2); then the chunks,
  // moved to the first chunk's Kq ---------------------------------------------
  const int nchunk = (B + kCoopMergeChunk - 1) / kCoopMergeChunk;
  float4* s_cp = reinterpret_cast<float4*>(smem);      // nchunk * groups
  float* s_gK = smem + nchunk * a.groups * 4;
  float* s_gd = s_gK + a.groups;
  float* s_grstd = s_gd + a.groups;
  const float4* src = a.part + static_cast<int64_t>(n) * B * a.groups;
  for (int idx = threadIdx.x; idx < nchunk * a.groups; idx += blockDim.x) {
    const int gg = idx % a.groups, q = idx / a.groups;
    const int b0 = q * kCoopMergeChunk;
    float4 u[kCoopMergeChunk];
#pragma unroll
    for (int j = 0; j < kCoopMergeChunk; ++j)
      if (b0 + j < B) u[j] = __ldcg(src + static_cast<int64_t>(b0 + j) * a.groups + gg);
    const float Kq = piece_mean(u[0]);
    MergeAcc m{0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < kCoopMergeChunk; ++j)
      if (b0 + j < B) merge_add(m, u[j], Kq);
    s_cp[idx] = make_float4(Kq, m.n, m.s1, m.s2);
  }
  __syncthreads();
  for (int gg = threadIdx.x; gg < a.groups; gg += blockDim.x) {
    const float Kc = s_cp[gg].x;
    MergeAcc m{0.0f, 0.0f, 0.0f};
    for (int q = 0; q < nchunk; ++q) merge_add_moved(m, s_cp[q * a.groups + gg], Kc);
    GStats st = merge_finish(m, Kc);
    if (merge_ill(st))  // pathological spread of the pieces: merge them all afresh
      st = merge_pieces_global(src, a.groups, gg, B);
    s_gK[gg] = st.K;
    s_gd[gg] = st.d;
    s_grstd[gg] = rsqrtf(st.var + a.eps);
  }
  __syncthreads();
  // --- normalize what this thread holds; store Y ---------------------------
  float Kg[VE], mu[VE], rs[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) {
    const unsigned ge = fdiv(c0 + e, a.cpg_div);
    Kg[e] = s_gK[ge];
    mu[e] = s_gd[ge];
    rs[e] = s_grstd[ge];
  }
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int p = p0 + tp + k * PL;
    if (p < p1) {
      const int64_t off = nbase + static_cast<int64_t>(p) * C + c0;
      float ga[VE], be[VE];
      lds_vec<VE>(s_ga + c0, ga);
      lds_vec<VE>(s_be + c0, be);
      Pack<T, VE> out;
#pragma unroll
      for (int e = 0; e < VE; ++e)
        out.v[e] = from_f32<T>(sgn_out(to_f32(sv[k].v[e]), Kg[e], mu[e], rs[e], ga[e], be[e],
                                       a.act));
      st_stream<T, VE>(a.y + off, out);
    }
  }
  grid_depart(a.ctl, departure);
}

// ---------------------------------------------------------------------------
// Route 6: NHWC, cooperative grid, the CTA's slab resident in shared memory
// ---------------------------------------------------------------------------
// Route 2's pixel ranges, pieces, bounded grid barrier and merge, but the
// CTA's slab of X -- and its S, formed in place -- lives in shared memory
// rather than registers, so a slab may hold as many pixels as shared memory
// takes (route 2: at most eight per thread) and nothing is read twice from
// HBM or L2.  With 16-byte vectors the slab (and a full-shape skip's) comes
// in by bulk copies and S goes back out by one bulk store, issued between the
// CTA's arrival at the grid barrier and its wait; otherwise every thread
// moves its own vectors.
// Dynamic shared memory: route 2's pieces / merge area and tail (up to the
// end of beta), then the copy's mbarrier (16 bytes) | S slab [ppc][C] |
// (full-shape skip) skip slab [ppc][C].
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from this CTA's shared memory to global memory, as one bulk async-group.
__device__ __forceinline__ void bulk_store_group(void* dst, const void* src, unsigned bytes) {
  asm volatile(
      "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\t"
      "cp.async.bulk.commit_group;"
      :: "l"(dst), "r"(smem_addr(src)), "r"(bytes) : "memory");
}

// Waits until every bulk store of this thread has read its shared memory.
__device__ __forceinline__ void bulk_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

template <typename T, typename M, int VE>
__global__ void __launch_bounds__(kCoopMaxThreads, 1)
sgn_nhwc_slab(const SgnArgs<T, M> a, int B, int ppc, int k_offset) {
  pdl_wait();
  pdl_trigger();
  using P = Pack<T, VE>;
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  float* s_R0 = smem + k_offset;
  float* s_R = s_R0 + a.groups;
  __shared__ int s_again;
  const int C = a.C;
  const int CV = C / VE;
  const int PL = blockDim.x / CV;
  const int tc = threadIdx.x % CV;
  const int tp = threadIdx.x / CV;
  const int n = blockIdx.x / B;
  const int p0 = (blockIdx.x % B) * ppc;
  const int p1 = min(p0 + ppc, a.HW);
  const int np = p1 - p0;
  const int64_t nbase = static_cast<int64_t>(n) * a.HW * C;
  const int c0 = tc * VE;
  constexpr bool kBulk = VE * sizeof(T) == 16;
  float* s_ga = s_R0 + coop_tail_floats(a.groups);  // 16-byte aligned
  float* s_be = s_ga + C;
  unsigned long long* s_bar = reinterpret_cast<unsigned long long*>(s_be + C);
  P* s_S = reinterpret_cast<P*>(s_bar + 2);             // [ppc][CV]: X, then S
  P* s_K = s_S + static_cast<int64_t>(ppc) * CV;       // [ppc][CV]: full-shape skip
  const unsigned slab = static_cast<unsigned>(np) * static_cast<unsigned>(C) * sizeof(T);

  // --- the slab into shared memory ------------------------------------------
  if constexpr (kBulk) {
    if (threadIdx.x == 0) {
      mbar_init(s_bar, 1u);
      mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      const int64_t at = nbase + static_cast<int64_t>(p0) * C;
      mbar_arrive_expect_tx(s_bar, a.bcast ? slab : 2u * slab);
      bulk_load(s_S, a.x + at, slab, s_bar);
      if (!a.bcast) bulk_load(s_K, a.skip + at, slab, s_bar);
    }
  } else {
    for (int q = tp; q < np; q += PL) {
      const int64_t off = nbase + static_cast<int64_t>(p0 + q) * C + c0;
      s_S[q * CV + tc] = ld_stream<T, VE>(a.x + off);
      if (!a.bcast) s_K[q * CV + tc] = ld_stream<T, VE>(a.skip + off);
    }
  }
  P skb, bv;
  if (a.bcast) skb = ld_reuse<T, VE>(a.skip + static_cast<int64_t>(n) * C + c0);
  if (a.bias) bv = ld_reuse<T, VE>(a.bias + c0);
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    s_ga[c] = to_f32(__ldg(a.gamma + c));
    s_be[c] = to_f32(__ldg(a.beta + c));
  }
  for (int gg = threadIdx.x; gg < a.groups; gg += blockDim.x) s_R0[gg] = nhwc_ref(a, n, gg, p0, p1);
  if (threadIdx.x == 0) s_again = 0;
  __syncthreads();
  bool landed = true;
  if constexpr (kBulk) {
    // a copy that has not landed within the limit is recorded and the CTA
    // carries on (its outputs are then undefined) so that the grid barrier
    // still completes; it waits for the copy again before it leaves
    landed = mbar_wait(s_bar, 0u, a.limit_ns);
    if (!landed) {
      atomicExch(&a.ctl->error, kStatusDeviceTimeout);
      atomicExch(&a.ctl->error_site, 6u);
    }
  }

  // --- S in place, and the sums of S - R and (S - R)^2 ----------------------
  float Kl[VE], lsum[VE], lsq[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) {
    Kl[e] = s_R0[fdiv(c0 + e, a.cpg_div)];
    lsum[e] = lsq[e] = 0.0f;
  }
#pragma unroll 2
  for (int q = tp; q < np; q += PL) {
    const P xv = s_S[q * CV + tc];
    P kv;
    if (!a.bcast) kv = s_K[q * CV + tc];
    P sv;
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      const float sk = a.bcast ? to_f32(skb.v[e]) : to_f32(kv.v[e]);
      sv.v[e] = sgn_sum_b<T>(to_f32(xv.v[e]), sk, to_f32(bv.v[e]), a.bias != nullptr);
      const float d = to_f32(sv.v[e]) - Kl[e];
      lsum[e] += d;
      lsq[e] = fmaf(d, d, lsq[e]);
    }
    s_S[q * CV + tc] = sv;
  }

  // --- this CTA's pieces, per group (route 2's combine; a second round
  // re-reads S from shared memory) --------------------------------------------
  float* s_acc = smem;
  float* s_col = smem + 2 * PL * C;
  const int nthr = PL * CV;
  const float n_cta = static_cast<float>(np) * static_cast<float>(a.cpg);
  for (int round = 0; round < 2; ++round) {
    if (round == 1) {
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        Kl[e] = s_R[fdiv(c0 + e, a.cpg_div)];
        lsum[e] = lsq[e] = 0.0f;
      }
      for (int q = tp; q < np; q += PL) {
        const P sv = s_S[q * CV + tc];
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float d = to_f32(sv.v[e]) - Kl[e];
          lsum[e] += d;
          lsq[e] = fmaf(d, d, lsq[e]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      s_acc[(e * PL + tp) * CV + tc] = lsum[e];
      s_acc[nthr * VE + (e * PL + tp) * CV + tc] = lsq[e];
    }
    __syncthreads();
    for (int j = threadIdx.x; j < C; j += blockDim.x) {
      const int e = j / CV, q0 = j % CV;
      float t1 = 0.0f, t2 = 0.0f;
      for (int q = 0; q < PL; ++q) {
        t1 += s_acc[(e * PL + q) * CV + q0];
        t2 += s_acc[nthr * VE + (e * PL + q) * CV + q0];
      }
      s_col[q0 * VE + e] = t1;
      s_col[C + q0 * VE + e] = t2;
    }
    __syncthreads();
    for (int gg = threadIdx.x; gg < a.groups; gg += blockDim.x) {
      float t1 = 0.0f, t2 = 0.0f;
      for (int cc = 0; cc < a.cpg; ++cc) {
        t1 += s_col[gg * a.cpg + cc];
        t2 += s_col[C + gg * a.cpg + cc];
      }
      const float R = round == 0 ? s_R0[gg] : s_R[gg];
      const float4 piece = piece_from_sums(n_cta, R, t1, t2);
      a.part[static_cast<int64_t>(blockIdx.x) * a.groups + gg] = piece;
      if (round == 0) {
        s_R[gg] = R + piece.z;
        if (piece_ill(piece)) s_again = 1;
      }
    }
    __syncthreads();
    if (!s_again) break;
  }
  // S out while the other CTAs arrive: with bulk copies one bulk store of the
  // slab (its writers make their shared-memory writes visible to the copy
  // engine before the arrival's barrier)
  if (kBulk && a.s) fence_proxy_async_smem();
  grid_arrive(a.ctl);
  if (a.s) {
    if constexpr (kBulk) {
      if (threadIdx.x == 0) bulk_store_group(a.s + nbase + static_cast<int64_t>(p0) * C, s_S, slab);
    } else {
      for (int q = tp; q < np; q += PL)
        st_stream<T, VE>(a.s + nbase + static_cast<int64_t>(p0 + q) * C + c0, s_S[q * CV + tc]);
    }
  }
  unsigned departure = 0u;
  if (!grid_wait(a.ctl, gridDim.x, a.limit_ns, 6u, departure)) {
    if (kBulk && threadIdx.x == 0) {
      if (!landed) mbar_wait(s_bar, 0u, a.limit_ns);
      if (a.s) bulk_store_wait_read();
    }
    grid_depart(a.ctl, departure);
    return;
  }

  // --- merge the batch item's B pieces per group (route 2's merge) ----------
  const int nchunk = (B + kCoopMergeChunk - 1) / kCoopMergeChunk;
  float4* s_cp = reinterpret_cast<float4*>(smem);      // nchunk * groups
  float* s_gK = smem + nchunk * a.groups * 4;
  float* s_gd = s_gK + a.groups;
  float* s_grstd = s_gd + a.groups;
  const float4* src = a.part + static_cast<int64_t>(n) * B * a.groups;
  for (int idx = threadIdx.x; idx < nchunk * a.groups; idx += blockDim.x) {
    const int gg = idx % a.groups, q = idx / a.groups;
    const int b0 = q * kCoopMergeChunk;
    float4 u[kCoopMergeChunk];
#pragma unroll
    for (int j = 0; j < kCoopMergeChunk; ++j)
      if (b0 + j < B) u[j] = __ldcg(src + static_cast<int64_t>(b0 + j) * a.groups + gg);
    const float Kq = piece_mean(u[0]);
    MergeAcc m{0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < kCoopMergeChunk; ++j)
      if (b0 + j < B) merge_add(m, u[j], Kq);
    s_cp[idx] = make_float4(Kq, m.n, m.s1, m.s2);
  }
  __syncthreads();
  for (int gg = threadIdx.x; gg < a.groups; gg += blockDim.x) {
    const float Kc = s_cp[gg].x;
    MergeAcc m{0.0f, 0.0f, 0.0f};
    for (int q = 0; q < nchunk; ++q) merge_add_moved(m, s_cp[q * a.groups + gg], Kc);
    GStats st = merge_finish(m, Kc);
    if (merge_ill(st))  // pathological spread of the pieces: merge them all afresh
      st = merge_pieces_global(src, a.groups, gg, B);
    s_gK[gg] = st.K;
    s_gd[gg] = st.d;
    s_grstd[gg] = rsqrtf(st.var + a.eps);
  }
  __syncthreads();
  // --- normalize the slab; store Y ------------------------------------------
  float Kg[VE], mu[VE], rs[VE], ga[VE], be[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) {
    const unsigned ge = fdiv(c0 + e, a.cpg_div);
    Kg[e] = s_gK[ge];
    mu[e] = s_gd[ge];
    rs[e] = s_grstd[ge];
  }
  lds_vec<VE>(s_ga + c0, ga);
  lds_vec<VE>(s_be + c0, be);
#pragma unroll 2
  for (int q = tp; q < np; q += PL) {
    const P sv = s_S[q * CV + tc];
    P out;
#pragma unroll
    for (int e = 0; e < VE; ++e)
      out.v[e] = from_f32<T>(sgn_out(to_f32(sv.v[e]), Kg[e], mu[e], rs[e], ga[e], be[e], a.act));
    st_stream<T, VE>(a.y + nbase + static_cast<int64_t>(p0 + q) * C + c0, out);
  }
  if (kBulk && threadIdx.x == 0) {
    if (!landed) mbar_wait(s_bar, 0u, a.limit_ns);
    if (a.s) bulk_store_wait_read();  // the S store has read the slab
  }
  grid_depart(a.ctl, departure);
}

// ---------------------------------------------------------------------------
// Route 4: NHWC through L2, two kernels
// ---------------------------------------------------------------------------
// For NHWC tensors small enough to stay in L2 between two kernels.  Both
// kernels map blockDim.x = CV * PL threads like route 2 (thread t covers the
// VE channels (t % CV) * VE .. +VE of pixel lane t / CV) and give CTA b of
// batch item n = b / B the pixels [(b % B) * ppc, +ppc), walked kL2Passes
// pixel lanes at a time; the grid is about what the GPU holds at once.
//
// sgn_nhwc_stats forms S (not stored) and accumulates, per group, the sums of
// S - K[g] and (S - K[g])^2 over its pixels (K[g] the group's first residual
// sum, the same for every CTA), and writes them to the workspace.  The last
// CTA of a batch item to finish (counted with an atomic) adds the item's B
// partials in a fixed order and writes each group's (K, d, rstd):
// mean = K + d, var = sum((S-K)^2)/n - d^2.  X and skip are read with the
// default cache policy so that the second kernel finds them in L2.
//
// sgn_nhwc_apply loads its inputs before waiting for the first kernel (it
// writes none of them), then reads the group statistics, re-forms S, and
// stores S and Y.
//
// Workspace: float4 slots after the control block hold the partials
// [N * B * groups] and the statistics [N * groups]; the control block holds
// one counter per batch item (N <= kL2MaxItems), zero between calls.
constexpr int kL2Passes = 2;       // pixels per thread in flight
// the same in route 5: three (measured on GB300 against two and four: 1-3%
// faster on (4, 64, 64, 320) / (2, 64, 64, 640) fp16 and (2, 64, 64, 320) fp32;
// four spills more and is slower)
constexpr int kCoopL2Passes = 3;
constexpr int kL2MaxThreads = 512;
constexpr int64_t kL2RouteMaxBytes = 48ll << 20;  // re-read through the 129 MB L2

// Shared memory of the per-CTA statistics: per-thread sums [2][VE][PL][CV],
// later the merge slices' pieces [S][groups] (float4).
template <int VE>
__host__ __device__ constexpr int nhwc_red_floats() {
  return 2 * kL2MaxThreads * VE > 3 * 1024 ? 2 * kL2MaxThreads * VE : 3 * 1024;
}

// One CTA's pieces over pixels [p0, p1) of batch item n (routes 4 and 5):
// each group's reference (the mean of four of its residual sums in the range)
// into s_ref[g], then per group the piece (count, R, mu, m2) of its residual
// sums, written to part[b * groups + g]; when some group's R was far from its
// mean, the pixel range is walked again (from L2) around R + mu, kept in
// s_ref[groups + g].  X and skip are read with the default cache policy, so that later
// passes find them in L2.  Every thread of the CTA calls it; it ends with a
// CTA barrier after the piece stores.
template <typename T, typename M, int VE, bool BC, int PASSES = kL2Passes>
__device__ __forceinline__ void nhwc_partials(const SgnArgs<T, M>& a, int n, int b, int p0,
                                              int p1, float* s_ref, float* s_red, float* s_col,
                                              float4* part) {
  __shared__ int s_again;
  const int C = a.C;
  const int CV = C / VE;
  const int PL = blockDim.x / CV;
  const int tc = threadIdx.x % CV;
  const int tp = threadIdx.x / CV;
  const int64_t nbase = static_cast<int64_t>(n) * a.HW * C;
  const int c0 = tc * VE;
  const bool active = tp < PL;
  float* s_R0 = s_ref;
  float* s_R = s_ref + a.groups;

  for (int g = threadIdx.x; g < a.groups; g += blockDim.x) s_R0[g] = nhwc_ref(a, n, g, p0, p1);
  if (threadIdx.x == 0) s_again = 0;
  Pack<T, VE> skb, bv;
  if (active) {
    if constexpr (BC) skb = ld_reuse<T, VE>(a.skip + static_cast<int64_t>(n) * C + c0);
    if (a.bias) bv = ld_reuse<T, VE>(a.bias + c0);
  }
  __syncthreads();
  float Kl[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) Kl[e] = s_R0[fdiv(c0 + e, a.cpg_div)];
  const int nthr = PL * CV;
  const float cnt = static_cast<float>(p1 - p0) * static_cast<float>(a.cpg);
  for (int round = 0; round < 2; ++round) {
    if (round == 1) {
#pragma unroll
      for (int e = 0; e < VE; ++e) Kl[e] = s_R[fdiv(c0 + e, a.cpg_div)];
    }
    float s1[VE], s2[VE];
#pragma unroll
    for (int e = 0; e < VE; ++e) s1[e] = s2[e] = 0.0f;
    if (active) {
      for (int q = p0 + tp; q < p1; q += PASSES * PL) {
        Pack<T, VE> xv[PASSES], kv[BC ? 1 : PASSES];
#pragma unroll
        for (int k = 0; k < PASSES; ++k) {
          const int p = q + k * PL;
          if (p < p1) {
            const int64_t off = nbase + static_cast<int64_t>(p) * C + c0;
            xv[k] = ld_reuse<T, VE>(a.x + off);
            if constexpr (!BC) kv[k] = ld_reuse<T, VE>(a.skip + off);
          }
        }
#pragma unroll
        for (int k = 0; k < PASSES; ++k) {
          if (q + k * PL < p1) {
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              const float sk = BC ? to_f32(skb.v[e]) : to_f32(kv[BC ? 0 : k].v[e]);
              const float d = to_f32(sgn_sum_b<T>(to_f32(xv[k].v[e]), sk, to_f32(bv.v[e]),
                                                  a.bias != nullptr)) -
                              Kl[e];
              s1[e] += d;
              s2[e] = fmaf(d, d, s2[e]);
            }
          }
        }
      }
    }
    // per channel (over the pixel lanes), then per group
    if (active) {
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        s_red[(e * PL + tp) * CV + tc] = s1[e];
        s_red[nthr * VE + (e * PL + tp) * CV + tc] = s2[e];
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < C; j += blockDim.x) {
      const int e = j / CV, q0 = j % CV;
      float t1 = 0.0f, t2 = 0.0f;
      for (int q = 0; q < PL; ++q) {
        t1 += s_red[(e * PL + q) * CV + q0];
        t2 += s_red[nthr * VE + (e * PL + q) * CV + q0];
      }
      s_col[q0 * VE + e] = t1;
      s_col[C + q0 * VE + e] = t2;
    }
    __syncthreads();
    for (int g = threadIdx.x; g < a.groups; g += blockDim.x) {
      float t1 = 0.0f, t2 = 0.0f;
      for (int cc = 0; cc < a.cpg; ++cc) {
        t1 += s_col[g * a.cpg + cc];
        t2 += s_col[C + g * a.cpg + cc];
      }
      const float R = round == 0 ? s_R0[g] : s_R[g];
      const float4 piece = piece_from_sums(cnt, R, t1, t2);
      part[static_cast<int64_t>(b) * a.groups + g] = piece;
      if (round == 0) {
        s_R[g] = R + piece.z;
        if (piece_ill(piece)) s_again = 1;
      }
    }
    __syncthreads();
    if (!s_again) break;
  }
}

// Merges a batch item's B pieces per group in a fixed order: slice j of group
// g sums pieces j, j + S, j + 2S, ... (S slices per group, the block's
// threads spread over groups x slices) around the mean Kq of its first piece,
// kept as (Kq, n, s1, s2); then the slices are moved to the first slice's Kq
// and added in order, so every CTA that merges gets the same bits.  Leaves the
// centre K, the offset d of the mean and rstd of group g in s_out[g],
// s_out[groups + g] and s_out[2 * groups + g]; ends with a barrier.  s_m holds
// S * groups float4.
template <typename T, typename M>
__device__ __forceinline__ void nhwc_merge(const SgnArgs<T, M>& a, const float4* part, int B,
                                           float4* s_m, float* s_out) {
  const int S = max(1, static_cast<int>(blockDim.x) / a.groups);
  for (int idx = threadIdx.x; idx < S * a.groups; idx += blockDim.x) {
    const int g = idx % a.groups, j = idx / a.groups;
    MergeAcc m{0.0f, 0.0f, 0.0f};
    float Kq = 0.0f;
    // eight loads in flight per batch; slots past B are empty pieces centred
    // on Kq, which add +0 to every sum
    for (int q = j; q < B; q += 8 * S) {
      float4 u[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        u[i] = q + i * S < B ? __ldcg(part + static_cast<int64_t>(q + i * S) * a.groups + g)
                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (q == j) Kq = piece_mean(u[0]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (q + i * S >= B) u[i].y = Kq;
        merge_add(m, u[i], Kq);
      }
    }
    s_m[j * a.groups + g] = make_float4(Kq, m.n, m.s1, m.s2);
  }
  __syncthreads();
  for (int g = threadIdx.x; g < a.groups; g += blockDim.x) {
    const float Kc = s_m[g].x;
    MergeAcc m{0.0f, 0.0f, 0.0f};
    for (int j = 0; j < min(S, B); ++j) merge_add_moved(m, s_m[j * a.groups + g], Kc);
    GStats st = merge_finish(m, Kc);
    if (merge_ill(st))  // pathological spread of the pieces: merge them all afresh
      st = merge_pieces_global(part, a.groups, g, B);
    s_out[g] = st.K;
    s_out[a.groups + g] = st.d;
    s_out[2 * a.groups + g] = rsqrtf(st.var + a.eps);
  }
  __syncthreads();
}

template <typename T, typename M, int VE, bool BC>
__global__ void __launch_bounds__(kL2MaxThreads, 2)
sgn_nhwc_stats(const SgnArgs<T, M> a, int B, int ppc) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(16) float s_red[nhwc_red_floats<VE>()];
  __shared__ float s_col[3 * 1024];  // [2][C], C <= 1024; then (K, d, rstd) per group
  __shared__ unsigned s_last;
  extern __shared__ float s_ref[];  // [2 * groups]
  const int n = blockIdx.x / B;
  const int b = blockIdx.x % B;
  const int p0 = b * ppc;
  const int p1 = min(p0 + ppc, a.HW);
  float4* part = a.part + static_cast<int64_t>(n) * B * a.groups;
  nhwc_partials<T, M, VE, BC>(a, n, b, p0, p1, s_ref, s_red, s_col, part);
  // The last CTA of this batch item merges its pieces.  The barrier at the
  // end of nhwc_partials orders every thread's piece stores before thread 0's
  // fence, and the fence (cumulative) makes them visible GPU-wide before the
  // count goes up; on the merging side the fence after the count orders the
  // reads after it.
  float4* stats = a.part + a.N * B * a.groups;
  unsigned* counter = a.ctl->item_done + n;
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(counter, 1u) == static_cast<unsigned>(B - 1);
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  nhwc_merge(a, part, B, reinterpret_cast<float4*>(s_red), s_col);
  for (int g = threadIdx.x; g < a.groups; g += blockDim.x)
    stats[static_cast<int64_t>(n) * a.groups + g] =
        make_float4(s_col[g], s_col[a.groups + g], s_col[2 * a.groups + g], 0.0f);
  if (threadIdx.x == 0) *counter = 0u;  // ready for the next call
}

template <typename T, typename M, int VE, bool BC>
__global__ void __launch_bounds__(kL2MaxThreads, 2)
sgn_nhwc_apply(const SgnArgs<T, M> a, int B, int ppc) {
  // per channel c, at [(c % VE) * CV + c / VE] (the threads of a warp read
  // consecutive entries): (K, d, rstd * gamma[c], beta[c]) of c's group
  extern __shared__ float4 s_coef[];
  const int C = a.C;
  const int CV = C / VE;
  const int PL = blockDim.x / CV;
  const int tc = threadIdx.x % CV;
  const int tp = threadIdx.x / CV;
  const int n = blockIdx.x / B;
  const int b = blockIdx.x % B;
  const int p0 = b * ppc;
  const int p1 = min(p0 + ppc, a.HW);
  const int64_t nbase = static_cast<int64_t>(n) * a.HW * C;
  const int c0 = tc * VE;
  const bool active = tp < PL;
  // The first pixels' inputs before the wait: the kernel before this one (the
  // statistics kernel) writes none of them, and it waited for everything
  // before it.
  Pack<T, VE> xv[kL2Passes], kv[BC ? 1 : kL2Passes], skb, bv;
  if (active) {
#pragma unroll
    for (int k = 0; k < kL2Passes; ++k) {
      const int p = p0 + tp + k * PL;
      if (p < p1) {
        const int64_t off = nbase + static_cast<int64_t>(p) * C + c0;
        xv[k] = ld_stream<T, VE>(a.x + off);
        if constexpr (!BC) kv[k] = ld_stream<T, VE>(a.skip + off);
      }
    }
    if constexpr (BC) skb = ld_reuse<T, VE>(a.skip + static_cast<int64_t>(n) * C + c0);
    if (a.bias) bv = ld_reuse<T, VE>(a.bias + c0);
  }
  pdl_wait();
  pdl_trigger();
  const float4* stats = a.part + a.N * B * a.groups + static_cast<int64_t>(n) * a.groups;
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    const float4 st = __ldcg(stats + c / a.cpg);
    s_coef[(c % VE) * CV + c / VE] =
        make_float4(st.x, st.y, st.z * to_f32(__ldg(a.gamma + c)), to_f32(__ldg(a.beta + c)));
  }
  __syncthreads();
  if (!active) return;
  for (int q = p0 + tp; q < p1; q += kL2Passes * PL) {
    if (q != p0 + tp) {
#pragma unroll
      for (int k = 0; k < kL2Passes; ++k) {
        const int p = q + k * PL;
        if (p < p1) {
          const int64_t off = nbase + static_cast<int64_t>(p) * C + c0;
          xv[k] = ld_stream<T, VE>(a.x + off);
          if constexpr (!BC) kv[k] = ld_stream<T, VE>(a.skip + off);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kL2Passes; ++k) {
      const int p = q + k * PL;
      if (p < p1) {
        const int64_t off = nbase + static_cast<int64_t>(p) * C + c0;
        Pack<T, VE> sv, out;
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float sk = BC ? to_f32(skb.v[e]) : to_f32(kv[BC ? 0 : k].v[e]);
          sv.v[e] = sgn_sum_b<T>(to_f32(xv[k].v[e]), sk, to_f32(bv.v[e]), a.bias != nullptr);
          const float4 cf = s_coef[e * CV + tc];
          out.v[e] = from_f32<T>(sgn_out(to_f32(sv.v[e]), cf.x, cf.y, cf.z, 1.0f, cf.w, a.act));
        }
        if (a.s) st_stream<T, VE>(a.s + off, sv);
        st_stream<T, VE>(a.y + off, out);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Route 5: NHWC, one cooperative grid re-reading its inputs through L2
// ---------------------------------------------------------------------------
// Route 4's work in one launch: every CTA takes the statistics of its pixel
// range (nhwc_partials), meets the grid at one bounded barrier, adds its
// batch item's partials itself (nhwc_merge, the same order in every CTA),
// turns them into the per-channel table (K, d, rstd * gamma[c], beta[c]) and
// walks its pixel range again -- X and skip now come from L2 -- forming S and
// writing S and Y.  No second launch, and no last-CTA merge that the rest of
// the grid waits for.  Needs every CTA resident at once (a cooperative
// launch) and the inputs to stay in L2 between the passes (as route 4).
// Dynamic shared memory: table [C] float4 | references [2 * groups] float.
template <typename T, typename M, int VE, bool BC>
__global__ void __launch_bounds__(kL2MaxThreads, 2)
sgn_nhwc_coop_l2(const SgnArgs<T, M> a, int B, int ppc) {
  __shared__ __align__(16) float s_red[nhwc_red_floats<VE>()];
  __shared__ float s_col[3 * 1024];  // [2][C], C <= 1024; then (K, d, rstd) per group
  extern __shared__ float4 s_dyn[];
  float4* s_coef = s_dyn;
  float* s_ref = reinterpret_cast<float*>(s_dyn + a.C);  // [2 * groups]
  const int C = a.C;
  const int CV = C / VE;
  const int PL = blockDim.x / CV;
  const int tc = threadIdx.x % CV;
  const int tp = threadIdx.x / CV;
  const int n = blockIdx.x / B;
  const int b = blockIdx.x % B;
  const int p0 = b * ppc;
  const int p1 = min(p0 + ppc, a.HW);
  const int64_t nbase = static_cast<int64_t>(n) * a.HW * C;
  const int c0 = tc * VE;
  float4* part = a.part + static_cast<int64_t>(n) * B * a.groups;

  nhwc_partials<T, M, VE, BC, kCoopL2Passes>(a, n, b, p0, p1, s_ref, s_red, s_col, part);
  // the arrival's release (after a CTA barrier) publishes the partials
  grid_arrive(a.ctl);
  unsigned departure = 0u;
  if (!grid_wait(a.ctl, gridDim.x, a.limit_ns, 5u, departure)) {
    grid_depart(a.ctl, departure);
    return;
  }
  nhwc_merge(a, part, B, reinterpret_cast<float4*>(s_red), s_col);
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    const int g = c / a.cpg;
    s_coef[(c % VE) * CV + c / VE] =
        make_float4(s_col[g], s_col[a.groups + g],
                    s_col[2 * a.groups + g] * to_f32(__ldg(a.gamma + c)),
                    to_f32(__ldg(a.beta + c)));
  }
  __syncthreads();
  if (tp < PL) {
    Pack<T, VE> skb, bv;
    if constexpr (BC) skb = ld_reuse<T, VE>(a.skip + static_cast<int64_t>(n) * C + c0);
    if (a.bias) bv = ld_reuse<T, VE>(a.bias + c0);
    for (int q = p0 + tp; q < p1; q += kCoopL2Passes * PL) {
      Pack<T, VE> xv[kCoopL2Passes], kv[BC ? 1 : kCoopL2Passes];
#pragma unroll
      for (int k = 0; k < kCoopL2Passes; ++k) {
        const int p = q + k * PL;
        if (p < p1) {
          const int64_t off = nbase + static_cast<int64_t>(p) * C + c0;
          xv[k] = ld_stream<T, VE>(a.x + off);
          if constexpr (!BC) kv[k] = ld_stream<T, VE>(a.skip + off);
        }
      }
#pragma unroll
      for (int k = 0; k < kCoopL2Passes; ++k) {
        const int p = q + k * PL;
        if (p < p1) {
          const int64_t off = nbase + static_cast<int64_t>(p) * C + c0;
          Pack<T, VE> sv, out;
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            const float sk = BC ? to_f32(skb.v[e]) : to_f32(kv[BC ? 0 : k].v[e]);
            sv.v[e] = sgn_sum_b<T>(to_f32(xv[k].v[e]), sk, to_f32(bv.v[e]), a.bias != nullptr);
            const float4 cf = s_coef[e * CV + tc];
            out.v[e] = from_f32<T>(sgn_out(to_f32(sv.v[e]), cf.x, cf.y, cf.z, 1.0f, cf.w, a.act));
          }
          if (a.s) st_stream<T, VE>(a.s + off, sv);
          st_stream<T, VE>(a.y + off, out);
        }
      }
    }
  }
  grid_depart(a.ctl, departure);
}

// ---------------------------------------------------------------------------
// Route 3: two-phase, any layout
// ---------------------------------------------------------------------------
// Element j of group instance (n, g), j in [0, cpg*HW):
//   NCHW: offset (n*C + g*cpg)*HW + j,                 channel g*cpg + j / HW
//   NHWC: offset (n*HW + j / cpg)*C + g*cpg + j % cpg,  channel g*cpg + j % cpg
template <typename T, typename M>
__device__ __forceinline__ void sgn_locate(const SgnArgs<T, M>& a, int64_t n, int g, int64_t j,
                                           bool cl, int64_t* off, int* c) {
  if (cl) {
    const int64_t p = j / a.cpg;
    const int cc = static_cast<int>(j % a.cpg);
    *c = g * a.cpg + cc;
    *off = (n * a.HW + p) * a.C + *c;
  } else {
    *c = g * a.cpg + static_cast<int>(j / a.HW);
    *off = (n * a.C + static_cast<int64_t>(g) * a.cpg) * a.HW + j;
  }
}

template <typename T, typename M>
__device__ __forceinline__ float sgn_form(const SgnArgs<T, M>& a, int64_t n, int64_t off, int c) {
  const float x = to_f32(__ldcs(a.x + off));
  const float sk = a.bcast ? to_f32(a.skip[n * a.C + c]) : to_f32(__ldcs(a.skip + off));
  return to_f32(sgn_sum<T>(x, sk, a.bias, c));
}

// Merge `count` moments held in shared memory (tree, fixed order); result in [0].
__device__ __forceinline__ void smem_merge(float* mn, float* mm, float* m2, int count) {
  for (int stride = 1; stride < count; stride <<= 1) {
    for (int i = threadIdx.x; i < count; i += blockDim.x) {
      if ((i % (2 * stride)) == 0 && i + stride < count) {
        const Moments r = merge(Moments{mn[i], mm[i], m2[i]},
                                Moments{mn[i + stride], mm[i + stride], m2[i + stride]});
        mn[i] = r.n;
        mm[i] = r.mean;
        m2[i] = r.m2;
      }
    }
    __syncthreads();
  }
}

// Kernel A: the piece (count, R, mu, m2) of one chunk of kTwoPhaseChunk
// elements of a group instance, R the chunk's first residual sum: each
// thread's elements are held in registers and summed twice (mean, then the
// squared deviations from it), and the threads' moments meet in a tree of
// Chan merges, all around R.
template <typename T, typename M, bool CL>
__global__ void __launch_bounds__(kTwoPhaseThreads)
sgn_partials(const SgnArgs<T, M> a, int chunks) {
  pdl_wait();
  pdl_trigger();
  __shared__ float mn[kTwoPhaseThreads], mm[kTwoPhaseThreads], m2s[kTwoPhaseThreads];
  const int64_t inst = blockIdx.x / chunks;
  const int q = blockIdx.x % chunks;
  const int64_t n = inst / a.groups;
  const int g = static_cast<int>(inst % a.groups);
  const int64_t L = static_cast<int64_t>(a.cpg) * a.HW;
  const int64_t j0 = static_cast<int64_t>(q) * kTwoPhaseChunk;
  int64_t off0;
  int cr;
  sgn_locate(a, n, g, j0, CL, &off0, &cr);
  const float R = sgn_form(a, n, off0, cr);
  float v[kTwoPhaseEpt];
  int cnt = 0;
  float sum = 0.0f;
#pragma unroll
  for (int i = 0; i < kTwoPhaseEpt; ++i) {
    const int64_t j = j0 + threadIdx.x + static_cast<int64_t>(i) * kTwoPhaseThreads;
    v[i] = 0.0f;
    if (j < L) {
      int64_t off;
      int c;
      sgn_locate(a, n, g, j, CL, &off, &c);
      const float x = to_f32(__ldcs(a.x + off));
      const float sk = a.bcast ? to_f32(a.skip[n * a.C + c]) : to_f32(__ldcs(a.skip + off));
      const T sT = sgn_sum<T>(x, sk, a.bias, c);
      if (a.s) a.s[off] = sT;
      v[i] = to_f32(sT) - R;
      sum += v[i];
      ++cnt;
    }
  }
  const float mu = cnt ? sum / static_cast<float>(cnt) : 0.0f;
  float m2 = 0.0f;
#pragma unroll
  for (int i = 0; i < kTwoPhaseEpt; ++i) {
    const int64_t j = j0 + threadIdx.x + static_cast<int64_t>(i) * kTwoPhaseThreads;
    if (j < L) {
      const float d = v[i] - mu;
      m2 = fmaf(d, d, m2);
    }
  }
  mn[threadIdx.x] = static_cast<float>(cnt);
  mm[threadIdx.x] = mu;
  m2s[threadIdx.x] = m2;
  __syncthreads();
  smem_merge(mn, mm, m2s, blockDim.x);
  if (threadIdx.x == 0) a.part[blockIdx.x] = make_float4(mn[0], R, mm[0], m2s[0]);
}

// Kernel B: merges the instance's chunk pieces around the first chunk's mean
// (again around the merged mean when that was far from it), re-forms S from
// the inputs and writes Y.
template <typename T, typename M, bool CL>
__global__ void __launch_bounds__(kTwoPhaseThreads)
sgn_normalize(const SgnArgs<T, M> a, int chunks) {
  pdl_wait();
  pdl_trigger();
  __shared__ float2 red2[33];
  const int64_t inst = blockIdx.x / chunks;
  const int q = blockIdx.x % chunks;
  const int64_t n = inst / a.groups;
  const int g = static_cast<int>(inst % a.groups);
  const int64_t L = static_cast<int64_t>(a.cpg) * a.HW;
  const float4* cp = a.part + inst * chunks;
  float Kc = piece_mean(__ldcg(cp));
  GStats st{};
  for (int round = 0; round < 3; ++round) {
    MergeAcc m{0.0f, 0.0f, 0.0f};
    for (int i = threadIdx.x; i < chunks; i += blockDim.x) merge_add(m, __ldcg(cp + i), Kc);
    const float2 t = cta_sum2(make_float2(m.n, m.s1), red2);
    const float2 u = cta_sum2(make_float2(m.s2, 0.0f), red2);
    st = merge_finish(MergeAcc{t.x, t.y, u.x}, Kc);
    if (!merge_ill(st)) break;  // uniform: every thread holds the same totals
    Kc = Kc + st.d;
  }
  const float rstd = rsqrtf(st.var + a.eps);
  const int64_t j0 = static_cast<int64_t>(q) * kTwoPhaseChunk;
#pragma unroll 4
  for (int i = 0; i < kTwoPhaseEpt; ++i) {
    const int64_t j = j0 + threadIdx.x + static_cast<int64_t>(i) * kTwoPhaseThreads;
    if (j < L) {
      int64_t off;
      int c;
      sgn_locate(a, n, g, j, CL, &off, &c);
      const float sv = sgn_form(a, n, off, c);
      a.y[off] = from_f32<T>(
          sgn_out(sv, st.K, st.d, rstd, to_f32(a.gamma[c]), to_f32(a.beta[c]), a.act));
    }
  }
}

// ---------------------------------------------------------------------------
// Kernel selection and typed launch (host)
// ---------------------------------------------------------------------------
// Offset (in floats) of the samples | R | gamma | beta tail of route 2's
// dynamic shared memory: past both the pieces area and the merge area.
inline size_t coop_k_offset(int PL, int C, int B, int groups) {
  const size_t passes = 2 * (static_cast<size_t>(PL) * C + C);
  const size_t nchunk = (static_cast<size_t>(B) + kCoopMergeChunk - 1) / kCoopMergeChunk;
  const size_t merge = nchunk * groups * 4 + 3ull * groups;
  const size_t off = passes > merge ? passes : merge;
  return (off + 3) & ~static_cast<size_t>(3);  // 16-byte aligned tail
}

template <typename T, typename M, int VE, int NV>
inline void* coop_fn() {
  return reinterpret_cast<void*>(sgn_nhwc_coop<T, M, VE, NV>);
}

template <typename T, typename M>
inline void* pick_coop(int ve, int nv) {
  constexpr int V16 = static_cast<int>(16 / sizeof(T));
  if (ve == 1) {
    switch (nv) {
      case 1: return coop_fn<T, M, 1, 1>();
      case 2: return coop_fn<T, M, 1, 2>();
      case 4: return coop_fn<T, M, 1, 4>();
      case 8: return coop_fn<T, M, 1, 8>();
    }
    return nullptr;
  }
  // 3, 5 and 6 pixels per thread too: the tightest count that holds a slab
  // keeps the fewest registers live (the NHWC fp16 workload's 54-pixel slabs
  // over 12 pixel lanes take 5; 8 spills)
  switch (nv) {
    case 1: return coop_fn<T, M, V16, 1>();
    case 2: return coop_fn<T, M, V16, 2>();
    case 3: return coop_fn<T, M, V16, 3>();
    case 4: return coop_fn<T, M, V16, 4>();
    case 5: return coop_fn<T, M, V16, 5>();
    case 6: return coop_fn<T, M, V16, 6>();
    case 8: return coop_fn<T, M, V16, 8>();
  }
  return nullptr;
}

template <typename T, typename M>
inline void* pick_slab(int ve) {
  constexpr int V16 = static_cast<int>(16 / sizeof(T));
  return ve == 1 ? reinterpret_cast<void*>(sgn_nhwc_slab<T, M, 1>)
                 : reinterpret_cast<void*>(sgn_nhwc_slab<T, M, V16>);
}

template <typename T, typename M>
inline void* pick_resident(int ve) {
  constexpr int V16 = static_cast<int>(16 / sizeof(T));
  return ve == 1 ? reinterpret_cast<void*>(sgn_nchw_smem<T, M, 1>)
                 : reinterpret_cast<void*>(sgn_nchw_smem<T, M, V16>);
}

// Route 4 kernels for vectors of `ve` elements and (N, C) or full skip:
// {statistics, apply}.
template <typename T, typename M, int VE>
inline void pick_l2_ve(bool bcast, void** stats, void** apply) {
  if (bcast) {
    *stats = reinterpret_cast<void*>(sgn_nhwc_stats<T, M, VE, true>);
    *apply = reinterpret_cast<void*>(sgn_nhwc_apply<T, M, VE, true>);
  } else {
    *stats = reinterpret_cast<void*>(sgn_nhwc_stats<T, M, VE, false>);
    *apply = reinterpret_cast<void*>(sgn_nhwc_apply<T, M, VE, false>);
  }
}

template <typename T, typename M>
inline void* pick_coop_l2(int ve, bool bcast) {
  constexpr int V16 = static_cast<int>(16 / sizeof(T));
  if (ve == 1)
    return bcast ? reinterpret_cast<void*>(sgn_nhwc_coop_l2<T, M, 1, true>)
                 : reinterpret_cast<void*>(sgn_nhwc_coop_l2<T, M, 1, false>);
  return bcast ? reinterpret_cast<void*>(sgn_nhwc_coop_l2<T, M, V16, true>)
               : reinterpret_cast<void*>(sgn_nhwc_coop_l2<T, M, V16, false>);
}

template <typename T, typename M>
inline void pick_l2(int ve, bool bcast, void** stats, void** apply) {
  constexpr int V16 = static_cast<int>(16 / sizeof(T));
  if (ve == 1) pick_l2_ve<T, M, 1>(bcast, stats, apply);
  else pick_l2_ve<T, M, V16>(bcast, stats, apply);
}

template <typename T, typename M>
inline cudaError_t launch_group_typed(const SkipGroupCall& c, const GroupPlan& p,
                                      cudaStream_t stream) {
  SgnArgs<T, M> a;
  a.x = static_cast<const T*>(c.x);
  a.skip = static_cast<const T*>(c.skip);
  a.bias = static_cast<const T*>(c.bias);
  a.gamma = static_cast<const M*>(c.gamma);
  a.beta = static_cast<const M*>(c.beta);
  a.y = static_cast<T*>(c.y);
  a.s = static_cast<T*>(c.s);
  a.N = c.N;
  a.C = static_cast<int>(c.C);
  a.HW = static_cast<int>(c.H * c.W);
  a.cpg = static_cast<int>(c.C / c.groups);
  a.groups = c.groups;
  a.cpg_div = make_fastdiv(static_cast<unsigned>(a.cpg));
  a.bcast = c.bcast ? 1 : 0;
  a.act = c.activation;
  a.eps = c.eps;
  a.ctl = static_cast<Control*>(c.workspace);
  a.part = reinterpret_cast<float4*>(static_cast<char*>(c.workspace) + kControlBytes);
  a.limit_ns = kWaitLimitNs;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
  cfg.blockDim = dim3(p.block);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];

  if (p.route == 1) {
    void* fn = pick_resident<T, M>(p.ve);
    if (!fn) return cudaErrorInvalidConfiguration;
    unsigned nattr = 0;
    if (p.csize > 1) {
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = p.csize;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      nattr = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = add_pdl_attr(attr, nattr);
    int span = p.nv;
    FastDiv vpc = make_fastdiv(static_cast<unsigned>(a.HW / p.ve));
    void* args[] = {&a, &span, &vpc};
    return cudaLaunchKernelExC(&cfg, fn, args);
  }
  if (p.route == 2) {
    // A cooperative launch keeps plain stream order (no early scheduling).
    void* fn = pick_coop<T, M>(p.ve, p.nv);
    if (!fn) return cudaErrorInvalidConfiguration;
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int B = p.ctas_per_item, ppc = p.pix_per_cta;
    const int PL = p.block / static_cast<int>(c.C / p.ve);
    int koff = static_cast<int>(coop_k_offset(PL, static_cast<int>(c.C), B, c.groups));
    void* args[] = {&a, &B, &ppc, &koff};
    return cudaLaunchKernelExC(&cfg, fn, args);
  }
  if (p.route == 6) {
    // A cooperative launch keeps plain stream order (no early scheduling).
    void* fn = pick_slab<T, M>(p.ve);
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int B = p.ctas_per_item, ppc = p.pix_per_cta;
    const int PL = p.block / static_cast<int>(c.C / p.ve);
    int koff = static_cast<int>(coop_k_offset(PL, static_cast<int>(c.C), B, c.groups));
    void* args[] = {&a, &B, &ppc, &koff};
    return cudaLaunchKernelExC(&cfg, fn, args);
  }
  if (p.route == 5) {
    // A cooperative launch keeps plain stream order (no early scheduling).
    void* fn = pick_coop_l2<T, M>(p.ve, c.bcast);
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int B = p.ctas_per_item, ppc = p.pix_per_cta;
    void* args[] = {&a, &B, &ppc};
    return cudaLaunchKernelExC(&cfg, fn, args);
  }
  if (p.route == 4) {
    void *stats = nullptr, *apply = nullptr;
    pick_l2<T, M>(p.ve, c.bcast, &stats, &apply);
    int B = p.ctas_per_item, ppc = p.pix_per_cta;
    void* args[] = {&a, &B, &ppc};
    cfg.attrs = attr;
    cfg.numAttrs = add_pdl_attr(attr, 0);
    cfg.dynamicSmemBytes = static_cast<size_t>(2 * c.groups) * sizeof(float);
    cudaError_t e = cudaLaunchKernelExC(&cfg, stats, args);
    if (e != cudaSuccess) return e;
    cfg.dynamicSmemBytes = p.smem;
    return cudaLaunchKernelExC(&cfg, apply, args);
  }
  // route 3
  int chunks = p.chunks;
  cfg.attrs = attr;
  cfg.numAttrs = add_pdl_attr(attr, 0);
  void* args[] = {&a, &chunks};
  void* first = c.channels_last ? reinterpret_cast<void*>(sgn_partials<T, M, true>)
                                : reinterpret_cast<void*>(sgn_partials<T, M, false>);
  void* second = c.channels_last ? reinterpret_cast<void*>(sgn_normalize<T, M, true>)
                                 : reinterpret_cast<void*>(sgn_normalize<T, M, false>);
  cudaError_t e = cudaLaunchKernelExC(&cfg, first, args);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelExC(&cfg, second, args);
}

// Kernel pointers and typed launches per element type T of X (group_f32.cu,
// group_f16.cu, group_bf16.cu).  Pointers are null for (M, ve, nv) without
// an instantiation.
void* group_coop_kernel_f32(DType m, int ve, int nv);
void* group_coop_kernel_f16(DType m, int ve, int nv);
void* group_coop_kernel_bf16(DType m, int ve, int nv);
void* group_resident_kernel_f32(DType m, int ve);
void* group_resident_kernel_f16(DType m, int ve);
void* group_resident_kernel_bf16(DType m, int ve);
void* group_slab_kernel_f32(DType m, int ve);
void* group_slab_kernel_f16(DType m, int ve);
void* group_slab_kernel_bf16(DType m, int ve);
void* group_coop_l2_kernel_f32(DType m, int ve, bool bcast);
void* group_coop_l2_kernel_f16(DType m, int ve, bool bcast);
void* group_coop_l2_kernel_bf16(DType m, int ve, bool bcast);
cudaError_t launch_group_f32(const SkipGroupCall& c, const GroupPlan& p, cudaStream_t stream);
cudaError_t launch_group_f16(const SkipGroupCall& c, const GroupPlan& p, cudaStream_t stream);
cudaError_t launch_group_bf16(const SkipGroupCall& c, const GroupPlan& p, cudaStream_t stream);

}  // namespace b200norm
