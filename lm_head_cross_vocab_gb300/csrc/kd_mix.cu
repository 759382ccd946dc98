// Multi-teacher mixing (orda-kernel README, "Cross-vocabulary distillation",
// multi-teacher mixing): K cached teacher logit rows over one vocabulary are
// mixed into one distribution, written as its log-probabilities,
//   arithmetic (probability average):  out = log sum_k w_k softmax(z_k)
//   geometric (product of experts):    out = g - logsumexp(g),  g = sum_k w_k z_k
// with the weights normalised to sum to 1 (the product of the teachers'
// softmaxes differs from exp(g) by a per-row factor only, which the
// normalisation removes).  A token the mixture gives no probability gets the
// most negative finite value of the output type, as the projection writes it.
//
// Every output needs the logsumexp of whole teacher rows (or of g).  A cluster
// of C CTAs (C = 1, 2, 4 or 8) therefore holds one token row of all K
// teachers in shared memory -- CTA r columns [r*sc, r*sc + sc), one bulk copy
// per teacher -- reduces its columns to a (max, sum of exp) pair per stream,
// exchanges the pairs through distributed shared memory, and writes its
// columns of the output with vector stores: each input byte is read from HBM
// once and each output byte written once.  Two shapes exist: two CTAs per SM
// with 100 KiB of staging each, and, for rows that need more than 8 x 100 KiB,
// a wide shape of one CTA per SM with 200 KiB.  Rows too long for an 8-CTA
// cluster of the wide shape take a one-CTA-per-row kernel that reads the row
// from global memory twice.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstring>

#include "../../include/kd.h"
#include "kd_internal.h"
#include "kd_ptx.cuh"

namespace kd {
namespace {

constexpr int kMaxT = KD_MIX_MAX_TEACHERS;
constexpr int kMT = 512;                  // threads per CTA (two CTAs per SM)
constexpr int kMW = kMT / 32;             // warps per CTA
constexpr int64_t kMixBuf = 100 * 1024;   // bytes of staged teacher rows per CTA (two per SM)
constexpr int64_t kMixBufWide = 200 * 1024;  // one CTA per SM, for longer rows
constexpr float kLN2 = 0.6931471805599453f;

struct MixParams {
  const void* z[kMaxT];  // teacher logits [n, v], K of them (weights > 0 only)
  float w[kMaxT];        // weights, normalised to sum to 1
  float lw[kMaxT];       // log w
  int k;
  int64_t n, v;
  int64_t sc;            // columns per CTA of the cluster kernel
  void* out;             // [n, v]
  uint32_t* status;
};

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16(x);
}
template <typename T>
__device__ __forceinline__ float lowest_of();
template <>
__device__ __forceinline__ float lowest_of<float>() {
  return -FLT_MAX;
}
template <>
__device__ __forceinline__ float lowest_of<__nv_bfloat16>() {
  return __uint_as_float(0xff7f0000u);  // most negative finite bf16
}

__device__ __forceinline__ float fast_exp(float x) { return ex2(x * kL2E); }

// (m, s) running pair of a logsumexp: the maximum and sum_v exp(x_v - m)
struct Lse {
  float m, s;
};
__device__ __forceinline__ Lse lse_merge(Lse a, Lse b) {
  if (b.s == 0.f) return a;
  if (a.s == 0.f) return b;
  const float m = fmaxf(a.m, b.m);
  return {m, a.s * fast_exp(a.m - m) + b.s * fast_exp(b.m - m)};
}
__device__ __forceinline__ float lse_value(Lse a) {
  return a.s > 0.f ? a.m + __logf(a.s) : -INFINITY;
}
// block-wide merge of one pair per thread; every thread gets the result
__device__ Lse block_lse(Lse v, Lse* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Lse u{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.s, o)};
    v = lse_merge(v, u);
  }
  __syncthreads();  // red[] may still be read from the previous call
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  Lse r = red[0];
#pragma unroll
  for (int i = 1; i < kMW; ++i) r = lse_merge(r, red[i]);
  return r;
}

// Pass 1 over columns [0, len) of one stream: stream t < K is teacher t,
// stream K (geometric) is g = sum_k w_k z_k.  get(k, j) reads teacher k at
// column j.  Thread-local maximum first, then the sum at that maximum.
template <bool GEO, typename Get>
__device__ __forceinline__ Lse stream_lse(const MixParams& P, int t, int64_t len, Get get) {
  auto val = [&](int64_t j) {
    if (!GEO) return get(t, j);
    float g = 0.f;
    for (int k = 0; k < P.k; ++k) g = fmaf(P.w[k], get(k, j), g);
    return g;
  };
  float m = -INFINITY;
  for (int64_t j = threadIdx.x; j < len; j += kMT) m = fmaxf(m, val(j));
  float s = 0.f;
  if (m > -INFINITY)
    for (int64_t j = threadIdx.x; j < len; j += kMT) s += fast_exp(val(j) - m);
  return {m, s};
}

// output value at one column from the row logsumexps lse[] (per teacher, or
// of g in slot 0 for the geometric mode)
template <bool GEO, typename TO, typename Get>
__device__ __forceinline__ float mix_value(const MixParams& P, const float* lse, int64_t j,
                                           Get get) {
  float r;
  if (GEO) {
    float g = 0.f;
    for (int k = 0; k < P.k; ++k) g = fmaf(P.w[k], get(k, j), g);
    r = g - lse[0];
  } else {
    // log sum_k exp(t_k), t_k = z_k - lse_k + log w_k, folded one teacher at a
    // time around the running maximum (K - 1 exponentials and one logarithm)
    float m = -INFINITY, s = 0.f;
    for (int k = 0; k < P.k; ++k) {
      const float t = get(k, j) - lse[k] + P.lw[k];
      if (!(t > -INFINITY)) continue;  // no probability (or a teacher row without any)
      if (s == 0.f) {
        m = t;
        s = 1.f;
        continue;
      }
      const float e = fast_exp(-fabsf(t - m));
      if (t > m) {
        s = fmaf(s, e, 1.f);
        m = t;
      } else {
        s += e;
      }
    }
    r = s > 0.f ? m + __logf(s) : -INFINITY;
  }
  return r > kNoMass ? r : lowest_of<TO>();
}


__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cl_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// a float of CTA `rank`'s shared memory (read between cluster barriers)
__device__ __forceinline__ float cl_load(const float* p, uint32_t rank) {
  uint32_t a = ptx::smem_u32(p);
  asm("mapa.shared::cluster.u32 %0, %0, %1;" : "+r"(a) : "r"(rank));
  float v;  // (volatile: never moved above the cluster barrier that publishes it)
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 8 consecutive staged fp32 values (16-byte aligned shared memory); bf16
// teachers take the packed passes below
__device__ __forceinline__ void ld8(const float* p, float v[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// the stream's values at 8 columns: teacher t, or g = sum_k w_k z_k
template <bool GEO, typename TI>
__device__ __forceinline__ void stream8(const MixParams& P, const TI* zs, int t, int64_t j0,
                                        float x[8]) {
  if (!GEO) {
    ld8(zs + t * P.sc + j0, x);
    return;
  }
  float y[8];
  ld8(zs + j0, y);
#pragma unroll
  for (int q = 0; q < 8; ++q) x[q] = P.w[0] * y[q];
  for (int k = 1; k < P.k; ++k) {
    ld8(zs + k * P.sc + j0, y);
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] = fmaf(P.w[k], y[q], x[q]);
  }
}

// Pass 1 of the cluster kernel: this thread's (max, sum of exp) of one stream
// over the staged columns [0, clen), 8 columns a step, one exponential per
// value (the running sum is rescaled when a step raises the maximum).
template <bool GEO, typename TI>
__device__ __forceinline__ Lse pass1(const MixParams& P, const TI* zs, int t, int64_t lo,
                                     int64_t hi, Lse acc) {
  float m = acc.m, s = acc.s;
  for (int64_t j0 = lo + (int64_t)threadIdx.x * 8; j0 < hi; j0 += (int64_t)kMT * 8) {
    float x[8];
    stream8<GEO>(P, zs, t, j0, x);
    if (j0 + 8 > hi) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (j0 + q >= hi) x[q] = -INFINITY;
    }
    float m8 = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                     fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
    // values at or below kNoMass carry no probability: they never set the
    // maximum (so m * log2(e) below stays finite) and their terms are 0
    if (m8 > m && m8 > kNoMass) {
      s *= ex2((m - m8) * kL2E);  // 0 while m is still -inf (s is 0 then too)
      m = m8;
    }
    // (x - m first: exact near the maximum, whatever the logits' magnitude)
    if (m > -INFINITY) {
#pragma unroll
      for (int q = 0; q < 8; ++q) s += ex2((x[q] - m) * kL2E);
    }
  }
  return {m, s};
}

// Pass 2 of the cluster kernel: 8 output values at columns j0.. from the row
// logsumexps lse[] (per teacher, or of g in slot 0).
template <bool GEO, typename TI, typename TO>
__device__ __forceinline__ void pass2_8(const MixParams& P, const TI* zs, const float* lse,
                                        int64_t j0, float r[8]) {
  if (GEO) {
    float g[8];
    stream8<true>(P, zs, 0, j0, g);
#pragma unroll
    for (int q = 0; q < 8; ++q) r[q] = g[q] - lse[0];
  } else {
    // log sum_k exp(t_k), t_k = z_k - lse_k + log w_k, folded teacher by
    // teacher around the running maximum in base 2 (K - 1 exponentials and
    // one logarithm); z_k - lse_k first, exact for a row's dominant token.
    // Terms are clamped below at kNoMass (base 2), so the fold needs no
    // special case: a clamped term adds 2^-huge = 0 beside any real one, and
    // a token with only clamped terms stays at or below kNoMass.
    constexpr float kFloor = kNoMass * kL2E;
    float m[8], s[8], x[8];
    ld8(zs + j0, x);
    const float l0 = lse[0], w0 = P.lw[0] * kL2E;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      m[q] = fmaxf(fmaf(x[q] - l0, kL2E, w0), kFloor);
      s[q] = 1.f;
    }
    for (int k = 1; k < P.k; ++k) {
      ld8(zs + k * P.sc + j0, x);
      const float lk = lse[k], wk = P.lw[k] * kL2E;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float t = fmaxf(fmaf(x[q] - lk, kL2E, wk), kFloor);
        const float d = t - m[q];
        const float e = ex2(-fabsf(d));
        s[q] = d > 0.f ? fmaf(s[q], e, 1.f) : s[q] + e;
        m[q] = fmaxf(m[q], t);
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) r[q] = m[q] > kFloor ? (m[q] + lg2(s[q])) * kLN2 : -INFINITY;
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) r[q] = r[q] > kNoMass ? r[q] : lowest_of<TO>();
}

// Packed passes for bf16 teachers: 32-bit slice indices, the values of a
// step taken as raw bf16x2 words, the fp32 work on f32x2 pairs (one
// instruction for two columns).
constexpr float kStaleMix = 8.f;  // log2 of the largest term a stale offset may leave

__device__ __forceinline__ float2 unpack2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }

// Pass 1, packed: this thread's (max, sum of exp) of one stream over the
// staged columns [lo, hi).  The sum is kept around an offset m that moves only
// when a step's maximum passes it by kStaleMix in base 2 (so no term exceeds
// 2^8; the sum is rescaled then): for a teacher stream the test runs on the
// raw words (max.bf16x2 against a threshold rounded down), for g on floats.
// Values at or below kNoMass never move the offset and add 0.
template <bool GEO, int KT>
__device__ __forceinline__ Lse pass1_bf16(const MixParams& P, const __nv_bfloat16* zs, int t,
                                          int lo, int hi, Lse acc) {
  const int sc = (int)P.sc;
  const int K = KT ? KT : P.k;  // KT: the teacher count when fixed at compile time
  float m = acc.m;
  float2 s2 = make_float2(acc.s, 0.f);
  float2 om = make_float2(-m * kL2E, -m * kL2E);
  uint32_t th = m > -INFINITY ? bf16x2_floor(m + kStaleMix * kLN2) : kNegInfX2;
  const float2 l2e = make_float2(kL2E, kL2E);
  for (int j0 = lo + (int)threadIdx.x * 8; j0 < hi; j0 += kMT * 8) {
    const bool tail = j0 + 8 > hi;
    float2 x[4];
    float m8;
    bool up;
    if (!GEO) {
      const uint4 u = *reinterpret_cast<const uint4*>(zs + t * sc + j0);
      uint32_t w[4] = {u.x, u.y, u.z, u.w};
      if (tail) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (j0 + 2 * i >= hi) w[i] = kNegInfX2;
          else if (j0 + 2 * i + 1 >= hi) w[i] = (w[i] & 0xffffu) | 0xff800000u;
        }
      }
      const uint32_t mx = max_bf16x2(max_bf16x2(w[0], w[1]), max_bf16x2(w[2], w[3]));
      up = max_bf16x2(mx, th) != th;
      m8 = fmaxf(bf16lo(mx), bf16hi(mx));
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = unpack2(w[i]);
    } else {  // g = sum_k w_k z_k
      const uint4 u = *reinterpret_cast<const uint4*>(zs + j0);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      const float2 w0 = make_float2(P.w[0], P.w[0]);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = mul2(unpack2(w[i]), w0);
#pragma unroll
      for (int k = 1; k < (KT ? KT : kMaxT); ++k) {
        if (!KT && k >= K) break;
        const uint4 v = *reinterpret_cast<const uint4*>(zs + k * sc + j0);
        const uint32_t y[4] = {v.x, v.y, v.z, v.w};
        const float2 wk = make_float2(P.w[k], P.w[k]);
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = fma2(unpack2(y[i]), wk, x[i]);
      }
      if (tail) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (j0 + 2 * i >= hi) x[i].x = -INFINITY;
          if (j0 + 2 * i + 1 >= hi) x[i].y = -INFINITY;
        }
      }
      m8 = fmaxf(fmaxf(fmaxf(x[0].x, x[0].y), fmaxf(x[1].x, x[1].y)),
                 fmaxf(fmaxf(x[2].x, x[2].y), fmaxf(x[3].x, x[3].y)));
      up = m8 > m + kStaleMix * kLN2 || !(m > -INFINITY);
    }
    if (up && m8 > m && m8 > kNoMass) {
      const float f = ex2((m - m8) * kL2E);  // 0 while m is still -inf (s is 0 then too)
      s2 = mul2(s2, make_float2(f, f));
      m = m8;
      om = make_float2(-m * kL2E, -m * kL2E);
      th = bf16x2_floor(m + kStaleMix * kLN2);
    }
    if (m > -INFINITY) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = fma2(x[i], l2e, om);
        s2 = add2(s2, make_float2(ex2(a.x), ex2(a.y)));
      }
    }
  }
  return {m, s2.x + s2.y};
}

// Pass 2, packed: 8 output values at columns j0.. (as pass2_8) from the row
// logsumexps lse_sh[] (per teacher, or of g in slot 0).
template <bool GEO, typename TO, int KT>
__device__ __forceinline__ void pass2_bf16(const MixParams& P, const __nv_bfloat16* zs,
                                           const float* lse_sh, int j0, float r[8]) {
  const int sc = (int)P.sc;
  const int K = KT ? KT : P.k;
  float2 res[4];
  const uint4 u0 = *reinterpret_cast<const uint4*>(zs + j0);
  const uint32_t w0[4] = {u0.x, u0.y, u0.z, u0.w};
  if (GEO) {
    const float2 wt = make_float2(P.w[0], P.w[0]);
#pragma unroll
    for (int i = 0; i < 4; ++i) res[i] = mul2(unpack2(w0[i]), wt);
#pragma unroll
    for (int k = 1; k < (KT ? KT : kMaxT); ++k) {
      if (!KT && k >= K) break;
      const uint4 v = *reinterpret_cast<const uint4*>(zs + k * sc + j0);
      const uint32_t y[4] = {v.x, v.y, v.z, v.w};
      const float2 wk = make_float2(P.w[k], P.w[k]);
#pragma unroll
      for (int i = 0; i < 4; ++i) res[i] = fma2(unpack2(y[i]), wk, res[i]);
    }
    const float2 nl = make_float2(-lse_sh[0], -lse_sh[0]);
#pragma unroll
    for (int i = 0; i < 4; ++i) res[i] = add2(res[i], nl);
  } else {
    // log sum_k exp(t_k), t_k = z_k - lse_k + log w_k, in base 2 around the
    // running maximum (K - 1 exponentials, one logarithm); z_k - lse_k first,
    // exact for a row's dominant token; terms clamped below at kNoMass
    constexpr float kFloor = kNoMass * kL2E;
    const float2 l2e = make_float2(kL2E, kL2E);
    float2 m[4], sum[4];
    {
      const float lw = P.lw[0] * kL2E;
      const float2 l = make_float2(lse_sh[0], lse_sh[0]), w = make_float2(lw, lw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 tt = fma2(sub2(unpack2(w0[i]), l), l2e, w);
        m[i] = make_float2(fmaxf(tt.x, kFloor), fmaxf(tt.y, kFloor));
        sum[i] = make_float2(1.f, 1.f);
      }
    }
#pragma unroll
    for (int k = 1; k < (KT ? KT : kMaxT); ++k) {
      if (!KT && k >= K) break;
      const uint4 v = *reinterpret_cast<const uint4*>(zs + k * sc + j0);
      const uint32_t y[4] = {v.x, v.y, v.z, v.w};
      const float lw = P.lw[k] * kL2E;
      const float2 l = make_float2(lse_sh[k], lse_sh[k]), w = make_float2(lw, lw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 tt = fma2(sub2(unpack2(y[i]), l), l2e, w);
        const float2 t2 = make_float2(fmaxf(tt.x, kFloor), fmaxf(tt.y, kFloor));
        const float2 d = sub2(t2, m[i]);
        const float2 e = make_float2(ex2(-fabsf(d.x)), ex2(-fabsf(d.y)));
        if (K == 2) {  // the sum starts at 1: either order gives 1 + e
          sum[i] = add2(sum[i], e);
        } else {
          sum[i].x = d.x > 0.f ? fmaf(sum[i].x, e.x, 1.f) : sum[i].x + e.x;
          sum[i].y = d.y > 0.f ? fmaf(sum[i].y, e.y, 1.f) : sum[i].y + e.y;
        }
        m[i] = make_float2(fmaxf(m[i].x, t2.x), fmaxf(m[i].y, t2.y));
      }
    }
    const float2 ln2 = make_float2(kLN2, kLN2);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 rr = mul2(add2(m[i], make_float2(lg2(sum[i].x), lg2(sum[i].y))), ln2);
      res[i].x = m[i].x > kFloor ? rr.x : -INFINITY;
      res[i].y = m[i].y > kFloor ? rr.y : -INFINITY;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r[2 * i] = res[i].x > kNoMass ? res[i].x : lowest_of<TO>();
    r[2 * i + 1] = res[i].y > kNoMass ? res[i].y : lowest_of<TO>();
  }
}

// Cluster kernel: see the top of this file.  Rows are taken cluster by
// cluster (all CTAs of a cluster loop over the same rows, so the cluster
// barriers match).  A CTA's columns are staged in two halves, each with its
// own barrier: pass 1 starts on the first half while the second lands, and
// pass 2 frees the first half (whose copy for the next row starts at once)
// before it writes the second.  So the staging of the next row runs under
// this row's pass 2 and the next row's pass 1, and two CTAs share an SM, so
// one CTA's waits are the other's compute.
template <typename TI, typename TO, bool GEO, bool WIDE, int KT>
__global__ void __launch_bounds__(kMT, WIDE ? 1 : 2) k_mix_cluster(const MixParams P) {
  extern __shared__ __align__(16) uint8_t mix_smem[];
  __shared__ __align__(8) uint64_t bars[2];  // one per half
  __shared__ Lse red_all[kMW][kMaxT];   // per warp and stream
  __shared__ float stats[2][kMaxT][2];  // this CTA's (max, sum) per stream, by row parity
  __shared__ float off_sh[kMaxT];       // the row logsumexp per stream
  __shared__ int abort_flag;
  const uint32_t rank = cl_rank(), csize = cl_size();
  const int64_t ncl = gridDim.x / csize;
  const int64_t c0 = (int64_t)rank * P.sc;
  const int64_t clen = P.v - c0 < P.sc ? (P.v - c0 > 0 ? P.v - c0 : 0) : P.sc;
  const int64_t h0 = clen / 2 / 8 * 8;  // halves [0, h0) and [h0, clen)
  const int nstreams = GEO ? 1 : (KT ? KT : P.k);
  TI* const zs = reinterpret_cast<TI*>(mix_smem);  // teacher k at zs + k * sc
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars[1]), 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  // stage half hh of `row`: the 16-byte-aligned bulk of each teacher's columns
  // by bulk copy, the rest (a ragged tail, or a whole unaligned row) by plain
  // loads
  // (returns whether some columns were plain-loaded: the wait then needs a
  // CTA barrier to see them; the bulk-copied ones come with the barrier wait)
  auto stage = [&](int64_t row, int hh) -> bool {
    const int64_t lo = hh ? h0 : 0, hi = hh ? clen : h0;
    const uint32_t bar = ptx::smem_u32(&bars[hh]);
    auto nbytes = [&](int k) -> int64_t {
      const TI* src = static_cast<const TI*>(P.z[k]) + row * P.v + c0 + lo;
      const bool al =
          ((reinterpret_cast<uintptr_t>(src) | ptx::smem_u32(zs + k * P.sc + lo)) & 15) == 0;
      return al ? (hi - lo) * (int64_t)sizeof(TI) / 16 * 16 : 0;
    };
    if (threadIdx.x == 0 && !*reinterpret_cast<volatile int*>(&abort_flag)) {
      // (after a timed-out wait no new copy starts; later waits give up)
      uint32_t total = 0;
      for (int k = 0; k < P.k; ++k) total += (uint32_t)nbytes(k);
      ptx::mbar_expect_tx(bar, total);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      for (int k = 0; k < P.k; ++k) {
        const int64_t nb = nbytes(k);
        if (nb > 0)
          ptx::bulk_load(ptx::smem_u32(zs + k * P.sc + lo),
                         static_cast<const TI*>(P.z[k]) + row * P.v + c0 + lo, (uint32_t)nb, bar);
      }
    }
    bool plain = false;
    for (int k = 0; k < P.k; ++k) {
      const TI* src = static_cast<const TI*>(P.z[k]) + row * P.v + c0;
      const int64_t q0 = lo + nbytes(k) / (int64_t)sizeof(TI);
      plain |= q0 < hi;
      for (int64_t q = q0 + threadIdx.x; q < hi; q += kMT) zs[k * P.sc + q] = src[q];
    }
    return plain;
  };
  uint32_t parity = 0;  // bit hh: phase parity to wait for on half hh
  // the first wait that gave up: its copies may still be in flight (none
  // starts after it, the abort flag being set by then)
  int pend_h = -1;
  uint32_t pend_p = 0;
  bool plain0 = false, plain1 = false;  // a half has plain-loaded columns
  auto wait_half = [&](int hh) {
    if (!ptx::warp_wait(ptx::smem_u32(&bars[hh]), (parity >> hh) & 1u, &abort_flag, P.status) &&
        pend_h < 0) {
      pend_h = hh;
      pend_p = (parity >> hh) & 1u;
    }
    parity ^= 1u << hh;
    if (hh ? plain1 : plain0) __syncthreads();  // the plain-loaded columns too
  };
  const int64_t first = blockIdx.x / csize;
  if (first < P.n) {
    plain0 = stage(first, 0);
    plain1 = stage(first, 1);
  }
  int it = 0;
  for (int64_t row = first; row < P.n; row += ncl, ++it) {
    // pass 1: this CTA's (max, sum) per stream, the first half as soon as it lands
    const int pb = it & 1;
    wait_half(0);
    // every stream's pair folded per thread, then per warp (shuffles), then
    // across the warps by one thread per stream: one CTA barrier for all
    for (int t = 0; t < nstreams; ++t) {
      Lse a;
      if constexpr (sizeof(TI) == 2) {  // bf16 teachers: the packed pass
        a = pass1_bf16<GEO, KT>(P, zs, t, 0, (int)h0, Lse{-INFINITY, 0.f});
        if (t == 0) wait_half(1);
        a = pass1_bf16<GEO, KT>(P, zs, t, (int)h0, (int)clen, a);
      } else {
        a = pass1<GEO>(P, zs, t, 0, h0, Lse{-INFINITY, 0.f});
        if (t == 0) wait_half(1);
        a = pass1<GEO>(P, zs, t, h0, clen, a);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        a = lse_merge(a, Lse{__shfl_xor_sync(0xffffffffu, a.m, o),
                             __shfl_xor_sync(0xffffffffu, a.s, o)});
      if ((threadIdx.x & 31) == 0) red_all[threadIdx.x >> 5][t] = a;
    }
    __syncthreads();
    if (threadIdx.x < (unsigned)nstreams) {
      Lse r = red_all[0][threadIdx.x];
      for (int w = 1; w < kMW; ++w) r = lse_merge(r, red_all[w][threadIdx.x]);
      stats[pb][threadIdx.x][0] = r.m;
      stats[pb][threadIdx.x][1] = r.s;
    }
    // every CTA's pairs of this row are written (and every CTA is done with
    // the previous row's pairs in this parity slot)
    cl_sync();
    // one thread per stream loads every CTA's pair (all loads issued before
    // any is used) and merges them
    if (threadIdx.x < (unsigned)nstreams) {
      Lse acc{-INFINITY, 0.f};
      for (uint32_t q0 = 0; q0 < csize; q0 += 4) {
        float pm[4], ps[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q0 + q < csize) {
            pm[q] = cl_load(&stats[pb][threadIdx.x][0], q0 + q);
            ps[q] = cl_load(&stats[pb][threadIdx.x][1], q0 + q);
          }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q0 + q < csize) acc = lse_merge(acc, Lse{pm[q], ps[q]});
      }
      off_sh[threadIdx.x] = lse_value(acc);
    }
    __syncthreads();
    // pass 2: the output columns, 8 per thread step (vector stores when
    // aligned), half by half; each half is restaged for the next row as soon
    // as every thread is done with it
    TO* o = static_cast<TO*>(P.out) + row * P.v + c0;
    const bool ov = (reinterpret_cast<uintptr_t>(o) & 15) == 0;
    for (int hh = 0; hh < 2; ++hh) {
      // (32-bit indices within the CTA's columns: sc is far below 2^31)
      const int lo = hh ? (int)h0 : 0, hi = hh ? (int)clen : (int)h0;
      for (int j0 = lo + (int)threadIdx.x * 8; j0 < hi; j0 += kMT * 8) {
        float r[8];
        if constexpr (sizeof(TI) == 2)
          pass2_bf16<GEO, TO, KT>(P, zs, off_sh, j0, r);
        else
          pass2_8<GEO, TI, TO>(P, zs, off_sh, j0, r);
        if (ov && j0 + 8 <= hi) {
          if constexpr (sizeof(TO) == 4) {
            reinterpret_cast<float4*>(o + j0)[0] = make_float4(r[0], r[1], r[2], r[3]);
            reinterpret_cast<float4*>(o + j0)[1] = make_float4(r[4], r[5], r[6], r[7]);
          } else {
            uint4 u;
            u.x = pack_bf16(r[0], r[1]);
            u.y = pack_bf16(r[2], r[3]);
            u.z = pack_bf16(r[4], r[5]);
            u.w = pack_bf16(r[6], r[7]);
            *reinterpret_cast<uint4*>(o + j0) = u;
          }
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (j0 + q < hi) o[j0 + q] = from_f<TO>(r[q]);
        }
      }
      __syncthreads();  // half hh is read
      if (row + ncl < P.n) (hh ? plain1 : plain0) = stage(row + ncl, hh);
    }
  }
  // no CTA leaves while another may still read its pairs, nor with a copy of
  // its own in flight (bounded, whatever the abort flag)
  cl_sync();
  if (pend_h >= 0 && threadIdx.x < 32)
    ptx::warp_wait(ptx::smem_u32(&bars[pend_h]), pend_p, &abort_flag, P.status, false);
}

// One CTA per row (grid-strided): pass 1 and pass 2 read the row from global
// memory, for rows of K teachers too long for a 16-CTA cluster.
template <typename TI, typename TO, bool GEO>
__global__ void __launch_bounds__(kMT) k_mix_rows(const MixParams P) {
  __shared__ Lse red[kMW];
  __shared__ float lse[kMaxT];
  const int nstreams = GEO ? 1 : P.k;
  for (int64_t row = blockIdx.x; row < P.n; row += gridDim.x) {
    auto get = [&](int k, int64_t j) {
      return to_f<TI>(static_cast<const TI*>(P.z[k])[row * P.v + j]);
    };
    for (int t = 0; t < nstreams; ++t) {
      const float l = lse_value(block_lse(stream_lse<GEO>(P, t, P.v, get), red));
      if (threadIdx.x == 0) lse[t] = l;
    }
    __syncthreads();
    TO* o = static_cast<TO*>(P.out) + row * P.v;
    for (int64_t j = threadIdx.x; j < P.v; j += kMT) o[j] = from_f<TO>(mix_value<GEO, TO>(P, lse, j, get));
    __syncthreads();  // lse[] is rewritten for the next row
  }
}

// smallest cluster (1, 2, 4 or 8 CTAs) whose per-CTA columns of all K
// teachers, sc a multiple of 8, fit `budget` bytes; 0 when none does.
// (Smaller clusters win over whole-row double buffering: more SMs can host
// them, and the per-row cluster barrier and reductions cost less; the
// two-half staging hides most of the copies instead.  Clusters of 16 CTAs
// measured worse than one wide CTA per SM in clusters of 8.)
int mix_cluster_for(int64_t v, int k, int64_t elem, int64_t budget, int64_t* sc) {
  for (int c = 1; c <= 8; c *= 2) {
    const int64_t cols = ((v + c - 1) / c + 7) / 8 * 8;
    if (cols * elem * k <= budget) {
      *sc = cols;
      return c;
    }
  }
  return 0;
}

// The cluster kernel in one shape (WIDE: one CTA per SM and twice the
// staging); returns 1 on a CUDA error, and sets *launched.
template <typename TI, typename TO, bool GEO, bool WIDE, int KT = 0>
int launch_mix_cluster(MixParams P, int c, int64_t sc, cudaStream_t s, bool* launched) {
  *launched = false;
  const int nsm = tc_num_sms() > 0 ? tc_num_sms() : 1;
  const size_t smem = (size_t)sc * sizeof(TI) * (size_t)P.k;
  auto kern = k_mix_cluster<TI, TO, GEO, WIDE, KT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return 1;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kMT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // co-resident clusters of this shape (cached per device, cluster size and
  // buffer bytes)
  cfg.gridDim = dim3((unsigned)(c * std::max(1, (WIDE ? 1 : 2) * nsm / c)));
  const int cached_max = max_active_clusters(reinterpret_cast<const void*>(kern), cfg);
  if (cached_max <= 0) return 0;
  P.sc = sc;
  const int64_t clusters = P.n < cached_max ? P.n : cached_max;
  cfg.gridDim = dim3((unsigned)(c * clusters));
  note_launch();
  if (cudaLaunchKernelEx(&cfg, kern, P) != cudaSuccess) return 1;
  *launched = true;
  return 0;
}

template <typename TI, typename TO, bool GEO>
int launch_mix(MixParams P, cudaStream_t s) {
  const int nsm = tc_num_sms() > 0 ? tc_num_sms() : 1;
  int64_t sc = 0;
  bool launched = false;
  int c = mix_cluster_for(P.v, P.k, (int64_t)sizeof(TI), kMixBuf, &sc);
  if constexpr (sizeof(TI) == 2) {  // two bf16 teachers: the teacher loops unrolled
    if (P.k == 2) {
      if (c > 0 && launch_mix_cluster<TI, TO, GEO, false, 2>(P, c, sc, s, &launched)) return 1;
      if (launched) return 0;
    }
  }
  if (c > 0 && launch_mix_cluster<TI, TO, GEO, false>(P, c, sc, s, &launched)) return 1;
  if (launched) return 0;
  c = mix_cluster_for(P.v, P.k, (int64_t)sizeof(TI), kMixBufWide, &sc);
  if (c > 0 && launch_mix_cluster<TI, TO, GEO, true>(P, c, sc, s, &launched)) return 1;
  if (launched) return 0;
  const int grid = (int)std::min<int64_t>(P.n, (int64_t)nsm * 2);
  note_launch();
  k_mix_rows<TI, TO, GEO><<<grid, kMT, 0, s>>>(P);
  return cudaGetLastError() != cudaSuccess;
}

}  // namespace
}  // namespace kd

using namespace kd;

extern "C" {

kd_status kd_mix_teacher_logits(const void* const* logits, int32_t k, const float* weights,
                                int64_t n_tokens, int64_t vocab, int32_t in_dtype,
                                int32_t mode, void* out, int32_t out_dtype,
                                uint32_t* dev_status, void* stream) {
  if (!logits || k < 1 || k > KD_MIX_MAX_TEACHERS || n_tokens < 0 || vocab < 1 ||
      vocab > ((int64_t)1 << 31) || (n_tokens > 0 && !out) ||
      (in_dtype != KD_BF16 && in_dtype != KD_FP32) ||
      (out_dtype != KD_BF16 && out_dtype != KD_FP32) ||
      (mode != KD_MIX_ARITHMETIC && mode != KD_MIX_GEOMETRIC))
    return KD_ERR_INVALID_ARG;
  MixParams P;
  memset(&P, 0, sizeof(P));
  double wsum = 0.0;
  for (int i = 0; i < k; ++i) {
    const double w = weights ? (double)weights[i] : 1.0;
    if (!(w >= 0.0 && w < 1e30)) return KD_ERR_INVALID_ARG;
    if (n_tokens > 0 && !logits[i]) return KD_ERR_INVALID_ARG;
    wsum += w;
  }
  if (!(wsum > 0.0)) return KD_ERR_INVALID_ARG;
  // teachers with weight 0 take no part
  for (int i = 0; i < k; ++i) {
    const double w = (weights ? (double)weights[i] : 1.0) / wsum;
    if (w <= 0.0) continue;
    P.z[P.k] = logits[i];
    P.w[P.k] = (float)w;
    P.lw[P.k] = (float)std::log(w);
    ++P.k;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || !kd_device_supported(dev)) return KD_ERR_NO_DEVICE;
  if (n_tokens == 0) return KD_OK;
  P.n = n_tokens;
  P.v = vocab;
  P.out = out;
  P.status = dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool geo = mode == KD_MIX_GEOMETRIC;
  int e;
  if (in_dtype == KD_BF16) {
    if (out_dtype == KD_BF16)
      e = geo ? launch_mix<__nv_bfloat16, __nv_bfloat16, true>(P, s)
              : launch_mix<__nv_bfloat16, __nv_bfloat16, false>(P, s);
    else
      e = geo ? launch_mix<__nv_bfloat16, float, true>(P, s)
              : launch_mix<__nv_bfloat16, float, false>(P, s);
  } else {
    if (out_dtype == KD_BF16)
      e = geo ? launch_mix<float, __nv_bfloat16, true>(P, s)
              : launch_mix<float, __nv_bfloat16, false>(P, s);
    else
      e = geo ? launch_mix<float, float, true>(P, s) : launch_mix<float, float, false>(P, s);
  }
  return e ? KD_ERR_CUDA : KD_OK;
}

}  // extern "C"
