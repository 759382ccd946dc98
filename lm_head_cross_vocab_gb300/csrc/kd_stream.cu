// HBM-streaming path for materialised logits (nemo_automodel KDLoss on
// student_logits / teacher_logits; flash_kd with upcast=True).
//
// Rows that are 16-byte aligned (the usual case) run the TMA-staged ring
// kernels of kd_ring.cuh: a producer warp streams each token row through a
// shared-memory ring with 1-D bulk copies while 16 consumer warps keep the
// online-softmax state (forward) or write d z_s (backward).  This file holds
// their generic per-chunk policies (any dtype, any temperature) and the
// dispatch; kd_stream_bf16.cu holds packed bf16 policies for T = 1 and T = 2.
// Rows that are not 16-byte aligned fall back to the plain kernels below: one
// CTA per row, per-thread loads, skew-JS re-reading the row from L2.
#include <cuda_bf16.h>

#include "kd_internal.h"
#include "kd_ring.cuh"

namespace kd {

namespace {

using ring::ld1;
using ring::st1;
constexpr int kThreads = 512;

// Merge every thread's state into thread 0 (result valid in thread 0 only).
__device__ __forceinline__ void block_merge(RowState& st, const Consts& c, float* sh) {
  for (int o = 16; o > 0; o >>= 1) merge(st, shfl_xor(st, o), c);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) st.store(sh + w * kRec);
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    if (l < nw) st.load(sh + l * kRec);
    else st.init();
    for (int o = 16; o > 0; o >>= 1) merge(st, shfl_xor(st, o), c);
  }
}

__device__ __forceinline__ float3 block_sum3(float a, float b, float d, float* sh) {
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
    d += __shfl_xor_sync(0xffffffffu, d, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    sh[3 * w] = a;
    sh[3 * w + 1] = b;
    sh[3 * w + 2] = d;
  }
  __syncthreads();
  float3 r = make_float3(0.f, 0.f, 0.f);
  if (threadIdx.x == 0)
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
      r.x += sh[3 * i];
      r.y += sh[3 * i + 1];
      r.z += sh[3 * i + 2];
    }
  return r;
}

}  // namespace

// Fallback for rows that are not 16-byte aligned: one CTA per row, plain
// per-thread loads.
template <typename T, bool HAS_T>
__global__ void __launch_bounds__(kThreads) k_stream_fwd(StreamArgs a) {
  __shared__ __align__(16) float sh[32 * kRec];
  __shared__ float sh_lse[2];
  const Consts c = a.c;
  const int64_t V = a.vocab;
  for (int64_t row = blockIdx.x; row < a.n; row += gridDim.x) {
    const T* zs = static_cast<const T*>(a.zs) + row * V;
    const T* zt = HAS_T ? static_cast<const T*>(a.zt) + row * V : nullptr;
    RowState st;
    st.init();
    for (int64_t e0 = threadIdx.x; e0 < V; e0 += 8 * kThreads) {
      float fs[8], ft[8];
      int nv = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t e = e0 + (int64_t)u * kThreads;
        fs[u] = ft[u] = 0.f;
        if (e < V) {
          fs[u] = ld1<T>(zs + e);
          if (HAS_T) ft[u] = ld1<T>(zt + e);
          nv = u + 1;
        }
      }
      update<8, HAS_T, true>(st, fs, ft, nv, c);
    }
    if (a.topk) {  // sparse cross term sum_S p a_s (ids validated by the prep kernel)
      const int32_t* ids = a.sidx + row * a.k;
      const float* ps = a.sp + row * a.k;
      for (int j = threadIdx.x; j < a.k; j += kThreads) {
        const int32_t id = ids[j];
        if (id >= 0 && (int64_t)id < V) st.tk = fmaf(ps[j], ld1<T>(zs + id) * c.inv_ts, st.tk);
      }
    }
    block_merge(st, c, sh);
    if (threadIdx.x == 0) {
      bool valid = true, bad = false;
      if (a.labels) {
        const int64_t y = a.labels[row];
        valid = y != a.ignore;
        bad = valid && (y < 0 || y >= V);
        if (valid && !bad) {
          st.zys = ld1<T>(zs + y);
          if (HAS_T) st.zyt = ld1<T>(zt + y);
        }
      }
      const float mass = a.topk ? a.mass[row] : 0.f, ent = a.topk ? a.ent[row] : 0.f;
      const RowOut o = finalize(st, c, a.variant, HAS_T, a.topk, mass, ent);
      const float nan = __int_as_float(0x7fc00000);
      if (a.ce_s) a.ce_s[row] = !valid ? 0.f : (bad ? nan : o.ce_s);
      if (a.ce_t) a.ce_t[row] = !valid ? 0.f : (bad ? nan : o.ce_t);
      if (a.kl && !(HAS_T && is_skew(a.variant))) a.kl[row] = valid ? o.kl : 0.f;
      float4* s4 = reinterpret_cast<float4*>(a.stats + row * KD_STATS_PER_TOKEN);
      s4[0] = make_float4(o.lse_s1, o.lse_sT, o.lse_t1, o.lse_tT);
      s4[1] = make_float4(o.kl_rev, 0.f, mass, o.dlse);
      sh_lse[0] = o.dlse;
      sh_lse[1] = o.lse_tT;
    }
    if (HAS_T && is_skew(a.variant)) {
      __syncthreads();
      const float dlse = sh_lse[0], lse_tT = sh_lse[1];
      const bool want_x = a.variant != KD_KL_SKEW_JS;
      float jq = 0.f, jp = 0.f, jx = 0.f;
      for (int64_t e = threadIdx.x; e < V; e += kThreads)
        js_terms(ld1<T>(zs + e), ld1<T>(zt + e), lse_tT, dlse, c, jq, jp, jx, want_x);
      const float3 r = block_sum3(jq, jp, jx, sh);
      if (threadIdx.x == 0) {
        const bool v_ok = !a.labels || a.labels[row] != a.ignore;
        a.stats[row * KD_STATS_PER_TOKEN + S_KL_PM] = r.y;
        if (want_x) a.stats[row * KD_STATS_PER_TOKEN + S_EPPM] = r.z;
        if (a.kl) a.kl[row] = v_ok ? skew_kl(a.variant, c.beta, r.x, r.y) : 0.f;
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- backward
// (fallback for unaligned rows)
// d z_s = s_row [ w_sce (softmax(z_s) - e_y) + w_kl T_s dKL/da_s ], exactly 0
// on ignored rows.  Top-K teachers: dKL/da = M softmax(a) - p; the -p part at
// the K support columns is applied by k_stream_bwd_topk afterwards.
template <typename T, bool HAS_T>
__global__ void __launch_bounds__(256) k_stream_bwd(StreamArgs a) {
  const Consts c = a.c;
  const int64_t V = a.vocab;
  constexpr int U = 4;  // 8-element groups per thread per CTA
  for (int64_t row = blockIdx.y; row < a.n; row += gridDim.y) {
    const T* zs = static_cast<const T*>(a.zs) + row * V;
    const T* zt = HAS_T ? static_cast<const T*>(a.zt) + row * V : nullptr;
    T* dz = static_cast<T*>(a.dz) + row * V;
    const float scale = a.row_scale[row];
    const float* stt = a.stats + row * KD_STATS_PER_TOKEN;
    const float lse_s1 = stt[S_LSE_S1], lse_sT = stt[S_LSE_ST], mass = stt[S_MASS];
    int64_t y = -1;
    if (a.labels) y = a.labels[row];
    const float wk = a.w_kl_ts, wc = a.w_sce;
    auto grad = [&](float s, float t, int64_t col) -> float {
      if (scale == 0.f) return 0.f;
      float g = 0.f;
      if (HAS_T) g = wk * kl_grad(s, t, stt, a.variant, c);
      else if (a.topk) g = wk * mass * ex2((s * c.inv_ts - lse_sT) * kL2E);
      if (wc != 0.f) g = fmaf(wc, ex2((s - lse_s1) * kL2E) - (col == y ? 1.f : 0.f), g);
      return scale * g;
    };
    const int64_t e0 = (int64_t)blockIdx.x * (blockDim.x * U * 8) + threadIdx.x;
    for (int u = 0; u < U * 8; ++u) {
      const int64_t e = e0 + (int64_t)u * blockDim.x;
      if (e < V) st1<T>(dz + e, grad(ld1<T>(zs + e), HAS_T ? ld1<T>(zt + e) : 0.f, e));
    }
  }
}

// Sparse correction of the top-K gradient at the support columns: recompute
// the full value in fp32 including the -p_k term (ids are distinct).
template <typename T>
__global__ void k_stream_bwd_topk(StreamArgs a) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= a.n * a.k) return;
  const int64_t row = i / a.k;
  const int32_t id = a.sidx[i];
  if (id < 0 || (int64_t)id >= a.vocab) return;
  const float scale = a.row_scale[row];
  if (scale == 0.f) return;
  const Consts c = a.c;
  const float* stt = a.stats + row * KD_STATS_PER_TOKEN;
  const T* zs = static_cast<const T*>(a.zs) + row * a.vocab;
  const float s = ld1<T>(zs + id);
  float g = a.w_kl_ts * (stt[S_MASS] * ex2((s * c.inv_ts - stt[S_LSE_ST]) * kL2E) - a.sp[i]);
  if (a.w_sce != 0.f) {
    const int64_t y = a.labels ? a.labels[row] : -1;
    g = fmaf(a.w_sce, ex2((s - stt[S_LSE_S1]) * kL2E) - (id == y ? 1.f : 0.f), g);
  }
  st1<T>(static_cast<T*>(a.dz) + row * a.vocab + id, scale * g);
}

// ------------------------------------------------- TMA-staged (aligned rows)
// Generic policies for the ring kernels (kd_ring.cuh): any dtype, any
// temperature.  bf16 problems with T = 1 or T = 2 take the packed policies of
// kd_stream_bf16.cu instead.
namespace {

// 16 bytes of staged values as floats
template <typename T>
__device__ __forceinline__ void raw_to_f(const uint4& u, float* v);
template <>
__device__ __forceinline__ void raw_to_f<__nv_bfloat16>(const uint4& u, float* v) {
  v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
}
template <>
__device__ __forceinline__ void raw_to_f<float>(const uint4& u, float* v) {
  v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
  v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
}

// The slots of a stage stay raw 16-byte words until their turn in step(),
// which converts and folds one slot at a time (registers).
template <typename T, bool HAS_T>
struct GenericAcc {
  static constexpr int EPT = ring::Chunk<T>::EPT;
  static constexpr bool kSecondSweep = true;  // serves every variant
  struct Frag {
    uint4 s, t;
  };
  RowState st;
  __device__ static void load(Frag& f, const uint8_t* buf, int ct, int piece) {
    f.s = *reinterpret_cast<const uint4*>(buf + ct * 16);
    if (HAS_T) f.t = *reinterpret_cast<const uint4*>(buf + piece + ct * 16);
  }
  __device__ static void pick(const Frag& f, int i, float& zs, float& zt) {
    float v[EPT];
    raw_to_f<T>(f.s, v);
#pragma unroll
    for (int u = 0; u < EPT; ++u)
      if (u == i) zs = v[u];
    if (HAS_T) {
      raw_to_f<T>(f.t, v);
#pragma unroll
      for (int u = 0; u < EPT; ++u)
        if (u == i) zt = v[u];
    }
  }
  __device__ void init() { st.init(); }
  template <int NS>
  __device__ void step(const Frag (&f)[NS], const int (&nv)[NS], const Consts& c) {
#pragma unroll 1
    for (int j = 0; j < NS; ++j) {
      float s[EPT], t[EPT];
      raw_to_f<T>(f[j].s, s);
      if (HAS_T) raw_to_f<T>(f[j].t, t);
      if (nv[j] == EPT) update<EPT, HAS_T, false>(st, s, t, EPT, c);
      else if (nv[j] > 0) update<EPT, HAS_T, true>(st, s, t, nv[j], c);
    }
  }
  __device__ RowState fold(const Consts&) const { return st; }
};

// d z_s = s_row [ w_sce (softmax(z_s) - e_y) + w_kl T_s dKL/da_s ] for one
// 16-byte slot; top-K teachers: dKL/da = M softmax(a), the -p part at the K
// support columns is applied by k_stream_bwd_topk afterwards.
template <typename T, bool HAS_T>
struct GenericGrad {
  static constexpr int EPT = ring::Chunk<T>::EPT;
  static constexpr int kSlotsFor = 0;  // from the problem's variant
  struct Frag {
    float s[EPT], t[EPT];
  };
  Consts c;
  float sv[KD_STATS_PER_TOKEN];
  float scale, sq_s, wk, wc;
  int64_t y;
  int variant, topk;
  __device__ static void load(Frag& f, const uint8_t* buf, int ct, int piece) {
    ring::Chunk<T>::load(buf, ct, f.s);
    if (HAS_T) ring::Chunk<T>::load(buf + piece, ct, f.t);
  }
  __device__ void row(const StreamArgs& a, int64_t r) {
    c = a.c;
    variant = a.variant;
    topk = a.topk;
    wk = a.w_kl_ts;
    wc = a.w_sce;
    scale = a.row_scale[r];
#pragma unroll
    for (int i = 0; i < KD_STATS_PER_TOKEN; ++i) sv[i] = a.stats[r * KD_STATS_PER_TOKEN + i];
    y = a.labels ? a.labels[r] : -1;
    sq_s = c.pw == 2 ? ex2((2.f * sv[S_LSE_ST] - sv[S_LSE_S1]) * kL2E) : 0.f;
  }
  __device__ void chunk(const Frag& f, int e0, int nv, T* dz) {
    float g[EPT];
#pragma unroll
    for (int u = 0; u < EPT; ++u) {
      float gg = 0.f;
      if (scale != 0.f) {
        const float lp = fmaf(f.s[u], c.inv_ts, -sv[S_LSE_ST]);
        const float p = ex2(lp * kL2E);
        if (HAS_T) {
          const float lq = fmaf(f.t[u], c.inv_tt, -sv[S_LSE_TT]);
          gg = wk * kl_grad_pq(f.s[u], f.t[u], lp, lq, p, ex2(lq * kL2E), sv, variant, c);
        } else if (topk) {
          gg = wk * sv[S_MASS] * p;
        }
        if (wc != 0.f)
          gg = fmaf(wc, softmax_t1(f.s[u], p, sv[S_LSE_S1], sq_s, c.pw) - (e0 + u == y ? 1.f : 0.f),
                    gg);
        gg *= scale;
      }
      g[u] = gg;
    }
    if (nv == EPT) {
      ring::Chunk<T>::store(dz + e0, g);
    } else {
#pragma unroll
      for (int u = 0; u < EPT; ++u)
        if (u < nv) ring::st1<T>(dz + e0 + u, g[u]);
    }
  }
};

}  // namespace

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
}  // namespace

template <typename T>
static void fwd_dispatch(const StreamArgs& a, cudaStream_t s) {
  const bool vec = (a.vocab % 8 == 0) && a.vocab < (1 << 30) && aligned16(a.zs) &&
                   (!a.zt || aligned16(a.zt));
  const unsigned grid = (unsigned)(a.n < 2147483647 ? a.n : 2147483647);
  const bool has_t = a.zt != nullptr;
  note_launch();
  if (vec) {  // rows 16-byte aligned: TMA-staged ring kernels
    if (launch_stream_fwd_packed(a, s)) return;
    if (has_t) ring::launch_fwd<T, true, GenericAcc<T, true>>(a, s);
    else ring::launch_fwd<T, false, GenericAcc<T, false>>(a, s);
  } else if (has_t) {
    k_stream_fwd<T, true><<<grid, kThreads, 0, s>>>(a);
  } else {
    k_stream_fwd<T, false><<<grid, kThreads, 0, s>>>(a);
  }
}

template <typename T>
static void bwd_dispatch(const StreamArgs& a, cudaStream_t s) {
  const bool vec = (a.vocab % 8 == 0) && a.vocab < (1 << 30) && aligned16(a.zs) &&
                   (!a.zt || aligned16(a.zt)) && aligned16(a.dz);
  const int64_t per_cta = 256 * 4 * 8;
  dim3 grid((unsigned)((a.vocab + per_cta - 1) / per_cta),
            (unsigned)(a.n < 65535 ? a.n : 65535));
  const bool has_t = a.zt != nullptr;
  note_launch();
  if (vec) {  // rows 16-byte aligned: TMA-staged ring kernels
    if (!launch_stream_bwd_packed(a, s)) {
      if (has_t) ring::launch_bwd<T, true, GenericGrad<T, true>>(a, s);
      else ring::launch_bwd<T, false, GenericGrad<T, false>>(a, s);
    }
  } else if (has_t) {
    k_stream_bwd<T, true><<<grid, 256, 0, s>>>(a);
  } else {
    k_stream_bwd<T, false><<<grid, 256, 0, s>>>(a);
  }
  if (a.topk && a.k > 0) {
    const int64_t tot = a.n * a.k;
    note_launch();
    k_stream_bwd_topk<T><<<(unsigned)((tot + 255) / 256), 256, 0, s>>>(a);
  }
}

void launch_stream_fwd(const StreamArgs& a, cudaStream_t s) {
  if (a.n <= 0) return;
  if (a.is_bf16) fwd_dispatch<__nv_bfloat16>(a, s);
  else fwd_dispatch<float>(a, s);
}

void launch_stream_bwd(const StreamArgs& a, cudaStream_t s) {
  if (a.n <= 0) return;
  if (a.is_bf16) bwd_dispatch<__nv_bfloat16>(a, s);
  else bwd_dispatch<float>(a, s);
}

}  // namespace kd
