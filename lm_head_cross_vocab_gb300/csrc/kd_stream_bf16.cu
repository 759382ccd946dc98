// Packed bf16 policies for the TMA-staged streaming kernels (kd_ring.cuh),
// for the common case T_s = T_t in {1, 2}.
//
// The arithmetic is the same as the generic policies (online softmax with the
// q- and p-weighted cross sums of d = a_t - a_s; closed-form gradients), but
// the variant, the temperature shortcut and whether the T = 1 (CE) sums are
// needed are template parameters, so no runtime branch stays in the inner
// loop, and the fp32 work runs on Blackwell's paired fp32 instructions
// (fma/add/mul .f32x2: one instruction for two columns).  Chunk maxima come
// from max.bf16x2 on the raw words.  A streamed logit costs about a dozen
// instructions this way instead of about forty, which is what lets the kernels
// keep up with HBM.
#include <cuda_bf16.h>

#include "kd_internal.h"
#include "kd_ring.cuh"

namespace kd {
namespace {

using bf16 = __nv_bfloat16;

__device__ __forceinline__ float2 splat(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 unpack(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }
__device__ __forceinline__ float2 ex2x2(float2 v) { return make_float2(ex2(v.x), ex2(v.y)); }
__device__ __forceinline__ float hsum(float2 v) { return v.x + v.y; }
// maxima of the even and odd elements of 8 bf16 values, as bf16x2
__device__ __forceinline__ uint32_t max4w(const uint4& u) {
  return max_bf16x2(max_bf16x2(u.x, u.y), max_bf16x2(u.z, u.w));
}
__device__ __forceinline__ float hmax(uint32_t w) { return fmaxf(bf16lo(w), bf16hi(w)); }
__device__ __forceinline__ uint32_t word(const uint4& u, int i) {
  return i == 0 ? u.x : (i == 1 ? u.y : (i == 2 ? u.z : u.w));
}

// ------------------------------------------------------------------ forward
// KLM: bit0 forward cross sums (q d, q (e^{-d} - 1)), bit1 reverse ones,
// bit2 only q (e^{-d} - 1) (the skew variants: the gap between the two
// log-normalisers, to the accuracy of a single term, for their second sweep).
// PW: 1 (T = 1, the CE sums are the tempered ones) or 2 (T = 2, e^{z-m} =
// (e^{(z-m)/2})^2).  NEED1: labels present, so the T = 1 sums are kept.
constexpr float kStale = 8.f;  // log2 of the largest term a stale maximum may leave

template <bool HAS_T, int KLM, int PW, bool NEED1>
struct PackedAcc {
  static constexpr int NA = 1;  // partial-sum sets, shared by the slots of a stage
  static constexpr bool kSecondSweep = KLM == 4;  // the skew variants' policy
  struct Frag {
    uint4 s, t;
  };
  float ms, mt, cq, cp;
  uint32_t ths, tht;  // bf16x2 rescale thresholds: offset + kStale (rounded down)
  float2 osT, otT;  // -m k_T per side (exponent offsets)
  float2 ls1[NA], lsT[NA], lt1[NA], ltT[NA], qd[NA], qx[NA], pd[NA], px[NA];

  __device__ static void load(Frag& f, const uint8_t* buf, int slot, int piece) {
    f.s = *reinterpret_cast<const uint4*>(buf + slot * 16);
    if (HAS_T) f.t = *reinterpret_cast<const uint4*>(buf + piece + slot * 16);
  }
  __device__ static void pick(const Frag& f, int i, float& zs, float& zt) {
    const uint32_t ws = word(f.s, i >> 1);
    zs = (i & 1) ? bf16hi(ws) : bf16lo(ws);
    if (HAS_T) {
      const uint32_t wt = word(f.t, i >> 1);
      zt = (i & 1) ? bf16hi(wt) : bf16lo(wt);
    }
  }
  __device__ void init() {
    ms = mt = neg_inf();
    ths = tht = kNegInfX2;
    cq = cp = 0.f;
    osT = otT = splat(0.f);
#pragma unroll
    for (int j = 0; j < NA; ++j)
      ls1[j] = lsT[j] = lt1[j] = ltT[j] = qd[j] = qx[j] = pd[j] = px[j] = splat(0.f);
  }
  // Rescale the running sums to a larger maximum (rare after a row's first
  // chunks); the same factors as update() in kd_common.cuh.
  __device__ __forceinline__ void grow(float cms, float cmt, const Consts& c) {
    bool grew = false;
    if (cms > ms) {
      const float2 fT = splat(ex2((ms - cms) * c.k_sT));
      const float2 f1 = splat(NEED1 ? ex2((ms - cms) * c.k_s1) : 0.f);
#pragma unroll
      for (int j = 0; j < NA; ++j) {
        lsT[j] = mul2(lsT[j], fT);
        if (KLM & 2) {
          pd[j] = mul2(pd[j], fT);
          px[j] = mul2(px[j], fT);
        }
        if (NEED1) ls1[j] = mul2(ls1[j], f1);
      }
      ms = cms;
      osT = splat(-ms * c.k_sT);
      ths = bf16x2_floor(ms + kStale / c.k_sT);
      grew = true;
    }
    if (HAS_T && cmt > mt && cmt > kNoMass) {  // no-mass chunks never set the offset
      const float2 fT = splat(ex2((mt - cmt) * c.k_tT));
      const float2 f1 = splat(NEED1 ? ex2((mt - cmt) * c.k_t1) : 0.f);
#pragma unroll
      for (int j = 0; j < NA; ++j) {
        ltT[j] = mul2(ltT[j], fT);
        if (KLM & 1) qd[j] = mul2(qd[j], fT);
        if (KLM & 5) qx[j] = mul2(qx[j], fT);
        if (NEED1) lt1[j] = mul2(lt1[j], f1);
      }
      mt = cmt;
      otT = splat(-mt * c.k_tT);
      tht = bf16x2_floor(mt + kStale / c.k_tT);
      grew = true;
    }
    if (HAS_T && grew) {
      const float dM = (ms * c.inv_ts - mt * c.inv_tt) * kL2E;
      cq = ex2(dM);
      cp = ex2(-dM);
    }
  }
  // With a teacher this path has T_s = T_t = T, so d = (t - s) / T: the
  // cross sums keep sum e (t - s) and fold() applies 1/T once.
  __device__ __forceinline__ void pair(int J, uint32_t ws, uint32_t wt, const Consts& c) {
    const float2 s = unpack(ws);
    const float2 es = ex2x2(fma2(s, splat(c.k_sT), osT));
    lsT[J] = add2(lsT[J], es);
    if (NEED1) ls1[J] = PW == 2 ? fma2(es, es, ls1[J]) : add2(ls1[J], es);
    if (HAS_T) {
      const float2 t = unpack(wt);
      const float2 et = ex2x2(fma2(t, splat(c.k_tT), otT));
      ltT[J] = add2(ltT[J], et);
      if (NEED1) lt1[J] = PW == 2 ? fma2(et, et, lt1[J]) : add2(lt1[J], et);
      const float2 dt = sub2(t, s);
      // e^{-d} - 1 terms as (sum + e_s c_q) - e_t: the partial sum is rounded
      // at the size of one term, as fine as ex2's own error
      if (KLM & 1) qd[J] = fma2(et, dt, qd[J]);
      if (KLM & 5) qx[J] = sub2(fma2(es, splat(cq), qx[J]), et);
      if (KLM & 2) {
        pd[J] = fma2(es, dt, pd[J]);  // sum of p d: the state keeps its negative
        px[J] = sub2(fma2(et, splat(cp), px[J]), es);
      }
    }
  }
  __device__ __forceinline__ void slot(int J, const Frag& f, const Consts& c) {
    pair(J, f.s.x, HAS_T ? f.t.x : 0u, c);
    pair(J, f.s.y, HAS_T ? f.t.y : 0u, c);
    pair(J, f.s.z, HAS_T ? f.t.z : 0u, c);
    pair(J, f.s.w, HAS_T ? f.t.w : 0u, c);
  }
  // nv is 0 or 8 here (the vocabulary is a multiple of 8)
  template <int NS>
  __device__ __forceinline__ void step(const Frag (&f)[NS], const int (&nv)[NS], const Consts& c) {
    uint32_t ws = kNegInfX2, wt = kNegInfX2;
#pragma unroll
    for (int j = 0; j < NS; ++j)
      if (nv[j] > 0) {
        ws = j == 0 ? max4w(f[j].s) : max_bf16x2(ws, max4w(f[j].s));
        if (HAS_T) wt = j == 0 ? max4w(f[j].t) : max_bf16x2(wt, max4w(f[j].t));
      }
    // The running maxima are only exponent offsets: a stale one is exact as
    // long as no term exceeds 2^8 (squares 2^16), so the sums are rescaled
    // only when a chunk's maximum passes the offset by that much -- after a
    // row's first chunk, almost never.  The test runs on the raw bf16x2
    // words against a threshold rounded down (a spurious rescale is harmless).
    if (max_bf16x2(ws, ths) != ths || (HAS_T && max_bf16x2(wt, tht) != tht))
      grow(hmax(ws), HAS_T ? hmax(wt) : neg_inf(), c);
#pragma unroll
    for (int j = 0; j < NS; ++j)
      if (nv[j] > 0) slot(j % NA, f[j], c);
  }
  __device__ static float total(const float2 (&v)[NA]) {
    float2 t = v[0];
#pragma unroll
    for (int j = 1; j < NA; ++j) t = add2(t, v[j]);
    return hsum(t);
  }
  __device__ RowState fold(const Consts& c) const {
    RowState st;
    st.init();
    st.ms = ms;
    st.ls1 = total(ls1);
    st.lsT = total(lsT);
    if (HAS_T) {
      st.mt = mt;
      st.lt1 = total(lt1);
      st.ltT = total(ltT);
      st.qd = total(qd) * c.inv_tt;
      st.qx = total(qx);
      st.pd = -total(pd) * c.inv_ts;
      st.px = total(px);
    }
    return st;
  }
};

// ----------------------------------------------------------------- backward
// VAR: KD_KL_FORWARD / REVERSE / JEFFREYS / SKEW_JS (teacher present; unused
// otherwise).  CE: w_sce != 0.  Gradients, with p = softmax(a_s), q =
// softmax(a_t), r = log p - log q - KL(p||q):
//   forward  p - q;   reverse  p r;   Jeffreys  p - q + p r;
//   skew-JS  b p (x - w(x) - KL_pm) (see kl_grad_pq);   top-K  M p;
// each times s_row w_kl T_s, plus s_row w_sce (softmax(z_s) - e_y).
template <bool HAS_T, int VAR, int PW, bool CE>
struct PackedGrad {
  static constexpr int kSlotsFor = HAS_T && (VAR == KD_KL_SKEW_JS || VAR == KD_KL_SKEW_FORWARD ||
                                             VAR == KD_KL_SKEW_REVERSE) ? 1 : 2;
  struct Frag {
    uint4 s, t;
  };
  float ks, ns, kt, nt;  // log2 p = s ks + ns, log2 q = t kt + nt
  float sw, swc, csq, kl_r;
  int64_t y;
  bool zero;
  float sv[KD_STATS_PER_TOKEN];  // skew-JS only
  Consts c;                      // skew-JS only

  __device__ static void load(Frag& f, const uint8_t* buf, int slot, int piece) {
    f.s = *reinterpret_cast<const uint4*>(buf + slot * 16);
    if (HAS_T) f.t = *reinterpret_cast<const uint4*>(buf + piece + slot * 16);
  }
  __device__ void row(const StreamArgs& a, int64_t r) {
    const float* st = a.stats + r * KD_STATS_PER_TOKEN;
    const float scale = a.row_scale[r];
    zero = scale == 0.f;
    ks = a.c.inv_ts * kL2E;
    ns = -st[S_LSE_ST] * kL2E;
    kt = a.c.inv_tt * kL2E;
    nt = HAS_T ? -st[S_LSE_TT] * kL2E : 0.f;
    sw = scale * a.w_kl_ts * (HAS_T ? 1.f : (a.topk ? st[S_MASS] : 0.f));
    swc = CE ? scale * a.w_sce : 0.f;
    csq = (CE && PW == 2) ? swc * ex2((2.f * st[S_LSE_ST] - st[S_LSE_S1]) * kL2E) : swc;
    kl_r = HAS_T ? st[S_KL_REV] : 0.f;
    y = (CE && a.labels) ? a.labels[r] : -1;
    if (HAS_T && is_skew(VAR)) {
      c = a.c;
#pragma unroll
      for (int i = 0; i < KD_STATS_PER_TOKEN; ++i) sv[i] = st[i];
    }
  }
  __device__ __forceinline__ float2 pair(uint32_t ws, uint32_t wt) const {
    const float2 s = unpack(ws);
    const float2 lp2 = fma2(s, splat(ks), splat(ns));
    const float2 p = ex2x2(lp2);
    float2 g = splat(0.f);
    if (HAS_T) {
      const float2 t = unpack(wt);
      const float2 lq2 = fma2(t, splat(kt), splat(nt));
      if (VAR == KD_KL_FORWARD) {
        g = mul2(sub2(p, ex2x2(lq2)), splat(sw));
      } else if (VAR == KD_KL_REVERSE || VAR == KD_KL_JEFFREYS) {
        const float2 r = fma2(sub2(lp2, lq2), splat(1.f / kL2E), splat(-kl_r));
        if (VAR == KD_KL_REVERSE) g = mul2(mul2(p, splat(sw)), r);
        else g = mul2(fma2(p, r, sub2(p, ex2x2(lq2))), splat(sw));
      } else {  // skew variants, two columns per .f32x2 instruction
        const float2 at = mul2(t, splat(c.inv_tt));
        const float2 x =
            add2(fma2(s, splat(c.inv_ts), make_float2(-at.x, -at.y)), splat(sv[S_DLSE]));
        float2 lqm, lpm;
        js_logs2(x, c, lqm, lpm);
        g = mul2(skew_grad2(VAR, p, lqm, lpm, sv[S_KL_PM], sv[S_EPPM], c), splat(sw));
      }
    } else {
      g = mul2(p, splat(sw));
    }
    if (CE) g = fma2(PW == 2 ? mul2(p, p) : p, splat(csq), g);
    return g;
  }
  __device__ __forceinline__ void chunk(const Frag& f, int e0, int, bf16* dz) {
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (!zero) {
      float2 g[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) g[i] = pair(word(f.s, i), HAS_T ? word(f.t, i) : 0u);
      if (CE && (uint64_t)(y - (int64_t)e0) < 8u) {  // the label column: - s_row w_sce
        const int j = (int)(y - e0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (j == 2 * i) g[i].x -= swc;
          if (j == 2 * i + 1) g[i].y -= swc;
        }
      }
      out.x = pack_bf16(g[0].x, g[0].y);
      out.y = pack_bf16(g[1].x, g[1].y);
      out.z = pack_bf16(g[2].x, g[2].y);
      out.w = pack_bf16(g[3].x, g[3].y);
    }
    *reinterpret_cast<uint4*>(dz + e0) = out;
  }
};

// ----------------------------------------------------------------- dispatch
template <bool HAS_T, int KLM, int PW>
void fwd_need(const StreamArgs& a, cudaStream_t s) {
  if (a.c.need_s1) ring::launch_fwd<bf16, HAS_T, PackedAcc<HAS_T, KLM, PW, true>>(a, s);
  else ring::launch_fwd<bf16, HAS_T, PackedAcc<HAS_T, KLM, PW, false>>(a, s);
}
template <bool HAS_T, int KLM>
void fwd_pw(const StreamArgs& a, cudaStream_t s) {
  if (a.c.pw == 2) fwd_need<HAS_T, KLM, 2>(a, s);
  else fwd_need<HAS_T, KLM, 1>(a, s);
}

template <bool HAS_T, int VAR, int PW>
void bwd_ce(const StreamArgs& a, cudaStream_t s) {
  if (a.w_sce != 0.f) ring::launch_bwd<bf16, HAS_T, PackedGrad<HAS_T, VAR, PW, true>>(a, s);
  else ring::launch_bwd<bf16, HAS_T, PackedGrad<HAS_T, VAR, PW, false>>(a, s);
}
template <bool HAS_T, int VAR>
void bwd_pw(const StreamArgs& a, cudaStream_t s) {
  if (a.c.pw == 2) bwd_ce<HAS_T, VAR, 2>(a, s);
  else bwd_ce<HAS_T, VAR, 1>(a, s);
}

bool packed_ok(const StreamArgs& a) {
  if (!a.is_bf16 || (a.c.pw != 1 && a.c.pw != 2)) return false;
  // with a teacher the T = 1 sums of both sides go together
  return a.zt == nullptr || a.c.need_s1 == a.c.need_t1;
}

}  // namespace

bool launch_stream_fwd_packed(const StreamArgs& a, cudaStream_t s) {
  if (!packed_ok(a)) return false;
  if (a.zt == nullptr) {
    fwd_pw<false, 0>(a, s);
    return true;
  }
  if (is_skew(a.variant)) {
    fwd_pw<true, 4>(a, s);
    return true;
  }
  switch (a.c.kl_mode) {
    case 1: fwd_pw<true, 1>(a, s); return true;
    case 2: fwd_pw<true, 2>(a, s); return true;
    case 3: fwd_pw<true, 3>(a, s); return true;
    default: return false;
  }
}

bool launch_stream_bwd_packed(const StreamArgs& a, cudaStream_t s) {
  if (!packed_ok(a)) return false;
  if (a.zt == nullptr) {
    bwd_pw<false, KD_KL_FORWARD>(a, s);
    return true;
  }
  switch (a.variant) {
    case KD_KL_FORWARD: bwd_pw<true, KD_KL_FORWARD>(a, s); return true;
    case KD_KL_REVERSE: bwd_pw<true, KD_KL_REVERSE>(a, s); return true;
    case KD_KL_JEFFREYS: bwd_pw<true, KD_KL_JEFFREYS>(a, s); return true;
    case KD_KL_SKEW_JS: bwd_pw<true, KD_KL_SKEW_JS>(a, s); return true;
    case KD_KL_SKEW_FORWARD: bwd_pw<true, KD_KL_SKEW_FORWARD>(a, s); return true;
    case KD_KL_SKEW_REVERSE: bwd_pw<true, KD_KL_SKEW_REVERSE>(a, s); return true;
    default: return false;
  }
}

}  // namespace kd
