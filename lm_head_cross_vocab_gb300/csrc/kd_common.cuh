// Device-side building blocks shared by every kernel of the fused LM-head +
// CE + KL loss: the per-token online-softmax state, its chunk update, the
// associative merge of two partial states, and the per-token finalisation.
//
// Online softmax (flash_kd API doc, module description): keep a running max
// and rescale the running sums whenever it grows, so that the vocabulary can
// be visited in any number of chunks with the full-row result.
//
// Per token the state carries, with a_s = z_s/T_s, a_t = z_t/T_t and
// d = a_t - a_s (orda-kernel README, "KL variants": p = student, q = teacher):
//   ms, ls1, lsT : max z_s, sum e^{z_s-ms} (T=1, for CE), sum e^{(z_s-ms)/T_s}
//   mt, lt1, ltT : the same for the teacher
//   qd = sum e^{a_t-Mt} d               -> E_q[d]
//   qx = sum (e^{a_s-Mt} - e^{a_t-Mt})  -> E_q[e^{-d}] - 1
//   pd = sum e^{a_s-Ms} (-d)            -> E_p[-d]
//   px = sum (e^{a_t-Ms} - e^{a_s-Ms})  -> E_p[e^{d}] - 1
// with Ms = ms/T_s, Mt = mt/T_t.  Then
//   KL(q||p) = E_q[d] + log E_q[e^{-d}],   KL(p||q) = E_p[-d] + log E_p[e^{d}],
// and both logs are taken as log1p of the small sums above, which keeps the
// relative error of small divergences at fp32 rounding level instead of the
// absolute error of a difference of two log-sum-exps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kd.h"

namespace kd {

constexpr float kL2E = 1.4426950408889634f;  // log2(e)
constexpr int kRec = 16;                     // floats per partial-state record
// Teacher logits at or below this carry no probability (ids a cross-vocabulary
// projection left unmatched): they never set a running maximum.
constexpr float kNoMass = -1e30f;

// fields of the saved per-token statistics (KD_STATS_PER_TOKEN floats)
// S_DLSE = logsumexp(a_t) - logsumexp(a_s), taken from the accurate log1p form
// of the forward-KL sums rather than from the difference of the two stored values.
// S_MASS holds the top-K mass M for top-K teachers and E_p[p/m] for the
// skew variants (never both).
enum StatField { S_LSE_S1 = 0, S_LSE_ST, S_LSE_T1, S_LSE_TT, S_KL_REV, S_KL_PM, S_MASS, S_DLSE };
constexpr int S_EPPM = S_MASS;

// Variants whose divergence is against the mixture m = (1-b) q + b p (a
// second sweep once both normalisers are known).
__host__ __device__ __forceinline__ bool is_skew(int v) {
  return v == KD_KL_SKEW_JS || v == KD_KL_SKEW_FORWARD || v == KD_KL_SKEW_REVERSE;
}
// The divergence of a skew variant from the second-sweep sums
// jq = KL(q||m) and jp = KL(p||m).
__host__ __device__ __forceinline__ float skew_kl(int v, float beta, float jq, float jp) {
  return v == KD_KL_SKEW_FORWARD ? jq : v == KD_KL_SKEW_REVERSE ? jp
                                                                : (1.f - beta) * jq + beta * jp;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Paired fp32 arithmetic (fma / add / sub / mul .f32x2): one instruction for
// two columns.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// three-input maximum (one instruction on sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// number of valid columns in a chunk of `width` that starts `rem` columns before the end
__device__ __forceinline__ int valid_cols(int64_t rem, int width) {
  return rem <= 0 ? 0 : (rem >= width ? width : (int)rem);
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
// raw bf16x2 words: the larger of each half; x rounded toward -inf into both
// halves; two -inf
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_floor(float x) {
  uint16_t h;
  asm("cvt.rm.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
  return ((uint32_t)h << 16) | h;
}
constexpr uint32_t kNegInfX2 = 0xff80ff80u;

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Constants of one problem, precomputed on the host.
struct Consts {
  float inv_ts, inv_tt;        // 1/T_s, 1/T_t
  float k_s1, k_sT;            // log2e, log2e/T_s   (exponent scales, student)
  float k_t1, k_tT;            // log2e, log2e/T_t
  float beta, log_b, log_1mb;  // b, log b, log(1-b)  (skew-JS)
  int need_s1, need_t1;        // student / teacher CE needed (T = 1 sums)
  int kl_mode;                 // bit0: forward cross sums, bit1: reverse cross sums
  int precise;                 // fp32 problems: libm expm1/log1p in the skew-JS terms
  int pw;                      // 1: T_s (= T_t) == 1, 2: T_s (= T_t) == 2, 0: otherwise
};

struct RowState {
  float ms, ls1, lsT, mt, lt1, ltT, qd, qx, pd, px, zys, zyt, tk, jq, jp, jx;
  float cq, cp;  // cached e^{Ms-Mt}, e^{Mt-Ms} for the current maxima (< 0: stale)

  __device__ __forceinline__ void init() {
    ms = mt = neg_inf();
    ls1 = lsT = lt1 = ltT = qd = qx = pd = px = zys = zyt = tk = jq = jp = jx = 0.f;
    cq = cp = -1.f;
  }
  __device__ __forceinline__ void store(float* r) const {
    float4* o = reinterpret_cast<float4*>(r);
    o[0] = make_float4(ms, ls1, lsT, mt);
    o[1] = make_float4(lt1, ltT, qd, qx);
    o[2] = make_float4(pd, px, zys, zyt);
    o[3] = make_float4(tk, jq, jp, jx);
  }
  __device__ __forceinline__ void load(const float* r) {
    const float4* i = reinterpret_cast<const float4*>(r);
    float4 a = i[0], b = i[1], c = i[2], d = i[3];
    ms = a.x; ls1 = a.y; lsT = a.z; mt = a.w;
    lt1 = b.x; ltT = b.y; qd = b.z; qx = b.w;
    pd = c.x; px = c.y; zys = c.z; zyt = c.w;
    tk = d.x; jq = d.y; jp = d.z; jx = d.w;
    cq = cp = -1.f;
  }
};

// e^{(old-new)*k} with the empty-state convention (old == new covers -inf).
__device__ __forceinline__ float rescale(float m_old, float m_new, float k) {
  return m_old == m_new ? 1.f : ex2((m_old - m_new) * k);
}

// Associative merge of b into a (shuffles, half tiles, vocabulary splits).
__device__ __forceinline__ void merge(RowState& a, const RowState& b, const Consts& c) {
  {
    const float m = fmaxf(a.ms, b.ms);
    const float fa1 = rescale(a.ms, m, c.k_s1), fb1 = rescale(b.ms, m, c.k_s1);
    const float faT = rescale(a.ms, m, c.k_sT), fbT = rescale(b.ms, m, c.k_sT);
    a.ls1 = a.ls1 * fa1 + b.ls1 * fb1;
    a.lsT = a.lsT * faT + b.lsT * fbT;
    a.pd = a.pd * faT + b.pd * fbT;
    a.px = a.px * faT + b.px * fbT;
    a.ms = m;
  }
  {
    const float m = fmaxf(a.mt, b.mt);
    const float fa1 = rescale(a.mt, m, c.k_t1), fb1 = rescale(b.mt, m, c.k_t1);
    const float faT = rescale(a.mt, m, c.k_tT), fbT = rescale(b.mt, m, c.k_tT);
    a.lt1 = a.lt1 * fa1 + b.lt1 * fb1;
    a.ltT = a.ltT * faT + b.ltT * fbT;
    a.qd = a.qd * faT + b.qd * fbT;
    a.qx = a.qx * faT + b.qx * fbT;
    a.mt = m;
  }
  a.zys += b.zys;
  a.zyt += b.zyt;
  a.tk += b.tk;
  a.jq += b.jq;
  a.jp += b.jp;
  a.jx += b.jx;
  a.cq = a.cp = -1.f;
}

__device__ __forceinline__ RowState shfl_xor(const RowState& s, int m) {
  RowState o;
  o.ms = __shfl_xor_sync(0xffffffffu, s.ms, m);
  o.ls1 = __shfl_xor_sync(0xffffffffu, s.ls1, m);
  o.lsT = __shfl_xor_sync(0xffffffffu, s.lsT, m);
  o.mt = __shfl_xor_sync(0xffffffffu, s.mt, m);
  o.lt1 = __shfl_xor_sync(0xffffffffu, s.lt1, m);
  o.ltT = __shfl_xor_sync(0xffffffffu, s.ltT, m);
  o.qd = __shfl_xor_sync(0xffffffffu, s.qd, m);
  o.qx = __shfl_xor_sync(0xffffffffu, s.qx, m);
  o.pd = __shfl_xor_sync(0xffffffffu, s.pd, m);
  o.px = __shfl_xor_sync(0xffffffffu, s.px, m);
  o.zys = __shfl_xor_sync(0xffffffffu, s.zys, m);
  o.zyt = __shfl_xor_sync(0xffffffffu, s.zyt, m);
  o.tk = __shfl_xor_sync(0xffffffffu, s.tk, m);
  o.jq = __shfl_xor_sync(0xffffffffu, s.jq, m);
  o.jp = __shfl_xor_sync(0xffffffffu, s.jp, m);
  o.jx = __shfl_xor_sync(0xffffffffu, s.jx, m);
  o.cq = o.cp = -1.f;
  return o;
}

// Merge the RowStates of the 32 lanes of a warp (result in every lane): the
// maxima first, then every lane rescales its sums once to the warp maxima,
// then plain sum reductions -- the same result as merge() over the lanes with
// one exponential per sum instead of one per level.
__device__ __forceinline__ void warp_merge(RowState& s, const Consts& c) {
  float m_s = s.ms, m_t = s.mt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m_s = fmaxf(m_s, __shfl_xor_sync(0xffffffffu, m_s, o));
    m_t = fmaxf(m_t, __shfl_xor_sync(0xffffffffu, m_t, o));
  }
  const float fs1 = rescale(s.ms, m_s, c.k_s1), fsT = rescale(s.ms, m_s, c.k_sT);
  const float ft1 = rescale(s.mt, m_t, c.k_t1), ftT = rescale(s.mt, m_t, c.k_tT);
  float v[14] = {s.ls1 * fs1, s.lsT * fsT, s.pd * fsT, s.px * fsT, s.lt1 * ft1, s.ltT * ftT,
                 s.qd * ftT, s.qx * ftT, s.zys, s.zyt, s.tk, s.jq, s.jp, s.jx};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int i = 0; i < 14; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
  }
  s.ms = m_s;
  s.mt = m_t;
  s.ls1 = v[0];
  s.lsT = v[1];
  s.pd = v[2];
  s.px = v[3];
  s.lt1 = v[4];
  s.ltT = v[5];
  s.qd = v[6];
  s.qx = v[7];
  s.zys = v[8];
  s.zyt = v[9];
  s.tk = v[10];
  s.jq = v[11];
  s.jp = v[12];
  s.jx = v[13];
  s.cq = s.cp = -1.f;
}

// Sums of one chunk against fixed maxima (see update()).  PW: how the T = 1
// sums follow from the tempered ones (0: own exponential, 1: equal, 2: square).
template <int NC, bool HAS_T, bool MASKED, int PW>
__device__ __forceinline__ void accum(const float* zs, const float* zt, int nvalid,
                                      const Consts& c, float os1, float osT, float ot1, float otT,
                                      float& ls1, float& lsT, float& lt1, float& ltT, float& qd,
                                      float& qx, float& pd, float& px, float cq, float cp) {
  if constexpr (!HAS_T) {
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      if (!MASKED || j < nvalid) {
        const float es = ex2(fmaf(zs[j], c.k_sT, osT));
        lsT += es;
        if (c.need_s1) {
          if (PW == 2) ls1 = fmaf(es, es, ls1);
          else if (PW == 1) ls1 += es;
          else ls1 += ex2(fmaf(zs[j], c.k_s1, os1));
        }
      }
    }
  } else {
    // e^{a_s-Mt} = e^{a_s-Ms} * cq and e^{a_t-Ms} = e^{a_t-Mt} * cp.  Both
    // directions' cross sums and (T = 1 or 2) the CE sums cost a few FMAs each,
    // less than a branch per element, so they are always formed; finalize()
    // reads only what the variant needs (an overflowed unused sum falls back to
    // the log-sum-exp difference there).
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      if (!MASKED || j < nvalid) {
        const float es = ex2(fmaf(zs[j], c.k_sT, osT));
        const float et = ex2(fmaf(zt[j], c.k_tT, otT));
        lsT += es;
        ltT += et;
        const float d = zt[j] * c.inv_tt - zs[j] * c.inv_ts;
        qd = fmaf(et, d, qd);
        qx += fmaf(es, cq, -et);
        pd = fmaf(es, -d, pd);
        px += fmaf(et, cp, -es);
        if (PW == 2) {
          ls1 = fmaf(es, es, ls1);
          lt1 = fmaf(et, et, lt1);
        } else if (PW == 1) {
          ls1 += es;
          lt1 += et;
        }
      }
    }
    if (PW == 0) {
      if (c.need_s1) {
#pragma unroll
        for (int j = 0; j < NC; ++j)
          if (!MASKED || j < nvalid) ls1 += ex2(fmaf(zs[j], c.k_s1, os1));
      }
      if (c.need_t1) {
#pragma unroll
        for (int j = 0; j < NC; ++j)
          if (!MASKED || j < nvalid) lt1 += ex2(fmaf(zt[j], c.k_t1, ot1));
      }
    }
  }
}

// accum() over NC columns (all valid, NC even) two at a time on the paired
// fp32 instructions, with a teacher: the same terms, each column pair's sums
// kept in a float2 and added up at the end.  The e^{-d} - 1 terms accumulate
// as (sum + e_s c_q) - e_t, so the partial sum is rounded at the size of one
// term (as fine as ex2's own error); pd is summed as e_s d and negated once.
template <int NC, int PW>
__device__ __forceinline__ void accum_pairs(const float* zs, const float* zt, const Consts& c,
                                            float osT, float otT, float& ls1, float& lsT,
                                            float& lt1, float& ltT, float& qd, float& qx,
                                            float& pd, float& px, float cq, float cp) {
  const float2 ksT = make_float2(c.k_sT, c.k_sT), oS = make_float2(osT, osT);
  const float2 ktT = make_float2(c.k_tT, c.k_tT), oT = make_float2(otT, otT);
  const float2 itt = make_float2(c.inv_tt, c.inv_tt), nits = make_float2(-c.inv_ts, -c.inv_ts);
  const float2 cq2 = make_float2(cq, cq), cp2 = make_float2(cp, cp);
  const float2 z = make_float2(0.f, 0.f);
  float2 s1 = z, sT = z, t1 = z, tT = z, sqd = z, sqx = z, spd = z, spx = z;
#pragma unroll
  for (int j = 0; j < NC; j += 2) {
    const float2 a_s = make_float2(zs[j], zs[j + 1]), a_t = make_float2(zt[j], zt[j + 1]);
    const float2 gs = fma2(a_s, ksT, oS), gt = fma2(a_t, ktT, oT);
    const float2 es = make_float2(ex2(gs.x), ex2(gs.y));
    const float2 et = make_float2(ex2(gt.x), ex2(gt.y));
    sT = add2(sT, es);
    tT = add2(tT, et);
    const float2 d = fma2(a_t, itt, mul2(a_s, nits));
    sqd = fma2(et, d, sqd);
    sqx = sub2(fma2(es, cq2, sqx), et);
    spd = fma2(es, d, spd);
    spx = sub2(fma2(et, cp2, spx), es);
    if (PW == 2) {
      s1 = fma2(es, es, s1);
      t1 = fma2(et, et, t1);
    } else if (PW == 1) {
      s1 = add2(s1, es);
      t1 = add2(t1, et);
    }
  }
  lsT += sT.x + sT.y;
  ltT += tT.x + tT.y;
  qd += sqd.x + sqd.y;
  qx += sqx.x + sqx.y;
  pd -= spd.x + spd.y;
  px += spx.x + spx.y;
  if (PW != 0) {
    ls1 += s1.x + s1.y;
    lt1 += t1.x + t1.y;
  }
}

// Chunk update of the online state with NC columns of student (and, when
// HAS_T, teacher) logits.  With MASKED, only the first `nvalid` columns count
// (the ragged end of the vocabulary).
template <int NC, bool HAS_T, bool MASKED, bool PAIRS = false>
__device__ __forceinline__ void update(RowState& st, const float* zs, const float* zt,
                                       int nvalid, const Consts& c) {
  static_assert(!PAIRS || (!MASKED && NC % 2 == 0), "paired columns: whole, even chunks");
  float cms = neg_inf(), cmt = neg_inf();
  if constexpr (PAIRS) {
#pragma unroll
    for (int j = 0; j < NC; j += 2) {
      cms = fmax3(cms, zs[j], zs[j + 1]);
      if (HAS_T) cmt = fmax3(cmt, zt[j], zt[j + 1]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      if (!MASKED || j < nvalid) {
        cms = fmaxf(cms, zs[j]);
        if (HAS_T) cmt = fmaxf(cmt, zt[j]);
      }
    }
  }
  if (MASKED && nvalid <= 0) return;
  // The running maxima are only exponent offsets: a stale one is exact while
  // no term exceeds 2^8, so the sums are rescaled only when a chunk's maximum
  // passes the offset by that much on either exponent scale (T = 1 or T) --
  // after a row's first chunk, almost never, and never divergently per chunk.
  const float kss = fmaxf(c.k_s1, c.k_sT), kst = fmaxf(c.k_t1, c.k_tT);
  const bool grow_s = (cms - st.ms) * kss > 8.f;
  const bool grow_t = HAS_T && cmt > kNoMass && (cmt - st.mt) * kst > 8.f;
  bool grew = false;
  if (grow_s) {
    const float f1 = ex2((st.ms - cms) * c.k_s1), fT = ex2((st.ms - cms) * c.k_sT);
    st.ls1 *= f1;
    st.lsT *= fT;
    st.pd *= fT;
    st.px *= fT;
    st.ms = cms;
    grew = true;
  }
  if (grow_t) {
    const float f1 = ex2((st.mt - cmt) * c.k_t1), fT = ex2((st.mt - cmt) * c.k_tT);
    st.lt1 *= f1;
    st.ltT *= fT;
    st.qd *= fT;
    st.qx *= fT;
    st.mt = cmt;
    grew = true;
  }
  const float ms = st.ms, mt = HAS_T ? st.mt : 0.f;
  if (HAS_T && (grew || st.cq < 0.f)) {
    const float dM = (ms * c.inv_ts - mt * c.inv_tt) * kL2E;
    st.cq = ex2(dM);
    st.cp = ex2(-dM);
  }
  const float cq = st.cq, cp = st.cp;
  const float os1 = -ms * c.k_s1, osT = -ms * c.k_sT;
  // a teacher offset never set (no teacher mass yet) contributes nothing: the
  // no-mass logits still give e^{...} = 0, without -inf + inf
  const float mt_off = mt > kNoMass ? mt : 0.f;
  const float ot1 = -mt_off * c.k_t1, otT = -mt_off * c.k_tT;
  float ls1 = 0.f, lsT = 0.f, lt1 = 0.f, ltT = 0.f, qd = 0.f, qx = 0.f, pd = 0.f, px = 0.f;
  // T = 1 sums (for CE): with T = 1 they are the tempered sums; with T = 2,
  // e^{z-m} = (e^{(z-m)/2})^2 exactly, so neither needs its own exponential.
  if (PAIRS && HAS_T && c.pw != 0) {
    if (c.pw == 2)
      accum_pairs<NC, 2>(zs, zt, c, osT, otT, ls1, lsT, lt1, ltT, qd, qx, pd, px, cq, cp);
    else
      accum_pairs<NC, 1>(zs, zt, c, osT, otT, ls1, lsT, lt1, ltT, qd, qx, pd, px, cq, cp);
  } else if (c.pw == 2) {
    accum<NC, HAS_T, MASKED, 2>(zs, zt, nvalid, c, os1, osT, ot1, otT, ls1, lsT, lt1, ltT, qd,
                                qx, pd, px, cq, cp);
  } else if (c.pw == 1) {
    accum<NC, HAS_T, MASKED, 1>(zs, zt, nvalid, c, os1, osT, ot1, otT, ls1, lsT, lt1, ltT, qd,
                                qx, pd, px, cq, cp);
  } else {
    accum<NC, HAS_T, MASKED, 0>(zs, zt, nvalid, c, os1, osT, ot1, otT, ls1, lsT, lt1, ltT, qd,
                                qx, pd, px, cq, cp);
  }
  st.ls1 += ls1;
  st.lsT += lsT;
  st.lt1 += lt1;
  st.ltT += ltT;
  st.qd += qd;
  st.qx += qx;
  st.pd += pd;
  st.px += px;
}

// log E[e^{x}] from its "minus 1" form when that is finite and well inside
// the log1p domain, else from the difference of the two log-sum-exps.
__device__ __forceinline__ float log_mean_exp(float x_minus_1, float lse_diff) {
  return (isfinite(x_minus_1) && x_minus_1 > -0.5f) ? log1pf(x_minus_1) : lse_diff;
}

struct RowOut {
  float ce_s, ce_t, kl, lse_s1, lse_sT, lse_t1, lse_tT, kl_rev, kl_pm, dlse;
};

// Finalise one token.  variant: KD_KL_*; topk: sparse objective with mass M
// and entropy E = sum_S p log p (Full-Chunked-KL-Loss README, "Methods").
__device__ __forceinline__ RowOut finalize(const RowState& s, const Consts& c, int variant,
                                           bool has_t, bool topk, float mass, float ent) {
  RowOut o;
  o.lse_s1 = s.ms + logf(s.ls1);
  o.lse_sT = s.ms * c.inv_ts + logf(s.lsT);
  o.ce_s = o.lse_s1 - s.zys;
  o.lse_t1 = o.lse_tT = 0.f;
  o.ce_t = 0.f;
  o.kl_rev = o.kl_pm = o.dlse = 0.f;
  o.kl = 0.f;
  if (topk) {
    o.kl = ent - s.tk + mass * o.lse_sT;
  } else if (has_t) {
    o.lse_t1 = s.mt + logf(s.lt1);
    o.lse_tT = s.mt * c.inv_tt + logf(s.ltT);
    o.ce_t = o.lse_t1 - s.zyt;
    // log E_q[e^{-d}] = logsumexp(a_s) - logsumexp(a_t)
    const float lme_q = log_mean_exp(s.qx / s.ltT, o.lse_sT - o.lse_tT);
    o.dlse = -lme_q;
    const float kl_f = s.qd / s.ltT + lme_q;
    const float kl_r = s.pd / s.lsT + log_mean_exp(s.px / s.lsT, o.lse_tT - o.lse_sT);
    o.kl_rev = kl_r;
    if (variant == KD_KL_FORWARD) o.kl = kl_f;
    else if (variant == KD_KL_REVERSE) o.kl = kl_r;
    else if (variant == KD_KL_JEFFREYS) o.kl = kl_f + kl_r;
    else {  // skew variants: second-pass sums jq = sum q log(q/m), jp = sum p log(p/m)
      o.kl_pm = s.jp;
      o.kl = skew_kl(variant, c.beta, s.jq, s.jp);
    }
  }
  return o;
}

// Skew-JS logarithms from x = log p - log q = (a_s - a_t) + (lse(a_t) - lse(a_s)),
// with m = (1-b) q + b p:
//   x <= 0:  l = log(m/q) = log1p(b expm1(x)),      log(q/m) = -l,  log(p/m) = x - l
//   x >  0:  l = log(m/p) = log1p((1-b) expm1(-x)),  log(p/m) = -l,  log(q/m) = -x - l
// No form subtracts two large values, and an id with q = 0 (a teacher id no
// token maps to: x huge) still gives log(p/m) = -log b exactly.  The precise
// form (fp32 problems: libm expm1 / log1p) keeps the relative accuracy of each
// term near x = 0.  The fast form (bf16 problems) takes e^{-|x|} from ex2 and
// the logarithm from __logf of 1 + coef (e - 1), each with an absolute error of
// about 1e-7 near x = 0; summed over a row this stays at the ~1e-7 absolute
// floor that the fp32 accumulation of every variant has anyway, so skew
// divergences below ~1e-4 per token are resolved to about 1e-7 absolute rather
// than to their relative tolerance (bf16 logits cannot hold distributions
// closer than their 2^-8 resolution).
__device__ __forceinline__ void js_logs(float x, const Consts& c, float& lqm, float& lpm) {
  const bool neg = x <= 0.f;
  const float coef = neg ? c.beta : 1.f - c.beta;
  const float y = neg ? x : -x;
  float l;
  if (c.precise) {
    l = log1pf(coef * expm1f(y));
  } else {
    l = __logf(fmaf(coef, ex2(y * kL2E) - 1.f, 1.f));
  }
  lqm = neg ? -l : -x - l;
  lpm = neg ? x - l : -l;
}

// Skew second pass: with the final normalisers known, accumulate
// jq += q log(q/m), jp += p log(p/m) and, when the variant's gradient needs
// E_p[p/m] (skew-forward, skew-reverse), jx += p (p/m).  p and q come each
// from its own log-normaliser, so neither inherits the other's range.
__device__ __forceinline__ void js_terms(float zs, float zt, float lse_tT, float dlse,
                                         const Consts& c, float& jq, float& jp, float& jx,
                                         bool want_x) {
  const float x = fmaf(zs, c.inv_ts, -zt * c.inv_tt) + dlse;
  const float lq = zt * c.inv_tt - lse_tT;
  const float lp = fmaf(zs, c.inv_ts, dlse - lse_tT);  // a_s - lse(a_s)
  float lqm, lpm;
  js_logs(x, c, lqm, lpm);
  const float q = ex2(lq * kL2E), p = ex2(lp * kL2E);
  jq = fmaf(q, lqm, jq);
  jp = fmaf(p, lpm, jp);
  if (want_x) jx = fmaf(p, ex2(lpm * kL2E), jx);
}

// js_logs for two columns (the fast path): log(q/m), log(p/m) from x = log p - log q
__device__ __forceinline__ void js_logs2(float2 x, const Consts& c, float2& lqm, float2& lpm) {
  const bool n0 = x.x <= 0.f, n1 = x.y <= 0.f;
  const float2 yl = make_float2(-fabsf(x.x) * kL2E, -fabsf(x.y) * kL2E);
  const float2 coef = make_float2(n0 ? c.beta : 1.f - c.beta, n1 ? c.beta : 1.f - c.beta);
  const float2 t = fma2(coef, make_float2(ex2(yl.x) - 1.f, ex2(yl.y) - 1.f), make_float2(1.f, 1.f));
  const float2 l = make_float2(__logf(t.x), __logf(t.y));
  const float2 xl = add2(x, l);
  lqm = make_float2(n0 ? -l.x : -xl.x, n1 ? -l.y : -xl.y);
  lpm = sub2(make_float2(n0 ? x.x : 0.f, n1 ? x.y : 0.f), l);
}

// skew_grad for two columns, p and the logs of js_logs2 given
__device__ __forceinline__ float2 skew_grad2(int variant, float2 p, float2 lqm, float2 lpm,
                                             float kl_pm, float eppm, const Consts& c) {
  const float b = c.beta;
  if (variant == KD_KL_SKEW_FORWARD) {
    const float eqm = (1.f - b * eppm) / (1.f - b);
    const float2 e = make_float2(ex2(lqm.x * kL2E) - eqm, ex2(lqm.y * kL2E) - eqm);
    return mul2(mul2(p, make_float2(-b, -b)), e);
  }
  const float2 d = sub2(lpm, make_float2(kl_pm, kl_pm));
  if (variant == KD_KL_SKEW_REVERSE) {
    const float2 e = make_float2(ex2(lpm.x * kL2E) - eppm, ex2(lpm.y * kL2E) - eppm);
    return mul2(p, fma2(make_float2(-b, -b), e, d));
  }
  return mul2(mul2(p, make_float2(b, b)), d);
}

// js_terms for two columns at once (the fast, non-precise path), the fp32
// arithmetic on .f32x2 pairs; the sums stay per lane.
__device__ __forceinline__ void js_terms2(float2 zs, float2 zt, float lse_tT, float dlse,
                                          const Consts& c, float2& jq, float2& jp, float2& jx,
                                          bool want_x) {
  const float2 its = make_float2(c.inv_ts, c.inv_ts), itt = make_float2(c.inv_tt, c.inv_tt);
  const float2 l2e = make_float2(kL2E, kL2E);
  const float2 at = mul2(zt, itt);
  const float2 x = add2(fma2(zs, its, make_float2(-at.x, -at.y)), make_float2(dlse, dlse));
  const float2 lq = sub2(at, make_float2(lse_tT, lse_tT));
  const float2 lp = fma2(zs, its, make_float2(dlse - lse_tT, dlse - lse_tT));
  // per column: y = -|x| and the weight of the smaller distribution
  const bool n0 = x.x <= 0.f, n1 = x.y <= 0.f;
  const float2 y = make_float2(-fabsf(x.x), -fabsf(x.y));
  const float2 coef = make_float2(n0 ? c.beta : 1.f - c.beta, n1 ? c.beta : 1.f - c.beta);
  const float2 yl = mul2(y, l2e);
  const float2 e = make_float2(ex2(yl.x), ex2(yl.y));
  const float2 t = fma2(coef, add2(e, make_float2(-1.f, -1.f)), make_float2(1.f, 1.f));
  const float2 l = make_float2(__logf(t.x), __logf(t.y));
  const float2 xl = add2(x, l);  // -(lqm) when x > 0
  const float2 lqm = make_float2(n0 ? -l.x : -xl.x, n1 ? -l.y : -xl.y);
  const float2 lpm = sub2(make_float2(n0 ? x.x : 0.f, n1 ? x.y : 0.f), l);
  const float2 a2 = mul2(lq, l2e), b2 = mul2(lp, l2e);
  const float2 q = make_float2(ex2(a2.x), ex2(a2.y));
  const float2 p = make_float2(ex2(b2.x), ex2(b2.y));
  jq = fma2(q, lqm, jq);
  jp = fma2(p, lpm, jp);
  if (want_x) {
    const float2 r = mul2(lpm, l2e);
    jx = fma2(p, make_float2(ex2(r.x), ex2(r.y)), jx);
  }
}

// Second sweep of the skew variants on bf16 rows, the fast form in base 2.
// Per column, with x2 = log2 p - log2 q, the larger of p and q is
// B = 2^max(log2 p, log2 q) and the smaller is B e, e = 2^-|x2|; m divided by
// the larger is t = 1 + w (e - 1), w the mixture weight of the smaller (b when
// p <= q, 1 - b otherwise), and l = log2 t.  Then, in base-2 units,
//   p <= q:  q log(q/m) = -B l,        p log(p/m) = -B v
//   p >  q:  p log(p/m) = -B l,        q log(q/m) = -B v,    v = e (|x2| + l)
// so the sums of the two sides are (S + D)/2 and (S - D)/2 with S = sum B (l + v)
// and D = sum B (v - l) sign(x2): the case split becomes a sign-bit transfer
// (w = 1/2 + (1/2 - b) sign(x2) likewise), no compare or select per column.
// With E_p[p/m]: p (p/m) = B g^2 / t, g = e (p <= q) or 1, 1/t = 2^-l.
// Three transcendentals a column (two ex2 and one lg2; one more ex2 for
// E_p[p/m]).  x2 is formed in the natural scale first (a_s - a_t + dlse, exact
// products for power-of-two temperatures) so that it keeps its absolute
// accuracy near 0; only the weight B comes from tempered logits minus their
// log-normalisers.  At x2 = 0 both cases agree (e = 1, t = 1, v = l = 0), so
// the sign of a zero does not matter.  A teacher logit at the lowest finite
// value (no mass) may overflow x2 to infinity: e is then 0 and only the sign
// of x2 and 2^-|x2| are taken from it.
struct SkewK {
  float2 its, nitt;  // 1/T_s and -1/T_t
  float2 dl, l2e;    // dlse, log2 e
  float2 ks, kt;     // log2 e / T_s, log2 e / T_t
  float2 cp, cq;     // (dlse - lse_tT) log2 e, -lse_tT log2 e
  float hb;          // 1/2 - b
};
__device__ __forceinline__ SkewK skew_consts(const Consts& c, float lse_tT, float dlse) {
  SkewK k;
  k.its = make_float2(c.inv_ts, c.inv_ts);
  k.nitt = make_float2(-c.inv_tt, -c.inv_tt);
  k.dl = make_float2(dlse, dlse);
  k.l2e = make_float2(kL2E, kL2E);
  k.ks = make_float2(c.inv_ts * kL2E, c.inv_ts * kL2E);
  k.kt = make_float2(c.inv_tt * kL2E, c.inv_tt * kL2E);
  const float cp = (dlse - lse_tT) * kL2E, cq = -lse_tT * kL2E;
  k.cp = make_float2(cp, cp);
  k.cq = make_float2(cq, cq);
  k.hb = 0.5f - c.beta;
  return k;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// a with the sign bit of b flipped into it (a xor (b & sign))
__device__ __forceinline__ float sign_xor(float a, float b) {
  return __uint_as_float(__float_as_uint(a) ^ (__float_as_uint(b) & 0x80000000u));
}
// Two columns: sv accumulates B (l + v), dv accumulates B (v - l) sign(x2)
// (base 2: jq = -ln2 (sv + dv) / 2, jp = -ln2 (sv - dv) / 2); ax accumulates
// p (p/m) when WANT_X.
template <bool WANT_X>
__device__ __forceinline__ void skew_pair_b2(float2 s, float2 t, const SkewK& k, float2& sv,
                                             float2& dv, float2& ax) {
  const float2 xn = add2(fma2(s, k.its, mul2(t, k.nitt)), k.dl);  // ln p - ln q
  const float2 x2 = mul2(xn, k.l2e);
  const float2 lp = fma2(s, k.ks, k.cp), lq = fma2(t, k.kt, k.cq);
  const float2 e = make_float2(ex2(-fabsf(x2.x)), ex2(-fabsf(x2.y)));
  const float2 B = make_float2(ex2(fmaxf(lp.x, lq.x)), ex2(fmaxf(lp.y, lq.y)));
  // w - 1/2 = (1/2 - b) sign(x2); t = 1 + w (e - 1) = (1 + e)/2 + (w - 1/2)(e - 1)
  const float2 h = make_float2(sign_xor(k.hb, x2.x), sign_xor(k.hb, x2.y));
  const float2 half = make_float2(0.5f, 0.5f);
  const float2 tt = fma2(h, add2(e, make_float2(-1.f, -1.f)), fma2(e, half, half));
  const float2 l = make_float2(lg2(tt.x), lg2(tt.y));
  // v = e l + (e log2 e) |xn|: xn stays finite where x2 may not (a projected
  // teacher's lowest finite logit at T_t = 1), and e = 0 there
  const float2 el = mul2(e, l), ek = mul2(e, k.l2e);
  const float2 v = make_float2(fmaf(ek.x, fabsf(xn.x), el.x), fmaf(ek.y, fabsf(xn.y), el.y));
  const float2 d = sub2(v, l);
  sv = fma2(B, add2(l, v), sv);
  dv = fma2(B, make_float2(sign_xor(d.x, x2.x), sign_xor(d.y, x2.y)), dv);
  if constexpr (WANT_X) {
    const float2 g = make_float2(x2.x <= 0.f ? e.x : 1.f, x2.y <= 0.f ? e.y : 1.f);
    const float2 r = make_float2(ex2(-l.x), ex2(-l.y));
    ax = fma2(mul2(mul2(B, g), g), r, ax);
  }
}

// d KL / d a_s of the skew variants (teacher detached), from p, log(q/m),
// log(p/m), KL(p||m) and E_p[p/m] (with (1-b) q/m + b p/m = 1):
//   skew-JS       b p (log(p/m) - KL(p||m))
//   skew-forward  -b p (q/m - E_p[q/m]),  E_p[q/m] = (1 - b E_p[p/m]) / (1 - b)
//   skew-reverse  p (log(p/m) - KL(p||m)) - b p (p/m - E_p[p/m])
__device__ __forceinline__ float skew_grad(int variant, float p, float lqm, float lpm,
                                           float kl_pm, float eppm, const Consts& c) {
  const float b = c.beta;
  if (variant == KD_KL_SKEW_FORWARD) {
    const float eqm = (1.f - b * eppm) / (1.f - b);
    return -b * p * (ex2(lqm * kL2E) - eqm);
  }
  if (variant == KD_KL_SKEW_REVERSE)
    return p * (lpm - kl_pm) - b * p * (ex2(lpm * kL2E) - eppm);
  return b * p * (lpm - kl_pm);
}

// Gradient of the KL part w.r.t. a_s (teacher detached), per element, from
// the saved statistics:
//   forward  p - q;  reverse p (log p - log q - KL(p||q));  Jeffreys the sum;
//   skew variants: skew_grad().
__device__ __forceinline__ float kl_grad(float zs, float zt, const float* stt, int variant,
                                         const Consts& c) {
  const float lp = zs * c.inv_ts - stt[S_LSE_ST];
  const float lq = zt * c.inv_tt - stt[S_LSE_TT];
  const float p = ex2(lp * kL2E);
  if (is_skew(variant)) {
    const float x = fmaf(zs, c.inv_ts, -zt * c.inv_tt) + stt[S_DLSE];
    float lqm, lpm;
    js_logs(x, c, lqm, lpm);
    return skew_grad(variant, p, lqm, lpm, stt[S_KL_PM], stt[S_EPPM], c);
  }
  float g = 0.f;
  if (variant != KD_KL_REVERSE) g = p - ex2(lq * kL2E);
  if (variant != KD_KL_FORWARD) g = fmaf(p, lp - lq - stt[S_KL_REV], g);
  return g;
}

// Same gradient from already computed lp = log p, lq = log q, p = e^lp, q = e^lq.
__device__ __forceinline__ float kl_grad_pq(float zs, float zt, float lp, float lq, float p,
                                            float q, const float* stt, int variant,
                                            const Consts& c) {
  if (is_skew(variant)) {
    const float x = fmaf(zs, c.inv_ts, -zt * c.inv_tt) + stt[S_DLSE];
    float lqm, lpm;
    js_logs(x, c, lqm, lpm);
    return skew_grad(variant, p, lqm, lpm, stt[S_KL_PM], stt[S_EPPM], c);
  }
  float g = 0.f;
  if (variant != KD_KL_REVERSE) g = p - q;
  if (variant != KD_KL_FORWARD) g = fmaf(p, lp - lq - stt[S_KL_REV], g);
  return g;
}

// softmax(z) = e^{z - lse(z)} from p = e^{z/T - lse(z/T)} when T is 1 or 2
// (pw as in Consts; sq = e^{2 lse(z/2) - lse(z)} per row), else directly.
__device__ __forceinline__ float softmax_t1(float z, float p, float lse1, float sq, int pw) {
  if (pw == 2) return p * p * sq;
  if (pw == 1) return p;
  return ex2((z - lse1) * kL2E);
}

__device__ __forceinline__ void set_status(uint32_t* st, uint32_t bits) {
  if (st) atomicOr(st, bits);
}

}  // namespace kd
