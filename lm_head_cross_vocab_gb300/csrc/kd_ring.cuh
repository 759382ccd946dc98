// TMA-staged streaming of materialised logit rows (kd_stream.cu and
// kd_stream_bf16.cu).
//
// One persistent CTA per SM.  A producer warp copies each token row in
// kChunk-byte pieces (z_s and, with a teacher, z_t) into a kStages-deep
// shared-memory ring with 1-D bulk copies (cp.async.bulk, completion counted
// on an mbarrier); kCW consumer warps read the ring, each thread owning
// kSlots 16-byte slots of every piece, and release each stage as soon as
// their registers hold it, so memory traffic never waits on the arithmetic.
// Two slots a stage halve the per-stage cost (barrier wait, release, loop)
// per byte; the policies fold the slots one at a time into one set of sums.  The per-chunk work is a
// policy: an accumulator (forward online softmax) or a gradient writer
// (backward), in a generic form (any dtype and temperature) or a packed bf16
// form.  Every wait is bounded (see kd_ptx.cuh); after a timeout the kernel
// drains its own copies and returns with KD_DEV_TIMEOUT set.
#pragma once

#include <cuda_bf16.h>

#include "kd_internal.h"
#include "kd_ptx.cuh"

namespace kd {
namespace ring {

constexpr int kCW = 24;                       // consumer warps
constexpr int kCT = 32 * kCW;                 // consumer threads
constexpr int kThreads = kCT + 32;            // + one producer warp
constexpr int kRingBytes = 192 * 1024;       // the ring: stages x 2 tensors x piece
constexpr int kMaxStages = 8;
// Ring geometry: NSL 16-byte slots per consumer thread per stage, pieces of
// NSL * 12 KiB per tensor, 8 / NSL stages.  Two slots halve the per-stage cost
// per byte (the one-sweep forwards and the backwards); one slot and eight
// stages leave the warps more slack between one another (the compute-bound
// two-sweep forward of the skew variants).
template <int NSL>
struct Geo {
  static constexpr int kSlots = NSL;
  static constexpr int kChunk = NSL * 16 * kCT;  // bytes of one tensor per stage
  static constexpr int kStages = kRingBytes / (2 * kChunk);
  static_assert(kStages * 2 * kChunk == kRingBytes && kStages <= kMaxStages, "ring geometry");
};
// Per-row merge records.  A consumer warp runs at most kStages + 1 chunks
// (so at most kStages + 2 rows) ahead of the slowest one, so 16 record sets
// are never reused while still being read.
constexpr int kMergeSlots = 16;
constexpr int kRecBytes = kMergeSlots * kCW * kRec * 4;
constexpr int kSmem = 128 + kRingBytes + 256 + kRecBytes + 64;
static_assert(kMergeSlots >= kMaxStages + 4, "merge records could be reused too early");
// control area after the ring: full / empty barriers, the abort word, the
// merge counters, all inside its 256 bytes and apart from one another
static_assert(16 * kMaxStages + 16 + 4 * kMergeSlots <= 256, "ring control words overlap");

template <typename T>
__device__ __forceinline__ float ld1(const T* p) {
  return static_cast<float>(*p);
}
template <>
__device__ __forceinline__ float ld1<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st1(T* p, float v) {
  *p = static_cast<T>(v);
}
template <>
__device__ __forceinline__ void st1<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16(v);
}

struct Ring {
  uint8_t* base;         // [stage][tensor][piece]
  uint32_t full, empty;  // mbarrier arrays (8 bytes each)
  volatile int* abort;
  uint64_t limit;        // time limit of every wait (ns)
  bool withhold;         // test hook: CTA 0's consumer warp 0 keeps its first release
  int* cnt;              // [kMergeSlots] arrivals per merge record set
  float* recs;           // [kMergeSlots][kCW][kRec] per-warp row states
  float* bcast;          // small broadcast area
};

__device__ __forceinline__ Ring make_ring(uint8_t* smem, const StreamArgs& a) {
  Ring r;
  r.limit = a.wait_limit_ns ? a.wait_limit_ns : ptx::kWaitLimitNs;
  r.withhold = a.debug_withhold_release != 0 && blockIdx.x == 0;
  const uint32_t raw = ptx::smem_u32(smem);
  const uint32_t pad = ((raw + 127u) & ~127u) - raw;
  r.base = smem + pad;
  uint8_t* tail = r.base + kRingBytes;
  r.full = ptx::smem_u32(tail);
  r.empty = r.full + 8 * kMaxStages;
  r.abort = reinterpret_cast<volatile int*>(tail + 16 * kMaxStages);
  r.cnt = reinterpret_cast<int*>(tail + 16 * kMaxStages + 16);
  r.recs = reinterpret_cast<float*>(tail + 256);
  r.bcast = r.recs + kMergeSlots * kCW * kRec;
  return r;
}

template <class G>
__device__ __forceinline__ void ring_init(const Ring& R) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < G::kStages; ++i) {
      ptx::mbar_init(R.full + 8 * i, 1);
      ptx::mbar_init(R.empty + 8 * i, kCW);  // one arrival per consumer warp
    }
    for (int i = 0; i < kMergeSlots; ++i) R.cnt[i] = 0;
    *R.abort = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
}

// Producer: stream `passes` sweeps of every row this CTA owns (rows
// blockIdx.x, +gridDim.x, ...) in G::kChunk pieces into the ring.  Rows are
// 16-byte aligned and the vocabulary a multiple of 16 bytes (the dispatch
// checks both), so every copy has a 16-byte aligned source, destination and
// size.
template <typename T, class G>
__device__ void producer(const Ring& R, const StreamArgs& a, bool has_t, int passes,
                         uint32_t* status) {
  constexpr int kChunk = G::kChunk, kStages = G::kStages;
  constexpr int EPC = kChunk / (int)sizeof(T);
  const int64_t V = a.vocab, nch = (V + EPC - 1) / EPC;
  const int lane = threadIdx.x & 31;
  int stage = 0;
  uint32_t phase = 0, issued = 0, par = 0;
  bool ok = true;
  for (int64_t row = blockIdx.x; ok && row < a.n; row += gridDim.x) {
    const T* zs = static_cast<const T*>(a.zs) + row * V;
    const T* zt = has_t ? static_cast<const T*>(a.zt) + row * V : nullptr;
    for (int pass = 0; ok && pass < passes; ++pass)
      for (int64_t ch = 0; ch < nch; ++ch) {
        if (!ptx::warp_wait(R.empty + 8 * stage, phase ^ 1, R.abort, status, true, R.limit)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const int64_t e0 = ch * EPC;
          const uint32_t bytes = (uint32_t)((V - e0 < EPC ? V - e0 : EPC) * (int64_t)sizeof(T));
          const uint32_t fb = R.full + 8 * stage;
          ptx::mbar_expect_tx(fb, has_t ? 2 * bytes : bytes);
          uint8_t* dst = R.base + (size_t)stage * 2 * kChunk;
          ptx::bulk_load(ptx::smem_u32(dst), zs + e0, bytes, fb);
          if (has_t) ptx::bulk_load(ptx::smem_u32(dst + kChunk), zt + e0, bytes, fb);
        }
        __syncwarp();
        issued |= 1u << stage;
        par = (par & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
  }
  if (!ok)  // let our own copies land before the CTA exits
    for (int st = 0; st < kStages; ++st)
      if (issued & (1u << st))
        ptx::warp_wait(R.full + 8 * st, (par >> st) & 1u, R.abort, status, false, R.limit);
}

// Consumer side of the ring.
template <class G>
struct Cursor {
  int stage = 0;
  uint32_t phase = 0;
  bool first = true;
  __device__ __forceinline__ const uint8_t* acquire(const Ring& R, uint32_t* status) {
    ptx::warp_wait(R.full + 8 * stage, phase, R.abort, status, true, R.limit);
    return R.base + (size_t)stage * 2 * G::kChunk;
  }
  __device__ __forceinline__ void release(const Ring& R) {
    __syncwarp();
    const bool keep = R.withhold && first && threadIdx.x < 32;  // test hook only
    first = false;
    if ((threadIdx.x & 31) == 0 && !keep) ptx::mbar_arrive(R.empty + 8 * stage);
    if (++stage == G::kStages) {
      stage = 0;
      phase ^= 1;
    }
  }
};

// Merge warp-reduced states (lane 0 of each consumer warp holds one) into
// consumer thread 0 behind a barrier (all consumers call).
__device__ __forceinline__ void consumer_merge(RowState& st, const Consts& c, const Ring& R) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) st.store(R.recs + w * kRec);
  ptx::named_sync(1, kCT);
  if (w == 0) {
    if (l < kCW) st.load(R.recs + l * kRec);
    else st.init();
    warp_merge(st, c);
  }
  ptx::named_sync(1, kCT);
}

// Barrier-free merge: every consumer warp leaves its warp-reduced state in
// the record set of this row and counts itself in; the last warp to arrive
// merges the set (returns true in that warp, merged state in its lane 0).
__device__ __forceinline__ bool async_merge(RowState& st, const Consts& c, const Ring& R,
                                            int local_row) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int slot = local_row & (kMergeSlots - 1);
  float* rec = R.recs + slot * kCW * kRec;
  int last = 0;
  if (l == 0) {
    st.store(rec + w * kRec);
    __threadfence_block();
    last = atomicAdd(R.cnt + slot, 1) == kCW - 1;
    __threadfence_block();
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return false;
  __syncwarp();  // orders the other lanes' reads after lane 0's observation
  if (l < kCW) st.load(rec + l * kRec);
  else st.init();
  warp_merge(st, c);
  if (l == 0) R.cnt[slot] = 0;  // released before this warp's next ring arrival
  return true;
}

__device__ __forceinline__ float3 consumer_sum3(float x, float y, float z, const Ring& R) {
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xffffffffu, x, o);
    y += __shfl_xor_sync(0xffffffffu, y, o);
    z += __shfl_xor_sync(0xffffffffu, z, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    R.recs[3 * w] = x;
    R.recs[3 * w + 1] = y;
    R.recs[3 * w + 2] = z;
  }
  ptx::named_sync(1, kCT);
  float3 r = make_float3(0.f, 0.f, 0.f);
  if (threadIdx.x == 0)
    for (int i = 0; i < kCW; ++i) {
      r.x += R.recs[3 * i];
      r.y += R.recs[3 * i + 1];
      r.z += R.recs[3 * i + 2];
    }
  ptx::named_sync(1, kCT);
  return r;
}

// 16 bytes of one staged tensor as floats.
template <typename T>
struct Chunk;
template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int EPT = 8;
  __device__ static void load(const uint8_t* p, int ct, float* v) {
    const uint4 u = *reinterpret_cast<const uint4*>(p + ct * 16);
    v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
    v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
  }
  __device__ static void store(__nv_bfloat16* dst, const float* g) {
    uint4 u;
    u.x = pack_bf16(g[0], g[1]);
    u.y = pack_bf16(g[2], g[3]);
    u.z = pack_bf16(g[4], g[5]);
    u.w = pack_bf16(g[6], g[7]);
    *reinterpret_cast<uint4*>(dst) = u;
  }
};
template <>
struct Chunk<float> {
  static constexpr int EPT = 4;
  __device__ static void load(const uint8_t* p, int ct, float* v) {
    const float4 f = *reinterpret_cast<const float4*>(p + ct * 16);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  }
  __device__ static void store(float* dst, const float* g) {
    *reinterpret_cast<float4*>(dst) = make_float4(g[0], g[1], g[2], g[3]);
  }
};

// Outputs of one token from its merged state (one thread).
// y: the row's label (no labels: -1 with has_label false); st.zys / st.zyt
// already hold the label's logits, picked up while the row streamed past.
template <typename T, bool HAS_T>
__device__ __forceinline__ RowOut finish_row(const StreamArgs& a, int64_t row, RowState& st,
                                             int64_t y, bool write_kl) {
  const Consts& c = a.c;
  const int64_t V = a.vocab;
  bool valid = true, bad = false;
  if (a.labels) {
    valid = y != a.ignore;
    bad = valid && (y < 0 || y >= V);
  }
  const float mass = a.topk ? a.mass[row] : 0.f, ent = a.topk ? a.ent[row] : 0.f;
  const RowOut o = finalize(st, c, a.variant, HAS_T, a.topk, mass, ent);
  const float nan = __int_as_float(0x7fc00000);
  if (a.ce_s) a.ce_s[row] = !valid ? 0.f : (bad ? nan : o.ce_s);
  if (a.ce_t) a.ce_t[row] = !valid ? 0.f : (bad ? nan : o.ce_t);
  if (a.kl && write_kl) a.kl[row] = valid ? o.kl : 0.f;
  float4* s4 = reinterpret_cast<float4*>(a.stats + row * KD_STATS_PER_TOKEN);
  s4[0] = make_float4(o.lse_s1, o.lse_sT, o.lse_t1, o.lse_tT);
  s4[1] = make_float4(o.kl_rev, 0.f, mass, o.dlse);
  return o;
}

// Second sweep of one row for the skew variants, once both normalisers are
// known: per-thread partial sums (jq, jp, jx) of q log(q/m), p log(p/m) and
// p (p/m) (the last only for want_x).
template <typename T, class G>
__device__ __forceinline__ float3 skew_sweep(const Ring& R, Cursor<G>& cur, uint32_t* status,
                                             int V, const Consts& c, float lse_tT, float dlse,
                                             bool want_x) {
  constexpr int EPT = 16 / (int)sizeof(T);
  constexpr int kSlots = G::kSlots, kChunk = G::kChunk;
  constexpr int EPC = kChunk / (int)sizeof(T);
  const int nch = (V + EPC - 1) / EPC, ct = threadIdx.x;
  float jq = 0.f, jp = 0.f, jx = 0.f;
  float2 jq2 = make_float2(0.f, 0.f), jp2 = jq2, jx2 = jq2;
  for (int ch = 0; ch < nch; ++ch) {
    const uint8_t* buf = cur.acquire(R, status);
    float fs[kSlots][EPT], ft[kSlots][EPT];
    int nv[kSlots];
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      const int slot = j * kCT + ct;
      nv[j] = valid_cols(V - (ch * EPC + slot * EPT), EPT);
      if (nv[j] > 0) {
        Chunk<T>::load(buf, slot, fs[j]);
        Chunk<T>::load(buf + kChunk, slot, ft[j]);
      }
    }
    cur.release(R);
    if (c.precise) {
#pragma unroll
      for (int j = 0; j < kSlots; ++j)
#pragma unroll
        for (int u = 0; u < EPT; ++u)
          if (u < nv[j]) js_terms(fs[j][u], ft[j][u], lse_tT, dlse, c, jq, jp, jx, want_x);
    } else {  // two columns per .f32x2 instruction
#pragma unroll
      for (int j = 0; j < kSlots; ++j)
#pragma unroll
        for (int u = 0; u < EPT; u += 2) {
          if (u + 1 < nv[j]) {
            js_terms2(make_float2(fs[j][u], fs[j][u + 1]), make_float2(ft[j][u], ft[j][u + 1]),
                      lse_tT, dlse, c, jq2, jp2, jx2, want_x);
          } else if (u < nv[j]) {
            js_terms(fs[j][u], ft[j][u], lse_tT, dlse, c, jq, jp, jx, want_x);
          }
        }
    }
  }
  return make_float3(jq + jq2.x + jq2.y, jp + jp2.x + jp2.y, jx + jx2.x + jx2.y);
}

// The same sweep over bf16 rows in the base-2 form of skew_pair_b2.  The
// dispatch keeps bf16 rows a multiple of 8 columns, so every slot is whole.
template <bool WANT_X, class G>
__device__ __forceinline__ float3 skew_sweep_bf16(const Ring& R, Cursor<G>& cur,
                                                  uint32_t* status, int V, const Consts& c,
                                                  float lse_tT, float dlse) {
  constexpr int kSlots = G::kSlots, kChunk = G::kChunk;
  constexpr int EPT = 8, EPC = kChunk / 2;
  const int nch = (V + EPC - 1) / EPC, ct = threadIdx.x;
  const SkewK k = skew_consts(c, lse_tT, dlse);
  float2 sv = make_float2(0.f, 0.f), dv = sv, ax = sv;
  for (int ch = 0; ch < nch; ++ch) {
    const uint8_t* buf = cur.acquire(R, status);
    uint4 us[kSlots], ut[kSlots];
    bool full[kSlots];
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      const int slot = j * kCT + ct;
      full[j] = ch * EPC + slot * EPT < V;
      if (full[j]) {
        us[j] = *reinterpret_cast<const uint4*>(buf + slot * 16);
        ut[j] = *reinterpret_cast<const uint4*>(buf + kChunk + slot * 16);
      }
    }
    cur.release(R);
#pragma unroll 1  // one slot's pairs live at a time (registers)
    for (int j = 0; j < kSlots; ++j)
      if (full[j]) {
        const uint32_t ws[4] = {us[j].x, us[j].y, us[j].z, us[j].w};
        const uint32_t wt[4] = {ut[j].x, ut[j].y, ut[j].z, ut[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          skew_pair_b2<WANT_X>(make_float2(bf16lo(ws[i]), bf16hi(ws[i])),
                               make_float2(bf16lo(wt[i]), bf16hi(wt[i])), k, sv, dv, ax);
      }
  }
  constexpr float kHalfLn2 = 0.34657359027997264f;
  const float S = sv.x + sv.y, D = dv.x + dv.y;
  return make_float3(-kHalfLn2 * (S + D), -kHalfLn2 * (S - D), ax.x + ax.y);
}

// Forward.  Acc: init(); static load(Frag&, buf, slot); static pick(const
// Frag&, i, zs, zt) (element i of a slot); step(const Frag[NS], const int
// nv[NS], c) for NS slots; RowState fold(c).  Frags are loaded from a stage
// by load(Frag&, buf, slot, piece bytes).  Column indices within a row are
// 32-bit (the dispatch keeps rows below 2^30 elements).  PASSES = 2 for
// skew-JS (a second sweep once both normalisers are known), else 1; a
// template parameter so single-pass kernels carry no second-sweep code.
template <typename T, bool HAS_T, class Acc, int PASSES, int NSL>
__global__ void __launch_bounds__(kThreads, 1) k_fwd(StreamArgs a, uint32_t* status) {
  using G = Geo<NSL>;
  constexpr int kSlots = G::kSlots, kChunk = G::kChunk;
  extern __shared__ uint8_t smem_raw[];
  const Ring R = make_ring(smem_raw, a);
  ring_init<G>(R);
  constexpr int passes = PASSES;
  if ((threadIdx.x >> 5) == kCW) {
    producer<T, G>(R, a, HAS_T, passes, status);
  } else {
    constexpr int EPT = 16 / (int)sizeof(T);
    constexpr int EPC = kChunk / (int)sizeof(T);
    const Consts c = a.c;
    const int V = (int)a.vocab, nch = (V + EPC - 1) / EPC;
    const int ct = threadIdx.x;
    Cursor<G> cur;
    int local_row = 0;
    // labels one row ahead: the load's latency hides behind a whole row
    int64_t y_next = (a.labels && (int64_t)blockIdx.x < a.n) ? a.labels[blockIdx.x] : -1;
    for (int64_t row = blockIdx.x; row < a.n; row += gridDim.x, ++local_row) {
      const int64_t y = y_next;
      if (a.labels && row + gridDim.x < a.n) y_next = a.labels[row + gridDim.x];
      // column of the label within the row, -1 if it is ignored or out of range
      const int yc = (a.labels && y != a.ignore && y >= 0 && y < a.vocab) ? (int)y : -1;
      Acc acc;
      acc.init();
      float zys = 0.f, zyt = 0.f;
      for (int ch = 0; ch < nch; ++ch) {
        const uint8_t* buf = cur.acquire(R, status);
        typename Acc::Frag f[kSlots];
        int nv[kSlots];
#pragma unroll
        for (int j = 0; j < kSlots; ++j) {
          const int slot = j * kCT + ct;
          const int e0 = ch * EPC + slot * EPT;
          nv[j] = valid_cols(V - e0, EPT);
          if (nv[j] > 0) {
            Acc::load(f[j], buf, slot, kChunk);
            // the label's logits, from the staged copy (one thread per row)
            if ((unsigned)(yc - e0) < (unsigned)EPT) Acc::pick(f[j], yc - e0, zys, zyt);
          }
        }
        cur.release(R);
        acc.step(f, nv, c);
      }
      RowState st = acc.fold(c);
      st.zys = zys;
      st.zyt = zyt;
      if (a.topk) {  // sparse cross term sum_S p a_s (ids validated by the prep kernel)
        const T* zs = static_cast<const T*>(a.zs) + row * a.vocab;
        const int32_t* ids = a.sidx + row * a.k;
        const float* ps = a.sp + row * a.k;
        for (int j = ct; j < a.k; j += kCT) {
          const int32_t id = ids[j];
          if (id >= 0 && id < V) st.tk = fmaf(ps[j], ld1<T>(zs + id) * c.inv_ts, st.tk);
        }
      }
      warp_merge(st, c);
      if constexpr (passes == 1) {
        // no CTA barrier: the last warp to finish the row finalises it
        if (async_merge(st, c, R, local_row) && (ct & 31) == 0)
          finish_row<T, HAS_T>(a, row, st, y, true);
        continue;
      }
      // skew-JS: both normalisers are needed before the second sweep
      consumer_merge(st, c, R);
      if (ct == 0) {
        const RowOut o = finish_row<T, HAS_T>(a, row, st, y, false);
        R.bcast[0] = o.dlse;
        R.bcast[1] = o.lse_tT;
      }
      ptx::named_sync(1, kCT);
      const float dlse = R.bcast[0], lse_tT = R.bcast[1];
      const bool want_x = a.variant != KD_KL_SKEW_JS;
      float3 part;
      if constexpr (sizeof(T) == 2) {  // bf16 problems take the fast (non-precise) forms
        part = want_x ? skew_sweep_bf16<true, G>(R, cur, status, V, c, lse_tT, dlse)
                      : skew_sweep_bf16<false, G>(R, cur, status, V, c, lse_tT, dlse);
      } else {
        part = skew_sweep<T, G>(R, cur, status, V, c, lse_tT, dlse, want_x);
      }
      const float3 r = consumer_sum3(part.x, part.y, part.z, R);
      if (ct == 0) {
        const bool v_ok = !a.labels || y != a.ignore;
        a.stats[row * KD_STATS_PER_TOKEN + S_KL_PM] = r.y;
        if (want_x) a.stats[row * KD_STATS_PER_TOKEN + S_EPPM] = r.z;
        if (a.kl) a.kl[row] = v_ok ? skew_kl(a.variant, c.beta, r.x, r.y) : 0.f;
      }
      ptx::named_sync(1, kCT);  // reduction slots are reused by the next row
    }
  }
  __syncthreads();
}

// Backward.  Grad: row(a, row) once per row; static load(Frag&, buf, slot,
// piece bytes); chunk(const Frag&, e0, nv, dz_row) writes the d z_s of one
// 16-byte slot.
template <typename T, bool HAS_T, class Grad, int NSL>
__global__ void __launch_bounds__(kThreads, 1) k_bwd(StreamArgs a, uint32_t* status) {
  using G = Geo<NSL>;
  constexpr int kSlots = G::kSlots, kChunk = G::kChunk;
  extern __shared__ uint8_t smem_raw[];
  const Ring R = make_ring(smem_raw, a);
  ring_init<G>(R);
  if ((threadIdx.x >> 5) == kCW) {
    producer<T, G>(R, a, HAS_T, 1, status);
  } else {
    constexpr int EPT = 16 / (int)sizeof(T);
    constexpr int EPC = kChunk / (int)sizeof(T);
    const int V = (int)a.vocab, nch = (V + EPC - 1) / EPC;
    const int ct = threadIdx.x;
    Cursor<G> cur;
    for (int64_t row = blockIdx.x; row < a.n; row += gridDim.x) {
      Grad g;
      g.row(a, row);
      T* dz = static_cast<T*>(a.dz) + row * a.vocab;
      for (int ch = 0; ch < nch; ++ch) {
        const uint8_t* buf = cur.acquire(R, status);
        typename Grad::Frag f[kSlots];
        int nv[kSlots], e0[kSlots];
#pragma unroll
        for (int j = 0; j < kSlots; ++j) {
          const int slot = j * kCT + ct;
          e0[j] = ch * EPC + slot * EPT;
          nv[j] = valid_cols(V - e0[j], EPT);
          if (nv[j] > 0) Grad::load(f[j], buf, slot, kChunk);
        }
        cur.release(R);
#pragma unroll
        for (int j = 0; j < kSlots; ++j)
          if (nv[j] > 0) g.chunk(f[j], e0[j], nv[j], dz);
      }
    }
  }
  __syncthreads();
}

// Forward with the pass count the variant needs.
template <typename T, bool HAS_T, class Acc>
inline void launch_fwd(const StreamArgs& a, cudaStream_t s);

// Launch one persistent CTA per SM (fewer for short batches).
template <typename K>
inline void launch(K kernel, const StreamArgs& a, cudaStream_t s) {
  const int sms = tc_num_sms() > 0 ? tc_num_sms() : 1;
  const int grid = (int)(a.n < sms ? a.n : sms);
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  kernel<<<grid, kThreads, kSmem, s>>>(a, a.status);
}

template <typename T, bool HAS_T, class Acc>
inline void launch_fwd(const StreamArgs& a, cudaStream_t s) {
  if constexpr (HAS_T && Acc::kSecondSweep) {  // (only policies that serve the skew variants)
    if (is_skew(a.variant)) {
      launch(k_fwd<T, HAS_T, Acc, 2, 1>, a, s);
      return;
    }
  }
  launch(k_fwd<T, HAS_T, Acc, 1, 2>, a, s);
}

// Backward: two slots a stage, one (and 8 stages) for the skew variants'
// heavier gradients.  Grad::kSlotsFor: 1 or 2 when its variant fixes it, 0 to
// decide from the problem's variant.
template <typename T, bool HAS_T, class Grad>
inline void launch_bwd(const StreamArgs& a, cudaStream_t s) {
  if constexpr (Grad::kSlotsFor == 1) {
    launch(k_bwd<T, HAS_T, Grad, 1>, a, s);
  } else if constexpr (Grad::kSlotsFor == 2) {
    launch(k_bwd<T, HAS_T, Grad, 2>, a, s);
  } else {
    if (HAS_T && is_skew(a.variant)) launch(k_bwd<T, HAS_T, Grad, 1>, a, s);
    else launch(k_bwd<T, HAS_T, Grad, 2>, a, s);
  }
}

}  // namespace ring
}  // namespace kd
