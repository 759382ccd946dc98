// Tensor-core (tcgen05 / TMA / TMEM) kernels for sm_103a.
//
// One persistent, warp-specialised kernel skeleton serves three jobs:
//   EPI_FWD   fused logits tile(s) -> online-softmax CE / KL state per row
//             (student tile z_s = H_s W_s^T and teacher tile z_t = H_t W_t^T
//             for the same 128 rows x BN vocabulary columns; either side may
//             instead be streamed from materialised logits) -> partial record
//             per (row, vocabulary split, half tile)
//   EPI_GRAD  recomputed logits tile(s) -> closed-form gradient G (bf16),
//             written row-major into a bounded chunk workspace (dH = G W and
//             dW = G^T H read it as stored)
//             (Full-Chunked-KL-Loss README, "Full Chunked KL": the backward
//             recomputes each chunk and applies M softmax(z) - p)
//   EPI_GEMM  plain C = A B^T with an fp32 / bf16 / accumulate epilogue
//             (dH and dW from the G chunks); each operand K-major or MN-major
//
// Roles (320 threads): warp 0 issues TMA loads into a STAGES-deep shared
// memory ring; warp 1 owns the TMEM allocation (512 columns: one or two
// accumulator stages) and issues tcgen05.mma; both warps run their loops
// converged, with warp-uniform operands, and one lane picked by elect.sync
// issues each copy, MMA and commit (a branch on lane 0 instead put the
// descriptors in per-thread registers and cost 10-15 % of the tensor pipe's
// time on GB300); warps 2..9 drain
// TMEM with tcgen05.ld (warp w reads TMEM lanes 32*(w%4).., half (w-2)/4 of
// the tile's columns); with two stages the epilogue of tile i overlaps the
// MMAs of tile i+1.
//
// PAIR = true runs the kernel on CTA pairs (clusters of 2, cta_group::2): one
// MMA of M = 256 rows x N = 256 columns spans both SMs; each CTA loads only its
// 128 rows of A and its half of the B columns, so each SM moves half the
// operand bytes per FLOP of a single-CTA 128 x 256 tile.  The even CTA issues
// the MMAs; both CTAs' TMA loads complete on its barriers, its commits arrive
// on both CTAs' barriers, and both CTAs' epilogues release the accumulator on
// its barrier.
// Every mbarrier wait is bounded in time; on expiry the kernel raises
// KD_DEV_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kd_internal.h"

namespace kd {

namespace {

constexpr int BM = 128;             // rows per tile (TMEM lanes)
constexpr int BK = 64;              // k elements per stage (one 128-byte swizzle row)
constexpr int kThreads = 320;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait

enum Epi { EPI_FWD = 0, EPI_GRAD = 1, EPI_GEMM = 2 };

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols));
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
// ---- CTA-pair (cta_group::2) forms
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// address of the same shared-memory variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols));
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// ---- issue forms for a whole warp: every lane executes them with the same
// (warp-uniform) operands and elect.sync picks the one lane that issues, so
// the operands stay in uniform registers and the issuing warps never diverge
// around their TMA / MMA / commit instructions.  The elected lane is always the
// lowest active one (lane 0 in a converged warp), so the commits track the
// MMAs that lane issued.
__device__ __forceinline__ void expect_tx_e(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_e(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                              int x, int y) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// TMA load into this CTA's shared memory, completing on a barrier of either
// CTA of the pair
__device__ __forceinline__ void tma_load_2d_pair_e(uint32_t dst, const CUtensorMap* map,
                                                   uint32_t bar_cluster, int x, int y) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
      ".mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void mma_bf16_e(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_bf16_pair_e(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit_e(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}
// arrive on the barrier at this offset in both CTAs of the pair
__device__ __forceinline__ void mma_commit_pair_both_e(uint32_t bar) {
  const uint16_t mask = 3;
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(bar),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void mma_commit_pair_local_e(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (tiles 1024-byte aligned).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;             // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
  return d;
}
// Shared-memory matrix descriptor of an MN-major operand (stored [K, M] or
// [K, N], M / N contiguous), staged as 64 x 64 TMA boxes with 128-byte swizzle:
// each box holds 64 k-rows of 128 bytes (64 consecutive M / N elements); boxes
// for successive 64-element blocks of M / N lie 8 KiB apart (leading byte
// offset), 8-row k groups 1024 bytes apart (stride byte offset).  One K = 16
// step advances the start by 16 rows = 2048 bytes.
constexpr int kMnBox = 64 * 64 * 2;  // bytes of one 64 x 64 bf16 box
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t addr) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(kMnBox >> 4) << 16;  // leading byte offset: next 64 M / N elements
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: next 8 k-rows
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor: kind::f16 with bf16 A/B, fp32 D, K-major A and B
// (bit 15 / bit 16 set: A / B MN-major).
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------------------ params
struct TcParams {  // (128-byte aligned by its tensor maps)
  CUtensorMap ma[2];
  CUtensorMap mb[2];
  int kb[2];          // k blocks per segment (0: segment absent)
  int acc_off[2];     // TMEM column offset of the segment's accumulator in a stage
  int a_row0[2];      // row offset added to the A tile row coordinate
  int b_row0[2];      // row offset added to the B tile row coordinate
  int seg_accum[2];   // 1: the segment adds to an accumulator an earlier segment wrote
  int a_mn[2], b_mn[2];  // 1: the operand is stored MN-major ([K, M] / [K, N])
  int m_tiles, n_tiles, n_splits, items;
  int m_band;         // row tiles per band of the item order (see item_range)
  int acc_stride;     // TMEM columns per accumulator stage
  int acc_stages;     // 1 or 2 accumulator stages in the 512 allocated columns
  int logits_vec;     // materialised logits rows are 16-byte aligned
  TcFwdArgs fwd;
  TcGradArgs grad;
  TcGemmArgs gemm;
};

template <int BN, bool PAIR>
struct Cfg {
  static constexpr int ROWS = PAIR ? 2 * BM : BM;     // tile rows (MMA M)
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;   // B rows this CTA loads
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TX_BYTES = PAIR ? 2 * STAGE_BYTES : STAGE_BYTES;  // per full barrier
  static constexpr int STAGES = (STAGE_BYTES <= 32768) ? 7 : 4;
  static constexpr int TILE_BYTES = STAGES * STAGE_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = TILE_BYTES + BAR_BYTES + 1024;  // + alignment slack
  static constexpr uint32_t IDESC = make_idesc(ROWS, BN);
};

struct Sync {
  uint32_t full, empty, acc_full, acc_empty, drain;  // smem addresses of barrier arrays
  volatile int* abort_flag;
  uint32_t* status;
  bool cluster_acquire;  // waits on barriers the peer CTA arrives on remotely
};

// Every lane tests the phase (each successful try_wait gives that lane acquire
// ordering on the data the barrier guards) and the warp leaves together once
// all lanes have seen it complete; the phase stays complete until this warp
// itself takes part in the next one, so no lane can miss it.  The wait is
// bounded in time: lane 0 checks the clock every 64 rounds and the warp gives
// up together.
__device__ __forceinline__ bool warp_wait(const Sync& s, uint32_t bar, uint32_t parity,
                                          bool honour_abort = true) {
  auto probe = [&]() {
    return s.cluster_acquire ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity);
  };
  if (__all_sync(0xffffffffu, probe())) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (__all_sync(0xffffffffu, probe())) return true;
    if ((it & 63) == 0) {
      int give_up = 0;
      if ((threadIdx.x & 31) == 0) {
        if (honour_abort && *s.abort_flag) {
          give_up = 1;
        } else if (globaltimer() - t0 > kWaitLimitNs) {
          *s.abort_flag = 1;
          set_status(s.status, KD_DEV_TIMEOUT);
          give_up = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
  }
}

// Items (row tile, vocabulary split) are ordered in bands of m_band row tiles:
// all splits of band 0 first, row tile fastest within a band.  The persistent
// CTAs work on consecutive items, so at any time they share a few row tiles,
// whose A rows (m_band of them, sized on the host to a slice of L2) stay
// resident while the B tiles stream past; with all row tiles in one band the
// A rows of every concurrent item could not all stay in L2.
__device__ __forceinline__ void item_range(const TcParams& P, int item, int& m_tile, int& split,
                                           int& t0, int& t1) {
  const int per_band = P.m_band * P.n_splits;
  const int band = item / per_band, idx = item - band * per_band;
  const int m0 = band * P.m_band;
  const int mb = min(P.m_band, P.m_tiles - m0);  // row tiles in this band
  m_tile = m0 + idx % mb;
  split = idx / mb;
  t0 = (int)((int64_t)P.n_tiles * split / P.n_splits);
  t1 = (int)((int64_t)P.n_tiles * (split + 1) / P.n_splits);
}

// v[j] for a runtime j in [0, 32) without dynamic register indexing
__device__ __forceinline__ float pick32(const float* v, int j) {
  float r = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) r = (i == j) ? v[i] : r;
  return r;
}

// 32 consecutive logits of one row from global memory (bf16)
__device__ __forceinline__ void load_logits32(const __nv_bfloat16* row, int64_t col0, int nv,
                                              bool vec, float* v) {
  if (vec && nv == 32) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = ldg_nc_v4(row + col0 + 8 * q);
      v[8 * q + 0] = bf16lo(u.x); v[8 * q + 1] = bf16hi(u.x);
      v[8 * q + 2] = bf16lo(u.y); v[8 * q + 3] = bf16hi(u.y);
      v[8 * q + 4] = bf16lo(u.z); v[8 * q + 5] = bf16hi(u.z);
      v[8 * q + 6] = bf16lo(u.w); v[8 * q + 7] = bf16hi(u.w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = j < nv ? __bfloat162float(row[col0 + j]) : 0.f;
  }
}

// ------------------------------------------------------------------ epilogues
// Fused forward: one RowState per (row, half) over the item's vocabulary tiles.
template <int BN>
struct FwdEpi {
  RowState st;
  int64_t row, y;
  bool row_ok;
  const int32_t* ids;
  const float* ps;
  int kp;

  __device__ __forceinline__ void begin(const TcParams& P, int64_t row_, int t0, int half) {
    const TcFwdArgs& a = P.fwd;
    st.init();
    row = row_;
    row_ok = row < a.n;
    y = (row_ok && a.labels) ? a.labels[row] : -1;
    ids = nullptr;
    ps = nullptr;
    kp = 0;
    if (a.topk && row_ok) {
      ids = a.sidx + row * a.k;
      ps = a.sp + row * a.k;
      const int64_t first = (int64_t)t0 * BN + half * (BN / 2);
      while (kp < a.k && (int64_t)ids[kp] < first) ++kp;
    }
  }

  template <bool HAS_T>
  __device__ __forceinline__ void chunk(const TcParams& P, const float* vs, const float* vt,
                                        int64_t col0) {
    const TcFwdArgs& a = P.fwd;
    if (!row_ok) return;
    const int nv = valid_cols(a.vocab - col0, 32);
    if (nv <= 0) return;
    if (a.js_pass) {
      const float* stt = a.stats + row * KD_STATS_PER_TOKEN;
      const float lt = stt[S_LSE_TT], dl = stt[S_DLSE];
      const bool want_x = a.variant != KD_KL_SKEW_JS;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < nv) js_terms(vs[j], vt[j], lt, dl, a.c, st.jq, st.jp, st.jx, want_x);
      return;
    }
    if (nv == 32) update<32, HAS_T, false, true>(st, vs, vt, 32, a.c);
    else update<32, HAS_T, true>(st, vs, vt, nv, a.c);
    if (y >= col0 && y < col0 + nv) {
      const int j = (int)(y - col0);
      st.zys += pick32(vs, j);
      if (HAS_T) st.zyt += pick32(vt, j);
    }
    if (ids) {
      // skip ids of the other half, then consume this chunk's matches
      while (kp < a.k && (int64_t)ids[kp] < col0) ++kp;
      while (kp < a.k && (int64_t)ids[kp] < col0 + nv) {
        st.tk = fmaf(ps[kp], pick32(vs, (int)(ids[kp] - col0)) * a.c.inv_ts, st.tk);
        ++kp;
      }
    }
  }

  __device__ __forceinline__ void end(const TcParams& P, int split, int half) {
    const TcFwdArgs& a = P.fwd;
    if (!row_ok) return;
    st.store(a.partials + ((int64_t)(split * 2 + half) * a.n + row) * kRec);
  }
};

// 32 consecutive values of one row as bf16 (16-byte stores when aligned);
// zeros instead when !keep (a masked row), selected on the packed words.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v, int nv,
                                              int64_t ld, bool keep = true) {
  const uint32_t mask = keep ? 0xffffffffu : 0u;
  if (nv == 32 && (ld % 8) == 0 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
    for (int qv = 0; qv < 4; ++qv) {
      uint4 u;
      u.x = pack_bf16(v[8 * qv + 0], v[8 * qv + 1]) & mask;
      u.y = pack_bf16(v[8 * qv + 2], v[8 * qv + 3]) & mask;
      u.z = pack_bf16(v[8 * qv + 4], v[8 * qv + 5]) & mask;
      u.w = pack_bf16(v[8 * qv + 6], v[8 * qv + 7]) & mask;
      *reinterpret_cast<uint4*>(dst + 8 * qv) = u;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nv) dst[j] = __float2bfloat16(keep ? v[j] : 0.f);
  }
}

// Gradient epilogue.  Per row, the constants of G with the row's upstream
// scale folded in; per 32 columns, one loop specialised on the KL form and the
// temperature shortcut, so no branch is left in the element loop.
//   G = wk dKL/da_s + wc (softmax(z_s) - e_y)
// with dKL/da_s = p - q (forward), p (log p - log q - KL(p||q)) (reverse),
// their sum (Jeffreys), b p (log(p/m) - KL(p||m)) (skew-JS), M p - p_S
// (top-K; the sparse part is subtracted at the matched ids).
enum GradVar { GV_FWD = 0, GV_REV = 1, GV_JEF = 2, GV_SJS = 3, GV_P = 4 };

struct GradRow {
  float ks, ns, kt, nt;  // log2 p = z_s ks + ns, log2 q = z_t kt + nt
  float wk;              // s w_kl T_s on the KL gradient (times M for top-K, 0 without KL)
  float wkp;             // s w_kl T_s (top-K matched-id terms)
  float wk_r, klr;       // s w_kl T_s ln 2, s w_kl T_s KL(p||q)   (reverse terms)
  float wc, cs, n1s;     // s w_sce; its p^2 coefficient (T = 2); -lse(z_s) log2 e
  float wt, ct, n1t;     // tied teacher CE: s w_tce; its q^2 coefficient; -lse(z_t) log2 e
  float dlse, klpm;      // skew variants: lse(a_t) - lse(a_s); KL(p||m)
  float eppm;            // skew-forward / skew-reverse: E_p[p/m]
  int var;               // kd_variant
  bool live;             // row inside the chunk with a nonzero scale
};

__device__ __forceinline__ GradRow grad_row(const TcGradArgs& a, int64_t row, bool row_ok,
                                            bool has_t) {
  GradRow r;
  const Consts& c = a.c;
  float sv[KD_STATS_PER_TOKEN];
  const float scale = row_ok ? a.row_scale[row] : 0.f;
#pragma unroll
  for (int i = 0; i < KD_STATS_PER_TOKEN; ++i)
    sv[i] = row_ok ? a.stats[row * KD_STATS_PER_TOKEN + i] : 0.f;
  r.live = scale != 0.f;
  r.ks = c.inv_ts * kL2E;
  r.ns = -sv[S_LSE_ST] * kL2E;
  r.kt = c.inv_tt * kL2E;
  r.nt = -sv[S_LSE_TT] * kL2E;
  const float wkl = scale * a.w_kl_ts;
  r.wkp = wkl;
  r.wk = a.topk ? wkl * sv[S_MASS] : (has_t ? wkl : 0.f);
  r.wk_r = wkl * 0.6931471805599453f;
  r.klr = wkl * sv[S_KL_REV];
  r.wc = scale * a.w_sce;
  const int pw = c.pw;
  r.cs = pw == 2 ? r.wc * ex2((2.f * sv[S_LSE_ST] - sv[S_LSE_S1]) * kL2E) : 0.f;
  r.n1s = -sv[S_LSE_S1] * kL2E;
  r.wt = scale * a.w_tce;
  r.ct = (pw == 2 && a.gt) ? r.wt * ex2((2.f * sv[S_LSE_TT] - sv[S_LSE_T1]) * kL2E) : 0.f;
  r.n1t = -sv[S_LSE_T1] * kL2E;
  r.dlse = sv[S_DLSE];
  r.klpm = sv[S_KL_PM];
  r.eppm = sv[S_EPPM];
  r.var = a.variant;
  return r;
}

// vs <- G for 32 columns (vt: teacher logits of the same columns), without the
// label term and the row mask, which the caller applies once per 32 columns.
// Columns go in pairs through the paired fp32 instructions (the same
// roundings as the scalar forms); the skew form stays per column.
template <int VAR, int PW>
__device__ __forceinline__ void grad32(float* vs, const float* vt, const GradRow& r,
                                       const Consts& c) {
  if constexpr (VAR == GV_SJS) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float p = ex2(fmaf(vs[j], r.ks, r.ns));
      const float x = fmaf(vs[j], c.inv_ts, -vt[j] * c.inv_tt) + r.dlse;
      float lqm, lpm;
      js_logs(x, c, lqm, lpm);
      float g = r.wk * skew_grad(r.var, p, lqm, lpm, r.klpm, r.eppm, c);
      if (PW == 2) g = fmaf(r.cs * p, p, g);
      else if (PW == 1) g = fmaf(r.wc, p, g);
      else g = fmaf(r.wc, ex2(fmaf(vs[j], kL2E, r.n1s)), g);
      vs[j] = g;
    }
  } else {
    const float2 ks = make_float2(r.ks, r.ks), ns = make_float2(r.ns, r.ns);
    const float2 kt = make_float2(r.kt, r.kt), nt = make_float2(r.nt, r.nt);
    const float2 wk = make_float2(r.wk, r.wk), wc = make_float2(r.wc, r.wc);
    const float2 wkr = make_float2(r.wk_r, r.wk_r), nklr = make_float2(-r.klr, -r.klr);
    const float2 cs = make_float2(r.cs, r.cs);
    const float2 l2e = make_float2(kL2E, kL2E), n1s = make_float2(r.n1s, r.n1s);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float2 zs = make_float2(vs[j], vs[j + 1]);
      const float2 l2p = fma2(zs, ks, ns);
      const float2 p = make_float2(ex2(l2p.x), ex2(l2p.y));
      float2 g;
      if constexpr (VAR == GV_P) {
        g = mul2(wk, p);
      } else {
        const float2 l2q = fma2(make_float2(vt[j], vt[j + 1]), kt, nt);
        if constexpr (VAR == GV_FWD) {
          g = mul2(wk, sub2(p, make_float2(ex2(l2q.x), ex2(l2q.y))));
        } else {
          const float2 rr = fma2(sub2(l2p, l2q), wkr, nklr);
          if constexpr (VAR == GV_REV)
            g = mul2(p, rr);
          else
            g = fma2(p, rr, mul2(wk, sub2(p, make_float2(ex2(l2q.x), ex2(l2q.y)))));
        }
      }
      if constexpr (PW == 2) {
        g = fma2(mul2(cs, p), p, g);
      } else if constexpr (PW == 1) {
        g = fma2(wc, p, g);
      } else {
        const float2 l1 = fma2(zs, l2e, n1s);
        g = fma2(wc, make_float2(ex2(l1.x), ex2(l1.y)), g);
      }
      vs[j] = g.x;
      vs[j + 1] = g.y;
    }
  }
}

// vt <- tied teacher-CE gradient s w_tce (softmax(z_t) - e_y) for 32 columns.
template <int PW>
__device__ __forceinline__ void grad32_teacher_ce(float* vt, const GradRow& r, int jy) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float g;
    if (PW == 2) {
      const float q = ex2(fmaf(vt[j], r.kt, r.nt));
      g = r.ct * q * q;
    } else if (PW == 1) {
      g = r.wt * ex2(fmaf(vt[j], r.kt, r.nt));
    } else {
      g = r.wt * ex2(fmaf(vt[j], kL2E, r.n1t));
    }
    if (j == jy) g -= r.wt;
    vt[j] = r.live ? g : 0.f;
  }
}

template <int VAR>
__device__ __forceinline__ void grad32_pw(int pw, float* vs, const float* vt, const GradRow& r,
                                          const Consts& c) {
  if (pw == 2) grad32<VAR, 2>(vs, vt, r, c);
  else if (pw == 1) grad32<VAR, 1>(vs, vt, r, c);
  else grad32<VAR, 0>(vs, vt, r, c);
}

template <bool HAS_T>
__device__ __forceinline__ void grad32_var(int gv, int pw, float* vs, const float* vt,
                                           const GradRow& r, const Consts& c) {
  if constexpr (HAS_T) {
    switch (gv) {
      case GV_FWD: grad32_pw<GV_FWD>(pw, vs, vt, r, c); return;
      case GV_REV: grad32_pw<GV_REV>(pw, vs, vt, r, c); return;
      case GV_JEF: grad32_pw<GV_JEF>(pw, vs, vt, r, c); return;
      case GV_SJS: grad32_pw<GV_SJS>(pw, vs, vt, r, c); return;
      default: break;
    }
  }
  grad32_pw<GV_P>(pw, vs, vt, r, c);
}

// G for 32 columns with the label's -w_ce (jy: the label's column within the
// 32, or -1; at most one column, so the element loop carries no compare)
template <bool HAS_T>
__device__ __forceinline__ void grad32_any(int gv, int pw, float* vs, const float* vt,
                                           const GradRow& r, const Consts& c, int jy) {
  grad32_var<HAS_T>(gv, pw, vs, vt, r, c);
  if (jy >= 0) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j == jy) vs[j] -= r.wc;
  }
}

// ------------------------------------------------------------------ kernel
template <int EPI, int BN, bool HAS_T, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) k_tc(const __grid_constant__ TcParams P) {
  using C = Cfg<BN, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + C::STAGES * C::A_BYTES;
  const uint32_t bars = base + C::TILE_BYTES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + C::TILE_BYTES + 200);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::TILE_BYTES + 208);

  Sync S;
  S.full = bars;                              // [STAGES]
  S.empty = bars + 8 * C::STAGES;             // [STAGES]
  S.acc_full = bars + 16 * C::STAGES;         // [2]
  S.acc_empty = bars + 16 * C::STAGES + 16;   // [2]
  S.drain = bars + 16 * C::STAGES + 32;       // [1]
  S.abort_flag = abort_flag;
  S.status = EPI == EPI_FWD ? P.fwd.status : EPI == EPI_GRAD ? P.grad.status : P.gemm.status;
  S.cluster_acquire = false;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // CTA rank within the pair
  const bool leader = rank == 0;                          // issues the MMAs
  const int cid = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ncl = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(S.full + 8 * i, 1);
      mbar_init(S.empty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(S.acc_full + 8 * i, 1);
      mbar_init(S.acc_empty + 8 * i, PAIR ? 16 : 8);  // one arrive per epilogue warp (both CTAs)
    }
    mbar_init(S.drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int s = 0; s < 2; ++s)
      if (P.kb[s] > 0) {
        prefetch_map(&P.ma[s]);
        prefetch_map(&P.mb[s]);
      }
  }
  if (warp == 1) {
    if (PAIR) {  // one warp of each CTA of the pair allocates collectively
      tmem_alloc_pair(smem_u32(tmem_holder), 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_holder), 512);
      tmem_relinquish();
    }
    tc_fence_before();
  }
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers and TMEM exist before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    int stage = 0;
    uint32_t phase = 0, issued = 0, par = 0;
    bool ok = true;
    for (int item = cid; ok && item < P.items; item += ncl) {
      int m_tile, split, t0, t1;
      item_range(P, item, m_tile, split, t0, t1);
      for (int t = t0; ok && t < t1; ++t)
        for (int sg = 0; ok && sg < 2; ++sg)
          for (int kb = 0; ok && kb < P.kb[sg]; ++kb) {
            if (!warp_wait(S, S.empty + 8 * stage, phase ^ 1)) {
              ok = false;
              break;
            }
            {  // the whole warp, one elected lane issuing
              const uint32_t fb = S.full + 8 * stage;
              const int ay = P.a_row0[sg] + m_tile * C::ROWS + (int)rank * BM;
              const int by = P.b_row0[sg] + t * BN + (int)rank * C::B_ROWS;
              // both CTAs' copies of a pair complete on the leader's barrier,
              // which expects the bytes of the whole pair
              const uint32_t fbar = PAIR ? mapa_shared(fb, 0) : fb;
              if (!PAIR || leader) expect_tx_e(fb, C::TX_BYTES);
              auto load = [&](uint32_t dst, const CUtensorMap* map, int x, int y) {
                if (PAIR) tma_load_2d_pair_e(dst, map, fbar, x, y);
                else tma_load_2d_e(dst, map, fbar, x, y);
              };
              const uint32_t dA = sA + stage * C::A_BYTES, dB = sB + stage * C::B_BYTES;
              // only the plain GEMM takes MN-major operands
              const bool a_mn = EPI == EPI_GEMM && P.a_mn[sg];
              const bool b_mn = EPI == EPI_GEMM && P.b_mn[sg];
              if (a_mn) {
                for (int h = 0; h < BM / 64; ++h) load(dA + h * kMnBox, &P.ma[sg], ay + 64 * h, kb * BK);
              } else {
                load(dA, &P.ma[sg], kb * BK, ay);
              }
              if (b_mn) {
                for (int h = 0; h < C::B_ROWS / 64; ++h)
                  load(dB + h * kMnBox, &P.mb[sg], by + 64 * h, kb * BK);
              } else {
                load(dB, &P.mb[sg], kb * BK, by);
              }
            }
            __syncwarp();
            issued |= 1u << stage;
            par = (par & ~(1u << stage)) | (phase << stage);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
    }
    if (!ok && leader) {  // wait for the copies in flight (the leader's barriers see both CTAs')
      for (int s = 0; s < C::STAGES; ++s)
        if (issued & (1u << s)) warp_wait(S, S.full + 8 * s, (par >> s) & 1u, false);
    }
  } else if (warp == 1 && leader) {
    // ---------------------------------------------------------- MMA issuer
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    Sync Sc = S;
    Sc.cluster_acquire = PAIR;  // the peer's epilogue arrives on acc_empty remotely
    for (int item = cid; ok && item < P.items; item += ncl) {
      int m_tile, split, t0, t1;
      item_range(P, item, m_tile, split, t0, t1);
      for (int t = t0; ok && t < t1; ++t) {
        if (!warp_wait(Sc, S.acc_empty + 8 * acc, acc_phase ^ 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int sg = 0; ok && sg < 2; ++sg) {
          const uint32_t d = tmem + acc * P.acc_stride + P.acc_off[sg];
          const bool a_mn = EPI == EPI_GEMM && P.a_mn[sg];
          const bool b_mn = EPI == EPI_GEMM && P.b_mn[sg];
          const uint32_t idesc = C::IDESC | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
          const uint32_t a_step = a_mn ? 128u : 2u;  // per K = 16, 16-byte units
          const uint32_t b_step = b_mn ? 128u : 2u;
          for (int kb = 0; kb < P.kb[sg]; ++kb) {
            if (!warp_wait(S, S.full + 8 * stage, phase)) {
              ok = false;
              break;
            }
            tc_fence_after();
            {  // the whole warp, one elected lane issuing
              const uint32_t a_addr = sA + stage * C::A_BYTES, b_addr = sB + stage * C::B_BYTES;
              const uint64_t ad = a_mn ? smem_desc_mn(a_addr) : smem_desc(a_addr);
              const uint64_t bd = b_mn ? smem_desc_mn(b_addr) : smem_desc(b_addr);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                const uint32_t accum = (kb > 0 || k > 0 || P.seg_accum[sg]) ? 1u : 0u;
                if (PAIR) mma_bf16_pair_e(d, ad + a_step * k, bd + b_step * k, idesc, accum);
                else mma_bf16_e(d, ad + a_step * k, bd + b_step * k, idesc, accum);
              }
              if (PAIR) mma_commit_pair_both_e(S.empty + 8 * stage);  // frees the stage in both CTAs
              else mma_commit_e(S.empty + 8 * stage);
            }
            __syncwarp();
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        if (!ok) break;
        if (PAIR) mma_commit_pair_both_e(S.acc_full + 8 * acc);
        else mma_commit_e(S.acc_full + 8 * acc);
        __syncwarp();
        if (++acc == P.acc_stages) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
    // wait until every MMA this thread issued has completed
    if (PAIR) mma_commit_pair_local_e(S.drain);
    else mma_commit_e(S.drain);
    __syncwarp();
    warp_wait(S, S.drain, 0, false);
  } else if (warp >= 2) {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;              // TMEM lane quarter
    const int half = (warp - 2) >> 2;    // column half of the tile
    const int r_in_tile = 32 * q + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const int r_in_pair = (int)rank * BM + r_in_tile;  // row within the (pair) tile
    for (int item = cid; ok && item < P.items; item += ncl) {
      int m_tile, split, t0, t1;
      item_range(P, item, m_tile, split, t0, t1);
      const int64_t tile_row = (int64_t)m_tile * C::ROWS + r_in_pair;
      FwdEpi<BN> fe;
      if (EPI == EPI_FWD) fe.begin(P, tile_row, t0, half);
      // gradient epilogue: the row's constants, loaded while the MMAs run
      GradRow gr;
      int64_t g_row = 0, g_y = -1;
      bool g_ok = false;
      if constexpr (EPI == EPI_GRAD) {
        const TcGradArgs& a = P.grad;
        g_row = a.r0 + tile_row;
        g_ok = g_row < a.r0 + a.rc;
        gr = grad_row(a, g_row, g_ok, HAS_T && (a.t_gemm || a.t_logits));
        g_y = (g_ok && a.labels) ? a.labels[g_row] : -1;
      }
      for (int t = t0; t < t1; ++t) {
        if (!warp_wait(S, S.acc_full + 8 * acc, acc_phase)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = lane_base + acc * P.acc_stride;
        if (EPI == EPI_FWD) {
          const TcFwdArgs& a = P.fwd;
          const int64_t row = tile_row;
#pragma unroll 1
          for (int cc = 0; cc < BN / 2; cc += 32) {
            const int col_in_tile = half * (BN / 2) + cc;
            const int64_t col0 = (int64_t)t * BN + col_in_tile;
            float vs[32], vt[32];
            __syncwarp();
            if (a.s_gemm) {
              tmem_ld16(tbase + P.acc_off[0] + col_in_tile, vs);
              tmem_ld16(tbase + P.acc_off[0] + col_in_tile + 16, vs + 16);
            }
            if (HAS_T && a.t_gemm) {
              const int off = P.acc_off[a.s_gemm ? 1 : 0];
              tmem_ld16(tbase + off + col_in_tile, vt);
              tmem_ld16(tbase + off + col_in_tile + 16, vt + 16);
            }
            tmem_ld_wait();
            const int nv = valid_cols(a.vocab - col0, 32);
            if (row < a.n) {
              if (a.s_logits)
                load_logits32(static_cast<const __nv_bfloat16*>(a.zs_logits) + row * a.vocab,
                              col0, nv, P.logits_vec, vs);
              if (HAS_T && a.t_logits)
                load_logits32(static_cast<const __nv_bfloat16*>(a.zt_logits) + row * a.vocab,
                              col0, nv, P.logits_vec, vt);
            }
            fe.template chunk<HAS_T>(P, vs, vt, col0);
          }
        } else if (EPI == EPI_GRAD) {
          const TcGradArgs& a = P.grad;
          const int64_t row = g_row, y = g_y;
          const bool row_ok = g_ok;
          const bool has_t = HAS_T && (a.t_gemm || a.t_logits);
          const int gv = !has_t ? GV_P
                         : a.variant == KD_KL_FORWARD ? GV_FWD
                         : a.variant == KD_KL_REVERSE ? GV_REV
                         : a.variant == KD_KL_JEFFREYS ? GV_JEF
                                                       : GV_SJS;
          const int pw = a.c.pw;
          const int32_t* ids = nullptr;
          const float* ps = nullptr;
          int kp = 0;
          if (a.topk && row_ok) {
            ids = a.sidx + row * a.k;
            ps = a.sp + row * a.k;
            const int64_t first = a.c0 + (int64_t)t * BN + half * (BN / 2);
            while (kp < a.k && (int64_t)ids[kp] < first) ++kp;
          }
#pragma unroll 1
          for (int cc = 0; cc < BN / 2; cc += 32) {
            const int col_in_tile = half * (BN / 2) + cc;
            const int64_t lc0 = (int64_t)t * BN + col_in_tile;   // column within the chunk
            const int64_t col0 = a.c0 + lc0;                       // vocabulary column
            float vs[32], vt[32];
            __syncwarp();
            if (a.s_gemm) {
              tmem_ld16(tbase + P.acc_off[0] + col_in_tile, vs);
              tmem_ld16(tbase + P.acc_off[0] + col_in_tile + 16, vs + 16);
            }
            if (HAS_T && a.t_gemm) {
              const int off = P.acc_off[a.s_gemm ? 1 : 0];
              tmem_ld16(tbase + off + col_in_tile, vt);
              tmem_ld16(tbase + off + col_in_tile + 16, vt + 16);
            }
            tmem_ld_wait();
            const int nv = valid_cols(a.cc - lc0, 32);
            if (row_ok && nv > 0) {
              if (a.s_logits)
                load_logits32(static_cast<const __nv_bfloat16*>(a.zs_logits) + row * a.vocab,
                              col0, nv, P.logits_vec, vs);
              if (HAS_T && a.t_logits)
                load_logits32(static_cast<const __nv_bfloat16*>(a.zt_logits) + row * a.vocab,
                              col0, nv, P.logits_vec, vt);
              const int jy = (y >= col0 && y < col0 + 32) ? (int)(y - col0) : -1;
              // G in place over vs first (it reads vt), then the tied
              // teacher-CE gradient in place over vt
              float* g = vs;
              grad32_any<HAS_T>(gv, pw, g, vt, gr, a.c, jy);
              const bool want_gt = HAS_T && a.gt != nullptr;
              if (want_gt) {
                if (pw == 2) grad32_teacher_ce<2>(vt, gr, jy);
                else if (pw == 1) grad32_teacher_ce<1>(vt, gr, jy);
                else grad32_teacher_ce<0>(vt, gr, jy);
              }
              if (ids && gr.live) {
                while (kp < a.k && (int64_t)ids[kp] < col0) ++kp;
                while (kp < a.k && (int64_t)ids[kp] < col0 + nv) {
                  const int jj = (int)(ids[kp] - col0);
                  const float sub = gr.wkp * ps[kp];
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    if (i == jj) g[i] -= sub;
                  ++kp;
                }
              }
              // row-major G (or d z_s) and G_t: 32 consecutive bf16 of this row
              store_bf16x32(a.g + (row - a.r0) * a.ldg + lc0, g, nv, a.ldg, gr.live);
              if (want_gt) store_bf16x32(a.gt + (row - a.r0) * a.ldg + lc0, vt, nv, a.ldg);
            }
          }
        } else {  // EPI_GEMM
          const TcGemmArgs& a = P.gemm;
          const int64_t row = tile_row;
#pragma unroll 1
          for (int cc = 0; cc < BN / 2; cc += 32) {
            const int col_in_tile = half * (BN / 2) + cc;
            const int64_t col0 = (int64_t)t * BN + col_in_tile;
            float v[32];
            __syncwarp();
            tmem_ld16(tbase + col_in_tile, v);
            tmem_ld16(tbase + col_in_tile + 16, v + 16);
            tmem_ld_wait();
            const int nv = valid_cols(a.N - col0, 32);
            if (row < a.M && nv > 0) {
              const bool full = nv == 32;
              if (a.mode != TC_OUT_BF16) {
                float* c = a.c32 + row * a.ldc32 + col0;
                const bool vec = full && (a.ldc32 % 4) == 0;
                if (a.mode != TC_OUT_F32) {
                  if (vec) {
#pragma unroll
                    for (int qv = 0; qv < 8; ++qv) {
                      const float4 o = *reinterpret_cast<const float4*>(c + 4 * qv);
                      v[4 * qv + 0] += o.x;
                      v[4 * qv + 1] += o.y;
                      v[4 * qv + 2] += o.z;
                      v[4 * qv + 3] += o.w;
                    }
                  } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                      if (j < nv) v[j] += c[j];
                  }
                }
                if (a.mode != TC_OUT_F32_ACC_BF16) {
                  if (vec) {
#pragma unroll
                    for (int qv = 0; qv < 8; ++qv)
                      *reinterpret_cast<float4*>(c + 4 * qv) =
                          make_float4(v[4 * qv], v[4 * qv + 1], v[4 * qv + 2], v[4 * qv + 3]);
                  } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                      if (j < nv) c[j] = v[j];
                  }
                }
              }
              if (a.mode == TC_OUT_BF16 || a.mode == TC_OUT_F32_ACC_BF16) {
                __nv_bfloat16* c = a.c16 + row * a.ldc16 + col0;
                if (full && (a.ldc16 % 8) == 0) {
#pragma unroll
                  for (int qv = 0; qv < 4; ++qv) {
                    uint4 u;
                    u.x = pack_bf16(v[8 * qv + 0], v[8 * qv + 1]);
                    u.y = pack_bf16(v[8 * qv + 2], v[8 * qv + 3]);
                    u.z = pack_bf16(v[8 * qv + 4], v[8 * qv + 5]);
                    u.w = pack_bf16(v[8 * qv + 6], v[8 * qv + 7]);
                    *reinterpret_cast<uint4*>(c + 8 * qv) = u;
                  }
                } else {
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    if (j < nv) c[j] = __float2bfloat16(v[j]);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR) mbar_arrive_cluster(mapa_shared(S.acc_empty + 8 * acc, 0));
          else mbar_arrive(S.acc_empty + 8 * acc);
        }
        if (++acc == P.acc_stages) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (EPI == EPI_FWD && ok) fe.end(P, split, half);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // no CTA leaves while its peer may still touch it
  tc_fence_after();
  if (warp == 1) {
    if (PAIR) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D bf16 map over a [rows, cols] matrix with row pitch `pitch` elements,
// box = 64 columns x box_rows rows, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t pitch,
              int box_rows) {
  if (!get_encoder()) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(pitch * 2)};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Map of an MN-major operand stored [k_rows, mn_cols] (pitch in elements),
// read in 64 (M / N) x 64 (K) boxes.
bool make_map_mn(CUtensorMap* m, const void* ptr, int64_t k_rows, int64_t mn_cols,
                 int64_t pitch) {
  if (!get_encoder()) return false;
  cuuint64_t dims[2] = {(cuuint64_t)mn_cols, (cuuint64_t)k_rows};
  cuuint64_t strides[1] = {(cuuint64_t)(pitch * 2)};
  cuuint32_t box[2] = {64u, (cuuint32_t)BK};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int EPI, int BN, bool HAS_T, bool PAIR>
int launch(const TcParams& P, int num_sms, cudaStream_t s) {
  using C = Cfg<BN, PAIR>;
  auto kern = k_tc<EPI, BN, HAS_T, PAIR>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return (int)e;
  if (P.items <= 0) return 0;
  if (!PAIR) {
    const int grid = P.items < num_sms ? P.items : num_sms;
    note_launch();
    kern<<<grid, kThreads, C::SMEM_BYTES, s>>>(P);
    return (int)cudaGetLastError();
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2 * (num_sms / 2));
  int max_clusters = max_active_clusters(reinterpret_cast<const void*>(kern), cfg);
  if (max_clusters <= 0) max_clusters = num_sms / 2;
  const int clusters = P.items < max_clusters ? P.items : max_clusters;
  cfg.gridDim = dim3(2 * clusters);
  note_launch();
  e = cudaLaunchKernelEx(&cfg, kern, P);
  if (e != cudaSuccess) return (int)e;
  return (int)cudaGetLastError();
}

bool logits_vec_ok(const void* p, int64_t vocab) {
  return p == nullptr || (((reinterpret_cast<uintptr_t>(p) & 15) == 0) && (vocab % 8) == 0);
}

int fail_map() { return (int)cudaErrorInvalidValue; }

// Row tiles per band of the item order: the A rows of one band (rows_per_tile
// x K bf16 per row tile, all segments) take at most 48 MiB of L2.
int band_tiles(const TcParams& P, int rows_per_tile) {
  const int64_t k = (int64_t)(P.kb[0] + P.kb[1]) * BK;
  const int64_t per_tile = std::max<int64_t>(1, (int64_t)rows_per_tile * k * 2);
  const int64_t b = ((int64_t)48 << 20) / per_tile;
  return (int)std::max<int64_t>(1, std::min<int64_t>(b, P.m_tiles));
}

// Segment setup shared by the fused forward and the gradient producer.
// bn = tile columns, b_box = B rows one CTA loads, rows_per_tile = MMA M.
template <class A>
bool setup_segments(TcParams& P, const A& a, int bn, int b_box, int rows_per_tile, int64_t r0,
                    int64_t rows, int64_t c0, int64_t cols) {
  int ns = 0;
  if (a.s_gemm) {
    if (!make_map(&P.ma[ns], a.h_s, a.n, a.d_s, a.d_s, BM) ||
        !make_map(&P.mb[ns], a.w_s, a.vocab, a.d_s, a.d_s, b_box))
      return false;
    P.kb[ns] = (int)((a.d_s + BK - 1) / BK);
    P.acc_off[ns] = 0;
    P.a_row0[ns] = (int)r0;
    P.b_row0[ns] = (int)c0;
    ++ns;
  }
  if (a.t_gemm) {
    const void* wt = a.w_t ? a.w_t : a.w_s;  // tied teachers use the student head
    if (!make_map(&P.ma[ns], a.h_t, a.n, a.d_t, a.d_t, BM) ||
        !make_map(&P.mb[ns], wt, a.vocab, a.d_t, a.d_t, b_box))
      return false;
    P.kb[ns] = (int)((a.d_t + BK - 1) / BK);
    P.acc_off[ns] = a.s_gemm ? bn : 0;
    P.a_row0[ns] = (int)r0;
    P.b_row0[ns] = (int)c0;
    ++ns;
  }
  const int sides = ns;
  P.acc_stride = sides * bn;             // 256 or 512 TMEM columns per stage
  P.acc_stages = 512 / P.acc_stride;     // 2 or 1
  P.m_tiles = (int)((rows + rows_per_tile - 1) / rows_per_tile);
  P.n_tiles = (int)((cols + bn - 1) / bn);
  return true;
}

}  // namespace

int tc_num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// CTA pairs unless KD_TC_PAIR=0 (debug override: single-CTA tiles).
bool tc_use_pairs() {
  const char* e = getenv("KD_TC_PAIR");
  return !(e && e[0] == '0');
}

// Tile columns of the fused kernels: two GEMM sides share the 512 TMEM
// columns (single CTA: 128 per side, double buffered; pairs: 256 per side,
// one stage); one side always gets 256 columns, double buffered.
int tc_fused_tile_cols(bool two_sides, bool pair) { return (two_sides && !pair) ? 128 : 256; }

// Gradient-producer tile columns.  Two GEMM sides on CTA pairs take 256
// columns per side (one TMEM stage, full-rate MMAs); the partial last wave of
// each chunk is covered by the next launch on the backward's second stream.
// KD_TC_GRAD_COLS=128 selects 128 columns per side with two TMEM stages.
int tc_grad_tile_cols(bool two_sides, bool pair) {
  if (!(two_sides && pair)) return tc_fused_tile_cols(two_sides, pair);
  const char* e = getenv("KD_TC_GRAD_COLS");
  return (e && e[0] == '1') ? 128 : 256;
}
int tc_tile_rows(bool pair) { return pair ? 2 * BM : BM; }

int launch_tc_fwd(const TcFwdArgs& a, int num_sms, cudaStream_t s) {
  TcParams P;
  memset(&P, 0, sizeof(P));
  const bool pair = tc_use_pairs();
  const bool two = a.s_gemm && a.t_gemm;
  const int bn = tc_fused_tile_cols(two, pair);
  if (!setup_segments(P, a, bn, pair ? bn / 2 : bn, tc_tile_rows(pair), 0, a.n, 0, a.vocab))
    return fail_map();
  P.n_splits = a.n_splits;
  P.items = P.m_tiles * P.n_splits;
  P.m_band = band_tiles(P, tc_tile_rows(pair));
  P.logits_vec = logits_vec_ok(a.zs_logits, a.vocab) && logits_vec_ok(a.zt_logits, a.vocab);
  P.fwd = a;
  const bool has_t = a.t_gemm || a.t_logits;
  if (pair)
    return has_t ? launch<EPI_FWD, 256, true, true>(P, num_sms, s)
                 : launch<EPI_FWD, 256, false, true>(P, num_sms, s);
  if (bn == 128)
    return has_t ? launch<EPI_FWD, 128, true, false>(P, num_sms, s)
                 : launch<EPI_FWD, 128, false, false>(P, num_sms, s);
  return has_t ? launch<EPI_FWD, 256, true, false>(P, num_sms, s)
               : launch<EPI_FWD, 256, false, false>(P, num_sms, s);
}

int launch_tc_grad(const TcGradArgs& a, int num_sms, cudaStream_t s) {
  TcParams P;
  memset(&P, 0, sizeof(P));
  const bool pair = tc_use_pairs();
  const bool two = a.s_gemm && a.t_gemm;
  const int bn = tc_grad_tile_cols(two, pair);
  if (!setup_segments(P, a, bn, pair ? bn / 2 : bn, tc_tile_rows(pair), a.r0, a.rc, a.c0, a.cc))
    return fail_map();
  P.n_splits = P.n_tiles;  // one tile per item
  P.items = P.m_tiles * P.n_tiles;
  P.m_band = band_tiles(P, tc_tile_rows(pair));
  P.logits_vec = logits_vec_ok(a.zs_logits, a.vocab) && logits_vec_ok(a.zt_logits, a.vocab);
  P.grad = a;
  const bool has_t = a.t_gemm || a.t_logits;
  if (pair && bn == 128) return launch<EPI_GRAD, 128, true, true>(P, num_sms, s);
  if (pair)
    return has_t ? launch<EPI_GRAD, 256, true, true>(P, num_sms, s)
                 : launch<EPI_GRAD, 256, false, true>(P, num_sms, s);
  if (bn == 128)
    return has_t ? launch<EPI_GRAD, 128, true, false>(P, num_sms, s)
                 : launch<EPI_GRAD, 128, false, false>(P, num_sms, s);
  return has_t ? launch<EPI_GRAD, 256, true, false>(P, num_sms, s)
               : launch<EPI_GRAD, 256, false, false>(P, num_sms, s);
}

int launch_tc_gemm(const TcGemmArgs& a, int num_sms, cudaStream_t s) {
  TcParams P;
  memset(&P, 0, sizeof(P));
  const bool pair = tc_use_pairs();
  constexpr int bn = 256;
  const int b_box = pair ? bn / 2 : bn;
  // operand maps: K-major [rows, K] or MN-major [K, rows]
  auto map = [&](CUtensorMap* m, const void* ptr, int64_t rows, int64_t k, int64_t ld, int box,
                 int mn) {
    return mn ? make_map_mn(m, ptr, k, rows, ld) : make_map(m, ptr, rows, k, ld, box);
  };
  if (!map(&P.ma[0], a.a0, a.M, a.K0, a.lda0, BM, a.a0_mn) ||
      !map(&P.mb[0], a.b0, a.N, a.K0, a.ldb0, b_box, a.b0_mn))
    return fail_map();
  P.kb[0] = (int)((a.K0 + BK - 1) / BK);
  P.a_mn[0] = a.a0_mn;
  P.b_mn[0] = a.b0_mn;
  if (a.K1 > 0) {
    if (!map(&P.ma[1], a.a1, a.M, a.K1, a.lda1, BM, a.a1_mn) ||
        !map(&P.mb[1], a.b1, a.N, a.K1, a.ldb1, b_box, a.b1_mn))
      return fail_map();
    P.kb[1] = (int)((a.K1 + BK - 1) / BK);
    P.a_mn[1] = a.a1_mn;
    P.b_mn[1] = a.b1_mn;
    P.seg_accum[1] = 1;  // both segments sum into the same accumulator
  }
  P.acc_stride = bn;
  P.acc_stages = 2;
  P.m_tiles = (int)((a.M + tc_tile_rows(pair) - 1) / tc_tile_rows(pair));
  P.n_tiles = (int)((a.N + bn - 1) / bn);
  P.n_splits = P.n_tiles;
  P.items = P.m_tiles * P.n_tiles;
  P.m_band = band_tiles(P, tc_tile_rows(pair));
  P.gemm = a;
  return pair ? launch<EPI_GEMM, 256, false, true>(P, num_sms, s)
              : launch<EPI_GEMM, 256, false, false>(P, num_sms, s);
}

}  // namespace kd
