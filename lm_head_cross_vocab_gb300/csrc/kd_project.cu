// Cross-vocabulary token-map projection (orda-kernel README, "Cross-vocabulary
// distillation", token-map projection): teacher logits over the teacher
// vocabulary are moved onto the student vocabulary.  map[j] is the student id
// of teacher token j, or -1.  For every token row n and student id i,
//   out[n, i] = log sum_{j : map[j] = i} exp(z_t[n, j] / T)
// (the teacher distribution tempered before aggregation, duplicates summed in
// probability space).  A student id that no teacher token maps to has
// probability 0: it is written as the most negative finite value of the
// output type, whose exponential is exactly 0 like that of -inf, so the
// distillation kernels need no special case for it (0 * log 0 terms stay 0).
//
// Every call first builds, in the caller's workspace, the inverse map (count
// -> exclusive scan -> scatter -> per-id sort, so summation orders are fixed
// and results deterministic) and the lists of one of two paths:
//
// * exchange (k_project_exchange, the normal path): a cluster of C <= 8 CTAs
//   shares each token row.  CTA r stages teacher columns [r*sc, r*sc + sc)
//   with one bulk copy, gathers the values its map edges need into a send
//   buffer ordered by destination CTA (random reads of its own shared memory
//   only), and ships each segment to the CTA that writes those student ids
//   with one shared::cta -> shared::cluster bulk copy; the owner then writes
//   its id range of the output row with 16-byte stores.  Random accesses
//   never leave an SM, and every output byte is written once in whole
//   sectors.
// * slices (k_project_slices, the fallback when a receive buffer would
//   overflow -- a map that sends most edges to one range, decided on the
//   device -- or when a row needs more than 8 CTAs or a CTA more than 32 Ki
//   student ids): work items (token row, slice); a CTA stages the slice and
//   stores each listed id's output straight to global memory.  Correct for any map, but its 2-byte stores leave
//   sectors partial, which costs DRAM read-modify-writes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <cstring>

#include "../../include/kd.h"
#include "kd_internal.h"
#include "kd_ptx.cuh"

namespace kd {
namespace {

constexpr int kT = 256;
constexpr int kPT = 1024;                 // threads per projection CTA (slice kernel, wide exchange)
constexpr int kXTNarrow = 512;            // threads per exchange CTA of the narrow shape
constexpr int64_t kSliceMax = 96 * 1024;  // bytes of a staged slice (two per CTA)
constexpr int kMaxSlices = 1024;          // teacher rows up to 96 MiB

__global__ void k_map_count(const int32_t* __restrict__ map, int64_t vt, int64_t vs,
                            int32_t* __restrict__ cnt, uint32_t* status) {
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < vt;
       j += (int64_t)gridDim.x * blockDim.x) {
    const int32_t i = map[j];
    if (i >= 0 && (int64_t)i < vs) atomicAdd(cnt + i, 1);
    else if (i != -1) set_status(status, KD_DEV_BAD_MAP);
  }
}

// off[0..vs] = exclusive scan of cnt[0..vs): one block of 1024 threads walks
// the array in tiles of 4096 (coalesced int4 loads, warp-shuffle scans of the
// per-thread sums, a scan of the 32 warp totals, a running carry).
__global__ void __launch_bounds__(1024) k_map_scan(const int32_t* __restrict__ cnt, int64_t vs,
                                                   int32_t* __restrict__ off) {
  __shared__ int32_t wsum[32];
  __shared__ int32_t carry_sh;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  int32_t carry = 0;
  for (int64_t base = 0; base < vs; base += 4096) {
    const int64_t i = base + 4 * (int64_t)t;
    int32_t v[4];
    if (i + 4 <= vs) {  // cnt is 256-byte aligned and i a multiple of 4
      const int4 q = *reinterpret_cast<const int4*>(cnt + i);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = i + k < vs ? cnt[i + k] : 0;
    }
    const int32_t own = v[0] + v[1] + v[2] + v[3];
    int32_t inc = own;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane == 31) wsum[w] = inc;
    __syncthreads();
    if (w == 0) {
      int32_t x = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += u;
      }
      wsum[lane] = x;  // inclusive warp-total prefix
      if (lane == 31) carry_sh = x;
    }
    __syncthreads();
    int32_t run = carry + (w > 0 ? wsum[w - 1] : 0) + inc - own;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (i + k < vs) off[i + k] = run;
      run += v[k];
    }
    carry += carry_sh;
    __syncthreads();  // wsum / carry_sh are rewritten by the next tile
  }
  if (t == 0) off[vs] = carry;
}

// Multi-block form of the same exclusive scan, for long arrays: tile sums
// (k_scan_tiles), the scan of those sums (k_map_scan on them), then every
// tile scanned from its offset (k_scan_apply).  Tiles are 4096 entries.
constexpr int kScanTile = 4096;

__device__ __forceinline__ void load4(const int32_t* __restrict__ in, int64_t i, int64_t n,
                                      int32_t v[4]) {
  if (i + 4 <= n) {  // in is 256-byte aligned and i a multiple of 4
    const int4 q = *reinterpret_cast<const int4*>(in + i);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = i + k < n ? in[i + k] : 0;
  }
}

__global__ void __launch_bounds__(1024) k_scan_tiles(const int32_t* __restrict__ in, int64_t n,
                                                     int32_t* __restrict__ tsum) {
  __shared__ int32_t ws[32];
  const int64_t i = (int64_t)blockIdx.x * kScanTile + 4 * (int64_t)threadIdx.x;
  int32_t v[4];
  load4(in, i, n, v);
  int32_t x = v[0] + v[1] + v[2] + v[3];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = x;
  __syncthreads();
  if (threadIdx.x < 32) {
    int32_t y = ws[threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
    if (threadIdx.x == 0) tsum[blockIdx.x] = y;
  }
}

__global__ void __launch_bounds__(1024) k_scan_apply(const int32_t* __restrict__ in, int64_t n,
                                                     const int32_t* __restrict__ toff,
                                                     int32_t* __restrict__ out) {
  __shared__ int32_t wsum[32];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int64_t i = (int64_t)blockIdx.x * kScanTile + 4 * (int64_t)t;
  int32_t v[4];
  load4(in, i, n, v);
  const int32_t own = v[0] + v[1] + v[2] + v[3];
  int32_t inc = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) wsum[w] = inc;
  __syncthreads();
  if (w == 0) {
    int32_t x = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += u;
    }
    wsum[lane] = x;
  }
  __syncthreads();
  int32_t run = toff[blockIdx.x] + (w > 0 ? wsum[w - 1] : 0) + inc - own;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (i + k < n) out[i + k] = run;
    run += v[k];
  }
  if (blockIdx.x == 0 && t == 0) out[n] = toff[gridDim.x];
}

// one[i] for student id i: its teacher column when exactly one teacher token
// maps to it, -1 when none does, -2 when several do; eid[e]: the student id of
// map edge e (the e-th entry of the id-sorted column list).
__global__ void k_map_single(const int32_t* __restrict__ off, const int32_t* __restrict__ cols,
                             int64_t vs, int32_t* __restrict__ one, int32_t* __restrict__ eid) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vs;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t b = off[i], e = off[i + 1];
    one[i] = e - b == 1 ? cols[b] : (e == b ? -1 : -2);
    for (int32_t k = b; k < e; ++k) eid[k] = (int32_t)i;
  }
}

__global__ void k_map_scatter(const int32_t* __restrict__ map, int64_t vt, int64_t vs,
                              const int32_t* __restrict__ off, int32_t* __restrict__ cur,
                              int32_t* __restrict__ cols) {
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < vt;
       j += (int64_t)gridDim.x * blockDim.x) {
    const int32_t i = map[j];
    if (i >= 0 && (int64_t)i < vs) cols[off[i] + atomicAdd(cur + i, 1)] = (int32_t)j;
  }
}

// ascending teacher columns within each student id's segment (segments are
// short: exact token maps send one teacher token, rarely a few, to an id)
__global__ void k_map_sort(const int32_t* __restrict__ off, int64_t vs, int32_t* __restrict__ cols) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vs;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t b = off[i], e = off[i + 1];
    for (int32_t k = b + 1; k < e; ++k) {
      const int32_t v = cols[k];
      int32_t p = k - 1;
      while (p >= b && cols[p] > v) {
        cols[p + 1] = cols[p];
        --p;
      }
      cols[p + 1] = v;
    }
  }
}

template <typename T>
__device__ __forceinline__ float ld(const T* p) {
  return static_cast<float>(*p);
}
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st(T* p, float v) {
  *p = static_cast<T>(v);
}
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16(v);
}
template <typename T>
__device__ __forceinline__ float lowest();
template <>
__device__ __forceinline__ float lowest<float>() {
  return -FLT_MAX;
}
template <>
__device__ __forceinline__ float lowest<__nv_bfloat16>() {
  return __uint_as_float(0xff7f0000u);  // most negative finite bf16
}


__device__ __forceinline__ float logaddexp(float a, float b) {
  if (a == -INFINITY) return b;
  const float m = fmaxf(a, b);
  return m + log1pf(expf(-fabsf(a - b)));
}

__device__ __forceinline__ void store_vec(float* o, const float* r) {
  reinterpret_cast<float4*>(o)[0] = make_float4(r[0], r[1], r[2], r[3]);
  reinterpret_cast<float4*>(o)[1] = make_float4(r[4], r[5], r[6], r[7]);
}
__device__ __forceinline__ void store_vec(__nv_bfloat16* o, const float* r) {
  uint4 u;
  u.x = pack_bf16(r[0], r[1]);
  u.y = pack_bf16(r[2], r[3]);
  u.z = pack_bf16(r[4], r[5]);
  u.w = pack_bf16(r[6], r[7]);
  *reinterpret_cast<uint4*>(o) = u;
}

// ---------------------------------------------------------------- exchange lists

// The exchange path (see k_project_exchange): a cluster of C <= kMaxC CTAs per
// token row; CTA r stages teacher columns [r*sc, r*sc + sc) and writes student
// ids [q*so, q*so + so) for q = r.  Map edge e (teacher column cols[e] ->
// student id eid[e]) travels from CTA r = cols[e] / sc to CTA q = eid[e] / so
// in segment (r, q).  Segments are padded to 8 elements so that every bulk
// copy starts and ends on 16 bytes.
constexpr int kMaxC = 8;
constexpr int kXSteps = 4;  // 8-id steps per thread: a CTA's range is at most 32 Ki ids
// ids with several teacher tokens that a CTA keeps in a shared-memory table
// (their receive slots; codes recv_cap + k name entry k)
constexpr int kMCap = 1024;
struct XLayout {
  int32_t cnt[kMaxC * kMaxC];      // edges of segment (r, q), at r * C + q
  int32_t sendoff[kMaxC * kMaxC];  // offset of segment (r, q) in CTA r's send buffer
  int32_t recvoff[kMaxC * kMaxC];  // offset of segment (r, q) in CTA q's receive buffer
  int32_t sendbase[kMaxC + 1];     // start of CTA r's gather list in send_src
  int32_t sendtot[kMaxC];          // padded elements CTA r sends
  int32_t recvtot[kMaxC];          // padded elements CTA q receives
  int32_t fits;                    // 1: every buffer fits, the exchange kernel runs
};
__host__ __device__ __forceinline__ int32_t pad8(int32_t x) { return (x + 7) & ~7; }

__device__ __forceinline__ int edge_key(int32_t e, const int32_t* __restrict__ cols,
                                        const int32_t* __restrict__ eid, int32_t sc, int32_t so,
                                        int C) {
  return (cols[e] / sc) * C + eid[e] / so;
}

__global__ void k_edge_count(const int32_t* __restrict__ off, const int32_t* __restrict__ cols,
                             const int32_t* __restrict__ eid, int64_t vs, int32_t sc, int32_t so,
                             int C, XLayout* __restrict__ X) {
  __shared__ int32_t h[kMaxC * kMaxC];
  for (int k = threadIdx.x; k < C * C; k += blockDim.x) h[k] = 0;
  __syncthreads();
  const int32_t E = off[vs];
  const int32_t stride = gridDim.x * blockDim.x;
  for (int32_t e0 = blockIdx.x * blockDim.x; e0 < E; e0 += stride) {
    const int32_t e = e0 + (int32_t)threadIdx.x;
    const int k = e < E ? edge_key(e, cols, eid, sc, so, C) : -1;
    const unsigned same = __match_any_sync(0xffffffffu, k);
    if (k >= 0 && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&h[k], __popc(same));
  }
  __syncthreads();
  for (int k = threadIdx.x; k < C * C; k += blockDim.x)
    if (h[k]) atomicAdd(&X->cnt[k], h[k]);
}

// padded offsets of every segment, and whether the buffers fit: send_cap and
// recv_cap are the elements the exchange kernel's shared memory holds
__global__ void k_exchange_layout(XLayout* X, int C, int32_t send_cap, int32_t recv_cap) {
  if (threadIdx.x != 0) return;
  int fits = 1;
  int32_t base = 0;
  for (int r = 0; r < C; ++r) {
    int32_t o = 0;
    for (int q = 0; q < C; ++q) {
      X->sendoff[r * C + q] = o;
      o += pad8(X->cnt[r * C + q]);
    }
    X->sendtot[r] = o;
    X->sendbase[r] = base;
    base += o;
    fits &= o <= send_cap;
  }
  X->sendbase[C] = base;
  for (int q = 0; q < C; ++q) {
    int32_t o = 0;
    for (int r = 0; r < C; ++r) {
      X->recvoff[r * C + q] = o;
      o += pad8(X->cnt[r * C + q]);
    }
    X->recvtot[q] = o;
    fits &= o <= recv_cap;
  }
  X->fits = fits;
}

// Block k = (r, q) places the edges of segment k in ascending edge order:
// CTA r's gather list gets the column offset within its slice, and epos[e]
// the edge's slot in CTA q's receive buffer.
__global__ void __launch_bounds__(1024) k_edge_partition(
    const int32_t* __restrict__ off, const int32_t* __restrict__ cols,
    const int32_t* __restrict__ eid, int64_t vs, int32_t sc, int32_t so, int C,
    const XLayout* __restrict__ X, int32_t* __restrict__ send_src, int32_t* __restrict__ epos) {
  __shared__ int32_t wsum[32];
  const int k = blockIdx.x, r = k / C;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int32_t E = off[vs];
  int32_t* dst = send_src + X->sendbase[r] + X->sendoff[k];
  const int32_t rbase = X->recvoff[k];
  int32_t base = 0;
  for (int32_t t0 = 0; t0 < E; t0 += 1024 * 8) {
    const int32_t e0 = t0 + (int32_t)threadIdx.x * 8;
    uint32_t hit = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (e0 + q < E && edge_key(e0 + q, cols, eid, sc, so, C) == k) hit |= 1u << q;
    const int32_t own = __popc(hit);
    int32_t inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane == 31) wsum[w] = inc;
    __syncthreads();
    if (w == 0) {
      int32_t x = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += u;
      }
      wsum[lane] = x;
    }
    __syncthreads();
    int32_t pos = base + (w > 0 ? wsum[w - 1] : 0) + inc - own;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (hit >> q & 1u) {
        dst[pos] = cols[e0 + q] - r * sc;
        epos[e0 + q] = rbase + pos;
        ++pos;
      }
    base += wsum[31];
    __syncthreads();  // wsum is rewritten by the next tile
  }
}

// code[i]: the receive-buffer slot of student id i's single edge; -1 for no
// teacher token; for k >= 2 tokens, -2 - (8 * off[i] + min(k, 9) - 2): their
// slots are epos[off[i] .. off[i] + k), and the count field 7 means "read
// off[i + 1]" (the exchange path holds at most 8 x 76 KiB of teacher row, so
// 8 * off[i] stays far below 2^31)
__global__ void k_exchange_codes(const int32_t* __restrict__ off,
                                 const int32_t* __restrict__ epos, int64_t vs,
                                 int32_t* __restrict__ code) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vs;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t b = off[i], k = off[i + 1] - b;
    code[i] = k == 1 ? epos[b] : (k == 0 ? -1 : -2 - (8 * b + (k < 9 ? k : 9) - 2));
  }
}

// Student ids with several teacher tokens, in ascending order: mflag[i] = 1
// for them; after an exclusive scan (k_map_scan) mpre[i] is the number of
// them below i, and mlist / mcode list each one with its code.
__global__ void k_multi_flag(const int32_t* __restrict__ code, int64_t vs,
                             int32_t* __restrict__ mflag) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vs;
       i += (int64_t)gridDim.x * blockDim.x)
    mflag[i] = code[i] <= -2;
}
__global__ void k_multi_scatter(const int32_t* __restrict__ code,
                                const int32_t* __restrict__ mpre, int64_t vs,
                                int32_t* __restrict__ mlist, int32_t* __restrict__ mcode) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vs;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t c = code[i];
    if (c <= -2) {
      mlist[mpre[i]] = (int32_t)i;
      mcode[mpre[i]] = c;
    }
  }
}

// ---------------------------------------------------------------- slice lists

// The slice that writes student id i: the one holding its teacher column (its
// first, for an id with several); unmatched ids are spread over the slices in
// contiguous id ranges.
__device__ __forceinline__ int slice_of(int64_t i, const int32_t* __restrict__ one,
                                        const int32_t* __restrict__ off,
                                        const int32_t* __restrict__ cols, int64_t vs, int32_t sc,
                                        int nsl) {
  const int32_t c = one[i];
  if (c >= 0) return c / sc;
  if (c == -2) return cols[off[i]] / sc;
  return (int)(i * nsl / vs);
}

// ids per slice: a shared-memory histogram per block (one atomic per warp
// and slice, via __match_any_sync), then one global atomic per block and slice
__global__ void k_slice_count(const int32_t* __restrict__ one, const int32_t* __restrict__ off,
                              const int32_t* __restrict__ cols, int64_t vs, int32_t sc, int nsl,
                              int32_t* __restrict__ slice_cnt, const XLayout* X) {
  if (X && X->fits) return;  // the exchange path runs instead
  __shared__ int32_t h[kMaxSlices];
  for (int s = threadIdx.x; s < nsl; s += blockDim.x) h[s] = 0;
  __syncthreads();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x; i0 < vs; i0 += stride) {
    const int64_t i = i0 + threadIdx.x;
    const int s = i < vs ? slice_of(i, one, off, cols, vs, sc, nsl) : -1;
    const unsigned same = __match_any_sync(0xffffffffu, s);
    if (s >= 0 && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&h[s], __popc(same));
  }
  __syncthreads();
  for (int s = threadIdx.x; s < nsl; s += blockDim.x)
    if (h[s]) atomicAdd(&slice_cnt[s], h[s]);
}

// Block r lists the ids of slice r in ascending order (a stable partition:
// 8 ids per thread per tile, block-wide prefix sums of the matches), with
// their column within the slice, or -1 (unmatched) / -2 (several columns).
// It also writes slice_off[r] (and slice_off[nsl] from the last block).
__global__ void __launch_bounds__(1024) k_slice_partition(
    const int32_t* __restrict__ one, const int32_t* __restrict__ off,
    const int32_t* __restrict__ cols, int64_t vs, int32_t sc, int nsl,
    const int32_t* __restrict__ slice_cnt, int32_t* __restrict__ slice_off,
    int32_t* __restrict__ list_id, int32_t* __restrict__ list_val, const XLayout* X) {
  if (X && X->fits) return;  // the exchange path runs instead
  __shared__ int32_t wsum[32];
  __shared__ int32_t base_sh;
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    int32_t b = 0;
    for (int s = 0; s < r; ++s) b += slice_cnt[s];
    base_sh = b;
    slice_off[r] = b;
    if (r == nsl - 1) slice_off[nsl] = b + slice_cnt[r];
  }
  __syncthreads();
  int32_t base = base_sh;
  for (int64_t t0 = 0; t0 < vs; t0 += 1024 * 8) {
    const int64_t i0 = t0 + (int64_t)threadIdx.x * 8;
    uint32_t hit = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (i0 + q < vs && slice_of(i0 + q, one, off, cols, vs, sc, nsl) == r) hit |= 1u << q;
    const int32_t own = __popc(hit);
    int32_t inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane == 31) wsum[w] = inc;
    __syncthreads();
    if (w == 0) {
      int32_t x = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += u;
      }
      wsum[lane] = x;
    }
    __syncthreads();
    int32_t pos = base + (w > 0 ? wsum[w - 1] : 0) + inc - own;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (hit >> q & 1u) {
        const int32_t c = one[i0 + q];
        list_id[pos] = (int32_t)(i0 + q);
        list_val[pos] = c >= 0 ? c - r * sc : c;
        ++pos;
      }
    base += wsum[31];
    __syncthreads();  // wsum is rewritten by the next tile
  }
}

// ---------------------------------------------------------------- projection

// Work items (token row, slice), grid-strided over one CTA per SM.  Each item
// stages its slice of the teacher row (buffer it & 1; the copy of the next
// item is started before this one is processed), then writes the output of
// every id on the slice's list: a single teacher column is read from shared
// memory, several are read from the row in global memory (still in L2, the
// other slices' CTAs having just streamed it) and folded in column order.
template <typename TI, typename TO>
__global__ void __launch_bounds__(kPT, 1)
    k_project_slices(const TI* __restrict__ zt, int64_t n, int64_t vt, int64_t vs, float inv_t,
                     const int32_t* __restrict__ off, const int32_t* __restrict__ cols,
                     const int32_t* __restrict__ list_id, const int32_t* __restrict__ list_val,
                     const int32_t* __restrict__ slice_off, int64_t sc, int nsl,
                     TO* __restrict__ out, uint32_t* status, const XLayout* X) {
  if (X && X->fits) return;  // the exchange path runs instead
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const size_t buf_bytes = (size_t)sc * sizeof(TI);
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars[1]), 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  const int64_t items = n * nsl;
  // stage item `item` into buffer b: the 16-byte-aligned bulk by one bulk
  // copy, a ragged tail (or a whole unaligned slice) by plain loads
  auto stage = [&](int64_t item, int b) {
    const int64_t row = item / nsl, c0 = (item % nsl) * sc;
    const int64_t clen = vt - c0 < sc ? vt - c0 : sc;
    const TI* src = zt + row * vt + c0;
    TI* dst = reinterpret_cast<TI*>(smem_raw + (size_t)b * buf_bytes);
    const bool al = ((reinterpret_cast<uintptr_t>(src) | ptx::smem_u32(dst)) & 15) == 0;
    const int64_t nb = al ? clen * (int64_t)sizeof(TI) / 16 * 16 : 0;
    if (threadIdx.x == 0 && !*reinterpret_cast<volatile int*>(&abort_flag)) {
      // (after a timed-out wait no new copy starts; later waits give up)
      const uint32_t bar = ptx::smem_u32(&bars[b]);
      ptx::mbar_expect_tx(bar, (uint32_t)nb);
      if (nb > 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        ptx::bulk_load(ptx::smem_u32(dst), src, (uint32_t)nb, bar);
      }
    }
    for (int64_t q = nb / (int64_t)sizeof(TI) + threadIdx.x; q < clen; q += kPT) dst[q] = src[q];
  };
  if (blockIdx.x < items) stage(blockIdx.x, 0);
  uint32_t parity = 0;  // bit b: phase parity to wait for on buffer b
  // the first wait that gave up: its copy may still be in flight (none starts
  // after it, the abort flag being set by then)
  int pend_b = -1;
  uint32_t pend_p = 0;
  int it = 0;
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
    const int b = it & 1;
    // buffer b ^ 1 held the previous item, which every thread is done with
    if (item + gridDim.x < items) stage(item + gridDim.x, b ^ 1);
    if (!ptx::warp_wait(ptx::smem_u32(&bars[b]), (parity >> b) & 1u, &abort_flag, status) &&
        pend_b < 0) {
      pend_b = b;
      pend_p = (parity >> b) & 1u;
    }
    parity ^= 1u << b;
    __syncthreads();  // the plain-loaded columns too
    const int64_t row = item / nsl;
    const int r = (int)(item % nsl);
    const TI* zs = reinterpret_cast<const TI*>(smem_raw + (size_t)b * buf_bytes);
    const TI* zrow = zt + row * vt;
    TO* o = out + row * vs;
    const int32_t k0 = slice_off[r], k1 = slice_off[r + 1];
    // four list entries per thread in flight; a warp's stores at each step
    // go to 32 consecutive entries, i.e. one short ascending run of ids
    for (int32_t k = k0 + (int32_t)threadIdx.x; k < k1; k += kPT * 4) {
      int32_t id[4], v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int32_t kk = k + u * kPT;
        id[u] = kk < k1 ? list_id[kk] : -1;
        v[u] = kk < k1 ? list_val[kk] : -1;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (id[u] < 0) continue;
        float r_;
        if (v[u] >= 0) {
          r_ = ld<TI>(zs + v[u]) * inv_t;
        } else if (v[u] == -2) {
          const int32_t e = off[id[u] + 1];
          r_ = -INFINITY;
#pragma unroll 1
          for (int32_t t = off[id[u]]; t < e; ++t)
            r_ = logaddexp(r_, ld<TI>(zrow + cols[t]) * inv_t);
        } else {
          r_ = -INFINITY;
        }
        st<TO>(o + id[u], r_ > -INFINITY ? r_ : lowest<TO>());
      }
    }
    __syncthreads();  // buffer b is read; the item after next overwrites it
  }
  if (pend_b >= 0 && threadIdx.x < 32)
    ptx::warp_wait(ptx::smem_u32(&bars[pend_b]), pend_p, &abort_flag, status, false);
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
__device__ __forceinline__ uint32_t cl_map(uint32_t a, uint32_t rank) {
  asm("mapa.shared::cluster.u32 %0, %0, %1;" : "+r"(a) : "r"(rank));
  return a;
}

// A CTA's outgoing segments, read once from the exchange layout: for each
// destination CTA q, the mapped receive address and barrier, the local
// source and the byte count (0: nothing to send).  Per row only thread 0
// reads them, from shared memory, so shipping a row's segments waits on no
// global load.
struct SendDesc {
  uint32_t dst[kMaxC], bar[kMaxC], src[kMaxC], bytes[kMaxC];
};
template <typename TI>
__device__ __forceinline__ void send_desc_init(SendDesc& d, const XLayout* X, uint32_t r,
                                               uint32_t C, const TI* send, const TI* recv,
                                               uint32_t bar_r) {
  const uint32_t q = threadIdx.x;
  if (q < C) {
    const int k = (int)(r * C + q);
    d.bytes[q] = (uint32_t)pad8(X->cnt[k]) * (uint32_t)sizeof(TI);
    d.dst[q] = cl_map(ptx::smem_u32(recv + X->recvoff[k]), q);
    d.bar[q] = cl_map(bar_r, q);
    d.src[q] = ptx::smem_u32(send + X->sendoff[k]);
  }
}
// Thread 0, after the CTA barrier that completes the send buffer: one
// shared::cta -> shared::cluster bulk copy per non-empty segment.
__device__ __forceinline__ void send_segments(const SendDesc& d, uint32_t C) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  for (uint32_t q = 0; q < C; ++q) {
    if (d.bytes[q] == 0) continue;
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(d.dst[q]),
        "r"(d.src[q]), "r"(d.bytes[q]), "r"(d.bar[q])
        : "memory");
  }
}

// Exchange path.  A cluster of C CTAs takes one token row at a time.  CTA r
// stages its slice of the teacher row (one bulk copy; the next row's copy
// starts as soon as the gather below has read the slice), gathers the values
// its map edges need into a send buffer ordered by destination CTA -- random
// reads of local shared memory only -- and ships segment (r, q) to CTA q with
// one shared::cta -> shared::cluster bulk copy completing on q's receive
// barrier.  CTA q then writes student ids [q*so, q*so + so) of the output row
// from its receive buffer with 16-byte stores.  One cluster barrier per row:
// after it every CTA has received (so every send buffer is free again) and
// read its receive buffer (so it may be refilled); the receive barrier of the
// next row is armed before it, so no copy can arrive early.
//
// Everything that depends only on the map stays on chip across rows: each
// thread's output codes in registers, and, for up to kMCap ids with several
// teacher tokens, their id and (with two tokens) both receive slots in a
// shared-memory table, so a row's output needs no global loads but its own
// gather list.  That list is read one 8-slot step ahead of the gather (the
// first step before the slice wait).
template <typename TI, typename TO, int XT>
__global__ void __launch_bounds__(XT, XT == kXTNarrow ? 2 : 1)
    k_project_exchange(const TI* __restrict__ zt, int64_t n, int64_t vt, int64_t vs,
                       float inv_t, const int32_t* __restrict__ off,
                       const int32_t* __restrict__ epos, const int32_t* __restrict__ code,
                       const int32_t* __restrict__ mpre, const int32_t* __restrict__ mlist,
                       const int32_t* __restrict__ mcode, const int32_t* __restrict__ send_src,
                       const XLayout* __restrict__ X, int64_t sc, int64_t so,
                       int64_t send_cap, int64_t recv_cap, TO* __restrict__ out,
                       uint32_t* status) {
  if (!X->fits) return;  // the slice path runs instead
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];  // 0: the staged slice, 1: the receive buffer
  __shared__ int abort_flag;
  __shared__ uint32_t mtab[kMCap];  // ids with several teacher tokens: 2 receive slots, or ~0
  __shared__ uint16_t mid[kMCap];   // ... their offsets in this CTA's id range
  __shared__ SendDesc sd;
  const uint32_t r = cl_rank(), C = cl_size();
  const int64_t ncl = gridDim.x / C;
  TI* const slice = reinterpret_cast<TI*>(smem_raw);
  TI* const send = slice + sc;        // sc and send_cap are multiples of 8
  TI* const recv = send + send_cap;
  const int64_t c0 = (int64_t)r * sc;
  const int64_t clen = vt - c0 < sc ? (vt - c0 > 0 ? vt - c0 : 0) : sc;
  const int64_t i_lo = (int64_t)r * so, i_hi = i_lo + so < vs ? i_lo + so : vs;
  const int32_t nsend = X->sendtot[r];
  const int32_t* gl = send_src + X->sendbase[r];
  const uint32_t rx_bytes = (uint32_t)X->recvtot[r] * (uint32_t)sizeof(TI);
  const uint32_t bar_s = ptx::smem_u32(&bars[0]), bar_r = ptx::smem_u32(&bars[1]);
  const uint32_t rcap = (uint32_t)recv_cap;  // < 0xfffe (planned)
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_s, 1);
    ptx::mbar_init(bar_r, 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  send_desc_init<TI>(sd, X, r, C, send, recv, bar_r);
  // ids with several teacher tokens: the first kMCap of this CTA's range get a
  // table entry (two receive slots; ~0 for three or more tokens)
  const int32_t m_lo = mpre[i_lo < i_hi ? i_lo : i_hi], m_hi = mpre[i_hi];
  const int32_t nm = m_hi - m_lo < kMCap ? m_hi - m_lo : kMCap;
  for (int32_t k = threadIdx.x; k < nm; k += XT) {
    const int32_t m = -2 - mcode[m_lo + k], e0 = m >> 3;
    mtab[k] = (m & 7) == 0 ? ((uint32_t)epos[e0] | ((uint32_t)epos[e0 + 1] << 16)) : ~0u;
    mid[k] = (uint16_t)(mlist[m_lo + k] - i_lo);
  }
  __syncthreads();
  // (returns whether some columns were plain-loaded: the wait then needs a
  // CTA barrier to see them; the bulk-copied ones come with the barrier wait)
  auto stage = [&](int64_t row) -> bool {
    const TI* src = zt + row * vt + c0;
    const bool al = ((reinterpret_cast<uintptr_t>(src) | ptx::smem_u32(slice)) & 15) == 0;
    const int64_t nb = al ? clen * (int64_t)sizeof(TI) / 16 * 16 : 0;
    if (threadIdx.x == 0 && !*reinterpret_cast<volatile int*>(&abort_flag)) {
      ptx::mbar_expect_tx(bar_s, (uint32_t)nb);
      if (nb > 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        ptx::bulk_load(ptx::smem_u32(slice), src, (uint32_t)nb, bar_s);
      }
    }
    const int64_t q0 = nb / (int64_t)sizeof(TI);
    for (int64_t q = q0 + threadIdx.x; q < clen; q += XT) slice[q] = src[q];
    return q0 < clen;
  };
  bool plain = false;
  const int64_t first = blockIdx.x / C;
  if (first < n) {
    plain = stage(first);
    if (threadIdx.x == 0) ptx::mbar_expect_tx(bar_r, rx_bytes);
  }
  cl_sync();  // every receive barrier is armed before any copy is sent
  // this thread's output ids are the same in every row: their codes, two
  // 16-bit slots per register, are loaded once (ranges longer than
  // kXSteps * 8 * XT ids are not planned for this kernel).  A code below
  // rcap is the receive slot of the id's single teacher token; 0xfffe marks
  // an id with several (written by the pass after the output), 0xffff one
  // that no teacher token reaches.
  uint32_t c16[kXSteps][4];
#pragma unroll
  for (int u = 0; u < kXSteps; ++u) {
    const int64_t j0 = i_lo + ((int64_t)u * XT + threadIdx.x) * 8;
#pragma unroll
    for (int q = 0; q < 4; ++q) c16[u][q] = 0xffffffffu;
    if (j0 >= i_hi) continue;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int32_t cq = j0 + q < i_hi ? code[j0 + q] : -1;
      const uint32_t h = cq >= 0 ? (uint32_t)cq : (cq == -1 ? 0xffffu : 0xfffeu);
      c16[u][q >> 1] = (c16[u][q >> 1] & ~(0xffffu << (16 * (q & 1)))) | (h << (16 * (q & 1)));
    }
  }
  // an id with several teacher tokens, folded from its edges in global memory
  auto fold = [&](int64_t id) -> float {
    const int32_t m = -2 - code[id], e0 = m >> 3;
    const int32_t e1 = (m & 7) == 7 ? off[id + 1] : e0 + (m & 7) + 2;
    float x = -INFINITY;
#pragma unroll 1
    for (int32_t e = e0; e < e1; ++e) x = logaddexp(x, ld<TI>(recv + epos[e]) * inv_t);
    return x;
  };
  uint32_t ps = 0, pr = 0;
  int pend = 0;  // bit 0 / 1: a wait on the slice / receive barrier gave up
  uint32_t pend_ps = 0, pend_pr = 0;
  const int32_t t_first = (int32_t)threadIdx.x * 8;
  for (int64_t row = first; row < n; row += ncl) {
    // the gather list's first step (the same in every row), ahead of the wait
    int4 ga = make_int4(0, 0, 0, 0), gb = ga;
    if (t_first < nsend) {
      ga = reinterpret_cast<const int4*>(gl + t_first)[0];
      gb = reinterpret_cast<const int4*>(gl + t_first)[1];
    }
    if (!ptx::warp_wait(bar_s, ps, &abort_flag, status) && !(pend & 1)) {
      pend |= 1;
      pend_ps = ps;
    }
    ps ^= 1u;
    if (plain) __syncthreads();  // the plain-loaded columns too
    // 8 slots per thread step: nsend, the list start and send are multiples of 8
    for (int32_t t0 = t_first; t0 < nsend; t0 += XT * 8) {
      const int32_t t1 = t0 + XT * 8;
      int4 na = ga, nb = gb;
      if (t1 < nsend) {
        na = reinterpret_cast<const int4*>(gl + t1)[0];
        nb = reinterpret_cast<const int4*>(gl + t1)[1];
      }
      const int32_t g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
      TI v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = slice[g[q]];
      if constexpr (sizeof(TI) == 2) {
        *reinterpret_cast<uint4*>(send + t0) = *reinterpret_cast<const uint4*>(v);
      } else {
        reinterpret_cast<uint4*>(send + t0)[0] = reinterpret_cast<const uint4*>(v)[0];
        reinterpret_cast<uint4*>(send + t0)[1] = reinterpret_cast<const uint4*>(v)[1];
      }
      ga = na;
      gb = nb;
    }
    __syncthreads();  // send is complete; the slice is free for the next row
    // the segments first (the cluster waits on them), then the next row's slice
    if (threadIdx.x == 0 && !*reinterpret_cast<volatile int*>(&abort_flag)) send_segments(sd, C);
    if (row + ncl < n) plain = stage(row + ncl);
    if (!ptx::warp_wait(bar_r, pr, &abort_flag, status) && !(pend & 2)) {
      pend |= 2;
      pend_pr = pr;
    }
    pr ^= 1u;
    // the output row: 8 ids per thread step, from the codes held in registers
    TO* o = out + row * vs;
#pragma unroll
    for (int u = 0; u < kXSteps; ++u) {
      const int64_t j0 = i_lo + ((int64_t)u * XT + threadIdx.x) * 8;
      if (j0 >= i_hi) break;
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t cq = (c16[u][q >> 1] >> (16 * (q & 1))) & 0xffffu;
        // slot 0 stands in for ids without a single slot (always in bounds)
        const float x = ld<TI>(recv + (cq < rcap ? cq : 0u)) * inv_t;
        v[q] = cq < rcap && x > -INFINITY ? x : lowest<TO>();
      }
      if (j0 + 8 <= i_hi && (reinterpret_cast<uintptr_t>(o + j0) & 15) == 0) {
        store_vec(o + j0, v);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (j0 + q < i_hi) st<TO>(o + j0 + q, v[q]);
      }
    }
    // ids with several teacher tokens: their columns' values are folded in
    // column order and overwrite the placeholders above (same CTA, after the
    // barrier, so the later store wins; the sectors are already whole)
    __syncthreads();
    for (int32_t k = threadIdx.x; k < m_hi - m_lo; k += XT) {
      float x;
      int64_t id;
      const uint32_t e = k < nm ? mtab[k] : ~0u;
      if (e != ~0u) {  // two tokens, both slots from the table
        id = i_lo + mid[k];
        x = logaddexp(ld<TI>(recv + (e & 0xffffu)) * inv_t, ld<TI>(recv + (e >> 16)) * inv_t);
      } else {  // three or more tokens, or beyond the table: edges from global memory
        id = k < nm ? i_lo + mid[k] : mlist[m_lo + k];
        x = fold(id);
      }
      st<TO>(o + id, x > -INFINITY ? x : lowest<TO>());
    }
    if (threadIdx.x == 0 && row + ncl < n) ptx::mbar_expect_tx(bar_r, rx_bytes);
    cl_sync();
  }
  // copies still in flight after a wait that gave up (bounded again)
  if (threadIdx.x < 32) {
    if (pend & 1) ptx::warp_wait(bar_s, pend_ps, &abort_flag, status, false);
    if (pend & 2) ptx::warp_wait(bar_r, pend_pr, &abort_flag, status, false);
  }
}

// ---------------------------------------------------------------- fused loss
// The projected teacher inside the distillation loss (orda-kernel README,
// "Cross-vocabulary distillation": token-map projection into a
// PrecomputedTeacher, whose logits the loss then reads at temperature 1).
// k_proj_loss runs the exchange of k_project_exchange -- the cluster shares a
// teacher row, CTA q receives the values of the teacher tokens that map into
// its student ids [q*so, q*so + so) -- and, instead of storing the projected
// values, uses them on chip against the student logits of the same ids:
//   forward:  the online-softmax state of each thread's ids (student at T_s,
//             projected teacher at 1), merged over the CTA and then over the
//             cluster in CTA 0, which finalises the token (CE, CE_t, KL,
//             saved statistics); the skew variants take a second sweep over
//             the same ids once CTA 0 has broadcast both normalisers;
//   backward: d z_s of each id from the saved statistics, stored directly.
// The projected [N, V_s] tensor never exists.  Ids no teacher token maps to
// take the lowest finite float, as the unfused projection writes them.
constexpr int kLT = 512;  // threads of the fused kernel (128 registers each)
// Student ids with several teacher tokens, per CTA, whose folded value is kept
// in shared memory for the row (beyond this, an id folds from global memory).
constexpr int64_t kPLSmem = 212 * 1024;  // dynamic shared memory of the fused kernel
struct PLParams {
  const void* zt;      // [n, vt] teacher logits
  const void* zs;      // [n, vs] student logits (same dtype)
  int64_t n, vt, vs;
  float inv_tp;        // 1 / projection temperature
  Consts c;            // the projected distribution enters at T = 1
  int variant;
  const int64_t* labels;
  int64_t ignore;
  float *ce_s, *ce_t, *kl, *stats;  // forward outputs (stats never NULL)
  const float* row_scale;           // backward
  float w_sce, w_kl_ts;
  void* dz;                         // [n, vs] d loss / d z_s
  const int32_t *off, *epos, *code, *send_src, *mpre, *mlist, *mcode;
  const XLayout* X;
  int64_t sc, so, send_cap, recv_cap;
  uint32_t* status;
};

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// the projected (tempered) teacher logits of ids j0 .. j0 + 7 from the
// receive buffer; ids with several teacher tokens fold their columns' values
// in column order (their edges from the code array), ids with none take the
// lowest finite float
template <typename TI>
__device__ __forceinline__ void proj_values(const PLParams& P, const TI* recv, const float* mval,
                                            uint32_t rcap, const uint32_t (&cw)[4], int64_t j0,
                                            int nv, float* v) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t cq = (cw[q >> 1] >> (16 * (q & 1))) & 0xffffu;
    float x;
    if (cq < rcap) {  // one teacher token: its receive slot
      x = ld<TI>(recv + cq) * P.inv_tp;
    } else if (cq < 0xfffeu) {  // several, folded for this row in shared memory
      x = mval[cq - rcap];
    } else if (cq == 0xfffeu && q < nv) {  // several, beyond the table: fold here
      const int64_t id = j0 + q;
      const int32_t m = -2 - P.code[id], e0 = m >> 3;
      const int32_t e1 = (m & 7) == 7 ? P.off[id + 1] : e0 + (m & 7) + 2;
      x = -INFINITY;
#pragma unroll 1
      for (int32_t e = e0; e < e1; ++e) x = logaddexp(x, ld<TI>(recv + P.epos[e]) * P.inv_tp);
    } else {
      x = -INFINITY;
    }
    v[q] = x > -INFINITY ? x : -FLT_MAX;
  }
}

// student logits of ids j0 .. j0 + nv - 1 of one row (16-byte loads when whole)
__device__ __forceinline__ void load8(const __nv_bfloat16* p, int nv, float* s) {
  if (nv == 8 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    s[0] = bf16lo(w.x); s[1] = bf16hi(w.x); s[2] = bf16lo(w.y); s[3] = bf16hi(w.y);
    s[4] = bf16lo(w.z); s[5] = bf16hi(w.z); s[6] = bf16lo(w.w); s[7] = bf16hi(w.w);
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) s[q] = q < nv ? __bfloat162float(p[q]) : 0.f;
  }
}
__device__ __forceinline__ void load8(const float* p, int nv, float* s) {
  if (nv == 8 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w; s[4] = b.x; s[5] = b.y; s[6] = b.z; s[7] = b.w;
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) s[q] = q < nv ? p[q] : 0.f;
  }
}

// 8 consecutive logits as raw 16-byte words (one for bf16, two for fp32),
// loaded ahead of their use and converted when needed
template <typename TI>
struct Vec8 {
  uint4 w[sizeof(TI) / 2];
};
template <typename TI>
__device__ __forceinline__ void ldv8(const TI* p, Vec8<TI>& v) {
#pragma unroll
  for (int i = 0; i < (int)(sizeof(TI) / 2); ++i) v.w[i] = reinterpret_cast<const uint4*>(p)[i];
}
__device__ __forceinline__ void cvt8(const Vec8<__nv_bfloat16>& v, float* s) {
  const uint4 w = v.w[0];
  s[0] = bf16lo(w.x); s[1] = bf16hi(w.x); s[2] = bf16lo(w.y); s[3] = bf16hi(w.y);
  s[4] = bf16lo(w.z); s[5] = bf16hi(w.z); s[6] = bf16lo(w.w); s[7] = bf16hi(w.w);
}
__device__ __forceinline__ void cvt8(const Vec8<float>& v, float* s) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    s[4 * i + 0] = __uint_as_float(v.w[i].x);
    s[4 * i + 1] = __uint_as_float(v.w[i].y);
    s[4 * i + 2] = __uint_as_float(v.w[i].z);
    s[4 * i + 3] = __uint_as_float(v.w[i].w);
  }
}

// Visit this thread's student ids, 8 per step (steps kLT * 8 ids apart), in a
// loop that is not unrolled (the per-step work is large: unrolled, it
// overflowed the instruction cache).  The step's receive codes are selected
// from the register array by compare (no dynamic register indexing), and the
// next step's student logits are loaded while this step computes.
// body(j0, nv, cw, s): ids j0 .. j0 + nv - 1, their codes and student logits.
template <typename TI, int STEPS, class Body>
__device__ __forceinline__ void for_ids(const TI* zsr, int64_t i_lo, int64_t i_hi, bool vec,
                                        const uint32_t (&c16)[STEPS][4], Body&& body) {
  Vec8<TI> cur, nxt;
  int64_t j0 = i_lo + (int64_t)threadIdx.x * 8;
  bool cur_ok = vec && j0 + 8 <= i_hi;
  if (cur_ok) ldv8(zsr + j0, cur);
#pragma unroll 1
  for (int u = 0; u < STEPS; ++u, j0 += (int64_t)kLT * 8) {
    if (j0 >= i_hi) break;
    const int nv = (int)(i_hi - j0 < 8 ? i_hi - j0 : 8);
    const int64_t j1 = j0 + (int64_t)kLT * 8;
    const bool nxt_ok = vec && u + 1 < STEPS && j1 + 8 <= i_hi;
    if (nxt_ok) ldv8(zsr + j1, nxt);
    uint32_t cw[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
#pragma unroll
    for (int k = 0; k < STEPS; ++k)
      if (k == u) {
        cw[0] = c16[k][0];
        cw[1] = c16[k][1];
        cw[2] = c16[k][2];
        cw[3] = c16[k][3];
      }
    float s[8];
    if (cur_ok) cvt8(cur, s);
    else load8(zsr + j0, nv, s);
    body(j0, nv, cw, s);
    cur = nxt;
    cur_ok = nxt_ok;
  }
}

// merge every thread's state into thread 0 (red: 16 x kRec floats)
__device__ __forceinline__ void pl_block_merge(RowState& st, const Consts& c, float* red) {
  warp_merge(st, c);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) st.store(red + w * kRec);
  __syncthreads();
  if (w == 0) {
    if (l < kLT / 32) st.load(red + l * kRec);
    else st.init();
    warp_merge(st, c);
  }
  __syncthreads();  // red is reused by the next merge
}
__device__ __forceinline__ float3 pl_block_sum3(float a, float b, float d, float* red) {
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
    d += __shfl_xor_sync(0xffffffffu, d, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    red[3 * w] = a;
    red[3 * w + 1] = b;
    red[3 * w + 2] = d;
  }
  __syncthreads();
  float3 r = make_float3(0.f, 0.f, 0.f);
  if (threadIdx.x == 0)
    for (int i = 0; i < kLT / 32; ++i) {
      r.x += red[3 * i];
      r.y += red[3 * i + 1];
      r.z += red[3 * i + 2];
    }
  __syncthreads();
  return r;
}

// per-token outputs from the cluster-merged state (CTA 0, thread 0)
__device__ __forceinline__ RowOut pl_finish(const PLParams& P, int64_t row, RowState& st,
                                            bool write_kl) {
  bool valid = true, bad = false;
  if (P.labels) {
    const int64_t y = P.labels[row];
    valid = y != P.ignore;
    bad = valid && (y < 0 || y >= P.vs);
  }
  const RowOut o = finalize(st, P.c, P.variant, true, false, 0.f, 0.f);
  const float nan = __int_as_float(0x7fc00000);
  if (P.ce_s) P.ce_s[row] = !valid ? 0.f : (bad ? nan : o.ce_s);
  if (P.ce_t) P.ce_t[row] = !valid ? 0.f : (bad ? nan : o.ce_t);
  if (P.kl && write_kl) P.kl[row] = valid ? o.kl : 0.f;
  float4* s4 = reinterpret_cast<float4*>(P.stats + row * KD_STATS_PER_TOKEN);
  s4[0] = make_float4(o.lse_s1, o.lse_sT, o.lse_t1, o.lse_tT);
  s4[1] = make_float4(o.kl_rev, 0.f, 0.f, o.dlse);
  return o;
}

template <typename TI, int MODE, bool SKEW, int STEPS>
__global__ void __launch_bounds__(kLT, 1) k_proj_loss(const __grid_constant__ PLParams P) {
  const XLayout* __restrict__ X = P.X;
  if (!X->fits) {  // the map overflows a receive buffer: the fused path cannot run it
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(P.status, KD_DEV_MAP_UNSUPPORTED);
    return;
  }
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];  // 0: the staged slice, 1: the receive buffer
  __shared__ int abort_flag;
  __shared__ __align__(16) float red[(kLT / 32) * kRec];   // block reductions
  __shared__ __align__(16) float mslot[2][kMaxC][kRec];    // CTA 0: each CTA's row state
  __shared__ __align__(16) float jslot[2][kMaxC][4];       // CTA 0: each CTA's skew sums
  __shared__ float bc[2][2];                               // skew: dlse, lse(a_t) from CTA 0
  __shared__ uint32_t mtab[kMCap];  // ids with several teacher tokens: 2 receive slots, or ~0
  __shared__ float mval[kMCap];     // ... their folded (tempered) values in the current row
  __shared__ SendDesc sd;
  const uint32_t r = cl_rank(), C = cl_size();
  const int64_t ncl = gridDim.x / C;
  const int64_t n = P.n, vt = P.vt, vs = P.vs, sc = P.sc;
  const TI* __restrict__ zt = static_cast<const TI*>(P.zt);
  TI* const slice = reinterpret_cast<TI*>(smem_raw);
  TI* const send = slice + sc;
  TI* const recv = send + P.send_cap;
  const int64_t c0 = (int64_t)r * sc;
  const int64_t clen = vt - c0 < sc ? (vt - c0 > 0 ? vt - c0 : 0) : sc;
  const int64_t i_lo = (int64_t)r * P.so, i_hi = i_lo + P.so < vs ? i_lo + P.so : vs;
  const int32_t nsend = X->sendtot[r];
  const int32_t* gl = P.send_src + X->sendbase[r];
  const uint32_t rx_bytes = (uint32_t)X->recvtot[r] * (uint32_t)sizeof(TI);
  const uint32_t bar_s = ptx::smem_u32(&bars[0]), bar_r = ptx::smem_u32(&bars[1]);
  uint32_t* status = P.status;
  const Consts c = P.c;
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_s, 1);
    ptx::mbar_init(bar_r, 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  send_desc_init<TI>(sd, X, r, C, send, recv, bar_r);
  __syncthreads();
  auto stage = [&](int64_t row) -> bool {
    const TI* src = zt + row * vt + c0;
    const bool al = ((reinterpret_cast<uintptr_t>(src) | ptx::smem_u32(slice)) & 15) == 0;
    const int64_t nb = al ? clen * (int64_t)sizeof(TI) / 16 * 16 : 0;
    if (threadIdx.x == 0 && !*reinterpret_cast<volatile int*>(&abort_flag)) {
      ptx::mbar_expect_tx(bar_s, (uint32_t)nb);
      if (nb > 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        ptx::bulk_load(ptx::smem_u32(slice), src, (uint32_t)nb, bar_s);
      }
    }
    const int64_t q0 = nb / (int64_t)sizeof(TI);
    for (int64_t q = q0 + threadIdx.x; q < clen; q += kLT) slice[q] = src[q];
    return q0 < clen;
  };
  bool plain = false;
  const int64_t first = blockIdx.x / C;
  if (first < n) {
    plain = stage(first);
    if (threadIdx.x == 0) ptx::mbar_expect_tx(bar_r, rx_bytes);
  }
  cl_sync();  // every receive barrier is armed before any copy is sent
  // this thread's student ids are the same in every row: their receive codes
  // (two 16-bit slots per register) are loaded once
  // ids with several teacher tokens: the first kMCap of this CTA's range get a
  // table entry (their two receive slots; ~0 for three or more tokens) and
  // codes rcap + k; the rest keep the marker 0xfffe (folded from global memory)
  const uint32_t rcap = (uint32_t)P.recv_cap;
  const int32_t m_lo = P.mpre[i_lo < i_hi ? i_lo : i_hi], m_hi = P.mpre[i_hi];
  const int32_t nm = m_hi - m_lo < kMCap ? m_hi - m_lo : kMCap;
  for (int32_t k = threadIdx.x; k < nm; k += kLT) {
    const int32_t m = -2 - P.mcode[m_lo + k], e0 = m >> 3;
    mtab[k] = (m & 7) == 0 ? ((uint32_t)P.epos[e0] | ((uint32_t)P.epos[e0 + 1] << 16)) : ~0u;
  }
  uint32_t c16[STEPS][4];
#pragma unroll
  for (int u = 0; u < STEPS; ++u) {
    const int64_t j0 = i_lo + ((int64_t)u * kLT + threadIdx.x) * 8;
#pragma unroll
    for (int q = 0; q < 4; ++q) c16[u][q] = 0xffffffffu;
    if (j0 >= i_hi) continue;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int32_t cq = j0 + q < i_hi ? P.code[j0 + q] : -1;
      uint32_t h = cq >= 0 ? (uint32_t)cq : 0xffffu;
      if (cq <= -2) {
        const int32_t k = P.mpre[j0 + q] - m_lo;
        h = k < nm ? rcap + (uint32_t)k : 0xfffeu;
      }
      c16[u][q >> 1] = (c16[u][q >> 1] & ~(0xffffu << (16 * (q & 1)))) | (h << (16 * (q & 1)));
    }
  }
  uint32_t ps = 0, pr = 0;
  int pend = 0;
  uint32_t pend_ps = 0, pend_pr = 0;
  int lr = 0;  // local row count (parity selects the merge slots)
  const int32_t t_first = (int32_t)threadIdx.x * 8;
  for (int64_t row = first; row < n; row += ncl, ++lr) {
    // the gather list's first step (the same in every row), ahead of the wait;
    // later steps are loaded one step ahead of the gather
    int4 ga = make_int4(0, 0, 0, 0), gb = ga;
    if (t_first < nsend) {
      ga = reinterpret_cast<const int4*>(gl + t_first)[0];
      gb = reinterpret_cast<const int4*>(gl + t_first)[1];
    }
    if (!ptx::warp_wait(bar_s, ps, &abort_flag, status) && !(pend & 1)) {
      pend |= 1;
      pend_ps = ps;
    }
    ps ^= 1u;
    if (plain) __syncthreads();
    for (int32_t t0 = t_first; t0 < nsend; t0 += kLT * 8) {
      const int32_t t1 = t0 + kLT * 8;
      int4 na = ga, nb = gb;
      if (t1 < nsend) {
        na = reinterpret_cast<const int4*>(gl + t1)[0];
        nb = reinterpret_cast<const int4*>(gl + t1)[1];
      }
      const int32_t g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
      TI v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = slice[g[q]];
      if constexpr (sizeof(TI) == 2) {
        *reinterpret_cast<uint4*>(send + t0) = *reinterpret_cast<const uint4*>(v);
      } else {
        reinterpret_cast<uint4*>(send + t0)[0] = reinterpret_cast<const uint4*>(v)[0];
        reinterpret_cast<uint4*>(send + t0)[1] = reinterpret_cast<const uint4*>(v)[1];
      }
      ga = na;
      gb = nb;
    }
    __syncthreads();  // send is complete; the slice is free for the next row
    // the segments first (the cluster waits on them), then the next row's slice
    if (threadIdx.x == 0 && !*reinterpret_cast<volatile int*>(&abort_flag)) send_segments(sd, C);
    if (row + ncl < n) plain = stage(row + ncl);
    if (!ptx::warp_wait(bar_r, pr, &abort_flag, status) && !(pend & 2)) {
      pend |= 2;
      pend_pr = pr;
    }
    pr ^= 1u;
    // this row's values of the tabled ids with several teacher tokens
    for (int32_t k = threadIdx.x; k < nm; k += kLT) {
      const uint32_t e = mtab[k];
      float x = -INFINITY;
      if (e != ~0u) {
        x = logaddexp(ld<TI>(recv + (e & 0xffffu)) * P.inv_tp, ld<TI>(recv + (e >> 16)) * P.inv_tp);
      } else {  // three or more tokens: their edges from global memory
        const int32_t id = P.mlist[m_lo + k], m = -2 - P.mcode[m_lo + k], e0 = m >> 3;
        const int32_t e1 = (m & 7) == 7 ? P.off[id + 1] : e0 + (m & 7) + 2;
#pragma unroll 1
        for (int32_t ed = e0; ed < e1; ++ed) x = logaddexp(x, ld<TI>(recv + P.epos[ed]) * P.inv_tp);
      }
      mval[k] = x;
    }
    __syncthreads();
    const TI* zsr = static_cast<const TI*>(P.zs) + row * vs;
    // whole 8-id groups load as 16-byte words when the rows are 16-byte aligned
    const bool vec = ((reinterpret_cast<uintptr_t>(zsr) | (uintptr_t)(i_lo * (int64_t)sizeof(TI))) & 15) == 0;
    const int par = lr & 1;
    const int64_t y = P.labels ? P.labels[row] : -1;
    if constexpr (MODE == 0) {
      // ---- forward: this thread's ids into one online-softmax state
      RowState st;
      st.init();
      float zys = 0.f, zyt = 0.f;
      for_ids<TI, STEPS>(zsr, i_lo, i_hi, vec, c16,
                         [&](int64_t j0, int nv, const uint32_t(&cw)[4], const float* s) {
                           float v[8];
                           proj_values<TI>(P, recv, mval, rcap, cw, j0, nv, v);
                           update<8, true, true>(st, s, v, nv, c);
                           if (y >= j0 && y < j0 + nv) {
                             const int jy = (int)(y - j0);
#pragma unroll
                             for (int q = 0; q < 8; ++q)
                               if (q == jy) {
                                 zys = s[q];
                                 zyt = v[q];
                               }
                           }
                         });
      st.zys = zys;
      st.zyt = zyt;
      pl_block_merge(st, c, red);
      if (threadIdx.x == 0) {  // this CTA's state into CTA 0's slot
        const uint32_t dst = cl_map(ptx::smem_u32(&mslot[par][r][0]), 0);
        st_cluster_v4(dst, make_float4(st.ms, st.ls1, st.lsT, st.mt));
        st_cluster_v4(dst + 16, make_float4(st.lt1, st.ltT, st.qd, st.qx));
        st_cluster_v4(dst + 32, make_float4(st.pd, st.px, st.zys, st.zyt));
        st_cluster_v4(dst + 48, make_float4(st.tk, st.jq, st.jp, st.jx));
      }
      if constexpr (SKEW) {
        // both normalisers before the second sweep: CTA 0 merges and
        // broadcasts them
        cl_sync();
        if (r == 0 && threadIdx.x == 0) {
          RowState m;
          m.load(&mslot[par][0][0]);
          for (uint32_t k = 1; k < C; ++k) {
            RowState o;
            o.load(&mslot[par][k][0]);
            merge(m, o, c);
          }
          const RowOut o = pl_finish(P, row, m, false);
          for (uint32_t k = 0; k < C; ++k) {
            st_cluster_f32(cl_map(ptx::smem_u32(&bc[par][0]), k), o.dlse);
            st_cluster_f32(cl_map(ptx::smem_u32(&bc[par][1]), k), o.lse_tT);
          }
        }
        cl_sync();
        const float dlse = bc[par][0], lse_tT = bc[par][1];
        const bool want_x = P.variant != KD_KL_SKEW_JS;
        float jq = 0.f, jp = 0.f, jx = 0.f;
        for_ids<TI, STEPS>(zsr, i_lo, i_hi, vec, c16,
                           [&](int64_t j0, int nv, const uint32_t(&cw)[4], const float* s) {
                             float v[8];
                             proj_values<TI>(P, recv, mval, rcap, cw, j0, nv, v);
#pragma unroll
                             for (int q = 0; q < 8; ++q)
                               if (q < nv) js_terms(s[q], v[q], lse_tT, dlse, c, jq, jp, jx, want_x);
                           });
        const float3 js = pl_block_sum3(jq, jp, jx, red);
        if (threadIdx.x == 0)
          st_cluster_v4(cl_map(ptx::smem_u32(&jslot[par][r][0]), 0),
                        make_float4(js.x, js.y, js.z, 0.f));
      }
    } else {
      // ---- backward: d z_s of this thread's ids
      const float scale = P.row_scale[row];
      float sv[KD_STATS_PER_TOKEN];
#pragma unroll
      for (int i = 0; i < KD_STATS_PER_TOKEN; ++i) sv[i] = P.stats[row * KD_STATS_PER_TOKEN + i];
      const float sq_s = c.pw == 2 ? ex2((2.f * sv[S_LSE_ST] - sv[S_LSE_S1]) * kL2E) : 0.f;
      TI* dzr = static_cast<TI*>(P.dz) + row * vs;
      for_ids<TI, STEPS>(zsr, i_lo, i_hi, vec, c16,
                         [&](int64_t j0, int nv, const uint32_t(&cw)[4], const float* s) {
        float v[8], g[8];
        proj_values<TI>(P, recv, mval, rcap, cw, j0, nv, v);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float gg = 0.f;
          if (scale != 0.f) {
            const float lp = fmaf(s[q], c.inv_ts, -sv[S_LSE_ST]);
            const float p = ex2(lp * kL2E);
            const float lq = fmaf(v[q], c.inv_tt, -sv[S_LSE_TT]);
            gg = P.w_kl_ts * kl_grad_pq(s[q], v[q], lp, lq, p, ex2(lq * kL2E), sv, P.variant, c);
            if (P.w_sce != 0.f)
              gg = fmaf(P.w_sce,
                        softmax_t1(s[q], p, sv[S_LSE_S1], sq_s, c.pw) - (j0 + q == y ? 1.f : 0.f),
                        gg);
            gg *= scale;
          }
          g[q] = gg;
        }
        if (nv == 8 && (reinterpret_cast<uintptr_t>(dzr + j0) & 15) == 0) {
          store_vec(dzr + j0, g);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q < nv) st<TI>(dzr + j0 + q, g[q]);
        }
      });
    }
    __syncthreads();
    if (threadIdx.x == 0 && row + ncl < n) ptx::mbar_expect_tx(bar_r, rx_bytes);
    cl_sync();
    if constexpr (MODE == 0) {
      if (r == 0 && threadIdx.x == 0) {
        if constexpr (SKEW) {
          float jq = 0.f, jp = 0.f, jx = 0.f;
          for (uint32_t k = 0; k < C; ++k) {
            jq += jslot[par][k][0];
            jp += jslot[par][k][1];
            jx += jslot[par][k][2];
          }
          const bool v_ok = !P.labels || y != P.ignore;
          P.stats[row * KD_STATS_PER_TOKEN + S_KL_PM] = jp;
          if (P.variant != KD_KL_SKEW_JS) P.stats[row * KD_STATS_PER_TOKEN + S_EPPM] = jx;
          if (P.kl) P.kl[row] = v_ok ? skew_kl(P.variant, c.beta, jq, jp) : 0.f;
        } else {
          RowState m;
          m.load(&mslot[par][0][0]);
          for (uint32_t k = 1; k < C; ++k) {
            RowState o;
            o.load(&mslot[par][k][0]);
            merge(m, o, c);
          }
          pl_finish(P, row, m, true);
        }
      }
    }
  }
  if (threadIdx.x < 32) {
    if (pend & 1) ptx::warp_wait(bar_s, pend_ps, &abort_flag, status, false);
    if (pend & 2) ptx::warp_wait(bar_r, pend_pr, &abort_flag, status, false);
  }
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// slices of a teacher row of vt elements: the fewest whose columns (sc, a
// multiple of 8) fit kSliceMax bytes; 0 when more than kMaxSlices are needed
int slices_for(int64_t vt, int64_t elem, int64_t* sc) {
  int64_t nsl = (vt * elem + kSliceMax - 1) / kSliceMax;
  if (nsl < 1) nsl = 1;
  const int64_t cols = ((vt + nsl - 1) / nsl + 7) / 8 * 8;
  nsl = (vt + cols - 1) / cols;
  if (nsl > kMaxSlices) return 0;
  *sc = cols;
  return (int)nsl;
}

struct ProjLayout {
  size_t cnt, off, cols, one, list_id, list_val, slice_cnt, slice_off, eid, epos, code, send_src,
      mflag, mpre, mlist, mcode, stmp, xl, bytes;
};
ProjLayout proj_layout(int64_t vt, int64_t vs) {
  ProjLayout L;
  L.cnt = 0;
  L.off = align256(L.cnt + (size_t)vs * 4);
  L.cols = align256(L.off + (size_t)(vs + 1) * 4);
  L.one = align256(L.cols + (size_t)vt * 4);
  L.list_id = align256(L.one + (size_t)vs * 4);
  L.list_val = align256(L.list_id + (size_t)vs * 4);
  L.slice_cnt = align256(L.list_val + (size_t)vs * 4);
  L.slice_off = align256(L.slice_cnt + (size_t)kMaxSlices * 4);
  L.eid = align256(L.slice_off + (size_t)(kMaxSlices + 1) * 4);
  L.epos = align256(L.eid + (size_t)vt * 4);
  L.code = align256(L.epos + (size_t)vt * 4);
  L.send_src = align256(L.code + (size_t)vs * 4);
  L.mflag = align256(L.send_src + ((size_t)vt + 8 * kMaxC * kMaxC) * 4);
  L.mpre = align256(L.mflag + (size_t)vs * 4);
  L.mlist = align256(L.mpre + (size_t)(vs + 1) * 4);
  L.mcode = align256(L.mlist + (size_t)vs * 4);
  L.stmp = align256(L.mcode + (size_t)vs * 4);
  L.xl = align256(L.stmp + (size_t)(2 * (vs / kScanTile + 2)) * 4);
  L.bytes = align256(L.xl + sizeof(XLayout));
  return L;
}

// Exchange plan: C = the fewest CTAs whose slices of a teacher row fit the
// slice bytes of a shape (at most kMaxC), the columns sc and student ids so
// per CTA, and the send / receive capacities that fill the rest of its shared
// memory.  The narrow shape (512 threads, two CTAs per SM, 38 KiB slices in
// 106 KiB) comes first: the two CTAs of an SM belong to different clusters and
// are in different phases of their rows, so one's waits are the other's work.
// Rows longer than 8 of its slices take the wide shape (1024 threads, one CTA
// per SM, 76 KiB slices in 220 KiB).  A CTA sends at most its sc columns
// (+ padding); what it receives depends on the map, so the device checks it
// (XLayout::fits) and the slice path runs otherwise.
struct XShape {
  int64_t slice, smem;  // bytes (the tables, about 6 KiB, come on top)
};
constexpr XShape kXNarrow{38 * 1024, 106 * 1024};  // kXTNarrow threads, two CTAs per SM
constexpr XShape kXWide{76 * 1024, 220 * 1024};    // kPT threads, one CTA per SM
struct XPlan {
  int C = 0;
  bool wide = false;
  int64_t sc = 0, so = 0, send_cap = 0, recv_cap = 0;
  size_t smem = 0;
  int max_clusters = 0;
};

template <typename TI, typename TO, int XT>
bool x_plan_shape(int64_t vt, int64_t vs, const XShape& sh, XPlan* P) {
  const int64_t elem = (int64_t)sizeof(TI);
  int64_t C = (vt * elem + sh.slice - 1) / sh.slice;
  if (C < 1) C = 1;
  if (C > kMaxC) return false;
  P->sc = ((vt + C - 1) / C + 7) / 8 * 8;
  C = (vt + P->sc - 1) / P->sc;
  P->C = (int)C;
  P->so = ((vs + C - 1) / C + 7) / 8 * 8;
  if (P->so > (int64_t)kXSteps * 8 * XT) return false;  // longer ranges: the slice path
  P->send_cap = P->sc + 8 * C;
  P->recv_cap = (sh.smem / elem - P->sc - P->send_cap) / 8 * 8;
  if (P->recv_cap > 65528) P->recv_cap = 65528;  // slots fit the kernel's 16-bit codes
  if (P->recv_cap < 8) return false;
  P->smem = (size_t)(P->sc + P->send_cap + P->recv_cap) * (size_t)elem;
  auto kern = k_project_exchange<TI, TO, XT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P->smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  // co-resident clusters of this shape (cached per device, cluster size and
  // buffer bytes)
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P->C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  const int nsm = tc_num_sms() > 0 ? tc_num_sms() : 1;
  const int per_sm = XT == kXTNarrow ? 2 : 1;
  cfg.gridDim = dim3((unsigned)(P->C * std::max(1, per_sm * nsm / P->C)));
  cfg.blockDim = dim3(XT);
  cfg.dynamicSmemBytes = P->smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int cached_max = max_active_clusters(reinterpret_cast<const void*>(kern), cfg);
  P->max_clusters = cached_max;
  return cached_max > 0;
}

template <typename TI, typename TO>
bool x_plan(int64_t vt, int64_t vs, XPlan* P) {
  *P = XPlan{};
  if (x_plan_shape<TI, TO, kXTNarrow>(vt, vs, kXNarrow, P)) return true;
  *P = XPlan{};
  P->wide = true;
  if (x_plan_shape<TI, TO, kPT>(vt, vs, kXWide, P)) return true;
  *P = XPlan{};
  return false;
}

template <typename TI, typename TO>
int launch_exchange(const XPlan& P, const void* zt, int64_t n, int64_t vt, int64_t vs,
                    float inv_t, const int32_t* off, const int32_t* epos, const int32_t* code,
                    const int32_t* mpre, const int32_t* mlist, const int32_t* mcode,
                    const int32_t* send_src, const XLayout* X, void* out, uint32_t* status,
                    cudaStream_t s) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  const int64_t clusters = n < P.max_clusters ? n : P.max_clusters;
  cfg.gridDim = dim3((unsigned)(P.C * clusters));
  cfg.blockDim = dim3(P.wide ? kPT : kXTNarrow);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch();
  auto kern = P.wide ? k_project_exchange<TI, TO, kPT> : k_project_exchange<TI, TO, kXTNarrow>;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const TI*>(zt), n, vt, vs, inv_t, off, epos,
                            code, mpre, mlist, mcode, send_src, X, P.sc, P.so, P.send_cap,
                            P.recv_cap, static_cast<TO*>(out), status) != cudaSuccess;
}

template <typename TI, typename TO>
int launch_project(const void* zt, int64_t n, int64_t vt, int64_t vs, float inv_t,
                   const int32_t* off, const int32_t* cols, const int32_t* list_id,
                   const int32_t* list_val, const int32_t* slice_off, int64_t sc, int nsl,
                   void* out, uint32_t* status, const XLayout* X, cudaStream_t s) {
  const size_t smem = 2 * (size_t)sc * sizeof(TI);
  auto kern = k_project_slices<TI, TO>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return 1;
  const int nsm = tc_num_sms() > 0 ? tc_num_sms() : 1;
  const int grid = (int)std::min<int64_t>(n * nsl, (int64_t)nsm);
  note_launch();
  kern<<<grid, kPT, smem, s>>>(static_cast<const TI*>(zt), n, vt, vs, inv_t, off, cols, list_id,
                               list_val, slice_off, sc, nsl, static_cast<TO*>(out), status, X);
  return cudaGetLastError() != cudaSuccess;
}

// out[0..n] = exclusive scan of in[0..n) with tile sums in tmp (2 * (n /
// kScanTile + 2) entries); one CTA does it alone when there is one tile.
void launch_scan(const int32_t* in, int64_t n, int32_t* out, int32_t* tmp, cudaStream_t s) {
  const int64_t tiles = (n + kScanTile - 1) / kScanTile;
  if (tiles <= 1) {
    note_launch();
    k_map_scan<<<1, 1024, 0, s>>>(in, n, out);
    return;
  }
  int32_t* tsum = tmp;
  int32_t* toff = tmp + tiles + 1;
  note_launch();
  k_scan_tiles<<<(unsigned)tiles, 1024, 0, s>>>(in, n, tsum);
  note_launch();
  k_map_scan<<<1, 1024, 0, s>>>(tsum, tiles, toff);
  note_launch();
  k_scan_apply<<<(unsigned)tiles, 1024, 0, s>>>(in, n, toff, out);
}

// The inverse map (count -> scan -> scatter -> per-id sort) and, with an
// exchange plan, the exchange lists (segments, send lists, receive slots,
// per-id codes); `multi`: also the list of ids with several teacher tokens
// (the exchange kernels fold those in a pass of their own, from a table in
// shared memory for the first kMCap of a CTA's range).  Returns 1 on a
// CUDA error.
int build_maps(const int32_t* token_map, int64_t vt, int64_t vs, char* ws, const ProjLayout& L,
               const XPlan* xp, bool multi, uint32_t* dev_status, cudaStream_t s) {
  int32_t* cnt = reinterpret_cast<int32_t*>(ws + L.cnt);
  int32_t* off = reinterpret_cast<int32_t*>(ws + L.off);
  int32_t* cols = reinterpret_cast<int32_t*>(ws + L.cols);
  int32_t* one = reinterpret_cast<int32_t*>(ws + L.one);
  int32_t* eid = reinterpret_cast<int32_t*>(ws + L.eid);
  int32_t* epos = reinterpret_cast<int32_t*>(ws + L.epos);
  int32_t* code = reinterpret_cast<int32_t*>(ws + L.code);
  int32_t* send_src = reinterpret_cast<int32_t*>(ws + L.send_src);
  int32_t* mflag = reinterpret_cast<int32_t*>(ws + L.mflag);
  int32_t* mpre = reinterpret_cast<int32_t*>(ws + L.mpre);
  int32_t* mlist = reinterpret_cast<int32_t*>(ws + L.mlist);
  int32_t* mcode = reinterpret_cast<int32_t*>(ws + L.mcode);
  int32_t* stmp = reinterpret_cast<int32_t*>(ws + L.stmp);
  XLayout* X = reinterpret_cast<XLayout*>(ws + L.xl);
  const int nsm = tc_num_sms() > 0 ? tc_num_sms() : 1;
  const int gmap = (int)std::min<int64_t>((vt + kT - 1) / kT, (int64_t)nsm * 8);
  const int gid = (int)std::min<int64_t>((vs + kT - 1) / kT, (int64_t)nsm * 8);
  if (cudaMemsetAsync(cnt, 0, (size_t)vs * 4, s) != cudaSuccess) return 1;
  note_launch();
  k_map_count<<<gmap, kT, 0, s>>>(token_map, vt, vs, cnt, dev_status);
  launch_scan(cnt, vs, off, stmp, s);
  if (cudaMemsetAsync(cnt, 0, (size_t)vs * 4, s) != cudaSuccess) return 1;
  note_launch();
  k_map_scatter<<<gmap, kT, 0, s>>>(token_map, vt, vs, off, cnt, cols);
  note_launch();
  k_map_sort<<<gid, kT, 0, s>>>(off, vs, cols);
  note_launch();
  k_map_single<<<gid, kT, 0, s>>>(off, cols, vs, one, eid);
  if (xp) {  // the exchange lists; X->fits then picks the path on the device
    if (cudaMemsetAsync(X, 0, sizeof(XLayout), s) != cudaSuccess ||
        cudaMemsetAsync(send_src, 0, ((size_t)vt + 8 * kMaxC * kMaxC) * 4, s) != cudaSuccess)
      return 1;
    note_launch();
    k_edge_count<<<gmap, kT, 0, s>>>(off, cols, eid, vs, (int32_t)xp->sc, (int32_t)xp->so, xp->C,
                                      X);
    note_launch();
    k_exchange_layout<<<1, 32, 0, s>>>(X, xp->C, (int32_t)xp->send_cap, (int32_t)xp->recv_cap);
    note_launch();
    k_edge_partition<<<xp->C * xp->C, 1024, 0, s>>>(off, cols, eid, vs, (int32_t)xp->sc,
                                                    (int32_t)xp->so, xp->C, X, send_src, epos);
    note_launch();
    k_exchange_codes<<<gid, kT, 0, s>>>(off, epos, vs, code);
    if (multi) {
      note_launch();
      k_multi_flag<<<gid, kT, 0, s>>>(code, vs, mflag);
      launch_scan(mflag, vs, mpre, stmp, s);
      note_launch();
      k_multi_scatter<<<gid, kT, 0, s>>>(code, mpre, vs, mlist, mcode);
    }
  }
  return cudaGetLastError() != cudaSuccess;
}

// the launches of one call, per dtype pair
struct ProjRun {
  const void* zt;
  int64_t n, vt, vs;
  float inv_t;
  const int32_t *off, *cols, *list_id, *list_val, *slice_off, *epos, *code, *mpre, *mlist, *mcode,
      *send_src;
  const XLayout* X;  // non-null when the exchange path may run
  int64_t sc;        // slice path: columns per slice
  int nsl;
  void* out;
  uint32_t* status;
  cudaStream_t s;
};
template <typename TI, typename TO>
struct ProjOps {
  static bool plan(int64_t vt, int64_t vs, XPlan* P) { return x_plan<TI, TO>(vt, vs, P); }
  static int run(const XPlan* xp, const ProjRun& a) {
    if (xp && launch_exchange<TI, TO>(*xp, a.zt, a.n, a.vt, a.vs, a.inv_t, a.off, a.epos, a.code,
                                      a.mpre, a.mlist, a.mcode, a.send_src, a.X, a.out,
                                      a.status, a.s))
      return 1;
    return launch_project<TI, TO>(a.zt, a.n, a.vt, a.vs, a.inv_t, a.off, a.cols, a.list_id,
                                  a.list_val, a.slice_off, a.sc, a.nsl, a.out, a.status, a.X,
                                  a.s);
  }
};


// Exchange plan of the fused kernel: as x_plan, with the fused kernel's own
// thread count (STEPS 8-id steps per thread cover a CTA's student ids).
template <typename TI>
bool pl_plan(int64_t vt, int64_t vs, XPlan* P, int* steps) {
  const int64_t elem = (int64_t)sizeof(TI);
  int64_t C = (vt * elem + kXWide.slice - 1) / kXWide.slice;
  if (C < 1) C = 1;
  if (C > kMaxC) return false;
  P->sc = ((vt + C - 1) / C + 7) / 8 * 8;
  C = (vt + P->sc - 1) / P->sc;
  P->C = (int)C;
  P->so = ((vs + C - 1) / C + 7) / 8 * 8;
  const int64_t st = (P->so + 8 * kLT - 1) / (8 * kLT);
  if (st > 8) return false;
  *steps = st <= 1 ? 1 : st <= 2 ? 2 : st <= 4 ? 4 : 8;
  P->send_cap = P->sc + 8 * C;
  P->recv_cap = (kPLSmem / elem - P->sc - P->send_cap) / 8 * 8;
  // receive slots and table codes share the 16-bit code space below 0xfffe
  if (P->recv_cap > 0xfffe - kMCap) P->recv_cap = (0xfffe - kMCap) / 8 * 8;
  if (P->recv_cap < 8) return false;
  P->smem = (size_t)(P->sc + P->send_cap + P->recv_cap) * (size_t)elem;
  return true;
}

template <typename TI, int MODE, bool SKEW, int STEPS>
int launch_pl(const XPlan& xp, const PLParams& P, cudaStream_t s) {
  auto kern = k_proj_loss<TI, MODE, SKEW, STEPS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)xp.smem) !=
      cudaSuccess)
    return 1;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)xp.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  const int nsm = tc_num_sms() > 0 ? tc_num_sms() : 1;
  cfg.gridDim = dim3((unsigned)(xp.C * std::max(1, nsm / xp.C)));
  cfg.blockDim = dim3(kLT);
  cfg.dynamicSmemBytes = xp.smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int maxc = max_active_clusters(reinterpret_cast<const void*>(kern), cfg);
  if (maxc <= 0) return 1;
  const int64_t clusters = P.n < maxc ? P.n : maxc;
  cfg.gridDim = dim3((unsigned)(xp.C * clusters));
  note_launch();
  return cudaLaunchKernelEx(&cfg, kern, P) != cudaSuccess;
}

template <typename TI, int MODE, bool SKEW>
int launch_pl_steps(const XPlan& xp, int steps, const PLParams& P, cudaStream_t s) {
  switch (steps) {
    case 1: return launch_pl<TI, MODE, SKEW, 1>(xp, P, s);
    case 2: return launch_pl<TI, MODE, SKEW, 2>(xp, P, s);
    case 4: return launch_pl<TI, MODE, SKEW, 4>(xp, P, s);
    default: return launch_pl<TI, MODE, SKEW, 8>(xp, P, s);
  }
}

template <typename TI>
int launch_pl_any(const XPlan& xp, int steps, const PLParams& P, int mode, cudaStream_t s) {
  if (mode == 1) return launch_pl_steps<TI, 1, false>(xp, steps, P, s);
  return is_skew(P.variant) ? launch_pl_steps<TI, 0, true>(xp, steps, P, s)
                            : launch_pl_steps<TI, 0, false>(xp, steps, P, s);
}

}  // namespace

size_t proj_loss_workspace_bytes(int64_t vt, int64_t vs) { return proj_layout(vt, vs).bytes; }

bool proj_loss_supported(int64_t vt, int64_t vs, bool bf16) {
  XPlan xp;
  int steps = 0;
  return bf16 ? pl_plan<__nv_bfloat16>(vt, vs, &xp, &steps) : pl_plan<float>(vt, vs, &xp, &steps);
}

int launch_proj_loss(const ProjLossArgs& a, void* workspace, cudaStream_t s) {
  XPlan xp;
  int steps = 0;
  const bool ok = a.is_bf16 ? pl_plan<__nv_bfloat16>(a.vt, a.vs, &xp, &steps)
                            : pl_plan<float>(a.vt, a.vs, &xp, &steps);
  if (!ok) return 1;
  const ProjLayout L = proj_layout(a.vt, a.vs);
  char* ws = static_cast<char*>(workspace);
  if (build_maps(a.token_map, a.vt, a.vs, ws, L, &xp, true, a.status, s)) return 1;
  if (a.n <= 0) return 0;
  PLParams P;
  memset(&P, 0, sizeof(P));
  P.zt = a.zt;
  P.zs = a.zs;
  P.n = a.n;
  P.vt = a.vt;
  P.vs = a.vs;
  P.inv_tp = a.inv_tp;
  P.c = a.c;
  P.variant = a.variant;
  P.labels = a.labels;
  P.ignore = a.ignore;
  P.ce_s = a.ce_s;
  P.ce_t = a.ce_t;
  P.kl = a.kl;
  P.stats = a.stats;
  P.row_scale = a.row_scale;
  P.w_sce = a.w_sce;
  P.w_kl_ts = a.w_kl_ts;
  P.dz = a.dz;
  P.off = reinterpret_cast<const int32_t*>(ws + L.off);
  P.epos = reinterpret_cast<const int32_t*>(ws + L.epos);
  P.code = reinterpret_cast<const int32_t*>(ws + L.code);
  P.send_src = reinterpret_cast<const int32_t*>(ws + L.send_src);
  P.mpre = reinterpret_cast<const int32_t*>(ws + L.mpre);
  P.mlist = reinterpret_cast<const int32_t*>(ws + L.mlist);
  P.mcode = reinterpret_cast<const int32_t*>(ws + L.mcode);
  P.X = reinterpret_cast<const XLayout*>(ws + L.xl);
  P.sc = xp.sc;
  P.so = xp.so;
  P.send_cap = xp.send_cap;
  P.recv_cap = xp.recv_cap;
  P.status = a.status;
  return a.is_bf16 ? launch_pl_any<__nv_bfloat16>(xp, steps, P, a.mode, s)
                   : launch_pl_any<float>(xp, steps, P, a.mode, s);
}

}  // namespace kd

using namespace kd;

extern "C" {

kd_status kd_project_workspace_size(int64_t v_teacher, int64_t v_student, size_t* bytes) {
  if (!bytes || v_teacher < 1 || v_student < 1 || v_teacher > ((int64_t)1 << 30) ||
      v_student > ((int64_t)1 << 30))
    return KD_ERR_INVALID_ARG;
  *bytes = proj_layout(v_teacher, v_student).bytes;
  return KD_OK;
}

kd_status kd_project_teacher_logits(const int32_t* token_map, int64_t v_teacher,
                                    int64_t v_student, const void* logits_t, int64_t n_tokens,
                                    int32_t in_dtype, float temperature, void* out,
                                    int32_t out_dtype, uint32_t* dev_status, void* workspace,
                                    size_t ws_bytes, void* stream) {
  size_t need = 0;
  if (kd_project_workspace_size(v_teacher, v_student, &need) != KD_OK || n_tokens < 0 ||
      !token_map || (n_tokens > 0 && (!logits_t || !out)) ||
      (in_dtype != KD_BF16 && in_dtype != KD_FP32) ||
      (out_dtype != KD_BF16 && out_dtype != KD_FP32) ||
      !(temperature > 0.f && temperature < FLT_MAX))
    return KD_ERR_INVALID_ARG;
  int64_t sc = 0;
  const int nsl = slices_for(v_teacher, in_dtype == KD_BF16 ? 2 : 4, &sc);
  if (nsl == 0) return KD_ERR_UNSUPPORTED;  // a teacher row above 96 MiB
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KD_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || !kd_device_supported(dev)) return KD_ERR_NO_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const ProjLayout L = proj_layout(v_teacher, v_student);
  char* ws = static_cast<char*>(workspace);
  int32_t* off = reinterpret_cast<int32_t*>(ws + L.off);
  int32_t* cols = reinterpret_cast<int32_t*>(ws + L.cols);
  int32_t* one = reinterpret_cast<int32_t*>(ws + L.one);
  int32_t* list_id = reinterpret_cast<int32_t*>(ws + L.list_id);
  int32_t* list_val = reinterpret_cast<int32_t*>(ws + L.list_val);
  int32_t* slice_cnt = reinterpret_cast<int32_t*>(ws + L.slice_cnt);
  int32_t* slice_off = reinterpret_cast<int32_t*>(ws + L.slice_off);
  int32_t* epos = reinterpret_cast<int32_t*>(ws + L.epos);
  int32_t* code = reinterpret_cast<int32_t*>(ws + L.code);
  int32_t* send_src = reinterpret_cast<int32_t*>(ws + L.send_src);
  int32_t* mpre = reinterpret_cast<int32_t*>(ws + L.mpre);
  int32_t* mlist = reinterpret_cast<int32_t*>(ws + L.mlist);
  int32_t* mcode = reinterpret_cast<int32_t*>(ws + L.mcode);
  XLayout* X = reinterpret_cast<XLayout*>(ws + L.xl);
  bool (*plan)(int64_t, int64_t, XPlan*);
  int (*run)(const XPlan*, const ProjRun&);
  if (in_dtype == KD_BF16) {
    plan = out_dtype == KD_BF16 ? ProjOps<__nv_bfloat16, __nv_bfloat16>::plan
                                : ProjOps<__nv_bfloat16, float>::plan;
    run = out_dtype == KD_BF16 ? ProjOps<__nv_bfloat16, __nv_bfloat16>::run
                               : ProjOps<__nv_bfloat16, float>::run;
  } else {
    plan = out_dtype == KD_BF16 ? ProjOps<float, __nv_bfloat16>::plan : ProjOps<float, float>::plan;
    run = out_dtype == KD_BF16 ? ProjOps<float, __nv_bfloat16>::run : ProjOps<float, float>::run;
  }
  XPlan xp;
  const bool xok = plan(v_teacher, v_student, &xp);
  if (cudaMemsetAsync(slice_cnt, 0, (size_t)nsl * 4, s) != cudaSuccess) return KD_ERR_CUDA;
  if (build_maps(token_map, v_teacher, v_student, ws, L, xok ? &xp : nullptr, true, dev_status,
                 s))
    return KD_ERR_CUDA;
  const int nsm = tc_num_sms() > 0 ? tc_num_sms() : 1;
  const int gid = (int)std::min<int64_t>((v_student + kT - 1) / kT, (int64_t)nsm * 8);
  const XLayout* Xp = xok ? X : nullptr;
  note_launch();
  k_slice_count<<<gid, kT, 0, s>>>(one, off, cols, v_student, (int32_t)sc, nsl, slice_cnt, Xp);
  note_launch();
  k_slice_partition<<<nsl, 1024, 0, s>>>(one, off, cols, v_student, (int32_t)sc, nsl, slice_cnt,
                                         slice_off, list_id, list_val, Xp);
  if (n_tokens > 0) {
    ProjRun a{logits_t, n_tokens, v_teacher, v_student, 1.f / temperature, off, cols, list_id,
              list_val, slice_off, epos, code, mpre, mlist, mcode, send_src, Xp, sc, nsl, out,
              dev_status, s};
    if (run(xok ? &xp : nullptr, a)) return KD_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

}  // extern "C"
