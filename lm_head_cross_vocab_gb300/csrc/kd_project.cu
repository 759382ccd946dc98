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
// The inverse map is built on the device in the caller's workspace on every
// call (count -> exclusive scan -> scatter -> per-id sort, so the summation
// order and the result are deterministic, plus a per-id column for the common
// case of exactly one teacher token); then one CTA per SM takes token rows in
// turn, stages each in shared memory and takes, for every student id, the
// log-sum-exp over the teacher columns of its id.
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

// one[i] for student id i: -1 when no teacher token maps to it, -2 when
// several do, and when exactly one does, its teacher column c -- or, for the
// cluster kernel (sc > 0), where that column is staged: the CTA c / sc of the
// cluster in bits 17.. and the element c % sc in bits 0..16.
constexpr int kEncBits = 17;
__global__ void k_map_single(const int32_t* __restrict__ off, const int32_t* __restrict__ cols,
                             int64_t vs, int32_t sc, int32_t* __restrict__ one) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vs;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t b = off[i], e = off[i + 1];
    int32_t v = e == b ? -1 : -2;
    if (e - b == 1) {
      v = cols[b];
      if (sc > 0) v = (v / sc) << kEncBits | (v % sc);
    }
    one[i] = v;
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

// One CTA per SM, one token row at a time.  The teacher row is staged in
// shared memory in slices of at most kSlice bytes (one slice when it fits, two
// for a 152k bf16 vocabulary), with coalesced 16-byte loads; every student id
// then folds the teacher tokens of its segment that fall in the slice into a
// running log-sum-exp (logaddexp; a single token gives z / T exactly).
// Between slices the running values live in a per-CTA fp32 scratch row (it
// stays in L2); the last slice writes the output row with vector stores.  So
// the random gathers hit shared memory and all global traffic is coalesced.
constexpr int kPT = 1024;               // threads per projection CTA
constexpr int kIds = 8;                 // student ids per thread per step
constexpr int64_t kSlice = 200 * 1024;  // bytes of a staged teacher-row slice

__host__ __device__ __forceinline__ int64_t scratch_pitch(int64_t vs) { return (vs + 7) / 8 * 8; }

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

template <typename TI, typename TO>
__global__ void __launch_bounds__(kPT, 1) k_project(const TI* __restrict__ zt, int64_t n,
                                                    int64_t vt, int64_t vs, float inv_t,
                                                    const int32_t* __restrict__ off,
                                                    const int32_t* __restrict__ cols,
                                                    const int32_t* __restrict__ one,
                                                    TO* __restrict__ out,
                                                    float* __restrict__ scratch, int64_t span) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TI* zsm = reinterpret_cast<TI*>(smem_raw);
  // scratch rows have a pitch of vs rounded up to 8 floats, so every row and
  // every 8-id group in it is 16-byte aligned for the float4 accesses below
  float* part = scratch ? scratch + (int64_t)blockIdx.x * scratch_pitch(vs) : nullptr;
  const int passes = (int)((vt + span - 1) / span);
  constexpr int EV = 16 / (int)sizeof(TI);  // elements per 16-byte vector
  for (int64_t row = blockIdx.x; row < n; row += gridDim.x) {
    const TI* z = zt + row * vt;
    TO* o = out + row * vs;
    for (int p = 0; p < passes; ++p) {
      const int64_t lo = (int64_t)p * span, hi = lo + span < vt ? lo + span : vt;
      const int64_t len = hi - lo;
      __syncthreads();  // the previous slice is no longer read
      if ((reinterpret_cast<uintptr_t>(z + lo) & 15) == 0) {
        const int64_t nvec = len / EV;
        for (int64_t q = threadIdx.x; q < nvec; q += kPT)
          reinterpret_cast<uint4*>(zsm)[q] = reinterpret_cast<const uint4*>(z + lo)[q];
        for (int64_t q = nvec * EV + threadIdx.x; q < len; q += kPT) zsm[q] = z[lo + q];
      } else {
        for (int64_t q = threadIdx.x; q < len; q += kPT) zsm[q] = z[lo + q];
      }
      __syncthreads();
      const bool last = p + 1 == passes;
      for (int64_t i0 = (int64_t)threadIdx.x * kIds; i0 < vs; i0 += (int64_t)kPT * kIds) {
        const bool full = i0 + kIds <= vs;
        // one coalesced load classifies the 8 ids; only ids with several
        // teacher tokens read their segment bounds
        int32_t oc[kIds];
        if (full) {
          const int4 a = reinterpret_cast<const int4*>(one + i0)[0];
          const int4 b = reinterpret_cast<const int4*>(one + i0)[1];
          oc[0] = a.x; oc[1] = a.y; oc[2] = a.z; oc[3] = a.w;
          oc[4] = b.x; oc[5] = b.y; oc[6] = b.z; oc[7] = b.w;
        } else {
#pragma unroll
          for (int k = 0; k < kIds; ++k) oc[k] = i0 + k < vs ? one[i0 + k] : -1;
        }
        float r[kIds];
        if (p == 0) {
#pragma unroll
          for (int k = 0; k < kIds; ++k) r[k] = -INFINITY;
        } else if (full) {
          const float4 a = reinterpret_cast<const float4*>(part + i0)[0];
          const float4 b = reinterpret_cast<const float4*>(part + i0)[1];
          r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
          r[4] = b.x; r[5] = b.y; r[6] = b.z; r[7] = b.w;
        } else {
#pragma unroll
          for (int k = 0; k < kIds; ++k) r[k] = i0 + k < vs ? part[i0 + k] : -INFINITY;
        }
#pragma unroll
        for (int k = 0; k < kIds; ++k) {
          const int64_t c = oc[k];
          if (c >= lo && c < hi) {  // the id's only teacher token lies in this slice
            r[k] = logaddexp(r[k], ld<TI>(zsm + (c - lo)) * inv_t);
          } else if (c == -2) {
            const int32_t e = off[i0 + k + 1];
#pragma unroll 1
            for (int32_t t = off[i0 + k]; t < e; ++t) {
              const int64_t ct = cols[t];
              if (ct >= lo && ct < hi) r[k] = logaddexp(r[k], ld<TI>(zsm + (ct - lo)) * inv_t);
            }
          }
        }
        if (last) {
#pragma unroll
          for (int k = 0; k < kIds; ++k)
            if (r[k] == -INFINITY) r[k] = lowest<TO>();
          if (full && (reinterpret_cast<uintptr_t>(o + i0) & 15) == 0) {
            store_vec(o + i0, r);
          } else {
#pragma unroll
            for (int k = 0; k < kIds; ++k)
              if (i0 + k < vs) st<TO>(o + i0 + k, r[k]);
          }
        } else if (full) {
          store_vec(part + i0, r);
        } else {
#pragma unroll
          for (int k = 0; k < kIds; ++k)
            if (i0 + k < vs) part[i0 + k] = r[k];
        }
      }
    }
  }
}

// Cluster projection.  A cluster of C CTAs (C = 1, 2, 4 or 8, one CTA per SM)
// works on one token row at a time: CTA r holds teacher columns
// [r*sc, r*sc + sc) of the row in its shared memory, brought in by one bulk
// copy (double-buffered, so the copy of the cluster's next row runs under the
// gathers of this one), and writes student ids [r*so, r*so + so) of the output
// row.  Each id's teacher column is read from whichever CTA of the cluster
// holds it (distributed shared memory), so the row is read from HBM once, the
// output written once with vector stores, and no partial results are kept.
constexpr int64_t kBuf = 104 * 1024;  // bytes of one staged slice (two per CTA)
constexpr int kGroups = 1;  // groups of 8 ids per thread whose gathers are in flight together

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster; release / acquire at cluster scope
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// element `e` of the staged-row buffer at shared-memory offset `base` of
// CTA `r` of the cluster.  (Plain loads, free to be batched by the compiler:
// the buffers do not change between the cluster barriers that bracket them.)
template <typename TI>
__device__ __forceinline__ float dsmem_get(uint32_t base, uint32_t r, uint32_t e) {
  uint32_t a = base + e * (uint32_t)sizeof(TI);
  asm("mapa.shared::cluster.u32 %0, %0, %1;" : "+r"(a) : "r"(r));
  if constexpr (sizeof(TI) == 2) {
    uint16_t v;
    asm("ld.shared::cluster.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return __bfloat162float(__ushort_as_bfloat16(v));
  } else {
    float v;
    asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
  }
}
// teacher value at column c of the staged row
template <typename TI>
__device__ __forceinline__ float dsmem_col(uint32_t base, uint32_t c, uint32_t sc) {
  const uint32_t r = c / sc;
  return dsmem_get<TI>(base, r, c - r * sc);
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(kPT, 1)
    k_project_cluster(const TI* __restrict__ zt, int64_t n, int64_t vt, int64_t vs, float inv_t,
                      const int32_t* __restrict__ off, const int32_t* __restrict__ cols,
                      const int32_t* __restrict__ one, TO* __restrict__ out, int64_t sc,
                      int64_t so, uint32_t* status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const uint32_t rank = cluster_rank(), csize = cluster_size();
  const int64_t ncl = gridDim.x / csize;
  const int64_t c0 = (int64_t)rank * sc;
  const int64_t clen = vt - c0 < sc ? (vt - c0 > 0 ? vt - c0 : 0) : sc;  // my columns
  const int64_t i_lo = (int64_t)rank * so, i_hi = i_lo + so < vs ? i_lo + so : vs;
  const uint32_t buf_sa = ptx::smem_u32(smem_raw);
  const uint32_t buf_bytes = (uint32_t)(sc * (int64_t)sizeof(TI));
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars[1]), 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  // stage my columns of `row` into buffer b: the 16-byte-aligned bulk by one
  // bulk copy, a ragged tail (or a whole unaligned row) by plain loads
  auto stage = [&](int64_t row, int b) {
    const TI* src = zt + row * vt + c0;
    TI* dst = reinterpret_cast<TI*>(smem_raw + (size_t)b * buf_bytes);
    const bool al = ((reinterpret_cast<uintptr_t>(src) | ptx::smem_u32(dst)) & 15) == 0;
    const int64_t nb = al ? clen * (int64_t)sizeof(TI) / 16 * 16 : 0;
    if (threadIdx.x == 0 && !*reinterpret_cast<volatile int*>(&abort_flag)) {
      // (after a timed-out wait no new copy starts; later waits give up)
      const uint32_t bar = ptx::smem_u32(&bars[b]);
      ptx::mbar_expect_tx(bar, (uint32_t)nb);
      if (nb > 0) {
        fence_proxy_async();
        ptx::bulk_load(ptx::smem_u32(dst), src, (uint32_t)nb, bar);
      }
    }
    for (int64_t q = nb / (int64_t)sizeof(TI) + threadIdx.x; q < clen; q += kPT) dst[q] = src[q];
  };
  const int64_t first = blockIdx.x / csize;
  if (first < n) stage(first, 0);
  uint32_t parity = 0;  // bit b: phase parity to wait for on buffer b
  // the first wait that gave up: its copy may still be in flight (none starts
  // after it, the abort flag being set by then)
  int pend_b = -1;
  uint32_t pend_p = 0;
  int k = 0;
  for (int64_t row = first; row < n; row += ncl, ++k) {
    const int b = k & 1;
    if (!ptx::warp_wait(ptx::smem_u32(&bars[b]), (parity >> b) & 1u, &abort_flag, status) &&
        pend_b < 0) {
      pend_b = b;
      pend_p = (parity >> b) & 1u;
    }
    parity ^= 1u << b;
    // every CTA's slice of this row has landed, and every CTA is done with
    // the row before it, whose buffer the next copy reuses
    cluster_sync();
    if (row + ncl < n) stage(row + ncl, b ^ 1);
    const uint32_t base = buf_sa + (uint32_t)b * buf_bytes;
    TO* o = out + row * vs;
    for (int64_t g0 = i_lo + (int64_t)threadIdx.x * kIds; g0 < i_hi; g0 += (int64_t)kPT * kIds * kGroups) {
      // the entries of up to kGroups groups of 8 ids, loaded together
      int32_t oc[kGroups][kIds];
#pragma unroll
      for (int j = 0; j < kGroups; ++j) {
        const int64_t i0 = g0 + (int64_t)j * kPT * kIds;
        if (i0 + kIds <= i_hi) {  // one is 256-byte aligned, i0 - i_lo a multiple of 8
          const int4 a = reinterpret_cast<const int4*>(one + i0)[0];
          const int4 c = reinterpret_cast<const int4*>(one + i0)[1];
          oc[j][0] = a.x; oc[j][1] = a.y; oc[j][2] = a.z; oc[j][3] = a.w;
          oc[j][4] = c.x; oc[j][5] = c.y; oc[j][6] = c.z; oc[j][7] = c.w;
        } else {
#pragma unroll
          for (int q = 0; q < kIds; ++q) oc[j][q] = i0 + q < i_hi ? one[i0 + q] : -1;
        }
      }
      // all single-token gathers of the groups first (each entry's
      // register then holds its value), then the rest; bit 8j+q of `multi` /
      // `none` marks an id with several / no teacher tokens
      float v[kGroups][kIds];
      uint32_t multi = 0, none = 0;
#pragma unroll
      for (int j = 0; j < kGroups; ++j)
#pragma unroll
        for (int q = 0; q < kIds; ++q) {
          const int32_t c = oc[j][q];
          multi |= (c == -2 ? 1u : 0u) << (8 * j + q);
          none |= (c == -1 ? 1u : 0u) << (8 * j + q);
          v[j][q] = c >= 0 ? dsmem_get<TI>(base, (uint32_t)c >> kEncBits,
                                           (uint32_t)c & ((1u << kEncBits) - 1))
                           : 0.f;
        }
#pragma unroll
      for (int j = 0; j < kGroups; ++j) {
        const int64_t i0 = g0 + (int64_t)j * kPT * kIds;
        if (i0 >= i_hi) break;
        float r[kIds];
#pragma unroll
        for (int q = 0; q < kIds; ++q) {
          if (!((multi | none) >> (8 * j + q) & 1u)) {
            r[q] = v[j][q] * inv_t;
          } else if (multi >> (8 * j + q) & 1u) {  // several teacher tokens: fold in column order
            const int32_t e = off[i0 + q + 1];
            float acc = -INFINITY;
#pragma unroll 1
            for (int32_t t = off[i0 + q]; t < e; ++t)
              acc = logaddexp(acc, dsmem_col<TI>(base, (uint32_t)cols[t], (uint32_t)sc) * inv_t);
            r[q] = acc;
          } else {
            r[q] = -INFINITY;
          }
          if (r[q] == -INFINITY) r[q] = lowest<TO>();
        }
        if (i0 + kIds <= i_hi && (reinterpret_cast<uintptr_t>(o + i0) & 15) == 0) {
          store_vec(o + i0, r);
        } else {
#pragma unroll
          for (int q = 0; q < kIds; ++q)
            if (i0 + q < i_hi) st<TO>(o + i0 + q, r[q]);
        }
      }
    }
  }
  // no CTA leaves while another may still read its shared memory, nor with
  // a copy of its own still in flight (bounded again, whatever the abort flag)
  cluster_sync();
  if (pend_b >= 0 && threadIdx.x < 32)
    ptx::warp_wait(ptx::smem_u32(&bars[pend_b]), pend_p, &abort_flag, status, false);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// teacher columns per staged slice (a multiple of 8, so every slice of an
// aligned row starts 16-byte aligned)
template <typename TI>
int64_t slice_cols() {
  return kSlice / (int64_t)sizeof(TI) / 8 * 8;
}

// smallest cluster (1, 2, 4, 8 CTAs) whose per-CTA share of a teacher row,
// sc columns (a multiple of 8), fits one staging buffer; 0 when eight CTAs
// cannot hold the row (the sliced kernel takes it then)
int cluster_for(int64_t vt, int64_t elem, int64_t* sc) {
  for (int c = 1; c <= 8; c *= 2) {
    const int64_t cols = ((vt + c - 1) / c + 7) / 8 * 8;
    if (cols * elem <= kBuf) {
      if (sc) *sc = cols;
      return c;
    }
  }
  return 0;
}

struct ProjLayout {
  size_t cnt, off, cols, one, scratch, bytes;
};
// inverse map, plus one fp32 scratch row per CTA when the sliced kernel may
// take the row in more than one slice (sized for fp32 logits, the larger
// element, which needs a cluster soonest)
ProjLayout proj_layout(int64_t vt, int64_t vs, int ctas) {
  ProjLayout L;
  L.cnt = 0;
  L.off = align256(L.cnt + (size_t)vs * 4);
  L.cols = align256(L.off + (size_t)(vs + 1) * 4);
  L.one = align256(L.cols + (size_t)vt * 4);
  L.scratch = align256(L.one + (size_t)vs * 4);
  const bool multi = cluster_for(vt, 4, nullptr) == 0 && vt > slice_cols<float>();
  L.bytes = align256(L.scratch + (multi ? (size_t)ctas * (size_t)scratch_pitch(vs) * 4 : 0));
  return L;
}

int proj_ctas() { return tc_num_sms() > 0 ? tc_num_sms() : 1; }

// Launch shape of the cluster kernel: cluster size, columns and student ids
// per CTA, staging bytes, co-resident clusters.
struct ClusterPlan {
  int c = 0;
  int64_t sc = 0, so = 0;
  size_t smem = 0;
  int max_clusters = 0;
};

template <typename TI, typename TO>
cudaLaunchConfig_t cluster_config(const ClusterPlan& P, cudaLaunchAttribute* attr,
                                  cudaStream_t s) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P.c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kPT);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// true when a cluster of at most 8 CTAs can hold a teacher row and such
// clusters can be resident (the cluster kernel takes the rows); false leaves
// them to the sliced kernel.  *err is set on a CUDA error.
template <typename TI, typename TO>
bool cluster_plan(int64_t vt, int64_t vs, ClusterPlan* P, bool* err) {
  *err = false;
  P->c = cluster_for(vt, (int64_t)sizeof(TI), &P->sc);
  if (P->c == 0) return false;
  P->so = ((vs + P->c - 1) / P->c + 7) / 8 * 8;
  P->smem = 2 * (size_t)P->sc * sizeof(TI);
  auto kern = k_project_cluster<TI, TO>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P->smem) !=
      cudaSuccess) {
    *err = true;
    return false;
  }
  // co-resident clusters of this shape (cached per cluster size and buffer)
  static int cached_c = 0, cached_max = 0;
  static size_t cached_smem = 0;
  if (cached_c != P->c || cached_smem != P->smem) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config<TI, TO>(*P, attr, nullptr);
    const int nsm = proj_ctas();
    cfg.gridDim = dim3((unsigned)(P->c * (nsm / P->c > 0 ? nsm / P->c : 1)));
    int m = 0;
    if (cudaOccupancyMaxActiveClusters(&m, kern, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      m = 0;
    }
    cached_c = P->c;
    cached_smem = P->smem;
    cached_max = m;
  }
  P->max_clusters = cached_max;
  return cached_max > 0;
}

template <typename TI, typename TO>
int launch_cluster(const ClusterPlan& P, const void* zt, int64_t n, int64_t vt, int64_t vs,
                   float inv_t, const int32_t* off, const int32_t* cols, const int32_t* one,
                   void* out, uint32_t* status, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config<TI, TO>(P, attr, s);
  const int64_t clusters = n < P.max_clusters ? n : P.max_clusters;
  cfg.gridDim = dim3((unsigned)(P.c * clusters));
  note_launch();
  return cudaLaunchKernelEx(&cfg, k_project_cluster<TI, TO>, static_cast<const TI*>(zt), n, vt,
                            vs, inv_t, off, cols, one, static_cast<TO*>(out), P.sc, P.so,
                            status) != cudaSuccess;
}

template <typename TI, typename TO>
int launch_sliced(const void* zt, int64_t n, int64_t vt, int64_t vs, float inv_t,
                  const int32_t* off, const int32_t* cols, const int32_t* one, void* out,
                  float* scratch, int grid, cudaStream_t s) {
  const int64_t span = slice_cols<TI>();
  const size_t smem = (size_t)(vt < span ? vt : span) * sizeof(TI);
  auto kern = k_project<TI, TO>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return 1;
  note_launch();
  kern<<<grid, kPT, smem, s>>>(static_cast<const TI*>(zt), n, vt, vs, inv_t, off, cols, one,
                               static_cast<TO*>(out), vt > span ? scratch : nullptr, span);
  return 0;
}

// Map the build-time plan and the projection itself onto one dtype pair.
struct ProjArgs {
  const void* zt;
  int64_t n, vt, vs;
  float inv_t;
  const int32_t *off, *cols, *one;
  void* out;
  float* scratch;
  uint32_t* status;
  cudaStream_t s;
};
template <typename TI, typename TO>
struct ProjOps {
  static bool plan(const ProjArgs& A, ClusterPlan* P, bool* err) {
    return cluster_plan<TI, TO>(A.vt, A.vs, P, err);
  }
  static int run(const ProjArgs& A, const ClusterPlan* P) {
    if (P)
      return launch_cluster<TI, TO>(*P, A.zt, A.n, A.vt, A.vs, A.inv_t, A.off, A.cols, A.one,
                                    A.out, A.status, A.s);
    const int grid = (int)std::min<int64_t>(A.n, (int64_t)proj_ctas());
    return launch_sliced<TI, TO>(A.zt, A.n, A.vt, A.vs, A.inv_t, A.off, A.cols, A.one, A.out,
                                 A.scratch, grid, A.s);
  }
};

}  // namespace
}  // namespace kd

using namespace kd;

extern "C" {

kd_status kd_project_workspace_size(int64_t v_teacher, int64_t v_student, size_t* bytes) {
  if (!bytes || v_teacher < 1 || v_student < 1 || v_teacher > ((int64_t)1 << 30) ||
      v_student > ((int64_t)1 << 30))
    return KD_ERR_INVALID_ARG;
  *bytes = proj_layout(v_teacher, v_student, proj_ctas()).bytes;
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
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KD_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || !kd_device_supported(dev)) return KD_ERR_NO_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const ProjLayout L = proj_layout(v_teacher, v_student, proj_ctas());
  char* ws = static_cast<char*>(workspace);
  int32_t* cnt = reinterpret_cast<int32_t*>(ws + L.cnt);
  int32_t* off = reinterpret_cast<int32_t*>(ws + L.off);
  int32_t* cols = reinterpret_cast<int32_t*>(ws + L.cols);
  int32_t* one = reinterpret_cast<int32_t*>(ws + L.one);
  float* scratch = reinterpret_cast<float*>(ws + L.scratch);
  const int nsm = tc_num_sms() > 0 ? tc_num_sms() : 1;
  const int gmap = (int)std::min<int64_t>((v_teacher + kT - 1) / kT, (int64_t)nsm * 8);
  const int gid = (int)std::min<int64_t>((v_student + kT - 1) / kT, (int64_t)nsm * 8);
  ProjArgs A{logits_t, n_tokens, v_teacher, v_student, 1.f / temperature, off, cols, one,
             out, scratch, dev_status, s};
  bool (*plan)(const ProjArgs&, ClusterPlan*, bool*);
  int (*run)(const ProjArgs&, const ClusterPlan*);
  if (in_dtype == KD_BF16) {
    plan = out_dtype == KD_BF16 ? ProjOps<__nv_bfloat16, __nv_bfloat16>::plan
                                : ProjOps<__nv_bfloat16, float>::plan;
    run = out_dtype == KD_BF16 ? ProjOps<__nv_bfloat16, __nv_bfloat16>::run
                               : ProjOps<__nv_bfloat16, float>::run;
  } else {
    plan = out_dtype == KD_BF16 ? ProjOps<float, __nv_bfloat16>::plan : ProjOps<float, float>::plan;
    run = out_dtype == KD_BF16 ? ProjOps<float, __nv_bfloat16>::run : ProjOps<float, float>::run;
  }
  ClusterPlan P;
  bool err = false;
  const bool clustered = n_tokens > 0 && plan(A, &P, &err);
  if (err) return KD_ERR_CUDA;
  if (cudaMemsetAsync(cnt, 0, (size_t)v_student * 4, s) != cudaSuccess) return KD_ERR_CUDA;
  note_launch();
  k_map_count<<<gmap, kT, 0, s>>>(token_map, v_teacher, v_student, cnt, dev_status);
  note_launch();
  k_map_scan<<<1, 1024, 0, s>>>(cnt, v_student, off);
  if (cudaMemsetAsync(cnt, 0, (size_t)v_student * 4, s) != cudaSuccess) return KD_ERR_CUDA;
  note_launch();
  k_map_scatter<<<gmap, kT, 0, s>>>(token_map, v_teacher, v_student, off, cnt, cols);
  note_launch();
  k_map_sort<<<gid, kT, 0, s>>>(off, v_student, cols);
  note_launch();
  k_map_single<<<gid, kT, 0, s>>>(off, cols, v_student, clustered ? (int32_t)P.sc : 0, one);
  if (n_tokens > 0 && run(A, clustered ? &P : nullptr)) return KD_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

}  // extern "C"
