// Small CUDA-core kernels around the fused loss: label validation and count,
// top-K preparation, the split-vocabulary combine + per-token finalisation,
// the scalar loss reduction, per-row gradient scales and a bf16 transpose.
#include <cuda_bf16.h>

#include "kd_internal.h"

namespace kd {

// ---------------------------------------------------------------- labels
// orda-kernel README, "Parameters": ignore_index is excluded from CE/KL and
// never used as a memory index; other out-of-range labels are errors.
__global__ void k_label_check(const int64_t* __restrict__ labels, int64_t n, int64_t vocab,
                              int64_t ignore, int32_t* count, uint32_t* status) {
  int local = 0;
  bool bad = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t y = labels[i];
    if (y != ignore) {
      ++local;
      if (y < 0 || y >= vocab) bad = true;
    }
  }
  for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
  if ((threadIdx.x & 31) == 0 && local) atomicAdd(count, local);
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_status(status, KD_DEV_BAD_LABEL);
}

void launch_label_check(const int64_t* labels, int64_t n, int64_t vocab, int64_t ignore,
                        int32_t* count, uint32_t* status, cudaStream_t s) {
  if (n <= 0) return;
  int blocks = (int)((n + 1023) / 1024);
  if (blocks > 256) blocks = 256;
  note_launch();
  k_label_check<<<blocks, 1024, 0, s>>>(labels, n, vocab, ignore, count, status);
}

// ---------------------------------------------------------------- top-K
// Rank sort of one row's K ids (K <= 1024) in shared memory.  Repeated or
// out-of-range ids flag KD_DEV_BAD_TOPK and are replaced by INT32_MAX, which
// no kernel ever matches or dereferences (the row's result is then invalid,
// as the status word reports).
__global__ void k_topk_prep(const int32_t* __restrict__ idx, const float* __restrict__ p,
                            int k, int64_t vocab, int32_t* __restrict__ sidx,
                            float* __restrict__ sp, float* __restrict__ mass,
                            float* __restrict__ ent, uint32_t* status) {
  extern __shared__ int32_t sh[];
  const int64_t row = blockIdx.x;
  const int32_t* ri = idx + row * k;
  const float* rp = p + row * k;
  for (int j = threadIdx.x; j < k; j += blockDim.x) sh[j] = ri[j];
  __syncthreads();
  float m = 0.f, e = 0.f;
  bool bad = false;
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    int32_t id = sh[j];
    const float pj = rp[j];
    int rank = 0;
    bool dup = false;
    for (int i = 0; i < k; ++i) {
      const int32_t o = sh[i];
      rank += (o < id) || (o == id && i < j);
      dup |= (o == id && i != j);
    }
    const bool oob = id < 0 || (int64_t)id >= vocab;
    if (dup || oob) {
      bad = true;
      id = INT32_MAX;
    }
    sidx[row * k + rank] = id;
    sp[row * k + rank] = pj;
    m += pj;
    if (pj > 0.f) e += pj * logf(pj);
  }
  __shared__ float red[2][32];
  for (int o = 16; o > 0; o >>= 1) {
    m += __shfl_xor_sync(0xffffffffu, m, o);
    e += __shfl_xor_sync(0xffffffffu, e, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    red[0][w] = m;
    red[1][w] = e;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(status, KD_DEV_BAD_TOPK);
  if (threadIdx.x == 0) {
    float mm = 0.f, ee = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
      mm += red[0][i];
      ee += red[1][i];
    }
    mass[row] = mm;
    ent[row] = ee;
  }
}

void launch_topk_prep(const int32_t* idx, const float* p, int64_t n, int k, int64_t vocab,
                      int32_t* sidx, float* sp, float* mass, float* ent, uint32_t* status,
                      cudaStream_t s) {
  if (n <= 0) return;
  int threads = k <= 128 ? 128 : (k <= 256 ? 256 : 512);
  note_launch();
  k_topk_prep<<<(unsigned)n, threads, k * sizeof(int32_t), s>>>(idx, p, k, vocab, sidx, sp,
                                                                 mass, ent, status);
}

// ---------------------------------------------------------------- combine
__global__ void k_combine(CombineArgs a) {
  // one warp per row: lane i folds parts i, i + 32, ..., then the warp merges
  // its lanes (a fixed tree, so the result does not depend on timing)
  const int64_t r = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= a.n) return;  // (r is the same in the whole warp)
  RowState st;
  st.init();
  for (int i = lane; i < a.n_parts; i += 32) {
    RowState o;
    o.load(a.partials + ((int64_t)i * a.n + r) * kRec);
    merge(st, o, a.c);
  }
  warp_merge(st, a.c);
  if (lane != 0) return;
  bool valid = true, bad = false;
  if (a.labels) {
    const int64_t y = a.labels[r];
    valid = y != a.ignore;
    bad = valid && (y < 0 || y >= a.vocab);
  }
  float* srow = a.stats + r * KD_STATS_PER_TOKEN;
  if (a.js_pass) {
    // skew variants: the first pass already wrote the log-normalisers
    const float kl = skew_kl(a.variant, a.c.beta, st.jq, st.jp);
    srow[S_KL_PM] = st.jp;
    if (a.variant != KD_KL_SKEW_JS) srow[S_EPPM] = st.jx;
    if (a.kl) a.kl[r] = valid ? kl : 0.f;
    return;
  }
  const float mass = a.topk ? a.mass[r] : 0.f;
  const float ent = a.topk ? a.ent[r] : 0.f;
  const RowOut o = finalize(st, a.c, a.variant, a.has_t, a.topk, mass, ent);
  const float nan = __int_as_float(0x7fc00000);
  if (a.ce_s) a.ce_s[r] = !valid ? 0.f : (bad ? nan : o.ce_s);
  if (a.ce_t) a.ce_t[r] = !valid ? 0.f : (bad ? nan : o.ce_t);
  if (a.kl) a.kl[r] = valid ? o.kl : 0.f;
  float4* s4 = reinterpret_cast<float4*>(srow);
  s4[0] = make_float4(o.lse_s1, o.lse_sT, o.lse_t1, o.lse_tT);
  s4[1] = make_float4(o.kl_rev, o.kl_pm, mass, o.dlse);
}

void launch_combine(const CombineArgs& a, cudaStream_t s) {
  if (a.n <= 0) return;
  note_launch();
  k_combine<<<(unsigned)((a.n + 7) / 8), 256, 0, s>>>(a);  // 8 rows (warps) a block
}

// ---------------------------------------------------------------- loss
// loss = sum_valid(w_sce CE_s + w_tce CE_t + w_kl T_s^2 KL) / denom, with
// denom = N_valid (mean), num_batch_labels (override) or 1 (sum).  One block,
// fixed summation order (deterministic).
__global__ void k_loss_reduce(ReduceArgs a) {
  double acc = 0.0;
  for (int64_t r = threadIdx.x; r < a.n; r += blockDim.x) {
    if (a.labels && a.labels[r] == a.ignore) continue;
    float v = 0.f;
    if (a.w_sce != 0.f) v += a.w_sce * a.ce_s[r];
    if (a.w_tce != 0.f) v += a.w_tce * a.ce_t[r];
    if (a.w_kl_t2 != 0.f) v += a.w_kl_t2 * a.kl[r];
    acc += (double)v;
  }
  __shared__ double red[32];
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
    double denom = 1.0;
    if (a.reduction == KD_REDUCE_MEAN) {
      if (a.num_batch_labels > 0) denom = (double)a.num_batch_labels;
      else {
        const int64_t c = a.labels ? (int64_t)*a.count : a.n;
        denom = c > 0 ? (double)c : 1.0;
      }
    }
    *a.loss = (float)(t / denom);
  }
}

void launch_loss_reduce(const ReduceArgs& a, cudaStream_t s) {
  note_launch();
  k_loss_reduce<<<1, 1024, 0, s>>>(a);
}

__global__ void k_row_scale(const int64_t* labels, int64_t n, int64_t ignore, float grad_scale,
                            const float* d_loss, int reduction, int64_t nbl,
                            const int32_t* count, float* scale) {
  const int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (r >= n) return;
  double denom = 1.0;
  if (reduction == KD_REDUCE_MEAN) {
    if (nbl > 0) denom = (double)nbl;
    else {
      const int64_t c = labels ? (int64_t)*count : n;
      denom = c > 0 ? (double)c : 1.0;
    }
  }
  const double up = (double)grad_scale * (d_loss ? (double)*d_loss : 1.0);
  const bool valid = !labels || labels[r] != ignore;
  scale[r] = valid ? (float)(up / denom) : 0.f;
}

void launch_row_scale(const int64_t* labels, int64_t n, int64_t ignore, float grad_scale,
                      const float* d_loss, int reduction, int64_t num_batch_labels,
                      const int32_t* count, float* scale, cudaStream_t s) {
  if (n <= 0) return;
  note_launch();
  k_row_scale<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(labels, n, ignore, grad_scale, d_loss,
                                                           reduction, num_batch_labels, count,
                                                           scale);
}

// ---------------------------------------------------------------- transpose
// 64 x 64 tiles, 256 threads.  Rows come in as 16-byte vectors (a warp reads
// 4 rows x 128 bytes), go through shared memory, and leave as 16-byte vectors
// of 8 transposed elements; a warp gathers 32 consecutive columns of one row
// group, so neither shared-memory phase has bank conflicts.  Ragged edges and
// unaligned pitches take element-wise accesses.
__global__ void __launch_bounds__(256) k_transpose_bf16(const uint16_t* __restrict__ src,
                                                        int64_t rows, int64_t cols, int64_t lds,
                                                        uint16_t* __restrict__ dst, int64_t ldd,
                                                        int vec) {
  __shared__ __align__(16) uint16_t t[64][72];
  const int64_t r0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
  const int tid = threadIdx.x;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int row = tid / 8 + 32 * k, cg = tid % 8;
    const int64_t r = r0 + row, c = c0 + 8 * cg;
    if (vec && r < rows && c + 8 <= cols) {
      *reinterpret_cast<uint4*>(&t[row][8 * cg]) =
          *reinterpret_cast<const uint4*>(src + r * lds + c);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        t[row][8 * cg + i] = (r < rows && c + i < cols) ? src[r * lds + c + i] : (uint16_t)0;
    }
  }
  __syncthreads();
  const int oc = tid % 32;  // column of the tile = row of the output
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int ocol = oc + 32 * k;        // tile column -> output row c0 + ocol
    const int rg = tid / 32;             // rows 8 rg .. 8 rg + 7 -> output columns
    const int64_t orow = c0 + ocol, ocol0 = r0 + 8 * rg;
    if (orow >= cols) continue;
    uint16_t e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = t[8 * rg + i][ocol];
    if (vec && ocol0 + 8 <= rows) {
      uint4 u;
      u.x = e[0] | ((uint32_t)e[1] << 16);
      u.y = e[2] | ((uint32_t)e[3] << 16);
      u.z = e[4] | ((uint32_t)e[5] << 16);
      u.w = e[6] | ((uint32_t)e[7] << 16);
      *reinterpret_cast<uint4*>(dst + orow * ldd + ocol0) = u;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (ocol0 + i < rows) dst[orow * ldd + ocol0 + i] = e[i];
    }
  }
}

void launch_transpose_bf16(const __nv_bfloat16* src, int64_t rows, int64_t cols, int64_t lds,
                           __nv_bfloat16* dst, int64_t ldd, cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return;
  const int vec = (lds % 8) == 0 && (ldd % 8) == 0 &&
                  (reinterpret_cast<uintptr_t>(src) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(dst) & 15) == 0;
  dim3 grid((unsigned)((cols + 63) / 64), (unsigned)((rows + 63) / 64));
  note_launch();
  k_transpose_bf16<<<grid, 256, 0, s>>>(reinterpret_cast<const uint16_t*>(src), rows, cols, lds,
                                        reinterpret_cast<uint16_t*>(dst), ldd, vec);
}

}  // namespace kd
