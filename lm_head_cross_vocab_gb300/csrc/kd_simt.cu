// fp32 path on CUDA cores.  tcgen05 has no true-fp32 MMA kind (tf32 drops
// mantissa bits), so fp32 problems -- whose per-token tolerance is 1e-5 --
// run a plain FFMA-tiled projection with the same online-softmax epilogue as
// the tensor-core path:
//   k_simt_fwd    logits tile (32 rows x 64 columns) -> online state per row
//                 over one vocabulary split -> partial record
//   k_simt_gprod  logits tile -> closed-form gradient tile G (fp32) for a
//                 (row chunk x vocab chunk) of the backward
//   k_simt_gemm   dH += G W, dW += G^T H with element strides
#include "kd_internal.h"

namespace kd {

namespace {

constexpr int BM = 32, BN = 64, BK = 32, NT = 256;

// z[BM][BN] tile = H[r0 .. r0+BM) . W[c0 .. c0+BN)^T into smem Z (row pitch BN+1)
__device__ __forceinline__ void tile_logits(const float* __restrict__ H,
                                            const float* __restrict__ W, int64_t n,
                                            int64_t vocab, int64_t d, int64_t r0, int64_t c0,
                                            float (*Hs)[BM + 1], float (*Ws)[BN + 1],
                                            float (*Z)[BN + 1]) {
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[2][4] = {};
  for (int64_t k0 = 0; k0 < d; k0 += BK) {
    for (int i = tid; i < BM * BK; i += NT) {
      const int r = i / BK, k = i % BK;
      const int64_t gr = r0 + r, gk = k0 + k;
      Hs[k][r] = (gr < n && gk < d) ? H[gr * d + gk] : 0.f;
    }
    for (int i = tid; i < BN * BK; i += NT) {
      const int c = i / BK, k = i % BK;
      const int64_t gc = c0 + c, gk = k0 + k;
      Ws[k][c] = (gc < vocab && gk < d) ? W[gc * d + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < BK; ++k) {
      const float h0 = Hs[k][ty], h1 = Hs[k][ty + 16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float w = Ws[k][tx + 16 * j];
        acc[0][j] = fmaf(h0, w, acc[0][j]);
        acc[1][j] = fmaf(h1, w, acc[1][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    Z[ty][tx + 16 * j] = acc[0][j];
    Z[ty + 16][tx + 16 * j] = acc[1][j];
  }
}

// first index i in sorted ids[0..k) with ids[i] >= x
__device__ __forceinline__ int lower_bound(const int32_t* ids, int k, int64_t x) {
  int lo = 0, hi = k;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)ids[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

}  // namespace

__global__ void __launch_bounds__(NT) k_simt_fwd(SimtArgs a) {
  __shared__ float Hs[BK][BM + 1];
  __shared__ float Ws[BK][BN + 1];
  __shared__ float Zs[BM][BN + 1];
  __shared__ float Zt[BM][BN + 1];
  const Consts c = a.c;
  const int64_t r0 = (int64_t)blockIdx.x * BM;
  const int split = blockIdx.y;
  const int64_t n_tiles = (a.vocab + BN - 1) / BN;
  const int64_t t0 = n_tiles * split / a.n_splits, t1 = n_tiles * (split + 1) / a.n_splits;
  const int tid = threadIdx.x, er = tid >> 3, seg = tid & 7;  // epilogue: row, 8-col segment
  const int64_t row = r0 + er;
  const bool row_ok = row < a.n;
  const bool has_t_gemm = a.teacher == KD_TEACHER_TIED || a.teacher == KD_TEACHER_SEPARATE;
  const bool has_t = has_t_gemm || a.teacher == KD_TEACHER_LOGITS;
  const bool topk = a.teacher == KD_TEACHER_TOPK;
  int64_t y = -1;
  if (row_ok && a.labels) y = a.labels[row];
  const float* stt = (a.js_pass && row_ok) ? a.stats + row * KD_STATS_PER_TOKEN : nullptr;
  const int32_t* ids = (topk && row_ok) ? a.sidx + row * a.k : nullptr;
  const float* ps = (topk && row_ok) ? a.sp + row * a.k : nullptr;
  int kp = 0;
  if (ids) kp = lower_bound(ids, a.k, t0 * BN + seg * 8);
  RowState st;
  st.init();
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t c0 = t * BN;
    tile_logits(a.h_s, a.w_s, a.n, a.vocab, a.d_s, r0, c0, Hs, Ws, Zs);
    if (has_t_gemm) {
      const float* wt = a.teacher == KD_TEACHER_TIED ? a.w_s : a.w_t;
      const int64_t dt = a.teacher == KD_TEACHER_TIED ? a.d_s : a.d_t;
      tile_logits(a.h_t, wt, a.n, a.vocab, dt, r0, c0, Hs, Ws, Zt);
    }
    __syncthreads();
    if (row_ok) {
      const int64_t col0 = c0 + seg * 8;
      const int nv = valid_cols(a.vocab - col0, 8);
      float zs[8], zt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        zs[j] = Zs[er][seg * 8 + j];
        zt[j] = 0.f;
        if (has_t_gemm) zt[j] = Zt[er][seg * 8 + j];
        else if (has_t && j < nv) zt[j] = a.zt[row * a.vocab + col0 + j];
      }
      if (a.js_pass) {
        for (int j = 0; j < nv; ++j)
          js_terms(zs[j], zt[j], stt[S_LSE_TT], stt[S_DLSE], c, st.jq, st.jp, st.jx,
                   a.variant != KD_KL_SKEW_JS);
      } else {
        if (has_t) update<8, true, true>(st, zs, zt, nv, c);
        else update<8, false, true>(st, zs, zt, nv, c);
        if (y >= col0 && y < col0 + nv) {
          st.zys += zs[y - col0];
          st.zyt += zt[y - col0];
        }
        if (ids) {
          while (kp < a.k && (int64_t)ids[kp] < col0 + nv) {
            const int64_t id = ids[kp];
            if (id >= col0) st.tk = fmaf(ps[kp], zs[id - col0] * c.inv_ts, st.tk);
            ++kp;
          }
        }
      }
    }
    __syncthreads();
    if (ids) kp = lower_bound(ids, a.k, (t + 1) * BN + seg * 8);
  }
  // reduce the 8 segments of each row (lanes 8r .. 8r+7 of one warp)
  for (int o = 4; o > 0; o >>= 1) merge(st, shfl_xor(st, o), c);
  if (row_ok && seg == 0) st.store(a.partials + ((int64_t)split * a.n + row) * kRec);
}

__global__ void __launch_bounds__(NT) k_simt_gprod(SimtArgs a) {
  __shared__ float Hs[BK][BM + 1];
  __shared__ float Ws[BK][BN + 1];
  __shared__ float Zs[BM][BN + 1];
  __shared__ float Zt[BM][BN + 1];
  const Consts c = a.c;
  const int64_t r0 = a.r0 + (int64_t)blockIdx.x * BM;
  const int64_t c0 = a.c0 + (int64_t)blockIdx.y * BN;
  const bool has_t_gemm = a.teacher == KD_TEACHER_TIED || a.teacher == KD_TEACHER_SEPARATE;
  const bool has_t = has_t_gemm || a.teacher == KD_TEACHER_LOGITS;
  const bool topk = a.teacher == KD_TEACHER_TOPK;
  const int64_t r_end = a.r0 + a.rc, c_end = a.c0 + a.cc;
  tile_logits(a.h_s, a.w_s, r_end, c_end, a.d_s, r0, c0, Hs, Ws, Zs);
  if (has_t_gemm) {
    const float* wt = a.teacher == KD_TEACHER_TIED ? a.w_s : a.w_t;
    const int64_t dt = a.teacher == KD_TEACHER_TIED ? a.d_s : a.d_t;
    tile_logits(a.h_t, wt, r_end, c_end, dt, r0, c0, Hs, Ws, Zt);
  }
  __syncthreads();
  const int tid = threadIdx.x, er = tid >> 3, seg = tid & 7;
  const int64_t row = r0 + er;
  if (row >= r_end) return;
  const float scale = a.row_scale[row];
  const float* stt = a.stats + row * KD_STATS_PER_TOKEN;
  const int64_t y = a.labels ? a.labels[row] : -1;
  const int64_t col0 = c0 + seg * 8;
  const int32_t* ids = topk ? a.sidx + row * a.k : nullptr;
  int kp = ids ? lower_bound(ids, a.k, col0) : 0;
  for (int j = 0; j < 8; ++j) {
    const int64_t col = col0 + j;
    if (col >= c_end) break;
    const float zs = Zs[er][seg * 8 + j];
    float zt = 0.f;
    if (has_t_gemm) zt = Zt[er][seg * 8 + j];
    else if (has_t) zt = a.zt[row * a.vocab + col];
    float g = 0.f, gt = 0.f;
    if (scale != 0.f) {
      if (has_t) {
        g = a.w_kl_ts * kl_grad(zs, zt, stt, a.variant, c);
      } else if (topk) {
        float pk = 0.f;
        if (kp < a.k && (int64_t)ids[kp] == col) pk = a.sp[row * a.k + kp++];
        g = a.w_kl_ts * (stt[S_MASS] * ex2((zs * c.inv_ts - stt[S_LSE_ST]) * kL2E) - pk);
      }
      const float ey = col == y ? 1.f : 0.f;
      if (a.w_sce != 0.f) g = fmaf(a.w_sce, ex2((zs - stt[S_LSE_S1]) * kL2E) - ey, g);
      g *= scale;
      if (a.gt) gt = scale * a.w_tce * (ex2((zt - stt[S_LSE_T1]) * kL2E) - ey);
    }
    const int64_t o = (row - a.r0) * a.cc + (col - a.c0);
    a.g[o] = g;
    if (a.gt) a.gt[o] = gt;
  }
}

void launch_simt_fwd(const SimtArgs& a, cudaStream_t s) {
  if (a.n <= 0) return;
  dim3 grid((unsigned)((a.n + BM - 1) / BM), (unsigned)a.n_splits);
  note_launch();
  k_simt_fwd<<<grid, NT, 0, s>>>(a);
}

void launch_simt_gprod(const SimtArgs& a, cudaStream_t s) {
  if (a.rc <= 0 || a.cc <= 0) return;
  dim3 grid((unsigned)((a.rc + BM - 1) / BM), (unsigned)((a.cc + BN - 1) / BN));
  note_launch();
  k_simt_gprod<<<grid, NT, 0, s>>>(a);
}

// ---------------------------------------------------------------- GEMM
namespace {
constexpr int GM = 64, GN = 64, GK = 16;
}

__global__ void __launch_bounds__(NT) k_simt_gemm(const float* __restrict__ A, int64_t sam,
                                                  int64_t sak, const float* __restrict__ B,
                                                  int64_t sbk, int64_t sbn, float* C,
                                                  int64_t ldc, int64_t M, int64_t N, int64_t K,
                                                  int accumulate) {
  __shared__ float As[GK][GM + 1];
  __shared__ float Bs[GK][GN + 1];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int64_t m0 = (int64_t)blockIdx.x * GM, n0 = (int64_t)blockIdx.y * GN;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += GK) {
    for (int i = tid; i < GM * GK; i += NT) {
      const int m = i % GM, k = i / GM;
      const int64_t gm = m0 + m, gk = k0 + k;
      As[k][m] = (gm < M && gk < K) ? A[gm * sam + gk * sak] : 0.f;
    }
    for (int i = tid; i < GN * GK; i += NT) {
      const int nn = i % GN, k = i / GN;
      const int64_t gn = n0 + nn, gk = k0 + k;
      Bs[k][nn] = (gn < N && gk < K) ? B[gk * sbk + gn * sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < GK; ++k) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = As[k][ty + 16 * i];
        bv[i] = Bs[k][tx + 16 * i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t m = m0 + ty + 16 * i, nn = n0 + tx + 16 * j;
      if (m < M && nn < N) {
        float* p = C + m * ldc + nn;
        *p = accumulate ? *p + acc[i][j] : acc[i][j];
      }
    }
}

void launch_simt_gemm(const float* A, int64_t sam, int64_t sak, const float* B, int64_t sbk,
                      int64_t sbn, float* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                      bool accumulate, cudaStream_t s) {
  if (M <= 0 || N <= 0) return;
  dim3 grid((unsigned)((M + GM - 1) / GM), (unsigned)((N + GN - 1) / GN));
  note_launch();
  k_simt_gemm<<<grid, NT, 0, s>>>(A, sam, sak, B, sbk, sbn, C, ldc, M, N, K, accumulate ? 1 : 0);
}

}  // namespace kd
