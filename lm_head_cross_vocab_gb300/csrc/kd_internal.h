// Host-side internal interface between the C ABI (kd_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kd.h"
#include "kd_common.cuh"

namespace kd {

// Count `k` kernel launches (reported by kd_launch_count()).
void note_launch(int k = 1);

// Clusters of `kern` that can be co-resident on the current device when it is
// launched with `cfg` (its cluster dimension attribute and dynamic shared
// memory); 0 if the query fails.  Cached per (kernel, device, cluster size,
// shared memory bytes) under a mutex, so host threads driving different
// devices at the same time each see their own device's answer.
int max_active_clusters(const void* kern, const cudaLaunchConfig_t& cfg);

// ---------------------------------------------------------------- aux kernels
// Count valid labels into *count (int32, zeroed by the caller) and flag bad ones.
void launch_label_check(const int64_t* labels, int64_t n, int64_t vocab, int64_t ignore,
                        int32_t* count, uint32_t* status, cudaStream_t s);
// Sort each row's top-K ids ascending (probabilities follow), validate them,
// and write M = sum p and E = sum p log p per row.
void launch_topk_prep(const int32_t* idx, const float* p, int64_t n, int k, int64_t vocab,
                      int32_t* sidx, float* sp, float* mass, float* ent, uint32_t* status,
                      cudaStream_t s);
// Merge per-split partial records [n_parts][n][kRec] and finalise every row.
struct CombineArgs {
  const float* partials;
  int n_parts;
  int64_t n, vocab;
  Consts c;
  int variant;
  int has_t, topk;
  int js_pass;            // 1: records hold skew-JS second-pass sums only
  const int64_t* labels;  // may be NULL
  int64_t ignore;
  const float* mass;      // top-K
  const float* ent;
  float *ce_s, *ce_t, *kl, *stats;  // stats must be non-NULL
};
void launch_combine(const CombineArgs& a, cudaStream_t s);
// Weighted, reduced scalar loss from the per-token outputs.
struct ReduceArgs {
  const float *ce_s, *ce_t, *kl;
  const int64_t* labels;
  int64_t n, ignore;
  float w_sce, w_tce, w_kl_t2;
  int reduction;
  int64_t num_batch_labels;
  const int32_t* count;
  float* loss;
};
void launch_loss_reduce(const ReduceArgs& a, cudaStream_t s);
// Per-row gradient scale: valid ? grad_scale * (*d_loss) / denom : 0.
void launch_row_scale(const int64_t* labels, int64_t n, int64_t ignore, float grad_scale,
                      const float* d_loss, int reduction, int64_t num_batch_labels,
                      const int32_t* count, float* scale, cudaStream_t s);
// dst[c][r] = src[r][c] for a [rows, cols] bf16 matrix (pitches in elements).
void launch_transpose_bf16(const __nv_bfloat16* src, int64_t rows, int64_t cols, int64_t lds,
                           __nv_bfloat16* dst, int64_t ldd, cudaStream_t s);

// ---------------------------------------------------------- streaming path
struct StreamArgs {
  const void* zs;       // [n, vocab]
  const void* zt;       // [n, vocab] or NULL
  int64_t n, vocab;
  Consts c;
  int variant;
  int is_bf16;
  int topk;             // top-K teacher: use sidx/sp/mass/ent
  int k;
  const int32_t* sidx;
  const float* sp;
  const float* mass;
  const float* ent;
  const int64_t* labels;
  int64_t ignore;
  float *ce_s, *ce_t, *kl, *stats;
  // backward
  const float* row_scale;
  float w_sce, w_kl_ts;  // w_sce, w_kl * T_s
  void* dz;              // [n, vocab] gradient of the student logits
  uint32_t* status;      // device status word (bounded-wait timeouts)
  // test hooks of the ring kernels (0 in normal use): a shorter limit for
  // every bounded wait, and one withheld consumer release (CTA 0, consumer
  // warp 0, its first stage), so that a test can make the producer's wait for
  // that stage run out with no copy in flight
  uint64_t wait_limit_ns;
  int debug_withhold_release;
};
void launch_stream_fwd(const StreamArgs& a, cudaStream_t s);
void launch_stream_bwd(const StreamArgs& a, cudaStream_t s);
// Packed bf16 ring kernels for T = 1 / T = 2 (16-byte aligned rows); return
// false, launching nothing, when the problem needs the generic kernels.
bool launch_stream_fwd_packed(const StreamArgs& a, cudaStream_t s);
bool launch_stream_bwd_packed(const StreamArgs& a, cudaStream_t s);

// ------------------------------------------- projected teacher (fused loss)
// Logit students against teacher logits over another vocabulary, moved onto
// the student vocabulary by a token map inside the loss kernels
// (kd_project.cu, k_proj_loss): the forward writes the per-token outputs and
// statistics, the backward d z_s; no projected [n, vs] tensor is stored.
struct ProjLossArgs {
  const int32_t* token_map;  // [vt]
  const void* zt;            // [n, vt]
  const void* zs;            // [n, vs]
  int64_t n, vt, vs;
  int is_bf16;
  float inv_tp;              // 1 / projection temperature
  Consts c;                  // teacher side at T = 1
  int variant;
  const int64_t* labels;
  int64_t ignore;
  float *ce_s, *ce_t, *kl, *stats;
  const float* row_scale;
  float w_sce, w_kl_ts;
  void* dz;
  int mode;                  // 0 forward, 1 backward
  uint32_t* status;
};
size_t proj_loss_workspace_bytes(int64_t vt, int64_t vs);
// false: a teacher row needs more than 8 CTAs or a CTA more than 32 Ki ids
bool proj_loss_supported(int64_t vt, int64_t vs, bool bf16);
// Builds the maps in `workspace` and launches the fused kernel; 1 on error.
int launch_proj_loss(const ProjLossArgs& a, void* workspace, cudaStream_t s);

// ------------------------------------------------------------- fp32 SIMT path
struct SimtArgs {
  // student: hidden (h_s, w_s, d_s); teacher: hidden (h_t, w_t, d_t) or logits zt
  const float *h_s, *w_s, *h_t, *w_t, *zt;
  int64_t n, vocab, d_s, d_t;
  int teacher;           // kd_teacher_kind
  Consts c;
  int variant;
  const int64_t* labels;
  int64_t ignore;
  const int32_t* sidx;
  const float* sp;
  int k;
  int n_splits;
  float* partials;       // [n_splits][n][kRec]
  const float* stats;    // pass-2 / backward
  int js_pass;
  // backward G producer over rows [r0, r0+rc) x cols [c0, c0+cc)
  int64_t r0, rc, c0, cc;
  const float* row_scale;
  float w_sce, w_tce, w_kl_ts;
  float* g;              // [rc, cc] student gradient tile
  float* gt;             // [rc, cc] tied teacher-CE gradient tile or NULL
};
void launch_simt_fwd(const SimtArgs& a, cudaStream_t s);
void launch_simt_gprod(const SimtArgs& a, cudaStream_t s);
// C[m, n] (+)= sum_k A(m, k) B(k, n) with element strides.
void launch_simt_gemm(const float* A, int64_t sam, int64_t sak, const float* B, int64_t sbk,
                      int64_t sbn, float* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                      bool accumulate, cudaStream_t s);

// ------------------------------------------------------------ tcgen05 path
int tc_num_sms();
bool tc_use_pairs();                                  // CTA-pair (cta_group::2) tiles
int tc_fused_tile_cols(bool two_sides, bool pair);    // vocabulary columns per tile (forward)
int tc_grad_tile_cols(bool two_sides, bool pair);     // ... of the gradient producer
int tc_tile_rows(bool pair);                          // token rows per tile (MMA M)
struct TcFwdArgs {
  const void *h_s, *w_s, *h_t, *w_t, *zs_logits, *zt_logits;
  int64_t n, vocab, d_s, d_t;
  int s_gemm, t_gemm;      // sides computed by tcgen05
  int s_logits, t_logits;  // sides read from materialised logits
  int topk;
  Consts c;
  int variant;
  const int64_t* labels;
  int64_t ignore;
  const int32_t* sidx;
  const float* sp;
  int k;
  int n_splits;
  float* partials;
  const float* stats;      // js pass
  int js_pass;
  uint32_t* status;
};
// Returns a cudaError_t-compatible code (0 = success).
int launch_tc_fwd(const TcFwdArgs& a, int num_ctas, cudaStream_t s);

struct TcGradArgs {
  const void *h_s, *w_s, *h_t, *w_t, *zs_logits, *zt_logits;
  int64_t n, vocab, d_s, d_t;
  int s_gemm, t_gemm, s_logits, t_logits, topk;
  Consts c;
  int variant;
  const int64_t* labels;
  int64_t ignore;
  const int32_t* sidx;
  const float* sp;
  int k;
  const float* stats;
  const float* row_scale;
  float w_sce, w_tce, w_kl_ts;
  int64_t r0, rc, c0, cc;  // chunk
  __nv_bfloat16* g;        // [rc, ldg] row-major student G (or d z_s)
  int64_t ldg;
  __nv_bfloat16* gt;       // [rc, ldg] row-major tied teacher-CE gradient, or NULL
  uint32_t* status;
};
int launch_tc_grad(const TcGradArgs& a, int num_ctas, cudaStream_t s);

// Tensor-core GEMM: C[M, N] = sum_k A[M, K] B[N, K] (+ A1 B1 over K1); each
// operand K-major ([M, K] / [N, K]) or, with its _mn flag, MN-major ([K, M] /
// [K, N]); bf16 operands, ld = pitch of the stored layout in elements, fp32
// accumulate.
enum TcOutMode { TC_OUT_BF16 = 0, TC_OUT_F32 = 1, TC_OUT_F32_ACC = 2, TC_OUT_F32_ACC_BF16 = 3 };
struct TcGemmArgs {
  const __nv_bfloat16 *a0, *b0, *a1, *b1;
  int64_t lda0, ldb0, lda1, ldb1;
  int64_t M, N, K0, K1;    // K1 = 0: single segment
  int a0_mn, b0_mn, a1_mn, b1_mn;
  int mode;
  float* c32;              // fp32 accumulator / output [M, ldc32]
  int64_t ldc32;
  __nv_bfloat16* c16;      // bf16 output [M, ldc16]
  int64_t ldc16;
  uint32_t* status;
};
int launch_tc_gemm(const TcGemmArgs& a, int num_ctas, cudaStream_t s);

}  // namespace kd
