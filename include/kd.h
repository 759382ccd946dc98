/*
 * kd.h -- C ABI of the GB300 (sm_103a) fused LM-head + cross-entropy + KL
 * knowledge-distillation loss.
 *
 * What it computes (per token n, vocabulary column v):
 *   z_s = H_s W_s^T (or given student logits), z_t = H_t W_t^T (or given
 *   teacher logits, or a cached top-K teacher), a_s = z_s / T_s,
 *   a_t = z_t / T_t, p = softmax(a_s) (student), q = softmax(a_t) (teacher).
 *   CE_s = logsumexp(z_s) - z_s[y], CE_t likewise on z_t (T = 1)
 *     -- flash_kd API doc, flash_ce_kd_loss, "labels" / "Returns".
 *   KL variants forward KL(q||p), reverse KL(p||q), Jeffreys (their sum),
 *   skew-JS (1-b) KL(q||m) + b KL(p||m), m = (1-b) q + b p
 *     -- orda-kernel README, "KL variants" (skew-JS's split is this
 *        library's reading: the page names it and its two halves only).
 *   Sparse top-K objective sum_S p log p - sum_S p a + M logsumexp(a),
 *   gradient M softmax(a) - p -- Full-Chunked-KL-Loss README, "Methods",
 *   "Full Chunked KL".
 *   loss = sum_valid (w_sce CE_s + w_tce CE_t + w_kl T_s^2 KL) / denom
 *     -- orda-kernel README, "Parameters" (each KL row scales by T_s^2,
 *        reduction "mean"/"sum"); nemo_automodel KDLoss (T^2, mean over
 *        valid tokens or sum / num_batch_labels).
 * The (tokens x vocab) logits are never stored: the forward keeps running
 * online-softmax statistics per token (flash_kd: "online-softmax (running
 * max + rescale)"), the backward recomputes each logit tile and applies the
 * closed-form gradient (Full-Chunked-KL-Loss README, "Full Chunked KL").
 *
 * Conventions
 *   - Every pointer in kd_inputs and every output/workspace pointer is a
 *     DEVICE pointer on the current CUDA device, owned by the caller.  The
 *     library never allocates device memory; scratch space is the caller's
 *     `workspace` of at least the size kd_workspace_size() reports.
 *   - All matrices are dense row-major with the last dimension contiguous:
 *     H_s [N, D_s], W_s [V, D_s], H_t [N, D_t], W_t [V, D_t],
 *     logits [N, V], labels int64 [N], topk_idx int32 [N, K],
 *     topk_p fp32 [N, K].  Element type of H / W / logits is kd_problem.dtype.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  Host-checkable errors (shapes, NULL
 *     pointers, parameter ranges, unsupported combinations, a workspace that
 *     is too small) return synchronously and enqueue nothing.
 *   - Data-dependent errors are OR-ed into the device word `dev_status`
 *     (KD_DEV_* bits), never raised: a label that is neither ignore_index
 *     nor in [0, V) (its CE becomes NaN; it is never used as a memory
 *     index -- orda-kernel README, "Parameters", ignore_index), a top-K id
 *     outside [0, V) or repeated in a row, a bounded device wait that timed
 *     out.  The caller zeroes dev_status before the call and reads it after
 *     synchronising (unless assume_valid_labels is set and it opts out).
 *   - No exception crosses this ABI.
 */
#ifndef KD_H_
#define KD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KD_ABI_VERSION 5

typedef enum kd_status {
  KD_OK = 0,
  KD_ERR_INVALID_ARG = 1,  /* bad shape, NULL pointer, parameter out of range   */
  KD_ERR_UNSUPPORTED = 2,  /* valid but unsupported combination / layout      */
  KD_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than required          */
  KD_ERR_BAD_LABEL = 4,    /* reported through dev_status only                 */
  KD_ERR_BAD_TOPK = 5,     /* reported through dev_status only                 */
  KD_ERR_TIMEOUT = 6,      /* reported through dev_status only                 */
  KD_ERR_CUDA = 7,         /* a CUDA runtime/driver call failed                */
  KD_ERR_NO_DEVICE = 8     /* current device is not an sm_103 GPU              */
} kd_status;

/* bits OR-ed into *dev_status by the kernels */
#define KD_DEV_BAD_LABEL 0x1u
#define KD_DEV_BAD_TOPK 0x2u
#define KD_DEV_TIMEOUT 0x4u
#define KD_DEV_BAD_MAP 0x8u   /* token map entry outside [-1, V_student) */
#define KD_DEV_MAP_UNSUPPORTED 0x10u /* KD_TEACHER_PROJECTED: the token map sends more
                                     * teacher tokens into one student id range
                                     * than the fused kernel's receive buffers
                                     * hold; nothing was computed (use
                                     * kd_project_teacher_logits + a
                                     * KD_TEACHER_LOGITS teacher instead) */

typedef enum kd_dtype { KD_BF16 = 0, KD_FP32 = 1 } kd_dtype;

/* orda-kernel README, "Quickstart" (student hidden + weight) and flash_kd
 * (already-materialised student logits). */
typedef enum kd_student_kind { KD_STUDENT_HIDDEN = 0, KD_STUDENT_LOGITS = 1 } kd_student_kind;

/* orda-kernel README, "Teacher descriptors": TiedTeacher (teacher hidden
 * through the student's W_s), SeparateTeacher / PrecomputedTeacher with
 * teacher_hidden + teacher_weight (own W_t), PrecomputedTeacher(logits=...);
 * Full-Chunked-KL-Loss README, "Methods": cached top-K probabilities.
 * KD_TEACHER_NONE: plain fused linear + CE (no KL, no teacher).
 * KD_TEACHER_PROJECTED: teacher logits over another vocabulary
 * (kd_inputs.logits_t [N, vocab_teacher]) moved onto the student vocabulary
 * by kd_inputs.token_map inside the loss kernels (orda-kernel README,
 * "Cross-vocabulary distillation": token-map projection into a
 * PrecomputedTeacher with logits_temperature = t_teacher):
 *   z_p[n, i] = log sum_{j : token_map[j] = i} exp(logits_t[n, j] / t_teacher),
 * an id no teacher token maps to having probability 0.  z_p is then the
 * teacher's logits at temperature 1 (CE_t = logsumexp(z_p) - z_p[y]); the
 * student is KD_STUDENT_LOGITS at t_student.  Results equal
 * kd_project_teacher_logits followed by a KD_TEACHER_LOGITS teacher with
 * t_teacher = 1, but the projected [N, V] tensor is never stored. */
typedef enum kd_teacher_kind {
  KD_TEACHER_NONE = 0,
  KD_TEACHER_TIED = 1,
  KD_TEACHER_SEPARATE = 2,
  KD_TEACHER_LOGITS = 3,
  KD_TEACHER_TOPK = 4,
  KD_TEACHER_PROJECTED = 5
} kd_teacher_kind;

/* orda-kernel README, "KL variants" (teacher-detached subset). */
typedef enum kd_variant {
  KD_KL_FORWARD = 0,  /* KL(q||p)                                   */
  KD_KL_REVERSE = 1,  /* KL(p||q)                                   */
  KD_KL_JEFFREYS = 2, /* KL(q||p) + KL(p||q)                        */
  KD_KL_SKEW_JS = 3,  /* (1-b) KL(q||m) + b KL(p||m), m=(1-b)q+bp   */
  KD_KL_SKEW_FORWARD = 4, /* KL(q||m) (orda "skew_forward")              */
  KD_KL_SKEW_REVERSE = 5  /* KL(p||m) (orda "skew_reverse")              */
} kd_variant;

typedef enum kd_reduction { KD_REDUCE_MEAN = 0, KD_REDUCE_SUM = 1 } kd_reduction;

/* Problem description (host memory, read during the call only). */
typedef struct kd_problem {
  int64_t n_tokens;      /* N >= 0                                            */
  int64_t vocab;         /* V >= 1                                            */
  int64_t d_student;     /* D_s (hidden students), multiple of 8 for bf16     */
  int64_t d_teacher;     /* D_t (separate teachers; tied uses D_s)            */
  int64_t topk;          /* K (top-K teachers), 1..1024                       */
  int32_t dtype;         /* kd_dtype of H, W and logits                       */
  int32_t student;       /* kd_student_kind                                   */
  int32_t teacher;       /* kd_teacher_kind                                   */
  int32_t variant;       /* kd_variant                                        */
  int32_t reduction;     /* kd_reduction                                      */
  float t_student;       /* T_s > 0 (kl_temperature)                          */
  float t_teacher;       /* T_t > 0 (kl_teacher_temperature; set = T_s)       */
  float w_student_ce;    /* >= 0, finite                                      */
  float w_teacher_ce;    /* >= 0, finite; 0 for top-K                         */
  float w_kl;            /* >= 0, finite                                      */
  float beta;            /* skew variants: b in (0,1) (kl_beta)              */
  int64_t ignore_index;  /* label value excluded from CE and KL               */
  int64_t num_batch_labels; /* > 0: mean divides by this instead of N_valid  */
  int32_t assume_valid_labels; /* 1: caller promises labels in range          */
  int32_t teacher_grads;  /* 1: kd_bwd_grads may be asked for d_h_t / d_w_t  */
                         /* (the workspace is sized for them); else 0        */
  int64_t vocab_chunk;   /* backward G-workspace vocab chunk (0 = auto); the  */
  int64_t seq_chunk;     /* token chunk (0 = auto). Results do not depend on  */
                         /* either beyond rounding (flash_kd chunk_size,      */
                         /* Full-Chunked-KL-Loss --chunk-sizes: memory knobs). */
  int64_t vocab_teacher; /* V_t of a KD_TEACHER_PROJECTED teacher, else 0     */
} kd_problem;

/* Input tensors (device pointers; NULL where the problem does not use one). */
typedef struct kd_inputs {
  const void* h_s;       /* [N, D_s]  student hidden (KD_STUDENT_HIDDEN)      */
  const void* w_s;       /* [V, D_s]  student head weight                     */
  const void* logits_s;  /* [N, V]    student logits (KD_STUDENT_LOGITS)      */
  const void* h_t;       /* [N, D_t]  teacher hidden (TIED: D_t = D_s)        */
  const void* w_t;       /* [V, D_t]  teacher head weight (SEPARATE)          */
  const void* logits_t;  /* [N, V]    teacher logits (KD_TEACHER_LOGITS)      */
  const int64_t* labels; /* [N] or NULL: every token valid, no CE allowed     */
  const int32_t* topk_idx; /* [N, K] distinct ids in [0, V), any order        */
  const float* topk_p;   /* [N, K] teacher probabilities (not renormalised)   */
  const int32_t* token_map; /* [V_t] KD_TEACHER_PROJECTED: student id of each  */
                         /* teacher token, or -1 (logits_t is then [N, V_t])  */
} kd_inputs;

/* Number of floats per token in the saved statistics written by kd_fwd and
 * read by kd_bwd: logsumexp(z_s), logsumexp(a_s), logsumexp(z_t),
 * logsumexp(a_t), KL(p||q), KL(p||m), top-K mass M (skew variants: E_p[p/m]),
 * and logsumexp(a_t) - logsumexp(a_s) evaluated to full relative precision. */
#define KD_STATS_PER_TOKEN 8

/* Bytes of device workspace kd_fwd and kd_bwd need for this problem on the
 * current device.  Either output pointer may be NULL. */
kd_status kd_workspace_size(const kd_problem* problem, size_t* fwd_bytes, size_t* bwd_bytes);

/* Forward.  Writes per-token outputs (fp32 [N]; any may be NULL to skip):
 *   ce_s  student CE (0 on ignored tokens; NaN on a bad label),
 *   ce_t  teacher CE (tied / separate / logits teachers),
 *   kl    raw per-token divergence of `variant` (NOT multiplied by T_s^2,
 *         flash_kd "Returns"; 0 on ignored tokens),
 *   stats [N, KD_STATS_PER_TOKEN] saved statistics for kd_bwd,
 *   loss  one fp32 device scalar (the weighted, reduced loss).
 * workspace: device scratch of ws_bytes >= kd_workspace_size().fwd_bytes,
 * 256-byte aligned.  Its contents need not be initialised. */
kd_status kd_fwd(const kd_problem* problem, const kd_inputs* inputs, float* ce_s, float* ce_t,
                 float* kl, float* stats, float* loss, uint32_t* dev_status, void* workspace,
                 size_t ws_bytes, void* stream);

/* Backward.  Reads `stats` from a kd_fwd on the same inputs (it may be
 * reused for several backward calls).  The upstream gradient of `loss` is
 * grad_scale * (*d_loss) (d_loss is a device fp32 scalar, or NULL for 1).
 * Writes (overwrites) the requested gradients, each in kd_problem.dtype;
 * NULL skips that gradient:
 *   d_h_s      [N, D_s] d loss / d H_s      (hidden students)
 *   d_w_s      [V, D_s] d loss / d W_s      (hidden students; a tied
 *              teacher's CE term also flows into it -- orda-kernel README,
 *              "Teacher descriptors", tied teachers share the weight)
 *   d_logits_s [N, V]   d loss / d z_s      (logit students)
 * The teacher is detached from every KL variant (orda-kernel README, "KL
 * variants").  Ignored tokens get exactly zero gradient rows. */
kd_status kd_bwd(const kd_problem* problem, const kd_inputs* inputs, const float* stats,
                 const float* d_loss, float grad_scale, void* d_h_s, void* d_w_s,
                 void* d_logits_s, uint32_t* dev_status, void* workspace, size_t ws_bytes,
                 void* stream);

/* Gradients kd_bwd_grads may write; NULL skips one. */
typedef struct kd_grads {
  void* d_h_s;       /* [N, D_s] d loss / d H_s (hidden students)             */
  void* d_w_s;       /* [V, D_s] d loss / d W_s (hidden students; with a tied  */
                     /* teacher's CE term included, as in kd_bwd)             */
  void* d_logits_s;  /* [N, V]   d loss / d z_s (logit students)               */
  void* d_h_t;       /* [N, D_t] d loss / d H_t: tied or separate teachers     */
  void* d_w_t;       /* [V, D_t] d loss / d W_t: separate teachers             */
} kd_grads;

/* Backward with teacher gradients (orda-kernel README, "Teacher descriptors":
 * a teacher whose teacher_ce_weight is > 0 is trained by its CE term;
 * "Parameters" list teacher_ce_weight).  Everything kd_bwd writes, plus the
 * teacher's: the teacher is detached from every KL variant, so its gradient
 * is that of w_teacher_ce * CE_t alone, G_t = d loss / d z_t =
 * s_n w_teacher_ce (softmax(z_t) - e_y) per valid token (s_n the row scale
 * of the reduction), and
 *   d_h_t = G_t W_t   (W_s for a tied teacher)     [N, D_t]
 *   d_w_t = G_t^T H_t (separate teachers only)     [V, D_t]
 * in kd_problem.dtype.  They need a hidden student, a tied or separate
 * teacher and problem->teacher_grads = 1 (KD_ERR_INVALID_ARG otherwise); with
 * w_teacher_ce = 0 they are written as zeros. */
kd_status kd_bwd_grads(const kd_problem* problem, const kd_inputs* inputs, const float* stats,
                       const float* d_loss, float grad_scale, const kd_grads* grads,
                       uint32_t* dev_status, void* workspace, size_t ws_bytes, void* stream);

/* Plan introspection: how kd_fwd / kd_bwd will run this problem on the current
 * device.  path: 0 logits streaming, 1 fp32 CUDA cores, 2 tensor cores;
 * vocab_splits: forward vocabulary splits; chunk_rows x chunk_cols: the
 * backward gradient chunk (tokens x vocabulary columns) staged in the
 * workspace, always smaller than the full tokens x vocab matrix.  Any output
 * pointer may be NULL. */
kd_status kd_plan_info(const kd_problem* problem, int32_t* path, int32_t* vocab_splits,
                       int64_t* chunk_rows, int64_t* chunk_cols);

/* Cross-vocabulary token-map projection (orda-kernel README, "Cross-vocabulary
 * distillation", token-map projection -> PrecomputedTeacher).  When student and
 * teacher tokenizers differ, per-column KL is undefined; the teacher
 * distribution is moved onto the student vocabulary instead:
 *   out[n, i] = log sum_{j : token_map[j] = i} exp(logits_t[n, j] / temperature)
 * for every token row n < n_tokens and student id i < v_student.  Duplicate
 * teacher tokens of one student id sum in probability space; the tempering is
 * applied before the aggregation, so pass the result to kd_fwd / kd_bwd as a
 * KD_TEACHER_LOGITS teacher with t_teacher = 1 (the pages declare it with
 * logits_temperature = T).  A student id no teacher token maps to has
 * probability 0: it gets the most negative finite value of out_dtype (its
 * exponential is exactly 0, as -inf's would be, and the divergences of the
 * distillation kernels need no special case for it).
 *   token_map  device int32 [v_teacher]: student id of teacher token j, or -1
 *              (entries outside [-1, v_student) set KD_DEV_BAD_MAP in
 *              *dev_status and are skipped)
 *   logits_t   device [n_tokens, v_teacher] in in_dtype (KD_BF16 / KD_FP32)
 *   out        device [n_tokens, v_student] in out_dtype
 *   workspace  >= kd_project_workspace_size() bytes, 256-byte aligned; the
 *              inverse map is rebuilt in it on every call (its contents need
 *              not be initialised)
 * Asynchronous on `stream`; host-checkable errors return synchronously. */
kd_status kd_project_workspace_size(int64_t v_teacher, int64_t v_student, size_t* bytes);
kd_status kd_project_teacher_logits(const int32_t* token_map, int64_t v_teacher,
                                    int64_t v_student, const void* logits_t, int64_t n_tokens,
                                    int32_t in_dtype, float temperature, void* out,
                                    int32_t out_dtype, uint32_t* dev_status, void* workspace,
                                    size_t ws_bytes, void* stream);

/* Multi-teacher mixing (orda-kernel README, "Cross-vocabulary distillation",
 * multi-teacher mixing -> PrecomputedTeacher).  K cached teacher logit rows
 * over one vocabulary are mixed into one distribution, written as its
 * log-probabilities (pass them to kd_fwd / kd_bwd as a KD_TEACHER_LOGITS
 * teacher with t_teacher = 1):
 *   KD_MIX_ARITHMETIC  probability average: out = log sum_k w_k softmax(z_k)
 *   KD_MIX_GEOMETRIC   product of experts:  out = log of prod_k softmax(z_k)^w_k,
 *                      renormalised (= g - logsumexp(g), g = sum_k w_k z_k)
 * with the weights normalised to sum to 1.  A token the mixture gives no
 * probability gets the most negative finite value of out_dtype, as
 * kd_project_teacher_logits writes unmatched ids; teacher values at or below
 * -1e30 count as probability 0.
 *   logits     host array of k device pointers, each [n_tokens, vocab] in
 *              in_dtype (KD_BF16 / KD_FP32), row-major, rows contiguous
 *   k          1 .. KD_MIX_MAX_TEACHERS
 *   weights    host array of k non-negative finite floats, not all 0 (a
 *              teacher with weight 0 takes no part), or NULL for uniform
 *   out        device [n_tokens, vocab] in out_dtype; may not alias an input
 * No workspace.  Asynchronous on `stream`; argument errors return
 * KD_ERR_INVALID_ARG synchronously. */
#define KD_MIX_MAX_TEACHERS 8
typedef enum kd_mix_mode { KD_MIX_ARITHMETIC = 0, KD_MIX_GEOMETRIC = 1 } kd_mix_mode;
kd_status kd_mix_teacher_logits(const void* const* logits, int32_t k, const float* weights,
                                int64_t n_tokens, int64_t vocab, int32_t in_dtype,
                                int32_t mode, void* out, int32_t out_dtype,
                                uint32_t* dev_status, void* stream);

/* Static description of a status code. */
const char* kd_status_string(kd_status status);

/* 1 if `device` is a GPU this library's kernels run on (compute capability
 * 10.3, i.e. sm_103), else 0 -- the analogue of orda-kernel's
 * is_available() (orda-kernel README, "Installation"). */
int kd_device_supported(int device);

/* KD_ABI_VERSION of the loaded library. */
int kd_abi_version(void);

/* Diagnostic for validating the tensor-core GEMM core on its own (not part of
 * the loss): C[M, N] = sum_k A(m, k) B(n, k) with bf16 operands and fp32 C
 * (row-major, pitch N), accumulated in fp32 on tcgen05 tensor cores.
 * `layout` bit 0 clear: A stored [M, K] (K contiguous); set: A stored [K, M]
 * (M contiguous).  Bit 1 likewise for B: [N, K] or [K, N].  The contiguous
 * extent of each stored operand must be a multiple of 8 and the pointers
 * 16-byte aligned.  Device pointers, asynchronous on `stream`.  The backward
 * forms dH = G W (G [R, C] as stored, W^T: layout 0) and dW = G^T H (G as
 * stored, H^T: layout 1) this way. */
kd_status kd_diag_gemm_bf16(const void* a, const void* b, float* c, int64_t m, int64_t n,
                            int64_t k, int layout, void* stream);

/* Size of the fixed device scratch array used by kd_fwd_static_scratch. */
#define KD_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/* Forward that allocates nothing and takes no workspace (the pages have no
 * counterpart: this exists for callers of this library, not for the method).
 * For callers that cannot allocate device memory -- a plugin inside a host
 * program that owns every device buffer and passes only the step's tensors,
 * or a runtime that must not call cudaMalloc mid-step because it can
 * synchronise the device and fail -- it runs exactly kd_fwd, with kd_fwd's
 * scratch taken from a fixed KD_STATIC_SCRATCH_BYTES array in the library's
 * device image (held by every GPU that loads the library until the process
 * exits).  Inputs and outputs are the caller's, as for kd_fwd.
 *   - Returns KD_ERR_WORKSPACE, without launching anything, when the problem
 *     needs more scratch than KD_STATIC_SCRATCH_BYTES (kd_workspace_size()'s
 *     fwd_bytes tells in advance).
 *   - The first call on a device looks up the array's device address with that
 *     device current and caches it; make that first call before any stream
 *     capture.
 *   - Every call on a device shares the one array and the array keeps the last
 *     call's contents; the call clears what must start at zero.  Calls whose
 *     work overlaps on the GPU (for example on two streams at once) race on the
 *     array: order them on one stream or with events. */
kd_status kd_fwd_static_scratch(const kd_problem* problem, const kd_inputs* inputs, float* ce_s,
                                float* ce_t, float* kl, float* stats, float* loss,
                                uint32_t* dev_status, void* stream);

/* Profiling aid.  When the events are non-NULL (cudaEvent_t handles created by
 * the caller), every later kd_fwd records fwd_start right before and fwd_stop
 * right after its fused projection launch(es) on the call's stream, and
 * kd_bwd records bwd_start / bwd_stop around its recompute + dH / dW section.
 * Pass NULLs to stop recording.  Process-wide setting. */
kd_status kd_set_profile_events(void* fwd_start, void* fwd_stop, void* bwd_start,
                                void* bwd_stop);

/* Profiling aid for the tensor-core backward.  kind 0: kd_bwd records
 * starts[k] / stops[k] (cudaEvent_t handles) right before / after the launch
 * of the gradient producer for chunk k, on the call's stream; kind 1: around
 * backward GEMM launch j (2k: dH of chunk k, 2k + 1: dW of chunk k) on the
 * stream that GEMM runs on.  Launches with an index >= n record nothing.  The
 * arrays stay owned by the caller and must outlive every kd_bwd enqueued
 * while they are set; n = 0 stops recording.  Process-wide setting;
 * KD_ERR_INVALID_ARG for an unknown kind or a NULL handle. */
kd_status kd_set_profile_launch_events(int kind, void* const* starts, void* const* stops, int n);

/* Number of kernel launches this library has enqueued in this process. */
uint64_t kd_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KD_H_ */
