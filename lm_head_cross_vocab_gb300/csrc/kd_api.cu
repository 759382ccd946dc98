// C ABI of the fused LM-head + CE + KL distillation loss: argument
// validation, the per-problem plan (which kernel family, vocabulary splits,
// backward chunking, workspace layout) and the launch sequence on the
// caller's stream.  The library never allocates device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cmath>
#include <cstring>

#include "../../include/kd.h"
#include "kd_internal.h"

#include <atomic>
#include <mutex>
#include <vector>

using namespace kd;

namespace kd {
namespace {
std::atomic<uint64_t> g_launches{0};
}
void note_launch(int k) { g_launches.fetch_add((uint64_t)k, std::memory_order_relaxed); }

int max_active_clusters(const void* kern, const cudaLaunchConfig_t& cfg) {
  struct Entry {
    const void* kern;
    int dev;
    unsigned cluster;
    size_t smem;
    int value;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  unsigned cluster = 1;
  for (unsigned i = 0; i < cfg.numAttrs; ++i)
    if (cfg.attrs[i].id == cudaLaunchAttributeClusterDimension)
      cluster = cfg.attrs[i].val.clusterDim.x * cfg.attrs[i].val.clusterDim.y *
                cfg.attrs[i].val.clusterDim.z;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.kern == kern && e.dev == dev && e.cluster == cluster && e.smem == cfg.dynamicSmemBytes)
      return e.value;
  int m = 0;
  if (cudaOccupancyMaxActiveClusters(&m, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    m = 0;
  }
  cache.push_back(Entry{kern, dev, cluster, cfg.dynamicSmemBytes, m});
  return m;
}
}  // namespace kd

namespace {

// profiling events set by kd_set_profile_events (fwd start/stop, bwd start/stop)
std::atomic<void*> g_prof[4] = {};

void prof_record(int i, cudaStream_t s) {
  void* e = g_prof[i].load(std::memory_order_relaxed);
  if (e) cudaEventRecord(static_cast<cudaEvent_t>(e), s);
}

// per-launch events set by kd_set_profile_launch_events: [kind] = (starts,
// stops, n); kind 0 = gradient producer launches, 1 = backward GEMM launches
struct LaunchEvents {
  void* const* starts;
  void* const* stops;
  int n;
};
std::mutex g_lprof_mu;
LaunchEvents g_lprof[2] = {};

// Records start (stop = false) or stop event `idx` of kind `kind` on `s`.
void launch_record(int kind, int64_t idx, bool stop, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_lprof_mu);
  const LaunchEvents& e = g_lprof[kind];
  if (idx < e.n) cudaEventRecord(static_cast<cudaEvent_t>(stop ? e.stops[idx] : e.starts[idx]), s);
}

enum Path { PATH_STREAM = 0, PATH_SIMT = 1, PATH_TC = 2, PATH_PROJ = 3 };

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Layout {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  }
};

struct Plan {
  Path path;
  bool s_gemm, s_logits, t_gemm, t_logits, topk, has_t, tied, is_bf16;
  int64_t n, v, ds, dt;
  Consts c;
  int nsm;
  int n_splits;   // forward vocabulary splits
  int n_parts;    // partial records per row
  int64_t R, C;   // backward chunk (rows x vocabulary columns)
  // forward workspace
  size_t f_count, f_ce_s, f_ce_t, f_kl, f_stats, f_part, f_sidx, f_sp, f_mass, f_ent, f_proj,
      f_bytes;
  // backward workspace
  size_t b_count, b_scale, b_sidx, b_sp, b_mass, b_ent, b_g, b_gt, b_wt, b_hst, b_htt, b_dh,
      b_dw, b_dht, b_dwt, b_proj, b_bytes;
  int64_t ldv, ldn;  // pitches of W^T [D, ldv] and H^T [D, ldn]
  bool kmajor_b;     // backward GEMMs take W^T / H^T (transposed per backward) as B
  bool two_streams;  // backward GEMMs of chunk k on a side stream beside chunk k+1
};

bool finite_nonneg(float x) { return std::isfinite(x) && x >= 0.f; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

kd_status check_problem(const kd_problem* p) {
  if (!p) return KD_ERR_INVALID_ARG;
  if (p->n_tokens < 0 || p->vocab < 1 || p->n_tokens > (int64_t)1 << 31 ||
      p->vocab > (int64_t)1 << 30)
    return KD_ERR_INVALID_ARG;
  if (p->dtype != KD_BF16 && p->dtype != KD_FP32) return KD_ERR_INVALID_ARG;
  if (p->student != KD_STUDENT_HIDDEN && p->student != KD_STUDENT_LOGITS)
    return KD_ERR_INVALID_ARG;
  if (p->teacher < KD_TEACHER_NONE || p->teacher > KD_TEACHER_PROJECTED) return KD_ERR_INVALID_ARG;
  if (p->variant < KD_KL_FORWARD || p->variant > KD_KL_SKEW_REVERSE) return KD_ERR_INVALID_ARG;
  if (p->reduction != KD_REDUCE_MEAN && p->reduction != KD_REDUCE_SUM) return KD_ERR_INVALID_ARG;
  // orda-kernel README, "Parameters": term weights finite and >= 0
  if (!finite_nonneg(p->w_student_ce) || !finite_nonneg(p->w_teacher_ce) ||
      !finite_nonneg(p->w_kl))
    return KD_ERR_INVALID_ARG;
  if (!(std::isfinite(p->t_student) && p->t_student > 0.f) ||
      !(std::isfinite(p->t_teacher) && p->t_teacher > 0.f))
    return KD_ERR_INVALID_ARG;
  // orda-kernel README, "KL variants": kl_beta in (0, 1) for the skew family
  if (is_skew(p->variant) && !(p->beta > 0.f && p->beta < 1.f)) return KD_ERR_INVALID_ARG;
  if (p->student == KD_STUDENT_HIDDEN && p->d_student < 1) return KD_ERR_INVALID_ARG;
  if (p->teacher == KD_TEACHER_SEPARATE && p->d_teacher < 1) return KD_ERR_INVALID_ARG;
  if (p->teacher == KD_TEACHER_TIED) {
    if (p->student != KD_STUDENT_HIDDEN) return KD_ERR_INVALID_ARG;
    if (p->d_teacher != 0 && p->d_teacher != p->d_student) return KD_ERR_INVALID_ARG;
  }
  if (p->teacher == KD_TEACHER_TOPK) {
    if (p->topk < 1 || p->topk > 1024 || p->topk > p->vocab) return KD_ERR_INVALID_ARG;
    if (p->w_teacher_ce != 0.f) return KD_ERR_UNSUPPORTED;  // no teacher logits
  }
  if (p->teacher == KD_TEACHER_NONE && p->w_teacher_ce != 0.f) return KD_ERR_INVALID_ARG;
  if (p->teacher == KD_TEACHER_PROJECTED) {
    // orda-kernel README, "Cross-vocabulary distillation": teacher logits over
    // their own vocabulary, moved onto the student's by a token map
    if (p->vocab_teacher < 1 || p->vocab_teacher > (int64_t)1 << 30) return KD_ERR_INVALID_ARG;
    if (p->student != KD_STUDENT_LOGITS) return KD_ERR_UNSUPPORTED;  // project, then kd_fwd
    if (!proj_loss_supported(p->vocab_teacher, p->vocab, p->dtype == KD_BF16))
      return KD_ERR_UNSUPPORTED;
  }
  return KD_OK;
}

kd_status check_inputs(const kd_problem* p, const kd_inputs* in) {
  if (!in) return KD_ERR_INVALID_ARG;
  if (p->n_tokens == 0) return KD_OK;
  if (p->student == KD_STUDENT_HIDDEN && (!in->h_s || !in->w_s)) return KD_ERR_INVALID_ARG;
  if (p->student == KD_STUDENT_LOGITS && !in->logits_s) return KD_ERR_INVALID_ARG;
  switch (p->teacher) {
    case KD_TEACHER_TIED:
      if (!in->h_t) return KD_ERR_INVALID_ARG;
      break;
    case KD_TEACHER_SEPARATE:
      if (!in->h_t || !in->w_t) return KD_ERR_INVALID_ARG;
      break;
    case KD_TEACHER_LOGITS:
      if (!in->logits_t) return KD_ERR_INVALID_ARG;
      break;
    case KD_TEACHER_TOPK:
      if (!in->topk_idx || !in->topk_p) return KD_ERR_INVALID_ARG;
      break;
    case KD_TEACHER_PROJECTED:
      if (!in->logits_t || !in->token_map) return KD_ERR_INVALID_ARG;
      break;
    default:
      break;
  }
  // CE needs labels (flash_kd: per-token CE against ground-truth labels)
  if (!in->labels && (p->w_student_ce != 0.f || p->w_teacher_ce != 0.f)) return KD_ERR_INVALID_ARG;
  return KD_OK;
}

// Host copy of the constants the kernels use.
Consts make_consts(const kd_problem* p, bool has_labels, bool has_t) {
  Consts c;
  c.inv_ts = 1.f / p->t_student;
  c.inv_tt = 1.f / p->t_teacher;
  c.k_s1 = kL2E;
  c.k_sT = kL2E / p->t_student;
  c.k_t1 = kL2E;
  c.k_tT = kL2E / p->t_teacher;
  c.beta = p->beta;
  const float b = (p->beta > 0.f && p->beta < 1.f) ? p->beta : 0.5f;
  c.log_b = std::log(b);
  c.log_1mb = std::log1p(-b);
  c.need_s1 = has_labels ? 1 : 0;
  c.need_t1 = (has_labels && has_t) ? 1 : 0;
  c.kl_mode = 0;
  if (has_t) {
    if (p->variant == KD_KL_FORWARD) c.kl_mode = 1;
    else if (p->variant == KD_KL_REVERSE) c.kl_mode = 2;
    else if (p->variant == KD_KL_JEFFREYS) c.kl_mode = 3;
    else c.kl_mode = 1;  // skew variants: forward sums give the accurate normaliser gap
  }
  c.precise = p->dtype == KD_FP32 ? 1 : 0;
  // exact shortcuts for the T = 1 sums when the temperature is 1 or 2 (both sides)
  const int pw_s = p->t_student == 1.f ? 1 : (p->t_student == 2.f ? 2 : 0);
  const int pw_t = p->t_teacher == 1.f ? 1 : (p->t_teacher == 2.f ? 2 : 0);
  c.pw = (!has_t || pw_s == pw_t) ? pw_s : 0;
  return c;
}

// Forward vocabulary split: m_tiles * splits items spread over the persistent
// CTAs with the smallest makespan in tiles (plus a small per-item cost for the
// partial record).
int choose_splits(int64_t m_tiles, int64_t n_tiles, int nsm) {
  int best = 1;
  double best_cost = 1e300;
  const int64_t max_s = std::min<int64_t>(n_tiles, 4096);
  for (int64_t s = 1; s <= max_s; ++s) {
    const int64_t items = m_tiles * s;
    const double waves = (double)cdiv(items, nsm);
    const double cost = waves * (double)cdiv(n_tiles, s) + 0.02 * waves;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = (int)s;
    }
  }
  return best;
}

// Backward chunk (R rows x C columns of G).  Cost model in bytes: every extra
// vocabulary chunk re-reads and re-writes the fp32 dH accumulator, every extra
// row chunk the fp32 dW accumulator, plus a fixed cost per chunk.  A chunk
// holds at most budget_elems elements and never more than N*V/8, so no
// (tokens x vocab) matrix is ever allocated.
void choose_chunk(const kd_problem* p, int64_t budget_elems, int64_t col_quant, int64_t cap_div,
                  int64_t& R, int64_t& C) {
  const int64_t n = std::max<int64_t>(p->n_tokens, 1), v = p->vocab;
  const int64_t d = p->student == KD_STUDENT_HIDDEN ? p->d_student : 1;
  const int64_t cap =
      std::max<int64_t>(col_quant * 128, std::min<int64_t>(budget_elems, n * v / cap_div));
  int64_t best_r = 128, best_c = col_quant;
  double best = 1e300;
  for (int64_t r = round_up(n, 128);; r = round_up(r / 2, 128)) {
    int64_t rr = p->seq_chunk > 0 ? round_up(p->seq_chunk, 128) : r;
    int64_t c = std::min<int64_t>(round_up(v, col_quant), cap / rr / col_quant * col_quant);
    if (c < col_quant) c = col_quant;
    if (p->vocab_chunk > 0) c = round_up(p->vocab_chunk, col_quant);
    const int64_t nr = cdiv(n, rr), nc = cdiv(v, c);
    const double cost = (nc > 1 ? (double)nc * n * d * 8.0 : 0.0) +
                        (nr > 1 ? (double)nr * v * d * 8.0 : 0.0) + (double)nr * nc * 1.5e8;
    if (cost < best) {
      best = cost;
      best_r = rr;
      best_c = c;
    }
    if (p->seq_chunk > 0 || r <= 128) break;
  }
  R = std::min<int64_t>(best_r, round_up(n, 128));
  C = std::min<int64_t>(best_c, round_up(v, col_quant));
  // same number of chunks, sizes evened out (no small last chunk)
  if (p->seq_chunk <= 0) R = std::min(R, round_up(cdiv(n, cdiv(n, R)), 128));
  if (p->vocab_chunk <= 0) C = std::min(C, round_up(cdiv(v, cdiv(v, C)), col_quant));
}

kd_status make_plan(const kd_problem* p, bool has_labels, Plan& P) {
  memset(&P, 0, sizeof(P));
  P.n = p->n_tokens;
  P.v = p->vocab;
  P.is_bf16 = p->dtype == KD_BF16;
  P.s_gemm = p->student == KD_STUDENT_HIDDEN;
  P.s_logits = !P.s_gemm;
  P.t_gemm = p->teacher == KD_TEACHER_TIED || p->teacher == KD_TEACHER_SEPARATE;
  P.t_logits = p->teacher == KD_TEACHER_LOGITS;
  const bool proj = p->teacher == KD_TEACHER_PROJECTED;
  P.topk = p->teacher == KD_TEACHER_TOPK;
  P.tied = p->teacher == KD_TEACHER_TIED;
  P.has_t = P.t_gemm || P.t_logits || proj;
  P.ds = P.s_gemm ? p->d_student : 0;
  P.dt = p->teacher == KD_TEACHER_TIED ? p->d_student
         : p->teacher == KD_TEACHER_SEPARATE ? p->d_teacher
                                             : 0;
  if (proj) {  // the projected distribution enters the loss at temperature 1
    kd_problem q = *p;
    q.t_teacher = 1.f;
    P.c = make_consts(&q, has_labels, true);
  } else {
    P.c = make_consts(p, has_labels, P.has_t);
  }
  P.nsm = std::max(1, tc_num_sms());
  if (proj) P.path = PATH_PROJ;
  else if (!P.s_gemm && !P.t_gemm) P.path = PATH_STREAM;
  else if (!P.is_bf16) P.path = PATH_SIMT;
  else P.path = PATH_TC;
  if (P.path == PATH_TC) {
    // TMA: row pitches must be multiples of 16 bytes
    if ((P.s_gemm && P.ds % 8) || (P.t_gemm && P.dt % 8)) return KD_ERR_UNSUPPORTED;
  }
  if (P.path == PATH_SIMT && P.s_logits) return KD_ERR_UNSUPPORTED;  // fp32 logits + GEMM teacher
  const int64_t n = P.n, v = P.v;
  // ---- forward
  Layout f;
  P.f_count = f.take(16);
  P.f_ce_s = f.take(n * 4);
  P.f_ce_t = f.take(n * 4);
  P.f_kl = f.take(n * 4);
  P.f_stats = f.take(n * KD_STATS_PER_TOKEN * 4);
  if (P.topk) {
    P.f_sidx = f.take(n * p->topk * 4);
    P.f_sp = f.take(n * p->topk * 4);
    P.f_mass = f.take(n * 4);
    P.f_ent = f.take(n * 4);
  }
  if (P.path == PATH_TC) {
    const bool pair = tc_use_pairs();
    const int bn = tc_fused_tile_cols(P.s_gemm && P.t_gemm, pair);
    const int rows = tc_tile_rows(pair);
    P.n_splits = choose_splits(cdiv(std::max<int64_t>(n, 1), rows), cdiv(v, bn),
                               pair ? std::max(1, P.nsm / 2) : P.nsm);
    P.n_parts = 2 * P.n_splits;
  } else if (P.path == PATH_SIMT) {
    const int64_t mt = cdiv(std::max<int64_t>(n, 1), 32), nt = cdiv(v, 64);
    P.n_splits = (int)std::max<int64_t>(1, std::min<int64_t>(nt, cdiv(4 * P.nsm, mt)));
    P.n_parts = P.n_splits;
  }
  if (P.n_parts) P.f_part = f.take((size_t)P.n_parts * n * kRec * 4);
  if (proj) P.f_proj = f.take(proj_loss_workspace_bytes(p->vocab_teacher, v));
  P.f_bytes = f.off;
  // ---- backward
  Layout b;
  P.b_count = b.take(16);
  P.b_scale = b.take(n * 4);
  if (P.topk) {
    P.b_sidx = b.take(n * p->topk * 4);
    P.b_sp = b.take(n * p->topk * 4);
    P.b_mass = b.take(n * 4);
    P.b_ent = b.take(n * 4);
  }
  if (P.path == PATH_TC) {
    // Two bf16 gradient chunks (the producer fills one while the GEMMs read
    // the other), each at most N*V/4 elements (N*V/8 with a tied teacher-CE
    // chunk beside it): never more than half a bf16 (tokens x vocab) matrix.
    // a teacher-CE gradient chunk G_t: into d W_s for a tied teacher, and
    // for d H_t / d W_t when those are requested (tied or separate teachers)
    const bool tce = P.t_gemm && p->w_teacher_ce != 0.f && (P.tied || p->teacher_grads);
    choose_chunk(p, (int64_t)64 << 20, 256, tce ? 8 : 4, P.R, P.C);
    if (P.s_gemm) {
      // The tensor cores read an MN-major B operand about 6 % slower than a
      // K-major one.  Transposing W and H once per backward moves
      // 4 D (V + N) bytes against that 6 % of 4 N V D GEMM FLOPs, so it pays
      // when N V / (N + V) is large (measured on GB300: 3.6k -> read W and H
      // as stored, 27k -> transpose).
      P.kmajor_b = (double)n * v / (double)(n + v) > 4096.0;
      if (const char* e = getenv("KD_TC_KMAJOR_B")) P.kmajor_b = e[0] == '1';  // debug override
      P.two_streams = true;
      P.ldv = round_up(v, 8);
      P.ldn = round_up(n, 8);
      if (P.kmajor_b) {
        P.b_wt = b.take(P.ds * P.ldv * 2);            // W_s^T (B operand of dH)
        P.b_hst = b.take(P.ds * P.ldn * 2);           // H_s^T (B operand of dW)
        if (tce && P.tied) P.b_htt = b.take(P.ds * P.ldn * 2);  // H_t^T
      }
      P.b_g = b.take(2 * P.R * P.C * 2);
      if (tce) P.b_gt = b.take(2 * P.R * P.C * 2);
      if (cdiv(v, P.C) > 1) P.b_dh = b.take(n * P.ds * 4);
      if (cdiv(n, P.R) > 1) P.b_dw = b.take(v * P.ds * 4);
      // fp32 accumulators of d H_t (over vocab chunks) and d W_t (over token chunks)
      if (tce && cdiv(v, P.C) > 1) P.b_dht = b.take(n * P.dt * 4);
      if (tce && !P.tied && cdiv(n, P.R) > 1) P.b_dwt = b.take(v * P.dt * 4);
    }
  } else if (P.path == PATH_SIMT) {
    choose_chunk(p, (int64_t)8 << 20, 64, 8, P.R, P.C);
    P.b_g = b.take(P.R * P.C * 4);
    if (P.tied || (P.t_gemm && p->teacher_grads))
      P.b_gt = b.take(P.R * P.C * 4);  // teacher-CE gradient tile
  }
  if (proj) P.b_proj = b.take(proj_loss_workspace_bytes(p->vocab_teacher, v));
  P.b_bytes = b.off;
  return KD_OK;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

kd_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KD_OK : KD_ERR_CUDA; }

// Per-device side stream and events of the backward's two-stream schedule
// (created once per device, never freed: they live as long as the process).
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, ready[2] = {}, consumed[2] = {};
};

kd_status side_stream(SideStream** out) {
  static SideStream per_dev[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  SideStream& ss = per_dev[dev];
  if (!ss.stream) {
    const unsigned f = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.fork, f) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, f) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.ready[0], f) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.ready[1], f) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.consumed[0], f) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.consumed[1], f) != cudaSuccess) {
      ss.stream = nullptr;
      return KD_ERR_CUDA;
    }
  }
  *out = &ss;
  return KD_OK;
}

}  // namespace

extern "C" {

int kd_abi_version(void) { return KD_ABI_VERSION; }

const char* kd_status_string(kd_status s) {
  switch (s) {
    case KD_OK: return "ok";
    case KD_ERR_INVALID_ARG: return "invalid argument";
    case KD_ERR_UNSUPPORTED: return "unsupported combination or layout";
    case KD_ERR_WORKSPACE: return "workspace missing or too small";
    case KD_ERR_BAD_LABEL: return "label outside [0, vocab) that is not ignore_index";
    case KD_ERR_BAD_TOPK: return "top-K id outside [0, vocab) or repeated in a row";
    case KD_ERR_TIMEOUT: return "a bounded device wait timed out";
    case KD_ERR_CUDA: return "CUDA error";
    case KD_ERR_NO_DEVICE: return "no supported (sm_103) CUDA device";
  }
  return "unknown status";
}

int kd_device_supported(int device) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess)
    return 0;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
    return 0;
  return (major == 10 && minor == 3) ? 1 : 0;
}

}  // extern "C"

namespace {
kd_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KD_ERR_NO_DEVICE;
  return kd_device_supported(dev) ? KD_OK : KD_ERR_NO_DEVICE;
}
}  // namespace

extern "C" {

kd_status kd_workspace_size(const kd_problem* problem, size_t* fwd_bytes, size_t* bwd_bytes) {
  kd_status st = check_problem(problem);
  if (st != KD_OK) return st;
  Plan P;
  st = make_plan(problem, true, P);
  if (st != KD_OK) return st;
  if (fwd_bytes) *fwd_bytes = P.f_bytes;
  if (bwd_bytes) *bwd_bytes = P.b_bytes;
  return KD_OK;
}

kd_status kd_plan_info(const kd_problem* problem, int32_t* path, int32_t* vocab_splits,
                       int64_t* chunk_rows, int64_t* chunk_cols) {
  kd_status st = check_problem(problem);
  if (st != KD_OK) return st;
  Plan P;
  st = make_plan(problem, true, P);
  if (st != KD_OK) return st;
  if (path) *path = (int32_t)P.path;
  if (vocab_splits) *vocab_splits = P.n_splits;
  if (chunk_rows) *chunk_rows = P.R;
  if (chunk_cols) *chunk_cols = P.C;
  return KD_OK;
}

kd_status kd_fwd(const kd_problem* problem, const kd_inputs* in, float* ce_s, float* ce_t,
                 float* kl, float* stats, float* loss, uint32_t* dev_status, void* workspace,
                 size_t ws_bytes, void* stream_) {
  kd_status st = check_problem(problem);
  if (st != KD_OK) return st;
  st = check_inputs(problem, in);
  if (st != KD_OK) return st;
  const kd_problem* p = problem;
  Plan P;
  st = make_plan(p, in->labels != nullptr, P);
  if (st != KD_OK) return st;
  if (!workspace || ws_bytes < P.f_bytes || (reinterpret_cast<uintptr_t>(workspace) % kAlign))
    return KD_ERR_WORKSPACE;
  st = check_device();
  if (st != KD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  const int64_t n = P.n;
  float* w_ce_s = ce_s ? ce_s : at<float>(workspace, P.f_ce_s);
  float* w_ce_t = ce_t ? ce_t : at<float>(workspace, P.f_ce_t);
  float* w_kl = kl ? kl : at<float>(workspace, P.f_kl);
  float* w_stats = stats ? stats : at<float>(workspace, P.f_stats);
  int32_t* count = at<int32_t>(workspace, P.f_count);
  if (n == 0) {
    if (loss && cudaMemsetAsync(loss, 0, sizeof(float), s) != cudaSuccess) return KD_ERR_CUDA;
    return KD_OK;
  }
  if (cudaMemsetAsync(count, 0, 16, s) != cudaSuccess) return KD_ERR_CUDA;
  if (in->labels) launch_label_check(in->labels, n, P.v, p->ignore_index, count, dev_status, s);
  int32_t* sidx = nullptr;
  float *sp = nullptr, *mass = nullptr, *ent = nullptr;
  if (P.topk) {
    sidx = at<int32_t>(workspace, P.f_sidx);
    sp = at<float>(workspace, P.f_sp);
    mass = at<float>(workspace, P.f_mass);
    ent = at<float>(workspace, P.f_ent);
    launch_topk_prep(in->topk_idx, in->topk_p, n, (int)p->topk, P.v, sidx, sp, mass, ent,
                     dev_status, s);
  }
  const bool js = P.has_t && is_skew(p->variant);
  if (P.path == PATH_PROJ) {
    ProjLossArgs a;
    memset(&a, 0, sizeof(a));
    a.token_map = in->token_map;
    a.zt = in->logits_t;
    a.zs = in->logits_s;
    a.n = n;
    a.vt = p->vocab_teacher;
    a.vs = P.v;
    a.is_bf16 = P.is_bf16;
    a.inv_tp = 1.f / p->t_teacher;
    a.c = P.c;
    a.variant = p->variant;
    a.labels = in->labels;
    a.ignore = p->ignore_index;
    a.ce_s = w_ce_s;
    a.ce_t = w_ce_t;
    a.kl = w_kl;
    a.stats = w_stats;
    a.mode = 0;
    a.status = dev_status;
    prof_record(0, s);
    if (launch_proj_loss(a, at<char>(workspace, P.f_proj), s)) return KD_ERR_CUDA;
    prof_record(1, s);
  } else if (P.path == PATH_STREAM) {
    StreamArgs a;
    memset(&a, 0, sizeof(a));
    a.zs = in->logits_s;
    a.zt = P.t_logits ? in->logits_t : nullptr;
    a.n = n;
    a.vocab = P.v;
    a.c = P.c;
    a.variant = p->variant;
    a.is_bf16 = P.is_bf16;
    a.topk = P.topk;
    a.k = (int)p->topk;
    a.sidx = sidx;
    a.sp = sp;
    a.mass = mass;
    a.ent = ent;
    a.labels = in->labels;
    a.ignore = p->ignore_index;
    a.ce_s = w_ce_s;
    a.ce_t = w_ce_t;
    a.kl = w_kl;
    a.stats = w_stats;
    a.status = dev_status;
    // test hooks of the ring kernels: a shorter wait limit and one withheld
    // consumer release (tests of the bounded-wait timeout path)
    if (const char* e = getenv("KD_TEST_WAIT_LIMIT_NS")) a.wait_limit_ns = strtoull(e, nullptr, 10);
    if (const char* e = getenv("KD_TEST_WITHHOLD_RELEASE")) a.debug_withhold_release = e[0] == '1';
    prof_record(0, s);
    launch_stream_fwd(a, s);
    prof_record(1, s);
  } else {
    float* part = at<float>(workspace, P.f_part);
    CombineArgs cb;
    memset(&cb, 0, sizeof(cb));
    cb.partials = part;
    cb.n_parts = P.n_parts;
    cb.n = n;
    cb.vocab = P.v;
    cb.c = P.c;
    cb.variant = p->variant;
    cb.has_t = P.has_t;
    cb.topk = P.topk;
    cb.labels = in->labels;
    cb.ignore = p->ignore_index;
    cb.mass = mass;
    cb.ent = ent;
    cb.ce_s = w_ce_s;
    cb.ce_t = w_ce_t;
    cb.kl = w_kl;
    cb.stats = w_stats;
    for (int pass = 0; pass < (js ? 2 : 1); ++pass) {
      if (pass == 0) prof_record(0, s);
      if (P.path == PATH_SIMT) {
        SimtArgs a;
        memset(&a, 0, sizeof(a));
        a.h_s = static_cast<const float*>(in->h_s);
        a.w_s = static_cast<const float*>(in->w_s);
        a.h_t = static_cast<const float*>(in->h_t);
        a.w_t = static_cast<const float*>(in->w_t);
        a.zt = static_cast<const float*>(in->logits_t);
        a.n = n;
        a.vocab = P.v;
        a.d_s = P.ds;
        a.d_t = P.dt;
        a.teacher = p->teacher;
        a.c = P.c;
        a.variant = p->variant;
        a.labels = in->labels;
        a.ignore = p->ignore_index;
        a.sidx = sidx;
        a.sp = sp;
        a.k = (int)p->topk;
        a.n_splits = P.n_splits;
        a.partials = part;
        a.stats = w_stats;
        a.js_pass = pass;
        launch_simt_fwd(a, s);
      } else {
        TcFwdArgs a;
        memset(&a, 0, sizeof(a));
        a.h_s = in->h_s;
        a.w_s = in->w_s;
        a.h_t = in->h_t;
        a.w_t = p->teacher == KD_TEACHER_SEPARATE ? in->w_t : nullptr;
        a.zs_logits = P.s_logits ? in->logits_s : nullptr;
        a.zt_logits = P.t_logits ? in->logits_t : nullptr;
        a.n = n;
        a.vocab = P.v;
        a.d_s = P.ds;
        a.d_t = P.dt;
        a.s_gemm = P.s_gemm;
        a.t_gemm = P.t_gemm;
        a.s_logits = P.s_logits;
        a.t_logits = P.t_logits;
        a.topk = P.topk;
        a.c = P.c;
        a.variant = p->variant;
        a.labels = in->labels;
        a.ignore = p->ignore_index;
        a.sidx = sidx;
        a.sp = sp;
        a.k = (int)p->topk;
        a.n_splits = P.n_splits;
        a.partials = part;
        a.stats = w_stats;
        a.js_pass = pass;
        a.status = dev_status;
        if (launch_tc_fwd(a, P.nsm, s) != 0) return KD_ERR_CUDA;
      }
      if (pass == (js ? 1 : 0)) prof_record(1, s);
      cb.js_pass = pass;
      launch_combine(cb, s);
    }
  }
  if (loss) {
    ReduceArgs r;
    memset(&r, 0, sizeof(r));
    r.ce_s = w_ce_s;
    r.ce_t = w_ce_t;
    r.kl = w_kl;
    r.labels = in->labels;
    r.n = n;
    r.ignore = p->ignore_index;
    r.w_sce = p->w_student_ce;
    r.w_tce = P.has_t ? p->w_teacher_ce : 0.f;
    r.w_kl_t2 = (P.has_t || P.topk) ? p->w_kl * p->t_student * p->t_student : 0.f;
    r.reduction = p->reduction;
    r.num_batch_labels = p->num_batch_labels;
    r.count = count;
    r.loss = loss;
    launch_loss_reduce(r, s);
  }
  return cuda_status(cudaGetLastError());
}

static kd_status bwd_impl(const kd_problem* problem, const kd_inputs* in, const float* stats,
                          const float* d_loss, float grad_scale, void* d_h_s, void* d_w_s,
                          void* d_logits_s, void* d_h_t, void* d_w_t, uint32_t* dev_status,
                          void* workspace, size_t ws_bytes, void* stream_) {
  kd_status st = check_problem(problem);
  if (st != KD_OK) return st;
  st = check_inputs(problem, in);
  if (st != KD_OK) return st;
  const kd_problem* p = problem;
  if (!std::isfinite(grad_scale)) return KD_ERR_INVALID_ARG;
  if (p->student == KD_STUDENT_HIDDEN && d_logits_s) return KD_ERR_INVALID_ARG;
  if (p->student == KD_STUDENT_LOGITS && (d_h_s || d_w_s)) return KD_ERR_INVALID_ARG;
  // teacher gradients: hidden student, tied / separate teacher, workspace
  // sized for them; d W_t only for a separate teacher (a tied teacher's
  // weight is W_s, whose gradient d_w_s carries)
  if ((d_h_t || d_w_t) &&
      (p->student != KD_STUDENT_HIDDEN || !p->teacher_grads ||
       (p->teacher != KD_TEACHER_TIED && p->teacher != KD_TEACHER_SEPARATE) ||
       (d_w_t && p->teacher != KD_TEACHER_SEPARATE)))
    return KD_ERR_INVALID_ARG;
  Plan P;
  st = make_plan(p, in->labels != nullptr, P);
  if (st != KD_OK) return st;
  if (!d_h_s && !d_w_s && !d_logits_s && !d_h_t && !d_w_t) return KD_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  const size_t esz = P.is_bf16 ? 2 : 4;
  // no tokens (or a teacher CE weight of 0): the weight / teacher gradients
  // are zero, written as such
  const bool no_tce = p->w_teacher_ce == 0.f;
  if (P.n == 0 || (no_tce && (d_h_t || d_w_t))) {
    st = check_device();
    if (st != KD_OK) return st;
    if (P.n == 0 && d_w_s && cudaMemsetAsync(d_w_s, 0, (size_t)P.v * P.ds * esz, s) != cudaSuccess)
      return KD_ERR_CUDA;
    if (d_w_t && cudaMemsetAsync(d_w_t, 0, (size_t)P.v * P.dt * esz, s) != cudaSuccess)
      return KD_ERR_CUDA;
    if (d_h_t && P.n > 0 &&
        cudaMemsetAsync(d_h_t, 0, (size_t)P.n * P.dt * esz, s) != cudaSuccess)
      return KD_ERR_CUDA;
    d_h_t = d_w_t = nullptr;
    if (P.n == 0 || (!d_h_s && !d_w_s && !d_logits_s)) return KD_OK;
  }
  if (!stats) return KD_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < P.b_bytes || (reinterpret_cast<uintptr_t>(workspace) % kAlign))
    return KD_ERR_WORKSPACE;
  st = check_device();
  if (st != KD_OK) return st;
  const int64_t n = P.n, v = P.v;
  int32_t* count = at<int32_t>(workspace, P.b_count);
  float* scale = at<float>(workspace, P.b_scale);
  if (cudaMemsetAsync(count, 0, 16, s) != cudaSuccess) return KD_ERR_CUDA;
  if (in->labels) launch_label_check(in->labels, n, v, p->ignore_index, count, dev_status, s);
  launch_row_scale(in->labels, n, p->ignore_index, grad_scale, d_loss, p->reduction,
                   p->num_batch_labels, count, scale, s);
  int32_t* sidx = nullptr;
  float *sp = nullptr, *mass = nullptr, *ent = nullptr;
  if (P.topk) {
    sidx = at<int32_t>(workspace, P.b_sidx);
    sp = at<float>(workspace, P.b_sp);
    mass = at<float>(workspace, P.b_mass);
    ent = at<float>(workspace, P.b_ent);
    launch_topk_prep(in->topk_idx, in->topk_p, n, (int)p->topk, v, sidx, sp, mass, ent,
                     dev_status, s);
  }
  const float w_kl_ts = (P.has_t || P.topk) ? p->w_kl * p->t_student : 0.f;
  // the teacher-CE gradient chunk G_t is made when something consumes it
  const float w_tce = ((P.tied && d_w_s) || d_h_t || d_w_t) ? p->w_teacher_ce : 0.f;
  const bool tied_tce = P.tied && d_w_s && w_tce != 0.f;  // G_t^T H_t into d W_s
  const void* w_teach = P.tied ? in->w_s : in->w_t;      // the teacher's head weight
  if (P.path == PATH_PROJ) {
    if (!d_logits_s) return cuda_status(cudaGetLastError());
    ProjLossArgs a;
    memset(&a, 0, sizeof(a));
    a.token_map = in->token_map;
    a.zt = in->logits_t;
    a.zs = in->logits_s;
    a.n = n;
    a.vt = p->vocab_teacher;
    a.vs = v;
    a.is_bf16 = P.is_bf16;
    a.inv_tp = 1.f / p->t_teacher;
    a.c = P.c;
    a.variant = p->variant;
    a.labels = in->labels;
    a.ignore = p->ignore_index;
    a.stats = const_cast<float*>(stats);  // read only by the backward
    a.row_scale = scale;
    a.w_sce = p->w_student_ce;
    a.w_kl_ts = w_kl_ts;
    a.dz = d_logits_s;
    a.mode = 1;
    a.status = dev_status;
    prof_record(2, s);
    if (launch_proj_loss(a, at<char>(workspace, P.b_proj), s)) return KD_ERR_CUDA;
    prof_record(3, s);
    return cuda_status(cudaGetLastError());
  }
  if (P.path == PATH_STREAM) {
    StreamArgs a;
    memset(&a, 0, sizeof(a));
    a.zs = in->logits_s;
    a.zt = P.t_logits ? in->logits_t : nullptr;
    a.n = n;
    a.vocab = v;
    a.c = P.c;
    a.variant = p->variant;
    a.is_bf16 = P.is_bf16;
    a.topk = P.topk;
    a.k = (int)p->topk;
    a.sidx = sidx;
    a.sp = sp;
    a.labels = in->labels;
    a.ignore = p->ignore_index;
    a.stats = const_cast<float*>(stats);
    a.row_scale = scale;
    a.w_sce = p->w_student_ce;
    a.w_kl_ts = w_kl_ts;
    a.dz = d_logits_s;
    a.status = dev_status;
    prof_record(2, s);
    launch_stream_bwd(a, s);
    prof_record(3, s);
    return cuda_status(cudaGetLastError());
  }
  const int64_t R = P.R, C = P.C;
  const int64_t nr = cdiv(n, R), nc = cdiv(v, C);
  if (P.path == PATH_SIMT) {
    float* g = at<float>(workspace, P.b_g);
    float* gt = w_tce != 0.f ? at<float>(workspace, P.b_gt) : nullptr;
    const int64_t D = P.ds;
    prof_record(2, s);
    for (int64_t ri = 0; ri < nr; ++ri) {
      const int64_t r0 = ri * R, rc = std::min(R, n - r0);
      for (int64_t ci = 0; ci < nc; ++ci) {
        const int64_t c0 = ci * C, cc = std::min(C, v - c0);
        SimtArgs a;
        memset(&a, 0, sizeof(a));
        a.h_s = static_cast<const float*>(in->h_s);
        a.w_s = static_cast<const float*>(in->w_s);
        a.h_t = static_cast<const float*>(in->h_t);
        a.w_t = static_cast<const float*>(in->w_t);
        a.zt = static_cast<const float*>(in->logits_t);
        a.n = n;
        a.vocab = v;
        a.d_s = P.ds;
        a.d_t = P.dt;
        a.teacher = p->teacher;
        a.c = P.c;
        a.variant = p->variant;
        a.labels = in->labels;
        a.ignore = p->ignore_index;
        a.sidx = sidx;
        a.sp = sp;
        a.k = (int)p->topk;
        a.stats = stats;
        a.r0 = r0;
        a.rc = rc;
        a.c0 = c0;
        a.cc = cc;
        a.row_scale = scale;
        a.w_sce = p->w_student_ce;
        a.w_tce = w_tce;
        a.w_kl_ts = w_kl_ts;
        a.g = g;
        a.gt = gt;
        launch_simt_gprod(a, s);
        const float* W = static_cast<const float*>(in->w_s);
        const float* H = static_cast<const float*>(in->h_s);
        if (d_h_s)  // dH[r0.., :] (+)= G W[c0.., :]
          launch_simt_gemm(g, cc, 1, W + c0 * D, D, 1, static_cast<float*>(d_h_s) + r0 * D, D,
                           rc, D, cc, ci > 0, s);
        if (d_w_s) {  // dW[c0.., :] (+)= G^T H[r0.., :]
          float* dw = static_cast<float*>(d_w_s) + c0 * D;
          launch_simt_gemm(g, 1, cc, H + r0 * D, D, 1, dw, D, cc, D, rc, ri > 0, s);
          if (gt && tied_tce)
            launch_simt_gemm(gt, 1, cc, static_cast<const float*>(in->h_t) + r0 * D, D, 1, dw, D,
                             cc, D, rc, true, s);
        }
        const int64_t Dt = P.dt;
        if (gt && d_h_t)  // dH_t[r0.., :] (+)= G_t W_t[c0.., :]
          launch_simt_gemm(gt, cc, 1, static_cast<const float*>(w_teach) + c0 * Dt, Dt, 1,
                           static_cast<float*>(d_h_t) + r0 * Dt, Dt, rc, Dt, cc, ci > 0, s);
        if (gt && d_w_t)  // dW_t[c0.., :] (+)= G_t^T H_t[r0.., :]
          launch_simt_gemm(gt, 1, cc, static_cast<const float*>(in->h_t) + r0 * Dt, Dt, 1,
                           static_cast<float*>(d_w_t) + c0 * Dt, Dt, cc, Dt, rc, ri > 0, s);
      }
    }
    prof_record(3, s);
    return cuda_status(cudaGetLastError());
  }
  // ---------------------------------------------------------------- tcgen05
  const int64_t D = P.ds;
  __nv_bfloat16* g = P.s_gemm ? at<__nv_bfloat16>(workspace, P.b_g) : nullptr;
  __nv_bfloat16* gt = (w_tce != 0.f && P.s_gemm) ? at<__nv_bfloat16>(workspace, P.b_gt) : nullptr;
  const bool kb = P.s_gemm && P.kmajor_b;
  __nv_bfloat16* wT = (kb && d_h_s) ? at<__nv_bfloat16>(workspace, P.b_wt) : nullptr;
  __nv_bfloat16* hsT = (kb && d_w_s) ? at<__nv_bfloat16>(workspace, P.b_hst) : nullptr;
  __nv_bfloat16* htT = (kb && tied_tce) ? at<__nv_bfloat16>(workspace, P.b_htt) : nullptr;
  if (wT)
    launch_transpose_bf16(static_cast<const __nv_bfloat16*>(in->w_s), v, D, D, wT, P.ldv, s);
  if (hsT)
    launch_transpose_bf16(static_cast<const __nv_bfloat16*>(in->h_s), n, D, D, hsT, P.ldn, s);
  if (htT)
    launch_transpose_bf16(static_cast<const __nv_bfloat16*>(in->h_t), n, D, D, htT, P.ldn, s);
  float* dh_acc = (P.s_gemm && nc > 1) ? at<float>(workspace, P.b_dh) : nullptr;
  float* dw_acc = (P.s_gemm && nr > 1) ? at<float>(workspace, P.b_dw) : nullptr;
  float* dht_acc = (d_h_t && nc > 1) ? at<float>(workspace, P.b_dht) : nullptr;
  float* dwt_acc = (d_w_t && nr > 1) ? at<float>(workspace, P.b_dwt) : nullptr;
  prof_record(2, s);
  // Two-stream schedule: gradient chunk k is produced on the caller's stream
  // into buffer k%2 while the dH / dW GEMMs of chunk k-1 run on a side
  // stream, so each launch's last partial wave overlaps the next launch.
  SideStream* ss = nullptr;
  cudaStream_t s2 = s;
  const char* env_streams = getenv("KD_BWD_STREAMS");  // debug override: 1 = one stream
  const bool two_streams = (P.two_streams && !(env_streams && env_streams[0] == '1')) ||
                           (env_streams && env_streams[0] == '2');
  if (!P.s_logits && two_streams) {
    if (side_stream(&ss) != KD_OK) return KD_ERR_CUDA;
    s2 = ss->stream;
    if (cudaEventRecord(ss->fork, s) != cudaSuccess ||
        cudaStreamWaitEvent(s2, ss->fork, 0) != cudaSuccess)
      return KD_ERR_CUDA;
  }
  int64_t k = 0;
  for (int64_t ri = 0; ri < nr; ++ri) {
    const int64_t r0 = ri * R, rc = std::min(R, n - r0);
    for (int64_t ci = 0; ci < nc; ++ci, ++k) {
      const int64_t c0 = ci * C, cc = std::min(C, v - c0);
      const int buf = (int)(k & 1);
      __nv_bfloat16* gk = g ? g + (size_t)buf * R * C : nullptr;
      __nv_bfloat16* gtk = gt ? gt + (size_t)buf * R * C : nullptr;
      if (ss && k >= 2 && cudaStreamWaitEvent(s, ss->consumed[buf], 0) != cudaSuccess)
        return KD_ERR_CUDA;
      TcGradArgs a;
      memset(&a, 0, sizeof(a));
      a.h_s = in->h_s;
      a.w_s = in->w_s;
      a.h_t = in->h_t;
      a.w_t = p->teacher == KD_TEACHER_SEPARATE ? in->w_t : nullptr;
      a.zs_logits = P.s_logits ? in->logits_s : nullptr;
      a.zt_logits = P.t_logits ? in->logits_t : nullptr;
      a.n = n;
      a.vocab = v;
      a.d_s = P.ds;
      a.d_t = P.dt;
      a.s_gemm = P.s_gemm;
      a.s_logits = P.s_logits;
      a.t_gemm = P.t_gemm;
      a.t_logits = P.t_logits;
      a.topk = P.topk;
      a.c = P.c;
      a.variant = p->variant;
      a.labels = in->labels;
      a.ignore = p->ignore_index;
      a.sidx = sidx;
      a.sp = sp;
      a.k = (int)p->topk;
      a.stats = stats;
      a.row_scale = scale;
      a.w_sce = p->w_student_ce;
      a.w_tce = w_tce;
      a.w_kl_ts = w_kl_ts;
      a.r0 = r0;
      a.rc = rc;
      a.c0 = c0;
      a.cc = cc;
      if (P.s_logits) {  // logit students: G is the requested d z_s itself
        a.g = static_cast<__nv_bfloat16*>(d_logits_s) + c0;
        a.ldg = v;
        a.gt = nullptr;
      } else {
        a.g = gk;
        a.ldg = C;
        a.gt = gtk;
      }
      a.status = dev_status;
      launch_record(0, k, false, s);
      if (launch_tc_grad(a, P.nsm, s) != 0) return KD_ERR_CUDA;
      launch_record(0, k, true, s);
      if (P.s_logits) continue;
      if (ss && (cudaEventRecord(ss->ready[buf], s) != cudaSuccess ||
                 cudaStreamWaitEvent(s2, ss->ready[buf], 0) != cudaSuccess))
        return KD_ERR_CUDA;
      // dW = G^T H reads G as stored, as an MN-major A (full rate): no
      // transposed copy of a gradient chunk is made.  B is W^T / H^T from the
      // transposes above, or W / H as stored (MN-major) when those don't pay.
      if (d_h_s) {  // dH[r0.., :] (+)= G[:, chunk] W[chunk, :]
        TcGemmArgs m;
        memset(&m, 0, sizeof(m));
        m.a0 = gk;
        m.lda0 = C;
        if (wT) {
          m.b0 = wT + c0;
          m.ldb0 = P.ldv;
        } else {
          m.b0 = static_cast<const __nv_bfloat16*>(in->w_s) + c0 * D;
          m.ldb0 = D;
          m.b0_mn = 1;
        }
        m.M = rc;
        m.N = D;
        m.K0 = cc;
        m.status = dev_status;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(d_h_s) + r0 * D;
        if (nc == 1) {
          m.mode = TC_OUT_BF16;
        } else {
          m.mode = ci == 0 ? TC_OUT_F32 : (ci + 1 < nc ? TC_OUT_F32_ACC : TC_OUT_F32_ACC_BF16);
          m.c32 = dh_acc + r0 * D;
          m.ldc32 = D;
        }
        m.c16 = out;
        m.ldc16 = D;
        launch_record(1, 2 * k, false, s2);
        if (launch_tc_gemm(m, P.nsm, s2) != 0) return KD_ERR_CUDA;
        launch_record(1, 2 * k, true, s2);
      }
      if (d_w_s) {  // dW[chunk, :] (+)= G[:, chunk]^T H[r0.., :] (+ G_t^T H_t)
        TcGemmArgs m;
        memset(&m, 0, sizeof(m));
        m.a0 = gk;
        m.lda0 = C;
        m.a0_mn = 1;
        if (hsT) {
          m.b0 = hsT + r0;
          m.ldb0 = P.ldn;
        } else {
          m.b0 = static_cast<const __nv_bfloat16*>(in->h_s) + r0 * D;
          m.ldb0 = D;
          m.b0_mn = 1;
        }
        m.M = cc;
        m.N = D;
        m.K0 = rc;
        if (gtk && tied_tce) {
          m.a1 = gtk;
          m.lda1 = C;
          m.a1_mn = 1;
          if (htT) {
            m.b1 = htT + r0;
            m.ldb1 = P.ldn;
          } else {
            m.b1 = static_cast<const __nv_bfloat16*>(in->h_t) + r0 * D;
            m.ldb1 = D;
            m.b1_mn = 1;
          }
          m.K1 = rc;
        }
        m.status = dev_status;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(d_w_s) + c0 * D;
        if (nr == 1) {
          m.mode = TC_OUT_BF16;
        } else {
          m.mode = ri == 0 ? TC_OUT_F32 : (ri + 1 < nr ? TC_OUT_F32_ACC : TC_OUT_F32_ACC_BF16);
          m.c32 = dw_acc + c0 * D;
          m.ldc32 = D;
        }
        m.c16 = out;
        m.ldc16 = D;
        launch_record(1, 2 * k + 1, false, s2);
        if (launch_tc_gemm(m, P.nsm, s2) != 0) return KD_ERR_CUDA;
        launch_record(1, 2 * k + 1, true, s2);
      }
      const int64_t Dt = P.dt;
      if (gtk && d_h_t) {  // dH_t[r0.., :] (+)= G_t[:, chunk] W_t[chunk, :] (W_t as stored)
        TcGemmArgs m;
        memset(&m, 0, sizeof(m));
        m.a0 = gtk;
        m.lda0 = C;
        m.b0 = static_cast<const __nv_bfloat16*>(w_teach) + c0 * Dt;
        m.ldb0 = Dt;
        m.b0_mn = 1;
        m.M = rc;
        m.N = Dt;
        m.K0 = cc;
        m.status = dev_status;
        if (nc == 1) {
          m.mode = TC_OUT_BF16;
        } else {
          m.mode = ci == 0 ? TC_OUT_F32 : (ci + 1 < nc ? TC_OUT_F32_ACC : TC_OUT_F32_ACC_BF16);
          m.c32 = dht_acc + r0 * Dt;
          m.ldc32 = Dt;
        }
        m.c16 = static_cast<__nv_bfloat16*>(d_h_t) + r0 * Dt;
        m.ldc16 = Dt;
        if (launch_tc_gemm(m, P.nsm, s2) != 0) return KD_ERR_CUDA;
      }
      if (gtk && d_w_t) {  // dW_t[chunk, :] (+)= G_t[:, chunk]^T H_t[r0.., :] (H_t as stored)
        TcGemmArgs m;
        memset(&m, 0, sizeof(m));
        m.a0 = gtk;
        m.lda0 = C;
        m.a0_mn = 1;
        m.b0 = static_cast<const __nv_bfloat16*>(in->h_t) + r0 * Dt;
        m.ldb0 = Dt;
        m.b0_mn = 1;
        m.M = cc;
        m.N = Dt;
        m.K0 = rc;
        m.status = dev_status;
        if (nr == 1) {
          m.mode = TC_OUT_BF16;
        } else {
          m.mode = ri == 0 ? TC_OUT_F32 : (ri + 1 < nr ? TC_OUT_F32_ACC : TC_OUT_F32_ACC_BF16);
          m.c32 = dwt_acc + c0 * Dt;
          m.ldc32 = Dt;
        }
        m.c16 = static_cast<__nv_bfloat16*>(d_w_t) + c0 * Dt;
        m.ldc16 = Dt;
        if (launch_tc_gemm(m, P.nsm, s2) != 0) return KD_ERR_CUDA;
      }
      if (ss && cudaEventRecord(ss->consumed[buf], s2) != cudaSuccess) return KD_ERR_CUDA;
    }
  }
  if (ss && (cudaEventRecord(ss->join, s2) != cudaSuccess ||
             cudaStreamWaitEvent(s, ss->join, 0) != cudaSuccess))
    return KD_ERR_CUDA;
  prof_record(3, s);
  return cuda_status(cudaGetLastError());
}

kd_status kd_bwd(const kd_problem* problem, const kd_inputs* in, const float* stats,
                 const float* d_loss, float grad_scale, void* d_h_s, void* d_w_s,
                 void* d_logits_s, uint32_t* dev_status, void* workspace, size_t ws_bytes,
                 void* stream) {
  return bwd_impl(problem, in, stats, d_loss, grad_scale, d_h_s, d_w_s, d_logits_s, nullptr,
                  nullptr, dev_status, workspace, ws_bytes, stream);
}

kd_status kd_bwd_grads(const kd_problem* problem, const kd_inputs* in, const float* stats,
                       const float* d_loss, float grad_scale, const kd_grads* grads,
                       uint32_t* dev_status, void* workspace, size_t ws_bytes, void* stream) {
  if (!grads) return KD_ERR_INVALID_ARG;
  return bwd_impl(problem, in, stats, d_loss, grad_scale, grads->d_h_s, grads->d_w_s,
                  grads->d_logits_s, grads->d_h_t, grads->d_w_t, dev_status, workspace, ws_bytes,
                  stream);
}

kd_status kd_set_profile_launch_events(int kind, void* const* starts, void* const* stops,
                                       int n) {
  if (kind < 0 || kind > 1 || n < 0 || (n > 0 && (!starts || !stops))) return KD_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!starts[i] || !stops[i]) return KD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_lprof_mu);
  g_lprof[kind] = LaunchEvents{n ? starts : nullptr, n ? stops : nullptr, n};
  return KD_OK;
}

kd_status kd_set_profile_events(void* fwd_start, void* fwd_stop, void* bwd_start,
                                void* bwd_stop) {
  if ((fwd_start == nullptr) != (fwd_stop == nullptr) ||
      (bwd_start == nullptr) != (bwd_stop == nullptr))
    return KD_ERR_INVALID_ARG;
  g_prof[0] = fwd_start;
  g_prof[1] = fwd_stop;
  g_prof[2] = bwd_start;
  g_prof[3] = bwd_stop;
  return KD_OK;
}

uint64_t kd_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

// Diagnostic: C[M, N] = A[M, K] B[N, K]^T on the tensor-core GEMM core.
kd_status kd_diag_gemm_bf16(const void* a, const void* b, float* c, int64_t m, int64_t n,
                            int64_t k, int layout, void* stream) {
  const int a_mn = layout & 1, b_mn = (layout >> 1) & 1;
  if (!a || !b || !c || m < 1 || n < 1 || k < 1 || (layout & ~3) || !aligned16(a) ||
      !aligned16(b) || ((a_mn ? m : k) % 8) || ((b_mn ? n : k) % 8))
    return KD_ERR_INVALID_ARG;
  kd_status st = check_device();
  if (st != KD_OK) return st;
  TcGemmArgs g;
  memset(&g, 0, sizeof(g));
  g.a0 = static_cast<const __nv_bfloat16*>(a);
  g.b0 = static_cast<const __nv_bfloat16*>(b);
  g.lda0 = a_mn ? m : k;
  g.ldb0 = b_mn ? n : k;
  g.a0_mn = a_mn;
  g.b0_mn = b_mn;
  g.M = m;
  g.N = n;
  g.K0 = k;
  g.mode = TC_OUT_F32;
  g.c32 = c;
  g.ldc32 = n;
  if (launch_tc_gemm(g, std::max(1, tc_num_sms()), static_cast<cudaStream_t>(stream)) != 0)
    return KD_ERR_CUDA;
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
