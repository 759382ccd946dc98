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
// order and the result are deterministic); then one CTA per token row takes,
// for each student id, the log-sum-exp over the teacher columns of its id,
// reading the row (resident in L2 while the CTA works on it) by gathers and
// writing the output row coalesced.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <cstring>

#include "../../include/kd.h"
#include "kd_internal.h"

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

// off[0..vs] = exclusive scan of cnt[0..vs); one block of 1024 threads, each
// summing a contiguous run, then a block scan of the run totals.
__global__ void __launch_bounds__(1024) k_map_scan(const int32_t* __restrict__ cnt, int64_t vs,
                                                   int32_t* __restrict__ off) {
  __shared__ int32_t tot[1024];
  const int t = threadIdx.x;
  const int64_t per = (vs + 1023) / 1024;
  const int64_t b = t * per, e = b + per < vs ? b + per : vs;
  int32_t s = 0;
  for (int64_t i = b; i < e; ++i) s += cnt[i];
  tot[t] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {  // inclusive Hillis-Steele scan of the totals
    const int32_t v = t >= o ? tot[t - o] : 0;
    __syncthreads();
    tot[t] += v;
    __syncthreads();
  }
  int32_t run = t > 0 ? tot[t - 1] : 0;
  for (int64_t i = b; i < e; ++i) {
    off[i] = run;
    run += cnt[i];
  }
  if (t == 1023) off[vs] = tot[1023];
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

template <typename TI, typename TO>
__global__ void __launch_bounds__(kT) k_project(const TI* __restrict__ zt, int64_t n, int64_t vt,
                                                int64_t vs, float inv_t,
                                                const int32_t* __restrict__ off,
                                                const int32_t* __restrict__ cols,
                                                TO* __restrict__ out) {
  for (int64_t row = blockIdx.x; row < n; row += gridDim.x) {
    const TI* z = zt + row * vt;
    TO* o = out + row * vs;
    for (int64_t i = threadIdx.x; i < vs; i += kT) {
      const int32_t b = off[i], e = off[i + 1];
      float r = lowest<TO>();
      if (e > b) {
        float m = ld<TI>(z + cols[b]) * inv_t;
        for (int32_t k = b + 1; k < e; ++k) m = fmaxf(m, ld<TI>(z + cols[k]) * inv_t);
        float s = 0.f;
        for (int32_t k = b; k < e; ++k) s += expf(ld<TI>(z + cols[k]) * inv_t - m);
        r = m + logf(s);
      }
      st<TO>(o + i, r);
    }
  }
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct ProjLayout {
  size_t cnt, off, cols, bytes;
};
ProjLayout proj_layout(int64_t vt, int64_t vs) {
  ProjLayout L;
  L.cnt = 0;
  L.off = align256(L.cnt + (size_t)vs * 4);
  L.cols = align256(L.off + (size_t)(vs + 1) * 4);
  L.bytes = align256(L.cols + (size_t)vt * 4);
  return L;
}

template <typename TI, typename TO>
void launch_project(const void* zt, int64_t n, int64_t vt, int64_t vs, float inv_t,
                    const int32_t* off, const int32_t* cols, void* out, int grid, cudaStream_t s) {
  note_launch();
  k_project<TI, TO><<<grid, kT, 0, s>>>(static_cast<const TI*>(zt), n, vt, vs, inv_t, off, cols,
                                        static_cast<TO*>(out));
}

}  // namespace
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
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KD_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || !kd_device_supported(dev)) return KD_ERR_NO_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const ProjLayout L = proj_layout(v_teacher, v_student);
  char* ws = static_cast<char*>(workspace);
  int32_t* cnt = reinterpret_cast<int32_t*>(ws + L.cnt);
  int32_t* off = reinterpret_cast<int32_t*>(ws + L.off);
  int32_t* cols = reinterpret_cast<int32_t*>(ws + L.cols);
  const int nsm = tc_num_sms() > 0 ? tc_num_sms() : 1;
  const int gmap = (int)std::min<int64_t>((v_teacher + kT - 1) / kT, (int64_t)nsm * 8);
  const int gid = (int)std::min<int64_t>((v_student + kT - 1) / kT, (int64_t)nsm * 8);
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
  if (n_tokens > 0) {
    const int grid = (int)std::min<int64_t>(n_tokens, (int64_t)nsm * 8);
    const float inv_t = 1.f / temperature;
    if (in_dtype == KD_BF16) {
      if (out_dtype == KD_BF16)
        launch_project<__nv_bfloat16, __nv_bfloat16>(logits_t, n_tokens, v_teacher, v_student,
                                                     inv_t, off, cols, out, grid, s);
      else
        launch_project<__nv_bfloat16, float>(logits_t, n_tokens, v_teacher, v_student, inv_t,
                                             off, cols, out, grid, s);
    } else {
      if (out_dtype == KD_BF16)
        launch_project<float, __nv_bfloat16>(logits_t, n_tokens, v_teacher, v_student, inv_t,
                                             off, cols, out, grid, s);
      else
        launch_project<float, float>(logits_t, n_tokens, v_teacher, v_student, inv_t, off, cols,
                                     out, grid, s);
    }
  }
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

}  // extern "C"
