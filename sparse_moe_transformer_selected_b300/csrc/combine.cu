// K5 — weighted unpermute-combine.
//
// out[t] = bf16( Σ_j w[t,j] · y[inv[t,j]] ): the softmax-weighted sum of the
// selected experts' outputs ("OpenAI 最新开源模型 gpt-oss 架构与训练解析", 模型架构,
// MoE bullet; no shared expert is added, section 更少的大专家 vs 更多的小专家).
// fp32 accumulation in slot order j = 0..k-1, one rounding to bf16 (nearest
// even).  Bandwidth-bound: k rows of fp32 read, one bf16 row written.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;

// Grid (T, ceil(d/4 / kThreads)): a CTA takes one token and kThreads groups of
// 4 columns, so each thread has a single round of dependent loads (its k rows
// of y), whatever d is.
__global__ void __launch_bounds__(kThreads)
combine_kernel(const float* __restrict__ y, const float* __restrict__ topk_w,
               const int32_t* __restrict__ inv, int d, int k, int R,
               __nv_bfloat16* __restrict__ out, int32_t* __restrict__ status) {
  const int t = blockIdx.x;
  const int i = blockIdx.y * kThreads + threadIdx.x;   // group of 4 columns
  pdl_wait();
  int32_t rows[8];
  float w[8];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      rows[j] = inv[(size_t)t * k + j];
      w[j] = topk_w[(size_t)t * k + j];
      if (rows[j] < 0 || rows[j] >= R) {   // a row the permutation never wrote
        bad = true;
        rows[j] = 0;
        w[j] = 0.f;
      }
    }
  }
  if (bad && threadIdx.x == 0 && blockIdx.y == 0) atomicMax(status, kStatusBounds);
  if (i >= d / 4) return;
  float4 v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < k) v[j] = *reinterpret_cast<const float4*>(y + (size_t)rows[j] * d + 4 * i);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {                         // slot order j = 0..k-1
      acc.x = fmaf(w[j], v[j].x, acc.x);
      acc.y = fmaf(w[j], v[j].y, acc.y);
      acc.z = fmaf(w[j], v[j].z, acc.z);
      acc.w = fmaf(w[j], v[j].w, acc.w);
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out + (size_t)t * d + 4 * i) = pk;
}

}  // namespace

cudaError_t launch_combine(const float* y, const float* topk_w, const int32_t* inv, int T,
                           int d, int k, __nv_bfloat16* out, int32_t* status, cudaStream_t s) {
  const int groups = (d / 4 + kThreads - 1) / kThreads;
  return launch_pdl(combine_kernel, dim3(T, groups), dim3(kThreads), 0, s, y, topk_w, inv, d, k,
                    T * k, out, status);
}

}  // namespace moe
