// K1 — router logits, top-k selection, softmax over the selected logits, and the
// per-tile expert histogram the permutation is built from.
//
// Follows "OpenAI 最新开源模型 gpt-oss 架构与训练解析", section 模型架构, MoE bullet
// (top-4 routing, softmax weighting of the selected experts) and
// "【LLM】GPT-OSS架构变化详解" section 2.4.1 (a router chooses each token's
// experts).  Ties go to the lower expert index; slots are ordered by
// (logit desc, index asc).
//
// One CTA = 32 tokens x all E experts.  fp32 FMA on CUDA cores: the router is
// 2·T·d·E flops, well under 1% of the block, and fp32 keeps the selection
// faithful to the exact logits except at true near-ties.
#include "common.cuh"

#include <math.h>

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kKC = 32;                  // K chunk staged in shared memory
constexpr int kTT = kRouterTile;         // tokens per CTA (32)
constexpr int kMaxE = 256;
constexpr int kLgStride = kMaxE + 8;     // floats per row of the logits / W tile

template <int NPER>   // experts per lane: e = lane + 32*i, i < NPER
__global__ void __launch_bounds__(kThreads)
router_topk_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ rw,
                   const float* __restrict__ rb, int T, int d, int E, int k,
                   int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                   int32_t* __restrict__ rank, int32_t* __restrict__ tile_counts,
                   int32_t* __restrict__ xexp, int32_t* __restrict__ status) {
  __shared__ float xs[kTT][kKC + 1];
  __shared__ float wl[kKC * kLgStride];  // W chunk [k][e]; later logits [t][e]
  __shared__ uint32_t mask[kMaxE];       // bit t: token t of this tile picked e
  __shared__ int32_t sel[kTT][8];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTT;
  if (blockIdx.x == 0 && tid == 0) status[0] = 0;
  for (int e = tid; e < kMaxE; e += kThreads) mask[e] = 0u;

  float xmax = 0.f;   // max |x| over this thread's share of token (tid >> 3)
  float acc[4][NPER];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < NPER; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < d; k0 += kKC) {
    {  // x chunk: 32 tokens x 32 k, 4 bf16 per thread
      const int tl = tid >> 3, kq = (tid & 7) * 4, t = t0 + tl;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < T) {
        const uint2 raw = *reinterpret_cast<const uint2*>(x + (size_t)t * d + k0 + kq);
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
        v[0] = __low2float(a); v[1] = __high2float(a);
        v[2] = __low2float(b); v[3] = __high2float(b);
        xmax = fmaxf(xmax, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) xs[tl][kq + c] = v[c];
    }
    for (int idx = tid; idx < E * (kKC / 4); idx += kThreads) {  // W chunk, transposed
      const int e = idx >> 3, kq = (idx & 7) * 4;
      const float4 w4 = *reinterpret_cast<const float4*>(rw + (size_t)e * d + k0 + kq);
      wl[(kq + 0) * kLgStride + e] = w4.x;
      wl[(kq + 1) * kLgStride + e] = w4.y;
      wl[(kq + 2) * kLgStride + e] = w4.z;
      wl[(kq + 3) * kLgStride + e] = w4.w;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kKC; ++kk) {
      float xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = xs[warp * 4 + i][kk];
#pragma unroll
      for (int j = 0; j < NPER; ++j) {
        const float wv = wl[kk * kLgStride + lane + 32 * j];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][j] = fmaf(xv[i], wv, acc[i][j]);
      }
    }
    __syncthreads();
  }

  // per-token exponent for holding x in f16: largest |x| scaled into [2^14, 2^15)
  xmax = fmaxf(xmax, __shfl_xor_sync(0xffffffffu, xmax, 1));
  xmax = fmaxf(xmax, __shfl_xor_sync(0xffffffffu, xmax, 2));
  xmax = fmaxf(xmax, __shfl_xor_sync(0xffffffffu, xmax, 4));
  if ((tid & 7) == 0 && t0 + (tid >> 3) < T) {
    const int et = (xmax > 0.f && isfinite(xmax)) ? 14 - ilogbf(xmax) : 0;
    xexp[t0 + (tid >> 3)] = max(-126, min(126, et));
  }

  // logits (+ bias) into shared memory, row per token
#pragma unroll
  for (int j = 0; j < NPER; ++j) {
    const int e = lane + 32 * j;
    if (e < E) {
      const float b = rb[e];
#pragma unroll
      for (int i = 0; i < 4; ++i) wl[(warp * 4 + i) * kLgStride + e] = acc[i][j] + b;
    }
  }
  __syncthreads();

  // top-k per token: warp w owns tokens 4w..4w+3
  for (int i = 0; i < 4; ++i) {
    const int tl = warp * 4 + i, t = t0 + tl;
    if (t >= T) break;
    float v[NPER];
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
      const int e = lane + 32 * j;
      float lv = (e < E) ? wl[tl * kLgStride + e] : -INFINITY;
      v[j] = isnan(lv) ? -INFINITY : lv;
    }
    uint32_t taken = 0;
    float sv[8];
    int se[8];
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int q = 0; q < NPER; ++q) {
        const int e = lane + 32 * q;
        if (e < E && !((taken >> q) & 1u) && (v[q] > bv || (v[q] == bv && e < be))) {
          bv = v[q];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      sv[j] = bv;
      se[j] = be;
    }
    if (lane == 0) {
      const float m = sv[0];
      float p[8], s = 0.f;
      for (int j = 0; j < k; ++j) {
        p[j] = expf(sv[j] - m);
        s += p[j];
      }
      const float inv_s = 1.0f / s;
      for (int j = 0; j < k; ++j) {
        topk_idx[(size_t)t * k + j] = se[j];
        topk_w[(size_t)t * k + j] = p[j] * inv_s;
        sel[tl][j] = se[j];
      }
    }
    if (lane < k) atomicOr(&mask[se[lane]], 1u << tl);  // order-free: deterministic
  }
  __syncthreads();

  const int ntok = min(kTT, T - t0);
  for (int e = tid; e < E; e += kThreads)
    tile_counts[(size_t)blockIdx.x * E + e] = __popc(mask[e]);
  for (int q = tid; q < ntok * k; q += kThreads) {
    const int tl = q / k, j = q - tl * k;
    const int e = sel[tl][j];
    rank[(size_t)(t0 + tl) * k + j] = __popc(mask[e] & ((1u << tl) - 1u));
  }
}

}  // namespace

cudaError_t launch_router_topk(const __nv_bfloat16* x, const float* router_w,
                               const float* router_b, int T, int d, int E, int k,
                               int32_t* topk_idx, float* topk_w, int32_t* rank,
                               int32_t* tile_counts, int32_t* xexp, int32_t* status,
                               cudaStream_t s) {
  const int grid = (T + kTT - 1) / kTT;
  const int nper = (E + 31) / 32;
#define MOE_ROUTER_CASE(N)                                                          \
  case N:                                                                           \
    router_topk_kernel<N><<<grid, kThreads, 0, s>>>(x, router_w, router_b, T, d, E, \
                                                    k, topk_idx, topk_w, rank,      \
                                                    tile_counts, xexp, status);     \
    break;
  switch (nper) {
    MOE_ROUTER_CASE(1)
    MOE_ROUTER_CASE(2)
    MOE_ROUTER_CASE(3)
    MOE_ROUTER_CASE(4)
    MOE_ROUTER_CASE(5)
    MOE_ROUTER_CASE(6)
    MOE_ROUTER_CASE(7)
    MOE_ROUTER_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_ROUTER_CASE
  return cudaGetLastError();
}

}  // namespace moe
