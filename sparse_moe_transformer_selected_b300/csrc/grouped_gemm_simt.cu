// K3 / K4 — grouped expert GEMMs, plain CUDA-core version.
//
// Each expert's segment of permuted rows is multiplied by that expert's MXFP4
// weights, dequantised exactly to fp32 in shared memory, with fp32
// accumulation.  K3 ends in the clamped SwiGLU ("OpenAI 最新开源模型 gpt-oss
// 架构与训练解析", 模型架构, MoE bullet: gated-SwiGLU with clamping and the +1
// residual term on the up branch); K4 adds the down bias.
#include "common.cuh"

#include <math.h>

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kBM = kGemmBM;   // 128 rows per tile
constexpr int kKC = 32;        // one MX block of K per stage

__device__ __forceinline__ float e2m1_value(uint32_t c) {
  // magnitude {0, .5, 1, 1.5, 2, 3, 4, 6} from exponent bits 2..1, mantissa bit 0
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const float mag = (e == 0) ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, (int)e - 1);
  return (c & 8u) ? -mag : mag;
}

// Global row tile g -> expert e with mtile_off[e] <= g < mtile_off[e+1].
__device__ __forceinline__ int expert_of_tile(const int32_t* mtile_off, int E, int g) {
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mtile_off[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Dequantise 8 codes (one 32-bit word) with a shared E8M0 scale.
__device__ __forceinline__ void dequant8(uint32_t word, int scale, float* v) {
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = ldexpf(e2m1_value((word >> (4 * i)) & 15u), scale - 127);
}

__global__ void __launch_bounds__(kThreads)
gateup_simt_kernel(GemmArgs a) {
  __shared__ float As[kKC][kBM + 4];
  __shared__ float Bg[kKC][33];
  __shared__ float Bu[kKC][33];
  const int g = blockIdx.y;
  if (g >= a.mtile_off[a.E]) return;
  const int e = expert_of_tile(a.mtile_off, a.E, g);
  const int seg_end = a.offsets[e + 1];
  const int r0 = a.offsets[e] + (g - a.mtile_off[e]) * kBM;
  const int n0 = blockIdx.x * 32;
  const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;
  const int d = a.d, W = a.W;
  float accg[4][4] = {}, accu[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += kKC) {
    {  // A: 128 rows x 32 k
      const int row = tid >> 1, kh = (tid & 1) * 16, r = r0 + row;
      float v[16];
      if (r < seg_end) {
        const __nv_bfloat16* src = a.x_perm + (size_t)r * d + k0 + kh;
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __bfloat162float(src[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) As[kh + i][row] = v[i];
    }
    {  // B: 32 gate rows + 32 up rows x 32 k
      const int row = tid >> 2, word = tid & 3;
      const int n = row < 32 ? n0 + row : W + n0 + row - 32;
      const size_t wrow = (size_t)e * 2 * W + n;
      const uint32_t cw = *reinterpret_cast<const uint32_t*>(a.w_gu + wrow * (d / 2) + k0 / 2 + word * 4);
      const int sc = a.w_gu_scale[wrow * (d / 32) + k0 / 32];
      float v[8];
      dequant8(cw, sc, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (row < 32) Bg[word * 8 + i][row] = v[i];
        else Bu[word * 8 + i][row - 32] = v[i];
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKC; ++kk) {
      float av[4], bg[4], bu[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) { bg[j] = Bg[kk][tx * 4 + j]; bu[j] = Bu[kk][tx * 4 + j]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          accg[i][j] = fmaf(av[i], bg[j], accg[i][j]);
          accu[i][j] = fmaf(av[i], bu[j], accu[i][j]);
        }
    }
    __syncthreads();
  }
  const float limit = a.limit, alpha = a.alpha;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty * 4 + i;
    if (r >= seg_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      const float zg = accg[i][j] + __bfloat162float(a.b_gu[(size_t)e * 2 * W + n]);
      const float zu = accu[i][j] + __bfloat162float(a.b_gu[(size_t)e * 2 * W + W + n]);
      const float gg = fminf(zg, limit);
      const float uu = fminf(fmaxf(zu, -limit), limit);
      const float h = gg * (1.0f / (1.0f + expf(-alpha * gg))) * (uu + 1.0f);
      const __nv_bfloat16 hi = __float2bfloat16_rn(h);
      const __nv_bfloat16 lo = __float2bfloat16_rn(h - __bfloat162float(hi));
      a.h_hi[(size_t)r * W + n] = hi;
      a.h_lo[(size_t)r * W + n] = lo;
    }
  }
}

__global__ void __launch_bounds__(kThreads)
down_simt_kernel(GemmArgs a) {
  __shared__ float As[kKC][kBM + 4];
  __shared__ float Bs[kKC][65];
  const int g = blockIdx.y;
  if (g >= a.mtile_off[a.E]) return;
  const int e = expert_of_tile(a.mtile_off, a.E, g);
  const int seg_end = a.offsets[e + 1];
  const int r0 = a.offsets[e] + (g - a.mtile_off[e]) * kBM;
  const int n0 = blockIdx.x * 64;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int d = a.d, W = a.W;
  float acc[8][4] = {};
  for (int k0 = 0; k0 < W; k0 += kKC) {
    {
      const int row = tid >> 1, kh = (tid & 1) * 16, r = r0 + row;
      float v[16];
      if (r < seg_end) {
        const __nv_bfloat16* ph = a.h_hi + (size_t)r * W + k0 + kh;
        const __nv_bfloat16* pl = a.h_lo + (size_t)r * W + k0 + kh;
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __bfloat162float(ph[i]) + __bfloat162float(pl[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) As[kh + i][row] = v[i];
    }
    {
      const int row = tid >> 2, word = tid & 3, n = n0 + row;
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (n < d) {
        const size_t wrow = (size_t)e * d + n;
        const uint32_t cw = *reinterpret_cast<const uint32_t*>(a.w_dn + wrow * (W / 2) + k0 / 2 + word * 4);
        dequant8(cw, a.w_dn_scale[wrow * (W / 32) + k0 / 32], v);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) Bs[word * 8 + i][row] = v[i];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKC; ++kk) {
      float av[8], bv[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) av[i] = As[kk][ty * 8 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + ty * 8 + i;
    if (r >= seg_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < d) a.y[(size_t)r * d + n] = acc[i][j] + __bfloat162float(a.b_dn[(size_t)e * d + n]);
    }
  }
}

}  // namespace

cudaError_t launch_gateup(const GemmArgs& a, cudaStream_t s) {
  dim3 grid(a.W / 32, a.R / kBM + a.E + 1);
  gateup_simt_kernel<<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_down(const GemmArgs& a, cudaStream_t s) {
  dim3 grid((a.d + 63) / 64, a.R / kBM + a.E + 1);
  down_simt_kernel<<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
