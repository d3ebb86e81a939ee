// K2 — expert histogram scan and token permutation.
//
// The pages fix only that each token is processed by its selected experts
// ("OpenAI 最新开源模型 gpt-oss 架构与训练解析", 模型架构, MoE bullet); grouping the
// routed rows by expert is what lets each expert run as one dense GEMM.  Rows
// are ordered by (expert, token, slot).  Since a token never picks an expert
// twice, a row's place is offsets[e] + (rows of e in earlier router tiles) +
// (rank inside its tile), all integer and order-free, so the permutation is
// deterministic without atomics.
#include "common.cuh"
#include "route_scan.cuh"

#include <cuda_fp16.h>
#include <math.h>

namespace moe {
namespace {

constexpr int kScanThreads = 1024;

// One CTA.  Thread (g, e) sums expert e over a contiguous range of tiles,
// then the partial sums are scanned in tile order and in expert order.
__global__ void __launch_bounds__(kScanThreads)
route_scan_kernel(const int32_t* __restrict__ tile_counts, int ntiles, int E, int chunk,
                  int chunk2, int32_t* __restrict__ tile_base, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ mtile_off) {
  __shared__ int32_t part[kScanThreads];
  __shared__ int32_t total[257];
  __shared__ int32_t off[257];
  pdl_wait();
  scan_tiles<kScanThreads>(tile_counts, ntiles, E, chunk, chunk2, tile_base, offsets, mtile_off, part,
                           total, off);
}

// One warp per token t: for each of its k routed rows (t, j) write perm / inv
// and copy x[t] to the row, converted to f16 after an exact power-of-two
// scaling by 2^e_t (e_t puts the token's largest |x| in [2^14, 2^15), so every
// bf16 value is held exactly).  The token is read and converted once for its
// k rows.  A slot whose expert or row is out of range is skipped and recorded.
__global__ void __launch_bounds__(256, 2)
route_scatter_kernel(const __nv_bfloat16* __restrict__ x, int T, int d, int E, int k,
                     const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ rank,
                     const int32_t* __restrict__ tile_base,
                     int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                     __half* __restrict__ x_perm, int32_t* __restrict__ rowexp,
                     int32_t* __restrict__ status) {
  const int64_t R = (int64_t)T * k;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_wait();
  if (t >= T) return;
  // the token's rows (-1: a slot left out); k <= 8, loops unrolled so the
  // rows stay in registers
  int64_t rows[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    rows[j] = -1;
    if (j >= k) continue;
    const int64_t q = t * k + j;
    const int e = topk_idx[q];
    int64_t row = -1;
    if (e >= 0 && e < E) row = (int64_t)tile_base[(size_t)(t / kRouterTile) * E + e] + rank[q];
    if (row < 0 || row >= R) {
      if (lane == 0) atomicMax(status, kStatusBounds);
      row = -1;
    } else if (lane == 0) {
      if (perm) perm[row] = (int32_t)q;
      if (inv) inv[q] = (int32_t)row;
    }
    rows[j] = row;
  }
  if (!x_perm) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
  const int n16 = d / 8;
  auto absmax8 = [](const uint4& v, float m) {
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      m = fmaxf(m, fmaxf(fabsf(__uint_as_float(in[c] << 16)), fabsf(__uint_as_float(in[c] & 0xFFFF0000u))));
    return m;
  };
  auto to_f16 = [](const uint4& v, float f) {
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float lo = __uint_as_float(in[c] << 16) * f;
      const float hi = __uint_as_float(in[c] & 0xFFFF0000u) * f;
      const __half2 h = __floats2half2_rn(lo, hi);
      o[c] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
  auto exponent = [&](float xmax) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) xmax = fmaxf(xmax, __shfl_xor_sync(0xffffffffu, xmax, off));
    return (xmax > 0.f && isfinite(xmax)) ? max(-126, min(126, 14 - ilogbf(xmax))) : 0;
  };
  // A row of up to 32 x kRowRegs 16-byte pieces (d <= 3072) is read once into
  // registers, all loads in flight together, and converted once; longer rows
  // take a pass for the maximum and one per routed row.
  constexpr int kRowRegs = 12;
  if (n16 <= 32 * kRowRegs) {
    uint4 v[kRowRegs];
    float xmax = 0.f;                                  // largest |x| of the token
#pragma unroll
    for (int j = 0; j < kRowRegs; ++j) {
      const int i = lane + 32 * j;
      v[j] = i < n16 ? src[i] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kRowRegs; ++j) xmax = absmax8(v[j], xmax);
    const int et = exponent(xmax);
    const float f = __int_as_float((et + 127) << 23);  // 2^e_t, |e_t| <= 126
#pragma unroll
    for (int j = 0; j < kRowRegs; ++j) v[j] = to_f16(v[j], f);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (rows[s] < 0) continue;
      if (lane == 0) rowexp[rows[s]] = et;
      uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)rows[s] * d);
#pragma unroll
      for (int j = 0; j < kRowRegs; ++j) {
        const int i = lane + 32 * j;
        if (i < n16) dst[i] = v[j];
      }
    }
  } else {
    float xmax = 0.f;
    for (int i = lane; i < n16; i += 32) xmax = absmax8(src[i], xmax);
    const int et = exponent(xmax);
    const float f = __int_as_float((et + 127) << 23);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (rows[s] < 0) continue;
      if (lane == 0) rowexp[rows[s]] = et;
      uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)rows[s] * d);
      for (int i = lane; i < n16; i += 32) dst[i] = to_f16(src[i], f);
    }
  }
}

}  // namespace

cudaError_t launch_route_scan(const int32_t* tile_counts, int ntiles, int E, int chunk, int chunk2,
                              int32_t* tile_base, int32_t* offsets, int32_t* mtile_off,
                              cudaStream_t s) {
  return launch_pdl(route_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, tile_counts, ntiles, E,
                    chunk, chunk2, tile_base, offsets, mtile_off);
}

cudaError_t launch_route_scatter(const __nv_bfloat16* x, int T, int d, int E, int k,
                                 const int32_t* topk_idx, const int32_t* rank,
                                 const int32_t* tile_base, int32_t* perm, int32_t* inv,
                                 void* x_perm, int32_t* rowexp, int32_t* status,
                                 cudaStream_t s) {
  if (k < 1 || k > 8) return cudaErrorInvalidValue;   // a warp keeps at most 8 rows of its token
  const int warps_per_block = 8;
  const int64_t grid = ((int64_t)T + warps_per_block - 1) / warps_per_block;
  return launch_pdl(route_scatter_kernel, dim3((unsigned)grid), dim3(warps_per_block * 32), 0, s,
                    x, T, d, E, k, topk_idx, rank, tile_base, perm, inv,
                    static_cast<__half*>(x_perm), rowexp, status);
}

}  // namespace moe
