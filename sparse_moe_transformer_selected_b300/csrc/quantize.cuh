// The block-scaled design's activation format, written per token.
//
// A token's row of the MoE input (bf16) goes out as two E4M3 tables with one
// UE8M0 scale per 32-element block: the OCP MX block of 32 elements sharing a
// power-of-two scale, the format "OpenAI 最新开源模型 gpt-oss 架构与训练解析"
// (模型架构, weight-quantisation bullet) gives the weights, here carried by two
// terms.  For block b with largest |x| = m_b > 0, e_b = floor(log2 m_b) - 7,
// so x 2^-e_b has magnitude below 256 (E4M3 holds up to 448);
// hi = E4M3(x 2^-e_b), lo = E4M3((x 2^-e_b - hi) 16), and x = (hi + lo / 16) 2^e_b,
// exact for a bf16 x within 2^-7 of its block's largest, else within 2^-13 of
// that largest (the E4M3 subnormal step).  The scale bytes are 127 + e_b (hi)
// and 123 + e_b (lo).  The grouped gate_up GEMM gathers each chunk's token rows
// of these tables.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint32_t e4m3_rn(float v) {
  return uint32_t(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(__nv_fp8_storage_t(b), __NV_E4M3)));
}

// Rows row0 .. row0 + nrows - 1 of x [*, d] into the term tables (rows of d
// bytes) and the scale tables (rows of ld_sx bytes), by all threads of the
// calling CTA (blockDim.x a multiple of 32).  Eight consecutive threads take
// one 32-element block, four elements each.
__device__ __forceinline__ void quantize_rows_mx(const __nv_bfloat16* __restrict__ x, int row0,
                                                 int nrows, int d, uint8_t* __restrict__ xq_hi,
                                                 uint8_t* __restrict__ xq_lo,
                                                 uint8_t* __restrict__ sx_hi,
                                                 uint8_t* __restrict__ sx_lo, int ld_sx) {
  const int nblk = d / 32;
  const int total = nrows * nblk * 8;
  const int lane = threadIdx.x & 31;
  const uint32_t group = 0xFFu << (lane & 24);     // the 8 lanes of this block
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int row = row0 + idx / (nblk * 8);
    const int rem = idx % (nblk * 8);
    const int b = rem >> 3, q = rem & 7;           // block, piece of 4 elements
    const size_t off = size_t(row) * d + b * 32 + q * 4;
    const uint2 raw = *reinterpret_cast<const uint2*>(x + off);
    float f[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                  __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
    float m = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
    m = fmaxf(m, __shfl_xor_sync(group, m, 1));
    m = fmaxf(m, __shfl_xor_sync(group, m, 2));
    m = fmaxf(m, __shfl_xor_sync(group, m, 4));
    const int eb = (m > 0.f && isfinite(m)) ? max(-120, min(120, ilogbf(m) - 7)) : 0;
    const float sc = __int_as_float((127 - eb) << 23);       // 2^-e_b
    uint32_t hi = 0, lo = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float v = f[c] * sc;
      const uint32_t hb = e4m3_rn(v);
      const uint32_t lb = e4m3_rn((v - e4m3_value(hb)) * 16.f);
      hi |= hb << (8 * c);
      lo |= lb << (8 * c);
    }
    *reinterpret_cast<uint32_t*>(xq_hi + off) = hi;
    *reinterpret_cast<uint32_t*>(xq_lo + off) = lo;
    if (q == 0) {
      sx_hi[size_t(row) * ld_sx + b] = uint8_t(127 + eb);
      sx_lo[size_t(row) * ld_sx + b] = uint8_t(123 + eb);
    }
  }
}

}  // namespace moe
