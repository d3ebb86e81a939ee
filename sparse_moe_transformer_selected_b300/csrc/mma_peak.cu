// Peak dense rate of the tensor-core MMA forms the grouped GEMMs issue,
// measured with the GEMMs' own instructions: kind::f16 (bf16 x bf16) with both
// operands in shared memory at 128 x 256, kind::mxf8f6f4 with block scales
// (E2M1 x E4M3, the block-scaled design) at 128 x 256, and kind::f16 with A
// read from tensor memory (the TMEM design's form) at 128 x 128 and
// 128 x 256.  One CTA per SM; one thread issues `iters` rounds of four
// back-to-back MMAs (K = 64 per round for kind::f16, 128 for kind::mxf8f6f4)
// into one TMEM accumulator; the host times the launch with CUDA events.  The
// operand values (zeros, scales 2^0) do not matter to the rate.  This is a
// measurement aid of the library: a GEMM's roofline can be read against the
// rate of the very instruction form it issues.
#include "common.cuh"
#include "moe.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kM = 128, kN = 256;
constexpr int kTileA = kM * 128, kTileB = kN * 128;   // one 128-byte swizzle row per operand row
constexpr long long kWaitCycles = 4000000000ll;

// KIND: 0 kind::f16 A, B in shared memory, N = 256; 1 kind::mxf8f6f4, N = 256;
// 2 kind::f16, A in TMEM, N = 128; 3 kind::f16, A in TMEM, N = 256.
template <int KIND>
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int32_t* status) {
  constexpr bool MX = KIND == 1;
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = sm;
  uint8_t* sb = sm + kTileA;
  uint64_t* done = reinterpret_cast<uint64_t*>(sm + kTileA + kTileB);
  uint32_t* tbase = reinterpret_cast<uint32_t*>(sm + kTileA + kTileB + 8);
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (kTileA + kTileB) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    ptx::mbar_init(done, 1);
    ptx::fence_mbar_init();
  }
  ptx::fence_proxy_async_smem();
  if (warp == 0) {
    ptx::tmem_alloc(tbase, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tbase;
  if (KIND >= 2) {
    // A in TMEM: columns 256..287, zeros
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0u;
    ptx::tmem_st_32x32b_x32(tmem + (uint32_t(warp * 32) << 16) + 256, z);
    ptx::tmem_st_wait();
  }
  if (MX) {
    // UE8M0 scale columns 256..271 (A: 256..259, B: 264..271) hold 2^0
    const uint32_t lane_addr = uint32_t(warp * 32) << 16;
    ptx::tmem_st_32x32b_x4(tmem + lane_addr + 256, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    ptx::tmem_st_32x32b_x4(tmem + lane_addr + 264, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    ptx::tmem_st_32x32b_x4(tmem + lane_addr + 268, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    ptx::tmem_st_wait();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (threadIdx.x == 0) {
    const uint64_t ad = ptx::desc_kmajor_sw128(ptx::smem_u32(sa));
    const uint64_t bd = ptx::desc_kmajor_sw128(ptx::smem_u32(sb));
    if (MX) {
      uint32_t idesc[4];
      for (int j = 0; j < 4; ++j) idesc[j] = ptx::idesc_mx(kM, kN, j, j);
      for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int j = 0; j < 4; ++j)               // K = 32 each: 32 bytes of the row
          ptx::mma_mx(tmem, ad + 2 * j, bd + 2 * j, idesc[j], tmem + 256, tmem + 264, it | j);
    } else if (KIND >= 2) {
      const uint32_t idesc = ptx::idesc_f16(kM, KIND == 2 ? 128 : kN, true);
      for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int j = 0; j < 4; ++j)               // K = 16 each: 8 TMEM columns of A
          ptx::mma_f16_tmem_a(tmem, tmem + 256 + 8 * j, bd + 2 * j, idesc, it | j);
    } else {
      const uint32_t idesc = ptx::idesc_f16(kM, kN, true);
      for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int j = 0; j < 4; ++j)               // K = 16 each: 32 bytes of the row
          ptx::mma_f16(tmem, ad + 2 * j, bd + 2 * j, idesc, it | j);
    }
    ptx::mma_commit(done);
    const long long t0 = clock64();
    bool ok;
    while (!(ok = ptx::mbar_try_wait(done, 0)) && clock64() - t0 < kWaitCycles) {
    }
    if (!ok) atomicMax(status, kStatusTimeout);
  }
  __syncwarp();                   // warp 0 reaches the barrier converged
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_mma_peak(int kind, int iters, double* tflops, void* workspace,
                                   void* stream) {
  if (kind < 0 || kind > 3 || iters < 1 || iters > (1 << 24)) return MOE_ERR_SHAPE;
  if (!tflops || !workspace) return MOE_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // more shared memory than two CTAs could share, so each SM runs exactly one
  const int smem = 120 * 1024;
  const void* fns[4] = {reinterpret_cast<const void*>(moe::mma_peak_kernel<0>),
                        reinterpret_cast<const void*>(moe::mma_peak_kernel<1>),
                        reinterpret_cast<const void*>(moe::mma_peak_kernel<2>),
                        reinterpret_cast<const void*>(moe::mma_peak_kernel<3>)};
  const void* fn = fns[kind];
  if (moe::set_smem_limit_once(fn, smem) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* status = static_cast<int32_t*>(workspace);
  if (cudaMemsetAsync(status, 0, 4, s) != cudaSuccess) return MOE_ERR_CUDA;
  const int grid = moe::device_sm_count();
  cudaEvent_t a, b;
  if (cudaEventCreate(&a) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaEventCreate(&b) != cudaSuccess) {
    cudaEventDestroy(a);
    return MOE_ERR_CUDA;
  }
  // one untimed launch (clocks up, first-touch costs), then the timed one
  moe_status st = MOE_OK;
  float ms = 0.f;
  for (int rep = 0; rep < 2 && st == MOE_OK; ++rep) {
    if (rep == 1 && cudaEventRecord(a, s) != cudaSuccess) st = MOE_ERR_CUDA;
    switch (kind) {
      case 0: moe::mma_peak_kernel<0><<<grid, 128, smem, s>>>(iters, status); break;
      case 1: moe::mma_peak_kernel<1><<<grid, 128, smem, s>>>(iters, status); break;
      case 2: moe::mma_peak_kernel<2><<<grid, 128, smem, s>>>(iters, status); break;
      default: moe::mma_peak_kernel<3><<<grid, 128, smem, s>>>(iters, status); break;
    }
    if (cudaGetLastError() != cudaSuccess) st = MOE_ERR_CUDA;
  }
  if (st == MOE_OK && cudaEventRecord(b, s) != cudaSuccess) st = MOE_ERR_CUDA;
  if (st == MOE_OK && cudaEventSynchronize(b) != cudaSuccess) st = MOE_ERR_CUDA;
  if (st == MOE_OK && cudaEventElapsedTime(&ms, a, b) != cudaSuccess) st = MOE_ERR_CUDA;
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  if (st != MOE_OK) return st;
  const double k_per_round = kind == 1 ? 128.0 : 64.0;
  const double n = kind == 2 ? 128.0 : double(moe::kN);
  const double flops = 2.0 * moe::kM * n * k_per_round * double(iters) * grid;
  *tflops = flops / (double(ms) * 1e-3) / 1e12;
  return MOE_OK;
}
