// A stand-alone launch of the combine that K4 runs in its epilogue
// (combine.cuh), on tables the caller supplies: a test hook, so the combine's
// own bounds check can be shown to catch a permuted-row index outside [0, T·k)
// (status word MOE_ERR_DEVICE_BOUNDS, the bad slot left out of the sum) with
// tables the host corrupted on purpose, without running the GEMMs on them.
#include "combine.cuh"
#include "common.cuh"
#include "moe.h"

namespace moe {
namespace {

constexpr int kChunk = 16;

// One CTA of 128 threads per (chunk of 16 permuted rows, output column tile),
// all resident at once or not: the counts decide which CTA sums a token.
__global__ void __launch_bounds__(128) combine_check_kernel(const GemmArgs a) {
  __shared__ __align__(16) uint8_t sm[combine_smem_bytes(kChunk, 8)];
  const int r0 = blockIdx.x * kChunk;
  const int n = min(kChunk, a.R - r0);
  combine_tile<4>(a, r0, n, blockIdx.y, threadIdx.x, sm, kChunk, 1);
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_debug_combine(const float* y, const int32_t* perm, const int32_t* inv,
                                        const float* topk_w, int64_t T, int d, int k,
                                        void* out_bf16, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  if (T <= 0 || d <= 0 || d % 32 || k < 1 || k > 8 || T * k >= (int64_t(1) << 31))
    return MOE_ERR_SHAPE;
  if (!y || !perm || !inv || !topk_w || !out_bf16 || !workspace) return MOE_ERR_NULL;
  const int R = int(T * k), n_mt = moe::down_col_tiles(d);
  const size_t cnt_off = 256, need = cnt_off + size_t(T) * n_mt * 4;
  if (workspace_bytes < need) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the status word and the counts start at zero
  if (cudaMemsetAsync(workspace, 0, need, s) != cudaSuccess) return MOE_ERR_CUDA;
  moe::GemmArgs a{};
  a.R = R;
  a.d = d;
  a.k = k;
  a.y = const_cast<float*>(y);
  a.perm = perm;
  a.inv = inv;
  a.topk_w = topk_w;
  a.status = static_cast<int32_t*>(workspace);
  a.cnt = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + cnt_off);
  a.n_mt_dn = n_mt;
  a.out = static_cast<__nv_bfloat16*>(out_bf16);
  a.resid = nullptr;
  const dim3 grid((R + moe::kChunk - 1) / moe::kChunk, n_mt);
  moe::combine_check_kernel<<<grid, 128, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
