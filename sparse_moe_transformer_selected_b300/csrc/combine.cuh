// K5 folded into K4's epilogue — the weighted unpermute-combine.
//
// out[t] = bf16( Σ_j w[t,j] · y[inv[t,j]] (+ resid[t]) ): the softmax-weighted
// sum of the selected experts' outputs ("OpenAI 最新开源模型 gpt-oss 架构与训练解析",
// 模型架构, MoE bullet; no shared expert is added, section 更少的大专家 vs
// 更多的小专家), plus the block's residual input when the caller runs the
// pre-norm block (section 更深对比更宽: residual connections).
//
// A token's k expert rows are produced by k different down-GEMM work units,
// in no fixed order.  Each unit, once its rows of y for output columns
// [mt·128, mt·128 + 128) are stored, counts itself against every token of its
// chunk in cnt[t, mt]; the unit that brings a count to k adds that token's k
// rows in slot order j = 0..k-1 (fp32 fma from 0, then the residual, one
// rounding to bf16).  Which unit is last varies from run to run; the sum it
// computes does not, so the output is bitwise reproducible without floating-
// point atomics.  The k rows are read back from L2 (ld.global.cg: other SMs
// wrote them during this kernel).
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {

// Shared memory of combine_tile for chunks of up to `nb` rows and k <= 8
// experts per token: count, token list, then k rows and k weights per token.
__host__ __device__ constexpr int combine_smem_bytes(int nb, int k) {
  return 16 + nb * 4 + nb * k * 4 * 2;
}

// Tokens i = i0, i0 + 4, ... < m of the list, columns c .. c + 3: a batch of B
// tokens loads its k <= KMAX rows (16 bytes each) before any is summed.
template <int B, int KMAX>
__device__ __forceinline__ void combine_batches(const GemmArgs& a, int m, int c, int i0,
                                                const int* tok, const int* rows, const float* wts) {
  const int k = a.k;
  const float* __restrict__ y = a.y;
  __nv_bfloat16* __restrict__ out = a.out;
  const __nv_bfloat16* __restrict__ resid = a.resid;
  for (int ib = i0; ib < m; ib += 4 * B) {
    float4 v[B][KMAX];
#pragma unroll
    for (int u = 0; u < B; ++u)
#pragma unroll
      for (int s = 0; s < KMAX; ++s) {
        const int i = ib + 4 * u;
        v[u][s] = (i < m && s < k)
                      ? __ldcg(reinterpret_cast<const float4*>(y + size_t(rows[i * k + s]) * a.d + c))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int i = ib + 4 * u;
      if (i >= m) break;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s = 0; s < KMAX; ++s) {             // slot order
        if (s < k) {
          const float w = wts[i * k + s];
          acc.x = fmaf(w, v[u][s].x, acc.x);
          acc.y = fmaf(w, v[u][s].y, acc.y);
          acc.z = fmaf(w, v[u][s].z, acc.z);
          acc.w = fmaf(w, v[u][s].w, acc.w);
        }
      }
      const size_t o = size_t(tok[i]) * a.d + c;
      if (resid) {
        const uint2 rr = *reinterpret_cast<const uint2*>(resid + o);
        acc.x += __uint_as_float(rr.x << 16);
        acc.y += __uint_as_float(rr.x & 0xFFFF0000u);
        acc.z += __uint_as_float(rr.y << 16);
        acc.w += __uint_as_float(rr.y & 0xFFFF0000u);
      }
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&lo);
      pk.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(out + o) = pk;
    }
  }
}

// Called by the 128 epilogue threads of a CTA (tid 0..127) after each has
// stored its y values of rows r0 .. r0 + n - 1 (n <= nb), output columns
// [mt·128, mt·128 + 128).  `sm` is combine_smem_bytes(nb, a.k) bytes of
// shared memory; `bar_id` a named barrier free for these 128 threads.
//
// The tokens this unit completes are listed first, with their k rows and
// weights, by one thread per token; then each warp takes a quarter of them,
// each thread four columns, with the rows of a batch of tokens loaded
// together so their round trips overlap.
// B tokens per batch (k <= 4; half as many for k > 4): as many as the calling
// kernel's registers allow.
template <int B>
__device__ __forceinline__ void combine_tile(const GemmArgs& a, int r0, int n, int mt, int tid,
                                             uint8_t* sm, int nb, uint32_t bar_id) {
  const int k = a.k;
  int* nlast = reinterpret_cast<int*>(sm);
  int* tok = reinterpret_cast<int*>(sm + 16);
  int* rows = tok + nb;                            // [nb][k]
  float* wts = reinterpret_cast<float*>(rows + nb * k);
  if (tid == 0) *nlast = 0;
  __threadfence();                                 // this thread's y stores, before the count
  ptx::named_barrier(bar_id, 128);
  for (int j = tid; j < n; j += 128) {
    const int t = __ldg(a.perm + r0 + j) / k;
    if (atomicAdd(a.cnt + size_t(t) * a.n_mt_dn + mt, 1) == k - 1) {
      const int i = atomicAdd(nlast, 1);
      tok[i] = t;
      for (int s = 0; s < k; ++s) {
        int row = __ldg(a.inv + size_t(t) * k + s);
        float w = __ldg(a.topk_w + size_t(t) * k + s);
        if (row < 0 || row >= a.R) {               // a row the permutation never wrote
          atomicMax(a.status, kStatusBounds);
          row = 0;
          w = 0.f;
        }
        rows[i * k + s] = row;
        wts[i * k + s] = w;
      }
    }
  }
  __threadfence();                                 // the other units' y stores, after the count
  ptx::named_barrier(bar_id, 128);
  const int m = *nlast;
  // four columns per thread (a warp covers the tile's 128 columns), tokens
  // warp, warp + 4, ...; a batch of tokens has all its k slots' loads in flight
  const int c = mt * 128 + (tid & 31) * 4;
  if (c < a.d) {                                   // d % 32 == 0: all four columns valid
    if (k <= 4) combine_batches<B, 4>(a, m, c, tid >> 5, tok, rows, wts);
    else combine_batches<(B > 1 ? B / 2 : 1), 8>(a, m, c, tid >> 5, tok, rows, wts);
  }
  ptx::named_barrier(bar_id, 128);                 // the lists are reused by the next unit
}

}  // namespace moe
