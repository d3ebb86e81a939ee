// Expert scan of the routing histogram, shared by the scan kernel and the
// router's top-k kernel (whose last CTA runs it when there are few token tiles).
#pragma once

#include "common.cuh"

namespace moe {

// Token tiles up to which the top-k kernel's last CTA does the scan itself.
constexpr int kFuseScanTiles = 8;

// With NT threads of one CTA: per-expert offsets (exclusive scan of the counts
// over experts), the base row of every (tile, expert) (scan over tiles), and
// the prefixes of ceil(count / chunk) and ceil(count / chunk2) token chunks
// (mtile_off[0..E] and mtile_off[E+1..2E+1]).  Integer and in a fixed order.
template <int NT>
__device__ __forceinline__ void scan_tiles(const int32_t* tile_counts, int ntiles, int E, int chunk,
                                           int chunk2, int32_t* tile_base, int32_t* offsets,
                                           int32_t* mtile_off, int32_t* part, int32_t* total,
                                           int32_t* off) {
  const int tid = threadIdx.x;
  const int G = NT / E;                       // thread groups over tiles (E <= NT)
  const int g = tid / E, e = tid - g * E;
  const bool active = g < G;
  const int span = (ntiles + G - 1) / G;      // router tiles per thread
  const int ta = min(ntiles, g * span), tb = min(ntiles, ta + span);
  int32_t sum = 0;
  if (active)
    for (int t = ta; t < tb; ++t) sum += __ldcg(tile_counts + (size_t)t * E + e);
  part[tid] = sum;
  __syncthreads();
  if (tid < E) {
    int32_t run = 0;
    for (int q = 0; q < G; ++q) {
      const int32_t v = part[q * E + tid];
      part[q * E + tid] = run;
      run += v;
    }
    total[tid] = run;
  }
  __syncthreads();
  // exclusive scans over experts of the counts and of their token chunks:
  // inclusive scans inside each warp (shuffles), then the warps' totals in
  // order (E <= 256: at most 8 warps)
  {
    const int lane = tid & 31, wid = tid >> 5;
    const int32_t v = tid < E ? total[tid] : 0;
    const int32_t c = tid < E ? (v + chunk - 1) / chunk : 0;
    const int32_t c2 = tid < E ? (v + chunk2 - 1) / chunk2 : 0;
    int32_t iv = v, ic = c, ic2 = c2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t pv = __shfl_up_sync(0xffffffffu, iv, o);
      const int32_t pc = __shfl_up_sync(0xffffffffu, ic, o);
      const int32_t pc2 = __shfl_up_sync(0xffffffffu, ic2, o);
      if (lane >= o) { iv += pv; ic += pc; ic2 += pc2; }
    }
    __shared__ int32_t wsum_v[8], wsum_c[8], wsum_c2[8];
    if (lane == 31 && wid < 8) { wsum_v[wid] = iv; wsum_c[wid] = ic; wsum_c2[wid] = ic2; }
    __syncthreads();
    if (tid < E) {
      int32_t bv = 0, bc = 0, bc2 = 0;
      for (int w = 0; w < wid; ++w) { bv += wsum_v[w]; bc += wsum_c[w]; bc2 += wsum_c2[w]; }
      const int32_t ev = bv + iv - v, ec = bc + ic - c, ec2 = bc2 + ic2 - c2;   // exclusive
      off[tid] = ev;
      offsets[tid] = ev;
      mtile_off[tid] = ec;
      mtile_off[E + 1 + tid] = ec2;
      if (tid == E - 1) {
        offsets[E] = ev + v;
        mtile_off[E] = ec + c;
        mtile_off[2 * E + 1] = ec2 + c2;
      }
    }
  }
  __syncthreads();
  if (active) {
    int32_t base = off[e] + part[tid];
    for (int t = ta; t < tb; ++t) {
      tile_base[(size_t)t * E + e] = base;
      base += __ldcg(tile_counts + (size_t)t * E + e);
    }
  }
}

}  // namespace moe
