// Expert scan of the routing histogram, shared by the scan kernel and the
// router's top-k kernel (whose last CTA runs it when there are few token tiles).
#pragma once

#include "common.cuh"

namespace moe {

// Token tiles up to which the top-k kernel's last CTA does the scan itself.
constexpr int kFuseScanTiles = 8;

// With NT threads of one CTA: per-expert offsets (exclusive scan of the counts
// over experts), the base row of every (tile, expert) (scan over tiles), and
// the prefix of ceil(count / chunk) token chunks.  Integer and in a fixed order.
template <int NT>
__device__ __forceinline__ void scan_tiles(const int32_t* tile_counts, int ntiles, int E, int chunk,
                                           int32_t* tile_base, int32_t* offsets, int32_t* mtile_off,
                                           int32_t* part, int32_t* total, int32_t* off) {
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
  if (tid == 0) {
    int32_t run = 0, mrun = 0;
    for (int q = 0; q < E; ++q) {
      off[q] = run;
      offsets[q] = run;
      mtile_off[q] = mrun;
      run += total[q];
      mrun += (total[q] + chunk - 1) / chunk;
    }
    offsets[E] = run;
    mtile_off[E] = mrun;
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
