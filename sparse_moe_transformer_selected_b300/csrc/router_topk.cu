// K1 — router logits, top-k selection, softmax over the selected logits, and the
// per-tile expert histogram the permutation is built from.
//
// Follows "OpenAI 最新开源模型 gpt-oss 架构与训练解析", section 模型架构, MoE bullet
// (top-4 routing, softmax weighting of the selected experts) and
// "【LLM】GPT-OSS架构变化详解" section 2.4.1 (a router chooses each token's
// experts).  Ties go to the lower expert index; slots are ordered by
// (logit desc, index asc).
//
// Two kernels.  router_logits: a CTA takes 32 tokens x all E experts over one
// range of K and writes that range's partial dot products (fp32 FMA on CUDA
// cores); small T is split over many K ranges so the few tokens of a decode
// step still spread over the GPU.  router_topk: a CTA sums the partials of 32
// tokens in a fixed order, adds the bias, and selects.  The router is 2·T·d·E
// flops, well under 1% of the block; fp32 keeps the selection faithful to the
// exact logits except at true near-ties.
//
// The pre-norm block ("【LLM】GPT-OSS架构变化详解" 2.7.1: RMSNorm divides by the
// root mean square, with no mean and no bias) feeds the MoE the bf16 values of
// x / sqrt(mean(x²) + eps) · g.  At decode sizes the logits kernel computes
// them on the fly (1/rms in fp64, then rms_scaled_bf16) and its first expert
// group writes them out for the later stages; larger batches run
// rms_norm_kernel first and route on its table.
#include "common.cuh"
#include "quantize.cuh"
#include "route_scan.cuh"

#include <math.h>

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kKC = 32;                  // K chunk staged in shared memory
constexpr int kTT = kRouterTile;         // tokens per CTA (32)
constexpr int kMaxE = 256;
constexpr int kLgStride = kMaxE + 8;     // floats per row of the logits / W tile

// The first kernel of a call clears the status word and the combine counts
// (grid-stride over all CTAs of the launch).
__device__ __forceinline__ void clear_call_state(const RouteArgs& r) {
  const int64_t cta = (int64_t(blockIdx.z) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  const int64_t nthr = int64_t(gridDim.x) * gridDim.y * gridDim.z * blockDim.x;
  if (cta == 0 && threadIdx.x == 0) {
    r.status[0] = 0;                             // first kernel of a call
    r.status[1] = 0;                             // top-k tiles done (fused scan)
    r.status[4] = 0;                             // which wait of a GEMM timed out, if one did
  }
  for (int64_t i = cta * blockDim.x + threadIdx.x; i < r.ncnt; i += nthr) r.cnt[i] = 0;
}

template <int NPER>   // experts per lane: e = lane + 32*i, i < NPER
__global__ void __launch_bounds__(kThreads)
router_logits_kernel(const RouteArgs r, int kc, int eg) {
  __shared__ float xs[kTT][kKC + 1];
  __shared__ float wl[kKC * kLgStride];  // W chunk [k][e]

  const __nv_bfloat16* __restrict__ x = r.x;
  const float* __restrict__ rw = r.router_w;
  const int T = r.T, d = r.d, E = r.E;
  float* __restrict__ part = r.logit_part;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTT;
  const int ks = blockIdx.y;
  const int kb = ks * kc, ke = min(d, kb + kc);
  const int e0 = blockIdx.z * eg;                // this CTA's experts: e0 .. e0+eg-1
  const int ne = min(eg, E - e0);
  pdl_wait();
  clear_call_state(r);

  float acc[4][NPER];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < NPER; ++j) acc[i][j] = 0.f;

  // A decode-sized CTA (one group of 32 experts, at most 8 chunks of 32 K)
  // issues all of its global loads first, then stages each chunk through
  // shared memory: one round of memory latency instead of one per chunk.
  const int nchunks = (ke - kb + kKC - 1) / kKC;
  if (NPER == 1 && nchunks <= 8) {
    uint2 xr[8];
    float4 wr[8];
    const int tl = tid >> 3, kq = (tid & 7) * 4, t = t0 + tl;
    const int we = tid >> 3;                      // expert of this thread's W piece
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int k0 = kb + c * kKC;
      xr[c] = make_uint2(0, 0);
      wr[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < nchunks) {
        if (t < T) xr[c] = *reinterpret_cast<const uint2*>(x + (size_t)t * d + k0 + kq);
        if (we < ne) wr[c] = *reinterpret_cast<const float4*>(rw + (size_t)(e0 + we) * d + k0 + kq);
      }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      if (c >= nchunks) break;
      const __nv_bfloat162 a2 = *reinterpret_cast<const __nv_bfloat162*>(&xr[c].x);
      const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&xr[c].y);
      xs[tl][kq + 0] = __low2float(a2);
      xs[tl][kq + 1] = __high2float(a2);
      xs[tl][kq + 2] = __low2float(b2);
      xs[tl][kq + 3] = __high2float(b2);
      wl[(kq + 0) * kLgStride + we] = wr[c].x;
      wl[(kq + 1) * kLgStride + we] = wr[c].y;
      wl[(kq + 2) * kLgStride + we] = wr[c].z;
      wl[(kq + 3) * kLgStride + we] = wr[c].w;
      __syncthreads();
#pragma unroll 4
      for (int kk = 0; kk < kKC; ++kk) {
        float xv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) xv[i] = xs[warp * 4 + i][kk];
        const float wv = wl[kk * kLgStride + lane];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][0] = fmaf(xv[i], wv, acc[i][0]);
      }
      __syncthreads();
    }
  } else
  for (int k0 = kb; k0 < ke; k0 += kKC) {
    {  // x chunk: 32 tokens x 32 k, 4 bf16 per thread
      const int tl = tid >> 3, kq = (tid & 7) * 4, t = t0 + tl;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < T) {
        const uint2 raw = *reinterpret_cast<const uint2*>(x + (size_t)t * d + k0 + kq);
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
        v[0] = __low2float(a); v[1] = __high2float(a);
        v[2] = __low2float(b); v[3] = __high2float(b);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) xs[tl][kq + c] = v[c];
    }
    for (int idx = tid; idx < ne * (kKC / 4); idx += kThreads) {  // W chunk, transposed
      const int e = idx >> 3, kq = (idx & 7) * 4;
      const float4 w4 = *reinterpret_cast<const float4*>(rw + (size_t)(e0 + e) * d + k0 + kq);
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

  // this K range's contribution to the logits of the tile's tokens
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + warp * 4 + i;
    if (t >= T) break;
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
      const int e = lane + 32 * j;
      if (e < ne) part[((size_t)ks * T + t) * E + e0 + e] = acc[i][j];
    }
  }
}

// Decode-sized batches (at most 8 router tiles): whole dot products, no
// partial slabs.  A CTA takes one token and 4 experts; its 8 warps split d
// into 8 ranges, so each lane has at most kRowIt 4-element pieces and loads all
// of them (token row and the 4 expert rows) before it multiplies: one round of
// memory latency.  Each warp adds its lanes in a fixed shuffle tree and warp 0
// adds the 8 ranges in order.  The result is the logits without bias, the one
// partial slab the top-k kernel adds the bias to.
constexpr int kRowExp = 4, kRowParts = kThreads / 32, kRowIt = 4;

__global__ void __launch_bounds__(kThreads)
router_logits_rows_kernel(const RouteArgs r) {
  __shared__ float red[kRowParts][kRowExp];
  __shared__ double red_ss[kRowParts];
  const bool norm = r.x_pre != nullptr;
  const __nv_bfloat16* __restrict__ x = norm ? r.x_pre : r.x;
  const float* __restrict__ rw = r.router_w;
  const float* __restrict__ g = r.norm_w;
  const int d = r.d, E = r.E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x;
  const int e0 = blockIdx.y * kRowExp;
  pdl_wait();
  clear_call_state(r);
  const int np = d / 4;                          // 4-element pieces of a row
  const int per = (np + kRowParts - 1) / kRowParts;
  const int p0 = warp * per, p1 = min(np, p0 + per);
  const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)t * d);
  // the block's RMSNorm: 1/rms(x_t) in fp64 (every square of a bf16 value is
  // exact in fp32; the sum is kept in fp64 so the bf16 rounding of x·g/rms
  // below is decided as for the exact value)
  float r32 = 1.f;
  double r64 = 1.0;
  if (norm) {
    double ss = 0.0;
    for (int pc = p0 + lane; pc < p1; pc += 32) {
      const uint2 v = __ldg(xr + pc);
      const float a0 = __uint_as_float(v.x << 16), a1 = __uint_as_float(v.x & 0xFFFF0000u);
      const float a2 = __uint_as_float(v.y << 16), a3 = __uint_as_float(v.y & 0xFFFF0000u);
      ss += double(a0 * a0) + double(a1 * a1) + double(a2 * a2) + double(a3 * a3);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) red_ss[warp] = ss;
    __syncthreads();
    double tot = 0.0;
#pragma unroll
    for (int q = 0; q < kRowParts; ++q) tot += red_ss[q];
    r64 = 1.0 / sqrt(tot / double(d) + double(r.eps));
    r32 = float(r64);
    if (blockIdx.y == 0 && threadIdx.x == 0) r.rnorm[t] = r32;
  }
  float acc[kRowExp] = {0.f, 0.f, 0.f, 0.f};
  for (int base = p0; base < p1; base += 32 * kRowIt) {
    uint2 xv[kRowIt];
    float4 wv[kRowExp][kRowIt];
    float4 gv[kRowIt];
#pragma unroll
    for (int it = 0; it < kRowIt; ++it) {
      const int pc = base + lane + 32 * it;
      const bool in = pc < p1;
      xv[it] = in ? __ldg(xr + pc) : make_uint2(0, 0);
      gv[it] = (in && norm) ? __ldg(reinterpret_cast<const float4*>(g) + pc)
                            : make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
      for (int j = 0; j < kRowExp; ++j)
        wv[j][it] = (in && e0 + j < E)
                        ? __ldg(reinterpret_cast<const float4*>(rw + (size_t)(e0 + j) * d) + pc)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int it = 0; it < kRowIt; ++it) {
      const int pc = base + lane + 32 * it;
      const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&xv[it].x);
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&xv[it].y);
      float x0 = __low2float(a), x1 = __high2float(a), x2 = __low2float(b), x3 = __high2float(b);
      if (norm) {                                // the MoE input: bf16(x·g/rms)
        x0 = rms_scaled_bf16(x0, gv[it].x, r32, r64);
        x1 = rms_scaled_bf16(x1, gv[it].y, r32, r64);
        x2 = rms_scaled_bf16(x2, gv[it].z, r32, r64);
        x3 = rms_scaled_bf16(x3, gv[it].w, r32, r64);
        if (blockIdx.y == 0 && pc < p1) {
          const __nv_bfloat162 lo = __floats2bfloat162_rn(x0, x1), hi = __floats2bfloat162_rn(x2, x3);
          uint2 o;
          o.x = *reinterpret_cast<const uint32_t*>(&lo);
          o.y = *reinterpret_cast<const uint32_t*>(&hi);
          reinterpret_cast<uint2*>(r.xn + (size_t)t * d)[pc] = o;
        }
      }
#pragma unroll
      for (int j = 0; j < kRowExp; ++j)
        acc[j] = fmaf(x3, wv[j][it].w, fmaf(x2, wv[j][it].z, fmaf(x1, wv[j][it].y, fmaf(x0, wv[j][it].x, acc[j]))));
    }
  }
#pragma unroll
  for (int j = 0; j < kRowExp; ++j)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < kRowExp; ++j) red[warp][j] = acc[j];
  }
  __syncthreads();
  if (warp == 0 && lane < kRowExp && e0 + lane < E) {
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < kRowParts; ++q) v += red[q][lane];
    r.logit_part[(size_t)t * E + e0 + lane] = v;
  }
  // the block-scaled design's token tables (the xn row this CTA wrote above is
  // visible to all its threads after the barrier)
  if (blockIdx.y == 0 && r.xq_hi)
    quantize_rows_mx(r.x, t, 1, d, r.xq_hi, r.xq_lo, r.sx_hi, r.sx_lo, r.ld_sx);
}

// The block's RMSNorm for larger batches, before the split logits kernel: one
// warp per token writes xn = bf16(x·g/rms) and 1/rms (as the rows kernel does).
__global__ void __launch_bounds__(kThreads)
rms_norm_kernel(const RouteArgs r) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kThreads / 32) + warp;
  pdl_wait();
  if (t >= r.T) return;
  const int np = r.d / 4;
  const uint2* xr = reinterpret_cast<const uint2*>(r.x_pre + (size_t)t * r.d);
  double ss = 0.0;
  for (int pc = lane; pc < np; pc += 32) {
    const uint2 v = __ldg(xr + pc);
    const float a0 = __uint_as_float(v.x << 16), a1 = __uint_as_float(v.x & 0xFFFF0000u);
    const float a2 = __uint_as_float(v.y << 16), a3 = __uint_as_float(v.y & 0xFFFF0000u);
    ss += double(a0 * a0) + double(a1 * a1) + double(a2 * a2) + double(a3 * a3);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const double r64 = 1.0 / sqrt(ss / double(r.d) + double(r.eps));
  const float r32 = float(r64);
  if (lane == 0) r.rnorm[t] = r32;
  uint2* dst = reinterpret_cast<uint2*>(r.xn + (size_t)t * r.d);
  for (int pc = lane; pc < np; pc += 32) {
    const uint2 v = __ldg(xr + pc);
    const float4 gv = __ldg(reinterpret_cast<const float4*>(r.norm_w) + pc);
    const float x0 = rms_scaled_bf16(__uint_as_float(v.x << 16), gv.x, r32, r64);
    const float x1 = rms_scaled_bf16(__uint_as_float(v.x & 0xFFFF0000u), gv.y, r32, r64);
    const float x2 = rms_scaled_bf16(__uint_as_float(v.y << 16), gv.z, r32, r64);
    const float x3 = rms_scaled_bf16(__uint_as_float(v.y & 0xFFFF0000u), gv.w, r32, r64);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x0, x1), hi = __floats2bfloat162_rn(x2, x3);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&lo);
    o.y = *reinterpret_cast<const uint32_t*>(&hi);
    dst[pc] = o;
  }
}

// quantize: write the block-scaled design's token tables for this tile (when
// the logits kernel did not).  One warp per token of the tile.
constexpr int kTopkThreads = 32 * kTT;

template <int NPER>
__global__ void __launch_bounds__(kTopkThreads)
router_topk_kernel(const RouteArgs r, int nks, bool quantize, int32_t* __restrict__ tiles_done) {
  __shared__ float wl[kTT * kLgStride];  // logits [t][e]
  __shared__ uint32_t mask[kMaxE];       // bit t: token t of this tile picked e
  __shared__ int32_t sel[kTT][8];
  __shared__ int32_t scan_part[kTopkThreads], scan_total[257], scan_off[257];
  static_assert(kTopkThreads >= 24, "the one-tile scan keeps 3 x 8 warp totals in scan_part");
  __shared__ int last_cta;

  const float* __restrict__ part = r.logit_part;
  const float* __restrict__ rb = r.router_b;
  const int T = r.T, E = r.E, k = r.k;
  int32_t* __restrict__ topk_idx = r.topk_idx;
  float* __restrict__ topk_w = r.topk_w;
  int32_t* __restrict__ rank = r.rank;
  int32_t* __restrict__ tile_counts = r.tile_counts;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTT;
  const int ntok = min(kTT, T - t0);
  for (int e = tid; e < kMaxE; e += kTopkThreads) mask[e] = 0u;
  pdl_wait();

  // logits = the K-range partial sums in a fixed order, then the bias (up to
  // 8 partials are all loaded before any is added, one round of loads)
  for (int idx = tid; idx < ntok * E; idx += kTopkThreads) {
    const int tl = idx / E, e = idx - tl * E;
    const float* p = part + (size_t)(t0 + tl) * E + e;
    const size_t stride = (size_t)T * E;
    float v = 0.f;
    if (nks <= 8) {
      float pv[8];
#pragma unroll
      for (int s = 0; s < 8; ++s) pv[s] = s < nks ? p[s * stride] : 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (s < nks) v += pv[s];
    } else {
      for (int s = 0; s < nks; ++s) v += p[s * stride];
    }
    wl[tl * kLgStride + e] = v + rb[e];
  }
  __syncthreads();

  // top-k of token `warp`: k rounds of a warp-wide (logit desc, index asc)
  // maximum over the experts not yet taken; lane j keeps slot j.  A logit is
  // compared through an order-preserving unsigned key (NaN as -inf, -0 as +0,
  // taken experts as key 0, below every logit), so a round is one warp max of
  // the keys and one warp min of the indices holding that key.
  if (warp < ntok) {
    const int tl = warp, t = t0 + tl;
    uint32_t key[NPER];
#pragma unroll
    for (int j = 0; j < NPER; ++j) {
      const int e = lane + 32 * j;
      float lv = (e < E) ? wl[tl * kLgStride + e] : -INFINITY;
      lv = isnan(lv) ? -INFINITY : lv + 0.0f;
      const uint32_t u = __float_as_uint(lv);
      key[j] = (e < E) ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
    }
    int my_e = 0;
    float my_l = -INFINITY;
    for (int j = 0; j < k; ++j) {
      uint32_t bk = 0u, be = 0xFFFFFFFFu;        // this lane's best (lowest expert on ties)
#pragma unroll
      for (int q = 0; q < NPER; ++q)
        if (key[q] > bk) { bk = key[q]; be = uint32_t(lane + 32 * q); }
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
      const uint32_t emin = __reduce_min_sync(0xffffffffu, bk == kmax ? be : 0xFFFFFFFFu);
      if ((emin & 31u) == uint32_t(lane)) {
#pragma unroll
        for (int q = 0; q < NPER; ++q)
          if (q == int(emin >> 5)) key[q] = 0u;
      }
      if (lane == j) {
        my_e = int(emin);
        my_l = __uint_as_float((kmax & 0x80000000u) ? (kmax & 0x7FFFFFFFu) : ~kmax);
      }
    }
    // softmax over the k selected logits: exp(l_j - l_0), summed in slot order
    const float m = __shfl_sync(0xffffffffu, my_l, 0);
    const float pj = lane < k ? expf(my_l - m) : 0.f;
    float ssum = 0.f;
    for (int j = 0; j < k; ++j) ssum += __shfl_sync(0xffffffffu, pj, j);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = my_e;
      topk_w[(size_t)t * k + lane] = pj * (1.0f / ssum);
      sel[tl][lane] = my_e;
      atomicOr(&mask[my_e], 1u << tl);             // order-free: deterministic
    }
  }
  __syncthreads();

  for (int e = tid; e < E; e += kTopkThreads)
    tile_counts[(size_t)blockIdx.x * E + e] = __popc(mask[e]);
  for (int q = tid; q < ntok * k; q += kTopkThreads) {
    const int tl = q / k, j = q - tl * k;
    const int e = sel[tl][j];
    rank[(size_t)(t0 + tl) * k + j] = __popc(mask[e] & ((1u << tl) - 1u));
  }

  if (tiles_done != nullptr && gridDim.x == 1) {
    // One router tile (T <= 32): the expert scan and the permutation from this
    // CTA's shared tables; no other CTA to count or wait for.
    __syncthreads();
    const int lane_e = tid & 31, wid = tid >> 5;
    const int32_t v = tid < E ? __popc(mask[tid]) : 0;
    const int32_t c = tid < E ? (v + r.chunk - 1) / r.chunk : 0;
    const int32_t c2 = tid < E ? (v + r.chunk2 - 1) / r.chunk2 : 0;
    int32_t iv = v, ic = c, ic2 = c2;            // inclusive scans inside each warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t pv = __shfl_up_sync(0xffffffffu, iv, o);
      const int32_t pc = __shfl_up_sync(0xffffffffu, ic, o);
      const int32_t pc2 = __shfl_up_sync(0xffffffffu, ic2, o);
      if (lane_e >= o) { iv += pv; ic += pc; ic2 += pc2; }
    }
    if (lane_e == 31 && wid < 8) { scan_part[wid] = iv; scan_part[8 + wid] = ic; scan_part[16 + wid] = ic2; }
    __syncthreads();
    if (tid < E) {
      int32_t bv = 0, bc = 0, bc2 = 0;           // the earlier warps' totals, in order
      for (int w2 = 0; w2 < wid; ++w2) {
        bv += scan_part[w2];
        bc += scan_part[8 + w2];
        bc2 += scan_part[16 + w2];
      }
      const int32_t ev = bv + iv - v, ec = bc + ic - c, ec2 = bc2 + ic2 - c2;
      scan_off[tid] = ev;
      r.offsets[tid] = ev;
      r.tile_base[tid] = ev;
      r.mtile_off[tid] = ec;
      r.mtile_off[E + 1 + tid] = ec2;
      if (tid == E - 1) {
        r.offsets[E] = ev + v;
        r.mtile_off[E] = ec + c;
        r.mtile_off[2 * E + 1] = ec2 + c2;
      }
    }
    __syncthreads();
    if (r.perm) {                                // row = expert base + rank among its tokens
      for (int q = tid; q < ntok * k; q += kTopkThreads) {
        const int tl = q / k, j = q - tl * k;
        const int e = sel[tl][j];
        const int row = scan_off[e] + __popc(mask[e] & ((1u << tl) - 1u));
        r.perm[row] = q;
        r.inv[q] = row;
      }
    }
  } else if (tiles_done != nullptr) {
    // With few tiles the CTA that finishes last also runs the expert scan (the
    // counter was zeroed by the logits kernel of this call).
    __threadfence();
    __syncthreads();
    if (tid == 0) last_cta = atomicAdd(tiles_done, 1) == int(gridDim.x) - 1;
    __syncthreads();
    if (last_cta) {
      __threadfence();
      scan_tiles<kTopkThreads>(tile_counts, int(gridDim.x), E, r.chunk, r.chunk2, r.tile_base,
                               r.offsets, r.mtile_off, scan_part, scan_total, scan_off);
      if (r.perm) {
        // every routed row's place: the (tile, expert) base this CTA just
        // wrote plus the row's rank in its tile (other CTAs wrote those)
        __syncthreads();
        const int R = T * k;
        for (int q = tid; q < R; q += kTopkThreads) {
          const int e = __ldcg(topk_idx + q);
          const int row = __ldcg(r.tile_base + (size_t)(q / k / kTT) * E + e) + __ldcg(rank + q);
          if (e < 0 || e >= E || row < 0 || row >= R) {
            atomicMax(r.status, kStatusBounds);
            continue;
          }
          r.perm[row] = q;
          r.inv[q] = row;
        }
      }
    }
  }
  if (quantize)
    quantize_rows_mx(r.x, t0, ntok, r.d, r.xq_hi, r.xq_lo, r.sx_hi, r.sx_lo, r.ld_sx);
}

}  // namespace

cudaError_t launch_router_topk(const RouteArgs& r, bool* scanned, cudaStream_t s) {
  const int T = r.T, d = r.d, E = r.E;
  const int ntiles = (T + kTT - 1) / kTT;
  const bool rows = ntiles <= kFuseScanTiles;   // decode-sized: whole dot products
  const bool tc = !rows && router_tc_fits(T, d, E) && r.rw_terms != nullptr;
  int nks = rows ? 1 : router_splits(T, d, E);
  const int kc = router_split_len(T, d, E);
  const int eg = router_expert_group(T, E);
  const dim3 g1(ntiles, nks, (E + eg - 1) / eg);
  const int nper_g = eg / 32;                    // experts per lane in the logits kernel
  const int nper = (E + 31) / 32;                // ... and in the top-k kernel
  if (nper_g < 1 || nper_g > 8 || nper > 8) return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  if (rows) {
    e = launch_pdl(router_logits_rows_kernel, dim3(T, (E + kRowExp - 1) / kRowExp), dim3(kThreads), 0,
                   s, r);
  } else if (r.x_pre) {
    // the block: the normalised table first; the logits kernel reads it
    e = launch_pdl(rms_norm_kernel, dim3((T + kThreads / 32 - 1) / (kThreads / 32)), dim3(kThreads),
                   0, s, r);
  }
#define MOE_LOGITS_CASE(N)                                                                   \
  case N:                                                                                    \
    e = launch_pdl(router_logits_kernel<N>, g1, dim3(kThreads), 0, s, r, kc, eg);             \
    break;
  if (tc) e = launch_router_logits_tc(r, &nks, s);
  switch (rows || tc ? 0 : nper_g) {
    MOE_LOGITS_CASE(1)
    MOE_LOGITS_CASE(2)
    MOE_LOGITS_CASE(3)
    MOE_LOGITS_CASE(4)
    MOE_LOGITS_CASE(5)
    MOE_LOGITS_CASE(6)
    MOE_LOGITS_CASE(7)
    MOE_LOGITS_CASE(8)
  }
#undef MOE_LOGITS_CASE
  if (e != cudaSuccess) return e;
  // few tiles: the last top-k CTA runs the expert scan (no separate launch)
  const bool fuse = ntiles <= kFuseScanTiles && r.tile_base != nullptr;
  int32_t* done = fuse ? r.status + 1 : nullptr;
  if (scanned) *scanned = fuse;
  RouteArgs rt = r;
  if (!fuse) rt.perm = rt.inv = nullptr;          // the scatter kernel writes them
  const bool quantize = !rows && r.xq_hi != nullptr;
#define MOE_TOPK_CASE(N)                                                                     \
  case N:                                                                                    \
    e = launch_pdl(router_topk_kernel<N>, dim3(ntiles), dim3(kTopkThreads), 0, s, rt, nks,   \
                   quantize, done);                                                          \
    break;
  switch (nper) {
    MOE_TOPK_CASE(1)
    MOE_TOPK_CASE(2)
    MOE_TOPK_CASE(3)
    MOE_TOPK_CASE(4)
    MOE_TOPK_CASE(5)
    MOE_TOPK_CASE(6)
    MOE_TOPK_CASE(7)
    MOE_TOPK_CASE(8)
  }
#undef MOE_TOPK_CASE
  return e;
}

}  // namespace moe
