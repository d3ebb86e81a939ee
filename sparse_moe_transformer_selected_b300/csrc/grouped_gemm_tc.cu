// K3 / K4 — grouped expert GEMMs on the 5th-generation tensor cores (tcgen05).
//
// Each expert's segment of the permuted rows is multiplied by that expert's
// MXFP4 weights ("OpenAI 最新开源模型 gpt-oss 架构与训练解析", 模型架构: MoE
// weights in MXFP4, experts are gated-SwiGLU FFNs with clamping and the +1
// term on the up branch; the same page's 更深对比更宽 section: d = W = 2880).
//
// Persistent kernel, one CTA per SM, warp-specialised:
//   warp 0      TMA producer: activation tiles (128 rows x 64 K, 128B swizzle)
//   warp 1      MMA issuer: tcgen05.mma kind::f16, M=128 N=256 K=16, fp32 in TMEM
//   warp 2      TMEM allocator (512 columns: two 256-column accumulators)
//   warps 4-7   epilogue: tcgen05.ld, scale, bias, SwiGLU (K3) / store y (K4)
//   warps 8-15  dequantisers: MXFP4 codes streamed from HBM through registers,
//               converted to f16/bf16 and written to the B tile (128B swizzle)
// Work unit = (row tile of one expert, N tile); units are dealt round-robin.
//
// Number formats (exact):
//   K3: A = x in f16, each token pre-scaled by 2^e_t so its largest |x| is in
//       [2^14, 2^15) (a bf16 value has 8 significant bits, so this is exact);
//       B = E2M1 codes -> f16 (cvt.rn.f16x2.e2m1x2) times 2^(s - r_n), r_n the
//       largest scale byte of weight row n; the epilogue multiplies by
//       2^(-e_t) * 2^(r_n - 127).  Exact whenever the scales of a row lie within
//       2^23 of each other.
//   K4: A = h as two bf16 terms (hi + lo); B = E2M1 -> f16 -> bf16 bit pattern
//       (a power-of-two rescale) times 2^(s - 15), exact for every scale < 143.
#include "common.cuh"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <math.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kBM = kGemmBM;     // 128
constexpr int kBK = 64;          // K per stage: one 128-byte swizzle row of 16-bit values
constexpr int kBN = 256;         // MMA N
constexpr int kThreads = 512;
constexpr int kWarpTMA = 0, kWarpMMA = 1, kWarpTmem = 2, kWarpEpi0 = 4, kWarpDq0 = 8;
constexpr int kDqWarps = 8;
constexpr int kATileBytes = kBM * kBK * 2;   // 16 KB
constexpr int kBTileBytes = kBN * kBK * 2;   // 32 KB
constexpr int kTmemCols = 512;
constexpr long long kSpinLimit = 4000000000ll;   // clock cycles (~2 s) before giving up

enum class Mode { GateUp, Down };

template <Mode M>
struct Cfg;
template <>
struct Cfg<Mode::GateUp> {
  static constexpr int NA = 1;        // A tiles per stage: x
  static constexpr int STAGES = 4;
  static constexpr bool kBf16 = false;
};
template <>
struct Cfg<Mode::Down> {
  static constexpr int NA = 2;        // h_hi, h_lo
  static constexpr int STAGES = 3;
  static constexpr bool kBf16 = true;
};

template <Mode M>
struct Smem {
  static constexpr int NA = Cfg<M>::NA, STAGES = Cfg<M>::STAGES;
  static constexpr int kRing = STAGES + 3;
  static constexpr int kStageBytes = NA * kATileBytes + kBTileBytes;
  static constexpr int kTiles = STAGES * kStageBytes;
  static constexpr int kColfac = kTiles;                                   // float[kRing][kBN]
  static constexpr int kBars = kColfac + kRing * kBN * 4;                  // uint64 barriers
  static constexpr int kNumBars = 3 * STAGES + 4 + 1 + kRing;
  static constexpr int kMisc = kBars + kNumBars * 8;                       // tmem base, abort
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;                             // alignment slack
};

struct Unit {
  int e, r0, seg_end, n0;
};

__device__ __forceinline__ int expert_of_tile(const int32_t* mtile_off, int E, int g) {
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(mtile_off + mid) <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Units are dealt row-tile-major: the CTAs in flight share a few activation
// row tiles (and the weights of one or two experts), which stay in L2.
__device__ __forceinline__ Unit unit_of(const GemmArgs& a, int n_tiles, int u, int n_step) {
  const int g = u / n_tiles, nt = u - g * n_tiles;
  Unit w;
  w.e = expert_of_tile(a.mtile_off, a.E, g);
  const int off = __ldg(a.offsets + w.e);
  w.r0 = off + (g - __ldg(a.mtile_off + w.e)) * kBM;
  w.seg_end = __ldg(a.offsets + w.e + 1);
  w.n0 = nt * n_step;
  return w;
}

// Bounded wait: true when the phase completed; false after a timeout (which is
// recorded in the status word) or when another thread of the CTA gave up.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           int32_t* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kSpinLimit) {
      *abort_flag = 1;
      atomicMax(status, kStatusTimeout);
      return false;
    }
  }
}

// ------------------------------------------------------------- dequant --

// 2^delta as an f16x2 pair (delta <= 0); 0 below the f16 subnormal range.
__device__ __forceinline__ uint32_t f16x2_pow2(int delta) {
  uint32_t b;
  if (delta >= -14) b = uint32_t(delta + 15) << 10;
  else if (delta >= -24) b = 1u << (delta + 24);
  else b = 0;
  return b | (b << 16);
}

// 2^p as a bf16x2 pair, -126 <= p <= 127.
__device__ __forceinline__ uint32_t bf16x2_pow2(int p) {
  const uint32_t b = uint32_t(p + 127) << 7;
  return b | (b << 16);
}

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hmul2_bf16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 8 E2M1 codes (one 32-bit word, even K index in the low nibble of each byte)
// -> 4 f16x2 words holding K pairs (0,1), (2,3), (4,5), (6,7).
__device__ __forceinline__ uint4 e2m1x8_to_f16(uint32_t w) {
  uint4 r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "r"(w));
  return r;
}

// f16 bit pattern of an E2M1 value -> bf16 bit pattern of the same value times
// 2^-112 (move the exponent/mantissa field right by 3, keep the sign).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_scaled(uint32_t t) {
  return ((t >> 3) & 0x0FFF0FFFu) ^ (t & 0x80008000u);
}

template <Mode M>
struct Dequant;

template <>
struct Dequant<Mode::GateUp> {
  // factor for one 32-element block: 2^(s - r_n) in f16
  __device__ __forceinline__ static uint32_t factor(int s, int rn) { return f16x2_pow2(s - rn); }
  __device__ __forceinline__ static uint4 convert(uint32_t w, uint32_t f) {
    uint4 v = e2m1x8_to_f16(w);
    v.x = hmul2_f16(v.x, f);
    v.y = hmul2_f16(v.y, f);
    v.z = hmul2_f16(v.z, f);
    v.w = hmul2_f16(v.w, f);
    return v;
  }
};

template <>
struct Dequant<Mode::Down> {
  // factor 2^(s - 15) in bf16 (the bit move left a factor 2^-112); rn unused.
  __device__ __forceinline__ static uint32_t factor(int s, int) {
    return bf16x2_pow2(min(s - 15, 127));
  }
  __device__ __forceinline__ static uint4 convert(uint32_t w, uint32_t f) {
    uint4 v = e2m1x8_to_f16(w);
    v.x = hmul2_bf16(f16x2_to_bf16x2_scaled(v.x), f);
    v.y = hmul2_bf16(f16x2_to_bf16x2_scaled(v.y), f);
    v.z = hmul2_bf16(f16x2_to_bf16x2_scaled(v.z), f);
    v.w = hmul2_bf16(f16x2_to_bf16x2_scaled(v.w), f);
    return v;
  }
};

// ------------------------------------------------------------- kernel --

template <Mode M>
__global__ void __launch_bounds__(kThreads, 1)
moe_gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a0,
                   const __grid_constant__ CUtensorMap map_a1, const GemmArgs a) {
  using C = Cfg<M>;
  using S = Smem<M>;
  constexpr int NA = C::NA, STAGES = C::STAGES;
  constexpr bool kGateUp = (M == Mode::GateUp);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* colfac = reinterpret_cast<float*>(smem + S::kColfac);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBars);
  uint64_t* a_full = bars;                    // [STAGES] TMA bytes landed
  uint64_t* b_full = bars + STAGES;           // [STAGES] dequantised B written (8 warps)
  uint64_t* empty = bars + 2 * STAGES;        // [STAGES] MMAs reading the stage done
  uint64_t* acc_full = bars + 3 * STAGES;     // [2]
  uint64_t* acc_empty = acc_full + 2;         // [2]
  uint64_t* mma_done = acc_full + 4;          // [1] final drain
  uint64_t* cf_ready = acc_full + 5;          // [kRing] column factors of a unit written
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(smem + S::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = kGateUp ? a.d : a.W;                    // reduction length
  const int KB = (K + kBK - 1) / kBK;
  const int n_step = kGateUp ? kBN / 2 : kBN;           // output columns per unit
  const int n_out = kGateUp ? a.W : a.d;
  const int n_tiles = (n_out + n_step - 1) / n_step;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&a_full[s], 1);
      ptx::mbar_init(&b_full[s], kDqWarps);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&acc_full[b], 1);
      ptx::mbar_init(&acc_empty[b], 4);
    }
    ptx::mbar_init(mma_done, 1);
    for (int r = 0; r < S::kRing; ++r) ptx::mbar_init(&cf_ready[r], kDqWarps);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpTmem) {
    ptx::tmem_alloc(tmem_base_p, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_base_p;
  pdl_wait();
  const int units = __ldg(a.mtile_off + a.E) * n_tiles;   // row tiles x N tiles

  if (warp == kWarpTMA) {
    // ------------------------------------------------------ TMA producer --
    if (ptx::elect_one()) {
      ptx::tma_prefetch_desc(&map_a0);
      if (NA > 1) ptx::tma_prefetch_desc(&map_a1);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;    // bit s: stage s received a load
      uint32_t lastph = 0;    // bit s: phase parity of that last load
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_of(a, n_tiles, u, n_step);
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_phase(&empty[stage], phase ^ 1, abort_flag, a.status)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&a_full[stage], NA * kATileBytes);
          uint8_t* st = smem + stage * S::kStageBytes;
          ptx::tma_load_2d(st, &map_a0, &a_full[stage], kb * kBK, w.r0);
          if (NA > 1) ptx::tma_load_2d(st + kATileBytes, &map_a1, &a_full[stage], kb * kBK, w.r0);
          issued |= 1u << stage;
          lastph = (lastph & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // on abort, the loads already issued must land before the CTA exits
        const long long t0 = clock64();
        for (int st = 0; st < STAGES; ++st) {
          if (!(issued >> st & 1u)) continue;
          while (!ptx::mbar_try_wait(&a_full[st], (lastph >> st) & 1u) &&
                 clock64() - t0 < kSpinLimit) {
          }
        }
      }
    }
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------- MMA issuer --
    if (ptx::elect_one()) {
      constexpr uint32_t idesc = ptx::idesc_f16(kBM, kBN, C::kBf16);
      int stage = 0;
      uint32_t phase = 0;
      int q = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++q) {
        const int buf = q & 1;
        if (!wait_phase(&acc_empty[buf], ((q >> 1) & 1) ^ 1, abort_flag, a.status)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kBN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_phase(&a_full[stage], phase, abort_flag, a.status) ||
              !wait_phase(&b_full[stage], phase, abort_flag, a.status)) { ok = false; break; }
          ptx::tc_fence_after();
          uint8_t* st = smem + stage * S::kStageBytes;
          const uint64_t bdesc = ptx::desc_kmajor_sw128(ptx::smem_u32(st + NA * kATileBytes));
#pragma unroll
          for (int t = 0; t < NA; ++t) {
            const uint64_t adesc = ptx::desc_kmajor_sw128(ptx::smem_u32(st + t * kATileBytes));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              // +32 bytes per K=16 step inside the 128-byte swizzled row
              ptx::mma_f16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                           (kb | kk | t) != 0 ? 1u : 0u);
            }
          }
          ptx::mma_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        ptx::mma_commit(&acc_full[buf]);
      }
      // all issued MMAs complete before TMEM is released
      ptx::mma_commit(mma_done);
      const long long t0 = clock64();
      while (!ptx::mbar_try_wait(mma_done, 0) && clock64() - t0 < kSpinLimit) {
      }
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
    // --------------------------------------------------------- epilogue --
    const int quarter = warp - kWarpEpi0;       // == warp % 4: TMEM lanes 32*quarter..
    const int row = quarter * 32 + lane;
    int q = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++q) {
      const Unit w = unit_of(a, n_tiles, u, n_step);
      const int buf = q & 1;
      bool ok = wait_phase(&acc_full[buf], (q >> 1) & 1, abort_flag, a.status) &&
                wait_phase(&cf_ready[q % S::kRing], (q / S::kRing) & 1, abort_flag, a.status);
      if (!__all_sync(0xffffffffu, ok)) break;     // warp-uniform: tcgen05.ld is .sync.aligned
      ptx::tc_fence_after();
      const int r = w.r0 + row;
      const bool valid = r < w.seg_end;
      const float* cf = colfac + (q % S::kRing) * kBN;
      const uint32_t tbase = tmem_base + (uint32_t(quarter * 32) << 16) + buf * kBN;
      if constexpr (kGateUp) {
        const float rowf = valid ? ldexpf(1.0f, -a.rowexp[r]) : 0.f;
        const __nv_bfloat16* bg = a.b_gu + size_t(w.e) * 2 * a.W;
#pragma unroll 1
        for (int c = 0; c < kBN / 2; c += 32) {
          uint32_t g[32], up[32];
          ptx::tmem_ld_32x32b_x32(tbase + c, g);
          ptx::tmem_ld_32x32b_x32(tbase + kBN / 2 + c, up);
          ptx::tmem_ld_wait();
          const int nb = w.n0 + c;
          if (valid && nb < a.W) {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float hv[2];
#pragma unroll
              for (int p = 0; p < 2; ++p) {
                const int jj = j + p;
                const int n = min(nb + jj, a.W - 1);
                const float zg = __uint_as_float(g[jj]) * rowf * cf[c + jj] + __bfloat162float(bg[n]);
                const float zu = __uint_as_float(up[jj]) * rowf * cf[kBN / 2 + c + jj] +
                                 __bfloat162float(bg[a.W + n]);
                const float gg = fminf(zg, a.limit);
                const float uu = fminf(fmaxf(zu, -a.limit), a.limit);
                hv[p] = gg * (1.0f / (1.0f + expf(-a.alpha * gg))) * (uu + 1.0f);
              }
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(hv[0], hv[1]);
              const float2 hf = __bfloat1622float2(h2);
              const __nv_bfloat162 l2 = __floats2bfloat162_rn(hv[0] - hf.x, hv[1] - hf.y);
              hi[j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
              lo[j / 2] = *reinterpret_cast<const uint32_t*>(&l2);
            }
            __nv_bfloat16* ph = a.h_hi + size_t(r) * a.W + nb;
            __nv_bfloat16* pl = a.h_lo + size_t(r) * a.W + nb;
            if (nb + 32 <= a.W) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                reinterpret_cast<uint4*>(ph)[v] = make_uint4(hi[4 * v], hi[4 * v + 1], hi[4 * v + 2], hi[4 * v + 3]);
                reinterpret_cast<uint4*>(pl)[v] = make_uint4(lo[4 * v], lo[4 * v + 1], lo[4 * v + 2], lo[4 * v + 3]);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (nb + j < a.W) {
                  reinterpret_cast<uint16_t*>(ph)[j] = uint16_t(hi[j / 2] >> (16 * (j & 1)));
                  reinterpret_cast<uint16_t*>(pl)[j] = uint16_t(lo[j / 2] >> (16 * (j & 1)));
                }
              }
            }
          }
        }
      } else {
        const __nv_bfloat16* bd = a.b_dn + size_t(w.e) * a.d;
#pragma unroll 1
        for (int c = 0; c < kBN; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tbase + c, v);
          ptx::tmem_ld_wait();
          const int nb = w.n0 + c;
          if (valid && nb < a.d) {
            float* py = a.y + size_t(r) * a.d + nb;
            if (nb + 32 <= a.d) {
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                float4 o;
                o.x = __uint_as_float(v[j + 0]) * cf[c + j + 0] + __bfloat162float(bd[nb + j + 0]);
                o.y = __uint_as_float(v[j + 1]) * cf[c + j + 1] + __bfloat162float(bd[nb + j + 1]);
                o.z = __uint_as_float(v[j + 2]) * cf[c + j + 2] + __bfloat162float(bd[nb + j + 2]);
                o.w = __uint_as_float(v[j + 3]) * cf[c + j + 3] + __bfloat162float(bd[nb + j + 3]);
                *reinterpret_cast<float4*>(py + j) = o;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (nb + j < a.d)
                  py[j] = __uint_as_float(v[j]) * cf[c + j] + __bfloat162float(bd[nb + j]);
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_empty[buf]);
    }
  } else if (warp >= kWarpDq0) {
    // ------------------------------------------------------ dequantisers --
    const int i = threadIdx.x - kWarpDq0 * 32;      // B row of the tile, 0..255
    const int rows_per_expert = kGateUp ? 2 * a.W : a.d;
    const uint8_t* wcodes = kGateUp ? a.w_gu : a.w_dn;
    const uint8_t* wscale = kGateUp ? a.w_gu_scale : a.w_dn_scale;
    const int nsb = K / 32;                         // scale bytes per row
    int stage = 0;
    uint32_t phase = 0;
    int q = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++q) {
      const Unit w = unit_of(a, n_tiles, u, n_step);
      int nrow;
      bool valid;
      if constexpr (kGateUp) {
        const int h = i & (kBN / 2 - 1);
        valid = w.n0 + h < a.W;
        nrow = (i < kBN / 2) ? w.n0 + h : a.W + w.n0 + h;
      } else {
        nrow = w.n0 + i;
        valid = nrow < a.d;
      }
      const size_t wrow = size_t(w.e) * rows_per_expert + (valid ? nrow : 0);
      const uint8_t* crow = wcodes + wrow * (K / 2);
      const uint8_t* srow = wscale + wrow * nsb;
      int rn = 0;
      if (valid) {
#pragma unroll 8
        for (int j = 0; j < nsb; ++j) rn = max(rn, int(__ldg(srow + j)));
      }
      colfac[(q % S::kRing) * kBN + i] = valid ? (kGateUp ? ldexpf(1.0f, rn - 127) : 1.0f) : 0.f;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&cf_ready[q % S::kRing]);

      // register prefetch ring: 4 K-blocks of codes (2 x 16 B) and their 2 scales
      uint4 ca[4], cb[4];
      uint32_t sc[4];
      auto load = [&](int kb, uint4& x0, uint4& x1, uint32_t& s) {
        x0 = make_uint4(0, 0, 0, 0);
        x1 = make_uint4(0, 0, 0, 0);
        s = 0;
        if (!valid || kb >= KB) return;
        const int k0 = kb * kBK;
        const uint4* p = reinterpret_cast<const uint4*>(crow + k0 / 2);
        x0 = __ldg(p);
        s = __ldg(srow + k0 / 32);
        if (k0 + 32 < K) {
          x1 = __ldg(p + 1);
          s |= uint32_t(__ldg(srow + k0 / 32 + 1)) << 8;
        }
      };
#pragma unroll
      for (int p = 0; p < 4; ++p) load(p, ca[p], cb[p], sc[p]);
      for (int kb0 = 0; kb0 < KB && ok; kb0 += 4) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int kb = kb0 + p;
          if (kb >= KB) break;
          const uint4 x0 = ca[p], x1 = cb[p];
          const uint32_t s = sc[p];
          load(kb + 4, ca[p], cb[p], sc[p]);
          ok = __all_sync(0xffffffffu, wait_phase(&empty[stage], phase ^ 1, abort_flag, a.status));
          if (!ok) break;
          const uint32_t f0 = Dequant<M>::factor(int(s & 0xFF), rn);
          const uint32_t f1 = Dequant<M>::factor(int(s >> 8), rn);
          uint8_t* bt = smem + stage * S::kStageBytes + NA * kATileBytes;
          const uint32_t wv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = Dequant<M>::convert(wv[c], c < 4 ? f0 : f1);
            *reinterpret_cast<uint4*>(bt + ptx::sw128_offset(i, c)) = v;
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&b_full[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpTmem) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host --

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major [rows, cols] 16-bit matrix, box 64 x 128, 128-byte swizzle.
cudaError_t make_map(CUtensorMap* map, const void* base, int rows, int cols, bool bf16) {
  auto enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  const cuuint32_t box[2] = {cuuint32_t(kBK), cuuint32_t(kBM)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <Mode M>
cudaError_t launch(const GemmArgs& a, cudaStream_t s) {
  using S = Smem<M>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_tc_kernel<M>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  CUtensorMap m0, m1;
  cudaError_t e;
  if (M == Mode::GateUp) {
    e = make_map(&m0, a.x_perm, a.R, a.d, false);
    m1 = m0;
  } else {
    e = make_map(&m0, a.h_hi, a.R, a.W, true);
    if (e == cudaSuccess) e = make_map(&m1, a.h_lo, a.R, a.W, true);
  }
  if (e != cudaSuccess) return e;
  const int n_step = (M == Mode::GateUp) ? kBN / 2 : kBN;
  const int n_out = (M == Mode::GateUp) ? a.W : a.d;
  const long long units_bound = (long long)(a.R / kBM + a.E) * ((n_out + n_step - 1) / n_step);
  const int grid = int(units_bound < num_sms() ? units_bound : num_sms());
  return launch_pdl(moe_gemm_tc_kernel<M>, dim3(grid), dim3(kThreads), S::kAlloc, s, m0, m1, a);
}

}  // namespace

cudaError_t launch_gateup(const GemmArgs& a, cudaStream_t s) { return launch<Mode::GateUp>(a, s); }
cudaError_t launch_down(const GemmArgs& a, cudaStream_t s) { return launch<Mode::Down>(a, s); }

}  // namespace moe
