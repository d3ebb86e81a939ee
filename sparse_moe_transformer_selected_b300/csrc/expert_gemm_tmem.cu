// K3 / K4 — grouped expert GEMMs with the dequantised weights held in tensor
// memory (tcgen05 "A from TMEM" form).
//
// Each expert's segment of the permuted rows is multiplied by that expert's
// MXFP4 weights ("OpenAI 最新开源模型 gpt-oss 架构与训练解析", 模型架构: MoE
// weights in MXFP4, experts are gated-SwiGLU FFNs with clamping and the +1
// term on the up branch; 更深对比更宽: d = W = 2880).
//
// The weights are the M side of the MMA and the tokens the N side:
//   D[weight row, token] = Σ_k A[weight row, k] · B[token, k]
// A (128 weight rows x 128 K per A stage) is never written to shared memory:
// the packed E2M1 codes arrive by TMA (128 rows x 256 K = 16 KB per code
// stage), sixteen dequantiser warps convert them in registers and store them
// into TMEM with tcgen05.st, and tcgen05.mma reads A from TMEM.  B (a chunk of
// nb tokens x 64 K per sub-tile, 128-byte swizzle) arrives by TMA.  The chunk
// nb is 16 when experts get a few tokens each (a decode step: the kernel
// streams weights and the activation ring is many small stages deep) and up to
// 192 when they get many (prefill): every chunk costs one dequantisation of
// the expert's weights, so the fewer chunks the better, up to the point where
// two accumulators of nb columns leave tensor memory too few A stages.
//
// Persistent kernel, one CTA per SM, 24 warps:
//   warp 0      producer: scales (1-D bulk copy) and codes (TMA)
//   warp 1      MMA issuer (one elected thread)
//   warp 2      TMEM allocator (512 columns: 2 accumulators of nb columns,
//               then as many A stages of 64 columns as fit, at most 6)
//   warp 3      producer: activations (TMA, one nb-row box per operand and stage)
//   warps 4-7   epilogue, TMEM lane quarter = warp % 4
//   warps 8-23  dequantisers, lane quarter = warp % 4, K quarter of each A
//               stage = (warp - 8) / 4
// Work unit = (token chunk of one expert, weight M tile), chunk-major so a
// chunk's activations and an expert's weights stay in L2 while they are reused.
//
// Number formats (exact products, fp32 accumulation):
//   gate_up: A = E2M1 -> f16 (cvt.rn.f16x2.e2m1x2) times 2^(s - r_n), r_n the
//            largest scale byte of weight row n; B = x · 2^e_t in f16 (the
//            permute stage scales each token so its largest |x| lies in
//            [2^14, 2^15), which holds every bf16 value).  The epilogue
//            multiplies by 2^(r_n - 127) · 2^(-e_t).  Exact for every scale
//            byte whose block lies within 2^14 of its row's largest; a block
//            further below contributes nothing (its factor would be an f16
//            subnormal): each of its terms is below 2^-14 of the largest
//            weights of the row.
//   down:    when the clamp bounds h inside the f16 range, as gate_up with
//            B = h as two f16 terms (hi + lo); otherwise A = E2M1 -> f16 bits
//            moved into a bf16 field (a factor 2^-112) times 2^(s - c_n) with
//            c_n = max(15, r_n - 127), exact for every scale byte (blocks more
//            than 2^253 below the row's largest aside), the epilogue
//            multiplying by 2^(c_n - 15); B = h as two bf16 terms.  Two MMAs
//            per K step (hi, lo).
#include "combine.cuh"
#include "common.cuh"
#include "map_cache.cuh"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <math.h>

#include <cmath>
#include <mutex>

namespace moe {
namespace {

constexpr int kNBMax = 192;                  // largest token chunk (MMA N)
constexpr int kMW = 128;                     // weight rows per unit (MMA M, TMEM lanes)
constexpr int kSK = 256;                     // K per code stage: 128 B of codes per row
constexpr int kAK = 128;                     // K per A stage
constexpr int kACols = kAK / 2;              // TMEM columns per A stage (f16 pairs)
constexpr int kMaxC = 12;                    // code-ring depth, most
constexpr int kMaxA = 6;                     // A-ring depth, most
constexpr int kMaxB = 16;                    // activation-ring depth, most
constexpr int kRing = 4;                     // per-unit row-factor ring
constexpr int kThreads = 768;
constexpr int kWarpProd = 0, kWarpMMA = 1, kWarpTmem = 2, kWarpProdB = 3, kWarpEpi0 = 4,
              kWarpDq0 = 8;
// 16 dequantiser warps: 4 per TMEM lane quarter, each converting a quarter
// (32 K, 16 columns) of every 128-K A stage for its 32 weight rows, two A
// stages per code stage.  Every warp takes part in every A stage, so each
// follows the A ring slot by slot.  Four warps per SM partition hide the
// latency of each warp's load -> convert -> store chain, which two could not.
constexpr int kDqWarps = 16;
constexpr int kTmemCols = 512;
constexpr int kCodeStageBytes = kMW * kSK / 2;   // 16 KB
constexpr int kCodeBoxRows = 64;
// code, A and B rings (full + empty each), scales and accumulators (2 + 2
// each), the row-factor ring, and the final MMA drain
constexpr int kNumBars = 2 * kMaxC + 2 * kMaxA + 2 * kMaxB + 4 + 4 + 2 * kRing + 1;
constexpr long long kSpinLimit = 4000000000ll;   // clock cycles: the final drains
constexpr int kMaxSmem = 232448;                 // 227 KB opt-in per CTA

// K of one activation stage, at most one A stage: 128 for small chunks and
// for one operand (gate_up: each stage wait and release then covers 8 MMAs;
// measured faster than 64), 64 for large chunks with two operands (down: a
// 128-K stage of h hi and lo would leave only two stages in the ring;
// measured slower).
__host__ __device__ inline int act_stage_k(int nb, int nops) {
  return (nb <= 32 || nops == 1) ? 128 : 64;
}
// A stages that fit in TMEM next to two accumulators of nb columns.
__host__ __device__ inline int a_stages(int nb) {
  const int n = (kTmemCols - 2 * nb) / kACols;
  return n < kMaxA ? n : kMaxA;
}

enum class Mode { GateUp, Down };

template <Mode M>
struct Cfg;
template <>
struct Cfg<Mode::GateUp> {
  static constexpr int NOPS = 1;      // B operands per K step: x
};
template <>
struct Cfg<Mode::Down> {
  static constexpr int NOPS = 2;      // h_hi, h_lo
};

struct Lay {
  int codes, bt, bstage, sc, scbuf, rf, bars, misc, total;
};

// Shared-memory plan for reduction length K (nsb = K/32 scale bytes per row),
// token chunk nb, k experts per token and ring depths nc (codes) and nbs
// (activations).
template <Mode M>
__host__ __device__ inline Lay layout(int nsb, int nb, int k, int nc, int nbs) {
  Lay l{};
  int off = 0;
  l.codes = off;
  off += nc * kCodeStageBytes;
  l.bstage = Cfg<M>::NOPS * (act_stage_k(nb, Cfg<M>::NOPS) / 64) * nb * 128;
  l.bt = off;
  off += nbs * l.bstage;
  l.scbuf = (kMW * nsb + 15) / 16 * 16;
  l.sc = off;
  off += 2 * l.scbuf;
  l.rf = off;
  off += kRing * kMW * 4;
  off = (off + 7) & ~7;
  l.bars = off;
  off += kNumBars * 8;
  l.misc = off;
  off += 16;                          // TMEM base, abort flag
  off += (M == Mode::Down) ? combine_smem_bytes(nb, k) : 0;   // combine lists
  l.total = off;
  return l;
}

struct Unit {
  int e, r0, n, mt;   // expert, first permuted row of the chunk, tokens in it, weight tile
};

__device__ __forceinline__ int expert_of_chunk(const int32_t* mtile_off, int E, int g) {
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(mtile_off + mid) <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ Unit unit_of(const GemmArgs& a, int n_mt, int u) {
  const int g = u / n_mt;
  Unit w;
  w.mt = u - g * n_mt;
  w.e = expert_of_chunk(a.mtile_off, a.E, g);
  w.r0 = __ldg(a.offsets + w.e) + (g - __ldg(a.mtile_off + w.e)) * a.nb;
  w.n = min(a.nb, __ldg(a.offsets + w.e + 1) - w.r0);
  return w;
}

// Bounded wait: true when the phase completed; false after limit_ns
// nanoseconds (recorded in the status word) or when another thread of the CTA
// gave up.
// The thread sleeps inside the wait instruction (woken when the phase
// completes) and wakes at least every 20 us to check the abort flag and the
// time limit.  `backoff_ns` > 0 also sleeps that long between polls: for
// waits that usually last a whole work unit (the epilogue) or that run far
// ahead (the producers), so polling does not take issue slots from the
// dequantisers that share the SM partition.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           int32_t* status, long long limit_ns,
                                           uint32_t backoff_ns = 0) {
  if (ptx::mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t n = 1;; ++n) {
    if (backoff_ns) __nanosleep(backoff_ns);
    if (ptx::mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if ((n & 31) == 0) {                        // the abort flag and the clock, now and then
      if (*abort_flag) return false;
      if ((long long)(global_ns() - t0) > limit_ns) {
        *abort_flag = 1;
        atomicMax(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Ring position: slot and phase parity, advanced in step by every role.
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) { slot = 0; phase ^= 1; }
  }
};

// Record of the loads a producer ring has in flight, so an aborting producer
// can wait for them to land before the CTA exits.
struct Inflight {
  uint32_t issued = 0, parity = 0;
  __device__ __forceinline__ void mark(int slot, uint32_t phase) {
    issued |= 1u << slot;
    parity = (parity & ~(1u << slot)) | (phase << slot);
  }
  __device__ __forceinline__ void drain(uint64_t* bars, int n) const {
    const long long t0 = clock64();
    for (int s = 0; s < n; ++s) {
      if (!(issued >> s & 1u)) continue;
      while (!ptx::mbar_try_wait(&bars[s], (parity >> s) & 1u) && clock64() - t0 < kSpinLimit) {
      }
    }
  }
};

// ------------------------------------------------------------- dequant --

// 2^delta as an f16x2 pair (delta <= 0); 0 below the f16 subnormal range.
// Branch-free: lanes of a warp hold different rows' scales.
__device__ __forceinline__ uint32_t f16x2_pow2(int delta) {
  const int e = delta + 15;                                   // biased exponent
  const uint32_t normal = uint32_t(max(e, 0)) << 10;
  const uint32_t sub = (e <= 0 && e > -10) ? (1u << (e + 9)) : 0u;   // 2^(delta+24) ulps
  const uint32_t b = e > 0 ? normal : sub;
  return b | (b << 16);
}

// 2^p as a bf16x2 pair for p <= 127; 0 below the bf16 normal range.
__device__ __forceinline__ uint32_t bf16x2_pow2(int p) {
  const uint32_t b = uint32_t(max(p + 127, 0)) << 7;
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

// 8 E2M1 codes (one 32-bit word, the even K index in the low nibble of each
// byte) -> 4 f16x2 words holding K pairs (0,1), (2,3), (4,5), (6,7).
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
// 2^-112 (the exponent/mantissa field moves right by 3; the sign stays).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_scaled(uint32_t t) {
  return ((t >> 3) & 0x0FFF0FFFu) ^ (t & 0x80008000u);
}

template <Mode M>
struct Dequant;

template <>
struct Dequant<Mode::GateUp> {
  // 2^(s - r_n) in f16
  __device__ __forceinline__ static uint32_t factor(int s, int rn) { return f16x2_pow2(s - rn); }
  __device__ __forceinline__ static void convert(uint32_t w, uint32_t f, uint32_t* out) {
    const uint4 v = e2m1x8_to_f16(w);
    out[0] = hmul2_f16(v.x, f);
    out[1] = hmul2_f16(v.y, f);
    out[2] = hmul2_f16(v.z, f);
    out[3] = hmul2_f16(v.w, f);
  }
};

// The bf16 form's row offset c_n = max(15, r_n - 127): weights scale by
// 2^(s - c_n) in bf16 (the bit move left a factor 2^-112, so the product is
// the weight times 2^(15 - c_n)), at most 2^127 for every scale byte, and the
// epilogue multiplies by 2^(c_n - 15) (1 unless r_n > 142).
__device__ __forceinline__ int bf16_row_offset(int rn) { return max(15, rn - 127); }

template <>
struct Dequant<Mode::Down> {
  __device__ __forceinline__ static uint32_t factor(int s, int rn) {
    return bf16x2_pow2(s - bf16_row_offset(rn));
  }
  __device__ __forceinline__ static void convert(uint32_t w, uint32_t f, uint32_t* out) {
    const uint4 v = e2m1x8_to_f16(w);
    out[0] = hmul2_bf16(f16x2_to_bf16x2_scaled(v.x), f);
    out[1] = hmul2_bf16(f16x2_to_bf16x2_scaled(v.y), f);
    out[2] = hmul2_bf16(f16x2_to_bf16x2_scaled(v.z), f);
    out[3] = hmul2_bf16(f16x2_to_bf16x2_scaled(v.w), f);
  }
};

// Largest byte of the `nsb` bytes at smem byte offset `base` (4-aligned buffer).
__device__ __forceinline__ int row_max_byte(const uint32_t* buf, uint32_t base, int nsb) {
  const uint32_t end = base + uint32_t(nsb);
  const uint32_t w0 = base >> 2, w1 = (end + 3) >> 2;
  const uint32_t mlo = 0xFFFFFFFFu << (8 * (base & 3));
  const uint32_t mhi = (end & 3) ? (0xFFFFFFFFu >> (8 * (4 - (end & 3)))) : 0xFFFFFFFFu;
  uint32_t m;
  if (w1 - w0 == 1) {
    m = buf[w0] & mlo & mhi;
  } else {
    m = __vmaxu4(buf[w0] & mlo, buf[w1 - 1] & mhi);
    for (uint32_t i = w0 + 1; i + 1 < w1; ++i) m = __vmaxu4(m, buf[i]);
  }
  m = __vmaxu4(m, m >> 16);
  m = __vmaxu4(m, m >> 8);
  return int(m & 0xFF);
}

// ------------------------------------------------------------- kernel --

// F16: the operands are f16 (weights scaled per row by 2^(s - r_n), gate_up's
// activations x·2^e_t, down's h as an f16 pair); otherwise bf16 (weights at
// full scale, h as a bf16 pair), which down uses when h is not bounded.
template <Mode M, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
moe_expert_gemm_tmem(const __grid_constant__ CUtensorMap map_w,
                     const __grid_constant__ CUtensorMap map_b0,
                     const __grid_constant__ CUtensorMap map_b1, const GemmArgs a) {
  constexpr int NOPS = Cfg<M>::NOPS;
  constexpr bool kGateUp = (M == Mode::GateUp);
  constexpr Mode DQ = F16 ? Mode::GateUp : Mode::Down;   // dequantiser format

  const int K = kGateUp ? a.d : a.W;                 // reduction length
  const int nsb = K / 32;                            // scale bytes per weight row
  const int nS = (K + kSK - 1) / kSK;                // code stages per unit
  const int nA = (K + kAK - 1) / kAK;                // A stages per unit
  const int bk = act_stage_k(a.nb, NOPS);            // K per activation stage
  const int nKB = (K + bk - 1) / bk;                 // activation stages per unit
  const int rpe = kGateUp ? 2 * a.W : a.d;           // weight rows per expert
  const int n_out = kGateUp ? a.W : a.d;
  const int rows_per_tile = kGateUp ? kMW / 2 : kMW; // output features per unit
  const int n_mt = (n_out + rows_per_tile - 1) / rows_per_tile;
  const int NC = a.stages_c, NBS = a.stages_b;
  const int NAS = a_stages(a.nb);
  const int a_col0 = 2 * a.nb;                       // TMEM: accumulators first, then A
  const Lay L = layout<M>(nsb, a.nb, a.k, NC, NBS);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* codes = smem + L.codes;
  uint8_t* bt = smem + L.bt;
  uint8_t* scb = smem + L.sc;
  float* rf = reinterpret_cast<float*>(smem + L.rf);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* code_full = bars;
  uint64_t* code_empty = code_full + kMaxC;
  uint64_t* a_full = code_empty + kMaxC;
  uint64_t* a_empty = a_full + kMaxA;
  uint64_t* b_full = a_empty + kMaxA;
  uint64_t* b_empty = b_full + kMaxB;
  uint64_t* sc_full = b_empty + kMaxB;
  uint64_t* sc_empty = sc_full + 2;
  uint64_t* acc_full = sc_empty + 2;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* rf_full = acc_empty + 2;
  uint64_t* rf_empty = rf_full + kRing;
  uint64_t* mma_done = rf_empty + kRing;
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  uint8_t* comb = smem + L.misc + 16;                // combine lists (down)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxC; ++s) {
      ptx::mbar_init(&code_full[s], 1);
      ptx::mbar_init(&code_empty[s], kDqWarps);
    }
    for (int s = 0; s < kMaxA; ++s) {
      ptx::mbar_init(&a_full[s], kDqWarps);
      ptx::mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < kMaxB; ++s) {
      ptx::mbar_init(&b_full[s], 1);
      ptx::mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sc_full[s], 1);
      ptx::mbar_init(&sc_empty[s], kDqWarps);
      ptx::mbar_init(&acc_full[s], 1);
      ptx::mbar_init(&acc_empty[s], 4);
    }
    for (int s = 0; s < kRing; ++s) {
      ptx::mbar_init(&rf_full[s], 4);
      ptx::mbar_init(&rf_empty[s], 4);
    }
    ptx::mbar_init(mma_done, 1);
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
  // Everything above overlapped the previous kernel; from here on global
  // memory written by earlier kernels is read.  gate_up lets the down kernel
  // start its own prologue now (its CTAs take an SM as this kernel's leave).
  pdl_wait();
  if (kGateUp) pdl_trigger();
  const int units = __ldg(a.mtile_off + a.E) * n_mt;   // token chunks x weight tiles

  if (warp == kWarpProd) {
    // ------------------------------------------- producer: scales and codes --
    if (ptx::elect_one() && !(kGateUp && a.inject == 1)) {
      ptx::tma_prefetch_desc(&map_w);
      Ring cr;
      Inflight c_in, s_in;
      bool ok = true;
      int q = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++q) {
        const Unit w = unit_of(a, n_mt, u);
        // the unit's scale rows (1-D bulk copies of contiguous rows)
        const int sb = q & 1;
        if (!wait_phase(&sc_empty[sb], ((q >> 1) & 1) ^ 1, abort_flag, a.status, a.wait_ns, 64)) { ok = false; break; }
        const uint8_t* wscale = kGateUp ? a.w_gu_scale : a.w_dn_scale;
        int row_a, row_b;
        if constexpr (kGateUp) {
          const int n0 = w.mt * (kMW / 2);
          const int nrows = min(kMW / 2, a.W - n0);
          row_a = w.e * rpe + n0;
          row_b = w.e * rpe + a.W + n0;
          const uint32_t bytes = uint32_t(nrows * nsb);
          ptx::mbar_arrive_expect_tx(&sc_full[sb], 2 * bytes);
          uint8_t* dst = scb + sb * L.scbuf;
          ptx::bulk_load(dst, wscale + size_t(row_a) * nsb, bytes, &sc_full[sb]);
          ptx::bulk_load(dst + (kMW / 2) * nsb, wscale + size_t(row_b) * nsb, bytes, &sc_full[sb]);
        } else {
          const int m0 = w.mt * kMW;
          const int nrows = min(kMW, a.d - m0);
          row_a = w.e * rpe + m0;
          row_b = row_a + kCodeBoxRows;
          const uint32_t bytes = uint32_t(nrows * nsb);
          ptx::mbar_arrive_expect_tx(&sc_full[sb], bytes);
          ptx::bulk_load(scb + sb * L.scbuf, wscale + size_t(row_a) * nsb, bytes, &sc_full[sb]);
        }
        s_in.mark(sb, (q >> 1) & 1);
        for (int cs = 0; cs < nS; ++cs) {
          if (!wait_phase(&code_empty[cr.slot], cr.phase ^ 1, abort_flag, a.status, a.wait_ns, 64)) { ok = false; break; }
          uint8_t* cdst = codes + cr.slot * kCodeStageBytes;
          ptx::mbar_arrive_expect_tx(&code_full[cr.slot], kCodeStageBytes);
          ptx::tma_load_2d(cdst, &map_w, &code_full[cr.slot], cs * (kSK / 2), row_a);
          ptx::tma_load_2d(cdst + kCodeStageBytes / 2, &map_w, &code_full[cr.slot], cs * (kSK / 2), row_b);
          c_in.mark(cr.slot, cr.phase);
          cr.next(NC);
        }
      }
      if (!ok) {
        c_in.drain(code_full, NC);
        s_in.drain(sc_full, 2);
      }
    }
    __syncwarp();                 // the warp reaches the final barrier converged
  } else if (warp == kWarpProdB) {
    // --------------------------------------------- producer: activations --
    if (ptx::elect_one()) {
      ptx::tma_prefetch_desc(&map_b0);
      if (NOPS > 1) ptx::tma_prefetch_desc(&map_b1);
      Ring br;
      Inflight b_in;
      bool ok = true;
      const int subs_per_stage = bk / 64;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_of(a, n_mt, u);
        for (int jb = 0; jb < nKB; ++jb) {
          if (!wait_phase(&b_empty[br.slot], br.phase ^ 1, abort_flag, a.status, a.wait_ns, 64)) { ok = false; break; }
          // one box of nb rows x 64 K per sub-tile and operand (rows past the
          // chunk are other experts' tokens or zero fill, and only feed
          // accumulator columns the epilogue ignores); sub-tiles past K are
          // not loaded and not read
          const int k0 = jb * bk;
          const int subs = min(subs_per_stage, (K - k0 + 63) / 64);
          ptx::mbar_arrive_expect_tx(&b_full[br.slot], uint32_t(NOPS * subs * a.nb * 128));
          uint8_t* bdst = bt + br.slot * L.bstage;
          for (int sb2 = 0; sb2 < subs; ++sb2) {
            ptx::tma_load_2d(bdst + (sb2 * NOPS) * a.nb * 128, &map_b0, &b_full[br.slot], k0 + 64 * sb2, w.r0);
            if (NOPS > 1)
              ptx::tma_load_2d(bdst + (sb2 * NOPS + 1) * a.nb * 128, &map_b1, &b_full[br.slot],
                               k0 + 64 * sb2, w.r0);
          }
          b_in.mark(br.slot, br.phase);
          br.next(NBS);
        }
      }
      if (!ok) b_in.drain(b_full, NBS);
    }
    __syncwarp();
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------------ MMA issuer --
    // One thread's instruction stream sets the pace for short MMAs, so the
    // loop keeps per-MMA work to a few adds: descriptors are built once per
    // activation stage and the K16 loop is unrolled.
    if (ptx::elect_one()) {
      Ring ar, br;
      bool ok = true;
      int q = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++q) {
        const Unit w = unit_of(a, n_mt, u);
        const int N = (w.n + 15) & ~15;
        const uint32_t idesc = ptx::idesc_f16(kMW, N, !F16);
        const int buf = q & 1;
        if (!wait_phase(&acc_empty[buf], ((q >> 1) & 1) ^ 1, abort_flag, a.status, a.wait_ns)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * a.nb;
        uint32_t accumulate = 0;
        int jb = 0;                                  // activation stage of the unit
        for (int ja = 0; ja < nA && ok; ++ja) {
          if (!wait_phase(&a_full[ar.slot], ar.phase, abort_flag, a.status, a.wait_ns)) { ok = false; break; }
          const uint32_t a_stage = tmem_base + a_col0 + ar.slot * kACols;
          // the activation stages inside this A stage
          for (int kb = ja * kAK; kb < min(K, (ja + 1) * kAK); kb += bk, ++jb) {
            if (!wait_phase(&b_full[br.slot], br.phase, abort_flag, a.status, a.wait_ns)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t bsm = ptx::smem_u32(bt + br.slot * L.bstage);
            const int nk = min(bk, K - kb) / 16;         // K16 steps in this stage
            const uint32_t a_cols = a_stage + (kb - ja * kAK) / 2;
            for (int kk0 = 0; kk0 < nk; kk0 += 4) {      // one 64-K sub-tile at a time
              const uint32_t sub = bsm + uint32_t((kk0 / 4) * NOPS * a.nb * 128);
              const uint64_t bdesc0 = ptx::desc_kmajor_sw128(sub);
              const uint64_t bdesc1 = ptx::desc_kmajor_sw128(sub + uint32_t(a.nb * 128));
              // a full 64-K sub-tile (4 K16 steps) or a 32-K tail (K % 32 == 0),
              // each a straight run of MMAs: a branch between the MMAs of a
              // run slows their issue far below the tensor pipe's rate
              if (nk - kk0 >= 4) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  ptx::mma_f16_tmem_a(d_tmem, a_cols + (kk0 + kk) * 8, bdesc0 + 2 * kk, idesc, accumulate);
                  if (NOPS > 1) ptx::mma_f16_tmem_a(d_tmem, a_cols + (kk0 + kk) * 8, bdesc1 + 2 * kk, idesc, 1u);
                  accumulate = 1u;
                }
              } else {
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                  ptx::mma_f16_tmem_a(d_tmem, a_cols + (kk0 + kk) * 8, bdesc0 + 2 * kk, idesc, accumulate);
                  if (NOPS > 1) ptx::mma_f16_tmem_a(d_tmem, a_cols + (kk0 + kk) * 8, bdesc1 + 2 * kk, idesc, 1u);
                  accumulate = 1u;
                }
              }
            }
            ptx::mma_commit(&b_empty[br.slot]);
            br.next(NBS);
          }
          if (!ok) break;
          ptx::mma_commit(&a_empty[ar.slot]);
          ar.next(NAS);
        }
        if (!ok) break;
        ptx::mma_commit(&acc_full[buf]);
      }
      // every issued MMA completes before TMEM is released
      ptx::mma_commit(mma_done);
      const long long t0 = clock64();
      while (!ptx::mbar_try_wait(mma_done, 0) && clock64() - t0 < kSpinLimit) {
      }
    }
    __syncwarp();
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
    // ------------------------------------------------------------- epilogue --
    const int quarter = warp & 3;
    const int Ln = quarter * 32 + lane;          // TMEM lane = weight row of the tile
    int q = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++q) {
      const Unit w = unit_of(a, n_mt, u);
      const int buf = q & 1, ring = q % kRing;
      const bool ok = wait_phase(&acc_full[buf], (q >> 1) & 1, abort_flag, a.status, a.wait_ns, 256) &&
                      wait_phase(&rf_full[ring], (q / kRing) & 1, abort_flag, a.status, a.wait_ns);
      // the four warps leave together (tcgen05.ld is .sync.aligned, and down's
      // combine synchronises all 128 threads)
      if (!ptx::group_all(1, 128, ok)) break;
      ptx::tc_fence_after();
      const float rowf = rf[ring * kMW + Ln];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&rf_empty[ring]);
      const uint32_t taddr = tmem_base + (uint32_t(quarter * 32) << 16) + buf * a.nb;
      if constexpr (kGateUp) {
        const bool is_up = Ln & 1;
        const int n = w.mt * (kMW / 2) + (Ln >> 1);
        const bool nvalid = n < a.W;
        const float bias =
            nvalid ? __bfloat162float(a.b_gu[size_t(w.e) * 2 * a.W + (is_up ? a.W : 0) + n]) : 0.f;
        for (int c = 0; c < w.n; c += 16) {
          uint32_t v[16];
          ptx::tmem_ld_32x32b_x16(taddr + c, v);
          // the token factors 2^-e_t of these 16 columns: lane j loads column
          // c + j % 16 (during the TMEM load) and the others take it by shuffle
          const int cl = c + (lane & 15);
          const float colf_l = cl < w.n ? __int_as_float((127 - __ldg(a.rowexp + w.r0 + cl)) << 23) : 0.f;
          ptx::tmem_ld_wait();
          float z[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float colf = __shfl_sync(0xffffffffu, colf_l, j);
            // the token's factor first: (acc 2^-e_t) is the dot product with
            // the row's weights scaled to its largest block, whose scale
            // 2^(r_n - 127) then overflows only if the true value does
            z[j] = (__uint_as_float(v[j]) * colf) * rowf + bias;
          }
          // gate lanes are even, up lanes odd: the even lane finishes tokens
          // c..c+7, the odd lane tokens c+8..c+15
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float send = is_up ? z[jj] : z[8 + jj];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const float zg = is_up ? recv : z[jj];
            const float zu = is_up ? z[8 + jj] : recv;
            const int col = c + (is_up ? 8 + jj : jj);
            const float gg = fminf(zg, a.limit);
            const float uu = fminf(fmaxf(zu, -a.limit), a.limit);
            // the sigmoid from the fast exponential and reciprocal (about 15
            // ulps at most while it is not negligible, alpha * g <= 12 for a
            // gate clamped at 7; far inside the layer's tolerance): with the
            // full-precision forms this epilogue set the kernel's pace
            const float sg = __fdividef(1.0f, 1.0f + __expf(-a.alpha * gg));
            const float hv = gg * sg * (uu + 1.0f);
            if (nvalid && col < w.n) {
              const size_t o = size_t(w.r0 + col) * a.W + n;
              if (a.h_f16) {                       // h = hi + lo, two f16 terms
                const __half hh = __float2half_rn(hv);
                const __half hl = __float2half_rn(hv - __half2float(hh));
                reinterpret_cast<__half*>(a.h_hi)[o] = hh;
                reinterpret_cast<__half*>(a.h_lo)[o] = hl;
              } else {                             // h = hi + lo, two bf16 terms
                const __nv_bfloat16 hh = __float2bfloat16_rn(hv);
                a.h_hi[o] = hh;
                a.h_lo[o] = __float2bfloat16_rn(hv - __bfloat162float(hh));
              }
            }
          }
        }
      } else {
        const int n = w.mt * kMW + Ln;
        const bool nvalid = n < a.d;
        const float bias = nvalid ? __bfloat162float(a.b_dn[size_t(w.e) * a.d + n]) : 0.f;
        for (int c = 0; c < w.n; c += 16) {
          uint32_t v[16];
          ptx::tmem_ld_32x32b_x16(taddr + c, v);
          ptx::tmem_ld_wait();
          if (nvalid) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c + j < w.n) a.y[size_t(w.r0 + c + j) * a.d + n] = __uint_as_float(v[j]) * rowf + bias;
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_empty[buf]);
      // K5: the weighted sum of each token whose k rows are now all stored
      // (after the accumulator is released, so the next unit's MMAs run meanwhile)
      if constexpr (!kGateUp)
        combine_tile<2>(a, w.r0, w.n, w.mt, Ln, comb, a.nb, 2);
    }
  } else if (warp >= kWarpDq0) {
    // --------------------------------------------------------- dequantisers --
    // Warp (quarter, part) converts K range [part*32, part*32+32) of each
    // 128-K half of every 256-K code stage for its 32 weight rows: 32 codes
    // -> 16 TMEM columns of one A stage, one tcgen05.st per half.
    const int quarter = warp & 3;
    const int part = (warp - kWarpDq0) >> 2;
    const int Ln = quarter * 32 + lane;          // TMEM lane = weight row of the tile
    const int sr = kGateUp ? ((Ln & 1) ? kMW / 2 + (Ln >> 1) : (Ln >> 1)) : Ln;   // smem row
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    const uint32_t choff0 = ptx::sw128_offset(sr, part);          // K half 0: chunk part
    const uint32_t choff1 = ptx::sw128_offset(sr, 4 + part);      // K half 1: chunk 4 + part
    Ring cr, ar;
    bool ok = true;
    int q = 0;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++q) {
      const Unit w = unit_of(a, n_mt, u);
      const bool valid = kGateUp ? (w.mt * (kMW / 2) + (Ln >> 1) < a.W) : (w.mt * kMW + Ln < a.d);
      const int sb = q & 1, ring = q % kRing;
      ok = __all_sync(0xffffffffu, wait_phase(&sc_full[sb], (q >> 1) & 1, abort_flag, a.status, a.wait_ns));
      if (!ok) break;
      const uint8_t* srow = scb + sb * L.scbuf + sr * nsb;
      int rn = 0;                                  // the row's largest scale byte
      if (valid)
        rn = row_max_byte(reinterpret_cast<const uint32_t*>(scb + sb * L.scbuf), uint32_t(sr * nsb), nsb);
      const uint32_t rnb = uint32_t(rn) * 0x0101u;   // r_n in the two low bytes
      if (part == 0) {
        ok = __all_sync(0xffffffffu, wait_phase(&rf_empty[ring], ((q / kRing) & 1) ^ 1, abort_flag, a.status, a.wait_ns));
        if (!ok) break;
        rf[ring * kMW + Ln] =
            valid ? (F16 ? ldexpf(1.0f, rn - 127) : ldexpf(1.0f, bf16_row_offset(rn) - 15)) : 0.f;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&rf_full[ring]);
      }
      for (int cs = 0; cs < nS; ++cs) {
        ok = __all_sync(0xffffffffu, wait_phase(&code_full[cr.slot], cr.phase, abort_flag, a.status, a.wait_ns, 32));
        if (!ok) break;
        const uint8_t* cst = codes + cr.slot * kCodeStageBytes;
        // this thread's scale blocks: one per K half
        const int b0 = cs * (kSK / 32) + part, b1 = b0 + 4;
        const bool v0 = valid && b0 < nsb, v1 = valid && b1 < nsb;
        const uint32_t s01 = (v0 ? uint32_t(srow[b0]) : 0u) | (v1 ? uint32_t(srow[b1]) << 8 : 0u);
        uint32_t f0, f1;
        if (F16) {
          // 2^(s - r_n) as f16x2 for both blocks at once: byte-wise
          // 15 - (r_n - s) (s <= r_n, so neither subtraction wraps for any
          // scale byte; clamped at 0 below the f16 normal range, where the
          // factor becomes 0), moved into both halves' exponent fields
          const uint32_t e2 = __vsubus4(0x0F0Fu, __vsubus4(rnb, s01)) & 0x1F1Fu;
          f0 = v0 ? (__byte_perm(e2, 0, 0x4040) << 10) : 0u;
          f1 = v1 ? (__byte_perm(e2, 0, 0x4141) << 10) : 0u;
        } else {
          f0 = v0 ? Dequant<DQ>::factor(int(s01 & 0xFF), rn) : 0u;
          f1 = v1 ? Dequant<DQ>::factor(int(s01 >> 8), rn) : 0u;
        }
        // 2 x 32 codes: one 16-byte chunk of the 128-byte swizzled row per half
        const uint4 x0 = *reinterpret_cast<const uint4*>(cst + choff0);
        const uint4 x1 = *reinterpret_cast<const uint4*>(cst + choff1);
        // the code stage has been read
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&code_empty[cr.slot]);
        cr.next(NC);
        uint32_t r[32];
        Dequant<DQ>::convert(x0.x, f0, &r[0]);
        Dequant<DQ>::convert(x0.y, f0, &r[4]);
        Dequant<DQ>::convert(x0.z, f0, &r[8]);
        Dequant<DQ>::convert(x0.w, f0, &r[12]);
        Dequant<DQ>::convert(x1.x, f1, &r[16]);
        Dequant<DQ>::convert(x1.y, f1, &r[20]);
        Dequant<DQ>::convert(x1.z, f1, &r[24]);
        Dequant<DQ>::convert(x1.w, f1, &r[28]);
        // the code stage's two A stages (the second only while it holds K)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (2 * cs + h >= nA) break;
          ok = __all_sync(0xffffffffu, wait_phase(&a_empty[ar.slot], ar.phase ^ 1, abort_flag, a.status, a.wait_ns, 32));
          if (!ok) break;
          ptx::tmem_st_32x32b_x16(tmem_base + lane_addr + a_col0 + ar.slot * kACols + part * 16, &r[16 * h]);
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&a_full[ar.slot]);
          ar.next(NAS);
        }
        if (!ok) break;
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sc_empty[sb]);
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

// Row-major [rows, cols] matrix of `esize`-byte elements, box {box_cols, box_rows},
// 128-byte swizzle.
cudaError_t make_map(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base,
                     long long rows, long long cols, int box_cols, int box_rows) {
  auto enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(cols) * esize};
  const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Ring depths for one launch.  Small chunks (decode-sized loads): a modest
// activation ring, then every remaining byte of shared memory holds code
// stages in flight (the weights stream from HBM, whose latency under load is
// several microseconds): about 10 x 16 KB.  Large chunks: as many activation
// stages as fit beside 3 code stages (gate_up) or 2 (down, whose stages carry
// h hi and lo: 4 stages of 64 K at 160 tokens with 2 code stages measured 5-9%
// faster than 3 with 4), then the rest as code stages.
template <Mode M>
void plan(GemmArgs& a) {
  const int K = (M == Mode::GateUp) ? a.d : a.W;
  const int per_b = layout<M>(K / 32, a.nb, a.k, 0, 1).bstage;
  int nbs;
  if (a.nb <= 32) {
    nbs = (48 * 1024) / per_b;                              // ~48 KB of activations
  } else {
    const Lay base = layout<M>(K / 32, a.nb, a.k, M == Mode::Down ? 2 : 3, 0);
    nbs = (kMaxSmem - 1024 - base.total) / per_b;
  }
  nbs = nbs < 2 ? 2 : nbs;
  nbs = nbs < kMaxB ? nbs : kMaxB;
  const Lay base1 = layout<M>(K / 32, a.nb, a.k, 0, nbs);
  int nc = (kMaxSmem - 1024 - base1.total) / kCodeStageBytes;
  nc = nc < kMaxC ? nc : kMaxC;
  a.stages_b = nbs;
  a.stages_c = nc;
}

template <Mode M>
size_t smem_bytes(const GemmArgs& a) {
  const int K = (M == Mode::GateUp) ? a.d : a.W;
  return size_t(layout<M>(K / 32, a.nb, a.k, a.stages_c, a.stages_b).total) + 1024;
}

template <Mode M, bool F16>
cudaError_t launch(const GemmArgs& args, cudaStream_t s) {
  GemmArgs a = args;
  plan<M>(a);
  const size_t smem = smem_bytes<M>(a);
  if (a.stages_b < 2 || a.stages_c < 2 || smem > size_t(kMaxSmem) || a.nb < 16 || a.nb > kNBMax ||
      a.nb % 16 || a_stages(a.nb) < 2)
    return cudaErrorInvalidConfiguration;
  {
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(moe_expert_gemm_tmem<M, F16>), kMaxSmem);
    if (e != cudaSuccess) return e;
  }
  // the three maps, from the cache when this layer's buffers were seen before
  struct Key {
    const void* p[4];
    int R, d, W, E, nb;
  } key;
  memset(&key, 0, sizeof(key));
  key.p[0] = (M == Mode::GateUp) ? a.w_gu : a.w_dn;
  key.p[1] = a.x_perm;
  key.p[2] = a.h_hi;
  key.p[3] = a.h_lo;
  key.R = a.R;
  key.d = a.d;
  key.W = a.W;
  key.E = a.E;
  key.nb = a.nb;
  static MapCache<Key, 3> cache;
  CUtensorMap maps[3];
  cudaError_t e = cudaSuccess;
  if (!cache.find(key, maps)) {
    CUtensorMap mw, m0, m1;
    if (M == Mode::GateUp) {
      e = make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.w_gu, (long long)a.E * 2 * a.W, a.d / 2,
                   kSK / 2, kCodeBoxRows);
      if (e == cudaSuccess)
        e = make_map(&m0, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.x_perm, a.R, a.d, 64, a.nb);
      m1 = m0;
    } else {
      e = make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.w_dn, (long long)a.E * a.d, a.W / 2,
                   kSK / 2, kCodeBoxRows);
      if (e == cudaSuccess)
        e = make_map(&m0, F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     a.h_hi, a.R, a.W, 64, a.nb);
      if (e == cudaSuccess)
        e = make_map(&m1, F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     a.h_lo, a.R, a.W, 64, a.nb);
    }
    if (e != cudaSuccess) return e;
    maps[0] = mw;
    maps[1] = m0;
    maps[2] = m1;
    cache.put(key, maps);
  }
  const CUtensorMap &mw = maps[0], &m0 = maps[1], &m1 = maps[2];
  const int n_out = (M == Mode::GateUp) ? a.W : a.d;
  const int rows_per_tile = (M == Mode::GateUp) ? kMW / 2 : kMW;
  const long long n_mt = (n_out + rows_per_tile - 1) / rows_per_tile;
  const long long units_bound = (long long)(a.R / a.nb + a.E) * n_mt;
  const int grid = int(units_bound < device_sm_count() ? units_bound : device_sm_count());
  return launch_pdl(moe_expert_gemm_tmem<M, F16>, dim3(grid), dim3(kThreads), smem, s, mw, m0, m1, a);
}

}  // namespace

// Down takes smaller large chunks than gate_up: its activation stages carry
// two operands (h hi and lo), and at 192 tokens only two of them fit in
// shared memory beside the code ring (measured: 160 best for down, 192 for
// gate_up).
int expert_gemm_tmem_chunk(int64_t R, int E, bool gate_up) {
  const int64_t avg = R / (E > 0 ? E : 1);
  return avg <= 8 ? 16 : avg <= 16 ? 32 : avg <= 32 ? 64 : (gate_up ? 192 : 160);
}

bool expert_gemm_tmem_fits(const GemmArgs& args) {
  GemmArgs g = args, d = args;
  g.nb = expert_gemm_tmem_chunk(args.R, args.E, true);
  d.nb = expert_gemm_tmem_chunk(args.R, args.E, false);
  plan<Mode::GateUp>(g);
  plan<Mode::Down>(d);
  return g.stages_b >= 2 && d.stages_b >= 2 && g.stages_c >= 2 && d.stages_c >= 2 &&
         smem_bytes<Mode::GateUp>(g) <= size_t(kMaxSmem) &&
         smem_bytes<Mode::Down>(d) <= size_t(kMaxSmem);
}
cudaError_t launch_gateup_tmem(const GemmArgs& a, cudaStream_t s) { return launch<Mode::GateUp, true>(a, s); }
cudaError_t launch_down_tmem(const GemmArgs& a, cudaStream_t s) {
  return a.h_f16 ? launch<Mode::Down, true>(a, s) : launch<Mode::Down, false>(a, s);
}

bool hidden_fits_f16(float limit) {
  // |h| = |g·σ(αg)·(u+1)| <= limit·(limit+1) once g <= limit and |u| <= limit
  return std::isfinite(limit) && limit >= 0.f && limit * (limit + 1.f) < 16384.f;
}

}  // namespace moe
