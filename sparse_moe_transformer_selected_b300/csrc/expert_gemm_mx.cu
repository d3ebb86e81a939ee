// K3 / K4 — grouped expert GEMMs on the block-scaled tensor-core path.
//
// Each expert's segment of the permuted rows is multiplied by that expert's
// MXFP4 weights ("OpenAI 最新开源模型 gpt-oss 架构与训练解析", 模型架构: MoE
// weights in MXFP4, 32 E2M1 codes sharing one E8M0 scale; experts are
// gated-SwiGLU FFNs with clamping and the +1 term on the up branch;
// 更深对比更宽: d = W = 2880).
//
// The MXFP4 format is what tcgen05.mma kind::mxf8f6f4 consumes: A is E2M1
// codes, each 32-element K block with a UE8M0 scale held in tensor memory, so
// the weights go from HBM to the tensor core without being converted.  The
// activations are the B side as sums of E4M3 terms, each term with its own
// block scales, stacked along N, and the epilogue adds a token's term columns.
// A work unit is a chunk of up to 8 tokens of one expert.
//   gate_up: x = hi + lo / 16 (2 terms; exact for bf16 values within 2^-7
//            of their 32-block's largest)
//   down:    h = (t0 + t1 / 16 + t2 / 256 + t3 / 4096) 2^h_exp (4 terms,
//            about 16 significant bits)
// One MMA covers M = 128 weight rows, N = 32, K = 32.
//
//   D[weight row, j] = Σ_k A[row, k] 2^(sa - 127) · B[j, k] 2^(sb - 127)
//
// Operands in shared memory, 128-byte swizzle, K-major:
//   A  TMA with the 4-bit "16U4_ALIGN16B" type: every 16 packed codes (8 bytes)
//      land in 16 bytes (8 bytes of codes, 8 bytes of padding), the layout
//      the MMA reads E2M1 from.  A box is 128 codes x 128 rows: gate_up's is
//      3-D, 64 gate rows and the 64 up rows W below them; down's 2-D.  The
//      type wants the tensor's row length a multiple of 128, so the map covers
//      the first K - K % 128 codes of each row and a second map, whose base
//      is the row's last 128 codes, serves the tail.
//   B  gate_up: the chunk's token rows of the per-token E4M3 tables (the router
//      quantises each token once), gathered by TMA tile::gather4: four token
//      rows of 128 K land in the first four rows of a 1024-byte swizzle atom,
//      so term t holds tokens 0-3 in rows 16t .. 16t + 3 and tokens 4-7 in
//      rows 16t + 8 .. 16t + 11 (B row of token j: 16t + 8 (j / 4) + j % 4);
//      the other rows only feed accumulator columns the epilogue ignores.
//      down: TMA boxes of 128 K x 8 rows of the h term tables (permuted rows,
//      written by gate_up), term t in rows 8t .. 8t + 7.
// Scales in tensor memory, written once per unit by four warps with tcgen05.st
// (a row's 4 scale bytes of 4 consecutive K blocks share a 32-bit column; the
// MMA picks the byte with the descriptor's scale-factor ID).
//
// One persistent kernel runs both GEMMs, one CTA per SM, 12 warps:
//   warp 0      producer: per stage A and B (TMA); one ring of stages of 256 K
//   warp 1      MMA issuer (one elected thread)
//   warp 2      TMEM allocator: 512 columns (2 accumulators of 64, then two
//               sets of A and B scale columns)
//   warp 3      unit scheduler (one elected thread): decodes this CTA's next
//               unit (routing tables, the chunk's token indices; for a down
//               unit, the wait for its chunk's h), hands it to the producer
//               through a two-entry queue in shared memory, and copies its
//               weight scale rows; so the producer issues stages only, never
//               stalled on a global load
//   warps 4-7   epilogue, TMEM lane quarter = warp % 4
//   warps 8-11  scale writers, TMEM lane quarter = warp % 4 (gate_up's
//               activation scales read from L2, one token row per lane)
// Work units: first every gate_up unit, then every down unit, each list
// chunk-major (token chunk of one expert x weight tile); CTA c takes units
// c, c + grid, ...  A down unit needs the whole h of its chunk: the gate_up
// epilogue of each (chunk, tile) releases a per-chunk count once its h rows
// are stored, and the producer acquires the full count before it loads the
// chunk's h.  Every CTA finishes its gate_up units before it reaches a down
// unit, so the waits form no cycle; the launch is cooperative (all CTAs
// resident), and each wait is bounded.  CTAs that finish their gate_up share
// early start on the first chunks' down units while the others finish, so
// the two GEMMs share one ramp and one tail.
#include "combine.cuh"
#include "common.cuh"
#include "map_cache.cuh"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kMW = 128;                      // weight rows per unit (MMA M)
constexpr int kBoxK = 128;                    // K per box: one 128-byte swizzle row
constexpr int kBoxBytesA = kMW * kBoxK;       // 16 KB, one byte per code in shared memory
constexpr int kNB = 8;                        // token chunk
constexpr int kBRows = 32;                    // MMA N: B rows of a box
constexpr int kHTerms = 4;                    // E4M3 terms of h
constexpr int kXTerms = 2;                    // E4M3 terms of x
constexpr int kAccCols = 64;                  // TMEM columns per accumulator
constexpr int kMaxStages = 8;
constexpr int kMaxExperts = 256;
constexpr int kThreads = 384;
constexpr int kWarpProd = 0, kWarpMMA = 1, kWarpTmem = 2, kWarpSched = 3, kWarpEpi0 = 4, kWarpSf0 = 8;
constexpr int kTmemCols = 512;
constexpr int kMaxGroups = (kTmemCols - 2 * kAccCols) / 16;   // SF groups (4 K blocks each)
constexpr long long kSpinLimit = 4000000000ll;   // clock cycles: the final drains
constexpr int kMaxSmem = 232448;
// stage ring (full + empty), scales (2 + 2), scale columns (2 + 2),
// accumulators (2 + 2), final drain, unit queue (2 + 2)
constexpr int kNumBars = 2 * kMaxStages + 4 + 4 + 4 + 1 + 4;

// Bounded wait: true when the phase completed; false after limit_ns
// nanoseconds (code in status[0], the waiting role's tag in status[4]) or when
// another thread of the CTA gave up.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           int32_t* status, long long limit_ns,
                                           uint32_t backoff_ns = 0, int tag = 0) {
  if (ptx::mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t n = 1;; ++n) {
    if (backoff_ns) __nanosleep(backoff_ns);
    if (ptx::mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if ((n & 31) == 0) {
      if (*abort_flag) return false;
      if ((long long)(global_ns() - t0) > limit_ns) {
        *abort_flag = 1;
        atomicMax(status, kStatusTimeout);
        atomicExch(status + 4, tag);
        return false;
      }
    }
  }
}

struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) { slot = 0; phase ^= 1; }
  }
};

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

__device__ __forceinline__ uint32_t to_e4m3(float v) {
  return uint32_t(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float from_e4m3(uint32_t b) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(__nv_fp8_storage_t(b), __NV_E4M3)));
}

// Geometry of one GEMM (gate_up or down), the same on host and device.
struct ModeGeo {
  int K, nsb, groups;        // reduction length, scale bytes per weight row, SF groups
  int nbox_main, tail;       // 128-K boxes from the main map; K % 128 (0: no tail box)
  int nbox, nstage;          // boxes per unit (main + tail), stages of 2 boxes
  int NT, rpt;               // B terms, B rows per term (N = NT rpt = kBRows)
  int n_out, rows_per_tile;  // output columns; weight rows of one tile's output
  int n_mt;                  // weight tiles per chunk
  int rpe;                   // weight rows per expert
  int sc_a;                  // scale bytes of a unit's weight rows (16-byte multiple)
};

__host__ __device__ inline ModeGeo mode_geo(bool gate_up, int d, int W) {
  ModeGeo g{};
  g.K = gate_up ? d : W;
  g.nsb = g.K / 32;
  g.groups = (g.nsb + 3) / 4;
  g.nbox_main = g.K / kBoxK;
  g.tail = g.K % kBoxK;
  g.nbox = g.nbox_main + (g.tail ? 1 : 0);
  g.nstage = (g.nbox + 1) / 2;
  g.NT = gate_up ? kXTerms : kHTerms;
  g.rpt = kBRows / g.NT;                   // gate_up: two atoms of 4 tokens; down: 8 rows
  g.n_out = gate_up ? W : d;
  g.rows_per_tile = gate_up ? kMW / 2 : kMW;
  g.n_mt = (g.n_out + g.rows_per_tile - 1) / g.rows_per_tile;
  g.rpe = gate_up ? 2 * W : d;
  g.sc_a = (kMW * g.nsb + 15) / 16 * 16;
  return g;
}

// A unit as the scheduler warp hands it to the producer.
struct UnitInfo {
  int gu;                    // gate_up (else down)
  int row_a, row_b;          // first weight rows of the two A boxes (gate, up) or of the one
  int r0;                    // first permuted row of the chunk
  int tok[kNB];              // gate_up: the chunk's tokens (rows past it repeat its first)
};

// Shared-memory plan of the launch (both GEMMs share the ring).
struct Geo {
  int groups;                // SF groups of the larger K (TMEM scale columns)
  int a_stage, b_stage;      // bytes per stage
  int stages;                // ring depth
  int off_b, off_sc, off_xch, off_bars, off_comb, off_info, off_tab, total;
};

__host__ __device__ inline Geo geometry(int d, int W, int stages) {
  const ModeGeo gu = mode_geo(true, d, W), dn = mode_geo(false, d, W);
  Geo g{};
  g.groups = gu.groups > dn.groups ? gu.groups : dn.groups;
  g.a_stage = 2 * kBoxBytesA;
  g.b_stage = 2 * kBRows * kBoxK;
  g.stages = stages;
  int off = stages * g.a_stage;
  g.off_b = off;
  off += stages * g.b_stage;
  g.off_sc = off;
  off += gu.sc_a > dn.sc_a ? gu.sc_a : dn.sc_a;
  g.off_xch = off;
  off += (kMW / 2) * kNB * 4;
  off = (off + 7) & ~7;
  g.off_bars = off;
  off += kNumBars * 8 + 16;           // barriers, TMEM base, abort flag
  g.off_comb = off;
  off += combine_smem_bytes(kNB, 8);
  off = (off + 15) & ~15;
  g.off_info = off;
  off += 2 * int(sizeof(UnitInfo));
  off = (off + 15) & ~15;
  g.off_tab = off;
  off += 2 * (kMaxExperts + 1) * 4;   // expert offsets and chunk prefix
  g.total = off;
  return g;
}

struct Unit {
  int e, r0, n, mt;   // expert, first permuted row of the chunk, tokens in it, weight tile
  int g;              // chunk index (over all experts)
  bool gu;            // a gate_up unit (else down)
};

// The routing tables of the launch, copied into shared memory once.
struct Tables {
  const int32_t* off;   // [E + 1] first permuted row of each expert
  const int32_t* mto;   // [E + 1] first chunk of each expert
};

__device__ __forceinline__ int expert_of_chunk(const int32_t* mto, int E, int g) {
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mto[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Unit u of the launch: gate_up units [0, u_gu), then down units.
__device__ __forceinline__ Unit unit_of(const GemmArgs& a, const Tables& tb, const ModeGeo& MG,
                                        const ModeGeo& MD, int u_gu, int u) {
  Unit w;
  w.gu = u < u_gu;
  const int n_mt = w.gu ? MG.n_mt : MD.n_mt;
  const int ul = w.gu ? u : u - u_gu;
  w.g = ul / n_mt;
  w.mt = ul - w.g * n_mt;
  w.e = expert_of_chunk(tb.mto, a.E, w.g);
  w.r0 = tb.off[w.e] + (w.g - tb.mto[w.e]) * a.nb;
  w.n = min(a.nb, tb.off[w.e + 1] - w.r0);
  return w;
}

// Scale bytes 4g..4g+3 of a row (bytes at or past nsb read as 0).
__device__ __forceinline__ uint32_t scale_word(const uint8_t* row, int g, int nsb) {
  uint32_t w = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (4 * g + j < nsb) w |= uint32_t(row[4 * g + j]) << (8 * j);
  return w;
}

// Bounded wait until *count >= target (acquire): false after limit_ns
// (status word MOE_ERR_TIMEOUT, the waiting role's tag in status[4]) or when
// another thread of the CTA gave up.
__device__ __forceinline__ bool wait_count(const int32_t* count, int target, volatile int* abort_flag,
                                           int32_t* status, long long limit_ns, int tag) {
  if (ptx::ld_acquire_gpu(count) >= target) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t n = 1;; ++n) {
    __nanosleep(128);
    if (ptx::ld_acquire_gpu(count) >= target) return true;
    if ((n & 31) == 0) {
      if (*abort_flag) return false;
      if ((long long)(global_ns() - t0) > limit_ns) {
        *abort_flag = 1;
        atomicMax(status, kStatusTimeout);
        atomicExch(status + 4, tag);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------- kernel --

__global__ void __launch_bounds__(kThreads, 1)
moe_expert_mx(const __grid_constant__ CUtensorMap map_wg,     // gate_up codes, main and tail
              const __grid_constant__ CUtensorMap map_wgt,
              const __grid_constant__ CUtensorMap map_wd,     // down codes, main and tail
              const __grid_constant__ CUtensorMap map_wdt,
              const __grid_constant__ CUtensorMap map_x0,     // x term token tables
              const __grid_constant__ CUtensorMap map_x1,
              const __grid_constant__ CUtensorMap map_h0,     // h term tables
              const __grid_constant__ CUtensorMap map_h1,
              const __grid_constant__ CUtensorMap map_h2,
              const __grid_constant__ CUtensorMap map_h3,
              const GemmArgs a, const int stages) {
  const ModeGeo MG = mode_geo(true, a.d, a.W), MD = mode_geo(false, a.d, a.W);
  const Geo G = geometry(a.d, a.W, stages);
  const int S = G.stages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + G.off_b;
  uint8_t* scb = smem + G.off_sc;
  float* xch = reinterpret_cast<float*>(smem + G.off_xch);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G.off_bars);
  uint64_t* full = bars;
  uint64_t* empty = full + kMaxStages;
  uint64_t* sc_full = empty + kMaxStages;
  uint64_t* sc_empty = sc_full + 2;
  uint64_t* sf_full = sc_empty + 2;
  uint64_t* sf_empty = sf_full + 2;
  uint64_t* acc_full = sf_empty + 2;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint64_t* info_full = mma_done + 1;
  uint64_t* info_empty = info_full + 2;
  UnitInfo* info = reinterpret_cast<UnitInfo*>(smem + G.off_info);
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(smem + G.off_bars + kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G.off_bars + kNumBars * 8 + 4);
  uint8_t* comb = smem + G.off_comb;             // combine lists (down units)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sc_full[s], 1);
      ptx::mbar_init(&sc_empty[s], 4);
      ptx::mbar_init(&sf_full[s], 4);
      ptx::mbar_init(&sf_empty[s], 1);
      ptx::mbar_init(&acc_full[s], 1);
      ptx::mbar_init(&acc_empty[s], 4);
      ptx::mbar_init(&info_full[s], 1);
      ptx::mbar_init(&info_empty[s], 1);
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
  // TMEM columns: accumulators, then per SF set (2) the A and the B columns
  const uint32_t sfa_col0 = 2 * kAccCols;
  const uint32_t sfb_col0 = 2 * kAccCols + 2 * 4 * G.groups;
  pdl_wait();
  // the routing tables, once, for every role's unit lookups
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + G.off_tab);
  int32_t* s_mto = s_off + kMaxExperts + 1;
  for (int i = threadIdx.x; i <= a.E; i += kThreads) {
    s_off[i] = __ldg(a.offsets + i);
    s_mto[i] = __ldg(a.mtile_off + i);
  }
  __syncthreads();
  const Tables tabs{s_off, s_mto};
  const int chunks = s_mto[a.E];
  const int u_gu = chunks * MG.n_mt;
  const int units = u_gu + chunks * MD.n_mt;

  // weight rows of a unit: gate and up halves (gate_up) or one block (down)
  auto rows_of = [&](const Unit& w, int& ra, int& rb, int& nrows) {
    if (w.gu) {
      const int n0 = w.mt * (kMW / 2);
      nrows = min(kMW / 2, a.W - n0);
      ra = w.e * MG.rpe + n0;
      rb = w.e * MG.rpe + a.W + n0;
    } else {
      const int m0 = w.mt * kMW;
      nrows = min(kMW, a.d - m0);
      ra = w.e * MD.rpe + m0;
      rb = ra;
    }
  };

  if (warp == kWarpSched) {
    // ------------------------------------------------------- unit scheduler --
    if (ptx::elect_one() && a.inject != 1) {
      Inflight in_sc;
      bool ok = true;
      int q = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++q) {
        const Unit w = unit_of(a, tabs, MG, MD, u_gu, u);
        int ra, rb, nrows;
        rows_of(w, ra, rb, nrows);
        UnitInfo& inf = info[q & 1];
        if (!wait_phase(&info_empty[q & 1], ((q >> 1) & 1) ^ 1, abort_flag, a.status, a.wait_ns, 64, 10)) { ok = false; break; }
        inf.gu = w.gu;
        inf.row_a = ra;
        inf.row_b = rb;
        inf.r0 = w.r0;
        if (w.gu) {
#pragma unroll
          for (int j = 0; j < kNB; ++j) inf.tok[j] = __ldg(a.perm + w.r0 + (j < w.n ? j : 0)) / a.k;
        } else {
          // every gate_up tile of this chunk has stored its h rows
          if (!wait_count(a.ready + w.g, MG.n_mt, abort_flag, a.status, a.wait_ns, 9)) { ok = false; break; }
          ptx::fence_proxy_async_global();
        }
        ptx::mbar_arrive(&info_full[q & 1]);
        // the unit's weight scale rows, into the staging buffer once the
        // scale writers have copied the previous unit's into TMEM (the
        // activations' scales are read by the writers)
        if (!wait_phase(&sc_empty[0], (q & 1) ^ 1, abort_flag, a.status, a.wait_ns, 64, 5)) { ok = false; break; }
        const int nsb = w.gu ? MG.nsb : MD.nsb;
        const uint8_t* wscale = w.gu ? a.w_gu_scale : a.w_dn_scale;
        const uint32_t bytes = uint32_t(nrows * nsb);
        if (w.gu) {
          ptx::mbar_arrive_expect_tx(&sc_full[0], 2 * bytes);
          ptx::bulk_load(scb, wscale + size_t(ra) * nsb, bytes, &sc_full[0]);
          ptx::bulk_load(scb + (kMW / 2) * nsb, wscale + size_t(rb) * nsb, bytes, &sc_full[0]);
        } else {
          ptx::mbar_arrive_expect_tx(&sc_full[0], bytes);
          ptx::bulk_load(scb, wscale + size_t(ra) * nsb, bytes, &sc_full[0]);
        }
        in_sc.mark(0, q & 1);
      }
      if (!ok) in_sc.drain(sc_full, 1);
    }
    __syncwarp();                 // the warp reaches the final barrier converged
  } else if (warp == kWarpProd) {
    // ------------------------------------------------------------ producer --
    if (ptx::elect_one() && a.inject != 1) {
      ptx::tma_prefetch_desc(&map_wg);
      ptx::tma_prefetch_desc(&map_x0);
      ptx::tma_prefetch_desc(&map_x1);
      Ring st;
      Inflight in_st;
      const CUtensorMap* mh[4] = {&map_h0, &map_h1, &map_h2, &map_h3};
      bool ok = true;
      bool down_maps = false;
      int q = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++q) {
        if (!wait_phase(&info_full[q & 1], (q >> 1) & 1, abort_flag, a.status, a.wait_ns, 0, 11)) { ok = false; break; }
        const UnitInfo& inf = info[q & 1];
        const bool gu = inf.gu != 0;
        const int row_a = inf.row_a, r0 = inf.r0;
        int tok[kNB];
#pragma unroll
        for (int j = 0; j < kNB; ++j) tok[j] = inf.tok[j];
        ptx::mbar_arrive(&info_empty[q & 1]);
        const ModeGeo& M = gu ? MG : MD;
        if (!gu) {
          if (!down_maps) {
            ptx::tma_prefetch_desc(&map_wd);
            for (int t = 0; t < kHTerms; ++t) ptx::tma_prefetch_desc(mh[t]);
            down_maps = true;
          }
          ptx::fence_proxy_async_global();     // h rows of other CTAs, read by TMA
        }
        const CUtensorMap* mw = gu ? &map_wg : &map_wd;
        const CUtensorMap* mwt = gu ? &map_wgt : &map_wdt;
        for (int s = 0; s < M.nstage; ++s) {
          if (!wait_phase(&empty[st.slot], st.phase ^ 1, abort_flag, a.status, a.wait_ns, 64, 4)) { ok = false; break; }
          const int i0 = 2 * s, i1 = min(2 * s + 2, M.nbox);
          // the 4-bit TMA counts the packed bytes it reads (half of what it
          // writes); gate_up's B is two gathers of 4 rows per term
          const uint32_t b_box = gu ? uint32_t(MG.NT * 2 * 4 * kBoxK) : uint32_t(kBRows * kBoxK);
          ptx::mbar_arrive_expect_tx(&full[st.slot], uint32_t(i1 - i0) * (kBoxBytesA / 2 + b_box));
          uint8_t* da = sa + st.slot * G.a_stage;
          uint8_t* db = sb + st.slot * G.b_stage;
          for (int i = i0; i < i1; ++i) {
            uint8_t* dai = da + (i - i0) * kBoxBytesA;
            uint8_t* dbi = db + (i - i0) * kBRows * kBoxK;
            const bool main_box = i < M.nbox_main;
            const CUtensorMap* mwi = main_box ? mw : mwt;
            const int xa = main_box ? i * kBoxK : 0;
            const int xb = i * kBoxK;
            if (gu) {
              ptx::tma_load_3d(dai, mwi, &full[st.slot], xa, row_a, 0);   // gate and up rows
              for (int t = 0; t < MG.NT; ++t) {
                const CUtensorMap* mb = t ? &map_x1 : &map_x0;
                ptx::tma_gather4(dbi + t * MG.rpt * kBoxK, mb, &full[st.slot], xb, tok[0], tok[1],
                                 tok[2], tok[3]);
                ptx::tma_gather4(dbi + t * MG.rpt * kBoxK + 1024, mb, &full[st.slot], xb, tok[4],
                                 tok[5], tok[6], tok[7]);
              }
            } else {
              ptx::tma_load_2d(dai, mwi, &full[st.slot], xa, row_a);
              for (int t = 0; t < MD.NT; ++t)
                ptx::tma_load_2d(dbi + t * MD.rpt * kBoxK, mh[t], &full[st.slot], xb, r0);
            }
          }
          in_st.mark(st.slot, st.phase);
          st.next(S);
        }
      }
      if (!ok) in_st.drain(full, S);
    }
    __syncwarp();                 // the warp reaches the final barrier converged
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------------ MMA issuer --
    if (ptx::elect_one()) {
      uint32_t idesc[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) idesc[j] = ptx::idesc_mx(kMW, kBRows, j, j);
      Ring st;
      bool ok = true;
      int q = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++q) {
        const ModeGeo& M = u < u_gu ? MG : MD;
        const int tail_off = kBoxK - M.tail;          // first tail code inside the tail box
        const int buf = q & 1;
        if (!wait_phase(&acc_empty[buf], ((q >> 1) & 1) ^ 1, abort_flag, a.status, a.wait_ns, 0, 2)) { ok = false; break; }
        if (!wait_phase(&sf_full[buf], (q >> 1) & 1, abort_flag, a.status, a.wait_ns, 0, 3)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kAccCols;
        const uint32_t sfa = tmem_base + sfa_col0 + buf * 4 * G.groups;
        const uint32_t sfb = tmem_base + sfb_col0 + buf * 4 * G.groups;
        uint32_t acc = 0;
        for (int s = 0; s < M.nstage; ++s) {
          if (!wait_phase(&full[st.slot], st.phase, abort_flag, a.status, a.wait_ns, 0, 1)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(sa + st.slot * G.a_stage);
          const uint32_t b_addr = ptx::smem_u32(sb + st.slot * G.b_stage);
          const int i0 = 2 * s, i1 = min(2 * s + 2, M.nbox);
          for (int i = i0; i < i1; ++i) {
            const uint64_t adesc = ptx::desc_kmajor_sw128(a_addr + uint32_t((i - i0) * kBoxBytesA));
            const uint64_t bdesc = ptx::desc_kmajor_sw128(b_addr + uint32_t((i - i0) * kBRows * kBoxK));
            const uint32_t sf_off = uint32_t(4 * i);     // SF group i: K blocks 4i..4i+3
            if (i < M.nbox_main) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                ptx::mma_mx(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc[j], sfa + sf_off, sfb + sf_off, acc);
                acc = 1;
              }
            } else {
              for (int j = 0; j < M.tail / 32; ++j) {
                ptx::mma_mx(d_tmem, adesc + uint64_t((tail_off + 32 * j) >> 4), bdesc + 2 * j, idesc[j],
                            sfa + sf_off, sfb + sf_off, acc);
                acc = 1;
              }
            }
          }
          ptx::mma_commit(&empty[st.slot]);
          st.next(S);
        }
        if (!ok) break;
        ptx::mma_commit(&acc_full[buf]);
        ptx::mma_commit(&sf_empty[buf]);
      }
      ptx::mma_commit(mma_done);
      const long long t0 = clock64();
      while (!ptx::mbar_try_wait(mma_done, 0) && clock64() - t0 < kSpinLimit) {
      }
    }
    __syncwarp();
  } else if (warp >= kWarpSf0 && warp < kWarpSf0 + 4) {
    // ------------------------------------------------------ scale writers --
    const int quarter = warp & 3;
    const uint32_t lane_addr = uint32_t(quarter * 32) << 16;
    const int m = quarter * 32 + lane;             // weight row of the tile = TMEM lane
    int q = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++q) {
      const bool gu = u < u_gu;
      const ModeGeo& M = gu ? MG : MD;
      const int sbuf = q & 1;                      // TMEM scale set
      // B: row n = lane of B at lane n of every lane quarter, column 4g
      // (N = 32).  x terms: row n is term n / 16, token 4 ((n % 16) / 8) +
      // n % 4 of the chunk (rows with n % 8 >= 4 are unused), whose scale row
      // of that term's table this lane reads from L2 (before the waits below,
      // so these loads overlap the weight scales' copy); h terms: row n is
      // term n / 8, scale 2^(h_exp - 4t) for every block.
      const int t0 = lane / M.rpt;
      uint32_t sw[kMaxGroups];
      if (gu) {
        const Unit w = unit_of(a, tabs, MG, MD, u_gu, u);
        const int jx = 4 * ((lane % 16) / 8) + (lane % 4);
        const int tk = __ldg(a.perm + w.r0 + (jx < w.n ? jx : 0)) / a.k;
        const uint32_t* srow =
            reinterpret_cast<const uint32_t*>((t0 ? a.sx_lo : a.sx_hi) + size_t(tk) * a.ld_sx);
#pragma unroll
        for (int g = 0; g < kMaxGroups; ++g)
          if (g < MG.groups) sw[g] = __ldg(srow + g);
      }
      const bool ok = wait_phase(&sc_full[0], q & 1, abort_flag, a.status, a.wait_ns, 64, 6) &&
                      wait_phase(&sf_empty[sbuf], ((q >> 1) & 1) ^ 1, abort_flag, a.status, a.wait_ns, 64, 7);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint32_t ta = tmem_base + lane_addr + sfa_col0 + sbuf * 4 * G.groups;
      const uint32_t tb = tmem_base + lane_addr + sfb_col0 + sbuf * 4 * G.groups;
      // A: row m's word of group g in all four columns 4g..4g+3 (the MMA reads
      // column 4g + m / 32)
      const uint8_t* ra = scb + m * M.nsb;
      for (int g = 0; g < M.groups; ++g) {
        const uint32_t wa = scale_word(ra, g, M.nsb);
        ptx::tmem_st_32x32b_x4(ta + 4 * g, wa, wa, wa, wa);
      }
      if (gu) {
#pragma unroll
        for (int g = 0; g < kMaxGroups; ++g)
          if (g < MG.groups) ptx::tmem_st_32x32b_x1(tb + 4 * g, sw[g]);
      } else {
        const uint32_t c0 = uint32_t(127 + a.h_exp - 4 * t0) * 0x01010101u;
        for (int g = 0; g < MD.groups; ++g) ptx::tmem_st_32x32b_x1(tb + 4 * g, c0);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(&sc_empty[0]);
        ptx::mbar_arrive(&sf_full[sbuf]);
      }
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
    // ------------------------------------------------------------ epilogue --
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;             // TMEM lane = weight row of the tile
    const float hscale = __int_as_float((127 - a.h_exp) << 23);   // 2^-h_exp
    int q = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++q) {
      const Unit w = unit_of(a, tabs, MG, MD, u_gu, u);
      const int buf = q & 1;
      const bool ok0 = wait_phase(&acc_full[buf], (q >> 1) & 1, abort_flag, a.status, a.wait_ns, 256, 8);
      if (!ptx::group_all(1, 128, ok0)) break;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t(quarter * 32) << 16) + buf * kAccCols;
      // D column n holds B row n: gate_up term n / 16 of token
      // 4 ((n % 16) / 8) + n % 4; down term n / 8 of token n % 8
      float z[kNB];
      {
        uint32_t v[2][16];
        ptx::tmem_ld_32x32b_x16(taddr, v[0]);
        ptx::tmem_ld_32x32b_x16(taddr + 16, v[1]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < kNB; ++j) {
          if (w.gu) {
            const int c = 8 * (j / 4) + j % 4;
            z[j] = __uint_as_float(v[0][c]) + __uint_as_float(v[1][c]);
          } else {
            z[j] = (__uint_as_float(v[0][j]) + __uint_as_float(v[0][8 + j])) +
                   (__uint_as_float(v[1][j]) + __uint_as_float(v[1][8 + j]));
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_empty[buf]);
      if (w.gu) {
        const bool is_up = m >= kMW / 2;
        const int n = w.mt * (kMW / 2) + (m & (kMW / 2 - 1));
        const bool nvalid = n < a.W;
        const float bias =
            nvalid ? __bfloat162float(a.b_gu[size_t(w.e) * 2 * a.W + (is_up ? a.W : 0) + n]) : 0.f;
        if (is_up) {
#pragma unroll
          for (int j = 0; j < kNB; ++j) xch[(m - kMW / 2) * kNB + j] = z[j] + bias;
        }
        ptx::named_barrier(2, 128);
        if (!is_up && nvalid) {
#pragma unroll
          for (int j = 0; j < kNB; ++j) {
            if (j < w.n) {
              const float gg = fminf(z[j] + bias, a.limit);
              const float uu = fminf(fmaxf(xch[m * kNB + j], -a.limit), a.limit);
              const float hv = gg * (1.0f / (1.0f + expf(-a.alpha * gg))) * (uu + 1.0f);
              float v = hv * hscale;
              uint8_t* o = a.hq + size_t(w.r0 + j) * a.W + n;
#pragma unroll
              for (int t = 0; t < kHTerms; ++t) {         // v = t0 + t1/16 + t2/256 + t3/4096
                const uint32_t b = to_e4m3(v);
                o[size_t(t) * a.R * a.W] = uint8_t(b);
                v = (v - from_e4m3(b)) * 16.f;
              }
            }
          }
          // the down units read these rows with TMA (the async proxy)
          ptx::fence_proxy_async_global();
        }
        ptx::named_barrier(3, 128);              // h stored; xch is reused by the next unit
        if (m == 0) ptx::red_release_gpu_add(a.ready + w.g, 1);
      } else {
        const int n = w.mt * kMW + m;
        const bool nvalid = n < a.d;
        if (nvalid) {
          const float bias = __bfloat162float(a.b_dn[size_t(w.e) * a.d + n]);
#pragma unroll
          for (int j = 0; j < kNB; ++j)
            if (j < w.n) a.y[size_t(w.r0 + j) * a.d + n] = z[j] + bias;
        }
        // K5: the weighted sum of each token whose k rows are now all stored
        combine_tile<4>(a, w.r0, w.n, w.mt, m, comb, kNB, 2);
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

// [rows, cols] matrix, box {box_cols, box_rows}, 128-byte swizzle; cols and
// box_cols count elements of type dt; row_bytes is the row stride.
cudaError_t make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, long long rows,
                     long long cols, long long row_bytes, int box_cols, int box_rows) {
  auto enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
  const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int plan_stages(const GemmArgs& a) {
  const Geo g0 = geometry(a.d, a.W, 0);
  const int per = g0.a_stage + g0.b_stage;
  int s = (kMaxSmem - 1024 - g0.total) / per;
  return s < kMaxStages ? s : kMaxStages;
}

// gate_up's codes as a 3-D tensor [half][row][code] over the [E 2W, d] table:
// the half dimension steps W rows, so one box at (x, row, 0) holds 64 gate rows
// and the 64 up rows W below them, in that order (one TMA instead of two).
cudaError_t make_gate_up_map(CUtensorMap* map, const void* base, long long rows, long long cols,
                             long long row_bytes, long long half_bytes) {
  auto enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {cuuint64_t(cols), cuuint64_t(rows), 2};
  const cuuint64_t strides[2] = {cuuint64_t(row_bytes), cuuint64_t(half_bytes)};
  const cuuint32_t box[3] = {cuuint32_t(kBoxK), cuuint32_t(kMW / 2), 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The weight maps of one GEMM: the main map and the tail map.
cudaError_t make_weight_maps(bool gu, const GemmArgs& a, CUtensorMap* mw, CUtensorMap* mwt) {
  const int K = gu ? a.d : a.W;
  const uint8_t* w = gu ? a.w_gu : a.w_dn;
  const long long rows = gu ? (long long)a.E * 2 * a.W : (long long)a.E * a.d;
  const int kmain = K / kBoxK * kBoxK;
  if (gu) {
    // the last 128 codes of each row: base at code K - 128 of row 0
    const long long half = (long long)a.W * (K / 2);
    cudaError_t e = make_gate_up_map(mw, w, rows, kmain, K / 2, half);
    if (e != cudaSuccess) return e;
    if (K % kBoxK) return make_gate_up_map(mwt, w + (K - kBoxK) / 2, rows, kBoxK, K / 2, half);
    *mwt = *mw;
    return cudaSuccess;
  }
  cudaError_t e = make_map(mw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w, rows, kmain, K / 2, kBoxK,
                           kMW);
  if (e != cudaSuccess) return e;
  if (K % kBoxK)       // the last 128 codes of each row: base at code K - 128 of row 0
    return make_map(mwt, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w + (K - kBoxK) / 2, rows, kBoxK,
                    K / 2, kBoxK, kMW);
  *mwt = *mw;
  return cudaSuccess;
}

// The ten tensor maps of one launch: gate_up and down weights (main, tail),
// gate_up's token tables [T, d] (a one-row box per gather4 coordinate), down's
// h term tables [R, W] (boxes of a chunk's 8 rows).
cudaError_t make_maps(const GemmArgs& a, CUtensorMap* maps) {
  cudaError_t e = make_weight_maps(true, a, &maps[0], &maps[1]);
  if (e == cudaSuccess) e = make_weight_maps(false, a, &maps[2], &maps[3]);
  const long long T = a.R / a.k;
  for (int t = 0; t < 2 && e == cudaSuccess; ++t)
    e = make_map(&maps[4 + t], CU_TENSOR_MAP_DATA_TYPE_UINT8, t ? a.xq_lo : a.xq_hi, T, a.d, a.d,
                 kBoxK, 1);
  for (int t = 0; t < kHTerms && e == cudaSuccess; ++t)
    e = make_map(&maps[6 + t], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.hq + size_t(t) * a.R * a.W, a.R,
                 a.W, a.W, kBoxK, a.nb);
  return e;
}

bool fits_mode(bool gu, const GemmArgs& a) {
  const int K = gu ? a.d : a.W;
  const int nsb = K / 32;
  if (K < kBoxK || K % 32 || (K / 2) % 16) return false;
  if ((K % kBoxK) && ((K - kBoxK) / 2) % 32) return false;      // tail map base alignment
  if ((nsb + 3) / 4 > kMaxGroups) return false;
  // 1-D copies of scale rows: 16-byte sizes and starts
  const int rpe = gu ? 2 * a.W : a.d;
  if ((size_t(rpe) * nsb) % 16) return false;
  if (gu) {
    if ((64 * nsb) % 16 || ((a.W % 64) * nsb) % 16) return false;
  } else {
    if ((128 * nsb) % 16 || ((a.d % 128) * nsb) % 16) return false;
  }
  return true;
}

struct MapKey {
  const void* p[5];
  int R, d, W, E, nb, k;
};

}  // namespace

int mx_chunk(int64_t, int) { return kNB; }

int mx_hidden_exp(float limit) {
  // |h| = |g sigmoid(alpha g) (u + 1)| <= limit (limit + 1) for the clamped g, u
  const double bound = double(limit) * (double(limit) + 1.0);
  int e = 0;
  while (bound * std::ldexp(1.0, -e) > 448.0) ++e;
  while (e > -20 && bound * std::ldexp(1.0, -(e - 1)) <= 448.0) --e;
  return e;
}

int mx_chunk_bound(int64_t R, int E) { return int(R / kNB + E + 1); }

bool mx_fits(const GemmArgs& args, float limit) {
  // h is carried with a fixed scale, so the clamp must bound it, and tightly
  // enough that typical values stay far above the E4M3 subnormals
  if (!(limit > 0.f) || !std::isfinite(limit) || limit > 16.f) return false;
  GemmArgs a = args;
  a.nb = mx_chunk(a.R, a.E);
  if (a.R / (a.E > 0 ? a.E : 1) > 8) return false;              // a decode-sized load
  if (a.E > kMaxExperts) return false;
  a.ld_sx = scale_row_bytes(a.d);
  return fits_mode(true, a) && fits_mode(false, a) && plan_stages(a) >= 2;
}

cudaError_t launch_experts_mx(const GemmArgs& a, cudaStream_t s) {
  if (a.nb != kNB || a.E > kMaxExperts || !fits_mode(true, a) || !fits_mode(false, a) || !a.ready)
    return cudaErrorInvalidConfiguration;
  const int stages = plan_stages(a);
  if (stages < 2) return cudaErrorInvalidConfiguration;
  const Geo g = geometry(a.d, a.W, stages);
  const size_t smem = size_t(g.total) + 1024;
  if (smem > size_t(kMaxSmem)) return cudaErrorInvalidConfiguration;
  {
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(moe_expert_mx), kMaxSmem);
    if (e != cudaSuccess) return e;
  }
  // the ten maps, from the cache when this layer's buffers were seen before
  MapKey key;
  memset(&key, 0, sizeof(key));
  key.p[0] = a.w_gu;
  key.p[1] = a.w_dn;
  key.p[2] = a.xq_hi;
  key.p[3] = a.xq_lo;
  key.p[4] = a.hq;
  key.R = a.R;
  key.d = a.d;
  key.W = a.W;
  key.E = a.E;
  key.nb = a.nb;
  key.k = a.k;
  static MapCache<MapKey, 10> cache;
  CUtensorMap m[10];
  if (!cache.find(key, m)) {
    cudaError_t e = make_maps(a, m);
    if (e != cudaSuccess) return e;
    cache.put(key, m);
  }
  const ModeGeo MG = mode_geo(true, a.d, a.W), MD = mode_geo(false, a.d, a.W);
  const long long units_bound = (long long)(a.R / a.nb + a.E) * (MG.n_mt + MD.n_mt);
  const int grid = int(units_bound < device_sm_count() ? units_bound : device_sm_count());
  // CTAs wait on each other's gate_up units: all must be resident at once
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, moe_expert_mx, m[0], m[1], m[2], m[3], m[4], m[5], m[6],
                                     m[7], m[8], m[9], a, stages);
  if (e == cudaErrorInvalidValue || e == cudaErrorNotSupported) {
    // a driver that does not combine the two attributes: cooperative alone
    (void)cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, moe_expert_mx, m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7],
                           m[8], m[9], a, stages);
  }
  return e;
}

}  // namespace moe
