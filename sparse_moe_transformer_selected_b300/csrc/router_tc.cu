// K1 router logits on the tensor cores, for batches of more than 8 router
// tiles ("OpenAI 最新开源模型 gpt-oss 架构与训练解析", 模型架构: the router is
// a linear layer giving one logit per expert; top-4 of them are taken).
//
//   logits[t, e] = Σ_k x[t, k] · W_r[e, k]        x bf16, W_r fp32
//
// W_r is split once per call into three bf16 terms, W = hi + mid + lo
// (hi = bf16(W), mid = bf16(W - hi), lo = bf16(W - hi - mid)); each
// difference is exact in fp32 and the three terms hold W's 24 significant
// bits, so hi + mid + lo = W for every normal fp32 value.  Each product of a
// bf16 x with a bf16 term is exact in fp32, and tcgen05.mma kind::f16 sums
// them in fp32: the logits are fp32 sums of the exact products, as the CUDA-
// core kernel's are, in another order.
//
// MMA: M = 128 experts (A = the three W terms, K-major), N = 128 tokens (B =
// x, K-major, straight from the [T, d] table), K = 16 per instruction, three
// instructions (hi, mid, lo) per K step into one fp32 accumulator in TMEM.
// One CTA per (token tile, d range, expert tile); the d ranges' partial sums
// go to the partial-logit slabs the top-k kernel adds in order, with the bias.
//   warp 0      TMA producer: per 64-K stage the three A tiles and the B tile
//   warp 1      TMEM allocator and MMA issuer (one elected thread)
//   warps 2-5   epilogue: TMEM lane quarter = warp % 4, lanes = experts
#include "common.cuh"
#include "map_cache.cuh"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

namespace moe {
namespace {

constexpr int kM = 128;                        // experts per tile (MMA M)
constexpr int kN = 128;                        // tokens per tile (MMA N)
constexpr int kK = 64;                         // K per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 3;
constexpr int kTileA = kM * kK * 2;            // 16 KB per W term
constexpr int kTileB = kN * kK * 2;            // 16 KB of x
constexpr int kStage = 3 * kTileA + kTileB;    // 64 KB
constexpr int kThreads = 192;
constexpr long long kWaitCycles = 4000000000ll;
constexpr int kSmem = kStages * kStage + 1024 + 256;

// W_r [E, d] fp32 -> terms [3][E_pad][d] bf16 (rows E .. E_pad - 1 zero).
// Also the first kernel of the call on this path: clears the call's status
// words and combine counts.
__global__ void __launch_bounds__(256) router_w_split_kernel(const RouteArgs r, __nv_bfloat16* terms,
                                                             int e_pad) {
  pdl_wait();
  const int64_t n = int64_t(e_pad) * r.d;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t first = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (first == 0) {
    r.status[0] = 0;
    r.status[1] = 0;
    r.status[4] = 0;
  }
  for (int64_t i = first; i < r.ncnt; i += stride) r.cnt[i] = 0;
  for (int64_t i = first; i < n; i += stride) {
    const int64_t e = i / r.d;
    const float w = e < r.E ? r.router_w[i] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    terms[i] = hi;
    terms[n + i] = mid;
    terms[2 * n + i] = lo;
  }
}

__device__ __forceinline__ bool spin(uint64_t* bar, uint32_t parity, int32_t* status) {
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicMax(status, kStatusTimeout);
      return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
router_logits_tc_kernel(const __grid_constant__ CUtensorMap map_w,   // terms [3 E_pad, d]
                        const __grid_constant__ CUtensorMap map_x,   // x [T, d]
                        const RouteArgs r, int e_pad, int k_len) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kStages * kStage);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint32_t* tbase = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tbase + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kN, ks = blockIdx.y, e0 = blockIdx.z * kM;
  const int kb = ks * k_len, ke = min(r.d, kb + k_len);
  const int nst = (ke - kb) / kK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tbase, kN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tbase;
  pdl_wait();

  if (warp == 0) {
    if (ptx::elect_one()) {
      ptx::tma_prefetch_desc(&map_w);
      ptx::tma_prefetch_desc(&map_x);
      int slot = 0;
      uint32_t ph = 0;
      uint32_t issued = 0, parity = 0;         // stages in flight, for a drain on abort
      bool ok = true;
      for (int s = 0; s < nst; ++s) {
        if (!spin(&empty[slot], ph ^ 1, r.status) || *abort_flag) { *abort_flag = 1; ok = false; break; }
        uint8_t* st = sm + slot * kStage;
        ptx::mbar_arrive_expect_tx(&full[slot], kStage);
        const int k = kb + s * kK;
        for (int t = 0; t < 3; ++t) ptx::tma_load_2d(st + t * kTileA, &map_w, &full[slot], k, t * e_pad + e0);
        ptx::tma_load_2d(st + 3 * kTileA, &map_x, &full[slot], k, t0);
        issued |= 1u << slot;
        parity = (parity & ~(1u << slot)) | (ph << slot);
        if (++slot == kStages) { slot = 0; ph ^= 1; }
      }
      if (!ok) {                               // let the copies in flight land
        const long long t0c = clock64();
        for (int s = 0; s < kStages; ++s)
          if (issued >> s & 1u)
            while (!ptx::mbar_try_wait(&full[s], (parity >> s) & 1u) && clock64() - t0c < kWaitCycles) {
            }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (ptx::elect_one()) {
      const uint32_t idesc = ptx::idesc_f16(kM, kN, true);
      int slot = 0;
      uint32_t ph = 0;
      uint32_t acc = 0;
      for (int s = 0; s < nst; ++s) {
        if (!spin(&full[slot], ph, r.status)) { *abort_flag = 1; break; }
        ptx::tc_fence_after();
        const uint32_t base = ptx::smem_u32(sm + slot * kStage);
        const uint64_t bdesc = ptx::desc_kmajor_sw128(base + 3 * kTileA);
#pragma unroll
        for (int kk = 0; kk < kK / 16; ++kk) {            // 32 bytes of the row per K16
#pragma unroll
          for (int t = 0; t < 3; ++t) {
            const uint64_t adesc = ptx::desc_kmajor_sw128(base + t * kTileA);
            ptx::mma_f16(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, acc);
            acc = 1;
          }
        }
        ptx::mma_commit(&empty[slot]);
        if (++slot == kStages) { slot = 0; ph ^= 1; }
      }
      ptx::mma_commit(done);                              // also when nothing was issued
    }
    __syncwarp();
  } else {
    // epilogue: lane = expert e0 + 32 q + lane, column c = token t0 + c
    const int q = warp & 3;
    const int e = e0 + 32 * q + lane;
    const bool ok = spin(done, 0, r.status) && !*abort_flag;
    ptx::tc_fence_after();
    if (__all_sync(0xffffffffu, ok) && nst > 0) {
      float* part = r.logit_part + size_t(ks) * r.T * r.E;
      for (int c0 = 0; c0 < kN; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tmem + (uint32_t(32 * q) << 16) + c0, v);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int t = t0 + c0 + j;
          if (t < r.T && e < r.E) part[size_t(t) * r.E + e] = __uint_as_float(v[j]);
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kN);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// bf16 [rows, cols] row-major, box {64, 128}, 128-byte swizzle.
cudaError_t make_bf16_map(CUtensorMap* map, const void* base, long long rows, long long cols) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(cols * 2)};
  const cuuint32_t box[2] = {cuuint32_t(kK), cuuint32_t(kN)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult res = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

struct MapKey {
  const void* p[2];
  int64_t T;
  int d, E;
};

}  // namespace

bool router_tc_fits(int64_t T, int d, int E) {
  return (T + kRouterTile - 1) / kRouterTile > 8 && d % kK == 0 && d >= kK && E >= 1 && E <= 256;
}

int router_tc_e_pad(int E) { return (E + kM - 1) / kM * kM; }

int router_tc_splits(int64_t T, int d, int E, int* k_len) {
  const int64_t tiles = ((T + kN - 1) / kN) * (router_tc_e_pad(E) / kM);
  // as many d ranges as keep the CTAs within one wave (a CTA per SM): a
  // partial second wave of these short, latency-bound CTAs costs a whole CTA time
  int64_t want = int64_t(device_sm_count()) / tiles;
  const int64_t stages = d / kK;
  if (want > stages) want = stages;
  if (want > kRouterTcMaxSplits) want = kRouterTcMaxSplits;
  if (want < 1) want = 1;
  const int64_t per = (stages + want - 1) / want;         // stages per d range
  if (k_len) *k_len = int(per * kK);
  return int((stages + per - 1) / per);                  // every range has a stage
}

cudaError_t launch_router_logits_tc(const RouteArgs& r, int* nks_out, cudaStream_t s) {
  const int e_pad = router_tc_e_pad(r.E);
  int k_len = 0;
  const int nks = router_tc_splits(r.T, r.d, r.E, &k_len);
  *nks_out = nks;
  __nv_bfloat16* terms = r.rw_terms;
  if (!terms) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(router_w_split_kernel, dim3(4 * device_sm_count()), dim3(256), 0, s,
                             r, terms, e_pad);
  if (e != cudaSuccess) return e;
  if ((e = set_smem_limit_once(reinterpret_cast<const void*>(router_logits_tc_kernel), kSmem)) !=
      cudaSuccess)
    return e;
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.p[0] = terms;
  key.p[1] = r.x;
  key.T = r.T;
  key.d = r.d;
  key.E = r.E;
  static MapCache<MapKey, 2> cache;
  CUtensorMap m[2];
  if (!cache.find(key, m)) {
    if ((e = make_bf16_map(&m[0], terms, 3LL * e_pad, r.d)) != cudaSuccess) return e;
    if ((e = make_bf16_map(&m[1], r.x, r.T, r.d)) != cudaSuccess) return e;
    cache.put(key, m);
  }
  const dim3 grid(unsigned((r.T + kN - 1) / kN), unsigned(nks), unsigned(e_pad / kM));
  return launch_pdl(router_logits_tc_kernel, grid, dim3(kThreads), size_t(kSmem), s, m[0], m[1], r,
                    e_pad, k_len);
}

}  // namespace moe
