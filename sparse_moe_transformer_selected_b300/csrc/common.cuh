// Shared device/host definitions of libmoe_b300 (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

// Programmatic dependent launch.  Every kernel of the block is launched with
// the programmatic-serialization attribute, so its launch and prologue overlap
// the previous kernel's tail; each kernel calls pdl_wait() before its first
// global-memory access (it returns once the previous kernel has completed and
// its writes are visible).  A kernel that calls pdl_trigger() lets the next
// one launch once every one of its CTAs has triggered or exited: the TMEM
// design's gate_up does, after its own wait; the others let the next kernel
// launch when they exit.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Host helpers shared by the launchers (defined in moe_abi.cu).
// Sets `kernel`'s dynamic shared-memory limit to `bytes` once per device: the
// attribute belongs to each device's context, so a process that drives
// several GPUs sets it on each.  Thread-safe.
cudaError_t set_smem_limit_once(const void* kernel, int bytes);
// Number of SMs of the current device (cached per device).
int device_sm_count();

// Router tile: tokens per CTA of the router kernel.  Also the granularity of
// the per-tile expert histogram the permutation is built from.
constexpr int kRouterTile = 32;
// Token chunk the routing-only call scans for, and the one the design checks
// start from.  A grouped GEMM cuts each expert's segment of the permuted rows
// into ceil(count / chunk) chunks of its own chunk size.
constexpr int kGemmBM = 128;

// Router work split.  A CTA of the logits kernel takes 32 tokens x a group of
// experts x a range of d.  A decode-sized batch has one or two 32-token tiles,
// so it uses groups of 32 experts and cuts d into ranges (at least 256 long,
// multiples of 32) to give the GPU a few dozen CTAs; the partial sums are added
// in a fixed order.  A prefill batch takes all experts per CTA (more reuse of
// each loaded x value) and few or no d ranges.
inline int router_expert_group(int64_t T, int E) {
  return (T <= 256 || E <= 32) ? 32 : (E + 31) / 32 * 32;
}
inline int router_split_len(int64_t T, int d, int E) {
  const int64_t ntiles = (T + kRouterTile - 1) / kRouterTile;
  const int64_t groups = (E + router_expert_group(T, E) - 1) / router_expert_group(T, E);
  int64_t want = (4 * 148 + ntiles * groups - 1) / (ntiles * groups);
  if (want < 1) want = 1;
  int64_t len = (d + want - 1) / want;
  len = (len + 31) / 32 * 32;
  if (len < 256) len = 256;
  return int(len < d ? len : (d + 31) / 32 * 32);
}
// The tensor-core logits kernel (router_tc.cu): more than 8 router tiles,
// d a multiple of 64.  It cuts d into at most kRouterTcMaxSplits ranges.
constexpr int kRouterTcMaxSplits = 8;
bool router_tc_fits(int64_t T, int d, int E);
int router_tc_e_pad(int E);
inline int router_splits(int64_t T, int d, int E) {
  // at most 8 router tiles: whole dot products, one slab (router_topk.cu)
  if ((T + kRouterTile - 1) / kRouterTile <= 8) return 1;
  if (router_tc_fits(T, d, E)) return kRouterTcMaxSplits;   // slabs reserved; the launch uses <=
  const int len = router_split_len(T, d, E);
  return (d + len - 1) / len;
}

// Device status word codes (values equal the public moe_status codes).
constexpr int kStatusTimeout = 7;
constexpr int kStatusBounds = 8;

// Workspace layout (every region 256-byte aligned).
struct Workspace {
  size_t status;       // int32[64]
  size_t topk_idx;     // int32[T*k]
  size_t topk_w;       // float[T*k]
  size_t logit_part;   // float[nks*T*E] router partial sums, one slab per K range
  size_t rank;         // int32[T*k]   rank of (t,j) inside its router tile
  size_t tile_counts;  // int32[ntiles*E]  rows of expert e in router tile
  size_t tile_base;    // int32[ntiles*E]  first permuted row of (tile, e)
  size_t offsets;      // int32[E+1]
  size_t mtile_off;    // int32[2(E+1)] prefixes of ceil(count/chunk), then of ceil(count/chunk2)
  size_t perm;         // int32[R]
  size_t inv;          // int32[R]
  size_t rowexp;       // int32[R]   e_t of the token of each permuted row
  size_t x_perm;       // f16[R, d]  x[t] * 2^e_t; block-scaled design: E4M3 hi [T, d] then lo [T, d]
  size_t h_hi;         // bf16[R, W]; block-scaled design: 4 E4M3 term tables [R, W] over h_hi and h_lo
  size_t h_lo;         // bf16[R, W]
  size_t y;            // float[R, d]
  size_t sx_hi;        // uint8[T, ld_sx]  UE8M0 block scales of x hi (block-scaled design)
  size_t sx_lo;        // uint8[T, ld_sx]  ... of x lo
  size_t cnt;          // int32[T, ceil(d/128)]  combine counts per (token, output column tile),
                      // then int32[T k / 8 + E + 1]: per token chunk of 8 rows, the gate_up
                      // tiles whose h is stored (block-scaled design)
  size_t rnorm;        // float[T]  1/rms of each token (the block's RMSNorm)
  size_t rw_terms;     // bf16[3, E_pad, d] the router weights as hi, mid, lo (tensor-core router)
  // The block's MoE input bf16(RMSNorm(x)) [T, d] lives at the start of the y
  // region: it is read only by the routing stages, before K4 writes y.
  size_t total;
};

// Output column tiles of the down GEMM (its weight tile is 128 rows of d).
inline int down_col_tiles(int d) { return (d + 127) / 128; }

// Row stride of the activation block-scale tables: d/32 bytes rounded up to a
// multiple of 16 (the rows of a chunk are copied with 1-D bulk copies).
inline int scale_row_bytes(int d) { return (d / 32 + 15) / 16 * 16; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline Workspace workspace_layout(int64_t T, int d, int W, int E, int k) {
  Workspace ws{};
  const int64_t R = T * k;
  const int64_t ntiles = (T + kRouterTile - 1) / kRouterTile;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  ws.status = take(64 * sizeof(int32_t));
  ws.topk_idx = take(size_t(R) * 4);
  ws.topk_w = take(size_t(R) * 4);
  ws.logit_part = take(size_t(router_splits(T, d, E)) * size_t(T) * E * 4);
  ws.rank = take(size_t(R) * 4);
  ws.tile_counts = take(size_t(ntiles) * E * 4);
  ws.tile_base = take(size_t(ntiles) * E * 4);
  ws.offsets = take(size_t(E + 1) * 4);
  ws.mtile_off = take(size_t(E + 1) * 8);
  ws.perm = take(size_t(R) * 4);
  ws.inv = take(size_t(R) * 4);
  ws.rowexp = take(size_t(R) * 4);
  ws.x_perm = take(size_t(R) * d * 2);
  ws.h_hi = take(size_t(R) * W * 2);
  ws.h_lo = take(size_t(R) * W * 2);
  ws.y = take(size_t(R) * d * 4);
  ws.sx_hi = take(size_t(T) * scale_row_bytes(d));
  ws.sx_lo = take(size_t(T) * scale_row_bytes(d));
  ws.cnt = take((size_t(T) * down_col_tiles(d) + size_t(R) / 8 + E + 1) * 4);
  ws.rnorm = take(size_t(T) * 4);
  ws.rw_terms = take(router_tc_fits(T, d, E) ? size_t(3) * router_tc_e_pad(E) * d * 2 : 0);
  ws.total = off;
  return ws;
}

// ---------------------------------------------------------------- kernels --
// Host-side launchers, one per stage.  All return the launch's cudaError_t.

// Arguments of K1 (router_topk.cu).
struct RouteArgs {
  const __nv_bfloat16* x;      // [T, d] the MoE input (for the block: the xn table below)
  const float* router_w;       // [E, d]
  const float* router_b;       // [E]
  // The pre-norm block: x_pre is the residual stream and K1 writes the MoE
  // input xn = bf16(RMSNorm(x_pre)) = bf16(x_pre / sqrt(mean(x_pre²) + eps) · g)
  // into the table x points at.  Null x_pre: x is given as is.
  const __nv_bfloat16* x_pre;  // [T, d] or null
  __nv_bfloat16* xn;           // [T, d] the table x points at (written when x_pre is given)
  const float* norm_w;         // [d]
  float eps;
  int T, d, E, k;
  int chunk;                   // token chunk of gate_up (for mtile_off[0..E])
  int chunk2;                  // token chunk of down (for mtile_off[E+1..2E+1])
  float* logit_part;           // [splits, T, E]
  int32_t* topk_idx;           // [T, k]
  float* topk_w;               // [T, k]
  int32_t* rank;               // [T, k]  rank of (t, j) among its tile's rows of expert e
  int32_t* tile_counts;        // [ntiles, E]
  int32_t* tile_base;          // [ntiles, E]
  int32_t* offsets;            // [E + 1]
  int32_t* mtile_off;          // [2 (E + 1)]
  int32_t* status;             // status word (cleared by the first kernel)
  float* rnorm;                // [T] 1 / rms of each token, written with xn
  int32_t* cnt;                // combine counts, zeroed by the first kernel
  int64_t ncnt;
  // Block-scaled design: the MoE input of every token as two E4M3 term tables
  // [T, d] with UE8M0 block scales [T, ld_sx] (quantize.cuh), or null.
  uint8_t* xq_hi;
  uint8_t* xq_lo;
  uint8_t* sx_hi;
  uint8_t* sx_lo;
  int ld_sx;
  // perm [R] / inv [T k]: written by the last top-k CTA when it runs the scan
  // (null: left to the scatter kernel)
  int32_t* perm;
  int32_t* inv;
  __nv_bfloat16* rw_terms;     // [3, E_pad, d] workspace of the tensor-core router
};

// bf16 (nearest, ties to even) of x·g·r for a bf16 value x, an fp32 g and
// r = 1/rms held in fp64 (r32 = (float)r), decided as for the exact product:
// the fp32 product lies within 2 ulps of it, so its own rounding is the
// exact one unless its low 16 bits are within 4 ulps of the halfway point;
// then the product is recomputed in fp64 (exact for x·g) and rounded there.
__device__ __forceinline__ float rms_scaled_bf16(float x, float g, float r32, double r64) {
  const float p = (x * g) * r32;
  const uint32_t low = __float_as_uint(p) & 0xFFFFu;
  if (low - 0x7FFCu > 8u) return __bfloat162float(__float2bfloat16_rn(p));
  const double v = double(x) * double(g) * r64;
  if (v == 0.0) return 0.f;
  int e;
  const double m = frexp(v, &e);                           // v = m 2^e, 0.5 <= |m| < 1
  return float(ldexp(rint(ldexp(m, 8)), e - 8));           // 8 significant bits, ties to even
}

// K1: logits (K-split partial sums, then summed in order with the bias), top-k,
// selected softmax, per-tile histogram and in-tile ranks.  The first kernel
// also clears the status word and the combine counts.  With norm_w, the
// logits are those of RMSNorm(x) = x / sqrt(mean(x²) + eps) · norm_w.
// When T has at most kFuseScanTiles tiles and tile_base is given, the last
// top-k CTA also runs the expert scan (tile_base, offsets, mtile_off for
// `chunk` and `chunk2`) and, when r.perm is given, writes perm and inv;
// *scanned is set.
// Otherwise the caller launches the scan and the scatter.  With r.xq_hi the
// token tables of the block-scaled design are written too.
cudaError_t launch_router_topk(const RouteArgs& r, bool* scanned, cudaStream_t s);
// K1's logits on the tensor cores (router_tc.cu), when router_tc_fits: the
// weight split, then the partial-logit slabs; *nks = the slabs written.
int router_tc_splits(int64_t T, int d, int E, int* k_len);
cudaError_t launch_router_logits_tc(const RouteArgs& r, int* nks, cudaStream_t s);

// K2a: expert offsets, per-(tile, expert) bases, prefixes of chunks of `chunk`
// rows (mtile_off[0..E]) and of `chunk2` rows (mtile_off[E+1..2E+1]).
cudaError_t launch_route_scan(const int32_t* tile_counts, int ntiles, int E, int chunk, int chunk2,
                              int32_t* tile_base, int32_t* offsets, int32_t* mtile_off,
                              cudaStream_t s);

// K2b: perm / inv tables and (optionally) the gathered activations in f16,
// x_perm[row] = x[t] * 2^e_t with e_t = 14 - floor(log2 max|x_t|) (so the
// token's largest |x| lies in [2^14, 2^15) and every bf16 value is held
// exactly), rowexp[row] = e_t.
cudaError_t launch_route_scatter(const __nv_bfloat16* x, int T, int d, int E, int k,
                                 const int32_t* topk_idx, const int32_t* rank,
                                 const int32_t* tile_base, int32_t* perm, int32_t* inv,
                                 void* x_perm, int32_t* rowexp, int32_t* status,
                                 cudaStream_t s);

struct GemmArgs {
  int R, d, W, E;
  int nb;                     // token chunk (TMEM design: multiple of 16, <= 192; block-scaled: 8)
  int stages_c, stages_b;     // ring depths of the TMEM design (set by its launcher)
  const int32_t* offsets;     // [E+1]
  const int32_t* mtile_off;   // [E+1] prefix of ceil(count / nb)
  const void* x_perm;         // f16 [R, d], each row scaled by 2^rowexp[row]
  const int32_t* rowexp;      // [R]
  const uint8_t* w_gu; const uint8_t* w_gu_scale; const __nv_bfloat16* b_gu;
  const uint8_t* w_dn; const uint8_t* w_dn_scale; const __nv_bfloat16* b_dn;
  float limit, alpha;
  int h_f16;                  // h carried as an f16 pair (else bf16), TMEM design only
  __nv_bfloat16* h_hi; __nv_bfloat16* h_lo;
  float* y;
  int32_t* status;
  // block-scaled design (expert_gemm_mx.cu): activations as sums of E4M3
  // terms, x = (hi + lo / 16) * 2^(s - 127) with s the hi block's UE8M0 byte
  // (the lo table holds s - 4), h = (t0 + t1 / 16 + t2 / 256 + t3 / 4096) * 2^h_exp
  const uint8_t* xq_hi; const uint8_t* xq_lo;   // [T, d], one row per token
  const uint8_t* sx_hi; const uint8_t* sx_lo;   // [T, ld_sx]
  int ld_sx;
  uint8_t* hq;                                  // 4 tables [R, W], term t at hq + t R W
  int h_exp;
  // K5, run by K4's epilogue (combine.cuh): out[t] = bf16(Σ_j w[t,j] y[inv[t,j]]
  // (+ resid[t])), counted per (token, output column tile) in cnt
  int k;
  const int32_t* perm;        // [R]   permuted row -> t k + j
  const int32_t* inv;         // [T k] (t, j) -> permuted row
  const float* topk_w;        // [T k]
  int32_t* cnt;               // [T, n_mt_dn], zero when K4 starts
  int n_mt_dn;
  // block-scaled design: per token chunk, the gate_up tiles whose h rows are
  // stored (zero when the expert kernel starts); a down unit waits for all
  int32_t* ready;
  __nv_bfloat16* out;         // [T, d]
  const __nv_bfloat16* resid; // [T, d] or null
  // failure detection: a bounded wait gives up after wait_ns nanoseconds
  // (status word MOE_ERR_TIMEOUT); inject = 1 (a test hook) makes gate_up's
  // weight producer issue nothing, so the waits for its stages run out
  long long wait_ns;
  int inject;
};

// Nanoseconds of the GPU's global timer (for wait limits).
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// K3: h = swiglu(x_perm · W_gu^T + b_gu), per expert segment, and
// K4: y = (h_hi + h_lo) · W_dn^T + b_dn with the combine in its epilogue,
// with the dequantised weights as the MMA's A operand in tensor memory
// (expert_gemm_tmem.cu); usable when its shared-memory plan fits (the
// reduction length sets the size of the per-unit scale buffers).
bool expert_gemm_tmem_fits(const GemmArgs& a);
// Token chunk of the TMEM design's gate_up (or down) for R routed rows over E
// experts: small chunks (N = 16) when experts get few tokens, so an activation
// stage is a few KB and the ring can be deep; 192 (down: 160) when they get
// many, since each chunk costs one dequantisation of the expert's weights.
int expert_gemm_tmem_chunk(int64_t R, int E, bool gate_up);
// Whether the clamp bounds h well inside the f16 range, so the TMEM design
// carries h as an f16 pair and runs the down GEMM in f16.
bool hidden_fits_f16(float limit);
cudaError_t launch_gateup_tmem(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_down_tmem(const GemmArgs& a, cudaStream_t s);

// K3 / K4 on the block-scaled tensor-core path (expert_gemm_mx.cu): the MXFP4
// weights are consumed as E2M1 codes with their UE8M0 scales by tcgen05.mma
// kind::mxf8f6f4, the activations as E4M3 hi / lo pairs with block scales.
// Usable when mx_fits() holds; gate_up writes h in the pair format down reads.
bool mx_fits(const GemmArgs& a, float limit);
int mx_chunk(int64_t R, int E);
// Exponent of the fixed power-of-two scale of h: |h| <= limit * (limit + 1)
// maps inside the E4M3 range.
int mx_hidden_exp(float limit);
// Chunks the block-scaled design can have for R rows over E experts (the
// length of GemmArgs::ready).
int mx_chunk_bound(int64_t R, int E);
// K3, K4 and K5 of the block-scaled design in one persistent kernel.
cudaError_t launch_experts_mx(const GemmArgs& a, cudaStream_t s);


}  // namespace moe
