// Shared device/host definitions of libmoe_b300 (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

// Router tile: tokens per CTA of the router kernel.  Also the granularity of
// the per-tile expert histogram the permutation is built from.
constexpr int kRouterTile = 32;
// Row tile of the grouped GEMMs (tcgen05 M).  An expert's segment of the
// permuted rows is cut into ceil(count / kGemmBM) row tiles.
constexpr int kGemmBM = 128;

// Device status word codes (values equal the public moe_status codes).
constexpr int kStatusTimeout = 7;
constexpr int kStatusBounds = 8;

// Workspace layout (every region 256-byte aligned).
struct Workspace {
  size_t status;       // int32[64]
  size_t topk_idx;     // int32[T*k]
  size_t topk_w;       // float[T*k]
  size_t rank;         // int32[T*k]   rank of (t,j) inside its router tile
  size_t tile_counts;  // int32[ntiles*E]  rows of expert e in router tile
  size_t tile_base;    // int32[ntiles*E]  first permuted row of (tile, e)
  size_t offsets;      // int32[E+1]
  size_t mtile_off;    // int32[E+1]   prefix of ceil(count/kGemmBM)
  size_t perm;         // int32[R]
  size_t inv;          // int32[R]
  size_t xexp;         // int32[T]   per-token exponent e_t of the f16 scaling
  size_t rowexp;       // int32[R]   e_t of the token of each permuted row
  size_t x_perm;       // f16[R, d]  x[t] * 2^e_t
  size_t h_hi;         // bf16[R, W]
  size_t h_lo;         // bf16[R, W]
  size_t y;            // float[R, d]
  size_t total;
};

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
  ws.rank = take(size_t(R) * 4);
  ws.tile_counts = take(size_t(ntiles) * E * 4);
  ws.tile_base = take(size_t(ntiles) * E * 4);
  ws.offsets = take(size_t(E + 1) * 4);
  ws.mtile_off = take(size_t(E + 1) * 4);
  ws.perm = take(size_t(R) * 4);
  ws.inv = take(size_t(R) * 4);
  ws.xexp = take(size_t(T) * 4);
  ws.rowexp = take(size_t(R) * 4);
  ws.x_perm = take(size_t(R) * d * 2);
  ws.h_hi = take(size_t(R) * W * 2);
  ws.h_lo = take(size_t(R) * W * 2);
  ws.y = take(size_t(R) * d * 4);
  ws.total = off;
  return ws;
}

// ---------------------------------------------------------------- kernels --
// Host-side launchers, one per stage.  All return the launch's cudaError_t.

// K1: logits, top-k, selected softmax, per-tile histogram and in-tile ranks,
// and the per-token exponent e_t = 14 - floor(log2 max|x_t|) used to hold x in
// f16 exactly.  Also clears the status word (the first kernel of every call).
cudaError_t launch_router_topk(const __nv_bfloat16* x, const float* router_w,
                               const float* router_b, int T, int d, int E, int k,
                               int32_t* topk_idx, float* topk_w, int32_t* rank,
                               int32_t* tile_counts, int32_t* xexp, int32_t* status,
                               cudaStream_t s);

// K2a: expert offsets, per-(tile, expert) bases, row-tile prefix.
cudaError_t launch_route_scan(const int32_t* tile_counts, int ntiles, int E,
                              int32_t* tile_base, int32_t* offsets, int32_t* mtile_off,
                              cudaStream_t s);

// K2b: perm / inv tables and (optionally) the gathered activations in f16,
// x_perm[row] = x[t] * 2^e_t, rowexp[row] = e_t.
cudaError_t launch_route_scatter(const __nv_bfloat16* x, int T, int d, int E, int k,
                                 const int32_t* topk_idx, const int32_t* rank,
                                 const int32_t* tile_base, const int32_t* xexp, int32_t* perm,
                                 int32_t* inv, void* x_perm, int32_t* rowexp, int32_t* status,
                                 cudaStream_t s);

struct GemmArgs {
  int R, d, W, E;
  const int32_t* offsets;     // [E+1]
  const int32_t* mtile_off;   // [E+1]
  const void* x_perm;         // f16 [R, d], each row scaled by 2^rowexp[row]
  const int32_t* rowexp;      // [R]
  const uint8_t* w_gu; const uint8_t* w_gu_scale; const __nv_bfloat16* b_gu;
  const uint8_t* w_dn; const uint8_t* w_dn_scale; const __nv_bfloat16* b_dn;
  float limit, alpha;
  __nv_bfloat16* h_hi; __nv_bfloat16* h_lo;
  float* y;
  int32_t* status;
};

// K3: h = swiglu(x_perm · W_gu^T + b_gu), per expert segment.
cudaError_t launch_gateup(const GemmArgs& a, cudaStream_t s);
// K4: y = (h_hi + h_lo) · W_dn^T + b_dn, per expert segment.
cudaError_t launch_down(const GemmArgs& a, cudaStream_t s);

// K5: out[t] = bf16(Σ_j w[t,j] · y[inv[t,j]]); a row index outside [0, T·k)
// is skipped and recorded in the status word.
cudaError_t launch_combine(const float* y, const float* topk_w, const int32_t* inv,
                           int T, int d, int k, __nv_bfloat16* out, int32_t* status,
                           cudaStream_t s);

}  // namespace moe
