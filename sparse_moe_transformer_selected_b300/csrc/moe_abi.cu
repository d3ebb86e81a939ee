// C ABI of libmoe_b300 (declared in include/moe.h): argument checking, the
// workspace layout and the launch sequence K1 -> K4 (K5 runs in K4's
// epilogue) on the caller's stream.
#include "moe.h"
#include "common.cuh"

#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

namespace {

thread_local std::string g_last_error;
// failure detection: the GEMMs' wait limit and the test hook (per thread)
constexpr long long kDefaultWaitNs = 2000000000ll;
thread_local long long g_wait_ns = kDefaultWaitNs;
thread_local int g_inject = 0;
constexpr int kTraceEvents = 7;
thread_local cudaEvent_t g_trace[kTraceEvents];
thread_local bool g_trace_on = false;

cudaError_t trace(int i, cudaStream_t s) {
  return g_trace_on ? cudaEventRecord(g_trace[i], s) : cudaSuccess;
}

moe_status fail(moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

moe_status check_shape(int64_t T, int d, int W, int E, int k) {
  if (T < 0) return fail(MOE_ERR_SHAPE, "T = %lld < 0", (long long)T);
  if (d <= 0 || d % 32) return fail(MOE_ERR_SHAPE, "d = %d must be a positive multiple of 32", d);
  if (W <= 0 || W % 32) return fail(MOE_ERR_SHAPE, "W = %d must be a positive multiple of 32", W);
  if (E < 1 || E > 256) return fail(MOE_ERR_SHAPE, "E = %d outside [1, 256]", E);
  if (k < 1 || k > 8 || k > E) return fail(MOE_ERR_SHAPE, "k = %d outside [1, min(E, 8)]", k);
  if (T * k >= (int64_t(1) << 31)) return fail(MOE_ERR_SHAPE, "T*k = %lld too large", (long long)(T * k));
  return MOE_OK;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// sm_103 check, once per device.
moe_status check_device() {
  static std::mutex mu;
  static int arch_ok[64];  // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(MOE_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    arch_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
    if (arch_ok[dev] == 2) {
      g_last_error = "device is sm_" + std::to_string(major) + std::to_string(minor) +
                     "; this library is built for sm_103a only";
    }
  }
  if (arch_ok[dev] != 1) return fail(MOE_ERR_UNSUPPORTED, "device is not sm_103 (B300)");
  return MOE_OK;
}

// Which grouped-GEMM design runs K3/K4:
//   Mx    block-scaled MMA on the E2M1 codes (expert_gemm_mx.cu): decode-sized
//         loads (a few rows per expert) with a clamp that bounds h
//   Tmem  dequantised weights as the MMA's A operand in tensor memory
//         (expert_gemm_tmem.cu): everything else
// MOE_GEMM=tmem skips the first (a diagnostic knob; both meet the same
// tolerances).  None: no design's shared-memory plan fits the shape.
enum class Design { None, Tmem, Mx };

moe::GemmArgs gemm_args(int64_t T, int d, int W, int E, int k) {
  moe::GemmArgs a{};
  a.R = int(T * k);
  a.d = d;
  a.W = W;
  a.E = E;
  a.k = k;
  a.nb = moe::kGemmBM;
  return a;
}

Design gemm_design(int64_t T, int d, int W, int E, int k, float limit) {
  const moe::GemmArgs a = gemm_args(T, d, W, E, k);
  const char* s = getenv("MOE_GEMM");
  const bool no_mx = s && strcmp(s, "tmem") == 0;
  if (!no_mx && moe::mx_fits(a, limit)) return Design::Mx;
  if (moe::expert_gemm_tmem_fits(a)) return Design::Tmem;
  return Design::None;
}

template <class T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

// Routing tables inside the workspace, as K1/K2 arguments.
// norm_w != null: x is the block's residual stream and the routing stages
// read its normalised copy, written by K1 at the start of the y region.
moe::RouteArgs route_args(void* ws, const moe::Workspace& L, const void* x, int64_t T, int d,
                          const float* rw, const float* rb, const float* norm_w, float eps,
                          int E, int k, int chunk, int chunk2) {
  moe::RouteArgs r{};
  r.router_w = rw;
  r.router_b = rb;
  r.norm_w = norm_w;
  r.eps = eps;
  if (norm_w) {
    r.x_pre = static_cast<const __nv_bfloat16*>(x);
    r.xn = at<__nv_bfloat16>(ws, L.y);
    r.x = r.xn;
  } else {
    r.x = static_cast<const __nv_bfloat16*>(x);
  }
  r.T = int(T);
  r.d = d;
  r.E = E;
  r.k = k;
  r.chunk = chunk;
  r.chunk2 = chunk2;
  r.logit_part = at<float>(ws, L.logit_part);
  r.topk_idx = at<int32_t>(ws, L.topk_idx);
  r.topk_w = at<float>(ws, L.topk_w);
  r.rank = at<int32_t>(ws, L.rank);
  r.tile_counts = at<int32_t>(ws, L.tile_counts);
  r.tile_base = at<int32_t>(ws, L.tile_base);
  r.offsets = at<int32_t>(ws, L.offsets);
  r.mtile_off = at<int32_t>(ws, L.mtile_off);
  r.status = at<int32_t>(ws, L.status);
  r.rnorm = at<float>(ws, L.rnorm);
  r.cnt = at<int32_t>(ws, L.cnt);
  r.ncnt = T * moe::down_col_tiles(d);
  r.perm = at<int32_t>(ws, L.perm);
  r.inv = at<int32_t>(ws, L.inv);
  r.rw_terms = moe::router_tc_fits(T, d, E) ? at<__nv_bfloat16>(ws, L.rw_terms) : nullptr;
  return r;
}

// K1, K2a, K2b on stream s (trace events 1..3 after each stage).  x_perm:
// the TMEM design's gathered f16 rows (null for the block-scaled design, whose
// token tables K1 writes).  The scan and the scatter run as kernels of their
// own only when K1's last top-k CTA did not run them (more than 8 router
// tiles, or rows to gather).
moe_status run_route(const moe::RouteArgs& r, int32_t* rowexp, void* x_perm, cudaStream_t s) {
  const int ntiles = int((r.T + moe::kRouterTile - 1) / moe::kRouterTile);
  bool scanned = false;
  cudaError_t e = moe::launch_router_topk(r, &scanned, s);
  if (e != cudaSuccess) return cuda_fail(e, "router_topk launch");
  if ((e = trace(1, s)) != cudaSuccess) return cuda_fail(e, "trace event");
  if (!scanned) {
    e = moe::launch_route_scan(r.tile_counts, ntiles, r.E, r.chunk, r.chunk2, r.tile_base,
                               r.offsets, r.mtile_off, s);
    if (e != cudaSuccess) return cuda_fail(e, "route_scan launch");
  }
  if ((e = trace(2, s)) != cudaSuccess) return cuda_fail(e, "trace event");
  if (x_perm || !scanned || !r.perm) {
    e = moe::launch_route_scatter(r.x, r.T, r.d, r.E, r.k, r.topk_idx, r.rank, r.tile_base,
                                  r.perm, r.inv, x_perm, rowexp, r.status, s);
    if (e != cudaSuccess) return cuda_fail(e, "route_scatter launch");
  }
  if ((e = trace(3, s)) != cudaSuccess) return cuda_fail(e, "trace event");
  return MOE_OK;
}

// Checks shared by moe_forward and moe_block_forward.
moe_status check_forward_args(const void* x_bf16, int64_t T, int d, int W, const float* router_w,
                              const float* router_b, const uint8_t* w_gu_fp4,
                              const uint8_t* w_gu_scale, const void* b_gu_bf16,
                              const uint8_t* w_dn_fp4, const uint8_t* w_dn_scale,
                              const void* b_dn_bf16, int E, int k, float limit, float alpha,
                              const void* out_bf16, const void* workspace) {
  moe_status st = check_shape(T, d, W, E, k);
  if (st != MOE_OK) return st;
  const void* ptrs[] = {x_bf16, router_w, router_b, w_gu_fp4, w_gu_scale, b_gu_bf16,
                        w_dn_fp4, w_dn_scale, b_dn_bf16, out_bf16, workspace};
  const char* names[] = {"x", "router_w", "router_b", "w_gu", "w_gu_scale", "b_gu",
                         "w_dn", "w_dn_scale", "b_dn", "out", "workspace"};
  for (int i = 0; i < 11; ++i) {
    if (T > 0 && !ptrs[i]) return fail(MOE_ERR_NULL, "%s is NULL", names[i]);
    if (misaligned(ptrs[i])) return fail(MOE_ERR_ALIGN, "%s is not 16-byte aligned", names[i]);
  }
  if (alpha != alpha || limit != limit) return fail(MOE_ERR_SHAPE, "limit/alpha is NaN");
  return MOE_OK;
}

// The whole block (arguments already checked, T > 0).  norm_w == null: x is
// the MoE input (moe_forward); otherwise x is the residual stream, the MoE
// reads RMSNorm(x) and out = x + MoE (moe_block_forward).
moe_status forward_impl(const void* x_bf16, int64_t T, int d, int W, const float* norm_w,
                        float eps, const float* router_w, const float* router_b,
                        const uint8_t* w_gu_fp4, const uint8_t* w_gu_scale, const void* b_gu_bf16,
                        const uint8_t* w_dn_fp4, const uint8_t* w_dn_scale, const void* b_dn_bf16,
                        int E, int k, float limit, float alpha, void* out_bf16, void* workspace,
                        size_t workspace_bytes, void* stream) {
  const moe::Workspace L = moe::workspace_layout(T, d, W, E, k);
  if (workspace_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, L.total);
  moe_status st = check_device();
  if (st != MOE_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  moe::GemmArgs a = gemm_args(T, d, W, E, k);
  Design design = gemm_design(T, d, W, E, k, limit);
  // the block-scaled path reads the weights with 4-bit TMA maps, whose base
  // addresses want 32-byte alignment (the tail map starts inside a row)
  if (design == Design::Mx &&
      ((reinterpret_cast<uintptr_t>(w_gu_fp4) | reinterpret_cast<uintptr_t>(w_dn_fp4)) & 31u))
    design = moe::expert_gemm_tmem_fits(a) ? Design::Tmem : Design::None;
  if (design == Design::None)
    return fail(MOE_ERR_UNSUPPORTED, "no grouped-GEMM design fits d = %d, W = %d", d, W);
  const bool mx = design == Design::Mx;
  // token chunks: one for both GEMMs in the block-scaled design; the TMEM
  // design's gate_up and down take their own (the scan writes both prefixes)
  a.nb = mx ? moe::mx_chunk(a.R, E) : moe::expert_gemm_tmem_chunk(a.R, E, true);
  const int nb_dn = mx ? a.nb : moe::expert_gemm_tmem_chunk(a.R, E, false);
  moe::RouteArgs r = route_args(workspace, L, x_bf16, T, d, router_w, router_b, norm_w, eps, E,
                                k, a.nb, nb_dn);
  // the block-scaled design's per-chunk counts follow the combine counts and
  // are zeroed with them
  if (mx) r.ncnt += moe::mx_chunk_bound(a.R, E);
  int32_t* rowexp = at<int32_t>(workspace, L.rowexp);
  void* x_perm = nullptr;
  if (mx) {                                    // token tables of the E4M3 terms
    r.xq_hi = at<uint8_t>(workspace, L.x_perm);
    r.xq_lo = at<uint8_t>(workspace, L.x_perm + size_t(T) * d);
    r.sx_hi = at<uint8_t>(workspace, L.sx_hi);
    r.sx_lo = at<uint8_t>(workspace, L.sx_lo);
    r.ld_sx = moe::scale_row_bytes(d);
  } else {
    x_perm = at<void>(workspace, L.x_perm);
  }
  cudaError_t e = trace(0, s);
  if (e != cudaSuccess) return cuda_fail(e, "trace event");
  st = run_route(r, rowexp, x_perm, s);
  if (st != MOE_OK) return st;

  a.offsets = r.offsets;
  a.mtile_off = r.mtile_off;
  a.x_perm = x_perm;
  a.rowexp = rowexp;
  a.w_gu = w_gu_fp4;
  a.w_gu_scale = w_gu_scale;
  a.b_gu = static_cast<const __nv_bfloat16*>(b_gu_bf16);
  a.w_dn = w_dn_fp4;
  a.w_dn_scale = w_dn_scale;
  a.b_dn = static_cast<const __nv_bfloat16*>(b_dn_bf16);
  a.limit = limit;
  a.alpha = alpha;
  a.h_f16 = !mx && moe::hidden_fits_f16(limit) ? 1 : 0;
  a.h_hi = at<__nv_bfloat16>(workspace, L.h_hi);
  a.h_lo = at<__nv_bfloat16>(workspace, L.h_lo);
  a.y = at<float>(workspace, L.y);
  a.status = r.status;
  a.perm = r.perm;
  a.inv = r.inv;
  a.topk_w = r.topk_w;
  a.cnt = r.cnt;
  a.n_mt_dn = moe::down_col_tiles(d);
  a.ready = mx ? r.cnt + T * a.n_mt_dn : nullptr;
  a.out = static_cast<__nv_bfloat16*>(out_bf16);
  a.resid = norm_w ? static_cast<const __nv_bfloat16*>(x_bf16) : nullptr;
  a.wait_ns = g_wait_ns;
  a.inject = g_inject;
  if (mx) {
    a.xq_hi = r.xq_hi;
    a.xq_lo = r.xq_lo;
    a.sx_hi = r.sx_hi;
    a.sx_lo = r.sx_lo;
    a.ld_sx = r.ld_sx;
    a.hq = at<uint8_t>(workspace, L.h_hi);
    a.h_exp = moe::mx_hidden_exp(limit);
  }
  if (mx) {
    // K3, K4 and K5 in one kernel: trace events 4 and 5 both follow it
    e = moe::launch_experts_mx(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "expert kernel launch");
    if ((e = trace(4, s)) != cudaSuccess) return cuda_fail(e, "trace event");
  } else {
    e = moe::launch_gateup_tmem(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "gate_up launch");
    if ((e = trace(4, s)) != cudaSuccess) return cuda_fail(e, "trace event");
    // K4 with K5 in its epilogue, over chunks of nb_dn rows
    moe::GemmArgs ad = a;
    ad.nb = nb_dn;
    ad.mtile_off = r.mtile_off + E + 1;
    e = moe::launch_down_tmem(ad, s);
    if (e != cudaSuccess) return cuda_fail(e, "down launch");
  }
  if ((e = trace(5, s)) != cudaSuccess) return cuda_fail(e, "trace event");
  if ((e = trace(6, s)) != cudaSuccess) return cuda_fail(e, "trace event");
  return MOE_OK;
}

}  // namespace

namespace moe {
// Lets other translation units of the library report through moe_last_error().
void set_last_error(const std::string& msg) { g_last_error = msg; }

cudaError_t set_smem_limit_once(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;   // (kernel, device)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& kd : done)
    if (kd.first == kernel && kd.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.emplace_back(kernel, dev);
  return e;
}

int device_sm_count() {
  static std::atomic<int> count[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = count[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}
}  // namespace moe

extern "C" {

size_t moe_workspace_bytes(int64_t T, int d, int W, int E, int k) {
  if (check_shape(T, d, W, E, k) != MOE_OK) return 0;
  if (T == 0) return 0;
  return moe::workspace_layout(T, d, W, E, k).total;
}

moe_status moe_workspace_region(int64_t T, int d, int W, int E, int k, int which,
                                size_t* offset, size_t* bytes) {
  moe_status st = check_shape(T, d, W, E, k);
  if (st != MOE_OK) return st;
  if (!offset || !bytes) return fail(MOE_ERR_NULL, "offset/bytes pointer is NULL");
  const moe::Workspace L = moe::workspace_layout(T, d, W, E, k);
  const size_t R = size_t(T) * k;
  switch (which) {
    case 0: *offset = L.topk_idx; *bytes = R * 4; break;
    case 1: *offset = L.topk_w; *bytes = R * 4; break;
    case 2: *offset = L.offsets; *bytes = size_t(E + 1) * 4; break;
    case 3: *offset = L.perm; *bytes = R * 4; break;
    case 4: *offset = L.inv; *bytes = R * 4; break;
    case 5: *offset = L.x_perm; *bytes = R * d * 2; break;
    case 6: *offset = L.h_hi; *bytes = R * W * 2; break;
    case 7: *offset = L.h_lo; *bytes = R * W * 2; break;
    case 8: *offset = L.y; *bytes = R * d * 4; break;
    default: return fail(MOE_ERR_SHAPE, "unknown workspace region %d", which);
  }
  return MOE_OK;
}

moe_status moe_forward(const void* x_bf16, int64_t T, int d, int W, const float* router_w,
                       const float* router_b, const uint8_t* w_gu_fp4, const uint8_t* w_gu_scale,
                       const void* b_gu_bf16, const uint8_t* w_dn_fp4, const uint8_t* w_dn_scale,
                       const void* b_dn_bf16, int E, int k, float limit, float alpha,
                       void* out_bf16, void* workspace, size_t workspace_bytes, void* stream) {
  moe_status st = check_forward_args(x_bf16, T, d, W, router_w, router_b, w_gu_fp4, w_gu_scale,
                                     b_gu_bf16, w_dn_fp4, w_dn_scale, b_dn_bf16, E, k, limit,
                                     alpha, out_bf16, workspace);
  if (st != MOE_OK || T == 0) return st;
  return forward_impl(x_bf16, T, d, W, nullptr, 0.f, router_w, router_b, w_gu_fp4, w_gu_scale,
                      b_gu_bf16, w_dn_fp4, w_dn_scale, b_dn_bf16, E, k, limit, alpha, out_bf16,
                      workspace, workspace_bytes, stream);
}

moe_status moe_block_forward(const void* x_bf16, int64_t T, int d, int W, const float* norm_w,
                             float eps, const float* router_w, const float* router_b,
                             const uint8_t* w_gu_fp4, const uint8_t* w_gu_scale,
                             const void* b_gu_bf16, const uint8_t* w_dn_fp4,
                             const uint8_t* w_dn_scale, const void* b_dn_bf16, int E, int k,
                             float limit, float alpha, void* out_bf16, void* workspace,
                             size_t workspace_bytes, void* stream) {
  moe_status st = check_forward_args(x_bf16, T, d, W, router_w, router_b, w_gu_fp4, w_gu_scale,
                                     b_gu_bf16, w_dn_fp4, w_dn_scale, b_dn_bf16, E, k, limit,
                                     alpha, out_bf16, workspace);
  if (st != MOE_OK) return st;
  if (T > 0 && !norm_w) return fail(MOE_ERR_NULL, "norm_w is NULL");
  if (misaligned(norm_w)) return fail(MOE_ERR_ALIGN, "norm_w is not 16-byte aligned");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(MOE_ERR_SHAPE, "eps must be finite and >= 0");
  if (T == 0) return MOE_OK;
  return forward_impl(x_bf16, T, d, W, norm_w, eps, router_w, router_b, w_gu_fp4, w_gu_scale,
                      b_gu_bf16, w_dn_fp4, w_dn_scale, b_dn_bf16, E, k, limit, alpha, out_bf16,
                      workspace, workspace_bytes, stream);
}

moe_status moe_route(const void* x_bf16, int64_t T, int d, const float* router_w,
                     const float* router_b, int E, int k, int32_t* topk_idx, float* topk_w,
                     int32_t* offsets, int32_t* perm, int32_t* inv, void* workspace,
                     size_t workspace_bytes, void* stream) {
  // The route tables do not depend on W; use the smallest legal width for sizing.
  moe_status st = check_shape(T, d, 32, E, k);
  if (st != MOE_OK) return st;
  const void* ptrs[] = {x_bf16, router_w, router_b, workspace, topk_idx, topk_w, offsets, perm, inv};
  const char* names[] = {"x", "router_w", "router_b", "workspace", "topk_idx", "topk_w",
                         "offsets", "perm", "inv"};
  for (int i = 0; i < 9; ++i) {
    if (i < 4 && T > 0 && !ptrs[i]) return fail(MOE_ERR_NULL, "%s is NULL", names[i]);
    if (misaligned(ptrs[i])) return fail(MOE_ERR_ALIGN, "%s is not 16-byte aligned", names[i]);
  }
  if (T == 0) return MOE_OK;
  const moe::Workspace L = moe::workspace_layout(T, d, 32, E, k);
  // Only the routing prefix of the layout is touched: everything before x_perm.
  if (workspace_bytes < L.x_perm)
    return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, L.x_perm);
  st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  moe::RouteArgs r = route_args(workspace, L, x_bf16, T, d, router_w, router_b, nullptr, 0.f, E,
                                k, moe::kGemmBM, moe::kGemmBM);
  r.ncnt = 0;                                  // no combine follows
  st = run_route(r, nullptr, nullptr, s);
  if (st != MOE_OK) return st;
  const size_t R = size_t(T) * k;
  struct { void* dst; const void* src; size_t n; } copies[] = {
      {topk_idx, r.topk_idx, R * 4}, {topk_w, r.topk_w, R * 4},
      {offsets, r.offsets, size_t(E + 1) * 4}, {perm, r.perm, R * 4}, {inv, r.inv, R * 4}};
  for (auto& c : copies) {
    if (!c.dst) continue;
    cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync of a route table");
  }
  return MOE_OK;
}

moe_status moe_poll_status(const void* workspace, void* stream) {
  if (!workspace) return fail(MOE_ERR_NULL, "workspace is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int32_t word = 0;
  e = cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy of the status word");
  if (word == MOE_ERR_TIMEOUT) return fail(MOE_ERR_TIMEOUT, "a device-side wait ran out");
  if (word == MOE_ERR_DEVICE_BOUNDS) return fail(MOE_ERR_DEVICE_BOUNDS, "a device index was out of range");
  if (word != 0) return fail(MOE_ERR_CUDA, "unexpected device status %d", word);
  return MOE_OK;
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

moe_status moe_hidden_format(int64_t T, int d, int W, int E, int k, float limit, int* format,
                             int* exponent) {
  moe_status st = check_shape(T, d, W, E, k);
  if (st != MOE_OK) return st;
  if (!format) return fail(MOE_ERR_NULL, "format is NULL");
  const Design design = T > 0 ? gemm_design(T, d, W, E, k, limit) : Design::Tmem;
  int f = MOE_HIDDEN_BF16_PAIR, x = 0;
  if (design == Design::Mx) {
    f = MOE_HIDDEN_E4M3_TERMS;
    x = moe::mx_hidden_exp(limit);
  } else if (design == Design::Tmem && moe::hidden_fits_f16(limit)) {
    f = MOE_HIDDEN_F16_PAIR;
  }
  *format = f;
  if (exponent) *exponent = x;
  return MOE_OK;
}

moe_status moe_set_wait_limit(double seconds) {
  if (seconds == 0.0) {
    g_wait_ns = kDefaultWaitNs;
    return MOE_OK;
  }
  if (!(seconds >= 1e-4 && seconds <= 60.0))
    return fail(MOE_ERR_SHAPE, "wait limit %g s outside [1e-4, 60] (0 restores 2 s)", seconds);
  g_wait_ns = (long long)(seconds * 1e9);
  return MOE_OK;
}

moe_status moe_set_fault_injection(int mode) {
  if (mode < 0 || mode > 1) return fail(MOE_ERR_SHAPE, "unknown fault-injection mode %d", mode);
  g_inject = mode;
  return MOE_OK;
}

moe_status moe_set_trace_events(void* const* events, int n) {
  if (n == 0 || events == nullptr) {
    g_trace_on = false;
    return MOE_OK;
  }
  if (n != kTraceEvents) return fail(MOE_ERR_SHAPE, "need %d trace events, got %d", kTraceEvents, n);
  for (int i = 0; i < kTraceEvents; ++i) {
    if (!events[i]) return fail(MOE_ERR_NULL, "trace event %d is NULL", i);
    g_trace[i] = static_cast<cudaEvent_t>(events[i]);
  }
  g_trace_on = true;
  return MOE_OK;
}

}  // extern "C"
