// The exported C ABI (include/moe_pft.h): host-side argument checks, workspace layout and
// launches.  Every check happens before any launch; the library allocates nothing.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* msg) {
  snprintf(g_err, sizeof(g_err), "%s", msg);
  return code;
}

int check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(g_err, sizeof(g_err), "%s: %s", what, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round256(size_t b) { return (b + 255) & ~size_t(255); }
size_t esize(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }
bool dtype_ok(int dtype) { return dtype == MOE_F32 || dtype == MOE_BF16; }

int* status_of(void* ws) { return &static_cast<WsHeader*>(ws)->status; }

// bf16 expert GEMMs with h and f multiples of 128 run on the tcgen05 engine; everything else
// (fp32, other shapes) on the SIMT engine.  MOE_PFT_GEMM=simt forces the SIMT engine.
int tc_failure(const char* what) {
  const int rc = check_launch(what);
  if (rc != MOE_OK) return rc;
  snprintf(g_err, sizeof(g_err), "%s: tensor map encoding or kernel attribute setup failed", what);
  return MOE_ERR_CUDA;
}

// Shapes the tensor-core router takes (the workspace is sized for them whatever the engine).
bool router_tc_shape(int dtype, int h, int E) {
  return (dtype == MOE_BF16 || dtype == MOE_F32) && h % 64 == 0 && E % 16 == 0 && E >= 64;
}

bool use_tensor_cores(int dtype, int h, int f) {
  const char* env = getenv("MOE_PFT_GEMM");
  if (env && strcmp(env, "simt") == 0) return false;
  return tc_supported(dtype, h, f);
}

// Shapes whose expert FFN can gather its token rows from x: the bf16 tensor-core engine, and the
// fp32 forward on the tensor cores (its backward gathers the rows into dxbuf for the FMA engine).
bool gather_engine(int dtype, int h, int f) {
  return use_tensor_cores(dtype, h, f) || f32tc_supported(dtype, h, f, 1);
}

#define REQUIRE(cond, code, msg)                                        \
  do {                                                                  \
    if (!(cond)) return fail(code, msg);                                \
  } while (0)

#define REQUIRE_PTR(p) REQUIRE((p) != nullptr && aligned16(p), MOE_ERR_INVALID_ARG, \
                               #p " is NULL or not 16-byte aligned")

}  // namespace

static std::atomic<unsigned long long> g_launches{0};

// Timing ring installed by moe_profile_events (diagnostic; one host thread at a time).
static cudaEvent_t* g_prof_events = nullptr;
static int g_prof_capacity = 0;
static std::atomic<unsigned long long> g_prof_count{0};

void count_launch(cudaStream_t st) {
  g_launches.fetch_add(1ull, std::memory_order_relaxed);
  if (g_prof_events != nullptr && g_prof_capacity > 0) {
    const unsigned long long n = g_prof_count.fetch_add(1ull, std::memory_order_relaxed);
    cudaEventRecord(g_prof_events[n % (unsigned long long)g_prof_capacity], st);
  }
}

void set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

// moe_debug_withhold_stage: tcgen05 launches still to withhold a stage, and their wait limit.
static std::atomic<int> g_withhold{0};
static std::atomic<unsigned long long> g_withhold_wait_ns{0};

bool debug_take_withhold(unsigned long long* wait_ns) {
  *wait_ns = 0;
  int n = g_withhold.load(std::memory_order_relaxed);
  while (n > 0) {
    if (g_withhold.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) {
      *wait_ns = g_withhold_wait_ns.load(std::memory_order_relaxed);
      return true;
    }
  }
  return false;
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return MOE_PFT_ABI_VERSION; }

uint64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_profile_events(void* const* events, int capacity) {
  if (events != nullptr && capacity <= 0) {
    set_last_error("moe_profile_events: capacity must be positive");
    return MOE_ERR_INVALID_ARG;
  }
  g_prof_events = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(events));
  g_prof_capacity = events ? capacity : 0;
  g_prof_count.store(0ull, std::memory_order_relaxed);
  return MOE_OK;
}

uint64_t moe_profile_count(void) { return g_prof_count.load(std::memory_order_relaxed); }

int moe_debug_withhold_stage(int launches, unsigned long long wait_limit_ns) {
  if (launches < 0 || (launches > 0 && wait_limit_ns != 0 && wait_limit_ns < 1000000ull) ||
      wait_limit_ns > 2000000000ull) {
    set_last_error("moe_debug_withhold_stage: need launches >= 0 and a wait limit of 0 or 1 ms .. 2 s");
    return MOE_ERR_INVALID_ARG;
  }
  g_withhold_wait_ns.store(wait_limit_ns, std::memory_order_relaxed);
  g_withhold.store(launches, std::memory_order_relaxed);
  return MOE_OK;
}

const char* moe_last_error(void) { return g_err; }

size_t moe_workspace_size(int op, int T, int h, int E, int k, int f, int dtype) {
  const size_t hdr = sizeof(WsHeader);
  const long long Tk = (long long)std::max(T, 0) * std::max(k, 0);
  switch (op) {
    case MOE_OP_ROUTE: {
      const int sp = (T > 0 && h > 0 && E > 0) ? router_splits(T, E, h) : 1;
      size_t b = sp > 1 ? round256((size_t)sp * T * E * sizeof(float)) : 0;
      if (T > 0 && router_tc_shape(dtype, h, E)) b = std::max(b, tc_router_scratch(0, T, h, E, dtype));
      return hdr + b;
    }
    case MOE_OP_ROUTE_BWD: {
      const int sp = (T > 0 && h > 0 && E > 0) ? router_splits(h, E, T) : 1;
      size_t b = sp > 1 ? round256((size_t)sp * h * E * sizeof(float)) : 0;
      if (T > 0 && router_tc_shape(dtype, h, E)) b = std::max(b, tc_router_scratch(1, T, h, E, dtype));
      return hdr + b;
    }
    case MOE_OP_PFT_BUILD:
      return hdr + round256(pft_scratch_bytes(std::max(Tk, 1LL), std::max(E, 1)));
    case MOE_OP_EXPERT_FFN:
      // the fp32 forward on the tensor cores keeps bf16 planes of its operands in the workspace
      return hdr + (Tk > 0 && f32tc_supported(dtype, h, f, E) ? f32tc_scratch(Tk, E, h, f) : 0);
    case MOE_OP_EXPERT_FFN_BWD:
      return hdr + 2 * round256((size_t)Tk * std::max(f, 0) * esize(dtype));
    case MOE_OP_GSHARD:
      return hdr + round256((size_t)Tk * sizeof(int));
    case MOE_OP_ALL: {
      size_t m = 0;
      for (int o = 0; o < MOE_OP_ALL; ++o) m = std::max(m, moe_workspace_size(o, T, h, E, k, f, dtype));
      return m;
    }
    default:
      return hdr;
  }
}

int moe_status_reset(void* ws, void* stream) {
  REQUIRE(ws != nullptr, MOE_ERR_WORKSPACE, "workspace is NULL");
  cudaMemsetAsync(ws, 0, sizeof(WsHeader), (cudaStream_t)stream);
  return check_launch("moe_status_reset");
}

int moe_check_status(const void* ws, void* stream, int* code) {
  REQUIRE(ws != nullptr && code != nullptr, MOE_ERR_INVALID_ARG, "ws or code is NULL");
  int host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, ws, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) {
    snprintf(g_err, sizeof(g_err), "moe_check_status: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  *code = host;
  return host == 0 ? MOE_OK : MOE_ERR_DEVICE;
}

int moe_route(const void* x, const float* Wg, const float* bias, int T, int h, int E, int k,
              int dtype, int flags, float* logits, float* probs, int32_t* topk_idx,
              float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  const cudaStream_t st = (cudaStream_t)stream;
  const bool from_logits = (flags & MOE_ROUTE_FROM_LOGITS) != 0;
  REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E, MOE_ERR_INVALID_ARG,
          "moe_route: need T >= 0 and 1 <= k <= E <= 1024");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_route: bad dtype");
  REQUIRE(ws != nullptr && ws_bytes >= moe_workspace_size(MOE_OP_ROUTE, T, h, E, k, 0, dtype),
          MOE_ERR_WORKSPACE, "moe_route: workspace too small");
  if (T == 0) return MOE_OK;
  REQUIRE_PTR(logits); REQUIRE_PTR(probs); REQUIRE_PTR(topk_idx); REQUIRE_PTR(topk_w);
  const float* partial = nullptr;  // K-split partials the top-k kernel finishes (tensor-core router)
  int slices = 1;
  if (!from_logits) {
    REQUIRE_PTR(x); REQUIRE_PTR(Wg);
    REQUIRE(h >= 8 && h % 8 == 0, MOE_ERR_UNSUPPORTED, "moe_route: h must be a multiple of 8");
    REQUIRE(E % 4 == 0, MOE_ERR_UNSUPPORTED, "moe_route: E must be a multiple of 4");
    REQUIRE(bias == nullptr || aligned16(bias), MOE_ERR_INVALID_ARG, "moe_route: bias not aligned");
    REQUIRE(aligned16(ws), MOE_ERR_WORKSPACE, "moe_route: workspace not 16-byte aligned");
    char* scratch = static_cast<char*>(ws) + sizeof(WsHeader);
    if (tc_router_supported(dtype, h, E)) {
      REQUIRE(aligned16(x) && aligned16(logits), MOE_ERR_INVALID_ARG, "moe_route: x or logits not aligned");
      if (tc_router_logits(x, Wg, bias, T, h, E, dtype, logits, scratch, &partial, &slices, status_of(ws), st) != 0)
        return tc_failure("moe_route");
    } else {
      simt_router_logits(dtype, x, Wg, bias, T, h, E, logits, reinterpret_cast<float*>(scratch), st);
    }
  }
  launch_softmax_topk(logits, partial, slices, partial != nullptr ? bias : nullptr, T, E, k,
                      (flags & MOE_ROUTE_SIGMOID) != 0, (flags & MOE_ROUTE_RENORM) != 0, probs, topk_idx, topk_w,
                      st);
  return check_launch("moe_route");
}

int moe_route_bwd(const void* x, const float* Wg, const float* probs, const int32_t* topk_idx,
                  const float* d_topk_w, int T, int h, int E, int k, int dtype, int flags,
                  float* d_logits, float* dWg, float* dx_router, void* ws, size_t ws_bytes,
                  void* stream) {
  const cudaStream_t st = (cudaStream_t)stream;
  REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E && h >= 8, MOE_ERR_INVALID_ARG,
          "moe_route_bwd: need T >= 0, 1 <= k <= E <= 1024, h >= 8");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_route_bwd: bad dtype");
  REQUIRE(h % 8 == 0 && E % 4 == 0, MOE_ERR_UNSUPPORTED,
          "moe_route_bwd: h must be a multiple of 8 and E of 4");
  REQUIRE(ws != nullptr && ws_bytes >= moe_workspace_size(MOE_OP_ROUTE_BWD, T, h, E, k, 0, dtype),
          MOE_ERR_WORKSPACE, "moe_route_bwd: workspace too small");
  REQUIRE_PTR(Wg); REQUIRE_PTR(dWg);
  if (T == 0) {  // no tokens: dW_g is exactly zero (x, like every [T, ...] array, may be empty)
    cudaMemsetAsync(dWg, 0, sizeof(float) * (size_t)h * E, st);
    return check_launch("moe_route_bwd");
  }
  REQUIRE_PTR(x); REQUIRE_PTR(probs); REQUIRE_PTR(topk_idx); REQUIRE_PTR(d_topk_w); REQUIRE_PTR(d_logits);
  REQUIRE(dx_router == nullptr || aligned16(dx_router), MOE_ERR_INVALID_ARG,
          "moe_route_bwd: dx_router not aligned");
  REQUIRE(aligned16(ws), MOE_ERR_WORKSPACE, "moe_route_bwd: workspace not 16-byte aligned");
  char* scratch = static_cast<char*>(ws) + sizeof(WsHeader);
  const bool tc = tc_router_supported(dtype, h, E);
  REQUIRE(!tc || (aligned16(x) && aligned16(d_logits) && aligned16(dWg)), MOE_ERR_INVALID_ARG,
          "moe_route_bwd: x, d_logits or dWg not aligned");
  // the tensor-core router reads d_logits as three bf16 planes at the start of the scratch:
  // the gate's backward writes them beside d_logits
  launch_route_dlogits(probs, topk_idx, d_topk_w, T, E, k, (flags & MOE_ROUTE_SIGMOID) != 0,
                       (flags & MOE_ROUTE_RENORM) != 0, d_logits, tc ? scratch : nullptr, status_of(ws), st);
  if (tc) {
    if (tc_router_bwd(x, Wg, d_logits, T, h, E, dtype, dWg, dx_router, scratch, true, status_of(ws), st) != 0)
      return tc_failure("moe_route_bwd");
  } else {
    simt_router_dwg(dtype, x, d_logits, T, h, E, dWg, reinterpret_cast<float*>(scratch), st);
    if (dx_router) simt_router_dx(d_logits, Wg, T, h, E, dx_router, st);
  }
  return check_launch("moe_route_bwd");
}

int moe_pft_build(const int32_t* topk_idx, int T, int E, int k, int32_t* num_ids,
                  int32_t* offsets, int32_t* token_ids, int32_t* expert_ids, int32_t* slot_of,
                  void* ws, size_t ws_bytes, void* stream) {
  const cudaStream_t st = (cudaStream_t)stream;
  REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E, MOE_ERR_INVALID_ARG,
          "moe_pft_build: need T >= 0 and 1 <= k <= E <= 1024");
  REQUIRE((long long)T * k <= (1LL << 30), MOE_ERR_UNSUPPORTED, "moe_pft_build: T*k above 2^30");
  REQUIRE(ws != nullptr && aligned16(ws) &&
              ws_bytes >= moe_workspace_size(MOE_OP_PFT_BUILD, T, 0, E, k, 0, MOE_F32),
          MOE_ERR_WORKSPACE, "moe_pft_build: workspace too small");
  REQUIRE_PTR(num_ids); REQUIRE_PTR(offsets);
  if (T == 0) {
    cudaMemsetAsync(num_ids, 0, sizeof(int) * E, st);
    cudaMemsetAsync(offsets, 0, sizeof(int) * (E + 1), st);
    return check_launch("moe_pft_build");
  }
  REQUIRE_PTR(topk_idx); REQUIRE_PTR(token_ids); REQUIRE_PTR(expert_ids); REQUIRE_PTR(slot_of);
  launch_pft_build(topk_idx, T, E, k, num_ids, offsets, token_ids, expert_ids, slot_of, ws, st);
  return check_launch("moe_pft_build");
}

int moe_dispatch(const void* x, const int32_t* token_ids, int T, int k, int h, int dtype,
                 void* xbuf, void* ws, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0 && k >= 1 && h >= 8, MOE_ERR_INVALID_ARG, "moe_dispatch: need T >= 0, k >= 1, h >= 8");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_dispatch: bad dtype");
  REQUIRE(h % 8 == 0, MOE_ERR_UNSUPPORTED, "moe_dispatch: h must be a multiple of 8");
  REQUIRE(ws != nullptr && ws_bytes >= moe_workspace_size(MOE_OP_DISPATCH, T, h, 1, k, 0, dtype),
          MOE_ERR_WORKSPACE, "moe_dispatch: workspace too small");
  if (T == 0) return MOE_OK;
  REQUIRE_PTR(x); REQUIRE_PTR(token_ids); REQUIRE_PTR(xbuf);
  launch_dispatch(dtype, x, token_ids, T, T * k, h, xbuf, status_of(ws), (cudaStream_t)stream);
  return check_launch("moe_dispatch");
}

int moe_dispatch_bwd(const void* dxbuf, const int32_t* slot_of, const float* dx_add, int T,
                     int k, int h, int dtype, void* dx, void* ws, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0 && k >= 1 && h >= 8, MOE_ERR_INVALID_ARG, "moe_dispatch_bwd: need T >= 0, k >= 1, h >= 8");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_dispatch_bwd: bad dtype");
  REQUIRE(h % 8 == 0, MOE_ERR_UNSUPPORTED, "moe_dispatch_bwd: h must be a multiple of 8");
  REQUIRE(ws != nullptr && ws_bytes >= moe_workspace_size(MOE_OP_DISPATCH_BWD, T, h, 1, k, 0, dtype),
          MOE_ERR_WORKSPACE, "moe_dispatch_bwd: workspace too small");
  if (T == 0) return MOE_OK;
  REQUIRE_PTR(dxbuf); REQUIRE_PTR(slot_of); REQUIRE_PTR(dx);
  REQUIRE(dx_add == nullptr || aligned16(dx_add), MOE_ERR_INVALID_ARG, "moe_dispatch_bwd: dx_add not aligned");
  launch_dispatch_bwd(dtype, dxbuf, slot_of, dx_add, T, k, h, dx, status_of(ws), (cudaStream_t)stream);
  return check_launch("moe_dispatch_bwd");
}

namespace {

int expert_ffn_impl(const char* fn, TokenRows xr, const int32_t* offsets, const void* W1, const void* W3,
                    const void* W2, int Tk, int E, int h, int f, int dtype, void* ybuf, void* h1, void* h3,
                    void* a, void* ws, size_t ws_bytes, cudaStream_t st, const CombineFold* fold = nullptr) {
  REQUIRE(Tk >= 0 && E >= 1 && E <= 1024 && h >= 8 && f >= 8, MOE_ERR_INVALID_ARG,
          "moe_expert_ffn: need Tk >= 0, 1 <= E <= 1024, h >= 8, f >= 8");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_expert_ffn: bad dtype");
  REQUIRE(h % 8 == 0 && f % 8 == 0, MOE_ERR_UNSUPPORTED, "moe_expert_ffn: h and f must be multiples of 8");
  REQUIRE(ws != nullptr && ws_bytes >= moe_workspace_size(MOE_OP_EXPERT_FFN, Tk, h, E, 1, f, dtype),
          MOE_ERR_WORKSPACE, "moe_expert_ffn: workspace too small");
  if (Tk == 0) return MOE_OK;
  REQUIRE(xr.xbuf != nullptr || gather_engine(dtype, h, f), MOE_ERR_UNSUPPORTED,
          "moe_expert_ffn_gather: needs a tensor-core engine (bf16 or fp32, h and f multiples of 128)");
  if (xr.xbuf == nullptr) {
    REQUIRE(xr.T >= 1, MOE_ERR_INVALID_ARG, "moe_expert_ffn_gather: need T >= 1");
    REQUIRE((long long)xr.T * h < (1LL << 31), MOE_ERR_UNSUPPORTED, "moe_expert_ffn_gather: T * h >= 2^31");
    REQUIRE_PTR(xr.x); REQUIRE_PTR(xr.token_ids);
  }
  REQUIRE_PTR(offsets); REQUIRE_PTR(W1); REQUIRE_PTR(W3); REQUIRE_PTR(W2);
  REQUIRE_PTR(ybuf); REQUIRE_PTR(h1); REQUIRE_PTR(h3); REQUIRE_PTR(a);
  if (use_tensor_cores(dtype, h, f)) {
    if (tc_expert_ffn(xr, offsets, W1, W3, W2, Tk, E, h, f, ybuf, h1, h3, a, status_of(ws), st, fold) != 0)
      return tc_failure(fn);
  } else if (f32tc_supported(dtype, h, f, E)) {
    REQUIRE(aligned16(ws), MOE_ERR_WORKSPACE, "moe_expert_ffn: workspace not 16-byte aligned");
    if (f32tc_expert_ffn(static_cast<const float*>(xr.xbuf), static_cast<const float*>(xr.x), xr.token_ids, xr.T,
                         offsets, static_cast<const float*>(W1), static_cast<const float*>(W3),
                         static_cast<const float*>(W2), Tk, E, h, f, static_cast<float*>(ybuf),
                         static_cast<float*>(h1), static_cast<float*>(h3), static_cast<float*>(a),
                         static_cast<char*>(ws) + sizeof(WsHeader), status_of(ws), st) != 0)
      return tc_failure(fn);
  } else {
    simt_expert_ffn(dtype, xr.xbuf, offsets, W1, W3, W2, Tk, E, h, f, ybuf, h1, h3, a, st);
  }
  return check_launch(fn);
}

int expert_ffn_bwd_impl(const char* fn, const void* dybuf, TokenRows xr, const void* h1, const void* h3,
                        const void* a, const int32_t* offsets, const void* W1, const void* W3, const void* W2,
                        int Tk, int E, int h, int f, int dtype, void* dxbuf, void* dW1, void* dW3, void* dW2,
                        void* ws, size_t ws_bytes, cudaStream_t st) {
  REQUIRE(Tk >= 0 && E >= 1 && E <= 1024 && h >= 8 && f >= 8, MOE_ERR_INVALID_ARG,
          "moe_expert_ffn_bwd: need Tk >= 0, 1 <= E <= 1024, h >= 8, f >= 8");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_expert_ffn_bwd: bad dtype");
  REQUIRE(h % 8 == 0 && f % 8 == 0, MOE_ERR_UNSUPPORTED, "moe_expert_ffn_bwd: h and f must be multiples of 8");
  REQUIRE(ws != nullptr && aligned16(ws) &&
              ws_bytes >= moe_workspace_size(MOE_OP_EXPERT_FFN_BWD, Tk, h, E, 1, f, dtype),
          MOE_ERR_WORKSPACE, "moe_expert_ffn_bwd: workspace too small");
  REQUIRE_PTR(dW1); REQUIRE_PTR(dW3); REQUIRE_PTR(dW2);
  if (Tk == 0) {
    const size_t wb = (size_t)E * h * f * esize(dtype);
    cudaMemsetAsync(dW1, 0, wb, st);
    cudaMemsetAsync(dW3, 0, wb, st);
    cudaMemsetAsync(dW2, 0, wb, st);
    return check_launch(fn);
  }
  REQUIRE(xr.xbuf != nullptr || gather_engine(dtype, h, f), MOE_ERR_UNSUPPORTED,
          "moe_expert_ffn_bwd_gather: needs a tensor-core engine (bf16 or fp32, h and f multiples of 128)");
  if (xr.xbuf == nullptr) {
    REQUIRE(xr.T >= 1, MOE_ERR_INVALID_ARG, "moe_expert_ffn_bwd_gather: need T >= 1");
    REQUIRE((long long)xr.T * h < (1LL << 31), MOE_ERR_UNSUPPORTED, "moe_expert_ffn_bwd_gather: T * h >= 2^31");
    REQUIRE_PTR(xr.x); REQUIRE_PTR(xr.token_ids);
  }
  REQUIRE_PTR(dybuf); REQUIRE_PTR(h1); REQUIRE_PTR(h3); REQUIRE_PTR(a);
  REQUIRE_PTR(offsets); REQUIRE_PTR(W1); REQUIRE_PTR(W3); REQUIRE_PTR(W2); REQUIRE_PTR(dxbuf);
  char* base = static_cast<char*>(ws) + sizeof(WsHeader);
  void* dh1 = base;
  void* dh3 = base + round256((size_t)Tk * f * esize(dtype));
  if (use_tensor_cores(dtype, h, f)) {
    if (tc_expert_ffn_bwd(dybuf, xr, h1, h3, a, offsets, W1, W3, W2, Tk, E, h, f, dxbuf, dW1, dW3, dW2,
                          dh1, dh3, status_of(ws), st) != 0)
      return tc_failure(fn);
  } else {
    // the gathered fp32 backward: the FMA engine reads the token rows from dxbuf, gathered there
    // first; it takes dW1/dW3 (their only reader) before dX overwrites them
    const void* rows = xr.xbuf;
    if (rows == nullptr) {
      launch_dispatch(dtype, xr.x, xr.token_ids, xr.T, Tk, h, dxbuf, status_of(ws), st);
      rows = dxbuf;
    }
    simt_expert_ffn_bwd(dtype, dybuf, rows, h1, h3, a, offsets, W1, W3, W2, Tk, E, h, f, dxbuf, dW1,
                        dW3, dW2, dh1, dh3, st);
  }
  return check_launch(fn);
}

}  // namespace

int moe_expert_ffn(const void* xbuf, const int32_t* offsets, const void* W1, const void* W3,
                   const void* W2, int Tk, int E, int h, int f, int dtype, void* ybuf, void* h1,
                   void* h3, void* a, void* ws, size_t ws_bytes, void* stream) {
  if (xbuf == nullptr && Tk > 0) return fail(MOE_ERR_INVALID_ARG, "moe_expert_ffn: null xbuf");
  return expert_ffn_impl("moe_expert_ffn", TokenRows{xbuf, nullptr, nullptr, 0}, offsets, W1, W3, W2, Tk, E, h, f,
                         dtype, ybuf, h1, h3, a, ws, ws_bytes, (cudaStream_t)stream);
}

int moe_expert_ffn_gather(const void* x, const int32_t* token_ids, int T, const int32_t* offsets,
                          const void* W1, const void* W3, const void* W2, int Tk, int E, int h, int f,
                          int dtype, void* ybuf, void* h1, void* h3, void* a, void* ws, size_t ws_bytes,
                          void* stream) {
  return expert_ffn_impl("moe_expert_ffn_gather", TokenRows{nullptr, x, token_ids, T}, offsets, W1, W3, W2, Tk,
                         E, h, f, dtype, ybuf, h1, h3, a, ws, ws_bytes, (cudaStream_t)stream);
}

int moe_expert_ffn_bwd(const void* dybuf, const void* xbuf, const void* h1, const void* h3,
                       const void* a, const int32_t* offsets, const void* W1, const void* W3,
                       const void* W2, int Tk, int E, int h, int f, int dtype, void* dxbuf,
                       void* dW1, void* dW3, void* dW2, void* ws, size_t ws_bytes, void* stream) {
  if (xbuf == nullptr && Tk > 0) return fail(MOE_ERR_INVALID_ARG, "moe_expert_ffn_bwd: null xbuf");
  return expert_ffn_bwd_impl("moe_expert_ffn_bwd", dybuf, TokenRows{xbuf, nullptr, nullptr, 0}, h1, h3, a,
                             offsets, W1, W3, W2, Tk, E, h, f, dtype, dxbuf, dW1, dW3, dW2, ws, ws_bytes,
                             (cudaStream_t)stream);
}

int moe_expert_ffn_bwd_gather(const void* dybuf, const void* x, const int32_t* token_ids, int T,
                              const void* h1, const void* h3, const void* a, const int32_t* offsets,
                              const void* W1, const void* W3, const void* W2, int Tk, int E, int h, int f,
                              int dtype, void* dxbuf, void* dW1, void* dW3, void* dW2, void* ws,
                              size_t ws_bytes, void* stream) {
  return expert_ffn_bwd_impl("moe_expert_ffn_bwd_gather", dybuf, TokenRows{nullptr, x, token_ids, T}, h1, h3,
                             a, offsets, W1, W3, W2, Tk, E, h, f, dtype, dxbuf, dW1, dW3, dW2, ws, ws_bytes,
                             (cudaStream_t)stream);
}

int moe_expert_ffn_fused(const void* xbuf, const void* x, const int32_t* token_ids, int T, int k,
                         const int32_t* slot_of, const float* topk_w, const int32_t* offsets, const void* W1,
                         const void* W3, const void* W2, int Tk, int E, int h, int f, int dtype, void* ybuf,
                         void* h1, void* h3, void* a, void* y, void* ws, size_t ws_bytes, void* stream) {
  const char* fn = "moe_expert_ffn_fused";
  REQUIRE(T >= 1 && k >= 1 && (long long)T * k == Tk, MOE_ERR_INVALID_ARG, "moe_expert_ffn_fused: need Tk == T * k");
  REQUIRE(use_tensor_cores(dtype, h, f), MOE_ERR_UNSUPPORTED,
          "moe_expert_ffn_fused: needs the tensor-core engine (bf16, h and f multiples of 128)");
  REQUIRE(y == nullptr || h % 256 == 0, MOE_ERR_UNSUPPORTED, "moe_expert_ffn_fused: the combine fold needs h % 256 == 0");
  REQUIRE_PTR(token_ids);
  CombineFold cf{};
  if (y != nullptr) {
    REQUIRE_PTR(slot_of); REQUIRE_PTR(topk_w);
    const size_t need = sizeof(WsHeader) + (size_t)T * (h / 128) * sizeof(int);
    REQUIRE(ws != nullptr && aligned16(ws) && ws_bytes >= need, MOE_ERR_WORKSPACE,
            "moe_expert_ffn_fused: workspace too small for the combine counters");
    cf = CombineFold{y, token_ids, slot_of, topk_w, T, k, reinterpret_cast<int*>(static_cast<char*>(ws) + sizeof(WsHeader))};
  }
  const TokenRows xr = xbuf != nullptr ? TokenRows{xbuf, nullptr, nullptr, 0} : TokenRows{nullptr, x, token_ids, T};
  return expert_ffn_impl(fn, xr, offsets, W1, W3, W2, Tk, E, h, f, dtype, ybuf, h1, h3, a, ws, ws_bytes,
                         (cudaStream_t)stream, y != nullptr ? &cf : nullptr);
}

int moe_expert_ffn_gather_supported(int h, int f, int dtype) {
  return dtype_ok(dtype) && h >= 8 && f >= 8 && gather_engine(dtype, h, f) ? 1 : 0;
}

int moe_combine(const void* ybuf, const int32_t* slot_of, const float* topk_w, int T, int k,
                int h, int dtype, void* y, void* ws, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0 && k >= 1 && h >= 8, MOE_ERR_INVALID_ARG, "moe_combine: need T >= 0, k >= 1, h >= 8");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_combine: bad dtype");
  REQUIRE(h % 8 == 0, MOE_ERR_UNSUPPORTED, "moe_combine: h must be a multiple of 8");
  REQUIRE(ws != nullptr && ws_bytes >= moe_workspace_size(MOE_OP_COMBINE, T, h, 1, k, 0, dtype),
          MOE_ERR_WORKSPACE, "moe_combine: workspace too small");
  if (T == 0) return MOE_OK;
  REQUIRE_PTR(ybuf); REQUIRE_PTR(slot_of); REQUIRE_PTR(topk_w); REQUIRE_PTR(y);
  launch_combine(dtype, ybuf, slot_of, topk_w, T, k, h, y, status_of(ws), (cudaStream_t)stream);
  return check_launch("moe_combine");
}

int moe_combine_bwd(const void* dy, const void* ybuf, const int32_t* slot_of,
                    const float* topk_w, int T, int k, int h, int dtype, void* dybuf,
                    float* d_topk_w, void* ws, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0 && k >= 1 && k <= 32 && h >= 8, MOE_ERR_INVALID_ARG,
          "moe_combine_bwd: need T >= 0, 1 <= k <= 32, h >= 8");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_combine_bwd: bad dtype");
  REQUIRE(h % 8 == 0, MOE_ERR_UNSUPPORTED, "moe_combine_bwd: h must be a multiple of 8");
  REQUIRE(ws != nullptr && ws_bytes >= moe_workspace_size(MOE_OP_COMBINE_BWD, T, h, 1, k, 0, dtype),
          MOE_ERR_WORKSPACE, "moe_combine_bwd: workspace too small");
  if (T == 0) return MOE_OK;
  REQUIRE_PTR(dy); REQUIRE_PTR(ybuf); REQUIRE_PTR(slot_of); REQUIRE_PTR(topk_w);
  REQUIRE_PTR(dybuf); REQUIRE_PTR(d_topk_w);
  launch_combine_bwd(dtype, dy, ybuf, slot_of, topk_w, T, k, h, dybuf, d_topk_w, status_of(ws),
                     (cudaStream_t)stream);
  return check_launch("moe_combine_bwd");
}

int moe_gshard_gate(const int32_t* topk_idx, const float* topk_w, int T, int E, int k, int C, int dtype,
                    void* dispatch_mask, float* combine_w, int32_t* loads, void* ws, size_t ws_bytes,
                    void* stream) {
  REQUIRE(T >= 1 && E >= 1 && E <= 1024 && k >= 1 && k <= E && C >= 1, MOE_ERR_INVALID_ARG,
          "moe_gshard_gate: need T >= 1, 1 <= k <= E <= 1024, C >= 1");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_gshard_gate: bad dtype");
  REQUIRE((long long)T * k <= (1LL << 30), MOE_ERR_UNSUPPORTED, "moe_gshard_gate: T*k above 2^30");
  REQUIRE(ws != nullptr && aligned16(ws) &&
              ws_bytes >= moe_workspace_size(MOE_OP_GSHARD, T, 0, E, k, 0, dtype),
          MOE_ERR_WORKSPACE, "moe_gshard_gate: workspace too small");
  REQUIRE_PTR(topk_idx); REQUIRE_PTR(topk_w); REQUIRE_PTR(dispatch_mask); REQUIRE_PTR(combine_w);
  REQUIRE_PTR(loads);
  int* slot = reinterpret_cast<int*>(static_cast<char*>(ws) + sizeof(WsHeader));
  launch_gshard_gate(dtype, topk_idx, topk_w, T, E, k, C, dispatch_mask, combine_w, loads, slot, status_of(ws),
                     (cudaStream_t)stream);
  return check_launch("moe_gshard_gate");
}

int moe_gshard_dispatch(const void* x, const void* dispatch_mask, int T, int E, int C, int h, int dtype,
                        void* xe, void* ws, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 1 && E >= 1 && C >= 1 && h >= 8, MOE_ERR_INVALID_ARG,
          "moe_gshard_dispatch: need T >= 1, E >= 1, C >= 1, h >= 8");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_gshard_dispatch: bad dtype");
  REQUIRE(h % 8 == 0, MOE_ERR_UNSUPPORTED, "moe_gshard_dispatch: h must be a multiple of 8");
  REQUIRE(ws != nullptr && ws_bytes >= sizeof(WsHeader), MOE_ERR_WORKSPACE, "moe_gshard_dispatch: workspace too small");
  REQUIRE_PTR(x); REQUIRE_PTR(dispatch_mask); REQUIRE_PTR(xe);
  launch_gshard_dispatch(dtype, x, dispatch_mask, T, E, C, h, xe, status_of(ws), (cudaStream_t)stream);
  return check_launch("moe_gshard_dispatch");
}

int moe_gshard_combine(const float* combine_w, const void* ye, int T, int E, int C, int h, int dtype, void* y,
                       void* ws, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 1 && E >= 1 && C >= 1 && h >= 8, MOE_ERR_INVALID_ARG,
          "moe_gshard_combine: need T >= 1, E >= 1, C >= 1, h >= 8");
  REQUIRE(dtype_ok(dtype), MOE_ERR_INVALID_ARG, "moe_gshard_combine: bad dtype");
  REQUIRE(h % 8 == 0, MOE_ERR_UNSUPPORTED, "moe_gshard_combine: h must be a multiple of 8");
  REQUIRE((long long)E * C < (1LL << 31), MOE_ERR_UNSUPPORTED, "moe_gshard_combine: E*C at or above 2^31");
  REQUIRE(ws != nullptr && ws_bytes >= sizeof(WsHeader), MOE_ERR_WORKSPACE, "moe_gshard_combine: workspace too small");
  REQUIRE_PTR(combine_w); REQUIRE_PTR(ye); REQUIRE_PTR(y);
  launch_gshard_combine(dtype, combine_w, ye, T, E, C, h, y, status_of(ws), (cudaStream_t)stream);
  return check_launch("moe_gshard_combine");
}

}  // extern "C"
