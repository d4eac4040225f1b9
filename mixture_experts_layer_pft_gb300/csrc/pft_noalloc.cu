// moe_pft_build_noalloc: the PFT build with its scratch in a fixed static device array, for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: a host framework that
// owns every device allocation and gives its plugins no scratch, or a service whose memory
// plan is fixed at start-up and forbids allocation afterwards.  This entry point needs only the
// caller's inputs and outputs.  Its scratch (the per-chunk histograms and the 256-byte header
// holding the status word and the last-block counter) lives in g_pft_scratch below, which every
// GPU that loads the library holds until the process exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;  // 1 MiB: 256-byte header + histograms

static __device__ __align__(256) unsigned char g_pft_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
// Per device: the array's device address and the id of the CUDA context it was looked up in.
// A device reset (or any teardown and re-creation of the primary context) gives the device a
// new context id, and the address is looked up again in the new context.
void* g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};

// Driver entry points for the current context and its id (looked up once; no libcuda link).
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};
const CtxFns& ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  return fns;
}

// Id of the CUDA context current on this thread; false when there is none yet (the runtime
// makes the device's primary context current on its first call that needs one).
bool current_ctx_id(unsigned long long* id) {
  const CtxFns& fns = ctx_fns();
  CUcontext ctx = nullptr;
  return fns.get_current && fns.get_id && fns.get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
         fns.get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_pft_scratch on the current device.  The first call on a device (in a
// given context) looks it up with cudaGetSymbolAddress, that device being current; later calls
// in the same context reuse it.  A changed context id triggers a fresh lookup.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long ctx_id = 0;
  const bool have_id = current_ctx_id(&ctx_id);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr || !have_id || g_scratch_ctx[dev] != ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pft_scratch);  // also makes the primary context current
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
    unsigned long long now = 0;
    g_scratch_ctx[dev] = current_ctx_id(&now) ? now : 0;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_pft_build_noalloc(const int32_t* topk_idx, int T, int E, int k, int32_t* num_ids,
                                     int32_t* offsets, int32_t* token_ids, int32_t* expert_ids,
                                     int32_t* slot_of, void* stream) {
  const cudaStream_t st = (cudaStream_t)stream;
  if (!(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E) || !num_ids || !offsets) {
    set_last_error("moe_pft_build_noalloc: need T >= 0, 1 <= k <= E <= 1024 and non-NULL num_ids, offsets");
    return MOE_ERR_INVALID_ARG;
  }
  // the same size limit as moe_pft_build: positions and offsets are int32
  if ((long long)T * k > (1LL << 30)) {
    set_last_error("moe_pft_build_noalloc: T*k above 2^30");
    return MOE_ERR_UNSUPPORTED;
  }
  if (T == 0) {  // the empty batch: every expert gets no rows, as moe_pft_build does
    cudaError_t e = cudaMemsetAsync(num_ids, 0, sizeof(int) * E, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int) * (E + 1), st);
    if (e != cudaSuccess) {
      set_last_error(cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  if (!topk_idx || !token_ids || !expert_ids || !slot_of) {
    set_last_error("moe_pft_build_noalloc: NULL topk_idx, token_ids, expert_ids or slot_of");
    return MOE_ERR_INVALID_ARG;
  }
  const size_t need = moe_workspace_size(MOE_OP_PFT_BUILD, T, 0, E, k, 0, MOE_F32);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "moe_pft_build_noalloc: T=%d, k=%d, E=%d needs %zu bytes of scratch, above the "
             "%zu-byte static maximum",
             T, k, E, need, kNoAllocScratchBytes);
    set_last_error(msg);
    return MOE_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, sizeof(WsHeader), st);  // status + counter
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  launch_pft_build(topk_idx, T, E, k, num_ids, offsets, token_ids, expert_ids, slot_of, scratch, st);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
