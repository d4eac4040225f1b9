// moe_pft_build_noalloc: the PFT build with its scratch in a fixed static device array, for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: a host framework that
// owns every device allocation and gives its plugins no scratch, or a service whose memory
// plan is fixed at start-up and forbids allocation afterwards.  This entry point needs only the
// caller's inputs and outputs.  Its scratch (the per-chunk histograms and the 256-byte header
// holding the status word and the last-block counter) lives in g_pft_scratch below, which every
// GPU that loads the library holds until the process exits.
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
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_pft_scratch on the current device.  The first call on a device looks it
// up (cudaGetSymbolAddress, with that device current); later calls reuse it.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pft_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
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
  if (!(T >= 1 && E >= 1 && E <= 1024 && k >= 1 && k <= E) || !topk_idx || !num_ids || !offsets ||
      !token_ids || !expert_ids || !slot_of) {
    set_last_error("moe_pft_build_noalloc: need T >= 1, 1 <= k <= E <= 1024 and non-NULL pointers");
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
