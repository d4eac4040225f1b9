// Host-side launchers behind the C ABI (not exported).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace moe {

int num_sms();  // SM count of the current device (cached per device)
// After each kernel launch on `st`: bump the moe_kernel_launches counter and, while a timing
// ring is installed (moe_profile_events), record its next event on `st`.
void count_launch(cudaStream_t st);
void set_last_error(const char* msg);  // the text moe_last_error() returns on this thread
// Test hook behind moe_debug_withhold_stage: true when the tcgen05 launch being prepared must
// withhold its first pipeline stage (one pending request is used up); *wait_ns gets the wait
// limit for that launch (0: the default).
bool debug_take_withhold(unsigned long long* wait_ns);

// gather.cu
void launch_dispatch(int dtype, const void* x, const int* token_ids, int T, int rows, int h,
                     void* xbuf, int* status, cudaStream_t st);
void launch_combine(int dtype, const void* ybuf, const int* slot_of, const float* w, int T, int k,
                    int h, void* y, int* status, cudaStream_t st);
void launch_dispatch_bwd(int dtype, const void* dxbuf, const int* slot_of, const float* dx_add,
                         int T, int k, int h, void* dx, int* status, cudaStream_t st);
void launch_combine_bwd(int dtype, const void* dy, const void* ybuf, const int* slot_of,
                        const float* w, int T, int k, int h, void* dybuf, float* d_w,
                        int* status, cudaStream_t st);

// route.cu
// With `partial` (K-split router partials [slices][T][E]) the logits are summed there in slice
// order, plus `bias`, and written to `logits`; otherwise `logits` is read.
void launch_softmax_topk(float* logits, const float* partial, int slices, const float* bias, int T, int E,
                         int k, bool sigmoid, bool renorm, float* probs, int* topk_idx, float* topk_w,
                         cudaStream_t st);
// With `dl_planes` ([3][T][E] bf16) the kernel also writes the exact three-plane split of d_logits.
void launch_route_dlogits(const float* probs, const int* topk_idx, const float* d_topk_w, int T,
                          int E, int k, bool sigmoid, bool renorm, float* d_logits, void* dl_planes,
                          int* status, cudaStream_t st);

// gshard.cu -- the capacity-buffer (GShard-style) comparison path
void launch_gshard_gate(int dtype, const int* idx, const float* w, int T, int E, int k, int C, void* mask,
                        float* cw, int* loads, int* slot, int* status, cudaStream_t st);
void launch_gshard_dispatch(int dtype, const void* x, const void* mask, int T, int E, int C, int h, void* xe,
                            int* status, cudaStream_t st);
void launch_gshard_combine(int dtype, const float* cw, const void* ye, int T, int E, int C, int h, void* y,
                           int* status, cudaStream_t st);

// pft.cu
int pft_num_chunks(long long Tk);
size_t pft_scratch_bytes(long long Tk, int E);
void launch_pft_build(const int* topk_idx, int T, int E, int k, int* num_ids, int* offsets,
                      int* token_ids, int* expert_ids, int* slot_of, void* ws, cudaStream_t st);

// gemm_simt.cu -- fp32-accumulating SIMT GEMMs (all shapes, both dtypes)
int router_splits(int M, int N, int K);  // split-K factor of a router GEMM (>= 1)
// out[i] = sum over z ascending of partial[z * count + i] (+ bias[i % N]), fp32
void launch_splitk_reduce(const float* partial, int splits, long long count, int N, const float* bias,
                          float* out, cudaStream_t st);
void simt_router_logits(int dtype, const void* x, const float* Wg, const float* bias, int T, int h,
                        int E, float* logits, float* partial, cudaStream_t st);
void simt_router_dwg(int dtype, const void* x, const float* d_logits, int T, int h, int E,
                     float* dWg, float* partial, cudaStream_t st);
void simt_router_dx(const float* d_logits, const float* Wg, int T, int h, int E, float* dx,
                    cudaStream_t st);
void simt_expert_ffn(int dtype, const void* xbuf, const int* offsets, const void* W1,
                     const void* W3, const void* W2, int Tk, int E, int h, int f, void* ybuf,
                     void* h1, void* h3, void* a, cudaStream_t st);
void simt_expert_ffn_bwd(int dtype, const void* dybuf, const void* xbuf, const void* h1,
                         const void* h3, const void* a, const int* offsets, const void* W1,
                         const void* W3, const void* W2, int Tk, int E, int h, int f, void* dxbuf,
                         void* dW1, void* dW3, void* dW2, void* dh1, void* dh3, cudaStream_t st);

// router_tc.cu -- router GEMMs on tcgen05 over exact three-plane bf16 splits (bf16 or fp32
// activations, h a multiple of 64, E of 16).  The scratch follows the workspace header, 256-byte aligned.
bool tc_router_supported(int dtype, int h, int E);
size_t tc_router_scratch(int op, int T, int h, int E, int dtype);  // op 0: forward, 1: backward
// The forward leaves several K slices' partials for launch_softmax_topk to add (*partial_out,
// *slices_out; nullptr and 1 when the logits were written directly).  The backward splits
// d_logits itself unless route_dlogits already wrote its planes at the start of `scratch`.
int tc_router_logits(const void* x, const float* Wg, const float* bias, int T, int h, int E, int dtype,
                     float* logits, void* scratch, const float** partial_out, int* slices_out, int* status,
                     cudaStream_t st);
int tc_router_bwd(const void* x, const float* Wg, const float* d_logits, int T, int h, int E, int dtype,
                  float* dWg, float* dx_router, void* scratch, bool dl_planes_ready, int* status, cudaStream_t st);

// gemm_f32tc.cu -- the fp32 expert forward on tcgen05 over exact three-plane bf16 splits (h and f
// multiples of 128).  The scratch (token planes of the rows and of a, two weight-plane buffers,
// two split counters) follows the workspace header.  The token rows are xbuf, or, with xbuf
// NULL, x[token_ids[p]] (T rows of x).
bool f32tc_supported(int dtype, int h, int f, int E);
size_t f32tc_scratch(long long Tk, int E, int h, int f);
int f32tc_expert_ffn(const float* xbuf, const float* x, const int* token_ids, int T, const int* offsets,
                     const float* W1, const float* W3, const float* W2, int Tk, int E, int h, int f, float* ybuf,
                     float* h1, float* h3, float* a, void* scratch, int* status, cudaStream_t st);

// gemm_tc.cu -- tcgen05/TMEM/TMA grouped GEMMs (bf16; h and f multiples of 128)
bool tc_supported(int dtype, int h, int f);
// Token rows of the padding-free buffer: either xbuf itself ([Tk,h]), or, with xbuf null, row p
// read as x[token_ids[p]] (x: [T,h]) by the GEMMs that consume it (gate/up, dW1/dW3).
struct TokenRows {
  const void* xbuf;
  const void* x;
  const int* token_ids;
  int T;
};
// The combine folded into the down projection (h % 256 == 0): y[t] from ybuf by the unit that
// completes token t's k rows of each 128-row M tile; cnt is [T * h/128] int scratch.
struct CombineFold {
  void* y;
  const int* token_ids;
  const int* slot_of;
  const float* topk_w;
  int T, k;
  int* cnt;
};
int tc_expert_ffn(TokenRows xr, const int* offsets, const void* W1, const void* W3, const void* W2,
                  int Tk, int E, int h, int f, void* ybuf, void* h1, void* h3, void* a, int* status,
                  cudaStream_t st, const CombineFold* fold = nullptr);
int tc_expert_ffn_bwd(const void* dybuf, TokenRows xr, const void* h1, const void* h3, const void* a,
                      const int* offsets, const void* W1, const void* W3, const void* W2, int Tk, int E,
                      int h, int f, void* dxbuf, void* dW1, void* dW3, void* dW2, void* dh1, void* dh3,
                      int* status, cudaStream_t st);

}  // namespace moe
