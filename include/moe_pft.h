/*
 * moe_pft.h -- C ABI of the padding-free (PFT) Mixture-of-Experts layer for GB300 (sm_103a).
 *
 * The layer is the one the X-MoE review describes (§3 "Training pipeline": PFT build,
 * padding-free gating, padding-free dispatch, expert compute over the uneven buffer,
 * padding-free combine), split into the Gate / Order / Dispatch / Expert / Combine / I-Order
 * modules of the FSMoE report (part 3, item 1 "Modular and non-intrusive design"), on one
 * GPU.  Each forward stage has a backward entry point.
 *
 * Conventions shared by every function:
 *   - Every pointer argument is a DEVICE pointer unless marked "host".  The caller owns all
 *     memory; the library allocates and frees nothing.  Device pointers must be 16-byte
 *     aligned (PyTorch allocations are).
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is the legacy
 *     default stream) and never synchronise the host, except moe_check_status.
 *   - Row-major layouts; indices are int32.  T tokens, h hidden size, E experts, k experts per
 *     token, f expert FFN width, Tk = T*k rows of the padding-free buffer.
 *   - `dtype` (MOE_F32 or MOE_BF16) is the type of activations, expert weights, expert
 *     intermediates and their gradients.  Gating tensors (router weight W_g, bias, logits,
 *     probabilities, gate weights and their gradients) are always fp32.  Arithmetic
 *     accumulates in fp32; each stored tensor is rounded once (round to nearest even).
 *   - `ws` is a workspace of at least moe_workspace_size(op, ...) bytes.  Its first 256 bytes
 *     hold a sticky device status word (the rest is unused): zero them once with
 *     moe_status_reset before the first call.  One workspace sized for the largest op may serve every op on
 *     one stream; calls that share a workspace must not overlap on the GPU.
 *   - Return value: MOE_OK, or a negative MOE_ERR_* code for errors found on the host before
 *     any launch (bad argument, unsupported shape or alignment, small workspace) or reported
 *     by the CUDA runtime at launch (moe_last_error() then has the message).  Errors found on
 *     the device (an index out of range, a bounded wait that gave up) never trap: the kernel
 *     skips the bad element, sets a bit in the status word and carries on; moe_check_status
 *     reads it.
 */
#ifndef MOE_PFT_H
#define MOE_PFT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_PFT_ABI_VERSION 2

enum moe_status_code {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, k > E, ... */
  MOE_ERR_UNSUPPORTED = -2, /* shape or alignment the kernels do not handle */
  MOE_ERR_WORKSPACE = -3,   /* ws is NULL or smaller than moe_workspace_size */
  MOE_ERR_CUDA = -4,        /* a CUDA runtime call failed; see moe_last_error() */
  MOE_ERR_DEVICE = -5       /* moe_check_status found a device-side error bit */
};

enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 };

/* Bits of the device status word (sticky until moe_status_reset). */
enum moe_device_status {
  MOE_STATUS_BAD_INDEX = 1, /* an expert id, token id or slot was out of range; element skipped */
  MOE_STATUS_TIMEOUT = 2    /* a bounded on-device wait gave up; results are invalid */
};

/* moe_route flags */
enum moe_route_flags {
  MOE_ROUTE_FROM_LOGITS = 1, /* `logits` is an input: skip the router GEMM and the bias */
  MOE_ROUTE_SIGMOID = 2,     /* scores p_e = sigmoid(l_e) per expert instead of the softmax */
  MOE_ROUTE_RENORM = 4       /* divide the k selected scores by their sum (weights sum to 1) */
};

/* Operation ids for moe_workspace_size. */
enum moe_op {
  MOE_OP_ROUTE = 0,
  MOE_OP_ROUTE_BWD = 1,
  MOE_OP_PFT_BUILD = 2,
  MOE_OP_DISPATCH = 3,
  MOE_OP_DISPATCH_BWD = 4,
  MOE_OP_EXPERT_FFN = 5,
  MOE_OP_EXPERT_FFN_BWD = 6,
  MOE_OP_COMBINE = 7,
  MOE_OP_COMBINE_BWD = 8,
  MOE_OP_ALL = 9, /* the largest of the above: one workspace for the whole layer */
  MOE_OP_GSHARD = 10 /* the capacity-buffer comparison path (moe_gshard_*) */
};

/* Workspace bytes `op` needs at these sizes (always >= 256, a multiple of 256). */
size_t moe_workspace_size(int op, int T, int h, int E, int k, int f, int dtype);

/* Zero the status word at the start of `ws` (asynchronous on `stream`). */
int moe_status_reset(void* ws, void* stream);

/* Synchronise `stream`, read the status word into *code (host) and return MOE_OK when it is
 * zero, MOE_ERR_DEVICE otherwise.  Not for the hot path. */
int moe_check_status(const void* ws, void* stream, int* code);

/* Message of the last MOE_ERR_CUDA / MOE_ERR_UNSUPPORTED on the calling host thread. */
const char* moe_last_error(void);

int moe_abi_version(void);

/* Diagnostic: number of kernels this library has launched in this process so far (all
 * devices, all host threads; an atomic counter, the only process-wide state it keeps). */
uint64_t moe_kernel_launches(void);

/* Diagnostic per-kernel timing.  `events` is a host array of `capacity` cudaEvent_t handles
 * (created by the caller with timing enabled; the caller keeps the array and the events alive
 * while installed).  While installed, right after its n-th kernel launch (n counting from 0 at
 * installation) the library records events[n % capacity] on the stream of that launch, so the
 * time between consecutive records is one kernel's duration in stream order.  NULL uninstalls.
 * Process-wide; install and use it from one host thread at a time. */
int moe_profile_events(void* const* events, int capacity);

/* Launches recorded since the current moe_profile_events installation. */
uint64_t moe_profile_count(void);

/* Test hook for the bounded waits of the tensor-core kernels (failure injected on the host; off
 * unless called).  The next `launches` tcgen05 kernel launches (expert GEMMs and router GEMMs,
 * in launch order, from any host thread) run with their TMA producer withholding the first
 * pipeline stage of each CTA's first unit: the stage's barrier is never completed, so the MMA
 * warp's wait for it can only end by running out.  The kernel then sets MOE_STATUS_TIMEOUT in
 * the status word, every warp role unwinds, loads already in flight are given time to land, the
 * tensor memory is released and the CTAs exit; the outputs of that launch are invalid.  Those
 * launches wait at most `wait_limit_ns` (1 ms .. 2 s; 0 keeps the default of about 2 s) per wait.
 * A CUDA graph captured while a request is pending keeps the hook in its launches.  Returns
 * MOE_ERR_INVALID_ARG for a negative count or a limit outside that range; 0 launches cancels. */
int moe_debug_withhold_stage(int launches, unsigned long long wait_limit_ns);

/*
 * Gate -- X-MoE review §3 "Training pipeline" step 2 (padding-free gating, no dispatch_mask)
 * and the FlashDMoE blog §1.1 "DMoE operator definition" (each token picks a few experts).
 *   logits[t,e] = sum_c x[t,c] * Wg[c,e] (+ bias[e]);  probs = softmax over the E experts;
 *   topk_idx[t,0..k-1] = the k largest logits, descending, ties to the lower expert index
 *   (selection compares the fp32 logits); topk_w[t,j] = probs[t, topk_idx[t,j]], not
 *   renormalised.  Router variants (the FSMoE report, part 6, lists several routers, sigmoid
 *   among them): MOE_ROUTE_SIGMOID makes probs[t,e] = sigmoid(logits[t,e]) (the selection is
 *   unchanged: both maps are monotone); MOE_ROUTE_RENORM divides the k selected scores by their
 *   sum.  The same gate flags must be passed to moe_route_bwd.
 * x: [T,h] dtype.  Wg: [h,E] fp32.  bias: [E] fp32 or NULL.  logits, probs: [T,E] fp32
 * (logits is an input when flags has MOE_ROUTE_FROM_LOGITS; x, Wg, bias may then be NULL).
 * topk_idx: [T,k] int32.  topk_w: [T,k] fp32.  Requires 1 <= k <= E <= 1024, h % 8 == 0, and,
 * when the logits are computed from x, E % 4 == 0 (16-byte rows of W_g); MOE_ERR_UNSUPPORTED
 * otherwise.
 */
int moe_route(const void* x, const float* Wg, const float* bias, int T, int h, int E, int k,
              int dtype, int flags, float* logits, float* probs, int32_t* topk_idx,
              float* topk_w, void* ws, size_t ws_bytes, void* stream);

/*
 * Gate backward (the adjoint of moe_route; the selection itself has no gradient):
 *   g[t,e] = d_topk_w[t,j] where e = topk_idx[t,j], else 0 (with MOE_ROUTE_RENORM,
 *   g = (d_topk_w[t,j] - sum_i d_topk_w[t,i] topk_w[t,i]) / S, S = sum of the selected probs);
 *   d_logits = probs * (g - sum_e probs*g) (MOE_ROUTE_SIGMOID: probs * (1 - probs) * g);
 *   dWg = x^T d_logits;  dx_router = d_logits Wg^T.  `flags`: the gate flags given to moe_route
 *   (MOE_ROUTE_FROM_LOGITS is ignored here).
 * d_logits: [T,E] fp32 (written).  dWg: [h,E] fp32 (overwritten).  dx_router: [T,h] fp32
 * (overwritten; NULL skips it).  Feed dx_router to moe_dispatch_bwd as `dx_add` so that dx is
 * rounded once.  Same limits as moe_route.
 */
int moe_route_bwd(const void* x, const float* Wg, const float* probs, const int32_t* topk_idx,
                  const float* d_topk_w, int T, int h, int E, int k, int dtype, int flags,
                  float* d_logits, float* dWg, float* dx_router, void* ws, size_t ws_bytes,
                  void* stream);

/*
 * PFT build (Order) -- X-MoE review §3 "Training pipeline" step 1 (flatten and sort
 * top_experts into token_ids / expert_ids) and §3 "Model components" (PFT holds token_ids,
 * expert_ids and num_ids, valid tokens only; memory O(B x H) with B = T*k routed rows,
 * §3 "Core formulas").  The flattened pairs (t, topk_idx[t,j]) are sorted by the unique key
 * (expert, token):
 *   num_ids[e] = #tokens routed to e;  offsets = exclusive prefix sum of num_ids, E+1 entries;
 *   token_ids[p], expert_ids[p] for p in [offsets[e], offsets[e+1]) list expert e's tokens in
 *   ascending order;  slot_of[t*k+j] = p, the row holding (t, topk_idx[t,j]) (I-Order).
 * topk_idx: [T,k] int32, each row k distinct ids in [0,E).  Outputs int32: num_ids [E],
 * offsets [E+1], token_ids [Tk], expert_ids [Tk], slot_of [Tk].  Deterministic.  An id
 * outside [0,E) sets MOE_STATUS_BAD_INDEX and is dropped (the outputs are then incomplete).
 * An id repeated within a row also sets MOE_STATUS_BAD_INDEX; num_ids and offsets then count
 * every entry, the copies share one row of token_ids and one row of that expert's bucket stays
 * unwritten (every write stays inside the arrays).
 * Requires E <= 1024, T*k <= 2^30.
 */
int moe_pft_build(const int32_t* topk_idx, int T, int E, int k, int32_t* num_ids,
                  int32_t* offsets, int32_t* token_ids, int32_t* expert_ids, int32_t* slot_of,
                  void* ws, size_t ws_bytes, void* stream);

/*
 * PFT build without a workspace.  The paper has no counterpart: this is a variant of
 * moe_pft_build for callers that cannot allocate device memory, such as plugins whose host
 * framework owns every allocation and offers no scratch space, or services whose memory plan
 * is fixed at start-up.  It computes exactly what moe_pft_build computes, from the same
 * arguments minus the workspace.  Its scratch is a 1 MiB array in the library's static device
 * memory, which every GPU that loads the library keeps until the process exits.
 *   - Limits: T*k <= 2^30, as for moe_pft_build, and the scratch needed,
 *     moe_workspace_size(MOE_OP_PFT_BUILD, T, 0, E, k, 0, 0), must not exceed 1 MiB
 *     (1,048,576 bytes).  With E <= 431 every T*k up to 2^30 fits; with E = 1024, T*k up to
 *     261,120.  Larger requests return MOE_ERR_UNSUPPORTED and moe_last_error() says why.
 *     T = 0 (an empty batch) zero-fills num_ids and offsets, as moe_pft_build does.
 *   - No allocation: it calls no cudaMalloc, cudaFree or allocating library routine.  The first
 *     call on each device looks up the array's device address (with that device current); make
 *     that first call before any stream capture.  The address is kept per device together with
 *     the id of the CUDA context it belongs to; after a device reset (a new primary context) the
 *     next call looks it up again, so that call too should come before any stream capture.
 *   - Shared state: every call on a device uses the same array.  Each call clears the array's
 *     header (its status word) on `stream` before its kernels run, so calls queued one
 *     after another on one stream are safe; calls that overlap on the GPU (different streams,
 *     or different host threads without ordering) race and corrupt each other's results.
 *   - Errors: an expert id outside [0,E) is dropped and its slot_of entry set to -1, as in
 *     moe_pft_build; there is no status word to read back.
 * Requires T >= 0 and 1 <= k <= E <= 1024.
 */
int moe_pft_build_noalloc(const int32_t* topk_idx, int T, int E, int k, int32_t* num_ids,
                          int32_t* offsets, int32_t* token_ids, int32_t* expert_ids,
                          int32_t* slot_of, void* stream);

/*
 * Dispatch -- X-MoE review §3 "Training pipeline" step 3 and the FlashDMoE blog §5
 * ("payload-efficient data handling": only tokens that need an expert move):
 *   xbuf[p,:] = x[token_ids[p],:] for p < T*k -- one contiguous, expert-major, uneven buffer.
 * x: [T,h] dtype.  xbuf: [T*k,h] dtype.  Bit-exact copy.  Requires h % 8 == 0.
 */
int moe_dispatch(const void* x, const int32_t* token_ids, int T, int k, int h, int dtype,
                 void* xbuf, void* ws, size_t ws_bytes, void* stream);

/*
 * Dispatch backward (adjoint of the gather):
 *   dx[t,:] = dx_add[t,:] + sum_{j=0..k-1} dxbuf[slot_of[t*k+j],:], fp32 sum, rounded once.
 * dxbuf: [T*k,h] dtype.  dx_add: [T,h] fp32 or NULL.  dx: [T,h] dtype (overwritten).
 */
int moe_dispatch_bwd(const void* dxbuf, const int32_t* slot_of, const float* dx_add, int T,
                     int k, int h, int dtype, void* dx, void* ws, size_t ws_bytes, void* stream);

/*
 * Expert compute -- X-MoE review §3 "Training pipeline" step 5 (GEMMs over the uneven
 * token buffer) with FlashDMoE's local in-place tile padding (blog §5): per expert e, rows
 * R = [offsets[e], offsets[e+1]) of xbuf, SwiGLU:
 *   h1 = X_R W1[e];  h3 = X_R W3[e];  a = silu(h1) * h3;  ybuf_R = a W2[e];  silu(z) = z*sigmoid(z).
 * xbuf: [Tk,h].  W1, W3: [E,h,f].  W2: [E,f,h].  ybuf: [Tk,h].  h1, h3, a: [Tk,f] (saved for
 * the backward; a is computed from the fp32 h1, h3 before they are rounded).  All dtype.
 * offsets: [E+1] int32 from moe_pft_build (read on the device; counts never reach the host).
 * Requires h % 8 == 0 and f % 8 == 0.
 */
int moe_expert_ffn(const void* xbuf, const int32_t* offsets, const void* W1, const void* W3,
                   const void* W2, int Tk, int E, int h, int f, int dtype, void* ybuf, void* h1,
                   void* h3, void* a, void* ws, size_t ws_bytes, void* stream);

/*
 * Expert compute backward, from the saved h1, h3, a:
 *   dA = dY W2[e]^T;  dh1 = dA * h3 * silu'(h1);  dh3 = dA * silu(h1);
 *   dxbuf_R = dh1 W1[e]^T + dh3 W3[e]^T;  dW1[e] = X_R^T dh1;  dW3[e] = X_R^T dh3;
 *   dW2[e] = a_R^T dY;  silu'(z) = s(1 + z(1-s)), s = sigmoid(z).
 * dybuf: [Tk,h].  dxbuf: [Tk,h] (overwritten).  dW1, dW3: [E,h,f], dW2: [E,f,h] (overwritten;
 * an expert with no rows gets exact zeros).  All dtype.  The workspace holds dh1 and dh3.
 */
int moe_expert_ffn_bwd(const void* dybuf, const void* xbuf, const void* h1, const void* h3,
                       const void* a, const int32_t* offsets, const void* W1, const void* W3,
                       const void* W2, int Tk, int E, int h, int f, int dtype, void* dxbuf,
                       void* dW1, void* dW3, void* dW2, void* ws, size_t ws_bytes, void* stream);

/*
 * Dispatch folded into the expert GEMMs -- the fused single-GPU path of FlashDMoE's blog (§4,
 * the persistent kernel that gathers its tokens itself instead of staging a dispatched copy).
 * The same results, bit for bit, as moe_dispatch(x, token_ids) followed by moe_expert_ffn /
 * moe_expert_ffn_bwd on the xbuf it writes, without materialising xbuf: the GEMMs that read it
 * (gate/up in the forward, dW1/dW3 in the backward) load row p as x[token_ids[p]].
 * x: [T,h] dtype.  token_ids: [Tk] int32 from moe_pft_build (an id outside [0,T) reads as a
 * zero row and sets MOE_STATUS_BAD_INDEX, as moe_dispatch does).  Other arguments as in
 * moe_expert_ffn / moe_expert_ffn_bwd.  Runs where a tensor-core engine does
 * (moe_expert_ffn_gather_supported): bf16 or fp32 with h and f multiples of 128, and
 * T * h < 2^31; otherwise MOE_ERR_UNSUPPORTED.  In fp32 the forward splits the gathered rows
 * straight into the bf16 planes its GEMMs read; the backward (FMA engine) gathers the rows
 * into dxbuf, takes dW1/dW3 from them, then overwrites dxbuf with dX.
 */
int moe_expert_ffn_gather(const void* x, const int32_t* token_ids, int T, const int32_t* offsets,
                          const void* W1, const void* W3, const void* W2, int Tk, int E, int h, int f,
                          int dtype, void* ybuf, void* h1, void* h3, void* a, void* ws, size_t ws_bytes,
                          void* stream);
int moe_expert_ffn_bwd_gather(const void* dybuf, const void* x, const int32_t* token_ids, int T,
                              const void* h1, const void* h3, const void* a, const int32_t* offsets,
                              const void* W1, const void* W3, const void* W2, int Tk, int E, int h, int f,
                              int dtype, void* dxbuf, void* dW1, void* dW3, void* dW2, void* ws,
                              size_t ws_bytes, void* stream);
/* 1 when moe_expert_ffn_gather / moe_expert_ffn_bwd_gather run for this shape and dtype, else 0
 * (host only; no device access). */
int moe_expert_ffn_gather_supported(int h, int f, int dtype);

/*
 * The fused single-GPU forward of FlashDMoE's blog (§5: one kernel gathers its tokens and
 * combines its results): moe_expert_ffn with the dispatch and/or the combine folded in.
 * xbuf non-NULL: the gate/up GEMM reads xbuf; xbuf NULL: it gathers row p as x[token_ids[p]]
 * (as moe_expert_ffn_gather).  y non-NULL: the down projection also writes
 *   y[t,:] = sum_j topk_w[t,j] * ybuf[slot_of[t*k+j],:]
 * bit for bit as moe_combine does (j ascending, fp32, one rounding); the unit that completes
 * token t's k rows of a 128-row tile of h sums that tile (contribution counters in the
 * workspace, zeroed by the call).  ybuf is written either way.
 * token_ids: [Tk] and slot_of: [Tk] int32 from moe_pft_build; topk_w: [T,k] fp32; Tk == T*k.
 * Tensor-core engine only (bf16, h and f multiples of 128); the combine fold also needs
 * h % 256 == 0; otherwise MOE_ERR_UNSUPPORTED.  The workspace (16-byte aligned) needs
 * moe_workspace_size(MOE_OP_EXPERT_FFN, ...) bytes and, with y, at least 256 + 4*T*(h/128).
 */
int moe_expert_ffn_fused(const void* xbuf, const void* x, const int32_t* token_ids, int T, int k,
                         const int32_t* slot_of, const float* topk_w, const int32_t* offsets, const void* W1,
                         const void* W3, const void* W2, int Tk, int E, int h, int f, int dtype, void* ybuf,
                         void* h1, void* h3, void* a, void* y, void* ws, size_t ws_bytes, void* stream);

/*
 * Combine -- X-MoE review §3 "Training pipeline" step 6 and the FlashDMoE blog §1.1 (results
 * return to the origin and are merged with the gate weights):
 *   y[t,:] = sum_{j=0..k-1} topk_w[t,j] * ybuf[slot_of[t*k+j],:], j ascending, fp32, rounded once.
 * ybuf: [Tk,h] dtype.  topk_w: [T,k] fp32.  y: [T,h] dtype.
 */
int moe_combine(const void* ybuf, const int32_t* slot_of, const float* topk_w, int T, int k,
                int h, int dtype, void* y, void* ws, size_t ws_bytes, void* stream);

/*
 * Combine backward (adjoint of the weighted gather):
 *   dybuf[slot_of[t*k+j],:] = topk_w[t,j] * dy[t,:];  d_topk_w[t,j] = <dy[t,:], ybuf[slot_of[t*k+j],:]>.
 * dy: [T,h] dtype.  dybuf: [Tk,h] dtype (every row written).  d_topk_w: [T,k] fp32.
 */
int moe_combine_bwd(const void* dy, const void* ybuf, const int32_t* slot_of,
                    const float* topk_w, int T, int k, int h, int dtype, void* dybuf,
                    float* d_topk_w, void* ws, size_t ws_bytes, void* stream);

/*
 * The capacity-buffer (GShard-style) data path, the comparison system the padding-free buffers
 * replace -- X-MoE review §3 "Core formulas" (GShard-style dispatching keeps an E x C x H buffer,
 * C a fixed capacity, against the PFT's B x H) and §3 "Training pipeline" step 2 (the PFT gate
 * builds no dispatch_mask); §5 "Ablation" times gating, dispatch and combine against it.  With C
 * the largest expert load nothing is dropped and the layer equals the padding-free one: the
 * experts run on the E*C padded rows (moe_expert_ffn with offsets e*C), and
 * moe_gshard_combine's y equals moe_combine's up to the order of the fp32 sums.
 *
 * moe_gshard_gate: from a top-k selection (topk_idx [T,k] int32, topk_w [T,k] fp32, as moe_route
 * writes them), token t's slot c in expert e is the number of tokens before t that chose e; each
 * (t, j) with c < C sets dispatch_mask[t,e,c] = 1 and combine_w[t,e,c] = topk_w[t,j]; slots at or
 * beyond C are dropped.  dispatch_mask: [T,E,C] dtype; combine_w: [T,E,C] fp32 (both overwritten,
 * zeros elsewhere); loads: [E] int32, the tokens that chose each expert (dropped ones included).
 * An id outside [0,E), or an expert listed twice in a row, sets MOE_STATUS_BAD_INDEX and is
 * skipped.  Workspace: moe_workspace_size(MOE_OP_GSHARD, T, h, E, k, f, dtype).
 */
int moe_gshard_gate(const int32_t* topk_idx, const float* topk_w, int T, int E, int k, int C, int dtype,
                    void* dispatch_mask, float* combine_w, int32_t* loads, void* ws, size_t ws_bytes,
                    void* stream);

/*
 * moe_gshard_dispatch: xe[e,c,:] = sum_t dispatch_mask[t,e,c] * x[t,:] for the one token per
 * padded row a gate mask holds (a row with no token is written as zeros; a column with more than
 * one non-zero sets MOE_STATUS_BAD_INDEX and keeps the first).  x: [T,h]; dispatch_mask:
 * [T,E,C]; xe: [E,C,h]; all dtype.  A mask of 1 copies the row bit for bit.
 */
int moe_gshard_dispatch(const void* x, const void* dispatch_mask, int T, int E, int C, int h, int dtype,
                        void* xe, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_gshard_combine: y[t,:] = sum_{e,c} combine_w[t,e,c] * ye[e,c,:], summed in fp32 in
 * ascending (e, c) order over the non-zero weights (at most 256 per token; more set
 * MOE_STATUS_BAD_INDEX), rounded once.  combine_w: [T,E,C] fp32; ye: [E,C,h] dtype; y: [T,h] dtype.
 */
int moe_gshard_combine(const float* combine_w, const void* ye, int T, int E, int C, int h, int dtype, void* y,
                       void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PFT_H */
