// Gating: softmax over E experts and top-k selection, one warp per token; and the gate's
// backward through the softmax Jacobian.  The router GEMMs (x·W_g, x^T·d_logits,
// d_logits·W_g^T) run elsewhere (tensor-core or FP32 FMA engines); the top-k kernel can finish a
// K-split logits GEMM (adding its partials in slice order), and the backward can emit the bf16
// planes the tensor-core engine consumes.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kWarpsPerBlock = 8;

// PL logits per lane (expert e = lane + 32*i), E <= 32*PL.  The k winners are found by k
// rounds of a warp arg-max under the order (logit descending, expert index ascending), so
// ties go to the lower index and the result equals a full stable sort's first k entries.
// Scores: softmax over the E experts, or (sigmoid) each expert's logistic score on its own;
// both are monotone in the logit, so the selection is the same.  With renorm the k selected
// scores are divided by their sum.
template <int PL>
__global__ void __launch_bounds__(kWarpsPerBlock * kWarp) softmax_topk_kernel(
    float* __restrict__ logits, const float* __restrict__ partial, int slices, const float* __restrict__ bias,
    int T, int E, int k, bool sigmoid, bool renorm, float* __restrict__ probs, int* __restrict__ topk_idx,
    float* __restrict__ topk_w) {
  const int lane = threadIdx.x % kWarp;
  const int t = blockIdx.x * kWarpsPerBlock + threadIdx.x / kWarp;
  if (t >= T) return;  // warp-uniform
  float* lt = logits + (size_t)t * E;
  float v[PL], p[PL];
  float m = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + kWarp * i;
    if (e < E && partial != nullptr) {
      // the logits GEMM left K slices: add them in slice order, then the bias
      float s = 0.f;
      for (int z = 0; z < slices; ++z) s += __ldg(partial + ((size_t)z * T + t) * E + e);
      if (bias != nullptr) s += __ldg(bias + e);
      lt[e] = s;
      v[i] = s;
    } else {
      v[i] = e < E ? lt[e] : -INFINITY;
    }
    m = fmaxf(m, v[i]);
  }
  float* pt = probs + (size_t)t * E;
  if (sigmoid) {
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + kWarp * i;
      p[i] = e < E ? 1.0f / (1.0f + expf(-v[i])) : 0.f;
      if (e < E) pt[e] = p[i];
    }
  } else {
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + kWarp * i;
      p[i] = e < E ? expf(v[i] - m) : 0.f;
      s += p[i];
    }
    s = warp_sum(s);
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + kWarp * i;
      p[i] = p[i] / s;
      if (e < E) pt[e] = p[i];
    }
  }
  float sel_sum = 0.f;  // sum of the selected scores, in selection order (same in every lane)
  unsigned taken = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY, bp = 0.f;
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + kWarp * i;
      const bool free_ = e < E && !((taken >> i) & 1u);
      if (free_ && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i]; bi = e; bp = p[i];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const float op = __shfl_xor_sync(0xffffffffu, bp, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; bp = op; }
    }
    if (bi != INT_MAX && lane == (bi % kWarp)) taken |= 1u << (bi / kWarp);
    sel_sum += bp;
    if (lane == 0) {
      topk_idx[(size_t)t * k + j] = bi == INT_MAX ? -1 : bi;
      topk_w[(size_t)t * k + j] = bp;
    }
  }
  if (renorm) {
    __syncwarp();  // lane 0's weights above are visible to the whole warp
    float* wt = topk_w + (size_t)t * k;
    for (int j = lane; j < k; j += kWarp) wt[j] = wt[j] / sel_sum;
  }
}

// Gradient of the scores: g[t,e] = d_w[t,j] at e = idx[t,j] (0 elsewhere); with renorm
// (w_j = p_j / S, S = sum of the selected scores) g_j = (d_w[t,j] - sum_i d_w[t,i] w_i) / S.
// Softmax: d_logits = p * (g - s_t), s_t = sum_j p[idx_j] g_j -- pass 1 writes p*(0 - s)
// everywhere and pass 2 overwrites the k selected entries.  Sigmoid: d_logits = p(1-p) g, zero
// off the selection.
__global__ void __launch_bounds__(kWarpsPerBlock * kWarp) route_dlogits_kernel(
    const float* __restrict__ probs, const int* __restrict__ topk_idx,
    const float* __restrict__ d_w, int T, int E, int k, bool sigmoid, bool renorm,
    float* __restrict__ d_logits, __nv_bfloat16* __restrict__ dl_planes, int* status) {
  const int lane = threadIdx.x % kWarp;
  const int t = blockIdx.x * kWarpsPerBlock + threadIdx.x / kWarp;
  if (t >= T) return;
  const float* pt = probs + (size_t)t * E;
  const int* it = topk_idx + (size_t)t * k;
  const float* dwt = d_w + (size_t)t * k;
  float S = 1.f, dwm = 0.f;
  if (renorm) {
    float a = 0.f, b = 0.f;
    for (int j = lane; j < k; j += kWarp) {
      const int e = __ldg(it + j);
      if ((unsigned)e < (unsigned)E) {
        const float pe = __ldg(pt + e);
        a += pe;
        b = fmaf(__ldg(dwt + j), pe, b);
      }
    }
    S = warp_sum(a);
    dwm = warp_sum(b) / S;  // sum_i d_w_i w_i
  }
  float s = 0.f;
  if (!sigmoid) {
    for (int j = lane; j < k; j += kWarp) {
      const int e = __ldg(it + j);
      if ((unsigned)e < (unsigned)E) {
        const float g = renorm ? (__ldg(dwt + j) - dwm) / S : __ldg(dwt + j);
        s = fmaf(__ldg(pt + e), g, s);
      }
    }
    s = warp_sum(s);
  }
  float* dl = d_logits + (size_t)t * E;
  for (int e = lane; e < E; e += kWarp) dl[e] = sigmoid ? 0.f : __ldg(pt + e) * (0.f - s);
  __syncwarp();
  for (int j = lane; j < k; j += kWarp) {
    const int e = __ldg(it + j);
    if ((unsigned)e >= (unsigned)E) {
      flag_status(status, MOE_STATUS_BAD_INDEX);
      continue;
    }
    const float g = renorm ? (__ldg(dwt + j) - dwm) / S : __ldg(dwt + j);
    const float pe = __ldg(pt + e);
    dl[e] = sigmoid ? pe * (1.f - pe) * g : pe * (g - s);
  }
  if (dl_planes != nullptr) {  // the row is final: its three bf16 planes ([3][T][E])
    __syncwarp();
    const size_t n = (size_t)T * E;
    for (int e = lane; e < E; e += kWarp) {
      const size_t o = (size_t)t * E + e;
      split3_value(dl[e], dl_planes + o, dl_planes + n + o, dl_planes + 2 * n + o);
    }
  }
}

}  // namespace

void launch_softmax_topk(float* logits, const float* partial, int slices, const float* bias, int T, int E,
                         int k, bool sigmoid, bool renorm, float* probs, int* topk_idx, float* topk_w,
                         cudaStream_t st) {
  const int grid = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int block = kWarpsPerBlock * kWarp;
#define MOE_TOPK(PLV)                                                                                     \
  softmax_topk_kernel<PLV><<<grid, block, 0, st>>>(logits, partial, slices, bias, T, E, k, sigmoid, renorm, \
                                                   probs, topk_idx, topk_w)
  if (E <= 32) MOE_TOPK(1);
  else if (E <= 64) MOE_TOPK(2);
  else if (E <= 128) MOE_TOPK(4);
  else if (E <= 256) MOE_TOPK(8);
  else if (E <= 512) MOE_TOPK(16);
  else MOE_TOPK(32);
#undef MOE_TOPK
  count_launch(st);
}

void launch_route_dlogits(const float* probs, const int* topk_idx, const float* d_topk_w, int T,
                          int E, int k, bool sigmoid, bool renorm, float* d_logits, void* dl_planes,
                          int* status, cudaStream_t st) {
  const int grid = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  route_dlogits_kernel<<<grid, kWarpsPerBlock * kWarp, 0, st>>>(
      probs, topk_idx, d_topk_w, T, E, k, sigmoid, renorm, d_logits, static_cast<__nv_bfloat16*>(dl_planes), status);
  count_launch(st);
}

}  // namespace moe
