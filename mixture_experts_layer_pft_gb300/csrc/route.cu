// Gating: softmax over E experts and top-k selection, one warp per token; and the gate's
// backward through the softmax Jacobian.  The router GEMMs (x·W_g, x^T·d_logits,
// d_logits·W_g^T) run on the SIMT GEMM engine in fp32.
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
template <int PL>
__global__ void __launch_bounds__(kWarpsPerBlock * kWarp) softmax_topk_kernel(
    const float* __restrict__ logits, int T, int E, int k, float* __restrict__ probs,
    int* __restrict__ topk_idx, float* __restrict__ topk_w) {
  const int lane = threadIdx.x % kWarp;
  const int t = blockIdx.x * kWarpsPerBlock + threadIdx.x / kWarp;
  if (t >= T) return;  // warp-uniform
  const float* lt = logits + (size_t)t * E;
  float v[PL], p[PL];
  float m = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + kWarp * i;
    v[i] = e < E ? __ldg(lt + e) : -INFINITY;
    m = fmaxf(m, v[i]);
  }
  m = warp_max(m);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + kWarp * i;
    p[i] = e < E ? expf(v[i] - m) : 0.f;
    s += p[i];
  }
  s = warp_sum(s);
  float* pt = probs + (size_t)t * E;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + kWarp * i;
    p[i] = p[i] / s;
    if (e < E) pt[e] = p[i];
  }
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
    if (lane == 0) {
      topk_idx[(size_t)t * k + j] = bi == INT_MAX ? -1 : bi;
      topk_w[(size_t)t * k + j] = bp;
    }
  }
}

// d_logits[t,e] = p[t,e] * (g[t,e] - s_t),  s_t = sum_j p[t,idx[t,j]] * d_w[t,j],
// g[t,e] = d_w[t,j] at e = idx[t,j] (0 elsewhere).  Pass 1 writes p*(0 - s) everywhere;
// pass 2 overwrites the k selected entries.
__global__ void __launch_bounds__(kWarpsPerBlock * kWarp) route_dlogits_kernel(
    const float* __restrict__ probs, const int* __restrict__ topk_idx,
    const float* __restrict__ d_w, int T, int E, int k, float* __restrict__ d_logits,
    int* status) {
  const int lane = threadIdx.x % kWarp;
  const int t = blockIdx.x * kWarpsPerBlock + threadIdx.x / kWarp;
  if (t >= T) return;
  const float* pt = probs + (size_t)t * E;
  float s = 0.f;
  for (int j = lane; j < k; j += kWarp) {
    const int e = __ldg(topk_idx + (size_t)t * k + j);
    if ((unsigned)e < (unsigned)E) s = fmaf(__ldg(pt + e), __ldg(d_w + (size_t)t * k + j), s);
  }
  s = warp_sum(s);
  float* dl = d_logits + (size_t)t * E;
  for (int e = lane; e < E; e += kWarp) dl[e] = __ldg(pt + e) * (0.f - s);
  __syncwarp();
  for (int j = lane; j < k; j += kWarp) {
    const int e = __ldg(topk_idx + (size_t)t * k + j);
    if ((unsigned)e >= (unsigned)E) {
      flag_status(status, MOE_STATUS_BAD_INDEX);
      continue;
    }
    dl[e] = __ldg(pt + e) * (__ldg(d_w + (size_t)t * k + j) - s);
  }
}

}  // namespace

void launch_softmax_topk(const float* logits, int T, int E, int k, float* probs, int* topk_idx,
                         float* topk_w, cudaStream_t st) {
  const int grid = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int block = kWarpsPerBlock * kWarp;
  if (E <= 32) softmax_topk_kernel<1><<<grid, block, 0, st>>>(logits, T, E, k, probs, topk_idx, topk_w);
  else if (E <= 64) softmax_topk_kernel<2><<<grid, block, 0, st>>>(logits, T, E, k, probs, topk_idx, topk_w);
  else if (E <= 128) softmax_topk_kernel<4><<<grid, block, 0, st>>>(logits, T, E, k, probs, topk_idx, topk_w);
  else if (E <= 256) softmax_topk_kernel<8><<<grid, block, 0, st>>>(logits, T, E, k, probs, topk_idx, topk_w);
  else if (E <= 512) softmax_topk_kernel<16><<<grid, block, 0, st>>>(logits, T, E, k, probs, topk_idx, topk_w);
  else softmax_topk_kernel<32><<<grid, block, 0, st>>>(logits, T, E, k, probs, topk_idx, topk_w);
  count_launch(st);
}

void launch_route_dlogits(const float* probs, const int* topk_idx, const float* d_topk_w, int T,
                          int E, int k, float* d_logits, int* status, cudaStream_t st) {
  const int grid = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  route_dlogits_kernel<<<grid, kWarpsPerBlock * kWarp, 0, st>>>(probs, topk_idx, d_topk_w, T, E,
                                                                 k, d_logits, status);
  count_launch(st);
}

}  // namespace moe
