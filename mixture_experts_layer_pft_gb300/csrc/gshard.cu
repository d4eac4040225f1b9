// The capacity-buffer (GShard-style) MoE data path that the padding-free buffers replace: the
// comparison system of the X-MoE review (§3 "Core formulas": O(E x C x H) padded dispatch against
// O(B x H); §5 ablation "PFT effect": gating, dispatch and combine timed against it).
//
//   gate      dispatch_mask [T,E,C] (0/1 in the activation type) and combine_weights [T,E,C] fp32
//             from the top-k selection: token t's slot in expert e is the number of earlier
//             tokens that chose e; a slot at or beyond the capacity C is dropped.  The masks are
//             zero-filled (the T*E*C write that the padded format costs), then the T*k ones set.
//   dispatch  xe[e,c,:] = sum_t dispatch_mask[t,e,c] x[t,:], the contraction over the tokens,
//             evaluated column by column: one thread per padded row (e, c) reads the mask down
//             the tokens (T*E*C reads, coalesced across c) and copies the row it selects, or
//             writes zeros for a padding row.
//   combine   y[t,:] = sum_{e,c} combine_weights[t,e,c] ye[e,c,:]: one CTA per token reads its
//             E*C weights (coalesced), lists the non-zero ones in (e, c) order and sums those
//             rows in fp32, rounded once.
// The experts run on all E*C padded rows through the grouped GEMMs with offsets e*C.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kGBlock = 256;
constexpr int kMaxList = 256;  // non-zero combine weights one token may carry

// ---------------------------------------------------------------------------- gate
// One CTA per expert walks the tokens in tiles of 256: a token that chose e gets the running
// count of earlier such tokens as its slot (block-wide exclusive scan of the choice flags).
__global__ void __launch_bounds__(kGBlock) gshard_slots_kernel(const int* __restrict__ idx, int T, int k, int E,
                                                               int* __restrict__ slot, int* __restrict__ loads) {
  __shared__ int warp_cnt[kGBlock / kWarp];
  __shared__ int s_base;
  const int e = blockIdx.x;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  if (threadIdx.x == 0) s_base = 0;
  __syncthreads();
  for (int t0 = 0; t0 < T; t0 += kGBlock) {
    const int t = t0 + threadIdx.x;
    int jsel = -1;
    if (t < T) {
      for (int j = 0; j < k; ++j)
        if (__ldg(idx + (size_t)t * k + j) == e) { jsel = j; break; }
    }
    const unsigned b = __ballot_sync(0xffffffffu, jsel >= 0);
    if (lane == 0) warp_cnt[warp] = __popc(b);
    __syncthreads();
    int before = s_base;
    for (int w = 0; w < warp; ++w) before += warp_cnt[w];
    if (jsel >= 0) slot[(size_t)t * k + jsel] = before + __popc(b & ((1u << lane) - 1u));
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int w = 0; w < kGBlock / kWarp; ++w) tot += warp_cnt[w];
      s_base += tot;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) loads[e] = s_base;
}

template <typename T_>
__global__ void __launch_bounds__(kGBlock) gshard_fill_kernel(const int* __restrict__ idx, const float* __restrict__ w,
                                                              const int* __restrict__ slot, long long Tk, int k,
                                                              int E, int C, T_* __restrict__ mask,
                                                              float* __restrict__ cw, int* status) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= Tk) return;
  const int e = __ldg(idx + i);
  if ((unsigned)e >= (unsigned)E) {
    flag_status(status, MOE_STATUS_BAD_INDEX);
    return;
  }
  const int c = __ldg(slot + i);
  if (c < 0) {  // no slot: the token lists expert e more than once
    flag_status(status, MOE_STATUS_BAD_INDEX);
    return;
  }
  if (c >= C) return;  // over capacity: dropped
  const size_t q = ((size_t)(i / k) * E + e) * (size_t)C + c;
  mask[q] = from_f<T_>(1.0f);
  cw[q] = __ldg(w + i);
}

// ---------------------------------------------------------------------------- dispatch
// CTA (e, c-block): thread c scans mask[t, e, c] over t (unrolled loads keep several in
// flight), then the CTA writes its rows xe[e, c, :] = mask * x[t_c, :] (zeros when no token).
template <typename T_>
__global__ void __launch_bounds__(kGBlock) gshard_dispatch_kernel(const T_* __restrict__ x,
                                                                  const T_* __restrict__ mask, int T, int E, int C,
                                                                  int nvec, T_* __restrict__ xe, int* status) {
  __shared__ int s_tok[kGBlock];
  __shared__ float s_val[kGBlock];
  const int cblocks = (C + kGBlock - 1) / kGBlock;
  const int e = blockIdx.x / cblocks;
  const int c0 = (blockIdx.x % cblocks) * kGBlock;
  const int c = c0 + threadIdx.x;
  int tok = -1;
  float val = 0.f;
  if (c < C) {
    const size_t stride = (size_t)E * C;
    const T_* col = mask + (size_t)e * C + c;
    constexpr int U = 8;
    int t = 0;
    for (; t + U <= T; t += U) {
      float m[U];
#pragma unroll
      for (int u = 0; u < U; ++u) m[u] = to_f(col[(size_t)(t + u) * stride]);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (m[u] != 0.f) {
          if (tok < 0) { tok = t + u; val = m[u]; }
          else flag_status(status, MOE_STATUS_BAD_INDEX);  // not one token per padded row
        }
    }
    for (; t < T; ++t) {
      const float m = to_f(col[(size_t)t * stride]);
      if (m != 0.f) {
        if (tok < 0) { tok = t; val = m; }
        else flag_status(status, MOE_STATUS_BAD_INDEX);
      }
    }
  }
  s_tok[threadIdx.x] = tok;
  s_val[threadIdx.x] = val;
  __syncthreads();
  const int rows = min(kGBlock, C - c0);
  const uint4* xs = reinterpret_cast<const uint4*>(x);
  uint4* dst = reinterpret_cast<uint4*>(xe) + ((size_t)e * C + c0) * nvec;
  for (long long q = threadIdx.x; q < (long long)rows * nvec; q += blockDim.x) {
    const int r = (int)(q / nvec), v = (int)(q % nvec);
    const int tr = s_tok[r];
    uint4 out = make_uint4(0, 0, 0, 0);
    if (tr >= 0) {
      const uint4 in = __ldg(xs + (size_t)tr * nvec + v);
      const float m = s_val[r];
      if (m == 1.0f) {
        out = in;
      } else {
        float f[Vec<T_>::N];
        unpack(in, f, T_{});
#pragma unroll
        for (int i = 0; i < Vec<T_>::N; ++i) f[i] *= m;
        out = pack(f, T_{});
      }
    }
    dst[(size_t)r * nvec + v] = out;
  }
}

// ---------------------------------------------------------------------------- combine
// CTA per token: list the non-zero combine weights of the token's E*C row in (e, c) order,
// then sum those rows of ye in fp32 in that order, rounding once.
template <typename T_>
__global__ void __launch_bounds__(kGBlock) gshard_combine_kernel(const float* __restrict__ cw,
                                                                 const T_* __restrict__ ye, int E, int C,
                                                                 int nvec, T_* __restrict__ y, int* status) {
  constexpr int VN = Vec<T_>::N;
  __shared__ int s_row[kMaxList];
  __shared__ float s_w[kMaxList];
  __shared__ int warp_cnt[kGBlock / kWarp];
  __shared__ int s_n;
  const int t = blockIdx.x;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const long long EC = (long long)E * C;
  const float* row = cw + (size_t)t * EC;
  if (threadIdx.x == 0) s_n = 0;
  __syncthreads();
  for (long long q0 = 0; q0 < EC; q0 += kGBlock) {
    const long long q = q0 + threadIdx.x;
    const float v = q < EC ? __ldg(row + q) : 0.f;
    const bool nz = v != 0.f;
    const unsigned b = __ballot_sync(0xffffffffu, nz);
    if (lane == 0) warp_cnt[warp] = __popc(b);
    __syncthreads();
    int pos = s_n;
    for (int w = 0; w < warp; ++w) pos += warp_cnt[w];
    pos += __popc(b & ((1u << lane) - 1u));
    if (nz) {
      if (pos < kMaxList) { s_row[pos] = (int)q; s_w[pos] = v; }
      else flag_status(status, MOE_STATUS_BAD_INDEX);  // more terms than the list holds
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int w = 0; w < kGBlock / kWarp; ++w) tot += warp_cnt[w];
      s_n += tot;
    }
    __syncthreads();
  }
  const int n = min(s_n, kMaxList);
  const uint4* yb = reinterpret_cast<const uint4*>(ye);
  uint4* dst = reinterpret_cast<uint4*>(y) + (size_t)t * nvec;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    float acc[VN];
#pragma unroll
    for (int i = 0; i < VN; ++i) acc[i] = 0.f;
    for (int l = 0; l < n; ++l) {
      float f[VN];
      unpack(__ldg(yb + (size_t)s_row[l] * nvec + v), f, T_{});
      const float wl = s_w[l];
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] = fmaf(wl, f[i], acc[i]);
    }
    dst[v] = pack(acc, T_{});
  }
}

}  // namespace

void launch_gshard_gate(int dtype, const int* idx, const float* w, int T, int E, int k, int C, void* mask,
                        float* cw, int* loads, int* slot, int* status, cudaStream_t st) {
  const size_t cells = (size_t)T * E * C;
  cudaMemsetAsync(mask, 0, cells * (dtype == MOE_BF16 ? 2 : 4), st);
  cudaMemsetAsync(cw, 0, cells * sizeof(float), st);
  cudaMemsetAsync(slot, 0xFF, (size_t)T * k * sizeof(int), st);  // -1: no slot
  gshard_slots_kernel<<<E, kGBlock, 0, st>>>(idx, T, k, E, slot, loads);
  count_launch(st);
  const long long Tk = (long long)T * k;
  const int blocks = (int)((Tk + kGBlock - 1) / kGBlock);
  if (dtype == MOE_BF16)
    gshard_fill_kernel<__nv_bfloat16><<<blocks, kGBlock, 0, st>>>(idx, w, slot, Tk, k, E, C,
                                                                   static_cast<__nv_bfloat16*>(mask), cw, status);
  else
    gshard_fill_kernel<float><<<blocks, kGBlock, 0, st>>>(idx, w, slot, Tk, k, E, C, static_cast<float*>(mask), cw,
                                                          status);
  count_launch(st);
}

void launch_gshard_dispatch(int dtype, const void* x, const void* mask, int T, int E, int C, int h, void* xe,
                            int* status, cudaStream_t st) {
  const int cblocks = (C + kGBlock - 1) / kGBlock;
  const int grid = E * cblocks;
  if (dtype == MOE_BF16)
    gshard_dispatch_kernel<__nv_bfloat16><<<grid, kGBlock, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(mask), T, E, C, h / 8,
        static_cast<__nv_bfloat16*>(xe), status);
  else
    gshard_dispatch_kernel<float><<<grid, kGBlock, 0, st>>>(static_cast<const float*>(x),
                                                            static_cast<const float*>(mask), T, E, C, h / 4,
                                                            static_cast<float*>(xe), status);
  count_launch(st);
}

void launch_gshard_combine(int dtype, const float* cw, const void* ye, int T, int E, int C, int h, void* y,
                           int* status, cudaStream_t st) {
  if (dtype == MOE_BF16)
    gshard_combine_kernel<__nv_bfloat16><<<T, kGBlock, 0, st>>>(cw, static_cast<const __nv_bfloat16*>(ye), E, C,
                                                                 h / 8, static_cast<__nv_bfloat16*>(y), status);
  else
    gshard_combine_kernel<float><<<T, kGBlock, 0, st>>>(cw, static_cast<const float*>(ye), E, C, h / 4,
                                                        static_cast<float*>(y), status);
  count_launch(st);
}

}  // namespace moe
