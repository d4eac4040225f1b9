// PFT build: sort the flattened (token, expert) pairs by the key (expert, token).
//
// Flattened entry i = t*k + j carries expert e_i = topk_idx[t][j].  For a fixed expert the
// entries are distinct tokens, so ascending i is ascending t and a STABLE counting sort on e
// gives the unique (expert, token) order.  Two launches, no spin-waits:
//   1. pft_hist: each CTA counts its chunk of entries per expert (shared-memory atomics) and
//      writes the chunk's histogram row.  The last CTA to finish (a ticket from an atomic
//      counter in the workspace header) sums the rows into num_ids, scans them into
//      offsets, turns every histogram entry into that chunk's base position for the expert,
//      and resets the counter for the next call.
//   2. pft_scatter: each CTA walks its chunk again in rounds of one entry per thread.  Inside
//      a warp, __match_any_sync groups the lanes with the same expert; a lane's rank is the
//      number of matching lanes below it.  Per-warp counts in shared memory give the rank
//      offset contributed by earlier warps of the round.  The position is
//      base[e] + earlier warps + rank; token_ids, expert_ids and slot_of are written there.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kHistBlock = 256;
constexpr int kScatBlock = 512;
constexpr int kScatWarps = kScatBlock / kWarp;
constexpr int kMaxE = 1024;

__global__ void __launch_bounds__(kHistBlock) pft_hist_kernel(
    const int* __restrict__ idx, long long Tk, int E, int chunk, int nchunks,
    int* __restrict__ hist, int* __restrict__ num_ids, int* __restrict__ offsets, WsHeader* hdr) {
  __shared__ int cnt[kMaxE];
  __shared__ int is_last;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const long long beg = (long long)blockIdx.x * chunk;
  const long long end = min(beg + chunk, Tk);
  bool bad = false;
  for (long long i = beg + threadIdx.x; i < end; i += blockDim.x) {
    const int e = __ldg(idx + i);
    if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);
    else bad = true;
  }
  if (bad) flag_status(&hdr->status, MOE_STATUS_BAD_INDEX);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = cnt[e];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&hdr->pft_done, 1u) == (unsigned)(nchunks - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // totals per expert (thread e walks the chunk rows; reads bypass L1)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int tot = 0;
    for (int c = 0; c < nchunks; ++c) tot += __ldcg(hist + (size_t)c * E + e);
    cnt[e] = tot;
    num_ids[e] = tot;
  }
  __syncthreads();
  // exclusive scan of cnt[0..E) by warp 0 (E <= 1024: 32 entries per lane)
  if (threadIdx.x < kWarp) {
    const int lane = threadIdx.x;
    const int per = (E + kWarp - 1) / kWarp;
    const int b0 = lane * per, b1 = min(b0 + per, E);
    int local = 0;
    for (int e = b0; e < b1; ++e) local += cnt[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int run = incl - local;
    for (int e = b0; e < b1; ++e) {
      const int c = cnt[e];
      cnt[e] = run;  // now the exclusive offset
      offsets[e] = run;
      run += c;
    }
    if (lane == kWarp - 1) offsets[E] = incl;
  }
  __syncthreads();
  // histogram entry (c, e) -> base position of chunk c's entries for expert e
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = cnt[e];
    for (int c = 0; c < nchunks; ++c) {
      const size_t q = (size_t)c * E + e;
      const int h = __ldcg(hist + q);
      hist[q] = run;
      run += h;
    }
  }
  if (threadIdx.x == 0) hdr->pft_done = 0u;
}

__global__ void __launch_bounds__(kScatBlock) pft_scatter_kernel(
    const int* __restrict__ idx, long long Tk, int k, int E, int chunk,
    const int* __restrict__ base_g, int* __restrict__ token_ids, int* __restrict__ expert_ids,
    int* __restrict__ slot_of) {
  extern __shared__ int sm[];
  int* base = sm;               // [E]
  int* wcnt = sm + E;           // [kScatWarps][E]
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  for (int e = threadIdx.x; e < E; e += blockDim.x) base[e] = __ldcg(base_g + (size_t)blockIdx.x * E + e);
  for (int q = threadIdx.x; q < kScatWarps * E; q += blockDim.x) wcnt[q] = 0;
  __syncthreads();
  const long long beg = (long long)blockIdx.x * chunk;
  const long long end = min(beg + chunk, Tk);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (long long r0 = beg; r0 < end; r0 += kScatBlock) {
    const long long i = r0 + threadIdx.x;
    int e = -1;
    if (i < end) {
      e = __ldg(idx + i);
      if ((unsigned)e >= (unsigned)E) {
        slot_of[i] = -1;  // flagged by pft_hist
        e = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    const bool leader = rank == 0;
    if (leader && e >= 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int pos = base[e] + rank;
      for (int w = 0; w < warp; ++w) pos += wcnt[w * E + e];
      token_ids[pos] = (int)(i / k);
      expert_ids[pos] = e;
      slot_of[i] = pos;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
      int add = 0;
      for (int w = 0; w < kScatWarps; ++w) add += wcnt[w * E + x];
      base[x] += add;
    }
    __syncthreads();
    if (leader && e >= 0) wcnt[warp * E + e] = 0;
    __syncwarp();
  }
}

}  // namespace

int pft_chunk_size(long long Tk) {
  // at least 1024 entries per CTA; larger chunks keep the grid near four waves of CTAs
  long long c = (Tk + 607) / 608;
  c = ((c + kScatBlock - 1) / kScatBlock) * kScatBlock;
  return (int)(c < 1024 ? 1024 : c);
}

int pft_num_chunks(long long Tk) {
  const long long c = pft_chunk_size(Tk);
  return (int)((Tk + c - 1) / c);
}

size_t pft_scratch_bytes(long long Tk, int E) {
  return (size_t)pft_num_chunks(Tk) * (size_t)E * sizeof(int);
}

void launch_pft_build(const int* topk_idx, int T, int E, int k, int* num_ids, int* offsets,
                      int* token_ids, int* expert_ids, int* slot_of, void* ws, cudaStream_t st) {
  const long long Tk = (long long)T * k;
  const int chunk = pft_chunk_size(Tk);
  const int nchunks = pft_num_chunks(Tk);
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  int* hist = reinterpret_cast<int*>(static_cast<char*>(ws) + sizeof(WsHeader));
  pft_hist_kernel<<<nchunks, kHistBlock, 0, st>>>(topk_idx, Tk, E, chunk, nchunks, hist, num_ids,
                                                  offsets, hdr);
  count_launch(st);
  const size_t smem = (size_t)(1 + kScatWarps) * E * sizeof(int);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(pft_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  pft_scatter_kernel<<<nchunks, kScatBlock, smem, st>>>(topk_idx, Tk, k, E, chunk, hist, token_ids,
                                                        expert_ids, slot_of);
  count_launch(st);
}

}  // namespace moe
