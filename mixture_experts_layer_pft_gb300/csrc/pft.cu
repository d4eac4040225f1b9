// PFT build: sort the flattened (token, expert) pairs by the key (expert, token).
//
// Flattened entry i = t*k + j carries expert e_i = topk_idx[t][j].  For a fixed expert the
// entries are distinct tokens, so ascending i is ascending t and a STABLE counting sort on e
// gives the unique (expert, token) order.  The entries are cut into G contiguous ranges, one per
// CTA, and three launches sort them with no spin-waits (two when G <= 64: the count kernel's last
// CTA does the scan):
//   1. pft_count: each CTA counts its range per expert (shared-memory atomic adds, eight loads in
//      flight per thread) and writes one column of the expert-major table hist[e][c].
//   2. pft_scan: one CTA per expert turns its row of the table into the exclusive prefix over
//      the ranges (the expert's rows that earlier ranges hold) and writes the expert's total to
//      num_ids; the last CTA to finish (a ticket from an atomic counter in the workspace header)
//      scans num_ids into offsets and resets the counter for the next call.
//   3. pft_scatter: each CTA walks its range in tiles of 2048 entries.  A warp owns 256
//      consecutive entries of a tile; per-warp counts in shared memory, and the lanes that share an
//      expert in each round of 32 (ballots over the bits of the id), give every entry its rank
//      among the same expert's entries of the tile, in index order.  slot_of is written in index order; token_ids and expert_ids go through a
//      tile-local sorted copy in shared memory and are written as runs of consecutive rows per
//      expert, so the scattered writes coalesce.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kPBlock = 512;                 // threads of the count CTAs
constexpr int kSBlock = 256;                 // threads of the scatter CTAs
constexpr int kPWarps = kSBlock / kWarp;     // 8 warps per scatter CTA
constexpr int kTile = 2048;                  // entries of one scatter tile
constexpr int kPerWarp = kTile / kPWarps;    // 256 consecutive entries per warp
constexpr int kRounds = kPerWarp / kWarp;    // 8 rounds of 32
constexpr int kMaxRanges = 608;              // 4 CTAs on each of 152 SMs (fixed: sizes the workspace)
constexpr int kScanBlock = 256;

// ---------------------------------------------------------------------------- 1. count
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total);
__device__ void scan_ranges_and_experts(int* hist, int G, int E, int* num_ids, int* offsets, int* warp_tot);

// With fused_scan (few ranges) the last CTA to finish (a ticket from the workspace header's
// counter) also does pft_scan's work, so that small builds take two launches.
__global__ void __launch_bounds__(kPBlock) pft_count_kernel(const int* __restrict__ idx, long long Tk, int E,
                                                            long long range, int G, int* __restrict__ hist,
                                                            WsHeader* hdr, bool fused_scan, int* __restrict__ num_ids,
                                                            int* __restrict__ offsets) {
  extern __shared__ int cnt[];  // [E]
  __shared__ int warp_tot[kPBlock / kWarp];
  __shared__ int is_last;
  int* status = &hdr->status;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const long long beg = (long long)blockIdx.x * range;
  const long long end = min(beg + range, Tk);
  bool bad = false;
  // eight loads in flight per thread (coalesced across the block), then the shared-memory adds
  constexpr int U = 8;
  for (long long i0 = beg + threadIdx.x; i0 < end; i0 += (long long)U * blockDim.x) {
    int ev[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = i0 + (long long)u * blockDim.x;
      ev[u] = i < end ? __ldg(idx + i) : -1;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = i0 + (long long)u * blockDim.x;
      if (i < end) {
        if ((unsigned)ev[u] < (unsigned)E) atomicAdd(&cnt[ev[u]], 1);
        else bad = true;
      }
    }
  }
  if (bad) flag_status(status, MOE_STATUS_BAD_INDEX);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)e * G + blockIdx.x] = cnt[e];
  if (!fused_scan) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&hdr->pft_done, 1u) == (unsigned)(G - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  scan_ranges_and_experts(hist, G, E, num_ids, offsets, warp_tot);
  if (threadIdx.x == 0) hdr->pft_done = 0u;
}

// ---------------------------------------------------------------------------- 2. scan
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
  int incl = v;
#pragma unroll
  for (int o = 1; o < kWarp; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == kWarp - 1) warp_tot[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
  for (int w = 0; w < (int)(blockDim.x / kWarp); ++w) {
    const int t = warp_tot[w];
    if (w < warp) before += t;
    all += t;
  }
  __syncthreads();
  *total = all;
  return before + incl - v;
}

// One CTA: each expert's row of the table turned into its exclusive prefix over the ranges (a
// thread per expert walks its G <= 64 entries), the totals into num_ids, their scan into offsets.
__device__ void scan_ranges_and_experts(int* hist, int G, int E, int* num_ids, int* offsets, int* warp_tot) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int* row = hist + (size_t)e * G;
    int run = 0;
    for (int c = 0; c < G; ++c) {
      const int v = __ldcg(row + c);
      row[c] = run;
      run += v;
    }
    num_ids[e] = run;
  }
  __syncthreads();
  int carry = 0;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int q = e0 + threadIdx.x;
    const int v = q < E ? num_ids[q] : 0;
    int tot;
    const int ex = block_exclusive_scan(v, warp_tot, &tot);
    if (q < E) offsets[q] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) offsets[E] = carry;
}

__global__ void __launch_bounds__(kScanBlock) pft_scan_kernel(int* __restrict__ hist, int G, int E,
                                                              int* __restrict__ num_ids, int* __restrict__ offsets,
                                                              WsHeader* hdr) {
  __shared__ int warp_tot[kScanBlock / kWarp];
  __shared__ int is_last;
  const int e = blockIdx.x;
  int* row = hist + (size_t)e * G;
  int run = 0;
  for (int c0 = 0; c0 < G; c0 += kScanBlock) {
    const int c = c0 + threadIdx.x;
    const int v = c < G ? __ldcg(row + c) : 0;
    int tot;
    const int ex = block_exclusive_scan(v, warp_tot, &tot);
    if (c < G) row[c] = run + ex;
    run += tot;
  }
  if (threadIdx.x == 0) num_ids[e] = run;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&hdr->pft_done, 1u) == (unsigned)(E - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // the last CTA: offsets = exclusive scan of num_ids (E <= 1024: four per thread)
  int carry = 0;
  for (int e0 = 0; e0 < E; e0 += kScanBlock) {
    const int q = e0 + threadIdx.x;
    const int v = q < E ? __ldcg(num_ids + q) : 0;
    int tot;
    const int ex = block_exclusive_scan(v, warp_tot, &tot);
    if (q < E) offsets[q] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    offsets[E] = carry;
    hdr->pft_done = 0u;
  }
}

// ---------------------------------------------------------------------------- 3. scatter
// Lanes of the warp holding the same expert id as this lane: the AND over the id's NB bits of
// the ballot of that bit (or of its complement), restricted to lanes with a valid id (NB bits
// cover every id below E).  Lanes with e < 0 get an unused mask.
template <int NB>
__device__ __forceinline__ unsigned same_expert_lanes(int e) {
  unsigned m = __ballot_sync(0xffffffffu, e >= 0);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const bool bit = ((e >> b) & 1) != 0;
    const unsigned bb = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bb : ~bb;
  }
  return m;
}

constexpr int kWStride = kPWarps + 1;  // per-expert row of the per-warp count table (padded)

// Shared memory: base[E] (next global row of each expert for this CTA), wcnt[E][kWStride]
// (per-warp counts, then each warp's start inside the tile's bucket), delta[E] (global row minus
// position in the tile's sorted copy), tcnt[E], stok[kTile], sexp[kTile] (uint16).
template <int NB>
__global__ void __launch_bounds__(kSBlock, 4) pft_scatter_kernel(const int* __restrict__ idx, int Tk, int k, int E,
                                                                 int range, int G, const int* __restrict__ hist,
                                                                 const int* __restrict__ offsets,
                                                                 int* __restrict__ token_ids,
                                                                 int* __restrict__ expert_ids,
                                                                 int* __restrict__ slot_of) {
  extern __shared__ int sm[];
  int* base = sm;
  int* wcnt = base + E;
  int* delta = wcnt + kWStride * E;
  int* tcnt = delta + E;
  int* stok = tcnt + E;
  unsigned short* sexp = reinterpret_cast<unsigned short*>(stok + kTile);
  __shared__ int warp_tot[kPWarps];
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    base[e] = __ldg(offsets + e) + __ldcg(hist + (size_t)e * G + blockIdx.x);
  __syncthreads();
  const int beg = blockIdx.x * range;
  const int end = min(beg + range, Tk);
  const int dt = kWarp / k, dj = kWarp % k;
  // this warp's 256 consecutive entries of a tile, 8 per lane in rounds of 32 (the next tile's
  // ids are loaded while the current one is written out)
  int nx[kRounds];
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int i = beg + warp * kPerWarp + r * kWarp + lane;
    nx[r] = i < end ? __ldg(idx + i) : -1;
  }
  for (int t0 = beg; t0 < end; t0 += kTile) {
    // (a) per-warp counts of the tile
    for (int q = threadIdx.x; q < kWStride * E; q += blockDim.x) wcnt[q] = 0;
    const int w0 = t0 + warp * kPerWarp;
    int ev[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int i = w0 + r * kWarp + lane;
      int e = nx[r];
      if (i < end && (unsigned)e >= (unsigned)E) {
        slot_of[i] = -1;  // reported by pft_count
        e = -1;
      }
      ev[r] = i < end ? e : -1;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRounds; ++r)
      if (ev[r] >= 0) atomicAdd(&wcnt[ev[r] * kWStride + warp], 1);
    __syncthreads();
    // (b) per expert: each warp's start inside the tile's bucket, the bucket size
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int* row = wcnt + e * kWStride;
      int run = 0;
#pragma unroll
      for (int w = 0; w < kPWarps; ++w) {
        const int c = row[w];
        row[w] = run;
        run += c;
      }
      tcnt[e] = run;
    }
    __syncthreads();
    // bucket starts of the tile's sorted copy: exclusive scan of tcnt over the experts
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += kSBlock) {
      const int q = e0 + threadIdx.x;
      const int v = q < E ? tcnt[q] : 0;
      int tot;
      const int ex = block_exclusive_scan(v, warp_tot, &tot);
      if (q < E) delta[q] = base[q] - (carry + ex);
      carry += tot;
    }
    __syncthreads();
    // (c) ranks in index order: slot_of directly, token and expert into the sorted copy.  The
    // token of entry i = w0 + 32 r + lane is t = i / k, stepped from round to round.
    int t_cur = (w0 + lane) / k, j_cur = (w0 + lane) % k;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int e = ev[r];
      const unsigned peers = same_expert_lanes<NB>(e);
      const unsigned below = peers & lt_mask;
      int pos = 0;
      if (e >= 0) pos = wcnt[e * kWStride + warp] + __popc(below);
      __syncwarp();
      if (e >= 0 && below == 0u) wcnt[e * kWStride + warp] = pos + __popc(peers);  // the group's first lane
      __syncwarp();
      if (e >= 0) {
        const int row = base[e] + pos;
        slot_of[w0 + r * kWarp + lane] = row;
        const int q = row - delta[e];
        stok[q] = t_cur;
        sexp[q] = (unsigned short)e;
      }
      t_cur += dt;
      j_cur += dj;
      if (j_cur >= k) { j_cur -= k; ++t_cur; }
    }
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int i = w0 + kTile + r * kWarp + lane;
      nx[r] = i < end ? __ldg(idx + i) : -1;
    }
    __syncthreads();
    // (d) write the sorted copy: consecutive entries of one expert go to consecutive rows
    for (int q = threadIdx.x; q < carry; q += blockDim.x) {
      const int e = sexp[q];
      const int row = q + delta[e];
      if ((unsigned)row < (unsigned)Tk) {  // always true when the counts agree; guards the writes
        token_ids[row] = stok[q];
        expert_ids[row] = e;
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) base[e] += tcnt[e];
    __syncthreads();
  }
}

size_t scatter_smem(int E) {
  return (size_t)(E + kWStride * E + 2 * E + kTile) * sizeof(int) + (size_t)kTile * sizeof(unsigned short);
}

template <int NB>
void launch_scatter(const int* idx, int Tk, int k, int E, int range, int G, const int* hist, const int* offsets,
                    int* token_ids, int* expert_ids, int* slot_of, cudaStream_t st) {
  const size_t smem = scatter_smem(E);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(pft_scatter_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  pft_scatter_kernel<NB><<<G, kSBlock, smem, st>>>(idx, Tk, k, E, range, G, hist, offsets, token_ids, expert_ids,
                                                   slot_of);
}

}  // namespace

// Ranges (CTAs) for Tk entries: at least 1024 entries each, at most kMaxRanges of them.
int pft_num_chunks(long long Tk) {
  const long long g = (Tk + 1023) / 1024;
  return (int)(g < 1 ? 1 : (g > kMaxRanges ? kMaxRanges : g));
}

int pft_chunk_size(long long Tk) {
  const long long g = pft_num_chunks(Tk);
  return (int)((Tk + g - 1) / g);
}

size_t pft_scratch_bytes(long long Tk, int E) {
  return (size_t)pft_num_chunks(Tk) * (size_t)E * sizeof(int);
}

void launch_pft_build(const int* topk_idx, int T, int E, int k, int* num_ids, int* offsets,
                      int* token_ids, int* expert_ids, int* slot_of, void* ws, cudaStream_t st) {
  const long long Tk = (long long)T * k;
  const int G = pft_num_chunks(Tk);
  const long long range = pft_chunk_size(Tk);
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  int* hist = reinterpret_cast<int*>(static_cast<char*>(ws) + sizeof(WsHeader));
  const bool fused_scan = G <= 64;  // few ranges: the count kernel's last CTA scans them
  pft_count_kernel<<<G, kPBlock, (size_t)E * sizeof(int), st>>>(topk_idx, Tk, E, range, G, hist, hdr, fused_scan,
                                                                 num_ids, offsets);
  count_launch(st);
  if (!fused_scan) {
    pft_scan_kernel<<<E, kScanBlock, 0, st>>>(hist, G, E, num_ids, offsets, hdr);
    count_launch(st);
  }
  // bits that hold every id below E (at most 10: E <= 1024)
  const int Tk32 = (int)Tk, range32 = (int)range;
  if (E <= 64) launch_scatter<6>(topk_idx, Tk32, k, E, range32, G, hist, offsets, token_ids, expert_ids, slot_of, st);
  else if (E <= 128) launch_scatter<7>(topk_idx, Tk32, k, E, range32, G, hist, offsets, token_ids, expert_ids, slot_of, st);
  else if (E <= 256) launch_scatter<8>(topk_idx, Tk32, k, E, range32, G, hist, offsets, token_ids, expert_ids, slot_of, st);
  else if (E <= 512) launch_scatter<9>(topk_idx, Tk32, k, E, range32, G, hist, offsets, token_ids, expert_ids, slot_of, st);
  else launch_scatter<10>(topk_idx, Tk32, k, E, range32, G, hist, offsets, token_ids, expert_ids, slot_of, st);
  count_launch(st);
}

}  // namespace moe
