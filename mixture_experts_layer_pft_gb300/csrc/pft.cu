// PFT build: sort the flattened (token, expert) pairs by the key (expert, token).
//
// Flattened entry i = t*k + j carries expert e_i = topk_idx[t][j].  For a fixed expert the
// entries are distinct tokens, so ascending i is ascending t and a STABLE counting sort on e
// gives the unique (expert, token) order.  The tokens are cut into G contiguous ranges, one per
// CTA, and three launches sort them with no spin-waits:
//   1. pft_count: each CTA counts its range's entries per expert (16-byte loads, shared-memory
//      atomic adds) and writes one column of the expert-major table hist[e][c].
//   2. pft_scan: a warp per expert turns its row of the table into the exclusive prefix over
//      the ranges (the expert's rows that earlier ranges hold) and writes the expert's total to
//      num_ids.  Every scatter CTA scans num_ids into offsets for itself (CTA 0 writes them).
//      (A last-CTA ticket that let the count kernel do this scan cost more in fences and
//      barriers than the launch it saved.)
//   3. pft_scatter: each CTA walks its range in tiles of at most 512 tokens.  A tile sets one bit
//      per entry in a per-expert bitmap over its tokens (bit t of expert e: token t chose e).
//      Because a token's k experts are distinct, an entry's rank among its expert's entries of
//      the tile is the number of bits below its own: a popcount of its word plus the prefix of
//      the words before it, which one pass per expert computes (each word's cell then holds the
//      global row of its first entry).  slot_of is written in index order; token_ids goes through
//      a tile-sorted copy in shared memory, so consecutive lanes write consecutive rows of a
//      bucket; expert_ids depends on offsets alone and each CTA fills its share of it as plain
//      runs.  A repeated id inside a row (which the bitmap would merge) is reported as a bad
//      index.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kPBlock = 512;                 // threads of the count CTAs
constexpr int kSBlock = 256;                 // threads of the scatter CTAs
constexpr int kTileEntries = 4096;           // entries of one scatter tile at most
constexpr int kPerThread = kTileEntries / kSBlock;  // 16 entries a thread
constexpr int kBitWords = 4096;              // bitmap words of one tile at most (E x words per expert)
constexpr int kMaxRanges = 608;              // 4 CTAs on each of 152 SMs (fixed: sizes the workspace)
constexpr int kScanBlock = 256;

// ---------------------------------------------------------------------------- 1. count
__global__ void __launch_bounds__(kPBlock, 4) pft_count_kernel(const int* __restrict__ idx, long long Tk, int E,
                                                            long long range, int G, int* __restrict__ hist,
                                                            int* status) {
  extern __shared__ int cnt[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const long long beg = (long long)blockIdx.x * range;
  const long long end = min(beg + range, Tk);
  bool bad = false;
  auto add = [&](int e) {
    if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);
    else bad = true;
  };
  // a scalar head up to a 16-byte boundary, 16-byte loads (four in flight per thread), a tail
  const long long head = (long long)((4u - (unsigned)(((uintptr_t)(idx + beg) >> 2) & 3u)) & 3u);
  const long long a0 = min(end, beg + head);
  const long long nv = (end - a0) / 4;
  const long long a1 = a0 + 4 * nv;
  for (long long i = beg + threadIdx.x; i < a0; i += blockDim.x) add(__ldg(idx + i));
  const int4* v = reinterpret_cast<const int4*>(idx + a0);
  constexpr int U = 4;
  for (long long j0 = threadIdx.x; j0 < nv; j0 += (long long)U * blockDim.x) {
    int4 q[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long j = j0 + (long long)u * blockDim.x;
      q[u] = j < nv ? __ldg(v + j) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (j0 + (long long)u * blockDim.x < nv) {
        add(q[u].x);
        add(q[u].y);
        add(q[u].z);
        add(q[u].w);
      }
  }
  for (long long i = a1 + threadIdx.x; i < end; i += blockDim.x) add(__ldg(idx + i));
  if (bad) flag_status(status, MOE_STATUS_BAD_INDEX);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)e * G + blockIdx.x] = cnt[e];
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

// A warp per expert: its row of the table in place into the exclusive prefix over the ranges,
// the total into num_ids.  The row moves through shared memory (coalesced loads and stores, every
// load in flight at once) so that lane l can scan ranges [kScanPer l, kScanPer (l+1)) on its own;
// one warp scan of the lane sums places each lane's prefix.  (kScanPer is odd: the blocked
// accesses are free of bank conflicts.)
constexpr int kScanPer = (kMaxRanges + kWarp - 1) / kWarp;  // 19
__global__ void __launch_bounds__(kScanBlock) pft_scan_kernel(int* __restrict__ hist, int G, int E,
                                                              int* __restrict__ num_ids) {
  __shared__ int tile[kScanBlock / kWarp][kScanPer * kWarp];
  const int lane = threadIdx.x % kWarp, wid = threadIdx.x / kWarp;
  const int e = blockIdx.x * (kScanBlock / kWarp) + wid;
  if (e >= E) return;
  int* row = hist + (size_t)e * G;
  int* t = tile[wid];
  int v[kScanPer];
#pragma unroll
  for (int u = 0; u < kScanPer; ++u) {
    const int c = u * kWarp + lane;
    v[u] = c < G ? __ldcg(row + c) : 0;
  }
#pragma unroll
  for (int u = 0; u < kScanPer; ++u) t[u * kWarp + lane] = v[u];
  __syncwarp();
  int sum = 0;
#pragma unroll
  for (int u = 0; u < kScanPer; ++u) {
    v[u] = t[lane * kScanPer + u];
    sum += v[u];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < kWarp; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  int run = incl - sum;
#pragma unroll
  for (int u = 0; u < kScanPer; ++u) {
    t[lane * kScanPer + u] = run;
    run += v[u];
  }
  __syncwarp();
#pragma unroll
  for (int u = 0; u < kScanPer; ++u) {
    const int c = u * kWarp + lane;
    if (c < G) row[c] = t[u * kWarp + lane];
  }
  if (lane == kWarp - 1) num_ids[e] = incl;
}

// ---------------------------------------------------------------------------- 3. scatter
// Shared memory: cell[E][S] (S = words per expert + 1, odd, so that a pass over one word of
// every expert is free of bank conflicts), each cell {bitmap word, global row of the word's
// first entry}; soff[E+1] (offsets); base[E] (the next global row of each expert for this CTA);
// delta[E] (global row minus position in the tile's sorted copy); srt[kTileEntries] (the tile
// in (expert, token) order: expert << 16 | token in tile).
//
// A tile is tt tokens starting at t0 (its entries t0*k ... ), at most 32 << lg tokens and
// kTileEntries entries; thread x holds the tile's entries x, x + 256, ... in registers, the
// next tile's loaded while the current one is written out.  Entry q of a tile is token q / k,
// stepped from one of a thread's entries to the next (256 / k tokens and 256 % k columns).
__global__ void __launch_bounds__(kSBlock, 4) pft_scatter_kernel(const int* __restrict__ idx, int T, int k, int E,
                                                                 int range_t, int G, int lg, int tt,
                                                                 const int* __restrict__ hist,
                                                                 const int* __restrict__ num_ids,
                                                                 int* __restrict__ offsets,
                                                                 int* __restrict__ token_ids,
                                                                 int* __restrict__ expert_ids,
                                                                 int* __restrict__ slot_of, int* status) {
  extern __shared__ __align__(16) int sm[];
  const int wpe = 1 << lg, S = wpe + 1;
  uint2* cell = reinterpret_cast<uint2*>(sm);  // .x: bitmap word, .y: global row of its first bit
  int* soff = sm + 2 * E * S;
  int* base = soff + E + 1;
  int* delta = base + E;
  unsigned* srt = reinterpret_cast<unsigned*>(delta + E);
  __shared__ int warp_tot[kSBlock / kWarp];
  const int Tk = T * k;
  const int tb = blockIdx.x * range_t;
  const int te = min(tb + range_t, T);
  // token and column of this thread's first entry of a tile, and the steps between its entries
  const int lt0 = threadIdx.x / k, j0 = threadIdx.x % k;
  const int dt = kSBlock / k, dj = kSBlock % k;
  bool dup = false;
  int ev[kPerThread];
  // ids of the tile starting at token t0: -1 past the tile; an id outside [0,E) gets slot -1
  auto load_ids = [&](int t0) {
    const int e0 = t0 * k, e1 = min(t0 + tt, te) * k;
#pragma unroll
    for (int r = 0; r < kPerThread; ++r) {
      const int i = e0 + r * kSBlock + threadIdx.x;
      ev[r] = i < e1 ? __ldg(idx + i) : -1;
    }
#pragma unroll
    for (int r = 0; r < kPerThread; ++r) {
      const int i = e0 + r * kSBlock + threadIdx.x;
      if (i < e1 && (unsigned)ev[r] >= (unsigned)E) {
        slot_of[i] = -1;  // reported by pft_count
        ev[r] = -1;
      }
    }
  };
  // the first tile's ids and this range's column of the table load while num_ids is scanned
  if (tb < te) load_ids(tb);
  for (int e = threadIdx.x; e < E; e += kSBlock) base[e] = __ldcg(hist + (size_t)e * G + blockIdx.x);
  // offsets: the exclusive scan of num_ids
  {
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += kSBlock) {
      const int e = e0 + threadIdx.x;
      const int v = e < E ? __ldcg(num_ids + e) : 0;
      int tot;
      const int ex = block_exclusive_scan(v, warp_tot, &tot);
      if (e < E) soff[e] = carry + ex;
      carry += tot;
    }
    if (threadIdx.x == 0) soff[E] = carry;
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += kSBlock) offsets[e] = soff[e];
  for (int e = threadIdx.x; e < E; e += kSBlock) base[e] += soff[e];
  // expert_ids depends on offsets alone: this CTA fills rows [lo, hi), one expert's run at a time
  {
    const int per = (Tk + G - 1) / G;
    const int lo = min(blockIdx.x * per, Tk), hi = min(lo + per, Tk);
    if (lo < hi) {
      int a = 0, z = E;  // the expert holding row lo: the last e with soff[e] <= lo
      while (z - a > 1) {
        const int m = (a + z) >> 1;
        if (soff[m] <= lo) a = m;
        else z = m;
      }
      for (int e = a; e < E && soff[e] < hi; ++e) {
        const int r1 = min(soff[e + 1], hi);
        for (int r = max(soff[e], lo) + threadIdx.x; r < r1; r += kSBlock) expert_ids[r] = e;
      }
    }
  }
  for (int t0 = tb; t0 < te; t0 += tt) {
    const int nw = (min(tt, te - t0) + 31) >> 5;  // words of the tile's tokens
    // (a) clear the bitmap (nothing reads it after the previous tile's barrier)
    {
      uint4* c4 = reinterpret_cast<uint4*>(cell);  // two cells each
      const int n4 = E * S / 2;
      for (int q = threadIdx.x; q < n4; q += kSBlock) c4[q] = make_uint4(0u, 0u, 0u, 0u);
      if ((E * S) & 1)
        if (threadIdx.x == 0) cell[E * S - 1] = make_uint2(0u, 0u);
    }
    __syncthreads();
    // (b) one bit per entry
    {
      int lt = lt0, j = j0;
#pragma unroll
      for (int r = 0; r < kPerThread; ++r) {
        const int e = ev[r];
        if (e >= 0) {
          const unsigned m = 1u << (lt & 31);
          const unsigned old = atomicOr(&cell[e * S + (lt >> 5)].x, m);
          dup |= (old & m) != 0u;
        }
        lt += dt;
        j += dj;
        if (j >= k) { j -= k; ++lt; }
      }
    }
    __syncthreads();
    // (c) per expert: the tile's count, its place in the tile's sorted copy (a scan over the
    // experts), and each word's first global row; the expert's next row moves past the tile
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += kSBlock) {
      const int e = e0 + threadIdx.x;
      uint2* c = cell + e * S;
      int run = 0;
      if (e < E)
        for (int w = 0; w < nw; ++w) run += __popc(c[w].x);
      int tot;
      const int ex = block_exclusive_scan(run, warp_tot, &tot);
      if (e < E) {
        int row = base[e];
        delta[e] = row - (carry + ex);
        base[e] = row + run;
        for (int w = 0; w < nw; ++w) {
          const unsigned x = c[w].x;
          c[w] = make_uint2(x, (unsigned)row);
          row += __popc(x);
        }
      }
      carry += tot;
    }
    __syncthreads();
    // (d) the entry's row: its word's first row plus the bits below its own; slot_of in index
    // order, and the entry into the sorted copy
    {
      const int e0 = t0 * k;
      int lt = lt0, j = j0;
#pragma unroll
      for (int r = 0; r < kPerThread; ++r) {
        const int e = ev[r];
        if (e >= 0) {
          const uint2 c = cell[e * S + (lt >> 5)];
          const int row = (int)c.y + __popc(c.x & ((1u << (lt & 31)) - 1u));
          slot_of[e0 + r * kSBlock + threadIdx.x] = row;
          srt[row - delta[e]] = ((unsigned)e << 16) | (unsigned)lt;
        }
        lt += dt;
        j += dj;
        if (j >= k) { j -= k; ++lt; }
      }
    }
    if (t0 + tt < te) load_ids(t0 + tt);
    __syncthreads();
    // (e) token_ids from the sorted copy: consecutive entries of one expert to consecutive rows
    for (int q = threadIdx.x; q < carry; q += kSBlock) {
      const unsigned v = srt[q];
      const int row = q + delta[v >> 16];
      if ((unsigned)row < (unsigned)Tk) token_ids[row] = t0 + (int)(v & 0xffffu);  // guards the write
    }
  }
  if (dup) flag_status(status, MOE_STATUS_BAD_INDEX);
}

// Tile shape of the scatter: lg = log2 of the bitmap words per expert (E << lg <= kBitWords,
// lg <= 4, no more words than a range's tokens need) and tt tokens per tile (32 << lg, fewer
// when k would take a tile past kTileEntries).
void scatter_shape(int E, int k, int range_t, int* lg, int* tt) {
  int l = 4;
  while (l > 0 && (E << l) > kBitWords) --l;
  while (l > 0 && (32 << (l - 1)) >= range_t) --l;
  int t = 32 << l;
  const int by_k = kTileEntries / k;
  if (by_k < t) t = by_k < 1 ? 1 : by_k;
  *lg = l;
  *tt = t;
}

size_t scatter_smem(int E, int lg) {
  return (size_t)(2 * E * ((1 << lg) + 1) + 3 * E + 1 + kTileEntries) * sizeof(int);
}

}  // namespace

// Ranges (CTAs) for Tk entries: at least 1024 entries each, at most kMaxRanges of them.  The
// build cuts whole tokens: ceil(T / pft_num_chunks) tokens a range, which never makes more.
int pft_num_chunks(long long Tk) {
  const long long g = (Tk + 1023) / 1024;
  return (int)(g < 1 ? 1 : (g > kMaxRanges ? kMaxRanges : g));
}

size_t pft_scratch_bytes(long long Tk, int E) {
  return (size_t)pft_num_chunks(Tk) * (size_t)E * sizeof(int);
}

void launch_pft_build(const int* topk_idx, int T, int E, int k, int* num_ids, int* offsets,
                      int* token_ids, int* expert_ids, int* slot_of, void* ws, cudaStream_t st) {
  const long long Tk = (long long)T * k;
  const int gmax = pft_num_chunks(Tk);
  const int range_t = (T + gmax - 1) / gmax;  // tokens of one range
  const int G = (T + range_t - 1) / range_t;
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  int* hist = reinterpret_cast<int*>(static_cast<char*>(ws) + sizeof(WsHeader));
  pft_count_kernel<<<G, kPBlock, (size_t)E * sizeof(int), st>>>(topk_idx, Tk, E, (long long)range_t * k, G, hist,
                                                                 &hdr->status);
  count_launch(st);
  constexpr int per_cta = kScanBlock / kWarp;
  pft_scan_kernel<<<(E + per_cta - 1) / per_cta, kScanBlock, 0, st>>>(hist, G, E, num_ids);
  count_launch(st);
  int lg, tt;
  scatter_shape(E, k, range_t, &lg, &tt);
  const size_t smem = scatter_smem(E, lg);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(pft_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  pft_scatter_kernel<<<G, kSBlock, smem, st>>>(topk_idx, T, k, E, range_t, G, lg, tt, hist, num_ids, offsets,
                                               token_ids, expert_ids, slot_of, &hdr->status);
  count_launch(st);
}

}  // namespace moe
