// fp32 expert FFN forward on the tensor cores (sm_103a: tcgen05 + TMEM + TMA), TF32-free.
//
// The fp32 layer's GEMMs h1 = X W1[e], h3 = X W3[e] and y = a W2[e] run over exact three-plane
// bf16 splits of both operands, v = v0 + v1 + v2 (v0 = bf16(v), v1 = bf16(v - v0), v2 = bf16(v - v0
// - v1): every difference is exact in fp32 and the last plane keeps the remaining bits).  Each
// product of two planes is exact in the fp32 accumulator, and the operand product is the sum of
// six plane products,
//   a b = a0 b0 + a0 b1 + a1 b0 + a0 b2 + a1 b1 + a2 b0,
// the dropped a1 b2, a2 b1, a2 b2 lying below 2^-32 of it.  The tensor core adds with truncation,
// so the leading product and the five small ones go to two TMEM accumulators and every 256 of K
// (16 MMA steps) the epilogue drains both into fp32 registers with round-to-nearest adds: no
// truncated chain is longer than 16 steps.  That keeps the sums at fp32 accuracy.
//
// Grouped over the padding-free buffer with the experts' tokens on the MMA's N (swap-AB, as the
// bf16 engine): a unit is (expert e, 128-row tile of the weight dimension, chunk of at most 128
// of the expert's tokens), the chunk padded to a multiple of 16 columns in place.
//
//   mode   D (fp32, TMEM)   A (M x K): weight planes, MN-major    B (N x K): token planes, K-major   K
//   H1     h1^T [f x n]     W1[e] planes [h, f]                   xbuf planes [Tk, h]                 h
//   H3A    h3^T [f x n]     W3[e] planes [h, f]                   xbuf planes                         h
//   Y      y^T  [h x n]     W2[e] planes [f, h]                   a planes [Tk, f]                    f
// H3A's epilogue reads h1 back and writes h3, a = silu(h1) h3 and the three planes of a.  The
// token planes come from xbuf, or, with the dispatch folded in, straight from x[token_ids[p]].
//
// Warp roles (one CTA per SM): warp 0 issues the TMA loads (three A and three B planes per stage),
// warp 1 owns TMEM (two buffers of the accumulator pair) and issues the MMAs, warps 2-9 drain the
// accumulators, two warps per TMEM lane quarter each holding its row's 64 running sums of half the
// token columns, and warp 10 splits the next GEMM's weight tensor into its planes meanwhile (the
// GEMMs are bound by the L2 -> SM stream, with DRAM bandwidth to spare).  That split is a queue of
// 4096-value chunks taken with an atomic counter: the side warp takes chunks while the CTA's GEMM
// warps work, and once they are done (TMEM released) all eleven warps drain what is left, so a
// short GEMM never waits on one warp's split.  Every wait is bounded.
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "planes.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace ptx;

constexpr int FBM = 128;       // MMA M: rows of the weight dimension per unit
constexpr int FBN = 128;       // tokens per chunk (MMA N up to 128)
constexpr int FBK = 64;        // K per stage (one 128-byte swizzle row of bf16)
constexpr int kFSteps = 4;     // stages per drain: 256 of K
constexpr int kFEpiWarps = 8;   // two per TMEM lane quarter, each draining half the columns
constexpr int kFCols = FBN / 2;  // columns per epilogue warp
constexpr int kFSplitWarp = 2 + kFEpiWarps;  // the side warp that splits the next weight tensor
constexpr int kFGemmWarps = 2 + kFEpiWarps;  // producer, MMA, epilogue
constexpr int kFThreads = 32 * kFGemmWarps + 32;
constexpr int kSplitItem = 4096;  // values of one chunk of the next weight tensor's split
constexpr uint32_t kFBox = 8192;   // one 64 x 64 bf16 box
constexpr uint32_t kFPlaneA = 2 * kFBox;  // 128 weight columns x 64 K rows
constexpr uint32_t kFPlaneB = 2 * kFBox;  // 128 token rows x 64 K
constexpr uint32_t kFStage = 3 * kFPlaneA + 3 * kFPlaneB;  // 96 KB
constexpr int kFStages = 2;
constexpr int kFMaxE = 1024;

enum FMode { H1 = 0, H3A = 1, Y = 2 };

struct F32Params {
  CUtensorMap mapA[3];  // weight planes, [E * Krows, M] each
  CUtensorMap mapB[3];  // token planes, [Tk, K] each
  const int* offsets;
  int E, M, K;          // M: weight columns (f or h); K: h or f
  float* out;           // h1 | h3 | ybuf, [Tk, M]
  const float* h1;      // H3A: h1 to read back
  float* a;             // H3A: a = silu(h1) h3, [Tk, M]
  __nv_bfloat16* a_planes;  // H3A: three planes of a, [3][Tk][M]
  long long Tk;
  // the next GEMM's weight tensor, split into its planes by this launch (nullptr: none):
  // nsrc [E][nper] fp32 -> ndst [3][E][nper] bf16, nper a multiple of kSplitItem; chunks are
  // taken with split_ctr, zero at launch
  const float* nsrc;
  __nv_bfloat16* ndst;
  long long nper;
  int* split_ctr;
  int* status;
  unsigned long long wait_ns;
  int withhold;
};

// Chunks of the next weight tensor's planes, over the experts with rows (s_act[0..nact)), taken
// from the launch's counter by whole warps until none are left, or until *stop reaches
// kFGemmWarps (the side warp: the CTA's GEMM warps are done and the whole CTA takes over).
// Nothing in this GEMM reads the planes; the next launch does.
__device__ __noinline__ void split_next_weights(const F32Params& p, const int* s_act, int nact, int lane,
                                                const volatile int* stop) {
  if (p.nsrc == nullptr) return;
  constexpr int G8 = kSplitItem / 8;  // 8-value groups of a chunk: 16 a lane, in two rounds of 8
  constexpr int U = 8;
  const int ipe = (int)(p.nper / kSplitItem);
  const int nitems = nact * ipe;
  const long long n = (long long)p.E * p.nper;
  const float4* src = reinterpret_cast<const float4*>(p.nsrc);
  uint4* d0 = reinterpret_cast<uint4*>(p.ndst);
  uint4* d1 = reinterpret_cast<uint4*>(p.ndst + n);
  uint4* d2 = reinterpret_cast<uint4*>(p.ndst + 2 * n);
  for (;;) {
    // lane 0 alone reads the stop flag and takes the chunk, so the warp stays converged
    int it = nitems;
    if (lane == 0 && (stop == nullptr || *stop < kFGemmWarps)) it = atomicAdd(p.split_ctr, 1);
    it = __shfl_sync(0xffffffffu, it, 0);
    if (it >= nitems) break;
    const long long g0 = (long long)s_act[it / ipe] * (p.nper / 8) + (long long)(it % ipe) * G8;
#pragma unroll 1
    for (int r = 0; r < G8 / (32 * U); ++r) {
      float4 a[U], b[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long j = g0 + (r * U + u) * 32 + lane;
        a[u] = __ldcs(src + 2 * j);  // read once: keep it out of the GEMM's L2 working set
        b[u] = __ldcs(src + 2 * j + 1);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long j = g0 + (r * U + u) * 32 + lane;
        split3_vec8(a[u], b[u], d0 + j, d1 + j, d2 + j);
      }
    }
  }
}

struct FUnit {
  int e, m0, row0, rows, nmma;
};

__device__ __forceinline__ FUnit fdecode(int u, const int* s_pref, const int* s_off, int E, int mt) {
  int lo = 0, hi = E - 1;  // largest e with s_pref[e] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pref[mid] <= u) lo = mid; else hi = mid - 1;
  }
  FUnit w;
  w.e = lo;
  const int n = s_off[lo + 1] - s_off[lo];
  const int nc = (n + FBN - 1) / FBN;
  const int cs = ((n + nc - 1) / nc + 15) & ~15;
  const int local = u - s_pref[lo];
  const int mtile = local / nc, c = local % nc;
  (void)mt;
  w.m0 = mtile * FBM;
  w.row0 = s_off[lo] + c * cs;
  w.rows = min(cs, n - c * cs);
  w.nmma = (w.rows + 15) & ~15;
  return w;
}

template <int MODE>
__global__ void __launch_bounds__(kFThreads, 1) f32tc_kernel(const __grid_constant__ F32Params p) {
  extern __shared__ __align__(1024) uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kFStages];
  __shared__ __align__(8) uint64_t empty_bar[kFStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_off[kFMaxE + 1];
  __shared__ int s_pref[kFMaxE + 1];
  __shared__ int s_act[kFMaxE];  // experts with rows, ascending
  __shared__ int s_total, s_nact;
  __shared__ volatile int s_gemm_done;  // GEMM warps past their loops

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t ring = (smem_u32(dsmem) + 1023u) & ~1023u;
  const int mt = p.M / FBM;

  // ------------------------------------------------------------------ schedule
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_off[i] = __ldg(p.offsets + i);
  __syncthreads();
  if (warp == 0) {
    const int per = (p.E + 31) / 32;
    const int b0 = min(lane * per, p.E), b1 = min(b0 + per, p.E);
    int local = 0;
    for (int e = b0; e < b1; ++e) {
      const int ue = ((s_off[e + 1] - s_off[e] + FBN - 1) / FBN) * mt;
      s_pref[e + 1] = ue;
      local += ue;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int e = b0; e < b1; ++e) {
      const int ue = s_pref[e + 1];
      s_pref[e] = run;
      run += ue;
    }
    if (lane == 31) {
      s_pref[p.E] = incl;
      s_total = incl;
    }
  } else if (warp == 1) {
    // the experts with rows, in order (ballot compaction)
    int nact = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      const bool act = e < p.E && s_off[e + 1] > s_off[e];
      const unsigned m = __ballot_sync(0xffffffffu, act);
      if (act) s_act[nact + __popc(m & ((1u << lane) - 1u))] = e;
      nact += __popc(m);
    }
    if (lane == 0) {
      s_nact = nact;
      s_gemm_done = 0;
    }
  }
  __syncthreads();
  const int total = s_total;
  const int nact = s_nact;
  if ((int)blockIdx.x >= total) {  // no unit for this CTA (before any TMEM use): every warp splits
    split_next_weights(p, s_act, nact, lane, nullptr);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kFStages; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&tfull_bar[b], 1); mbar_init(&tempty_bar[b], kFEpiWarps); }
    mbar_init(&drain_bar, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;
  const int nsteps = p.K / FBK;

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const FUnit w = fdecode(u, s_pref, s_off, p.E, mt);
        const int nbB = (w.nmma + 63) / 64;
        const uint32_t tx = 3 * kFPlaneA + 3 * (uint32_t)nbB * kFBox;
        for (int ks = 0; ks < nsteps; ++ks) {
          if (!mbar_wait(&empty_bar[s], ph ^ 1u, &s_abort, p.status, p.wait_ns)) { ok = false; break; }
          if (p.withhold && u == (int)blockIdx.x && ks == 0) {  // test hook: a stage nobody fills
            if (++s == kFStages) { s = 0; ph ^= 1u; }
            continue;
          }
          mbar_expect_tx(&full_bar[s], tx);
          const uint32_t a_sm = ring + s * kFStage;
          const uint32_t b_sm = a_sm + 3 * kFPlaneA;
          const int k0 = ks * FBK;
          const int y = w.e * p.K + k0;
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            tma_load_2d(a_sm + i * kFPlaneA, &p.mapA[i], &full_bar[s], w.m0, y);
            tma_load_2d(a_sm + i * kFPlaneA + kFBox, &p.mapA[i], &full_bar[s], w.m0 + 64, y);
            for (int j = 0; j < nbB; ++j)
              tma_load_2d(b_sm + i * kFPlaneB + j * kFBox, &p.mapB[i], &full_bar[s], k0, w.row0 + 64 * j);
          }
          if (++s == kFStages) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok || s_abort) {  // give the loads already in flight time to land
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 2000000ull) {
        }
      }
      atomicAdd((int*)&s_gemm_done, 1);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    int s = 0;
    uint32_t ph = 0;
    int cc = 0;  // drain chunks issued so far (accumulator buffer = cc & 1)
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const FUnit w = fdecode(u, s_pref, s_off, p.E, mt);
      const uint32_t idesc = idesc_bf16(w.nmma, true, false);
      for (int c0 = 0; c0 < nsteps && ok; c0 += kFSteps, ++cc) {
        const int b = cc & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&tempty_bar[b], ((uint32_t)(cc >> 1) & 1u) ^ 1u, &s_abort,
                                               p.status, p.wait_ns))) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_main = tmem_base + (uint32_t)(b * 2 * FBN);
        const uint32_t d_corr = d_main + FBN;
        const int c1 = min(nsteps, c0 + kFSteps);
        for (int ks = c0; ks < c1; ++ks) {
          if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[s], ph, &s_abort, p.status, p.wait_ns))) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a_sm = ring + s * kFStage;
            const uint32_t b_sm = a_sm + 3 * kFPlaneA;
#pragma unroll
            for (int kk = 0; kk < FBK / 16; ++kk) {
              const bool first = (ks == c0 && kk == 0);
              // (A plane, B plane): the leading product, then the small ones from the smallest
              const int qa[6] = {0, 2, 1, 0, 1, 0};
              const int qb[6] = {0, 0, 1, 2, 0, 1};
#pragma unroll
              for (int t = 0; t < 6; ++t) {
                const uint64_t ad = sdesc(a_sm + qa[t] * kFPlaneA + kk * 2048, kFBox, 1024);
                const uint64_t bd = sdesc(b_sm + qb[t] * kFPlaneB + kk * 32, 16, 1024);
                const bool lead = (t == 0);
                umma(lead ? d_main : d_corr, ad, bd, idesc, (first && (lead || t == 1)) ? 0u : 1u);
              }
            }
            umma_commit(&empty_bar[s]);  // the stage is free once these MMAs have read it
          }
          __syncwarp();
          if (++s == kFStages) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) umma_commit(&tfull_bar[b]);
        __syncwarp();
      }
    }
    if (lane == 0) {
      umma_commit(&drain_bar);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(&drain_bar, 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
      atomicAdd((int*)&s_gemm_done, 1);
    }
    __syncwarp();
  } else if (warp == kFSplitWarp) {
    // ================================================================ side splitter
    split_next_weights(p, s_act, nact, lane, &s_gemm_done);
  } else {
    // ================================================================ epilogue (warps 2..9)
    const int q = warp & 3;              // TMEM lane quarter
    const int cb = ((warp - 2) >> 2) * kFCols;  // this warp's first column
    int cc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const FUnit w = fdecode(u, s_pref, s_off, p.E, mt);
      float run[kFCols];
#pragma unroll
      for (int i = 0; i < kFCols; ++i) run[i] = 0.f;
      for (int c0 = 0; c0 < nsteps; c0 += kFSteps, ++cc) {
        const int b = cc & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull_bar[b], (uint32_t)(cc >> 1) & 1u, &s_abort, p.status,
                                               p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t0 = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * 2 * FBN + cb);
#pragma unroll
        for (int g = 0; g < kFCols / 16; ++g) {
          if (cb + 16 * g < w.nmma) {
            float vm[16], vc[16];
            tmem_ld16(t0 + 16 * g, vm);
            tmem_ld16(t0 + FBN + 16 * g, vc);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) run[16 * g + i] += vm[i] + vc[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[b]);
      }
      if (!ok) break;
      // element (token n, weight column m) of the output; lanes hold consecutive m, so each store
      // instruction writes 32 consecutive floats of one token row
      const int m = w.m0 + q * 32 + lane;
      if (MODE == H3A) {
        // h1 in groups of 16 columns, all loads issued before the group's stores
#pragma unroll
        for (int g = 0; g < kFCols / 16; ++g) {
          if (cb + 16 * g >= w.rows) break;
          float z1[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = cb + 16 * g + i;
            z1[i] = n < w.rows ? __ldg(p.h1 + (size_t)(w.row0 + n) * p.M + m) : 0.f;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = cb + 16 * g + i;
            if (n < w.rows) {
              const size_t o = (size_t)(w.row0 + n) * p.M + m;
              const float v = run[16 * g + i];
              const float av = z1[i] * sigmoidf_(z1[i]) * v;
              p.out[o] = v;
              p.a[o] = av;
              split3_value(av, p.a_planes + o, p.a_planes + p.Tk * p.M + o, p.a_planes + 2 * p.Tk * p.M + o);
            }
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < kFCols; ++i)
          if (cb + i < w.rows) p.out[(size_t)(w.row0 + cb + i) * p.M + m] = run[i];
      }
    }
    __syncwarp();
    if (lane == 0) atomicAdd((int*)&s_gemm_done, 1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
  }
  // what is left of the next tensor's split, with every warp
  split_next_weights(p, s_act, nact, lane, nullptr);
}

// Three-plane split of the experts' weight matrices, skipping experts without rows: expert
// blockIdx.y, dst[p][e][i] = plane p of src[e][i] for its `per` elements (a multiple of 8), eight
// elements a thread with 16-byte loads and plane stores.
__global__ void __launch_bounds__(256) split3_experts_kernel(const float* __restrict__ src, const int* __restrict__ offsets,
                                                             long long per, long long n, __nv_bfloat16* __restrict__ dst) {
  const int e = blockIdx.y;
  if (__ldg(offsets + e + 1) == __ldg(offsets + e)) return;  // no rows: its planes are never read
  const size_t o = (size_t)e * per;
  const float4* s = reinterpret_cast<const float4*>(src + o);
  uint4* d0 = reinterpret_cast<uint4*>(dst + o);
  uint4* d1 = reinterpret_cast<uint4*>(dst + n + o);
  uint4* d2 = reinterpret_cast<uint4*>(dst + 2 * n + o);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < per / 8; i += (long long)gridDim.x * blockDim.x)
    split3_vec8(__ldg(s + 2 * i), __ldg(s + 2 * i + 1), d0 + i, d1 + i, d2 + i);
}

// The same for n contiguous values (n a multiple of 8): dst[p][i] = plane p of src[i].
__global__ void __launch_bounds__(256) split3_rows_kernel(const float* __restrict__ src, long long n,
                                                          __nv_bfloat16* __restrict__ dst, int* zero2) {
  if (zero2 != nullptr && blockIdx.x == 0 && threadIdx.x < 2) zero2[threadIdx.x] = 0;  // the next launches' counters
  const float4* s = reinterpret_cast<const float4*>(src);
  uint4* d0 = reinterpret_cast<uint4*>(dst);
  uint4* d1 = reinterpret_cast<uint4*>(dst + n);
  uint4* d2 = reinterpret_cast<uint4*>(dst + 2 * n);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n / 8; i += (long long)gridDim.x * blockDim.x)
    split3_vec8(__ldg(s + 2 * i), __ldg(s + 2 * i + 1), d0 + i, d1 + i, d2 + i);
}

// The dispatch folded into the split of the token rows: dst[p][row] = plane p of
// x[token_ids[row]], a CTA per row at a time with the next row's id loaded ahead.  An id outside
// [0,T) gives zero planes and sets MOE_STATUS_BAD_INDEX, as moe_dispatch does.  Also zeroes the
// next launches' two split counters (zero2).
__global__ void __launch_bounds__(256) split3_gather_kernel(const float* __restrict__ x,
                                                            const int* __restrict__ token_ids, int T,
                                                            long long Tk, int h, __nv_bfloat16* __restrict__ dst,
                                                            int* zero2, int* status) {
  if (blockIdx.x == 0 && threadIdx.x < 2) zero2[threadIdx.x] = 0;
  const int hv = h / 8;  // 8-value items per row
  const long long n = Tk * h;
  uint4* d0 = reinterpret_cast<uint4*>(dst);
  uint4* d1 = reinterpret_cast<uint4*>(dst + n);
  uint4* d2 = reinterpret_cast<uint4*>(dst + 2 * n);
  long long row = blockIdx.x;
  int t = row < Tk ? __ldg(token_ids + row) : 0;
  for (; row < Tk; row += gridDim.x) {
    const long long nxt = row + gridDim.x;
    const int tn = nxt < Tk ? __ldg(token_ids + nxt) : 0;
    const long long o = row * hv;
    if ((unsigned)t < (unsigned)T) {
      const float4* s = reinterpret_cast<const float4*>(x + (size_t)t * h);
      for (int c = threadIdx.x; c < hv; c += blockDim.x)
        split3_vec8(__ldg(s + 2 * c), __ldg(s + 2 * c + 1), d0 + o + c, d1 + o + c, d2 + o + c);
    } else {
      if (threadIdx.x == 0) flag_status(status, MOE_STATUS_BAD_INDEX);
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int c = threadIdx.x; c < hv; c += blockDim.x) {
        d0[o + c] = z;
        d1[o + c] = z;
        d2[o + c] = z;
      }
    }
    t = tn;
  }
}

template <int MODE>
int flaunch(const F32Params& p0, cudaStream_t st) {
  F32Params p = p0;
  p.withhold = debug_take_withhold(&p.wait_ns) ? 1 : 0;
  const int smem = (int)(kFStages * kFStage + 1024);
  if (cudaFuncSetAttribute(f32tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -1;
  f32tc_kernel<MODE><<<num_sms(), kFThreads, smem, st>>>(p);
  count_launch(st);
  return 0;
}

bool make_plane_maps(CUtensorMap* maps, const __nv_bfloat16* planes, long long rows, long long cols) {
  for (int i = 0; i < 3; ++i)
    if (!tc_make_map(&maps[i], planes + (size_t)i * rows * cols, rows, cols, 64, 64)) return false;
  return true;
}

size_t r256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

bool f32tc_supported(int dtype, int h, int f, int E) {
  const char* env = getenv("MOE_PFT_GEMM");
  if (env && strcmp(env, "simt") == 0) return false;
  return dtype == MOE_F32 && h % 128 == 0 && f % 128 == 0 && E <= kFMaxE && tc_encode_available();
}

size_t f32tc_scratch(long long Tk, int E, int h, int f) {
  // token planes of xbuf and of a, and two weight-plane buffers: one GEMM reads one while its
  // side warp (then the whole CTA) fills the other for the next GEMM
  return r256((size_t)3 * Tk * h * 2) + r256((size_t)3 * Tk * f * 2) + 2 * r256((size_t)3 * E * h * f * 2) + 256;
}

int f32tc_expert_ffn(const float* xbuf, const float* x, const int* token_ids, int T, const int* offsets,
                     const float* W1, const float* W3, const float* W2, int Tk, int E, int h, int f, float* ybuf,
                     float* h1, float* h3, float* a, void* scratch, int* status, cudaStream_t st) {
  char* sp = static_cast<char*>(scratch);
  const size_t wbytes = r256((size_t)3 * E * h * f * 2);
  __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(sp);
  __nv_bfloat16* ap = reinterpret_cast<__nv_bfloat16*>(sp + r256((size_t)3 * Tk * h * 2));
  char* wbase = sp + r256((size_t)3 * Tk * h * 2) + r256((size_t)3 * Tk * f * 2);
  __nv_bfloat16* wpA = reinterpret_cast<__nv_bfloat16*>(wbase);            // W1, then W2
  __nv_bfloat16* wpB = reinterpret_cast<__nv_bfloat16*>(wbase + wbytes);   // W3
  int* ctr = reinterpret_cast<int*>(wbase + 2 * wbytes);                    // the two split queues
  const int blocks = 8 * num_sms();
  const long long per = (long long)h * f;
  if (xbuf != nullptr) split3_rows_kernel<<<blocks, 256, 0, st>>>(xbuf, (long long)Tk * h, xp, ctr);
  else split3_gather_kernel<<<blocks, 256, 0, st>>>(x, token_ids, T, Tk, h, xp, ctr, status);
  count_launch(st);
  const dim3 wgrid(16, E);
  split3_experts_kernel<<<wgrid, 256, 0, st>>>(W1, offsets, per, (long long)E * per, wpA);
  count_launch(st);

  F32Params g;
  memset(&g, 0, sizeof(g));
  g.offsets = offsets; g.E = E; g.Tk = Tk; g.status = status;
  g.M = f; g.K = h; g.nper = per;
  // h1 = xbuf W1, while W3 is split into the second buffer
  bool ok = make_plane_maps(g.mapB, xp, Tk, h) && make_plane_maps(g.mapA, wpA, (long long)E * h, f);
  if (!ok) return -1;
  g.out = h1; g.nsrc = W3; g.ndst = wpB; g.split_ctr = ctr;
  if (flaunch<H1>(g, st)) return -1;
  // h3 = xbuf W3, a = silu(h1) h3 and its planes, while W2 is split into the first buffer
  ok = make_plane_maps(g.mapA, wpB, (long long)E * h, f);
  if (!ok) return -1;
  g.out = h3; g.h1 = h1; g.a = a; g.a_planes = ap; g.nsrc = W2; g.ndst = wpA; g.split_ctr = ctr + 1;
  if (flaunch<H3A>(g, st)) return -1;
  // y = a W2
  F32Params d;
  memset(&d, 0, sizeof(d));
  d.offsets = offsets; d.E = E; d.Tk = Tk; d.status = status;
  ok = make_plane_maps(d.mapB, ap, Tk, f) && make_plane_maps(d.mapA, wpA, (long long)E * f, h);
  if (!ok) return -1;
  d.M = h; d.K = f;
  d.out = ybuf;
  return flaunch<Y>(d, st);
}

}  // namespace moe
