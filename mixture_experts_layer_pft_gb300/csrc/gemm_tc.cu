// Tensor-core grouped GEMM engine for the bf16 expert FFN (sm_103a: tcgen05 + TMEM + TMA).
//
// One persistent, warp-specialised kernel template serves the six GEMMs of the expert FFN
// forward and backward over the padding-free buffer.  Every GEMM is arranged so that a weight
// (or weight-gradient) dimension is the MMA's M = 128 and the expert's tokens are either the
// MMA's N (forward, dgrad) or its K (wgrad).  With tokens on N, an expert segment of n rows
// costs round_up(n, 16) columns: the in-place tile padding is at most 15 columns per segment
// and each 128-row weight tile streams from HBM once per chunk of its expert's tokens (128 for
// the gate/up GEMM, 256 for the others; the chunks of one tile run side by side and share L2).
//
//   mode      D (fp32 in TMEM)            A operand (M x K)          B operand (N x K)
//   GATEUP    H1^T, H3^T [f x n]          W1[e], W3[e] ([h,f]: MN)   xbuf rows   (K-major)
//   DOWN      Y^T [h x n]                 W2[e] ([f,h]: MN)          a rows      (K-major)
//   DA        dA^T [f x n]                W2[e] ([f,h]: K-major)     dybuf rows  (K-major)
//   DX        dX^T [h x n], K = 2f        W1[e] then W3[e] (K-maj)   dh1 then dh3 rows (K-major)
//   WGRAD13   dW1^T, dW3^T [f x h-tile]   dh1, dh3 rows ([n,f]: MN)  xbuf rows ([n,h]: MN), K = n
//   WGRAD2    dW2^T [h x f-tile]          dybuf rows ([n,h]: MN)     a rows ([n,f]: MN), K = n
//
// Warp roles (one CTA per SM): warp 0 issues TMA loads into a ring of shared-memory stages;
// warp 1 owns the TMEM allocation and one lane issues tcgen05.mma into fp32 accumulators in
// TMEM; the epilogue warps (4, or 8 = two per TMEM lane quarter splitting the columns) drain
// TMEM (tcgen05.ld), apply the epilogue (SwiGLU, its derivative, or a plain store) and
// transpose each block through shared memory: token-N outputs go out in 32 x 16 blocks with
// 16-byte stores, four lanes per 64-byte column segment; weight gradients in 32 x 32 blocks as
// TMA tensor stores (wider blocks halve the per-block latency that bounds that epilogue).  Stages
// and accumulators hand over through mbarriers.  Every wait is bounded (about two seconds of
// %globaltimer): on expiry the kernel sets MOE_STATUS_TIMEOUT, every role unwinds, and the
// TMEM is released before the CTA exits.  No cluster, no multicast.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace ptx;

constexpr int BM = 128;           // MMA M: rows of the weight dimension per tile
constexpr int BK = 64;            // K per stage: one 128-byte swizzle row of bf16
constexpr uint32_t kBox = 8192;   // bytes of one 64 x 64 bf16 box
constexpr uint32_t kATile = 16384;  // bytes of one 128 x 64 A tile
constexpr int kTmemCols = 512;
constexpr int kMaxE = 1024;
constexpr uint32_t kStageRegion = 196608;  // shared memory given to the stage ring

// GATEUP_WIDE is the gate/up GEMM with 256-token chunks: each weight tile streams once per
// expert when experts hold up to 256 tokens, at the price of one accumulator set (its epilogue is
// not overlapped with the next unit's MMAs) and three stages in place of four.  The host picks it
// when experts average more than 96 tokens (every X-MoE shape measured: -5% to -22% against the
// 128-token chunks).
// DOWN_PAIR, DA_PAIR and DX_PAIR are DOWN, DA and DX with two 128-row M tiles per unit: the two
// accumulators share each token-chunk stage, so the chunk streams into shared memory once per 256
// rows of the weight dimension instead of once per 128 (one accumulator set, three stages).
enum Mode {
  GATEUP = 0, DOWN = 1, DA = 2, DX = 3, WGRAD13 = 4, WGRAD2 = 5, GATEUP_WIDE = 6,
  DOWN_PAIR = 7, DA_PAIR = 8, DX_PAIR = 9, WGRAD13_WIDE = 10, WGRAD2_PAIR = 11
};

template <int MODE> struct Cfg {
  static constexpr int BASE = MODE == GATEUP_WIDE ? GATEUP : MODE == DOWN_PAIR ? DOWN
                              : MODE == DA_PAIR ? DA : MODE == DX_PAIR ? DX
                              : MODE == WGRAD13_WIDE ? WGRAD13 : MODE == WGRAD2_PAIR ? WGRAD2 : MODE;
  static constexpr bool PAIR = (MODE == DOWN_PAIR || MODE == DA_PAIR || MODE == DX_PAIR);  // token-N pairs
  static constexpr bool MPAIR = PAIR || MODE == WGRAD2_PAIR;  // two 128-row M tiles per unit
  static constexpr bool GU = (BASE == GATEUP);
  static constexpr int NUM_A = (GU || BASE == WGRAD13 || MPAIR) ? 2 : 1;  // accumulators per unit
  static constexpr bool A_MN = (GU || BASE == DOWN || BASE == WGRAD13 || BASE == WGRAD2);
  static constexpr bool B_MN = (BASE == WGRAD13 || BASE == WGRAD2);
  static constexpr bool TOKEN_N = (BASE <= DX);
  static constexpr int MT = MPAIR ? 2 * BM : BM;  // rows of the weight (M) dimension per unit
  // gate/up and dW1/dW3 keep two accumulators per unit; 128-column tiles leave room to
  // double-buffer them (the _WIDE variants take 256 columns and one accumulator set)
  static constexpr int BN = (MODE == WGRAD13 || MODE == GATEUP) ? 128 : 256;
  static constexpr uint32_t A_BYTES = NUM_A * kATile;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + (BN / 64) * kBox;
  static constexpr int STAGES = kStageRegion / STAGE_BYTES;
  static constexpr int ACC_BUFS = kTmemCols / (NUM_A * BN);
  // epilogue: two warps per TMEM lane quarter (splitting the columns), except for the gate/up
  // GEMM, whose three outputs per element need more transpose buffer than shared memory has left
  static constexpr int EPI_WARPS = (MODE == GATEUP) ? 4 : 8;  // GATEUP_WIDE: 3 stages leave room for 8
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  // epilogue chunk: columns per TMEM load and per tensor store.  Weight gradients drain 32 at a
  // time and alternate between two transpose slots per warp, so two tensor stores are in flight.
  static constexpr int CW = TOKEN_N ? 16 : 32;
  static constexpr int NSLOT = (GU || !TOKEN_N) ? (GU ? 3 : 2) : (BASE == DA) ? 2 : 1;
  // per-expert tables in shared memory: token-N modes search the unit prefix sums; weight
  // gradients have the same unit count per expert and read the two offsets they need directly
  static constexpr int TABLE = TOKEN_N ? kMaxE + 1 : 1;
  static_assert(ACC_BUFS >= 1 && STAGES >= 2, "tile configuration");
};

struct TcParams {
  CUtensorMap mapA0;  // GATEUP W1 | DOWN W2 | DA W2 | DX W1 | WGRAD13 dh1 | WGRAD2 dybuf
  CUtensorMap mapA1;  // GATEUP W3 | DX W3 | WGRAD13 dh3
  CUtensorMap mapB0;  // GATEUP xbuf | DOWN a | DA dybuf | DX dh1 | WGRAD13 xbuf | WGRAD2 a
  CUtensorMap mapB1;  // DX dh3
  CUtensorMap mapO0;  // wgrad: dW1 | dW2 viewed [E * rows, cols], 32 x 32 boxes (TMA stores)
  CUtensorMap mapO1;  // WGRAD13: dW3
  const int* offsets;
  int E;
  int M;           // total rows of the M (weight) dimension per expert
  int K;           // token-N modes: K of one operand pair (DX: f per half)
  int Nw;          // wgrad modes: total N (weight) columns
  int a_rows;      // rows per expert in the 2D view of the weight map(s) (token-N modes)
  __nv_bfloat16* out0;
  __nv_bfloat16* out1;
  __nv_bfloat16* out2;
  const __nv_bfloat16* in0;
  const __nv_bfloat16* in1;
  int ld_out;
  long long out_expert_stride;  // wgrad: elements between consecutive experts' outputs
  int* status;
  // gate/up and dW1/dW3 with gathered token rows: row p of the padding-free buffer is read as
  // gx[gids[p]] (gx: [gx_rows, gx_ld]); null gx means the buffer comes through mapB0
  const __nv_bfloat16* gx;
  const int* gids;
  int gx_rows;
  int gx_ld;
  // down projection with the combine folded in (paired M tiles): y[t, m] = sum_j w[t,j] ybuf[slot(t,j), m]
  // is summed by the unit that completes token t's k rows of a 128-row M tile (c_cnt counts them)
  __nv_bfloat16* c_y;  // null: no combine
  const int* c_tok;    // token of each buffer row (the PFT's token_ids)
  const int* c_slot;   // [T*k] buffer row of (t, j)
  const float* c_w;    // [T*k] gate weights
  int* c_cnt;          // [T * c_mt] contribution counters, zero at launch
  int c_T, c_k, c_mt;  // tokens, top-k, 128-row M tiles per token row
  // bounded waits: limit per wait in ns (0: the default); withhold != 0 is the test hook of
  // moe_debug_withhold_stage (the producer never fills the first stage of the first unit)
  unsigned long long wait_ns;
  int withhold;
};

// Logistic function for the bf16 epilogues: the fast exponential and division are accurate to a
// few fp32 ulps, far below the bf16 rounding of every value they feed.
__device__ __forceinline__ float sigmoid_bf16_epilogue(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// ---------------------------------------------------------------------------- work units

struct Unit {
  int e;        // expert
  int m0;       // first row of the weight (M) dimension
  int row0;     // token-N: first buffer row of the chunk; wgrad: first buffer row of the expert
  int rows;     // token-N: rows in the chunk; wgrad: rows of the expert (K)
  int n0;       // wgrad: first N column
  int ncols;    // columns of D to produce (token-N: rows; wgrad: N tile width)
  int nmma;     // MMA N (multiple of 16)
  int nk;       // K steps of BK
  int na;       // accumulators (A tiles) in use: NUM_A, or 1 for a paired mode's split unit
};

// Token-N modes: expert e has nc_e = ceil(n_e / BN) chunks of about equal size (a multiple of
// 16 rows, the last one shorter); its units are (m-tile, chunk) pairs, chunks innermost, so
// the CTAs that stream one weight tile for different chunks run side by side.
//
// Paired modes balance the last wave: when the paired units leave a last wave at most half
// full, each of its units is split into its two 128-row M tiles, which go after all full
// pairs, so no CTA runs more than half a pair beyond the others.
struct Sched {
  int total;
  int mt;     // M tiles per expert
  int nt;     // wgrad: N tiles
  int pairs;  // paired modes: units that keep both M tiles (the rest are split)
};

template <int MODE>
__device__ __forceinline__ Unit decode(int u, const Sched& sc, const int* s_pref, const int* s_off,
                                       const TcParams& p) {
  using C = Cfg<MODE>;
  Unit w;
  w.na = C::NUM_A;
  int half = 0;  // paired modes: which M tile a split unit keeps
  if (C::PAIR && u >= sc.pairs) {
    const int v = u - sc.pairs;
    u = sc.pairs + (v >> 1);
    half = v & 1;
    w.na = 1;
  }
  if (C::TOKEN_N) {
    int lo = 0, hi = p.E - 1;  // largest e with s_pref[e] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pref[mid] <= u) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int n = s_off[e + 1] - s_off[e];
    const int nc = (n + C::BN - 1) / C::BN;
    const int cs = ((n + nc - 1) / nc + 15) & ~15;
    const int local = u - s_pref[e];
    const int mtile = local / nc, c = local % nc;
    w.e = e;
    w.m0 = mtile * C::MT + half * BM;
    w.row0 = s_off[e] + c * cs;
    w.rows = min(cs, n - c * cs);
    w.n0 = 0;
    w.ncols = w.rows;
    w.nmma = (w.rows + 15) & ~15;
    w.nk = (C::BASE == DX) ? 2 * p.K / BK : p.K / BK;
  } else {
    const int per = sc.mt * sc.nt;
    w.e = u / per;
    const int r = u % per;
    w.m0 = (r / sc.nt) * C::MT;
    w.n0 = (r % sc.nt) * C::BN;
    w.row0 = __ldg(p.offsets + w.e);
    w.rows = __ldg(p.offsets + w.e + 1) - w.row0;
    w.ncols = min(C::BN, p.Nw - w.n0);
    w.nmma = w.ncols;
    w.nk = (w.rows + BK - 1) / BK;
  }
  return w;
}

// ---------------------------------------------------------------------------- combine fold
// Down projection with the combine folded in (kept out of line, away from the epilogue's
// registers).  fold_count: count this unit's (token row, M tile) contributions; a cell reaching
// k contributions joins this CTA's list.  fold_sum: one warp per listed cell sums the token's k
// rows of that 128-row M tile from ybuf (read through L2), j ascending in fp32, one rounding,
// as the combine kernel does.
static __device__ __noinline__ void fold_count(const TcParams* pp, int row0, int ncols, int na, int tile0,
                                               int et, int nthreads, int* own, int* nown) {
  const TcParams& p = *pp;
  for (int cq = et; cq < ncols * na; cq += nthreads) {
    const int c = cq % ncols, tl = cq / ncols;
    const int t = __ldg(p.c_tok + row0 + c);
    if ((unsigned)t < (unsigned)p.c_T) {
      const int cell = t * p.c_mt + tile0 + tl;
      if (atomicAdd(p.c_cnt + cell, 1) == p.c_k - 1) own[atomicAdd(nown, 1)] = cell;
    } else {
      flag_status(p.status, MOE_STATUS_BAD_INDEX);
    }
  }
}

static __device__ __noinline__ void fold_sum(const TcParams* pp, const int* own, int nown, int ew, int nwarps,
                                             int lane) {
  const TcParams& p = *pp;
  for (int i = ew; i < nown; i += nwarps) {
    const int cell = own[i];
    const int t = cell / p.c_mt;
    const size_t m = (size_t)(cell % p.c_mt) * BM + 4 * lane;  // this lane's 4 outputs
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < p.c_k; j0 += 4) {
      int sj[4];
      float wj[4];
      uint2 r[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        sj[jj] = -1;
        wj[jj] = 0.f;
        if (j0 + jj < p.c_k) {
          const int sl = __ldg(p.c_slot + (size_t)t * p.c_k + j0 + jj);
          wj[jj] = __ldg(p.c_w + (size_t)t * p.c_k + j0 + jj);
          if ((unsigned)sl < (unsigned)(p.c_T * p.c_k)) sj[jj] = sl;
          else flag_status(p.status, MOE_STATUS_BAD_INDEX);
        }
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
        if (sj[jj] >= 0) r[jj] = __ldcg(reinterpret_cast<const uint2*>(p.out0 + (size_t)sj[jj] * p.ld_out + m));
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        if (sj[jj] < 0) continue;
        acc[0] = fmaf(wj[jj], __uint_as_float(r[jj].x << 16), acc[0]);
        acc[1] = fmaf(wj[jj], __uint_as_float(r[jj].x & 0xFFFF0000u), acc[1]);
        acc[2] = fmaf(wj[jj], __uint_as_float(r[jj].y << 16), acc[2]);
        acc[3] = fmaf(wj[jj], __uint_as_float(r[jj].y & 0xFFFF0000u), acc[3]);
      }
    }
    *reinterpret_cast<uint2*>(p.c_y + (size_t)t * p.ld_out + m) =
        make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
  }
}

// ---------------------------------------------------------------------------- the kernel

template <int MODE>
__global__ void __launch_bounds__(Cfg<MODE>::THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  using C = Cfg<MODE>;
  extern __shared__ __align__(1024) uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[C::STAGES];
  __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[C::ACC_BUFS];
  __shared__ __align__(8) uint64_t tempty_bar[C::ACC_BUFS];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_off[C::TABLE];
  __shared__ int s_pref[C::TABLE];
  __shared__ Sched s_sched;
  // epilogue transpose buffers: one 16-column x 32-row bf16 block per warp and output slot
  __shared__ __align__(128) __nv_bfloat16 s_stage[C::EPI_WARPS][C::NSLOT][C::CW][32];
  // down projection with the combine folded in: (token, M tile) cells this CTA owns, per unit parity
  constexpr int kOwn = (C::PAIR && C::BASE == DOWN) ? 2 * C::BN : 1;
  __shared__ int s_own[2][kOwn];
  __shared__ int s_nown[2];
  __shared__ __align__(8) uint64_t comb_bar;  // the epilogue warps meet here

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // stage ring aligned to 1024 bytes (the swizzle atom)
  const uint32_t ring = (smem_u32(dsmem) + 1023u) & ~1023u;
  uint8_t* ring_ptr = dsmem + (ring - smem_u32(dsmem));

  // ------------------------------------------------------------------ schedule
  if constexpr (!C::TOKEN_N) {
    if (threadIdx.x == 0) {
      s_sched.mt = p.M / C::MT;
      s_sched.nt = (p.Nw + C::BN - 1) / C::BN;
      s_sched.total = p.E * s_sched.mt * s_sched.nt;
      s_sched.pairs = s_sched.total;
    }
  } else {
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_off[i] = __ldg(p.offsets + i);
    __syncthreads();
    if (warp == 0) {
      // units per expert, then an inclusive scan into s_pref[1..E] (s_pref[0] = 0)
      const int per = (p.E + 31) / 32;
      const int b0 = min(lane * per, p.E), b1 = min(b0 + per, p.E);
      const int mt = p.M / C::MT;
      int local = 0;
      for (int e = b0; e < b1; ++e) {
        const int ue = ((s_off[e + 1] - s_off[e] + C::BN - 1) / C::BN) * mt;
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
        const int rem = incl % (int)gridDim.x;
        const int pairs = (C::PAIR && rem > 0 && 2 * rem <= (int)gridDim.x) ? incl - rem : incl;
        s_sched.pairs = pairs;
        s_sched.total = pairs + 2 * (incl - pairs);
        s_sched.mt = mt;
        s_sched.nt = 0;
      }
    }
  }
  __syncthreads();
  const Sched sc = s_sched;
  if ((int)blockIdx.x >= sc.total) return;  // nothing for this CTA (before any TMEM use)

  // ------------------------------------------------------------------ barriers + TMEM
  if (threadIdx.x == 0) {
    // gathered token rows: a stage's full barrier also takes one arrival per producer lane, made
    // by the hardware once that lane's row copies have landed
    const uint32_t full_count = ((C::GU || C::BASE == WGRAD13) && p.gx != nullptr) ? 33u : 1u;
    for (int s = 0; s < C::STAGES; ++s) { mbar_init(&full_bar[s], full_count); mbar_init(&empty_bar[s], 1); }
    for (int b = 0; b < C::ACC_BUFS; ++b) { mbar_init(&tfull_bar[b], 1); mbar_init(&tempty_bar[b], C::EPI_WARPS); }
    mbar_init(&drain_bar, 1);
    mbar_init(&comb_bar, C::EPI_WARPS);
    s_nown[0] = 0;
    s_nown[1] = 0;
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;

  if (warp == 0) {
    if ((C::GU || C::BASE == WGRAD13) && p.gx != nullptr) {
      // ============================================================== producer, gathered rows
      // The weight-side tiles come by TMA (lane 0).  The token-side tile is gathered from gx by
      // the whole warp with 16-byte copies, written in the 128-byte swizzled layout a tensor
      // map would produce (16-byte chunk c of row r lands at chunk c ^ (r & 7) of the row).
      // Rows past the segment and columns past the matrix are zero-filled.  Every lane then
      // arrives on the stage's full barrier through its copies' completion (cp.async arrive),
      // so the warp never waits for its own copies; the MMA warp fences the landed rows into the
      // async proxy before multiplying them.
      constexpr int NR = C::GU ? C::BN / 32 : 2;  // row offsets per lane: rows lane + 32 j
      const int g = lane >> 3, c = lane & 7;      // row group of 8 lanes; 16-byte chunk of the row
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      // element offset of buffer row p in gx, or -1 for a zero row (past the segment, bad id)
      auto row_offset = [&](int rel, int limit, int prow) -> int {
        if (rel >= limit) return -1;
        const int t = __ldg(p.gids + prow);
        if ((unsigned)t < (unsigned)p.gx_rows) return t * p.gx_ld;
        flag_status(p.status, MOE_STATUS_BAD_INDEX);
        return -1;
      };
      for (int u = blockIdx.x; u < sc.total && ok; u += gridDim.x) {
        const Unit w = decode<MODE>(u, sc, s_pref, s_off, p);
        const uint32_t tx = (uint32_t)w.na * kATile;
        int roff[NR];
        if (C::GU) {  // gate/up: the chunk's rows serve every K step of the unit
#pragma unroll
          for (int j = 0; j < NR; ++j) roff[j] = row_offset(lane + 32 * j, w.rows, w.row0 + lane + 32 * j);
        }
        for (int ks = 0; ks < w.nk; ++ks) {
          const int k0 = ks * BK;
          if (!C::GU) {  // dW1/dW3: this K step's 64 token rows
#pragma unroll
            for (int j = 0; j < NR; ++j)
              roff[j] = row_offset(k0 + lane + 32 * j, w.rows, w.row0 + k0 + lane + 32 * j);
          }
          if (!__all_sync(0xffffffffu, mbar_wait(&empty_bar[s], ph ^ 1u, &s_abort, p.status, p.wait_ns))) {
            ok = false;
            break;
          }
          if (p.withhold && u == (int)blockIdx.x && ks == 0) {  // test hook: a stage nobody fills
            if (++s == C::STAGES) { s = 0; ph ^= 1u; }
            continue;
          }
          const uint32_t a_sm = ring + s * C::STAGE_BYTES;
          const uint32_t b_sm = a_sm + C::A_BYTES;
          if (lane == 0) {
            mbar_expect_tx(&full_bar[s], tx);
            const int y = C::GU ? w.e * p.a_rows + k0 : w.row0 + k0;
            tma_load_2d(a_sm, &p.mapA0, &full_bar[s], w.m0, y);
            tma_load_2d(a_sm + kBox, &p.mapA0, &full_bar[s], w.m0 + 64, y);
            tma_load_2d(a_sm + kATile, &p.mapA1, &full_bar[s], w.m0, y);
            tma_load_2d(a_sm + kATile + kBox, &p.mapA1, &full_bar[s], w.m0 + 64, y);
          }
          // copy i moves chunk c of one row; the row's offset comes from the lane that loaded it
          if (C::GU) {
            // gate/up: row rr = 4 i + g of the chunk (K-major, one 64-row box per 64 rows), K = k0..
#pragma unroll
            for (int i = 0; i < C::BN / 4; ++i) {
              const int rr = 4 * i + g;
              const int off = __shfl_sync(0xffffffffu, roff[i >> 3], 4 * (i & 7) + g);
              if (rr < w.nmma) {
                const bool live = off >= 0;
                cp_async_16(b_sm + (rr >> 6) * kBox + (rr & 63) * 128 + ((c ^ (rr & 7)) << 4),
                            live ? p.gx + off + k0 + 8 * c : p.gx, live ? 16u : 0u);
              }
            }
          } else {
            // dW1/dW3: token row r = 4 m + g of the step (MN-major, one box per 64 columns of h)
#pragma unroll
            for (int i = 0; i < C::BN / 4; ++i) {
              const int box = i >> 4, m = i & 15, r = 4 * m + g;
              const int off = __shfl_sync(0xffffffffu, roff[m >> 3], 4 * (m & 7) + g);
              const int col = w.n0 + 64 * box;
              if (64 * box < w.ncols) {
                const bool live = off >= 0 && col < p.Nw;
                cp_async_16(b_sm + box * kBox + r * 128 + ((c ^ (r & 7)) << 4),
                            live ? p.gx + off + col + 8 * c : p.gx, live ? 16u : 0u);
              }
            }
          }
          cp_async_arrive_noinc(&full_bar[s]);
          if (++s == C::STAGES) { s = 0; ph ^= 1u; }
        }
      }
      cp_async_wait<0>();  // no copy of this warp outlives it
      if (lane == 0) {
        if (!ok || s_abort) {
          const unsigned long long t0 = globaltimer();
          while (globaltimer() - t0 < 2000000ull) {
          }
        }
      }
    } else if (lane == 0) {
      // ============================================================== TMA producer
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < sc.total && ok; u += gridDim.x) {
        const Unit w = decode<MODE>(u, sc, s_pref, s_off, p);
        const int nbB = C::TOKEN_N ? (w.nmma + 63) / 64 : C::BN / 64;
        const uint32_t tx = (uint32_t)w.na * kATile + (uint32_t)nbB * kBox;
        for (int ks = 0; ks < w.nk; ++ks) {
          if (!mbar_wait(&empty_bar[s], ph ^ 1u, &s_abort, p.status, p.wait_ns)) { ok = false; break; }
          if (p.withhold && u == (int)blockIdx.x && ks == 0) {  // test hook: a stage nobody fills
            if (++s == C::STAGES) { s = 0; ph ^= 1u; }
            continue;
          }
          mbar_expect_tx(&full_bar[s], tx);
          const uint32_t a_sm = ring + s * C::STAGE_BYTES;
          const uint32_t b_sm = a_sm + C::A_BYTES;
          const int k0 = ks * BK;
          if (C::GU || C::BASE == DOWN) {
            const int y = w.e * p.a_rows + k0;
            tma_load_2d(a_sm, &p.mapA0, &full_bar[s], w.m0, y);
            tma_load_2d(a_sm + kBox, &p.mapA0, &full_bar[s], w.m0 + 64, y);
            if (C::GU) {
              tma_load_2d(a_sm + kATile, &p.mapA1, &full_bar[s], w.m0, y);
              tma_load_2d(a_sm + kATile + kBox, &p.mapA1, &full_bar[s], w.m0 + 64, y);
            } else if (C::PAIR && w.na == 2) {
              tma_load_2d(a_sm + kATile, &p.mapA0, &full_bar[s], w.m0 + 128, y);
              tma_load_2d(a_sm + kATile + kBox, &p.mapA0, &full_bar[s], w.m0 + 192, y);
            }
            for (int j = 0; j < nbB; ++j) tma_load_2d(b_sm + j * kBox, &p.mapB0, &full_bar[s], k0, w.row0 + 64 * j);
          } else if (C::BASE == DA) {
            for (int a = 0; a < w.na; ++a)
              tma_load_2d(a_sm + a * kATile, &p.mapA0, &full_bar[s], k0, w.e * p.a_rows + w.m0 + a * BM);
            for (int j = 0; j < nbB; ++j) tma_load_2d(b_sm + j * kBox, &p.mapB0, &full_bar[s], k0, w.row0 + 64 * j);
          } else if (C::BASE == DX) {
            const bool second = k0 >= p.K;
            const int kk = second ? k0 - p.K : k0;
            for (int a = 0; a < w.na; ++a)
              tma_load_2d(a_sm + a * kATile, second ? &p.mapA1 : &p.mapA0, &full_bar[s], kk, w.e * p.a_rows + w.m0 + a * BM);
            for (int j = 0; j < nbB; ++j)
              tma_load_2d(b_sm + j * kBox, second ? &p.mapB1 : &p.mapB0, &full_bar[s], kk, w.row0 + 64 * j);
          } else {  // wgrad: K runs over the expert's token rows
            const int y = w.row0 + k0;
            tma_load_2d(a_sm, &p.mapA0, &full_bar[s], w.m0, y);
            tma_load_2d(a_sm + kBox, &p.mapA0, &full_bar[s], w.m0 + 64, y);
            if (C::BASE == WGRAD13) {
              tma_load_2d(a_sm + kATile, &p.mapA1, &full_bar[s], w.m0, y);
              tma_load_2d(a_sm + kATile + kBox, &p.mapA1, &full_bar[s], w.m0 + 64, y);
            } else if (C::MPAIR) {
              tma_load_2d(a_sm + kATile, &p.mapA0, &full_bar[s], w.m0 + 128, y);
              tma_load_2d(a_sm + kATile + kBox, &p.mapA0, &full_bar[s], w.m0 + 192, y);
            }
            for (int j = 0; j < nbB; ++j) tma_load_2d(b_sm + j * kBox, &p.mapB0, &full_bar[s], w.n0 + 64 * j, y);
          }
          if (++s == C::STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok || s_abort) {
        // give the loads already in flight (a few microseconds each) time to land
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    int s = 0;
    uint32_t ph = 0;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < sc.total && ok; u += gridDim.x, ++it) {
      const Unit w = decode<MODE>(u, sc, s_pref, s_off, p);
      const int b = it % C::ACC_BUFS;
      const uint32_t aph = (uint32_t)(it / C::ACC_BUFS) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&tempty_bar[b], aph ^ 1u, &s_abort, p.status, p.wait_ns))) { ok = false; break; }
      tc_fence_after();
      if (w.nk == 0) {  // an expert without rows (wgrad): nothing to multiply
        if (lane == 0) mbar_arrive(&tfull_bar[b]);
        continue;
      }
      const uint32_t idesc = idesc_bf16(w.nmma, C::A_MN, C::B_MN);
      const uint32_t d0 = tmem_base + (uint32_t)(b * C::NUM_A * C::BN);
      for (int ks = 0; ks < w.nk; ++ks) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[s], ph, &s_abort, p.status, p.wait_ns))) { ok = false; break; }
        if ((C::GU || C::BASE == WGRAD13) && p.gx != nullptr) {
          // gathered rows were written by cp.async (generic proxy); the MMAs read them through
          // the async proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        const uint32_t a_sm = ring + s * C::STAGE_BYTES;
        const uint32_t b_sm = a_sm + C::A_BYTES;
        int nsl = BK / 16;  // K slices of 16 to multiply in this stage
        if (!C::TOKEN_N && ks == w.nk - 1 && (w.rows & (BK - 1)) != 0) {
          // the last K step ends inside the stage: multiply only the slices that hold valid
          // token rows, and zero the rows of the last slice that belong to the next expert
          const int valid = w.rows & (BK - 1);
          nsl = (valid + 15) / 16;
          const int zrows = nsl * 16 - valid;
          if (zrows > 0) {
            const int nbox = C::NUM_A * 2 + C::BN / 64;
            for (int q = lane; q < nbox * zrows * 8; q += 32) {
              const int box = q / (zrows * 8);
              const int r = valid + (q / 8) % zrows;
              const int c16 = q % 8;
              uint4* dst = reinterpret_cast<uint4*>(ring_ptr + (a_sm - ring) + box * kBox + r * 128 + c16 * 16);
              *dst = make_uint4(0, 0, 0, 0);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
          }
        }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int a = 0; a < C::NUM_A; ++a) {
            if (a >= w.na) break;
            const uint32_t a_base = a_sm + a * kATile;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              if (kk >= nsl) break;
              uint64_t ad, bd;
              if (C::A_MN) ad = sdesc(a_base + kk * 2048, kBox, 1024);
              else ad = sdesc(a_base + kk * 32, 16, 1024);
              if (C::B_MN) bd = sdesc(b_sm + kk * 2048, kBox, 1024);
              else bd = sdesc(b_sm + kk * 32, 16, 1024);
              umma(d0 + a * C::BN, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
            }
          }
          umma_commit(&empty_bar[s]);  // the stage is free once these MMAs have read it
        }
        __syncwarp();
        if (++s == C::STAGES) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(&tfull_bar[b]);
      __syncwarp();
    }
    // make sure no MMA is still writing TMEM before the teardown
    if (lane == 0) {
      umma_commit(&drain_bar);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(&drain_bar, 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue (warps 2..)
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int cg = (warp - 2) >> 2;      // column group: chunks cg, cg + G, cg + 2G, ...
    constexpr int G = C::EPI_WARPS / 4;  // warps per lane quarter
    __nv_bfloat16 (*stg)[C::CW][32] = s_stage[warp - 2];  // this warp's transpose buffers
    int slot = 0;  // weight gradients: the transpose slot of the next tensor store
    uint32_t cph = 0;  // combine fold: phase of comb_bar
    int it = 0;
    for (int u = blockIdx.x; u < sc.total; u += gridDim.x, ++it) {
      const Unit w = decode<MODE>(u, sc, s_pref, s_off, p);
      const int b = it % C::ACC_BUFS;
      const uint32_t aph = (uint32_t)(it / C::ACC_BUFS) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull_bar[b], aph, &s_abort, p.status, p.wait_ns))) break;
      tc_fence_after();
      const uint32_t t0u = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * C::NUM_A * C::BN);
      const bool zero = (w.nk == 0);
      // output element (m, c) lives at [colbase + c][mbase + lane] (+ the expert's base for wgrad)
      const size_t colbase = C::TOKEN_N ? (size_t)w.row0 : (size_t)w.n0;
      const size_t ebase = C::TOKEN_N ? 0 : (size_t)w.e * (size_t)p.out_expert_stride;
      if constexpr (!C::TOKEN_N) {
        // weight gradients: the warp's whole share of the accumulators (dW1 then dW3, one or two
        // M tiles of dW2; 32 columns per TMEM load) goes to registers as bf16 pairs, TMEM goes
        // back to the MMA warp, and the 32 x 32 tensor stores overlap the next unit's main loop
        constexpr int NOUT = C::NUM_A;
        constexpr int NCH = C::BN / (C::CW * G);  // 32-column chunks per warp
        const int mbase = w.m0 + q * 32;
        uint32_t pk[NOUT][NCH][16];
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int c0 = C::CW * (cg + G * j);
#pragma unroll
          for (int a = 0; a < NOUT; ++a) {
            float vv[32];
            if (!zero && c0 < w.ncols) {
              tmem_ld32(t0u + a * C::BN + c0, vv);
              tmem_wait_ld();
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) vv[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[a][j][i] = pack_bf16x2(vv[2 * i], vv[2 * i + 1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[b]);
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int c0 = C::CW * (cg + G * j);
          if (c0 >= w.ncols) break;
#pragma unroll
          for (int a = 0; a < NOUT; ++a) {
            // the two slots alternate store by store; the store two back has read this one
            unsigned short* sw = reinterpret_cast<unsigned short*>(&stg[slot][0][0]);
            slot ^= 1;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              sw[(2 * i) * 32 + lane] = (unsigned short)(pk[a][j][i] & 0xFFFFu);
              sw[(2 * i + 1) * 32 + lane] = (unsigned short)(pk[a][j][i] >> 16);
            }
            __syncwarp();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
              if (C::BASE == WGRAD13)
                tma_store_2d(a == 0 ? &p.mapO0 : &p.mapO1, smem_u32(sw), mbase, w.e * p.a_rows + w.n0 + c0);
              else
                tma_store_2d(&p.mapO0, smem_u32(sw), mbase + a * BM, w.e * p.a_rows + w.n0 + c0);
              bulk_commit();
            }
          }
        }
      } else if constexpr (C::PAIR && C::BASE != DA) {
        // down projection and dX with paired M tiles write the accumulators themselves: both
        // tiles' columns (16 per TMEM load) go to registers as bf16 pairs, TMEM goes back to the
        // MMA warp, and the 16-byte stores of the token rows overlap the next unit's main loop
        constexpr int NCH = C::BN / (C::CW * G);  // 16-column chunks per warp and tile
        uint32_t pk[2][NCH][8];
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int c0 = C::CW * (cg + G * j);
          float v0[16], v1[16];
          if (!zero && c0 < w.ncols) {
            tmem_ld16(t0u + c0, v0);
            if (w.na == 2) {
              tmem_ld16(t0u + C::BN + c0, v1);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) v1[i] = 0.f;
            }
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) { v0[i] = 0.f; v1[i] = 0.f; }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            pk[0][j][i] = pack_bf16x2(v0[2 * i], v0[2 * i + 1]);
            pk[1][j][i] = pack_bf16x2(v1[2 * i], v1[2 * i + 1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[b]);
        unsigned short* sw = reinterpret_cast<unsigned short*>(&stg[0][0][0]);
#pragma unroll
        for (int mtl = 0; mtl < 2; ++mtl) {
          if (mtl >= w.na) break;
          const int mbase = w.m0 + mtl * BM + q * 32;
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            const int c0 = C::CW * (cg + G * j);
            if (c0 >= w.ncols) break;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              sw[(2 * i) * 32 + lane] = (unsigned short)(pk[mtl][j][i] & 0xFFFFu);
              sw[(2 * i + 1) * 32 + lane] = (unsigned short)(pk[mtl][j][i] >> 16);
            }
            __syncwarp();
            // four lanes cover one token row's 32 outputs (64 contiguous bytes)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int v = lane + 32 * r, ci = v >> 2, part = v & 3;
              if (c0 + ci < w.ncols) {
                const size_t o = (colbase + c0 + ci) * (size_t)p.ld_out + mbase + part * 8;
                *reinterpret_cast<uint4*>(p.out0 + o) = *reinterpret_cast<const uint4*>(sw + ci * 32 + part * 8);
              }
            }
            __syncwarp();
          }
        }
        if (C::BASE == DOWN && p.c_y != nullptr) {
          // Combine folded in.  Every epilogue thread fences its ybuf stores device-wide; after
          // the warps meet, the contributions are counted, and after they meet again the cells
          // this unit completed are summed (fold_count, fold_sum).
          const int et = (warp - 2) * 32 + lane, ew = warp - 2;
          const int par = it & 1;
          __threadfence();
          __syncwarp();
          if (lane == 0) mbar_arrive(&comb_bar);
          if (!__all_sync(0xffffffffu, mbar_wait(&comb_bar, cph, &s_abort, p.status, p.wait_ns))) break;
          cph ^= 1u;
          fold_count(&p, w.row0, w.ncols, w.na, w.m0 / BM, et, C::EPI_WARPS * 32, s_own[par], &s_nown[par]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&comb_bar);
          if (!__all_sync(0xffffffffu, mbar_wait(&comb_bar, cph, &s_abort, p.status, p.wait_ns))) break;
          cph ^= 1u;
          __threadfence();
          const int nown = s_nown[par];
          if (et == 0) s_nown[par ^ 1] = 0;  // the next unit's list; its readers are past this unit's meetings
          fold_sum(&p, s_own[par], nown, ew, C::EPI_WARPS, lane);
        }
      } else {
      // a paired unit's two M tiles go out one after the other (accumulators at t0 and t0 + BN)
      for (int mtl = 0; mtl < (C::PAIR ? w.na : 1); ++mtl) {
      const uint32_t t0 = t0u + (uint32_t)(mtl * C::BN);
      const int mbase = w.m0 + mtl * BM + q * 32;
      for (int c0 = C::CW * cg; c0 < w.ncols; c0 += C::CW * G) {
        {
        // (1) DA: start the coalesced 16-byte loads of h1, h3 for these 16 columns
        uint4 in_a[2], in_b[2];
        if (C::BASE == DA) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int v = lane + 32 * r, ci = v >> 2, part = v & 3;
            in_a[r] = make_uint4(0, 0, 0, 0);
            in_b[r] = in_a[r];
            if (c0 + ci < w.ncols) {
              const size_t o = ebase + (colbase + c0 + ci) * (size_t)p.ld_out + mbase + part * 8;
              in_a[r] = __ldg(reinterpret_cast<const uint4*>(p.in0 + o));
              in_b[r] = __ldg(reinterpret_cast<const uint4*>(p.in1 + o));
            }
          }
        }
        // (2) the accumulator columns
        float v0[16], v1[16];
        if (!zero) {
          tmem_ld16(t0 + c0, v0);
          if (C::GU) tmem_ld16(t0 + C::BN + c0, v1);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) { v0[i] = 0.f; v1[i] = 0.f; }
        }
        // (3) DA: transpose h1, h3 through shared memory to this lane's row
        float z1[16], z3[16];
        if (C::BASE == DA) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int v = lane + 32 * r, ci = v >> 2, part = v & 3;
            *reinterpret_cast<uint4*>(&stg[0][ci][part * 8]) = in_a[r];
            *reinterpret_cast<uint4*>(&stg[1][ci][part * 8]) = in_b[r];
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            z1[i] = __bfloat162float(stg[0][i][lane]);
            z3[i] = __bfloat162float(stg[1][i][lane]);
          }
          __syncwarp();  // the outputs below reuse these two slots
        }
        // (4) the epilogue math, written to shared memory as [column][m]
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (C::GU) {
            const float h1 = v0[i], h3 = v1[i];
            stg[0][i][lane] = __float2bfloat16_rn(h1);
            stg[1][i][lane] = __float2bfloat16_rn(h3);
            stg[2][i][lane] = __float2bfloat16_rn(h1 * sigmoid_bf16_epilogue(h1) * h3);
          } else if (C::BASE == DA) {
            const float sg = sigmoid_bf16_epilogue(z1[i]);
            const float da = v0[i];
            stg[0][i][lane] = __float2bfloat16_rn(da * z3[i] * sg * (1.f + z1[i] * (1.f - sg)));
            stg[1][i][lane] = __float2bfloat16_rn(da * z1[i] * sg);
          } else {
            stg[0][i][lane] = __float2bfloat16_rn(v0[i]);
          }
        }
        __syncwarp();
        // (5) 16-byte stores: four lanes cover one column's 32 rows (64 contiguous bytes)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int v = lane + 32 * r, ci = v >> 2, part = v & 3;
          if (c0 + ci < w.ncols) {
            const size_t o = ebase + (colbase + c0 + ci) * (size_t)p.ld_out + mbase + part * 8;
            if (C::GU) {
              *reinterpret_cast<uint4*>(p.out0 + o) = *reinterpret_cast<const uint4*>(&stg[0][ci][part * 8]);
              *reinterpret_cast<uint4*>(p.out1 + o) = *reinterpret_cast<const uint4*>(&stg[1][ci][part * 8]);
              *reinterpret_cast<uint4*>(p.out2 + o) = *reinterpret_cast<const uint4*>(&stg[2][ci][part * 8]);
            } else if (C::BASE == DA) {
              *reinterpret_cast<uint4*>(p.out0 + o) = *reinterpret_cast<const uint4*>(&stg[0][ci][part * 8]);
              *reinterpret_cast<uint4*>(p.out1 + o) = *reinterpret_cast<const uint4*>(&stg[1][ci][part * 8]);
            } else {
              *reinterpret_cast<uint4*>(p.out0 + o) = *reinterpret_cast<const uint4*>(&stg[0][ci][part * 8]);
            }
          }
        }
        __syncwarp();
        }
      }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[b]);
      }  // token-N
    }
  }

  // ------------------------------------------------------------------ teardown
  if (!C::TOKEN_N && warp >= 2 && lane == 0) bulk_wait_all();  // this warp's tensor stores
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

bool tc_encode_available() { return encode_fn() != nullptr; }

bool tc_make_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_cols, int box_rows,
                 bool swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


namespace {

template <int MODE>
int launch(const TcParams& p0, cudaStream_t st) {
  using C = Cfg<MODE>;
  TcParams p = p0;
  p.withhold = debug_take_withhold(&p.wait_ns) ? 1 : 0;
  const int smem = (int)(C::STAGES * C::STAGE_BYTES + 1024);
  if (cudaFuncSetAttribute(tc_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -1;
  tc_gemm_kernel<MODE><<<num_sms(), C::THREADS, smem, st>>>(p);
  count_launch(st);
  return 0;
}

TcParams blank_params() {
  TcParams p;
  memset(&p, 0, sizeof(p));
  return p;
}

}  // namespace

bool tc_supported(int dtype, int h, int f) {
  return dtype == MOE_BF16 && h % 128 == 0 && f % 128 == 0 && encode_fn() != nullptr;
}

namespace {
// The token-side operand of gate/up and dW1/dW3: the buffer's tensor map, or the gather source.
bool set_token_rows(TcParams* p, const TokenRows& xr, int Tk, int h) {
  if (xr.xbuf != nullptr) return tc_make_map(&p->mapB0, xr.xbuf, Tk, h, 64, 64);
  p->gx = static_cast<const __nv_bfloat16*>(xr.x);
  p->gids = xr.token_ids;
  p->gx_rows = xr.T;
  p->gx_ld = h;
  return xr.x != nullptr && xr.token_ids != nullptr;
}
}  // namespace

int tc_expert_ffn(TokenRows xr, const int* offsets, const void* W1, const void* W3, const void* W2, int Tk,
                  int E, int h, int f, void* ybuf, void* h1, void* h3, void* a, int* status, cudaStream_t st,
                  const CombineFold* fold) {
  if (fold != nullptr && h % 256 != 0) return -1;  // the fold lives in the paired down projection
  TcParams g = blank_params();
  bool ok = tc_make_map(&g.mapA0, W1, (long long)E * h, f, 64, 64) &&
            tc_make_map(&g.mapA1, W3, (long long)E * h, f, 64, 64) && set_token_rows(&g, xr, Tk, h);
  if (!ok) return -1;
  g.offsets = offsets; g.E = E; g.M = f; g.K = h; g.a_rows = h;
  g.out0 = static_cast<__nv_bfloat16*>(h1); g.out1 = static_cast<__nv_bfloat16*>(h3);
  g.out2 = static_cast<__nv_bfloat16*>(a); g.ld_out = f; g.status = status;
  // experts averaging more than 96 tokens: one 256-token chunk per expert in most cases
  if ((Tk > 96LL * E ? launch<GATEUP_WIDE>(g, st) : launch<GATEUP>(g, st)) != 0) return -1;

  TcParams d = blank_params();
  ok = tc_make_map(&d.mapA0, W2, (long long)E * f, h, 64, 64) && tc_make_map(&d.mapB0, a, Tk, f, 64, 64);
  if (!ok) return -1;
  d.offsets = offsets; d.E = E; d.M = h; d.K = f; d.a_rows = f;
  d.out0 = static_cast<__nv_bfloat16*>(ybuf); d.ld_out = h; d.status = status;
  if (fold != nullptr) {
    d.c_y = static_cast<__nv_bfloat16*>(fold->y);
    d.c_tok = fold->token_ids; d.c_slot = fold->slot_of; d.c_w = fold->topk_w; d.c_cnt = fold->cnt;
    d.c_T = fold->T; d.c_k = fold->k; d.c_mt = h / BM;
    if (cudaMemsetAsync(fold->cnt, 0, (size_t)fold->T * (h / BM) * sizeof(int), st) != cudaSuccess) return -1;
  }
  return h % 256 == 0 ? launch<DOWN_PAIR>(d, st) : launch<DOWN>(d, st);
}

int tc_expert_ffn_bwd(const void* dybuf, TokenRows xr, const void* h1, const void* h3, const void* a,
                      const int* offsets, const void* W1, const void* W3, const void* W2, int Tk, int E, int h,
                      int f, void* dxbuf, void* dW1, void* dW3, void* dW2, void* dh1, void* dh3, int* status,
                      cudaStream_t st) {
  // dA^T = W2[e] dY^T, fused with the SwiGLU backward -> dh1, dh3
  TcParams da = blank_params();
  bool ok = tc_make_map(&da.mapA0, W2, (long long)E * f, h, 64, 128) && tc_make_map(&da.mapB0, dybuf, Tk, h, 64, 64);
  if (!ok) return -1;
  da.offsets = offsets; da.E = E; da.M = f; da.K = h; da.a_rows = f;
  da.out0 = static_cast<__nv_bfloat16*>(dh1); da.out1 = static_cast<__nv_bfloat16*>(dh3);
  da.in0 = static_cast<const __nv_bfloat16*>(h1); da.in1 = static_cast<const __nv_bfloat16*>(h3);
  da.ld_out = f; da.status = status;
  if ((f % 256 == 0 ? launch<DA_PAIR>(da, st) : launch<DA>(da, st)) != 0) return -1;

  // dX^T = W1[e] dh1^T + W3[e] dh3^T
  TcParams dx = blank_params();
  ok = tc_make_map(&dx.mapA0, W1, (long long)E * h, f, 64, 128) && tc_make_map(&dx.mapA1, W3, (long long)E * h, f, 64, 128) &&
       tc_make_map(&dx.mapB0, dh1, Tk, f, 64, 64) && tc_make_map(&dx.mapB1, dh3, Tk, f, 64, 64);
  if (!ok) return -1;
  dx.offsets = offsets; dx.E = E; dx.M = h; dx.K = f; dx.a_rows = h;
  dx.out0 = static_cast<__nv_bfloat16*>(dxbuf); dx.ld_out = h; dx.status = status;
  if ((h % 256 == 0 ? launch<DX_PAIR>(dx, st) : launch<DX>(dx, st)) != 0) return -1;

  // dW1[e]^T = dh1^T X, dW3[e]^T = dh3^T X  (stored as dW1[e][h][f])
  TcParams w13 = blank_params();
  ok = tc_make_map(&w13.mapA0, dh1, Tk, f, 64, 64) && tc_make_map(&w13.mapA1, dh3, Tk, f, 64, 64) &&
       set_token_rows(&w13, xr, Tk, h);
  if (!ok) return -1;
  ok = tc_make_map(&w13.mapO0, dW1, (long long)E * h, f, 32, Cfg<WGRAD13>::CW, false) &&
       tc_make_map(&w13.mapO1, dW3, (long long)E * h, f, 32, Cfg<WGRAD13>::CW, false);
  if (!ok) return -1;
  w13.offsets = offsets; w13.E = E; w13.M = f; w13.Nw = h; w13.a_rows = h;
  w13.out0 = static_cast<__nv_bfloat16*>(dW1); w13.out1 = static_cast<__nv_bfloat16*>(dW3);
  w13.ld_out = f; w13.out_expert_stride = (long long)h * f; w13.status = status;
  if ((h % 256 == 0 ? launch<WGRAD13_WIDE>(w13, st) : launch<WGRAD13>(w13, st)) != 0) return -1;

  // dW2[e]^T = dY^T a  (stored as dW2[e][f][h])
  TcParams w2 = blank_params();
  ok = tc_make_map(&w2.mapA0, dybuf, Tk, h, 64, 64) && tc_make_map(&w2.mapB0, a, Tk, f, 64, 64);
  if (!ok) return -1;
  ok = tc_make_map(&w2.mapO0, dW2, (long long)E * f, h, 32, Cfg<WGRAD2>::CW, false);
  if (!ok) return -1;
  w2.offsets = offsets; w2.E = E; w2.M = h; w2.Nw = f; w2.a_rows = f;
  w2.out0 = static_cast<__nv_bfloat16*>(dW2); w2.ld_out = h; w2.out_expert_stride = (long long)f * h;
  w2.status = status;
  return h % 256 == 0 ? launch<WGRAD2_PAIR>(w2, st) : launch<WGRAD2>(w2, st);
}

}  // namespace moe
