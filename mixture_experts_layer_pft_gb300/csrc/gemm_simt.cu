// SIMT grouped GEMM engine: fp32 FFMA with fp32 accumulation, for both element types.
//
// It serves the fp32 layer (no TF32 anywhere: every product is an fp32 FMA), the router
// GEMMs in every precision (gating is fp32), and any bf16 shape the tensor-core engine does
// not take.  A 256-thread CTA computes a 128x128 tile of C, 8x8 per thread, from 128x8 / 8x128
// operand tiles double-buffered in shared memory.
//
// Two grouping modes over the padding-free buffer (segments [offsets[g], offsets[g+1])):
//   ROWS: C_g[rows of segment g, N] = A_g[rows, K] * B_g  -- B_g is expert g's weight matrix,
//         stored [K,N] or, with TRANS_B, [N,K].  Used for the expert FFN forward, the dgrad
//         and the router GEMMs (one group).  Optionally two K segments are concatenated
//         (KCAT: C = A0*B0 + A1*B1, the dX = dh1*W1^T + dh3*W3^T of the backward).
//   KSEG: C_g[M,N] = A_seg^T * B_seg, K = the segment's rows -- the weight gradients
//         (A, B stored [rows, M] / [rows, N]).  An empty segment writes zeros.
// DUAL computes two products that share A (C = A*B0, C2 = A*B1) for the SwiGLU pair.
// SPLIT-K (router GEMMs, whose N = E is small): gridDim.z CTAs share one output tile, each
// over a contiguous slice of K, and write fp32 partials; splitk_reduce_kernel then adds the
// slices in a fixed order (and the bias), so the result does not depend on scheduling.
#include <string.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int BM = 128, BN = 128, NT = 256;
// K depth of one shared-memory tile: BK for the single-product kernels (the two-product DUAL
// ones stay at 8, which keeps their three double-buffered tiles under 48 KB of static shared
// memory).  Each thread loads KT/2 consecutive elements of each operand per tile.
#ifndef MOE_SIMT_BK
#define MOE_SIMT_BK 16
#endif
// Single-product kernels fit two CTAs per SM (at most 128 registers); the DUAL ones need more.
#ifndef MOE_SIMT_MINB
#define MOE_SIMT_MINB 2
#endif
constexpr int BK = MOE_SIMT_BK;

// EPI_SWIGLU_H3: the product is h3; with h1 read back from X1 it also writes a = silu(h1) * h3.
enum Epi { EPI_STORE = 0, EPI_BIAS = 1, EPI_SWIGLU = 2, EPI_DSWIGLU = 3, EPI_STORE2 = 4, EPI_SWIGLU_H3 = 5 };

struct Args {
  const void* A0;
  const void* A1;     // KCAT: A of the second K segment (nullptr: none)
  const void* B0;
  const void* B1;     // KCAT: B of the second K segment; DUAL: the second B
  long long strideB;  // elements between consecutive groups' B (ROWS mode)
  int lda, ldb;
  int K0, K1;         // ROWS: K of the two segments (K1 = 0 without KCAT); KSEG: K0 = rows when no offsets
  int M;              // ROWS without offsets: rows; KSEG: rows of C
  int N;
  const int* offsets;  // [G+1] or nullptr (one group)
  int G;
  void* C;
  void* C2;
  void* C3;
  int ldc;
  long long strideC;  // KSEG: elements between consecutive groups' C
  const void* X1;     // DSWIGLU: stored h1
  const void* X2;     // DSWIGLU: stored h3
  const float* bias;  // EPI_BIAS: [N]
  int splits;         // > 1: write fp32 partials [splits][rows][N] to `partial`
  float* partial;
};

__device__ __forceinline__ float4 zero4() { return make_float4(0.f, 0.f, 0.f, 0.f); }

template <typename TA, typename TB, typename TC, bool KSEG, bool TRANS_B, bool DUAL, int EPI>
__global__ void __launch_bounds__(NT, DUAL ? 1 : MOE_SIMT_MINB) simt_gemm_kernel(const Args args) {
  constexpr int KT = DUAL ? 8 : BK;  // K depth of a tile
  constexpr int VPT = KT / 2;        // elements of each operand a thread loads per tile
  constexpr int NL = VPT / 4;        // 4-element loads per operand
  constexpr int TPR = NT / KT;       // threads per k-row of a [KT x 128] tile
  __shared__ __align__(16) float As[2][KT][BM];
  __shared__ __align__(16) float Bs[2][KT][BN];
  __shared__ __align__(16) float Bs2[DUAL ? 2 : 1][KT][DUAL ? BN : 4];
  __shared__ int s_g, s_mt;

  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;

  // ------------------------------------------------------------------ tile decode
  int g = 0, mt = 0;
  if (KSEG) {
    const int mtiles = (args.M + BM - 1) / BM;
    g = blockIdx.x / mtiles;
    mt = blockIdx.x % mtiles;
  } else if (args.offsets == nullptr) {
    mt = blockIdx.x;
  } else {
    if (tid < kWarp) {
      const int lane = tid;
      if (lane == 0) s_g = -1;
      __syncwarp();
      const int G = args.G;
      const int per = (G + kWarp - 1) / kWarp;
      const int b0 = min(lane * per, G), b1 = min(b0 + per, G);
      int local = 0;
      for (int q = b0; q < b1; ++q) {
        const int n = __ldg(args.offsets + q + 1) - __ldg(args.offsets + q);
        local += (n + BM - 1) / BM;
      }
      int incl = local;
#pragma unroll
      for (int o = 1; o < kWarp; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int bx = blockIdx.x;
      int run = incl - local;
      if (bx >= run && bx < incl) {
        for (int q = b0; q < b1; ++q) {
          const int n = __ldg(args.offsets + q + 1) - __ldg(args.offsets + q);
          const int tq = (n + BM - 1) / BM;
          if (bx < run + tq) { s_g = q; s_mt = bx - run; break; }
          run += tq;
        }
      }
    }
    __syncthreads();
    g = s_g;
    mt = s_mt;
    if (g < 0) return;  // beyond the last tile (the grid is an upper bound)
  }

  const int n0 = blockIdx.y * BN;
  const int N = args.N;
  // ROWS: rows [row0, row0 + rows_valid) of the buffer; KSEG: C rows [m0, m0+BM), K range [kb, ke)
  size_t row0 = 0;
  int rows_valid = 0, m0 = 0, kb = 0, ke = 0, Ktot = 0;
  if (KSEG) {
    m0 = mt * BM;
    kb = args.offsets ? __ldg(args.offsets + g) : 0;
    ke = args.offsets ? __ldg(args.offsets + g + 1) : args.K0;
    Ktot = ke - kb;
  } else {
    const int seg_beg = args.offsets ? __ldg(args.offsets + g) : 0;
    const int seg_end = args.offsets ? __ldg(args.offsets + g + 1) : args.M;
    row0 = (size_t)seg_beg + (size_t)mt * BM;
    rows_valid = min(BM, seg_end - (int)row0);
    Ktot = args.K0 + args.K1;
  }
  // this CTA's slice of K (all of it without split-K); slices are multiples of BK
  int kbeg = 0, kend = Ktot;
  if (args.splits > 1) {
    const int per = (((Ktot + args.splits - 1) / args.splits) + KT - 1) / KT * KT;
    kbeg = min(Ktot, (int)blockIdx.z * per);
    kend = min(Ktot, kbeg + per);
  }
  const TA* A0 = static_cast<const TA*>(args.A0);
  const TA* A1 = static_cast<const TA*>(args.A1);
  const TB* B0 = static_cast<const TB*>(args.B0);
  const TB* B1 = static_cast<const TB*>(args.B1);
  if (!KSEG && args.offsets) {
    B0 += (size_t)g * args.strideB;
    if (B1) B1 += (size_t)g * args.strideB;
  }

  // ------------------------------------------------------------------ tile loaders
  // Tiles stored along K in memory ([rows, K]: the A rows, or B with TRANS_B) are read by two
  // threads per row, VPT consecutive k each, and transposed into shared memory as [k][row].
  // Tiles stored along M / N ([K, cols]: KSEG operands, B without TRANS_B) are read by TPR
  // threads per k-row, VPT consecutive columns each.
  float4 ra[NL], rb[NL], rb2[DUAL ? NL : 1];
  auto load_tiles = [&](int k0) {
    if (KSEG) {
      const int kr = tid / TPR, c = (tid % TPR) * VPT;
      const int tok = kb + k0 + kr;
      const bool kv = tok < ke && k0 + kr < kend;
#pragma unroll
      for (int q = 0; q < NL; ++q) {
        const int cc = c + 4 * q;
        ra[q] = (kv && m0 + cc < args.M) ? load4(A0 + (size_t)tok * args.lda + m0 + cc) : zero4();
        const bool nv = kv && n0 + cc < N;
        rb[q] = nv ? load4(B0 + (size_t)tok * args.ldb + n0 + cc) : zero4();
        if (DUAL) rb2[q] = nv ? load4(B1 + (size_t)tok * args.ldb + n0 + cc) : zero4();
      }
    } else {
      // KCAT: k < K0 reads (A0, B0) at k, k >= K0 reads (A1, B1) at k - K0.  K0 is a multiple
      // of 4, so each 4-element load lies in one segment (a tile may straddle the two).
      const bool kcat = A1 != nullptr;
      {
        const int r = tid >> 1, kc = (tid & 1) * VPT;
#pragma unroll
        for (int q = 0; q < NL; ++q) {
          const int ka = k0 + kc + 4 * q;
          const bool s1 = kcat && ka >= args.K0;
          const bool v = r < rows_valid && ka < kend;
          ra[q] = v ? load4((s1 ? A1 : A0) + (row0 + r) * (size_t)args.lda + (s1 ? ka - args.K0 : ka)) : zero4();
        }
      }
      if (TRANS_B) {  // B stored [N, ldb]
        const int n = tid >> 1, kc = (tid & 1) * VPT;
#pragma unroll
        for (int q = 0; q < NL; ++q) {
          const int ka = k0 + kc + 4 * q;
          const bool s1 = kcat && ka >= args.K0;
          const int kl = s1 ? ka - args.K0 : ka;
          const bool v = n0 + n < N && ka < kend;
          rb[q] = v ? load4((s1 ? B1 : B0) + (size_t)(n0 + n) * args.ldb + kl) : zero4();
          if (DUAL) rb2[q] = v ? load4(B1 + (size_t)(n0 + n) * args.ldb + kl) : zero4();
        }
      } else {  // B stored [K, ldb]
        const int kr = tid / TPR, c = (tid % TPR) * VPT;
        const int ka = k0 + kr;
        const bool s1 = kcat && ka >= args.K0;
        const int kl = s1 ? ka - args.K0 : ka;
#pragma unroll
        for (int q = 0; q < NL; ++q) {
          const bool v = ka < kend && n0 + c + 4 * q < N;
          rb[q] = v ? load4((s1 ? B1 : B0) + (size_t)kl * args.ldb + n0 + c + 4 * q) : zero4();
          if (DUAL) rb2[q] = v ? load4(B1 + (size_t)kl * args.ldb + n0 + c + 4 * q) : zero4();
        }
      }
    }
  };
  auto store_tiles = [&](int buf) {
    if (KSEG) {
      const int kr = tid / TPR, c = (tid % TPR) * VPT;
#pragma unroll
      for (int q = 0; q < NL; ++q) {
        *reinterpret_cast<float4*>(&As[buf][kr][c + 4 * q]) = ra[q];
        *reinterpret_cast<float4*>(&Bs[buf][kr][c + 4 * q]) = rb[q];
        if (DUAL) *reinterpret_cast<float4*>(&Bs2[buf][kr][c + 4 * q]) = rb2[q];
      }
    } else {
      {
        const int r = tid >> 1, kc = (tid & 1) * VPT;
#pragma unroll
        for (int q = 0; q < NL; ++q) {
          As[buf][kc + 4 * q + 0][r] = ra[q].x; As[buf][kc + 4 * q + 1][r] = ra[q].y;
          As[buf][kc + 4 * q + 2][r] = ra[q].z; As[buf][kc + 4 * q + 3][r] = ra[q].w;
        }
      }
      if (TRANS_B) {
        const int n = tid >> 1, kc = (tid & 1) * VPT;
#pragma unroll
        for (int q = 0; q < NL; ++q) {
          Bs[buf][kc + 4 * q + 0][n] = rb[q].x; Bs[buf][kc + 4 * q + 1][n] = rb[q].y;
          Bs[buf][kc + 4 * q + 2][n] = rb[q].z; Bs[buf][kc + 4 * q + 3][n] = rb[q].w;
          if (DUAL) {
            Bs2[buf][kc + 4 * q + 0][n] = rb2[q].x; Bs2[buf][kc + 4 * q + 1][n] = rb2[q].y;
            Bs2[buf][kc + 4 * q + 2][n] = rb2[q].z; Bs2[buf][kc + 4 * q + 3][n] = rb2[q].w;
          }
        }
      } else {
        const int kr = tid / TPR, c = (tid % TPR) * VPT;
#pragma unroll
        for (int q = 0; q < NL; ++q) {
          *reinterpret_cast<float4*>(&Bs[buf][kr][c + 4 * q]) = rb[q];
          if (DUAL) *reinterpret_cast<float4*>(&Bs2[buf][kr][c + 4 * q]) = rb2[q];
        }
      }
    }
  };

  // ------------------------------------------------------------------ main loop
  float acc[8][8];
  float acc2[DUAL ? 8 : 1][DUAL ? 8 : 1];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  if (DUAL) {
#pragma unroll
    for (int i = 0; i < (DUAL ? 8 : 1); ++i)
#pragma unroll
      for (int j = 0; j < (DUAL ? 8 : 1); ++j) acc2[i][j] = 0.f;
  }

  const int ntiles = (kend - kbeg + KT - 1) / KT;
  if (ntiles > 0) {
    load_tiles(kbeg);
    store_tiles(0);
    __syncthreads();
    for (int kt = 0; kt < ntiles; ++kt) {
      const int buf = kt & 1;
      if (kt + 1 < ntiles) load_tiles(kbeg + (kt + 1) * KT);
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        float a[8], b[8];
        const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
        const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
        const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
        const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
        a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
        a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
        b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
        b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        if (DUAL) {
          float c[8];
          const float4 c0 = *reinterpret_cast<const float4*>(&Bs2[buf][kk][tx * 4]);
          const float4 c1 = *reinterpret_cast<const float4*>(&Bs2[buf][kk][64 + tx * 4]);
          c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
          c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
#pragma unroll
          for (int i = 0; i < (DUAL ? 8 : 1); ++i)
#pragma unroll
            for (int j = 0; j < (DUAL ? 8 : 1); ++j) acc2[i][j] = fmaf(a[i], c[j], acc2[i][j]);
        }
      }
      if (kt + 1 < ntiles) store_tiles(buf ^ 1);
      __syncthreads();
    }
  }

  // ------------------------------------------------------------------ epilogue
  TC* C = static_cast<TC*>(args.C);
  TC* C2 = static_cast<TC*>(args.C2);
  TC* C3 = static_cast<TC*>(args.C3);
  if (KSEG) {
    C += (size_t)g * args.strideC;
    if (C2) C2 += (size_t)g * args.strideC;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = (i < 4) ? ty * 4 + i : 64 + ty * 4 + (i - 4);
    size_t crow;
    if (KSEG) {
      if (m0 + m >= args.M) continue;
      crow = (size_t)(m0 + m);
    } else {
      if (m >= rows_valid) continue;
      crow = row0 + m;
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int n = n0 + hh * 64 + tx * 4;
      if (n >= N) continue;
      const size_t off = crow * (size_t)args.ldc + n;
      float4 v = make_float4(acc[i][hh * 4 + 0], acc[i][hh * 4 + 1], acc[i][hh * 4 + 2], acc[i][hh * 4 + 3]);
      if (args.splits > 1) {
        *reinterpret_cast<float4*>(args.partial + ((size_t)blockIdx.z * args.M + crow) * args.N + n) = v;
      } else if (EPI == EPI_STORE) {
        store4(C + off, v);
      } else if (EPI == EPI_BIAS) {
        const float4 b = *reinterpret_cast<const float4*>(args.bias + n);
        v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
        store4(C + off, v);
      } else if (EPI == EPI_SWIGLU || EPI == EPI_STORE2) {
        const int ii = DUAL ? i : 0;
        const int jb = DUAL ? hh * 4 : 0;
        const float4 u = make_float4(acc2[ii][jb], acc2[ii][DUAL ? jb + 1 : 0],
                                     acc2[ii][DUAL ? jb + 2 : 0], acc2[ii][DUAL ? jb + 3 : 0]);
        store4(C + off, v);
        store4(C2 + off, u);
        if (EPI == EPI_SWIGLU) {
          float4 a;
          a.x = v.x * sigmoidf_(v.x) * u.x;
          a.y = v.y * sigmoidf_(v.y) * u.y;
          a.z = v.z * sigmoidf_(v.z) * u.z;
          a.w = v.w * sigmoidf_(v.w) * u.w;
          store4(C3 + off, a);
        }
      } else if (EPI == EPI_SWIGLU_H3) {
        const float4 z1 = load4(static_cast<const TC*>(args.X1) + off);
        float4 a;
        a.x = z1.x * sigmoidf_(z1.x) * v.x;
        a.y = z1.y * sigmoidf_(z1.y) * v.y;
        a.z = z1.z * sigmoidf_(z1.z) * v.z;
        a.w = z1.w * sigmoidf_(z1.w) * v.w;
        store4(C + off, v);
        store4(C2 + off, a);
      } else if (EPI == EPI_DSWIGLU) {
        const float4 z1 = load4(static_cast<const TC*>(args.X1) + off);
        const float4 z3 = load4(static_cast<const TC*>(args.X2) + off);
        float4 d1, d3;
        float s;
        s = sigmoidf_(z1.x); d1.x = v.x * z3.x * s * (1.f + z1.x * (1.f - s)); d3.x = v.x * z1.x * s;
        s = sigmoidf_(z1.y); d1.y = v.y * z3.y * s * (1.f + z1.y * (1.f - s)); d3.y = v.y * z1.y * s;
        s = sigmoidf_(z1.z); d1.z = v.z * z3.z * s * (1.f + z1.z * (1.f - s)); d3.z = v.z * z1.z * s;
        s = sigmoidf_(z1.w); d1.w = v.w * z3.w * s * (1.f + z1.w * (1.f - s)); d3.w = v.w * z1.w * s;
        store4(C + off, d1);
        store4(C2 + off, d3);
      }
    }
  }
}

// out[r][n] = sum_{z ascending} partial[z][r][n] (+ bias[n]), fp32.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ partial, int splits,
                                                            long long count, int N,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ out) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (long long)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int z = 0; z < splits; ++z) s += __ldg(partial + (size_t)z * count + i);
    if (bias) s += __ldg(bias + (int)(i % N));
    out[i] = s;
  }
}

template <typename TA, typename TB, typename TC, bool KSEG, bool TRANS_B, bool DUAL, int EPI>
void run(const Args& a, cudaStream_t st) {
  dim3 grid;
  if (KSEG) {
    grid.x = (unsigned)(a.G * ((a.M + BM - 1) / BM));
  } else if (a.offsets == nullptr) {
    grid.x = (unsigned)((a.M + BM - 1) / BM);
  } else {
    long long rows = 0;  // upper bound on sum_g ceil(n_g / BM): floor(Tk / BM) + G
    rows = a.M / BM + a.G;
    grid.x = (unsigned)rows;
  }
  grid.y = (unsigned)((a.N + BN - 1) / BN);
  grid.z = (unsigned)(a.splits > 1 ? a.splits : 1);
  if (grid.x == 0 || grid.y == 0) return;
  simt_gemm_kernel<TA, TB, TC, KSEG, TRANS_B, DUAL, EPI><<<grid, NT, 0, st>>>(a);
  count_launch(st);
  if (a.splits > 1)
    launch_splitk_reduce(a.partial, a.splits, (long long)a.M * a.N, a.N, EPI == EPI_BIAS ? a.bias : nullptr,
                         static_cast<float*>(a.C), st);
}

Args blank() {
  Args a;
  memset(&a, 0, sizeof(a));
  return a;
}

template <typename T>
void expert_ffn_t(const void* xbuf, const int* offsets, const void* W1, const void* W3,
                  const void* W2, int Tk, int E, int h, int f, void* ybuf, void* h1, void* h3,
                  void* a, cudaStream_t st) {
  Args g1 = blank();
  g1.A0 = xbuf; g1.lda = h; g1.K0 = h;
  g1.B0 = W1; g1.B1 = W3; g1.ldb = f; g1.strideB = (long long)h * f;
  g1.M = Tk; g1.N = f; g1.offsets = offsets; g1.G = E;
  g1.C = h1; g1.C2 = h3; g1.C3 = a; g1.ldc = f;
  if (std::is_same<T, float>::value && (long long)Tk * f >= (1LL << 22)) {
    // fp32 at scale: two single-product GEMMs (16-deep tiles, two CTAs per SM) beat the
    // two-product one (the long-sequence layer's gate/up: 34 -> 41 TFLOP/s); h1 is stored
    // exactly, so a = silu(h1) * h3 from the stored h1 is the same value.  Small problems keep
    // one launch.
    g1.B1 = nullptr; g1.C2 = nullptr; g1.C3 = nullptr;
    run<T, T, T, false, false, false, EPI_STORE>(g1, st);
    Args g3 = g1;
    g3.B0 = W3; g3.C = h3; g3.C2 = a; g3.X1 = h1;
    run<T, T, T, false, false, false, EPI_SWIGLU_H3>(g3, st);
  } else {
    run<T, T, T, false, false, true, EPI_SWIGLU>(g1, st);
  }
  Args g2 = blank();
  g2.A0 = a; g2.lda = f; g2.K0 = f;
  g2.B0 = W2; g2.ldb = h; g2.strideB = (long long)f * h;
  g2.M = Tk; g2.N = h; g2.offsets = offsets; g2.G = E;
  g2.C = ybuf; g2.ldc = h;
  run<T, T, T, false, false, false, EPI_STORE>(g2, st);
}

template <typename T>
void expert_ffn_bwd_t(const void* dybuf, const void* xbuf, const void* h1, const void* h3,
                      const void* a, const int* offsets, const void* W1, const void* W3,
                      const void* W2, int Tk, int E, int h, int f, void* dxbuf, void* dW1,
                      void* dW3, void* dW2, void* dh1, void* dh3, cudaStream_t st) {
  // dA = dY W2^T (W2[e] stored [f,h] = [N,K]) fused with the SwiGLU backward
  Args da = blank();
  da.A0 = dybuf; da.lda = h; da.K0 = h;
  da.B0 = W2; da.ldb = h; da.strideB = (long long)f * h;
  da.M = Tk; da.N = f; da.offsets = offsets; da.G = E;
  da.C = dh1; da.C2 = dh3; da.ldc = f; da.X1 = h1; da.X2 = h3;
  run<T, T, T, false, true, false, EPI_DSWIGLU>(da, st);
  // dW1[e] = X^T dh1, dW3[e] = X^T dh3 (K = the expert's rows).  It runs before dX: the gathered
  // backward passes its token rows in dxbuf, which dX then overwrites.
  Args w13 = blank();
  w13.A0 = xbuf; w13.lda = h; w13.M = h;
  w13.B0 = dh1; w13.B1 = dh3; w13.ldb = f; w13.N = f;
  w13.offsets = offsets; w13.G = E;
  w13.C = dW1; w13.C2 = dW3; w13.ldc = f; w13.strideC = (long long)h * f;
  run<T, T, T, true, false, true, EPI_STORE2>(w13, st);
  // dX = dh1 W1^T + dh3 W3^T (W1[e] stored [h,f] = [N,K])
  Args dx = blank();
  dx.A0 = dh1; dx.A1 = dh3; dx.lda = f; dx.K0 = f; dx.K1 = f;
  dx.B0 = W1; dx.B1 = W3; dx.ldb = f; dx.strideB = (long long)h * f;
  dx.M = Tk; dx.N = h; dx.offsets = offsets; dx.G = E;
  dx.C = dxbuf; dx.ldc = h;
  run<T, T, T, false, true, false, EPI_STORE>(dx, st);
  // dW2[e] = a^T dY
  Args w2 = blank();
  w2.A0 = a; w2.lda = f; w2.M = f;
  w2.B0 = dybuf; w2.ldb = h; w2.N = h;
  w2.offsets = offsets; w2.G = E;
  w2.C = dW2; w2.ldc = h; w2.strideC = (long long)f * h;
  run<T, T, T, true, false, false, EPI_STORE>(w2, st);
}

}  // namespace

void launch_splitk_reduce(const float* partial, int splits, long long count, int N, const float* bias,
                          float* out, cudaStream_t st) {
  const int blocks = (int)std::min<long long>((count + 255) / 256, 4096);
  splitk_reduce_kernel<<<blocks, 256, 0, st>>>(partial, splits, count, N, bias, out);
  count_launch(st);
}

// K slices for a router GEMM with an M x N output and K-long sums (one CTA per SM; 152 SMs):
// at least 128 of K per slice, and the count whose last wave of CTAs is fullest among those
// giving two waves or more (fewer slices on ties).  The same count sizes the workspace.
int router_splits(int M, int N, int K) {
  constexpr int kSms = 152;
  const long long base = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int smax = std::max(1, std::min(64, K / 128));
  int best = 1;
  double best_score = -1.0;
  for (int sp = 1; sp <= smax; ++sp) {
    const long long ctas = base * sp;
    const long long waves = (ctas + kSms - 1) / kSms;
    double score = (double)ctas / (double)(waves * kSms);  // fill of the waves
    if (ctas < 2 * kSms) score *= (double)ctas / (2.0 * kSms);
    if (score > best_score + 1e-9) { best_score = score; best = sp; }
  }
  return best;
}

void simt_router_logits(int dtype, const void* x, const float* Wg, const float* bias, int T, int h,
                        int E, float* logits, float* partial, cudaStream_t st) {
  Args a = blank();
  a.A0 = x; a.lda = h; a.K0 = h;
  a.B0 = Wg; a.ldb = E;
  a.M = T; a.N = E; a.G = 1;
  a.C = logits; a.ldc = E; a.bias = bias;
  a.splits = router_splits(T, E, h);
  a.partial = partial;
  if (dtype == MOE_BF16) {
    if (bias) run<__nv_bfloat16, float, float, false, false, false, EPI_BIAS>(a, st);
    else run<__nv_bfloat16, float, float, false, false, false, EPI_STORE>(a, st);
  } else {
    if (bias) run<float, float, float, false, false, false, EPI_BIAS>(a, st);
    else run<float, float, float, false, false, false, EPI_STORE>(a, st);
  }
}

void simt_router_dwg(int dtype, const void* x, const float* d_logits, int T, int h, int E,
                     float* dWg, float* partial, cudaStream_t st) {
  Args a = blank();
  a.A0 = x; a.lda = h; a.M = h;
  a.B0 = d_logits; a.ldb = E; a.N = E;
  a.K0 = T; a.G = 1;
  a.C = dWg; a.ldc = E;
  a.splits = router_splits(h, E, T);
  a.partial = partial;
  if (dtype == MOE_BF16) run<__nv_bfloat16, float, float, true, false, false, EPI_STORE>(a, st);
  else run<float, float, float, true, false, false, EPI_STORE>(a, st);
}

void simt_router_dx(const float* d_logits, const float* Wg, int T, int h, int E, float* dx,
                    cudaStream_t st) {
  Args a = blank();
  a.A0 = d_logits; a.lda = E; a.K0 = E;
  a.B0 = Wg; a.ldb = E;  // Wg [h,E] read as [N=h, K=E]
  a.M = T; a.N = h; a.G = 1;
  a.C = dx; a.ldc = h;
  run<float, float, float, false, true, false, EPI_STORE>(a, st);
}

void simt_expert_ffn(int dtype, const void* xbuf, const int* offsets, const void* W1,
                     const void* W3, const void* W2, int Tk, int E, int h, int f, void* ybuf,
                     void* h1, void* h3, void* a, cudaStream_t st) {
  if (dtype == MOE_BF16)
    expert_ffn_t<__nv_bfloat16>(xbuf, offsets, W1, W3, W2, Tk, E, h, f, ybuf, h1, h3, a, st);
  else expert_ffn_t<float>(xbuf, offsets, W1, W3, W2, Tk, E, h, f, ybuf, h1, h3, a, st);
}

void simt_expert_ffn_bwd(int dtype, const void* dybuf, const void* xbuf, const void* h1,
                         const void* h3, const void* a, const int* offsets, const void* W1,
                         const void* W3, const void* W2, int Tk, int E, int h, int f, void* dxbuf,
                         void* dW1, void* dW3, void* dW2, void* dh1, void* dh3, cudaStream_t st) {
  if (dtype == MOE_BF16)
    expert_ffn_bwd_t<__nv_bfloat16>(dybuf, xbuf, h1, h3, a, offsets, W1, W3, W2, Tk, E, h, f,
                                    dxbuf, dW1, dW3, dW2, dh1, dh3, st);
  else expert_ffn_bwd_t<float>(dybuf, xbuf, h1, h3, a, offsets, W1, W3, W2, Tk, E, h, f, dxbuf,
                               dW1, dW3, dW2, dh1, dh3, st);
}

}  // namespace moe
