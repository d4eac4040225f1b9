// Router GEMMs on the tensor cores with fp32-faithful sums (sm_103a: tcgen05 + TMEM + TMA).
//
// Gating is an fp32 computation: logits = x Wg (+ bias), and in the backward dWg = x^T dL and
// dx = dL Wg^T, with x in bf16 or fp32 and Wg, dL in fp32.  Every fp32 operand is first split exactly into
// three bf16 planes, v = v0 + v1 + v2 with v0 = bf16(v), v1 = bf16(v - v0), v2 = v - v0 - v1, so
// that every product of two planes is exact in fp32 and the operand products the layer needs are
// sums of plane products:
//   x w      = x w0 + x w1 + x w2                             (bf16 x: one plane; fp32 x is split
//                                                              too and takes the six-term sum below)
//   a b      = a0 b0 + a0 b1 + a1 b0 + a0 b2 + a1 b1 + a2 b0   (both fp32; the dropped terms
//                                                              a1 b2, a2 b1, a2 b2 are below 2^-32
//                                                              of the product)
// The tensor core adds into its fp32 accumulator with truncation, so the error of a TMEM sum grows
// with the number of MMA steps that feed it.  Two accumulators keep the leading product (x w0, or
// a0 b0) apart from the small ones, and every 256 of K the epilogue drains both into fp32
// registers with round-to-nearest adds: no truncated chain is longer than 16 MMA steps.
//
//   mode   C [M x N] fp32     A (M x K)                           B (N x K)
//   FWD    logits [T x E]     x [T, h] bf16 (K-major)             Wg planes [h, E] (MN-major)
//   DWG    dWg [h x E]        x [T, h] bf16 (MN-major), K = T     dL planes [T, E] (MN-major)
//   DX     dx [T x h]         dL planes [T, E] (K-major), K = E   Wg planes [h, E] (K-major)
//   FWD3, DWG3: FWD and DWG with three planes of fp32 x
//
// One persistent CTA per SM walks units (slice z of K, M tile, N tile of 128): warp 0 issues the
// TMA loads, warp 1 owns TMEM (two buffers of the accumulator pair) and issues the MMAs, warps 2-5
// drain one TMEM lane quarter each and hold their row's 128 running sums in registers.  With
// several K slices a unit writes fp32 partials [slice][M][N] that the split-K reduction adds in a
// fixed order (with the bias), so results do not depend on scheduling.  Every wait is bounded.
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "planes.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace ptx;

constexpr int RBM = 128;      // MMA M
constexpr int RBN = 128;      // N tile
constexpr int RBK = 64;       // K per stage (one 128-byte swizzle row of bf16)
constexpr int kChunkSteps = 4;  // stages per drain: 256 of K
constexpr int kRThreads = 192;  // producer, MMA, four epilogue warps
constexpr uint32_t kPlane = 16384;  // bytes of one 128 x 64 bf16 plane tile

// FWD3 and DWG3 are FWD and DWG for fp32 activations: x is split into three planes too, and
// every product is the six-term plane sum that DX uses.
enum RMode { FWD = 0, DWG = 1, DX = 2, FWD3 = 3, DWG3 = 4 };

template <int MODE> struct RCfg {
  static constexpr int NA = (MODE == DX || MODE == FWD3 || MODE == DWG3) ? 3 : 1;  // A planes
  static constexpr int NB = 3;                     // B planes
  static constexpr bool A_MN = (MODE == DWG || MODE == DWG3);
  static constexpr bool B_MN = (MODE != DX);
  static constexpr uint32_t STAGE_BYTES = (NA + NB) * kPlane;
  static constexpr int STAGES = 196608 / STAGE_BYTES;
  static_assert(STAGES >= 2, "stage ring");
};

struct RouterParams {
  CUtensorMap mapA[3];
  CUtensorMap mapB[3];
  int M, N, K;
  int mt, nt, z;    // M tiles, N tiles, K slices
  int kslice;       // K of one slice (a multiple of 256)
  float* out;       // z > 1: partials [z][M][N]; else the result [M][N]
  const float* bias;  // FWD with one slice: [N] added to the result (nullable)
  int* status;
  // bounded waits: limit per wait in ns (0: the default); withhold != 0 is the test hook of
  // moe_debug_withhold_stage (the producer never fills the first stage of the first unit)
  unsigned long long wait_ns;
  int withhold;
};

struct RUnit {
  int m0, n0, z;
  int kb, nsteps;  // first K, stages of RBK
  int ncols;       // valid N columns (a multiple of 16)
};

__device__ __forceinline__ RUnit rdecode(int u, const RouterParams& p) {
  RUnit w;
  const int nt = u % p.nt;
  const int r = u / p.nt;
  w.n0 = nt * RBN;
  w.m0 = (r % p.mt) * RBM;
  w.z = r / p.mt;
  w.kb = w.z * p.kslice;
  const int ke = min(p.K, w.kb + p.kslice);
  w.nsteps = (ke - w.kb + RBK - 1) / RBK;
  w.ncols = min(RBN, p.N - w.n0);
  return w;
}

template <int MODE>
__global__ void __launch_bounds__(kRThreads, 1) router_tc_kernel(const __grid_constant__ RouterParams p) {
  using C = RCfg<MODE>;
  extern __shared__ __align__(1024) uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[C::STAGES];
  __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t ring = (smem_u32(dsmem) + 1023u) & ~1023u;
  const int total = p.mt * p.nt * p.z;
  if ((int)blockIdx.x >= total) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&tfull_bar[b], 1); mbar_init(&tempty_bar[b], 4); }
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

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const RUnit w = rdecode(u, p);
        const int nbB = C::B_MN ? (w.ncols + 63) / 64 : 2;  // 64-column boxes per B plane
        const uint32_t tx = C::NA * kPlane + C::NB * (uint32_t)nbB * 8192u;
        for (int ks = 0; ks < w.nsteps; ++ks) {
          if (!mbar_wait(&empty_bar[s], ph ^ 1u, &s_abort, p.status, p.wait_ns)) { ok = false; break; }
          if (p.withhold && u == (int)blockIdx.x && ks == 0) {  // test hook: a stage nobody fills
            if (++s == C::STAGES) { s = 0; ph ^= 1u; }
            continue;
          }
          mbar_expect_tx(&full_bar[s], tx);
          const uint32_t a_sm = ring + s * C::STAGE_BYTES;
          const uint32_t b_sm = a_sm + C::NA * kPlane;
          const int k0 = w.kb + ks * RBK;
#pragma unroll
          for (int i = 0; i < C::NA; ++i) {
            if (C::A_MN) {  // x [T, h]: rows are K, columns are M
              tma_load_2d(a_sm + i * kPlane, &p.mapA[i], &full_bar[s], w.m0, k0);
              tma_load_2d(a_sm + i * kPlane + 8192, &p.mapA[i], &full_bar[s], w.m0 + 64, k0);
            } else {  // rows are M, columns are K: one 64 x 128 box
              tma_load_2d(a_sm + i * kPlane, &p.mapA[i], &full_bar[s], k0, w.m0);
            }
          }
#pragma unroll
          for (int j = 0; j < C::NB; ++j) {
            if (C::B_MN) {  // rows are K, columns are N
              for (int q = 0; q < nbB; ++q)
                tma_load_2d(b_sm + j * kPlane + q * 8192, &p.mapB[j], &full_bar[s], w.n0 + 64 * q, k0);
            } else {  // rows are N, columns are K
              tma_load_2d(b_sm + j * kPlane, &p.mapB[j], &full_bar[s], k0, w.n0);
            }
          }
          if (++s == C::STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok || s_abort) {  // give the loads already in flight time to land
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    int s = 0;
    uint32_t ph = 0;
    int cc = 0;  // drain chunks issued so far (accumulator buffer = cc & 1)
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const RUnit w = rdecode(u, p);
      const uint32_t idesc = idesc_bf16((w.ncols + 15) & ~15, C::A_MN, C::B_MN);
      for (int c0 = 0; c0 < w.nsteps && ok; c0 += kChunkSteps, ++cc) {
        const int b = cc & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&tempty_bar[b], ((uint32_t)(cc >> 1) & 1u) ^ 1u, &s_abort,
                                               p.status, p.wait_ns))) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_main = tmem_base + (uint32_t)(b * 2 * RBN);
        const uint32_t d_corr = d_main + RBN;
        const int c1 = min(w.nsteps, c0 + kChunkSteps);
        for (int ks = c0; ks < c1; ++ks) {
          if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[s], ph, &s_abort, p.status, p.wait_ns))) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a_sm = ring + s * C::STAGE_BYTES;
            const uint32_t b_sm = a_sm + C::NA * kPlane;
#pragma unroll
            for (int kk = 0; kk < RBK / 16; ++kk) {
              const bool first = (ks == c0 && kk == 0);
              // (A plane, B plane): the leading product, then the small ones from the smallest
              constexpr int NP = (C::NA == 3) ? 6 : 3;
              const int pa[6] = {0, 0, 0, 2, 1, 1};
              const int pb[6] = {0, 2, 1, 0, 1, 0};
              const int qa[6] = {0, 2, 1, 0, 1, 0};  // NA == 3: a2 b0, a1 b1, a0 b2, a1 b0, a0 b1
              const int qb[6] = {0, 0, 1, 2, 0, 1};
#pragma unroll
              for (int t = 0; t < NP; ++t) {
                const int ia = (C::NA == 3) ? qa[t] : pa[t];
                const int ib = (C::NA == 3) ? qb[t] : pb[t];
                uint64_t ad, bd;
                if (C::A_MN) ad = sdesc(a_sm + ia * kPlane + kk * 2048, 8192, 1024);
                else ad = sdesc(a_sm + ia * kPlane + kk * 32, 16, 1024);
                if (C::B_MN) bd = sdesc(b_sm + ib * kPlane + kk * 2048, 8192, 1024);
                else bd = sdesc(b_sm + ib * kPlane + kk * 32, 16, 1024);
                const bool lead = (t == 0);
                umma(lead ? d_main : d_corr, ad, bd, idesc, (first && (lead || t == 1)) ? 0u : 1u);
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
    }
    if (lane == 0) {
      umma_commit(&drain_bar);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(&drain_bar, 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter
    int cc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const RUnit w = rdecode(u, p);
      float run[RBN];
#pragma unroll
      for (int i = 0; i < RBN; ++i) run[i] = 0.f;
      for (int c0 = 0; c0 < w.nsteps; c0 += kChunkSteps, ++cc) {
        const int b = cc & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull_bar[b], (uint32_t)(cc >> 1) & 1u, &s_abort, p.status, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t0 = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * 2 * RBN);
#pragma unroll
        for (int g = 0; g < RBN / 16; ++g) {
          if (16 * g < w.ncols) {
            float vm[16], vc[16];
            tmem_ld16(t0 + 16 * g, vm);
            tmem_ld16(t0 + RBN + 16 * g, vc);
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
      const int row = w.m0 + q * 32 + lane;
      if (row < p.M) {
        const bool add_bias = (MODE == FWD || MODE == FWD3) && p.z == 1 && p.bias != nullptr;
        float* dst = p.out + ((size_t)w.z * p.M + row) * (size_t)p.N + w.n0;
#pragma unroll
        for (int g = 0; g < RBN / 4; ++g) {
          if (4 * g < w.ncols) {
            float4 v = make_float4(run[4 * g], run[4 * g + 1], run[4 * g + 2], run[4 * g + 3]);
            if (add_bias) {
              const float4 bb = __ldg(reinterpret_cast<const float4*>(p.bias + w.n0 + 4 * g));
              v.x += bb.x; v.y += bb.y; v.z += bb.z; v.w += bb.w;
            }
            *reinterpret_cast<float4*>(dst + 4 * g) = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
  }
}

// Exact three-plane split of fp32 values: dst[p * n + i] = plane p of src[i], p = 0, 1, 2.  Each
// difference below is exact in fp32, and the last plane holds the remaining at most 8 significant
// bits, so v0 + v1 + v2 == v for every normal fp32 value above 2^-100 in magnitude.
__global__ void __launch_bounds__(256) split3_kernel(const float* __restrict__ src, long long n,
                                                     __nv_bfloat16* __restrict__ dst) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    split3_value(__ldg(src + i), dst + i, dst + n + i, dst + 2 * n + i);
  }
}

// n a multiple of 8: eight values a thread, 16-byte loads and plane stores.
__global__ void __launch_bounds__(256) split3_vec_kernel(const float* __restrict__ src, long long n,
                                                         __nv_bfloat16* __restrict__ dst) {
  const float4* s = reinterpret_cast<const float4*>(src);
  uint4* d0 = reinterpret_cast<uint4*>(dst);
  uint4* d1 = reinterpret_cast<uint4*>(dst + n);
  uint4* d2 = reinterpret_cast<uint4*>(dst + 2 * n);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n / 8; i += (long long)gridDim.x * blockDim.x)
    split3_vec8(__ldg(s + 2 * i), __ldg(s + 2 * i + 1), d0 + i, d1 + i, d2 + i);
}

void launch_split3(const float* src, long long n, __nv_bfloat16* dst, cudaStream_t st) {
  if (n % 8 == 0) {  // every plane starts 16-byte aligned (the planes are n values apart)
    const int blocks = (int)std::min<long long>((n / 8 + 255) / 256, 8 * num_sms());
    split3_vec_kernel<<<blocks, 256, 0, st>>>(src, n, dst);
  } else {
    const int blocks = (int)std::min<long long>((n + 255) / 256, 8 * num_sms());
    split3_kernel<<<blocks, 256, 0, st>>>(src, n, dst);
  }
  count_launch(st);
}

// K slices for `tiles` output tiles over K: slices are whole drain chunks (256 of K); the count
// minimises (waves of one CTA per SM) x (chunks per slice), fewer slices on ties.
// The count depends on the shape alone (152 SMs assumed), so that the workspace size, which
// holds the partials, does not depend on the device.
void pick_slices(int tiles, int K, int* kslice, int* z) {
  constexpr int sms = 152;
  const int chunks = (K + 255) / 256;
  int best_per = chunks;
  long long best_cost = -1;
  for (int per = chunks; per >= 1; --per) {
    const int zz = (chunks + per - 1) / per;
    const long long ctas = (long long)tiles * zz;
    const long long cost = ((ctas + sms - 1) / sms) * per;
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_per = per; }
  }
  *kslice = best_per * 256;
  *z = (K + *kslice - 1) / *kslice;
}

template <int MODE>
int rlaunch(const RouterParams& p0, cudaStream_t st) {
  using C = RCfg<MODE>;
  RouterParams p = p0;
  p.withhold = debug_take_withhold(&p.wait_ns) ? 1 : 0;
  const int smem = (int)(C::STAGES * C::STAGE_BYTES + 1024);
  if (cudaFuncSetAttribute(router_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -1;
  const int total = p.mt * p.nt * p.z;
  router_tc_kernel<MODE><<<std::min(total, num_sms()), kRThreads, smem, st>>>(p);
  count_launch(st);
  return 0;
}

RouterParams rblank(int* status) {
  RouterParams p;
  memset(&p, 0, sizeof(p));
  p.status = status;
  return p;
}

size_t r256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

// bf16 or fp32 activations (fp32 ones are split into planes too), h a multiple of 64, 64 <= E <= 1024 a
// multiple of 16 (MMA N); MOE_PFT_GEMM=simt forces the fp32 FFMA path.
bool tc_router_supported(int dtype, int h, int E) {
  const char* env = getenv("MOE_PFT_GEMM");
  if (env && strcmp(env, "simt") == 0) return false;
  return (dtype == MOE_BF16 || dtype == MOE_F32) && h % 64 == 0 && E % 16 == 0 && E >= 64 && E <= 1024 &&
         tc_encode_available();
}

// Scratch bytes after the workspace header: op 0 = forward, 1 = backward.  fp32 activations add
// the three planes of x.
size_t tc_router_scratch(int op, int T, int h, int E, int dtype) {
  const size_t planes_w = r256((size_t)3 * h * E * 2);
  const size_t planes_d = r256((size_t)3 * T * E * 2);
  const size_t planes_x = dtype == MOE_F32 ? r256((size_t)3 * T * h * 2) : 0;
  int ks, z;
  if (op == 0) {  // forward: Wg planes, x planes, partials [z][T][E]
    pick_slices(((T + RBM - 1) / RBM) * ((E + RBN - 1) / RBN), h, &ks, &z);
    return planes_w + planes_x + (z > 1 ? r256((size_t)z * T * E * 4) : 0);
  }
  // backward: dL planes, Wg planes, x planes, partials [z][h][E]
  pick_slices(((h + RBM - 1) / RBM) * ((E + RBN - 1) / RBN), T, &ks, &z);
  return planes_d + planes_w + planes_x + (z > 1 ? r256((size_t)z * h * E * 4) : 0);
}

int tc_router_logits(const void* x, const float* Wg, const float* bias, int T, int h, int E, int dtype,
                     float* logits, void* scratch, const float** partial_out, int* slices_out, int* status,
                     cudaStream_t st) {
  const bool f32 = dtype == MOE_F32;
  char* sp = static_cast<char*>(scratch);
  __nv_bfloat16* wp = reinterpret_cast<__nv_bfloat16*>(sp);
  __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(sp + r256((size_t)3 * h * E * 2));
  float* partial = reinterpret_cast<float*>(sp + r256((size_t)3 * h * E * 2) +
                                            (f32 ? r256((size_t)3 * T * h * 2) : 0));
  launch_split3(Wg, (long long)h * E, wp, st);
  if (f32) launch_split3(static_cast<const float*>(x), (long long)T * h, xp, st);
  RouterParams p = rblank(status);
  bool ok = true;
  if (f32) {
    for (int i = 0; i < 3; ++i) ok = ok && tc_make_map(&p.mapA[i], xp + (size_t)i * T * h, T, h, 64, 128);
  } else {
    ok = tc_make_map(&p.mapA[0], x, T, h, 64, 128);
  }
  for (int j = 0; j < 3; ++j) ok = ok && tc_make_map(&p.mapB[j], wp + (size_t)j * h * E, h, E, 64, 64);
  if (!ok) return -1;
  p.M = T; p.N = E; p.K = h;
  p.mt = (T + RBM - 1) / RBM; p.nt = (E + RBN - 1) / RBN;
  pick_slices(p.mt * p.nt, h, &p.kslice, &p.z);
  p.out = p.z > 1 ? partial : logits;
  p.bias = bias;
  if (f32 ? rlaunch<FWD3>(p, st) : rlaunch<FWD>(p, st)) return -1;
  // several K slices: the caller adds the partials (with the bias) where it reads the logits
  *partial_out = p.z > 1 ? partial : nullptr;
  *slices_out = p.z;
  return 0;
}

int tc_router_bwd(const void* x, const float* Wg, const float* d_logits, int T, int h, int E, int dtype,
                  float* dWg, float* dx_router, void* scratch, bool dl_planes_ready, int* status, cudaStream_t st) {
  const bool f32 = dtype == MOE_F32;
  char* sp = static_cast<char*>(scratch);
  __nv_bfloat16* dp = reinterpret_cast<__nv_bfloat16*>(sp);
  __nv_bfloat16* wp = reinterpret_cast<__nv_bfloat16*>(sp + r256((size_t)3 * T * E * 2));
  __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<char*>(wp) + r256((size_t)3 * h * E * 2));
  float* partial = reinterpret_cast<float*>(reinterpret_cast<char*>(xp) + (f32 ? r256((size_t)3 * T * h * 2) : 0));
  if (!dl_planes_ready) launch_split3(d_logits, (long long)T * E, dp, st);
  if (f32) launch_split3(static_cast<const float*>(x), (long long)T * h, xp, st);
  // dWg = x^T dL: M = h, N = E, K = T
  RouterParams g = rblank(status);
  bool ok = true;
  if (f32) {
    for (int i = 0; i < 3; ++i) ok = ok && tc_make_map(&g.mapA[i], xp + (size_t)i * T * h, T, h, 64, 64);
  } else {
    ok = tc_make_map(&g.mapA[0], x, T, h, 64, 64);
  }
  for (int j = 0; j < 3; ++j) ok = ok && tc_make_map(&g.mapB[j], dp + (size_t)j * T * E, T, E, 64, 64);
  if (!ok) return -1;
  g.M = h; g.N = E; g.K = T;
  g.mt = (h + RBM - 1) / RBM; g.nt = (E + RBN - 1) / RBN;
  pick_slices(g.mt * g.nt, T, &g.kslice, &g.z);
  g.out = g.z > 1 ? partial : dWg;
  if (f32 ? rlaunch<DWG3>(g, st) : rlaunch<DWG>(g, st)) return -1;
  if (g.z > 1) launch_splitk_reduce(partial, g.z, (long long)h * E, E, nullptr, dWg, st);
  if (dx_router == nullptr) return 0;
  // dx = dL Wg^T: M = T, N = h, K = E
  launch_split3(Wg, (long long)h * E, wp, st);
  RouterParams d = rblank(status);
  ok = true;
  for (int i = 0; i < 3; ++i) {
    ok = ok && tc_make_map(&d.mapA[i], dp + (size_t)i * T * E, T, E, 64, 128);
    ok = ok && tc_make_map(&d.mapB[i], wp + (size_t)i * h * E, h, E, 64, 128);
  }
  if (!ok) return -1;
  d.M = T; d.N = h; d.K = E;
  d.mt = (T + RBM - 1) / RBM; d.nt = (h + RBN - 1) / RBN;
  d.kslice = ((E + 255) / 256) * 256;
  d.z = 1;
  d.out = dx_router;
  return rlaunch<DX>(d, st);
}

}  // namespace moe
