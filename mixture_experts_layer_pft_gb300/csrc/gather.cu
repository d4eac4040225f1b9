// Dispatch and combine over the padding-free token buffer, and their adjoints.
//
// All four are row gathers: every row of h elements moves as 16-byte vectors, a group of
// `tpr` threads per row (tpr is a power of two, 32..256, chosen so each thread handles at
// most two vectors per pass; rows wider than 256 x 2 vectors take several passes),
// `256 / tpr` rows per 256-thread block.  Loads are issued before the dependent stores, and
// the k-way gathers issue the loads of four source rows before summing any of them, so that
// each thread keeps several 16-byte requests in flight.  Sums run in fp32 in a fixed order
// (j ascending), so results are bitwise reproducible; no atomics.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kBlock = 256;
constexpr int kMaxVecPerThread = 2;
// The k-way gathers (combine, dispatch backward) issue the loads of kJB source rows before
// consuming any, with at most kGatherVec vectors per thread per row, so each thread keeps
// kJB * kGatherVec 16-byte loads in flight.
constexpr int kJB = 4;
constexpr int kGatherVec = 2;

struct RowGeom {
  int tpr;       // threads per row
  int rows_per_block;
};

RowGeom row_geom(int nvec, int maxvec = kMaxVecPerThread) {
  int tpr = 32;
  while (tpr < kBlock && tpr * maxvec < nvec) tpr *= 2;
  return {tpr, kBlock / tpr};
}

// ---------------------------------------------------------------------------- dispatch
// xbuf[p,:] = x[token_ids[p],:]
template <typename T>
__global__ void __launch_bounds__(kBlock) dispatch_kernel(const T* __restrict__ x,
                                                          const int* __restrict__ token_ids,
                                                          int T_, int rows, int nvec, int tpr,
                                                          T* __restrict__ xbuf, int* status) {
  const int rpb = kBlock / tpr;
  const int p = blockIdx.x * rpb + threadIdx.x / tpr;
  const int lt = threadIdx.x % tpr;
  if (p >= rows) return;
  const int t = __ldg(token_ids + p);
  uint4* dst = reinterpret_cast<uint4*>(xbuf) + (size_t)p * nvec;
  if ((unsigned)t >= (unsigned)T_) {
    if (lt == 0) flag_status(status, MOE_STATUS_BAD_INDEX);
    for (int v = lt; v < nvec; v += tpr) dst[v] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x) + (size_t)t * nvec;
  for (int vb = 0; vb < nvec; vb += tpr * kMaxVecPerThread) {
    uint4 r[kMaxVecPerThread];
#pragma unroll
    for (int u = 0; u < kMaxVecPerThread; ++u) {
      const int v = vb + lt + u * tpr;
      if (v < nvec) r[u] = __ldg(src + v);
    }
    // streaming stores (evict first): the buffer is written once, while the rows of x it copies
    // are read k times and should stay in L2
#pragma unroll
    for (int u = 0; u < kMaxVecPerThread; ++u) {
      const int v = vb + lt + u * tpr;
      if (v < nvec) __stcs(reinterpret_cast<int4*>(dst + v), *reinterpret_cast<const int4*>(&r[u]));
    }
  }
}

// ---------------------------------------------------------------------------- combine
// y[t,:] = sum_j w[t,j] * ybuf[slot_of[t*k+j],:]
template <typename T>
__global__ void __launch_bounds__(kBlock) combine_kernel(const T* __restrict__ ybuf,
                                                         const int* __restrict__ slot_of,
                                                         const float* __restrict__ w, int T_,
                                                         int k, int nvec, int tpr, int Tk,
                                                         T* __restrict__ y, int* status) {
  constexpr int VN = Vec<T>::N;
  constexpr int MV = kGatherVec;
  const int rpb = kBlock / tpr;
  const int t = blockIdx.x * rpb + threadIdx.x / tpr;
  const int lt = threadIdx.x % tpr;
  if (t >= T_) return;
  const uint4* yb = reinterpret_cast<const uint4*>(ybuf);
  uint4* dst = reinterpret_cast<uint4*>(y) + (size_t)t * nvec;
  for (int vb = 0; vb < nvec; vb += tpr * MV) {
    float acc[MV][VN];
#pragma unroll
    for (int u = 0; u < MV; ++u)
#pragma unroll
      for (int q = 0; q < VN; ++q) acc[u][q] = 0.f;
    for (int j0 = 0; j0 < k; j0 += kJB) {
      // slots and weights of up to kJB rows, then all their loads, then the sums (j ascending)
      int sj[kJB];
      float wj[kJB];
#pragma unroll
      for (int jj = 0; jj < kJB; ++jj) {
        sj[jj] = -1;
        wj[jj] = 0.f;
        if (j0 + jj < k) {
          const int s = __ldg(slot_of + (size_t)t * k + j0 + jj);
          wj[jj] = __ldg(w + (size_t)t * k + j0 + jj);
          if ((unsigned)s < (unsigned)Tk) sj[jj] = s;
          else if (lt == 0 && vb == 0) flag_status(status, MOE_STATUS_BAD_INDEX);
        }
      }
      uint4 r[kJB][MV];
#pragma unroll
      for (int jj = 0; jj < kJB; ++jj)
#pragma unroll
        for (int u = 0; u < MV; ++u) {
          const int v = vb + lt + u * tpr;
          if (sj[jj] >= 0 && v < nvec) r[jj][u] = __ldg(yb + (size_t)sj[jj] * nvec + v);
        }
#pragma unroll
      for (int jj = 0; jj < kJB; ++jj) {
        if (sj[jj] < 0) continue;
#pragma unroll
        for (int u = 0; u < MV; ++u) {
          const int v = vb + lt + u * tpr;
          if (v < nvec) {
            float f[VN];
            unpack(r[jj][u], f, T());
#pragma unroll
            for (int q = 0; q < VN; ++q) acc[u][q] = fmaf(wj[jj], f[q], acc[u][q]);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < MV; ++u) {
      const int v = vb + lt + u * tpr;
      if (v < nvec) dst[v] = pack(acc[u], T());
    }
  }
}

// ---------------------------------------------------------------------------- dispatch bwd
// dx[t,:] = dx_add[t,:] + sum_j dxbuf[slot_of[t*k+j],:]
template <typename T>
__global__ void __launch_bounds__(kBlock) dispatch_bwd_kernel(
    const T* __restrict__ dxbuf, const int* __restrict__ slot_of, const float* __restrict__ dx_add,
    int T_, int k, int nvec, int tpr, int Tk, T* __restrict__ dx, int* status) {
  constexpr int VN = Vec<T>::N;
  constexpr int MV = kGatherVec;
  const int rpb = kBlock / tpr;
  const int t = blockIdx.x * rpb + threadIdx.x / tpr;
  const int lt = threadIdx.x % tpr;
  if (t >= T_) return;
  const uint4* src = reinterpret_cast<const uint4*>(dxbuf);
  uint4* dst = reinterpret_cast<uint4*>(dx) + (size_t)t * nvec;
  for (int vb = 0; vb < nvec; vb += tpr * MV) {
    float acc[MV][VN];
#pragma unroll
    for (int u = 0; u < MV; ++u) {
      const int v = vb + lt + u * tpr;
#pragma unroll
      for (int q = 0; q < VN; ++q) acc[u][q] = 0.f;
      if (dx_add != nullptr && v < nvec) {
        const float4* a4 = reinterpret_cast<const float4*>(dx_add + ((size_t)t * nvec + v) * VN);
#pragma unroll
        for (int q = 0; q < VN / 4; ++q) {
          const float4 a = __ldg(a4 + q);
          acc[u][4 * q] = a.x; acc[u][4 * q + 1] = a.y; acc[u][4 * q + 2] = a.z; acc[u][4 * q + 3] = a.w;
        }
      }
    }
    for (int j0 = 0; j0 < k; j0 += kJB) {
      int sj[kJB];
#pragma unroll
      for (int jj = 0; jj < kJB; ++jj) {
        sj[jj] = -1;
        if (j0 + jj < k) {
          const int s = __ldg(slot_of + (size_t)t * k + j0 + jj);
          if ((unsigned)s < (unsigned)Tk) sj[jj] = s;
          else if (lt == 0 && vb == 0) flag_status(status, MOE_STATUS_BAD_INDEX);
        }
      }
      uint4 r[kJB][MV];
#pragma unroll
      for (int jj = 0; jj < kJB; ++jj)
#pragma unroll
        for (int u = 0; u < MV; ++u) {
          const int v = vb + lt + u * tpr;
          if (sj[jj] >= 0 && v < nvec) r[jj][u] = __ldg(src + (size_t)sj[jj] * nvec + v);
        }
#pragma unroll
      for (int jj = 0; jj < kJB; ++jj) {
        if (sj[jj] < 0) continue;
#pragma unroll
        for (int u = 0; u < MV; ++u) {
          const int v = vb + lt + u * tpr;
          if (v < nvec) {
            float f[VN];
            unpack(r[jj][u], f, T());
#pragma unroll
            for (int q = 0; q < VN; ++q) acc[u][q] += f[q];
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < MV; ++u) {
      const int v = vb + lt + u * tpr;
      if (v < nvec) dst[v] = pack(acc[u], T());
    }
  }
}

// ---------------------------------------------------------------------------- combine bwd
template <typename T, int KMAX>
__global__ void __launch_bounds__(kBlock) combine_bwd_kernel(
    const T* __restrict__ dy, const T* __restrict__ ybuf, const int* __restrict__ slot_of,
    const float* __restrict__ w, int T_, int k, int nvec, int tpr, int Tk, T* __restrict__ dybuf,
    float* __restrict__ d_w, int* status) {
  constexpr int VN = Vec<T>::N;
  __shared__ float red[kBlock / kWarp][KMAX];
  const int rpb = kBlock / tpr;
  const int row_in_block = threadIdx.x / tpr;
  const int t = blockIdx.x * rpb + row_in_block;
  const int lt = threadIdx.x % tpr;
  const bool active = t < T_;
  float dwp[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) dwp[j] = 0.f;
  for (int vb = 0; active && vb < nvec; vb += tpr * kMaxVecPerThread) {
    float g[kMaxVecPerThread][VN];
    const uint4* dyv = reinterpret_cast<const uint4*>(dy) + (size_t)t * nvec;
#pragma unroll
    for (int u = 0; u < kMaxVecPerThread; ++u) {
      const int v = vb + lt + u * tpr;
      if (v < nvec) unpack(__ldg(dyv + v), g[u], T());
    }
    const uint4* yb = reinterpret_cast<const uint4*>(ybuf);
    uint4* db = reinterpret_cast<uint4*>(dybuf);
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j >= k) break;
      const int s = __ldg(slot_of + (size_t)t * k + j);
      const float wj = __ldg(w + (size_t)t * k + j);
      if ((unsigned)s >= (unsigned)Tk) {
        if (lt == 0 && vb == 0) flag_status(status, MOE_STATUS_BAD_INDEX);
        continue;
      }
      uint4 r[kMaxVecPerThread];
#pragma unroll
      for (int u = 0; u < kMaxVecPerThread; ++u) {
        const int v = vb + lt + u * tpr;
        if (v < nvec) r[u] = __ldg(yb + (size_t)s * nvec + v);
      }
#pragma unroll
      for (int u = 0; u < kMaxVecPerThread; ++u) {
        const int v = vb + lt + u * tpr;
        if (v < nvec) {
          float f[VN], o[VN];
          unpack(r[u], f, T());
#pragma unroll
          for (int q = 0; q < VN; ++q) {
            dwp[j] = fmaf(g[u][q], f[q], dwp[j]);
            o[q] = wj * g[u][q];
          }
          db[(size_t)s * nvec + v] = pack(o, T());
        }
      }
    }
  }
  // reduce dwp over the tpr threads of the row: warp shuffles, then across the row's warps
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const float s = warp_sum(dwp[j]);
    if (lane == 0) red[warp][j] = s;
  }
  __syncthreads();
  const int wpr = tpr / kWarp;  // warps per row
  if (active && lt < k) {
    float s = 0.f;
    for (int q = 0; q < wpr; ++q) s += red[row_in_block * wpr + q][lt];
    d_w[(size_t)t * k + lt] = s;
  }
}

template <typename T>
void launch_dispatch_t(const void* x, const int* token_ids, int T_, int rows, int h,
                       void* xbuf, int* status, cudaStream_t st) {
  const int nvec = h / Vec<T>::N;
  const RowGeom g = row_geom(nvec);
  const int grid = (rows + g.rows_per_block - 1) / g.rows_per_block;
  dispatch_kernel<T><<<grid, kBlock, 0, st>>>(static_cast<const T*>(x), token_ids, T_, rows,
                                              nvec, g.tpr, static_cast<T*>(xbuf), status);
  count_launch(st);
}

template <typename T>
void launch_combine_t(const void* ybuf, const int* slot_of, const float* w, int T_, int k, int h,
                      void* y, int* status, cudaStream_t st) {
  const int nvec = h / Vec<T>::N;
  const RowGeom g = row_geom(nvec, kGatherVec);
  const int grid = (T_ + g.rows_per_block - 1) / g.rows_per_block;
  combine_kernel<T><<<grid, kBlock, 0, st>>>(static_cast<const T*>(ybuf), slot_of, w, T_, k,
                                             nvec, g.tpr, T_ * k, static_cast<T*>(y), status);
  count_launch(st);
}

template <typename T>
void launch_dispatch_bwd_t(const void* dxbuf, const int* slot_of, const float* dx_add, int T_,
                           int k, int h, void* dx, int* status, cudaStream_t st) {
  const int nvec = h / Vec<T>::N;
  const RowGeom g = row_geom(nvec, kGatherVec);
  const int grid = (T_ + g.rows_per_block - 1) / g.rows_per_block;
  dispatch_bwd_kernel<T><<<grid, kBlock, 0, st>>>(static_cast<const T*>(dxbuf), slot_of, dx_add,
                                                  T_, k, nvec, g.tpr, T_ * k,
                                                  static_cast<T*>(dx), status);
  count_launch(st);
}

template <typename T, int KMAX>
void launch_combine_bwd_k(const void* dy, const void* ybuf, const int* slot_of, const float* w,
                          int T_, int k, int h, void* dybuf, float* d_w, int* status,
                          cudaStream_t st) {
  const int nvec = h / Vec<T>::N;
  const RowGeom g = row_geom(nvec);
  const int grid = (T_ + g.rows_per_block - 1) / g.rows_per_block;
  combine_bwd_kernel<T, KMAX><<<grid, kBlock, 0, st>>>(
      static_cast<const T*>(dy), static_cast<const T*>(ybuf), slot_of, w, T_, k, nvec, g.tpr,
      T_ * k, static_cast<T*>(dybuf), d_w, status);
  count_launch(st);
}

template <typename T>
void launch_combine_bwd_t(const void* dy, const void* ybuf, const int* slot_of, const float* w,
                          int T_, int k, int h, void* dybuf, float* d_w, int* status,
                          cudaStream_t st) {
  if (k <= 2) launch_combine_bwd_k<T, 2>(dy, ybuf, slot_of, w, T_, k, h, dybuf, d_w, status, st);
  else if (k <= 4) launch_combine_bwd_k<T, 4>(dy, ybuf, slot_of, w, T_, k, h, dybuf, d_w, status, st);
  else if (k <= 8) launch_combine_bwd_k<T, 8>(dy, ybuf, slot_of, w, T_, k, h, dybuf, d_w, status, st);
  else if (k <= 16) launch_combine_bwd_k<T, 16>(dy, ybuf, slot_of, w, T_, k, h, dybuf, d_w, status, st);
  else launch_combine_bwd_k<T, 32>(dy, ybuf, slot_of, w, T_, k, h, dybuf, d_w, status, st);
}

}  // namespace

void launch_dispatch(int dtype, const void* x, const int* token_ids, int T_, int rows, int h,
                     void* xbuf, int* status, cudaStream_t st) {
  if (dtype == MOE_BF16) launch_dispatch_t<__nv_bfloat16>(x, token_ids, T_, rows, h, xbuf, status, st);
  else launch_dispatch_t<float>(x, token_ids, T_, rows, h, xbuf, status, st);
}

void launch_combine(int dtype, const void* ybuf, const int* slot_of, const float* w, int T_, int k,
                    int h, void* y, int* status, cudaStream_t st) {
  if (dtype == MOE_BF16) launch_combine_t<__nv_bfloat16>(ybuf, slot_of, w, T_, k, h, y, status, st);
  else launch_combine_t<float>(ybuf, slot_of, w, T_, k, h, y, status, st);
}

void launch_dispatch_bwd(int dtype, const void* dxbuf, const int* slot_of, const float* dx_add,
                         int T_, int k, int h, void* dx, int* status, cudaStream_t st) {
  if (dtype == MOE_BF16)
    launch_dispatch_bwd_t<__nv_bfloat16>(dxbuf, slot_of, dx_add, T_, k, h, dx, status, st);
  else launch_dispatch_bwd_t<float>(dxbuf, slot_of, dx_add, T_, k, h, dx, status, st);
}

void launch_combine_bwd(int dtype, const void* dy, const void* ybuf, const int* slot_of,
                        const float* w, int T_, int k, int h, void* dybuf, float* d_w,
                        int* status, cudaStream_t st) {
  if (dtype == MOE_BF16)
    launch_combine_bwd_t<__nv_bfloat16>(dy, ybuf, slot_of, w, T_, k, h, dybuf, d_w, status, st);
  else launch_combine_bwd_t<float>(dy, ybuf, slot_of, w, T_, k, h, dybuf, d_w, status, st);
}

}  // namespace moe
