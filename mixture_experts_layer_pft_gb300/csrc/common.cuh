// Device helpers shared by the PFT MoE kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_pft.h"

namespace moe {

// Layout of the 256-byte workspace header.
struct WsHeader {
  int status;           // sticky MOE_STATUS_* bits
  int pad[63];          // unused
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr int kWarp = 32;

__device__ __forceinline__ void flag_status(int* status, int bit) {
  if (status) atomicOr(status, bit);
}

// Exact split of an fp32 value into three bf16 planes, v = p0 + p1 + p2: p0 = bf16(v),
// p1 = bf16(v - p0), p2 = bf16(v - p0 - p1).  Each difference is exact in fp32 and the last
// plane holds the remaining at most 8 significant bits (normal values above 2^-100).
__device__ __forceinline__ void split3_value(float v, __nv_bfloat16* p0, __nv_bfloat16* p1, __nv_bfloat16* p2) {
  *p0 = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(*p0);
  *p1 = __float2bfloat16_rn(r1);
  *p2 = __float2bfloat16_rn(r1 - __bfloat162float(*p1));
}

// ---------------------------------------------------------------------------- element types

template <typename T> struct Vec;  // 16-byte vector of T
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Unpack a 16-byte vector into Vec<T>::N floats, and pack back (rounding to nearest even).
__device__ __forceinline__ void unpack(const uint4& u, float* out, float) {
  out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
  out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack(const uint4& u, float* out, __nv_bfloat16) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint4 pack(const float* in, float) {
  return make_uint4(__float_as_uint(in[0]), __float_as_uint(in[1]), __float_as_uint(in[2]),
                    __float_as_uint(in[3]));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint4 pack(const float* in, __nv_bfloat16) {
  return make_uint4(pack_bf16x2(in[0], in[1]), pack_bf16x2(in[2], in[3]),
                    pack_bf16x2(in[4], in[5]), pack_bf16x2(in[6], in[7]));
}

// Four consecutive elements as float4 (8-byte load for bf16, 16-byte for fp32).
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}
__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
  uint2 u;
  u.x = pack_bf16x2(v.x, v.y);
  u.y = pack_bf16x2(v.z, v.w);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

}  // namespace moe
