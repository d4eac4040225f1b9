// Vectorised exact three-plane bf16 split of fp32 values (the planes the tensor-core kernels
// multiply for fp32 operands; split3_value in common.cuh defines one value's planes).
#pragma once

#include "common.cuh"

namespace moe {

// Eight consecutive fp32 values (two 16-byte loads) split into their three bf16 planes, each
// plane's eight values packed into one 16-byte vector.
__device__ __forceinline__ void split3_vec8(const float4& a, const float4& b, uint4* p0, uint4* p1, uint4* p2) {
  const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t w0[4], w1[4], w2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat16 q0[2], q1[2], q2[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) split3_value(v[2 * i + j], &q0[j], &q1[j], &q2[j]);
    w0[i] = (uint32_t)__bfloat16_as_ushort(q0[0]) | ((uint32_t)__bfloat16_as_ushort(q0[1]) << 16);
    w1[i] = (uint32_t)__bfloat16_as_ushort(q1[0]) | ((uint32_t)__bfloat16_as_ushort(q1[1]) << 16);
    w2[i] = (uint32_t)__bfloat16_as_ushort(q2[0]) | ((uint32_t)__bfloat16_as_ushort(q2[1]) << 16);
  }
  *p0 = make_uint4(w0[0], w0[1], w0[2], w0[3]);
  *p1 = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  *p2 = make_uint4(w2[0], w2[1], w2[2], w2[3]);
}

}  // namespace moe
