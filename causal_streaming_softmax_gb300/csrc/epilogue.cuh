// epilogue.cuh - storing a 64-wide gradient row into a token-major block of
// a projection gradient, in binary32 and/or bfloat16 (the projection-fused
// epilogues of the key and dQ passes).
#pragma once

#include "attn_internal.h"
#include "sm103.cuh"

namespace css {

// The 64 values r0[0..31], r1[0..31] (binary32 bits), each times `scale`
// when `scaled`, written to p.f32 + off and, rounded to nearest even, to
// p.bf16 + off (either may be null).
__device__ __forceinline__ void store_projection_row(const Projection& p, size_t off,
                                                     const uint32_t (&r0)[32],
                                                     const uint32_t (&r1)[32], float scale,
                                                     bool scaled) {
  float v[64];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = scaled ? __fmul_rn(__uint_as_float(r0[i]), scale) : __uint_as_float(r0[i]);
    v[32 + i] = scaled ? __fmul_rn(__uint_as_float(r1[i]), scale) : __uint_as_float(r1[i]);
  }
  if (p.f32) {
    float4* dst = reinterpret_cast<float4*>(p.f32 + off);
#pragma unroll
    for (int u = 0; u < 16; ++u) dst[u] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
  }
  if (p.bf16) {
    uint4* dst = reinterpret_cast<uint4*>(p.bf16 + off);
#pragma unroll
    for (int u = 0; u < 8; ++u)
      dst[u] = make_uint4(pack_bf16x2(v[8 * u], v[8 * u + 1]), pack_bf16x2(v[8 * u + 2], v[8 * u + 3]),
                          pack_bf16x2(v[8 * u + 4], v[8 * u + 5]),
                          pack_bf16x2(v[8 * u + 6], v[8 * u + 7]));
  }
}

}  // namespace css
