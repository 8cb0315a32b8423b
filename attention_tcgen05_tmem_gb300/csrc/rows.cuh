// rows.cuh -- per-row helpers for epilogues and the TTT suffix passes:
// row addressing in [B, H, S, D] views, bf16 row dot products (fp32
// accumulate) and 16-column stores of fp32 results as fp32 or bf16.
#pragma once
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

constexpr int kDiagBatch = 8;  // TTT suffix diagonals folded per epilogue pass

__device__ __forceinline__ const __nv_bfloat16* row_ptr(const View& v, int b, int h, int64_t s) {
  return reinterpret_cast<const __nv_bfloat16*>(v.ptr) + b * v.sb + h * v.sh + s * v.ss;
}

// Dot product of two bf16 rows of length D (fp32 accumulate, fixed order).
template <int D>
__device__ __forceinline__ float dot_rows(const __nv_bfloat16* x, const __nv_bfloat16* y) {
  float acc = 0.f;
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 8) {
    const uint4 xa = *reinterpret_cast<const uint4*>(x + c0);
    const uint4 ya = *reinterpret_cast<const uint4*>(y + c0);
    const __nv_bfloat162* xv = reinterpret_cast<const __nv_bfloat162*>(&xa);
    const __nv_bfloat162* yv = reinterpret_cast<const __nv_bfloat162*>(&ya);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 xf = __bfloat1622float2(xv[e]);
      const float2 yf = __bfloat1622float2(yv[e]);
      acc = fmaf(xf.x, yf.x, acc);
      acc = fmaf(xf.y, yf.y, acc);
    }
  }
  return acc;
}

// x[0..15] += w * row[0..15] (bf16 row).
__device__ __forceinline__ void axpy16(float* x, float w, const __nv_bfloat16* row) {
#pragma unroll
  for (int e = 0; e < 16; e += 8) {
    const uint4 ra = *reinterpret_cast<const uint4*>(row + e);
    const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&ra);
#pragma unroll
    for (int f = 0; f < 4; ++f) {
      const float2 rf = __bfloat1622float2(r2[f]);
      x[e + 2 * f] = fmaf(w, rf.x, x[e + 2 * f]);
      x[e + 2 * f + 1] = fmaf(w, rf.y, x[e + 2 * f + 1]);
    }
  }
}

// Store 16 fp32 values (times mul) at columns c0 .. c0+15 of an output row,
// as fp32 or bf16.
__device__ __forceinline__ void store16(const View& v, int b, int h, int64_t s, int c0,
                                        const float* x, float mul, bool f32) {
  const int64_t off = b * v.sb + h * v.sh + s * v.ss + c0;
  if (f32) {
    float* row = reinterpret_cast<float*>(v.ptr) + off;
#pragma unroll
    for (int e = 0; e < 16; e += 4)
      *reinterpret_cast<float4*>(row + e) =
          make_float4(x[e] * mul, x[e + 1] * mul, x[e + 2] * mul, x[e + 3] * mul);
  } else {
    __nv_bfloat16* row = reinterpret_cast<__nv_bfloat16*>(v.ptr) + off;
#pragma unroll
    for (int e = 0; e < 16; e += 8) {
      uint4 pkt;
      pkt.x = pack_bf16x2(x[e + 0] * mul, x[e + 1] * mul);
      pkt.y = pack_bf16x2(x[e + 2] * mul, x[e + 3] * mul);
      pkt.z = pack_bf16x2(x[e + 4] * mul, x[e + 5] * mul);
      pkt.w = pack_bf16x2(x[e + 6] * mul, x[e + 7] * mul);
      *reinterpret_cast<uint4*>(row + e) = pkt;
    }
  }
}

}  // namespace attn
