// rows.cuh -- per-row helpers for epilogues and the TTT suffix passes:
// row addressing in [B, H, S, D] views, the additive mask row, bf16 row dot
// products (fp32 accumulate), 16-column stores of fp32 results as fp32 or
// bf16, and coalesced row staging through shared memory in both directions.
#pragma once
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

__device__ __forceinline__ const __nv_bfloat16* row_ptr(const View& v, int b, int h, int64_t s) {
  return reinterpret_cast<const __nv_bfloat16*>(v.ptr) + b * v.sb + h * v.sh + s * v.ss;
}

// Additive mask (HOT-Step section 3: an arbitrary additive [S_kv, S] mask).  The raw
// scores s enter the exponent as s * scale * log2(e), so M is folded in as
// s + M / scale (M = -inf gives -inf).
__device__ __forceinline__ float bf16_bits(uint32_t h) { return __uint_as_float(h << 16); }

// s[c] += M[col0 + c] / scale for one row of a bf16 table (the additive mask by
// query row for the forward and dQ, its transpose by key row for dK/dV).  row:
// the row's first element, 16-byte aligned; col0 a multiple of 8; columns at
// or past ncols read nothing (those scores are masked or never stored).
template <int N>
__device__ __forceinline__ void add_bias_row(uint32_t* s, const uint16_t* row, int col0, int ncols,
                                             float inv_scale) {
  const uint16_t* r = row + col0;
  if (col0 + N <= ncols) {
#pragma unroll
    for (int c0 = 0; c0 < N; c0 += 8) {
      const uint4 m = *reinterpret_cast<const uint4*>(r + c0);
      const uint32_t w[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[c0 + 2 * e] = __float_as_uint(
            fmaf(bf16_bits(w[e] & 0xffffu), inv_scale, __uint_as_float(s[c0 + 2 * e])));
        s[c0 + 2 * e + 1] = __float_as_uint(
            fmaf(bf16_bits(w[e] >> 16), inv_scale, __uint_as_float(s[c0 + 2 * e + 1])));
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < N; ++c)
      if (col0 + c < ncols)
        s[c] = __float_as_uint(fmaf(bf16_bits(r[c]), inv_scale, __uint_as_float(s[c])));
  }
}

// The same in two halves, for loads issued well before the scores arrive:
// load_bias_row fetches M[col0 .. col0 + N) of a row into registers (16-byte
// loads; zeros past ncols), apply_bias_row adds them as add_bias_row does.
template <int N>
__device__ __forceinline__ void load_bias_row(uint4* m, const uint16_t* row, int col0, int ncols) {
  const uint16_t* r = row + col0;
  if (col0 + N <= ncols) {
#pragma unroll
    for (int c = 0; c < N / 8; ++c) m[c] = *reinterpret_cast<const uint4*>(r + 8 * c);
  } else {
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = 8 * c + 2 * e;
        const uint32_t lo = col0 + k < ncols ? r[k] : 0u;
        const uint32_t hi = col0 + k + 1 < ncols ? r[k + 1] : 0u;
        w[e] = lo | (hi << 16);
      }
      m[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

template <int N>
__device__ __forceinline__ void apply_bias_row(uint32_t* s, const uint4* m, float inv_scale) {
#pragma unroll
  for (int c = 0; c < N / 8; ++c) {
    const uint32_t w[4] = {m[c].x, m[c].y, m[c].z, m[c].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s[8 * c + 2 * e] = __float_as_uint(
          fmaf(bf16_bits(w[e] & 0xffffu), inv_scale, __uint_as_float(s[8 * c + 2 * e])));
      s[8 * c + 2 * e + 1] = __float_as_uint(
          fmaf(bf16_bits(w[e] >> 16), inv_scale, __uint_as_float(s[8 * c + 2 * e + 1])));
    }
  }
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

// Coalesced row stores for epilogues in which lane i of a warp holds row
// row0 + i (the TMEM lane layout): storing straight from the lanes makes every
// store instruction touch 32 rows.  Instead each lane puts its row -- NC
// columns, fp32 or bf16 -- into a warp-private shared-memory staging area, and
// the warp then copies rows out with each instruction covering consecutive
// 16-byte chunks of one or two rows.  Chunk c of staged row r sits at chunk
// position c ^ (r % CPR) (CPR = chunks per row, a power of two), so the lane
// writes (fixed c, 32 rows) and the copy-out reads (fixed row, consecutive c)
// both run at the minimum of four wavefronts per 512-byte instruction.
template <int NC>
struct RowStage {
  uint8_t* base;  // 32 * NC * 4 bytes of shared memory, 16-byte aligned
  bool f32;       // element type of the destination (fp32, else bf16)

  __device__ int row_bytes() const { return NC * (f32 ? 4 : 2); }
  // columns c0 .. c0 + 15 (c0 a multiple of 16, < NC) of this lane's row, times mul
  __device__ void put16(int lane, int c0, const float* x, float mul) const {
    const int rb = row_bytes(), cpr = rb / 16;
    uint8_t* row = base + lane * rb;
    if (f32) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = c0 / 4 + e;
        *reinterpret_cast<float4*>(row + 16 * (c ^ (lane & (cpr - 1)))) =
            make_float4(x[4 * e] * mul, x[4 * e + 1] * mul, x[4 * e + 2] * mul,
                        x[4 * e + 3] * mul);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = c0 / 8 + e;
        uint4 pkt;
        pkt.x = pack_bf16x2(x[8 * e + 0] * mul, x[8 * e + 1] * mul);
        pkt.y = pack_bf16x2(x[8 * e + 2] * mul, x[8 * e + 3] * mul);
        pkt.z = pack_bf16x2(x[8 * e + 4] * mul, x[8 * e + 5] * mul);
        pkt.w = pack_bf16x2(x[8 * e + 6] * mul, x[8 * e + 7] * mul);
        *reinterpret_cast<uint4*>(row + 16 * (c ^ (lane & (cpr - 1)))) = pkt;
      }
    }
  }
  // rows 0 .. nrows-1 of the stage to rows row0 .. of the view (columns col0 ..
  // col0 + NC - 1); call after every lane's put16 and a __syncwarp
  __device__ void copy_out(int lane, const View& v, int b, int h, int64_t row0, int nrows,
                           int col0) const {
    const int rb = row_bytes(), cpr = rb / 16, es = f32 ? 4 : 2;
    char* dst0 = reinterpret_cast<char*>(v.ptr) + (b * v.sb + h * v.sh + row0 * v.ss + col0) * es;
    for (int k = lane; k < nrows * cpr; k += 32) {
      const int r = k / cpr, c = k % cpr;
      const uint4 val = *reinterpret_cast<const uint4*>(base + r * rb + 16 * (c ^ (r & (cpr - 1))));
      *reinterpret_cast<uint4*>(dst0 + (int64_t)r * v.ss * es + 16 * c) = val;
    }
  }
};

// The reverse direction, for epilogues that need other rows of the same 32
// query positions (the TTT suffix segments' k or v rows): the warp fetches
// rows row0 .. row0 + nvalid - 1 (bf16, columns col0 .. col0 + NC - 1) with
// 16-byte asynchronous copies, each instruction covering consecutive chunks of
// one or two rows, into a warp-private area where row r keeps its chunks
// XOR-swizzled by r (the RowStage layout); lane r then reads its own row from
// there.  Rows at or past nvalid are not fetched and must not be read.
template <int NC>
struct RowFetch {
  static constexpr int RB = NC * 2;    // bytes per staged row
  static constexpr int CPR = RB / 16;  // 16-byte chunks per row (a power of two)
  uint8_t* base;                       // 32 * RB bytes of shared memory, 16-byte aligned

  __device__ void issue(int lane, const View& v, int b, int h, int64_t row0, int nvalid,
                        int col0) const {
    const char* src0 = reinterpret_cast<const char*>(v.ptr) +
                       (b * v.sb + h * v.sh + row0 * v.ss + col0) * 2;
    for (int k = lane; k < nvalid * CPR; k += 32) {
      const int r = k / CPR, c = k % CPR;
      cp_async16(base + r * RB + 16 * (c ^ (r & (CPR - 1))), src0 + (int64_t)r * v.ss * 2 + 16 * c);
    }
  }
  // x[0..15] += w * (columns 16 c2 .. 16 c2 + 15 of this lane's row)
  __device__ void axpy16(int lane, int c2, float w, float* x) const {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * c2 + h;
      const uint4 ra = *reinterpret_cast<const uint4*>(base + lane * RB + 16 * (c ^ (lane & (CPR - 1))));
      const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&ra);
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        const float2 rf = __bfloat1622float2(r2[f]);
        x[8 * h + 2 * f] = fmaf(w, rf.x, x[8 * h + 2 * f]);
        x[8 * h + 2 * f + 1] = fmaf(w, rf.y, x[8 * h + 2 * f + 1]);
      }
    }
  }
};

// Skipped work is made visible: a CTA that computes nothing (the device error
// word was already set when it started) or gave up part-way (one of its waits
// ran out of budget) writes NaN where its results would go, so that stale
// memory can never pass for a result.
__device__ __forceinline__ float nan_f32() { return __int_as_float(0x7fc00000); }

// NaN over columns c_begin, c_begin + step, ... (16-column chunks) of one row.
__device__ __forceinline__ void poison_row(const View& v, int b, int h, int64_t s, int c_begin,
                                           int c_step, int D, bool f32) {
  float x[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) x[e] = nan_f32();
  for (int c0 = c_begin; c0 < D; c0 += c_step) store16(v, b, h, s, c0, x, 1.f, f32);
}

// NaN over rows [s0, s0 + n) of an output view, by all threads of the CTA.
__device__ __forceinline__ void poison_rows(const View& v, int b, int h, int64_t s0, int n, int D,
                                            bool f32) {
  const int chunks = D / 16;
  float x[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) x[e] = nan_f32();
  for (int i = threadIdx.x; i < n * chunks; i += blockDim.x)
    store16(v, b, h, s0 + i / chunks, (i % chunks) * 16, x, 1.f, f32);
}

}  // namespace attn
