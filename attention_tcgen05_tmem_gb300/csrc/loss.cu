// loss.cu -- soft-target log-softmax loss over logits [rows, V] (fp32) with
// an in-place backward (SpecForge long-context post, "In-place Gradient
// Calculation": the EAGLE3 loss of a TTT step,
//     loss = -mean_r mask[r] * sum_v target[r, v] * log_softmax(logits[r])_v,
// computed with an online softmax that keeps per-row statistics, and a
// backward that overwrites the logits with their gradient).
//
// Both passes stream HBM once: one CTA per row reads the row with 16-byte
// evict-first loads.  The forward needs a single pass where the page's
// listing makes two, because
//     sum_v p_v (x_v - lse) = sum_v p_v x_v - lse * sum_v p_v
// so the running max / sum, sum p x and sum p are accumulated together and
// combined at the end.  Instead of the page's (m, d) the forward stores
// lse = m + ln d (the backward only needs exp(x - m) / d = exp(x - lse)) and
// sum_v p_v.  Reductions run in a fixed order: the result is bitwise
// reproducible.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kLossThreads = 256;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.69314718055994531f;

// Online softmax state in the log2 domain: max of x*log2(e) and the sum of
// 2^(x*log2(e) - max).
struct Online {
  float m, d;
};

__device__ __forceinline__ Online combine(Online a, Online b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return Online{m, 0.f};
  return Online{m, a.d * ex2_approx(a.m - m) + b.d * ex2_approx(b.m - m)};
}

__device__ __forceinline__ void add4(Online& s, float& spx, float& sp, float4 x, float4 p) {
  const float x0 = x.x * kLog2eF, x1 = x.y * kLog2eF, x2 = x.z * kLog2eF, x3 = x.w * kLog2eF;
  const float mx = fmaxf(fmax3(x0, x1, x2), x3);
  if (mx > s.m) {
    s.d = (s.m == -INFINITY) ? 0.f : s.d * ex2_approx(s.m - mx);
    s.m = mx;
  }
  s.d += ex2_approx(x0 - s.m) + ex2_approx(x1 - s.m) + ex2_approx(x2 - s.m) + ex2_approx(x3 - s.m);
  spx = fmaf(p.x, x.x, fmaf(p.y, x.y, fmaf(p.z, x.z, fmaf(p.w, x.w, spx))));
  sp += (p.x + p.y) + (p.z + p.w);
}

__device__ __forceinline__ void add1(Online& s, float& spx, float& sp, float x, float p) {
  const float xl = x * kLog2eF;
  if (xl > s.m) {
    s.d = (s.m == -INFINITY) ? 0.f : s.d * ex2_approx(s.m - xl);
    s.m = xl;
  }
  s.d += ex2_approx(xl - s.m);
  spx = fmaf(p, x, spx);
  sp += p;
}

// VEC: every row of logits and target starts on a 16-byte boundary, so the
// rows stream as float4; otherwise as coalesced single floats.
template <bool VEC>
__global__ void __launch_bounds__(kLossThreads)
    logsoftmax_loss_fwd_kernel(LossArgs a) {
  const int64_t r = blockIdx.x;
  const float* x = a.logits + r * a.ld_logits;
  const float* p = a.target + r * a.ld_target;
  const int n4 = VEC ? (int)(a.V / 4) : 0;
  Online s{-INFINITY, 0.f};
  float spx = 0.f, sp = 0.f;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const float4* p4 = reinterpret_cast<const float4*>(p);
  int i = threadIdx.x;
  // four 16-byte pairs in flight per thread
  for (; i + 3 * kLossThreads < n4; i += 4 * kLossThreads) {
    float4 xv[4], pv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      xv[u] = __ldcs(x4 + i + u * kLossThreads);
      pv[u] = __ldcs(p4 + i + u * kLossThreads);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) add4(s, spx, sp, xv[u], pv[u]);
  }
  for (; i < n4; i += kLossThreads) add4(s, spx, sp, __ldcs(x4 + i), __ldcs(p4 + i));
  for (int v = 4 * n4 + threadIdx.x; v < a.V; v += kLossThreads) add1(s, spx, sp, x[v], p[v]);

  // fixed-order reduction: warp butterflies, then warp 0 over the warps
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const Online o{__shfl_xor_sync(0xffffffffu, s.m, off), __shfl_xor_sync(0xffffffffu, s.d, off)};
    s = combine(s, o);
    spx += __shfl_xor_sync(0xffffffffu, spx, off);
    sp += __shfl_xor_sync(0xffffffffu, sp, off);
  }
  __shared__ float red[4][kLossThreads / 32];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[0][w] = s.m;
    red[1][w] = s.d;
    red[2][w] = spx;
    red[3][w] = sp;
  }
  __syncthreads();
  if (w == 0) {
    constexpr int NW = kLossThreads / 32;
    Online t = lane < NW ? Online{red[0][lane], red[1][lane]} : Online{-INFINITY, 0.f};
    float tpx = lane < NW ? red[2][lane] : 0.f, tp = lane < NW ? red[3][lane] : 0.f;
#pragma unroll
    for (int off = NW / 2; off > 0; off >>= 1) {
      const Online o{__shfl_xor_sync(0xffffffffu, t.m, off), __shfl_xor_sync(0xffffffffu, t.d, off)};
      t = combine(t, o);
      tpx += __shfl_xor_sync(0xffffffffu, tpx, off);
      tp += __shfl_xor_sync(0xffffffffu, tp, off);
    }
    if (lane == 0) {
      const float lse = (t.m + lg2_approx(t.d)) * kLn2F;  // natural log
      a.row_lse[r] = lse;
      a.row_tsum[r] = tp;
      a.row_loss[r] = lse * tp - tpx;  // -sum_v p_v (x_v - lse)
    }
  }
}

// loss = sum_r mask[r] * row_loss[r] / rows, accumulated in fp64 in a fixed order.
__global__ void __launch_bounds__(1024) logsoftmax_loss_mean_kernel(LossArgs a) {
  double acc = 0.0;
  for (int64_t r = threadIdx.x; r < a.rows; r += blockDim.x)
    acc += (double)(a.mask ? a.mask[r] : 1.f) * (double)a.row_loss[r];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  __shared__ double red[32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    acc = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (threadIdx.x == 0) a.loss[0] = (float)(acc / (double)a.rows);
  }
}

// logits[r, v] <- -(g_r) (target[r, v] - softmax_v * tsum[r]),
// g_r = grad_loss * mask[r] / rows (the page's per-row grad_output).
__device__ __forceinline__ float4 grad4(float4 x, float4 p, float nlse2, float g, float c) {
  float4 o;
  o.x = fmaf(ex2_approx(fmaf(x.x, kLog2eF, nlse2)), c, -p.x * g);
  o.y = fmaf(ex2_approx(fmaf(x.y, kLog2eF, nlse2)), c, -p.y * g);
  o.z = fmaf(ex2_approx(fmaf(x.z, kLog2eF, nlse2)), c, -p.z * g);
  o.w = fmaf(ex2_approx(fmaf(x.w, kLog2eF, nlse2)), c, -p.w * g);
  return o;
}

template <bool VEC>
__global__ void __launch_bounds__(kLossThreads)
    logsoftmax_loss_bwd_kernel(LossArgs a) {
  const int64_t r = blockIdx.x;
  float* x = a.logits_out + r * a.ld_logits;
  const float* p = a.target + r * a.ld_target;
  const float gl = a.grad_loss ? a.grad_loss[0] : 1.f;
  const float g = gl * (a.mask ? a.mask[r] : 1.f) / (float)a.rows;
  const float c = g * a.row_tsum[r];
  const float nlse2 = -a.row_lse[r] * kLog2eF;
  const int n4 = VEC ? (int)(a.V / 4) : 0;
  float4* x4 = reinterpret_cast<float4*>(x);
  const float4* p4 = reinterpret_cast<const float4*>(p);
  int i = threadIdx.x;
  for (; i + 3 * kLossThreads < n4; i += 4 * kLossThreads) {
    float4 xv[4], pv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      xv[u] = __ldcs(x4 + i + u * kLossThreads);
      pv[u] = __ldcs(p4 + i + u * kLossThreads);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) __stcs(x4 + i + u * kLossThreads, grad4(xv[u], pv[u], nlse2, g, c));
  }
  for (; i < n4; i += kLossThreads) __stcs(x4 + i, grad4(__ldcs(x4 + i), __ldcs(p4 + i), nlse2, g, c));
  for (int v = 4 * n4 + threadIdx.x; v < a.V; v += kLossThreads)
    x[v] = fmaf(ex2_approx(fmaf(x[v], kLog2eF, nlse2)), c, -p[v] * g);
}

bool rows_16b_aligned(const LossArgs& a, const float* logits) {
  return a.ld_logits % 4 == 0 && a.ld_target % 4 == 0 &&
         reinterpret_cast<uintptr_t>(logits) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(a.target) % 16 == 0;
}

}  // namespace

cudaError_t launch_logsoftmax_loss_fwd(const LossArgs& a, cudaStream_t s) {
  if (rows_16b_aligned(a, a.logits))
    logsoftmax_loss_fwd_kernel<true><<<(unsigned)a.rows, kLossThreads, 0, s>>>(a);
  else
    logsoftmax_loss_fwd_kernel<false><<<(unsigned)a.rows, kLossThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.loss == nullptr) return e;
  logsoftmax_loss_mean_kernel<<<1, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_logsoftmax_loss_bwd(const LossArgs& a, cudaStream_t s) {
  if (rows_16b_aligned(a, a.logits_out))
    logsoftmax_loss_bwd_kernel<true><<<(unsigned)a.rows, kLossThreads, 0, s>>>(a);
  else
    logsoftmax_loss_bwd_kernel<false><<<(unsigned)a.rows, kLossThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace attn
