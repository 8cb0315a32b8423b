// bwd.cu -- deterministic fused attention backward on tcgen05 (sm_103a).
//
// The backward recomputes the weights from the saved LSE (CS336 README,
// "Flash Attention (Triton)": P is recomputed from L) and never stores the
// S x S score matrix.  It uses no atomics and a fixed schedule, so results are
// bitwise reproducible (HOT-Step flash-attn-training, section 1, asks the same
// of its backward: no floating-point atomics, a fixed order of accumulation):
//
//   1. prep:  Delta[q] = sum_d dO[q,d] O[q,d]               (fp32, from bf16)
//   2. dK/dV: one CTA per (b, kv head, 128-key tile) owns its dK and dV rows.
//             It walks the group's q heads in ascending order and, for each,
//             its visible query tiles in ascending order:
//               S^T = K Q^T,  P^T = exp(c S^T - LSE),  dV += P^T dO,
//               dP^T = V dO^T,  dS^T = P^T (dP^T - Delta),  dK += dS^T Q
//             and writes dK (times c) and dV once.
//   3. dQ:    one CTA per (b, q head, 128-query tile) walks its visible key
//             tiles in ascending order:
//               S = Q K^T, dP = dO V^T, dS = P (dP - Delta), dQ += dS K
//             then adds the TTT suffix-diagonal terms and writes c dQ once.
//   4. TTT:   the keys of appended segments (one diagonal each) get
//             dV = sum_g p dO and dK = c sum_g dS q, summed over the group's
//             q heads in ascending order; one warp per key row r serves the
//             key i*Sq + r of every segment i, reading each q and dO row once.
//
// Tensor-core kernels use 12 warps: 0-7 elementwise (two warpgroups split the
// 128 columns of each S / dP tile; thread = TMEM lane = row), 8 TMA producer,
// 9 tcgen05 issuer, 10-11 idle (their registers go to the elementwise warps).
// P^T, dS^T and dS are written back to tensor memory as bf16 and used as the
// A operand of the next MMA directly from there.
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"
#include "rows.cuh"
#include "sched.cuh"
#include "tile.cuh"
#include "trace.cuh"

namespace attn {
namespace {

constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) break;
  }
}


// ===================================================================== prep
// Dot product of two 8-element bf16 chunks (fp32 accumulate).
__device__ __forceinline__ float dot8(const uint4& x, const uint4& y) {
  const __nv_bfloat162* xv = reinterpret_cast<const __nv_bfloat162*>(&x);
  const __nv_bfloat162* yv = reinterpret_cast<const __nv_bfloat162*>(&y);
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 xf = __bfloat1622float2(xv[e]);
    const float2 yf = __bfloat1622float2(yv[e]);
    acc = fmaf(xf.x, yf.x, acc);
    acc = fmaf(xf.y, yf.y, acc);
  }
  return acc;
}

// Delta[b, h, q] = sum_d dO * O.  D/8 threads per row, 16-byte loads.  For a
// TTT step t > 0 the same row group also computes, for each suffix diagonal
// i = 1..t (key row i*Sq + q), p_i = exp(c q.k_i - LSE) and
// ds_i = p_i (dO.v_i - Delta), for the dQ epilogue and the suffix-key pass.
// TTT: instantiated separately for steps with suffix diagonals, so that their
// registers do not lower the occupancy of the plain Delta pass.
template <int D, bool TTT>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BwdArgs a) {
  constexpr int TPR = D / 8;  // threads per row
  constexpr int RPB = 256 / TPR;
  const int64_t total = (int64_t)a.d.B * a.d.Hq * a.d.Sq;
  const int64_t row = (int64_t)blockIdx.x * RPB + threadIdx.x / TPR;
  const int sub = threadIdx.x % TPR;
  const bool in = row < total;
  float acc = 0.f;
  int q = 0, h = 0, b = 0;
  uint4 ga = make_uint4(0u, 0u, 0u, 0u);
  // TTT: the q row, LSE and the k, v rows of the first diagonal are loaded
  // together with dO and O, and each later diagonal's rows one step ahead of
  // its reduction, so that the loads' latencies overlap
  uint4 qa = make_uint4(0u, 0u, 0u, 0u), kk = qa, vv = qa;
  float lse2 = 0.f;
  if (in) {
    q = (int)(row % a.d.Sq);
    const int bh = (int)(row / a.d.Sq);
    h = bh % a.d.Hq;
    b = bh / a.d.Hq;
    if constexpr (TTT) {
      const int hk = h / a.d.G;
      qa = *reinterpret_cast<const uint4*>(row_ptr(a.q, b, h, q) + sub * 8);
      lse2 = a.lse[row] * kLog2e;
      kk = *reinterpret_cast<const uint4*>(row_ptr(a.k, b, hk, (int64_t)a.d.Sq + q) + sub * 8);
      vv = *reinterpret_cast<const uint4*>(row_ptr(a.v, b, hk, (int64_t)a.d.Sq + q) + sub * 8);
    }
    const __nv_bfloat16* g = row_ptr(a.dout, b, h, q) + sub * 8;
    ga = *reinterpret_cast<const uint4*>(g);
    const __nv_bfloat162* gv = reinterpret_cast<const __nv_bfloat162*>(&ga);
    float of[8];
    if (a.d.out_f32) {
      const float* o = reinterpret_cast<const float*>(a.o.ptr) + b * a.o.sb + h * a.o.sh +
                       (int64_t)q * a.o.ss + sub * 8;
      const float4 o0 = *reinterpret_cast<const float4*>(o);
      const float4 o1 = *reinterpret_cast<const float4*>(o + 4);
      of[0] = o0.x; of[1] = o0.y; of[2] = o0.z; of[3] = o0.w;
      of[4] = o1.x; of[5] = o1.y; of[6] = o1.z; of[7] = o1.w;
    } else {
      const uint4 oa = *reinterpret_cast<const uint4*>(row_ptr(a.o, b, h, q) + sub * 8);
      const __nv_bfloat162* ov = reinterpret_cast<const __nv_bfloat162*>(&oa);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(ov[e]);
        of[2 * e] = f.x;
        of[2 * e + 1] = f.y;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 gf = __bfloat1622float2(gv[e]);
      acc = fmaf(of[2 * e], gf.x, acc);
      acc = fmaf(of[2 * e + 1], gf.y, acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, TPR);
  if (in && sub == 0) a.delta[row] = acc;

  if constexpr (TTT) {
    const int t = a.d.geom.ttt;  // uniform over the grid, > 0
    const int hk = h / a.d.G;
    const bool diag_vis = in && q < with_len(a.d.geom, a.d.seqlens, b).kv_len;
    for (int i = 1; i <= t; ++i) {
      const uint4 kc = kk, vc = vv;
      if (in && i < t) {
        const int64_t kr = (int64_t)(i + 1) * a.d.Sq + q;
        kk = *reinterpret_cast<const uint4*>(row_ptr(a.k, b, hk, kr) + sub * 8);
        vv = *reinterpret_cast<const uint4*>(row_ptr(a.v, b, hk, kr) + sub * 8);
      }
      float s = dot8(qa, kc), dp = dot8(ga, vc);
#pragma unroll
      for (int off = TPR / 2; off > 0; off >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, off, TPR);
        dp += __shfl_xor_sync(0xffffffffu, dp, off, TPR);
      }
      if (in && sub == 0) {
        // the diagonals of rows at or past the batch entry's key length are masked
        // (their weight and score gradient are 0, and so are their dK, dV and dQ terms)
        const float p = diag_vis ? ex2_approx(fmaf(s, a.d.scale_log2, -lse2)) : 0.f;
        a.ttt_p[row * t + (i - 1)] = p;
        a.ttt_ds[row * t + (i - 1)] = p * (dp - acc);
      }
    }
  }
}

// Additive mask transpose for the dK/dV pass (which reads the mask by key
// row): M [Bm][Sq][Skv] -> workspace [Bm][Skv][SqT], 64 x 64 tiles through
// shared memory, both sides coalesced; columns q >= Sq of the copy are zero.
__global__ void __launch_bounds__(256) mask_transpose_kernel(const BwdArgs a) {
  __shared__ uint16_t tile[64][65];
  const Dims& d = a.d;
  const int k0 = blockIdx.x * 64, q0 = blockIdx.y * 64, b = blockIdx.z;
  const uint16_t* src = d.addm + b * d.addm_sb;
  uint16_t* dst = a.addm_t + b * a.addm_t_sb;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;  // 64 x 4 threads
  for (int r = ty; r < 64; r += 4) {
    const int q = q0 + r, kv = k0 + tx;
    tile[r][tx] = (q < d.Sq && kv < d.Skv) ? src[(int64_t)q * d.addm_sq + kv] : (uint16_t)0;
  }
  __syncthreads();
  for (int r = ty; r < 64; r += 4) {
    const int kv = k0 + r, q = q0 + tx;
    if (kv < d.Skv && q < a.addm_t_sq) dst[(int64_t)kv * a.addm_t_sq + q] = tile[tx][r];
  }
}

// ===================================================================== dK/dV
template <int D>
struct DkdvLayout {
  using TG = TileGeom<D>;
  static constexpr int NST = (D == 128) ? 2 : (D == 64 ? 4 : 6);
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TG::TILE_BYTES;
  static constexpr int ST_OFF = 2 * TG::TILE_BYTES;              // stages: Q, dO
  static constexpr int STAGE_BYTES = 2 * TG::TILE_BYTES;
  static constexpr int STAT_OFF = ST_OFF + NST * STAGE_BYTES;  // per stage: -lse2[128], delta[128]
  static constexpr int BAR_OFF = STAT_OFF + NST * 2 * 128 * 4;
  // kv_full, qdo_full[NST], qdo_empty[NST], s_full[2], dp_full, p_ready[2], ds_ready, done, drain
  static constexpr int NBAR = 1 + 2 * NST + 8;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BYTES = MISC_OFF + 16;
  // at least 116 KB so that only one CTA fits per SM: each holds all 512 TMEM columns
  static constexpr int ALLOC = (BYTES + 1024 > 116 * 1024) ? BYTES + 1024 : 116 * 1024;
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

// W: the mask has a lower key bound (window) or per-batch key lengths; the
// other masks take the one-sided form of the tile arithmetic.
// W: general mask arithmetic (window, key lengths, additive mask); M (implies
// W): an additive mask is present, in an instantiation of its own.
// NaN over rows [k0, k0 + n) of dK and dV (a CTA that skips its work); kept
// out of line so that it costs the kernel's register allocation nothing.
__device__ __noinline__ void poison_key_rows(const BwdArgs& a, int b, int hk, int k0, int n,
                                             int D) {
  poison_rows(a.dk, b, hk, k0, n, D, a.d.out_f32 != 0);
  poison_rows(a.dv, b, hk, k0, n, D, a.d.out_f32 != 0);
}

template <int D, bool W, bool M>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const BwdArgs a) {
  using TG = TileGeom<D>;
  using L = DkdvLayout<D>;
  constexpr int NST = L::NST;
  // tensor memory: S^T (two buffers at D <= 64, where the columns allow), dP^T,
  // then the dV and dK accumulators
  constexpr bool DB = D <= 64;
  constexpr uint32_t T_DP = DB ? 256 : 128;
  constexpr uint32_t T_DV = DB ? 384 : 256;
  extern __shared__ uint8_t smem_raw[];

  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* kv_full = bars;
  uint64_t* qdo_full = bars + 1;
  uint64_t* qdo_empty = qdo_full + NST;
  uint64_t* s_full = qdo_empty + NST;  // [2]
  uint64_t* dp_full = s_full + 2;
  // p_ready alternates between two barriers: with S^T double-buffered a warp
  // can reach iteration it + 1 before a slower warp has arrived for it, and one
  // barrier would count that early arrival toward the wrong phase (S^T of
  // iteration it + 2 is issued only after p_ready(it) completes, so two suffice)
  uint64_t* p_ready = dp_full + 1;  // [2]
  uint64_t* ds_ready = p_ready + 2;
  uint64_t* done = ds_ready + 1;
  uint64_t* drain = done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  float* stats = reinterpret_cast<float*>(smem + L::STAT_OFF);  // [NST][2][128]

  const Dims& d = a.d;
  const int BH = d.B * d.Hkv;
  // heaviest key tiles (smallest k0 under causal/TTT) first
  const int kt = (int)(blockIdx.x / BH);
  const int bh = blockIdx.x % BH;
  const int hk = bh % d.Hkv;
  const int b = bh / d.Hkv;
  const int k0 = kt * kBN;
  if (*reinterpret_cast<volatile uint32_t*>(a.ctl.err) != 0) {
    // sticky device error: no work; NaN over this CTA's dK and dV rows
    poison_key_rows(a, b, hk, k0, min(kBN, d.geom.kv_main - k0), D);
    return;
  }
  // the work item must exist (ATTN_DEBUG)
  if (!ATTN_CHECK(a.ctl.err, k0 < d.geom.kv_main && hk < d.Hkv && b < d.B, 7)) return;
  // this batch entry's geometry; query tiles qt_begin .. qt_begin + n_q - 1 see the key tile
  const MaskGeom g = W ? with_len(d.geom, d.seqlens, b) : d.geom;
  int qt_begin, n_q;
  sched_q_tiles<W>(g, k0, &qt_begin, &n_q);
  const int N = n_q * d.G;

  const int warp = warp_id();
  const int lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&qdo_full[s], 2);  // the copies' expect_tx and the LSE / Delta rows
      mbar_init(&qdo_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(dp_full, 1);
    mbar_init(&p_ready[0], 256);
    mbar_init(&p_ready[1], 256);
    mbar_init(ds_ready, 256);
    mbar_init(done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{a.ctl.err, abort_flag, a.ctl.budget_ns};

  auto iter_head = [&](int it) { return hk * d.G + it / n_q; };
  auto iter_q0 = [&](int it) { return (qt_begin + it % n_q) * kBM; };

  if (warp >= 8) {
    regs_shrink();  // producer / MMA warpgroup (warps 10, 11 idle)
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (N > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tdo);
        mbar_arrive_expect_tx(kv_full, 2 * TG::TILE_BYTES);
        TG::load(smem + L::K_OFF, &tk, kv_full, k0, hk, b, d.geom.kv_main, d.Hkv, d.B,
                 a.ctl.err, 5);
        TG::load(smem + L::V_OFF, &tv, kv_full, k0, hk, b, d.geom.kv_main, d.Hkv, d.B,
                 a.ctl.err, 5);
      }
      int issued = 0;
      for (int it = 0; it < N; ++it) {
        const int s = it % NST;
        const uint32_t ph = (uint32_t)(it / NST) & 1u;
        if (!mbar_wait_warp(&qdo_empty[s], ph ^ 1u, ctl)) break;
        const int h = iter_head(it);
        const int q0 = iter_q0(it);
        // the copies go out first; the LSE / Delta rows (plain loads, an L2 round
        // trip) follow and are published by a second arrival on the same barrier
        if (lane == 0) {
          mbar_arrive_expect_tx(&qdo_full[s], 2 * TG::TILE_BYTES);
          uint8_t* dst = smem + L::ST_OFF + s * L::STAGE_BYTES;
          TG::load(dst, &tq, &qdo_full[s], q0, h, b, d.Sq, d.Hq, d.B, a.ctl.err, 6);
          TG::load(dst + TG::TILE_BYTES, &tdo, &qdo_full[s], q0, h, b, d.Sq, d.Hq, d.B,
                   a.ctl.err, 6);
        }
        float* st = stats + s * 256;
        const int64_t rbase = ((int64_t)b * d.Hq + h) * d.Sq;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = lane * 4 + e;
          const int qq = q0 + r;
          const bool in = qq < d.Sq;
          st[r] = in ? -a.lse[rbase + qq] * kLog2e : -INFINITY;  // -LSE in log2 units
          st[128 + r] = in ? a.delta[rbase + qq] : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&qdo_full[s]);
        issued = it + 1;
      }
      if (lane == 0 && *abort_flag) {
        drain_wait(kv_full, 0);
        for (int it = issued - NST < 0 ? 0 : issued - NST; it < issued; ++it)
          drain_wait(&qdo_full[it % NST], (uint32_t)(it / NST) & 1u);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------- MMA
    if (lane == 0 && N > 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_g = make_idesc_bf16(128, D, false, true);
      const uint64_t dK = TG::kmajor_base(smem_u32(smem + L::K_OFF));
      const uint64_t dV = TG::kmajor_base(smem_u32(smem + L::V_OFF));
      const uint64_t dSTk = TG::kmajor_base(smem_u32(smem + L::ST_OFF));   // stage 0, K-major
      const uint64_t dSTm = TG::mnmajor_base(smem_u32(smem + L::ST_OFF));  // stage 0, MN-major
      auto stage = [&](int it) { return TG::bytes((it % NST) * L::STAGE_BYTES); };
      constexpr uint64_t kDo = TG::bytes(TG::TILE_BYTES);  // dO follows Q in a stage
      auto issue_st = [&](int it) {  // S^T = K Q^T into buffer it % 2 (one buffer at D = 128)
        const uint64_t qd = dSTk + stage(it);
        const uint32_t col = DB ? 128u * (uint32_t)(it & 1) : 0u;
#pragma unroll
        for (int kk = 0; kk < TG::KSTEPS; ++kk)
          umma_ss(tmem + col, dK + TG::kmajor_step(kk), qd + TG::kmajor_step(kk), idesc_s, kk > 0);
        umma_commit(&s_full[DB ? (it & 1) : 0]);
      };
      auto issue_dpt = [&](int it) {  // dP^T = V dO^T
        const uint64_t od = dSTk + stage(it) + kDo;
#pragma unroll
        for (int kk = 0; kk < TG::KSTEPS; ++kk)
          umma_ss(tmem + T_DP, dV + TG::kmajor_step(kk), od + TG::kmajor_step(kk), idesc_s,
                  kk > 0);
        umma_commit(dp_full);
      };
      // A operand in TMEM: q columns 16kk.. of warpgroup kk/4 live at 64*(kk/4) + 8*(kk%4)
      auto issue_grad = [&](uint32_t acc_col, uint32_t a_col, uint64_t bd, bool acc) {
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          umma_ts(tmem + acc_col, tmem + a_col + 64 * (kk / 4) + 8 * (kk % 4),
                  bd + TG::mnmajor_step(kk), idesc_g, (acc || kk > 0) ? 1u : 0u);
      };
      auto wait_stage = [&](int it) {
        return mbar_wait(&qdo_full[it % NST], (uint32_t)(it / NST) & 1u, ctl);
      };
      // Issue order.  D = 128: S^T(0), dP^T(0), then per query tile: dV(it),
      // S^T(it+1) (its columns held P^T(it)), dK(it), dP^T(it+1) (its columns held
      // dS^T(it)).  D <= 64, two S^T buffers: S^T(0), dP^T(0), S^T(1), then per tile:
      // dV(it), S^T(it+2) into the buffer dV(it) just read, dK(it), dP^T(it+1) -- the
      // elementwise warps find S^T(it+1) ready when they finish tile it.
      bool ok = mbar_wait(kv_full, 0, ctl) && wait_stage(0);
      if (ok) {
        tc_fence_after();
        issue_st(0);
        issue_dpt(0);
        if (DB && N > 1 && (ok = wait_stage(1))) {
          tc_fence_after();
          issue_st(1);
        }
      }
      for (int it = 0; ok && it < N; ++it) {
        ATTN_TR(1, 0, it);
        if (!(ok = mbar_wait(&p_ready[it & 1], (uint32_t)(it >> 1) & 1u, ctl))) break;
        ATTN_TR(1, 1, it);
        tc_fence_after();
        issue_grad(T_DV, DB ? 128u * (uint32_t)(it & 1) : 0u, dSTm + stage(it) + kDo,
                   it > 0);  // dV += P^T dO
        const int next_s = DB ? it + 2 : it + 1;
        if (next_s < N) {
          if (!(ok = wait_stage(next_s))) break;
          ATTN_TR(1, 2, it);
          tc_fence_after();
          issue_st(next_s);
        }
        if (!(ok = mbar_wait(ds_ready, (uint32_t)it & 1u, ctl))) break;
        ATTN_TR(1, 3, it);
        tc_fence_after();
        issue_grad(T_DV + D, T_DP, dSTm + stage(it), it > 0);  // dK += dS^T Q
        umma_commit(&qdo_empty[it % NST]);
        if (it + 1 < N) issue_dpt(it + 1);
        ATTN_TR(1, 4, it);
      }
      if (ok) {
        umma_commit(done);
      } else {
        umma_commit(drain);
        drain_wait(drain, 0);
      }
    }
  }
  } else {
    regs_grow();  // elementwise warpgroups
    // ------------------------------------------------------- elementwise
    const int wg = warp >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int kv = k0 + r;
    const FullRange full_q = full_rows_for_keys(g, k0);  // query tiles without masking (W)
    const float inv_scale = 1.f / d.scale;                // additive mask as M / scale (W)
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tdP = tmem + lane_base + T_DP + 64 * wg;  // dP^T / dS^T columns of this WG
    const float sl2 = d.scale_log2;
    bool ok = true;
    for (int it = 0; it < N; ++it) {
      const int s = it % NST;
      const int q0 = iter_q0(it);
      const float* nlse2 = stats + s * 256 + 64 * wg;  // -LSE * log2(e)
      const float* dl = stats + s * 256 + 128 + 64 * wg;
      const bool tr = lane == 0 && quad == 0;
      if (tr) ATTN_TR(2 + wg, 0, it);
      // additive mask (transposed copy, by key row): loaded before the wait for S^T
      const bool addm = M && kv < d.Skv;
      uint4 mreg[M ? 8 : 1];
      if constexpr (M) {
        if (addm)
          load_bias_row<64>(mreg, a.addm_t + b * a.addm_t_sb + (int64_t)kv * a.addm_t_sq,
                            q0 + 64 * wg, d.Sq);
      }
      if (!(ok = mbar_wait_warp(&s_full[DB ? (it & 1) : 0],
                                (uint32_t)(DB ? (it >> 1) : it) & 1u, ctl)))
        break;
      // S^T / P^T columns of this WG (buffer it % 2 at D <= 64)
      const uint32_t tS = tmem + lane_base + (DB ? 128u * (uint32_t)(it & 1) : 0u) + 64 * wg;
      if (tr) ATTN_TR(2 + wg, 1, it);
      tc_fence_after();
      uint32_t raw[64];
      if constexpr (D <= 64) tmem_ld64(tS, raw); else tmem_ld32x2(tS, tS + 32, raw);
      // key row kv sees query columns [clo, chi] of the tile; rows past Sq have
      // -lse2 = -inf.  Masked scores go to -inf (exponential 0) in a pass of its own,
      // so that the exponential loop of full tiles carries no per-element select.
      if constexpr (M) {
        if (addm) apply_bias_row<64>(raw, mreg, inv_scale);
      }
      if (sched_col_tile_masked<W>(g, full_q, q0, k0)) {
        int clo, chi;
        sched_col_rows<W>(g, kv, q0 + 64 * wg, &clo, &chi);
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < clo || c > chi) raw[c] = __float_as_uint(-INFINITY);
      }
      float p[64];
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + c);
        float x[4];
        fma2(x[0], x[1], __uint_as_float(raw[c]), __uint_as_float(raw[c + 1]), sl2, sl2, l4.x, l4.y);
        fma2(x[2], x[3], __uint_as_float(raw[c + 2]), __uint_as_float(raw[c + 3]), sl2, sl2, l4.z,
             l4.w);
#pragma unroll
        for (int e = 0; e < 4; ++e) p[c + e] = ex2_approx(x[e]);
      }
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(p[2 * c], p[2 * c + 1]);
      tmem_st32(tS, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_ready[it & 1]);
      if (tr) ATTN_TR(2 + wg, 2, it);

      if (!(ok = mbar_wait_warp(dp_full, (uint32_t)it & 1u, ctl))) break;
      if (tr) ATTN_TR(2 + wg, 3, it);
      tc_fence_after();
      if constexpr (D <= 64) tmem_ld64(tdP, raw); else tmem_ld32x2(tdP, tdP + 32, raw);
      // dS = P (dP - Delta); packed pairs measure faster except at D = 128, where
      // they cost registers the kernel does not have to spare
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 d4 = *reinterpret_cast<const float4*>(dl + c);
        if constexpr (D == 128) {
          p[c + 0] = p[c + 0] * (__uint_as_float(raw[c + 0]) - d4.x);
          p[c + 1] = p[c + 1] * (__uint_as_float(raw[c + 1]) - d4.y);
          p[c + 2] = p[c + 2] * (__uint_as_float(raw[c + 2]) - d4.z);
          p[c + 3] = p[c + 3] * (__uint_as_float(raw[c + 3]) - d4.w);
        } else {
          sub_mul2(p[c], p[c + 1], __uint_as_float(raw[c]), __uint_as_float(raw[c + 1]), d4.x,
                   d4.y, p[c], p[c + 1]);
          sub_mul2(p[c + 2], p[c + 3], __uint_as_float(raw[c + 2]), __uint_as_float(raw[c + 3]),
                   d4.z, d4.w, p[c + 2], p[c + 3]);
        }
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(p[2 * c], p[2 * c + 1]);
      tmem_st32(tdP, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(ds_ready);
      if (tr) ATTN_TR(2 + wg, 4, it);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && N > 0) ok = mbar_wait_warp(done, 0, ctl);
    if (ok) {
      const bool store = kv < g.kv_main;
      const bool f32 = d.out_f32 != 0;
      if (N > 0) tc_fence_after();
      for (int c0 = 16 * wg; c0 < D; c0 += 32) {
        float vals[16];
        uint32_t raw[16];
        if (N > 0) {
          tmem_ld16(tmem + lane_base + T_DV + c0, raw);
#pragma unroll
          for (int e = 0; e < 16; ++e) vals[e] = __uint_as_float(raw[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) vals[e] = 0.f;
        }
        if (store) store16(a.dv, b, hk, kv, c0, vals, 1.f, f32);
        if (N > 0) {
          tmem_ld16(tmem + lane_base + T_DV + D + c0, raw);
#pragma unroll
          for (int e = 0; e < 16; ++e) vals[e] = __uint_as_float(raw[e]);
        }
        if (store) store16(a.dk, b, hk, kv, c0, vals, d.scale, f32);
      }
    } else if (kv < g.kv_main) {
      // a wait of this CTA ran out of budget: NaN instead of a partial result
      poison_row(a.dv, b, hk, kv, 16 * wg, 32, D, d.out_f32 != 0);
      poison_row(a.dk, b, hk, kv, 16 * wg, 32, D, d.out_f32 != 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ======================================================================= dQ
template <int D>
struct DqLayout {
  using TG = TileGeom<D>;
  // K and V have their own rings: a K tile is held until dQ += dS K of its
  // iteration retires, a V tile only until dP = dO V^T does, so K needs the
  // deeper ring to keep the copies a full iteration ahead
  static constexpr int NK = (D == 128) ? 3 : (D == 64 ? 5 : 8);
  static constexpr int NV = (D == 128) ? 2 : (D == 64 ? 4 : (D == 32 ? 6 : 8));
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = TG::TILE_BYTES;
  static constexpr int K_OFF = 2 * TG::TILE_BYTES;
  static constexpr int V_OFF = K_OFF + NK * TG::TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + NV * TG::TILE_BYTES;
  // qdo_full, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_full[2], dp_full,
  // dp_free, ds_ready[2], done, drain
  static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 8;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BYTES = MISC_OFF + 16;
  // at least 116 KB so that only one CTA fits per SM: each holds all 512 TMEM columns
  static constexpr int ALLOC = (BYTES + 1024 > 116 * 1024) ? BYTES + 1024 : 116 * 1024;
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

template <int D, bool W, bool M>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const BwdArgs a) {
  using TG = TileGeom<D>;
  using L = DqLayout<D>;
  constexpr int NK = L::NK, NV = L::NV;
  // tensor memory: S in two buffers (S(j) in buffer j % 2), dP, the dQ
  // accumulator.  Once the elementwise warps have read S(j), its buffer takes
  // dS(j) (bf16) as the A operand of dQ += dS K, so that dP(j+1) can be
  // computed as soon as dP(j) has been read and S(j+1) long before it is needed.
  constexpr int T_S = 0, T_DP = 256, T_DQ = 384;
  extern __shared__ uint8_t smem_raw[];

  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* qdo_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;  // [2]
  uint64_t* dp_full = s_full + 2;
  uint64_t* dp_free = dp_full + 1;
  // ds_ready alternates between two barriers: dP(j + 1) is issued once every
  // warp has read dP(j), so a warp can finish tile j + 1 before a slower one has
  // arrived for tile j; dP(j + 2) waits for dp_free(j + 1), which every warp
  // signals after its ds_ready(j), so two barriers keep the phases apart
  uint64_t* ds_ready = dp_free + 1;  // [2]
  uint64_t* done = ds_ready + 2;
  uint64_t* drain = done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);

  const Dims& d = a.d;
  const int n_qt = cdiv(d.Sq, kBM);
  const int BH = d.B * d.Hq;
  int qt, bh;
  if (d.geom.kind == kMaskFull || d.geom.kind == kMaskWindow) {
    qt = blockIdx.x % n_qt;
    bh = blockIdx.x / n_qt;
  } else {
    qt = n_qt - 1 - (int)(blockIdx.x / BH);
    bh = blockIdx.x % BH;
  }
  const int h = bh % d.Hq;
  const int b = bh / d.Hq;
  const int hk = h / d.G;
  const int q0 = qt * kBM;
  if (*reinterpret_cast<volatile uint32_t*>(a.ctl.err) != 0) {
    // sticky device error: no work; NaN over this CTA's dQ rows
    poison_rows(a.dq, b, h, q0, min(kBM, d.Sq - q0), D, d.out_f32 != 0);
    return;
  }
  // the work item must exist (ATTN_DEBUG)
  if (!ATTN_CHECK(a.ctl.err, q0 < d.Sq && h < d.Hq && b < d.B, 10)) return;
  // this batch entry's geometry; key tiles kt0 .. kt0 + n_kv - 1
  const MaskGeom g = W ? with_len(d.geom, d.seqlens, b) : d.geom;
  int kt0, n_kv;
  sched_kv_tiles<W>(g, q0, kBM, &kt0, &n_kv);

  const int warp = warp_id();
  const int lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(qdo_full, 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) mbar_init(&s_full[x], 1);
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 8);  // one arrival per elementwise warp
    mbar_init(&ds_ready[0], 8);
    mbar_init(&ds_ready[1], 8);
    mbar_init(done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{a.ctl.err, abort_flag, a.ctl.budget_ns};

  if (warp >= 8) {
    regs_shrink();  // producer / MMA warpgroup (warps 10, 11 idle)
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_kv > 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_expect_tx(qdo_full, 2 * TG::TILE_BYTES);
      TG::load(smem + L::Q_OFF, &tq, qdo_full, q0, h, b, d.Sq, d.Hq, d.B, a.ctl.err, 8);
      TG::load(smem + L::DO_OFF, &tdo, qdo_full, q0, h, b, d.Sq, d.Hq, d.B, a.ctl.err, 8);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        if (!mbar_wait(&k_empty[j % NK], ((uint32_t)(j / NK) & 1u) ^ 1u, ctl)) break;
        mbar_arrive_expect_tx(&k_full[j % NK], TG::TILE_BYTES);
        TG::load(smem + L::K_OFF + (j % NK) * TG::TILE_BYTES, &tk, &k_full[j % NK],
                 (kt0 + j) * kBN, hk, b, g.kv_main, d.Hkv, d.B, a.ctl.err, 9);
        k_issued = j + 1;
        if (!mbar_wait(&v_empty[j % NV], ((uint32_t)(j / NV) & 1u) ^ 1u, ctl)) break;
        mbar_arrive_expect_tx(&v_full[j % NV], TG::TILE_BYTES);
        TG::load(smem + L::V_OFF + (j % NV) * TG::TILE_BYTES, &tv, &v_full[j % NV],
                 (kt0 + j) * kBN, hk, b, g.kv_main, d.Hkv, d.B, a.ctl.err, 9);
        v_issued = j + 1;
      }
      if (*abort_flag) {
        drain_wait(qdo_full, 0);
        for (int j = k_issued - NK < 0 ? 0 : k_issued - NK; j < k_issued; ++j)
          drain_wait(&k_full[j % NK], (uint32_t)(j / NK) & 1u);
        for (int j = v_issued - NV < 0 ? 0 : v_issued - NV; j < v_issued; ++j)
          drain_wait(&v_full[j % NV], (uint32_t)(j / NV) & 1u);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------- MMA
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_g = make_idesc_bf16(128, D, false, true);
      const uint64_t dQd = TG::kmajor_base(smem_u32(smem + L::Q_OFF));
      const uint64_t dDO = TG::kmajor_base(smem_u32(smem + L::DO_OFF));
      const uint64_t dKk = TG::kmajor_base(smem_u32(smem + L::K_OFF));   // K slot 0, K-major
      const uint64_t dKm = TG::mnmajor_base(smem_u32(smem + L::K_OFF));  // K slot 0, MN-major
      const uint64_t dVk = TG::kmajor_base(smem_u32(smem + L::V_OFF));   // V slot 0, K-major
      auto kslot = [](int j) { return TG::bytes((j % NK) * TG::TILE_BYTES); };
      auto vslot = [](int j) { return TG::bytes((j % NV) * TG::TILE_BYTES); };
      // dS(j) (bf16) of keys 16kk.. sits in S buffer j % 2, in the columns of warpgroup
      // kk/4: 64 (kk/4) + 8 (kk%4)
      auto issue_dq = [&](int j) {  // dQ += dS(j) K_j
        const uint64_t kd = dKm + kslot(j);
        const uint32_t ta = tmem + T_S + 128 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_ts(tmem + T_DQ, ta + 64 * (kk / 4) + 8 * (kk % 4), kd + TG::mnmajor_step(kk),
                  idesc_g, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&k_empty[j % NK]);
      };
      auto issue_s = [&](int j) {  // S(j) = Q K_j^T into buffer j % 2
        const uint64_t kd = dKk + kslot(j);
#pragma unroll
        for (int kk = 0; kk < TG::KSTEPS; ++kk)
          umma_ss(tmem + T_S + 128 * (j & 1), dQd + TG::kmajor_step(kk),
                  kd + TG::kmajor_step(kk), idesc_s, kk > 0);
        umma_commit(&s_full[j & 1]);
      };
      auto issue_dp = [&](int j) {  // dP(j) = dO V_j^T
        const uint64_t vd = dVk + vslot(j);
#pragma unroll
        for (int kk = 0; kk < TG::KSTEPS; ++kk)
          umma_ss(tmem + T_DP, dDO + TG::kmajor_step(kk), vd + TG::kmajor_step(kk), idesc_s,
                  kk > 0);
        umma_commit(dp_full);
        umma_commit(&v_empty[j % NV]);
      };
      // issue order: S(0), dP(0), S(1), then per tile j: dP(j+1), dQ(j), S(j+2).
      // dP(j+1) waits only until dP(j) has been read; S(j+2) reuses the buffer of
      // S(j) and dS(j), so it follows dQ(j)
      bool ok = mbar_wait(qdo_full, 0, ctl) && mbar_wait(&k_full[0], 0, ctl);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = mbar_wait(&v_full[0], 0, ctl);
      }
      if (ok) {
        tc_fence_after();
        issue_dp(0);
        if (n_kv > 1 && (ok = mbar_wait(&k_full[1 % NK], (uint32_t)(1 / NK) & 1u, ctl))) {
          tc_fence_after();
          issue_s(1);
        }
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        ATTN_TR(1, 0, j);
        if (j + 1 < n_kv) {
          const int m = j + 1;
          ok = mbar_wait(dp_free, (uint32_t)j & 1u, ctl) &&
               mbar_wait(&v_full[m % NV], (uint32_t)(m / NV) & 1u, ctl);
          if (!ok) break;
          ATTN_TR(1, 1, j);
          tc_fence_after();
          issue_dp(m);
        }
        ATTN_TR(1, 2, j);
        if (!(ok = mbar_wait(&ds_ready[j & 1], (uint32_t)(j >> 1) & 1u, ctl))) break;
        ATTN_TR(1, 3, j);
        tc_fence_after();
        issue_dq(j);
        ATTN_TR(1, 4, j);
        if (j + 2 < n_kv) {
          const int m = j + 2;
          if (!(ok = mbar_wait(&k_full[m % NK], (uint32_t)(m / NK) & 1u, ctl))) break;
          ATTN_TR(1, 5, j);
          tc_fence_after();
          issue_s(m);
        }
        ATTN_TR(1, 6, j);
      }
      if (ok) {
        umma_commit(done);
      } else {
        umma_commit(drain);
        drain_wait(drain, 0);
      }
    }
  }
  } else {
    regs_grow();  // elementwise warpgroups
    // ------------------------------------------------------- elementwise
    const int wg = warp >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int q = q0 + r;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float sl2 = d.scale_log2;
    const int64_t rrow = ((int64_t)b * d.Hq + h) * d.Sq + q;
    const bool qin = q < d.Sq;
    const float lse2 = qin ? a.lse[rrow] * kLog2e : INFINITY;
    const float delta = qin ? a.delta[rrow] : 0.f;
    const FullRange full_k = full_keys_for_rows(g, q0);  // key tiles without masking (W)
    const float inv_scale = 1.f / d.scale;                // additive mask as M / scale (W)
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      // P first (needs only S), while the dP MMA may still be running
      const bool tr = lane == 0 && quad == 0;
      if (tr) ATTN_TR(2 + wg, 0, j);
      const int k0 = (kt0 + j) * kBN;
      // additive mask: this row's 64 values loaded before the wait for S
      const bool addm = M && qin;
      uint4 mreg[M ? 8 : 1];
      if constexpr (M) {
        if (addm)
          load_bias_row<64>(mreg, d.addm + b * d.addm_sb + (int64_t)q * d.addm_sq, k0 + 64 * wg,
                            d.Skv);
      }
      if (!(ok = mbar_wait_warp(&s_full[j & 1], (uint32_t)(j >> 1) & 1u, ctl))) break;
      if (tr) ATTN_TR(2 + wg, 1, j);
      tc_fence_after();
      uint32_t rs[64];
      const uint32_t tS = tmem + lane_base + T_S + 128 * (j & 1) + 64 * wg;
      tmem_ld32x2(tS, tS + 32, rs);
      // masked scores to -inf (their exponential is 0) in a pass of its own, so that
      // the exponential loop of full tiles carries no per-element select
      if constexpr (M) {
        if (addm) apply_bias_row<64>(rs, mreg, inv_scale);
      }
      if (sched_row_tile_masked<W>(g, full_k, q0, k0)) {
        int clo, chi;
        sched_row_cols<W>(g, q, k0 + 64 * wg, &clo, &chi);
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < clo || c > chi) rs[c] = __float_as_uint(-INFINITY);
      }
      float p[64];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float x0, x1;
        fma2_bc(x0, x1, __uint_as_float(rs[c]), __uint_as_float(rs[c + 1]), sl2, -lse2);
        p[c] = ex2_approx(x0);
        p[c + 1] = ex2_approx(x1);
      }
      if (tr) ATTN_TR(2 + wg, 2, j);
      if (!(ok = mbar_wait_warp(dp_full, (uint32_t)j & 1u, ctl))) break;
      if (tr) ATTN_TR(2 + wg, 3, j);
      tc_fence_after();
      uint32_t rp[64];
      const uint32_t tP = tmem + lane_base + T_DP + 64 * wg;
      tmem_ld32x2(tP, tP + 32, rp);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dp_free);  // dP columns free for dP(j+1)
      if (tr) ATTN_TR(2 + wg, 4, j);
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float ds0, ds1;
        sub_mul2(ds0, ds1, __uint_as_float(rp[c]), __uint_as_float(rp[c + 1]), delta, delta, p[c],
                 p[c + 1]);
        pk[c / 2] = pack_bf16x2(ds0, ds1);
      }
      if (tr) ATTN_TR(2 + wg, 5, j);
      // dS over the first half of this warpgroup's S(j) columns (already read)
      tmem_st32(tS, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_ready[j & 1]);
      if (tr) ATTN_TR(2 + wg, 6, j);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n_kv > 0) ok = mbar_wait_warp(done, 0, ctl);
    if (ok) {
      if (n_kv > 0) tc_fence_after();
      // this warpgroup's dQ columns: the contiguous half [cbeg, cend) (all of them
      // for warpgroup 0 at D = 16)
      constexpr int NCW = D >= 32 ? D / 2 : 16;
      const int cbeg = wg * NCW, cend = min(D, cbeg + NCW);
      const uint32_t tq = tmem + lane_base + T_DQ;
      if (n_kv == 0 && g.ttt > 0) {  // accumulator never written by an MMA: start at zero
        uint32_t z[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) z[e] = 0u;
        for (int c0 = cbeg; c0 < cend; c0 += 16) tmem_st16(tq + c0, z);
        tmem_st_wait();
      }
      // TTT suffix diagonals: dQ += ds_i k_i with ds_i = p_i (dO . v_i - Delta) from the
      // prep pass.  The k rows of the warp's 32 query positions (this warpgroup's
      // columns) are fetched two segments at a time into the warp's output staging
      // area (every MMA has completed, so the Q and dO tiles are free) and folded
      // into the TMEM accumulator in one pass per pair, in segment order.
      if (g.ttt > 0 && cbeg < cend) {
        const int row0 = q0 + quad * 32;
        const int nvalid = max(0, min(32, d.Sq - row0));
        uint8_t* fbase = smem + L::Q_OFF + warp * (32 * NCW * 4);
        const RowFetch<NCW> fk[2] = {{fbase}, {fbase + 32 * NCW * 2}};
        for (int i0 = 1; i0 <= g.ttt; i0 += 2) {
          const int nseg = min(2, g.ttt - i0 + 1);
          for (int u = 0; u < nseg; ++u)
            fk[u].issue(lane, a.k, b, hk, (int64_t)(i0 + u) * d.Sq + row0, nvalid, cbeg);
          cp_async_commit();
          float dsv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u)
            dsv[u] = (qin && u < nseg) ? a.ttt_ds[rrow * g.ttt + (i0 + u - 1)] : 0.f;
          cp_async_wait_all();
          __syncwarp();
          for (int c0 = cbeg; c0 < cend; c0 += 16) {
            uint32_t raw[16];
            float vals[16];
            tmem_ld16(tq + c0, raw);
#pragma unroll
            for (int e = 0; e < 16; ++e) vals[e] = __uint_as_float(raw[e]);
            if (qin) {
#pragma unroll
              for (int u = 0; u < 2; ++u)
                if (u < nseg) fk[u].axpy16(lane, (c0 - cbeg) / 16, dsv[u], vals);
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) raw[e] = __float_as_uint(vals[e]);
            tmem_st16(tq + c0, raw);
          }
          tmem_st_wait();
          __syncwarp();  // every lane has read the pair before it is refilled
        }
      }
      // the warp's 32 rows of its half go through shared memory (every MMA has
      // completed, so the Q and dO tiles are free) for coalesced global stores
      const RowStage<NCW> stage{smem + L::Q_OFF + warp * (32 * NCW * 4), d.out_f32 != 0};
      for (int c0 = cbeg; c0 < cend; c0 += 16) {
        float acc[16];
        if (n_kv > 0 || g.ttt > 0) {
          uint32_t raw[16];
          tmem_ld16(tq + c0, raw);
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] = __uint_as_float(raw[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] = 0.f;
        }
        stage.put16(lane, c0 - cbeg, acc, d.scale);
      }
      __syncwarp();
      if (cbeg < cend) {
        const int row0 = q0 + quad * 32;
        stage.copy_out(lane, a.dq, b, h, row0, min(32, max(0, d.Sq - row0)), cbeg);
      }
    } else if (qin) {
      // a wait of this CTA ran out of budget: NaN instead of a partial result
      poison_row(a.dq, b, h, q, 16 * wg, 32, D, d.out_f32 != 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================ TTT diag
// dK/dV of the keys of appended segments i = 1..t: key row i*Sq + r is seen
// only by query row r of every q head of its group.  One warp per (batch
// entry, kv head, row r) serves all t segments of that row, so each q and dO
// row is read once: lane l holds columns [l*VEC, l*VEC + VEC).  The sums over
// the group's q heads run in ascending head order.
template <int D>
struct SuffixVec {
  static constexpr int VEC = D >= 32 ? D / 32 : 1;  // columns per lane
  static constexpr int LANES = D / VEC;             // lanes holding columns
};

template <int VEC>
__device__ __forceinline__ void store_cols(void* base, int64_t off, bool f32, const float* v) {
  if (f32) {
    float* o = reinterpret_cast<float*>(base) + off;
    if constexpr (VEC == 4) {
      *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
    } else if constexpr (VEC == 2) {
      *reinterpret_cast<float2*>(o) = make_float2(v[0], v[1]);
    } else {
      o[0] = v[0];
    }
  } else {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(base) + off;
    if constexpr (VEC == 4) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]), hi = __floats2bfloat162_rn(v[2], v[3]);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(o) = u;
    } else if constexpr (VEC == 2) {
      *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(v[0], v[1]);
    } else {
      o[0] = __float2bfloat16_rn(v[0]);
    }
  }
}

// Raw bf16 columns of one lane (VEC = 4, 2 or 1), loaded in one instruction
// and widened to fp32 only when used, so that the loads of several q heads can
// be in flight together at little register cost.
template <int VEC>
struct RawCols {
  using T = typename std::conditional<VEC == 4, uint2,
                                      typename std::conditional<VEC == 2, uint32_t,
                                                                uint16_t>::type>::type;
  T v;
  __device__ void load(const __nv_bfloat16* p) { v = *reinterpret_cast<const T*>(p); }
  __device__ void widen(float* f) const {
    if constexpr (VEC == 4) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else if constexpr (VEC == 2) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
      f[0] = a.x; f[1] = a.y;
    } else {
      f[0] = bf16_bits(v);
    }
  }
};

// CH: segments per pass over the q and dO rows (1, 2, 4 or 8, the smallest
// that covers t up to 8), so that the accumulators' registers scale with t.
// The q heads of the group are taken HB at a time: their q and dO rows and
// their p / ds values (lane u holds segment i0 + u, handed to every lane by a
// shuffle) are all requested before the first is used, so that each warp
// keeps several rows of memory traffic in flight.  The sums still run over
// the heads in ascending order, one fused multiply-add per head.
template <int D, int CH>
__global__ void __launch_bounds__(256) ttt_diag_bwd_kernel(const BwdArgs a) {
  constexpr int VEC = SuffixVec<D>::VEC, LANES = SuffixVec<D>::LANES;
  constexpr int HB = CH >= 4 ? 4 : 2;  // fewer at small CH, where registers set the occupancy
  static_assert(CH <= 32, "one lane per segment of a pass");
  const Dims& d = a.d;
  const int t = d.geom.ttt;
  const int64_t rows = (int64_t)d.B * d.Hkv * d.Sq;
  const int64_t wrow = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wrow >= rows) return;
  const int lane = threadIdx.x & 31;
  const bool act = lane < LANES;
  const int c0 = lane * VEC;
  const int r = (int)(wrow % d.Sq);
  const int64_t bk = wrow / d.Sq;
  const int hk = (int)(bk % d.Hkv);
  const int b = (int)(bk / d.Hkv);
  for (int i0 = 1; i0 <= t; i0 += CH) {
    const int nch = min(CH, t - i0 + 1);  // segments in this pass
    float dk[CH][VEC], dv[CH][VEC];
#pragma unroll
    for (int u = 0; u < CH; ++u)
#pragma unroll
      for (int e = 0; e < VEC; ++e) dk[u][e] = dv[u][e] = 0.f;
    for (int g0 = 0; g0 < d.G; g0 += HB) {
      RawCols<VEC> qr[HB], gr[HB];
      float pl[HB], dsl[HB];
#pragma unroll
      for (int j = 0; j < HB; ++j) {
        const int gq = g0 + j;
        const bool hv = gq < d.G;
        const int h = hk * d.G + gq;
        const int64_t rrow = ((int64_t)b * d.Hq + h) * d.Sq + r;
        if (hv && act) {
          qr[j].load(row_ptr(a.q, b, h, r) + c0);
          gr[j].load(row_ptr(a.dout, b, h, r) + c0);
        }
        // p and ds of (query row r of q head h, segment i0 + lane) from the prep pass
        const bool pv = hv && lane < nch;
        pl[j] = pv ? a.ttt_p[rrow * t + (i0 - 1 + lane)] : 0.f;
        dsl[j] = pv ? a.ttt_ds[rrow * t + (i0 - 1 + lane)] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < HB; ++j) {
        if (g0 + j >= d.G) break;  // uniform over the warp
        float qv[VEC], gv[VEC];
        qr[j].widen(qv);
        gr[j].widen(gv);
#pragma unroll
        for (int u = 0; u < CH; ++u) {
          const float p = __shfl_sync(0xffffffffu, pl[j], u);
          const float ds = __shfl_sync(0xffffffffu, dsl[j], u);
          if (act && u < nch) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              dv[u][e] = fmaf(p, gv[e], dv[u][e]);
              dk[u][e] = fmaf(ds, qv[e], dk[u][e]);
            }
          }
        }
      }
    }
    if (act) {
#pragma unroll
      for (int u = 0; u < CH; ++u) {
        const int i = i0 + u;
        if (i > t) break;
        const int64_t kr = (int64_t)i * d.Sq + r;
        float k_out[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) k_out[e] = dk[u][e] * d.scale;
        store_cols<VEC>(a.dk.ptr, b * a.dk.sb + hk * a.dk.sh + kr * a.dk.ss + c0,
                        d.out_f32 != 0, k_out);
        store_cols<VEC>(a.dv.ptr, b * a.dv.sb + hk * a.dv.sh + kr * a.dv.ss + c0,
                        d.out_f32 != 0, dv[u]);
      }
    }
  }
}

template <int D, bool W, bool M>
cudaError_t launch_bwd_dw(const BwdArgs& a, const Maps& m, unsigned passes, cudaStream_t s) {
  cudaError_t e;
  if (passes & 1u) {
    constexpr int RPB = 256 / (D / 8);
    const int64_t rows = (int64_t)a.d.B * a.d.Hq * a.d.Sq;
    if (a.d.geom.ttt > 0)
      bwd_prep_kernel<D, true><<<(unsigned)((rows + RPB - 1) / RPB), 256, 0, s>>>(a);
    else
      bwd_prep_kernel<D, false><<<(unsigned)((rows + RPB - 1) / RPB), 256, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.addm_t != nullptr) {
      const dim3 grid((unsigned)cdiv(a.d.Skv, 64), (unsigned)cdiv((int)a.addm_t_sq, 64),
                      a.addm_t_sb == 0 ? 1u : (unsigned)a.d.B);
      mask_transpose_kernel<<<grid, 256, 0, s>>>(a);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  if (passes & 2u) {
    using L = DkdvLayout<D>;
    auto kern = bwd_dkdv_kernel<D, W, M>;
    static const cudaError_t regs_ok = check_launch_regs(reinterpret_cast<const void*>(kern));
    if (regs_ok != cudaSuccess) return regs_ok;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC)) !=
        cudaSuccess)
      return e;
    const unsigned grid = (unsigned)(cdiv(a.d.geom.kv_main, kBN) * a.d.B * a.d.Hkv);
    kern<<<grid, kThreads, L::ALLOC, s>>>(m.q, m.k, m.v, m.dout, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (passes & 4u) {
    using L = DqLayout<D>;
    auto kern = bwd_dq_kernel<D, W, M>;
    static const cudaError_t regs_ok = check_launch_regs(reinterpret_cast<const void*>(kern));
    if (regs_ok != cudaSuccess) return regs_ok;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC)) !=
        cudaSuccess)
      return e;
    const unsigned grid = (unsigned)(cdiv(a.d.Sq, kBM) * a.d.B * a.d.Hq);
    kern<<<grid, kThreads, L::ALLOC, s>>>(m.q, m.k, m.v, m.dout, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((passes & 8u) && a.d.geom.ttt > 0) {
    const int64_t rows = (int64_t)a.d.B * a.d.Hkv * a.d.Sq;  // one warp per key row r
    const unsigned grid = (unsigned)((rows + 7) / 8);
    const int t = a.d.geom.ttt;
    if (t <= 1)
      ttt_diag_bwd_kernel<D, 1><<<grid, 256, 0, s>>>(a);
    else if (t <= 2)
      ttt_diag_bwd_kernel<D, 2><<<grid, 256, 0, s>>>(a);
    else if (t <= 4)
      ttt_diag_bwd_kernel<D, 4><<<grid, 256, 0, s>>>(a);
    else
      ttt_diag_bwd_kernel<D, 8><<<grid, 256, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, const Maps& m, unsigned passes, cudaStream_t s) {
  if (a.d.addm != nullptr) return launch_bwd_dw<D, true, true>(a, m, passes, s);
  return needs_general_mask(a.d) ? launch_bwd_dw<D, true, false>(a, m, passes, s)
                                 : launch_bwd_dw<D, false, false>(a, m, passes, s);
}

}  // namespace

// Pipeline depths of the backward's tensor-core passes, for the plan description.
template <int D>
BwdShape bwd_shape_d() {
  BwdShape b;
  b.dkdv_stages = DkdvLayout<D>::NST;
  b.dq_k_ring = DqLayout<D>::NK;
  b.dq_v_ring = DqLayout<D>::NV;
  b.dkdv_smem = DkdvLayout<D>::ALLOC;
  b.dq_smem = DqLayout<D>::ALLOC;
  return b;
}
BwdShape bwd_shape(int D) {
  return D == 128 ? bwd_shape_d<128>() : D == 64 ? bwd_shape_d<64>()
         : D == 32 ? bwd_shape_d<32>() : bwd_shape_d<16>();
}

cudaError_t launch_bwd(const BwdArgs& a, const Maps& m, unsigned passes, cudaStream_t s) {
  switch (a.d.D) {
    case 16: return launch_bwd_d<16>(a, m, passes, s);
    case 32: return launch_bwd_d<32>(a, m, passes, s);
    case 64: return launch_bwd_d<64>(a, m, passes, s);
    case 128: return launch_bwd_d<128>(a, m, passes, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn

ATTN_TRACE_READER(attn_trace_read_bwd)
