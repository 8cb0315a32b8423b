// fwd_impl.cuh -- fused attention forward on tcgen05 (sm_103a): the kernels and
// their launch templates, instantiated unsplit by fwd.cu and split by
// fwd_split.cu (two translation units, compiled in parallel).
//
// Computes, per (b, q head), O = softmax(c Q K^T + mask) V and the per-row
// natural-log LSE, streaming K/V tiles through an online softmax (CS336
// README, "Flash Attention (Triton)": running max and sum, O rescaled as tiles
// stream, LSE kept for the backward; SpecForge post, "Flex Attention": empty
// tiles skipped, full tiles skip the mask test).  The TTT suffix diagonals of
// the EAGLE3 mask (SpecForge post, "EAGLE3 Training" and "Flex Attention")
// are merged per row in the epilogue by log-sum-exp, without a dense mask.
//
// One CTA owns two 128-row query tiles of one (b, h) and 10 warps:
//   warps 0-3  softmax for query tile 0 (thread = row = TMEM lane)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q0, Q1 once, then K_j, V_j into a slot ring
//   warp  9    tcgen05 issuer (one thread) and TMEM owner
// Tensor memory (512 columns x 128 lanes of 32 bit), two S buffers:
//   [0,128) S0 / P0   [128,256) S1 / P1   [256,256+D) O0   [256+D,256+2D) O1
// (all 512 columns at D = 128)
// P (bf16, two per column) overwrites the first 64 columns of its S tile and
// is the A operand of O += P V straight from tensor memory.
//
// MMA issue order per key tile j (FA-style ping-pong, so one tile's softmax
// overlaps the other tile's MMAs):  PV0(j-1), S0(j), PV1(j-1), S1(j).
// Because tcgen05 MMAs of one thread run in issue order, S_x(j) completing
// implies PV_x(j-1) completed, which makes the O rescale wait free.
//
// D <= 64 leaves room for a third S buffer, used by the general masks
// (window, key lengths, additive): [0,384) three S / P buffers,
// [384,384+D) O0, [384+D,384+2D) O1.  Score tile n = 2j + x (tile x, key
// tile j) lives in buffer n % 3, and the issue order becomes
//     PV0(j), S1(j+1), PV1(j), S0(j+2)
// so each score tile is computed a full step before its softmax needs it,
// instead of after the previous P of the same query tile.  The O rescale
// then waits for PV_x(j-1) explicitly (rarely: only when the max grows).
// s_full and p_ready are per buffer: a buffer is refilled only after its P
// was consumed, so neither barrier can run two phases ahead of a waiter.
// o_done: S_x(j) completing implies only PV_x(j-2); the rescale wait for
// PV_x(j-1) at step j is unambiguous (PV_x(j-2) done, PV_x(j) not yet
// issued), but at the end of the row two o_done phases may be open, so the
// epilogue waits for o_last, committed once after the last PV_x.
//
// The running max is refreshed only when it grows by more than 8 (log2
// units); otherwise the stale max is kept and P stays <= 256.  O, l and m
// always share one reference, so the result is exact up to rounding.
#pragma once
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "rows.cuh"
#include "sched.cuh"
#include "tile.cuh"
#include "trace.cuh"

namespace attn {
namespace {

constexpr int kFwdThreads = 384;
constexpr float kRescaleThreshold = 8.0f;

// The TTT suffix-diagonal scores of a query row (t fp32 values) are parked in
// that row of O between the scores pre-pass and the main kernel when they fit.
__host__ __device__ inline bool ttt_scores_fit(int t, int D, int out_f32) {
  return t > 0 && t * 4 <= D * (out_f32 ? 4 : 2);
}

// Scores pre-pass: for every query row q and suffix diagonal i = 1..t (key
// row i*Sq + q), c log2(e) q . k_i, written as fp32 into the first t slots of
// the row's O storage.  D/8 threads per row, 16-byte loads, shuffle reduction.
template <int D>
__global__ void __launch_bounds__(256) ttt_scores_kernel(const FwdArgs a) {
  constexpr int TPR = D / 8;
  constexpr int RPB = 256 / TPR;
  const Dims& d = a.d;
  const int t = d.geom.ttt;
  const int64_t total = (int64_t)d.B * d.Hq * d.Sq;
  const int64_t row = (int64_t)blockIdx.x * RPB + threadIdx.x / TPR;
  const int sub = threadIdx.x % TPR;
  const bool in = row < total;
  int q = 0, h = 0, b = 0;
  uint4 qa = make_uint4(0u, 0u, 0u, 0u);
  if (in) {
    q = (int)(row % d.Sq);
    const int bh = (int)(row / d.Sq);
    h = bh % d.Hq;
    b = bh / d.Hq;
    qa = *reinterpret_cast<const uint4*>(row_ptr(a.q, b, h, q) + sub * 8);
  }
  const int hk = h / d.G;
  float* parked = reinterpret_cast<float*>(static_cast<char*>(a.o.ptr) +
                                           (b * a.o.sb + h * a.o.sh + (int64_t)q * a.o.ss) *
                                               (d.out_f32 ? 4 : 2));
  for (int i = 1; i <= t; ++i) {
    float s = 0.f;
    if (in) {
      const uint4 ka =
          *reinterpret_cast<const uint4*>(row_ptr(a.k, b, hk, (int64_t)i * d.Sq + q) + sub * 8);
      const __nv_bfloat162* qv = reinterpret_cast<const __nv_bfloat162*>(&qa);
      const __nv_bfloat162* kv = reinterpret_cast<const __nv_bfloat162*>(&ka);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 qf = __bfloat1622float2(qv[e]);
        const float2 kf = __bfloat1622float2(kv[e]);
        s = fmaf(qf.x, kf.x, s);
        s = fmaf(qf.y, kf.y, s);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off, TPR);
    if (in && sub == 0) parked[i - 1] = s * d.scale_log2;
  }
}

template <int D>
struct FwdLayout {
  using TG = TileGeom<D>;
  static constexpr int NSLOT = (D == 128) ? 5 : (D == 64 ? 6 : 8);
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = 2 * TG::TILE_BYTES;
  static constexpr int BAR_OFF = KV_OFF + NSLOT * TG::TILE_BYTES;
  // q_full, kv_full[NSLOT], kv_empty[NSLOT], s_full[3], p_ready[3], o_done[2], o_last[2],
  // drain
  static constexpr int NBAR = 1 + 2 * NSLOT + 11;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BYTES = MISC_OFF + 16;
  // at least 116 KB so that only one CTA fits per SM: each holds all 512 TMEM columns
  static constexpr int ALLOC = (BYTES + 1024 > 116 * 1024) ? BYTES + 1024 : 116 * 1024;
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

// Wait for a barrier phase with a fixed budget, ignoring the abort flag (used
// to drain copies and MMAs still in flight before the CTA exits).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) break;
  }
}

__device__ __forceinline__ float neg_inf() { return -INFINITY; }

// W: the mask has a lower key bound (window), per-batch key lengths or an
// additive mask; the other masks take the one-sided form of the tile
// arithmetic.  M (implies W): an additive mask is present (its own
// instantiation, so that the registers holding the mask row cost the other
// general masks nothing).  S: the key-range split (one CTA per chunk of a
// pair's key tiles, partial results for the merge pass); its own
// instantiation, so that the unsplit kernels carry none of its registers.
template <int D, bool W, bool M, bool S>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const FwdArgs a) {
  using TG = TileGeom<D>;
  using L = FwdLayout<D>;
  constexpr int NSLOT = L::NSLOT;
  // three rotating S buffers: for the general masks at D <= 64, whose rows
  // are short or partly masked; on long full rows the tensor pipe is the
  // bound and the two-buffer order measures faster
  constexpr bool TB = W && D <= 64;
  constexpr uint32_t O_COL = TB ? 384u : 256u;   // first O accumulator column
  extern __shared__ uint8_t smem_raw[];

  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + NSLOT;
  uint64_t* s_full = kv_empty + NSLOT;  // [3]: per tile x (D = 128) or per buffer (D <= 64)
  uint64_t* p_ready = s_full + 3;       // [3], indexed like s_full
  uint64_t* o_done = p_ready + 3;       // [2]: per query tile, one phase per PV
  uint64_t* o_last = o_done + 2;        // [2]: per query tile, after its last PV (D <= 64)
  uint64_t* drain = o_last + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);

  const Dims& d = a.d;
  // ---- work decode: causal/TTT launch the longest query-tile pairs first; with a
  // key-range split, CTA blockIdx.x takes chunk blockIdx.x % nchunk of its pair
  constexpr bool split = S;
  const int chunk = split ? (int)(blockIdx.x % (unsigned)a.nchunk) : 0;
  const unsigned bid = split ? blockIdx.x / (unsigned)a.nchunk : blockIdx.x;
  const int n_qp = cdiv(d.Sq, 2 * kBM);
  const int BH = d.B * d.Hq;
  int qp, bh;
  if (d.geom.kind == kMaskFull || d.geom.kind == kMaskWindow) {
    qp = bid % n_qp;
    bh = bid / n_qp;
  } else {
    qp = n_qp - 1 - (int)(bid / BH);
    bh = bid % BH;
  }
  const int h = bh % d.Hq;
  const int b = bh / d.Hq;
  const int hk = h / d.G;
  const int q0 = qp * 2 * kBM;
  if (*reinterpret_cast<volatile uint32_t*>(a.ctl.err) != 0) {
    // sticky device error: no work; NaN over this CTA's O and LSE rows (with a
    // split, the merge pass writes them)
    if (!split) {
      const int nrows = min(2 * kBM, d.Sq - q0);
      poison_rows(a.o, b, h, q0, nrows, D, d.out_f32 != 0);
      for (int i = threadIdx.x; i < nrows; i += blockDim.x)
        a.lse[((int64_t)b * d.Hq + h) * d.Sq + q0 + i] = nan_f32();
    }
    return;
  }
  // the work item must exist (ATTN_DEBUG)
  if (!ATTN_CHECK(a.ctl.err, q0 < d.Sq && h < d.Hq && b < d.B && (!split || chunk < a.nchunk), 3))
    return;
  // this batch entry's geometry; key tiles kt0 .. kt0 + n_kv - 1
  const MaskGeom g = W ? with_len(d.geom, d.seqlens, b) : d.geom;
  int kt0, n_kv;
  sched_kv_tiles<W>(g, q0, 2 * kBM, &kt0, &n_kv);
  if (split) {
    // this CTA's chunk of the pair's key tiles; a chunk past the range has no work
    // (the merge pass derives the pair's chunk count from the same range)
    const int c0 = chunk * a.split;
    if (c0 >= n_kv) return;
    kt0 += c0;
    n_kv = min(a.split, n_kv - c0);
  }

  const int warp = warp_id();
  const int lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int x = 0; x < 3; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_ready[x], 128);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&o_done[x], 1);
      mbar_init(&o_last[x], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  const bool scores_parked = ttt_scores_fit(g.ttt, D, d.out_f32);
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
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_expect_tx(q_full, 2 * TG::TILE_BYTES);
      TG::load(smem + L::Q_OFF, &tq, q_full, q0, h, b, d.Sq, d.Hq, d.B, a.ctl.err, 1);
      TG::load(smem + L::Q_OFF + TG::TILE_BYTES, &tq, q_full, q0 + kBM, h, b, d.Sq, d.Hq, d.B,
               a.ctl.err, 1);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        bool ok = true;
        for (int w = 0; w < 2; ++w) {
          const int idx = 2 * j + w;
          const int s = idx % NSLOT;
          const uint32_t ph = (uint32_t)(idx / NSLOT) & 1u;
          if (!mbar_wait(&kv_empty[s], ph ^ 1u, ctl)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&kv_full[s], TG::TILE_BYTES);
          TG::load(smem + L::KV_OFF + s * TG::TILE_BYTES, w == 0 ? &tk : &tv, &kv_full[s],
                   (kt0 + j) * kBN, hk, b, g.kv_main, d.Hkv, d.B, a.ctl.err, 2);
          issued = idx + 1;
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        // let every copy in flight land before the CTA can exit
        drain_wait(q_full, 0);
        for (int idx = issued - NSLOT < 0 ? 0 : issued - NSLOT; idx < issued; ++idx)
          drain_wait(&kv_full[idx % NSLOT], (uint32_t)(idx / NSLOT) & 1u);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------- MMA
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = make_idesc_bf16(128, D, false, true);
      // descriptors of Q tile 0 and of ring slot 0; tiles and slots are offsets
      const uint64_t dQ0 = TG::kmajor_base(smem_u32(smem + L::Q_OFF));
      const uint64_t dK0 = TG::kmajor_base(smem_u32(smem + L::KV_OFF));
      const uint64_t dV0 = TG::mnmajor_base(smem_u32(smem + L::KV_OFF));
      auto slot_of = [](int idx) { return idx % NSLOT; };
      auto phase_of = [](int idx) { return (uint32_t)(idx / NSLOT) & 1u; };
      // S of query tile x into S buffer `buf`; O_x += P V with P in buffer `buf`
      auto issue_s = [&](int x, int slot, int buf) {
        const uint64_t qd = dQ0 + TG::bytes(x * TG::TILE_BYTES);
        const uint64_t kd = dK0 + TG::bytes(slot * TG::TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < TG::KSTEPS; ++kk)
          umma_ss(tmem + buf * 128, qd + TG::kmajor_step(kk), kd + TG::kmajor_step(kk), idesc_s,
                  kk > 0);
      };
      auto issue_pv = [&](int x, int slot, bool acc, int buf) {
        const uint64_t vd = dV0 + TG::bytes(slot * TG::TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_ts(tmem + O_COL + x * D, tmem + buf * 128 + kk * 8, vd + TG::mnmajor_step(kk),
                  idesc_o, (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(q_full, 0, ctl);
      if (ok) ok = mbar_wait(&kv_full[slot_of(0)], phase_of(0), ctl);
      if constexpr (TB) {
        // score tile n = 2j + x in buffer n % 3; p_ready / s_full per buffer,
        // phase n / 3
        auto bar_par = [](int n) { return (uint32_t)(n / 3) & 1u; };
        if (ok) {
          tc_fence_after();
          issue_s(0, slot_of(0), 0);
          umma_commit(&s_full[0]);
          issue_s(1, slot_of(0), 1);
          umma_commit(&s_full[1]);
          umma_commit(&kv_empty[slot_of(0)]);
          if (n_kv > 1 && (ok = mbar_wait(&kv_full[slot_of(2)], phase_of(2), ctl))) {
            tc_fence_after();
            issue_s(0, slot_of(2), 2);  // S0(1)
            umma_commit(&s_full[2]);
          }
        }
        for (int j = 0; ok && j < n_kv; ++j) {
          const int vi = 2 * j + 1, n0 = 2 * j, n1 = 2 * j + 1;
          ATTN_TR(1, 0, j);
          if (!(ok = mbar_wait(&kv_full[slot_of(vi)], phase_of(vi), ctl))) break;
          ATTN_TR(1, 1, j);
          if (!(ok = mbar_wait(&p_ready[n0 % 3], bar_par(n0), ctl))) break;
          ATTN_TR(1, 2, j);
          tc_fence_after();
          issue_pv(0, slot_of(vi), j > 0, n0 % 3);
          umma_commit(&o_done[0]);
          if (j + 1 == n_kv) umma_commit(&o_last[0]);
          if (j + 1 < n_kv) {  // S1(j+1) takes the buffer P0(j) just left
            const int ki = 2 * (j + 1), n = n0 + 3;
            issue_s(1, slot_of(ki), n % 3);
            umma_commit(&s_full[n % 3]);
            umma_commit(&kv_empty[slot_of(ki)]);
          }
          ATTN_TR(1, 3, j);
          if (!(ok = mbar_wait(&p_ready[n1 % 3], bar_par(n1), ctl))) break;
          ATTN_TR(1, 4, j);
          tc_fence_after();
          issue_pv(1, slot_of(vi), j > 0, n1 % 3);
          umma_commit(&o_done[1]);
          if (j + 1 == n_kv) umma_commit(&o_last[1]);
          umma_commit(&kv_empty[slot_of(vi)]);
          if (j + 2 < n_kv) {  // S0(j+2) takes the buffer P1(j) just left
            const int ki = 2 * (j + 2), n = n1 + 3;
            if (!(ok = mbar_wait(&kv_full[slot_of(ki)], phase_of(ki), ctl))) break;
            tc_fence_after();
            issue_s(0, slot_of(ki), n % 3);
            umma_commit(&s_full[n % 3]);
          }
        }
      } else {
      if (ok) {
        tc_fence_after();
        issue_s(0, slot_of(0), 0);
        umma_commit(&s_full[0]);
        issue_s(1, slot_of(0), 1);
        umma_commit(&s_full[1]);
        umma_commit(&kv_empty[slot_of(0)]);
      }
      for (int j = 1; ok && j < n_kv; ++j) {
        const int vi = 2 * (j - 1) + 1, ki = 2 * j;
        ATTN_TR(1, 0, j);
        ok = mbar_wait(&kv_full[slot_of(vi)], phase_of(vi), ctl) &&
             mbar_wait(&kv_full[slot_of(ki)], phase_of(ki), ctl);
        ATTN_TR(1, 1, j);
        ok = ok && mbar_wait(&p_ready[0], (uint32_t)(j - 1) & 1u, ctl);
        if (!ok) break;
        ATTN_TR(1, 2, j);
        tc_fence_after();
        issue_pv(0, slot_of(vi), j - 1 > 0, 0);
        umma_commit(&o_done[0]);
        issue_s(0, slot_of(ki), 0);
        umma_commit(&s_full[0]);
        ATTN_TR(1, 3, j);
        if (!(ok = mbar_wait(&p_ready[1], (uint32_t)(j - 1) & 1u, ctl))) break;
        ATTN_TR(1, 4, j);
        tc_fence_after();
        issue_pv(1, slot_of(vi), j - 1 > 0, 1);
        umma_commit(&o_done[1]);
        umma_commit(&kv_empty[slot_of(vi)]);
        issue_s(1, slot_of(ki), 1);
        umma_commit(&s_full[1]);
        umma_commit(&kv_empty[slot_of(ki)]);
      }
      if (ok) {
        const int vi = 2 * (n_kv - 1) + 1;
        ok = mbar_wait(&kv_full[slot_of(vi)], phase_of(vi), ctl) &&
             mbar_wait(&p_ready[0], (uint32_t)(n_kv - 1) & 1u, ctl);
        if (ok) {
          tc_fence_after();
          issue_pv(0, slot_of(vi), n_kv - 1 > 0, 0);
          umma_commit(&o_done[0]);
          ok = mbar_wait(&p_ready[1], (uint32_t)(n_kv - 1) & 1u, ctl);
        }
        if (ok) {
          tc_fence_after();
          issue_pv(1, slot_of(vi), n_kv - 1 > 0, 1);
          umma_commit(&o_done[1]);
          umma_commit(&kv_empty[slot_of(vi)]);
        }
      }
      }  // TB
      if (!ok) {
        // every MMA issued so far must finish before tensor memory is freed
        umma_commit(drain);
        drain_wait(drain, 0);
      }
    }
  }
  } else {
    regs_grow();  // elementwise warpgroups
    // ---------------------------------------------------------- softmax
    const int x = warp >> 2;    // query tile of this warpgroup
    const int quad = warp & 3;  // TMEM lane quadrant
    const int r = quad * 32 + lane;
    const int qt0 = q0 + x * kBM;
    const int q = qt0 + r;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tO = tmem + lane_base + O_COL + x * D;
    const float sl2 = d.scale_log2;

    const FullRange full_k = full_keys_for_rows(g, qt0);  // key tiles without masking (W)
    const float inv_scale = 1.f / d.scale;                 // additive mask as M / scale (W)
    float m_run = neg_inf();  // running max of c*log2(e)*s
    float l_run = 0.f;
    bool ok = true;
    const bool tr = lane == 0 && quad == 0;
    for (int j = 0; j < n_kv; ++j) {
      if (tr) ATTN_TR(2 + x, 0, j);
      // score tile n = 2j + x: buffer n % 3, barrier phase n / 3 (D <= 64);
      // buffer and barrier x, phase j (D = 128)
      const int n = 2 * j + x;
      const int sb = TB ? n % 3 : x;
      const uint32_t spar = TB ? (uint32_t)(n / 3) & 1u : (uint32_t)j & 1u;
      const uint32_t tS = tmem + lane_base + sb * 128;
      const int k0 = (kt0 + j) * kBN;
      if (!(ok = mbar_wait_warp(&s_full[sb], spar, ctl))) break;
      if (tr) ATTN_TR(2 + x, 1, j);
      tc_fence_after();
      uint32_t sr[128];  // S row as raw fp32 bits; columns k0 .. k0+127
      tmem_ld64x2(tS + 0, tS + 64, sr);

      if constexpr (M) {
        if (q < d.Sq)
          add_bias_row<128>(sr, d.addm + b * d.addm_sb + (int64_t)q * d.addm_sq, k0, d.Skv,
                            inv_scale);
      }
      if (sched_row_tile_masked<W>(g, full_k, qt0, k0)) {
        int clo, chi;
        sched_row_cols<W>(g, q, k0, &clo, &chi);
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < clo || c > chi) sr[c] = __float_as_uint(neg_inf());
      }
      // row max over 8 independent chains of three-input max (a single chain of
      // 127 dependent max operations is latency-bound)
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = fmaxf(__uint_as_float(sr[i]), __uint_as_float(sr[8 + i]));
#pragma unroll
      for (int c = 16; c < 128; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          m8[i] = fmax3(m8[i], __uint_as_float(sr[c + i]), __uint_as_float(sr[c + 8 + i]));
      const float mt = fmaxf(fmax3(m8[0], m8[1], m8[2]),
                             fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
      const float m_new = mt * sl2;  // -inf stays -inf (sl2 > 0)
      const bool need = m_new > m_run + kRescaleThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = (m_run == neg_inf()) ? 0.f : ex2_approx(m_run - m_new);
        m_run = m_new;
        l_run *= alpha;
      }
      const float mu = (m_run == neg_inf()) ? 0.f : m_run;
      if (tr) ATTN_TR(2 + x, 2, j);
      // P = 2^(c log2(e) s - mu), argument by packed FMA; row sum in four packed
      // partial sums (eight independent chains)
      float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int qtr = 0; qtr < 4; ++qtr) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float x0, x1;
          fma2_bc(x0, x1, __uint_as_float(sr[qtr * 32 + 2 * c]),
                  __uint_as_float(sr[qtr * 32 + 2 * c + 1]), sl2, -mu);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          add2(rs[2 * (c & 3)], rs[2 * (c & 3) + 1], p0, p1);
          pk[c] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tS + qtr * 16, pk);
      }
      l_run += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      if (tr) ATTN_TR(2 + x, 3, j);
      if (j > 0) {
        // O must hold PV(j-1) before it is rescaled.  D = 128: the commit that
        // signalled S(j) tracks every MMA issued before it, PV(j-1) included, so
        // no wait.  D <= 64: S(j) was issued before PV(j-1); wait for it
        if (__any_sync(0xffffffffu, need)) {
          if constexpr (TB) {
            if (!(ok = mbar_wait_warp(&o_done[x], (uint32_t)(j - 1) & 1u, ctl))) break;
          }
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t ov[16];
            tmem_ld16(tO + c0, ov);
#pragma unroll
            for (int c = 0; c < 16; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st16(tO + c0, ov);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_ready[sb]);
      if (tr) ATTN_TR(2 + x, 4, j);
    }

    // ------------------------------------------------------------ epilogue
    // O_x is final once PV_x(n_kv - 1) has completed.  At D = 128 the last S_x
    // implies PV_x(n_kv - 2), so the o_done phase of the last PV is unambiguous;
    // with three S buffers two phases may still be open, hence o_last.
    if (ok && n_kv > 0)
      ok = TB ? mbar_wait_warp(&o_last[x], 0u, ctl)
              : mbar_wait_warp(&o_done[x], (uint32_t)(n_kv - 1) & 1u, ctl);
    if constexpr (split) {
      // partial result of this key chunk (never a TTT mask, n_kv > 0): the
      // unnormalised O row and the running max and sum it is relative to
      if (ok) {
        tc_fence_after();
        // partial rows are indexed by CTA: (blockIdx.x, row of the pair)
        const int64_t slot = (int64_t)blockIdx.x * (2 * kBM) + x * kBM + r;
        // staged like the final O rows (see below), stored as dense fp32 rows
        const RowStage<D> stage{smem + (x == 0 ? L::Q_OFF : L::KV_OFF) + quad * (32 * D * 4),
                                true};
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          uint32_t raw[16];
          float vals[16];
          tmem_ld16(tO + c0, raw);
#pragma unroll
          for (int e = 0; e < 16; ++e) vals[e] = __uint_as_float(raw[e]);
          stage.put16(lane, c0, vals, 1.f);
        }
        __syncwarp();
        const View part{a.part_o, 0, 0, D};
        const int row0 = qt0 + quad * 32;
        stage.copy_out(lane, part, 0, 0, slot - r + quad * 32, min(32, max(0, d.Sq - row0)), 0);
        if (q < d.Sq) a.part_ml[slot] = make_float2(m_run, l_run);
      }
    } else if (ok) {
      if (n_kv > 0) tc_fence_after();
      const bool qin = q < d.Sq;
      // suffix diagonals exist for rows inside the batch entry's key length
      const bool qdiag = qin && q < g.kv_len;
      if (g.ttt > 0) {
        // TTT suffix diagonals (key/value row i*Sq + q of segment i = 1..t), merged into
        // the unnormalised O accumulator in TMEM by log-sum-exp
        if (n_kv == 0) {  // accumulator never written by an MMA: start at zero
          uint32_t z[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16) tmem_st16(tO + c0, z);
          tmem_st_wait();
        }
        const __nv_bfloat16* qrow = row_ptr(a.q, b, h, q);
        // scaled score c log2(e) q . k_i of diagonal i: parked in this row of O by the
        // scores pre-pass when it fits there (read before this thread writes the row)
        const float* parked = reinterpret_cast<const float*>(
            static_cast<const char*>(a.o.ptr) +
            (b * a.o.sb + h * a.o.sh + (int64_t)q * a.o.ss) * (d.out_f32 ? 4 : 2));
        auto diag_score = [&](int i) {
          return scores_parked ? parked[i - 1]
                               : dot_rows<D>(qrow, row_ptr(a.k, b, hk, (int64_t)i * d.Sq + q)) * sl2;
        };
        float m_star = m_run;  // pass 1: the merged running max
        if (qdiag)
          for (int i = 1; i <= g.ttt; ++i) m_star = fmaxf(m_star, diag_score(i));
        const float alpha = (m_run == neg_inf()) ? 0.f : ex2_approx(m_run - m_star);
        l_run *= alpha;
        // pass 2: O = alpha O + sum_i w_i v_i.  The v rows of the warp's 32 query
        // positions are fetched two segments at a time into the warp's output
        // staging area (coalesced copies, one round trip per pair) and folded
        // into the TMEM accumulator in one pass per pair, in segment order.
        const int row0 = qt0 + quad * 32;
        const int nvalid = max(0, min(32, min(d.Sq, g.kv_len) - row0));
        uint8_t* fbase = smem + (x == 0 ? L::Q_OFF : L::KV_OFF) + quad * (32 * D * 4);
        const RowFetch<D> fv[2] = {{fbase}, {fbase + 32 * D * 2}};
        for (int i0 = 1; i0 <= g.ttt; i0 += 2) {
          const int nseg = min(2, g.ttt - i0 + 1);
          for (int u = 0; u < nseg; ++u)
            fv[u].issue(lane, a.v, b, hk, (int64_t)(i0 + u) * d.Sq + row0, nvalid, 0);
          cp_async_commit();
          float w[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            w[u] = 0.f;
            if (qdiag && u < nseg) {
              w[u] = ex2_approx(diag_score(i0 + u) - m_star);
              l_run += w[u];
            }
          }
          cp_async_wait_all();
          __syncwarp();
          const float scale0 = (i0 == 1) ? alpha : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t raw[16];
            float vals[16];
            tmem_ld16(tO + c0, raw);
#pragma unroll
            for (int e = 0; e < 16; ++e) vals[e] = __uint_as_float(raw[e]) * scale0;
            if (qdiag) {
#pragma unroll
              for (int u = 0; u < 2; ++u)
                if (u < nseg) fv[u].axpy16(lane, c0 / 16, w[u], vals);
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) raw[e] = __float_as_uint(vals[e]);
            tmem_st16(tO + c0, raw);
          }
          tmem_st_wait();
          __syncwarp();  // every lane has read the pair before it is refilled
        }
        m_run = m_star;
      }
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      const bool have_acc = n_kv > 0 || g.ttt > 0;
      // the warp's 32 rows go through shared memory so that the global stores are
      // coalesced: query tile 0 stages in the Q tiles (their last reader, S1 of the
      // last key tile, was issued before PV0 of that tile, which has completed),
      // query tile 1 in the K/V ring (free: its own last PV was the last MMA)
      const RowStage<D> stage{smem + (x == 0 ? L::Q_OFF : L::KV_OFF) + quad * (32 * D * 4),
                              d.out_f32 != 0};
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 16) {
        float vals[16];
        if (have_acc) {
          uint32_t raw[16];
          tmem_ld16(tO + c0, raw);
#pragma unroll
          for (int e = 0; e < 16; ++e) vals[e] = __uint_as_float(raw[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) vals[e] = 0.f;
        }
        stage.put16(lane, c0, vals, inv);
      }
      __syncwarp();
      const int row0 = qt0 + quad * 32;
      stage.copy_out(lane, a.o, b, h, row0, min(32, max(0, d.Sq - row0)), 0);
      if (qin) {
        const float lse = (l_run > 0.f) ? (m_run + lg2_approx(l_run)) * 0.69314718055994531f : 0.f;
        a.lse[((int64_t)b * d.Hq + h) * d.Sq + q] = lse;
      }
    } else if (q < d.Sq) {
      // a wait of this CTA ran out of budget: NaN instead of a partial result
      // (with a split, the merge pass sees the error word and writes NaN)
      poison_row(a.o, b, h, q, 0, 16, D, d.out_f32 != 0);
      a.lse[((int64_t)b * d.Hq + h) * d.Sq + q] = nan_f32();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge pass of the split forward.  Chunk c of a row holds O_c (unnormalised),
// its running max m_c and sum l_c, both in the log2 domain of the scaled scores
// (P = 2^(c log2(e) s - m_c)); the chunks combine as
//     m = max_c m_c,  l = sum_c l_c 2^(m_c - m),  O = sum_c O_c 2^(m_c - m) / l,
// the same log-sum-exp merge as the online softmax, taken in chunk order so the
// result is bitwise reproducible.  One thread per 16 columns of a query row.
template <int D, bool W>
__global__ void __launch_bounds__(256) fwd_merge_kernel(const FwdArgs a) {
  constexpr int TPR = D / 16;
  const Dims& d = a.d;
  const int64_t rows = (int64_t)d.B * d.Hq * d.Sq;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = idx / TPR;
  if (row >= rows) return;
  const int c0 = (int)(idx % TPR) * 16;
  const int q = (int)(row % d.Sq);
  const int bh = (int)(row / d.Sq);
  const int h = bh % d.Hq;
  const int b = bh / d.Hq;
  const bool f32 = d.out_f32 != 0;
  if (*reinterpret_cast<volatile uint32_t*>(a.ctl.err) != 0) {
    // a chunk was skipped or gave up: NaN, not a partial result
    poison_row(a.o, b, h, q, c0, D, D, f32);
    if (c0 == 0) a.lse[row] = nan_f32();
    return;
  }
  const int n_qp = cdiv(d.Sq, 2 * kBM);
  const int qp = q / (2 * kBM), rr = q % (2 * kBM);
  const MaskGeom g = W ? with_len(d.geom, d.seqlens, b) : d.geom;
  int kt0, n_kv;
  sched_kv_tiles<W>(g, qp * 2 * kBM, 2 * kBM, &kt0, &n_kv);
  const int nc = n_kv > 0 ? cdiv(n_kv, a.split) : 0;
  // the forward's CTA of (pair, chunk 0): its work decode inverted
  const int bid = (d.geom.kind == kMaskFull || d.geom.kind == kMaskWindow)
                      ? bh * n_qp + qp
                      : (n_qp - 1 - qp) * (d.B * d.Hq) + bh;
  const int64_t slot0 = (int64_t)bid * a.nchunk;
  // the chunks read must be slots the forward wrote (ATTN_DEBUG)
  if (!ATTN_CHECK(a.ctl.err, nc <= a.nchunk && bid < n_qp * d.B * d.Hq, 4)) return;
  float m = -INFINITY;
  for (int c = 0; c < nc; ++c) m = fmaxf(m, a.part_ml[(slot0 + c) * (2 * kBM) + rr].x);
  float l = 0.f;
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  for (int c = 0; c < nc; ++c) {
    const int64_t slot = (slot0 + c) * (2 * kBM) + rr;
    const float2 ml = a.part_ml[slot];
    if (ml.x == -INFINITY) continue;  // the row sees no key of this chunk
    const float w = ex2_approx(ml.x - m);
    l = fmaf(ml.y, w, l);
    const float4* po = reinterpret_cast<const float4*>(a.part_o + slot * D + c0);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 v = po[e];
      acc[4 * e] = fmaf(v.x, w, acc[4 * e]);
      acc[4 * e + 1] = fmaf(v.y, w, acc[4 * e + 1]);
      acc[4 * e + 2] = fmaf(v.z, w, acc[4 * e + 2]);
      acc[4 * e + 3] = fmaf(v.w, w, acc[4 * e + 3]);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  store16(a.o, b, h, q, c0, acc, inv, f32);
  if (c0 == 0) a.lse[row] = l > 0.f ? (m + lg2_approx(l)) * 0.69314718055994531f : 0.f;
}

template <int D, bool W, bool M, bool S>
cudaError_t launch_fwd_dw(const FwdArgs& a, const Maps& m, cudaStream_t s) {
  using L = FwdLayout<D>;
  auto kern = fwd_kernel<D, W, M, S>;
  static const cudaError_t regs_ok = check_launch_regs(reinterpret_cast<const void*>(kern));
  if (regs_ok != cudaSuccess) return regs_ok;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  if (ttt_scores_fit(a.d.geom.ttt, D, a.d.out_f32)) {
    constexpr int RPB = 256 / (D / 8);
    const int64_t rows = (int64_t)a.d.B * a.d.Hq * a.d.Sq;
    ttt_scores_kernel<D><<<(unsigned)((rows + RPB - 1) / RPB), 256, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int n_qp = cdiv(a.d.Sq, 2 * kBM);
  const int64_t pairs = (int64_t)n_qp * a.d.B * a.d.Hq;
  const unsigned grid = (unsigned)(pairs * (S ? a.nchunk : 1));
  kern<<<grid, kFwdThreads, L::ALLOC, s>>>(m.q, m.k, m.v, a);
  if ((e = cudaGetLastError()) != cudaSuccess || !S) return e;
  const int64_t threads = (int64_t)a.d.B * a.d.Hq * a.d.Sq * (D / 16);
  fwd_merge_kernel<D, W><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, bool S>
cudaError_t launch_fwd_d(const FwdArgs& a, const Maps& m, cudaStream_t s) {
  if (a.d.addm != nullptr) return launch_fwd_dw<D, true, true, S>(a, m, s);
  return needs_general_mask(a.d) ? launch_fwd_dw<D, true, false, S>(a, m, s)
                                 : launch_fwd_dw<D, false, false, S>(a, m, s);
}

// All four head dims, split (S) or not.
template <bool S>
cudaError_t launch_fwd_any(const FwdArgs& a, const Maps& m, cudaStream_t s) {
  switch (a.d.D) {
    case 16: return launch_fwd_d<16, S>(a, m, s);
    case 32: return launch_fwd_d<32, S>(a, m, s);
    case 64: return launch_fwd_d<64, S>(a, m, s);
    case 128: return launch_fwd_d<128, S>(a, m, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace attn
