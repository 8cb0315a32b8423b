// fwd.cu -- the forward's unsplit instantiations, the key-range split plan and
// the forward launch (the kernels are in fwd_impl.cuh; the split instantiations
// in fwd_split.cu).
#include "fwd_impl.cuh"

namespace attn {

// The split's cost model, in units of one key-tile iteration of the forward:
// a CTA's fixed costs (tensor memory and barrier set-up, the Q load, pipeline
// fill, the epilogue) are worth about kCtaFixedTiles iterations and the merge
// pass, a launch of its own, about kMergeTiles.  A launch of n CTAs on the SMs
// takes ceil(n / SMs) waves of (chunk + fixed) each; unsplit, one CTA per pair
// (fewer than the SMs) takes the longest pair's tiles plus the fixed costs.
// Measured on GB300 with CUDA-graph replay (sweep S = 4096): a fixed chunk of
// 8 tiles gave 320 CTAs, three waves, and no gain; two full waves do.
constexpr int kMinSplitTiles = 4;
constexpr int kCtaFixedTiles = 3;
constexpr int kMergeTiles = 5;
constexpr int kMaxSlotsPerSM = 4;

FwdSplit fwd_split_plan(const Dims& d) {
  constexpr int num_sms = kPlanSMs;
  if (d.geom.ttt > 0) return FwdSplit{};  // TTT merges its diagonals per CTA
  const int n_qp = cdiv(d.Sq, 2 * kBM);
  const int64_t BH = (int64_t)d.B * d.Hq;
  if (n_qp * BH >= num_sms) return FwdSplit{};  // one CTA per pair already fills a wave
  // key tiles of every pair (the bound without per-batch key lengths, which only
  // shorten rows)
  int n_kv[2 * kPlanSMs];
  int nmax = 0;
  for (int qp = 0; qp < n_qp; ++qp) {
    int kt0;
    sched_kv_tiles<true>(d.geom, qp * 2 * kBM, 2 * kBM, &kt0, &n_kv[qp]);
    if (n_kv[qp] > nmax) nmax = n_kv[qp];
  }
  int64_t best = (int64_t)nmax + kCtaFixedTiles;
  int best_split = 0;
  for (int split = kMinSplitTiles; split < nmax; ++split) {
    // the partials take pairs x chunks slots of 2 kBM rows: at most four per SM
    // (at most 81 MB at D = 128, whatever the sequence length)
    if ((int64_t)n_qp * BH * cdiv(nmax, split) > kMaxSlotsPerSM * num_sms) continue;
    int64_t ctas = 0;
    for (int qp = 0; qp < n_qp; ++qp) ctas += n_kv[qp] > 0 ? cdiv(n_kv[qp], split) : 0;
    ctas *= BH;
    const int64_t waves = (ctas + num_sms - 1) / num_sms;
    const int64_t cost = waves * (split + kCtaFixedTiles) + kMergeTiles;
    if (cost < best) {
      best = cost;
      best_split = split;
    }
  }
  return fwd_split_with(d, best_split);
}

FwdSplit fwd_split_with(const Dims& d, int split) {
  FwdSplit sp;
  if (split <= 0 || d.geom.ttt > 0) return sp;
  const int n_qp = cdiv(d.Sq, 2 * kBM);
  int nmax = 0;
  for (int qp = 0; qp < n_qp; ++qp) {
    int kt0, n;
    sched_kv_tiles<true>(d.geom, qp * 2 * kBM, 2 * kBM, &kt0, &n);
    if (n > nmax) nmax = n;
  }
  sp.split = split;
  sp.nchunk = nmax > 0 ? cdiv(nmax, split) : 1;
  const int64_t slots = (int64_t)n_qp * d.B * d.Hq * sp.nchunk * 2 * kBM;
  sp.part_o_bytes = ((size_t)slots * d.D * 4 + 255) & ~(size_t)255;
  sp.part_ml_bytes = ((size_t)slots * 8 + 255) & ~(size_t)255;
  return sp;
}

// Depth of the forward's K/V ring (entries of one 128-key K or V tile) and
// whether the three-buffer score rotation is used, for the plan description.
FwdShape fwd_shape(const Dims& d) {
  FwdShape f;
  f.ring = d.D == 128 ? FwdLayout<128>::NSLOT
           : d.D == 64 ? FwdLayout<64>::NSLOT
           : d.D == 32 ? FwdLayout<32>::NSLOT : FwdLayout<16>::NSLOT;
  f.three_buffers = needs_general_mask(d) && d.D <= 64;
  f.smem = d.D == 128 ? FwdLayout<128>::ALLOC
           : d.D == 64 ? FwdLayout<64>::ALLOC
           : d.D == 32 ? FwdLayout<32>::ALLOC : FwdLayout<16>::ALLOC;
  return f;
}

cudaError_t launch_fwd(const FwdArgs& a, const Maps& m, cudaStream_t s) {
  return a.split > 0 ? launch_fwd_split(a, m, s) : launch_fwd_any<false>(a, m, s);
}

}  // namespace attn

ATTN_TRACE_READER(attn_trace_read_fwd)
