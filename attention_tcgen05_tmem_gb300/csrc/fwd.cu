// fwd.cu -- the forward's unsplit instantiations, the key-range split plan and
// the forward launch (the kernels are in fwd_impl.cuh; the split instantiations
// in fwd_split.cu).
#include "fwd_impl.cuh"

namespace attn {

// Fewest key tiles a chunk of the split forward takes: a CTA's fixed costs (tensor
// memory and barrier set-up, the Q load, pipeline fill, the epilogue) are worth
// several key tiles.
constexpr int kMinSplitTiles = 4;

FwdSplit fwd_split_plan(const Dims& d) {
  constexpr int num_sms = kPlanSMs;
  FwdSplit sp;
  if (d.geom.ttt > 0) return sp;  // TTT merges its diagonals per CTA
  const int n_qp = cdiv(d.Sq, 2 * kBM);
  const int64_t pairs = (int64_t)n_qp * d.B * d.Hq;
  if (pairs >= num_sms) return sp;  // one CTA per pair already fills a wave
  // key tiles of every pair (the bound without per-batch key lengths, which only
  // shorten rows), and the whole launch's
  int64_t total = 0;
  int nmax = 0;
  for (int qp = 0; qp < n_qp; ++qp) {
    int kt0, n;
    sched_kv_tiles<true>(d.geom, qp * 2 * kBM, 2 * kBM, &kt0, &n);
    total += n;
    if (n > nmax) nmax = n;
  }
  total *= (int64_t)d.B * d.Hq;
  // about two chunks per SM, each at least kMinSplitTiles key tiles
  int64_t split = (total + 2 * num_sms - 1) / (2 * num_sms);
  if (split < kMinSplitTiles) split = kMinSplitTiles;
  if (split >= nmax) return sp;
  return fwd_split_with(d, (int)split);
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

cudaError_t launch_fwd(const FwdArgs& a, const Maps& m, cudaStream_t s) {
  return a.split > 0 ? launch_fwd_split(a, m, s) : launch_fwd_any<false>(a, m, s);
}

}  // namespace attn

ATTN_TRACE_READER(attn_trace_read_fwd)
