// fwd_split.cu -- the forward's split instantiations (one CTA per chunk of a
// query-tile pair's key tiles, then the merge pass); a translation unit of its
// own so that it compiles in parallel with fwd.cu.
#include "fwd_impl.cuh"

namespace attn {

cudaError_t launch_fwd_split(const FwdArgs& a, const Maps& m, cudaStream_t s) {
  return launch_fwd_any<true>(a, m, s);
}

}  // namespace attn
