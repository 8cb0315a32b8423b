// abi_internal.h -- entry points shared between the C ABI's translation units
// (api.cu defines them; host_step.cu uses them).  Not installed.
#pragma once
#include <cstddef>

#include "attn_train.h"

namespace attn {

// Chunk length (key tiles) of the forward's key-range split planned for *p
// (0: no split); *p must be valid.
int fwd_split_tiles(const attn_problem* p);
// Workspace bytes of the forward of *p split into chunks of `split` key tiles.
size_t fwd_split_bytes(const attn_problem* p, int split);
// attn_train_fwd_ws with the chunk length fixed at `split` (0: no split), so that
// a slice of a larger problem (some of its GQA groups) can use the larger
// problem's chunks and give exactly its results.
attn_status fwd_with_split(const attn_problem* p, int split, attn_tensor q, attn_tensor k,
                           attn_tensor v, attn_tensor o, float* lse, void* workspace,
                           size_t ws_bytes, void* stream);

}  // namespace attn
