// sched_host.cpp -- a host build of the attention kernels' schedule functions
// (attention_tcgen05_tmem_gb300/csrc/sched.cuh) for the CPU tests: it
// evaluates, for every (query, key) pair of one batch entry, which pairs the
// forward, dK/dV and dQ passes visit unmasked, in the one-sided form and in the
// general form, exactly as the kernels and the device-side mask export do.
#define __host__
#define __device__
#include <cstddef>
#include <cstdint>

#include "sched.cuh"

// bits: 6 planes of Sq x Skv bytes, laid out like attn_train_mask_pattern's
// output: planes 0-2 the forward, dK/dV and dQ schedules in the form selected
// by `general`, planes 3-5 in the general form.  len < 0: no key length.
extern "C" void sched_pattern_host(int kind, int t, int wl, int wr, int Sq, int Skv, int len,
                                   int general, uint8_t* bits) {
  using namespace attn;
  MaskGeom g = make_geom(kind, t, wl, wr, Sq, Skv);
  const int lens[1] = {len};
  if (len >= 0) g = with_len(g, lens, 0);
  const size_t n = (size_t)Sq * Skv;
  for (int q = 0; q < Sq; ++q) {
    for (int kv = 0; kv < Skv; ++kv) {
      const size_t idx = (size_t)q * Skv + kv;
      uint8_t vis[6];
      sched_pattern_pair(g, q, kv, general != 0, vis);
      for (int p = 0; p < 6; ++p) bits[p * n + idx] = vis[p];
    }
  }
}
