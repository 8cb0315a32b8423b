// sched.cuh -- tile classification and iteration ranges (host and device).
//
// The attention grid is cut into 128-row query tiles and 128-column key
// tiles.  Masks are evaluated arithmetically, never from a mask tensor
// (FlexAttention's BlockMask idea -- skip empty blocks, and skip the mask
// test on full blocks -- from the SpecForge post, "Flex Attention"; the
// HOT-Step page, section 3, reports that skipping all -inf tiles halves the
// causal work).
//
// The tiled part of every mask is one band predicate:
//     visible(q, kv) = kv < kv_len  and  q - lo <= kv <= q + hi
//   full:    lo = hi = unbounded
//   causal:  lo unbounded, hi = 0
//   TTT t:   lo unbounded, hi = -t (segment 0's causal part shrinks by one
//            diagonal per appended segment: SpecForge "Flex Attention",
//            causal_mask with shift_left = t)
//   window:  lo = left, hi = right extent (the HOT-Step page's windowed
//            self-attention, section 4, read as a band around the diagonal)
// kv_len is the key length of the tiled part for one batch entry: Skv (Sq for
// TTT), cut to seq_lengths[b] when the caller passes per-batch lengths (the
// padding term kv < seq_lengths[b] of the eagle3 mask_mod).  The TTT suffix
// diagonals (kv = q + i*Sq, i = 1..t, visible for q < seq_lengths[b]) are not
// tiles: the kernels merge them in a separate per-row pass.
#pragma once
#include <cstdint>

namespace attn {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // key rows per tile

enum MaskKind : int { kMaskFull = 0, kMaskCausal = 1, kMaskTTT = 2, kMaskWindow = 3 };

// An extent that no problem reaches (sequence lengths stay below 2^30; the
// helpers below compute in 64 bits, so q + kUnbounded cannot overflow).
constexpr int kUnbounded = 1 << 30;

struct MaskGeom {
  int kind;      // MaskKind
  int Sq;        // query rows
  int kv_main;   // key rows of the tiled part (Skv, or Sq for TTT)
  int kv_len;    // kv_main cut to this batch entry's key length (see with_len)
  int ttt;       // number of suffix diagonals (t for TTT, else 0)
  int lo;        // band: kv >= q - lo
  int hi;        // band: kv <= q + hi
};

__host__ __device__ inline MaskGeom make_geom(int kind, int t, int wl, int wr, int Sq, int Skv) {
  MaskGeom g;
  g.kind = kind;
  g.Sq = Sq;
  g.kv_main = (kind == kMaskTTT) ? Sq : Skv;
  g.kv_len = g.kv_main;
  g.ttt = (kind == kMaskTTT) ? t : 0;
  g.lo = (kind == kMaskWindow) ? (wl < kUnbounded ? wl : kUnbounded) : kUnbounded;
  g.hi = kind == kMaskFull ? kUnbounded
       : kind == kMaskCausal ? 0
       : kind == kMaskTTT ? -t
                           : (wr < kUnbounded ? wr : kUnbounded);
  return g;
}

// The geometry of batch entry b: keys from seq_lengths[b] on are invisible
// (values are clamped to [0, kv_main]; null = every key).
__host__ __device__ inline MaskGeom with_len(MaskGeom g, const int* seq_lengths, int b) {
  if (seq_lengths != nullptr) {
    int L = seq_lengths[b];
    if (L < 0) L = 0;
    if (L > g.kv_main) L = g.kv_main;
    g.kv_len = L;
  }
  return g;
}

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

__host__ __device__ inline int64_t clamp64(int64_t x, int64_t a, int64_t b) {
  return x < a ? a : (x > b ? b : x);
}

// Keys [begin, end) that some query of rows [q0, q0 + rows) may see.
__host__ __device__ inline void kv_range_for_rows(const MaskGeom& g, int q0, int rows, int* begin,
                                                  int* end) {
  int64_t last_q = (int64_t)q0 + rows - 1;
  if (last_q > g.Sq - 1) last_q = g.Sq - 1;
  const int64_t e = clamp64(last_q + g.hi + 1, 0, g.kv_len);
  const int64_t b = clamp64((int64_t)q0 - g.lo, 0, e);
  *begin = (int)b;
  *end = (int)e;
}

// Key tiles [*kt0, *kt0 + *n) to visit for rows [q0, q0 + rows).
__host__ __device__ inline void kv_tiles_for_rows(const MaskGeom& g, int q0, int rows, int* kt0,
                                                  int* n) {
  int b, e;
  kv_range_for_rows(g, q0, rows, &b, &e);
  *kt0 = b / kBN;
  *n = e > b ? cdiv(e, kBN) - b / kBN : 0;
}

// A (query tile, key tile) pair needs no per-element test iff every pair in it
// is visible (rows beyond Sq are never stored, so they do not matter).
__host__ __device__ inline bool tile_is_full(const MaskGeom& g, int q0, int k0) {
  if (k0 + kBN > g.kv_len) return false;
  if ((int64_t)k0 < (int64_t)q0 + kBM - 1 - g.lo) return false;
  return (int64_t)k0 + kBN - 1 <= (int64_t)q0 + g.hi;
}

// Visible columns of query row q inside the key tile at k0: c (key k0 + c)
// is visible iff *clo <= c <= *chi (empty when *chi < *clo).
__host__ __device__ inline void col_range(const MaskGeom& g, int q, int k0, int* clo, int* chi) {
  const int64_t h = (int64_t)q + g.hi < (int64_t)g.kv_len - 1 ? (int64_t)q + g.hi
                                                              : (int64_t)g.kv_len - 1;
  *chi = (int)clamp64(h - k0, -1, kBN);
  *clo = (int)clamp64((int64_t)q - g.lo - k0, 0, kBN);
}

// Query rows [begin, end) that see some key of the key tile at k0.
__host__ __device__ inline void q_range_for_kv(const MaskGeom& g, int k0, int* begin, int* end) {
  if (k0 >= g.kv_len) {
    *begin = *end = 0;
    return;
  }
  const int64_t kv_last = (k0 + kBN < g.kv_len ? k0 + kBN : g.kv_len) - 1;
  // q sees kv iff kv - hi <= q <= kv + lo
  const int64_t e = clamp64(kv_last + g.lo + 1, 0, g.Sq);
  const int64_t b = clamp64((int64_t)k0 - g.hi, 0, e);
  *begin = (int)b;
  *end = (int)e;
}

// Visible query columns of key row kv inside the query tile starting at q0:
// column c (query q0 + c) is visible iff *clo <= c <= *chi.
__host__ __device__ inline void row_range_for_kv(const MaskGeom& g, int kv, int q0, int* clo,
                                                 int* chi) {
  if (kv >= g.kv_len) {
    *clo = kBM;
    *chi = -1;
    return;
  }
  *clo = (int)clamp64((int64_t)kv - g.hi - q0, 0, kBM);
  *chi = (int)clamp64((int64_t)kv + g.lo - q0, -1, kBM);
}

// tile_is_full folded into a range, for the kernels' inner loops: with the
// query tile fixed (forward, dQ), the key tile at k0 is full iff
// lo <= k0 <= hi; with the key tile fixed (dK/dV), the query tile at q0 is
// full iff lo <= q0 <= hi.  The two numbers depend on tile indices only (the
// compiler can keep them in uniform registers); the per-row bounds of partial
// tiles come from col_range / row_range_for_kv inside the rare masked branch.
struct FullRange {
  int lo, hi;
};

__host__ __device__ inline int clamp_int(int64_t x) {
  return (int)clamp64(x, -(int64_t)kUnbounded, (int64_t)kUnbounded);
}

// Key tiles k0 that are full for the query tile at qt0:
// k0 + kBN <= kv_len, k0 >= qt0 + kBM - 1 - lo, k0 + kBN - 1 <= qt0 + hi.
__host__ __device__ inline FullRange full_keys_for_rows(const MaskGeom& g, int qt0) {
  const int64_t a = (int64_t)qt0 + g.hi - (kBN - 1), b = (int64_t)g.kv_len - kBN;
  return FullRange{clamp_int((int64_t)qt0 + kBM - 1 - g.lo), clamp_int(a < b ? a : b)};
}
// Query tiles q0 that are full for the key tile at k0 (none when it runs past kv_len).
__host__ __device__ inline FullRange full_rows_for_keys(const MaskGeom& g, int k0) {
  if (k0 + kBN > g.kv_len) return FullRange{kUnbounded, -kUnbounded};
  return FullRange{clamp_int((int64_t)k0 + kBN - 1 - g.hi),
                   clamp_int((int64_t)k0 + g.lo - (kBM - 1))};
}
__host__ __device__ inline bool in_range(const FullRange& r, int x) { return x >= r.lo && x <= r.hi; }

// The one-sided forms: masks without a lower key bound (full, causal, TTT) and
// without per-batch key lengths (kv_len == kv_main).  The kernels are
// instantiated for this case of their own, so that the general window and
// length arithmetic costs the common masks nothing.  Both forms must select
// exactly the visible pairs; the mask export below evaluates each of them as
// the kernels do, and the tests compare every plane with the visibility
// predicate bit for bit.
__host__ __device__ inline int upper_kv_end(const MaskGeom& g, int q0, int rows) {
  int64_t last_q = (int64_t)q0 + rows - 1;
  if (last_q > g.Sq - 1) last_q = g.Sq - 1;
  return (int)clamp64(last_q + g.hi + 1, 0, g.kv_main);
}
__host__ __device__ inline bool upper_tile_full(const MaskGeom& g, int q0, int k0) {
  if (k0 + kBN > g.kv_main) return false;
  return g.kind == kMaskFull || (int64_t)k0 + kBN - 1 <= (int64_t)q0 + g.hi;
}
// Column c of the key tile at k0 is visible to query q iff c <= the limit.
__host__ __device__ inline int upper_col_limit(const MaskGeom& g, int q, int k0) {
  int64_t lim = (int64_t)g.kv_main - 1 - k0;
  if (g.kind != kMaskFull) {
    const int64_t c = (int64_t)q + g.hi - k0;
    if (c < lim) lim = c;
  }
  return (int)clamp64(lim, -1, kBN);
}
// First query row that sees key row kv (all of them for the full mask).
__host__ __device__ inline int upper_q_begin(const MaskGeom& g, int kv) {
  if (g.kind == kMaskFull) return 0;
  return (int)clamp64((int64_t)kv - g.hi, 0, g.Sq);
}

// ---- The schedules the attention kernels run ----------------------------
// Every decision a kernel takes about which tiles to visit and which scores
// to hide goes through these functions, and so does the test-only export of
// the mask pattern, so that the export shows exactly what the kernels compute.
// W selects the general form (window mask, per-batch key lengths, additive
// mask); without it the one-sided form (full, causal, TTT).

// Key tiles [*kt0, *kt0 + *n) visited by query rows [q0, q0 + rows): the
// forward (rows = 2 kBM, a query-tile pair) and dQ (rows = kBM).
template <bool W>
__host__ __device__ inline void sched_kv_tiles(const MaskGeom& g, int q0, int rows, int* kt0,
                                               int* n) {
  if constexpr (W) {
    kv_tiles_for_rows(g, q0, rows, kt0, n);
  } else {
    *kt0 = 0;
    *n = cdiv(upper_kv_end(g, q0, rows), kBN);
  }
}

// Query tiles [*qt0, *qt0 + *n) that the dK/dV pass visits for the key tile at k0.
template <bool W>
__host__ __device__ inline void sched_q_tiles(const MaskGeom& g, int k0, int* qt0, int* n) {
  if constexpr (W) {
    int lo, hi;
    q_range_for_kv(g, k0, &lo, &hi);
    *qt0 = lo / kBM;
    *n = hi > lo ? cdiv(hi, kBM) - *qt0 : 0;
  } else {
    *qt0 = upper_q_begin(g, k0) / kBM;
    const int m = cdiv(g.Sq, kBM) - *qt0;
    *n = m < 0 ? 0 : m;
  }
}

// Row side (forward, dQ): whether the key tile at k0 needs per-column masking
// for the query tile at qt0; full_k = full_keys_for_rows(g, qt0) (read by the
// general form only, so the kernels can keep it in uniform registers).
template <bool W>
__host__ __device__ inline bool sched_row_tile_masked(const MaskGeom& g, const FullRange& full_k,
                                                      int qt0, int k0) {
  if constexpr (W) return !in_range(full_k, k0);
  else return !upper_tile_full(g, qt0, k0);
}
// Row side, masked tile: columns c of the key block starting at k0 that query
// q sees are *clo <= c <= *chi.
template <bool W>
__host__ __device__ inline void sched_row_cols(const MaskGeom& g, int q, int k0, int* clo,
                                               int* chi) {
  if constexpr (W) {
    col_range(g, q, k0, clo, chi);
  } else {
    *clo = 0;
    *chi = upper_col_limit(g, q, k0);
  }
}

// Column side (dK/dV): whether the query tile at q0 needs per-row masking for
// the key tile at k0; full_q = full_rows_for_keys(g, k0) (general form only).
template <bool W>
__host__ __device__ inline bool sched_col_tile_masked(const MaskGeom& g, const FullRange& full_q,
                                                      int q0, int k0) {
  if constexpr (W) return !in_range(full_q, q0);
  else return !upper_tile_full(g, q0, k0);
}
// Column side, masked tile: query columns c of the block starting at q0 that
// key row kv is seen by are *clo <= c <= *chi.
template <bool W>
__host__ __device__ inline void sched_col_rows(const MaskGeom& g, int kv, int q0, int* clo,
                                               int* chi) {
  if constexpr (W) {
    row_range_for_kv(g, kv, q0, clo, chi);
  } else {
    *clo = upper_q_begin(g, kv) - q0;
    *chi = kBM;
  }
}

// The three schedules at one (q, kv) pair of the tiled part (kv < kv_main),
// through the same sched_* calls the kernels make (for the test-only mask
// export): vis[0] the forward (a pair of query tiles,
// whole 128-column key tiles), vis[1] the dK/dV pass (key tile fixed, 64-row
// query halves), vis[2] the dQ pass (64-column key halves).
template <bool W>
__host__ __device__ inline void sched_pattern_at(const MaskGeom& g, int q, int kv, uint8_t vis[3]) {
  const int kt = kv / kBN, k0 = kt * kBN;
  const int qt0 = (q / kBM) * kBM;
  // forward: the CTA of query tiles [qp0, qp0 + 2 kBM)
  {
    const int qp0 = (q / (2 * kBM)) * 2 * kBM;
    int kt0, n;
    sched_kv_tiles<W>(g, qp0, 2 * kBM, &kt0, &n);
    bool keep = kt >= kt0 && kt < kt0 + n;
    if (keep && sched_row_tile_masked<W>(g, full_keys_for_rows(g, qt0), qt0, k0)) {
      int clo, chi;
      sched_row_cols<W>(g, q, k0, &clo, &chi);
      keep = kv - k0 >= clo && kv - k0 <= chi;
    }
    vis[0] = keep ? 1 : 0;
  }
  // dK/dV: the CTA of key tile k0; warpgroup wg holds query columns q0 + 64 wg ..
  {
    int qtb, n;
    sched_q_tiles<W>(g, k0, &qtb, &n);
    bool keep = q / kBM >= qtb && q / kBM < qtb + n;
    if (keep && sched_col_tile_masked<W>(g, full_rows_for_keys(g, k0), qt0, k0)) {
      const int wg = (q - qt0) / 64;
      int clo, chi;
      sched_col_rows<W>(g, kv, qt0 + 64 * wg, &clo, &chi);
      const int c = q - qt0 - 64 * wg;
      keep = c >= clo && c <= chi;
    }
    vis[1] = keep ? 1 : 0;
  }
  // dQ: the CTA of query tile qt0; warpgroup wg holds key columns k0 + 64 wg ..
  {
    int kt0, n;
    sched_kv_tiles<W>(g, qt0, kBM, &kt0, &n);
    bool keep = kt >= kt0 && kt < kt0 + n;
    if (keep && sched_row_tile_masked<W>(g, full_keys_for_rows(g, qt0), qt0, k0)) {
      const int wg = (kv - k0) / 64;
      int clo, chi;
      sched_row_cols<W>(g, q, k0 + 64 * wg, &clo, &chi);
      const int c = kv - k0 - 64 * wg;
      keep = c >= clo && c <= chi;
    }
    vis[2] = keep ? 1 : 0;
  }
}

// One (q, kv) pair of the test-only mask export: vis[0..2] the forward, dK/dV
// and dQ schedules in the form the kernels run (general or one-sided),
// vis[3..5] the same in the general form.  Keys past the tiled part are the
// TTT suffix diagonals, key row i*Sq + q of segment i = 1..t, visible for
// rows below the key length, as the kernels' per-row diagonal passes address
// them.
__host__ __device__ inline void sched_pattern_pair(const MaskGeom& g, int q, int kv, bool general,
                                                   uint8_t vis[6]) {
  if (kv < g.kv_main) {
    sched_pattern_at<true>(g, q, kv, vis + 3);
    if (general) {
      vis[0] = vis[3];
      vis[1] = vis[4];
      vis[2] = vis[5];
    } else {
      sched_pattern_at<false>(g, q, kv, vis);
    }
    return;
  }
  const int64_t rel = (int64_t)kv - q;
  const bool diag = g.ttt > 0 && kv >= g.Sq && rel > 0 && rel % g.Sq == 0 &&
                    rel / g.Sq <= g.ttt && q < g.kv_len;
  for (int p = 0; p < 6; ++p) vis[p] = diag ? 1 : 0;
}

// Tile class for the test-only mask-pattern export: 0 empty, 1 partial, 2 full.
__host__ __device__ inline int tile_class(const MaskGeom& g, int q0, int k0) {
  int b, e;
  kv_range_for_rows(g, q0, kBM, &b, &e);
  if (k0 >= e || k0 + kBN <= b) return 0;
  return tile_is_full(g, q0, k0) ? 2 : 1;
}

}  // namespace attn
