// sched.cuh -- tile classification and iteration ranges (host and device).
//
// The attention grid is cut into 128-row query tiles and 128-column key
// tiles.  Masks are evaluated arithmetically, never from a mask tensor
// (FlexAttention's BlockMask idea -- skip empty blocks, and skip the mask
// test on full blocks -- from the SpecForge post, "Flex Attention"; the
// HOT-Step page, section 3, reports that skipping all -inf tiles halves the
// causal work).
//
// The tiled part of every mask is one predicate:
//     visible(q, kv) = kv < kv_main  and  (mask == FULL  or  kv <= q - shift)
// with shift = 0 (causal), shift = t (TTT step t: segment 0's causal part
// shrinks by one diagonal per appended segment, SpecForge "Flex Attention"
// causal_mask with shift_left = t), kv_main = Skv for full/causal and Sq for
// TTT.  The TTT suffix diagonals (kv = q + i*Sq, i = 1..t) are not tiles:
// the kernels merge them in a separate per-row pass.
#pragma once
#include <cstdint>

namespace attn {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // key rows per tile

enum MaskKind : int { kMaskFull = 0, kMaskCausal = 1, kMaskTTT = 2 };

struct MaskGeom {
  int kind;     // MaskKind
  int shift;    // 0 for causal, t for TTT, unused for full
  int Sq;       // query rows
  int kv_main;  // key rows of the tiled part
  int ttt;      // number of suffix diagonals (t for TTT, else 0)
};

__host__ __device__ inline MaskGeom make_geom(int kind, int t, int Sq, int Skv) {
  MaskGeom g;
  g.kind = kind;
  g.shift = (kind == kMaskTTT) ? t : 0;
  g.Sq = Sq;
  g.kv_main = (kind == kMaskTTT) ? Sq : Skv;
  g.ttt = (kind == kMaskTTT) ? t : 0;
  return g;
}

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Keys [0, end) that some query of rows [q0, q0 + rows) may see.
__host__ __device__ inline int kv_end_for_rows(const MaskGeom& g, int q0, int rows) {
  if (g.kind == kMaskFull) return g.kv_main;
  int last_q = q0 + rows - 1;
  if (last_q > g.Sq - 1) last_q = g.Sq - 1;
  long e = (long)last_q - g.shift + 1;
  if (e < 0) e = 0;
  if (e > g.kv_main) e = g.kv_main;
  return (int)e;
}

// A (query tile, key tile) pair needs no per-element test iff every pair in it
// is visible (rows beyond Sq are never stored, so they do not matter).
__host__ __device__ inline bool tile_is_full(const MaskGeom& g, int q0, int k0) {
  if (k0 + kBN > g.kv_main) return false;
  if (g.kind == kMaskFull) return true;
  return k0 + kBN - 1 <= q0 - g.shift;
}

// Per-row column limit inside a key tile: column c (key k0 + c) is visible to
// query q iff c <= limit.  Negative means nothing visible.
__host__ __device__ inline int col_limit(const MaskGeom& g, int q, int k0) {
  long lim = (long)g.kv_main - 1 - k0;
  if (g.kind != kMaskFull) {
    long c = (long)q - g.shift - k0;
    if (c < lim) lim = c;
  }
  if (lim < -1) lim = -1;
  if (lim > kBN) lim = kBN;
  return (int)lim;
}

// First query row that can see any key of the key tile starting at k0.
__host__ __device__ inline int q_begin_for_kv(const MaskGeom& g, int k0) {
  if (g.kind == kMaskFull) return 0;
  long b = (long)k0 + g.shift;
  return b > g.Sq ? g.Sq : (int)b;
}

// Tile class for the test-only mask-pattern export: 0 empty, 1 partial, 2 full.
__host__ __device__ inline int tile_class(const MaskGeom& g, int q0, int k0) {
  const int end = kv_end_for_rows(g, q0, kBM);
  if (k0 >= end) return 0;
  return tile_is_full(g, q0, k0) ? 2 : 1;
}

}  // namespace attn
