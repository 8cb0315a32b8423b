// tile.cuh -- shared-memory tile geometry for [128 rows x D] bf16 tiles and
// the tcgen05 descriptors that read them.
//
// A tile is loaded by TMA in boxes of [128 rows x min(D, 64) columns] with
// the hardware swizzle that matches the row width (128 B rows: 128-byte
// swizzle; 64 B rows (D = 32): 64-byte swizzle; 32 B rows (D = 16): 32-byte
// swizzle).  For D = 128 the two 64-column boxes sit back to back.  Every
// tile starts on a 1024-byte boundary, so the swizzle phase of a row is its
// index mod 8.
//
// The same tile serves two operand roles:
//  * K-major (the contraction runs over D): Q and K for S = Q K^T, dO and V
//    for dP = dO V^T, K and Q for S^T = K Q^T, V and dO for dP^T = V dO^T.
//  * MN-major (the contraction runs over the 128 rows, N = D): V in
//    O += P V, dO in dV += P^T dO, Q in dK += dS^T Q, K in dQ += dS K.
#pragma once
#include "ptx.cuh"

namespace attn {

template <int D>
struct TileGeom {
  static_assert(D == 16 || D == 32 || D == 64 || D == 128, "head dim");
  static constexpr int ROWB = (D >= 64) ? 128 : D * 2;  // bytes per row in one box
  static constexpr int BOXC = (D >= 64) ? 64 : D;       // columns per box
  static constexpr int NBOX = D / BOXC;                 // boxes per tile
  static constexpr int BOX_BYTES = 128 * ROWB;
  static constexpr int TILE_BYTES = NBOX * BOX_BYTES;  // = 128 * D * 2
  static constexpr uint32_t LAYOUT =
      (D >= 64) ? kSwizzle128 : (D == 32 ? kSwizzle64 : kSwizzle32);
  static constexpr uint32_t SBO = 8 * ROWB;  // stride between 8-row groups
  static constexpr int KSTEPS = D / 16;      // MMA k-steps over D

  // K-major descriptor for k-step kk (columns 16kk .. 16kk+15).
  __device__ static uint64_t kmajor(uint32_t tile, int kk) {
    constexpr int per_box = BOXC / 16;
    const uint32_t a = tile + (uint32_t)(kk / per_box) * BOX_BYTES + (uint32_t)(kk % per_box) * 32u;
    return make_sdesc(a, 16u, SBO, LAYOUT);
  }
  // MN-major descriptor for k-step kk (rows 16kk .. 16kk+15), N = D.  The
  // leading byte offset steps between 64-column boxes, the stride byte offset
  // between 8-row groups.
  __device__ static uint64_t mnmajor(uint32_t tile, int kk) {
    const uint32_t a = tile + (uint32_t)kk * 16u * ROWB;
    return make_sdesc(a, (uint32_t)BOX_BYTES, SBO, LAYOUT);
  }
  // Same descriptors built once per buffer: the start address is the only
  // field that changes between k-steps and ring slots, and it sits in the low
  // 14 bits (address >> 4; shared memory addresses stay below 2^18), so a
  // k-step or slot is one 64-bit add on a precomputed base.
  __device__ static uint64_t kmajor_base(uint32_t tile) { return make_sdesc(tile, 16u, SBO, LAYOUT); }
  __device__ static uint64_t mnmajor_base(uint32_t tile) {
    return make_sdesc(tile, (uint32_t)BOX_BYTES, SBO, LAYOUT);
  }
  __host__ __device__ static constexpr uint64_t kmajor_step(int kk) {
    return (uint64_t)(((kk / (BOXC / 16)) * BOX_BYTES + (kk % (BOXC / 16)) * 32) >> 4);
  }
  __host__ __device__ static constexpr uint64_t mnmajor_step(int kk) {
    return (uint64_t)((kk * 16 * ROWB) >> 4);
  }
  __host__ __device__ static constexpr uint64_t bytes(int n) { return (uint64_t)(n >> 4); }

  // Issue the TMA boxes of one tile (rows r0 .. r0+127 of head h, batch b).
  __device__ static void load(void* dst, const CUtensorMap* m, uint64_t* bar, int r0, int h,
                              int b) {
#pragma unroll
    for (int x = 0; x < NBOX; ++x)
      tma_load_4d(static_cast<char*>(dst) + x * BOX_BYTES, m, bar, x * BOXC, r0, h, b);
  }
  // The same, with the ATTN_DEBUG check that the tile overlaps the first rows +
  // 128 rows of the tensor (a pair's second query tile may lie just past its
  // end, read as zeros) and that head and batch entry exist; the copy is
  // skipped if not.
  __device__ static void load(void* dst, const CUtensorMap* m, uint64_t* bar, int r0, int h,
                              int b, int rows, int H, int B, uint32_t* err, int site) {
    if (ATTN_CHECK(err, r0 >= 0 && r0 < rows + 128 && h >= 0 && h < H && b >= 0 && b < B, site))
      load(dst, m, bar, r0, h, b);
    (void)rows, (void)H, (void)B, (void)err, (void)site;
  }
};

}  // namespace attn
