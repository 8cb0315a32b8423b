// aux.cu -- test-only kernels: the device view of the mask (the forward, dK/dV
// and dQ schedules, through the scheduling calls the kernels make), a one-tile
// tcgen05 descriptor probe, and a bounded-wait self-test that times out on
// purpose (nothing ever arrives on its barrier).
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "sched.cuh"
#include "tile.cuh"

namespace attn {
namespace {

// bits[p][q][kv], six planes of Sq x Skv: planes 0-2 the forward, dK/dV and
// dQ schedules in the form the kernels run for this problem (one-sided unless
// needs_general_mask), planes 3-5 the same three in the general form.  Every
// plane includes the TTT suffix diagonals exactly as the kernels address them
// (key row i*Sq + q, i = 1..t).  tiles[qt][kt] = tile class of the tiled part.
// With per-batch key lengths this is the view of batch entry 0.
__global__ void mask_pattern_kernel(const Dims d, bool general, uint8_t* bits, uint8_t* tiles) {
  const MaskGeom g = with_len(d.geom, d.seqlens, 0);
  const int64_t n = (int64_t)d.Sq * d.Skv;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int q = (int)(idx / d.Skv);
    const int kv = (int)(idx % d.Skv);
    uint8_t vis[6];
    sched_pattern_pair(g, q, kv, general, vis);
    for (int p = 0; p < 6; ++p) bits[p * n + idx] = vis[p];
  }
  if (tiles != nullptr) {
    const int nqt = cdiv(d.Sq, kBM), nkt = cdiv(g.kv_main, kBN);
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < (int64_t)nqt * nkt;
         idx += (int64_t)gridDim.x * blockDim.x) {
      const int qt = (int)(idx / nkt), kt = (int)(idx % nkt);
      tiles[idx] = (uint8_t)tile_class(g, qt * kBM, kt * kBN);
    }
  }
}

// ---------------------------------------------------------------- probe
template <int D>
__global__ void __launch_bounds__(128, 1)
    probe_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                 const __nv_bfloat16* a_global, float* c, int mode, Ctl cc) {
  using TG = TileGeom<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + (((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw));
  uint8_t* tA = smem;
  uint8_t* tB = smem + TG::TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * TG::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{cc.err, abort_flag, cc.budget_ns};
  const int r = threadIdx.x;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  if (mode == 1) {
    // A row r (128 bf16) into TMEM columns [128, 192), two values per column
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(a_global + (int64_t)r * 128);
    uint32_t v[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = arow[h * 32 + e];
      tmem_st32(tmem + lane_base + 128 + h * 32, v);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (threadIdx.x == 0) {
    if (mode == 0) {
      mbar_arrive_expect_tx(&bars[0], 2 * TG::TILE_BYTES);
      TG::load(tA, &ta, &bars[0], 0, 0, 0);
      TG::load(tB, &tb, &bars[0], 0, 0, 0);
    } else {
      mbar_arrive_expect_tx(&bars[0], TG::TILE_BYTES);
      TG::load(tB, &tb, &bars[0], 0, 0, 0);
    }
    if (mbar_wait(&bars[0], 0, ctl)) {
      tc_fence_after();
      if (mode == 0) {
        constexpr uint32_t idesc = make_idesc_bf16(128, 128, false, false);
        for (int kk = 0; kk < TG::KSTEPS; ++kk)
          umma_ss(tmem, TG::kmajor(smem_u32(tA), kk), TG::kmajor(smem_u32(tB), kk), idesc, kk > 0);
      } else {
        constexpr uint32_t idesc = make_idesc_bf16(128, D, false, true);
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem, tmem + 128 + 8 * kk, TG::mnmajor(smem_u32(tB), kk), idesc, kk > 0);
      }
      umma_commit(&bars[1]);
    } else {
      umma_commit(&bars[1]);
    }
  }
  __syncwarp();
  const bool ok = mbar_wait_warp(&bars[1], 0, ctl);
  if (ok) {
    tc_fence_after();
    const int ncol = (mode == 0) ? 128 : D;
    for (int c0 = 0; c0 < ncol; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + lane_base + c0, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) c[(int64_t)r * ncol + c0 + e] = __uint_as_float(v[e]);
    }
  }
  (void)lane;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ------------------------------------------------------- wait self-test
// Waits on a barrier that nothing will ever complete; the bounded wait must
// give up, record kErrWaitTimeout and let the kernel return normally.
__global__ void selftest_wait_kernel(Ctl cc) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{cc.err, &abort_flag, cc.budget_ns};
  mbar_wait_warp(&bar, 0, ctl);
}

// A device check that fails on purpose (ATTN_DEBUG builds; no memory access).
__global__ void selftest_check_kernel(Ctl cc) {
  (void)ATTN_CHECK(cc.err, threadIdx.x == 1u << 30, 99);
  (void)cc;
}

template <int D>
cudaError_t launch_probe_d(int mode, const CUtensorMap& ta, const CUtensorMap& tb,
                           const void* a_global, float* c, Ctl ctl, cudaStream_t s) {
  const int smem = 2 * TileGeom<D>::TILE_BYTES + 64 + 1024;
  auto kern = probe_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<1, 128, smem, s>>>(ta, tb, static_cast<const __nv_bfloat16*>(a_global), c, mode, ctl);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mask_pattern(const Dims& d, uint8_t* bits, uint8_t* tiles, cudaStream_t s) {
  const int64_t n = (int64_t)d.Sq * d.Skv;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  mask_pattern_kernel<<<(unsigned)blocks, 256, 0, s>>>(d, needs_general_mask(d), bits, tiles);
  return cudaGetLastError();
}

cudaError_t launch_probe(int mode, int D, const CUtensorMap& ta, const CUtensorMap& tb,
                         const void* a_global, float* c, Ctl ctl, cudaStream_t s) {
  switch (D) {
    case 16: return launch_probe_d<16>(mode, ta, tb, a_global, c, ctl, s);
    case 32: return launch_probe_d<32>(mode, ta, tb, a_global, c, ctl, s);
    case 64: return launch_probe_d<64>(mode, ta, tb, a_global, c, ctl, s);
    case 128: return launch_probe_d<128>(mode, ta, tb, a_global, c, ctl, s);
    default: return cudaErrorInvalidValue;
  }
}

bool debug_checks_built() {
#ifdef ATTN_DEBUG
  return true;
#else
  return false;
#endif
}

cudaError_t launch_selftest_check(Ctl ctl, cudaStream_t s) {
  selftest_check_kernel<<<1, 32, 0, s>>>(ctl);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(Ctl ctl, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(ctl);
  return cudaGetLastError();
}

}  // namespace attn
