// mma_rate.cu -- tensor-pipe microbenchmark (measurement tool, not part of the
// library): back-to-back tcgen05.mma throughput per SM for the shapes the
// attention kernels issue, the forward's own issue sequences, and what the
// issuing thread's barrier reads and shared-memory loads between MMA batches
// cost.  One CTA per SM; one thread issues; cycles from clock64 on that thread,
// median over the SMs.  Built and run by mma_rate.py.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <vector>

#include "csrc/ptx.cuh"
#include "csrc/tile.cuh"

using namespace attn;

namespace {

constexpr int kData = 128 * 1024;  // operand area of shared memory
constexpr int kSmem = kData + 1024 + 256;

enum Case : int {
  kSS = 0,          // A, B in shared memory (K-major), N = template N
  kTS = 1,          // A in tensor memory, B MN-major in shared memory, N = template N
  kSSCopies = 2,    // kSS N = 128 while warp 1 streams 32 KB bulk copies into shared memory
  kFwd128 = 3,      // head dim 128 forward order: PV0, S0, PV1, S1 (+ their commits)
  kFwd128Wait = 4,  // kFwd128 with warps 1-8 waiting on a barrier meanwhile
  kFwd64 = 5,       // head dim 64 forward order (S: N = 128, K = 64; PV: N = 64, K = 128)
  kFwd64Handoff = 6,   // kFwd64 + S_x -> warps -> P_x hand-off before every PV_x
  kFwd64Fence = 7,     // kFwd64 + tcgen05.fence::after_thread_sync before every PV_x
  kFwd64WaitDone = 8,  // kFwd64 + try_wait on an already completed phase before every PV_x
  kFwd64TestDone = 9,  // kFwd64 + test_wait on an already completed phase before every PV_x
  kFwd64LoadShared = 10,  // kFwd64 + a volatile shared-memory load before every PV_x
};

__device__ int g_random_operands = 1;

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// iters: MMA groups; cases kSS / kTS / kSSCopies issue 4 MMAs per group, the
// forward orders a whole key tile per group.
template <int CASE, int N>
__global__ void __launch_bounds__(384, 1) mma_loop(long long* cyc, uint32_t* err, int iters,
                                                  const uint8_t* gsrc, long long gbytes,
                                                  int* copies) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = raw + (((smem_u32(raw) + 1023u) & ~1023u) - smem_u32(raw));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kData);
  uint64_t* done = bars;            // the MMAs' final commit
  uint64_t* cbar = bars + 1;        // [2] bulk-copy regions
  uint64_t* gate = bars + 3;        // released after the MMAs (waiting warps)
  uint64_t* s_full = bars + 4;      // [2]
  uint64_t* p_ready = bars + 6;     // [2]
  uint64_t* completed = bars + 8;   // a phase completed before the timing
  volatile int* stop = reinterpret_cast<volatile int*>(bars + 9);
  volatile int* abort_flag = stop + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);

  const bool rnd = g_random_operands != 0;
  for (int i = threadIdx.x; i < kData / 4; i += blockDim.x) {
    uint32_t w = 0u;
    if (rnd) {  // bf16 pairs ~ U(-1, 1) from an integer hash
      uint32_t h = (uint32_t)i * 2654435761u ^ (blockIdx.x * 97u + 12345u);
      h ^= h >> 15;
      h *= 2246822519u;
      h ^= h >> 13;
      const float a = (h & 0xffffu) / 32768.0f - 1.0f, b = (h >> 16) / 32768.0f - 1.0f;
      w = (__float_as_uint(a) >> 16) | (__float_as_uint(b) & 0xffff0000u);
    }
    reinterpret_cast<uint32_t*>(smem)[i] = w;
  }
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    mbar_init(&cbar[0], 1);
    mbar_init(&cbar[1], 1);
    mbar_init(gate, 1);
    mbar_init(completed, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_ready[x], 128);
    }
    *stop = 0;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x / 32 == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{err, abort_flag, 2000000000ull};
  if (CASE == kTS && threadIdx.x < 128) {  // the A operand columns [256, 264): zeros
    uint32_t z[16];
    for (int e = 0; e < 16; ++e) z[e] = 0u;
    tmem_st16(tmem + ((uint32_t)(threadIdx.x / 32 * 32) << 16) + 256, z);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (threadIdx.x == 0) {
    mbar_arrive(completed);
    bool good = true;
    const long long t0 = clock64();
    if constexpr (CASE == kSS || CASE == kSSCopies) {
      using TG = TileGeom<128>;
      constexpr uint32_t idesc = make_idesc_bf16(128, N, false, false);
      const uint64_t a = TG::kmajor_base(smem_u32(smem));                     // [0, 32 KB)
      const uint64_t b = TG::kmajor_base(smem_u32(smem + TG::TILE_BYTES));   // [32, 64 KB)
      for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ss(tmem, a + TG::kmajor_step(kk), b + TG::kmajor_step(kk), idesc, (it | kk) != 0);
    } else if constexpr (CASE == kTS) {
      using TG = TileGeom<N>;
      constexpr uint32_t idesc = make_idesc_bf16(128, N, false, true);
      const uint64_t b = TG::mnmajor_base(smem_u32(smem));
      for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ts(tmem, tmem + 256, b + TG::mnmajor_step(kk), idesc, (it | kk) != 0);
    } else if constexpr (CASE == kFwd128 || CASE == kFwd128Wait) {
      // Q0 [0, 32K) Q1 [32K, 64K) K [64K, 96K) V [96K, 128K); S/P_x at 128x, O_x at 256 + 128x
      using TG = TileGeom<128>;
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = make_idesc_bf16(128, 128, false, true);
      const uint64_t dQ0 = TG::kmajor_base(smem_u32(smem));
      const uint64_t dK = TG::kmajor_base(smem_u32(smem + 2 * TG::TILE_BYTES));
      const uint64_t dV = TG::mnmajor_base(smem_u32(smem + 3 * TG::TILE_BYTES));
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + 256 + x * 128, tmem + x * 128 + kk * 8, dV + TG::mnmajor_step(kk),
                    idesc_o, 1u);
          umma_commit(&cbar[0]);
          const uint64_t qd = dQ0 + TG::bytes(x * TG::TILE_BYTES);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ss(tmem + x * 128, qd + TG::kmajor_step(kk), dK + TG::kmajor_step(kk), idesc_s,
                    kk > 0);
          umma_commit(&cbar[1]);
          umma_commit(&cbar[1]);
        }
      }
    } else {
      // head dim 64: Q0 [0, 16K) Q1 [16K, 32K) K [32K, 48K) V [48K, 64K);
      // S/P_x at 128x, O_x at 256 + 64x
      using TG = TileGeom<64>;
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = make_idesc_bf16(128, 64, false, true);
      const uint64_t dQ0 = TG::kmajor_base(smem_u32(smem));
      const uint64_t dK = TG::kmajor_base(smem_u32(smem + 2 * TG::TILE_BYTES));
      const uint64_t dV = TG::mnmajor_base(smem_u32(smem + 3 * TG::TILE_BYTES));
      auto issue_s = [&](int x) {
        const uint64_t qd = dQ0 + TG::bytes(x * TG::TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ss(tmem + x * 128, qd + TG::kmajor_step(kk), dK + TG::kmajor_step(kk), idesc_s,
                  kk > 0);
        umma_commit(&s_full[x]);
      };
      auto issue_pv = [&](int x) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + 256 + x * 64, tmem + x * 128 + kk * 8, dV + TG::mnmajor_step(kk),
                  idesc_o, 1u);
      };
      issue_s(0);
      issue_s(1);
      for (int it = 1; it < iters && good; ++it) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (CASE == kFwd64Handoff) {
            good = mbar_wait(&p_ready[x], (uint32_t)(it - 1) & 1u, ctl);
            tc_fence_after();
          }
          if (CASE == kFwd64Fence) tc_fence_after();
          if (CASE == kFwd64WaitDone) good = mbar_wait(completed, 0, ctl);
          if (CASE == kFwd64TestDone) good = mbar_test_wait(completed, 0) || mbar_wait(completed, 0, ctl);
          if (CASE == kFwd64LoadShared) good = *stop == 0;
          issue_pv(x);
          issue_s(x);
        }
      }
    }
    umma_commit(done);
    const bool ok = mbar_wait(done, 0, ctl) && good;
    const long long t1 = clock64();
    cyc[blockIdx.x] = ok ? (t1 - t0) : -1;
    *stop = 1;
    mbar_arrive(gate);
  }
  if (CASE == kFwd64Handoff && threadIdx.x >= 32 && threadIdx.x < 288) {
    // "softmax" warps 1-4 (tile 0) and 5-8 (tile 1): wait for S_x, release P_x at once
    const int x = (threadIdx.x / 32 - 1) / 4;
    for (int it = 0; it < iters - 1; ++it) {
      if (!mbar_wait_warp(&s_full[x], (uint32_t)it & 1u, ctl)) break;
      tc_fence_after();
      tc_fence_before();
      mbar_arrive(&p_ready[x]);
    }
  }
  if (CASE == kFwd128Wait && threadIdx.x >= 32 && threadIdx.x < 288) mbar_wait_warp(gate, 0, ctl);
  if (CASE == kSSCopies && threadIdx.x == 32) {
    // copies into [64 KB, 96 KB) and [96 KB, 128 KB) in turn, one in flight per region
    int n = 0;
    const long long chunks = gbytes / 32768;
    long long off = (long long)(blockIdx.x * 37) % chunks;
    while (!*stop) {
      const int r = n & 1;
      if (n >= 2 && !mbar_wait(&cbar[r], (uint32_t)((n - 2) / 2) & 1u, ctl)) break;
      mbar_arrive_expect_tx(&cbar[r], 32768);
      bulk_g2s(smem + 65536 + r * 32768, gsrc + off * 32768, 32768, &cbar[r]);
      off = (off + 1) % chunks;
      ++n;
    }
    for (int m = n - 2 < 0 ? 0 : n - 2; m < n; ++m)
      mbar_wait(&cbar[m & 1], (uint32_t)(m / 2) & 1u, ctl);
    copies[blockIdx.x] = n;
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x / 32 == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

struct Run {
  double cycles = 0;  // median over SMs of the timed region
  double copies = 0;  // median bulk copies (kSSCopies)
  bool ok = true;
};

template <int CASE, int N>
Run run(int nsm, int iters, int threads, const uint8_t* gsrc = nullptr, long long gbytes = 0) {
  static long long* dcyc = nullptr;
  static uint32_t* derr = nullptr;
  static int* dcop = nullptr;
  if (!dcyc) {
    cudaMalloc(&dcyc, nsm * 8);
    cudaMalloc(&derr, 4);
    cudaMalloc(&dcop, nsm * 4);
  }
  cudaMemset(derr, 0, 4);
  auto k = mma_loop<CASE, N>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  Run r;
  for (int rep = 0; rep < 2; ++rep) {
    k<<<nsm, threads, kSmem>>>(dcyc, derr, iters, gsrc, gbytes, dcop);
    if (cudaDeviceSynchronize() != cudaSuccess) {
      r.ok = false;
      return r;
    }
  }
  std::vector<long long> c(nsm);
  std::vector<int> n(nsm);
  cudaMemcpy(c.data(), dcyc, nsm * 8, cudaMemcpyDeviceToHost);
  cudaMemcpy(n.data(), dcop, nsm * 4, cudaMemcpyDeviceToHost);
  uint32_t herr = 0;
  cudaMemcpy(&herr, derr, 4, cudaMemcpyDeviceToHost);
  std::sort(c.begin(), c.end());
  std::sort(n.begin(), n.end());
  r.ok = herr == 0 && c[0] > 0;
  r.cycles = (double)c[nsm / 2];
  r.copies = (double)n[nsm / 2];
  return r;
}

void print_mma(const char* name, int n_dim, const Run& r, double mmas, bool random) {
  const double per = r.cycles / mmas;
  const double flop = 2.0 * 128 * n_dim * 16;
  printf("{\"case\": \"%s\", \"operands\": \"%s\", \"cycles_per_mma\": %.1f, "
         "\"flop_per_clk_sm\": %.0f, \"pct_of_8192\": %.1f, \"ok\": %s}\n",
         name, random ? "random" : "zeros", per, flop / per, 100.0 * flop / per / 8192,
         r.ok ? "true" : "false");
}

void print_seq(const char* name, const Run& r, double iterations, int mmas_per_iteration,
               bool random) {
  printf("{\"case\": \"%s\", \"operands\": \"%s\", \"cycles_per_key_tile\": %.1f, "
         "\"mmas_per_key_tile\": %d, \"ok\": %s}\n",
         name, random ? "random" : "zeros", r.cycles / iterations, mmas_per_iteration,
         r.ok ? "true" : "false");
}

}  // namespace

int main(int argc, char** argv) {
  int nsm = 0;
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  const int groups = 4096;  // 16384 MMAs in the single-shape cases
  for (int random = 0; random < 2; ++random) {
    cudaMemcpyToSymbol(g_random_operands, &random, sizeof(int));
    print_mma("SS M128 N64 K16", 64, run<kSS, 64>(nsm, groups, 128), groups * 4.0, random);
    print_mma("SS M128 N128 K16", 128, run<kSS, 128>(nsm, groups, 128), groups * 4.0, random);
    print_mma("SS M128 N256 K16", 256, run<kSS, 256>(nsm, groups, 128), groups * 4.0, random);
    print_mma("TS M128 N64 K16", 64, run<kTS, 64>(nsm, groups, 128), groups * 4.0, random);
    print_mma("TS M128 N128 K16", 128, run<kTS, 128>(nsm, groups, 128), groups * 4.0, random);
    {
      const long long gb = 32ll << 20;  // an L2-resident source
      uint8_t* g = nullptr;
      cudaMalloc(&g, gb);
      cudaMemset(g, 0, gb);
      const Run r = run<kSSCopies, 128>(nsm, groups, 128, g, gb);
      print_mma("SS M128 N128 K16 + bulk copies into shared memory", 128, r, groups * 4.0, random);
      printf("{\"case\": \"bulk copies during the MMAs\", \"bytes_per_clk_sm\": %.1f}\n",
             r.copies * 32768.0 / r.cycles);
      cudaFree(g);
    }
    const int it128 = groups / 8, it64 = groups / 6;  // 16384 MMAs again
    print_seq("forward order, head dim 128", run<kFwd128, 128>(nsm, it128, 128), it128, 32, random);
    print_seq("forward order, head dim 128, 8 warps waiting",
              run<kFwd128Wait, 128>(nsm, it128, 384), it128, 32, random);
    print_seq("forward order, head dim 64", run<kFwd64, 128>(nsm, it64, 128), it64, 24, random);
    print_seq("forward order, head dim 64, S -> warps -> P hand-off",
              run<kFwd64Handoff, 128>(nsm, it64, 384), it64, 24, random);
    print_seq("forward order, head dim 64, fence before each PV",
              run<kFwd64Fence, 128>(nsm, it64, 128), it64, 24, random);
    print_seq("forward order, head dim 64, try_wait on a completed phase before each PV",
              run<kFwd64WaitDone, 128>(nsm, it64, 128), it64, 24, random);
    print_seq("forward order, head dim 64, test_wait on a completed phase before each PV",
              run<kFwd64TestDone, 128>(nsm, it64, 128), it64, 24, random);
    print_seq("forward order, head dim 64, volatile shared load before each PV",
              run<kFwd64LoadShared, 128>(nsm, it64, 128), it64, 24, random);
  }
  (void)argc;
  (void)argv;
  return 0;
}
