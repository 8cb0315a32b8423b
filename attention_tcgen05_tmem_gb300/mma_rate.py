"""Tensor-pipe microbenchmark (measurement tool, not part of the library).

Compiles mma_rate.cu for sm_103a into _build/ and runs it on cuda:0: one CTA
per SM issues back-to-back tcgen05.mma from one thread, and the program prints
one JSON line per case (median over the SMs of clock64 cycles):

- cycles per 128 x N x 16 MMA for N = 64, 128, 256 with both operands in shared
  memory, and for N = 64, 128 with A in tensor memory (the P V shape);
- the same N = 128 MMAs while another warp streams bulk copies into shared
  memory, and the copy bytes per clock that reached the SM meanwhile;
- the forward's issue order per key tile at head dim 128 (P V0, S0, P V1, S1 with
  their commits), alone and with eight warps waiting on a barrier;
- the head-dim-64 forward order, alone, with the S -> elementwise warps -> P
  hand-off of the real kernel, and with one tcgen05 fence, one try_wait or
  test_wait on an already completed phase, or one volatile shared-memory load
  before every P V: what the issuing thread's reads between MMA batches cost.

Every case runs with zero and with random bf16 operands.

    python -m attention_tcgen05_tmem_gb300.mma_rate
"""
from __future__ import annotations

import os
import subprocess
import sys

from . import build as lib_build

HERE = os.path.dirname(os.path.abspath(__file__))


def build() -> str:
    out_dir = lib_build.BUILD_DIR
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "mma_rate")
    src = os.path.join(HERE, "mma_rate.cu")
    deps = [src] + [os.path.join(HERE, "csrc", f) for f in ("ptx.cuh", "tile.cuh")]
    if os.path.exists(exe) and all(os.path.getmtime(d) <= os.path.getmtime(exe) for d in deps):
        return exe
    cmd = [lib_build.nvcc(), *lib_build.ARCH, "-O3", "-std=c++17", "--expt-relaxed-constexpr",
           "-I", HERE, "-I", os.path.join(lib_build.ROOT, "include"), src, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for mma_rate.cu:\n{r.stdout}\n{r.stderr}")
    return exe


def main() -> int:
    exe = build()
    return subprocess.run([exe]).returncode


if __name__ == "__main__":
    sys.exit(main())
