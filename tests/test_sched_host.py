"""The kernels' tile schedules, compiled for the host, against the oracle's
visibility predicate bit for bit (no GPU needed).

tests/sched_host.cpp builds attention_tcgen05_tmem_gb300/csrc/sched.cuh --
the functions every attention kernel calls to pick its key or query tiles and
to mask partial tiles -- with a host compiler and evaluates the forward, dK/dV
and dQ schedules at every (query, key) pair, in the one-sided form (full,
causal and TTT masks without key lengths) and in the general form.  Each plane
must equal oracle.mask, the SpecForge eagle3 mask_mod read as a predicate.
The GPU test test_gpu_mask.py checks the same planes as the device computes
them."""
import ctypes
import os
import random
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KIND = {"full": 0, "causal": 1, "ttt": 2, "window": 3}


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("sched") / "libsched_host.so")
    subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-I",
                    os.path.join(ROOT, "attention_tcgen05_tmem_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "sched_host.cpp"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.sched_pattern_host.argtypes = [ctypes.c_int] * 8 + [ctypes.c_void_p]
    lib.sched_pattern_host.restype = None
    return lib


def planes(lib, mask, t, Sq, Skv, window=None, length=None, general=False):
    bits = np.zeros((6, Sq, Skv), dtype=np.uint8)
    wl, wr = window if window is not None else (0, 0)
    lib.sched_pattern_host(KIND[mask], t, wl, wr, Sq, Skv, -1 if length is None else length,
                           1 if general else 0, bits.ctypes.data)
    return bits


def check(lib, mask, t, Sq, Skv, window=None, length=None):
    want = oracle.mask(mask, t, Sq, Skv, window=window, length=length)
    one_sided = mask != "window" and length is None
    forms = [False, True] if one_sided else [True]
    for general in forms:
        bits = planes(lib, mask, t, Sq, Skv, window, length, general)
        for p, name in enumerate(("forward", "dK/dV", "dQ") * 2):
            form = "general" if (general or p >= 3) else "one-sided"
            got = bits[p]
            if not np.array_equal(got, want):
                q, kv = np.argwhere(got != want)[0]
                raise AssertionError(f"{mask} t={t} Sq={Sq} Skv={Skv} w={window} len={length}: "
                                     f"{name} ({form}) differs at q={q} kv={kv}: "
                                     f"{got[q, kv]} vs {want[q, kv]}")


# one-sided problems, TTT at every step of the EAGLE3 workload, ragged tails
ONE_SIDED = ([("causal", 0, S, S) for S in (1, 5, 127, 128, 129, 255, 256, 257, 700)] +
             [("causal", 0, 300, 700), ("causal", 0, 700, 300), ("causal", 0, 129, 1)] +
             [("full", 0, 333, 129), ("full", 0, 1, 257), ("full", 0, 256, 256)] +
             [("ttt", t, S, (t + 1) * S) for t in range(7) for S in (5, 128, 200, 257, 640)])
GENERAL = [("window", 0, 1000, 1000, (200, 0), None), ("window", 0, 900, 900, (130, 130), None),
           ("window", 0, 500, 777, (0, 300), None), ("window", 0, 450, 300, (5, 5), None),
           ("window", 0, 600, 600, (1, 0), 333), ("causal", 0, 700, 700, None, 321),
           ("full", 0, 333, 500, None, 129), ("causal", 0, 300, 300, None, 0),
           ("ttt", 2, 384, 1152, None, 200), ("ttt", 6, 260, 1820, None, 3),
           ("ttt", 4, 300, 1500, None, 129), ("ttt", 5, 257, 1542, None, 256)]


@pytest.mark.parametrize("mask,t,Sq,Skv", ONE_SIDED)
def test_one_sided_and_general_schedules_equal_the_mask(lib, mask, t, Sq, Skv):
    check(lib, mask, t, Sq, Skv)


@pytest.mark.parametrize("mask,t,Sq,Skv,window,length", GENERAL)
def test_general_schedule_equals_the_mask(lib, mask, t, Sq, Skv, window, length):
    check(lib, mask, t, Sq, Skv, window, length)


def test_random_problems(lib):
    """Random shapes of every mask kind, extents and key lengths included."""
    rng = random.Random(1234)
    for _ in range(150):
        mask = rng.choice(["full", "causal", "ttt", "window"])
        t = rng.randint(0, 6) if mask == "ttt" else 0
        Sq = rng.randint(1, 420)
        Skv = (t + 1) * Sq if mask == "ttt" else rng.randint(1, 420)
        window = (rng.randint(0, 300), rng.randint(0, 300)) if mask == "window" else None
        kv_main = Sq if mask == "ttt" else Skv
        length = rng.choice([None, rng.randint(0, kv_main)])
        check(lib, mask, t, Sq, Skv, window, length)
