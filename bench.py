#!/usr/bin/env python3
"""Fused training attention on GB300: forward + deterministic backward TFLOPS.

One step = one pass of the whole hot path over one batch of synthetic input:
attn_train_fwd (O, LSE) then the backward passes (Delta prep, dK/dV, dQ, and
the TTT suffix pass when the mask has one), all through the C ABI.  The
EAGLE3 TTT workload's step is the forward + backward of all seven TTT steps
(t = 0..6, K/V growing by one segment per step).

Throughput is mask-aware: F = 3.5 * 4 * D * N_vis FLOPs per step, N_vis the
exact number of visible (q, kv) pairs (forward 2 GEMMs, backward 5).  Inputs
are seeded N(0,1) draws rounded to bf16 (attention_tcgen05_tmem_gb300.synth).

Prints ONE JSON line on rank 0 (``--all``: one line per workload).  Under
torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas; attention needs no collective), the timed region is
bracketed by barriers and the max over ranks is taken.  ``--impl reference``
times the fp64 CPU oracle on the host cores on a bounded sample of the same
workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOPS (mask-aware, bf16) and % of GB300 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TTT_ALL = "eagle3_ttt_steps0-6"
# Host-device copies on GB300 (Grace host) pause for 20-80 ms about twice a
# second; the end-to-end session gets enough slots to keep computing through
# a pause this long
E2E_RIDE_MS = 80.0


def bench_workloads():
    """name -> list of synth.Workload run back to back in one step."""
    from attention_tcgen05_tmem_gb300 import synth
    d = {w.name: [w] for w in synth.ALL + synth.PROFILE}
    d[TTT_ALL] = list(synth.TTT_STEPS)
    return d


def headline_names():
    from attention_tcgen05_tmem_gb300 import synth
    return ([synth.TINY.name] + [w.name for w in synth.SWEEP] +
            [synth.LONG_GQA.name, TTT_ALL, synth.DIT_SELF.name, synth.DIT_CROSS.name,
             synth.DIT_WINDOW.name, synth.SWA_GQA.name, synth.VARLEN_GQA.name,
             synth.VARLEN_TTT.name, synth.DIT_ADDMASK.name])


def parse_args():
    from attention_tcgen05_tmem_gb300 import synth
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=synth.LONG_GQA.name,
                    help="one of: " + ", ".join(list(bench_workloads()) + list(loss_table())))
    ap.add_argument("--all", action="store_true", help="one line per workload of the pages")
    ap.add_argument("--out", choices=["fp32", "bf16"], default="fp32",
                    help="dtype of O, dQ, dK, dV (fp32 is the parity-gated configuration)")
    ap.add_argument("--repeats", type=int, default=3,
                    help="timed regions per workload (interleaved across workloads); the "
                         "line reports the median region and the spread")
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches (CUDA events between kernels) instead of a "
                         "CUDA-graph replay of each step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunk", type=int, default=0,
                    help="kv heads per chunk of the host-memory step (0 = automatic)")
    ap.add_argument("--e2e-slots", type=int, default=0,
                    help="device slots of the host-memory session (0 = enough for about "
                         f"{E2E_RIDE_MS:.0f} ms of compute, at most 16)")
    ap.add_argument("--e2e-seconds", type=float, default=1.0,
                    help="length of each timed end-to-end region")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 100 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, pw, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        try:
            lines = open(self.path).read().strip().splitlines()
        except OSError:
            lines = []
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if self.path:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "power_w_max": max(pw) if pw else None, "samples": len(sm)}


# ------------------------------------------------------------- CPU oracle
def cpu_sample(ws, target_s: float, inputs=None, rows=None):
    """Time the fp64 oracle (forward + backward) on a bounded sample of the
    workload's first (or only) shape: the q heads of the first kv-head
    groups (at least as many q heads as host threads) and the last R query
    rows (those with the most visible keys), R grown until the run takes
    about target_s seconds.  Returns (TFLOP/s, description, threads, per pass)
    with per pass = {"fwd": TFLOP/s, "bwd": TFLOP/s, "rows": R} (4 D and 10 D
    FLOP per visible pair).  rows=R skips the search and runs R rows once."""
    import oracle
    from attention_tcgen05_tmem_gb300 import flops, synth

    w = ws[-1]  # for TTT: the largest step (most keys per row)
    threads = oracle.num_threads()
    groups = min(w.Hkv, max(1, -(-threads // w.G)))
    hq = groups * w.G
    x = inputs or synth.make_inputs(w)
    q = x["q"][:, :hq].double().numpy()
    k = x["k"][:, :groups].double().numpy()
    v = x["v"][:, :groups].double().numpy()
    do = x["dout"][:, :hq].double().numpy()
    t = w.ttt_step
    lens = w.seq_lengths if w.seq_lengths is not None else (None,) * w.B
    kw = dict(window=w.window, seq_lengths=w.seq_lengths, add_mask=x.get("add_mask"))

    def pairs(r0):  # visible pairs of query rows [r0, Sq), one q head of every batch entry
        return sum(flops.visible_pairs_rows(w.mask, w.Sq, w.Skv, t, w.window, L, r0, w.Sq)
                   for L in lens)

    def run(R):
        r0 = w.Sq - R
        t0 = time.perf_counter()
        oracle.fwd(q, k, v, w.mask, t, rows=(r0, w.Sq), **kw)
        t1 = time.perf_counter()
        oracle.bwd(q, k, v, do, w.mask, t, rows=(r0, w.Sq), **kw)
        t2 = time.perf_counter()
        return t2 - t0, 14.0 * w.D * hq * pairs(r0), t1 - t0, t2 - t1

    if rows is not None:
        R = min(w.Sq, int(rows))
        dt, f, dtf, dtb = run(R)
    else:
        R = min(w.Sq, 8)
        dt, f, dtf, dtb = run(R)
        for _ in range(3):
            if dt >= 0.5 * target_s or R >= w.Sq:
                break
            R = int(min(w.Sq, max(2 * R, R * target_s / max(dt, 1e-3))))
            dt, f, dtf, dtb = run(R)
    desc = (f"fp64 oracle fwd+bwd on {w.name}: {w.B} batch x {hq} of {w.Hq} q heads "
            f"({groups} kv-head groups), last {R} of {w.Sq} query rows, {f / 1e9:.1f} GFLOP "
            f"mask-aware, {dt:.1f} s")
    per_pass = {"fwd": f * 4 / 14 / max(dtf, 1e-9) / 1e12, "bwd": f * 10 / 14 / max(dtb, 1e-9) / 1e12,
                "rows": R}
    return f / dt / 1e12, desc, threads, per_pass


# Seconds the reference arm (the CPU oracle) aims to spend over all its steps.
REF_BUDGET_S = 150.0


# --------------------------------------------------------------- GPU arm
def gpu_index_for(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [s.strip() for s in vis.split(",") if s.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


class Case:
    """Device buffers and the per-step launch sequence of one shape."""

    def __init__(self, w, dev, out, binding, synth):
        import torch
        self.w = w
        self.b = binding
        self.x = synth.make_inputs(w)
        self.q, self.k, self.v, self.do = (self.x[n].to(dev) for n in ("q", "k", "v", "dout"))
        # per-batch key lengths stay on the device for the whole run (the problem
        # holds their address)
        self.lens = self.x["seq_lengths"].to(dev) if "seq_lengths" in self.x else None
        self.add = self.x["add_mask"].to(dev) if "add_mask" in self.x else None
        odt = torch.float32 if out == "fp32" else torch.bfloat16
        self.p = binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, w.ttt_step, 0.0, out,
                                 w.window, self.lens, self.add)
        binding.check_supported(self.p)
        self.o = torch.empty(self.q.shape, dtype=odt, device=dev)
        self.lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device=dev)
        self.dq = torch.empty(self.q.shape, dtype=odt, device=dev)
        self.dk = torch.empty(self.k.shape, dtype=odt, device=dev)
        self.dv = torch.empty(self.v.shape, dtype=odt, device=dev)
        self.ws = torch.empty(binding.workspace_size(self.p), dtype=torch.uint8, device=dev)
        # the forward's key-range split (small grids) and its workspace
        nfw = binding.fwd_workspace_size(self.p)
        self.fws = torch.empty(nfw, dtype=torch.uint8, device=dev) if nfw else None
        has_ttt = w.mask == "ttt" and w.ttt_step > 0
        self.passes = [("bwd_prep", binding.BWD_PREP), ("bwd_dkdv", binding.BWD_DKDV),
                       ("bwd_dq", binding.BWD_DQ)]
        if has_ttt:
            self.passes.append(("ttt_diag_bwd", binding.BWD_TTT))
        self.names = ["fwd"] + [n for n, _ in self.passes]
        # kernels launched per step: a TTT forward adds its diagonal-scores pre-pass
        # when the t scores fit into an output row (t * 4 <= D * output element size)
        scores = has_ttt and w.ttt_step * 4 <= w.D * (4 if out == "fp32" else 2)
        self.launches = len(self.names) + (1 if scores else 0) + (1 if self.fws is not None else 0)

    def step(self, stream, evs=None, mark=None):
        """One forward + backward on `stream`; timing marks between the kernels:
        torch events (evs) or a callable mark(i) (events inside a CUDA graph)."""
        b = self.b
        if mark is None and evs:
            mark = lambda i: evs[i].record(stream)  # noqa: E731
        if mark:
            mark(0)
        b.fwd_ws_raw(self.p, self.q, self.k, self.v, self.o, self.lse, self.fws, stream.cuda_stream)
        if mark:
            mark(1)
        for i, (_, m) in enumerate(self.passes):
            b.bwd_passes_raw(self.p, m, self.q, self.k, self.v, self.o, self.do, self.lse, self.dq,
                             self.dk, self.dv, self.ws, stream.cuda_stream)
            if mark:
                mark(2 + i)


def cuda_runtime():
    """The CUDA runtime library the attention library loaded (so that events
    and streams are handled by the same runtime instance), via ctypes."""
    import ctypes
    path = None
    try:
        with open("/proc/self/maps") as f:
            for line in f:
                if "libcudart.so" in line:
                    path = line.split()[-1]
                    break
    except OSError:
        pass
    rt = ctypes.CDLL(path or "libcudart.so.13")
    vp = ctypes.c_void_p
    rt.cudaEventCreate.argtypes = [ctypes.POINTER(vp)]
    rt.cudaEventRecordWithFlags.argtypes = [vp, vp, ctypes.c_uint]
    rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), vp, vp]
    rt.cudaEventDestroy.argtypes = [vp]
    return rt


class GraphEvents:
    """Timing events stamped by every replay of a CUDA graph: event-record
    nodes captured with cudaEventRecordExternal, so per-kernel times exclude
    the host's launch gaps."""

    EXTERNAL = 0x1

    def __init__(self, rt, n):
        import ctypes
        self.rt, self.ev = rt, [ctypes.c_void_p() for _ in range(n)]
        for e in self.ev:
            self._check(rt.cudaEventCreate(ctypes.byref(e)), "cudaEventCreate")

    @staticmethod
    def _check(err, what):
        if err != 0:
            raise RuntimeError(f"{what} failed ({err})")

    def record(self, i, stream_handle):
        import ctypes
        self._check(self.rt.cudaEventRecordWithFlags(self.ev[i], ctypes.c_void_p(stream_handle),
                                                     self.EXTERNAL), "cudaEventRecordWithFlags")

    def elapsed_ms(self, i, j):
        import ctypes
        ms = ctypes.c_float()
        self._check(self.rt.cudaEventElapsedTime(ctypes.byref(ms), self.ev[i], self.ev[j]),
                    "cudaEventElapsedTime")
        return float(ms.value)

    def close(self):
        for e in self.ev:
            self.rt.cudaEventDestroy(e)
        self.ev = []


class Runner:
    """One workload on one GPU: device buffers, the timed device-only region
    (K steps of kernels with CUDA events between them) and the end-to-end
    region through the host-memory session.  Each region can be run several
    times; main() interleaves the repeats across workloads."""

    def __init__(self, args, ws, local_rank, dist):
        import torch

        from attention_tcgen05_tmem_gb300 import binding, synth
        from attention_tcgen05_tmem_gb300 import build as lib_build

        lib_build.build()
        self.args, self.ws, self.dist, self.local_rank = args, ws, dist, local_rank
        self.binding = binding
        self.dev = dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        self.stream = torch.cuda.current_stream(dev)
        self.cases = [Case(w, dev, args.out, binding, synth) for w in ws]
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > 129 MB L2
        self.hosts = None
        self.h2d = self.d2h = 0
        self.step_ms = None  # device-only time per step, once timed
        self.e2e_slots = self.e2e_count = None
        self.launches_per_step = sum(c.launches for c in self.cases)
        for _ in range(max(args.warmup, 3)):
            for c in self.cases:
                c.step(self.stream)
        torch.cuda.synchronize(dev)
        binding.device_status()
        self.graph, self.gevs, self.timing = None, None, "eager, CUDA events between kernels"
        if not args.eager:
            self._capture()

    def _capture(self):
        """The step as one CUDA graph, with timing events recorded inside it (small
        problems are otherwise timed with the host's launch gaps between kernels)."""
        import torch
        try:
            rt = cuda_runtime()
            self.gevs = [GraphEvents(rt, len(c.names) + 1) for c in self.cases]
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream(self.dev)
            s.wait_stream(self.stream)
            with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
                for c, gev in zip(self.cases, self.gevs):
                    c.step(s, mark=lambda i, gev=gev: gev.record(i, s.cuda_stream))
            for _ in range(2):
                g.replay()
            torch.cuda.synchronize(self.dev)
            self.binding.device_status()
            self.graph = g
            self.timing = "CUDA graph replay per step, events recorded inside the graph"
        except Exception as ex:  # noqa: BLE001 -- eager timing remains valid
            for gev in self.gevs or []:
                gev.close()
            self.graph, self.gevs = None, None
            self.timing = f"eager, CUDA events between kernels (graph capture failed: {ex!r})"[:200]

    def timed(self):
        """K steps, L2 flushed between steps outside the events; returns the
        summed event time of the steps, per-kernel sums and the clocks seen."""
        import torch
        K, dev, dist = self.args.steps, self.dev, self.dist
        per_kernel, total_ms = {}, 0.0
        if self.graph is not None:
            if dist:
                dist.barrier()
            torch.cuda.synchronize(dev)
            with ClockSampler(gpu_index_for(self.local_rank)) as clk:
                for i in range(K):
                    self.flush.zero_()  # evict L2 between steps (outside the events)
                    self.graph.replay()
                    torch.cuda.synchronize(dev)
                    for c, gev in zip(self.cases, self.gevs):
                        total_ms += gev.elapsed_ms(0, len(c.names))
                        for j, n in enumerate(c.names):
                            per_kernel[n] = per_kernel.get(n, 0.0) + gev.elapsed_ms(j, j + 1)
            if dist:
                dist.barrier()
            self.binding.device_status()
            total_ms, = max_over_ranks([total_ms], dist, dev)
            self.step_ms = total_ms / K
            return {"total_ms": total_ms, "per_kernel_ms": per_kernel, "clocks": clk.summary()}
        evsets = [[[torch.cuda.Event(enable_timing=True) for _ in range(len(c.names) + 1)]
                   for c in self.cases] for _ in range(K)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(gpu_index_for(self.local_rank)) as clk:
            for i in range(K):
                self.flush.zero_()  # evict L2 between steps (outside the events)
                for c, evs in zip(self.cases, evsets[i]):
                    c.step(self.stream, evs)
            torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        self.binding.device_status()
        for i in range(K):
            for c, evs in zip(self.cases, evsets[i]):
                total_ms += evs[0].elapsed_time(evs[-1])
                for j, n in enumerate(c.names):
                    per_kernel[n] = per_kernel.get(n, 0.0) + evs[j].elapsed_time(evs[j + 1])
        total_ms, = max_over_ranks([total_ms], dist, dev)
        self.step_ms = total_ms / K
        return {"total_ms": total_ms, "per_kernel_ms": per_kernel, "clocks": clk.summary()}

    def _pick_slots(self, hps):
        import torch
        b, args = self.binding, self.args
        free, _ = torch.cuda.mem_get_info(self.dev)
        return e2e_slots(args.e2e_slots, self.step_ms,
                         lambda n: sum(b.step_host_arena_size(hp, args.e2e_chunk, n) for hp in hps),
                         free, b.HOST_MAX_SLOTS)

    def _open_sessions(self):
        # end to end through the C ABI's host-memory session (attn_train_host_session_*):
        # every step copies q, k, v, dO (and key lengths / mask) in from pinned host
        # buffers and O, LSE, dQ, dK, dV out; the copies overlap the kernels of the
        # same and the neighbouring steps, and the timed region ends after the last
        # step's copies (join + synchronize)
        import torch
        b, args = self.binding, self.args
        self.hosts = []
        staged = []
        for c in self.cases:
            w = c.w
            pin = {n: c.x[n].pin_memory()
                   for n in ("q", "k", "v", "dout", "seq_lengths", "add_mask") if n in c.x}
            outs = {n: torch.empty(getattr(c, n).shape, dtype=getattr(c, n).dtype).pin_memory()
                    for n in ("o", "lse", "dq", "dk", "dv")}
            hp = b.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, w.ttt_step, 0.0, args.out,
                           w.window, pin.get("seq_lengths"), pin.get("add_mask"), host=True)
            io = {"q": pin["q"], "k": pin["k"], "v": pin["v"], "dout": pin["dout"], **outs}
            staged.append((hp, io, pin))
            self.h2d += sum(t.numel() * t.element_size() for t in pin.values())
            self.d2h += sum(t.numel() * t.element_size() for t in outs.values())
        self.e2e_slots = n = self._pick_slots([hp for hp, _, _ in staged])
        for hp, io, pin in staged:
            arena = torch.empty(b.step_host_arena_size(hp, args.e2e_chunk, n), dtype=torch.uint8,
                                device=self.dev)
            self.hosts.append((b.HostSession(hp, arena, args.e2e_chunk, n), io, pin))
        self.e2e_count = e2e_steps(args.e2e_seconds, self.step_ms)
        self._e2e_steps(2)  # first use of the sessions

    def _e2e_steps(self, n):
        for _ in range(n):
            for sess, io, _ in self.hosts:
                sess.step(io, self.stream.cuda_stream)
        for sess, _, _ in self.hosts:
            sess.join(self.stream.cuda_stream)

    def e2e(self):
        """Milliseconds for K end-to-end steps (e2e_count steps run, about a
        second, scaled to K) and the clocks sampled meanwhile.  The sampler
        starts first and the warm-up steps (one per slot) run right before the
        timed ones: the first copies after an idle host link are slow, and the
        link pauses about twice a second under load, so the region neither
        starts cold nor is short enough to miss or catch a pause by chance."""
        import torch
        if self.hosts is None:
            self._open_sessions()
        dev, dist, K = self.dev, self.dist, self.args.steps
        Ke = self.e2e_count
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        with ClockSampler(gpu_index_for(self.local_rank)) as clk:
            self._e2e_steps(max(3, self.e2e_slots))  # warm-up (outside the events)
            torch.cuda.synchronize(dev)
            if dist:
                dist.barrier()
            e0.record(self.stream)
            self._e2e_steps(Ke)
            e1.record(self.stream)
            torch.cuda.synchronize(dev)
        self.binding.device_status()
        ms, = max_over_ranks([e0.elapsed_time(e1) / Ke * K], dist, dev)
        return {"ms": ms, "clocks": clk.summary()}

    def close(self):
        for sess, _, _ in self.hosts or []:
            sess.close()
        self.hosts = None
        for gev in self.gevs or []:
            gev.close()
        self.graph, self.gevs = None, None


def e2e_slots(requested, step_ms, arena_bytes, free_bytes, max_slots):
    """Device slots of the end-to-end sessions: `requested` (clamped to 2 ..
    max_slots) if given, else enough for E2E_RIDE_MS of compute at the measured
    device step time (8 ms if not yet timed), reduced until the arenas
    (arena_bytes(n) for n slots) take at most a quarter of the free memory."""
    import math
    if requested:
        return min(max_slots, max(2, requested))
    est = step_ms or 8.0
    n = min(max_slots, max(2, math.ceil(E2E_RIDE_MS / est) + 1))
    while n > 2 and arena_bytes(n) > free_bytes / 4:
        n -= 1
    return n


def e2e_steps(seconds, step_ms):
    """Timed end-to-end steps: about `seconds` of device time (3 to 1000)."""
    import math
    return max(3, min(1000, math.ceil(seconds * 1e3 / (step_ms or 8.0))))


def median_run(runs):
    """The repeat with the median total time (its per-kernel times and clocks
    go with it)."""
    order = sorted(range(len(runs)), key=lambda i: runs[i]["total_ms"])
    return runs[order[(len(order) - 1) // 2]]


def max_over_ranks(values, dist, device="cpu"):
    """Element-wise max of per-rank timings (the slowest replica sets the
    time of the whole job)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_value(flops_per_step, steps, total_ms, n_gpus):
    """Whole-job throughput in TFLOP/s: every replica does flops_per_step per
    step, the job takes the slowest replica's time."""
    return n_gpus * flops_per_step * steps / (total_ms * 1e-3) / 1e12


def kernel_flops(ws, name):
    """Algorithmic FLOPs of one step of each kernel: the tensor-core work it
    must do on exactly the visible pairs it owns (2*D per pair and GEMM):
    forward 2 GEMMs; dK/dV 4 (S^T recompute, dP^T, dV, dK) on the tiled part;
    dQ 3 (S recompute, dP, dQ); the TTT suffix pass 4 on the diagonal pairs."""
    from attention_tcgen05_tmem_gb300 import flops
    tot = 0
    for w in ws:
        nvis = flops.visible_pairs(w)
        ndiag = flops.diagonal_pairs(w)
        per = {"fwd": 4 * nvis, "bwd_dkdv": 8 * (nvis - ndiag), "bwd_dq": 6 * nvis,
               "ttt_diag_bwd": 8 * ndiag, "bwd_prep": 0}[name]
        tot += per * w.D
    return tot


def prep_bytes(ws, out_bytes):
    return sum(w.B * w.Hq * w.Sq * (w.D * (out_bytes + 2) + 4) for w in ws)


# Host-only sources that no timed kernel runs (the host-memory step's copy
# orchestration): a change there leaves the kernels' DRAM traffic as it was.
HOST_ONLY_SOURCES = ("host_step.cu",)


def kernel_source_sha() -> str:
    """sha256 over the CUDA sources of the kernels and their launches: a capture
    taken on other sources is stale."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_tcgen05_tmem_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")) and name not in HOST_ONLY_SOURCES:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def load_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the
    committed ncu summary (profiles/traffic.json); None when there is no
    capture or it was taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    ent = t.get(workload, {}).get(kernel)
    if not ent or ent.get("src_sha") != kernel_source_sha():
        return None
    return ent.get("bytes")


# Dense bf16 tensor rate of one SM: 4096 multiply-adds per clock (a 128 x 256 x 16
# tcgen05 MMA every 128 cycles).
BF16_FLOP_PER_CLK_SM = 8192


def theoretical_peak(value_per_gpu, clocks, device):
    """Fraction of SMs x max SM clock x the per-SM dense bf16 rate, with the
    figures it is made of; empty when the max clock was not sampled."""
    import torch
    mhz = (clocks or {}).get("sm_max_mhz")
    if not mhz:
        return {}
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    peak = sms * mhz * 1e6 * BF16_FLOP_PER_CLK_SM / 1e12
    return {"theoretical": value_per_gpu / peak, "theoretical_tflops": peak,
            "theoretical_basis": f"{sms} SMs x {mhz:.0f} MHz x {BF16_FLOP_PER_CLK_SM} FLOP/clk"}


def clock_peak_tflops(clocks, device):
    """SMs x the median SM clock sampled under load x the per-SM dense bf16
    rate: the tensor peak at the clock the kernels actually ran at."""
    import torch
    mhz = (clocks or {}).get("sm_mhz")
    if not mhz:
        return None
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    return sms * mhz * 1e6 * BF16_FLOP_PER_CLK_SM / 1e12


def merge_clocks(samples):
    """Clock records of several timed regions as one: the median of their
    median SM clocks, the highest max clock and power, every throttle reason
    seen in any of them."""
    got = [c for c in samples if c.get("sm_mhz") is not None]
    if not got:
        return samples[0] if samples else {"sm_mhz": None, "reasons": ["unsampled"], "samples": 0}
    pw = [c["power_w_max"] for c in got if c.get("power_w_max") is not None]
    return {"sm_mhz": statistics.median(c["sm_mhz"] for c in got),
            "sm_max_mhz": max(c["sm_max_mhz"] for c in got),
            "reasons": sorted(set().union(*(c["reasons"] for c in got))),
            "power_w_max": max(pw) if pw else None,
            "samples": sum(c["samples"] for c in got)}


def kernel_plan(runner):
    """The kernels, tiles, grids and pipeline depths the library uses for each
    problem of the workload (attn_train_describe on the timed problems)."""
    plans = [runner.binding.describe(c.p) for c in runner.cases]
    return plans[0] if len(plans) == 1 else plans


def run_env(device):
    """GPU, driver, runtime and host the line was measured on."""
    import platform

    import torch
    env = {"torch": torch.__version__, "cuda_runtime": torch.version.cuda,
           "host_cores": os.cpu_count(), "host_arch": platform.machine()}
    try:
        prop = torch.cuda.get_device_properties(device)
        env.update({"gpu": prop.name, "sms": prop.multi_processor_count,
                    "gpu_mem_gib": round(prop.total_memory / 2**30, 1)})
    except Exception:  # noqa: BLE001 -- descriptive only
        pass
    try:
        r = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                            "-i", gpu_index_for(device)], capture_output=True, text=True,
                           timeout=20)
        if r.returncode == 0 and r.stdout.strip():
            env["driver"] = r.stdout.strip().splitlines()[0]
    except (OSError, subprocess.SubprocessError):
        pass
    try:  # lscpu names Arm cores ("Neoverse-V2"); /proc/cpuinfo gives only a part number there
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20)
        for ln in r.stdout.splitlines():
            if ln.lower().startswith("model name:"):
                env["host_cpu"] = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if "host_cpu" not in env:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    key = ln.split(":")[0].strip().lower()
                    if key in ("model name", "cpu model", "cpu part"):
                        env["host_cpu"] = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return env


def describe(name, ws, out, n_gpus):
    cfg = dict(ws[0].describe()) if len(ws) == 1 else {
        "workload": name, "B": ws[0].B, "Hq": ws[0].Hq, "Hkv": ws[0].Hkv, "Sq": ws[0].Sq,
        "Skv": [w.Skv for w in ws], "D": ws[0].D, "mask": ws[0].mask,
        "ttt_steps": [w.ttt_step for w in ws]}
    cfg["workload"] = name
    cfg.update({"outputs": out, "l2": "flushed between steps (256 MiB write)",
                "parallelism": f"replicas x{n_gpus}"})
    return cfg


# ------------------------------------------- soft-target log-softmax loss
LOSS_METRIC = "soft-target log-softmax loss fwd+bwd HBM throughput (algorithmic bytes)"


def loss_table():
    from attention_tcgen05_tmem_gb300 import synth
    return {w.name: w for w in synth.LOSS}


def loss_bytes(w):
    """Algorithmic HBM bytes of one forward + in-place backward over [rows, V]
    fp32: the forward reads logits and target and writes 3 row statistics; the
    backward reads logits, target and the statistics and writes the gradient;
    the mask is read by both."""
    n, V = w.rows, w.V
    return n * V * 4 * 2 + n * (4 + 12) + n * V * 4 * 3 + n * (4 + 8)


def loss_cpu_sample(w, x, target_s, rows=None):
    """The fp64 oracle on the first R rows (R grown to about target_s s, or
    rows=R fixed); returns (GB/s of the same algorithmic bytes per row,
    description, R)."""
    from oracle import softmax_loss as sl
    N, V = w.rows, w.V
    lg = x["logits"].reshape(N, V)
    tg = x["target"].reshape(N, V)
    mk = x["mask"].reshape(N)
    R = 8 if rows is None else min(N, int(rows))
    while True:
        t0 = time.perf_counter()
        sl.forward(lg[:R], tg[:R], mk[:R])
        sl.backward(lg[:R], tg[:R], mk[:R])
        dt = time.perf_counter() - t0
        if rows is not None or dt >= 0.5 * target_s or R >= N:
            break
        R = int(min(N, max(2 * R, R * target_s / max(dt, 1e-3))))
    gbs = loss_bytes(w) * R / N / dt / 1e9
    return gbs, f"fp64 oracle fwd+bwd on the first {R} of {N} rows of {w.name}, {dt:.1f} s", R


def run_loss(args, w, rank, local_rank, dist, n_gpus, peaks, peak_src):
    import torch

    from attention_tcgen05_tmem_gb300 import binding, synth
    from attention_tcgen05_tmem_gb300 import build as lib_build

    lib_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    x = synth.make_loss_inputs(w)
    pristine = x["logits"].to(dev)
    logits = torch.empty_like(pristine)
    target = x["target"].to(dev)
    mask = x["mask"].reshape(-1).to(dev)
    N = w.rows
    f = dict(dtype=torch.float32, device=dev)
    row_loss, row_lse, row_tsum, loss = (torch.empty(n, **f) for n in (N, N, N, 1))
    one = torch.ones(1, **f)

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        binding.logsoftmax_loss_fwd_raw(logits, target, mask, row_loss, row_lse, row_tsum, loss,
                                        stream.cuda_stream)
        if evs:
            evs[1].record(stream)
        binding.logsoftmax_loss_bwd_raw(logits, target, mask, row_lse, row_tsum, one,
                                        stream.cuda_stream)
        if evs:
            evs[2].record(stream)

    for _ in range(max(args.warmup, 3)):
        logits.copy_(pristine)
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_index_for(local_rank)) as clk:
        for i in range(K):
            logits.copy_(pristine)  # the backward overwrote the logits (outside the events)
            step(evsets[i])
        torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in evsets) / K
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in evsets) / K
    total_ms, = max_over_ranks([(fwd_ms + bwd_ms) * K], dist, dev)
    per = total_ms / K
    B = loss_bytes(w)
    value = n_gpus * B / (per * 1e-3) / 1e9
    peak_hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    fwd_bytes = N * w.V * 8 + N * 16
    bwd_bytes = B - fwd_bytes
    dom, dom_ms, dom_bytes = ("bwd", bwd_ms, bwd_bytes) if bwd_ms >= fwd_ms else ("fwd", fwd_ms, fwd_bytes)
    ach = dom_bytes / (dom_ms * 1e-3) / 1e9
    line = {
        "metric": LOSS_METRIC, "value": value, "unit": "GB/s", "n_gpus": n_gpus, "steps": K,
        "warmup": args.warmup, "ms_per_step": per, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(w.describe(), **{"l2": "inputs larger than L2 (no flush needed)",
                                        "parallelism": f"replicas x{n_gpus}"}),
        "kernel_ms": {"logsoftmax_loss_fwd": fwd_ms, "logsoftmax_loss_bwd": bwd_ms},
        "roofline": {"bound": "hbm", "kernel": f"logsoftmax_loss_{dom}", "achieved": ach,
                     "peak": peak_hbm, "unit": "GB/s", "frac": ach / peak_hbm, "traffic": None,
                     "peak_kind": f"HBM copy, of {peak_src}"},
        "gpu_launches": 3 * K,
        "clocks": clk.summary(),
    }
    if not args.no_e2e:
        pin = {n: x[n].pin_memory() for n in ("logits", "target", "mask")}
        out_grad = torch.empty(x["logits"].shape, dtype=torch.float32).pin_memory()
        out_loss = torch.empty(1, dtype=torch.float32).pin_memory()

        def e2e_step():
            logits.copy_(pin["logits"].reshape(logits.shape), non_blocking=True)
            target.copy_(pin["target"].reshape(target.shape), non_blocking=True)
            mask.copy_(pin["mask"].reshape(-1), non_blocking=True)
            step()
            out_loss.copy_(loss, non_blocking=True)
            out_grad.copy_(logits.reshape(out_grad.shape), non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        Ke = max(3, min(K, 10))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Ke):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms, = max_over_ranks([e0.elapsed_time(e1) / Ke], dist, dev)
        line["e2e"] = {"value": n_gpus * B / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                       "h2d_bytes_per_step": sum(t.numel() * 4 for t in pin.values()),
                       "d2h_bytes_per_step": out_grad.numel() * 4 + 4}
    if rank == 0 and n_gpus == 1 and not args.no_cpu_baseline:
        gbs, desc, _ = loss_cpu_sample(w, x, args.cpu_seconds)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    from attention_tcgen05_tmem_gb300 import flops
    table = bench_workloads()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    n_gpus = max(world, 1)
    names = headline_names() if args.all else [args.workload]
    losses = loss_table()
    loss_names = [n for n in names if n in losses]
    if args.all:
        loss_names = list(losses)
    names = [n for n in names if n not in losses]

    if args.impl == "reference":
        if rank != 0:
            return 0
        # the whole reference run stays near REF_BUDGET_S seconds: each step times the
        # oracle on a sample sized once per workload (calibrated outside the steps)
        n_lines = max(1, len(loss_names) + len(names))
        step_s = max(0.2, min(4.0, REF_BUDGET_S / n_lines / (args.warmup + args.steps)))
        for name in loss_names:
            from attention_tcgen05_tmem_gb300 import synth
            w = losses[name]
            x = synth.make_loss_inputs(w)
            per, desc = [], ""
            _, _, R = loss_cpu_sample(w, x, step_s)
            for i in range(args.warmup + args.steps):
                gbs, desc, _ = loss_cpu_sample(w, x, step_s, rows=R)
                if i >= args.warmup:
                    per.append(gbs)
            value = statistics.median(per)
            line = {"impl": "reference", "metric": LOSS_METRIC, "value": value, "unit": "GB/s",
                    "n_gpus": n_gpus, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": loss_bytes(w) / (value * 1e9) * 1e3, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                    "config": w.describe(),
                    "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                     "sample": desc},
                    "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        for name in names:
            ws = table[name]
            F = sum(flops.flops_fwd_bwd(w) for w in ws)
            per, per_f, per_b, desc, threads = [], [], [], "", 1
            from attention_tcgen05_tmem_gb300 import synth
            x = synth.make_inputs(ws[-1])
            R = cpu_sample(ws, step_s, x)[3]["rows"]
            for i in range(args.warmup + args.steps):
                tf, desc, threads, pp = cpu_sample(ws, step_s, x, rows=R)
                if i >= args.warmup:
                    per.append(tf)
                    per_f.append(pp["fwd"])
                    per_b.append(pp["bwd"])
            value = statistics.median(per)
            line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
                    "n_gpus": n_gpus, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": F / (value * 1e12) * 1e3, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                    "config": describe(name, ws, args.out, n_gpus),
                    "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads,
                                     "kind": "oracle", "sample": desc,
                                     "fwd_value": statistics.median(per_f),
                                     "bwd_value": statistics.median(per_b)},
                    "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        return 0

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
        dist = tdist
    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    for name in loss_names:
        run_loss(args, losses[name], rank, local_rank, dist, n_gpus, peaks, peak_src)
    # every timed region runs args.repeats times, the repeats interleaved across
    # workloads (arm drift between invocations shows as spread, not as bias)
    runners = {name: Runner(args, table[name], local_rank, dist) for name in names}
    runs = {name: [] for name in names}
    e2es = {name: [] for name in names}
    for _ in range(args.repeats):
        for name in names:
            runs[name].append(runners[name].timed())
    if not args.no_e2e:
        for _ in range(args.repeats):
            for name in names:
                e2es[name].append(runners[name].e2e())
    plans = {name: kernel_plan(runners[name]) for name in names}
    for name in names:
        runners[name].close()
    env = run_env(local_rank)
    for name in names:
        ws = table[name]
        F = sum(flops.flops_fwd_bwd(w) for w in ws)
        K = args.steps
        r = median_run(runs[name])
        clocks = merge_clocks([x["clocks"] for x in runs[name]])
        value = job_value(F, K, r["total_ms"], n_gpus)
        pk = r["per_kernel_ms"]
        dom = max(pk, key=lambda n: pk[n])
        dom_ms = pk[dom] / K
        if dom == "bwd_prep":
            ach = prep_bytes(ws, 4 if args.out == "fp32" else 2) / (dom_ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peak_hbm,
                    "unit": "GB/s", "frac": ach / peak_hbm, "traffic": None,
                    "peak_kind": f"HBM copy, of {peak_src}"}
        else:
            # the kernel is timed per launch (milliseconds) inside a short timed region,
            # so the burst figure is its peak; the sustained one is given beside it,
            # and frac_clock compares with SMs x the sampled SM clock x the dense rate
            ach = kernel_flops(ws, dom) / (dom_ms * 1e-3) / 1e12
            roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak_burst,
                    "unit": "TFLOP/s", "frac": ach / peak_burst, "traffic": None,
                    "peak_kind": f"bf16 burst, of {peak_src}",
                    "peak_sustained": peak_sus, "frac_sustained": ach / peak_sus}
            clk_peak = clock_peak_tflops(clocks, local_rank)
            if clk_peak:
                roof["frac_clock"] = ach / clk_peak
                roof["clock_peak"] = clk_peak
        traffic = load_traffic(name, dom)
        if traffic is not None:
            roof["traffic"] = traffic
        alg_bytes = sum(flops.bytes_fwd(w) + flops.bytes_bwd(w) for w in ws)
        totals = sorted(x["total_ms"] / K for x in runs[name])
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": n_gpus, "steps": K,
            "warmup": args.warmup, "ms_per_step": r["total_ms"] / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(describe(name, ws, args.out, n_gpus), timing=runners[name].timing),
            "pct_of_peak": {"bf16_burst": value / n_gpus / peak_burst,
                            "bf16_sustained": value / n_gpus / peak_sus, "source": peak_src,
                            **theoretical_peak(value / n_gpus, clocks, local_rank)},
            "fwd_tflops": sum(flops.flops_fwd(w) for w in ws) / (pk["fwd"] / K * 1e-3) / 1e12,
            "bwd_tflops": sum(flops.flops_bwd(w) for w in ws) /
                          (sum(v for n, v in pk.items() if n != "fwd") / K * 1e-3) / 1e12,
            "hbm_gbs_algorithmic": alg_bytes / (r["total_ms"] / K * 1e-3) / 1e9,
            "kernel_ms": {n: v / K for n, v in pk.items()},
            "roofline": roof,
            "kernels": plans[name],
            "env": env,
            "gpu_launches": runners[name].launches_per_step * K,
            "clocks": clocks,
            "repeats": {"n": len(totals), "steps_each": K,
                        "ms_per_step": {"median": r["total_ms"] / K, "min": totals[0],
                                        "max": totals[-1]}},
        }
        if e2es[name]:
            e = sorted(x["ms"] for x in e2es[name])
            e_med = e[(len(e) - 1) // 2]
            line["e2e"] = {"value": job_value(F, K, e_med, n_gpus), "unit": UNIT,
                           "h2d_bytes_per_step": runners[name].h2d,
                           "d2h_bytes_per_step": runners[name].d2h,
                           "steps_timed": runners[name].e2e_count,
                           "slots": runners[name].e2e_slots}
            line["repeats"]["e2e_ms_per_step"] = {"median": e_med / K, "min": e[0] / K,
                                                  "max": e[-1] / K}
            line["e2e_clocks"] = merge_clocks([x["clocks"] for x in e2es[name]])
        if rank == 0 and n_gpus == 1 and not args.no_cpu_baseline:
            tf, desc, threads, pp = cpu_sample(ws, args.cpu_seconds)
            line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": threads, "kind": "oracle",
                                    "sample": desc, "fwd_value": pp["fwd"], "bwd_value": pp["bwd"]}
        if rank == 0:
            print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
