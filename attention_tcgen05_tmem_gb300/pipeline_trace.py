"""Pipeline timeline of the tensor-core kernels (profiling tool).

Builds the library with -DATTN_TRACE (libattn_train_trace.so), runs each
tensor-core kernel of one workload on its own, reads the per-role SM-cycle
stamps the trace build records for the first CTAs of the launch, and prints
one JSON line per kernel: the mean cycles between consecutive probes of each
role (0 producer, 1 MMA issuer, 2 and 3 the elementwise warpgroups) and the
iteration period.  Probe numbering is the one in the kernels' ATTN_TR calls.

    python -m attention_tcgen05_tmem_gb300.pipeline_trace [--workload NAME]
"""
from __future__ import annotations

import argparse
import ctypes
import json

import numpy as np

C, R, E, I = 4, 4, 8, 64  # CTAs, roles, events, iterations (csrc/trace.cuh)


def main() -> int:
    import torch

    from . import binding, synth
    from . import build as lib_build

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=synth.LONG_GQA.name)
    args = ap.parse_args()
    w = synth.by_name(args.workload)
    path = lib_build.build_trace()
    binding._lib = None
    binding.load(path)
    raw = ctypes.CDLL(path)
    dev = torch.device("cuda:0")
    x = synth.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    p = binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, w.ttt_step, 0.0, "fp32")
    f32 = torch.float32
    o = torch.empty(q.shape, dtype=f32, device=dev)
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=f32, device=dev)
    dq = torch.empty(q.shape, dtype=f32, device=dev)
    dk = torch.empty(k.shape, dtype=f32, device=dev)
    dv = torch.empty(v.shape, dtype=f32, device=dev)
    ws = torch.empty(binding.workspace_size(p), dtype=torch.uint8, device=dev)
    binding.fwd_raw(p, q, k, v, o, lse)
    binding.bwd_passes_raw(p, binding.BWD_PREP, q, k, v, o, do, lse, dq, dk, dv, ws)
    torch.cuda.synchronize()
    kernels = {"fwd": ("attn_trace_read_fwd", None), "bwd_dkdv": ("attn_trace_read_bwd", 2),
               "bwd_dq": ("attn_trace_read_bwd", 4)}
    for kern, (reader, mask) in kernels.items():
        getattr(raw, reader + "_clear")()
        for _ in range(2):
            if mask is None:
                binding.fwd_raw(p, q, k, v, o, lse)
            else:
                binding.bwd_passes_raw(p, mask, q, k, v, o, do, lse, dq, dk, dv, ws)
        torch.cuda.synchronize()
        binding.device_status()
        buf = np.zeros((C, R, E, I), dtype=np.uint64)
        getattr(raw, reader)(buf.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(buf.nbytes))
        out = {"workload": w.name, "kernel": kern}
        for role in range(R):
            tr = buf[:, role].astype(np.float64)
            used = [e for e in range(E) if (tr[:, e, :] > 0).any()]
            if not used:
                continue
            d = {}
            for a_, b_ in zip(used, used[1:]):
                m = (tr[:, a_, :] > 0) & (tr[:, b_, :] > 0)
                d[f"{a_}->{b_}"] = round(float((tr[:, b_, :] - tr[:, a_, :])[m].mean()), 1)
            per = [np.diff(s[s > 0]).mean() for s in tr[:, used[0], :] if (s > 0).sum() > 1]
            d["period"] = round(float(np.mean(per)), 1) if per else None
            out[f"role{role}"] = d
        print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
