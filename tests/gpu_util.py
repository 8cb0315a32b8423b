"""Helpers shared by the GPU tests: device setup and the parity bar.

The bar is the one the library is held to: for bf16 O, dQ, dK, dV the max
absolute error <= 2e-2 and the relative L2 error <= 1e-2 against the fp64
oracle on the same bf16-rounded inputs; LSE within 1e-3 absolute.
"""
import numpy as np
import torch

ATOL = 2e-2
REL_L2 = 1e-2
LSE_ATOL = 1e-3


def device():
    from attention_tcgen05_tmem_gb300 import build as lib_build
    lib_build.build()
    return torch.device("cuda:0")


def compare(name, got, ref, atol=ATOL, rel_l2=REL_L2):
    g = got.detach().double().cpu().numpy() if hasattr(got, "detach") else np.asarray(got)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite output"
    err = np.abs(g - r).max() if g.size else 0.0
    den = np.linalg.norm(r.ravel())
    rel = np.linalg.norm((g - r).ravel()) / den if den > 0 else np.linalg.norm(g.ravel())
    assert err <= atol and rel <= rel_l2, f"{name}: max abs {err:.3e} (bar {atol}), rel L2 {rel:.3e} (bar {rel_l2})"
    return err, rel
