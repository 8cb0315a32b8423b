"""One-tile checks of the hand-built tcgen05 descriptors against a CPU
matmul: the shared-memory K-major and MN-major layouts written by TMA with
hardware swizzle, the instruction descriptor, and the A operand read from
tensor memory.  Every kernel in the library uses exactly these forms."""
import pytest
import torch

from attention_tcgen05_tmem_gb300 import binding
from tests.gpu_util import device


@pytest.mark.gpu
@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_probe_ss_kmajor(D):
    dev = device()
    g = torch.Generator().manual_seed(D)
    a = torch.randn(128, D, generator=g).to(torch.bfloat16)
    b = torch.randn(128, D, generator=g).to(torch.bfloat16)
    c = binding.probe_mma(0, a.to(dev), b.to(dev), D)
    binding.device_status()
    ref = a.float() @ b.float().T
    err = (c.cpu() - ref).abs().max().item()
    assert err < 1e-3 * max(1.0, ref.abs().max().item()), err


@pytest.mark.gpu
@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_probe_ts_mnmajor(D):
    dev = device()
    g = torch.Generator().manual_seed(100 + D)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    b = torch.randn(128, D, generator=g).to(torch.bfloat16)
    c = binding.probe_mma(1, a.to(dev), b.to(dev), D)
    binding.device_status()
    ref = a.float() @ b.float()
    err = (c.cpu() - ref).abs().max().item()
    assert err < 1e-3 * max(1.0, ref.abs().max().item()), err
