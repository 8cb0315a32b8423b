"""The profiling tools stay buildable: the tensor-pipe microbenchmark
(mma_rate.cu, a standalone sm_103a program that includes the kernels' PTX and
tile-descriptor headers) compiles with the same toolchain as the library."""
import os
import shutil

import pytest

from attention_tcgen05_tmem_gb300 import build as lib_build
from attention_tcgen05_tmem_gb300 import mma_rate


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc not available")
def test_mma_rate_compiles():
    exe = mma_rate.build()
    assert os.path.isfile(exe) and os.access(exe, os.X_OK)
    assert os.path.dirname(exe) == lib_build.BUILD_DIR
