"""The tensor-memory scale layout of the block-scaled FP4 MMA that the W4A4 kernels write
their scales in (tcgen05.mma kind::mxf4nvf4, scale_vec::4X, M = N = 128): A's scale of row m
sits in lane m, column m / 32; B's scale of column n in lane 32 q + n % 32 of every lane
quadrant q, column n / 32; the byte is the 16-element block within the 64-element K step.
A standalone probe (gpu_probes/mxf4_scale_layout.cu) decodes every (row, column, block) of 32
single MMAs and reports any position that differs."""
import os
import shutil
import subprocess
import tempfile

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_mxf4nvf4_scale_factor_layout():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "probe")
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-o", exe,
                               os.path.join(HERE, "gpu_probes", "mxf4_scale_layout.cu")])
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "LAYOUT OK" in r.stdout, r.stdout
