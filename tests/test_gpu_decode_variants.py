"""Parity of the alternative decode kernels, which a process selects with the
environment variable FTMOE_DECODE: "stream" (TMA-streamed register MMAs, separate
combine) or "tc" (tensor-core MMAs with the dequantised operand in tensor memory,
separate combine); the lean register-fed kernels are the default. Each case runs in a
child process so that the selection takes effect."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r"""
import sys
sys.path[:0] = [{root!r}, {here!r}]
import numpy as np, torch
import oracle, synth
import nvfp4_quantized_moe_gb300 as ft
from nvfp4_quantized_moe_gb300 import build
build.build(); ft.load()
from moe_cases import GpuLayer, assert_close, logits_for, oracle_banks
name, T, tp, want = {name!r}, {T}, {tp}, {want}
shape = synth.SHAPES[name]
for r in range(tp):
    L = GpuLayer(name, r, tp)
    logits = logits_for(name, T, name == "dsv4")
    x = synth.make_activations(T, shape.hidden)
    ids, w = L.route(logits)
    n0 = ft.ft_moe_launch_count()
    out, _ = L.forward(x, ids, w)
    launches = ft.ft_moe_launch_count() - n0
    assert launches == want, f"expected {{want}} launches, saw {{launches}}"
    ref_ids, ref_w = oracle.route(logits, shape.top_k)
    rb, sb = oracle_banks(name, r, tp)
    ref = oracle.moe_forward(rb, sb, shape.group, x, ref_ids, ref_w, nthreads=oracle.default_threads())
    rel, mx = assert_close(out.cpu().numpy(), ref, f"{{name}} T={{T}} tp={{tp}} rank={{r}}")
    print("ok", name, T, tp, r, rel, mx)
"""


@pytest.mark.parametrize("name,T,tp", [("qwen36", 1, 1), ("qwen36", 64, 1), ("qwen36", 32, 2), ("dsv4", 16, 1),
                                       ("dsv4", 16, 4)])
@pytest.mark.parametrize("mode,launches", [("stream", 4), ("tc", 4)])
def test_decode_variant_matches_oracle(mode, launches, name, T, tp):
    """Both: align, gate_up, down and a separate combine."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    env = dict(os.environ, FTMOE_DECODE=mode)
    code = CHILD.format(root=ROOT, here=HERE, name=name, T=T, tp=tp, want=launches)
    r = subprocess.run([sys.executable, "-c", code], env=env,
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert r.stdout.count("ok ") == tp
