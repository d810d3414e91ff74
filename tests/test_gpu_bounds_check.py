"""The bounds-checking build (FTMOE_BOUNDS_CHECK: every index the kernels derive from the
routing tables -- expert ids, sorted slots, padded position counts -- is checked before it
addresses memory, a bad one reported as FT_ERR_BOUNDS) on valid inputs: no false alarm
(status 0) and results bitwise equal to the regular build, on every regime (fused and
separate decode, tensor-core prefill, fp8_block, W4A4). Each library runs in its own process,
since a process loads one libftmoe."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import hashlib, json, os, sys
import numpy as np
import torch
root, lib = sys.argv[1], sys.argv[2]
sys.path.insert(0, root)
sys.path.insert(0, os.path.join(root, "tests"))
import nvfp4_quantized_moe_gb300 as ft
ft.LIB_PATH = lib
ft.load()
import synth
from moe_cases import GpuLayer, logits_for

def digest(t):
    return hashlib.sha256(t.contiguous().view(torch.uint8).cpu().numpy().tobytes()).hexdigest()

res = {}
for name, T, w4a4 in (("qwen36", 1, False), ("qwen36", 64, False), ("qwen36", 2048, False),
                      ("mini_w4a4", 256, False), ("mini_w4a4", 256, True),
                      ("mini_fp8", 8, False), ("mini_fp8", 512, False)):
    L = GpuLayer(name)
    H = L.shape.hidden
    x_bits = synth.make_activations(T, H, seed=5)
    ids, w = L.route(logits_for(name, T, True, seed=5))
    if w4a4:
        x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
        out = torch.empty((T, H), dtype=torch.float32, device="cuda")
        ws = torch.full((ft.ft_moe_workspace_size_w4a4(L.cfg, T),), 0xFF, dtype=torch.uint8, device="cuda")
        ft.ft_moe_forward_w4a4(L.cfg, L.routed, L.shared, x, ids, w, out, ws)
        st = ft.ft_moe_read_status(ws)
    else:
        out, st = L.forward(x_bits, ids, w, check_status=False)
    torch.cuda.synchronize()
    res[f"{name}/T{T}/{'w4a4' if w4a4 else 'w4a16'}"] = [int(st), digest(out)]
    del L
    torch.cuda.empty_cache()
print("RESULT " + json.dumps(res))
"""


def _run(lib: str) -> dict:
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT, lib], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")][-1]
    return json.loads(line[len("RESULT "):])


@pytest.mark.gpu
def test_bounds_check_build_agrees_with_regular_build():
    from nvfp4_quantized_moe_gb300 import build
    regular = build.build()
    checked = build.build(check=True)
    a, b = _run(regular), _run(checked)
    assert a.keys() == b.keys()
    for case in a:
        assert a[case][0] == 0, (case, "regular build status", a[case][0])
        assert b[case][0] == 0, (case, "bounds-checking build reported", b[case][0])
        assert a[case][1] == b[case][1], (case, "outputs differ between the builds")
