"""The error path of the kernels that wait on one another, without faulting the GPU.

A host-side fault injection (ft_moe_debug_inject_stall) shortens every wait to 5 ms and
withholds what the waits are for: the tensor-core (prefill) kernels issue no copies, and
the fused decode kernel's gate_up stage publishes no finished block, so every bounded
wait runs out.
The forward must then report FT_ERR_TIMEOUT through the status word, every CTA must
return (the stream synchronises), and the next, normal call on the same stream and
context must succeed and reproduce the earlier output bit for bit (tensor memory was
freed and nothing was left waiting).
"""
import numpy as np
import pytest
import torch

import synth
from moe_cases import GpuLayer, logits_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ft():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_quantized_moe_gb300 import build
    build.build()
    import nvfp4_quantized_moe_gb300 as ft
    ft.load()
    return ft


@pytest.mark.parametrize("name,T", [("mini", 256), ("qwen36", 2048), ("qwen36", 1), ("qwen36", 8)])
def test_stalled_pipeline_reports_timeout_and_recovers(ft, name, T):
    L = GpuLayer(name)
    shape = synth.SHAPES[name]
    x = synth.make_activations(T, shape.hidden, seed=21)
    ids, w = L.route(logits_for(name, T, True, seed=21))
    good, st = L.forward(x, ids, w)
    assert st == 0
    n0 = ft.ft_moe_launch_count()
    ft.ft_moe_debug_inject_stall(5_000_000, 1)
    _, st = L.forward(x, ids, w, check_status=False)
    assert ft.ft_moe_launch_count() > n0
    assert ft.STATUS[st] == "FT_ERR_TIMEOUT"
    again, st = L.forward(x, ids, w)          # disarmed: a normal call
    assert st == 0
    assert torch.equal(again, good)


def test_injection_without_skip_changes_nothing(ft):
    """A short limit alone (no skipped producer) leaves a healthy pipeline's output intact."""
    L = GpuLayer("mini")
    x = synth.make_activations(256, 256, seed=22)
    ids, w = L.route(logits_for("mini", 256, False, seed=22))
    good, _ = L.forward(x, ids, w)
    ft.ft_moe_debug_inject_stall(1_000_000_000, 0)
    again, st = L.forward(x, ids, w)
    assert st == 0 and torch.equal(again, good)
    assert np.isfinite(good.cpu().numpy()).all()
