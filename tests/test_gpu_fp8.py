"""Parity of the fp8_block expert path (e4m3 codes, 128 x 128-block scale_inv) against
the oracle: pack byte-exact, forward within the floating tolerance of the NVFP4 tests."""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_cases import GpuLayer, assert_close, logits_for, oracle_banks, pieces

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_quantized_moe_gb300 import build
    build.build()


_layers = {}


def layer(name, tp_rank=0, tp_size=1):
    key = (name, tp_rank, tp_size)
    if key not in _layers:
        if len(_layers) > 4:
            _layers.clear()
            torch.cuda.empty_cache()
        _layers[key] = GpuLayer(name, tp_rank, tp_size)
    return _layers[key]


@pytest.mark.parametrize("name,tp", [("mini_fp8", 1), ("qwen36_fp8", 2), ("qwen36_fp8", 4)])
@pytest.mark.parametrize("from_host", [True, False])
def test_fp8_pack_matches_oracle_slicer(name, tp, from_host):
    for r in range(tp):
        L = GpuLayer(name, r, tp, from_host=from_host)
        rb, sb = oracle_banks(name, r, tp)
        for i, key in ((0, "gu"), (1, "gu_scale"), (3, "dn"), (4, "dn_scale")):
            assert np.array_equal(L.routed[i].cpu().numpy(), rb[key]), (key, r)
            assert np.array_equal(L.shared[i].cpu().numpy(), sb[key]), (key, r)
        assert L.routed[2].numel() == 0 and L.routed[5].numel() == 0  # no globals


def _run(name, T, zipf, tp_rank=0, tp_size=1, sample=None, out_dtype=torch.float32):
    L = layer(name, tp_rank, tp_size)
    shape = synth.SHAPES[name]
    logits = logits_for(name, T, zipf)
    x = synth.make_activations(T, shape.hidden)
    ids, w = L.route(logits)
    out, _ = L.forward(x, ids, w, out_dtype=out_dtype)
    ref_ids, ref_w = oracle.route(logits, shape.top_k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    rb, sb = oracle_banks(name, tp_rank, tp_size)
    tokens = np.arange(T) if sample is None else sample
    ref = oracle.moe_forward(rb, sb, 128, x, ref_ids, ref_w, tokens=tokens, nthreads=oracle.default_threads())
    return out.float().cpu().numpy()[tokens], ref


@pytest.mark.parametrize("T,zipf", [(1, False), (16, False), (200, True), (256, False), (1000, True)])
def test_fp8_forward_mini_every_token(T, zipf):
    """T >= 128 routes through the tensor-core kernels (T * k >= 32 * E), below through the GEMV."""
    got, ref = _run("mini_fp8", T, zipf)
    assert_close(got, ref, f"mini_fp8 T={T}")


@pytest.mark.parametrize("T", [1, 8, 64])
def test_fp8_forward_qwen36_decode(T):
    got, ref = _run("qwen36_fp8", T, False)
    assert_close(got, ref, f"qwen36_fp8 T={T}")


def test_fp8_forward_bf16_output():
    got, ref = _run("qwen36_fp8", 8, False, out_dtype=torch.bfloat16)
    assert_close(got, ref, "qwen36_fp8 bf16 out")


@pytest.mark.parametrize("T", [2048, 8192])
def test_fp8_forward_qwen36_prefill_sampled(T):
    rng = np.random.default_rng(T)
    sample = np.sort(rng.choice(T, size=16, replace=False))
    sample[0], sample[-1] = 0, T - 1
    got, ref = _run("qwen36_fp8", T, True, sample=sample)
    assert_close(got, ref, f"qwen36_fp8 prefill T={T}")


@pytest.mark.parametrize("tp", [2, 4])
def test_fp8_tp_partials_sum_to_full(tp):
    T = 32
    shape = synth.SHAPES["qwen36_fp8"]
    total = 0
    for r in range(tp):
        got, ref = _run("qwen36_fp8", T, False, r, tp)
        assert_close(got, ref, f"fp8 rank {r}/{tp}")
        total = total + got.astype(np.float64)
    ids, w = oracle.route(logits_for("qwen36_fp8", T, False), shape.top_k)
    rb, sb = oracle_banks("qwen36_fp8")
    x = synth.make_activations(T, shape.hidden)
    full = oracle.moe_forward(rb, sb, 128, x, ids, w, nthreads=oracle.default_threads())
    assert_close(total, full, f"sum of {tp} fp8 partials vs tp=1")
