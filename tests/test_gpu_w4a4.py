"""The W4A4 variant (NVFP4 activations on the block-scaled FP4 tensor cores) against its
oracle: the activation quantizer bit for bit (codes, e4m3 scales, row scales) on bf16 and fp32
rows, and the forward (x and every expert's h quantized) within the stated floating-point
tolerance, every token, routed and shared experts, groups 16 and 32, tp = 1 and 2."""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_cases import GpuLayer, assert_close, logits_for, oracle_banks

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


def _e2m1_values(codes):
    lut = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])
    nib = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    nib[..., 0::2], nib[..., 1::2] = codes & 15, codes >> 4
    return lut[nib]


@pytest.mark.parametrize("src_dtype", ["bf16", "f32"])
def test_quantizer_matches_oracle_bit_exact(ft, src_dtype):
    rng = np.random.default_rng(61)
    rows, K = 96, 512
    x = (rng.standard_normal((rows, K)) * np.exp(rng.uniform(-6, 6, (rows, 1)))).astype(np.float32)
    x[3] = 0.0                      # an all-zero row
    x[5, 32:48] = 0.0               # an all-zero block
    x[7, :16] = [0.25, -0.75, 1.25, 1.75, 2.5, 3.5, 5, 6, 2688, 0.3, -0.3, 0, 7, -7, 100, 1e-6]
    if src_dtype == "bf16":
        bits = synth.bf16_bits_from_f32(x)
        xs = (bits.astype(np.uint32) << 16).view(np.float32)
        src = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        xs = x
        src = torch.from_numpy(x).cuda()
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, K // 16), dtype=torch.uint8, device="cuda")
    glob = torch.empty(rows, dtype=torch.float32, device="cuda")
    ft.ft_moe_quantize_nvfp4(src, codes, scales, glob)
    rc, rs, rg = oracle.quant_nvfp4(xs)
    assert np.array_equal(glob.cpu().numpy(), rg)
    assert np.array_equal(scales.cpu().numpy(), rs)
    # codes: bit-exact up to the sign of a zero (-0 and +0 are the same value)
    got = codes.cpu().numpy()
    assert np.array_equal(_e2m1_values(got), _e2m1_values(rc))
    nz = (got & 7) != 0
    assert np.array_equal(got[nz], rc[nz])


def _run(ft, name, T, zipf, tp_rank=0, tp_size=1, tokens=None):
    L = GpuLayer(name, tp_rank, tp_size)
    shape = synth.SHAPES[name]
    logits = logits_for(name, T, zipf, seed=4)
    x_bits = synth.make_activations(T, shape.hidden, seed=4)
    ids, w = L.route(logits)
    x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
    ws = torch.full((ft.ft_moe_workspace_size_w4a4(L.cfg, T),), 0xFF, dtype=torch.uint8, device="cuda")
    ft.ft_moe_forward_w4a4(L.cfg, L.routed, L.shared, x, ids, w, out, ws)
    assert ft.ft_moe_read_status(ws) == 0
    ref_ids, ref_w = oracle.route(logits, shape.top_k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    rb, sb = oracle_banks(name, tp_rank, tp_size)
    tokens = np.arange(T) if tokens is None else tokens
    ref = oracle.moe_forward(rb, sb, shape.group, x_bits, ref_ids, ref_w, tokens=tokens,
                             nthreads=oracle.default_threads(), w4a4=True)
    return out.cpu().numpy()[tokens], ref, x_bits, ref_ids, ref_w, rb, sb


@pytest.mark.parametrize("T,zipf", [(256, False), (1000, True), (3, False)])
def test_w4a4_forward_mini_every_token(ft, T, zipf):
    got, ref, *_ = _run(ft, "mini_w4a4", T, zipf)
    assert_close(got, ref, f"W4A4 mini T={T}")


def test_w4a4_forward_qwen36_prefill(ft):
    T = 2048
    got, ref, x_bits, ids, w, rb, sb = _run(ft, "qwen36", T, True)
    assert_close(got, ref, "W4A4 qwen36 T=2048")
    # the W4A4 numbers stay near the W4A16 layer's: only the noise of the two 4-bit activation
    # quantizations (x and h, each with a relative rounding error of about a tenth) separates them
    full = oracle.moe_forward(rb, sb, 16, x_bits, ids, w, tokens=np.arange(0, T, 64), nthreads=oracle.default_threads())
    rel = np.linalg.norm(got[::64] - full) / np.linalg.norm(full)
    assert 0.02 < rel < 0.25, rel


def test_w4a4_forward_tp2_and_group32(ft):
    for r in range(2):
        got, ref, *_ = _run(ft, "qwen36", 512, True, r, 2)
        assert_close(got, ref, f"W4A4 qwen36 tp=2 rank {r}")
    sample = np.arange(0, 256, 5)
    got, ref, *_ = _run(ft, "dsv4", 256, True, tokens=sample)
    assert_close(got, ref, "W4A4 dsv4 (group 32)")


def test_w4a4_rejects_unsupported_shapes(ft):
    cfg = ft.MoEConfig.of(synth.SHAPES["qwen36"], 0, 4)   # I_l = 128: not a whole 256-element stage
    with pytest.raises(ft.FtMoeError):
        ft.ft_moe_workspace_size_w4a4(cfg, 16)
