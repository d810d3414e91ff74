"""ft_moe_align_static: the align entry point that allocates nothing.

Some callers cannot allocate device memory: an engine that fixes every device
allocation at start-up may not allocate afterwards, and a caller that only owns the
buffers handed to it has nothing to size a workspace from. ft_moe_align_static serves
them with library-owned static scratch. This test calls it through the C ABI and checks,
on two calls in a row with different routings, that its outputs equal, bit for bit,
both those of ft_moe_align (the entry point with a caller workspace) and the oracle's
sort, on the one-CTA and the multi-pass sort (up to 32 chunks of 1024 experts), and that
device memory in use does not change across the calls.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_quantized_moe_gb300 import build
    build.build()
    import nvfp4_quantized_moe_gb300 as ft
    ft.load()
    L = ctypes.CDLL(ft.LIB_PATH)
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    L.ft_moe_align_static.argtypes = [P, I32, I32, I32, I32, P, P, P, P, P, P]
    L.ft_moe_align_static.restype = ctypes.c_int
    return L


def _bufs(T, k, E, B):
    cap = max(T * k + min(E, T * k) * (B - 1), 1)
    mk = lambda n: torch.full((n,), -5, dtype=torch.int32, device="cuda")
    return [mk(cap), mk(cap // B + 1), mk(E + 1), mk(1)]


def _ptrs(ts):
    return [ctypes.c_void_p(t.data_ptr()) for t in ts]


def _with_workspace(ids, E, B):
    import nvfp4_quantized_moe_gb300 as ft
    T, k = ids.shape
    out = _bufs(T, k, E, B)
    ws = torch.empty(ft.ft_moe_align_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    ft.ft_moe_align(ids, E, B, *out, ws)
    assert ft.ft_moe_read_status(ws) == 0
    return out


def _static_call(lib, ids, E, B, out, status):
    T, k = ids.shape
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.ft_moe_align_static(ctypes.c_void_p(ids.data_ptr()), T, k, E, B, *_ptrs(out),
                                 ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream))
    assert rc == 0
    torch.cuda.synchronize()


def _same(got, ref, B):
    n = int(ref[3].item())
    assert int(got[3].item()) == n
    assert torch.equal(got[0][:n], ref[0][:n])
    assert torch.equal(got[1][:n // B], ref[1][:n // B])
    assert torch.equal(got[2], ref[2])


def _matches_oracle(got, ids_np, E, B):
    ref_sorted, ref_block, ref_off, ref_n = oracle.align(ids_np, E, B)
    n = int(got[3].item())
    assert n == ref_n
    assert np.array_equal(got[0][:n].cpu().numpy(), ref_sorted)
    assert np.array_equal(got[1][:n // B].cpu().numpy(), ref_block)
    assert np.array_equal(got[2].cpu().numpy(), ref_off)


def _device_memory():
    free, _ = torch.cuda.mem_get_info()
    return free, torch.cuda.memory_allocated(), torch.cuda.memory_reserved()


@pytest.mark.parametrize("T,k,E,B", [(64, 8, 256, 8), (4096, 8, 256, 16), (8192, 8, 256, 128),
                                     (8192, 8, 1024, 64)])
def test_static_align_matches_workspace_align_and_oracle_twice(lib, T, k, E, B):
    routings = [oracle.route(synth.zipf_logits(T, E, seed=seed), k)[0] for seed in (11, 12)]
    ids = [torch.from_numpy(r).cuda() for r in routings]
    refs = [_with_workspace(i, E, B) for i in ids]
    outs = [_bufs(T, k, E, B) for _ in ids]
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _static_call(lib, ids[1], E, B, outs[1], status)  # first call on the device: address set-up
    torch.cuda.synchronize()
    before = _device_memory()
    for call in (0, 1):
        status.fill_(-1)
        _static_call(lib, ids[call], E, B, outs[call], status)
        assert int(status.item()) == 0, call
        _same(outs[call], refs[call], B)
        _matches_oracle(outs[call], routings[call], E, B)
    assert _device_memory() == before, "device memory in use changed across the calls"


def test_static_align_empty_input(lib):
    """T = 0: no slots, no blocks, every expert offset 0, status FT_OK."""
    E, B = 256, 8
    ids = torch.zeros((0, 8), dtype=torch.int32, device="cuda")
    out = _bufs(0, 8, E, B)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _static_call(lib, ids, E, B, out, status)
    assert int(status.item()) == 0
    assert int(out[3].item()) == 0
    assert not out[2].any()


def test_static_align_limits_and_status(lib):
    ids = torch.zeros((8193, 8), dtype=torch.int32, device="cuda")   # 65544 slots > 65536
    out = _bufs(1, 8, 256, 8)
    rc = lib.ft_moe_align_static(ctypes.c_void_p(ids.data_ptr()), 8193, 8, 256, 8, *_ptrs(out), None, None)
    assert rc == 3
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device="cuda")
    _static_call(lib, bad, 8, 4, _bufs(2, 2, 8, 4), status)
    assert int(status.item()) == 6
    good = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device="cuda")
    _static_call(lib, good, 8, 4, _bufs(2, 2, 8, 4), status)
    assert int(status.item()) == 0
