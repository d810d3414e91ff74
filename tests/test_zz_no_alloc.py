"""ft_moe_align_static: the align entry point that allocates nothing.

Some callers cannot allocate device memory: code running in a host callback on a
stream may not call the CUDA API at all, and engines that plan all device memory at
start-up forbid allocation afterwards. ft_moe_align_static serves them with library-
owned static scratch. This test calls it through the C ABI and checks that its outputs
equal those of ft_moe_align (which uses a caller workspace), bit for bit, on two calls
in a row with different routings, on both the one-CTA and the multi-pass sort.
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
    cap = T * k + min(E, T * k) * (B - 1)
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


def _static(lib, ids, E, B):
    T, k = ids.shape
    out = _bufs(T, k, E, B)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.ft_moe_align_static(ctypes.c_void_p(ids.data_ptr()), T, k, E, B, *_ptrs(out),
                                 ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream))
    assert rc == 0
    torch.cuda.synchronize()
    return out, int(status.item())


@pytest.mark.parametrize("T,k,E,B", [(64, 8, 256, 8), (4096, 8, 256, 16), (8192, 8, 256, 128)])
def test_static_align_matches_workspace_align_twice(lib, T, k, E, B):
    for call, seed in enumerate((11, 12)):
        ids_np, _ = oracle.route(synth.zipf_logits(T, E, seed=seed), k)
        ids = torch.from_numpy(ids_np).cuda()
        ref = _with_workspace(ids, E, B)
        got, status = _static(lib, ids, E, B)
        assert status == 0, call
        n = int(ref[3].item())
        assert int(got[3].item()) == n, call
        assert torch.equal(got[0][:n], ref[0][:n]), call
        assert torch.equal(got[1][:n // B], ref[1][:n // B]), call
        assert torch.equal(got[2], ref[2]), call


def test_static_align_limits_and_status(lib):
    ids = torch.zeros((8193, 8), dtype=torch.int32, device="cuda")   # 65544 slots > 65536
    out = _bufs(1, 8, 256, 8)
    rc = lib.ft_moe_align_static(ctypes.c_void_p(ids.data_ptr()), 8193, 8, 256, 8, *_ptrs(out), None, None)
    assert rc == 3
    bad = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device="cuda")
    _, status = _static(lib, bad, 8, 4)
    assert status == 6
    good = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device="cuda")
    _, status = _static(lib, good, 8, 4)
    assert status == 0
