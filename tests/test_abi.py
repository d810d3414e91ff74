"""Host-side checks of the C ABI: the library loads, exports every declared symbol,
and validates geometry and arguments before touching a GPU (no kernel runs here)."""
import ctypes
import json
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ft():
    from nvfp4_quantized_moe_gb300 import build
    build.build()
    import nvfp4_quantized_moe_gb300 as ft
    ft.load()
    return ft


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "ft_moe.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^(?:ft_status|const char \*|int64_t)\s*(ft_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(ft):
    declared = _declared_symbols()
    assert declared == sorted(ft.EXPORTS)
    lib = ctypes.CDLL(ft.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_bounds_checking_build_compiles_and_exports(ft):
    """The FTMOE_BOUNDS_CHECK variant (libftmoe_check.so) still compiles and exports the same
    ABI (its kernels run in tests/test_gpu_bounds_check.py)."""
    from nvfp4_quantized_moe_gb300 import build
    path = build.build(check=True)
    lib = ctypes.CDLL(path)
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_layout_matches_pages_bank_shapes(ft):
    with open(os.path.join(ROOT, "tests", "golden", "bank_layout_qwen36.json")) as f:
        g = json.load(f)
    for tp, want in g["per_tp"].items():
        cfg = ft.MoEConfig(g["hidden"], g["intermediate"], g["num_experts"], 8, g["group"], 512, 0, int(tp))
        got = {name: list(shape) for name, shape, _, _ in ft.ft_moe_layout(cfg, 0)}
        assert got == want, tp


def test_layout_bytes_and_shared(ft):
    cfg = ft.MoEConfig.of(synth.SHAPES["qwen36"])
    specs = ft.ft_moe_layout(cfg, 0)
    per_expert = sum(b for *_, b in specs) // 256
    assert per_expert == 1024 * 1024 + 1024 * 128 + 1024 * 4 + 2048 * 256 + 2048 * 32 + 2048 * 4 == 1781760
    sh = ft.ft_moe_layout(cfg, 1)
    assert [s for _, s, _, _ in sh][0] == (1, 1024, 1024)
    c4 = ft.MoEConfig.of(synth.SHAPES["dsv4"], 0, 4)
    assert sum(b for *_, b in ft.ft_moe_layout(c4, 0)) // 256 == (1024 * 2048 + 1024 * 128 + 1024 * 4 +
                                                                   4096 * 256 + 4096 * 16 + 4096 * 4)


def test_layout_follows_explicit_shard(ft):
    """An explicit range sizes the rank's banks by its own length, not intermediate/tp_size."""
    shape = synth.SHAPES["qwen36"]
    a = ft.MoEConfig.of(shape, 0, 2, shard=(0, 320), shared_shard=(0, 192))
    b = ft.MoEConfig.of(shape, 1, 2, shard=(320, 192), shared_shard=(192, 320))
    ra = {n: tuple(s) for n, s, _, _ in ft.ft_moe_layout(a, 0)}
    rb = {n: tuple(s) for n, s, _, _ in ft.ft_moe_layout(b, 0)}
    assert ra["gate_up"] == (256, 640, 1024) and rb["gate_up"] == (256, 384, 1024)
    assert ra["down"] == (256, 2048, 160) and rb["down"] == (256, 2048, 96)
    sa = {n: tuple(s) for n, s, _, _ in ft.ft_moe_layout(a, 1)}
    sb = {n: tuple(s) for n, s, _, _ in ft.ft_moe_layout(b, 1)}
    assert sa["gate_up"] == (1, 384, 1024) and sb["gate_up"] == (1, 640, 1024)


def test_layout_fp8_block(ft):
    """fp8_block banks: one code byte per weight, fp32 scale_inv per 128 x 128 block, no globals."""
    c = ft.MoEConfig.of(synth.SHAPES["qwen36_fp8"], 1, 2)
    got = {n: (tuple(sh), b) for n, sh, _, b in ft.ft_moe_layout(c, 0)}
    assert got["gate_up"] == ((256, 512, 2048), 256 * 512 * 2048)
    assert got["gate_up_scale"] == ((256, 4, 16), 256 * 4 * 16 * 4)
    assert got["down"] == ((256, 2048, 256), 256 * 2048 * 256)
    assert got["down_scale"] == ((256, 16, 2), 256 * 16 * 2 * 4)
    assert got["gate_up_global"][1] == 0 and got["down_global"][1] == 0


@pytest.mark.parametrize("fields,code", [
    (dict(format=1), 3),                                   # fp8_block needs group 128
    (dict(format=1, group=128, tp_size=4), 2),             # 512 / 4 = 128 is fine ...
    (dict(format=1, group=128, intermediate=384, tp_size=2), 2),  # ... 192 is not whole 128-blocks
    (dict(format=1, group=128, shard_begin=64, shard_size=128), 2),
    (dict(format=7), 1),
])
def test_layout_rejects_bad_fp8_geometry(ft, fields, code):
    base = dict(hidden=2048, intermediate=512, num_experts=256, top_k=8, group=16, shared_intermediate=512,
                tp_rank=0, tp_size=1, shard_begin=0, shard_size=0, shared_shard_begin=0, shared_shard_size=0,
                format=0)
    base.update(fields)
    cfg = ft.MoEConfig(*[base[n] for n, _ in ft.MoEConfig._fields_])
    if fields.get("tp_size") == 4 and fields.get("intermediate") is None:
        # shared 512 / 4 = 128 as well: valid
        assert len(ft.ft_moe_layout(cfg, 0)) == 6
        return
    with pytest.raises(ft.FtMoeError) as ei:
        ft.ft_moe_layout(cfg, 0)
    assert ei.value.status == code


@pytest.mark.parametrize("fields,code", [
    (dict(tp_size=3), 2),                      # 512 % 3
    (dict(tp_size=64), 2),                     # 512/64 = 8 not a multiple of 16
    (dict(group=8), 3),                        # unsupported block size
    (dict(num_experts=2048), 3),
    (dict(top_k=0), 1),
    (dict(tp_rank=2, tp_size=2), 1),
    (dict(hidden=2056), 2),                    # not a multiple of 16
    (dict(hidden=2064), 3),                    # multiple of 16, not of 128
    (dict(shared_intermediate=200), 2),        # 200 % 16 at tp=1
    (dict(shard_begin=8, shard_size=64), 2),   # begin not on a block boundary
    (dict(shard_begin=0, shard_size=40), 2),   # size not a whole number of blocks
    (dict(shard_begin=448, shard_size=128), 2),  # runs past the intermediate
    (dict(shard_size=-16), 1),
    (dict(shared_shard_begin=256, shared_shard_size=272), 2),  # shared range past 512
])
def test_layout_rejects_bad_geometry(ft, fields, code):
    base = dict(hidden=2048, intermediate=512, num_experts=256, top_k=8, group=16, shared_intermediate=512,
                tp_rank=0, tp_size=1, shard_begin=0, shard_size=0, shared_shard_begin=0, shared_shard_size=0,
                format=0)
    base.update(fields)
    cfg = ft.MoEConfig(*[base[n] for n, _ in ft.MoEConfig._fields_])
    with pytest.raises(ft.FtMoeError) as ei:
        ft.ft_moe_layout(cfg, 0)
    assert ei.value.status == code
    assert ft.ft_last_error()


def test_layout_shared_without_shared_expert(ft):
    cfg = ft.MoEConfig.of(synth.SHAPES["tiny"])
    with pytest.raises(ft.FtMoeError) as ei:
        ft.ft_moe_layout(cfg, 1)
    assert ei.value.status == 3


def test_forward_argument_checks_happen_before_launch(ft):
    lib = ft.load()
    cfg = ft.MoEConfig.of(synth.SHAPES["qwen36"])
    fake = ft._Banks()
    for i in range(6):
        fake.p[i] = 4096 * (i + 1)
    need = ctypes.c_size_t()
    assert lib.ft_moe_workspace_size(ctypes.byref(cfg), 64, ctypes.byref(need)) == 0
    assert need.value > 64 * 8 * 2048 * 4
    # T = 0 is a no-op
    assert lib.ft_moe_forward(ctypes.byref(cfg), ctypes.byref(fake), ctypes.byref(fake), None, 0, None, None,
                              None, ft.FT_DTYPE_F32, None, 0, None) == 0
    # missing shared banks when the layer has a shared expert
    assert lib.ft_moe_forward(ctypes.byref(cfg), ctypes.byref(fake), None, 4096, 4, 4096, 4096, 4096,
                              ft.FT_DTYPE_F32, 4096, need.value, None) == 1
    # misaligned activations
    assert lib.ft_moe_forward(ctypes.byref(cfg), ctypes.byref(fake), ctypes.byref(fake), 4098, 4, 4096, 4096,
                              4096, ft.FT_DTYPE_F32, 4096, 1 << 40, None) == 1
    # workspace too small
    assert lib.ft_moe_forward(ctypes.byref(cfg), ctypes.byref(fake), ctypes.byref(fake), 4096, 64, 4096, 4096,
                              8192, ft.FT_DTYPE_F32, 4096, need.value - 1, None) == 4
    # bad output dtype
    assert lib.ft_moe_forward(ctypes.byref(cfg), ctypes.byref(fake), ctypes.byref(fake), 4096, 4, 4096, 4096,
                              4096, 7, 4096, 1 << 40, None) == 1
    # routing limits
    assert lib.ft_moe_route(4096, 4, 2048, 8, 4096, 4096, None) == 3
    assert lib.ft_moe_route(4096, 4, 8, 9, 4096, 4096, None) == 3
    assert lib.ft_moe_route(None, 0, 8, 2, None, None, None) == 0
    n = ctypes.c_size_t()
    assert lib.ft_moe_align_workspace_size(8192, 8, 256, ctypes.byref(n)) == 0 and n.value > 8192 * 8 * 4
    assert lib.ft_moe_align(4096, 4, 2, 8, 0, 4096, 4096, 4096, 4096, 4096, 1 << 20, None) == 1


def test_route_gemm_argument_checks_happen_before_launch(ft):
    lib = ft.load()
    a = 4096  # aligned stand-in address; nothing is launched for these calls
    assert lib.ft_moe_route_gemm(None, 0, 2048, None, 256, 8, None, None, None, None) == 0   # T = 0
    assert lib.ft_moe_route_gemm(a, 4, 2040, a, 256, 8, a, a, a, None) == 1     # H not a multiple of 32
    assert lib.ft_moe_route_gemm(a, 4, 2048, a, 0, 8, a, a, a, None) == 1       # E = 0
    assert lib.ft_moe_route_gemm(a, 4, 2048, a, 2048, 8, a, a, a, None) == 3    # E > 1024
    assert lib.ft_moe_route_gemm(a, 4, 2048, a, 16, 17, a, a, a, None) == 3     # k > E
    assert lib.ft_moe_route_gemm(a + 8, 4, 2048, a, 256, 8, a, a, a, None) == 1  # x misaligned
    assert lib.ft_moe_route_gemm(a, 4, 2048, None, 256, 8, a, a, a, None) == 1  # no router weight


def test_pack_rejects_overlap(ft):
    lib = ft.load()
    cfg = ft.MoEConfig.of(synth.SHAPES["tiny"])
    banks = ft._Banks()
    for i in range(6):
        banks.p[i] = 1 << 20 + i
    pieces = ft._Pieces(*([1 << 20] * 9), 1)
    assert lib.ft_moe_pack(ctypes.byref(cfg), 0, ctypes.byref(pieces), ctypes.byref(banks), None) == 1


def test_align_static_rejects_sizes_beyond_its_array(ft):
    """The static entry point's limits (slots, experts, top_k) are checked on the host,
    before any CUDA call: sizes its fixed array cannot hold return FT_ERR_UNSUPPORTED."""
    lib = ctypes.CDLL(ft.LIB_PATH)
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    lib.ft_moe_align_static.argtypes = [P, I32, I32, I32, I32, P, P, P, P, P, P]
    lib.ft_moe_align_static.restype = ctypes.c_int
    dummy = ctypes.c_void_p(16)  # never dereferenced: the call returns before using it
    bufs = [dummy] * 4
    for T, k, E in ((1, 8, 1025), (1, 33, 64), (8193, 8, 256), (65537, 1, 8)):
        assert lib.ft_moe_align_static(dummy, T, k, E, 8, *bufs, None, None) == 3, (T, k, E)
    assert lib.ft_moe_align_static(dummy, -1, 8, 256, 8, *bufs, None, None) == 1
    assert lib.ft_moe_align_static(dummy, 4, 8, 256, 0, *bufs, None, None) == 1


def test_inject_stall_rejects_bad_arguments(ft):
    lib = ft.load()
    assert lib.ft_moe_debug_inject_stall(0, 2) == 1
    assert lib.ft_moe_debug_inject_stall(10, 1) == 1           # below 1 ms
    assert lib.ft_moe_debug_inject_stall(3 * 10 ** 9, 1) == 1  # above the default limit
