"""CPU oracle for the NVFP4 (and fp8_block) routed-MoE expert forward (TEST INFRASTRUCTURE ONLY).

A ctypes front end over ``ftmoe_oracle.c``, the plain fp64 C statement of the
layer. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline import this package; the CUDA library never does, and this package
never imports the CUDA library.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ftmoe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (portable C11, no target-specific flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


class Bank(ctypes.Structure):
    _fields_ = [("gu", ctypes.c_void_p), ("gu_scale", ctypes.c_void_p), ("gu_global", ctypes.c_void_p),
                ("dn", ctypes.c_void_p), ("dn_scale", ctypes.c_void_p), ("dn_global", ctypes.c_void_p),
                ("E", ctypes.c_int32), ("H", ctypes.c_int32), ("Il", ctypes.c_int32), ("g", ctypes.c_int32),
                ("fmt", ctypes.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            L.orc_e2m1.restype = D; L.orc_e2m1.argtypes = [ctypes.c_uint]
            L.orc_e4m3.restype = D; L.orc_e4m3.argtypes = [ctypes.c_uint]
            L.orc_dequant_bf16.restype = ctypes.c_uint16
            L.orc_dequant_bf16.argtypes = [ctypes.c_uint, ctypes.c_uint]
            L.orc_bf16_to_double.restype = D; L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_dequant_matrix.restype = None
            L.orc_dequant_matrix.argtypes = [P, P, P, I, I, I, P]
            L.orc_route.restype = I; L.orc_route.argtypes = [P, I, I, I, P, P]
            L.orc_router_logits.restype = None; L.orc_router_logits.argtypes = [P, P, I, I, I, P, P]
            L.orc_align.restype = I; L.orc_align.argtypes = [P, I, I, I, I, P, P, P, P]
            L.orc_slice.restype = I; L.orc_slice.argtypes = [I] * 6 + [P] * 15
            L.orc_slice_range.restype = I; L.orc_slice_range.argtypes = [I] * 6 + [P] * 15
            L.orc_slice_fp8_range.restype = I; L.orc_slice_fp8_range.argtypes = [I] * 5 + [P] * 10
            L.orc_dequant_fp8_matrix.restype = None
            L.orc_dequant_fp8_matrix.argtypes = [P, P, I, I, P]
            L.orc_expert_gate_up.restype = None
            L.orc_expert_gate_up.argtypes = [ctypes.POINTER(Bank), I, P, P]
            L.orc_swiglu.restype = None; L.orc_swiglu.argtypes = [P, I, P]
            L.orc_expert_gate_up_f64.restype = None
            L.orc_expert_gate_up_f64.argtypes = [ctypes.POINTER(Bank), I, P, P]
            L.orc_expert_down.restype = None
            L.orc_expert_down.argtypes = [ctypes.POINTER(Bank), I, P, P]
            L.orc_moe_forward.restype = I
            L.orc_moe_forward.argtypes = [ctypes.POINTER(Bank), ctypes.POINTER(Bank), P, I, P, P, I,
                                          P, I, P, I]
            L.orc_moe_forward_w4a4.restype = I
            L.orc_moe_forward_w4a4.argtypes = [ctypes.POINTER(Bank), ctypes.POINTER(Bank), P, I, P, P, I,
                                               P, I, P, I]
            L.orc_quant_nvfp4.restype = None
            L.orc_quant_nvfp4.argtypes = [P, I, I, P, P, P]
            L.orc_e4m3_code.restype = ctypes.c_uint; L.orc_e4m3_code.argtypes = [ctypes.c_float]
            L.orc_e2m1_code.restype = ctypes.c_uint; L.orc_e2m1_code.argtypes = [ctypes.c_float]
            _lib = L
        return _lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data


@contextlib.contextmanager
def mutation(code: int):
    """Plant one known mistake in the oracle for the duration of the block."""
    v = ctypes.c_int.in_dll(lib(), "orc_mutation")
    old = v.value
    v.value = code
    try:
        yield
    finally:
        v.value = old


MUTATIONS = {
    "nibble_order": 1, "swap_gate_up": 2, "drop_global": 3, "scale_index": 4, "e2m1_sign": 5,
    "no_renorm": 6, "tie_high": 7, "down_rows": 8, "drop_shared": 9, "drop_route_w": 10,
    "e4m3_bias": 11, "up_slice": 12, "router_transposed": 13, "fp8_block_transposed": 14,
    "dequant_transposed": 15, "w4a4_no_h_quant": 16, "e2m1_tie_up": 17, "row_scale_448": 18,
}


def e2m1(nibble: int) -> float:
    return lib().orc_e2m1(nibble)


def e4m3(byte: int) -> float:
    return lib().orc_e4m3(byte)


def dequant_bf16(nibble: int, scale_byte: int) -> int:
    return lib().orc_dequant_bf16(nibble, scale_byte)


def dequant_matrix(codes: np.ndarray, scales: np.ndarray, glob: np.ndarray, group: int) -> np.ndarray:
    """Dense fp64 [rows, K] of one expert matrix (codes [rows, K/2])."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    glob = np.ascontiguousarray(glob, np.float32)
    rows, K = codes.shape[0], codes.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    lib().orc_dequant_matrix(_p(codes), _p(scales), _p(glob), rows, K, group, _p(out))
    return out


def dequant_fp8_matrix(codes: np.ndarray, sinv: np.ndarray) -> np.ndarray:
    """Dense fp64 [rows, K] of one fp8_block expert matrix (codes [rows, K] u8,
    scale_inv [rows/128, K/128] f32)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    sinv = np.ascontiguousarray(sinv, np.float32)
    rows, K = codes.shape
    out = np.empty((rows, K), np.float64)
    lib().orc_dequant_fp8_matrix(_p(codes), _p(sinv), rows, K, _p(out))
    return out


def route(logits: np.ndarray, k: int):
    """(ids int32 [T,k], w float64 [T,k]) -- softmax, top-k, renormalise."""
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    if lib().orc_route(_p(logits), T, E, k, _p(ids), _p(w)) != 0:
        raise ValueError("bad routing arguments")
    return ids, w


def router_logits(x_bits: np.ndarray, w_bits: np.ndarray):
    """logits [T, E] = x [T, H] . W [E, H]^T over bf16 values in fp64, and absum
    [T, E] = sum |x * w| (the scale of rounding errors of lower-precision sums)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    T, H = x.shape
    E = w.shape[0]
    assert w.shape[1] == H
    logits = np.zeros((T, E), dtype=np.float64)
    absum = np.zeros((T, E), dtype=np.float64)
    lib().orc_router_logits(_p(x), _p(w), T, H, E, _p(logits), _p(absum))
    return logits, absum


def align(ids: np.ndarray, E: int, block: int):
    """(sorted_slot, block_expert, expert_off, n_padded) for ids [T, k]."""
    ids = np.ascontiguousarray(ids, np.int32)
    T, k = ids.shape
    cap = T * k + E * (block - 1)
    sorted_slot = np.full(max(cap, 1), -1, np.int32)
    block_expert = np.full(max(cap // block, 1), -1, np.int32)
    expert_off = np.zeros(E + 1, np.int32)
    n_padded = np.zeros(1, np.int32)
    if lib().orc_align(_p(ids), T, k, E, block, _p(sorted_slot), _p(block_expert),
                       _p(expert_off), _p(n_padded)) != 0:
        raise ValueError("invalid expert id or arguments")
    n = int(n_padded[0])
    return sorted_slot[:n].copy(), block_expert[:n // block].copy(), expert_off, n


def slice_bank(pieces: dict, group: int, tp_rank: int = 0, tp_size: int = 1, shard: tuple | None = None) -> dict:
    """Rank-local bank {gu, gu_scale, gu_global, dn, dn_scale, dn_global} from full pieces:
    the even split (tp_rank of tp_size) or, with shard = (begin, size), that explicit range."""
    c = {k: np.ascontiguousarray(v) for k, v in pieces.items()}
    E, I, H2 = c["gate"].shape
    H = H2 * 2
    if shard is None and I % tp_size:
        raise ValueError("intermediate not divisible by tp_size")
    Il = I // tp_size if shard is None else shard[1]
    out = {
        "gu": np.zeros((E, 2 * Il, H // 2), np.uint8),
        "gu_scale": np.zeros((E, 2 * Il, H // group), np.uint8),
        "gu_global": np.zeros((E, 2 * Il), np.float32),
        "dn": np.zeros((E, H, Il // 2), np.uint8),
        "dn_scale": np.zeros((E, H, Il // group), np.uint8),
        "dn_global": np.zeros((E, H), np.float32),
    }
    fn, a, b = (lib().orc_slice, tp_rank, tp_size) if shard is None else (lib().orc_slice_range, shard[0], shard[1])
    rc = fn(E, H, I, group, a, b,
            *[_p(c[n]) for n in ("gate", "gate_scale", "gate_global", "up", "up_scale",
                                 "up_global", "down", "down_scale", "down_global")],
            *[_p(out[n]) for n in ("gu", "gu_scale", "gu_global", "dn", "dn_scale",
                                   "dn_global")])
    if rc != 0:
        raise ValueError("indivisible or invalid tp geometry")
    return out


def slice_fp8_bank(pieces: dict, tp_rank: int = 0, tp_size: int = 1, shard: tuple | None = None) -> dict:
    """fp8_block rank-local bank {gu, gu_scale, dn, dn_scale, fmt} from full pieces
    (gate/up [E, I, H] u8 + [E, I/128, H/128] f32, down [E, H, I] u8 + [E, H/128, I/128]):
    the even split (tp_rank of tp_size) or the explicit range shard = (begin, size)."""
    c = {k: np.ascontiguousarray(v) for k, v in pieces.items()}
    E, I, H = c["gate"].shape
    if shard is None:
        if I % tp_size:
            raise ValueError("intermediate not divisible by tp_size")
        shard = (tp_rank * (I // tp_size), I // tp_size)
    b, n = shard
    out = {
        "gu": np.zeros((E, 2 * n, H), np.uint8),
        "gu_scale": np.zeros((E, 2 * n // 128, H // 128), np.float32),
        "dn": np.zeros((E, H, n), np.uint8),
        "dn_scale": np.zeros((E, H // 128, n // 128), np.float32),
        "fmt": "fp8_block",
    }
    rc = lib().orc_slice_fp8_range(E, H, I, b, n,
                                   *[_p(c[k]) for k in ("gate", "gate_scale", "up", "up_scale", "down",
                                                        "down_scale")],
                                   *[_p(out[k]) for k in ("gu", "gu_scale", "dn", "dn_scale")])
    if rc != 0:
        raise ValueError("range not made of whole 128-element blocks")
    return out


def _bank(b: dict, group: int) -> Bank:
    if b.get("fmt") == "fp8_block":
        E, rows, H = b["gu"].shape
        return Bank(_p(b["gu"]), _p(b["gu_scale"]), None, _p(b["dn"]), _p(b["dn_scale"]), None,
                    E, H, rows // 2, 128, 1)
    E, rows, H2 = b["gu"].shape
    return Bank(_p(b["gu"]), _p(b["gu_scale"]), _p(b["gu_global"]), _p(b["dn"]), _p(b["dn_scale"]),
                _p(b["dn_global"]), E, H2 * 2, rows // 2, group, 0)


def expert_gate_up(bank: dict, group: int, e: int, x_row: np.ndarray) -> np.ndarray:
    x_row = np.ascontiguousarray(x_row, np.uint16)
    G = np.zeros(bank["gu"].shape[1], np.float64)
    lib().orc_expert_gate_up(ctypes.byref(_bank(bank, group)), e, _p(x_row), _p(G))
    return G


def expert_gate_up_f64(bank: dict, group: int, e: int, x: np.ndarray) -> np.ndarray:
    """gate_up pre-activations of expert e on fp64 activations (the W4A4 path's dequantized x)."""
    x = np.ascontiguousarray(x, np.float64)
    G = np.zeros(bank["gu"].shape[1], np.float64)
    lib().orc_expert_gate_up_f64(ctypes.byref(_bank(bank, group)), e, _p(x), _p(G))
    return G


def swiglu(G: np.ndarray) -> np.ndarray:
    G = np.ascontiguousarray(G, np.float64)
    Il = G.shape[0] // 2
    h = np.zeros(Il, np.float64)
    lib().orc_swiglu(_p(G), Il, _p(h))
    return h


def expert_down(bank: dict, group: int, e: int, h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, np.float64)
    y = np.zeros(bank["dn"].shape[1], np.float64)
    lib().orc_expert_down(ctypes.byref(_bank(bank, group)), e, _p(h), _p(y))
    return y


def e4m3_code(v: float) -> int:
    """Nearest e4m3 code of a non-negative value (ties to even, saturating at 448)."""
    return int(lib().orc_e4m3_code(v))


def e2m1_code(v: float) -> int:
    """Nearest e2m1 code (sign bit 3; ties to even, saturating at 6)."""
    return int(lib().orc_e2m1_code(v))


def quant_nvfp4(x: np.ndarray):
    """NVFP4 quantization of fp32 rows [rows, K] (K % 16 == 0): (codes u8 [rows, K/2],
    e4m3 scales u8 [rows, K/16], fp32 row scales [rows])."""
    x = np.ascontiguousarray(x, np.float32)
    rows, K = x.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    scales = np.zeros((rows, K // 16), np.uint8)
    glob = np.zeros(rows, np.float32)
    lib().orc_quant_nvfp4(_p(x), rows, K, _p(codes), _p(scales), _p(glob))
    return codes, scales, glob


def moe_forward(routed: dict | None, shared: dict | None, group: int, x: np.ndarray,
                ids: np.ndarray | None = None, w: np.ndarray | None = None,
                tokens=None, nthreads: int = 1, w4a4: bool = False) -> np.ndarray:
    """Rank-local partial [len(tokens), H] in fp64 (x: bf16 bits [T, H]); w4a4 = True quantizes
    the activations (x, then each expert's h) to NVFP4 as the native FP4 variant does."""
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, np.int32)
    out = np.zeros((len(tokens), H), np.float64)
    rb = _bank(routed, group) if routed is not None else None
    sb = _bank(shared, group) if shared is not None else None
    if rb is not None:
        ids = np.ascontiguousarray(ids, np.int32)
        w = np.ascontiguousarray(w, np.float64)
        k = ids.shape[1]
        pids, pw = _p(ids), _p(w)
    else:
        k, pids, pw = 0, None, None
    fwd = lib().orc_moe_forward_w4a4 if w4a4 else lib().orc_moe_forward
    rc = fwd(ctypes.byref(rb) if rb is not None else None,
                               ctypes.byref(sb) if sb is not None else None,
                               _p(x), H, pids, pw, k, _p(tokens), len(tokens), _p(out), nthreads)
    if rc != 0:
        raise RuntimeError("oracle forward failed")
    return out


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
