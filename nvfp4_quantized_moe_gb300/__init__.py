"""Python binding of libftmoe, the sm_103a NVFP4 (W4A16) routed-MoE expert forward.

Argument marshalling only: every function forwards to the C entry point of the same
name in ``libftmoe.so`` (declared in ``include/ft_moe.h``), passing torch tensors'
device pointers and the current CUDA stream. All arithmetic runs in the library's
CUDA kernels; there is no Python or CPU fallback, and importing this package fails
loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "FtMoeError", "MoEConfig", "load", "ft_moe_layout", "ft_moe_pack", "ft_moe_route", "ft_moe_route_gemm",
    "ft_moe_workspace_size", "ft_moe_forward", "ft_moe_align_workspace_size", "ft_moe_align",
    "ft_moe_dequant", "ft_moe_read_status", "ft_last_error", "alloc_banks", "EXPORTS",
    "FT_GU", "FT_GU_SCALE", "FT_GU_GLOBAL", "FT_DN", "FT_DN_SCALE", "FT_DN_GLOBAL",
    "FT_DTYPE_BF16", "FT_DTYPE_F32", "STATUS", "ft_moe_set_stage_events", "ft_moe_launch_count",
    "FT_NSTAGES", "STAGES", "ft_moe_debug_inject_stall", "ft_moe_workspace_size_w4a4", "ft_moe_forward_w4a4",
    "ft_moe_quantize_nvfp4",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libftmoe.so")

FT_GU, FT_GU_SCALE, FT_GU_GLOBAL, FT_DN, FT_DN_SCALE, FT_DN_GLOBAL, FT_NBANKS = range(7)
FT_DTYPE_U8, FT_DTYPE_E4M3, FT_DTYPE_F32, FT_DTYPE_BF16 = range(4)
FT_FORMAT_NVFP4, FT_FORMAT_FP8_BLOCK = range(2)
STATUS = {0: "FT_OK", 1: "FT_ERR_INVALID_ARG", 2: "FT_ERR_INDIVISIBLE", 3: "FT_ERR_UNSUPPORTED",
          4: "FT_ERR_WORKSPACE", 5: "FT_ERR_CUDA", 6: "FT_ERR_INVALID_ROUTING", 7: "FT_ERR_TIMEOUT",
          8: "FT_ERR_BOUNDS"}
BANK_NAMES = ("gate_up", "gate_up_scale", "gate_up_global", "down", "down_scale", "down_global")

# Every symbol include/ft_moe.h declares.
EXPORTS = ("ft_moe_layout", "ft_moe_pack", "ft_moe_route", "ft_moe_route_gemm", "ft_moe_workspace_size",
           "ft_moe_forward", "ft_moe_align_workspace_size", "ft_moe_align", "ft_moe_dequant", "ft_moe_read_status",
           "ft_last_error", "ft_moe_set_stage_events", "ft_moe_launch_count", "ft_moe_align_static",
           "ft_moe_debug_inject_stall", "ft_moe_workspace_size_w4a4", "ft_moe_forward_w4a4", "ft_moe_quantize_nvfp4")
FT_NSTAGES = 6
STAGES = ("align", "gate_up", "shared_gate_up", "down", "shared_down", "combine")


class FtMoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class MoEConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("intermediate", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("group", ctypes.c_int32), ("shared_intermediate", ctypes.c_int32),
                ("tp_rank", ctypes.c_int32), ("tp_size", ctypes.c_int32), ("shard_begin", ctypes.c_int32),
                ("shard_size", ctypes.c_int32), ("shared_shard_begin", ctypes.c_int32),
                ("shared_shard_size", ctypes.c_int32), ("format", ctypes.c_int32)]

    @classmethod
    def of(cls, shape, tp_rank: int = 0, tp_size: int = 1, shard=None, shared_shard=None) -> "MoEConfig":
        """Even split (tp_rank of tp_size) or explicit (begin, size) ranges of the intermediate."""
        sb, ss = shard if shard else (0, 0)
        hb, hs = shared_shard if shared_shard else (0, 0)
        fmt = FT_FORMAT_FP8_BLOCK if getattr(shape, "fmt", "nvfp4") == "fp8_block" else FT_FORMAT_NVFP4
        return cls(shape.hidden, shape.intermediate, shape.num_experts, shape.top_k, shape.group,
                   shape.shared_intermediate, tp_rank, tp_size, sb, ss, hb, hs, fmt)


class _BankSpec(ctypes.Structure):
    _fields_ = [("shape", ctypes.c_int64 * 3), ("ndim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("bytes", ctypes.c_int64)]


class _Banks(ctypes.Structure):
    _fields_ = [("p", ctypes.c_void_p * FT_NBANKS)]


class _Pieces(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate", "gate_scale", "gate_global", "up", "up_scale", "up_global",
                                               "down", "down_scale", "down_global")] + [("on_device", ctypes.c_int32)]


_lib = None


def load():
    """Load libftmoe.so; raise if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libftmoe.so not built at {LIB_PATH}: run nvfp4_quantized_moe_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        sigs = {
            "ft_moe_layout": [P, I32, P],
            "ft_moe_pack": [P, I32, P, P, P],
            "ft_moe_route": [P, I32, I32, I32, P, P, P],
            "ft_moe_route_gemm": [P, I32, I32, P, I32, I32, P, P, P, P],
            "ft_moe_workspace_size": [P, I32, P],
            "ft_moe_forward": [P, P, P, P, I32, P, P, P, I32, P, SZ, P],
            "ft_moe_align_workspace_size": [I32, I32, I32, P],
            "ft_moe_align": [P, I32, I32, I32, I32, P, P, P, P, P, SZ, P],
            "ft_moe_dequant": [P, I32, P, I32, I32, P, P],
            "ft_moe_read_status": [P, P],
            "ft_moe_set_stage_events": [P],
            "ft_moe_debug_inject_stall": [ctypes.c_uint64, I32],
            "ft_moe_workspace_size_w4a4": [P, I32, P],
            "ft_moe_forward_w4a4": [P, P, P, P, I32, P, P, P, I32, P, SZ, P],
            "ft_moe_quantize_nvfp4": [P, I32, I32, I32, P, P, P, P],
        }
        for name, args in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.ft_last_error.argtypes = []
        L.ft_last_error.restype = ctypes.c_char_p
        L.ft_moe_launch_count.argtypes = []
        L.ft_moe_launch_count.restype = ctypes.c_int64
        _lib = L
    return _lib


def ft_last_error() -> str:
    return load().ft_last_error().decode()


def _check(status: int):
    if status != 0:
        raise FtMoeError(status, ft_last_error())


def _stream(stream, *tensors):
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    for t in tensors:
        if isinstance(t, torch.Tensor) and t.is_cuda:
            return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)
    return ctypes.c_void_p(0)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return ctypes.c_void_p(t.data_ptr())
    return ctypes.c_void_p(t.ctypes.data)  # numpy (host pieces)


_DTYPES = {FT_DTYPE_U8: torch.uint8, FT_DTYPE_E4M3: torch.uint8, FT_DTYPE_F32: torch.float32,
           FT_DTYPE_BF16: torch.bfloat16}


def ft_moe_layout(cfg: MoEConfig, shared: int = 0):
    """[(name, shape, torch dtype, bytes)] for the six rank-local banks."""
    specs = (_BankSpec * FT_NBANKS)()
    _check(load().ft_moe_layout(ctypes.byref(cfg), shared, specs))
    return [(BANK_NAMES[i], tuple(specs[i].shape[:specs[i].ndim]), _DTYPES[specs[i].dtype], specs[i].bytes)
            for i in range(FT_NBANKS)]


def alloc_banks(cfg: MoEConfig, shared: int = 0, device="cuda"):
    """Allocate (with torch) the six banks ft_moe_layout describes."""
    return [torch.empty(shape, dtype=dt, device=device) for _, shape, dt, _ in ft_moe_layout(cfg, shared)]


def _banks(tensors):
    if tensors is None:
        return None
    b = _Banks()
    for i, t in enumerate(tensors):
        b.p[i] = t.data_ptr()
    return b


def ft_moe_pack(cfg: MoEConfig, shared: int, pieces: dict, banks, stream=None):
    """Slice full checkpoint-shaped pieces (all host numpy/CPU tensors or all CUDA tensors) into banks."""
    names = ("gate", "gate_scale", "gate_global", "up", "up_scale", "up_global", "down", "down_scale", "down_global")
    vals = [pieces.get(n) for n in names]  # fp8_block pieces have no globals
    given = [v for v in vals if v is not None]
    on_dev = all(isinstance(v, torch.Tensor) and v.is_cuda for v in given)
    if not on_dev:
        vals = [v.numpy() if isinstance(v, torch.Tensor) else v for v in vals]
    for v in vals:
        if v is not None and not (v.is_contiguous() if isinstance(v, torch.Tensor) else v.flags.c_contiguous):
            raise ValueError("pieces must be contiguous")
    p = _Pieces(*[_ptr(v).value if v is not None else None for v in vals], 1 if on_dev else 0)
    _check(load().ft_moe_pack(ctypes.byref(cfg), shared, ctypes.byref(p), ctypes.byref(_banks(banks)),
                              _stream(stream, *banks)))


def ft_moe_route(logits: torch.Tensor, k: int, topk_ids: torch.Tensor, topk_w: torch.Tensor, stream=None):
    T, E = logits.shape
    _check(load().ft_moe_route(_ptr(logits), T, E, k, _ptr(topk_ids), _ptr(topk_w), _stream(stream, logits)))


def ft_moe_route_gemm(x: torch.Tensor, w_router: torch.Tensor, k: int, logits: torch.Tensor, topk_ids: torch.Tensor,
                      topk_w: torch.Tensor, stream=None):
    """Router logits = x . w_router^T (bf16 in, fp32 [T, E] out), then the top-k of ft_moe_route."""
    T, H = x.shape
    E = w_router.shape[0]
    _check(load().ft_moe_route_gemm(_ptr(x), T, H, _ptr(w_router), E, k, _ptr(logits), _ptr(topk_ids),
                                    _ptr(topk_w), _stream(stream, x)))


def ft_moe_workspace_size(cfg: MoEConfig, T: int) -> int:
    n = ctypes.c_size_t()
    _check(load().ft_moe_workspace_size(ctypes.byref(cfg), T, ctypes.byref(n)))
    return n.value


def ft_moe_forward(cfg: MoEConfig, routed, shared, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor,
                   out: torch.Tensor, workspace: torch.Tensor, stream=None):
    """Rank-local partial into `out` (bf16 or fp32 [T, H])."""
    out_dtype = {torch.bfloat16: FT_DTYPE_BF16, torch.float32: FT_DTYPE_F32}[out.dtype]
    rb, sb = _banks(routed), _banks(shared)
    _check(load().ft_moe_forward(ctypes.byref(cfg), ctypes.byref(rb), ctypes.byref(sb) if sb is not None else None,
                                 _ptr(x), x.shape[0], _ptr(topk_ids), _ptr(topk_w), _ptr(out), out_dtype,
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream, x)))


def ft_moe_workspace_size_w4a4(cfg: MoEConfig, T: int) -> int:
    n = ctypes.c_size_t()
    _check(load().ft_moe_workspace_size_w4a4(ctypes.byref(cfg), T, ctypes.byref(n)))
    return n.value


def ft_moe_forward_w4a4(cfg: MoEConfig, routed, shared, x: torch.Tensor, topk_ids: torch.Tensor,
                        topk_w: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor, stream=None):
    """Rank-local partial with NVFP4 activations (W4A4) into `out` (bf16 or fp32 [T, H])."""
    out_dtype = {torch.bfloat16: FT_DTYPE_BF16, torch.float32: FT_DTYPE_F32}[out.dtype]
    rb, sb = _banks(routed), _banks(shared)
    _check(load().ft_moe_forward_w4a4(ctypes.byref(cfg), ctypes.byref(rb),
                                      ctypes.byref(sb) if sb is not None else None, _ptr(x), x.shape[0],
                                      _ptr(topk_ids), _ptr(topk_w), _ptr(out), out_dtype, _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream, x)))


def ft_moe_quantize_nvfp4(src: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, glob: torch.Tensor,
                          stream=None):
    """NVFP4 codes [rows, K/2], e4m3 scales [rows, K/16] and row scales [rows] of bf16 or fp32 rows."""
    dt = {torch.bfloat16: FT_DTYPE_BF16, torch.float32: FT_DTYPE_F32}[src.dtype]
    rows, K = src.shape
    _check(load().ft_moe_quantize_nvfp4(_ptr(src), dt, rows, K, _ptr(codes), _ptr(scales), _ptr(glob),
                                        _stream(stream, src)))


def ft_moe_align_workspace_size(T: int, k: int, E: int) -> int:
    n = ctypes.c_size_t()
    _check(load().ft_moe_align_workspace_size(T, k, E, ctypes.byref(n)))
    return n.value


def ft_moe_align(topk_ids: torch.Tensor, E: int, block: int, sorted_slot, block_expert, expert_off, n_padded,
                 workspace: torch.Tensor, stream=None):
    T, k = topk_ids.shape
    _check(load().ft_moe_align(_ptr(topk_ids), T, k, E, block, _ptr(sorted_slot), _ptr(block_expert),
                               _ptr(expert_off), _ptr(n_padded), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream, topk_ids)))


def ft_moe_dequant(cfg: MoEConfig, shared: int, banks, which: int, expert: int, out: torch.Tensor, stream=None):
    _check(load().ft_moe_dequant(ctypes.byref(cfg), shared, ctypes.byref(_banks(banks)), which, expert, _ptr(out),
                                 _stream(stream, out)))


def ft_moe_set_stage_events(events):
    """Arm per-stage timing of the next ft_moe_forward on this thread (FT_NSTAGES + 1 torch.cuda.Event)."""
    if events is None:
        _check(load().ft_moe_set_stage_events(None))
        return
    arr = (ctypes.c_void_p * (FT_NSTAGES + 1))(*[ev.cuda_event for ev in events])
    _check(load().ft_moe_set_stage_events(arr))


def ft_moe_debug_inject_stall(wait_limit_ns: int, skip_producer: int):
    """Arm fault injection for the next ft_moe_forward on this thread (see ft_moe.h)."""
    _check(load().ft_moe_debug_inject_stall(wait_limit_ns, skip_producer))


def ft_moe_launch_count() -> int:
    return int(load().ft_moe_launch_count())


def ft_moe_read_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise and return the device status word (0 = FT_OK)."""
    return load().ft_moe_read_status(_ptr(workspace), _stream(stream, workspace))
