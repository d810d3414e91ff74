"""Shared fixtures for the parity tests: seeded layers, their CUDA banks and the oracle's view.

The same generator bytes feed both sides. The oracle side slices and computes with
``oracle`` only; the CUDA side packs and computes with the C ABI only.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import synth

RTOL_L2 = 1e-2        # relative L2 error bound on floating outputs
ATOL_RMS = 3e-2       # max-abs error bound, as a fraction of the oracle output's RMS
ROUTE_W_RTOL = 1e-6   # routing weights (fp32 on the GPU vs fp64 oracle)


@functools.lru_cache(maxsize=4)
def pieces(shape_name: str, seed: int = 0):
    shape = synth.SHAPES[shape_name]
    make = synth.make_fp8_pieces if shape.fmt == "fp8_block" else synth.make_pieces
    routed = make(shape, seed)
    shared = make(shape, seed, shared=True) if shape.shared_intermediate else None
    return routed, shared


def logits_for(shape_name: str, T: int, zipf: bool, seed: int = 0):
    E = synth.SHAPES[shape_name].num_experts
    return synth.zipf_logits(T, E, seed=seed) if zipf else synth.make_logits(T, E, seed=seed)


def oracle_banks(shape_name: str, tp_rank: int = 0, tp_size: int = 1, seed: int = 0, shard=None,
                 shared_shard=None):
    """Rank-local banks: even split (tp_rank of tp_size) or explicit (begin, size) ranges."""
    shape = synth.SHAPES[shape_name]
    routed, shared = pieces(shape_name, seed)
    if shape.fmt == "fp8_block":
        rb = oracle.slice_fp8_bank(routed, tp_rank, tp_size, shard=shard)
        sb = oracle.slice_fp8_bank(shared, tp_rank, tp_size, shard=shared_shard) if shared is not None else None
        return rb, sb
    rb = oracle.slice_bank(routed, shape.group, tp_rank, tp_size, shard=shard)
    sb = (oracle.slice_bank(shared, shape.group, tp_rank, tp_size, shard=shared_shard)
          if shared is not None else None)
    return rb, sb


def hot_block_sample(ids: np.ndarray, E: int, n: int, seed: int, block: int = 128, n_hot: int = 3):
    """Sorted token sample of size >= n that puts at least one token in every block of
    `block` expert-sorted positions of the n_hot most loaded experts (the blocks a
    tensor-core unit works on), the first and last token, and random others."""
    T, k = ids.shape
    counts = np.bincount(ids.reshape(-1), minlength=E)
    chosen = {0, T - 1}
    for e in np.argsort(-counts, kind="stable")[:n_hot]:
        slots = np.nonzero(ids.reshape(-1) == e)[0]  # slot order = the sort's order within e
        for b in range(0, len(slots), block):
            chosen.add(int(slots[b + (len(slots[b:b + block]) - 1) // 2]) // k)
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(T), np.fromiter(chosen, int))
    extra = max(0, n - len(chosen))
    chosen.update(rng.choice(rest, size=min(extra, len(rest)), replace=False).tolist())
    return np.array(sorted(chosen), dtype=np.int32)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.abs(got - ref).max())
    assert rel <= RTOL_L2, f"{what}: relative L2 error {rel:.3e} > {RTOL_L2}"
    assert mx <= ATOL_RMS * rms, f"{what}: max abs error {mx:.3e} > {ATOL_RMS} x RMS {rms:.3e}"
    return rel, mx / rms


class GpuLayer:
    """Rank-local banks of one layer on the GPU, packed through ft_moe_pack."""

    def __init__(self, shape_name: str, tp_rank: int = 0, tp_size: int = 1, seed: int = 0, from_host: bool = True,
                 shard=None, shared_shard=None):
        import nvfp4_quantized_moe_gb300 as ft
        self.ft = ft
        self.shape = synth.SHAPES[shape_name]
        self.cfg = ft.MoEConfig.of(self.shape, tp_rank, tp_size, shard=shard, shared_shard=shared_shard)
        routed, shared = pieces(shape_name, seed)
        self.routed = ft.alloc_banks(self.cfg, 0)
        src = routed if from_host else {k: torch.from_numpy(v).cuda() for k, v in routed.items()}
        ft.ft_moe_pack(self.cfg, 0, src, self.routed)
        self.shared = None
        if shared is not None:
            self.shared = ft.alloc_banks(self.cfg, 1)
            src = shared if from_host else {k: torch.from_numpy(v).cuda() for k, v in shared.items()}
            ft.ft_moe_pack(self.cfg, 1, src, self.shared)
        torch.cuda.synchronize()

    def route(self, logits: np.ndarray):
        T = logits.shape[0]
        k = self.shape.top_k
        lg = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        self.ft.ft_moe_route(lg, k, ids, w)
        return ids, w

    def forward(self, x_bits: np.ndarray, ids: torch.Tensor, w: torch.Tensor, out_dtype=torch.float32,
                check_status: bool = True):
        T, H = x_bits.shape
        x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
        out = torch.empty((T, H), dtype=out_dtype, device="cuda")
        # every byte 0xFF (a NaN in any float view): whatever the kernels read without
        # having written it first shows up in the output
        ws = torch.full((self.ft.ft_moe_workspace_size(self.cfg, T),), 0xFF, dtype=torch.uint8, device="cuda")
        self.ft.ft_moe_forward(self.cfg, self.routed, self.shared, x, ids, w, out, ws)
        st = self.ft.ft_moe_read_status(ws)
        if check_status:
            assert st == 0, self.ft.STATUS.get(st, st)
        return out, st
