"""Seeded synthetic inputs for the NVFP4 routed-MoE expert forward.

This module only draws random numbers and encodes them into the storage formats
the layer consumes (bf16 activations, fp32 logits, packed e2m1 code bytes, e4m3
scale bytes, fp32 per-row globals). It holds none of the layer's arithmetic and
is shared by the CUDA path's tests/bench and by the CPU oracle's tests: both
sides read the very same bytes.

Workload recipes (value distributions) follow the layer described on the
"[TP=2] Quantized MoE expert parallelism ... NVFP4 port" page, section 2
(hidden 2048, 256 experts, top-8, moe_intermediate 512, shared expert 512,
group size 16) and the "Offloaded MoE ignores tensor parallelism" page
(DeepSeek-V4-Flash FP4 experts with 32-element scale blocks):

* activations     bf16 ~ N(0, 1)
* router logits   fp32 ~ N(0, 1), optionally + ln Zipf(s) prior over a seeded
                  expert permutation (skewed prefill routing)
* code bytes      uniform over 0..255 (two independent uniform e2m1 nibbles)
* block scales    continuous U[0.25, 2] rounded to nearest-even e4m3
* weight_global   fp32 U[0.5, 1.5], one per output row
* router weights  bf16 ~ N(0, 1/H) [E, H] (replicated on every rank), so that with
                  N(0,1) activations the router logits are again ~ N(0, 1)

fp8_block experts (the Qwen3.6-35B-A3B-FP8 checkpoint of the "feat(qwen3_5_moe):
tensor-parallel weight sharding" page, Testing: same layer geometry, fp8 weights with a
128x128-block weight_scale_inv):

* weight codes    e4m3 (round-to-nearest-even, saturating at 448) of N(0, 1) * 32
* scale_inv       fp32 U[0.5, 1.5] * 2^-8, one per 128 x 128 block
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "LayerShape", "SHAPES", "rng_for", "bf16_bits_from_f32", "e4m3_rne_bytes",
    "make_pieces", "make_activations", "make_logits", "zipf_logits", "make_router_weights",
    "e4m3_rne_signed_bytes", "make_fp8_pieces",
]


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Geometry of one MoE layer (full intermediate, before any tp slicing)."""
    hidden: int
    intermediate: int
    num_experts: int
    top_k: int
    group: int = 16
    shared_intermediate: int = 0
    fmt: str = "nvfp4"  # or "fp8_block" (group is then the 128-element scale block)


# The layer families exercised by the tests and the bench.
SHAPES = {
    # tiny layer: T=16, H=256, E=8, top-2, I=64, no shared expert
    "tiny": LayerShape(hidden=256, intermediate=64, num_experts=8, top_k=2),
    # small layer whose tiles fit the 128-row tensor-core path (full-oracle parity)
    "mini": LayerShape(hidden=256, intermediate=256, num_experts=8, top_k=2, group=16, shared_intermediate=128),
    # Qwen3.6-35B-A3B-shaped MoE layer (decode and prefill)
    "qwen36": LayerShape(hidden=2048, intermediate=512, num_experts=256, top_k=8,
                         group=16, shared_intermediate=512),
    # DeepSeek-V4-Flash-like routed FP4 layer, 32-element scale blocks
    "dsv4": LayerShape(hidden=4096, intermediate=2048, num_experts=256, top_k=8,
                       group=32, shared_intermediate=2048),
    # hidden width not a multiple of 256 (the decode down stage's last row tile of a block
    # is partly out of range), small enough for full-oracle parity
    "odd_h": LayerShape(hidden=640, intermediate=512, num_experts=128, top_k=8, group=16,
                        shared_intermediate=512),
    # small layer whose every K is a whole 256-element stage of the W4A4 kernels (full-oracle parity)
    "mini_w4a4": LayerShape(hidden=256, intermediate=256, num_experts=8, top_k=2, group=16,
                            shared_intermediate=256),
    # fp8_block experts: a small layer (full-oracle parity) and the Qwen3.6-FP8 layer
    "mini_fp8": LayerShape(hidden=256, intermediate=256, num_experts=8, top_k=2, group=128,
                           shared_intermediate=128, fmt="fp8_block"),
    "qwen36_fp8": LayerShape(hidden=2048, intermediate=512, num_experts=256, top_k=8,
                             group=128, shared_intermediate=512, fmt="fp8_block"),
}


def rng_for(seed: int, *stream: int) -> np.random.Generator:
    """Independent PCG64 stream per (seed, tensor id, ...)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def e4m3_rne_bytes(v: np.ndarray) -> np.ndarray:
    """Encode positive values in [2^-6, 448] as OCP e4m3 bytes, round-to-nearest-even.

    Used only to draw the block scales. A normal e4m3 value is 2^(E-7) * (1 + M/8)
    with a 4-bit biased exponent E and a 3-bit mantissa M.
    """
    v = np.asarray(v, dtype=np.float64)
    if np.any(v < 2.0 ** -6) or np.any(v > 448.0):
        raise ValueError("scale outside the normal e4m3 range")
    e = np.floor(np.log2(v)).astype(np.int64)
    frac = v / np.exp2(e.astype(np.float64)) - 1.0          # in [0, 1)
    m = np.rint(frac * 8.0).astype(np.int64)                   # rint is half-to-even
    carry = m == 8
    m = np.where(carry, 0, m)
    e = np.where(carry, e + 1, e)
    return ((e + 7) << 3 | m).astype(np.uint8)


def e4m3_rne_signed_bytes(v: np.ndarray) -> np.ndarray:
    """Encode any finite values as OCP e4m3 bytes, round-to-nearest-even, saturating at
    +-448 (subnormals 2^-9 * m below 2^-6). Used only to draw fp8 weight codes."""
    v = np.asarray(v, dtype=np.float64)
    sign = (v < 0).astype(np.int64) << 7
    a = np.minimum(np.abs(v), 448.0)
    sub = a < 2.0 ** -6
    m_sub = np.rint(a * 2.0 ** 9).astype(np.int64)  # subnormal: a = m * 2^-9, m in 0..8
    safe = np.where(sub, 1.0, a)
    e = np.floor(np.log2(safe)).astype(np.int64)
    m = np.rint((safe / np.exp2(e.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
    carry = m == 8
    m = np.where(carry, 0, m)
    e = np.where(carry, e + 1, e)
    normal = ((e + 7) << 3) | m
    code = np.where(sub, m_sub, normal)  # m_sub == 8 is the smallest normal, byte 8
    return (sign | code).astype(np.uint8)


def _codes(rng, shape):
    return rng.integers(0, 256, size=shape, dtype=np.uint8)


def _scales(rng, shape):
    return e4m3_rne_bytes(rng.uniform(0.25, 2.0, size=shape))


def _globals(rng, shape):
    return rng.uniform(0.5, 1.5, size=shape).astype(np.float32)


def make_pieces(shape: LayerShape, seed: int = 0, shared: bool = False) -> dict[str, np.ndarray]:
    """Checkpoint-shaped expert tensors at full intermediate size, expert-major.

    Returns the nine tensors per expert of an NVFP4 checkpoint (weight, block
    scale, per-row global for each of gate, up and down):

      gate, up           u8  [E, I, H/2]   two e2m1 codes per byte
      gate_scale, ...    u8  [E, I, H/g]   e4m3 block scales
      gate_global, ...   f32 [E, I]        per output row
      down               u8  [E, H, I/2]
      down_scale         u8  [E, H, I/g]
      down_global        f32 [E, H]

    ``shared=True`` draws the always-on shared expert (E=1, I=shared_intermediate).
    """
    H, g = shape.hidden, shape.group
    if shared:
        E, I, base = 1, shape.shared_intermediate, 100
        if I == 0:
            raise ValueError("layer has no shared expert")
    else:
        E, I, base = shape.num_experts, shape.intermediate, 0
    r = lambda i: rng_for(seed, base + i)
    return {
        "gate": _codes(r(1), (E, I, H // 2)),
        "gate_scale": _scales(r(2), (E, I, H // g)),
        "gate_global": _globals(r(3), (E, I)),
        "up": _codes(r(4), (E, I, H // 2)),
        "up_scale": _scales(r(5), (E, I, H // g)),
        "up_global": _globals(r(6), (E, I)),
        "down": _codes(r(7), (E, H, I // 2)),
        "down_scale": _scales(r(8), (E, H, I // g)),
        "down_global": _globals(r(9), (E, H)),
    }


def make_fp8_pieces(shape: LayerShape, seed: int = 0, shared: bool = False) -> dict[str, np.ndarray]:
    """Checkpoint-shaped fp8_block expert tensors at full intermediate size, expert-major:

      gate, up           u8  [E, I, H]           e4m3 codes
      gate_scale, ...    f32 [E, I/128, H/128]   scale_inv per 128 x 128 block
      down               u8  [E, H, I]
      down_scale         f32 [E, H/128, I/128]
    """
    H = shape.hidden
    if shared:
        E, I, base = 1, shape.shared_intermediate, 700
        if I == 0:
            raise ValueError("layer has no shared expert")
    else:
        E, I, base = shape.num_experts, shape.intermediate, 600
    r = lambda i: rng_for(seed, base + i)
    codes = lambda g, sh: e4m3_rne_signed_bytes(g.standard_normal(sh) * 32.0)
    sinv = lambda g, sh: (g.uniform(0.5, 1.5, size=sh) * 2.0 ** -8).astype(np.float32)
    return {
        "gate": codes(r(1), (E, I, H)), "gate_scale": sinv(r(2), (E, I // 128, H // 128)),
        "up": codes(r(3), (E, I, H)), "up_scale": sinv(r(4), (E, I // 128, H // 128)),
        "down": codes(r(5), (E, H, I)), "down_scale": sinv(r(6), (E, H // 128, I // 128)),
    }


def make_activations(T: int, H: int, seed: int = 0, stream: int = 200) -> np.ndarray:
    """bf16 activations ~ N(0,1), returned as uint16 bit patterns [T, H]."""
    x = rng_for(seed, stream, T, H).standard_normal((T, H), dtype=np.float32)
    return bf16_bits_from_f32(x)


def make_logits(T: int, E: int, seed: int = 0, stream: int = 300) -> np.ndarray:
    """Router logits fp32 ~ N(0,1) [T, E] (near-uniform routing)."""
    return rng_for(seed, stream, T, E).standard_normal((T, E), dtype=np.float32)


def zipf_logits(T: int, E: int, s: float = 1.1, seed: int = 0, stream: int = 400) -> np.ndarray:
    """Skewed router logits: N(0,1) + ln p, p_{perm(r)} ~ (r+1)^-s over a seeded permutation."""
    rng = rng_for(seed, stream, T, E)
    perm = rng.permutation(E)
    ranks = np.arange(E, dtype=np.float64)
    prior = (ranks + 1.0) ** (-s)
    prior /= prior.sum()
    log_prior = np.empty(E, dtype=np.float64)
    log_prior[perm] = np.log(prior)
    noise = rng.standard_normal((T, E))
    return (noise + log_prior[None, :]).astype(np.float32)


def make_router_weights(E: int, H: int, seed: int = 0, stream: int = 500) -> np.ndarray:
    """Router weights bf16 ~ N(0, 1/H), returned as uint16 bit patterns [E, H]."""
    w = rng_for(seed, stream, E, H).standard_normal((E, H), dtype=np.float32) / np.float32(np.sqrt(H))
    return bf16_bits_from_f32(w)
