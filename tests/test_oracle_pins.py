"""Pins of the CPU oracle to facts outside itself.

Every pin compares the oracle with something it does not contain: library
routines (torch's float8_e4m3fn and bfloat16 conversions, torch fp64 softmax /
matmul / silu, Python's stable sort), closed forms, exact integer arithmetic,
brute force over all subsets, the OCP bit-field definitions, and the structural
properties the pages state (tp=1 is the identity; the sum of tp partials equals
the full-intermediate output; shards tile their axis). The last test plants known
mistakes in the oracle and checks that some pin catches each of them.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TINY = synth.SHAPES["tiny"]


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _e2m1_bitfield(nib):
    """OCP E2M1: S.EE.M, exponent bias 1, subnormal when E == 0."""
    s, e, m = (nib >> 3) & 1, (nib >> 1) & 3, nib & 1
    v = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -v if s else v


def _torch_e4m3(byte_array):
    t = torch.from_numpy(np.asarray(byte_array, np.uint8).copy()).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _nibbles(codes):
    """Independent unpacking: element 2m = low nibble of byte m (the stated convention)."""
    codes = np.asarray(codes, np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = codes & 15
    out[..., 1::2] = codes >> 4
    return out


def _dense(codes, scales, glob, group):
    """Test-side dequantisation: table lookup via the bit-field formula and torch's e4m3."""
    lut = np.array([_e2m1_bitfield(i) for i in range(16)])
    vals = lut[_nibbles(codes)]
    sc = np.repeat(_torch_e4m3(scales), group, axis=-1)
    return vals * sc * np.asarray(glob, np.float64)[..., None]


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def _tiny_layer(seed=0, shared=False, shape=TINY):
    pieces = synth.make_pieces(shape, seed)
    sp = synth.make_pieces(shape, seed, shared=True) if shared else None
    return pieces, sp


# ------------------------------------------------------------------ formats

def pin_e2m1():
    mags = _golden("e2m1_values.json")["magnitudes"]
    for n in range(16):
        v = oracle.e2m1(n)
        expect = (-1.0 if n & 8 else 1.0) * mags[n & 7]
        assert v == expect and math.copysign(1.0, v) == math.copysign(1.0, expect), n
        assert v == _e2m1_bitfield(n), n


def pin_e4m3():
    ref = _torch_e4m3(np.arange(256))
    for b in range(256):
        v = oracle.e4m3(b)
        if np.isnan(ref[b]):
            assert math.isnan(v), b
        else:
            assert v == ref[b] and math.copysign(1, v) == math.copysign(1, ref[b]), b
    g = _golden("e4m3_special_values.json")
    for code, val in g["values"].items():
        assert oracle.e4m3(int(code, 16)) == val, code
    for code in g["nan"]:
        assert math.isnan(oracle.e4m3(int(code, 16)))


def pin_dequant_bf16():
    sc = _torch_e4m3(np.arange(256))
    for s in range(256):
        if np.isnan(sc[s]):
            continue
        prods = np.array([_e2m1_bitfield(n) * sc[s] for n in range(16)])
        ref = torch.from_numpy(prods).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
        got = np.array([oracle.dequant_bf16(n, s) for n in range(16)], np.uint16)
        # exactness: the product survives the bf16 round trip unchanged
        assert np.array_equal(_bf16_to_f64(got), prods), s
        assert np.array_equal(got[np.abs(prods) > 0], ref[np.abs(prods) > 0]), s


# ------------------------------------------------------------------ routing

def pin_route_worked_example():
    g = _golden("routing_worked_example.json")
    logits = np.log(np.array([g["logits_ln_of"]], np.float64)).astype(np.float32)
    ids, w = oracle.route(logits, g["k"])
    assert ids[0].tolist() == g["ids"]
    assert np.allclose(w[0], g["weights"], rtol=1e-6, atol=0)


def pin_route_brute_force():
    T, E, k = 16, TINY.num_experts, TINY.top_k
    logits = synth.make_logits(T, E, seed=0)
    ids, w = oracle.route(logits, k)
    for t in range(T):
        p = torch.softmax(torch.from_numpy(logits[t].astype(np.float64)), 0).numpy()
        best = max(itertools.combinations(range(E), k), key=lambda c: (sum(p[list(c)]), [-i for i in c]))
        assert set(ids[t].tolist()) == set(best), t
        order = sorted(best, key=lambda i: (-p[i], i))
        assert ids[t].tolist() == order, t
        assert np.allclose(w[t], p[order] / p[order].sum(), rtol=1e-12, atol=0)
        assert abs(w[t].sum() - 1.0) < 1e-12


def pin_route_library():
    T, E, k = 64, 256, 8
    logits = synth.zipf_logits(T, E, seed=3)
    ids, w = oracle.route(logits, k)
    p = torch.softmax(torch.from_numpy(logits.astype(np.float64)), dim=1)
    vals, idx = torch.sort(p, dim=1, descending=True, stable=True)
    assert np.array_equal(ids, idx[:, :k].numpy().astype(np.int32))
    ref = (vals[:, :k] / vals[:, :k].sum(1, keepdim=True)).numpy()
    assert np.allclose(w, ref, rtol=1e-12, atol=0)


def pin_route_ties_and_shift():
    logits = np.array([[1.0, 3.0, 3.0, 0.5, 3.0, -2.0]], np.float32)
    ids, w = oracle.route(logits, 3)
    assert ids[0].tolist() == [1, 2, 4]
    assert np.allclose(w[0], [1 / 3] * 3, rtol=1e-12)
    ids2, w2 = oracle.route(logits + np.float32(5.0), 3)
    assert np.array_equal(ids, ids2) and np.allclose(w, w2, rtol=1e-12)


# ------------------------------------------------------------------ align

def pin_align():
    for T, E, k, B, seed in [(16, 8, 2, 4, 0), (33, 16, 4, 8, 1), (5, 64, 8, 16, 2), (1, 256, 8, 8, 3)]:
        ids, _ = oracle.route(synth.make_logits(T, E, seed=seed), k)
        sorted_slot, block_expert, expert_off, n = oracle.align(ids, E, B)
        flat = ids.reshape(-1)
        ref = sorted(range(T * k), key=lambda s: flat[s])   # Python's sort is stable
        real = sorted_slot[sorted_slot < T * k]
        assert real.tolist() == ref
        assert n % B == 0 and n == expert_off[E]
        assert np.all(sorted_slot[sorted_slot >= T * k] == T * k)
        for e in range(E):
            run = sorted_slot[expert_off[e]:expert_off[e + 1]]
            cnt = int((flat == e).sum())
            assert len(run) == (cnt + B - 1) // B * B
            assert all(flat[s] == e for s in run if s < T * k)
        for b, e in enumerate(block_expert):
            assert expert_off[e] <= b * B < expert_off[e + 1]
    with pytest.raises(ValueError):
        oracle.align(np.array([[0, 9]], np.int32), 8, 4)


# ------------------------------------------------------------------ tp slicing

def pin_slice_identity_and_tiling():
    pieces, _ = _tiny_layer()
    g = TINY.group
    b1 = oracle.slice_bank(pieces, g, 0, 1)
    # tp=1 is byte-identical to the plain concatenation [gate; up]
    assert np.array_equal(b1["gu"], np.concatenate([pieces["gate"], pieces["up"]], axis=1))
    assert np.array_equal(b1["gu_scale"], np.concatenate([pieces["gate_scale"], pieces["up_scale"]], 1))
    assert np.array_equal(b1["gu_global"], np.concatenate([pieces["gate_global"], pieces["up_global"]], 1))
    for n in ("dn", "dn_scale", "dn_global"):
        src = {"dn": "down", "dn_scale": "down_scale", "dn_global": "down_global"}[n]
        assert np.array_equal(b1[n], pieces[src])
    for tp in (2, 4):
        banks = [oracle.slice_bank(pieces, g, r, tp) for r in range(tp)]
        Il = TINY.intermediate // tp
        # gate rows / up rows tile the full intermediate axis in rank order
        assert np.array_equal(np.concatenate([b["gu"][:, :Il] for b in banks], 1), pieces["gate"])
        assert np.array_equal(np.concatenate([b["gu"][:, Il:] for b in banks], 1), pieces["up"])
        assert np.array_equal(np.concatenate([b["gu_scale"][:, Il:] for b in banks], 1), pieces["up_scale"])
        assert np.array_equal(np.concatenate([b["gu_global"][:, :Il] for b in banks], 1), pieces["gate_global"])
        # down is a column slice; its scales follow on the same axis; its global is whole
        assert np.array_equal(np.concatenate([b["dn"] for b in banks], 2), pieces["down"])
        assert np.array_equal(np.concatenate([b["dn_scale"] for b in banks], 2), pieces["down_scale"])
        for b in banks:
            assert np.array_equal(b["dn_global"], pieces["down_global"])
    with pytest.raises(ValueError):
        oracle.slice_bank(pieces, g, 0, 3)      # 64 % 3
    with pytest.raises(ValueError):
        oracle.slice_bank(pieces, g, 0, 8)      # 64/8 = 8 is not a multiple of the 16-element block


# ------------------------------------------------------------------ expert arithmetic

def pin_one_hot_columns():
    """x = e_k makes each pre-activation equal to column k of the dequantised matrix."""
    pieces, _ = _tiny_layer(seed=5)
    bank = oracle.slice_bank(pieces, TINY.group)
    dense = _dense(bank["gu"][3], bank["gu_scale"][3], bank["gu_global"][3], TINY.group)
    one = synth.bf16_bits_from_f32(np.array([1.0], np.float32))[0]
    for k in (0, 1, 15, 16, 17, 130, 255):
        x = np.zeros(TINY.hidden, np.uint16)
        x[k] = one
        G = oracle.expert_gate_up(bank, TINY.group, 3, x)
        assert np.array_equal(G, dense[:, k]), k


def _exact_dot(w_rows, x_vals):
    return [sum((Fraction(a) * Fraction(b) for a, b in zip(row, x_vals)), Fraction(0)) for row in w_rows]


def pin_linear_parts_exact():
    """Dyadic inputs make fp64 sums exact: compare bit-for-bit with rational arithmetic."""
    pieces, _ = _tiny_layer(seed=7)
    pieces = dict(pieces)
    rng = np.random.default_rng(11)
    for nm in ("gate_global", "up_global", "down_global"):
        pieces[nm] = rng.choice(np.array([0.5, 0.75, 1.0, 1.25, 1.5], np.float32), size=pieces[nm].shape)
    bank = oracle.slice_bank(pieces, TINY.group)
    xv = rng.integers(-12, 13, size=TINY.hidden) / 4.0
    x = synth.bf16_bits_from_f32(xv.astype(np.float32))
    e = 2
    W = _dense(bank["gu"][e], bank["gu_scale"][e], bank["gu_global"][e], TINY.group)
    G = oracle.expert_gate_up(bank, TINY.group, e, x)
    exact = _exact_dot(W.tolist(), xv.tolist())
    assert all(Fraction(g) == ex for g, ex in zip(G.tolist(), exact))
    hv = rng.integers(-40, 41, size=TINY.intermediate) / 8.0
    Wd = _dense(bank["dn"][e], bank["dn_scale"][e], bank["dn_global"][e], TINY.group)
    y = oracle.expert_down(bank, TINY.group, e, hv)
    exact = _exact_dot(Wd.tolist(), hv.tolist())
    assert all(Fraction(v) == ex for v, ex in zip(y.tolist(), exact))


def pin_dense_mlp_special_case():
    """E=1, k=1, weight 1 is a dense SwiGLU MLP: torch fp64 silu/matmul on test-side weights."""
    shape = synth.LayerShape(hidden=256, intermediate=96, num_experts=1, top_k=1)
    pieces = synth.make_pieces(shape, seed=9)
    bank = oracle.slice_bank(pieces, 16)
    x = synth.make_activations(5, 256, seed=9)
    ids = np.zeros((5, 1), np.int32)
    w = np.ones((5, 1))
    out = oracle.moe_forward(bank, None, 16, x, ids, w)
    Wg = torch.from_numpy(_dense(pieces["gate"][0], pieces["gate_scale"][0], pieces["gate_global"][0], 16))
    Wu = torch.from_numpy(_dense(pieces["up"][0], pieces["up_scale"][0], pieces["up_global"][0], 16))
    Wd = torch.from_numpy(_dense(pieces["down"][0], pieces["down_scale"][0], pieces["down_global"][0], 16))
    xt = torch.from_numpy(_bf16_to_f64(x))
    ref = (torch.nn.functional.silu(xt @ Wg.T) * (xt @ Wu.T)) @ Wd.T
    assert torch.allclose(torch.from_numpy(out), ref, rtol=1e-12, atol=1e-9 * ref.abs().max().item())
    # the same MLP as the shared expert (no routed experts) gives the same rows
    sh = oracle.moe_forward(None, bank, 16, x)
    assert np.array_equal(sh, out)


def pin_routed_combination():
    """Output = sum_j w_j * expert_j(x) + shared(x): checked against separate expert calls."""
    shape = synth.LayerShape(hidden=256, intermediate=64, num_experts=8, top_k=2, shared_intermediate=32)
    pieces, sp = _tiny_layer(seed=4, shared=True, shape=shape)
    bank = oracle.slice_bank(pieces, 16)
    sbank = oracle.slice_bank(sp, 16)
    T = 6
    x = synth.make_activations(T, 256, seed=4)
    ids, w = oracle.route(synth.make_logits(T, 8, seed=4), 2)
    out = oracle.moe_forward(bank, sbank, 16, x, ids, w)
    single = oracle.moe_forward(None, sbank, 16, x)
    for t in range(T):
        acc = np.zeros(256)
        for j in range(2):
            e = int(ids[t, j])
            Wg = _dense(pieces["gate"][e], pieces["gate_scale"][e], pieces["gate_global"][e], 16)
            Wu = _dense(pieces["up"][e], pieces["up_scale"][e], pieces["up_global"][e], 16)
            Wd = _dense(pieces["down"][e], pieces["down_scale"][e], pieces["down_global"][e], 16)
            xv = _bf16_to_f64(x[t])
            gt, ut = Wg @ xv, Wu @ xv
            acc += w[t, j] * (Wd @ (gt / (1 + np.exp(-gt)) * ut))
        assert np.allclose(out[t] - single[t], acc, rtol=1e-10, atol=1e-9 * np.abs(acc).max())


def pin_untouched_experts_and_tokens():
    pieces, _ = _tiny_layer(seed=2)
    bank = oracle.slice_bank(pieces, TINY.group)
    T = 16
    x = synth.make_activations(T, TINY.hidden, seed=2)
    ids, w = oracle.route(synth.make_logits(T, TINY.num_experts, seed=2)[:, :], TINY.top_k)
    out = oracle.moe_forward(bank, None, TINY.group, x, ids, w)
    # experts nobody routed to can hold anything
    used = set(ids.reshape(-1).tolist())
    junk = {k: v.copy() for k, v in pieces.items()}
    rng = np.random.default_rng(1)
    for e in range(TINY.num_experts):
        if e not in used:
            for nm in ("gate", "up", "down", "gate_scale", "up_scale", "down_scale"):
                junk[nm][e] = rng.integers(0, 127, size=junk[nm][e].shape, dtype=np.uint8)
    if len(used) < TINY.num_experts:
        out2 = oracle.moe_forward(oracle.slice_bank(junk, TINY.group), None, TINY.group, x, ids, w)
        assert np.array_equal(out, out2)
    # each token row is independent of the others
    for t in (0, 7, 15):
        one = oracle.moe_forward(bank, None, TINY.group, x[t:t + 1], ids[t:t + 1], w[t:t + 1])
        assert np.array_equal(one[0], out[t])
    sub = oracle.moe_forward(bank, None, TINY.group, x, ids, w, tokens=[15, 3], nthreads=2)
    assert np.array_equal(sub, out[[15, 3]])


def pin_tp_partial_sum():
    """Sum over ranks of rank-local partials equals the full-intermediate output."""
    shape = synth.LayerShape(hidden=256, intermediate=128, num_experts=8, top_k=2, shared_intermediate=64)
    pieces, sp = _tiny_layer(seed=6, shared=True, shape=shape)
    T = 8
    x = synth.make_activations(T, 256, seed=6)
    ids, w = oracle.route(synth.make_logits(T, 8, seed=6), 2)
    full = oracle.moe_forward(oracle.slice_bank(pieces, 16), oracle.slice_bank(sp, 16), 16, x, ids, w)
    for tp in (2, 4):
        parts = [oracle.moe_forward(oracle.slice_bank(pieces, 16, r, tp), oracle.slice_bank(sp, 16, r, tp),
                                    16, x, ids, w) for r in range(tp)]
        total = np.sum(parts, axis=0)
        rel = np.abs(total - full).max() / np.abs(full).max()
        assert rel < 1e-12, (tp, rel)
        # a single rank alone is not the answer (the check is sensitive)
        assert np.abs(parts[0] - full).max() / np.abs(full).max() > 1e-3


def pin_asymmetric_partition():
    """Explicit uneven ranges: equal to the even split when the range is the rank's share,
    tile the intermediate axis, and their partials sum to the full output (linearity)."""
    shape = synth.LayerShape(hidden=256, intermediate=128, num_experts=8, top_k=2, shared_intermediate=64)
    pieces, sp = _tiny_layer(seed=12, shared=True, shape=shape)
    for r in range(4):
        even, rng_ = oracle.slice_bank(pieces, 16, r, 4), oracle.slice_bank(pieces, 16, shard=(32 * r, 32))
        assert all(np.array_equal(even[n], rng_[n]) for n in even)
    cuts = [(0, 48), (48, 64), (112, 16)]
    banks = [oracle.slice_bank(pieces, 16, shard=c) for c in cuts]
    gate_rows = np.concatenate([b["gu"][:, :c[1]] for b, c in zip(banks, cuts)], axis=1)
    assert np.array_equal(gate_rows, pieces["gate"])
    T = 8
    x = synth.make_activations(T, 256, seed=12)
    ids, w = oracle.route(synth.make_logits(T, 8, seed=12), 2)
    full = oracle.moe_forward(oracle.slice_bank(pieces, 16), oracle.slice_bank(sp, 16), 16, x, ids, w)
    shared_cuts = [(0, 16), (16, 32), (48, 16)]
    parts = [oracle.moe_forward(b, oracle.slice_bank(sp, 16, shard=sc), 16, x, ids, w)
             for b, sc in zip(banks, shared_cuts)]
    rel = np.abs(np.sum(parts, axis=0) - full).max() / np.abs(full).max()
    assert rel < 1e-12, rel


def pin_router_logits_exact():
    """Router logits against exact rational arithmetic: with these magnitudes every
    bf16 product and every partial sum fits 53 bits, so fp64 must be exact; absum too.
    Square E == H so that a transposed read would still index inside W (and differ)."""
    T, H, E = 3, 16, 16
    x = synth.make_activations(T, H, seed=21)
    w = synth.make_router_weights(E, H, seed=21)
    logits, absum = oracle.router_logits(x, w)
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wv = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(T):
        for e in range(E):
            exact = sum((Fraction(a) * Fraction(b) for a, b in zip(xv[t], wv[e])), Fraction(0))
            mag = sum((abs(Fraction(a) * Fraction(b)) for a, b in zip(xv[t], wv[e])), Fraction(0))
            assert Fraction(logits[t, e]) == exact and Fraction(absum[t, e]) == mag


def pin_router_one_hot():
    """A one-hot token selects one column of the router weight: logits[e] = W[e][i]."""
    H = E = 16
    w = synth.make_router_weights(E, H, seed=22)
    wv = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    x = np.zeros((H, H), np.uint16)
    x[np.arange(H), np.arange(H)] = synth.bf16_bits_from_f32(np.ones(1, np.float32))[0]
    logits, _ = oracle.router_logits(x, w)
    assert np.array_equal(logits, wv.T)


# ------------------------------------------------------------------ fp8_block experts

FP8 = synth.LayerShape(hidden=256, intermediate=256, num_experts=4, top_k=2, group=128,
                       shared_intermediate=256, fmt="fp8_block")


def _dense_fp8(codes, sinv):
    """Test-side fp8_block dequantisation: torch's e4m3 times the 128 x 128 block grid
    expanded with np.kron (an independent statement of "one scale per block")."""
    return _torch_e4m3(codes) * np.kron(np.asarray(sinv, np.float64), np.ones((128, 128)))


def pin_fp8_slice_identity_and_tiling():
    pieces = synth.make_fp8_pieces(FP8, seed=31)
    b1 = oracle.slice_fp8_bank(pieces)
    assert np.array_equal(b1["gu"], np.concatenate([pieces["gate"], pieces["up"]], axis=1))
    assert np.array_equal(b1["gu_scale"], np.concatenate([pieces["gate_scale"], pieces["up_scale"]], 1))
    assert np.array_equal(b1["dn"], pieces["down"]) and np.array_equal(b1["dn_scale"], pieces["down_scale"])
    banks = [oracle.slice_fp8_bank(pieces, r, 2) for r in range(2)]
    assert np.array_equal(np.concatenate([b["gu"][:, :128] for b in banks], 1), pieces["gate"])
    assert np.array_equal(np.concatenate([b["gu"][:, 128:] for b in banks], 1), pieces["up"])
    assert np.array_equal(np.concatenate([b["gu_scale"][:, 1:] for b in banks], 1), pieces["up_scale"])
    assert np.array_equal(np.concatenate([b["dn"] for b in banks], 2), pieces["down"])
    assert np.array_equal(np.concatenate([b["dn_scale"] for b in banks], 2), pieces["down_scale"])
    with pytest.raises(ValueError):
        oracle.slice_fp8_bank(pieces, 0, 4)      # 64 is not a whole 128-element block
    with pytest.raises(ValueError):
        oracle.slice_fp8_bank(pieces, shard=(64, 128))


def pin_fp8_one_hot_columns():
    """x = e_k gives column k of the block-scaled fp8 matrix, for k in both K blocks and
    rows in all four row blocks of gate_up (and the same through down with h = e_i)."""
    pieces = synth.make_fp8_pieces(FP8, seed=32)
    bank = oracle.slice_fp8_bank(pieces)
    e = 2
    dense = _dense_fp8(bank["gu"][e], bank["gu_scale"][e])
    one = synth.bf16_bits_from_f32(np.array([1.0], np.float32))[0]
    for k in (0, 5, 127, 128, 200, 255):
        x = np.zeros(FP8.hidden, np.uint16)
        x[k] = one
        assert np.array_equal(oracle.expert_gate_up(bank, 128, e, x), dense[:, k]), k
    dd = _dense_fp8(bank["dn"][e], bank["dn_scale"][e])
    for i in (3, 130):
        h = np.zeros(FP8.intermediate)
        h[i] = 1.0
        assert np.array_equal(oracle.expert_down(bank, 128, e, h), dd[:, i]), i


def pin_fp8_dense_mlp_and_partials():
    """E=1, k=1, weight 1: a dense SwiGLU MLP (torch fp64 on test-side weights); and the
    tp=2 partials of a routed layer with a shared expert sum to the full output."""
    shape = synth.LayerShape(hidden=256, intermediate=256, num_experts=1, top_k=1, group=128, fmt="fp8_block")
    pieces = synth.make_fp8_pieces(shape, seed=33)
    x = synth.make_activations(4, 256, seed=33)
    out = oracle.moe_forward(oracle.slice_fp8_bank(pieces), None, 128, x, np.zeros((4, 1), np.int32), np.ones((4, 1)))
    Wg, Wu, Wd = (torch.from_numpy(_dense_fp8(pieces[n][0], pieces[n + "_scale"][0])) for n in ("gate", "up", "down"))
    xt = torch.from_numpy(_bf16_to_f64(x))
    ref = (torch.nn.functional.silu(xt @ Wg.T) * (xt @ Wu.T)) @ Wd.T
    assert torch.allclose(torch.from_numpy(out), ref, rtol=1e-12, atol=1e-9 * ref.abs().max().item())
    pieces = synth.make_fp8_pieces(FP8, seed=34)
    sp = synth.make_fp8_pieces(FP8, seed=34, shared=True)
    T = 6
    x = synth.make_activations(T, 256, seed=34)
    ids, w = oracle.route(synth.make_logits(T, FP8.num_experts, seed=34), 2)
    full = oracle.moe_forward(oracle.slice_fp8_bank(pieces), oracle.slice_fp8_bank(sp), 128, x, ids, w)
    parts = [oracle.moe_forward(oracle.slice_fp8_bank(pieces, r, 2), oracle.slice_fp8_bank(sp, r, 2), 128, x, ids, w)
             for r in range(2)]
    rel = np.abs(np.sum(parts, axis=0) - full).max() / np.abs(full).max()
    assert rel < 1e-12, rel
    assert np.abs(parts[0] - full).max() / np.abs(full).max() > 1e-3


def pin_dequant_matrices():
    """The oracle's dense matrix routines against the test-side dequantisers on
    non-square matrices (a row-stride or transposition slip changes the result): NVFP4
    with groups 16 and 32, its per-row global included, and fp8_block with three row
    blocks and two K blocks."""
    rng = np.random.default_rng(41)
    for rows, K, g in ((48, 96, 16), (40, 128, 32), (3, 256, 16)):
        codes = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
        scales = synth.e4m3_rne_bytes(rng.uniform(0.25, 2.0, (rows, K // g)))
        glob = rng.uniform(0.5, 1.5, rows).astype(np.float32)
        got = oracle.dequant_matrix(codes, scales, glob, g)
        assert got.shape == (rows, K)
        assert np.array_equal(got, _dense(codes, scales, glob, g)), (rows, K, g)
    codes = rng.integers(0, 256, (384, 256), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3F  # no NaN codes
    sinv = rng.uniform(0.5, 1.5, (3, 2)).astype(np.float32)
    got = oracle.dequant_fp8_matrix(codes, sinv)
    assert np.array_equal(got, _dense_fp8(codes, sinv))


# ------------------------------------------------------------------ W4A4 (NVFP4 activations)

def pin_nvfp4_code_rounding():
    """e2m1 codes against hand-derived round-to-nearest-even cases (golden), e4m3 codes against
    torch's float8_e4m3fn conversion at every code and at every midpoint between neighbours."""
    for v, want in _golden("e2m1_rounding.json")["cases"]:
        assert oracle.e2m1_code(v) == want, (v, want, oracle.e2m1_code(v))
    vals = _torch_e4m3(np.arange(0x7F, dtype=np.uint8))
    probes = list(vals) + [(vals[i] + vals[i + 1]) / 2 for i in range(0x7E)] + [447.0, 449.0, 470.0]
    ref = torch.tensor(np.minimum(np.array(probes), 448.0), dtype=torch.float32).to(torch.float8_e4m3fn)
    ref_codes = ref.view(torch.uint8).numpy()
    for v, want in zip(probes, ref_codes):
        assert oracle.e4m3_code(float(v)) == int(want), (v, int(want), oracle.e4m3_code(float(v)))


def _nvfp4_values(codes, scales, glob):
    """Test-side decoding of quantized rows (bit-field e2m1, torch e4m3, row scale)."""
    lut = np.array([_e2m1_bitfield(i) for i in range(16)])
    return lut[_nibbles(codes)] * np.repeat(_torch_e4m3(scales), 16, axis=-1) * np.asarray(glob, np.float64)[:, None]


def pin_nvfp4_exact_rows():
    """Rows that NVFP4 represents exactly come back unchanged: row max 2688 (row scale 1),
    each block = e2m1 magnitudes x signs x an e4m3 scale s with one element at 6 s."""
    rng = np.random.default_rng(51)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    svals = _torch_e4m3(np.arange(0x08, 0x7F, dtype=np.uint8))  # normal scales
    rows = []
    for r in range(6):
        blocks = []
        for b in range(8):
            # one block per row has scale 448, so that its 6 x 448 = 2688 makes the row scale 1
            s = 448.0 if b == r % 8 else float(rng.choice(svals[svals <= 448]))
            v = rng.choice(mags, 16) * rng.choice([-1, 1], 16) * s
            v[rng.integers(16)] = 6 * s * rng.choice([-1, 1])
            blocks.append(v)
        rows.append(np.concatenate(blocks))
    x = np.array(rows, np.float32)
    codes, scales, glob = oracle.quant_nvfp4(x)
    assert np.all(glob == 1.0)
    assert np.array_equal(_nvfp4_values(codes, scales, glob), x.astype(np.float64))


def pin_nvfp4_nearest_and_bounds():
    """Random rows: every block scale is the e4m3 value nearest its block max / (6 x row scale),
    every code the e2m1 value nearest x / (scale x row scale) (a brute-force search over the 15
    values; the quantizer multiplies by the rounded reciprocal, so a tie-breaking difference of
    one fp32 rounding is tolerated), and no element moves by more than one e2m1 step."""
    rng = np.random.default_rng(52)
    x = (rng.standard_normal((5, 64)) * np.exp(rng.uniform(-8, 8, (5, 1)))).astype(np.float32)
    x[2, 16:32] = 0.0  # an all-zero block
    codes, scales, glob = oracle.quant_nvfp4(x)
    assert np.allclose(glob, np.abs(x).max(1) / 2688.0, rtol=1e-7)
    svals = _torch_e4m3(np.arange(0x7F, dtype=np.uint8))
    lut = np.array([_e2m1_bitfield(i) for i in range(16)])
    xq = _nvfp4_values(codes, scales, glob)
    for r in range(x.shape[0]):
        for b in range(4):
            blk = x[r, 16 * b:16 * b + 16].astype(np.float64)
            want = np.abs(blk).max() / (6 * float(glob[r]))
            sv = _torch_e4m3(scales[r, b:b + 1])[0]
            assert abs(sv - want) <= np.abs(svals - want).min() * (1 + 1e-6) + 1e-30, (r, b)
            d = sv * float(glob[r])
            for i in range(16):
                if d == 0:
                    assert xq[r, 16 * b + i] == 0
                    continue
                err = abs(xq[r, 16 * b + i] / d - blk[i] / d)
                assert err <= np.abs(lut - blk[i] / d).min() * (1 + 1e-6) + 1e-6, (r, b, i)
                assert abs(xq[r, 16 * b + i] - blk[i]) <= 2 * d * (1 + 1e-6)


def pin_w4a4_forward_composition():
    """The W4A4 forward is the W4A16 chain with NVFP4 activations: quantized x into gate_up,
    SwiGLU, h rounded to fp32 and quantized into down, weighted sum then the shared expert --
    composed here from the separately pinned pieces (quantizer, gate_up, SwiGLU, down)."""
    shape = synth.SHAPES["mini"]
    pieces, sp = _tiny_layer(seed=53, shared=True, shape=shape)
    rb, sb = oracle.slice_bank(pieces, 16), oracle.slice_bank(sp, 16)
    T = 3
    x = synth.make_activations(T, shape.hidden, seed=53)
    ids, w = oracle.route(synth.make_logits(T, shape.num_experts, seed=53), shape.top_k)
    got = oracle.moe_forward(rb, sb, 16, x, ids, w, w4a4=True)
    xf = _bf16_to_f64(x).astype(np.float32)
    c, s_, g = oracle.quant_nvfp4(xf)
    xq = _nvfp4_values(c, s_, g)
    for t in range(T):
        ref = np.zeros(shape.hidden)
        for bank, e, wt in [(rb, int(ids[t, j]), w[t, j]) for j in range(shape.top_k)] + [(sb, 0, 1.0)]:
            h = oracle.swiglu(oracle.expert_gate_up_f64(bank, 16, e, xq[t])).astype(np.float32)
            hc, hs, hg = oracle.quant_nvfp4(h[None, :])
            ref += wt * oracle.expert_down(bank, 16, e, _nvfp4_values(hc, hs, hg)[0])
        assert np.allclose(got[t], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max()), t
    # and it stays within quantization noise of the W4A16 output (a few percent)
    full = oracle.moe_forward(rb, sb, 16, x, ids, w)
    rel = np.linalg.norm(got - full) / np.linalg.norm(full)
    assert 1e-3 < rel < 0.2, rel


PINS = [pin_e2m1, pin_e4m3, pin_dequant_bf16, pin_route_worked_example, pin_route_brute_force,
        pin_route_library, pin_route_ties_and_shift, pin_align, pin_slice_identity_and_tiling,
        pin_one_hot_columns, pin_linear_parts_exact, pin_dense_mlp_special_case,
        pin_routed_combination, pin_untouched_experts_and_tokens, pin_tp_partial_sum,
        pin_router_logits_exact, pin_router_one_hot, pin_asymmetric_partition,
        pin_fp8_slice_identity_and_tiling, pin_fp8_one_hot_columns, pin_fp8_dense_mlp_and_partials,
        pin_dequant_matrices, pin_nvfp4_code_rounding, pin_nvfp4_exact_rows, pin_nvfp4_nearest_and_bounds,
        pin_w4a4_forward_composition]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


@pytest.mark.parametrize("name", sorted(oracle.MUTATIONS))
def test_planted_mistake_is_caught(name):
    """Negative control: each planted oracle mistake makes at least one pin fail."""
    caught = []
    with oracle.mutation(oracle.MUTATIONS[name]):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                caught.append(pin.__name__)
    assert caught, f"mutation {name} escaped every pin"
