"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Integer stages (router ids, align order, pack bytes, dequantised bf16 values) must be
bit-exact; floating outputs must reach relative L2 error <= 1e-2 and max-abs error
<= 3e-2 x RMS of the oracle output; routing weights agree to 1e-6 relative.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_cases import ROUTE_W_RTOL, GpuLayer, assert_close, hot_block_sample, logits_for, oracle_banks, pieces

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_quantized_moe_gb300 import build
    build.build()
    import nvfp4_quantized_moe_gb300 as ft
    ft.load()


@pytest.fixture(scope="module")
def ft():
    import nvfp4_quantized_moe_gb300 as ft
    return ft


_layers = {}


def layer(name, tp_rank=0, tp_size=1, shard=None, shared_shard=None):
    key = (name, tp_rank, tp_size, shard, shared_shard)
    if key not in _layers:
        if len(_layers) > 6:
            _layers.clear()
            torch.cuda.empty_cache()
        _layers[key] = GpuLayer(name, tp_rank, tp_size, shard=shard, shared_shard=shared_shard)
    return _layers[key]


# ------------------------------------------------------------------ dequant (bit-exact)

def test_dequant_all_code_scale_pairs(ft):
    """Every (e2m1 code, e4m3 scale byte) pair through the kernels' dequant routine."""
    shape = synth.LayerShape(hidden=256, intermediate=64, num_experts=1, top_k=1)
    cfg = ft.MoEConfig.of(shape)
    rows, K, g = 128, 256, 16
    nib = np.arange(16, dtype=np.uint8)
    group_bytes = (nib[1::2] << 4 | nib[0::2]).astype(np.uint8)          # elements 0..15 = codes 0..15
    gu = np.tile(group_bytes, (rows, K // 16))
    sc = (np.arange(rows * (K // g)) % 256).astype(np.uint8).reshape(rows, K // g)
    banks = ft.alloc_banks(cfg, 0)
    banks[0].copy_(torch.from_numpy(gu.reshape(1, rows, K // 2)))
    banks[1].copy_(torch.from_numpy(sc.reshape(1, rows, K // g)))
    for b in banks[2:]:
        b.zero_()
    out = torch.empty((rows, K), dtype=torch.bfloat16, device="cuda")
    ft.ft_moe_dequant(cfg, 0, banks, ft.FT_GU, 0, out)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    checked = 0
    for n in range(rows):
        for kk in range(K):
            s = int(sc[n, kk // g])
            if s in (0x7F, 0xFF):
                continue
            assert got[n, kk] == oracle.dequant_bf16(kk % 16, s), (n, kk, s)
            checked += 1
    assert checked == rows * K - 2 * 8 * 16


def test_dequant_real_bank_matches_oracle(ft):
    L = layer("qwen36")
    rb, _ = oracle_banks("qwen36")
    for which, e in ((ft.FT_GU, 0), (ft.FT_GU, 255), (ft.FT_DN, 17)):
        rows, K = (1024, 2048) if which == ft.FT_GU else (2048, 512)
        out = torch.empty((rows, K), dtype=torch.bfloat16, device="cuda")
        ft.ft_moe_dequant(L.cfg, 0, L.routed, which, e, out)
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        codes = rb["gu"][e] if which == ft.FT_GU else rb["dn"][e]
        sc = rb["gu_scale"][e] if which == ft.FT_GU else rb["dn_scale"][e]
        ref = oracle.dequant_matrix(codes, sc, np.ones(rows, np.float32), 16)
        gotf = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.array_equal(gotf, ref)


# ------------------------------------------------------------------ pack (bit-exact)

@pytest.mark.parametrize("name,tp", [("tiny", 1), ("tiny", 2), ("tiny", 4), ("qwen36", 2)])
@pytest.mark.parametrize("from_host", [True, False])
def test_pack_matches_oracle_slicer(ft, name, tp, from_host):
    shape = synth.SHAPES[name]
    routed, shared = pieces(name)
    for r in range(tp):
        L = GpuLayer(name, r, tp, from_host=from_host)
        rb, sb = oracle_banks(name, r, tp)
        for i, key in enumerate(("gu", "gu_scale", "gu_global", "dn", "dn_scale", "dn_global")):
            assert np.array_equal(L.routed[i].cpu().numpy(), rb[key]), (key, r)
            if shared is not None:
                assert np.array_equal(L.shared[i].cpu().numpy(), sb[key]), (key, r)
        # banks own their storage
        assert all(b.untyped_storage().data_ptr() != 0 for b in L.routed)
    del shape


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("T,E,k,zipf", [(16, 8, 2, False), (1, 256, 8, False), (64, 256, 8, False),
                                        (2048, 256, 8, True), (37, 1024, 32, True), (5, 33, 3, False),
                                        (3, 32, 32, False)])
def test_route_matches_oracle(ft, T, E, k, zipf):
    logits = synth.zipf_logits(T, E, seed=T) if zipf else synth.make_logits(T, E, seed=T)
    lg = torch.from_numpy(logits).cuda()
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ft.ft_moe_route(lg, k, ids, w)
    ref_ids, ref_w = oracle.route(logits, k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy().astype(np.float64), ref_w, rtol=ROUTE_W_RTOL, atol=0)


def test_route_ties_go_to_lower_index(ft):
    logits = np.zeros((4, 64), np.float32)
    logits[1, ::3] = 2.0
    logits[2, [5, 9, 40]] = 1.0
    lg = torch.from_numpy(logits).cuda()
    ids = torch.empty((4, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((4, 8), dtype=torch.float32, device="cuda")
    ft.ft_moe_route(lg, 8, ids, w)
    ref_ids, ref_w = oracle.route(logits, 8)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=ROUTE_W_RTOL)


# ------------------------------------------------------------------ align (bit-exact)

@pytest.mark.parametrize("T,E,k,B,zipf", [(16, 8, 2, 8, False), (1, 256, 8, 8, False), (64, 256, 8, 8, False),
                                          (1024, 256, 8, 16, True), (2048, 256, 8, 8, True),
                                          (8192, 256, 8, 128, True), (3000, 1024, 8, 64, True),
                                          (7, 5, 3, 1, False)])
def test_align_matches_oracle(ft, T, E, k, B, zipf):
    logits = synth.zipf_logits(T, E, seed=1) if zipf else synth.make_logits(T, E, seed=1)
    ids_np, _ = oracle.route(logits, k)
    ids = torch.from_numpy(ids_np).cuda()
    cap = T * k + min(E, T * k) * (B - 1)
    sorted_slot = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    block_expert = torch.full((cap // B + 1,), -7, dtype=torch.int32, device="cuda")
    expert_off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    n_padded = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(ft.ft_moe_align_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    ft.ft_moe_align(ids, E, B, sorted_slot, block_expert, expert_off, n_padded, ws)
    assert ft.ft_moe_read_status(ws) == 0
    ref_sorted, ref_block, ref_off, ref_n = oracle.align(ids_np, E, B)
    n = int(n_padded.item())
    assert n == ref_n
    assert np.array_equal(sorted_slot[:n].cpu().numpy(), ref_sorted)
    assert np.array_equal(block_expert[:n // B].cpu().numpy(), ref_block)
    assert np.array_equal(expert_off.cpu().numpy(), ref_off)


@pytest.mark.parametrize("T,E,H", [(1, 256, 2048), (33, 256, 2048), (64, 256, 2048), (2048, 256, 2048),
                                   (16, 8, 256), (5, 40, 64), (16, 256, 4096)])
def test_route_gemm_matches_oracle(ft, T, E, H):
    """Router logit GEMM + top-k. Logits: within the fp32 summation bound H * 2^-23 * sum|x*w|
    of the oracle's fp64 logits. Top-k: bit-exact with the oracle routing the GPU's own fp32
    logits; against the fp64 logits the selected set may differ only where the boundary
    logits lie within that bound of each other (either choice is then a valid top-k)."""
    k = min(8, E)
    x_bits = synth.make_activations(T, H, seed=31)
    w_bits = synth.make_router_weights(E, H, seed=31)
    x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    wr = torch.from_numpy(w_bits.view(np.int16)).cuda().view(torch.bfloat16)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ft.ft_moe_route_gemm(x, wr, k, logits, ids, w)
    got = logits.cpu().numpy().astype(np.float64)
    ref, absum = oracle.router_logits(x_bits, w_bits)
    bound = H * 2.0 ** -23 * absum
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / np.maximum(absum, 1e-30)))
    own_ids, own_w = oracle.route(logits.cpu().numpy(), k)
    got_ids = ids.cpu().numpy()
    assert np.array_equal(got_ids, own_ids)
    assert np.allclose(w.cpu().numpy(), own_w, rtol=ROUTE_W_RTOL, atol=0)
    ref_ids, _ = oracle.route(ref.astype(np.float32), k)
    for t in np.nonzero(np.any(np.sort(got_ids, 1) != np.sort(ref_ids, 1), axis=1))[0]:
        kth = np.sort(ref[t])[::-1][k - 1]
        assert np.all(ref[t][got_ids[t]] >= kth - 2 * bound[t][got_ids[t]]), f"token {t}: not a valid top-{k}"


def test_align_flags_invalid_ids(ft):
    ids = torch.tensor([[0, 1], [2, 9], [3, 3]], dtype=torch.int32, device="cuda")
    E, B = 8, 4
    cap = 6 + 6 * (B - 1)
    bufs = [torch.empty(cap, dtype=torch.int32, device="cuda"), torch.empty(cap, dtype=torch.int32, device="cuda"),
            torch.empty(E + 1, dtype=torch.int32, device="cuda"), torch.empty(1, dtype=torch.int32, device="cuda")]
    ws = torch.empty(ft.ft_moe_align_workspace_size(3, 2, E), dtype=torch.uint8, device="cuda")
    ft.ft_moe_align(ids, E, B, *bufs, ws)
    assert ft.ft_moe_read_status(ws) == 6      # FT_ERR_INVALID_ROUTING
    # the out-of-range slot (expert 9) is skipped, the rest are placed
    n = int(bufs[3].item())
    placed = sorted(v for v in bufs[0][:n].cpu().tolist() if v < 6)
    assert placed == [0, 1, 2, 4, 5]


# ------------------------------------------------------------------ forward

def _run_and_compare(name, T, zipf, tp_rank=0, tp_size=1, sample=None, out_dtype=torch.float32, shard=None,
                     shared_shard=None):
    L = layer(name, tp_rank, tp_size, shard, shared_shard)
    shape = synth.SHAPES[name]
    logits = logits_for(name, T, zipf)
    x = synth.make_activations(T, shape.hidden)
    ids, w = L.route(logits)
    out, _ = L.forward(x, ids, w, out_dtype=out_dtype)
    ref_ids, ref_w = oracle.route(logits, shape.top_k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    rb, sb = oracle_banks(name, tp_rank, tp_size, shard=shard, shared_shard=shared_shard)
    tokens = np.arange(T) if sample is None else sample
    ref = oracle.moe_forward(rb, sb, shape.group, x, ref_ids, ref_w, tokens=tokens,
                             nthreads=oracle.default_threads())
    got = out.float().cpu().numpy()[tokens]
    return got, ref


@pytest.mark.parametrize("tp", [1, 2])
def test_forward_tiny(tp):
    for r in range(tp):
        got, ref = _run_and_compare("tiny", 16, False, r, tp)
        assert_close(got, ref, f"tiny tp={tp} rank={r}")


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_forward_qwen36_decode(T):
    got, ref = _run_and_compare("qwen36", T, False)
    assert_close(got, ref, f"qwen36 decode T={T}")


@pytest.mark.parametrize("T", [1, 64, 200])
def test_forward_odd_hidden_decode(T):
    """H = 640: the down stage's 256-row units of a block end half out of range (at T=64 and
    200 the down launch streams block runs of units, whose warps then stop early)."""
    got, ref = _run_and_compare("odd_h", T, False)
    assert_close(got, ref, f"odd_h decode T={T}")


def test_forward_bf16_output():
    got, ref = _run_and_compare("qwen36", 8, False, out_dtype=torch.bfloat16)
    assert_close(got, ref, "bf16 out")


@pytest.mark.parametrize("T,tp,zipf", [(256, 1, False), (1000, 1, True), (384, 2, True), (256, 1, True)])
def test_forward_mini_tensor_core_path(T, tp, zipf):
    """Every token against the oracle on a layer small enough for it (tensor-core path:
    T * k >= 32 * E and 128-row tiles)."""
    for r in range(tp):
        got, ref = _run_and_compare("mini", T, zipf, r, tp)
        assert_close(got, ref, f"mini T={T} tp={tp} rank={r}")


_oracle_cache = {}


def _oracle_full(name, T, zipf, tokens):
    """The oracle's tp = 1 output for these tokens (cached: several tests sum partials
    against it)."""
    key = (name, T, zipf, tokens.tobytes())
    if key not in _oracle_cache:
        shape = synth.SHAPES[name]
        ids, w = oracle.route(logits_for(name, T, zipf), shape.top_k)
        rb, sb = oracle_banks(name)
        x = synth.make_activations(T, shape.hidden)
        _oracle_cache.clear()
        _oracle_cache[key] = oracle.moe_forward(rb, sb, shape.group, x, ids, w, tokens=tokens,
                                                nthreads=oracle.default_threads())
    return _oracle_cache[key]


def _hot_sample(name, T, n=512):
    shape = synth.SHAPES[name]
    ids, _ = oracle.route(logits_for(name, T, True), shape.top_k)
    return hot_block_sample(ids, shape.num_experts, n, seed=T)


def test_forward_qwen36_prefill_every_token():
    """T = 2048 (tensor-core path, Zipf routing): every token against the oracle."""
    T = 2048
    got, ref = _run_and_compare("qwen36", T, True)
    assert_close(got, ref, f"qwen36 prefill T={T}")


def test_forward_qwen36_prefill_hot_blocks():
    """T = 8192: at least 512 tokens, with one in every 128-position block of the three
    most loaded experts (each such block is a separate tensor-core unit)."""
    T = 8192
    sample = _hot_sample("qwen36", T)
    assert len(sample) >= 512
    got, ref = _run_and_compare("qwen36", T, True, sample=sample)
    assert_close(got, ref, f"qwen36 prefill T={T}")


@pytest.mark.parametrize("tp,T,zipf", [(2, 32, False), (4, 32, False), (2, 2048, True), (4, 2048, True)])
def test_forward_tp_partials_sum_to_full(tp, T, zipf):
    """Each rank-local partial matches the oracle's on every token; their host sum
    matches the tp=1 output."""
    sample = np.arange(T, dtype=np.int32)
    total = 0
    for r in range(tp):
        got, ref = _run_and_compare("qwen36", T, zipf, r, tp, sample=sample)
        assert_close(got, ref, f"rank {r}/{tp}")
        total = total + got.astype(np.float64)
    assert_close(total, _oracle_full("qwen36", T, zipf, sample), f"sum of {tp} partials vs tp=1")


# Two ranks with unequal shares of the intermediate dimension (routed 320 + 192 of 512,
# shared 192 + 320 of 512): every range is whole scale blocks, and 320 / 192 are not
# multiples of the tensor-core path's 128-row tiles, so both paths see ragged K and N.
ASYM = [((0, 320), (0, 192)), ((320, 192), (192, 320))]


def test_pack_explicit_shard_matches_oracle_slicer(ft):
    for shard, shared_shard in ASYM:
        L = GpuLayer("qwen36", shard=shard, shared_shard=shared_shard)
        rb, sb = oracle_banks("qwen36", shard=shard, shared_shard=shared_shard)
        for i, key in enumerate(("gu", "gu_scale", "gu_global", "dn", "dn_scale", "dn_global")):
            assert np.array_equal(L.routed[i].cpu().numpy(), rb[key]), (key, shard)
            assert np.array_equal(L.shared[i].cpu().numpy(), sb[key]), (key, shared_shard)


@pytest.mark.parametrize("T,zipf", [(1, False), (32, False), (2048, True)])
def test_forward_asymmetric_shards_sum_to_full(T, zipf):
    """Partials over unequal ranges match the oracle's and add up to the unsharded output."""
    shape = synth.SHAPES["qwen36"]
    sample = np.arange(T) if T <= 64 else np.sort(np.random.default_rng(7).choice(T, 16, replace=False))
    total = 0
    for shard, shared_shard in ASYM:
        got, ref = _run_and_compare("qwen36", T, zipf, sample=sample, shard=shard, shared_shard=shared_shard)
        assert_close(got, ref, f"shard {shard} shared {shared_shard}")
        total = total + got.astype(np.float64)
    logits = logits_for("qwen36", T, zipf)
    ids, w = oracle.route(logits, shape.top_k)
    rb, sb = oracle_banks("qwen36")
    x = synth.make_activations(T, shape.hidden)
    full = oracle.moe_forward(rb, sb, shape.group, x, ids, w, tokens=sample, nthreads=oracle.default_threads())
    assert_close(total, full, "sum of asymmetric partials vs unsharded")


@pytest.mark.parametrize("T,tp", [(1, 1), (16, 1), (1, 4), (16, 4)])
def test_forward_dsv4_group32(T, tp):
    for r in range(tp) if T == 1 else [0, tp - 1]:
        got, ref = _run_and_compare("dsv4", T, True, r, tp)
        assert_close(got, ref, f"dsv4 T={T} tp={tp} rank={r}")


@pytest.mark.parametrize("tp", [1, 4])
def test_forward_dsv4_prefill_hot_blocks(tp):
    """dsv4 T = 4096 (g = 32): at least 512 tokens covering every 128-position block of the
    three most loaded experts; at tp = 4 every rank against the oracle and the sum of
    the partials against the tp = 1 output."""
    T = 4096
    sample = _hot_sample("dsv4", T)
    assert len(sample) >= 512
    total = 0
    for r in range(tp):
        got, ref = _run_and_compare("dsv4", T, True, r, tp, sample=sample)
        assert_close(got, ref, f"dsv4 T={T} tp={tp} rank={r}")
        total = total + got.astype(np.float64)
    if tp > 1:
        assert_close(total, _oracle_full("dsv4", T, True, sample), f"dsv4 sum of {tp} partials vs tp=1")


def _scale_rows_bf16(x_bits: np.ndarray, exps) -> np.ndarray:
    """Rows of bf16 bit patterns times 2**e (exact: power of two, no overflow); e=None
    zeroes the row."""
    f = (x_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t, e in enumerate(exps):
        f[t] = 0.0 if e is None else np.ldexp(f[t], e)
    return (f.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("T", [16, 256])
def test_forward_rows_of_mixed_magnitude(T):
    """Token rows 2^-40 .. 2^40 apart and all-zero rows, on the warp-MMA path (T=16) and
    the tensor-core path (T=256): both stage each activation row with its own
    power-of-two scale, so every row keeps its own relative accuracy."""
    L = layer("mini")
    shape = synth.SHAPES["mini"]
    cycle = [0, 40, -40, None, 17, -23]
    x = _scale_rows_bf16(synth.make_activations(T, shape.hidden, seed=11), [cycle[t % 6] for t in range(T)])
    logits = logits_for("mini", T, False, seed=11)
    ids, w = L.route(logits)
    out, _ = L.forward(x, ids, w)
    ref_ids, ref_w = oracle.route(logits, shape.top_k)
    rb, sb = oracle_banks("mini")
    ref = oracle.moe_forward(rb, sb, shape.group, x, ref_ids, ref_w, nthreads=oracle.default_threads())
    got = out.cpu().numpy()
    for t in range(T):
        if cycle[t % 6] is None:
            assert not got[t].any(), f"token {t}: zero row gives nonzero output"
        else:
            assert_close(got[t], ref[t], f"token {t} (row scale 2^{cycle[t % 6]})")


def test_forward_deterministic_and_untouched_experts():
    L = layer("qwen36")
    x = synth.make_activations(32, 2048, seed=3)
    ids, w = L.route(logits_for("qwen36", 32, False, seed=3))
    a, _ = L.forward(x, ids, w)
    b, _ = L.forward(x, ids, w)
    assert torch.equal(a, b)
    # scribble over an expert nobody uses: bitwise-identical output
    used = set(ids.cpu().numpy().reshape(-1).tolist())
    free = next(e for e in range(256) if e not in used)
    saved = [t[free].clone() for t in L.routed]
    for t in L.routed:
        t[free].copy_(torch.randint_like(t[free], 0, 100) if t.dtype == torch.uint8 else torch.rand_like(t[free]))
    c, _ = L.forward(x, ids, w)
    for t, s in zip(L.routed, saved):
        t[free].copy_(s)
    assert torch.equal(a, c)


def test_forward_invalid_ids_flagged():
    L = layer("tiny")
    x = synth.make_activations(4, 256)
    ids = torch.tensor([[0, 1], [2, 2], [3, 4], [5, 6]], dtype=torch.int32, device="cuda")
    w = torch.full((4, 2), 0.5, device="cuda")
    _, st = L.forward(x, ids, w, check_status=False)
    assert st == 6


def test_forward_in_cuda_graph():
    L = layer("qwen36")
    T = 8
    x_bits = synth.make_activations(T, 2048, seed=9)
    logits = torch.from_numpy(logits_for("qwen36", T, False, seed=9)).cuda()
    x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.empty((T, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 8), dtype=torch.float32, device="cuda")
    out = torch.empty((T, 2048), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.ft.ft_moe_workspace_size(L.cfg, T), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        L.ft.ft_moe_route(logits, 8, ids, w)
        L.ft.ft_moe_forward(L.cfg, L.routed, L.shared, x, ids, w, out, ws)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.ft.ft_moe_route(logits, 8, ids, w)
        L.ft.ft_moe_forward(L.cfg, L.routed, L.shared, x, ids, w, out, ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


def test_tensor_core_path_deterministic_and_graph_replay():
    """T = 2048 runs the tensor-core kernels: two eager runs are bitwise identical, and a
    CUDA-graph replay of route + forward reproduces the eager output bit for bit."""
    L = layer("qwen36")
    T, H = 2048, 2048
    x_bits = synth.make_activations(T, H, seed=13)
    logits = torch.from_numpy(logits_for("qwen36", T, True, seed=13)).cuda()
    x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.empty((T, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 8), dtype=torch.float32, device="cuda")
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = torch.full((L.ft.ft_moe_workspace_size(L.cfg, T),), 0xFF, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    runs = []
    with torch.cuda.stream(s):
        for _ in range(2):
            L.ft.ft_moe_route(logits, 8, ids, w)
            L.ft.ft_moe_forward(L.cfg, L.routed, L.shared, x, ids, w, out, ws)
            runs.append(out.clone())
    torch.cuda.synchronize()
    assert L.ft.ft_moe_read_status(ws) == 0
    assert torch.equal(runs[0], runs[1])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.ft.ft_moe_route(logits, 8, ids, w)
        L.ft.ft_moe_forward(L.cfg, L.routed, L.shared, x, ids, w, out, ws)
    out.zero_()
    ws.fill_(0xFF)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, runs[0])
