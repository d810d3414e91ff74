"""The bench's algorithmic byte and flop counts (the roofline numerators), checked against the
per-expert byte figures of the layer families (CPU only)."""
import importlib.util
import os

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_qwen36_expert_bytes(bench):
    # gate_up: 1024 rows x 1024 code bytes + 1024 x 128 scale bytes + 1024 fp32 globals;
    # down: 2048 rows x 256 code bytes + 2048 x 32 scale bytes + 2048 fp32 globals
    gu, dn = bench._expert_bytes(synth.SHAPES["qwen36"], 512)
    assert (gu, dn) == (1_183_744, 598_016)
    assert gu + dn == 1_781_760


def test_dsv4_expert_bytes(bench):
    # 32-element scale blocks: gate_up 4096 x 2048 + 4096 x 128 + 4096 x 4,
    # down 4096 x 1024 + 4096 x 64 + 4096 x 4
    gu, dn = bench._expert_bytes(synth.SHAPES["dsv4"], 2048)
    assert (gu, dn) == (8_388_608 + 524_288 + 16_384, 4_194_304 + 262_144 + 16_384)
    assert gu + dn == 13_402_112


def test_config_names_the_shape(bench):
    class Args:
        shape, T, layers = "dsv4", 16, 8
    cfg = bench._config(Args)
    assert cfg["workload"] == "dsv4-moe-decode-T16"
    assert (cfg["hidden"], cfg["intermediate"], cfg["group"]) == (4096, 2048, 32)
