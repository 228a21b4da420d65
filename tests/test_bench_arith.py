"""The benchmark's FLOP and byte counts against the worked numbers the pages
print (tests/golden/pages_arithmetic.txt, each line cited there)."""
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def golden():
    vals = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "pages_arithmetic.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (x.strip() for x in line.split("="))
            vals[k] = float(v)
    return vals


@pytest.fixture(scope="module")
def bench():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


@pytest.mark.parametrize("ms,tf", [("day26_flash_attn_v2_median_ms", "day26_flash_attn_v2_tflops"),
                                   ("day26_sdpa_median_ms", "day26_sdpa_tflops"),
                                   ("day26_naive_median_ms", "day26_naive_tflops")])
def test_day26_table_uses_unhalved_count(bench, ms, tf):
    g = golden()
    full = bench.attn_flops(g["day26_B"], g["day26_H"], g["day26_S"], g["day26_D"], causal=False)
    assert full / (g[ms] * 1e-3) / 1e12 == pytest.approx(g[tf], rel=0.01)
    # the causal convention this benchmark reports is exactly half of it
    half = bench.attn_flops(g["day26_B"], g["day26_H"], g["day26_S"], g["day26_D"], causal=True)
    assert half == full / 2


def test_kwkr_memory_arithmetic():
    g = golden()
    B, H, N, D = g["kwkr_B"], g["kwkr_H"], g["kwkr_N"], g["kwkr_D"]
    assert 4 * B * H * N * D * 2 / 1e6 == pytest.approx(g["kwkr_qkvo_total_mb"], rel=0.01)
    assert B * H * N * N / 1e9 == pytest.approx(g["kwkr_s_elements_billion"], rel=0.01)
    assert B * H * N * N * 2 / 1e9 == pytest.approx(g["kwkr_s_gb"], rel=0.03)
    assert B * H * (2 * N) ** 2 * 2 / 1e9 == pytest.approx(g["kwkr_s_gb_at_4096"], rel=0.01)


def test_chain_bytes(bench):
    """Residual traffic of the 4-layer block: kept (j <= i) fp32 logits are
    written by layers 0-2 and read by layers 1-3."""
    W = bench.EXTRA_WORKLOADS["residual_chain"]
    kept = W["N"] * (W["N"] + 1) // 2 * W["Hq"] * 4
    io = bench.chain_layer_bytes(W, 0) - kept
    assert [bench.chain_layer_bytes(W, i) - io for i in range(4)] == [kept, 2 * kept, 2 * kept, kept]
    assert 6 * kept / 1e9 == pytest.approx(4.03, rel=0.01)


def test_window_counts_reduce_to_causal():
    """A window of at least N keys is the causal mask: same FLOPs, same tile
    pairs; W = 128 on two tiles touches (0,0), (1,0), (1,1)."""
    import bench
    assert bench.attn_flops(1, 2, 1024, 64, True, 1024) == bench.attn_flops(1, 2, 1024, 64, True)
    assert bench.tile_pairs(1, 2, 1024, True, 4096) == bench.tile_pairs(1, 2, 1024, True)
    assert bench.tile_pairs(1, 1, 256, True, 128) == 3
    assert bench.tile_pairs(1, 1, 256, True, 1) == 2
    # W keys per row once i >= W: N*W - W^2/2 pairs in the continuous count
    assert bench.attn_flops(1, 1, 1000, 1, True, 100) == 4.0 * (1000 * 100 - 100 * 100 / 2)
