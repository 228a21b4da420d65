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


def test_median_p90_min(bench):
    """The pages' bench template reports median, p90 and min of the timed
    iterations; p90 by nearest rank."""
    st = bench.pct_stats([float(x) for x in range(10, 0, -1)])
    assert st == {"median": 5.5, "p90": 9.0, "min": 1.0}
    assert bench.pct_stats([2.0]) == {"median": 2.0, "p90": 2.0, "min": 2.0}


def test_profile_summary_is_read_only_at_its_own_digest(bench, tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k_x.md").write_text(
        "source_digest: abc123\ndram_bytes_per_launch: 1000\nunits_per_launch: 10\n"
        "tensor_pipe_active_pct: 61.5\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.profiled("k_x", "abc123", 40)
    assert p["traffic"] == 4000 and p["tensor_pipe_active_pct"] == 61.5
    assert "scaled" in p["traffic_basis"]
    assert bench.profiled("k_x", "abc123", 10)["traffic_basis"] == "measured at this size"
    assert bench.profiled("k_x", "ffffff", 10) == {}     # kernel changed since the capture
    assert bench.profiled("missing", "abc123", 10) == {}


def test_both_arms_print_the_same_config(bench):
    W = bench.WORKLOAD
    a = bench.line_config(W, 1, bench.wants_flush("auto", bench.workload_bytes(W)),
                          bench.workload_bytes(W))
    assert a["workload"] == W["name"] and a["step"] == "forward + backward"
    assert a["l2"].startswith("no flush")
