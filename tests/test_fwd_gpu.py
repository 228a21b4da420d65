"""GPU parity of the forward pass (C ABI) against the fp64 oracle, element by
element on shapes spanning several tiles and a ragged tail, and on sampled
rows at the full workload sizes."""
import math

import numpy as np
import pytest

from helpers import (check_lse, check_o, make_qkv, sample_rows, to_oracle)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tiled_attention_02_gb300 as ta
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ta.build()
    return ta


def run_fwd(ta, x, causal, scale=None, **kw):
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = ta.attn_fwd(q, k, v, scale=scale, causal=causal, **kw)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    return o, lse


def oracle_fwd(orc, x, causal, scale, rows=None):
    return orc.forward(to_oracle(x["q"]), to_oracle(x["k"]), to_oracle(x["v"]), scale=scale,
                       causal=causal, rows=rows)


def test_tiny_config(ta, orc):
    """B=1, H=1, N=128, D=64, non-causal, scale 1/8."""
    x = make_qkv(1, 1, 1, 128, 64, seed=0)
    o, lse = run_fwd(ta, x, causal=False)
    ref = oracle_fwd(orc, x, False, 1 / 8)
    check_o(o, ref["o"], "tiny")
    check_lse(lse, ref["lse"], "tiny")


SHAPES = [
    # B, Hq, Hkv, N
    (1, 2, 2, 384),     # several tiles
    (2, 4, 2, 256),     # GQA
    (1, 3, 1, 200),     # ragged tail, GQA 3:1
    (1, 1, 1, 1),       # single row
    (1, 2, 2, 129),     # one row past a tile
    (1, 1, 1, 1000),    # unaligned length from the kwkr.cn test matrix (4.3)
]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}H{s[1]}kv{s[2]}N{s[3]}" for s in SHAPES])
def test_parity_small(ta, orc, D, causal, shape):
    _parity(ta, orc, D, causal, shape)


# Head dims 80 and 96: rows padded to two 128-byte swizzle atoms in shared
# memory (zero-filled by TMA past D), stores clipped at D.
SHAPES_ODD_D = [(1, 2, 2, 384), (1, 3, 1, 200), (2, 2, 1, 129), (1, 1, 1, 1)]


@pytest.mark.parametrize("D", [80, 96])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES_ODD_D,
                         ids=[f"B{s[0]}H{s[1]}kv{s[2]}N{s[3]}" for s in SHAPES_ODD_D])
def test_parity_head_dim_80_96(ta, orc, D, causal, shape):
    _parity(ta, orc, D, causal, shape)


def _parity(ta, orc, D, causal, shape):
    B, Hq, Hkv, N = shape
    x = make_qkv(B, Hq, Hkv, N, D, seed=N + D)
    o, lse = run_fwd(ta, x, causal=causal)
    ref = oracle_fwd(orc, x, causal, 1 / math.sqrt(D))
    check_o(o, ref["o"], f"{shape} D{D} causal{causal}")
    check_lse(lse, ref["lse"], f"{shape} D{D} causal{causal}")


def test_nondefault_scale_and_no_lse(ta, orc):
    x = make_qkv(1, 2, 1, 300, 128, seed=7)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = ta.attn_fwd(q, k, v, scale=0.3, causal=True, want_lse=False)
    torch.cuda.synchronize()
    assert lse is None
    ref = oracle_fwd(orc, x, True, 0.3)
    check_o(o, ref["o"], "scale 0.3")


def test_every_output_written(ta, orc):
    """Outputs pre-filled with NaN must be fully overwritten (no tile missed)."""
    x = make_qkv(2, 3, 3, 333, 64, seed=3)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((2, 3, 333), float("nan"), device="cuda")
    ta.attn_fwd(q, k, v, causal=True, o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_deterministic(ta):
    x = make_qkv(1, 4, 2, 512, 128, seed=11)
    o1, l1 = run_fwd(ta, x, causal=True)
    o2, l2 = run_fwd(ta, x, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_causal_first_row_equals_first_value_row(ta):
    """Closed form on the GPU side too: causal row 0 attends only key 0."""
    x = make_qkv(1, 2, 2, 256, 128, seed=5)
    o, _ = run_fwd(ta, x, causal=True)
    assert torch.equal(o[:, :, 0].cpu(), x["v"][:, :, 0])


# ------------------------------------------------------ full-size workloads

FULL = [
    # name, B, Hq, Hkv, N, D, causal
    ("noncausal_8x32x2048x128", 8, 32, 32, 2048, 128, False),
    ("causal_2x16x4096x64", 2, 16, 16, 4096, 64, True),
    ("causal_1x16x16384x128", 1, 16, 16, 16384, 128, True),
]


@pytest.mark.parametrize("name,B,Hq,Hkv,N,D,causal", FULL, ids=[f[0] for f in FULL])
def test_parity_full_size_sampled(ta, orc, name, B, Hq, Hkv, N, D, causal):
    x = make_qkv(B, Hq, Hkv, N, D, seed=0)
    o, lse = run_fwd(ta, x, causal=causal)
    rows = sample_rows(B, Hq, N, 768, seed=1)
    ref = oracle_fwd(orc, x, causal, 1 / math.sqrt(D), rows=rows)
    check_o(o.reshape(-1, D)[torch.from_numpy(rows).cuda()], ref["o"], name)
    check_lse(lse.reshape(-1)[torch.from_numpy(rows).cuda()], ref["lse"], name)
    # properties at every row: finite, and LSE within its bounds
    # (max logit <= LSE <= max logit + ln |J_i|, so LSE <= |s|_max + ln N)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


# Rows of 64 key tiles or more take the variant whose K and V tiles share
# one stage ring (D >= 80; D = 64 always does): both sides of the threshold,
# ragged, causal and not, grouped heads, every head dim the variant has.
MERGE_EDGE = [
    # B, Hq, Hkv, N, D, causal
    (1, 4, 2, 8063, 128, True),    # 63 key tiles: separate K and V rings
    (1, 4, 2, 8065, 128, True),    # 64 key tiles, the last ragged: merged
    (1, 3, 3, 8192 + 37, 96, False),
    (1, 2, 1, 9000, 80, True),
]


@pytest.mark.parametrize("case", MERGE_EDGE,
                         ids=[f"B{c[0]}H{c[1]}kv{c[2]}N{c[3]}D{c[4]}{'c' if c[5] else 'nc'}"
                              for c in MERGE_EDGE])
def test_parity_merged_kv_stages(ta, orc, case):
    B, Hq, Hkv, N, D, causal = case
    x = make_qkv(B, Hq, Hkv, N, D, seed=7)
    o, lse = run_fwd(ta, x, causal=causal)
    rows = np.unique(np.concatenate([sample_rows(B, Hq, N, 160, seed=8),
                                     [0, N - 1, N - 128, B * Hq * N - 1]]))
    ref = oracle_fwd(orc, x, causal, 1 / math.sqrt(D), rows=rows)
    name = f"N={N} D={D} causal={causal}"
    check_o(o.reshape(-1, D)[torch.from_numpy(rows).cuda()], ref["o"], name)
    check_lse(lse.reshape(-1)[torch.from_numpy(rows).cuda()], ref["lse"], name)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


# More (query tile, head) items than SMs, so that the plain forward's
# persistent blocks each walk several items (the rings, S/P buffers and output
# buffers continue across item boundaries), with a ragged last tile, grouped
# heads, odd head dims and a sliding window.  Outputs start as NaN: every item
# of every block must be written.
MULTI_ITEM = [
    # B, Hq, Hkv, N, D, causal, window
    (3, 24, 8, 1000, 128, True, None),
    (3, 24, 8, 1000, 80, False, None),
    (2, 40, 40, 700, 64, True, None),
    (2, 48, 16, 1500, 96, True, 300),
]


@pytest.mark.parametrize("case", MULTI_ITEM,
                         ids=[f"B{c[0]}H{c[1]}kv{c[2]}N{c[3]}D{c[4]}{'c' if c[5] else 'nc'}"
                              f"{'W' + str(c[6]) if c[6] else ''}" for c in MULTI_ITEM])
def test_parity_more_items_than_sms(ta, orc, case):
    B, Hq, Hkv, N, D, causal, window = case
    n_items = B * Hq * ((N + 127) // 128)
    assert n_items > torch.cuda.get_device_properties(0).multi_processor_count
    x = make_qkv(B, Hq, Hkv, N, D, seed=B * N + D)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, N), float("nan"), device="cuda")
    ta.attn_fwd(q, k, v, causal=causal, o=o, lse=lse, window=window)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    ref = orc.forward(to_oracle(x["q"]), to_oracle(x["k"]), to_oracle(x["v"]),
                      scale=1 / math.sqrt(D), causal=causal, window=window)
    check_o(o, ref["o"], f"{case}")
    check_lse(lse, ref["lse"], f"{case}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_parity_growing_row_max(ta, orc, D, causal):
    """Keys ramped by position: a row's logits grow by about 8 (natural units,
    11.5 in log2) per 128-key tile, so each new tile raises the row max past
    the lazy-rescale threshold and the running output is rescaled at every
    tile, on top of the score MMAs running ahead of the PV MMAs."""
    B, H, N = 2, 3, 1000
    x = make_qkv(B, H, H, N, D, seed=11)
    c = 8.0 / math.sqrt(D)   # scale * D * c / 128 = 8 / 128 per key
    ramp = (torch.arange(N, dtype=torch.float32) / 128.0).view(1, 1, N, 1)
    x["q"] = (1.0 + 0.25 * x["q"].float()).to(torch.bfloat16)
    x["k"] = (c * ramp + 0.25 * x["k"].float()).to(torch.bfloat16)
    o, lse = run_fwd(ta, x, causal=causal)
    ref = oracle_fwd(orc, x, causal, 1 / math.sqrt(D))
    assert float(ref["lse"].max()) > 40.0   # the growth is really there
    check_o(o, ref["o"], f"growing max D{D} causal={causal}")
    check_lse(lse, ref["lse"], f"growing max D{D} causal={causal}")


def test_causal_head_chunked_order(ta, orc):
    """Causal items in chunks of heads (all heads' K/V well over twice the
    L2): B=2, H=32, N=16384, D=128 runs its 64 heads in chunks of about half
    the L2, the last chunk smaller.  Heads are independent problems, so every
    row must equal, bit for bit, a launch on that head alone (one chunk, the
    plain order); sampled rows are checked against the oracle."""
    B, H, N, D = 2, 32, 16384, 128
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    assert B * H * N * D * 4 > 2 * l2, "shape must take the head-chunked order"
    x = make_qkv(B, H, H, N, D, seed=7)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    ta.attn_fwd(q, k, v, causal=True, o=o, lse=lse)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    for b in range(B):
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            o1, lse1 = ta.attn_fwd(q[sl].contiguous(), k[sl].contiguous(), v[sl].contiguous(),
                                   causal=True)
            assert torch.equal(o[sl], o1), f"O of head ({b}, {h})"
            assert torch.equal(lse[sl], lse1), f"LSE of head ({b}, {h})"
    rows = sample_rows(B, H, N, 256, seed=8)
    ref = oracle_fwd(orc, x, True, 1 / math.sqrt(D), rows=rows)
    r = torch.from_numpy(rows).cuda()
    check_o(o.reshape(-1, D)[r], ref["o"], "head-chunked causal")
    check_lse(lse.reshape(-1)[r], ref["lse"], "head-chunked causal")


# Every element of the two forward configurations against the oracle, as
# the pages' own checks compare whole outputs (max-abs and mean-abs:
# blog.ans20xx.com day26, "数值对齐检查"; kwkr.cn/news/592482, 3.4).  The
# oracle takes about 70 GFLOP (C3) and 550 GFLOP (C2) of fp64 work.
FULL_EVERY_ELEMENT = [
    ("C2_noncausal_8x32x2048x128", 8, 32, 32, 2048, 128, False),
    ("C3_causal_2x16x4096x64", 2, 16, 16, 4096, 64, True),
]


@pytest.mark.parametrize("name,B,Hq,Hkv,N,D,causal", FULL_EVERY_ELEMENT,
                         ids=[f[0] for f in FULL_EVERY_ELEMENT])
def test_parity_full_size_every_element(ta, orc, name, B, Hq, Hkv, N, D, causal):
    x = make_qkv(B, Hq, Hkv, N, D, seed=0)
    o, lse = run_fwd(ta, x, causal=causal)
    ref = oracle_fwd(orc, x, causal, 1 / math.sqrt(D))
    mx, mean = check_o(o, ref["o"], name)
    lmx = check_lse(lse, ref["lse"], name)
    print(f"{name}: O max-abs {mx:.3e} mean-abs {mean:.3e}, LSE max-abs {lmx:.3e}")
