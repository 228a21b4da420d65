"""GPU parity of the causal sliding-window mask (attn_fwd_window /
attn_bwd_window) against the fp64 oracle.  Window reading: key j is kept for
query i iff i - W < j <= i ("FlashAttention原理与Triton实战" 3.1 and 7: a
window mask on the causal kernel; Block Attention Residual page, "实验结果":
an SWA baseline)."""
import math

import numpy as np
import pytest

from helpers import (check_grad, check_logits, check_lse, check_o, make_bias, make_qkv,
                     sample_rows, to_oracle)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tiled_attention_02_gb300 as ta
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ta.build()
    return ta


def dev(x, names=("q", "k", "v")):
    return tuple(x[n].cuda() for n in names)


def orc_in(x, names=("q", "k", "v")):
    return tuple(to_oracle(x[n]) for n in names)


CASES = [
    # B, Hq, Hkv, N, D, W
    (1, 2, 2, 384, 128, 1),      # only the diagonal
    (1, 2, 1, 384, 64, 100),     # window inside one tile
    (1, 2, 2, 500, 128, 128),    # exactly one tile, ragged N
    (1, 3, 1, 700, 64, 200),     # window spans tile edges, GQA 3:1
    (2, 2, 2, 300, 96, 257),     # D = 96, window past two tiles
    (1, 1, 1, 1000, 80, 333),    # D = 80, unaligned N
]
IDS = [f"B{c[0]}H{c[1]}kv{c[2]}N{c[3]}D{c[4]}W{c[5]}" for c in CASES]


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_window_forward(ta, orc, case):
    B, Hq, Hkv, N, D, W = case
    x = make_qkv(B, Hq, Hkv, N, D, seed=N + W)
    o, lse = ta.attn_fwd(*dev(x), causal=True, window=W)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    ref = orc.forward(*orc_in(x), scale=1 / math.sqrt(D), causal=True, window=W)
    check_o(o, ref["o"], f"window {case}")
    check_lse(lse, ref["lse"], f"window {case}")


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_window_backward(ta, orc, case):
    B, Hq, Hkv, N, D, W = case
    x = make_qkv(B, Hq, Hkv, N, D, seed=N + W + 1, with_do=True)
    q, k, v, do = dev(x, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=True, window=W)
    dq, dk, dv = ta.attn_bwd(q, k, v, o, lse, do, causal=True, window=W)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    ref = orc.backward(*orc_in(x, ("q", "k", "v", "do")), scale=1 / math.sqrt(D), causal=True,
                       window=W)
    check_grad(dq, ref["dq"], f"dq {case}")
    check_grad(dk, ref["dk"], f"dk {case}")
    check_grad(dv, ref["dv"], f"dv {case}")


@pytest.mark.parametrize("W", [384, 385, 5000])
def test_window_at_least_n_is_causal_bit_for_bit(ta, W):
    B, Hq, Hkv, N, D = 1, 2, 1, 384, 128
    x = make_qkv(B, Hq, Hkv, N, D, seed=3, with_do=True)
    q, k, v, do = dev(x, ("q", "k", "v", "do"))
    o1, l1 = ta.attn_fwd(q, k, v, causal=True)
    o2, l2 = ta.attn_fwd(q, k, v, causal=True, window=W)
    g1 = ta.attn_bwd(q, k, v, o1, l1, do, causal=True)
    g2 = ta.attn_bwd(q, k, v, o2, l2, do, causal=True, window=W)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])   # dK, dV (deterministic)
    assert (g1[0].float() - g2[0].float()).abs().max().item() < 1e-2  # dQ: reduction order


@pytest.mark.parametrize("off", [0, 1], ids=["staged", "direct"])
def test_window_bias_and_emit(ta, orc, off):
    """Residual variants under the window: O, LSE and the kept logits match,
    and tiles that hold no kept key keep their prior contents."""
    B, Hq, Hkv, N, D, W = 1, 2, 1, 640, 64, 150
    x = make_qkv(B, Hq, Hkv, N, D, seed=11)
    bias = make_bias(B, Hq, N, seed=12)
    n = B * Hq * N * N
    sentinel = 4321.0
    raw_e = torch.full((n + 4,), sentinel, device="cuda")
    emit = raw_e[off:off + n].view(B, Hq, N, N)
    raw_b = torch.empty(n + 4, device="cuda")
    b_dev = raw_b[off:off + n].view(B, Hq, N, N)
    b_dev.copy_(bias)
    o, lse = ta.attn_fwd(*dev(x), b_dev, causal=True, window=W, emit_logits=emit)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    ref = orc.forward(*orc_in(x), scale=1 / math.sqrt(D), causal=True, window=W,
                      bias=bias.numpy(), emit_logits=True)
    check_o(o, ref["o"], "window bias")
    check_lse(lse, ref["lse"], "window bias")
    check_logits(emit, ref["logits"], "window emit")
    for qt in range(N // 128):
        for kt in range(N // 128):
            blk = emit[..., qt * 128:(qt + 1) * 128, kt * 128:(kt + 1) * 128]
            # a kept key exists iff some query row i and key j in the tiles
            # have 0 <= i - j < W
            touched = kt <= qt and (qt * 128 - (kt * 128 + 127)) < W
            if not touched:
                assert bool((blk == sentinel).all()), (off, qt, kt)


def test_window_long_sequence_sampled(ta, orc):
    """N = 16384 with a 2048-key window: 256 sampled query rows (O, LSE, dQ)
    and 256 sampled key rows (dK, dV)."""
    B, Hq, Hkv, N, D, W = 1, 4, 4, 16384, 128, 2048
    x = make_qkv(B, Hq, Hkv, N, D, seed=5, with_do=True)
    q, k, v, do = dev(x, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=True, window=W)
    dq, dk, dv = ta.attn_bwd(q, k, v, o, lse, do, causal=True, window=W)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    qr = sample_rows(B, Hq, N, 256, seed=6)
    kr = sample_rows(B, Hkv, N, 256, seed=7)
    args = orc_in(x, ("q", "k", "v", "do"))
    ref = orc.forward(*args[:3], scale=1 / math.sqrt(D), causal=True, window=W, rows=qr)
    qr_t = torch.from_numpy(qr).cuda()
    kr_t = torch.from_numpy(kr).cuda()
    check_o(o.reshape(-1, D)[qr_t], ref["o"], "window long O")
    check_lse(lse.reshape(-1)[qr_t], ref["lse"], "window long LSE")
    g = orc.backward_sampled(*args, scale=1 / math.sqrt(D), causal=True, window=W, q_rows=qr,
                             k_rows=kr)
    check_grad(dq.reshape(-1, D)[qr_t], g["dq"], "window long dq")
    check_grad(dk.reshape(-1, D)[kr_t], g["dk"], "window long dk")
    check_grad(dv.reshape(-1, D)[kr_t], g["dv"], "window long dv")
