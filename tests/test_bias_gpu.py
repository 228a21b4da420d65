"""GPU parity of the additive logit bias and the emitted logits (block
attention residual: S_i = Q_i K_i^T / sqrt(d) + S_{i-1}, S_{-1} = 0,
Block Attention Residual Triton kernel, sections "Block Attention Residual
做了什么" and "v2: 优化 torch.cat + SRAM 复用") against the fp64 oracle."""
import math

import numpy as np
import pytest

from helpers import (check_logits, check_lse, check_o, make_bias, make_chain, make_qkv,
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


def dev(x):
    return tuple(x[n].cuda() for n in ("q", "k", "v"))


def orc_in(x):
    return tuple(to_oracle(x[n]) for n in ("q", "k", "v"))


CASES = [
    # B, Hq, Hkv, N, D, causal
    (1, 4, 2, 384, 128, True),
    (1, 4, 2, 384, 128, False),
    (2, 2, 1, 256, 64, True),
    (1, 2, 2, 203, 64, False),     # N % 4 != 0: scalar bias path, ragged tail
    (1, 3, 3, 130, 128, True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}kv{c[2]}N{c[3]}D{c[4]}c{int(c[5])}"
                                             for c in CASES])
def test_bias_and_emit(ta, orc, case):
    B, Hq, Hkv, N, D, causal = case
    x = make_qkv(B, Hq, Hkv, N, D, seed=N)
    bias = make_bias(B, Hq, N, seed=N + 1)
    q, k, v = dev(x)
    emit = torch.full((B, Hq, N, N), float("nan"), device="cuda")
    o, lse = ta.attn_fwd(q, k, v, bias.cuda(), causal=causal, emit_logits=emit)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    ref = orc.forward(*orc_in(x), scale=1 / math.sqrt(D), causal=causal, bias=bias.numpy(),
                      emit_logits=True)
    check_o(o, ref["o"], "bias")
    check_lse(lse, ref["lse"], "bias")
    check_logits(emit, ref["logits"], "emit")


def test_emit_without_bias(ta, orc):
    B, Hq, Hkv, N, D = 1, 2, 1, 300, 128
    x = make_qkv(B, Hq, Hkv, N, D, seed=9)
    q, k, v = dev(x)
    emit = torch.empty((B, Hq, N, N), device="cuda")
    o, lse = ta.attn_fwd(q, k, v, causal=True, emit_logits=emit)
    torch.cuda.synchronize()
    ref = orc.forward(*orc_in(x), scale=1 / math.sqrt(D), causal=True, emit_logits=True)
    check_o(o, ref["o"], "emit only")
    check_logits(emit, ref["logits"], "emit only")


def test_bias_without_emit_matches_emit_path(ta):
    """The bias-only variant and the bias+emit variant give identical O."""
    B, Hq, Hkv, N, D = 1, 2, 2, 256, 128
    x = make_qkv(B, Hq, Hkv, N, D, seed=4)
    bias = make_bias(B, Hq, N, seed=5).cuda()
    q, k, v = dev(x)
    o1, l1 = ta.attn_fwd(q, k, v, bias, causal=True)
    o2, l2 = ta.attn_fwd(q, k, v, bias, causal=True, emit_logits=torch.empty_like(bias))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_in_place_alias(ta, orc):
    """emit_logits may be the bias buffer itself (preallocated residual)."""
    B, Hq, Hkv, N, D = 1, 4, 4, 256, 64
    x = make_qkv(B, Hq, Hkv, N, D, seed=12)
    bias = make_bias(B, Hq, N, seed=13)
    buf = bias.cuda()
    q, k, v = dev(x)
    o, lse = ta.attn_fwd(q, k, v, buf, causal=True, emit_logits=buf)
    torch.cuda.synchronize()
    ref = orc.forward(*orc_in(x), scale=1 / 8, causal=True, bias=bias.numpy(), emit_logits=True)
    check_o(o, ref["o"], "alias")
    check_logits(buf, ref["logits"], "alias")


def test_zero_bias_equals_no_bias(ta):
    x = make_qkv(1, 2, 2, 256, 128, seed=21)
    q, k, v = dev(x)
    o1, l1 = ta.attn_fwd(q, k, v, causal=True)
    o2, l2 = ta.attn_fwd(q, k, v, torch.zeros(1, 2, 256, 256, device="cuda"), causal=True)
    torch.cuda.synchronize()
    check_o(o2, o1.double().cpu().numpy(), "zero bias")
    assert (l1 - l2).abs().max().item() < 1e-5


def run_chain_gpu(ta, layers, causal, snapshot_rows=None):
    """Block of chained layers with one in-place fp32 residual buffer."""
    q0 = layers[0]["q"]
    B, Hq, N, _ = q0.shape
    buf = torch.empty((B, Hq, N, N), device="cuda")
    outs, snaps = [], []
    for i, x in enumerate(layers):
        q, k, v = dev(x)
        bias = buf if i > 0 else None
        emit = buf if i < len(layers) - 1 else None
        o, lse = ta.attn_fwd(q, k, v, bias, causal=causal, emit_logits=emit)
        outs.append((o, lse))
        if emit is not None and snapshot_rows is not None:
            snaps.append(buf.reshape(-1, N)[snapshot_rows].clone())
        elif emit is not None:
            snaps.append(buf.clone())
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    return outs, snaps


def test_chain_small_full_compare(ta, orc):
    B, Hq, Hkv, N, D = 1, 10, 2, 384, 128
    layers = make_chain(B, Hq, Hkv, N, D, layers=4, seed=0)
    outs, snaps = run_chain_gpu(ta, layers, causal=True)
    prev = None
    for i, x in enumerate(layers):
        ref = orc.forward(*orc_in(x), scale=1 / math.sqrt(D), causal=True,
                          bias=None if prev is None else np.nan_to_num(prev), emit_logits=True)
        check_o(outs[i][0], ref["o"], f"chain layer {i}")
        check_lse(outs[i][1], ref["lse"], f"chain layer {i}")
        if i < 3:
            check_logits(snaps[i], ref["logits"], f"chain logits {i}")
        prev = ref["logits"]


def test_chain_full_size_sampled(ta, orc):
    """Block of 4 layers: B=1, 20 query heads, 4 kv heads, N=4096, D=128,
    causal; one 1.34 GB fp32 residual buffer updated in place.  Row i of S_L
    depends only on row i of S_{L-1}, so the oracle follows sampled rows
    through the whole block."""
    B, Hq, Hkv, N, D = 1, 20, 4, 4096, 128
    layers = make_chain(B, Hq, Hkv, N, D, layers=4, seed=0)
    rows = sample_rows(B, Hq, N, 256, seed=2)
    rows_t = torch.from_numpy(rows).cuda()
    outs, snaps = run_chain_gpu(ta, layers, causal=True, snapshot_rows=rows_t)
    prev = None
    for i, x in enumerate(layers):
        ref = orc.forward(*orc_in(x), scale=1 / math.sqrt(D), causal=True, rows=rows,
                          bias=None if prev is None else prev, emit_logits=True)
        check_o(outs[i][0].reshape(-1, D)[rows_t], ref["o"], f"layer {i}")
        check_lse(outs[i][1].reshape(-1)[rows_t], ref["lse"], f"layer {i}")
        if i < 3:
            check_logits(snaps[i], ref["logits"], f"logits {i}")
        prev = np.ascontiguousarray(ref["logits"])
