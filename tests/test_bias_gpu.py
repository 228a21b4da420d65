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
    (1, 2, 1, 260, 128, True),     # N % 32 != 0: ragged inside a staged fp32 chunk
    (1, 2, 2, 260, 128, False),
    (1, 2, 1, 640, 64, True),      # five key tiles: the staged ring wraps
    (1, 2, 2, 256, 80, True),      # head dims 80 and 96
    (1, 2, 1, 203, 96, False),
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


def test_staged_and_direct_paths_agree(ta):
    """Bias and emit rows that are 16-byte aligned go through the staged
    (TMA) path; the same values one float off a 16-byte boundary go through
    the direct per-thread path.  Both evaluate y = fma(qk, scale, bias) on the
    same accumulator, so O, LSE and every kept logit agree bit for bit."""
    B, Hq, Hkv, N, D = 1, 2, 1, 384, 128
    x = make_qkv(B, Hq, Hkv, N, D, seed=31)
    bias = make_bias(B, Hq, N, seed=32).cuda()
    q, k, v = dev(x)
    n = bias.numel()
    raw_b = torch.empty(n + 4, device="cuda")
    raw_e = torch.full((n + 4,), float("nan"), device="cuda")
    b_off = raw_b[1:n + 1].view(B, Hq, N, N)
    e_off = raw_e[1:n + 1].view(B, Hq, N, N)
    b_off.copy_(bias)
    assert b_off.data_ptr() % 16 == 4
    e_al = torch.full_like(bias, float("nan"))
    for causal in (True, False):
        o1, l1 = ta.attn_fwd(q, k, v, bias, causal=causal, emit_logits=e_al)
        o2, l2 = ta.attn_fwd(q, k, v, b_off, causal=causal, emit_logits=e_off)
        torch.cuda.synchronize()
        assert ta.attn_last_device_status() == 0
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        keep = torch.ones(N, N, dtype=torch.bool, device="cuda")
        if causal:
            keep = torch.tril(keep)
        assert torch.equal(e_al[..., keep], e_off[..., keep])


def test_causal_emit_leaves_upper_tiles(ta):
    """Under the causal mask the 128 x 128 logit tiles strictly above the
    diagonal are never written (both residual paths)."""
    B, Hq, Hkv, N, D = 1, 2, 2, 384, 64
    x = make_qkv(B, Hq, Hkv, N, D, seed=41)
    q, k, v = dev(x)
    sentinel = 12345.0
    for off in (0, 1):   # 0: staged path, 1: direct path (misaligned rows)
        raw = torch.full((B * Hq * N * N + 4,), sentinel, device="cuda")
        emit = raw[off:off + B * Hq * N * N].view(B, Hq, N, N)
        ta.attn_fwd(q, k, v, causal=True, emit_logits=emit)
        torch.cuda.synchronize()
        assert ta.attn_last_device_status() == 0
        for qt in range(3):
            for kt in range(3):
                blk = emit[..., qt * 128:(qt + 1) * 128, kt * 128:(kt + 1) * 128]
                if kt > qt:
                    assert bool((blk == sentinel).all()), (off, qt, kt)
                else:
                    assert bool(torch.isfinite(blk).all())


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


def test_chain_full_size_every_element(ta, orc):
    """The 4-layer block at full size (B=1, 20 query heads, 4 kv heads,
    N=4096, D=128, causal), every output element and every kept emitted logit
    against the oracle's own chain (fp64 logits carried layer to layer)."""
    B, Hq, Hkv, N, D = 1, 20, 4, 4096, 128
    layers = make_chain(B, Hq, Hkv, N, D, layers=4, seed=0)
    outs, snaps = run_chain_gpu(ta, layers, causal=True)
    prev = None
    for i, x in enumerate(layers):
        ref = orc.forward(*orc_in(x), scale=1 / math.sqrt(D), causal=True,
                          bias=prev, emit_logits=True)
        check_o(outs[i][0], ref["o"], f"layer {i}")
        check_lse(outs[i][1], ref["lse"], f"layer {i}")
        if i < 3:
            check_logits(snaps[i], ref["logits"], f"logits {i}")
            snaps[i] = None
            # The next layer's bias: the kept logits (masked entries never
            # reach a result; zero them so the oracle reads finite numbers).
            prev = np.nan_to_num(ref["logits"], nan=0.0, copy=False)
        del ref
