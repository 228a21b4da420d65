"""GPU parity of the recompute backward (C ABI) against the fp64 oracle's
exact gradient: every element on small shapes (several tiles, ragged tails,
grouped heads), and 256 query rows (dQ) plus 256 key rows (dK, dV) at the
full long-sequence size."""
import math

import numpy as np
import pytest

from helpers import check_grad, make_qkv, sample_rows, to_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tiled_attention_02_gb300 as ta
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ta.build()
    return ta


def gpu_fwd_bwd(ta, x, causal):
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = ta.attn_bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    return dq, dk, dv


SHAPES = [
    # B, Hq, Hkv, N, D
    (1, 2, 2, 256, 128),
    (1, 4, 2, 384, 64),      # grouped heads: dK, dV summed over the group
    (1, 3, 1, 200, 128),     # ragged tail
    (2, 2, 2, 129, 64),      # one row past a tile
    (1, 1, 1, 1, 128),       # single row
    (1, 6, 2, 256, 128),
    (1, 2, 1, 384, 80),      # head dims 80 and 96: padded swizzle atoms, clipped stores
    (1, 2, 2, 200, 96),      #   and a third fp32 dQ box clipped at D
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}H{s[1]}kv{s[2]}N{s[3]}D{s[4]}" for s in SHAPES])
def test_bwd_parity_small(ta, orc, shape, causal):
    B, Hq, Hkv, N, D = shape
    x = make_qkv(B, Hq, Hkv, N, D, seed=N + D + 1, with_do=True)
    dq, dk, dv = gpu_fwd_bwd(ta, x, causal)
    ref = orc.backward(*(to_oracle(x[n]) for n in ("q", "k", "v", "do")),
                       scale=1 / math.sqrt(D), causal=causal)
    check_grad(dq, ref["dq"], f"dq {shape}")
    check_grad(dk, ref["dk"], f"dk {shape}")
    check_grad(dv, ref["dv"], f"dv {shape}")


def test_bwd_every_output_written(ta):
    x = make_qkv(1, 2, 1, 333, 128, seed=2, with_do=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=True)
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    ta.attn_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()


def test_bwd_workspace_contents_do_not_matter(ta):
    """The workspace is fully initialised by the call itself."""
    x = make_qkv(1, 2, 2, 256, 64, seed=3, with_do=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=True)
    need = ta.attn_bwd_workspace_size(1, 2, 2, 256, 64)
    ws1 = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ws2 = torch.full((need,), 0x7F, dtype=torch.uint8, device="cuda")
    a = ta.attn_bwd(q, k, v, o, lse, do, causal=True, workspace=ws1)
    b = ta.attn_bwd(q, k, v, o, lse, do, causal=True, workspace=ws2)
    torch.cuda.synchronize()
    for u, w in zip(a, b):
        assert (u.float() - w.float()).abs().max().item() < 1e-2


FULL_SIZE = [
    # D, window: the default step's shape (B=1, H=16, N=16384, causal) at each head
    # dim the bench times, and its 4096-key sliding window
    (128, None), (80, None), (96, None), (128, 4096),
]


@pytest.mark.parametrize("D,window", FULL_SIZE,
                         ids=[f"D{d}" + (f"W{w}" if w else "") for d, w in FULL_SIZE])
def test_bwd_full_size_sampled(ta, orc, D, window):
    """B=1, H=16, N=16384, causal: O and LSE at 256 sampled query rows, dQ
    at the same rows and dK, dV at 256 sampled key rows against the oracle's
    exact values."""
    from helpers import check_lse, check_o
    B, H, N = 1, 16, 16384
    x = make_qkv(B, H, H, N, D, seed=0, with_do=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=True, window=window)
    dq, dk, dv = ta.attn_bwd(q, k, v, o, lse, do, causal=True, window=window)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    q_rows = sample_rows(B, H, N, 256, seed=3)
    rng = np.random.default_rng(4)
    heads = rng.choice(H, size=4, replace=False)
    k_rows = np.unique(np.concatenate([
        np.array([h * N, h * N + N - 1, h * N + 127, h * N + 128]) for h in heads] + [
        heads[rng.integers(0, 4, 240)] * N + rng.integers(0, N, 240)]))
    ox = [to_oracle(x[n]) for n in ("q", "k", "v", "do")]
    ref = orc.backward_sampled(*ox, scale=1 / math.sqrt(D), causal=True, window=window,
                               q_rows=q_rows, k_rows=k_rows)
    fw = orc.forward(*ox[:3], scale=1 / math.sqrt(D), causal=True, window=window, rows=q_rows)
    qr, kr = torch.from_numpy(q_rows).cuda(), torch.from_numpy(k_rows).cuda()
    check_o(o.reshape(-1, D)[qr], fw["o"], "O sampled")
    check_lse(lse.reshape(-1)[qr], fw["lse"], "LSE sampled")
    check_grad(dq.reshape(-1, D)[qr], ref["dq"], "dq sampled")
    check_grad(dk.reshape(-1, D)[kr], ref["dk"], "dk sampled")
    check_grad(dv.reshape(-1, D)[kr], ref["dv"], "dv sampled")


def _bf16_close(a, b, rel=2.0 ** -7):
    """Equal up to one bf16 rounding step (fp32 sums in another order)."""
    a, b = a.float(), b.float()
    return bool(((a - b).abs() <= rel * torch.maximum(a.abs(), b.abs()) + 1e-6).all())


def test_bwd_head_chunked_order(ta, orc):
    """Blocks in chunks of kv heads (the fp32 dQ accumulator, 537 MB, is
    over half the L2): B=4, H=16, N=16384, D=128 causal.  Heads are independent
    problems: dK and dV of every head equal, bit for bit, a launch on that
    head alone (the same blocks, in the plain order), and dQ does up to the
    order of its fp32 reduce-adds; sampled rows are checked against the
    oracle's exact gradient."""
    B, H, N, D = 4, 16, 16384, 128
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    assert B * H * N * D * 4 > 0.5 * l2, "shape must take the head-chunked order"
    x = make_qkv(B, H, H, N, D, seed=11, with_do=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=True)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    ta.attn_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    for b in range(B):
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            dq1, dk1, dv1 = ta.attn_bwd(*(t[sl].contiguous() for t in (q, k, v, o, lse, do)),
                                        causal=True)
            assert torch.equal(dk[sl], dk1), f"dK of head ({b}, {h})"
            assert torch.equal(dv[sl], dv1), f"dV of head ({b}, {h})"
            assert _bf16_close(dq[sl], dq1), f"dQ of head ({b}, {h})"
    q_rows = sample_rows(B, H, N, 256, seed=12)
    rng = np.random.default_rng(13)
    heads = rng.choice(B * H, size=3, replace=False)
    k_rows = np.unique(np.concatenate(
        [np.array([g * N, g * N + N - 1, g * N + 128]) for g in heads] +
        [heads[rng.integers(0, 3, 120)] * N + rng.integers(0, N, 120)]))
    ref = orc.backward_sampled(*(to_oracle(x[n]) for n in ("q", "k", "v", "do")),
                               scale=1 / math.sqrt(D), causal=True, q_rows=q_rows, k_rows=k_rows)
    qr, kr = torch.from_numpy(q_rows).cuda(), torch.from_numpy(k_rows).cuda()
    check_grad(dq.reshape(-1, D)[qr], ref["dq"], "dq sampled, head-chunked")
    check_grad(dk.reshape(-1, D)[kr], ref["dk"], "dk sampled, head-chunked")
    check_grad(dv.reshape(-1, D)[kr], ref["dv"], "dv sampled, head-chunked")


def test_bwd_head_chunked_grouped(ta, orc):
    """The chunked order with grouped heads: B=2, Hq=32, Hkv=8, N=16384,
    D=128 causal, one kv head (four query heads) per chunk.  Outputs start as
    NaN, so every block must have written its rows; sampled rows of one kv
    head against the oracle."""
    B, Hq, Hkv, N, D = 2, 32, 8, 16384, 128
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    assert B * Hq * N * D * 4 > 0.5 * l2, "shape must take the head-chunked order"
    x = make_qkv(B, Hq, Hkv, N, D, seed=21, with_do=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=True)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    ta.attn_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    q_rows = sample_rows(B, Hq, N, 256, seed=22)
    rng = np.random.default_rng(23)
    g = int(rng.integers(0, B * Hkv))
    k_rows = np.unique(np.concatenate([np.array([g * N, g * N + N - 1, g * N + 128]),
                                       g * N + rng.integers(0, N, 120)]))
    ref = orc.backward_sampled(*(to_oracle(x[n]) for n in ("q", "k", "v", "do")),
                               scale=1 / math.sqrt(D), causal=True, q_rows=q_rows, k_rows=k_rows)
    qr, kr = torch.from_numpy(q_rows).cuda(), torch.from_numpy(k_rows).cuda()
    check_grad(dq.reshape(-1, D)[qr], ref["dq"], "dq sampled, grouped head-chunked")
    check_grad(dk.reshape(-1, D)[kr], ref["dk"], "dk sampled, grouped head-chunked")
    check_grad(dv.reshape(-1, D)[kr], ref["dv"], "dv sampled, grouped head-chunked")
