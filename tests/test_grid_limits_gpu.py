"""Launch-shape limits: problems whose head count or row-tile count passes
65535 (the limit of a grid's y dimension), forward and backward through the C
ABI.  Inputs are drawn on the device; the oracle checks rows whose exact
value depends only on a part it can take in full: one head of independent
heads, or, under a sliding window, a slice of rows that holds every key the
compared rows see."""
import math

import numpy as np
import pytest

from helpers import check_grad, check_lse, check_o, to_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tiled_attention_02_gb300 as ta
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ta.build()
    return ta


def _run(ta, x, **kw):
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o, lse = ta.attn_fwd(q, k, v, **kw)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    ta.attn_bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, **kw)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    return o, lse, dq, dk, dv


def test_head_count_past_grid_y(ta, orc):
    """B=65537 heads (a prime) of N=128, D=64: the backward's fp32 dQ
    accumulator (2.1 GB) is past twice the L2, but no chunk of whole heads
    near half the L2 divides a prime, and 65537 one-head chunks would pass
    the grid's y limit.  Heads are independent problems: the first, the last
    and heads around 2^15 and 2^16 each match the oracle run on that head."""
    from tiled_attention_02_gb300.inputs import make_qkv_device
    B, H, N, D = 65537, 1, 128, 64
    x = make_qkv_device(B, H, H, N, D, seed=31, with_do=True)
    o, lse, dq, dk, dv = _run(ta, x, causal=False)
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    for b in (0, 1, 32768, 65535, 65536):
        xb = {n: x[n][b:b + 1].cpu() for n in ("q", "k", "v", "do")}
        ref = orc.backward(*(to_oracle(xb[n]) for n in ("q", "k", "v", "do")),
                           scale=1 / math.sqrt(D), causal=False)
        check_o(o[b:b + 1], ref["o"], f"O head {b}")
        check_lse(lse[b:b + 1], ref["lse"], f"LSE head {b}")
        check_grad(dq[b:b + 1], ref["dq"], f"dq head {b}")
        check_grad(dk[b:b + 1], ref["dk"], f"dk head {b}")
        check_grad(dv[b:b + 1], ref["dv"], f"dv head {b}")


def test_row_tiles_past_grid_y(ta, orc):
    """N = 65536*128 + 100 rows (65537 row tiles, the last ragged), D=64,
    sliding window W=256.  A query row sees only keys i-W+1 .. i, so on a
    slice of rows [a, a+L) the oracle fixes every row whose window lies in the
    slice (O, LSE, dQ at i >= a+W-1) and every key row whose attending query
    rows all do (dK, dV at a+W-1 <= j <= a+L-W).  Slices: the start, across
    tile 65535 -> 65536, and the ragged end."""
    from tiled_attention_02_gb300.inputs import make_qkv_device
    B, H, N, D, W, L = 1, 1, 65536 * 128 + 100, 64, 256, 2048
    x = make_qkv_device(B, H, H, N, D, seed=32, with_do=True)
    o, lse, dq, dk, dv = _run(ta, x, causal=True, window=W)
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    for a in (0, 65535 * 128 - 1000, N - L):
        xs = {n: x[n][:, :, a:a + L].cpu() for n in ("q", "k", "v", "do")}
        ref = orc.backward(*(to_oracle(xs[n]) for n in ("q", "k", "v", "do")),
                           scale=1 / math.sqrt(D), causal=True, window=W)
        lo = 0 if a == 0 else W - 1          # rows from the start see no keys before it
        r = slice(lo, L)
        check_o(o[:, :, a + lo:a + L], ref["o"][:, :, r], f"O slice {a}")
        check_lse(lse[:, :, a + lo:a + L], ref["lse"][:, :, r], f"LSE slice {a}")
        check_grad(dq[:, :, a + lo:a + L], ref["dq"][:, :, r], f"dq slice {a}")
        hi = L if a + L == N else L - W + 1  # key rows whose query rows are all in the slice
        kr = slice(lo, hi)
        check_grad(dk[:, :, a + lo:a + hi], ref["dk"][:, :, kr], f"dk slice {a}")
        check_grad(dv[:, :, a + lo:a + hi], ref["dv"][:, :, kr], f"dv slice {a}")
