"""GPU parity of the block-residual backward (attn_bwd_residual) against the
fp64 oracle.  Reading (Block Attention Residual page, "v1: Fuse Residual 进
Attention Kernel": the backward keeps the LSE statistics, corrected for the
residual): with S_l = scale Q_l K_l^T + S_{l-1}, the gradient reaching S_l is
dS_l = P_l o (dP_l - Delta_l) + dS_{l+1}; it gives dQ_l, dK_l and is the
gradient of layer l's bias."""
import math

import numpy as np
import pytest

from helpers import check_grad, make_bias, make_chain, make_qkv, to_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# dS is a gradient (of the bias), held to the gradient tolerance: P enters it
# rounded to bf16 (relative error <= 2^-9, the same P the dV MMA uses) and
# Delta comes from the bf16 O, so |error| ~ 2^-9 |dS| + ...; |dS| reaches ~6.
from helpers import GRAD_MAX_ABS as DLOGIT_ABS  # noqa: E402


@pytest.fixture(scope="module")
def ta():
    import tiled_attention_02_gb300 as ta
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ta.build()
    return ta


def check_dlogits(got, ref, causal, what):
    g = got.detach().cpu().numpy().astype(np.float64).reshape(ref.shape)
    N = ref.shape[-1]
    keep = np.tril(np.ones((N, N), dtype=bool)) if causal else np.ones((N, N), dtype=bool)
    assert np.isfinite(g[..., keep]).all(), f"{what}: non-finite dS"
    mx = float(np.abs(g[..., keep] - ref[..., keep]).max())
    assert mx <= DLOGIT_ABS, f"{what}: dS max-abs {mx:.3e} (max |ref| {np.abs(ref).max():.3g})"


CASES = [
    # B, Hq, Hkv, N, D, causal, bias, grad_in, grad_out
    (1, 2, 2, 256, 128, True, True, True, True),
    (1, 4, 2, 384, 64, True, True, False, True),     # last layer of a block
    (1, 2, 1, 300, 128, True, False, True, False),   # first layer: no bias, no dS out
    (1, 2, 2, 256, 64, False, True, True, True),     # non-causal
    (2, 2, 1, 200, 96, True, True, True, True),      # D = 96, ragged N
]


@pytest.mark.parametrize("case", CASES, ids=[
    f"B{c[0]}H{c[1]}kv{c[2]}N{c[3]}D{c[4]}c{int(c[5])}b{int(c[6])}gi{int(c[7])}go{int(c[8])}"
    for c in CASES])
def test_residual_backward_layer(ta, orc, case):
    B, Hq, Hkv, N, D, causal, has_b, has_gi, has_go = case
    x = make_qkv(B, Hq, Hkv, N, D, seed=N + D, with_do=True)
    bias = make_bias(B, Hq, N, seed=N + 5) if has_b else None
    gin = make_bias(B, Hq, N, seed=N + 6, std=0.05) if has_gi else None
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    b_dev = bias.cuda() if has_b else None
    o, lse = ta.attn_fwd(q, k, v, b_dev, causal=causal)
    gout = torch.full((B, Hq, N, N), float("nan"), device="cuda") if has_go else None
    dq, dk, dv = ta.attn_bwd(q, k, v, o, lse, do, causal=causal, bias=b_dev,
                             grad_in=gin.cuda() if has_gi else None, grad_out=gout)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    ref = orc.backward(*(to_oracle(x[n]) for n in ("q", "k", "v", "do")), scale=1 / math.sqrt(D),
                       causal=causal, bias=None if bias is None else bias.numpy(),
                       grad_in=None if gin is None else gin.numpy())
    check_grad(dq, ref["dq"], f"dq {case}")
    check_grad(dk, ref["dk"], f"dk {case}")
    check_grad(dv, ref["dv"], f"dv {case}")
    if has_go:
        check_dlogits(gout, ref["dlogits"], causal, f"dS {case}")


def test_residual_backward_in_place(ta, orc):
    """grad_out may be the grad_in buffer (one chain gradient buffer)."""
    B, Hq, Hkv, N, D = 1, 2, 2, 256, 128
    x = make_qkv(B, Hq, Hkv, N, D, seed=8, with_do=True)
    bias = make_bias(B, Hq, N, seed=9)
    gin = make_bias(B, Hq, N, seed=10, std=0.05)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, bias.cuda(), causal=True)
    buf = gin.cuda()
    dq, dk, dv = ta.attn_bwd(q, k, v, o, lse, do, causal=True, bias=bias.cuda(), grad_in=buf,
                             grad_out=buf)
    torch.cuda.synchronize()
    ref = orc.backward(*(to_oracle(x[n]) for n in ("q", "k", "v", "do")), scale=1 / math.sqrt(D),
                       causal=True, bias=bias.numpy(), grad_in=gin.numpy())
    check_grad(dq, ref["dq"], "in place dq")
    check_dlogits(buf, ref["dlogits"], True, "in place dS")


def test_residual_chain_backward(ta, orc):
    """A 4-layer block, forward then backward through the chain: each layer's
    bias is the previous layer's emitted logits (kept per layer), and one
    gradient buffer carries dS from layer l to layer l-1 in place."""
    B, Hq, Hkv, N, D, L = 1, 4, 2, 384, 128, 4
    layers = make_chain(B, Hq, Hkv, N, D, layers=L, seed=3, with_do=True)
    dev = [{n: x[n].cuda() for n in ("q", "k", "v", "do")} for x in layers]
    S = [torch.empty((B, Hq, N, N), device="cuda") for _ in range(L - 1)]
    fw = []
    for i, x in enumerate(dev):
        o, lse = ta.attn_fwd(x["q"], x["k"], x["v"], S[i - 1] if i > 0 else None, causal=True,
                             emit_logits=S[i] if i < L - 1 else None)
        fw.append((o, lse))
    gbuf = torch.empty((B, Hq, N, N), device="cuda")
    grads = [None] * L
    for i in reversed(range(L)):
        x, (o, lse) = dev[i], fw[i]
        grads[i] = ta.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=True,
                               bias=S[i - 1] if i > 0 else None,
                               grad_in=gbuf if i < L - 1 else None,
                               grad_out=gbuf if i > 0 else None)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    # oracle: forward chain for the biases, then the same backward recursion
    scale = 1 / math.sqrt(D)
    ox = [{n: to_oracle(x[n]) for n in ("q", "k", "v", "do")} for x in layers]
    biases, prev = [None], None
    for i in range(L - 1):
        f = orc.forward(ox[i]["q"], ox[i]["k"], ox[i]["v"], scale=scale, causal=True,
                        bias=prev, emit_logits=True)
        prev = np.nan_to_num(f["logits"])
        biases.append(prev)
    g_in = None
    for i in reversed(range(L)):
        r = orc.backward(ox[i]["q"], ox[i]["k"], ox[i]["v"], ox[i]["do"], scale=scale,
                         causal=True, bias=biases[i], grad_in=g_in)
        dq, dk, dv = grads[i]
        check_grad(dq, r["dq"], f"chain dq {i}")
        check_grad(dk, r["dk"], f"chain dk {i}")
        check_grad(dv, r["dv"], f"chain dv {i}")
        g_in = r.get("dlogits")


def test_residual_chain_backward_full_size_sampled(ta, orc):
    """The block-residual training step at full size: 4 layers, B=1, Hq=20,
    Hkv=4, N=4096, D=128, causal, forward then backward through the block
    with one gradient buffer passed down in place.  Row i of a layer's dQ
    and of its outgoing logit gradient depends only on row i of its bias
    (the layer below's logits) and of the gradient arriving from the layer
    above, so the oracle follows 256 sampled query rows through the whole
    block, up and back down."""
    from helpers import sample_rows
    B, Hq, Hkv, N, D, L = 1, 20, 4, 4096, 128, 4
    scale = 1 / math.sqrt(D)
    layers = make_chain(B, Hq, Hkv, N, D, layers=L, seed=9, with_do=True)
    dev = [{n: x[n].cuda() for n in ("q", "k", "v", "do")} for x in layers]
    S = [torch.empty((B, Hq, N, N), device="cuda") for _ in range(L - 1)]
    fw = []
    for i, x in enumerate(dev):
        fw.append(ta.attn_fwd(x["q"], x["k"], x["v"], S[i - 1] if i > 0 else None, causal=True,
                              emit_logits=S[i] if i < L - 1 else None))
    gbuf = torch.empty((B, Hq, N, N), device="cuda")
    dq = [None] * L
    for i in reversed(range(L)):
        x, (o, lse) = dev[i], fw[i]
        dq[i], dk, dv = ta.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=True,
                                    bias=S[i - 1] if i > 0 else None,
                                    grad_in=gbuf if i < L - 1 else None,
                                    grad_out=gbuf if i > 0 else None)
        assert torch.isfinite(dk.float()).all() and torch.isfinite(dv.float()).all()
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    rows = sample_rows(B, Hq, N, 256, seed=10)
    rows_t = torch.from_numpy(rows).cuda()
    ox = [{n: to_oracle(x[n]) for n in ("q", "k", "v", "do")} for x in layers]
    # up: the sampled rows' logits of layers 0..L-2, each the next one's bias
    bias_rows, prev = [None], None
    for i in range(L - 1):
        f = orc.forward(ox[i]["q"], ox[i]["k"], ox[i]["v"], scale=scale, causal=True, rows=rows,
                        bias=prev, emit_logits=True)
        prev = np.nan_to_num(f["logits"])
        bias_rows.append(prev)

    def at_rows(r):
        """A [B,Hq,N,N] array holding r at the sampled rows (zero pages elsewhere)."""
        if r is None:
            return None
        full = np.zeros((B, Hq, N, N))
        full.reshape(-1, N)[rows] = r
        return full
    # down: dQ and the outgoing logit gradient of the same rows
    g_rows = None
    for i in reversed(range(L)):
        r = orc.backward_sampled(ox[i]["q"], ox[i]["k"], ox[i]["v"], ox[i]["do"], scale=scale,
                                 causal=True, q_rows=rows, k_rows=[], bias=at_rows(bias_rows[i]),
                                 grad_in=at_rows(g_rows))
        check_grad(dq[i].reshape(-1, D)[rows_t], r["dq"], f"chain dq {i} sampled")
        g_rows = r["dlogits"]
        if i == 1:   # the buffer holds layer 1's outgoing gradient at the end
            got = gbuf.reshape(-1, N)[rows_t].cpu().numpy().astype(np.float64)
            keep = np.arange(N)[None, :] <= (rows % N)[:, None]
            err = np.abs(got - g_rows)[keep].max()
            assert err <= DLOGIT_ABS, f"layer 1 logit gradient max-abs {err:.3e}"
