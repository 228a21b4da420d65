"""GPU parity of the decode step (attn_decode, flash decode) against the
fp64 oracle: one query row per (batch, query head) at position N-1 over an
N-row cache is the last row of causal attention."""
import math

import numpy as np
import pytest

from helpers import check_lse, check_o, to_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tiled_attention_02_gb300 as ta
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ta.build()
    return ta


def oracle_decode(orc, x, scale):
    """Place each query row at position N-1 of an otherwise zero query
    tensor and take the causal forward's last row."""
    q = to_oracle(x["q"])
    k, v = to_oracle(x["k"]), to_oracle(x["v"])
    B, Hq, D = q.shape
    N = k.shape[2]
    qf = np.zeros((B, Hq, N, D))
    qf[:, :, N - 1] = q
    rows = np.arange(B * Hq) * N + (N - 1)
    ref = orc.forward(qf, k, v, scale=scale, causal=True, rows=rows)
    return ref["o"].reshape(B, Hq, D), ref["lse"].reshape(B, Hq)


CASES = [
    # B, Hq, Hkv, N, D
    (1, 1, 1, 1, 64),          # a single key
    (2, 4, 4, 100, 64),        # one ragged stage, plain multi-head
    (2, 8, 2, 1000, 128),      # GQA 4:1, ragged
    (1, 16, 1, 3000, 128),     # 16 query heads on one kv head
    (3, 6, 2, 777, 80),        # D = 80
    (2, 12, 4, 4096, 96),      # D = 96
    (1, 5, 1, 20000, 128),     # long cache: many splits
    (2, 16, 2, 4096, 64),      # D = 64 with 8:1 groups over several splits
    (40, 8, 8, 1000, 128),     # several kv heads per block, segments straddling blocks
    (8, 32, 8, 300, 96),       # short caches: blocks of one or two stages
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}kv{c[2]}N{c[3]}D{c[4]}" for c in CASES])
def test_decode_parity(ta, orc, case):
    from tiled_attention_02_gb300.inputs import make_decode
    B, Hq, Hkv, N, D = case
    x = make_decode(B, Hq, Hkv, N, D, seed=N + D)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = ta.attn_decode(q, k, v)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    ro, rl = oracle_decode(orc, x, 1 / math.sqrt(D))
    check_o(o, ro, f"decode {case}")
    check_lse(lse, rl, f"decode {case}")


def test_decode_equals_last_row_of_forward(ta):
    """The decode kernel and the causal forward agree on the last row."""
    from tiled_attention_02_gb300.inputs import make_qkv
    B, Hq, Hkv, N, D = 1, 8, 2, 1500, 128
    x = make_qkv(B, Hq, Hkv, N, D, seed=21)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    of, lf = ta.attn_fwd(q, k, v, causal=True)
    od, ld = ta.attn_decode(q[:, :, N - 1].contiguous(), k, v)
    torch.cuda.synchronize()
    assert (of[:, :, N - 1].float() - od.float()).abs().max().item() <= 1.6e-2
    assert (lf[:, :, N - 1] - ld).abs().max().item() <= 1e-3


def test_decode_workspace_contents_do_not_matter(ta):
    from tiled_attention_02_gb300.inputs import make_decode
    B, Hq, Hkv, N, D = 2, 4, 2, 2000, 64
    x = make_decode(B, Hq, Hkv, N, D, seed=4)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    need = ta.attn_decode_workspace_size(B, Hq, Hkv, N, D)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")   # NaN patterns
    o1, l1 = ta.attn_decode(q, k, v, workspace=ws)
    o2, l2 = ta.attn_decode(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_full_size(ta, orc):
    """The decode bench line's shape, B=16, Hq=32, Hkv=8, N=16384, D=128:
    every one of its 512 query rows against the oracle, one (batch, kv head)
    group of query heads at a time."""
    from tiled_attention_02_gb300.inputs import make_decode
    B, Hq, Hkv, N, D = 16, 32, 8, 16384, 128
    G = Hq // Hkv
    x = make_decode(B, Hq, Hkv, N, D, seed=5)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = ta.attn_decode(q, k, v)
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    ro = np.empty((B, Hq, D))
    rl = np.empty((B, Hq))
    for b in range(B):
        for g in range(Hkv):
            xg = {"q": x["q"][b:b + 1, g * G:(g + 1) * G], "k": x["k"][b:b + 1, g:g + 1],
                  "v": x["v"][b:b + 1, g:g + 1]}
            go, gl = oracle_decode(orc, xg, 1 / math.sqrt(D))
            ro[b, g * G:(g + 1) * G] = go[0]
            rl[b, g * G:(g + 1) * G] = gl[0]
    check_o(o, ro, "decode full size")
    check_lse(lse, rl, "decode full size")
