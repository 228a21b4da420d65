"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (an engine that owns all device allocations and gives libraries no
allocator, or code that must avoid the synchronisation cudaMalloc/cudaFree
can cause).  It uses the library's fixed device scratch instead of a
caller workspace.  Checked through the C ABI against attn_bwd on the same
inputs, on two calls in a row (the scratch keeps the previous call's
contents, which must not matter), and against the fp64 oracle on sampled
rows.  Kept in its own file, collected last."""
import math

import numpy as np
import pytest

from helpers import check_grad, make_qkv, to_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tiled_attention_02_gb300 as ta
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ta.build()
    return ta


def raw_noalloc(ta, q, k, v, o, lse, do, dq, dk, dv, causal):
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    return ta.raw_attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), B, Hq, Hkv, N, D, D ** -0.5, causal,
                                   torch.cuda.current_stream().cuda_stream)


def same_up_to_sum_order(got, want, name):
    """Two bf16 roundings of fp32 sums whose terms were added in different
    orders: equal, or one bf16 step apart (2^-7 relative at most), plus a
    floor of 1e-5 of the tensor's largest value for sums that cancel."""
    g, w = got.float(), want.float()
    tol = 2.0 ** -7 * torch.maximum(g.abs(), w.abs()) + 1e-5 * w.abs().max()
    bad = (g - w).abs() > tol
    assert not bool(bad.any()), f"{name}: {int(bad.sum())} elements differ beyond sum order"


def run_twice_and_compare(ta, q, k, v, o, lse, do, causal):
    ref = ta.attn_bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    grouped = q.shape[1] > k.shape[1]
    outs = []
    for call in range(2):
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
        st = raw_noalloc(ta, q, k, v, o, lse, do, dq, dk, dv, causal)
        assert st == ta.ATTN_OK, ta.attn_status_string(st)
        torch.cuda.synchronize()
        assert ta.attn_last_device_status() == 0
        # dQ is summed over key tiles by fp32 reduce-adds in no fixed order.
        same_up_to_sum_order(dq, ref[0], f"call {call}: dq")
        if grouped:
            # Grouped heads: a key tile's query heads are split over blocks,
            # and dK / dV are fp32 reduce-adds too.
            same_up_to_sum_order(dk, ref[1], f"call {call}: dk")
            same_up_to_sum_order(dv, ref[2], f"call {call}: dv")
        else:
            # One block owns each key tile: dK and dV come out of the same
            # kernels in the same order, bit for bit.
            assert torch.equal(dk, ref[1]), f"call {call}: dk"
            assert torch.equal(dv, ref[2]), f"call {call}: dv"
        outs.append((dq, dk, dv))
    return outs


@pytest.mark.parametrize("shape,causal", [((1, 4, 2, 384, 128), True),
                                          ((2, 2, 2, 200, 64), False)])
def test_noalloc_matches_workspace_backward_twice(ta, orc, shape, causal):
    B, Hq, Hkv, N, D = shape
    x = make_qkv(B, Hq, Hkv, N, D, seed=31, with_do=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=causal)
    outs = run_twice_and_compare(ta, q, k, v, o, lse, do, causal)
    # The second call's gradients against the exact fp64 gradient.
    rng = np.random.default_rng(5)
    q_rows = np.unique(np.concatenate([[0, B * Hq * N - 1], rng.integers(0, B * Hq * N, 24)]))
    k_rows = np.unique(np.concatenate([[0, B * Hkv * N - 1], rng.integers(0, B * Hkv * N, 24)]))
    ref = orc.backward_sampled(*(to_oracle(x[n]) for n in ("q", "k", "v", "do")),
                               scale=1 / math.sqrt(D), causal=causal, q_rows=q_rows, k_rows=k_rows)
    dq, dk, dv = outs[1]
    qr, kr = torch.from_numpy(q_rows).cuda(), torch.from_numpy(k_rows).cuda()
    check_grad(dq.reshape(-1, D)[qr], ref["dq"], "noalloc dq")
    check_grad(dk.reshape(-1, D)[kr], ref["dk"], "noalloc dk")
    check_grad(dv.reshape(-1, D)[kr], ref["dv"], "noalloc dv")


def test_noalloc_shape_that_fills_the_scratch(ta):
    """One head of D = 128 at N = 64526 needs exactly the scratch's size."""
    B, Hq, Hkv, N, D = 1, 1, 1, 64526, 128
    assert ta.attn_bwd_workspace_size(B, Hq, Hkv, N, D) == ta.ATTN_BWD_NOALLOC_SCRATCH_BYTES
    x = make_qkv(B, Hq, Hkv, N, D, seed=32, with_do=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=True)
    run_twice_and_compare(ta, q, k, v, o, lse, do, True)


def test_noalloc_rejects_shapes_beyond_the_scratch(ta):
    """Too large for the fixed scratch: a clear error, nothing launched."""
    B, Hq, Hkv, N, D = 1, 16, 16, 16384, 128
    assert ta.attn_bwd_workspace_size(B, Hq, Hkv, N, D) > ta.ATTN_BWD_NOALLOC_SCRATCH_BYTES
    A = 0x10000
    st = ta.raw_attn_bwd_noalloc(A, A, A, A, A, A, A, A, A, B, Hq, Hkv, N, D, 0.1, 1, None)
    assert st == ta.ATTN_ERR_UNSUPPORTED
