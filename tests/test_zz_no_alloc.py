"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (an engine that owns all device allocations and gives libraries no
allocator, or code that must avoid the synchronisation cudaMalloc/cudaFree
can cause).  It uses the library's fixed device scratch instead of a
caller workspace.  Checked through the C ABI against attn_bwd on the same
inputs, on two calls in a row (the scratch keeps the previous call's
contents, which must not matter).  Kept in its own file, collected last."""
import pytest

from helpers import GRAD_MAX_ABS, make_qkv

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


@pytest.mark.parametrize("shape,causal", [((1, 4, 2, 384, 128), True),
                                          ((2, 2, 2, 200, 64), False)])
def test_noalloc_matches_workspace_backward_twice(ta, shape, causal):
    B, Hq, Hkv, N, D = shape
    x = make_qkv(B, Hq, Hkv, N, D, seed=31, with_do=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(q, k, v, causal=causal)
    ref = ta.attn_bwd(q, k, v, o, lse, do, causal=causal)
    for call in range(2):
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
        st = raw_noalloc(ta, q, k, v, o, lse, do, dq, dk, dv, causal)
        assert st == ta.ATTN_OK, ta.attn_status_string(st)
        torch.cuda.synchronize()
        assert ta.attn_last_device_status() == 0
        for got, want, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
            err = (got.float() - want.float()).abs().max().item()
            assert err <= GRAD_MAX_ABS, f"call {call}: {name} max-abs {err:.3e}"


def test_noalloc_rejects_shapes_beyond_the_scratch(ta):
    """Too large for the fixed scratch: a clear error, nothing launched."""
    B, Hq, Hkv, N, D = 1, 16, 16, 16384, 128
    assert ta.attn_bwd_workspace_size(B, Hq, Hkv, N, D) > ta.ATTN_BWD_NOALLOC_SCRATCH_BYTES
    A = 0x10000
    st = ta.raw_attn_bwd_noalloc(A, A, A, A, A, A, A, A, A, B, Hq, Hkv, N, D, 0.1, 1, None)
    assert st == ta.ATTN_ERR_UNSUPPORTED
