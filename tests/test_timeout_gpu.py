"""The bounded-wait failure path on the GPU, without a fault: a test hook
leaves out thread block 0's first K tile load, so one pipeline wait can never
complete.  With every wait bounded by 1 ms, the kernel must record
ATTN_ERR_TIMEOUT in the device status word and return -- no trap, no hang --
the blocks that were not starved must still produce correct rows, and the
next ordinary call on the same stream must pass oracle parity."""
import math
import time

import numpy as np
import pytest

from helpers import check_lse, check_o, make_qkv, to_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ta():
    import tiled_attention_02_gb300 as ta
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ta.build()
    return ta


@pytest.mark.parametrize("D,causal", [(64, True), (128, False)])
def test_starved_wait_times_out_and_context_stays_usable(ta, orc, D, causal):
    B, Hq, Hkv, N = 1, 2, 2, 512
    x = make_qkv(B, Hq, Hkv, N, D, seed=41)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, N), float("nan"), device="cuda")
    stream = torch.cuda.current_stream()
    assert ta.attn_last_device_status() == ta.ATTN_OK   # nothing pending before

    t0 = time.monotonic()
    st = ta.raw_attn_debug_fwd_timeout(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), B, Hq, Hkv, N, D, 1 / math.sqrt(D),
                                       causal, 1_000_000, stream.cuda_stream)
    assert st == ta.ATTN_OK, ta.attn_status_string(st)
    status = ta.attn_last_device_status()   # synchronises the stream
    elapsed = time.monotonic() - t0
    assert status == ta.ATTN_ERR_TIMEOUT, ta.attn_status_string(status)
    assert elapsed < 10.0, f"the starved launch took {elapsed:.1f} s to return"
    # The status word was read and cleared.
    assert ta.attn_last_device_status() == ta.ATTN_OK

    # Block 0 gave up on its query tile(s): those rows stay NaN, in whole
    # 128-row tiles.  Every row another block wrote is correct.
    ref = orc.forward(to_oracle(x["q"]), to_oracle(x["k"]), to_oracle(x["v"]),
                      scale=1 / math.sqrt(D), causal=causal)
    rows_nan = torch.isnan(lse.reshape(-1)).cpu().numpy()
    assert 0 < rows_nan.sum() < B * Hq * N and rows_nan.sum() % 128 == 0
    written = ~rows_nan
    check_o(o.reshape(-1, D)[torch.from_numpy(written).cuda()],
            ref["o"].reshape(-1, D)[written], "rows of the blocks that were not starved")
    check_lse(lse.reshape(-1)[torch.from_numpy(written).cuda()],
              ref["lse"].reshape(-1)[written], "rows of the blocks that were not starved")

    # The context is still usable: an ordinary call on the same stream.
    o2, lse2 = ta.attn_fwd(q, k, v, causal=causal, stream=stream)
    assert ta.attn_last_device_status(stream) == ta.ATTN_OK
    check_o(o2, ref["o"], "ordinary call after the timeout")
    check_lse(lse2, ref["lse"], "ordinary call after the timeout")


def test_timeout_hook_rejects_a_zero_limit(ta):
    A = 0x10000
    assert ta.raw_attn_debug_fwd_timeout(A, A, A, A, None, 1, 1, 1, 128, 64, 0.125, 0, 0,
                                         None) == ta.ATTN_ERR_INVALID
