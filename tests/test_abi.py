"""Host-only checks of the C ABI: the library loads, exports every entry
point include/tattn.h declares, and rejects bad arguments before touching
any memory (no GPU needed: invalid calls return before any CUDA call)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ta():
    import tiled_attention_02_gb300 as ta
    ta.build()
    return ta


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(attn_\w+)\s*\(", text))
    return names


def test_header_declares_entry_points():
    assert {"attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_status_string",
            "attn_last_device_status"} <= declared_functions()


def test_library_exports_every_declared_symbol(ta):
    L = ta.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(ta.EXPORTED) == declared_functions()


def test_status_strings(ta):
    for code in range(6):
        s = ta.attn_status_string(code)
        assert s.startswith("ATTN_")
    assert "unknown" in ta.attn_status_string(99)


A = 0x10000   # fake, 16-byte aligned "device" addresses: never dereferenced


def fwd(ta, **kw):
    args = dict(q=A, k=A, v=A, bias=None, o=A, lse=None, B=1, Hq=2, Hkv=1, N=256, D=128,
                scale=0.125, causal=0, emit=None, stream=None)
    args.update(kw)
    return ta.raw_attn_fwd(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(o=None), 1),
    (dict(q=A + 2), 1), (dict(k=A + 8), 1), (dict(o=A + 4), 1),
    (dict(bias=A + 2), 1), (dict(emit=A + 1), 1), (dict(lse=A + 3), 1),
    (dict(D=72), 2), (dict(D=112), 2), (dict(D=256), 2), (dict(D=0), 1), (dict(D=-64), 1),
    (dict(Hkv=3), 1), (dict(Hkv=0), 1), (dict(B=-1), 1), (dict(N=-5), 1),
    (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1),
    # B*Hq*ceil(N/128) = 2^31, one past the bound: by heads and by length
    (dict(B=1 << 16, Hq=1 << 15, Hkv=1 << 15, N=128), 2),
    (dict(B=1, Hq=256, Hkv=256, N=1 << 30), 2),
])
def test_fwd_rejects_bad_arguments(ta, kw, code):
    assert fwd(ta, **kw) == code


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=0), dict(N=0), dict(B=0, q=None)])
def test_fwd_empty_problem_is_ok_without_launch(ta, kw):
    assert fwd(ta, **kw) == 0


def bwd(ta, **kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, do=A, dq=A, dk=A, dv=A, B=1, Hq=2, Hkv=2, N=256,
                D=64, scale=0.125, causal=1, ws=A, ws_bytes=1 << 30, stream=None)
    args.update(kw)
    return ta.raw_attn_bwd(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(lse=None), 1), (dict(do=None), 1), (dict(ws=None), 1), (dict(dk=A + 2), 1),
    (dict(ws=A + 16), 1), (dict(ws_bytes=1000), 1), (dict(D=32), 2), (dict(Hkv=3), 1),
    (dict(B=1 << 16, Hq=1 << 15, Hkv=1 << 15, N=128), 2),
    (dict(B=1, Hq=256, Hkv=256, N=1 << 30), 2),
])
def test_bwd_rejects_bad_arguments(ta, kw, code):
    assert bwd(ta, **kw) == code


def test_workspace_size(ta):
    # fp32 dQ accumulator + two fp32 per-row arrays padded to 128-row tiles,
    # each region rounded up to 256 bytes
    assert ta.attn_bwd_workspace_size(1, 16, 16, 16384, 128) == (16 * 16384 * 128 * 4
                                                                 + 2 * 16 * 16384 * 4)
    assert ta.attn_bwd_workspace_size(1, 1, 1, 3, 64) == 768 + 2 * 512
    assert ta.attn_bwd_workspace_size(1, 1, 1, 5, 64) == 1280 + 2 * 512
    # grouped heads: + fp32 dK and dV accumulators [B,Hkv,N,D] (66560 bytes each here)
    assert ta.attn_bwd_workspace_size(2, 3, 1, 130, 64) == (6 * 130 * 64 * 4 + 2 * 6 * 256 * 4
                                                            + 2 * 66560)
    assert ta.attn_bwd_workspace_size(0, 1, 1, 3, 64) == 0
    # D = 80 and 96 rows: 320- and 384-byte fp32 rows
    assert ta.attn_bwd_workspace_size(1, 1, 1, 3, 80) == 1024 + 2 * 512
    assert ta.attn_bwd_workspace_size(1, 1, 1, 3, 96) == 1280 + 2 * 512
    assert ta.attn_bwd_workspace_size(1, 1, 1, 3, 112) == 0


@pytest.mark.parametrize("window", [0, -1, -128])
def test_window_entry_points_reject_bad_window(ta, window):
    """window must be >= 1; rejected on the host before anything runs."""
    assert ta.raw_attn_fwd_window(A, A, A, None, A, A, 1, 2, 2, 256, 64, 0.125, window, None,
                                  None) == 1
    assert ta.raw_attn_bwd_window(A, A, A, A, A, A, A, A, A, 1, 2, 2, 256, 64, 0.125, window, A,
                                  1 << 30, None) == 1


def test_window_entry_points_check_shapes_like_the_plain_ones(ta):
    assert ta.raw_attn_fwd_window(A, A, A, None, A, A, 1, 2, 2, 256, 72, 0.125, 64, None,
                                  None) == 2
    assert ta.raw_attn_fwd_window(A, A, A, None, A, A, 1, 2, 2, 0, 64, 0.125, 64, None,
                                  None) == 0
    assert ta.raw_attn_bwd_window(A + 2, A, A, A, A, A, A, A, A, 1, 2, 2, 256, 64, 0.125, 64, A,
                                  1 << 30, None) == 1


def test_decode_workspace_size(ta):
    # slots = 512 + B*Hkv - 1 segments of G = Hq/Hkv heads: m and l [slots, G],
    # o [slots, G, D], fp32, each region rounded up to 256 bytes
    r256 = lambda x: (x + 255) // 256 * 256
    assert ta.attn_decode_workspace_size(1, 1, 1, 100, 64) == 2 * 512 * 4 + 512 * 64 * 4
    assert ta.attn_decode_workspace_size(2, 8, 2, 16384, 128) == 2 * r256(515 * 4 * 4) + 515 * 4 * 128 * 4
    assert ta.attn_decode_workspace_size(2, 8, 2, 100, 128) == ta.attn_decode_workspace_size(2, 8, 2, 16384, 128)
    assert ta.attn_decode_workspace_size(1, 32, 1, 1024, 64) == 0     # 32 query heads per kv head
    assert ta.attn_decode_workspace_size(1, 2, 2, 1024, 72) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(o=A + 2), 1), (dict(ws=None), 1), (dict(ws=A + 16), 1),
    (dict(ws_bytes=10), 1), (dict(D=72), 2), (dict(Hq=34, Hkv=2), 2), (dict(Hkv=3), 1),
    (dict(scale=float("nan")), 1),
])
def test_decode_rejects_bad_arguments(ta, kw, code):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, Hq=4, Hkv=2, N=1000, D=64, scale=0.125, ws=A,
                ws_bytes=1 << 30, stream=None)
    args.update(kw)
    assert ta.raw_attn_decode(**args) == code


def test_decode_empty_problem_is_ok(ta):
    assert ta.raw_attn_decode(A, A, A, A, A, 0, 4, 2, 100, 64, 0.125, A, 1 << 30, None) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(N=254), 2),            # residual rows must be 16-byte multiples
    (dict(bias=A + 4), 2),       # 16-byte aligned residual bases
    (dict(gout=A + 2), 1),       # fp32 alignment
    (dict(D=72), 2), (dict(lse=None), 1),
])
def test_bwd_residual_rejects(ta, kw, code):
    args = dict(q=A, k=A, v=A, o=A, lse=A, do=A, bias=A, gin=A, dq=A, dk=A, dv=A, gout=A, B=1,
                Hq=2, Hkv=2, N=256, D=64, scale=0.125, causal=1, ws=A, ws_bytes=1 << 30,
                stream=None)
    args.update(kw)
    assert ta.raw_attn_bwd_residual(args["q"], args["k"], args["v"], args["o"], args["lse"],
                                    args["do"], args["bias"], args["gin"], args["dq"], args["dk"],
                                    args["dv"], args["gout"], args["B"], args["Hq"], args["Hkv"],
                                    args["N"], args["D"], args["scale"], args["causal"],
                                    args["ws"], args["ws_bytes"], args["stream"]) == code


def noalloc(ta, **kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, do=A, dq=A, dk=A, dv=A, B=1, Hq=2, Hkv=2, N=256, D=64,
                scale=0.125, causal=1, stream=None)
    args.update(kw)
    return ta.raw_attn_bwd_noalloc(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0, D=0), 1),                      # D is checked before the empty shortcut
    (dict(B=0, scale=float("nan")), 1),       # and so is the scale
    (dict(N=0, D=72), 2),
    (dict(B=0), 0), (dict(Hq=0), 0), (dict(N=0), 0),
    (dict(B=-1), 1), (dict(Hkv=3), 1), (dict(D=72), 2), (dict(q=None), 1),
])
def test_noalloc_codes_match_attn_bwd(ta, kw, code):
    """attn_bwd_noalloc returns the code attn_bwd would for the same sizes,
    empty problems included, without launching anything."""
    assert noalloc(ta, **kw) == code
    b = dict(kw)
    for key in ("do", "dq", "dk", "dv"):
        b.pop(key, None)
    assert bwd(ta, **b) == code


def test_noalloc_scratch_constant_is_the_headers(ta):
    text = open(os.path.join(ROOT, "include", "tattn.h")).read()
    m = re.search(r"#define\s+ATTN_BWD_NOALLOC_SCRATCH_BYTES\s+(\d+)", text)
    assert m and int(m.group(1)) == ta.ATTN_BWD_NOALLOC_SCRATCH_BYTES


def test_noalloc_rejects_one_row_past_the_scratch(ta):
    """The C entry point's own limit sits exactly at the header's size: one
    head of D = 128 fits up to N = 64526 rows (workspace == scratch) and is
    refused at N = 64527, before any launch."""
    S = ta.ATTN_BWD_NOALLOC_SCRATCH_BYTES
    assert ta.attn_bwd_workspace_size(1, 1, 1, 64526, 128) == S
    assert ta.attn_bwd_workspace_size(1, 1, 1, 64527, 128) > S
    assert noalloc(ta, Hq=1, Hkv=1, N=64527, D=128) == ta.ATTN_ERR_UNSUPPORTED
    assert noalloc(ta, Hq=4, Hkv=2, N=64527, D=128) == ta.ATTN_ERR_UNSUPPORTED


def _cpu_bwd_args(B=1, Hq=2, Hkv=1, N=64, D=64):
    import torch
    bf = torch.bfloat16
    q = torch.zeros(B, Hq, N, D, dtype=bf)
    k = torch.zeros(B, Hkv, N, D, dtype=bf)
    return dict(q=q, k=k, v=k.clone(), o=q.clone(), lse=torch.zeros(B, Hq, N), do=q.clone())


@pytest.mark.parametrize("fn", ["attn_bwd", "attn_bwd_noalloc"])
@pytest.mark.parametrize("bad", ["dq_shape", "dk_shape", "dv_dtype", "dq_layout", "dk_device"])
def test_wrappers_reject_bad_output_buffers(ta, fn, bad):
    """Caller-given dq/dk/dv go through the same checks as the inputs, before
    any call into the library (CPU tensors here: nothing can launch)."""
    import torch
    a = _cpu_bwd_args()
    q, k = a["q"], a["k"]
    if bad == "dq_shape":
        a["dq"], err = torch.zeros(1, 2, 63, 64, dtype=torch.bfloat16), ValueError
    elif bad == "dk_shape":
        a["dk"], err = torch.zeros_like(q), ValueError
    elif bad == "dv_dtype":
        a["dv"], err = torch.zeros(k.shape), TypeError
    elif bad == "dq_layout":
        a["dq"], err = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16).transpose(2, 3), ValueError
    else:
        a["dk"], err = torch.zeros_like(k), TypeError   # right shape, but not on the device
    kw = {n: a.pop(n) for n in ("dq", "dk", "dv") if n in a}
    with pytest.raises(err):
        getattr(ta, fn)(*a.values(), **kw)
