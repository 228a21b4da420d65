"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

This package is the slow, obviously-correct statement of what the CUDA
library computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it.  It shares no code with the CUDA
path and never imports the product package; it takes plain numpy arrays.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, one
query row at a time from the definition).  This module only compiles it with
gcc, marshals numpy arrays, and composes its steps:

* :func:`forward` -- O, LSE and (optionally) the pre-softmax logits.
* :func:`backward` -- exact dQ, dK, dV for every row (small shapes).
* :func:`backward_sampled` -- dQ for chosen query rows and dK/dV for chosen
  key rows, for shapes too large to do in full.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, special cases, finite differences, brute force on
tiny inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
# Tests that plant a mistake in a copy of the C source point this at the
# mutant's library (see tests/test_oracle_mutants.py).
_LIB_OVERRIDE = os.environ.get("TATTN_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``_build/liboracle.so`` (gcc, OpenMP).

    ``-ffp-contract=off`` keeps multiply and add separate so the x86 and Arm
    builds round identically; no fast-math flags are used.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
               "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_LIB_OVERRIDE or build())
            lib.orc_set_threads.argtypes = [ctypes.c_int]
            lib.orc_get_threads.restype = ctypes.c_int
            lib.orc_fwd_rows.argtypes = [_ptr, _ptr, _ptr, _ptr, _i64, _i64, _i64, _i64, _i64,
                                         _dbl, ctypes.c_int, _i64, _ptr, _i64, ctypes.c_int,
                                         _ptr, _ptr, _ptr]
            lib.orc_delta_rows.argtypes = [_ptr, _ptr, _i64, _ptr, _i64, _ptr]
            lib.orc_bwd_dq_rows.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _i64,
                                            _i64, _i64, _i64, _i64, _dbl, ctypes.c_int, _i64,
                                            _ptr, _i64, _ptr, _ptr]
            lib.orc_bwd_dkv_rows.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                                             _i64, _i64, _i64, _i64, _i64, _dbl, ctypes.c_int,
                                             _i64, _ptr, _i64, _ptr, _ptr]
            _lib = lib
    return _lib


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def get_threads() -> int:
    return int(_load().orc_get_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a) -> int | None:
    return None if a is None else a.ctypes.data


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B,H,N,D]")
    B, Hq, N, D = q.shape
    Bk, Hkv, Nk, Dk = k.shape
    if (Bk, Nk, Dk) != (B, N, D) or v.shape != k.shape or Hkv == 0 or Hq % Hkv:
        raise ValueError(f"incompatible shapes q{q.shape} k{k.shape} v{v.shape}")
    return B, Hq, Hkv, N, D


def _window(causal, window) -> int:
    """0 for no window; else the window length W >= 1 (causal only)."""
    if window is None:
        return 0
    w = int(window)
    if w < 1 or not causal:
        raise ValueError("a sliding window needs causal=True and W >= 1")
    return w


def _rows(rows, total):
    if rows is None:
        return None, total
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    if r.size and (r.min() < 0 or r.max() >= total):
        raise ValueError("row index out of range")
    return r, int(r.size)


def forward(q, k, v, *, scale: float, causal: bool, bias=None, rows=None,
            emit_logits: bool = False, logits_out=None, window=None):
    """Exact attention forward in fp64.

    q [B,Hq,N,D], k/v [B,Hkv,N,D] (any float dtype; widened to float64, which
    holds bf16 and fp32 inputs exactly);
    bias [B,Hq,N,N] or None (widened to float64); with ``rows`` given, bias
    may instead be [nrows, N]: the bias rows of the requested rows only.
    rows: flat query-row indices ``(b*Hq + h)*N + i`` or None for all rows.
    window: None, or W >= 1 with causal=True: key j is kept for query i iff
    i - W < j <= i (sliding window over the W most recent keys).

    Returns dict with ``o`` ([B,Hq,N,D] when rows is None, else [nrows,D]),
    ``lse`` (matching) and, when ``emit_logits``, ``logits`` ([B,Hq,N,N] or
    [nrows,N]) holding s_ij for kept keys and NaN where the causal mask or
    the window hides the key.  ``logits_out`` may be given (float64, right shape) to reuse a
    buffer; it may be the same array as ``bias`` when rows is None.
    """
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, N, D = _shapes(q, k, v)
    w = _window(causal, window)
    total = B * Hq * N
    r, nrows = _rows(rows, total)
    if bias is not None:
        if not (isinstance(bias, np.ndarray) and bias.dtype == np.float64
                and bias.flags.c_contiguous):
            bias = _f64(bias)
        per_request = r is not None and bias.shape == (nrows, N)
        if bias.shape != (B, Hq, N, N) and not per_request:
            raise ValueError("bias must be [B,Hq,N,N] (or [nrows,N] with rows)")
    else:
        per_request = False
    o = np.empty((nrows, D), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    logits = None
    if emit_logits:
        if logits_out is not None:
            if (logits_out.dtype != np.float64 or not logits_out.flags.c_contiguous
                    or logits_out.size != nrows * N):
                raise ValueError("logits_out must be contiguous float64 of nrows*N")
            if logits_out is bias and r is not None and not per_request:
                raise ValueError("logits_out may alias a full bias only for all rows")
            logits = logits_out
        else:
            logits = np.empty((nrows, N), dtype=np.float64)
    lib.orc_fwd_rows(_p(q), _p(k), _p(v), _p(bias), B, Hq, Hkv, N, D, float(scale),
                     int(bool(causal)), w, _p(r), nrows, int(per_request), _p(o), _p(lse),
                     _p(logits))
    out = {}
    if r is None:
        out["o"] = o.reshape(B, Hq, N, D)
        out["lse"] = lse.reshape(B, Hq, N)
    else:
        out["o"], out["lse"] = o, lse
    if emit_logits:
        if causal:
            # Keys above the diagonal (and, with a window, keys j <= i - W)
            # are not part of J_i: mark them NaN.
            if r is None:
                iu = np.triu_indices(N, 1)
                il = np.tril_indices(N, -w) if w else None
                for lg in logits.reshape(B * Hq, N, N):
                    lg[iu] = np.nan
                    if w:
                        lg[il] = np.nan
            else:
                lg = logits.reshape(nrows, N)
                jj, ii = np.arange(N)[None, :], (r % N)[:, None]
                lg[jj > ii] = np.nan
                if w:
                    lg[jj <= ii - w] = np.nan
        out["logits"] = logits.reshape(B, Hq, N, N) if r is None else logits.reshape(nrows, N)
    return out


def delta(dO, o_rows, rows=None):
    """Delta_i = sum_d dO_i[d] O_i[d] for the given rows (o_rows in row order)."""
    lib = _load()
    dO = _f64(dO)
    D = dO.shape[-1]
    o_rows = _f64(o_rows).reshape(-1, D)
    r, nrows = _rows(rows, dO.size // D)
    if o_rows.shape[0] != nrows:
        raise ValueError("o_rows must hold one row per requested row")
    out = np.empty((nrows,), dtype=np.float64)
    lib.orc_delta_rows(_p(dO), _p(o_rows), D, _p(r), nrows, _p(out))
    return out


def backward(q, k, v, dO, *, scale: float, causal: bool, window=None, bias=None, grad_in=None):
    """Exact dQ, dK, dV (fp64) for every row; returns dict with o, lse too.

    bias [B,Hq,N,N] (the forward's additive logit bias) and grad_in
    [B,Hq,N,N] (the gradient arriving at this layer's logits from the next
    layer of a block residual chain) are optional.  With either given, the
    result also holds ``dlogits`` [B,Hq,N,N]: the total logit gradient
    dS = P o (dP - Delta) + grad_in on the kept keys and 0 elsewhere, which
    is the gradient w.r.t. the bias and the ``grad_in`` of the previous
    layer."""
    lib = _load()
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, Hq, Hkv, N, D = _shapes(q, k, v)
    w = _window(causal, window)
    bias = None if bias is None else _f64(bias)
    grad_in = None if grad_in is None else _f64(grad_in)
    for name, a in (("bias", bias), ("grad_in", grad_in)):
        if a is not None and a.shape != (B, Hq, N, N):
            raise ValueError(f"{name} must be [B,Hq,N,N]")
    fw = forward(q, k, v, scale=scale, causal=causal, window=window, bias=bias)
    lse = np.ascontiguousarray(fw["lse"].reshape(-1))
    dlt = delta(dO, fw["o"].reshape(-1, D))
    dq = np.empty((B * Hq * N, D), dtype=np.float64)
    dk = np.empty((B * Hkv * N, D), dtype=np.float64)
    dv = np.empty((B * Hkv * N, D), dtype=np.float64)
    res = bias is not None or grad_in is not None
    dl = np.empty((B * Hq * N, N), dtype=np.float64) if res else None
    lib.orc_bwd_dq_rows(_p(q), _p(k), _p(v), _p(dO), _p(lse), _p(dlt), _p(bias), _p(grad_in),
                        B, Hq, Hkv, N, D, float(scale), int(bool(causal)), w, None, B * Hq * N,
                        _p(dq), _p(dl))
    lib.orc_bwd_dkv_rows(_p(q), _p(k), _p(v), _p(dO), _p(lse), _p(dlt), _p(bias), _p(grad_in),
                         B, Hq, Hkv, N, D, float(scale), int(bool(causal)), w, None, B * Hkv * N,
                         _p(dk), _p(dv))
    out = {"o": fw["o"], "lse": fw["lse"], "dq": dq.reshape(B, Hq, N, D),
           "dk": dk.reshape(B, Hkv, N, D), "dv": dv.reshape(B, Hkv, N, D)}
    if res:
        out["dlogits"] = dl.reshape(B, Hq, N, N)
    return out


def backward_sampled(q, k, v, dO, *, scale: float, causal: bool, q_rows, k_rows, window=None,
                     bias=None, grad_in=None):
    """dQ at flat query rows ``q_rows`` and dK/dV at flat key rows ``k_rows``.

    bias and grad_in: as for ``backward`` ([B,Hq,N,N] or None), read only at
    the query rows involved, so an array filled at those rows alone serves.

    Key row flat index is ``(b*Hkv + g)*N + j``.  The statistics LSE and Delta
    are computed by the oracle's own forward pass over every query row of the
    heads involved (a key row needs all the query rows that attend to it).
    Returns dict with dq [len(q_rows), D], dk and dv [len(k_rows), D], and
    dlogits [len(q_rows), N]: the total logit gradient dS of those rows (0 at
    keys outside J_i), the grad_in of the layer below in a residual chain.
    """
    lib = _load()
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, Hq, Hkv, N, D = _shapes(q, k, v)
    w = _window(causal, window)
    group = Hq // Hkv
    bias = None if bias is None else _f64(bias)
    grad_in = None if grad_in is None else _f64(grad_in)
    for name, t in (("bias", bias), ("grad_in", grad_in)):
        if t is not None and t.shape != (B, Hq, N, N):
            raise ValueError(f"{name} must be [B,Hq,N,N]")
    qr, nq = _rows(q_rows, B * Hq * N)
    kr, nk = _rows(k_rows, B * Hkv * N)
    # Query rows whose statistics are needed.
    need = set() if qr is None else {int(x) for x in qr}
    # A key row j of kv head (b, g) needs every query row of the group's
    # heads that attends to it: j <= i < j + W under the causal mask (W = N
    # without a window), all i otherwise.
    spans = {}
    for x in (kr if kr is not None else []):
        bg, j = divmod(int(x), N)
        b, g = divmod(bg, Hkv)
        lo = j if causal else 0
        hi = min(N, j + w) if w else N
        for h in range(g * group, (g + 1) * group):
            spans.setdefault(b * Hq + h, []).append((lo, hi))
    for bh, sp in spans.items():
        for lo, hi in sp:
            need |= set(range(bh * N + lo, bh * N + hi))
    stat_rows = np.asarray(sorted(need), dtype=np.int64)
    lse = np.zeros((B * Hq * N,), dtype=np.float64)
    dlt = np.zeros((B * Hq * N,), dtype=np.float64)
    if stat_rows.size:
        fw = forward(q, k, v, scale=scale, causal=causal, rows=stat_rows, window=window,
                     bias=bias)
        lse[stat_rows] = fw["lse"]
        dlt[stat_rows] = delta(dO, fw["o"], stat_rows)
    dq = np.empty((nq, D), dtype=np.float64)
    dk = np.empty((nk, D), dtype=np.float64)
    dv = np.empty((nk, D), dtype=np.float64)
    dl = np.empty((nq, N), dtype=np.float64)
    if nq:
        lib.orc_bwd_dq_rows(_p(q), _p(k), _p(v), _p(dO), _p(lse), _p(dlt), _p(bias),
                            _p(grad_in), B, Hq, Hkv, N, D, float(scale), int(bool(causal)), w,
                            _p(qr), nq, _p(dq), _p(dl))
    if nk:
        lib.orc_bwd_dkv_rows(_p(q), _p(k), _p(v), _p(dO), _p(lse), _p(dlt), _p(bias),
                             _p(grad_in), B, Hq, Hkv, N, D, float(scale), int(bool(causal)), w,
                             _p(kr), nk, _p(dk), _p(dv))
    return {"dq": dq, "dk": dk, "dv": dv, "dlogits": dl}
