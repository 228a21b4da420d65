"""Pins for the fp64 oracle: checks against facts the pages and the mathematics
fix, none of which re-types the oracle's own formula.

Each pin names the passage it follows (page title and section):
  [FA-Triton]   "FlashAttention原理与Triton实战：突破Attention显存瓶颈"
  [FA-kwkr]     kwkr.cn/news/592482 (FlashAttention online-softmax tutorial)
  [BlockRes]    Block Attention Residual Triton kernel (iqiancheng.github.io)
  [Day26]       blog.ans20xx.com/posts/ai/day26 (operator-level speedups)
"""
import math

import numpy as np
import pytest

RNG = np.random.default_rng(1234)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(3, 3), (4, 2)])
def test_zero_query_gives_mean_of_values(orc, causal, Hq, Hkv):
    """Q = 0 makes every logit 0, so softmax is uniform over the kept keys:
    O_i is the mean of the kept rows of V and LSE_i = ln |J_i|
    ([FA-kwkr] 2.1 softmax definition; causal key set from [FA-kwkr] 3.4)."""
    B, N, D = 2, 7, 5
    q = np.zeros((B, Hq, N, D))
    k, v = rand(B, Hkv, N, D), rand(B, Hkv, N, D)
    out = orc.forward(q, k, v, scale=0.37, causal=causal)
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            for i in range(N):
                kept = v[b, h // g, : i + 1] if causal else v[b, h // g]
                np.testing.assert_allclose(out["o"][b, h, i], kept.mean(axis=0), rtol=0, atol=1e-14)
                assert abs(out["lse"][b, h, i] - math.log(len(kept))) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(orc, causal):
    """sum_j P_ij = 1: with every value row equal to 1, every output is 1
    ([FA-kwkr] 2.1, the division by l)."""
    B, H, N, D = 1, 2, 9, 3
    out = orc.forward(rand(B, H, N, D, scale=3), rand(B, H, N, D, scale=3), np.ones((B, H, N, D)),
                      scale=0.5, causal=causal)
    np.testing.assert_allclose(out["o"], 1.0, rtol=0, atol=1e-14)


def test_two_keys_is_logistic(orc):
    """Two keys: P_i0 = 1 / (1 + exp(s_i1 - s_i0)), the logistic function, so
    O_i = sigma(s0 - s1) v0 + sigma(s1 - s0) v1 and
    LSE_i = max(s) + log1p(exp(-|s0 - s1|))."""
    scale = 0.8
    q = np.array([[[[1.5], [-0.25]]]])          # B=H=1, N=2, D=1
    k = np.array([[[[0.5], [-2.0]]]])
    v = np.array([[[[3.0], [-7.0]]]])
    out = orc.forward(q, k, v, scale=scale, causal=False)
    for i in range(2):
        s0, s1 = scale * q[0, 0, i, 0] * k[0, 0, 0, 0], scale * q[0, 0, i, 0] * k[0, 0, 1, 0]
        p0 = 1.0 / (1.0 + math.exp(s1 - s0))
        want = p0 * 3.0 + (1.0 - p0) * -7.0
        assert abs(out["o"][0, 0, i, 0] - want) < 1e-14
        assert abs(out["lse"][0, 0, i] - (max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-14


def test_hard_attention_limit(orc):
    """A logit far above the others takes all the weight: O_i = v_{j*}."""
    B, H, N, D = 1, 2, 6, 4
    q, k, v = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    star = RNG.integers(0, N, size=(B, H, N))
    bias = np.zeros((B, H, N, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                bias[b, h, i, star[b, h, i]] = 2000.0
    out = orc.forward(q, k, v, scale=0.3, causal=False, bias=bias)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                np.testing.assert_array_equal(out["o"][b, h, i], v[b, h, star[b, h, i]])


# --------------------------------------------------------------- causal cases

def test_causal_first_row_is_first_value_row(orc):
    """Under the causal mask query 0 sees only key 0, so O_0 = v_0 exactly and
    LSE_0 = s_00 ([FA-kwkr] 3.4: triu(diagonal=1) is masked; [Day26] tril keep mask)."""
    B, H, N, D = 2, 3, 8, 16
    q, k, v = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    out = orc.forward(q, k, v, scale=0.25, causal=True)
    np.testing.assert_array_equal(out["o"][:, :, 0], v[:, :, 0])
    s00 = 0.25 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    np.testing.assert_allclose(out["lse"][:, :, 0], s00, rtol=0, atol=1e-13)


def test_causal_last_row_equals_unmasked(orc):
    """The last query row keeps every key, so it matches the unmasked result."""
    B, H, N, D = 1, 2, 11, 8
    q, k, v = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    c = orc.forward(q, k, v, scale=0.3, causal=True)
    f = orc.forward(q, k, v, scale=0.3, causal=False)
    np.testing.assert_array_equal(c["o"][:, :, -1], f["o"][:, :, -1])
    np.testing.assert_array_equal(c["lse"][:, :, -1], f["lse"][:, :, -1])


def test_causal_prefix_equals_truncated_sequence(orc):
    """Causal row i depends on keys 0..i only: it equals row i of the same
    problem cut to length i+1 and run without a mask."""
    B, H, N, D = 1, 2, 9, 4
    q, k, v = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    c = orc.forward(q, k, v, scale=0.7, causal=True)
    for i in range(N):
        t = orc.forward(q[:, :, : i + 1], k[:, :, : i + 1], v[:, :, : i + 1], scale=0.7, causal=False)
        np.testing.assert_allclose(c["o"][:, :, i], t["o"][:, :, i], rtol=0, atol=1e-14)
        np.testing.assert_allclose(c["lse"][:, :, i], t["lse"][:, :, i], rtol=0, atol=1e-14)


# ----------------------------------------------------- online-softmax merge

def online_two_block(q, k, v, scale, split):
    """The pages' block merge, written independently of the oracle: process
    keys [0, split) then [split, N) with m_new = max(m_old, m_blk),
    alpha = exp(m_old - m_new), l_new = alpha l_old + l_blk,
    O_new = alpha O_old + O_blk, and divide by l at the end
    ([FA-kwkr] 2.2 and 2.3; [FA-Triton] 2.2)."""
    N = k.shape[0]
    m = np.full(q.shape[0], -np.inf)
    l = np.zeros(q.shape[0])
    acc = np.zeros((q.shape[0], v.shape[1]))
    for lo, hi in ((0, split), (split, N)):
        s = scale * (q @ k[lo:hi].T)
        m_blk = s.max(axis=1)
        m_new = np.maximum(m, m_blk)
        alpha = np.exp(m - m_new)
        p = np.exp(s - m_new[:, None])
        l = alpha * l + p.sum(axis=1)
        acc = alpha[:, None] * acc + p @ v[lo:hi]
        m = m_new
    return acc / l[:, None], m + np.log(l)


@pytest.mark.parametrize("split", [1, 3, 6])
def test_merge_identity_matches_two_pass(orc, split):
    N, D = 7, 5
    q, k, v = rand(N, D, scale=2), rand(N, D, scale=2), rand(N, D)
    o_ref, lse_ref = online_two_block(q, k, v, 0.6, split)
    out = orc.forward(q[None, None], k[None, None], v[None, None], scale=0.6, causal=False)
    np.testing.assert_allclose(out["o"][0, 0], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["lse"][0, 0], lse_ref, rtol=0, atol=1e-12)


# ----------------------------------------------------------- invariances

def test_key_permutation_invariance(orc):
    """Unmasked attention is a sum over keys: permuting K and V rows together
    changes nothing; permuting query rows permutes the output rows."""
    B, H, N, D = 1, 2, 10, 6
    q, k, v = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    base = orc.forward(q, k, v, scale=0.4, causal=False)
    perm = RNG.permutation(N)
    pk = orc.forward(q, k[:, :, perm], v[:, :, perm], scale=0.4, causal=False)
    np.testing.assert_allclose(pk["o"], base["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(pk["lse"], base["lse"], rtol=0, atol=1e-13)
    pq = orc.forward(q[:, :, perm], k, v, scale=0.4, causal=False)
    np.testing.assert_allclose(pq["o"], base["o"][:, :, perm], rtol=0, atol=1e-15)


def test_linear_in_values(orc):
    B, H, N, D = 1, 1, 8, 3
    q, k = rand(B, H, N, D), rand(B, H, N, D)
    v1, v2 = rand(B, H, N, D), rand(B, H, N, D)
    o1 = orc.forward(q, k, v1, scale=0.5, causal=True)["o"]
    o2 = orc.forward(q, k, v2, scale=0.5, causal=True)["o"]
    o12 = orc.forward(q, k, v1 + 2.0 * v2, scale=0.5, causal=True)["o"]
    np.testing.assert_allclose(o12, o1 + 2.0 * o2, rtol=0, atol=1e-13)


def test_scale_moves_between_query_and_factor(orc):
    """scale * (q . k) is bilinear: (2q) with scale/2 is the same problem."""
    B, H, N, D = 1, 2, 6, 4
    q, k, v = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    a = orc.forward(q, k, v, scale=0.3, causal=True)
    b = orc.forward(2.0 * q, k, v, scale=0.15, causal=True)
    np.testing.assert_allclose(a["o"], b["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=0, atol=1e-14)


def test_scale_multiplies_logits_not_one(orc):
    """Catches a dropped scale: with scale s the logits are s q.k."""
    q = np.array([[[[1.0]]]]).repeat(2, axis=2)
    k = np.array([[[[2.0], [0.0]]]])
    v = np.array([[[[1.0], [0.0]]]])
    out = orc.forward(q, k, v, scale=0.5, causal=False)
    p0 = 1.0 / (1.0 + math.exp(-1.0))    # s = [1.0, 0.0]
    np.testing.assert_allclose(out["o"][0, 0, :, 0], p0, rtol=0, atol=1e-15)


def test_gqa_equals_repeated_kv(orc):
    """Grouped heads: query head h reads kv head h // (Hq/Hkv); this equals
    plain multi-head attention with each kv head repeated Hq/Hkv times
    (contiguous groups, every 5 query heads share one kv head in the
    block-residual model of [BlockRes])."""
    B, Hq, Hkv, N, D = 2, 6, 2, 5, 3
    q, k, v = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D)
    g = orc.forward(q, k, v, scale=0.5, causal=True)
    kr, vr = np.repeat(k, Hq // Hkv, axis=1), np.repeat(v, Hq // Hkv, axis=1)
    m = orc.forward(q, kr, vr, scale=0.5, causal=True)
    np.testing.assert_array_equal(g["o"], m["o"])
    np.testing.assert_array_equal(g["lse"], m["lse"])


# ------------------------------------------------------------------ bias

def softmax_rows(x):
    from scipy.special import softmax
    return softmax(x, axis=-1)


def test_bias_alone_is_softmax_of_bias(orc):
    """Q = 0: logits are the bias itself, O = softmax(bias) V (library softmax),
    and the emitted logits equal the bias ([BlockRes] formula)."""
    B, H, N, D = 1, 2, 6, 3
    q, k, v = np.zeros((B, H, N, D)), rand(B, H, N, D), rand(B, H, N, D)
    bias = rand(B, H, N, N, scale=2)
    out = orc.forward(q, k, v, scale=0.9, causal=False, bias=bias, emit_logits=True)
    np.testing.assert_allclose(out["o"], softmax_rows(bias) @ v, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(out["logits"], bias)


def test_constant_row_bias_shifts_lse_only(orc):
    """Adding c_i to every logit of row i leaves P (and so O) unchanged and
    adds c_i to LSE_i."""
    B, H, N, D = 1, 2, 7, 4
    q, k, v = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    c = rand(B, H, N, 1, scale=5)
    bias = np.broadcast_to(c, (B, H, N, N)).copy()
    a = orc.forward(q, k, v, scale=0.4, causal=True)
    b = orc.forward(q, k, v, scale=0.4, causal=True, bias=bias)
    np.testing.assert_allclose(b["o"], a["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(b["lse"], a["lse"] + c[..., 0], rtol=0, atol=1e-13)


def test_bias_is_not_scaled(orc):
    """The residual adds to the already-scaled logits ([BlockRes] formula:
    Q K^T / sqrt(d) + residual): bias b on key 0 of a zero-query row gives
    P_0 = 1/(1 + exp(-b)) for two keys, whatever the scale."""
    q = np.zeros((1, 1, 2, 1))
    k, v = np.ones((1, 1, 2, 1)), np.array([[[[1.0], [0.0]]]])
    bias = np.zeros((1, 1, 2, 2))
    bias[..., 0] = 1.3
    for scale in (0.1, 10.0):
        out = orc.forward(q, k, v, scale=scale, causal=False, bias=bias)
        np.testing.assert_allclose(out["o"][0, 0, :, 0], 1 / (1 + math.exp(-1.3)), rtol=0, atol=1e-15)


def test_emitted_logits_chain(orc):
    """A block of layers: S_i = scale Q_i K_i^T + S_{i-1}, S_{-1} = 0.  With
    Q_i = 0 in a layer its emitted logits are exactly its input; emitted
    logits are NaN-marked above the diagonal under the causal mask."""
    B, H, N, D = 1, 2, 5, 3
    q0, k0, v0 = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    s0 = orc.forward(q0, k0, v0, scale=0.5, causal=True, emit_logits=True)["logits"]
    s1 = orc.forward(np.zeros_like(q0), k0, v0, scale=0.5, causal=True,
                     bias=np.nan_to_num(s0), emit_logits=True)["logits"]
    np.testing.assert_array_equal(s1, s0)
    assert np.isnan(s0[0, 0, 0, 1]) and not np.isnan(s0[0, 0, 1, 1])


def test_emit_in_place_alias(orc):
    """The logits output may be the bias buffer itself (each row reads its
    bias before writing its logits)."""
    B, H, N, D = 1, 2, 6, 4
    q, k, v = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    bias = rand(B, H, N, N)
    ref = orc.forward(q, k, v, scale=0.3, causal=False, bias=bias.copy(), emit_logits=True)
    buf = bias.copy()
    out = orc.forward(q, k, v, scale=0.3, causal=False, bias=buf, emit_logits=True, logits_out=buf)
    np.testing.assert_array_equal(buf, ref["logits"])
    np.testing.assert_array_equal(out["o"], ref["o"])


# ------------------------------------------------------- brute force / rows

def test_matches_library_softmax_on_tiny_inputs(orc):
    """Brute force with library routines (scipy softmax, numpy matmul, a
    boolean tril mask as in [Day26]'s naive wrapper) on tiny inputs."""
    B, Hq, Hkv, N, D = 2, 4, 2, 6, 5
    q, k, v = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D)
    bias = rand(B, Hq, N, N)
    kr, vr = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    for causal in (False, True):
        s = 0.35 * np.matmul(q, np.swapaxes(kr, -1, -2)) + bias
        if causal:
            s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
        want = np.matmul(softmax_rows(s), vr)
        out = orc.forward(q, k, v, scale=0.35, causal=causal, bias=bias)
        np.testing.assert_allclose(out["o"], want, rtol=0, atol=1e-13)


def test_sampled_rows_equal_full(orc):
    B, Hq, Hkv, N, D = 2, 4, 2, 9, 4
    q, k, v = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D)
    bias = rand(B, Hq, N, N)
    full = orc.forward(q, k, v, scale=0.5, causal=True, bias=bias, emit_logits=True)
    rows = np.array([0, 5, 17, 40, B * Hq * N - 1])
    part = orc.forward(q, k, v, scale=0.5, causal=True, bias=bias, rows=rows, emit_logits=True)
    np.testing.assert_array_equal(part["o"], full["o"].reshape(-1, D)[rows])
    np.testing.assert_array_equal(part["lse"], full["lse"].reshape(-1)[rows])
    np.testing.assert_array_equal(part["logits"], full["logits"].reshape(-1, N)[rows])


# -------------------------------------------------------------- backward

def loss(orc, q, k, v, do, scale, causal):
    return float((orc.forward(q, k, v, scale=scale, causal=causal)["o"] * do).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(orc, causal):
    """Central differences of L = sum(O * dO) pin dQ, dK, dV (recompute
    backward of [FA-kwkr] 2.4 / [FA-Triton] 4.3 must be the true gradient)."""
    B, Hq, Hkv, N, D = 1, 4, 2, 5, 3
    scale = 0.6
    q, k, v, do = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D), rand(B, Hq, N, D)
    g = orc.backward(q, k, v, do, scale=scale, causal=causal)
    h = 1e-5
    for name, arr in (("dq", q), ("dk", k), ("dv", v)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a = arr.copy(); a[idx] += h
            b = arr.copy(); b[idx] -= h
            args = {"q": q, "k": k, "v": v}
            key = name[1]
            args[key] = a
            lp = loss(orc, args["q"], args["k"], args["v"], do, scale, causal)
            args[key] = b
            lm = loss(orc, args["q"], args["k"], args["v"], do, scale, causal)
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(g[name] - fd).max() / max(1.0, np.abs(fd).max())
        assert err < 1e-7, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_sum_invariants(orc, causal):
    """Rows of P sum to 1, so sum_j dV_j = sum_i dO_i over a head group; and
    sum_j dS_ij = 0, so sum_j dK_j = 0."""
    B, Hq, Hkv, N, D = 2, 4, 2, 7, 4
    q, k, v, do = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D), rand(B, Hq, N, D)
    g = orc.backward(q, k, v, do, scale=0.45, causal=causal)
    grp = Hq // Hkv
    for b in range(B):
        for j in range(Hkv):
            np.testing.assert_allclose(g["dv"][b, j].sum(axis=0),
                                       do[b, j * grp:(j + 1) * grp].sum(axis=(0, 1)),
                                       rtol=0, atol=1e-12)
            np.testing.assert_allclose(g["dk"][b, j].sum(axis=0), 0.0, rtol=0, atol=1e-12)


def test_backward_sampled_equals_full(orc):
    B, Hq, Hkv, N, D = 1, 4, 2, 8, 3
    q, k, v, do = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D), rand(B, Hq, N, D)
    full = orc.backward(q, k, v, do, scale=0.5, causal=True)
    qr, kr = np.array([0, 3, 9, 31]), np.array([0, 7, 8, 15])
    part = orc.backward_sampled(q, k, v, do, scale=0.5, causal=True, q_rows=qr, k_rows=kr)
    np.testing.assert_allclose(part["dq"], full["dq"].reshape(-1, D)[qr], rtol=0, atol=1e-14)
    np.testing.assert_allclose(part["dk"], full["dk"].reshape(-1, D)[kr], rtol=0, atol=1e-14)
    np.testing.assert_allclose(part["dv"], full["dv"].reshape(-1, D)[kr], rtol=0, atol=1e-14)


def test_backward_sampled_with_residual_equals_full(orc):
    """Sampled rows with a logit bias and an incoming logit gradient (filled
    only at the sampled query rows' heads, as a full-size test does) match
    the full residual backward, dlogits rows included."""
    B, Hq, Hkv, N, D = 1, 4, 2, 8, 3
    q, k, v, do = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D), rand(B, Hq, N, D)
    bias, gin = rand(B, Hq, N, N), rand(B, Hq, N, N)
    full = orc.backward(q, k, v, do, scale=0.5, causal=True, bias=bias, grad_in=gin)
    qr = np.array([0, 3, 9, 31])
    part = orc.backward_sampled(q, k, v, do, scale=0.5, causal=True, q_rows=qr, k_rows=[],
                                bias=bias, grad_in=gin)
    np.testing.assert_allclose(part["dq"], full["dq"].reshape(-1, D)[qr], rtol=0, atol=1e-14)
    np.testing.assert_allclose(part["dlogits"], full["dlogits"].reshape(-1, N)[qr], rtol=0,
                               atol=1e-14)
    # only the sampled rows of bias and grad_in are read
    sb, sg = np.full_like(bias, np.nan), np.full_like(gin, np.nan)
    sb.reshape(-1, N)[qr], sg.reshape(-1, N)[qr] = bias.reshape(-1, N)[qr], gin.reshape(-1, N)[qr]
    part2 = orc.backward_sampled(q, k, v, do, scale=0.5, causal=True, q_rows=qr, k_rows=[],
                                 bias=sb, grad_in=sg)
    np.testing.assert_array_equal(part2["dq"], part["dq"])


def test_backward_zero_output_grad(orc):
    B, H, N, D = 1, 2, 5, 3
    q, k, v = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    g = orc.backward(q, k, v, np.zeros((B, H, N, D)), scale=0.5, causal=True)
    for name in ("dq", "dk", "dv"):
        assert np.abs(g[name]).max() == 0.0


def test_per_request_bias_rows_equal_full_bias(orc):
    """Sampled rows with only their own bias rows give the same result as the
    full bias, and a block chain can be followed row by row (row i of S_L
    depends only on row i of S_{L-1})."""
    B, Hq, Hkv, N, D = 1, 4, 2, 7, 3
    bias = rand(B, Hq, N, N)
    rows = np.array([1, 8, 27])
    layers = [(rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D)) for _ in range(3)]
    full_bias, part_bias = bias.copy(), bias.reshape(-1, N)[rows].copy()
    for q, k, v in layers:
        f = orc.forward(q, k, v, scale=0.5, causal=True, bias=full_bias, emit_logits=True)
        p = orc.forward(q, k, v, scale=0.5, causal=True, bias=part_bias, rows=rows,
                        emit_logits=True, logits_out=part_bias)
        np.testing.assert_array_equal(p["o"], f["o"].reshape(-1, D)[rows])
        np.testing.assert_array_equal(p["logits"], f["logits"].reshape(-1, N)[rows])
        full_bias = f["logits"]


# ------------------------------------------------------- sliding window
# Reading of the pages: [FA-Triton] 3.1 / 7 name a window mask stacked on the
# causal kernel and [BlockRes] "实验结果" an SWA baseline, with no formula; the
# window is taken as the W most recent keys, the query's own included:
# key j is kept for query i iff i - W < j <= i.

def test_window_one_keeps_only_the_diagonal(orc):
    """W = 1: each query sees only its own key, so P_ii = 1, O_i = v_i and
    LSE_i = s_ii = scale q_i . k_i exactly."""
    B, Hq, Hkv, N, D = 1, 4, 2, 6, 3
    q, k, v = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D)
    out = orc.forward(q, k, v, scale=0.7, causal=True, window=1)
    for h in range(Hq):
        g = h // 2
        np.testing.assert_array_equal(out["o"][0, h], v[0, g])
        np.testing.assert_allclose(out["lse"][0, h], 0.7 * (q[0, h] * k[0, g]).sum(-1),
                                   rtol=0, atol=1e-14)


@pytest.mark.parametrize("W", [2, 3, 5])
def test_window_zero_query_gives_mean_of_last_w_values(orc, W):
    """Q = 0: uniform weights over the last min(i+1, W) keys, so O_i is the
    mean of v[max(0, i-W+1) .. i] and LSE_i = ln min(i+1, W)."""
    B, H, N, D = 1, 2, 8, 4
    q = np.zeros((B, H, N, D))
    k, v = rand(B, H, N, D), rand(B, H, N, D)
    out = orc.forward(q, k, v, scale=0.9, causal=True, window=W)
    for h in range(H):
        for i in range(N):
            lo = max(0, i - W + 1)
            np.testing.assert_allclose(out["o"][0, h, i], v[0, h, lo:i + 1].mean(axis=0),
                                       rtol=0, atol=1e-14)
            assert abs(out["lse"][0, h, i] - math.log(i + 1 - lo)) < 1e-14


def test_window_at_least_n_equals_causal(orc):
    B, Hq, Hkv, N, D = 1, 2, 1, 7, 3
    q, k, v = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D)
    bias = rand(B, Hq, N, N)
    c = orc.forward(q, k, v, scale=0.5, causal=True, bias=bias, emit_logits=True)
    for W in (N, N + 5):
        w = orc.forward(q, k, v, scale=0.5, causal=True, bias=bias, emit_logits=True, window=W)
        np.testing.assert_array_equal(w["o"], c["o"])
        np.testing.assert_array_equal(w["lse"], c["lse"])
        np.testing.assert_array_equal(w["logits"], c["logits"])


def test_window_matches_library_softmax_on_tiny_inputs(orc):
    """Brute force: an explicit band mask (numpy tril minus tril(-W)) applied
    to the full logit matrix, scipy-style softmax, matmul with V."""
    B, Hq, Hkv, N, D, W = 2, 4, 2, 9, 5, 3
    q, k, v = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D)
    bias = rand(B, Hq, N, N)
    kr, vr = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    band = np.tril(np.ones((N, N), dtype=bool)) & ~np.tril(np.ones((N, N), dtype=bool), -W)
    s = 0.35 * np.matmul(q, np.swapaxes(kr, -1, -2)) + bias
    want = np.matmul(softmax_rows(np.where(band, s, -np.inf)), vr)
    out = orc.forward(q, k, v, scale=0.35, causal=True, bias=bias, window=W, emit_logits=True)
    np.testing.assert_allclose(out["o"], want, rtol=0, atol=1e-13)
    lg = out["logits"]
    assert np.isnan(lg[..., ~band]).all()
    np.testing.assert_allclose(lg[..., band], s[..., band], rtol=0, atol=1e-13)


def test_window_backward_matches_finite_differences(orc):
    B, Hq, Hkv, N, D, W = 1, 2, 1, 6, 3, 2
    scale = 0.6
    q, k, v, do = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D), rand(B, Hq, N, D)
    g = orc.backward(q, k, v, do, scale=scale, causal=True, window=W)

    def L(qq, kk, vv):
        return float((orc.forward(qq, kk, vv, scale=scale, causal=True, window=W)["o"] * do).sum())

    h = 1e-5
    for name, arr in (("dq", q), ("dk", k), ("dv", v)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = {"q": q, "k": k, "v": v}
            a = arr.copy(); a[idx] += h
            b = arr.copy(); b[idx] -= h
            args[name[1]] = a
            lp = L(args["q"], args["k"], args["v"])
            args[name[1]] = b
            lm = L(args["q"], args["k"], args["v"])
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(g[name] - fd).max() / max(1.0, np.abs(fd).max())
        assert err < 1e-7, (name, err)


def test_window_backward_sampled_equals_full(orc):
    B, Hq, Hkv, N, D, W = 1, 4, 2, 10, 3, 3
    q, k, v, do = rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D), rand(B, Hq, N, D)
    full = orc.backward(q, k, v, do, scale=0.5, causal=True, window=W)
    qr, kr = np.array([0, 3, 12, 39]), np.array([0, 4, 9, 13, 19])
    part = orc.backward_sampled(q, k, v, do, scale=0.5, causal=True, q_rows=qr, k_rows=kr,
                                window=W)
    np.testing.assert_allclose(part["dq"], full["dq"].reshape(-1, D)[qr], rtol=0, atol=1e-14)
    np.testing.assert_allclose(part["dk"], full["dk"].reshape(-1, D)[kr], rtol=0, atol=1e-14)
    np.testing.assert_allclose(part["dv"], full["dv"].reshape(-1, D)[kr], rtol=0, atol=1e-14)


def test_window_needs_causal(orc):
    x = rand(1, 1, 4, 2)
    with pytest.raises(ValueError):
        orc.forward(x, x, x, scale=1.0, causal=False, window=2)
    with pytest.raises(ValueError):
        orc.forward(x, x, x, scale=1.0, causal=True, window=0)


# ------------------------------------------- block-residual backward
# Reading ([BlockRes] "v1: Fuse Residual 进 Attention Kernel": the backward
# keeps the LSE statistics, corrected for the residual; no formula printed):
# S_l = scale Q_l K_l^T + S_{l-1}.  S_l reaches the loss through layer l's
# softmax and, unscaled, through S_{l+1}, so the total logit gradient is
# dS_l = P_l o (dP_l - Delta_l) + dS_{l+1}; it drives dQ_l, dK_l and is the
# gradient of layer l's bias.

def chain_forward(orc, layers, scale, causal):
    outs, prev = [], None
    for q, k, v in layers:
        f = orc.forward(q, k, v, scale=scale, causal=causal,
                        bias=None if prev is None else np.nan_to_num(prev), emit_logits=True)
        outs.append(f["o"])
        prev = f["logits"]
    return outs


@pytest.mark.parametrize("causal", [False, True])
def test_residual_chain_backward_matches_finite_differences(orc, causal):
    """Two chained layers, L = sum_l sum(O_l * dO_l): layer 1's backward with
    bias S_0 gives dlogits_1, which enters layer 0's backward as grad_in;
    every input's gradient must equal central differences of L."""
    B, Hq, Hkv, N, D = 1, 2, 1, 5, 3
    scale = 0.7
    layers = [(rand(B, Hq, N, D), rand(B, Hkv, N, D), rand(B, Hkv, N, D)) for _ in range(2)]
    dos = [rand(B, Hq, N, D) for _ in range(2)]

    def L(ls):
        return float(sum((o * do).sum() for o, do in zip(chain_forward(orc, ls, scale, causal), dos)))

    f0 = orc.forward(*layers[0], scale=scale, causal=causal, emit_logits=True)
    g1 = orc.backward(*layers[1], dos[1], scale=scale, causal=causal,
                      bias=np.nan_to_num(f0["logits"]))
    g0 = orc.backward(*layers[0], dos[0], scale=scale, causal=causal, grad_in=g1["dlogits"])
    grads = [g0, g1]
    h = 1e-5
    for li in range(2):
        for ti, name in enumerate(("dq", "dk", "dv")):
            arr = layers[li][ti]
            fd = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                a = arr.copy(); a[idx] += h
                b = arr.copy(); b[idx] -= h
                lp = [list(x) for x in layers]; lp[li][ti] = a
                lm = [list(x) for x in layers]; lm[li][ti] = b
                fd[idx] = (L(lp) - L(lm)) / (2 * h)
            err = np.abs(grads[li][name] - fd).max() / max(1.0, np.abs(fd).max())
            assert err < 1e-7, (li, name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_bias_gradient_is_total_logit_gradient(orc, causal):
    """dL/dbias_ij by central differences equals dlogits on the kept keys
    and 0 on the masked ones; grad_in adds straight onto it."""
    B, H, N, D = 1, 1, 4, 3
    q, k, v, do = rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D), rand(B, H, N, D)
    bias, gin = rand(B, H, N, N), rand(B, H, N, N)

    def L(bb):
        return float((orc.forward(q, k, v, scale=0.5, causal=causal, bias=bb)["o"] * do).sum())

    g = orc.backward(q, k, v, do, scale=0.5, causal=causal, bias=bias)
    h = 1e-6
    fd = np.zeros_like(bias)
    for idx in np.ndindex(bias.shape):
        a = bias.copy(); a[idx] += h
        b = bias.copy(); b[idx] -= h
        fd[idx] = (L(a) - L(b)) / (2 * h)
    np.testing.assert_allclose(g["dlogits"], fd, rtol=0, atol=1e-8)
    g2 = orc.backward(q, k, v, do, scale=0.5, causal=causal, bias=bias, grad_in=gin)
    kept = np.tril(np.ones((N, N), dtype=bool)) if causal else np.ones((N, N), dtype=bool)
    np.testing.assert_allclose(g2["dlogits"][..., kept], (g["dlogits"] + gin)[..., kept],
                               rtol=0, atol=1e-14)
    assert (g2["dlogits"][..., ~kept] == 0).all()
