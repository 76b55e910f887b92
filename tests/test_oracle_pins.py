"""Pins for the fp64 oracle, against facts that do not come from the oracle.

Each check targets a plausible mistake in the oracle:
  * a second, matrix-form formulation (complex-number rotation, full T x T
    score matrix with a mask matrix, matrix-calculus gradients) on tiny
    shapes -> wrong index, transposed operand, dropped term or scale;
  * central finite differences in double precision (the method the pages use
    for their own backward, socker-news README "Verified backward") -> any
    gradient-formula mistake, independently of the formulas;
  * closed forms: T = 1, q = 0 (uniform causal average, LSE = ln(t + 1)),
    constant v, LSE_0 = scale * q_0 . k_0, the D = 2 rotation with theta = 1
    -> wrong mask boundary, wrong rotation sign, missing scale;
  * invariants: causality, GQA == MHA with repeated K/V, rotary norm
    preservation and relative-position dependence, R^T R = I, the identity
    sum_j P_tj dP_tj = dO_t . O_t.
"""
import math
import os

import numpy as np
import pytest

from causal_gqa_attention_flashattention_gb300 import inputs

BASE = 10000.0


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- second formulation
def _rot_complex(x, base, sign=1.0, half=False):
    """Rotary embedding as a complex phase: (x0 + i x1) * exp(i t theta), with
    pairs (x[2i], x[2i+1]) or, half-split, (x[i], x[i + D/2])."""
    B, T, H, D = x.shape
    theta = base ** (-np.arange(0, D, 2) / D)
    ang = np.arange(T)[:, None] * theta[None, :]
    ph = np.exp(1j * sign * ang)[None, :, None, :]
    lo, hi = (slice(0, D // 2), slice(D // 2, D)) if half else (slice(0, D, 2), slice(1, D, 2))
    z = (x[..., lo] + 1j * x[..., hi]) * ph
    out = np.empty_like(x)
    out[..., lo] = z.real
    out[..., hi] = z.imag
    return out


def bruteforce(q, k, v, do, base, half=False):
    """Whole-matrix causal GQA attention and its matrix-calculus gradients."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    qr, kr = _rot_complex(q, base, half=half), _rot_complex(k, base, half=half)
    mask = np.triu(np.ones((T, T), dtype=bool), 1)  # True where key > query
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, T))
    dqr = np.zeros_like(q)
    dkr = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            S = scale * qr[b, :, h] @ kr[b, :, g].T
            S[mask] = -np.inf
            mx = S.max(axis=1, keepdims=True)
            E = np.exp(S - mx)
            Z = E.sum(axis=1, keepdims=True)
            P = E / Z
            o[b, :, h] = P @ v[b, :, g]
            lse[b, h] = (mx + np.log(Z))[:, 0]
            dP = do[b, :, h] @ v[b, :, g].T
            dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
            dqr[b, :, h] = scale * dS @ kr[b, :, g]
            dkr[b, :, g] += scale * dS.T @ qr[b, :, h]
            dv[b, :, g] += P.T @ do[b, :, h]
    dq = _rot_complex(dqr, base, -1.0, half)
    dk = _rot_complex(dkr, base, -1.0, half)
    return o, lse, dq, dk, dv


def close(a, b, tol):
    a, b = np.asarray(a), np.asarray(b)
    err = np.max(np.abs(a - b)) / max(1.0, np.max(np.abs(b)))
    assert err <= tol, err


@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 2), (1, 4, 2, 1, 4), (2, 6, 4, 2, 4),
                                   (1, 5, 3, 3, 6), (2, 6, 4, 1, 8)])
def test_bruteforce_matrix_form(oracle_mod, shape):
    B, T, Hq, Hkv, D = shape
    q, k, v = rnd((B, T, Hq, D), 1), rnd((B, T, Hkv, D), 2), rnd((B, T, Hkv, D), 3)
    do = rnd((B, T, Hq, D), 4)
    for base in (BASE, 7.0):
        o, lse = oracle_mod.attn_fwd(q, k, v, base)
        g = oracle_mod.attn_bwd(q, k, v, do, base)
        bo, blse, bdq, bdk, bdv = bruteforce(q, k, v, do, base)
        close(o, bo, 1e-12)
        close(lse, blse, 1e-12)
        close(g["o"], bo, 1e-12)
        close(g["lse"], blse, 1e-12)
        close(g["dq"], bdq, 1e-12)
        close(g["dk"], bdk, 1e-12)
        close(g["dv"], bdv, 1e-12)


# ---------------------------------------------------------------- finite differences
def _load_pages_fd_figures():
    path = os.path.join(os.path.dirname(__file__), "golden", "pages_gradient_check.txt")
    vals = {}
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            name, val = line.split()
            vals[name] = float(val)
    return vals


def test_central_finite_differences(oracle_mod):
    """dq, dk, dv against central differences of L = sum(dO * O) in fp64."""
    pages = _load_pages_fd_figures()
    B, T, Hq, Hkv, D = 1, 5, 4, 2, 4
    q, k, v = rnd((B, T, Hq, D), 11), rnd((B, T, Hkv, D), 12), rnd((B, T, Hkv, D), 13)
    do = rnd((B, T, Hq, D), 14)
    base = 50.0  # a small base gives large angles at every frequency pair

    def loss(q_, k_, v_):
        o, _ = oracle_mod.attn_fwd(q_, k_, v_, base)
        return float(np.sum(do * o))

    g = oracle_mod.attn_bwd(q, k, v, do, base)
    eps = 1e-5
    worst = 0.0
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"dq": (xp, k, v), "dk": (q, xp, v), "dv": (q, k, xp)}[name]
            args_m = {"dq": (xm, k, v), "dk": (q, xm, v), "dv": (q, k, xm)}[name]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        rel = np.max(np.abs(fd - g[name])) / np.max(np.abs(fd))
        worst = max(worst, rel)
    assert worst <= 1e-6, worst
    assert worst < pages["overall_max"] < pages["pass_threshold"]


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("shape", [(2, 9, 4, 2, 4, 3), (1, 6, 3, 3, 2, 1), (1, 5, 2, 1, 4, 5)])
def test_decode_is_the_last_rows(oracle_mod, shape):
    """decode_fwd equals the last Tq rows of the whole-matrix formulation run on
    a query tensor whose earlier rows are random (they must not matter)."""
    B, T, Hq, Hkv, D, Tq = shape
    q, k, v, do = rnd((B, T, Hq, D), 21), rnd((B, T, Hkv, D), 22), rnd((B, T, Hkv, D), 23), rnd((B, T, Hq, D), 24)
    o_ref, lse_ref, _, _, _ = bruteforce(q, k, v, do, 10000.0)
    o, lse = oracle_mod.decode_fwd(q[:, T - Tq:], k, v, 10000.0)
    close(o, o_ref[:, T - Tq:], 1e-12)
    close(lse, lse_ref[:, :, T - Tq:], 1e-12)
    # the same with the half-split pair layout
    o_ref, lse_ref, _, _, _ = bruteforce(q, k, v, do, 10000.0, half=True)
    o, lse = oracle_mod.decode_fwd(q[:, T - Tq:], k, v, 10000.0, half=True)
    close(o, o_ref[:, T - Tq:], 1e-12)
    close(lse, lse_ref[:, :, T - Tq:], 1e-12)


@pytest.mark.parametrize("shape", [(1, 5, 2, 1, 4), (2, 7, 4, 2, 8), (1, 9, 3, 3, 6)])
def test_half_split_layout_matrix_form(oracle_mod, shape):
    """The half-split pair layout (x[i], x[i + D/2]) against the whole-matrix
    formulation with the same layout."""
    B, T, Hq, Hkv, D = shape
    q, k, v, do = rnd((B, T, Hq, D), 31), rnd((B, T, Hkv, D), 32), rnd((B, T, Hkv, D), 33), rnd((B, T, Hq, D), 34)
    o_r, lse_r, dq_r, dk_r, dv_r = bruteforce(q, k, v, do, 500.0, half=True)
    ref = oracle_mod.attn_bwd(q, k, v, do, 500.0, half=True)
    for name, r in (("o", o_r), ("lse", lse_r), ("dq", dq_r), ("dk", dk_r), ("dv", dv_r)):
        close(ref[name], r, 1e-12)


def test_half_split_is_a_feature_permutation(oracle_mod):
    """Half-split RoPE of x equals interleaved RoPE of P x read back through P,
    with (P x)[2i] = x[i] and (P x)[2i+1] = x[i + D/2]; the scores use both
    q and k in the same order, so o and lse agree and dq, dk map back by P."""
    B, T, Hq, Hkv, D = 2, 8, 4, 2, 8
    q, k, v, do = rnd((B, T, Hq, D), 41), rnd((B, T, Hkv, D), 42), rnd((B, T, Hkv, D), 43), rnd((B, T, Hq, D), 44)
    perm = np.empty(D, dtype=int)
    perm[0::2], perm[1::2] = np.arange(D // 2), np.arange(D // 2, D)  # P x = x[..., perm]
    half = oracle_mod.attn_bwd(q, k, v, do, 10000.0, half=True)
    inter = oracle_mod.attn_bwd(q[..., perm], k[..., perm], v, do, 10000.0)
    inv = np.argsort(perm)
    close(half["o"], inter["o"], 1e-12)
    close(half["lse"], inter["lse"], 1e-12)
    close(half["dq"], inter["dq"][..., inv], 1e-12)
    close(half["dk"], inter["dk"][..., inv], 1e-12)
    close(half["dv"], inter["dv"], 1e-12)
    x = rnd((B, T, Hq, D), 45)
    close(oracle_mod.rope(x, 10000.0, half=True), oracle_mod.rope(x[..., perm], 10000.0)[..., inv], 1e-12)
    y = rnd((B, T, Hq, 2), 46)  # with D = 2 the two layouts are the same rotation
    close(oracle_mod.rope(y, 10000.0, half=True), oracle_mod.rope(y, 10000.0), 1e-15)


def test_single_token(oracle_mod):
    """T = 1: O = v_0, LSE = s_00, dq = dk = 0, dv_0 = sum over the group of dO."""
    B, T, Hq, Hkv, D = 2, 1, 4, 2, 8
    q, k, v = rnd((B, T, Hq, D), 21), rnd((B, T, Hkv, D), 22), rnd((B, T, Hkv, D), 23)
    do = rnd((B, T, Hq, D), 24)
    g = oracle_mod.attn_bwd(q, k, v, do, BASE)
    G = Hq // Hkv
    for h in range(Hq):
        np.testing.assert_allclose(g["o"][:, 0, h], v[:, 0, h // G], rtol=0, atol=1e-15)
        s00 = np.sum(q[:, 0, h] * k[:, 0, h // G], axis=-1) / math.sqrt(D)
        np.testing.assert_allclose(g["lse"][:, h, 0], s00, rtol=1e-14, atol=1e-14)
    assert np.all(g["dq"] == 0.0) and np.all(g["dk"] == 0.0)
    np.testing.assert_allclose(g["dv"][:, 0], do[:, 0].reshape(B, Hkv, G, D).sum(2), atol=1e-14)


def test_zero_queries_give_causal_mean(oracle_mod):
    """q = 0: every visible score is 0, so O_t = mean_{j<=t} v_j, LSE_t = ln(t+1)."""
    B, T, Hq, Hkv, D = 1, 9, 2, 1, 4
    q = np.zeros((B, T, Hq, D))
    k, v = rnd((B, T, Hkv, D), 31), rnd((B, T, Hkv, D), 32)
    o, lse = oracle_mod.attn_fwd(q, k, v, BASE)
    for t in range(T):
        for h in range(Hq):
            np.testing.assert_allclose(o[0, t, h], v[0, : t + 1, 0].mean(0), atol=1e-14)
            assert abs(lse[0, h, t] - math.log(t + 1)) < 1e-14


def test_constant_values(oracle_mod):
    """v_j = c for all j: O_t = c and the score gradients vanish (dq = dk = 0)."""
    B, T, Hq, Hkv, D = 1, 7, 4, 2, 4
    q, k = rnd((B, T, Hq, D), 41), rnd((B, T, Hkv, D), 42)
    c = rnd((D,), 43)
    v = np.broadcast_to(c, (B, T, Hkv, D)).copy()
    do = rnd((B, T, Hq, D), 44)
    g = oracle_mod.attn_bwd(q, k, v, do, BASE)
    np.testing.assert_allclose(g["o"], np.broadcast_to(c, g["o"].shape), atol=1e-14)
    assert np.max(np.abs(g["dq"])) < 1e-14 and np.max(np.abs(g["dk"])) < 1e-14


def test_rope_two_dims_closed_form(oracle_mod):
    """D = 2 has theta_0 = base^0 = 1: R_t (x0, x1) = (x0 cos t - x1 sin t, x0 sin t + x1 cos t)."""
    T = 6
    x = rnd((1, T, 1, 2), 51)
    r = oracle_mod.rope(x, 12345.0)
    for t in range(T):
        x0, x1 = x[0, t, 0]
        exp = (x0 * math.cos(t) - x1 * math.sin(t), x0 * math.sin(t) + x1 * math.cos(t))
        np.testing.assert_allclose(r[0, t, 0], exp, rtol=0, atol=1e-15)


def test_rope_second_pair_frequency(oracle_mod):
    """D = 4: the second pair turns at theta_1 = base^(-1/2)."""
    base = 100.0
    x = np.zeros((1, 4, 1, 4))
    x[..., 2] = 1.0
    r = oracle_mod.rope(x, base)
    for t in range(4):
        a = t * base ** -0.5
        np.testing.assert_allclose(r[0, t, 0], [0, 0, math.cos(a), math.sin(a)], atol=1e-15)


# ---------------------------------------------------------------- invariants
def test_rope_invariants(oracle_mod):
    B, T, H, D = 1, 40, 3, 16
    x = rnd((B, T, H, D), 61)
    r = oracle_mod.rope(x, BASE)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-14)
    np.testing.assert_array_equal(r[:, 0], x[:, 0])                    # R_0 = I
    np.testing.assert_allclose(oracle_mod.rope(r, BASE, inverse=True), x, atol=1e-13)  # R^T R = I
    # <R_m q, R_n k> depends on m - n only: place the same q, k at (m, n) and (m+s, n+s)
    qv, kv = rnd((D,), 62), rnd((D,), 63)
    m, n, s = 7, 3, 25
    a = np.zeros((1, T, 1, D))
    b = np.zeros((1, T, 1, D))
    a[0, m, 0], b[0, n, 0] = qv, kv
    a[0, m + s, 0], b[0, n + s, 0] = qv, kv
    ra, rb = oracle_mod.rope(a, BASE), oracle_mod.rope(b, BASE)
    d1 = ra[0, m, 0] @ rb[0, n, 0]
    d2 = ra[0, m + s, 0] @ rb[0, n + s, 0]
    assert abs(d1 - d2) < 1e-12
    assert abs(d1 - qv @ kv) > 1e-6  # and it does depend on the offset


def test_causality(oracle_mod):
    """Perturbing q/k/v rows after t leaves O_t and LSE_t bit-for-bit unchanged."""
    B, T, Hq, Hkv, D = 1, 12, 4, 2, 8
    q, k, v = rnd((B, T, Hq, D), 71), rnd((B, T, Hkv, D), 72), rnd((B, T, Hkv, D), 73)
    o, lse = oracle_mod.attn_fwd(q, k, v, BASE)
    t = 5
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:, t + 1:] += rnd(q2[:, t + 1:].shape, 74)
    k2[:, t + 1:] += rnd(k2[:, t + 1:].shape, 75)
    v2[:, t + 1:] += rnd(v2[:, t + 1:].shape, 76)
    o2, lse2 = oracle_mod.attn_fwd(q2, k2, v2, BASE)
    np.testing.assert_array_equal(o2[:, : t + 1], o[:, : t + 1])
    np.testing.assert_array_equal(lse2[:, :, : t + 1], lse[:, :, : t + 1])
    assert not np.array_equal(o2[:, t + 1:], o[:, t + 1:])


def test_gqa_equals_mha_with_repeated_kv(oracle_mod):
    B, T, Hq, Hkv, D = 2, 10, 6, 2, 8
    G = Hq // Hkv
    q, k, v = rnd((B, T, Hq, D), 81), rnd((B, T, Hkv, D), 82), rnd((B, T, Hkv, D), 83)
    do = rnd((B, T, Hq, D), 84)
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    g1 = oracle_mod.attn_bwd(q, k, v, do, BASE)
    g2 = oracle_mod.attn_bwd(q, kr, vr, do, BASE)
    close(g1["o"], g2["o"], 1e-13)
    close(g1["lse"], g2["lse"], 1e-13)
    close(g1["dq"], g2["dq"], 1e-13)
    close(g1["dk"], g2["dk"].reshape(B, T, Hkv, G, D).sum(3), 1e-13)
    close(g1["dv"], g2["dv"].reshape(B, T, Hkv, G, D).sum(3), 1e-13)


def test_delta_identity_and_lse_bounds(oracle_mod):
    """sum_j P_tj dP_tj (computed from its definition) equals dO_t . O_t;
    LSE_t >= the largest visible score; LSE_0 = s_00."""
    B, T, Hq, Hkv, D = 1, 16, 2, 1, 8
    q, k, v = rnd((B, T, Hq, D), 91), rnd((B, T, Hkv, D), 92), rnd((B, T, Hkv, D), 93)
    do = rnd((B, T, Hq, D), 94)
    g = oracle_mod.attn_bwd(q, k, v, do, BASE)
    close(g["delta"], np.einsum("bthd,bthd->bht", do, g["o"]), 1e-13)
    qr, kr = oracle_mod.rope(q, BASE), oracle_mod.rope(k, BASE)
    for h in range(Hq):
        s = qr[0, :, h] @ kr[0, :, 0].T / math.sqrt(D)
        for t in range(T):
            assert g["lse"][0, h, t] >= s[t, : t + 1].max() - 1e-14
        assert abs(g["lse"][0, h, 0] - s[0, 0]) < 1e-14


def test_group_sampling_matches_full(oracle_mod):
    """Computing a subset of (batch, kv-head) groups gives the same numbers as the full run."""
    B, T, Hq, Hkv, D = 2, 20, 4, 2, 8
    q, k, v = rnd((B, T, Hq, D), 101), rnd((B, T, Hkv, D), 102), rnd((B, T, Hkv, D), 103)
    do = rnd((B, T, Hq, D), 104)
    full = oracle_mod.attn_bwd(q, k, v, do, BASE)
    part = oracle_mod.attn_bwd(q, k, v, do, BASE, groups=[(1, 0)])
    G = Hq // Hkv
    np.testing.assert_array_equal(part["dq"][1, :, 0:G], full["dq"][1, :, 0:G])
    np.testing.assert_array_equal(part["dk"][1, :, 0], full["dk"][1, :, 0])
    np.testing.assert_array_equal(part["dv"][1, :, 0], full["dv"][1, :, 0])
    assert np.isnan(part["dq"][0]).all() and np.isnan(part["dk"][1, :, 1]).all()


# ---------------------------------------------------------------- input recipe
def test_bf16_rounding_and_recipe():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e-3], dtype=np.float32)
    bits = inputs.bf16_round_bits(x)
    back = inputs.bf16_bits_to_f64(bits)
    # ties go to even: 1 + 2^-8 -> 1, 1 + 3*2^-8 -> 1 + 2^-6
    np.testing.assert_array_equal(back[:3], [1.0, 1.0, 1.0 + 2 ** -6])
    assert back[3] == -2.5 and abs(back[4] - 3.0e-3) < 3.0e-3 * 2 ** -8
    a = inputs.make_shape_inputs(1, 64, 2, 1, 16, seed=5, recipe="stress")
    b = inputs.make_shape_inputs(1, 64, 2, 1, 16, seed=5, recipe="stress")
    np.testing.assert_array_equal(a["q_bits"], b["q_bits"])
    assert np.max(np.abs(a["q"])) > 16.0  # outlier rows present at this size


# ---------------------------------------------------------------- RMSNorm + Q/K/V projection
def _stack_proj(*blocks):
    return np.concatenate(blocks, axis=0)


def test_rmsnorm_worked_example(oracle_mod):
    # x = (3, 4): mean of squares (9 + 16) / 2 = 12.5, so with w = 1 and eps = 0
    # the normalised row is (3, 4) / sqrt(12.5) = (0.848528137423857, 1.131370849898476).
    # Projection rows [I; 2 I; -I] read it back as q = xn, k = 2 xn, v = -xn.
    x = np.array([[[3.0, 4.0]]])
    I = np.eye(2)
    W = _stack_proj(I, 2 * I, -I)
    q, k, v, rstd = oracle_mod.qkv_rmsnorm(x, np.ones(2), W, Hq=1, Hkv=1, D=2, eps=0.0)
    xn = np.array([0.8485281374238571, 1.1313708498984762])
    np.testing.assert_allclose(rstd[0, 0], 0.28284271247461906, rtol=1e-15)  # 1 / sqrt(12.5)
    np.testing.assert_allclose(q[0, 0, 0], xn, rtol=1e-15)
    np.testing.assert_allclose(k[0, 0, 0], 2 * xn, rtol=1e-15)
    np.testing.assert_allclose(v[0, 0, 0], -xn, rtol=1e-15)
    # eps adds to the mean of squares: 1 / sqrt(12.5 + 0.5) = 1 / sqrt(13)
    _, _, _, r2 = oracle_mod.qkv_rmsnorm(x, np.ones(2), W, Hq=1, Hkv=1, D=2, eps=0.5)
    np.testing.assert_allclose(r2[0, 0], 0.2773500981126146, rtol=1e-15)
    # the norm weight scales feature c before the projection: w = (2, -1)
    q3, _, _, _ = oracle_mod.qkv_rmsnorm(x, np.array([2.0, -1.0]), W, Hq=1, Hkv=1, D=2, eps=0.0)
    np.testing.assert_allclose(q3[0, 0, 0], [2 * xn[0], -xn[1]], rtol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance(oracle_mod):
    # with w = 1, eps = 0 and the identity projection (N = C = 16), the
    # concatenated q | k | v of a row is the normalised row: mean square 1,
    # and scaling the row by any positive factor changes nothing.
    B, T, C, Hq, Hkv, D = 2, 5, 16, 2, 1, 4
    x = rnd((B, T, C), 31)
    q, k, v, _ = oracle_mod.qkv_rmsnorm(x, np.ones(C), np.eye(C), Hq, Hkv, D, eps=0.0)
    cat = np.concatenate([q.reshape(B, T, -1), k.reshape(B, T, -1), v.reshape(B, T, -1)], axis=-1)
    np.testing.assert_allclose(np.mean(cat * cat, axis=-1), 1.0, rtol=1e-14)
    q2, k2, v2, _ = oracle_mod.qkv_rmsnorm(7.25 * x, np.ones(C), np.eye(C), Hq, Hkv, D, eps=0.0)
    np.testing.assert_allclose(q2, q, rtol=1e-13)
    np.testing.assert_allclose(v2, v, rtol=1e-13)
    # a zero row stays zero and its rstd is 1 / sqrt(eps)
    x[0, 0] = 0.0
    q3, _, _, r3 = oracle_mod.qkv_rmsnorm(x, np.ones(C), np.eye(C), Hq, Hkv, D, eps=1e-4)
    assert np.all(q3[0, 0] == 0.0) and abs(r3[0, 0] - 100.0) < 1e-12


def test_projection_one_hot_rows_and_head_order(oracle_mod):
    # A row with one non-zero entry s at column c has mean square s^2 / C, so
    # (eps = 0) it normalises to sign(s) sqrt(C) w_c e_c and projects onto
    # sign(s) sqrt(C) w_c W[:, c]; the first Hq*D rows of W are the query
    # features (head h at rows h*D ..), then Hkv*D key rows, then the values.
    B, T, C, Hq, Hkv, D = 1, 3, 12, 3, 1, 2
    N = (Hq + 2 * Hkv) * D
    W = rnd((N, C), 32)
    w = 1.0 + 0.1 * rnd((C,), 33)
    x = np.zeros((B, T, C))
    cols, vals = [4, 0, 11], [-2.5, 0.75, 3.0]
    for t in range(T):
        x[0, t, cols[t]] = vals[t]
    q, k, v, rstd = oracle_mod.qkv_rmsnorm(x, w, W, Hq, Hkv, D, eps=0.0)
    for t in range(T):
        c, s = cols[t], vals[t]
        col = np.sign(s) * np.sqrt(C) * w[c] * W[:, c]
        np.testing.assert_allclose(rstd[0, t], np.sqrt(C) / abs(s), rtol=1e-15)
        for h in range(Hq):
            np.testing.assert_allclose(q[0, t, h], col[h * D:(h + 1) * D], rtol=1e-13)
        np.testing.assert_allclose(k[0, t, 0], col[Hq * D:(Hq + 1) * D], rtol=1e-13)
        np.testing.assert_allclose(v[0, t, 0], col[(Hq + 1) * D:], rtol=1e-13)


def test_prologue_inputs_recipe():
    a = inputs.make_prologue_inputs(2, 16, 64, 4, 2, 8, seed=3)
    b = inputs.make_prologue_inputs(2, 16, 64, 4, 2, 8, seed=3)
    np.testing.assert_array_equal(a["w_qkv_bits"], b["w_qkv_bits"])
    assert a["w_qkv"].shape == ((4 + 2 * 2) * 8, 64) and a["norm_w"].shape == (64,)
    assert 0.5 < np.std(a["w_qkv"]) * np.sqrt(64) < 1.5 and abs(np.mean(a["norm_w"]) - 1.0) < 0.1
