"""GPU parity of the step in front of attention: RMSNorm + the fused Q/K/V
projection (ne_attn_qkv_rmsnorm), against the fp64 oracle on the same seeded
bf16 inputs, and the whole chain projection -> attention forward -> backward
with the rotated q and k handed over in the workspace.

q, k, v and the rotated q, k must reach relative L2 <= 5e-3 and max abs
<= 2e-2 (the attention bound: they are bf16 / fp16 roundings of unit-scale
values, about 2^-9 relative, after a product with the bf16-rounded
norm-weighted projection); rstd is fp32 arithmetic on exact inputs
(relative 1e-5).

The chain adds one rounded stage in front of attention: its q, k, v differ
from the exact projections by about 2.3e-3 relative (the bf16 rounding of
w * W and of the outputs), which moves the attention outputs by about as much
as the attention's own bf16 rounding does.  So the chain keeps the relative
L2 bound of 5e-3 and doubles the absolute one to 4e-2 (the attention's
2e-2 for its own rounding plus as much again for its perturbed inputs).
"""
import numpy as np
import pytest

import _harness as H
from causal_gqa_attention_flashattention_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EPS = 1e-5
CHAIN_MAX_ABS_TOL = 2 * H.MAX_ABS_TOL

# (B, T, C, Hq, Hkv, D).  Row counts B*T that leave a ragged last 128-row tile,
# a width C that is not a multiple of the 64-wide K blocks, D = 32 and 64.  The
# two model-width shapes run with more than one tile per SM, where the tile
# width picker takes 192 (gpu_116m_model: 8192 rows, 1280 features) and 256
# (8192 rows, 1536 features) columns on a 152-SM part; the small ones take 128.
QKV_SHAPES = [
    (2, 200, 256, 4, 2, 64),
    (1, 130, 200, 6, 3, 32),
    (1, 77, 128, 4, 2, 32),
    (3, 129, 8, 2, 1, 64),
    (16, 512, 768, 12, 4, 64),
    (8, 1024, 1024, 16, 4, 64),
]


@pytest.fixture(scope="module")
def nb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_flashattention_gb300 import binding
    binding.lib()
    return binding


def half_perm(D):
    """Column j of a half-split rotated row holds feature j/2 (even j) or D/2 + j//2 (odd j)."""
    return np.array([j // 2 if j % 2 == 0 else D // 2 + j // 2 for j in range(D)])


def run(nb, x, Hq, Hkv, D, rotated, half, write_qk=True):
    dx, dw, dW = (H.to_device(x[n + "_bits"]) for n in ("x", "norm_w", "w_qkv"))
    q, k, v, rstd, ws = nb.qkv_rmsnorm(dx, dw, dW, Hq, Hkv, D, eps=EPS, rope_base=inputs.ROPE_BASE,
                                       rotated=rotated, rope_half=half, write_qk=write_qk)
    nb.check_status()
    return q, k, v, rstd, ws


def check(name, gpu, ref, tol_rel=H.REL_L2_TOL, tol_abs=H.MAX_ABS_TOL):
    rel, mx = H.errors(gpu, ref)
    print("QKV", name, "rel %.2e abs %.2e" % (rel, mx))
    assert np.isfinite(gpu).all() and rel <= tol_rel and mx <= tol_abs, (name, rel, mx)


@pytest.mark.parametrize("shape", QKV_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("half", [False, True])
def test_qkv_projection_parity(nb, oracle_mod, shape, half):
    B, T, C, Hq, Hkv, D = shape
    x = inputs.make_prologue_inputs(B, T, C, Hq, Hkv, D, seed=900 + T + C)
    q, k, v, rstd, ws = run(nb, x, Hq, Hkv, D, rotated=True, half=half)
    rq, rk, rv, rr = oracle_mod.qkv_rmsnorm(x["x"], x["norm_w"], x["w_qkv"], Hq, Hkv, D, eps=EPS)
    check("q", H.to_f64(q), rq)
    check("k", H.to_f64(k), rk)
    check("v", H.to_f64(v), rv)
    check("rstd", rstd.cpu().numpy().astype(np.float64), rr, tol_rel=1e-5, tol_abs=1e-4)
    # rotated fp16 copies, in the order the attention kernels take them
    qr, kr = nb.rotated_qk(ws, B, T, Hq, Hkv, D)
    oq = oracle_mod.rope(rq, inputs.ROPE_BASE, half=half)
    ok = oracle_mod.rope(rk, inputs.ROPE_BASE, half=half)
    if half:
        oq, ok = oq[..., half_perm(D)], ok[..., half_perm(D)]
    check("q rotated", H.to_f64(qr), oq)
    check("k rotated", H.to_f64(kr), ok)


def test_qkv_without_rotation(nb, oracle_mod):
    """Without NE_ATTN_QK_ROTATED only q, k, v and rstd are written (no workspace prefix)."""
    B, T, C, Hq, Hkv, D = 2, 300, 192, 4, 2, 64
    x = inputs.make_prologue_inputs(B, T, C, Hq, Hkv, D, seed=41)
    q, k, v, rstd, ws = run(nb, x, Hq, Hkv, D, rotated=False, half=False)
    assert ws.numel() == nb.qkv_workspace_size(B, T, C, Hq, Hkv, D)
    rq, rk, rv, rr = oracle_mod.qkv_rmsnorm(x["x"], x["norm_w"], x["w_qkv"], Hq, Hkv, D, eps=EPS)
    check("q", H.to_f64(q), rq)
    check("k", H.to_f64(k), rk)
    check("v", H.to_f64(v), rv)


def test_qkv_rows_outside_the_problem_untouched(nb):
    """Ragged last tile: rows past B*T and columns past N are never written."""
    B, T, C, Hq, Hkv, D = 1, 77, 64, 2, 1, 32
    x = inputs.make_prologue_inputs(B, T, C, Hq, Hkv, D, seed=3)
    dx, dw, dW = (H.to_device(x[n + "_bits"]) for n in ("x", "norm_w", "w_qkv"))
    pad = 4096
    bufs = {n: torch.full((B * T * h * D + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
            for n, h in (("q", Hq), ("k", Hkv), ("v", Hkv))}
    rs = torch.full((B * T + pad,), 7.0, dtype=torch.float32, device="cuda")
    q = bufs["q"][:B * T * Hq * D].view(B, T, Hq, D)
    k = bufs["k"][:B * T * Hkv * D].view(B, T, Hkv, D)
    v = bufs["v"][:B * T * Hkv * D].view(B, T, Hkv, D)
    nb.qkv_rmsnorm(dx, dw, dW, Hq, Hkv, D, eps=EPS, q=q, k=k, v=v, rstd=rs[:B * T].view(B, T))
    nb.check_status()
    for n, h in (("q", Hq), ("k", Hkv), ("v", Hkv)):
        assert (bufs[n][B * T * h * D:].float() == 7.0).all(), n
    assert (rs[B * T:] == 7.0).all()


@pytest.mark.parametrize("shape", [(2, 200, 256, 4, 2, 64), (1, 130, 128, 6, 3, 32), (4, 512, 768, 12, 4, 64)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("half", [False, True])
def test_projection_feeds_attention(nb, oracle_mod, shape, half):
    """The chain a block runs: RMSNorm + projection writing only the rotated q, k
    (and v), then the attention forward and backward taking q, k from the
    workspace, against the oracle's projection followed by the oracle's attention."""
    B, T, C, Hq, Hkv, D = shape
    x = inputs.make_prologue_inputs(B, T, C, Hq, Hkv, D, seed=77 + T)
    n_bwd = nb.bwd_workspace_size(B, T, Hq, Hkv, D)
    n_qkv = nb.qkv_workspace_size(B, T, C, Hq, Hkv, D, rotated=True, rope_half=half)
    ws = torch.empty(max(n_bwd, n_qkv), dtype=torch.uint8, device="cuda")
    dx, dw, dW = (H.to_device(x[n + "_bits"]) for n in ("x", "norm_w", "w_qkv"))
    _, _, v, _, _ = nb.qkv_rmsnorm(dx, dw, dW, Hq, Hkv, D, eps=EPS, rotated=True, rope_half=half,
                                   write_qk=False, workspace=ws)
    dout_bits = inputs.bf16_round_bits(np.random.default_rng(5 + T).standard_normal((B, T, Hq, D)).astype(np.float32))
    do = H.to_device(dout_bits)
    o, lse = nb.attn_fwd(None, None, v, inputs.ROPE_BASE, workspace=ws, qk_rotated=True, Hq=Hq, rope_half=half)
    dq, dk, dv = nb.attn_bwd(None, None, v, o, lse, do, inputs.ROPE_BASE, grad_dtype=torch.float32, workspace=ws,
                             qk_rotated=True, rope_half=half)
    nb.check_status()
    rq, rk, rv, _ = oracle_mod.qkv_rmsnorm(x["x"], x["norm_w"], x["w_qkv"], Hq, Hkv, D, eps=EPS)
    ref = oracle_mod.attn_bwd(rq, rk, rv, inputs.bf16_bits_to_f64(dout_bits), inputs.ROPE_BASE, half=half)
    gpu = dict(o=H.to_f64(o), dq=H.to_f64(dq), dk=H.to_f64(dk), dv=H.to_f64(dv))
    rep = {n: H.errors(gpu[n], ref[n]) for n in gpu}
    rep["lse"] = H.errors(lse.cpu().numpy().astype(np.float64), ref["lse"])
    print("CHAIN", shape, half, {n: ("%.2e" % a, "%.2e" % b) for n, (a, b) in rep.items()})
    bad = [n for n in ("o", "dq", "dk", "dv") if rep[n][0] > H.REL_L2_TOL or rep[n][1] > CHAIN_MAX_ABS_TOL]
    assert not bad and rep["lse"][1] <= H.LSE_ABS_TOL, rep


def test_qkv_bad_arguments(nb):
    x = inputs.make_prologue_inputs(1, 16, 64, 2, 1, 32, seed=1)
    dx, dw, dW = (H.to_device(x[n + "_bits"]) for n in ("x", "norm_w", "w_qkv"))
    with pytest.raises(nb.NeAttnError):
        nb.qkv_rmsnorm(dx, dw, dW, 2, 1, 32, eps=0.0)
    with pytest.raises(ValueError):
        nb.qkv_rmsnorm(dx, dw, dW, 2, 1, 32, write_qk=False)  # nothing would hold q and k
    nb.check_status()


@pytest.mark.parametrize("shape,base", [((4, 1, 64, 2, 1, 32), inputs.ROPE_BASE), ((2, 150, 128, 4, 2, 64), 500000.0)],
                         ids=["one_position", "base_500000"])
def test_qkv_other_sizes_and_base(nb, oracle_mod, shape, base):
    """Sequences of one position (four rows in all) and another rotary base."""
    B, T, C, Hq, Hkv, D = shape
    x = inputs.make_prologue_inputs(B, T, C, Hq, Hkv, D, seed=31 + T)
    dx, dw, dW = (H.to_device(x[n + "_bits"]) for n in ("x", "norm_w", "w_qkv"))
    q, k, v, rstd, ws = nb.qkv_rmsnorm(dx, dw, dW, Hq, Hkv, D, eps=EPS, rope_base=base, rotated=True)
    nb.check_status()
    rq, rk, rv, rr = oracle_mod.qkv_rmsnorm(x["x"], x["norm_w"], x["w_qkv"], Hq, Hkv, D, eps=EPS)
    check("q", H.to_f64(q), rq)
    check("v", H.to_f64(v), rv)
    qr, kr = nb.rotated_qk(ws, B, T, Hq, Hkv, D)
    check("q rotated", H.to_f64(qr), oracle_mod.rope(rq, base))
    check("k rotated", H.to_f64(kr), oracle_mod.rope(rk, base))
