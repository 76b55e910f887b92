"""GPU parity of the FP8 forward (NE_ATTN_FP8): e4m3 rotated q, k with one
scale per head, S on the 8-bit tensor-core path, v / P / O as in the default
forward.  Checked against the fp64 oracle on the same bf16 inputs with the
bound derived in test_fp8_tolerance.py (the e4m3 floor of the same inputs
with a 1.5x margin, plus the default path's bounds), and against the CPU
emulation of the same e4m3 rounding (oracle/fp8.py, written from the format's
definition and pinned by hand-worked values), which it must follow far more
closely than the exact oracle.
"""
import numpy as np
import pytest

import _harness as H
from causal_gqa_attention_flashattention_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FP8_SHAPES = [(2, 200, 4, 2, 64), (1, 384, 12, 4, 64), (3, 77, 8, 1, 64), (16, 512, 12, 4, 64)]


@pytest.fixture(scope="module")
def nb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_flashattention_gb300 import binding
    binding.lib()
    return binding


def fp8_run(nb, x, half=False, o_dtype=None):
    q, k, v = (H.to_device(x[n + "_bits"]) for n in ("q", "k", "v"))
    o, lse = nb.attn_fwd(q, k, v, inputs.ROPE_BASE, fp8=True, rope_half=half, o_dtype=o_dtype or torch.bfloat16)
    nb.check_status()
    return H.to_f64(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape", FP8_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("half", [False, True])
def test_fp8_forward_parity(nb, oracle_mod, shape, half):
    B, T, Hq, Hkv, D = shape
    x = H.make(B, T, Hq, Hkv, D, seed=300 + T)
    o, lse = fp8_run(nb, x, half)
    floor, ref_o, ref_l = H.fp8_floor(oracle_mod, x, inputs.ROPE_BASE, half)
    b_rel, b_mx, b_lse = H.fp8_bounds(floor)
    rel, mx = H.errors(o, ref_o)
    ls = float(np.max(np.abs(lse - ref_l)))
    print("FP8", shape, half, "o rel %.2e abs %.2e lse abs %.2e | floor %.2e %.2e %.2e" % ((rel, mx, ls) + floor))
    assert np.isfinite(o).all() and rel <= b_rel and mx <= b_mx and ls <= b_lse


@pytest.mark.parametrize("half", [False, True])
def test_fp8_follows_the_e4m3_emulation(nb, oracle_mod, half):
    """Against attention on the e4m3-rounded q, k (CPU emulation, per-head scales)
    the error is the default path's own (bf16 P, fp32 accumulation), not the
    3e-2 of the rounding: the kernel rounds what the emulation rounds."""
    B, T, Hq, Hkv, D = 2, 256, 4, 2, 64
    x = H.make(B, T, Hq, Hkv, D, seed=62)
    o, lse = fp8_run(nb, x, half)
    base = inputs.ROPE_BASE
    q8 = oracle_mod.rope(H.e4m3_per_head(oracle_mod.rope(x["q"], base, half=half)), base, inverse=True, half=half)
    k8 = oracle_mod.rope(H.e4m3_per_head(oracle_mod.rope(x["k"], base, half=half)), base, inverse=True, half=half)
    em_o, em_l = oracle_mod.attn_fwd(q8, k8, x["v"], base, half=half)
    ex_o, _ = oracle_mod.attn_fwd(x["q"], x["k"], x["v"], base, half=half)
    rel_em, mx_em = H.errors(o, em_o)
    rel_ex, _ = H.errors(o, ex_o)
    print("FP8 vs emulation rel %.2e abs %.2e lse %.2e | vs exact rel %.2e" % (
        rel_em, mx_em, float(np.max(np.abs(lse - em_l))), rel_ex))
    assert rel_em <= H.REL_L2_TOL and rel_em < 0.3 * rel_ex and float(np.max(np.abs(lse - em_l))) <= H.LSE_ABS_TOL


def test_fp8_fp32_output(nb, oracle_mod):
    B, T, Hq, Hkv, D = 1, 300, 6, 2, 64
    x = H.make(B, T, Hq, Hkv, D, seed=63)
    o, lse = fp8_run(nb, x, o_dtype=torch.float32)
    floor, ref_o, ref_l = H.fp8_floor(oracle_mod, x, inputs.ROPE_BASE)
    b_rel, b_mx, b_lse = H.fp8_bounds(floor)
    rel, mx = H.errors(o, ref_o)
    assert rel <= b_rel and mx <= b_mx and float(np.max(np.abs(lse - ref_l))) <= b_lse


def test_fp8_flag_rules(nb):
    x = H.make(1, 64, 2, 1, 32, seed=1)
    q, k, v = (H.to_device(x[n + "_bits"]) for n in ("q", "k", "v"))
    with pytest.raises(nb.NeAttnError):
        nb.attn_fwd(q, k, v, fp8=True)  # D = 32
    x = H.make(1, 64, 2, 1, 64, seed=1)
    q, k, v = (H.to_device(x[n + "_bits"]) for n in ("q", "k", "v"))
    with pytest.raises(nb.NeAttnError):
        nb.attn_fwd(q, k, v, fp8=True, precise=True)
    nb.check_status()
