"""The tolerance of the FP8 forward (NE_ATTN_FP8), derived on the CPU.

The pages fix no precision for an 8-bit variant, so its bound comes from the
arithmetic: e4m3 keeps 3 mantissa bits (relative rounding up to 2^-4), so
each rotated feature of q and k moves by up to 6 %.  For unit-normal q and k
the logits (sum of 64 products over sqrt(64)) then move by about 0.05, which
reaches O through softmax.  The emulation below rounds the oracle's rotated
q, k to e4m3 with one scale per head, rotates back and runs the exact
attention on them: that error floor is what the GPU path cannot beat.  The
bound in _harness.fp8_bounds is the floor of the same inputs with a 1.5x
margin plus the default path's own bounds (a floor measured on one small case
would be too tight for larger ones: the maximum error grows with the number
of outputs).  The e4m3 rounding
itself is pinned to values worked out from the format's definition, and the
per-head scale to a tensor worked by hand (oracle/fp8.py holds the emulation).
"""
import numpy as np

import _harness as H
from causal_gqa_attention_flashattention_gb300 import inputs


def test_e4m3_rounding_pins():
    # 1 + 1/16 lies halfway between 1 and 1.125: ties to the even mantissa (1.0);
    # 1.1875 lies halfway between 1.125 and 1.25: ties to 1.25 (mantissa 010)
    vals = np.array([1.0, 1.0625, 1.1875, 448.0, 464.0, 1000.0, 2.0 ** -9, 3 * 2.0 ** -10, -0.3, 0.0])
    want = np.array([1.0, 1.0, 1.25, 448.0, 448.0, 448.0, 2.0 ** -9, 2.0 ** -8, -0.3125, 0.0])
    np.testing.assert_array_equal(H.e4m3_round(vals), want)
    # every representable positive value is a fixed point
    grid = [m * 2.0 ** -9 for m in range(8)] + [(1 + m / 8) * 2.0 ** e for e in range(-6, 9) for m in range(8)]
    grid = np.array([g for g in grid if g <= 448.0])
    np.testing.assert_array_equal(H.e4m3_round(grid), grid)
    assert len(np.unique(grid)) == 127  # 0, 7 subnormals and 15 x 8 normals less 480 (codes 0x00..0x7e)


# A [B=2, T=2, H=2, D=2] tensor worked by hand.  Head 0 takes its largest
# |value| (3.5) at batch 1, position 0; head 1 its largest (0.7) at batch 0,
# position 1 (and -0.7 at batch 1).  Scales: 3.5 / 448 = 2^-7 (codes = value *
# 128) and 0.7 / 448 = 1 / 640 (codes = value * 640).  Codes on the e4m3 grid:
#   0.3 * 128 = 38.4   in [32, 64), step 4          -> 40    -> 0.3125
#   -1.1 * 128 = -140.8 in [128, 256), step 16      -> -144  -> -1.125
#   0.01 * 128 = 1.28  in [1, 2), step 1/8          -> 1.25  -> 0.009765625
#   3.5 * 128 = 448, 1.0 * 128 = 128, 2.0 * 128 = 256 (on the grid)
#   0.123 * 640 = 78.72 in [64, 128), step 8         -> 80    -> 0.125
#   3e-4 * 640 = 0.192 in [1/8, 1/4), step 1/64      -> 0.1875 -> 2.9296875e-4
#   0.1 * 640 = 64, -0.05 * 640 = -32, 0.7 * 640 = 448 (on the grid)
PER_HEAD_X = np.array([
    [[[0.3, -1.1], [0.1, 3e-4]],      # b=0, t=0: head 0, head 1
     [[0.01, 0.0], [0.7, -0.05]]],    # b=0, t=1
    [[[1.0, 3.5], [0.123, 0.0]],      # b=1, t=0
     [[-0.3, 2.0], [-0.7, 0.0]]],     # b=1, t=1
])
PER_HEAD_CODES = np.array([
    [[[40.0, -144.0], [64.0, 0.1875]],
     [[1.25, 0.0], [448.0, -32.0]]],
    [[[128.0, 448.0], [80.0, 0.0]],
     [[-40.0, 256.0], [-448.0, 0.0]]],
])
PER_HEAD_VALUES = np.array([
    [[[0.3125, -1.125], [0.1, 2.9296875e-4]],
     [[0.009765625, 0.0], [0.7, -0.05]]],
    [[[1.0, 3.5], [0.125, 0.0]],
     [[-0.3125, 2.0], [-0.7, 0.0]]],
])


def test_e4m3_per_head_scale_pins():
    from oracle import fp8
    np.testing.assert_array_equal(fp8.head_scales(PER_HEAD_X), [3.5, 0.7])
    vals, codes = fp8.e4m3_per_head(PER_HEAD_X, return_codes=True)
    np.testing.assert_allclose(codes, PER_HEAD_CODES, rtol=1e-12, atol=0)
    np.testing.assert_allclose(vals, PER_HEAD_VALUES, rtol=1e-12, atol=1e-18)
    # a scale per (batch, head) or per row rounds this tensor differently: the
    # reduction axes are pinned, not just the element rounding
    for axes in ((1, 3), (3,)):
        amax = np.max(np.abs(PER_HEAD_X), axis=axes, keepdims=True)
        s = np.where(amax > 0, amax / 448.0, 1.0)
        other = fp8.e4m3_round(PER_HEAD_X / s) * s
        assert np.max(np.abs(other - PER_HEAD_VALUES)) > 1e-3, axes
    # a head of zeros keeps zero codes
    z = np.zeros((1, 3, 2, 4))
    z[0, 1, 0, 2] = 0.5
    v, c = fp8.e4m3_per_head(z, return_codes=True)
    assert c[0, 1, 0, 2] == 448.0 and v[0, 1, 0, 2] == 0.5 and not np.any(c[:, :, 1])


def test_fp8_floor_level(oracle_mod):
    """The floor the FP8 bound is built on: about 3e-2 relative in O on
    unit-normal inputs, far above the default path's 5e-3, and the bound
    derived from it stays within about 2x of it."""
    B, T, Hq, Hkv, D = 2, 256, 4, 2, 64
    x = H.make(B, T, Hq, Hkv, D, seed=61)
    floor, _, _ = H.fp8_floor(oracle_mod, x, inputs.ROPE_BASE)
    rel, mx, lse = floor
    print("e4m3 floor: O rel %.3e abs %.3e, LSE abs %.3e" % floor)
    assert 0.02 < rel < 0.05 and 0.03 < mx < 0.3 and 0.02 < lse < 0.3
    b_rel, b_mx, b_lse = H.fp8_bounds(floor)
    assert b_rel <= 2.0 * rel and b_mx <= 2.0 * mx and b_lse <= 2.5 * lse
