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
itself is pinned to values worked out from the format's definition.
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
