"""e4m3 emulation for the FP8 forward's oracle (float64 numpy).

TEST INFRASTRUCTURE ONLY, like the rest of this package: the test-suite and
the CPU-baseline leg of ``bench.py`` may import it; the product path never
does, and it imports nothing of the product package.

The FP8 forward is an inference variant of the attention path.  The pages
name no 8-bit format: the variant and its one scale per head are this
library's reading.  What it computes is attention on the rotated q and k
after each has been rounded to the OCP FP8 E4M3 format with one scale per
head:

  scale_h = max |x| over all batches, positions and features of head h,
  code    = e4m3(x * 448 / scale_h)   (round to nearest, ties to even,
                                       saturating at 448),
  value   = code * scale_h / 448.

The format (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; the
exponent field 15 with mantissa 111 is NaN, so the largest finite value is
1.75 * 2^8 = 448; subnormals step by 2^-9) is written out in ``e4m3_round``
from that definition.  Pins (tests/test_fp8_tolerance.py): values worked by
hand from the format (ties, saturation, subnormals, the 127 non-negative
codes), and a hand-worked tensor whose heads take their maxima at different
batches and positions, which a scale per (batch, head) or per row would
round differently.
"""
import numpy as np

E4M3_MAX = 448.0


def e4m3_round(x):
    """Round to the E4M3 grid: for |x| >= 2^-6 the spacing is 2^(e - 3) with
    e = floor(log2 |x|) (at most 8); below 2^-6 it is the subnormal step 2^-9.
    Round to nearest, ties to even (numpy's round), saturate at 448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.clip(np.floor(np.log2(np.maximum(a, 2.0 ** -9))), -6, 8)
    step = 2.0 ** (e - 3)
    return np.sign(x) * np.minimum(np.round(a / step) * step, E4M3_MAX)


def head_scales(xr):
    """xr [B,T,H,D] -> [H] largest |value| of each head over its batches,
    positions and features (axes 0, 1 and 3)."""
    return np.max(np.abs(np.asarray(xr, dtype=np.float64)), axis=(0, 1, 3))


def e4m3_per_head(xr, return_codes=False):
    """xr [B,T,H,D] rotated values -> their e4m3 rounding with one scale per
    head, returned as values (code * scale_h / 448); with return_codes also
    the codes themselves (values on the e4m3 grid, |code| <= 448).  A head
    whose values are all zero keeps scale 1 (its codes are zero)."""
    xr = np.asarray(xr, dtype=np.float64)
    amax = head_scales(xr)[None, None, :, None]
    s = np.where(amax > 0, amax / E4M3_MAX, 1.0)
    codes = e4m3_round(xr / s)
    if return_codes:
        return codes * s, codes
    return codes * s
