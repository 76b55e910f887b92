"""Shared helpers for the GPU parity tests: seeded inputs -> device, error metrics."""
import numpy as np

from causal_gqa_attention_flashattention_gb300 import inputs
from oracle.fp8 import e4m3_per_head, e4m3_round  # noqa: F401  (the FP8 oracle)

# Tolerances for O, dQ, dK, dV against the fp64 oracle on the same bf16 inputs.
REL_L2_TOL = 5e-3
MAX_ABS_TOL = 2e-2
# LSE is not covered by the stated tolerance; the fp32 online softmax keeps it
# within a few fp32 ulps of ln(sum exp) times the row's dynamic range.
LSE_ABS_TOL = 1e-2

# The long-context stress workload in split precision (NE_ATTN_PRECISE_QK).  Its
# outlier rows reach logits |s| ~ 1.7e4.  The split-precision logits carry the
# rotated q, k as fp16 hi + lo (22 mantissa bits: 2^-22 relative per operand)
# and accumulate in fp32 (2^-24 per step at |s|), so a logit is off by up to
# ~2^-21 |s|, about 1e-2 at 1.7e4 (the LSE, measured: 1.1e-2).  A row's P then
# moves by that much relative, and dq = scale sum_j dS_tj k_j, dk (and the LSE)
# with it: on the few rows whose gradients reach 1e2 .. 3e2 the error is about
# 1e-3 of the value, above the absolute 2e-2 (measured 1.1e-3 relative at
# worst).  For dq and dk on that workload each element is held to
# 2e-2 + 2e-3 |value|; the LSE to 1e-2 + 2^-20 |lse|.  O and dv, and the
# relative L2 of every tensor, keep the stated bounds.
STRESS_GRAD_REL = 2e-3
STRESS_LSE_REL = 2.0 ** -20


def to_device(bits):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy())
    return t.view(torch.bfloat16).to("cuda")


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def errors(gpu, ref):
    d = gpu - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(d) / nref if nref > 0 else np.linalg.norm(d)
    return float(rel), float(np.max(np.abs(d))) if d.size else 0.0


def group_slices(B, Hq, Hkv, groups):
    """Index helpers selecting the query heads / kv head of each (b, g) group."""
    G = Hq // Hkv
    if groups is None:
        groups = [(b, g) for b in range(B) for g in range(Hkv)]
    qsel = [(b, slice(g * G, (g + 1) * G)) for b, g in groups]
    ksel = [(b, g) for b, g in groups]
    return qsel, ksel


def gather_q(x, qsel):      # x [B,T,Hq,D] -> stacked selection
    return np.stack([x[b, :, hs] for b, hs in qsel])


def gather_k(x, ksel):      # x [B,T,Hkv,D]
    return np.stack([x[b, :, g] for b, g in ksel])


def gather_lse(x, qsel):    # x [B,Hq,T]
    return np.stack([x[b, hs] for b, hs in qsel])


def make(B, T, Hq, Hkv, D, seed, recipe="normal"):
    return inputs.make_shape_inputs(B, T, Hq, Hkv, D, seed, recipe)


# ------------------------------------------------------------------ the FP8 forward
# The bound for NE_ATTN_FP8 (derived in tests/test_fp8_tolerance.py) is the error
# that the e4m3 rounding of the rotated q, k alone causes on the same inputs (the
# "floor": exact attention on the rounded values against exact attention), with a
# 1.5x margin, plus the default path's own bounds for everything after the rounding.
# On unit-normal inputs the floor is about 3e-2 relative in O.
FP8_FLOOR_MARGIN = 1.5


def fp8_bounds(floor):
    """floor = (O rel L2, O max abs, LSE max abs) of the e4m3 emulation -> bounds."""
    rel, mx, lse = floor
    return (FP8_FLOOR_MARGIN * rel + REL_L2_TOL, FP8_FLOOR_MARGIN * mx + MAX_ABS_TOL,
            FP8_FLOOR_MARGIN * lse + LSE_ABS_TOL)


def fp8_floor(oracle_mod, x, base, half=False):
    """Exact attention on e4m3-rounded rotated q, k (per-head scales) against
    exact attention: returns ((rel, max abs, LSE max abs), ref_o, ref_lse)."""
    ref_o, ref_l = oracle_mod.attn_fwd(x["q"], x["k"], x["v"], base, half=half)
    q8 = oracle_mod.rope(e4m3_per_head(oracle_mod.rope(x["q"], base, half=half)), base, inverse=True, half=half)
    k8 = oracle_mod.rope(e4m3_per_head(oracle_mod.rope(x["k"], base, half=half)), base, inverse=True, half=half)
    o8, l8 = oracle_mod.attn_fwd(q8, k8, x["v"], base, half=half)
    rel, mx = errors(o8, ref_o)
    return (rel, mx, float(np.max(np.abs(l8 - ref_l)))), ref_o, ref_l
