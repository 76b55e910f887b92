"""Shared helpers for the GPU parity tests: seeded inputs -> device, error metrics."""
import numpy as np

from causal_gqa_attention_flashattention_gb300 import inputs

# Tolerances for O, dQ, dK, dV against the fp64 oracle on the same bf16 inputs.
REL_L2_TOL = 5e-3
MAX_ABS_TOL = 2e-2
# LSE is not covered by the stated tolerance; the fp32 online softmax keeps it
# within a few fp32 ulps of ln(sum exp) times the row's dynamic range.
LSE_ABS_TOL = 1e-2


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
