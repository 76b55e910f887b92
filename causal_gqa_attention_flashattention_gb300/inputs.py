"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it draws normal samples, applies
the workload recipe (scaling, outlier rows), rounds to bfloat16 and returns
both the bf16 bit patterns (for the device) and their exact fp64 values (for
the CPU checker).  It imports neither the CUDA binding nor the checker.

The workloads are shaped like the NanoEuler models (socker-news README,
"Configuration" table: CPU model dim 128 with 4/2 heads, GPU model dim 768
with 12/4 heads and context 512; planned scale-up to ~270M parameters in the
"Roadmap"), with the long-context stress case added on top.
"""
import numpy as np

# name -> (B, T, Hq, Hkv, D, recipe)
WORKLOADS = {
    "tiny_cpu_model": (2, 128, 4, 2, 32, "normal"),
    "cpu_small_model_ctx512": (8, 512, 4, 2, 32, "normal"),
    "gpu_116m_model": (16, 512, 12, 4, 64, "normal"),
    "scaled_270m_synthetic": (8, 1024, 16, 4, 64, "normal"),
    "long_context_stress": (2, 8192, 12, 4, 64, "stress"),
}
WORKLOAD_ORDER = list(WORKLOADS)
ROPE_BASE = 10000.0


def bf16_round_bits(x32):
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16.  Inputs are finite here.
    """
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return ((u + rounding) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f64(bits):
    """Exact widening of bf16 bit patterns to float64."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _seed_for(name, seed):
    if seed is not None:
        return seed
    return 1234 + WORKLOAD_ORDER.index(name)


def make_shape_inputs(B, T, Hq, Hkv, D, seed, recipe="normal"):
    """Draw q, k, v, dO for one problem.

    recipe "normal": all four ~ N(0, 1).
    recipe "stress": q, k ~ 4 * N(0, 1), and every (b, t, h) D-vector of q and,
      independently, of k is multiplied by 16 with probability 0.01 (large
      logits); v, dO ~ N(0, 1).  Scaling happens before bf16 rounding.

    Returns a dict with "<name>_bits" (uint16 bf16 patterns) and "<name>"
    (float64 exact values) for name in q, k, v, dout.
    """
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, D), dtype=np.float32)
    k = rng.standard_normal((B, T, Hkv, D), dtype=np.float32)
    v = rng.standard_normal((B, T, Hkv, D), dtype=np.float32)
    do = rng.standard_normal((B, T, Hq, D), dtype=np.float32)
    if recipe == "stress":
        q *= np.float32(4.0)
        k *= np.float32(4.0)
        q *= np.where(rng.random((B, T, Hq, 1)) < 0.01, np.float32(16.0), np.float32(1.0))
        k *= np.where(rng.random((B, T, Hkv, 1)) < 0.01, np.float32(16.0), np.float32(1.0))
    elif recipe != "normal":
        raise ValueError("unknown recipe %r" % recipe)
    out = {}
    for name, arr in (("q", q), ("k", k), ("v", v), ("dout", do)):
        bits = bf16_round_bits(arr)
        out[name + "_bits"] = bits
        out[name] = bf16_bits_to_f64(bits)
    return out


def make_workload_inputs(name, seed=None):
    B, T, Hq, Hkv, D, recipe = WORKLOADS[name]
    return make_shape_inputs(B, T, Hq, Hkv, D, _seed_for(name, seed), recipe)


def workload_shape(name):
    B, T, Hq, Hkv, D, _ = WORKLOADS[name]
    return dict(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D)


# name -> (B, T, C, Hq, Hkv, D): the step in front of attention (RMSNorm and the
# Q/K/V projection) at the models' widths (socker-news README, "Configuration").
PROLOGUE_WORKLOADS = {
    "tiny_cpu_model": (2, 128, 128, 4, 2, 32),
    "gpu_116m_model": (16, 512, 768, 12, 4, 64),
}


def make_prologue_inputs(B, T, C, Hq, Hkv, D, seed):
    """Draw the inputs of RMSNorm + the fused Q/K/V projection.

    x ~ N(0, 1) [B, T, C] (a residual stream of unit scale); the norm weight
    ~ 1 + 0.1 N(0, 1) [C] (near its initial value of one); the projection
    w_qkv ~ N(0, 1) / sqrt(C) [(Hq + 2 Hkv) D, C], so the projected q, k, v
    are of unit scale like the attention workloads' inputs.  All rounded to
    bf16.  Returns "<name>_bits" and "<name>" (exact fp64) for x, norm_w, w_qkv.
    """
    rng = np.random.default_rng(seed)
    N = (Hq + 2 * Hkv) * D
    x = rng.standard_normal((B, T, C), dtype=np.float32)
    w = (1.0 + 0.1 * rng.standard_normal(C)).astype(np.float32)
    W = (rng.standard_normal((N, C), dtype=np.float32) / np.float32(np.sqrt(C))).astype(np.float32)
    out = {}
    for name, arr in (("x", x), ("norm_w", w), ("w_qkv", W)):
        bits = bf16_round_bits(arr)
        out[name + "_bits"] = bits
        out[name] = bf16_bits_to_f64(bits)
    return out
