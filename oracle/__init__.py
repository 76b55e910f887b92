"""fp64 CPU oracle for causal GQA attention with RoPE on Q/K, and for the
RMSNorm + Q/K/V projection step that feeds it.

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(the CUDA library and its Python binding) never does, and this package never
imports the product package.

The e4m3 rounding with one scale per head, the oracle of the FP8 forward,
is in ``fp8.py``.  The attention arithmetic lives in ``attn_oracle.c``
(plain C, double precision, OpenMP over rows); this module compiles it with gcc and marshals
numpy arrays.  The RMSNorm + projection step (``qkv_rmsnorm``) is written here
in float64 numpy, with one library matrix product.  The header of
``attn_oracle.c`` and the docstrings below name the passages of the NanoEuler
pages each step follows and the readings taken where the pages are silent.

Every function is pinned by ``tests/test_oracle_pins.py`` (brute force in a
second formulation, closed forms, invariants and central finite differences)
and the e4m3 emulation by ``tests/test_fp8_tolerance.py`` (values worked by
hand from the format and the per-head scale); no function here is "parity
unpinned".
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force=False):
    """Compile attn_oracle.c into _build/liboracle.so (gcc, -O2, OpenMP).

    No -ffast-math and no -march flags: the oracle keeps IEEE double
    semantics and builds the same way on x86-64 and AArch64 hosts.
    """
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        u8p = ctypes.POINTER(ctypes.c_ubyte)
        i = ctypes.c_int
        lib.oracle_rope.argtypes = [dp, dp, i, i, i, i, ctypes.c_double, i, i]
        lib.oracle_rope.restype = None
        lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i,
                                        ctypes.c_double, i, u8p, i]
        lib.oracle_attn_fwd.restype = None
        lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                        i, i, i, i, i, ctypes.c_double, i, u8p, i]
        lib.oracle_attn_bwd.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i
        _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _sel(B, Hkv, groups):
    """groups: None (all) or an iterable of (b, kv_head) pairs to compute."""
    if groups is None:
        return None
    s = np.zeros(B * Hkv, dtype=np.uint8)
    for b, g in groups:
        s[b * Hkv + g] = 1
    return s


def num_threads():
    return _load().oracle_num_threads()


def rope(x, base, inverse=False, half=False):
    """R_t x for x of shape [B, T, H, D] (interleaved pairs); R_t^T x if inverse."""
    lib = _load()
    x = _f64(x)
    B, T, H, D = x.shape
    out = np.empty_like(x)
    lib.oracle_rope(_p(x), _p(out), B, T, H, D, float(base), -1 if inverse else 1, int(bool(half)))
    return out


def attn_fwd(q, k, v, base=10000.0, groups=None, nthreads=0, half=False):
    """Causal GQA attention forward.  q [B,T,Hq,D], k/v [B,T,Hkv,D] (fp64).

    Returns (o [B,T,Hq,D], lse [B,Hq,T]); entries of groups not selected are NaN.
    """
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, T, Hkv, D) and v.shape == k.shape and Hq % Hkv == 0
    o = np.full(q.shape, np.nan)
    lse = np.full((B, Hq, T), np.nan)
    sel = _sel(B, Hkv, groups)
    lib.oracle_attn_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, T, Hq, Hkv, D,
                        float(base), int(bool(half)),
                        None if sel is None else sel.ctypes.data_as(
                            ctypes.POINTER(ctypes.c_ubyte)), int(nthreads))
    return o, lse


def decode_fwd(q_new, k, v, base=10000.0, groups=None, nthreads=0, half=False):
    """Decode step with a key/value cache (the engine's incremental generation
    with a KV cache: mynewscn README; socker-news README, GPU generation mode).

    The Tq queries q_new [B,Tq,Hq,D] sit at positions T-Tq .. T-1 of
    k/v [B,T,Hkv,D] and attend causally; the result is rows T-Tq .. T-1 of the
    forward over T positions.  Earlier query rows cannot reach those rows, so
    they are zero here.  Returns (o [B,Tq,Hq,D], lse [B,Hq,Tq]).
    """
    q_new = _f64(q_new)
    B, Tq, Hq, D = q_new.shape
    T = k.shape[1]
    assert 1 <= Tq <= T
    q = np.zeros((B, T, Hq, D))
    q[:, T - Tq:] = q_new
    o, lse = attn_fwd(q, k, v, base, groups, nthreads, half)
    return o[:, T - Tq:].copy(), lse[:, :, T - Tq:].copy()


def attn_bwd(q, k, v, dout, base=10000.0, groups=None, nthreads=0, half=False):
    """Causal GQA attention backward from the definition.

    Returns dict with dq, dk, dv and the forward by-products o, lse and
    delta (= sum_j P_tj dP_tj, shape [B,Hq,T]).  Unselected groups are NaN.
    """
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    assert dout.shape == q.shape and Hq % Hkv == 0
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(k.shape, np.nan)
    o = np.full(q.shape, np.nan)
    lse = np.full((B, Hq, T), np.nan)
    delta = np.full((B, Hq, T), np.nan)
    sel = _sel(B, Hkv, groups)
    lib.oracle_attn_bwd(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv),
                        _p(o), _p(lse), _p(delta), B, T, Hq, Hkv, D, float(base), int(bool(half)),
                        None if sel is None else sel.ctypes.data_as(
                            ctypes.POINTER(ctypes.c_ubyte)), int(nthreads))
    return dict(dq=dq, dk=dk, dv=dv, o=o, lse=lse, delta=delta)



def qkv_rmsnorm(x, norm_w, w_qkv, Hq, Hkv, D, eps=1e-5):
    """The step in front of attention: RMSNorm, then the fused Q/K/V projection.

    Each NanoEuler block computes x + attn(rmsnorm(x)) with a pre-norm
    RMSNorm and no bias anywhere (socker-news README, "Architecture" and
    "Block structure order"; mynewscn README, architecture list).  The pages
    name RMSNorm without writing it out; its definition (Zhang and Sennrich,
    "Root Mean Square Layer Normalization", 2019) is
        rstd_r = 1 / sqrt(mean_c x[r, c]^2 + eps),   xn[r, c] = x[r, c] * rstd_r * w[c].
    The projection is one matrix for all three (read here as rows
    [Hq*D query features | Hkv*D key features | Hkv*D value features] of
    w_qkv [N, C], the output-by-input layout), qkv = xn W^T, without bias.
    The rotary embedding is not part of this step: attn_fwd applies it.

    x [B, T, C], norm_w [C], w_qkv [(Hq + 2 Hkv) D, C], all taken exactly as
    float64.  Returns (q [B,T,Hq,D], k [B,T,Hkv,D], v [B,T,Hkv,D], rstd [B,T]).
    """
    x, w, W = _f64(x), _f64(norm_w), _f64(w_qkv)
    B, T, C = x.shape
    N = (Hq + 2 * Hkv) * D
    assert w.shape == (C,) and W.shape == (N, C)
    rstd = 1.0 / np.sqrt(np.mean(x * x, axis=-1) + float(eps))
    xn = x * rstd[..., None] * w
    qkv = xn.reshape(B * T, C) @ W.T
    q = qkv[:, :Hq * D].reshape(B, T, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(B, T, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].reshape(B, T, Hkv, D)
    return q.copy(), k.copy(), v.copy(), rstd
