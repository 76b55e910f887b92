"""ne_attn_bwd_noalloc: the backward pass for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc when they need the
backward pass, for example a plugin whose host process owns all device memory,
or a deployment that fixes its memory at start-up.  For them
the library has an entry point that takes no workspace and allocates nothing:
its scratch is one fixed device array inside the library.  These tests call it
through the C ABI and check that it returns what ne_attn_bwd (with a caller
workspace) returns, on two calls in a row, within the parity tolerances the
other tests use.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import _harness as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

NE_ERR_SCRATCH_LIMIT = -7


@pytest.fixture(scope="module")
def nb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_flashattention_gb300 import binding
    L = binding.lib()
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.ne_attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    L.ne_attn_bwd_noalloc.restype = i
    return binding


def _noalloc_bwd(nb, q, k, v, o, lse, do, flags):
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    gd = torch.float32 if flags & nb.GRAD_FP32 else torch.bfloat16
    dq = torch.full(q.shape, float("nan"), dtype=gd, device="cuda")
    dk = torch.full(k.shape, float("nan"), dtype=gd, device="cuda")
    dv = torch.full(k.shape, float("nan"), dtype=gd, device="cuda")
    st = nb.lib().ne_attn_bwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, T, Hq, Hkv, D, 10000.0, flags,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, nb.lib().ne_attn_status_string(st)
    nb.check_status()
    return dq, dk, dv


def _close(a, b):
    """a within the parity tolerances of the fp32 result b; a bf16 result also
    carries the half-ulp its own rounding adds (2^-9 of the value)."""
    half_ulp = 2.0 ** -9 if a.dtype == torch.bfloat16 else 0.0
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    rel, mx = H.errors(a, b)
    assert rel <= H.REL_L2_TOL, rel
    assert np.all(np.abs(a - b) <= H.MAX_ABS_TOL + np.abs(b) * half_ulp), mx


@pytest.mark.parametrize("shape,precise,half,fp32", [
    ((2, 300, 6, 2, 64), False, False, True), ((1, 200, 4, 2, 32), False, False, True),
    ((1, 257, 3, 1, 64), True, False, True),
    ((2, 300, 6, 2, 64), False, True, True),     # half-split rotary layout
    ((2, 300, 6, 2, 64), False, False, False),   # bf16 gradients
    ((16, 512, 12, 4, 64), False, False, True),  # the 116M model's attention shape
])
def test_noalloc_matches_workspace_entry_point(nb, shape, precise, half, fp32):
    B, T, Hq, Hkv, D = shape
    flags = ((nb.GRAD_FP32 if fp32 else 0) | ((nb.PRECISE_QK | nb.O_FP32) if precise else 0)
             | (nb.ROPE_HALF if half else 0))
    outs = []
    for call in range(2):  # two calls in a row: the fixed scratch keeps the previous call's contents
        x = H.make(*shape, seed=100 + call, recipe="stress" if precise else "normal")
        q, k, v, do = (H.to_device(x[n + "_bits"]) for n in ("q", "k", "v", "dout"))
        o, lse = nb.attn_fwd(q, k, v, o_dtype=torch.float32 if precise else torch.bfloat16, precise=precise,
                             rope_half=half)
        ref = nb.attn_bwd(q, k, v, o, lse, do, grad_dtype=torch.float32, precise=precise, rope_half=half)
        got = _noalloc_bwd(nb, q, k, v, o, lse, do, flags)
        for r, g in zip(ref, got):
            assert torch.isfinite(g).all()
            _close(g, r)
        outs.append(got)
    assert not torch.equal(outs[0][1], outs[1][1])  # the second call really computed new results


def test_noalloc_rejects_problems_beyond_its_scratch(nb):
    # 4 x 8192 x 16 heads at D = 64 needs ~330 MB of scratch: far past the fixed array.
    B, T, Hq, Hkv, D = 4, 8192, 16, 4, 64
    q = torch.empty((1, 16, 1, 64), dtype=torch.bfloat16, device="cuda")  # never touched
    st = nb.lib().ne_attn_bwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(),
                                      q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), B, T, Hq, Hkv, D,
                                      10000.0, 0, None)
    assert st == NE_ERR_SCRATCH_LIMIT
    assert b"scratch" in nb.lib().ne_attn_status_string(st)
