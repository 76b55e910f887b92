"""ctypes binding for libneattn.so (C ABI in include/ne_attn.h).

Argument marshalling only: every step of the attention runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  If the
library has not been built, or its kernels cannot run on this device, the
calls raise; there is no other implementation to fall back to.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libneattn.so")

NE_OK = 0
O_FP32 = 1       # flag bits, see include/ne_attn.h
GRAD_FP32 = 2
PRECISE_QK = 4
QK_ROTATED = 8
ROPE_HALF = 16
FP8 = 32
_lib = None


class NeAttnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = lib().ne_attn_status_string(status).decode() if _lib is not None else str(status)
        super().__init__("%s failed with status %d: %s" % (fn, status, msg))


def lib():
    """Loads the in-tree CUDA library (built by __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libneattn.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.ne_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        L.ne_attn_fwd.restype = i
        L.ne_attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
        L.ne_attn_fwd_ex.restype = i
        L.ne_attn_fwd_workspace_size.argtypes = [i, i, i, i, i, i]
        L.ne_attn_fwd_workspace_size.restype = sz
        L.ne_attn_bwd_workspace_size.argtypes = [i, i, i, i, i, i]
        L.ne_attn_bwd_workspace_size.restype = sz
        L.ne_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
        L.ne_attn_bwd.restype = i
        L.ne_attn_check_status.argtypes = [vp]
        L.ne_attn_check_status.restype = i
        L.ne_attn_status_string.argtypes = [i]
        L.ne_attn_status_string.restype = ctypes.c_char_p
        L.ne_attn_debug_timeout_probe.argtypes = [i, vp]
        L.ne_attn_debug_timeout_probe.restype = i
        L.ne_attn_profile_start.argtypes = [i]
        L.ne_attn_profile_start.restype = i
        L.ne_attn_profile_stop.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong)]
        L.ne_attn_profile_stop.restype = i
        L.ne_attn_profile_detach.argtypes = []
        L.ne_attn_profile_detach.restype = i
        L.ne_attn_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong)]
        L.ne_attn_profile_read.restype = i
        L.ne_attn_kv_append.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        L.ne_attn_kv_append.restype = i
        L.ne_attn_decode_workspace_size.argtypes = [i, i, i, i, i, i]
        L.ne_attn_decode_workspace_size.restype = sz
        L.ne_attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, sz, vp]
        L.ne_attn_decode.restype = i
        ip = ctypes.POINTER(ctypes.c_int)
        L.ne_attn_debug_fwd_schedule.argtypes = [i, i, i, i, i, ip, i, ip, ip]
        L.ne_attn_debug_fwd_schedule.restype = i
        L.ne_attn_qkv_workspace_size.argtypes = [i, i, i, i, i, i, i]
        L.ne_attn_qkv_workspace_size.restype = sz
        L.ne_attn_qkv_rmsnorm.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, i, vp, sz, vp]
        L.ne_attn_qkv_rmsnorm.restype = i
        _lib = L
    return _lib


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, st):
    if st != NE_OK:
        raise NeAttnError(fn, st)


def _ptr(t):
    return ctypes.c_void_p(None if t is None else t.data_ptr())


def _shape(q, k):
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    return B, T, Hq, Hkv, D


def fwd_workspace_size(B, T, Hq, Hkv, D, precise=False, fp8=False):
    flags = (PRECISE_QK if precise else 0) | (FP8 if fp8 else 0)
    return int(lib().ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, flags))


def attn_fwd(q, k, v, rope_base=10000.0, o=None, lse=None, o_dtype=torch.bfloat16, precise=False,
             workspace=None, rope_half=False, qk_rotated=False, Hq=None, fp8=False, stream=None):
    """o, lse = causal GQA attention of q [B,T,Hq,D], k/v [B,T,Hkv,D] (bf16, CUDA).

    o_dtype: bfloat16 or float32.  precise: hi+lo split of the rotated q, k
    for the logits (NE_ATTN_PRECISE_QK).  workspace: a uint8 CUDA tensor of at
    least fwd_workspace_size bytes (the rotated fp16 q, k land there); if None
    one is allocated for the call.  qk_rotated: `workspace` already holds the
    rotated q and k (written by qkv_rmsnorm with rotated=True); q and k may
    then be None, with the number of query heads given as Hq.  fp8: the
    e4m3 forward (NE_ATTN_FP8; D = 64, about 3e-2 relative error in o).
    """
    if qk_rotated and workspace is None:
        raise ValueError("qk_rotated needs the workspace that holds the rotated q and k")
    if q is None:
        if not qk_rotated or Hq is None:
            raise ValueError("q may be None only with qk_rotated and Hq")
        B, T, Hkv, D = v.shape
    else:
        B, T, Hq, Hkv, D = _shape(q, k)
    if o is None:
        o = torch.empty((B, T, Hq, D), dtype=o_dtype, device=v.device)
    if lse is None:
        # precise mode stores the LSE and its fp32 remainder: lse[0] is the LSE
        shape = (2, B, Hq, T) if precise else (B, Hq, T)
        lse = torch.empty(shape, dtype=torch.float32, device=v.device)
    assert lse.numel() == (2 if precise else 1) * B * Hq * T and o.shape == (B, T, Hq, D)
    for t in (q, k, v):
        assert t is None or (t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous())
    assert o.dtype in (torch.bfloat16, torch.float32) and o.is_contiguous()
    assert lse.dtype == torch.float32 and lse.is_contiguous()
    flags = ((O_FP32 if o.dtype == torch.float32 else 0) | (PRECISE_QK if precise else 0)
             | (ROPE_HALF if rope_half else 0) | (QK_ROTATED if qk_rotated else 0) | (FP8 if fp8 else 0))
    if workspace is None:
        n = fwd_workspace_size(B, T, Hq, Hkv, D, precise, fp8)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=v.device)
    assert workspace.dtype == torch.uint8 and workspace.is_cuda
    _check("ne_attn_fwd_ex", lib().ne_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                                  B, T, Hq, Hkv, D, float(rope_base), flags,
                                                  _ptr(workspace), workspace.numel(), _stream(stream)))
    return o, lse


def bwd_workspace_size(B, T, Hq, Hkv, D, precise=False):
    return int(lib().ne_attn_bwd_workspace_size(B, T, Hq, Hkv, D, PRECISE_QK if precise else 0))


def alloc_workspace(B, T, Hq, Hkv, D, precise=False, device="cuda"):
    n = bwd_workspace_size(B, T, Hq, Hkv, D, precise)
    if n == 0:
        raise ValueError("unsupported shape")
    return torch.empty(n, dtype=torch.uint8, device=device)


def attn_bwd(q, k, v, o, lse, dout, rope_base=10000.0, grad_dtype=torch.bfloat16, precise=False,
             dq=None, dk=None, dv=None, workspace=None, qk_rotated=False, rope_half=False, stream=None):
    """dq, dk, dv of the causal GQA attention given the forward's o and lse.

    o may be bfloat16 or float32; grad_dtype selects the gradient dtype.
    qk_rotated: `workspace` was also the forward's workspace (for these q, k)
    and still holds its rotated q and k (NE_ATTN_QK_ROTATED).
    """
    if qk_rotated and workspace is None:
        raise ValueError("qk_rotated needs the workspace the forward wrote")
    if (q is None or k is None) and not qk_rotated:
        raise ValueError("q and k may be None only with qk_rotated")
    B, T, Hq, D = dout.shape
    Hkv = v.shape[2]
    if grad_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("grad_dtype must be bfloat16 or float32")
    if dq is None:
        dq = torch.empty(dout.shape, dtype=grad_dtype, device=v.device)
    if dk is None:
        dk = torch.empty(v.shape, dtype=grad_dtype, device=v.device)
    if dv is None:
        dv = torch.empty(v.shape, dtype=grad_dtype, device=v.device)
    if workspace is None:
        workspace = alloc_workspace(B, T, Hq, Hkv, D, precise, v.device)
    for t in (q, k, v, dout):
        assert t is None or (t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous())
    assert o.dtype in (torch.bfloat16, torch.float32) and o.is_contiguous()
    assert lse.dtype == torch.float32 and lse.numel() == (2 if precise else 1) * B * Hq * T
    for t in (dq, dk, dv):
        assert t.dtype == grad_dtype and t.is_contiguous()
    flags = ((O_FP32 if o.dtype == torch.float32 else 0) | (GRAD_FP32 if grad_dtype == torch.float32 else 0)
             | (PRECISE_QK if precise else 0) | (QK_ROTATED if qk_rotated else 0) | (ROPE_HALF if rope_half else 0))
    _check("ne_attn_bwd", lib().ne_attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
        B, T, Hq, Hkv, D, float(rope_base), flags, _ptr(workspace), workspace.numel(), _stream(stream)))
    return dq, dk, dv


def check_status(stream=None):
    """Synchronises the stream; raises if a kernel reported a device-side timeout."""
    _check("ne_attn_check_status", lib().ne_attn_check_status(_stream(stream)))


def status_of_last_kernels(stream=None):
    """Like check_status but returns the raw status code (and clears it)."""
    return int(lib().ne_attn_check_status(_stream(stream)))


KERNEL_KINDS = ("fwd", "bwd_prep", "bwd_dkdv", "bwd_dq", "fwd_rope", "kv_append", "decode", "decode_aux",
                "qkv_prep", "qkv")


def profile_start(capacity):
    """Brackets each library kernel launch with CUDA events (see ne_attn_profile_start)."""
    _check("ne_attn_profile_start", lib().ne_attn_profile_start(int(capacity)))


def profile_stop():
    """Returns {kernel kind: (total device ms, launches)} for the launches since profile_start."""
    ms = (ctypes.c_double * len(KERNEL_KINDS))()
    n = (ctypes.c_longlong * len(KERNEL_KINDS))()
    _check("ne_attn_profile_stop", lib().ne_attn_profile_stop(ms, n))
    return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(KERNEL_KINDS)}


def profile_stop_deferred():
    """Closes a profile whose launches were captured into a CUDA graph: the
    events run (and are timed) each time the graph replays.  Returns a handle
    for profile_read, which reads the times of the most recent replay."""
    _check("ne_attn_profile_detach", lib().ne_attn_profile_detach())
    return True


def profile_read(handle):
    ms = (ctypes.c_double * len(KERNEL_KINDS))()
    n = (ctypes.c_longlong * len(KERNEL_KINDS))()
    _check("ne_attn_profile_read", lib().ne_attn_profile_read(ms, n))
    return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(KERNEL_KINDS)}


def debug_timeout_probe(limit_us, stream=None):
    _check("ne_attn_debug_timeout_probe", lib().ne_attn_debug_timeout_probe(int(limit_us), _stream(stream)))


def fwd_bwd_host(q, k, v, dout, rope_base=10000.0, grad_dtype=torch.bfloat16, o_dtype=torch.bfloat16,
                 precise=False, device="cuda", stream=None):
    """End-to-end call on host (CPU) bfloat16 tensors: copies in, forward +
    backward, copies out.  Pinned host memory makes the copies asynchronous.
    Returns host tensors (o, lse, dq, dk, dv).
    """
    s = torch.cuda.current_stream() if stream is None else stream
    with torch.cuda.stream(s):
        qd = q.to(device, non_blocking=True)
        kd = k.to(device, non_blocking=True)
        vd = v.to(device, non_blocking=True)
        dod = dout.to(device, non_blocking=True)
        ws = alloc_workspace(*_shape(qd, kd), precise=precise, device=device)
        o, lse = attn_fwd(qd, kd, vd, rope_base, o_dtype=o_dtype, precise=precise, workspace=ws, stream=s)
        dq, dk, dv = attn_bwd(qd, kd, vd, o, lse, dod, rope_base, grad_dtype, precise=precise, workspace=ws,
                              qk_rotated=not precise, stream=s)
        out = [t.to("cpu", non_blocking=False) for t in (o, lse, dq, dk, dv)]
    return tuple(out)


def kv_cache(B, Tcap, Hkv, D, device):
    """Empty head-major key (fp16, rotated) and value (bf16) caches [B, Hkv, Tcap, D]."""
    return (torch.zeros((B, Hkv, Tcap, D), dtype=torch.float16, device=device),
            torch.zeros((B, Hkv, Tcap, D), dtype=torch.bfloat16, device=device))


def kv_append(k_new, v_new, k_cache, v_cache, pos0, rope_base=10000.0, rope_half=False, stream=None):
    """Writes positions pos0 .. pos0 + Tn - 1 of the caches from k_new, v_new [B,Tn,Hkv,D] (bf16)."""
    B, Tn, Hkv, D = k_new.shape
    Tcap = k_cache.shape[2]
    for t in (k_new, v_new):
        assert t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous()
    assert k_cache.dtype == torch.float16 and v_cache.dtype == torch.bfloat16
    assert k_cache.is_contiguous() and v_cache.is_contiguous() and k_cache.shape == v_cache.shape
    _check("ne_attn_kv_append", lib().ne_attn_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                                        B, Tn, pos0, Tcap, Hkv, D, float(rope_base),
                                                        ROPE_HALF if rope_half else 0, _stream(stream)))


def decode_workspace_size(B, Tq, Tkv, Hq, Hkv, D):
    return int(lib().ne_attn_decode_workspace_size(B, Tq, Tkv, Hq, Hkv, D))


def attn_decode(q, k_cache, v_cache, Tkv, rope_base=10000.0, o=None, lse=None, o_dtype=torch.bfloat16,
                workspace=None, rope_half=False, stream=None):
    """o, lse for the Tq new queries q [B,Tq,Hq,D] (bf16, positions Tkv-Tq .. Tkv-1)
    against cache positions 0 .. Tkv-1 (see ne_attn_decode)."""
    B, Tq, Hq, D = q.shape
    Hkv, Tcap = k_cache.shape[1], k_cache.shape[2]
    assert q.dtype == torch.bfloat16 and q.is_cuda and q.is_contiguous()
    assert k_cache.dtype == torch.float16 and v_cache.dtype == torch.bfloat16
    if o is None:
        o = torch.empty(q.shape, dtype=o_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
    assert o.dtype in (torch.bfloat16, torch.float32) and o.is_contiguous()
    assert lse.dtype == torch.float32 and lse.is_contiguous() and lse.numel() == B * Hq * Tq
    if workspace is None:
        workspace = torch.empty(max(decode_workspace_size(B, Tq, Tkv, Hq, Hkv, D), 1), dtype=torch.uint8,
                                device=q.device)
    flags = (O_FP32 if o.dtype == torch.float32 else 0) | (ROPE_HALF if rope_half else 0)
    _check("ne_attn_decode", lib().ne_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse),
                                                  B, Tq, Tkv, Tcap, Hq, Hkv, D, float(rope_base), flags,
                                                  _ptr(workspace), workspace.numel(), _stream(stream)))
    return o, lse


def qkv_workspace_size(B, T, C, Hq, Hkv, D, rotated=False, rope_half=False):
    flags = (QK_ROTATED if rotated else 0) | (ROPE_HALF if rope_half else 0)
    return int(lib().ne_attn_qkv_workspace_size(B, T, C, Hq, Hkv, D, flags))


def qkv_rmsnorm(x, norm_w, w_qkv, Hq, Hkv, D, eps=1e-5, rope_base=10000.0, rotated=False, rope_half=False,
                write_qk=True, q=None, k=None, v=None, rstd=None, workspace=None, stream=None):
    """RMSNorm of x [B,T,C] and the fused projection w_qkv [(Hq+2Hkv)D, C] (bf16, CUDA).

    Returns (q, k, v, rstd, workspace): q [B,T,Hq,D], k and v [B,T,Hkv,D]
    (bf16; q and k are None when write_qk is False), rstd [B,T] fp32.
    rotated: also write the rotated q, k (fp16) at the start of `workspace`
    (allocated here if None; at least qkv_workspace_size bytes), where
    attn_fwd / attn_bwd with qk_rotated=True take them.
    """
    B, T, C = x.shape
    N = (Hq + 2 * Hkv) * D
    assert norm_w.shape == (C,) and w_qkv.shape == (N, C)
    for t in (x, norm_w, w_qkv):
        assert t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous()
    if not write_qk and not rotated:
        raise ValueError("write_qk=False needs rotated=True")
    dev = x.device
    if write_qk:
        q = torch.empty((B, T, Hq, D), dtype=torch.bfloat16, device=dev) if q is None else q
        k = torch.empty((B, T, Hkv, D), dtype=torch.bfloat16, device=dev) if k is None else k
    else:
        q = k = None
    v = torch.empty((B, T, Hkv, D), dtype=torch.bfloat16, device=dev) if v is None else v
    rstd = torch.empty((B, T), dtype=torch.float32, device=dev) if rstd is None else rstd
    for t in (q, k, v):
        assert t is None or (t.dtype == torch.bfloat16 and t.is_contiguous())
    assert rstd.dtype == torch.float32 and rstd.numel() == B * T
    if workspace is None:
        n = qkv_workspace_size(B, T, C, Hq, Hkv, D, rotated, rope_half)
        if n == 0:
            raise ValueError("unsupported shape")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    flags = (QK_ROTATED if rotated else 0) | (ROPE_HALF if rope_half else 0)
    _check("ne_attn_qkv_rmsnorm", lib().ne_attn_qkv_rmsnorm(
        _ptr(x), _ptr(norm_w), _ptr(w_qkv), _ptr(q), _ptr(k), _ptr(v), _ptr(rstd), B, T, C, Hq, Hkv, D,
        float(eps), float(rope_base), flags, _ptr(workspace), workspace.numel(), _stream(stream)))
    return q, k, v, rstd, workspace


def rotated_qk(workspace, B, T, Hq, Hkv, D):
    """Views of the rotated fp16 q [B,T,Hq,D] and k [B,T,Hkv,D] at the start of a
    forward / backward / projection workspace (NE_ATTN_QK_ROTATED layout)."""
    def up(n):
        return (n + 255) // 256 * 256
    nq, nk = 2 * B * T * Hq * D, 2 * B * T * Hkv * D
    qr = workspace[:nq].view(torch.float16).view(B, T, Hq, D)
    kr = workspace[up(nq):up(nq) + nk].view(torch.float16).view(B, T, Hkv, D)
    return qr, kr


class HostStepPipeline:
    """Forward + backward steps on host tensors, with the copies of one step
    overlapping the compute of the others.

    Inputs go up on one stream, the library's kernels run on a second, results
    come down on a third; `depth` device buffer sets rotate, and CUDA events
    order each set's reuse (a set is refilled only after its previous results
    have come down).  Host tensors should be pinned so the copies run
    asynchronously.  submit() only enqueues work; synchronize() waits for all
    of it and raises if a kernel reported a device-side timeout.  precise:
    split precision (NE_ATTN_PRECISE_QK) with an fp32 o, for inputs with very
    large logits; lse then holds the LSE and its remainder ([2 B, Hq, T]).
    """

    def __init__(self, B, T, Hq, Hkv, D, rope_base=10000.0, depth=3, grad_dtype=torch.float32,
                 o_dtype=torch.bfloat16, device="cuda", precise=False):
        self.shape = (B, T, Hq, Hkv, D)
        self.rope_base = float(rope_base)
        self.grad_dtype = grad_dtype
        self.precise = bool(precise)
        if self.precise:
            o_dtype = torch.float32
        self.device = torch.device(device)
        self.up = torch.cuda.Stream(self.device)
        self.comp = torch.cuda.Stream(self.device)
        self.down = torch.cuda.Stream(self.device)
        self.sets = []
        for _ in range(depth):
            def bf(h):
                return torch.empty((B, T, h, D), dtype=torch.bfloat16, device=self.device)
            self.sets.append(dict(
                q=bf(Hq), k=bf(Hkv), v=bf(Hkv), do=bf(Hq),
                o=torch.empty((B, T, Hq, D), dtype=o_dtype, device=self.device),
                lse=torch.empty(((2 if self.precise else 1) * B, Hq, T), dtype=torch.float32, device=self.device),
                dq=torch.empty((B, T, Hq, D), dtype=grad_dtype, device=self.device),
                dk=torch.empty((B, T, Hkv, D), dtype=grad_dtype, device=self.device),
                dv=torch.empty((B, T, Hkv, D), dtype=grad_dtype, device=self.device),
                ws=alloc_workspace(B, T, Hq, Hkv, D, precise=self.precise, device=self.device),
                up_done=torch.cuda.Event(), comp_done=torch.cuda.Event(), down_done=torch.cuda.Event(),
                used=False))
        self.n = 0

    def submit(self, q, k, v, dout, out):
        """Enqueue one step: q, k, v, dout are host bf16 tensors; `out` maps
        o, lse, dq, dk, dv to host tensors that receive the results."""
        s = self.sets[self.n % len(self.sets)]
        self.n += 1
        if s["used"]:
            self.up.wait_event(s["down_done"])  # the set's last results have come down
        with torch.cuda.stream(self.up):
            for name, src in (("q", q), ("k", k), ("v", v), ("do", dout)):
                s[name].copy_(src, non_blocking=True)
            s["up_done"].record(self.up)
        self.comp.wait_event(s["up_done"])
        attn_fwd(s["q"], s["k"], s["v"], self.rope_base, o=s["o"], lse=s["lse"], workspace=s["ws"],
                 o_dtype=s["o"].dtype, precise=self.precise, stream=self.comp)
        attn_bwd(s["q"], s["k"], s["v"], s["o"], s["lse"], s["do"], self.rope_base, grad_dtype=self.grad_dtype,
                 dq=s["dq"], dk=s["dk"], dv=s["dv"], workspace=s["ws"], qk_rotated=not self.precise,
                 precise=self.precise, stream=self.comp)
        s["comp_done"].record(self.comp)
        self.down.wait_event(s["comp_done"])
        with torch.cuda.stream(self.down):
            for name in ("o", "lse", "dq", "dk", "dv"):
                out[name].copy_(s[name], non_blocking=True)
            s["down_done"].record(self.down)
        s["used"] = True

    def synchronize(self):
        self.down.synchronize()
        check_status(self.comp)


def fwd_schedule(B, Hkv, G, nt, nsm):
    """The persistent forward's work items per CTA (host computation, no GPU):
    a list of `grid` lists of items (b, (h0, i0), (h1, i1) or None), each CTA's
    items in the order it runs them."""
    k, grid = ctypes.c_int(0), ctypes.c_int(0)
    lib().ne_attn_debug_fwd_schedule(B, Hkv, G, nt, nsm, None, 0, ctypes.byref(grid), ctypes.byref(k))
    n = max(1, 4 * grid.value * k.value)
    buf = (ctypes.c_int * n)()
    _check("ne_attn_debug_fwd_schedule",
           lib().ne_attn_debug_fwd_schedule(B, Hkv, G, nt, nsm, buf, n, ctypes.byref(grid), ctypes.byref(k)))
    out = []
    for c in range(grid.value):
        row = []
        for j in range(k.value):
            b, hh, i0, i1 = buf[4 * (c * k.value + j):4 * (c * k.value + j) + 4]
            if b < 0:
                continue
            h0, h1 = hh & 0xFFFF, (hh >> 16) - 1
            row.append((b, (h0, i0), (h1, i1) if h1 >= 0 else None))
        out.append(row)
    return out
