"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports
every entry point include/ne_attn.h declares, and rejects bad arguments on
the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libne():
    from causal_gqa_attention_flashattention_gb300 import build, binding
    build.build()
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ne_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ne_attn_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(libne):
    names = declared_functions()
    assert "ne_attn_fwd" in names and "ne_attn_bwd" in names
    for n in names:
        assert hasattr(libne, n), n


def test_workspace_size(libne):
    B, T, Hq, Hkv, D = 16, 512, 12, 4, 64
    n = libne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, D, 0)
    expect = 4 * B * Hq * T * D + 2 * B * T * (Hq + Hkv) * D + 2 * 4 * B * Hq * T
    assert expect <= n <= expect + 5 * 256
    n_precise = libne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, D, 4)
    assert n_precise - n >= 2 * B * T * (Hq + Hkv) * D  # fp16 remainders of rotated q and k
    assert libne.ne_attn_bwd_workspace_size(1, 77, 4, 2, 32, 0) >= 4 * 4 * 128 * 32  # padded to 128 rows
    assert libne.ne_attn_bwd_workspace_size(1, 16, 3, 2, 64, 0) == 0
    assert libne.ne_attn_bwd_workspace_size(1, 16, 2, 1, 48, 0) == 0
    assert libne.ne_attn_bwd_workspace_size(1, 16, 2, 1, 64, 32) == 0  # unknown flag
    assert libne.ne_attn_bwd_workspace_size(1, 16, 2, 1, 64, 8) == libne.ne_attn_bwd_workspace_size(1, 16, 2, 1, 64, 0)
    assert libne.ne_attn_bwd_workspace_size(1, 16, 2, 1, 64, 8 | 4) == 0  # reuse needs default precision


def test_fwd_workspace_size(libne):
    B, T, Hq, Hkv, D = 16, 512, 12, 4, 64
    n = libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 0)
    assert n == 2 * B * T * (Hq + Hkv) * D  # rotated fp16 q and k (both already 256-byte multiples)
    assert libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 1) == n  # fp32 o changes nothing
    assert libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 4) == 0  # precise kernel rotates in shared memory
    assert libne.ne_attn_fwd_workspace_size(1, 3, 1, 1, 32, 0) == 2 * 256  # each array rounded to 256 bytes
    assert libne.ne_attn_fwd_workspace_size(1, 16, 2, 1, 64, 2) == 0  # gradient flag is not a forward flag
    # the backward's workspace starts with the same two arrays
    assert libne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, D, 0) >= n + 4 * B * Hq * T * D


def test_host_argument_checks(libne):
    buf = ctypes.create_string_buffer(4096 + 64)
    base = (ctypes.addressof(buf) + 63) // 64 * 64
    p = ctypes.c_void_p(base)
    mis = ctypes.c_void_p(base + 2)
    null = None
    assert libne.ne_attn_fwd(null, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, null) == -1
    assert libne.ne_attn_fwd(p, p, p, p, p, 1, 16, 3, 2, 64, 10000.0, null) == -1
    assert libne.ne_attn_fwd(p, p, p, p, p, 1, 0, 2, 1, 64, 10000.0, null) == -1
    assert libne.ne_attn_fwd(p, p, p, p, p, 1, 16, 2, 1, 48, 10000.0, null) == -3
    assert libne.ne_attn_fwd(p, p, p, p, p, 1, 16, 2, 1, 64, 0.5, null) == -1
    assert libne.ne_attn_fwd(mis, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, null) == -2
    assert libne.ne_attn_fwd_ex(p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 2, null, 0, null) == -1  # grad flag on fwd
    assert libne.ne_attn_fwd_ex(p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 0, p, 16, null) == -5  # workspace too small
    assert libne.ne_attn_fwd_ex(p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 0, mis, 1 << 20, null) == -5  # misaligned
    assert libne.ne_attn_bwd(p, p, p, p, p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 32, p, 4096, null) == -1  # unknown flag
    assert libne.ne_attn_bwd(p, p, p, p, p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 8 | 4, p, 1 << 20, null) == -1
    assert libne.ne_attn_bwd(p, p, p, p, p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 0, p, 16, null) == -5
    assert libne.ne_attn_bwd(p, p, p, p, p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 0, mis, 1 << 20, null) == -5
    assert libne.ne_attn_debug_timeout_probe(0, null) == -1
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert libne.ne_attn_status_string(code)


def test_decode_workspace_size(libne):
    B, Tq, Tkv, Hq, Hkv, D = 2, 3, 1000, 12, 4, 64
    n = libne.ne_attn_decode_workspace_size(B, Tq, Tkv, Hq, Hkv, D)
    R, ntk = (Hq // Hkv) * Tq, (Tkv + 127) // 128
    # packed queries [B,Hkv,128,D] fp16 + per split: O (fp32 R x D) and (max, sum)
    assert n >= B * Hkv * 128 * D * 2 + B * Hkv * ntk * R * (D * 4 + 8)
    assert n % 256 == 0
    assert libne.ne_attn_decode_workspace_size(1, 129, 129, 1, 1, 64) == 0  # 129 query rows > one tile
    assert libne.ne_attn_decode_workspace_size(1, 3, 2, 4, 2, 64) == 0      # Tq > Tkv
    assert libne.ne_attn_decode_workspace_size(1, 1, 10, 3, 2, 64) == 0     # Hq % Hkv
    assert libne.ne_attn_decode_workspace_size(1, 1, 10, 4, 2, 48) == 0     # D


def test_decode_host_argument_checks(libne):
    buf = ctypes.create_string_buffer(4096 + 512)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)
    mis = ctypes.c_void_p(base + 2)
    null = None
    # ne_attn_kv_append(k_new, v_new, k_cache, v_cache, B, Tn, pos0, Tcap, Hkv, D, base, flags, stream)
    assert libne.ne_attn_kv_append(null, p, p, p, 1, 4, 0, 8, 2, 64, 10000.0, 0, null) == -1
    assert libne.ne_attn_kv_append(p, p, p, p, 1, 4, 5, 8, 2, 64, 10000.0, 0, null) == -1   # past the capacity
    assert libne.ne_attn_kv_append(p, p, p, p, 1, 0, 0, 8, 2, 64, 10000.0, 0, null) == -1   # nothing to append
    assert libne.ne_attn_kv_append(p, p, p, p, 1, 4, -1, 8, 2, 64, 10000.0, 0, null) == -1
    assert libne.ne_attn_kv_append(p, p, mis, p, 1, 4, 0, 8, 2, 64, 10000.0, 0, null) == -2
    assert libne.ne_attn_kv_append(p, p, p, p, 1, 4, 0, 8, 2, 48, 10000.0, 0, null) == -3
    # ne_attn_decode(q, kc, vc, o, lse, B, Tq, Tkv, Tcap, Hq, Hkv, D, base, flags, ws, ws_bytes, stream)
    ok = (1, 1, 10, 16, 4, 2, 64, 10000.0)
    assert libne.ne_attn_decode(p, p, p, p, p, *ok, 0, p, 4096, null) == -5  # workspace too small
    assert libne.ne_attn_decode(p, p, p, p, p, *ok, 0, null, 1 << 20, null) == -5  # workspace required
    assert libne.ne_attn_decode(p, p, p, p, p, *ok, 0, mis, 1 << 20, null) == -5  # misaligned workspace
    assert libne.ne_attn_decode(p, p, p, p, p, *ok, 2, p, 1 << 20, null) == -1  # gradient flag
    assert libne.ne_attn_decode(null, p, p, p, p, *ok, 0, p, 1 << 20, null) == -1
    assert libne.ne_attn_decode(p, p, p, p, p, 1, 11, 10, 16, 4, 2, 64, 10000.0, 0, p, 1 << 20, null) == -1  # Tq > Tkv
    assert libne.ne_attn_decode(p, p, p, p, p, 1, 1, 10, 9, 4, 2, 64, 10000.0, 0, p, 1 << 20, null) == -1  # Tkv > Tcap
    assert libne.ne_attn_decode(p, p, p, p, p, 1, 65, 100, 100, 4, 2, 64, 10000.0, 0, p, 1 << 20, null) == -3  # 130 rows
    assert libne.ne_attn_decode(p, p, p, mis, p, *ok, 0, p, 1 << 20, null) == -2
    assert libne.ne_attn_kv_append(p, p, p, p, 1, 4, 0, 8, 2, 64, 10000.0, 1, null) == -1  # only the layout flag
    assert libne.ne_attn_decode(p, p, p, p, p, *ok, 16, p, 4096, null) == -5  # layout flag accepted (then workspace)


def test_half_split_flag_rules(libne):
    buf = ctypes.create_string_buffer(4096 + 512)
    p = ctypes.c_void_p((ctypes.addressof(buf) + 255) // 256 * 256)
    null = None
    B, T, Hq, Hkv, D = 2, 200, 4, 2, 64
    assert libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 16) == libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 0)
    assert libne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, D, 16) == libne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, D, 0)
    assert libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 16 | 4) == 0  # not with split precision
    assert libne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, D, 16 | 4) == 0
    assert libne.ne_attn_fwd_ex(p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 16 | 4, null, 0, null) == -3
    assert libne.ne_attn_bwd(p, p, p, p, p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 16 | 4, p, 1 << 20, null) == -3
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    libne.ne_attn_bwd_noalloc.argtypes = [vp] * 9 + [i] * 5 + [f, i, vp]
    libne.ne_attn_bwd_noalloc.restype = i
    assert libne.ne_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 16 | 4, null) == -3
    # the fixed scratch never holds a forward's rotated q, k: the reuse flag is refused
    assert libne.ne_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 8, null) == -1



def test_qkv_workspace_size(libne):
    B, T, C, Hq, Hkv, D = 16, 512, 768, 12, 4, 64
    N = (Hq + 2 * Hkv) * D
    n = libne.ne_attn_qkv_workspace_size(B, T, C, Hq, Hkv, D, 0)
    assert n == N * C * 2  # the folded projection matrix (already a 256-byte multiple)
    fwd = libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 0)
    assert libne.ne_attn_qkv_workspace_size(B, T, C, Hq, Hkv, D, 8) == fwd + n  # rotated q, k first
    assert libne.ne_attn_qkv_workspace_size(B, T, C, Hq, Hkv, D, 8 | 16) == fwd + n
    assert libne.ne_attn_qkv_workspace_size(B, T, 100, Hq, Hkv, D, 0) == 0  # rows must be 16-byte multiples
    assert libne.ne_attn_qkv_workspace_size(B, T, C, Hq, Hkv, D, 1) == 0  # output-dtype flag is not accepted
    assert libne.ne_attn_qkv_workspace_size(B, T, C, 12, 5, D, 0) == 0  # Hq % Hkv
    # the forward accepts the reuse flag now (it changes nothing in the size)
    assert libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 8) == fwd
    assert libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 8 | 4) == 0


def test_qkv_host_argument_checks(libne):
    buf = ctypes.create_string_buffer(4096 + 512)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)
    mis = ctypes.c_void_p(base + 2)
    null = None
    ok = (1, 4, 64, 4, 2, 32)  # B, T, C, Hq, Hkv, D
    # ne_attn_qkv_rmsnorm(x, norm_w, w_qkv, q, k, v, rstd, B, T, C, Hq, Hkv, D, eps, base, flags, ws, bytes, stream)
    f = libne.ne_attn_qkv_rmsnorm
    assert f(null, p, p, p, p, p, p, *ok, 1e-5, 10000.0, 0, p, 1 << 20, null) == -1
    assert f(p, p, p, p, p, p, null, *ok, 1e-5, 10000.0, 0, p, 1 << 20, null) == -1  # rstd is an output
    assert f(p, p, p, null, p, p, p, *ok, 1e-5, 10000.0, 0, p, 1 << 20, null) == -1  # q needed without the flag
    assert f(p, p, p, p, p, p, p, *ok, 0.0, 10000.0, 0, p, 1 << 20, null) == -1      # eps > 0
    assert f(p, p, p, p, p, p, p, *ok, 1e-5, 1.0, 0, p, 1 << 20, null) == -1         # rope base
    assert f(p, p, p, p, p, p, p, *ok, 1e-5, 10000.0, 4, p, 1 << 20, null) == -1     # precise flag
    assert f(p, p, p, p, p, p, p, 1, 4, 60, 4, 2, 32, 1e-5, 10000.0, 0, p, 1 << 20, null) == -1  # C % 8
    assert f(p, p, p, p, p, p, p, 1, 4, 64, 4, 2, 48, 1e-5, 10000.0, 0, p, 1 << 20, null) == -3  # D
    assert f(p, mis, p, p, p, p, p, *ok, 1e-5, 10000.0, 0, p, 1 << 20, null) == -2
    assert f(p, p, p, p, p, p, p, *ok, 1e-5, 10000.0, 8, null, 0, null) == -5  # rotated q, k need a workspace
    assert f(p, p, p, null, null, p, p, *ok, 1e-5, 10000.0, 8, p, 64, null) == -5  # too small (q, k optional)
    assert f(p, p, p, p, p, p, p, *ok, 1e-5, 10000.0, 0, mis, 1 << 20, null) == -5
    # forward and backward: q, k may be NULL only with the reuse flag, which needs the workspace
    # ne_attn_fwd_ex(q, k, v, o, lse, B, T, Hq, Hkv, D, base, flags, ws, bytes, stream)
    fx = libne.ne_attn_fwd_ex
    assert fx(null, null, p, p, p, 1, 4, 4, 2, 32, 10000.0, 0, p, 1 << 20, null) == -1
    assert fx(null, null, p, p, p, 1, 4, 4, 2, 32, 10000.0, 8, null, 0, null) == -5
    assert fx(null, null, p, p, p, 1, 4, 4, 2, 32, 10000.0, 8 | 4, p, 1 << 20, null) == -1
    # ne_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, T, Hq, Hkv, D, base, flags, ws, bytes, stream)
    bx = libne.ne_attn_bwd
    assert bx(null, null, p, p, p, p, p, p, p, 1, 4, 4, 2, 32, 10000.0, 0, p, 1 << 20, null) == -1
    assert bx(null, null, p, p, p, p, p, p, p, 1, 4, 4, 2, 32, 10000.0, 8, p, 64, null) == -5


def test_fp8_flag_rules_on_the_host(libne):
    B, T, Hq, Hkv, D = 16, 512, 12, 4, 64
    n8 = libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 32)
    assert n8 == B * T * (Hq + Hkv) * D + 256  # e4m3 q and k, then the per-head maxima
    assert libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 32 | 16) == n8  # either rotary layout
    assert libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, 32, 32) == 0       # D = 64 only
    assert libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 32 | 4) == 0    # not with precise logits
    assert libne.ne_attn_fwd_workspace_size(B, T, Hq, Hkv, D, 32 | 8) == 0    # the library rotates
    assert libne.ne_attn_fwd_workspace_size(1, 16, 256, 1, D, 32) == 0        # at most 256 heads in all
    assert libne.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, D, 32) == 0        # forward only
    buf = ctypes.create_string_buffer(4096 + 512)
    p = ctypes.c_void_p((ctypes.addressof(buf) + 255) // 256 * 256)
    null = None
    fx = libne.ne_attn_fwd_ex
    assert fx(p, p, p, p, p, 1, 16, 2, 1, 32, 10000.0, 32, null, 0, null) == -3
    assert fx(p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 32 | 4, null, 0, null) == -1
    assert fx(p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 32, p, 64, null) == -5  # workspace too small
    assert fx(p, p, p, p, p, 1, 16, 2, 1, 64, 10000.0, 64, null, 0, null) == -1  # unknown flag


@pytest.mark.parametrize("B,Hkv,G,nt,nsm", [(16, 4, 3, 4, 152), (8, 4, 4, 8, 152), (2, 4, 3, 64, 152),
                                             (8, 2, 2, 4, 152), (1, 1, 8, 3, 152), (3, 2, 5, 5, 10),
                                             (1, 1, 1, 1, 152), (2, 3, 1, 7, 4)])
def test_forward_schedule(libne, B, Hkv, G, nt, nsm):
    """The forward's work table (host logic): every (batch, head, query tile)
    unit exactly once; the two units of an item share batch and key/value head
    and their first unit has the larger tile; head pairs sit at one tile and
    tile pairs of one head are adjacent; each CTA's items longest first; and
    the busiest CTA within one item of the average."""
    from causal_gqa_attention_flashattention_gb300 import binding
    lists = binding.fwd_schedule(B, Hkv, G, nt, nsm)
    units = []
    cost = lambda it: 2 * (it[1][1] + 1) + 1 + (2 * (it[2][1] + 1) + 1 if it[2] else 0)
    for l in lists:
        for b, u0, u1 in l:
            units.append((b, u0[0], u0[1]))
            if u1 is not None:
                units.append((b, u1[0], u1[1]))
                assert u0[0] // G == u1[0] // G and u0[1] >= u1[1]
                assert (u0[1] == u1[1] and u1[0] == u0[0] + 1) or (u0[0] == u1[0] and u1[1] == u0[1] - 1)
        assert [cost(it) for it in l] == sorted((cost(it) for it in l), reverse=True)
    want = sorted((b, h, i) for b in range(B) for h in range(Hkv * G) for i in range(nt))
    assert sorted(units) == want
    n_items = sum(len(l) for l in lists)
    assert len(lists) == min(n_items, nsm)
    loads = [sum(cost(it) for it in l) for l in lists]
    biggest = max(cost(it) for l in lists for it in l)
    assert max(loads) <= sum(loads) / len(lists) + biggest
