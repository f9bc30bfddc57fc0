"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every
function include/mf.h declares, and rejects bad arguments on the host before any
device work (CPU only)."""
import ctypes
import os
import re

import pytest

import packed_resolution_diffusion_pack_b300 as mf
from packed_resolution_diffusion_pack_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "mf.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mf_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol():
    lib = mf.load()
    names = _declared()
    assert len(names) >= 9
    for name in names:
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_status_strings_and_version():
    lib = mf.load()
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.mf_status_string(code).decode() == name
    assert lib.mf_version() == 10000


def test_pack_size_host():
    assert mf.pack_size([(5, 4, 6), (7, 8, 8), (3, 2, 16)]) == (135, 71)
    assert mf.pack_size([]) == (0, 0)
    assert mf.pack_size([(0, 0, 0), (3, 0, 5)]) == (3, 3)


@pytest.mark.parametrize("specs,code", [
    ([(1, 2, 3), (-1, 2, 2)], 1),
    ([(1, -2, 3)], 1),
    ([(0, 65536, 65536)], 3),
    ([(2 ** 31 - 1, 0, 0), (1, 0, 0)], 3),
])
def test_pack_size_errors(specs, code):
    with pytest.raises(mf.MFError) as ei:
        mf.pack_size(specs)
    assert ei.value.status == code


def _fwd(lib, q=16, k=16, v=16, o=16, lse=16, cu=16, n=1, T=8, max_len=8, h=1, d=64, ws=256,
         ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.mf_attn_workspace_bytes(T, n, h, d, 0)
    p = ctypes.c_void_p
    return lib.mf_varlen_attn_fwd(p(q), p(k), p(v), p(cu), None, n, T, max_len, h, d, 0.0, p(o),
                                  p(lse), p(ws), ws_bytes, None)


def test_attn_argument_errors_on_host():
    lib = mf.load()
    # fake, never dereferenced addresses: every case must be rejected before launch
    base = 1 << 20
    a = dict(q=base, k=base + 4096, v=base + 8192, o=base + 12288, lse=base + 16384,
             cu=base + 20480, ws=base + 24576)
    assert _fwd(lib, **a, d=96) == 2           # head_dim unsupported
    assert _fwd(lib, **{**a, "q": base + 8}) == 2  # misaligned tensor
    assert _fwd(lib, **{**a, "ws": base + 64}) == 2  # misaligned workspace
    assert _fwd(lib, **a, ws_bytes=16) == 1    # workspace too small
    assert _fwd(lib, **a, n=-1) == 1
    assert _fwd(lib, **a, h=0) == 1
    assert _fwd(lib, **{**a, "cu": 0}) == 1
    assert _fwd(lib, **{**a, "q": 0}) == 1
    assert _fwd(lib, **a, T=2 ** 30, h=64) == 3  # heads * T overflows int32
    assert lib.mf_attn_workspace_bytes(10, 1, 1, 96, 0) == 0
    # a backward workspace also serves the forward (the training step shares one)
    assert lib.mf_attn_workspace_bytes(10, 1, 2, 128, 1) >= lib.mf_attn_workspace_bytes(10, 1, 2, 128, 0)


def test_rope_argument_errors_on_host():
    lib = mf.load()
    p = ctypes.c_void_p
    assert lib.mf_rope2d_qk(p(1 << 20), None, p(1 << 21), None, p(1 << 22), 4, 2, 80, None) == 2
    assert lib.mf_rope2d_qk(p(1 << 20), None, None, None, p(1 << 22), 4, 2, 64, None) == 1
    assert lib.mf_rope2d_qk(p(1 << 20), None, p(1 << 21), None, None, 4, 2, 64, None) == 1
    assert lib.mf_rope2d_qk(p((1 << 20) + 2), None, p(1 << 21), None, p(1 << 22), 4, 2, 64, None) == 2
    assert lib.mf_rope2d_qk(None, None, None, None, None, 0, 2, 64, None) == 0  # nothing to do


def test_get_status_rejects_null():
    assert mf.load().mf_get_status(None, None) == 1


def test_neighbour_argument_errors_on_host():
    lib = mf.load()
    p = ctypes.c_void_p
    spec = lambda rows: (ctypes.c_int32 * (3 * len(rows)))(*[x for r in rows for x in r])  # noqa: E731
    good = spec([(1, 2, 3), (4, 2, 3)])
    base = 1 << 20
    # CFG step: every case rejected (or empty) before any launch
    assert lib.mf_cfg_euler_step(p(base), good, 1, 12, 2.0, 0.1, p(base + 4096), None) == 2  # C % 8
    assert lib.mf_cfg_euler_step(p(base), good, -1, 8, 2.0, 0.1, p(base + 4096), None) == 1
    assert lib.mf_cfg_euler_step(p(base), spec([(1, 2, 3), (4, 3, 2)]), 1, 8, 2.0, 0.1,
                                 p(base + 4096), None) == 1  # grids differ
    assert lib.mf_cfg_euler_step(p(base), spec([(1, 2, 3), (-4, 2, 3)]), 1, 8, 2.0, 0.1,
                                 p(base + 4096), None) == 1
    assert lib.mf_cfg_euler_step(p(base + 8), good, 1, 8, 2.0, 0.1, p(base + 4096), None) == 2
    assert lib.mf_cfg_euler_step(None, good, 1, 8, 2.0, 0.1, p(base + 4096), None) == 1
    assert lib.mf_cfg_euler_step(None, spec([(1, 0, 3), (4, 0, 3)]), 1, 8, 2.0, 0.1, None, None) == 0
    # adaptive LayerNorm / gated residual
    x, s1, s2, y = p(base), p(base + 4096), p(base + 8192), p(base + 12288)
    cu = p(base + 16384)
    assert lib.mf_adaln_modulate(x, cu, 2, 10, 12, s1, s2, 1e-6, y, None) == 2    # Dm % 8
    assert lib.mf_adaln_modulate(x, cu, 0, 10, 64, s1, s2, 1e-6, y, None) == 1    # no samples
    assert lib.mf_adaln_modulate(x, cu, 2, 10, 64, s1, s2, -1.0, y, None) == 1    # eps < 0
    assert lib.mf_adaln_modulate(p(base + 4), cu, 2, 10, 64, s1, s2, 1e-6, y, None) == 2
    assert lib.mf_adaln_modulate(x, None, 2, 10, 64, s1, s2, 1e-6, y, None) == 1
    assert lib.mf_adaln_modulate(None, None, 0, 0, 64, None, None, 1e-6, None, None) == 0
    assert lib.mf_gated_residual(x, s1, cu, 2, 10, 60, s2, y, None) == 2
    assert lib.mf_gated_residual(x, None, cu, 2, 10, 64, s2, y, None) == 1
    assert lib.mf_gated_residual(x, s1, cu, -1, 10, 64, s2, y, None) == 1


def test_pack3d_size_host():
    assert mf.pack3d_size([(2, 1, 2, 2, 1)]) == (6, 6)
    assert mf.pack3d_size([]) == (0, 0)
    with pytest.raises(mf.MFError) as ei:
        mf.pack3d_size([(1, 2, 3, -1, 1)])
    assert ei.value.status == 1
    with pytest.raises(mf.MFError) as ei:
        mf.pack3d_size([(0, 65536, 65536, 0, 0)])
    assert ei.value.status == 3
    lib = mf.load()
    p = ctypes.c_void_p
    assert lib.mf_rope3d_qk(p(1 << 20), None, p(1 << 21), None, p(1 << 22), 4, 2, 80, None) == 2
    assert lib.mf_rope3d_qk(p(1 << 20), None, p(1 << 21), None, None, 4, 2, 64, None) == 1
    assert lib.mf_varlen_attn_fwd_3d(p(1 << 20), p(1 << 21), p(1 << 22), p(1 << 23), None, 1, 8, 8,
                                     1, 64, 0.0, p(1 << 24), p(1 << 25), p(1 << 26), 1 << 20,
                                     None) == 1  # 3D positions are required


def test_fp8_argument_errors_on_host():
    """The 8-bit forward and its quantisation: head_dim 64, a bad pos_axes, null or
    misaligned buffers are rejected before any launch."""
    lib = mf.load()
    p = ctypes.c_void_p
    base = 1 << 20
    q, k, v, o, lse = (p(base + i * 4096) for i in range(5))
    cu, pos, ws = p(base + 40960), p(base + 45056), p(base + 65536)
    big = 1 << 40
    assert lib.mf_varlen_attn_fwd_fp8(q, k, v, cu, pos, 2, 1, 10, 10, 2, 64, 0.0, o, lse, ws, big,
                                      None) == 2
    assert lib.mf_varlen_attn_fwd_fp8(q, k, v, cu, pos, 4, 1, 10, 10, 2, 128, 0.0, o, lse, ws, big,
                                      None) == 1
    assert lib.mf_varlen_attn_fwd_fp8(q, None, v, cu, pos, 2, 1, 10, 10, 2, 128, 0.0, o, lse, ws,
                                      big, None) == 1
    assert lib.mf_varlen_attn_fwd_fp8(q, k, v, cu, pos, 2, 1, 10, 10, 2, 128, 0.0, o, lse, ws, 16,
                                      None) == 1  # workspace too small
    q8, k8, v8, qs, kv = (p(base + 8192 * (i + 1)) for i in range(5))
    assert lib.mf_quant_e4m3(q, k, v, pos, 2, 10, 2, 64, q8, k8, v8, qs, kv, None) == 2
    assert lib.mf_quant_e4m3(q, k, v, pos, 5, 10, 2, 128, q8, k8, v8, qs, kv, None) == 1
    assert lib.mf_quant_e4m3(q, k, v, pos, 2, 10, 2, 128, None, k8, v8, qs, kv, None) == 1
    assert lib.mf_quant_e4m3(q, k, v, pos, 2, 10, 2, 128, p(base + 8200), k8, v8, qs, kv,
                             None) == 2
    assert lib.mf_quant_e4m3(q, k, v, pos, 2, -1, 2, 128, q8, k8, v8, qs, kv, None) == 1


def test_binding_argument_counts_match_header():
    """Every declaration in mf.h has as many parameters as its ctypes binding
    declares (a drifted binding would shift every argument after the change)."""
    src = open(os.path.join(ROOT, "include", "mf.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    decls = dict(re.findall(r"\b(mf_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", src))
    assert len(decls) >= 9
    for name, params in decls.items():
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(_lib.SIGNATURES[name][1]) == n, (name, n, len(_lib.SIGNATURES[name][1]))


def test_noalloc_binding_rejects_editing_positions():
    """The allocation-free forward takes 2D positions only: an editing pack's
    [T, 3] table, or a table of the wrong dtype, is refused on the host before
    the C call (it would otherwise be read with a stride of 2)."""
    import torch
    T = 8
    q = torch.zeros((T, 1, 64), dtype=torch.bfloat16)
    cu = torch.tensor([0, T], dtype=torch.int32)
    with pytest.raises(ValueError, match="2D positions"):
        mf.varlen_attn_fwd_noalloc(q, q, q, cu, torch.zeros((T, 3), dtype=torch.int32), T)
    with pytest.raises(ValueError, match="int32"):
        mf.varlen_attn_fwd_noalloc(q, q, q, cu, torch.zeros((T, 2), dtype=torch.int64), T)


def test_fused_rope_forward_argument_errors_on_host():
    """The rotate-on-load forward: unsupported head_dim, misaligned or null buffers
    and a short workspace are rejected before any launch; 3D positions are refused
    by the binding."""
    import torch
    lib = mf.load()
    p = ctypes.c_void_p
    base = 1 << 20
    q, k, v, o, lse, cu, ws = (p(base + 4096 * i) for i in range(7))
    pos = p(base + 65536)
    fn = lib.mf_varlen_attn_fwd_fused_rope
    big = lib.mf_attn_workspace_bytes(8, 1, 1, 64, 0)
    assert fn(q, k, v, cu, pos, 1, 8, 8, 1, 96, 0.0, o, lse, ws, big, None) == 2
    assert fn(q, k, v, cu, p(base + 65540), 1, 8, 8, 1, 64, 0.0, o, lse, ws, big, None) == 2
    assert fn(q, None, v, cu, pos, 1, 8, 8, 1, 64, 0.0, o, lse, ws, big, None) == 1
    assert fn(q, k, v, cu, pos, 1, 8, 8, 1, 64, 0.0, o, lse, ws, 16, None) == 1
    assert fn(q, k, v, None, pos, 1, 8, 8, 1, 64, 0.0, o, lse, ws, big, None) == 1
    T = 8
    x = torch.zeros((T, 1, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="2D positions"):
        mf.varlen_attn_fwd_fused_rope(x, x, x, torch.tensor([0, T], dtype=torch.int32),
                                      torch.zeros((T, 3), dtype=torch.int32), T)


def test_stored_ds_workspace_size():
    """mf_attn_workspace_bytes_ds: the backward workspace (rounded up to 1 KB) plus
    heads (ceil(T / 128) + n) tiles of 128 keys x (max_len rounded up to 128)
    fp16 queries; 0 for invalid sizes."""
    lib = mf.load()
    T, n, h, d, L = 48019, 18, 24, 128, 4291
    base = lib.mf_attn_workspace_bytes(T, n, h, d, 1)
    got = lib.mf_attn_workspace_bytes_ds(T, n, h, d, L)
    ds = h * (-(-T // 128) + n) * 128 * (-(-L // 128) * 128) * 2
    assert got == -(-base // 1024) * 1024 + ds
    assert mf.attn_workspace_bytes_ds(T, n, h, d, L) == got
    assert lib.mf_attn_workspace_bytes_ds(T, n, h, 96, L) == 0
    assert lib.mf_attn_workspace_bytes_ds(T, n, h, d, -1) == 0
    assert lib.mf_attn_workspace_bytes_ds(-1, n, h, d, L) == 0
