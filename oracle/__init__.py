"""FP64 CPU oracle for packed native-resolution 2D-RoPE varlen attention and its
neighbours (frame-aware 3D RoPE for editing packs, packed-CFG Euler step,
adaptive LayerNorm, gated residual).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s cpu_baseline / reference leg may import this package.  The product
path (``packed_resolution_diffusion_pack_b300``) never imports it, and this
package never imports the product path: the two share nothing but the seeded
input generator in ``synth``.

The arithmetic lives in ``mf_oracle.c`` (plain C, double precision, one query row
at a time, OpenMP across (sample, head) pairs).  This module only compiles it with
gcc and marshals numpy arrays.  Each function cites the page passage it follows in
the C source.  Pins that tie the oracle to something other than itself are in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mf_oracle.c")
_BUILD = os.path.join(_HERE, "_build")

ROPE_BASE = 10000.0


def compile_source(src: str, so: str) -> str:
    """gcc -O2 -fopenmp a C source file into a shared library."""
    tmp = so + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-D_DEFAULT_SOURCE", src, "-o", tmp, "-lm"])
    os.replace(tmp, so)
    return so


def build(force: bool = False) -> str:
    """Compile mf_oracle.c into _build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    so = os.path.join(_BUILD, "liboracle.so")
    if force or not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(_SRC):
        compile_source(_SRC, so)
    return so


_libs: dict = {}


def lib(so: str | None = None):
    """The compiled oracle; ``so`` selects another build of the same source
    (tests that plant a mistake in a copy of the oracle use this)."""
    key = so or "default"
    if key not in _libs:
        L = ctypes.CDLL(so or build())
        p, i64, f64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
        L.oracle_pack.argtypes = [p, i64, p, p]
        L.oracle_rope2d.argtypes = [p, p, i64, i64, i64, f64, i32, p]
        L.oracle_attn_fwd.argtypes = [p, p, p, p, i64, p, i64, i64, i64, f64, f64, p, p]
        L.oracle_attn_bwd.argtypes = [p, p, p, p, p, i64, p, i64, i64, i64, f64, f64, p, p, p]
        L.oracle_attn_fwd_rows.argtypes = [p, p, p, p, i64, p, i64, i64, i64, f64, f64, p, i64, p, p]
        L.oracle_cfg_euler.argtypes = [p, p, i64, i64, f64, f64, p, p]
        L.oracle_pack3d.argtypes = [p, i64, p, p]
        L.oracle_rope3d.argtypes = [p, p, i64, i64, i64, f64, i32, p]
        L.oracle_adaln.argtypes = [p, p, i64, i64, p, p, f64, p]
        L.oracle_gated_residual.argtypes = [p, p, p, i64, i64, p, p]
        L.oracle_e4m3_array.argtypes = [p, i64, p]
        L.oracle_quant_e4m3.argtypes = [p, p, p, p, i64, i64, i64, i32, p, p, p, p, p, p]
        L.oracle_attn_fwd_e4m3.argtypes = [p, p, p, p, p, p, p, i64, i64, i64, i64, f64, i32, p,
                                           p]
        for f in (L.oracle_pack, L.oracle_rope2d, L.oracle_attn_fwd, L.oracle_attn_bwd,
                  L.oracle_attn_fwd_rows, L.oracle_cfg_euler, L.oracle_adaln,
                  L.oracle_gated_residual, L.oracle_pack3d, L.oracle_rope3d,
                  L.oracle_e4m3_array, L.oracle_quant_e4m3, L.oracle_attn_fwd_e4m3):
            f.restype = ctypes.c_int
        _libs[key] = L
    return _libs[key]


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data


def pack(specs, so: str | None = None):
    """(cu_seqlens int64[n+1], pos int64[T, 2]) for specs [(text_len, H, W)]."""
    s = np.ascontiguousarray(np.asarray(specs, dtype=np.int64).reshape(-1, 3))
    n = s.shape[0]
    cu = np.zeros(n + 1, dtype=np.int64)
    if lib(so).oracle_pack(s.ctypes.data, n, cu.ctypes.data, None) != 0:
        raise ValueError("negative spec entry")
    pos = np.zeros((int(cu[-1]), 2), dtype=np.int64)
    lib(so).oracle_pack(s.ctypes.data, n, cu.ctypes.data, pos.ctypes.data)
    return cu, pos


def rope2d(x, pos, inverse: bool = False, base: float = ROPE_BASE, so: str | None = None):
    """R(+theta) x (or R(-theta) x) for x [T, heads, d] float64, pos [T, 2]."""
    x = _f64(x)
    T, h, d = x.shape
    y = np.empty_like(x)
    p = np.ascontiguousarray(pos, dtype=np.int64)
    rc = lib(so).oracle_rope2d(x.ctypes.data, p.ctypes.data, T, h, d, base,
                                    -1 if inverse else 1, y.ctypes.data)
    if rc != 0:
        raise ValueError("head_dim must be a multiple of 4")
    return y


def attn_fwd(q, k, v, cu, pos, scale=None, base: float = ROPE_BASE, so: str | None = None):
    """O [T, h, d] and LSE [h, T] (float64).  pos=None: no rotation."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, h, d = q.shape
    cu = np.ascontiguousarray(cu, dtype=np.int64)
    p = None if pos is None else np.ascontiguousarray(pos, dtype=np.int64)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = np.zeros_like(q)
    lse = np.zeros((h, T), dtype=np.float64)
    lib(so).oracle_attn_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, cu.ctypes.data,
                                 len(cu) - 1, _ptr(p), T, h, d, scale, base, o.ctypes.data,
                                 lse.ctypes.data)
    return o, lse


def attn_fwd_rows(q, k, v, cu, pos, rows, scale=None, base: float = ROPE_BASE,
                  so: str | None = None):
    """O and LSE of selected query rows only; rows = [(token, head), ...].
    Returns (o_rows [m, d], lse_rows [m])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, h, d = q.shape
    cu = np.ascontiguousarray(cu, dtype=np.int64)
    p = None if pos is None else np.ascontiguousarray(pos, dtype=np.int64)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = np.zeros((len(r), d))
    lse = np.zeros(len(r))
    rc = lib(so).oracle_attn_fwd_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, cu.ctypes.data,
                                      len(cu) - 1, _ptr(p), T, h, d, scale, base, r.ctypes.data,
                                      len(r), o.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("row outside the pack")
    return o, lse


def attn_bwd(q, k, v, d_o, cu, pos, scale=None, base: float = ROPE_BASE, so: str | None = None):
    """dQ, dK, dV [T, h, d] (float64) with respect to the un-rotated q, k, v."""
    q, k, v, d_o = _f64(q), _f64(k), _f64(v), _f64(d_o)
    T, h, d = q.shape
    cu = np.ascontiguousarray(cu, dtype=np.int64)
    p = None if pos is None else np.ascontiguousarray(pos, dtype=np.int64)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(q), np.zeros_like(q)
    lib(so).oracle_attn_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, d_o.ctypes.data,
                                 cu.ctypes.data, len(cu) - 1, _ptr(p), T, h, d, scale, base,
                                 dq.ctypes.data, dk.ctypes.data, dv.ctypes.data)
    return dq, dk, dv


def pack3d(specs, so: str | None = None):
    """Editing packs: (cu_seqlens int64[n+1], pos int64[T, 3] = (frame, row, col)) for
    specs [(text_len, Hs, Ws, Ht, Wt)], each sample [text; source; target]."""
    s = np.ascontiguousarray(np.asarray(specs, dtype=np.int64).reshape(-1, 5))
    n = s.shape[0]
    cu = np.zeros(n + 1, dtype=np.int64)
    if lib(so).oracle_pack3d(s.ctypes.data, n, cu.ctypes.data, None) != 0:
        raise ValueError("negative spec entry")
    pos = np.zeros((int(cu[-1]), 3), dtype=np.int64)
    lib(so).oracle_pack3d(s.ctypes.data, n, cu.ctypes.data, pos.ctypes.data)
    return cu, pos


def rope3d(x, pos, inverse: bool = False, base: float = ROPE_BASE, so: str | None = None):
    """Frame-aware 3D rotation R(+theta) x (or R(-theta) x); x [T, heads, d] float64,
    pos [T, 3]."""
    x = _f64(x)
    T, h, d = x.shape
    y = np.empty_like(x)
    p = np.ascontiguousarray(pos, dtype=np.int64)
    if lib(so).oracle_rope3d(x.ctypes.data, p.ctypes.data, T, h, d, base,
                             -1 if inverse else 1, y.ctypes.data) != 0:
        raise ValueError("head_dim must be a multiple of 16")
    return y


def attn_fwd3d(q, k, v, cu, pos3, scale=None, base: float = ROPE_BASE, so: str | None = None):
    """Attention of an editing pack: the attention above on q' = R3 q, k' = R3 k
    (the definition written out: rotate, then attend without rotation)."""
    return attn_fwd(rope3d(q, pos3, base=base, so=so), rope3d(k, pos3, base=base, so=so), v, cu,
                    None, scale=scale, so=so)


def attn_bwd3d(q, k, v, d_o, cu, pos3, scale=None, base: float = ROPE_BASE,
               so: str | None = None):
    """Gradients of attn_fwd3d with respect to the un-rotated q, k, v: the gradients
    with respect to q', k' taken back through the rotation's transpose R3(-theta)."""
    dqr, dkr, dv = attn_bwd(rope3d(q, pos3, base=base, so=so), rope3d(k, pos3, base=base, so=so),
                            v, d_o, cu, None, scale=scale, so=so)
    return (rope3d(dqr, pos3, inverse=True, base=base, so=so),
            rope3d(dkr, pos3, inverse=True, base=base, so=so), dv)


def cfg_euler(v, specs, guidance: float, dt: float, z, so: str | None = None):
    """One packed-CFG rectified-flow Euler step: z + dt * (v_u + g (v_c - v_u)) on
    each (cond, uncond) pair's image rows.  v [T, C], z [N, C] (float64);
    specs = [(text_len, H, W)] * 2 pairs, cond then uncond per pair."""
    v, z = _f64(v), _f64(z)
    s = np.ascontiguousarray(np.asarray(specs, dtype=np.int64).reshape(-1, 3))
    if s.shape[0] % 2:
        raise ValueError("specs must hold (cond, uncond) pairs")
    out = np.empty_like(z)
    rc = lib(so).oracle_cfg_euler(v.ctypes.data, s.ctypes.data, s.shape[0] // 2, v.shape[1],
                                  float(guidance), float(dt), z.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError("a pair's two samples have different image grids")
    return out


def adaln(x, cu, shift, scale, eps: float = 1e-6, so: str | None = None):
    """LN(x) * (1 + scale_s) + shift_s per token of sample s; x [T, Dm] (float64)."""
    x, shift, scale = _f64(x), _f64(shift), _f64(scale)
    cu = np.ascontiguousarray(cu, dtype=np.int64)
    y = np.empty_like(x)
    lib(so).oracle_adaln(x.ctypes.data, cu.ctypes.data, len(cu) - 1, x.shape[1],
                         shift.ctypes.data, scale.ctypes.data, float(eps), y.ctypes.data)
    return y


def gated_residual(x, h, cu, gate, so: str | None = None):
    """x + gate_s * h per token of sample s; x, h [T, Dm] (float64)."""
    x, h, gate = _f64(x), _f64(h), _f64(gate)
    cu = np.ascontiguousarray(cu, dtype=np.int64)
    out = np.empty_like(x)
    lib(so).oracle_gated_residual(x.ctypes.data, h.ctypes.data, cu.ctypes.data, len(cu) - 1,
                                  x.shape[1], gate.ctypes.data, out.ctypes.data)
    return out


def e4m3(x, so: str | None = None):
    """Nearest OCP E4M3 value of each element (ties to even, saturating at +-448),
    as float64."""
    x = _f64(x)
    y = np.empty_like(x)
    lib(so).oracle_e4m3_array(x.ctypes.data, x.size, y.ctypes.data)
    return y


def quant_e4m3(q, k, v, pos, round: bool = True, base: float = ROPE_BASE,
               so: str | None = None):
    """The 8-bit variant's operands: (qh, sq, kh, sk, vh, sv) with qh, kh, vh
    [T, h, d] (e4m3 values as float64), sq [T, h], sk and sv [h].  q and k are
    rotated first (pos [T, 2]: 2D rotation, [T, 3]: frame-aware 3D, None: none)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, h, d = q.shape
    if pos is None:
        qr, kr = q, k
    elif np.asarray(pos).shape[1] == 3:
        qr, kr = rope3d(q, pos, base=base, so=so), rope3d(k, pos, base=base, so=so)
    else:
        qr, kr = rope2d(q, pos, base=base, so=so), rope2d(k, pos, base=base, so=so)
    qh, kh, vh = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    sq = np.empty((T, h))
    sk, sv = np.empty(h), np.empty(h)
    if lib(so).oracle_quant_e4m3(_f64(qr).ctypes.data, k.ctypes.data, _f64(kr).ctypes.data,
                                 v.ctypes.data, T, h, d, 1 if round else 0, qh.ctypes.data,
                                 sq.ctypes.data, kh.ctypes.data, sk.ctypes.data, vh.ctypes.data,
                                 sv.ctypes.data) != 0:
        raise ValueError("head_dim must be even")
    return qh, sq, kh, sk, vh, sv


def attn_fwd_e4m3(q, k, v, cu, pos, scale=None, round: bool = True, base: float = ROPE_BASE,
                  so: str | None = None):
    """O [T, h, d] and LSE [h, T] of the 8-bit variant of the forward (operands and
    probabilities rounded to e4m3; round=False keeps every value exact)."""
    qh, sq, kh, sk, vh, sv = quant_e4m3(q, k, v, pos, round=round, base=base, so=so)
    return attn_fwd_e4m3_quantized(qh, sq, kh, sk, vh, sv, cu, scale=scale, round=round, so=so)


def attn_fwd_e4m3_quantized(qh, sq, kh, sk, vh, sv, cu, scale=None, round: bool = True,
                            so: str | None = None):
    """The attention steps of the 8-bit variant on operands that quant_e4m3 made
    (for example over a whole head, then applied to one sample's slice)."""
    qh, sq, kh, sk, vh, sv = (_f64(a) for a in (qh, sq, kh, sk, vh, sv))
    T, h, d = qh.shape
    cu = np.ascontiguousarray(cu, dtype=np.int64)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = np.zeros_like(qh)
    lse = np.zeros((h, T))
    lib(so).oracle_attn_fwd_e4m3(qh.ctypes.data, sq.ctypes.data, kh.ctypes.data, sk.ctypes.data,
                                 vh.ctypes.data, sv.ctypes.data, cu.ctypes.data, len(cu) - 1, T,
                                 h, d, scale, 1 if round else 0, o.ctypes.data, lse.ctypes.data)
    return o, lse


def sample_head_slice(x, cu, i: int, a: int):
    """Rows of sample i, head a of a packed [T, h, d] array, as [L_i, 1, d]."""
    return x[int(cu[i]):int(cu[i + 1]), a:a + 1, :]


def attn_fwd_pair(q, k, v, cu, pos, i: int, a: int, **kw):
    """The oracle on one (sample, head) pair: exact because samples and heads are
    independent in the definition.  Returns O [L, d], LSE [L]."""
    sl = slice(int(cu[i]), int(cu[i + 1]))
    L = sl.stop - sl.start
    o, lse = attn_fwd(sample_head_slice(q, cu, i, a), sample_head_slice(k, cu, i, a),
                      sample_head_slice(v, cu, i, a), np.array([0, L]), pos[sl], **kw)
    return o[:, 0, :], lse[0]


def attn_bwd_pair(q, k, v, d_o, cu, pos, i: int, a: int, **kw):
    sl = slice(int(cu[i]), int(cu[i + 1]))
    L = sl.stop - sl.start
    dq, dk, dv = attn_bwd(sample_head_slice(q, cu, i, a), sample_head_slice(k, cu, i, a),
                          sample_head_slice(v, cu, i, a), sample_head_slice(d_o, cu, i, a),
                          np.array([0, L]), pos[sl], **kw)
    return dq[:, 0, :], dk[:, 0, :], dv[:, 0, :]
