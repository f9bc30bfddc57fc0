"""Packed native-resolution 2D-RoPE varlen attention on B300 (sm_103a).

The hot path of Mage-Flow's native-resolution MMDiT joint attention: pack many
[text; image-latent] samples into one token stream, rotate Q/K by each image
token's native (row, col) latent position, and run block-diagonal (per-sample)
attention forward and backward.  All compute runs in the hand-written CUDA
kernels of ``libmf.so`` (C ABI: ``include/mf.h``); this module only marshals
torch tensors (device memory, streams) into those calls.

Tensors are "THD": ``[T, heads, head_dim]`` bf16, contiguous, on a CUDA device.
"""
from __future__ import annotations

import ctypes

from ._lib import MFError, STATUS_NAMES, check, library_path, load

__all__ = [
    "MFError", "STATUS_NAMES", "load", "library_path", "pack_size", "pack", "rope2d_qk",
    "attn_workspace_bytes", "workspace", "varlen_attn_fwd", "varlen_attn_bwd", "get_status",
    "cfg_euler_step", "adaln_modulate", "gated_residual", "pack3d_size", "pack3d", "rope3d_qk",
    "varlen_attn_fwd_fp8", "quant_e4m3", "varlen_attn_fwd_noalloc", "noalloc_get_status",
    "varlen_attn_fwd_fused_rope", "attn_workspace_bytes_ds",
]


def _torch():
    import torch
    return torch


def _stream_ptr(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _specs_array(specs):
    flat = [int(x) for s in specs for x in s]
    if len(flat) != 3 * len(specs):
        raise ValueError("specs must be (text_len, H_lat, W_lat) triples")
    return (ctypes.c_int32 * max(1, len(flat)))(*flat), len(specs)


def _check_thd(name, t, T=None, heads=None, head_dim=None):
    torch = _torch()
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
        raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [T, heads, head_dim]")
    if (T is not None and t.shape[0] != T) or (heads is not None and t.shape[1] != heads) or \
            (head_dim is not None and t.shape[2] != head_dim):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected ({T}, {heads}, {head_dim})")


def pack_size(specs):
    """(T, max_len) of a pack of (text_len, H_lat, W_lat) samples (host only)."""
    arr, n = _specs_array(specs)
    T, mx = ctypes.c_int32(), ctypes.c_int32()
    check(load().mf_pack_size(arr, n, ctypes.byref(T), ctypes.byref(mx)), "mf_pack_size")
    return T.value, mx.value


def pack(specs, device=None, stream=None, with_pos: bool = True, cu=None, pos=None):
    """cu_seqlens int32 [n+1] and pos int32 [T, 2] built on the device by mf_pack
    (into `cu` / `pos` when given)."""
    torch = _torch()
    arr, n = _specs_array(specs)
    T, _ = pack_size(specs)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if cu is None:
        cu = torch.empty(n + 1, dtype=torch.int32, device=dev)
    if pos is None and with_pos:
        pos = torch.empty((T, 2), dtype=torch.int32, device=dev)
    if cu.numel() != n + 1 or cu.dtype != torch.int32 or (pos is not None and pos.shape != (T, 2)):
        raise ValueError("cu/pos buffers do not match the specs")
    check(load().mf_pack(arr, n, _ptr(cu), _ptr(pos) if pos is not None and T > 0 else None,
                         _stream_ptr(stream)), "mf_pack")
    return cu, pos


def _specs5_array(specs):
    flat = [int(x) for s in specs for x in s]
    if len(flat) != 5 * len(specs):
        raise ValueError("editing specs must be (text_len, Hs, Ws, Ht, Wt) tuples")
    return (ctypes.c_int32 * max(1, len(flat)))(*flat), len(specs)


def pack3d_size(specs):
    """(T, max_len) of an editing pack of (text_len, Hs, Ws, Ht, Wt) samples."""
    arr, n = _specs5_array(specs)
    T, mx = ctypes.c_int32(), ctypes.c_int32()
    check(load().mf_pack3d_size(arr, n, ctypes.byref(T), ctypes.byref(mx)), "mf_pack3d_size")
    return T.value, mx.value


def pack3d(specs, device=None, stream=None, cu=None, pos=None):
    """cu_seqlens int32 [n+1] and pos int32 [T, 3] = (frame, row, col) of an editing
    pack [text; source; target] built on the device by mf_pack3d."""
    torch = _torch()
    arr, n = _specs5_array(specs)
    T, _ = pack3d_size(specs)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    cu = torch.empty(n + 1, dtype=torch.int32, device=dev) if cu is None else cu
    pos = torch.empty((T, 3), dtype=torch.int32, device=dev) if pos is None else pos
    if cu.numel() != n + 1 or pos.shape != (T, 3):
        raise ValueError("cu/pos buffers do not match the specs")
    check(load().mf_pack3d(arr, n, _ptr(cu), _ptr(pos) if T > 0 else None, _stream_ptr(stream)),
          "mf_pack3d")
    return cu, pos


def rope3d_qk(q, k, pos3, q_out=None, k_out=None, stream=None):
    """Frame-aware 3D RoPE of q and k (either may be None); returns (q_out, k_out)."""
    torch = _torch()
    ref = q if q is not None else k
    _check_thd("q/k", ref)
    T, h, d = ref.shape
    if q is not None:
        q_out = torch.empty_like(q) if q_out is None else q_out
        _check_thd("q_out", q_out, T, h, d)
    if k is not None:
        k_out = torch.empty_like(k) if k_out is None else k_out
        _check_thd("k_out", k_out, T, h, d)
    check(load().mf_rope3d_qk(_ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), _ptr(pos3), T, h, d,
                              _stream_ptr(stream)), "mf_rope3d_qk")
    return q_out, k_out


def rope2d_qk(q, k, pos, q_out=None, k_out=None, stream=None):
    """Per-sample 2D RoPE of q and k (either may be None); returns (q_out, k_out)."""
    torch = _torch()
    ref = q if q is not None else k
    _check_thd("q/k", ref)
    T, h, d = ref.shape
    if q is not None:
        _check_thd("q", q, T, h, d)
        q_out = torch.empty_like(q) if q_out is None else q_out
        _check_thd("q_out", q_out, T, h, d)
    if k is not None:
        _check_thd("k", k, T, h, d)
        k_out = torch.empty_like(k) if k_out is None else k_out
        _check_thd("k_out", k_out, T, h, d)
    check(load().mf_rope2d_qk(_ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), _ptr(pos), T, h, d,
                              _stream_ptr(stream)), "mf_rope2d_qk")
    return q_out, k_out


def attn_workspace_bytes(T, n, heads, head_dim, bwd: bool) -> int:
    return int(load().mf_attn_workspace_bytes(T, n, heads, head_dim, 1 if bwd else 0))


def attn_workspace_bytes_ds(T, n, heads, head_dim, max_len) -> int:
    """Workspace bytes that select the backward's stored-dS form (0: unavailable)."""
    return int(load().mf_attn_workspace_bytes_ds(T, n, heads, head_dim, int(max_len)))


def workspace(T, n, heads, head_dim, bwd: bool, device=None, store_ds_max_len=None):
    """A device workspace of the size the library asks for (uint8 tensor).  With
    store_ds_max_len (the call's max_len), a backward workspace large enough for
    the stored-dS form (mf_attn_workspace_bytes_ds)."""
    torch = _torch()
    if store_ds_max_len is not None:
        nbytes = attn_workspace_bytes_ds(T, n, heads, head_dim, store_ds_max_len)
    else:
        nbytes = attn_workspace_bytes(T, n, heads, head_dim, bwd)
    if nbytes == 0:
        raise ValueError("invalid attention sizes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def _is_3d(pos) -> bool:
    """Positions with three coordinates per token select the editing-pack entry points."""
    if pos is None:
        return False
    if pos.dim() != 2 or pos.shape[1] not in (2, 3) or pos.dtype != _torch().int32:
        raise ValueError("pos must be an int32 tensor [T, 2] or [T, 3]")
    return pos.shape[1] == 3


def varlen_attn_fwd(q, k, v, cu_seqlens, pos, max_len, softmax_scale: float = 0.0, o=None,
                    lse=None, ws=None, stream=None):
    """Block-diagonal attention forward with per-sample 2D RoPE (pos [T, 2]; None:
    no rotation) or, for editing packs, the frame-aware 3D RoPE (pos [T, 3]).
    Returns (o [T, h, d] bf16, lse [h, T] fp32)."""
    torch = _torch()
    _check_thd("q", q)
    T, h, d = q.shape
    for name, t in (("k", k), ("v", v)):
        _check_thd(name, t, T, h, d)
    n = cu_seqlens.numel() - 1
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((h, T), dtype=torch.float32, device=q.device) if lse is None else lse
    ws = workspace(T, n, h, d, False, q.device) if ws is None else ws
    fn = "mf_varlen_attn_fwd_3d" if _is_3d(pos) else "mf_varlen_attn_fwd"
    check(getattr(load(), fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(pos), n, T,
                              int(max_len), h, d, float(softmax_scale), _ptr(o), _ptr(lse),
                              _ptr(ws), ws.numel(), _stream_ptr(stream)), fn)
    return o, lse


def varlen_attn_fwd_fused_rope(q, k, v, cu_seqlens, pos, max_len, softmax_scale: float = 0.0,
                               o=None, lse=None, ws=None, stream=None):
    """varlen_attn_fwd with the 2D RoPE applied on the attention kernel's tile load
    (no rotation pre-pass; pos [T, 2] int32 or None).  Same outputs, bit for bit.
    The workspace keeps no rotated operands: a backward after it is varlen_attn_bwd
    with after_fwd=False.  Returns (o [T, h, d] bf16, lse [h, T] fp32)."""
    torch = _torch()
    if _is_3d(pos):
        raise ValueError("varlen_attn_fwd_fused_rope takes 2D positions [T, 2]")
    _check_thd("q", q)
    T, h, d = q.shape
    for name, t in (("k", k), ("v", v)):
        _check_thd(name, t, T, h, d)
    n = cu_seqlens.numel() - 1
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((h, T), dtype=torch.float32, device=q.device) if lse is None else lse
    ws = workspace(T, n, h, d, False, q.device) if ws is None else ws
    check(load().mf_varlen_attn_fwd_fused_rope(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(pos), n, T, int(max_len), h, d,
        float(softmax_scale), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream_ptr(stream)),
        "mf_varlen_attn_fwd_fused_rope")
    return o, lse


def varlen_attn_bwd(q, k, v, o, lse, d_o, cu_seqlens, pos, max_len, softmax_scale: float = 0.0,
                    dq=None, dk=None, dv=None, ws=None, stream=None, after_fwd: bool = False):
    """Gradients (dq, dk, dv) with respect to the un-rotated q, k and v.

    after_fwd=True: `ws` is the workspace the forward of these q, k, pos just used
    (sized for the backward); the forward's rotated operands are reused and the
    backward's own rotation pre-pass is skipped (mf_varlen_attn_bwd_after_fwd)."""
    torch = _torch()
    _check_thd("q", q)
    T, h, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("d_o", d_o)):
        _check_thd(name, t, T, h, d)
    n = cu_seqlens.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if after_fwd:
        if ws is None:
            raise ValueError("after_fwd needs the workspace the forward used")
        check(load().mf_varlen_attn_bwd_after_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(cu_seqlens), _ptr(pos),
            3 if _is_3d(pos) else 2, n, T, int(max_len), h, d, float(softmax_scale), _ptr(dq),
            _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream_ptr(stream)),
            "mf_varlen_attn_bwd_after_fwd")
        return dq, dk, dv
    ws = workspace(T, n, h, d, True, q.device) if ws is None else ws
    fn = "mf_varlen_attn_bwd_3d" if _is_3d(pos) else "mf_varlen_attn_bwd"
    check(getattr(load(), fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o),
                              _ptr(cu_seqlens), _ptr(pos), n, T, int(max_len), h, d,
                              float(softmax_scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                              ws.numel(), _stream_ptr(stream)), fn)
    return dq, dk, dv


def varlen_attn_fwd_fp8(q, k, v, cu_seqlens, pos, max_len, softmax_scale: float = 0.0, o=None,
                        lse=None, ws=None, stream=None):
    """The 8-bit (E4M3) variant of varlen_attn_fwd (head_dim 128): same arguments
    and outputs, both GEMMs on E4M3 operands and probabilities (mf.h states its
    scaling and rounding steps).  Returns (o [T, h, d] bf16, lse [h, T] fp32)."""
    torch = _torch()
    _check_thd("q", q)
    T, h, d = q.shape
    for name, t in (("k", k), ("v", v)):
        _check_thd(name, t, T, h, d)
    n = cu_seqlens.numel() - 1
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((h, T), dtype=torch.float32, device=q.device) if lse is None else lse
    ws = workspace(T, n, h, d, False, q.device) if ws is None else ws
    axes = 3 if _is_3d(pos) else 2
    check(load().mf_varlen_attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(pos),
                                        axes, n, T, int(max_len), h, d, float(softmax_scale),
                                        _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                                        _stream_ptr(stream)), "mf_varlen_attn_fwd_fp8")
    return o, lse


def quant_e4m3(q, k, v, pos, stream=None):
    """The 8-bit forward's operands: (q8, k8, v8) uint8 [T, h, 128] (E4M3 codes),
    qscale fp32 [T, h] and kv_max2 fp32 [2, h] (squared largest pair norm of k and
    squared largest |v| per head)."""
    torch = _torch()
    _check_thd("q", q)
    T, h, d = q.shape
    for name, t in (("k", k), ("v", v)):
        _check_thd(name, t, T, h, d)
    q8, k8, v8 = (torch.empty((T, h, d), dtype=torch.uint8, device=q.device) for _ in range(3))
    qscale = torch.empty((T, h), dtype=torch.float32, device=q.device)
    kv_max2 = torch.empty((2, h), dtype=torch.float32, device=q.device)
    check(load().mf_quant_e4m3(_ptr(q), _ptr(k), _ptr(v), _ptr(pos), 3 if _is_3d(pos) else 2, T,
                               h, d, _ptr(q8), _ptr(k8), _ptr(v8), _ptr(qscale), _ptr(kv_max2),
                               _stream_ptr(stream)), "mf_quant_e4m3")
    return q8, k8, v8, qscale, kv_max2


def varlen_attn_fwd_noalloc(q, k, v, cu_seqlens, pos, max_len, softmax_scale: float = 0.0,
                            o=None, lse=None, stream=None):
    """The forward without a workspace, for callers that cannot allocate device
    memory (e.g. a plugin handed only its inputs and outputs): its scratch is a
    fixed array inside the library (limits MF_NOALLOC_* in mf.h).  Pass `o` and
    `lse` to keep this call itself free of allocations.  The call takes 2D
    positions only: pos must be None or int32 [T, 2] (an editing pack's [T, 3]
    table raises ValueError).  Device-side errors of the call are read back with
    noalloc_get_status."""
    torch = _torch()
    if _is_3d(pos):
        raise ValueError("the allocation-free forward takes 2D positions (int32 [T, 2]) only")
    _check_thd("q", q)
    T, h, d = q.shape
    for name, t in (("k", k), ("v", v)):
        _check_thd(name, t, T, h, d)
    n = cu_seqlens.numel() - 1
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((h, T), dtype=torch.float32, device=q.device) if lse is None else lse
    check(load().mf_varlen_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(pos),
                                            n, T, int(max_len), h, d, float(softmax_scale), _ptr(o),
                                            _ptr(lse), _stream_ptr(stream)),
          "mf_varlen_attn_fwd_noalloc")
    return o, lse


def cfg_euler_step(v, specs, guidance: float, dt: float, z, stream=None):
    """One packed-CFG rectified-flow Euler step, in place on z (fp32 [N, C]):
    z += dt * (v_u + guidance (v_c - v_u)) over each (cond, uncond) pair's image
    rows of the packed model output v (bf16 [T, C]).  specs: (text_len, H, W) of
    the 2 * pairs samples, cond then uncond per pair."""
    torch = _torch()
    if v.dtype != torch.bfloat16 or v.dim() != 2 or not v.is_cuda or not v.is_contiguous():
        raise ValueError("v must be a contiguous CUDA bf16 tensor [T, C]")
    if z.dtype != torch.float32 or z.dim() != 2 or not z.is_cuda or not z.is_contiguous():
        raise ValueError("z must be a contiguous CUDA fp32 tensor [N, C]")
    arr, n = _specs_array(specs)
    if n % 2:
        raise ValueError("specs must hold (cond, uncond) pairs")
    T, _ = pack_size(specs)
    N = sum(int(s[1]) * int(s[2]) for s in specs[0::2])
    C = v.shape[1]
    if v.shape[0] != T or z.shape != (N, C):
        raise ValueError(f"v {tuple(v.shape)} / z {tuple(z.shape)} do not match the specs ({T}, {N}, {C})")
    check(load().mf_cfg_euler_step(_ptr(v), arr, n // 2, C, float(guidance), float(dt), _ptr(z),
                                   _stream_ptr(stream)), "mf_cfg_euler_step")
    return z


def _check_rows(name, t, T=None, Dm=None):
    torch = _torch()
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 2:
        raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [rows, Dm]")
    if (T is not None and t.shape[0] != T) or (Dm is not None and t.shape[1] != Dm):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected ({T}, {Dm})")


def adaln_modulate(x, cu_seqlens, shift, scale, eps: float = 1e-6, y=None, stream=None):
    """LN(x) (1 + scale_s) + shift_s for every token of sample s (bf16 [T, Dm])."""
    torch = _torch()
    _check_rows("x", x)
    T, Dm = x.shape
    n = cu_seqlens.numel() - 1
    _check_rows("shift", shift, n, Dm)
    _check_rows("scale", scale, n, Dm)
    y = torch.empty_like(x) if y is None else y
    _check_rows("y", y, T, Dm)
    check(load().mf_adaln_modulate(_ptr(x), _ptr(cu_seqlens), n, T, Dm, _ptr(shift), _ptr(scale),
                                   float(eps), _ptr(y), _stream_ptr(stream)), "mf_adaln_modulate")
    return y


def gated_residual(x, h, cu_seqlens, gate, out=None, stream=None):
    """x + gate_s * h for every token of sample s (bf16 [T, Dm])."""
    torch = _torch()
    _check_rows("x", x)
    T, Dm = x.shape
    n = cu_seqlens.numel() - 1
    _check_rows("h", h, T, Dm)
    _check_rows("gate", gate, n, Dm)
    out = torch.empty_like(x) if out is None else out
    _check_rows("out", out, T, Dm)
    check(load().mf_gated_residual(_ptr(x), _ptr(h), _ptr(cu_seqlens), n, T, Dm, _ptr(gate),
                                   _ptr(out), _stream_ptr(stream)), "mf_gated_residual")
    return out


def get_status(ws, stream=None) -> None:
    """Synchronise and raise MFError if the last call on this workspace recorded a
    device-side error (malformed cu_seqlens, a wait that ran out)."""
    check(load().mf_get_status(_ptr(ws), _stream_ptr(stream)), "device status")


def noalloc_get_status(stream=None) -> None:
    """Synchronise and raise MFError if the last varlen_attn_fwd_noalloc call on
    the current device recorded a device-side error (its status word lives in the
    library's fixed scratch array)."""
    check(load().mf_noalloc_get_status(_stream_ptr(stream)), "device status (noalloc)")


def timing_enable(on: bool = True) -> None:
    """Bracket every kernel launch of the library with CUDA events (opt-in)."""
    check(load().mf_timing_enable(1 if on else 0), "mf_timing_enable")


def timing_reset() -> None:
    check(load().mf_timing_reset(), "mf_timing_reset")


def timing_read() -> dict:
    """{kernel name: (total device ms, launches)} since the last reset (syncs)."""
    from ._lib import KERNELS
    out = {}
    for i, name in enumerate(KERNELS):
        ms, n = ctypes.c_double(), ctypes.c_int64()
        check(load().mf_timing_read(i, ctypes.byref(ms), ctypes.byref(n)), "mf_timing_read")
        out[name] = (ms.value, n.value)
    return out
