"""Failure handling and out-of-bounds evidence on the GPU, without a fault.

- The time-out path: a test hook (mf_test_varlen_attn_fwd_stalled) makes one wait
  inside the attention kernel run out after a short limit.  The kernel must record
  MF_ERR_TIMEOUT, let its copies land, free its tensor memory and exit; the
  context must stay usable, and the next call must be correct.
- Guard bands: every output (O, LSE, dQ, dK, dV, the 8-bit, rotate-on-load and
  allocation-free forwards' outputs, the neighbours' outputs) and the caller's workspace are
  views into larger buffers whose head and tail hold a known bit pattern.  After
  the calls on ragged packs (last tiles cut short, zero-length and one-token
  samples, a short sample at the very end of the pack) the patterns must be
  untouched: no kernel writes outside its outputs.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import check_grad, check_lse, check_o, dev, f64, random_inputs

pytestmark = pytest.mark.gpu

GUARD = 512  # elements before and after each output (1 KB of bf16, 2 KB of fp32)
PAT16, PAT32 = 0x5A5A, 0x5A5A5A5A
# ragged: a one-token sample, lengths around the 128-row tiles, an empty sample,
# and a 3-token sample last, so the pack's final tile is almost all past its end
SPECS = [(1, 0, 0), (7, 8, 15), (0, 0, 0), (1, 8, 16), (15, 16, 15), (40, 24, 40), (3, 0, 0)]


def _guarded(shape, dtype):
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
    if dtype.itemsize == 2:
        buf.view(torch.int16).fill_(PAT16)
    elif dtype.itemsize == 4:
        buf.view(torch.int32).fill_(PAT32)
    else:
        buf.view(torch.uint8).fill_(0x5A)
    return buf, buf[GUARD:GUARD + n].view(shape)


def _intact(buf, what):
    torch.cuda.synchronize()
    n = buf.numel() - 2 * GUARD
    if buf.dtype.itemsize == 2:
        bits, pat = buf.view(torch.int16), PAT16
    elif buf.dtype.itemsize == 4:
        bits, pat = buf.view(torch.int32), PAT32
    else:
        bits, pat = buf.view(torch.uint8), 0x5A
    head, tail = bits[:GUARD], bits[GUARD + n:]
    assert bool((head == pat).all()), f"{what}: written before its start"
    assert bool((tail == pat).all()), f"{what}: written past its end"


def _guarded_ws(T, n, h, d, bwd):
    import packed_resolution_diffusion_pack_b300 as mf
    nbytes = mf.attn_workspace_bytes(T, n, h, d, bwd)
    buf, ws = _guarded((nbytes,), torch.uint8)
    assert ws.data_ptr() % 256 == 0
    return buf, ws


@pytest.mark.parametrize("d", [64, 128])
def test_outputs_and_workspace_keep_their_guard_bands(cuda_lib, d):
    mf = cuda_lib
    h = 3
    cu, pos = mf.pack(SPECS)
    T, max_len = mf.pack_size(SPECS)
    n = len(SPECS)
    q, k, v, do = (dev(x) for x in random_inputs(T, h, d, 81))
    bo, o = _guarded((T, h, d), torch.bfloat16)
    bl, lse = _guarded((h, T), torch.float32)
    bwf, wsf = _guarded_ws(T, n, h, d, False)
    mf.varlen_attn_fwd(q, k, v, cu, pos, max_len, o=o, lse=lse, ws=wsf)
    mf.get_status(wsf)
    for b, w in ((bo, "O"), (bl, "LSE"), (bwf, "forward workspace")):
        _intact(b, w)
    bq, dq = _guarded((T, h, d), torch.bfloat16)
    bk, dk = _guarded((T, h, d), torch.bfloat16)
    bv, dv = _guarded((T, h, d), torch.bfloat16)
    bwb, wsb = _guarded_ws(T, n, h, d, True)
    mf.varlen_attn_bwd(q, k, v, o, lse, do, cu, pos, max_len, dq=dq, dk=dk, dv=dv, ws=wsb)
    mf.get_status(wsb)
    for b, w in ((bq, "dQ"), (bk, "dK"), (bv, "dV"), (bwb, "backward workspace")):
        _intact(b, w)
    # the outputs themselves are right
    f = synth.bf16_bits_to_f64
    cu_r, pos_r = oracle.pack(SPECS)
    qb, kb, vb, dob = (synth.torch_to_bits(x.cpu()) for x in (q, k, v, do))
    o_ref, lse_ref = oracle.attn_fwd(f(qb), f(kb), f(vb), cu_r, pos_r)
    check_o(f64(o), o_ref)
    check_lse(lse.cpu().numpy(), lse_ref)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv),
                          oracle.attn_bwd(f(qb), f(kb), f(vb), f(dob), cu_r, pos_r)):
        check_grad(f64(g), r, name)


def test_fp8_and_noalloc_forwards_keep_their_guard_bands(cuda_lib):
    mf = cuda_lib
    h, d = 2, 128
    cu, pos = mf.pack(SPECS)
    T, max_len = mf.pack_size(SPECS)
    q, k, v, _ = (dev(x) if x is not None else None for x in random_inputs(T, h, d, 82, False))
    bo, o = _guarded((T, h, d), torch.bfloat16)
    bl, lse = _guarded((h, T), torch.float32)
    bw, ws = _guarded_ws(T, len(SPECS), h, d, False)
    mf.varlen_attn_fwd_fp8(q, k, v, cu, pos, max_len, o=o, lse=lse, ws=ws)
    mf.get_status(ws)
    for b, w in ((bo, "8-bit O"), (bl, "8-bit LSE"), (bw, "8-bit workspace")):
        _intact(b, w)
    bo2, o2 = _guarded((T, h, d), torch.bfloat16)
    bl2, lse2 = _guarded((h, T), torch.float32)
    mf.varlen_attn_fwd_noalloc(q, k, v, cu, pos, max_len, o=o2, lse=lse2)
    mf.noalloc_get_status()
    _intact(bo2, "allocation-free O")
    _intact(bl2, "allocation-free LSE")


@pytest.mark.parametrize("d", [64, 128])
def test_fused_rope_forward_keeps_its_guard_bands(cuda_lib, d):
    """The rotate-on-load forward writes O, LSE and its (cos, sin) table in the
    workspace, and nothing around them; its outputs equal the two-pass forward's."""
    mf = cuda_lib
    h = 2
    cu, pos = mf.pack(SPECS)
    T, max_len = mf.pack_size(SPECS)
    q, k, v, _ = (dev(x) if x is not None else None for x in random_inputs(T, h, d, 83, False))
    bo, o = _guarded((T, h, d), torch.bfloat16)
    bl, lse = _guarded((h, T), torch.float32)
    bw, ws = _guarded_ws(T, len(SPECS), h, d, False)
    mf.varlen_attn_fwd_fused_rope(q, k, v, cu, pos, max_len, o=o, lse=lse, ws=ws)
    mf.get_status(ws)
    for b, w in ((bo, "fused O"), (bl, "fused LSE"), (bw, "fused workspace")):
        _intact(b, w)
    o_ref, lse_ref = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_neighbours_keep_their_guard_bands(cuda_lib):
    mf = cuda_lib
    lens = [1, 0, 37, 300, 5]
    T, Dm, n = sum(lens), 136, len(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    x = dev(synth.normal_bf16_bits(3, 30, (T, Dm)))
    hh = dev(synth.normal_bf16_bits(3, 31, (T, Dm)))
    vec = dev(synth.normal_bf16_bits(3, 32, (n, Dm)))
    by, y = _guarded((T, Dm), torch.bfloat16)
    mf.adaln_modulate(x, cu, vec, vec, 1e-6, y=y)
    _intact(by, "adaLN output")
    bg, g = _guarded((T, Dm), torch.bfloat16)
    mf.gated_residual(x, hh, cu, vec, out=g)
    _intact(bg, "gated residual output")
    specs = [(3, 5, 7), (0, 5, 7), (1, 2, 3), (4, 2, 3)]
    Tc, _ = mf.pack_size(specs)
    C = 16
    vv = dev(synth.normal_bf16_bits(3, 33, (Tc, C)))
    N = 5 * 7 + 2 * 3
    bz, z = _guarded((N, C), torch.float32)
    z.zero_()
    mf.cfg_euler_step(vv, specs, 3.0, 0.1, z)
    _intact(bz, "CFG Euler latent")


@pytest.mark.parametrize("d", [64, 128])
def test_wait_that_runs_out_is_reported_and_the_next_call_is_right(cuda_lib, d):
    """The stalled forward returns MF_ERR_TIMEOUT through mf_get_status, writes
    nothing, and leaves the context usable: a normal call on the same workspace
    and one on a fresh workspace both match the oracle."""
    mf = cuda_lib
    lib = mf.load()
    h = 2
    cu, pos = mf.pack(SPECS)
    T, max_len = mf.pack_size(SPECS)
    n = len(SPECS)
    q, k, v, _ = (dev(x) if x is not None else None for x in random_inputs(T, h, d, 83, False))
    bo, o = _guarded((T, h, d), torch.bfloat16)
    bl, lse = _guarded((h, T), torch.float32)
    ws = mf.workspace(T, n, h, d, False)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.mf_test_varlen_attn_fwd_stalled(p(q), p(k), p(v), p(cu), p(pos), n, T, max_len, h, d,
                                             0.0, p(o), p(lse), p(ws), ws.numel(), 20000, stream)
    assert rc == 0, mf.STATUS_NAMES.get(rc, rc)
    with pytest.raises(mf.MFError) as ei:
        mf.get_status(ws)
    assert ei.value.status == 5  # MF_ERR_TIMEOUT
    # nothing was written: every element still holds the pattern
    torch.cuda.synchronize()
    assert bool((bo.view(torch.int16) == PAT16).all()) and bool((bl.view(torch.int32) == PAT32).all())
    # out-of-range limits are refused on the host
    for bad in (0, 1000001):
        assert lib.mf_test_varlen_attn_fwd_stalled(p(q), p(k), p(v), p(cu), p(pos), n, T, max_len,
                                                   h, d, 0.0, p(o), p(lse), p(ws), ws.numel(),
                                                   bad, stream) == 1
    f = synth.bf16_bits_to_f64
    cu_r, pos_r = oracle.pack(SPECS)
    qb, kb, vb = (synth.torch_to_bits(x.cpu()) for x in (q, k, v))
    o_ref, lse_ref = oracle.attn_fwd(f(qb), f(kb), f(vb), cu_r, pos_r)
    for w in (ws, mf.workspace(T, n, h, d, False)):
        o2, lse2 = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len, ws=w)
        mf.get_status(w)
        check_o(f64(o2), o_ref)
        check_lse(lse2.cpu().numpy(), lse_ref)


def test_backward_wait_that_runs_out_is_reported_and_the_next_call_is_right(cuda_lib):
    """The same for the backward's attention kernel: MF_ERR_TIMEOUT, dK and dV
    untouched, then a normal backward on the same workspace matches the oracle."""
    mf = cuda_lib
    lib = mf.load()
    h, d = 2, 128
    cu, pos = mf.pack(SPECS)
    T, max_len = mf.pack_size(SPECS)
    n = len(SPECS)
    q, k, v, do = (dev(x) for x in random_inputs(T, h, d, 84))
    o, lse = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len)
    dq = torch.empty_like(q)
    bk, dk = _guarded((T, h, d), torch.bfloat16)
    bv, dv = _guarded((T, h, d), torch.bfloat16)
    ws = mf.workspace(T, n, h, d, True)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.mf_test_varlen_attn_bwd_stalled(p(q), p(k), p(v), p(o), p(lse), p(do), p(cu), p(pos),
                                             n, T, max_len, h, d, 0.0, p(dq), p(dk), p(dv), p(ws),
                                             ws.numel(), 20000, stream)
    assert rc == 0, mf.STATUS_NAMES.get(rc, rc)
    with pytest.raises(mf.MFError) as ei:
        mf.get_status(ws)
    assert ei.value.status == 5  # MF_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert bool((bk.view(torch.int16) == PAT16).all()) and bool((bv.view(torch.int16) == PAT16).all())
    dq2, dk2, dv2 = mf.varlen_attn_bwd(q, k, v, o, lse, do, cu, pos, max_len, ws=ws)
    mf.get_status(ws)
    f = synth.bf16_bits_to_f64
    cu_r, pos_r = oracle.pack(SPECS)
    qb, kb, vb, dob = (synth.torch_to_bits(x.cpu()) for x in (q, k, v, do))
    for name, g, r in zip(("dq", "dk", "dv"), (dq2, dk2, dv2),
                          oracle.attn_bwd(f(qb), f(kb), f(vb), f(dob), cu_r, pos_r)):
        check_grad(f64(g), r, name)
