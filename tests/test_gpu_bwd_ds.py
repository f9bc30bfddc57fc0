"""The backward's stored-dS form (a workspace of mf_attn_workspace_bytes_ds): the
dK / dV kernel also writes each (sample, head)'s scaled fp16 dS^T, and dQ is one
streaming GEMM over it.  Checked against the FP64 oracle's gradients (rcap.io
listing "native-resolution packed step": the loss is back-propagated through the
packed attention) on ragged packs, large logits, editing packs, the training
step's shared workspace and the long samples of two workloads at full size; dK
and dV must equal the recompute form's bit for bit (the same kernel computes
them), and no byte around the outputs or the workspace may change."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import check_grad, dev, f64, random_inputs

pytestmark = pytest.mark.gpu

RAGGED_SPECS = [(1, 0, 0), (7, 8, 15), (0, 8, 16), (1, 8, 16), (15, 16, 15), (0, 16, 16),
                (1, 16, 16), (0, 12, 32), (1, 16, 32), (40, 24, 40)]


def _bwd_both(mf, specs, q, k, v, do, pos3=False):
    """Forward, then the backward in both forms; returns (recompute, stored-dS)."""
    if pos3:
        cu, pos = mf.pack3d(specs)
        T, max_len = mf.pack3d_size(specs)
    else:
        cu, pos = mf.pack(specs)
        T, max_len = mf.pack_size(specs)
    h, d = q.shape[1], q.shape[2]
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    o, lse = mf.varlen_attn_fwd(qd, kd, vd, cu, pos, max_len)
    ws_r = mf.workspace(T, len(specs), h, d, True)
    ws_s = mf.workspace(T, len(specs), h, d, True, store_ds_max_len=max_len)
    assert ws_s.numel() > ws_r.numel()
    rec = mf.varlen_attn_bwd(qd, kd, vd, o, lse, dod, cu, pos, max_len, ws=ws_r)
    mf.get_status(ws_r)
    sto = mf.varlen_attn_bwd(qd, kd, vd, o, lse, dod, cu, pos, max_len, ws=ws_s)
    mf.get_status(ws_s)
    torch.cuda.synchronize()
    return rec, sto


def _oracle_check(specs, q, k, v, do, grads, pos3=False):
    f = synth.bf16_bits_to_f64
    if pos3:
        cu_r, pos_r = oracle.pack3d(specs)
        g_ref = oracle.attn_bwd3d(f(q), f(k), f(v), f(do), cu_r, pos_r)
    else:
        cu_r, pos_r = oracle.pack(specs)
        g_ref = oracle.attn_bwd(f(q), f(k), f(v), f(do), cu_r, pos_r)
    for name, g, r in zip(("dq", "dk", "dv"), grads, g_ref):
        check_grad(f64(g), r, name)


@pytest.mark.parametrize("d", [64, 128])
def test_ragged_multi_tile(cuda_lib, d):
    T = int(oracle.pack(RAGGED_SPECS)[0][-1])
    q, k, v, do = random_inputs(T, 2, d, 61)
    rec, sto = _bwd_both(cuda_lib, RAGGED_SPECS, q, k, v, do)
    _oracle_check(RAGGED_SPECS, q, k, v, do, sto)
    assert torch.equal(rec[1], sto[1]) and torch.equal(rec[2], sto[2])


def test_large_logits(cuda_lib):
    specs = [(64, 16, 16), (100, 8, 40)]
    T = int(oracle.pack(specs)[0][-1])
    s = np.array([0.5, 2.0, 1.3])
    q = synth.normal_bf16_bits(5, 2, (T, 3, 128), s)
    k = synth.normal_bf16_bits(5, 3, (T, 3, 128), s[::-1].copy())
    v = synth.normal_bf16_bits(5, 4, (T, 3, 128), s)
    do = synth.normal_bf16_bits(5, 5, (T, 3, 128))
    rec, sto = _bwd_both(cuda_lib, specs, q, k, v, do)
    _oracle_check(specs, q, k, v, do, sto)
    assert torch.equal(rec[1], sto[1]) and torch.equal(rec[2], sto[2])


def test_editing_pack(cuda_lib):
    specs = [(7, 8, 16, 8, 16), (1, 16, 16, 12, 20), (3, 5, 7, 5, 7)]
    T = int(oracle.pack3d(specs)[0][-1])
    q, k, v, do = random_inputs(T, 2, 128, 62)
    rec, sto = _bwd_both(cuda_lib, specs, q, k, v, do, pos3=True)
    _oracle_check(specs, q, k, v, do, sto, pos3=True)
    assert torch.equal(rec[1], sto[1]) and torch.equal(rec[2], sto[2])


def test_training_step_shared_workspace(cuda_lib):
    """Forward and the stored-dS backward on one workspace (the backward reusing the
    forward's rotated operands), as the benchmarked step runs them."""
    mf = cuda_lib
    specs = RAGGED_SPECS
    cu, pos = mf.pack(specs)
    T, max_len = mf.pack_size(specs)
    q, k, v, do = random_inputs(T, 2, 128, 63)
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    ws = mf.workspace(T, len(specs), 2, 128, True, store_ds_max_len=max_len)
    o, lse = mf.varlen_attn_fwd(qd, kd, vd, cu, pos, max_len, ws=ws)
    g = mf.varlen_attn_bwd(qd, kd, vd, o, lse, dod, cu, pos, max_len, ws=ws, after_fwd=True)
    mf.get_status(ws)
    _oracle_check(specs, q, k, v, do, g)


def test_guard_bands(cuda_lib):
    """Outputs and the (larger) workspace as views into guarded buffers."""
    from test_gpu_guards import SPECS, _guarded, _guarded_ws, _intact  # noqa: F401
    mf = cuda_lib
    h, d = 2, 128
    cu, pos = mf.pack(SPECS)
    T, max_len = mf.pack_size(SPECS)
    q, k, v, do = (dev(x) for x in random_inputs(T, h, d, 64))
    o, lse = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len)
    nbytes = mf.attn_workspace_bytes_ds(T, len(SPECS), h, d, max_len)
    bw, ws = _guarded((nbytes,), torch.uint8)
    assert ws.data_ptr() % 256 == 0
    bufs = [_guarded((T, h, d), torch.bfloat16) for _ in range(3)]
    mf.varlen_attn_bwd(q, k, v, o, lse, do, cu, pos, max_len, dq=bufs[0][1], dk=bufs[1][1],
                       dv=bufs[2][1], ws=ws)
    mf.get_status(ws)
    _intact(bw, "stored-dS workspace")
    for (b, _), name in zip(bufs, ("dQ", "dK", "dV")):
        _intact(b, name)


def _full_pairs(name, pairs_fn):
    import packed_resolution_diffusion_pack_b300 as mf
    wl = synth.workload(name)
    q, k, v, do = synth.make_inputs(wl, with_do=True)
    cu, pos = mf.pack(wl.specs)
    T, max_len = wl.total, wl.max_len
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    ws = mf.workspace(T, len(wl.specs), wl.heads, wl.head_dim, True, store_ds_max_len=max_len)
    o, lse = mf.varlen_attn_fwd(qd, kd, vd, cu, pos, max_len, ws=ws)
    dq, dk, dv = mf.varlen_attn_bwd(qd, kd, vd, o, lse, dod, cu, pos, max_len, ws=ws,
                                    after_fwd=True)
    mf.get_status(ws)
    cu_r, pos_r = oracle.pack(wl.specs)
    f = synth.bf16_bits_to_f64
    for (i, a) in pairs_fn(wl):
        s, e = int(cu_r[i]), int(cu_r[i + 1])
        sl = lambda x: f(x[s:e, a:a + 1])  # noqa: E731
        g_ref = oracle.attn_bwd(sl(q), sl(k), sl(v), sl(do), np.array([0, e - s]), pos_r[s:e])
        for nm, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref):
            check_grad(f64(g[s:e, a:a + 1]), r, f"{nm} sample {i} head {a}")


def test_full_mixed_50k_long_and_short(cuda_lib):
    def pairs(wl):
        L = np.array(wl.lengths)
        return [(int(np.argmax(L)), 0), (int(np.argmax(L)), wl.heads - 1), (int(np.argmin(L)), 3)]
    _full_pairs("mixed_50k", pairs)


def test_full_extreme_aspect_big_sample(cuda_lib):
    """The 128x128 sample (about 16.5k tokens: 130 key tiles into every dQ row)."""
    def pairs(wl):
        return [(int(np.argmax(np.array(wl.lengths))), 5)]
    _full_pairs("extreme_aspect", pairs)


def test_zero_length_and_one_token_samples(cuda_lib):
    """Zero-length samples between others, one-token samples and a 3-token sample
    at the end of the pack (its last tile almost all past the pack)."""
    specs = [(1, 0, 0), (7, 8, 15), (0, 0, 0), (1, 8, 16), (15, 16, 15), (40, 24, 40), (3, 0, 0)]
    T = int(oracle.pack(specs)[0][-1])
    q, k, v, do = random_inputs(T, 2, 64, 65)
    rec, sto = _bwd_both(cuda_lib, specs, q, k, v, do)
    _oracle_check(specs, q, k, v, do, sto)
    assert torch.equal(rec[1], sto[1]) and torch.equal(rec[2], sto[2])


def test_empty_pack(cuda_lib):
    mf = cuda_lib
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    e = torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 0), dtype=torch.float32, device="cuda")
    ws = mf.workspace(0, 1, 2, 128, True, store_ds_max_len=0)
    dq, dk, dv = mf.varlen_attn_bwd(e, e, e, e, lse, e, cu, None, 0, ws=ws)
    mf.get_status(ws)
    assert dq.shape == (0, 2, 128)


def test_bad_seqlens_write_nothing(cuda_lib):
    """A malformed cu_seqlens with the stored-dS workspace: MF_ERR_BAD_SEQLENS, and no
    gradient row written."""
    from test_gpu_guards import PAT16, _guarded
    mf = cuda_lib
    T, h, d = 64, 1, 64
    q, k, v, do = (dev(x) for x in random_inputs(T, h, d, 66))
    cu_ok = torch.tensor([0, 40, 64], dtype=torch.int32, device="cuda")
    o, lse = mf.varlen_attn_fwd(q, k, v, cu_ok, None, 64)
    ws = mf.workspace(T, 2, h, d, True, store_ds_max_len=64)
    bufs = [_guarded((T, h, d), torch.bfloat16) for _ in range(3)]
    for b, _ in bufs:
        b.view(torch.int16).fill_(PAT16)
    cu_bad = torch.tensor([0, 40, 30], dtype=torch.int32, device="cuda")
    mf.varlen_attn_bwd(q, k, v, o, lse, do, cu_bad, None, 64, dq=bufs[0][1], dk=bufs[1][1],
                       dv=bufs[2][1], ws=ws)
    with pytest.raises(mf.MFError) as ei:
        mf.get_status(ws)
    assert ei.value.status == 6  # MF_ERR_BAD_SEQLENS
    torch.cuda.synchronize()
    for b, _ in bufs:
        assert bool((b.view(torch.int16) == PAT16).all())


def test_wait_that_runs_out_is_reported_and_the_next_call_is_right(cuda_lib):
    """The time-out path through both kernels of the stored-dS form (the test hook
    stalls every CTA's MMA thread): MF_ERR_TIMEOUT, no gradient written, then a normal
    backward on the same workspace matches the oracle."""
    import ctypes
    from test_gpu_guards import PAT16, SPECS, _guarded
    mf = cuda_lib
    lib = mf.load()
    h, d = 2, 128
    cu, pos = mf.pack(SPECS)
    T, max_len = mf.pack_size(SPECS)
    n = len(SPECS)
    qb, kb, vb, dob = random_inputs(T, h, d, 67)
    q, k, v, do = dev(qb), dev(kb), dev(vb), dev(dob)
    o, lse = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len)
    bufs = [_guarded((T, h, d), torch.bfloat16) for _ in range(3)]
    ws = mf.workspace(T, n, h, d, True, store_ds_max_len=max_len)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.mf_test_varlen_attn_bwd_stalled(p(q), p(k), p(v), p(o), p(lse), p(do), p(cu), p(pos),
                                             n, T, max_len, h, d, 0.0, p(bufs[0][1]),
                                             p(bufs[1][1]), p(bufs[2][1]), p(ws), ws.numel(),
                                             20000, stream)
    assert rc == 0, mf.STATUS_NAMES.get(rc, rc)
    with pytest.raises(mf.MFError) as ei:
        mf.get_status(ws)
    assert ei.value.status == 5  # MF_ERR_TIMEOUT
    torch.cuda.synchronize()
    for b, _ in bufs:
        assert bool((b.view(torch.int16) == PAT16).all())
    g = mf.varlen_attn_bwd(q, k, v, o, lse, do, cu, pos, max_len, ws=ws)
    mf.get_status(ws)
    _oracle_check(SPECS, qb, kb, vb, dob, g)
