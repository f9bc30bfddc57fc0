"""mf_varlen_attn_fwd_noalloc through the C ABI (GPU).

The call is for users who cannot allocate device memory themselves, for example
a plugin inside a framework that owns the allocator and hands it only inputs and
outputs.  Its scratch is a fixed device array inside the library.  These checks
compare it with mf_varlen_attn_fwd given a caller workspace, on two calls in a
row.  Between the two calls the array still holds the first call's data.  The
checks also cover the size limit.  This file is named to be collected last.  It
passes alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import check_lse, check_o, dev, f64

pytestmark = pytest.mark.gpu

PACKS = [
    ([(5, 4, 6), (7, 8, 8), (3, 2, 16)], 2, 64, 31),
    ([(1, 0, 0), (40, 24, 40), (0, 8, 16), (15, 16, 15)], 3, 128, 32),
]


def _inputs(specs, heads, d, seed):
    T = sum(t + h * w for t, h, w in specs)
    shape = (T, heads, d)
    return [dev(synth.normal_bf16_bits(seed, s, shape)) for s in (2, 3, 4)], T


def test_noalloc_matches_workspace_forward_twice():
    import packed_resolution_diffusion_pack_b300 as mf
    lib = mf.load()
    for specs, heads, d, seed in PACKS:  # two calls in a row, different packs
        (q, k, v), T = _inputs(specs, heads, d, seed)
        cu, pos = mf.pack(specs)
        _, max_len = mf.pack_size(specs)
        o_ref, lse_ref = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len)
        o = torch.empty_like(q)
        lse = torch.empty((heads, T), dtype=torch.float32, device="cuda")
        p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
        rc = lib.mf_varlen_attn_fwd_noalloc(p(q), p(k), p(v), p(cu), p(pos), len(specs), T,
                                            max_len, heads, d, 0.0, p(o), p(lse),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, mf.STATUS_NAMES.get(rc, rc)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: within the parity tolerance, and in
        # fact bit for bit
        check_o(f64(o), f64(o_ref), "noalloc O")
        check_lse(lse.cpu().numpy(), lse_ref.cpu().numpy())
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import packed_resolution_diffusion_pack_b300 as mf
    lib = mf.load()
    max_elems = 4194304
    heads, d = 64, 128
    T = max_elems // (heads * d) + 1  # one token over the limit
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: rejected before any launch
    rc = lib.mf_varlen_attn_fwd_noalloc(p, p, p, p, None, 1, T, T, heads, d, 0.0, p, p, None)
    assert rc == 2  # MF_ERR_UNSUPPORTED
    rc = lib.mf_varlen_attn_fwd_noalloc(p, p, p, p, None, 4097, 8, 8, 1, 64, 0.0, p, p, None)
    assert rc == 2


def test_noalloc_python_binding():
    import packed_resolution_diffusion_pack_b300 as mf
    specs, heads, d, seed = PACKS[0]
    (q, k, v), T = _inputs(specs, heads, d, seed)
    cu, pos = mf.pack(specs)
    _, max_len = mf.pack_size(specs)
    o, lse = mf.varlen_attn_fwd_noalloc(q, k, v, cu, pos, max_len)
    o_ref, lse_ref = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert np.isfinite(lse.cpu().numpy()).all()


def test_noalloc_status_reports_device_errors():
    """The status word in the scratch array reports what the last allocation-free
    forward found on the device: a malformed cu_seqlens is MF_ERR_BAD_SEQLENS,
    and the next well-formed call clears it."""
    import packed_resolution_diffusion_pack_b300 as mf
    T = 64
    q = dev(synth.normal_bf16_bits(0, 2, (T, 1, 64)))
    bad = torch.tensor([0, 40, 30], dtype=torch.int32, device="cuda")
    mf.varlen_attn_fwd_noalloc(q, q, q, bad, None, 64)
    with pytest.raises(mf.MFError) as ei:
        mf.noalloc_get_status()
    assert ei.value.status == 6  # MF_ERR_BAD_SEQLENS
    good = torch.tensor([0, 40, 64], dtype=torch.int32, device="cuda")
    o, lse = mf.varlen_attn_fwd_noalloc(q, q, q, good, None, 40)
    mf.noalloc_get_status()
    o_ref, lse_ref = mf.varlen_attn_fwd(q, q, q, good, None, 40)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
