"""A pack past 2^31 elements per tensor: 700 images of 32 x 32 latents (716,800
tokens) at 24 heads x 128, so q, k, v, O, dQ, dK, dV each hold 2.2e9 bf16 values
and every element offset past the first 2^31 needs 64-bit arithmetic (the
stored-dS array holds 35 GB).  The forward and the stored-dS backward run on the
whole pack; the first sample and the last one (whose rows all lie past 2^31
elements) are compared with the FP64 oracle run on that sample alone
(paperlayer.ai summary 3.2.1: attention stays within each packed sample, so a
sample's outputs depend on its own tokens only).  The rotate-on-load forward must
equal the two-pass one bit for bit; the 8-bit forward gets a coarse check."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import check_grad, check_lse, check_o, f64

pytestmark = pytest.mark.gpu

N_IMG, SIDE, HEADS, D = 700, 32, 24, 128


def test_pack_beyond_2_31_elements(cuda_lib):
    mf = cuda_lib
    specs = [(0, SIDE, SIDE)] * N_IMG
    T, max_len = mf.pack_size(specs)
    L = SIDE * SIDE
    assert T == N_IMG * L and T * HEADS * D > 2 ** 31
    cu, pos = mf.pack(specs)
    g = torch.Generator(device="cuda").manual_seed(21)
    shape = (T, HEADS, D)
    q, k, v, do = (torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
                   for _ in range(4))
    ws = mf.workspace(T, N_IMG, HEADS, D, True, store_ds_max_len=max_len)
    o, lse = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len, ws=ws)
    mf.get_status(ws)
    dq, dk, dv = mf.varlen_attn_bwd(q, k, v, o, lse, do, cu, pos, max_len, ws=ws, after_fwd=True)
    mf.get_status(ws)
    torch.cuda.synchronize()
    cu_1, pos_1 = oracle.pack([(0, SIDE, SIDE)])
    bits = synth.torch_to_bits
    f = synth.bf16_bits_to_f64
    for s in (0, N_IMG - 1):
        rows = slice(s * L, (s + 1) * L)
        qs, ks, vs, dos = (f(bits(t[rows].contiguous())) for t in (q, k, v, do))
        o_ref, lse_ref = oracle.attn_fwd(qs, ks, vs, cu_1, pos_1)
        check_o(f64(o[rows].contiguous()), o_ref)
        check_lse(lse[:, rows].cpu().numpy(), lse_ref)
        g_ref = oracle.attn_bwd(qs, ks, vs, dos, cu_1, pos_1)
        for name, gg, r in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref):
            check_grad(f64(gg[rows].contiguous()), r, f"{name} of sample {s}")
    # the rotate-on-load forward: bit for bit the two-pass one, over the whole pack
    o_r, lse_r = mf.varlen_attn_fwd_fused_rope(q, k, v, cu, pos, max_len, ws=ws)
    mf.get_status(ws)
    assert torch.equal(o_r, o) and torch.equal(lse_r, lse)
    # the 8-bit forward: a coarse check of its offsets past 2^31 elements (its error
    # bounds are checked on smaller packs): within 0.05 of the 16-bit O, whose
    # entries here are of order 0.1
    o8, lse8 = mf.varlen_attn_fwd_fp8(q, k, v, cu, pos, max_len, ws=ws)
    mf.get_status(ws)
    rows = slice((N_IMG - 1) * L, N_IMG * L)
    assert (o8[rows].float() - o[rows].float()).abs().max().item() <= 0.05
    assert (lse8[:, rows] - lse[:, rows]).abs().max().item() <= 0.05
