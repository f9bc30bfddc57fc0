"""The forward with the 2D RoPE applied on the attention kernel's tile load
(mf_varlen_attn_fwd_fused_rope): the same fp32 rotation and roundings as the
two-pass forward's pre-pass, so O and LSE must be bit-identical to
mf_varlen_attn_fwd's; and, on small packs, within the attention tolerances of
the FP64 oracle (paperlayer.ai summary 3.2.1; rotary positions per sample)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import check_lse, check_o, dev, f64, random_inputs

pytestmark = pytest.mark.gpu

RAGGED_SPECS = [(1, 0, 0), (7, 8, 15), (0, 8, 16), (1, 8, 16), (15, 16, 15), (0, 16, 16),
                (1, 16, 16), (0, 12, 32), (1, 16, 32), (40, 24, 40)]


def _both(mf, specs, qd, kd, vd, rope=True, scale=0.0):
    cu, pos = mf.pack(specs)
    T, max_len = mf.pack_size(specs)
    h, d = qd.shape[1], qd.shape[2]
    p = pos if rope else None
    ws_a = mf.workspace(T, len(specs), h, d, False)
    ws_b = mf.workspace(T, len(specs), h, d, False)
    o_a, lse_a = mf.varlen_attn_fwd(qd, kd, vd, cu, p, max_len, scale, ws=ws_a)
    o_b, lse_b = mf.varlen_attn_fwd_fused_rope(qd, kd, vd, cu, p, max_len, scale, ws=ws_b)
    mf.get_status(ws_a)
    mf.get_status(ws_b)
    torch.cuda.synchronize()
    return (o_a, lse_a), (o_b, lse_b), (cu, pos)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("rope", [True, False])
def test_bit_identical_to_two_pass_ragged(cuda_lib, d, rope):
    specs = RAGGED_SPECS
    T = int(oracle.pack(specs)[0][-1])
    q, k, v, _ = random_inputs(T, 3, d, 41, with_do=False)
    (o_a, l_a), (o_b, l_b), _ = _both(cuda_lib, specs, dev(q), dev(k), dev(v), rope=rope)
    assert torch.equal(o_a, o_b)
    assert torch.equal(l_a, l_b)


@pytest.mark.parametrize("d", [64, 128])
def test_oracle_parity_ragged(cuda_lib, d):
    specs = RAGGED_SPECS
    cu_ref, pos_ref = oracle.pack(specs)
    T = int(cu_ref[-1])
    q, k, v, _ = random_inputs(T, 2, d, 43, with_do=False)
    mf = cuda_lib
    cu, pos = mf.pack(specs)
    _, max_len = mf.pack_size(specs)
    ws = mf.workspace(T, len(specs), 2, d, False)
    o, lse = mf.varlen_attn_fwd_fused_rope(dev(q), dev(k), dev(v), cu, pos, max_len, ws=ws)
    mf.get_status(ws)
    f = synth.bf16_bits_to_f64
    o_ref, lse_ref = oracle.attn_fwd(f(q), f(k), f(v), cu_ref, pos_ref)
    check_o(f64(o), o_ref)
    check_lse(lse.cpu().numpy(), lse_ref)


def test_explicit_scale_and_large_values(cuda_lib):
    """Per-head scales up to 2 (logit std up to 4) and an explicit softmax scale."""
    specs = [(64, 16, 16), (100, 8, 40), (0, 3, 5)]
    T = int(oracle.pack(specs)[0][-1])
    s = np.array([0.5, 2.0, 1.3])
    q = dev(synth.normal_bf16_bits(6, 2, (T, 3, 128), s))
    k = dev(synth.normal_bf16_bits(6, 3, (T, 3, 128), s[::-1].copy()))
    v = dev(synth.normal_bf16_bits(6, 4, (T, 3, 128), s))
    (o_a, l_a), (o_b, l_b), _ = _both(cuda_lib, specs, q, k, v, scale=0.17)
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b)


@pytest.mark.parametrize("name", ["mixed_50k", "extreme_aspect", "cfg_2048", "single_1024"])
def test_bit_identical_full_size(cuda_lib, name):
    """The workloads at full size (24 heads x 128): fused and two-pass forwards agree
    bit for bit on every output row (inputs: seeded N(0, 1) bf16 made on the device)."""
    wl = synth.workload(name)
    T = int(sum(wl.lengths))
    g = torch.Generator(device="cuda").manual_seed(7)
    shape = (T, wl.heads, wl.head_dim)
    q, k, v = (torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    (o_a, l_a), (o_b, l_b), _ = _both(cuda_lib, wl.specs, q, k, v)
    assert torch.equal(o_a, o_b)
    assert torch.equal(l_a, l_b)


def test_position_outside_table_is_reported(cuda_lib):
    """A coordinate outside [0, min(max_len, T)) is an argument error recorded in the
    workspace (read as 0 in the kernel, so nothing is accessed out of range); the
    next call with valid positions runs normally."""
    mf = cuda_lib
    specs = [(3, 4, 5), (0, 6, 6)]
    cu, pos = mf.pack(specs)
    T, max_len = mf.pack_size(specs)
    q, k, v, _ = random_inputs(T, 2, 64, 47, with_do=False)
    qd, kd, vd = dev(q), dev(k), dev(v)
    ws = mf.workspace(T, len(specs), 2, 64, False)
    for bad in (max_len, -1, 1 << 20):
        p = pos.clone()
        p[5, 1] = bad
        mf.varlen_attn_fwd_fused_rope(qd, kd, vd, cu, p, max_len, ws=ws)
        with pytest.raises(mf.MFError) as ei:
            mf.get_status(ws)
        assert ei.value.status == 1  # MF_ERR_INVALID_ARG
    o_b, l_b = mf.varlen_attn_fwd_fused_rope(qd, kd, vd, cu, pos, max_len, ws=ws)
    mf.get_status(ws)
    o_a, l_a = mf.varlen_attn_fwd(qd, kd, vd, cu, pos, max_len)
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b)


def test_fp16_range_flag(cuda_lib):
    """A rotated value or V outside fp16's range is reported as by the two-pass
    forward (MF_ERR_OVERFLOW)."""
    mf = cuda_lib
    specs = [(5, 4, 4)]
    cu, pos = mf.pack(specs)
    T, max_len = mf.pack_size(specs)
    q, k, v, _ = random_inputs(T, 1, 64, 48, with_do=False)
    vd = dev(v)
    vd[3, 0, 7] = 1.0e5
    ws = mf.workspace(T, 1, 1, 64, False)
    mf.varlen_attn_fwd_fused_rope(dev(q), dev(k), vd, cu, pos, max_len, ws=ws)
    with pytest.raises(mf.MFError) as ei:
        mf.get_status(ws)
    assert ei.value.status == 3  # MF_ERR_OVERFLOW


def test_empty_and_zero_length_samples(cuda_lib):
    mf = cuda_lib
    specs = [(0, 0, 0), (2, 3, 3), (0, 0, 0)]
    cu, pos = mf.pack(specs)
    T, max_len = mf.pack_size(specs)
    q, k, v, _ = random_inputs(T, 1, 128, 49, with_do=False)
    (o_a, l_a), (o_b, l_b), _ = _both(mf, specs, dev(q), dev(k), dev(v))
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b)
    cu0 = torch.zeros(2, dtype=torch.int32, device="cuda")
    e = torch.empty((0, 1, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = mf.varlen_attn_fwd_fused_rope(e, e, e, cu0, None, 0)
    assert o.shape == (0, 1, 64) and lse.shape == (1, 0)
