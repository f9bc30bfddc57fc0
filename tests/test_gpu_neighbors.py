"""GPU parity of the attention's memory-bound neighbours, through the C-ABI
binding, against the FP64 oracle on the same seeded inputs: the packed-CFG
rectified-flow Euler step, the adaptive LayerNorm modulation and the gated
residual.

Tolerances, derived from the kernels' arithmetic:
  CFG step (fp32 out): fmaf(dt, fmaf(g, v_c - v_u, v_u), z) rounds twice (v_c - v_u of
      two bf16 values is exact in fp32), so |err| <= 2^-22 (|z'| + |dt| (|v_u| + |g| |v_c - v_u|)).
  adaLN (bf16 out): fp32 streamed mean / variance (chunk statistics merged
      pairwise) and rsqrt, then one bf16 rounding:
      |err| <= 1 bf16 ulp of the result + 1e-4.
  gated residual (bf16 out): one fp32 FMA, then one bf16 rounding: |err| <= 1 bf16 ulp.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_ulp, dev, f64

pytestmark = pytest.mark.gpu

S_V, S_Z, S_X, S_SHIFT, S_SCALE, S_H, S_GATE = 30, 31, 32, 33, 34, 35, 36


def _cfg_case(specs, C, seed=0):
    T = int(oracle.pack(specs)[0][-1])
    N = sum(s[1] * s[2] for s in specs[0::2])
    vb = synth.normal_bf16_bits(seed, S_V, (T, C))
    z = synth.normal_f64(seed, S_Z, N * C).astype(np.float32).reshape(N, C)
    return vb, z


CFG_SPECS = {
    "hand_sized": [(1, 1, 2), (2, 1, 2)],
    "cfg_2048": synth.cfg_2048().specs,
    "several_pairs_with_empties": [(3, 0, 5), (1, 0, 5), (0, 2, 3), (7, 2, 3), (5, 4, 4), (0, 4, 4),
                                   (9, 1, 1), (2, 1, 1)],
}


@pytest.mark.parametrize("name", list(CFG_SPECS))
@pytest.mark.parametrize("g", [0.0, 1.0, 4.5])
def test_cfg_euler_step(cuda_lib, name, g):
    mf = cuda_lib
    specs = CFG_SPECS[name]
    C, dt = 64 if name == "cfg_2048" else 16, 0.0625
    vb, z = _cfg_case(specs, C)
    zd = torch.from_numpy(z.copy()).cuda()
    mf.cfg_euler_step(dev(vb), specs, g, dt, zd)
    torch.cuda.synchronize()
    got = zd.cpu().numpy().astype(np.float64)
    v = synth.bf16_bits_to_f64(vb)
    ref = oracle.cfg_euler(v, specs, g, dt, z.astype(np.float64))
    # bound terms from the oracle's own inputs
    cu, _ = oracle.pack(specs)
    vc = np.concatenate([v[cu[2 * p] + specs[2 * p][0]: cu[2 * p] + specs[2 * p][0] + specs[2 * p][1] * specs[2 * p][2]]
                         for p in range(len(specs) // 2)] or [np.zeros((0, C))])
    vu = np.concatenate([v[cu[2 * p + 1] + specs[2 * p + 1][0]: cu[2 * p + 1] + specs[2 * p + 1][0] + specs[2 * p][1] * specs[2 * p][2]]
                         for p in range(len(specs) // 2)] or [np.zeros((0, C))])
    bound = 2.0 ** -22 * (np.abs(ref) + dt * (np.abs(vu) + abs(g) * np.abs(vc - vu))) + 1e-30
    assert np.all(np.abs(got - ref) <= bound), np.abs(got - ref).max()


def test_cfg_euler_two_steps_in_place(cuda_lib):
    """Two calls in a row on the same z: the state the second step starts from is
    the first step's output."""
    mf = cuda_lib
    specs = CFG_SPECS["several_pairs_with_empties"]
    vb, z = _cfg_case(specs, 8, seed=3)
    zd = torch.from_numpy(z.copy()).cuda()
    vd = dev(vb)
    mf.cfg_euler_step(vd, specs, 3.0, 0.1, zd)
    mid = zd.cpu().numpy().astype(np.float64)
    mf.cfg_euler_step(vd, specs, 3.0, 0.1, zd)
    ref = oracle.cfg_euler(synth.bf16_bits_to_f64(vb), specs, 3.0, 0.1, mid)
    assert np.abs(zd.cpu().numpy() - ref).max() <= 1e-5


def _rows_case(lens, Dm, seed=0):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, n = int(cu[-1]), len(lens)
    return (cu, synth.normal_bf16_bits(seed, S_X, (T, Dm)), synth.normal_bf16_bits(seed, S_SHIFT, (n, Dm)),
            synth.normal_bf16_bits(seed, S_SCALE, (n, Dm)), synth.normal_bf16_bits(seed, S_H, (T, Dm)),
            synth.normal_bf16_bits(seed, S_GATE, (n, Dm)))


ROW_CASES = {
    "tiny_pack_dm64": (synth.tiny().lengths, 64),
    "zero_length_samples_dm8": ([3, 0, 5, 0, 0, 1], 8),
    "one_row_dm4096": ([1], 4096),
    "wide_rows_dm6144": ([3, 2], 6144),
    "ragged_dm1032": ([17, 1, 64, 5], 1032),
    "mixed_50k_dm3072": (synth.mixed_50k().lengths, 3072),
}


@pytest.mark.parametrize("name", list(ROW_CASES))
def test_adaln_modulate(cuda_lib, name):
    mf = cuda_lib
    lens, Dm = ROW_CASES[name]
    cu, xb, shb, scb, _, _ = _rows_case(lens, Dm)
    cud = torch.from_numpy(cu.astype(np.int32)).cuda()
    y = mf.adaln_modulate(dev(xb), cud, dev(shb), dev(scb), eps=1e-6)
    torch.cuda.synchronize()
    f = synth.bf16_bits_to_f64
    ref = oracle.adaln(f(xb), cu, f(shb), f(scb), 1e-6)
    err = np.abs(f64(y) - ref)
    assert np.all(err <= bf16_ulp(ref) + 1e-4), err.max()


def test_adaln_in_place(cuda_lib):
    mf = cuda_lib
    cu, xb, shb, scb, _, _ = _rows_case([9, 4], 256, seed=5)
    x = dev(xb)
    cud = torch.from_numpy(cu.astype(np.int32)).cuda()
    mf.adaln_modulate(x, cud, dev(shb), dev(scb), eps=1e-6, y=x)
    f = synth.bf16_bits_to_f64
    ref = oracle.adaln(f(xb), cu, f(shb), f(scb), 1e-6)
    assert np.all(np.abs(f64(x) - ref) <= bf16_ulp(ref) + 1e-4)


@pytest.mark.parametrize("name", list(ROW_CASES))
def test_gated_residual(cuda_lib, name):
    mf = cuda_lib
    lens, Dm = ROW_CASES[name]
    cu, xb, _, _, hb, gb = _rows_case(lens, Dm, seed=1)
    cud = torch.from_numpy(cu.astype(np.int32)).cuda()
    out = mf.gated_residual(dev(xb), dev(hb), cud, dev(gb))
    torch.cuda.synchronize()
    f = synth.bf16_bits_to_f64
    ref = oracle.gated_residual(f(xb), f(hb), cu, f(gb))
    assert np.all(np.abs(f64(out) - ref) <= bf16_ulp(ref)), np.abs(f64(out) - ref).max()


def test_gated_residual_in_place(cuda_lib):
    mf = cuda_lib
    cu, xb, _, _, hb, gb = _rows_case([2, 0, 6], 64, seed=2)
    x = dev(xb)
    cud = torch.from_numpy(cu.astype(np.int32)).cuda()
    mf.gated_residual(x, dev(hb), cud, dev(gb), out=x)
    f = synth.bf16_bits_to_f64
    ref = oracle.gated_residual(f(xb), f(hb), cu, f(gb))
    assert np.all(np.abs(f64(x) - ref) <= bf16_ulp(ref))
