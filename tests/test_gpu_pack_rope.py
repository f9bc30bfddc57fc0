"""GPU parity of mf_pack (bit-exact tables) and mf_rope2d_qk (within 1 bf16 ulp
of the FP64 oracle), through the C-ABI binding."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_ulp, dev, f64

pytestmark = pytest.mark.gpu

EDGE_SPECS = {
    "single_token": [(1, 0, 0)],
    "text_only": [(5, 0, 0), (17, 0, 0)],
    "image_only": [(0, 3, 7), (0, 1, 1), (0, 64, 64)],
    "zero_length_inside": [(3, 2, 2), (0, 0, 0), (0, 5, 0), (2, 0, 9), (4, 1, 3), (0, 0, 0)],
    "wide_and_tall": [(7, 1, 300), (9, 300, 1)],
    "many_samples": [(i % 5, (i * 7) % 4, (i * 3) % 6) for i in range(700)],
}


def _pack_cases():
    cases = {k: v for k, v in EDGE_SPECS.items()}
    cases["tiny"] = synth.tiny().specs
    for s in range(2):
        cases[f"mixed_50k_seed{s}"] = synth.mixed_50k(s).specs
    cases["extreme_aspect"] = synth.extreme_aspect().specs
    cases["cfg_2048"] = synth.cfg_2048().specs
    return cases


@pytest.mark.parametrize("name,specs", list(_pack_cases().items()))
def test_pack_bit_exact(cuda_lib, name, specs):
    mf = cuda_lib
    cu, pos = mf.pack(specs)
    cu_ref, pos_ref = oracle.pack(specs)
    assert np.array_equal(cu.cpu().numpy().astype(np.int64), cu_ref)
    if pos_ref.shape[0]:
        assert np.array_equal(pos.cpu().numpy().astype(np.int64), pos_ref)
    T, mx = mf.pack_size(specs)
    assert T == int(cu_ref[-1]) and mx == int(np.diff(cu_ref).max(initial=0))


def test_pack_empty(cuda_lib):
    cu, pos = cuda_lib.pack([])
    assert cu.cpu().tolist() == [0] and pos.shape == (0, 2)


@pytest.mark.parametrize("d,heads,specs", [
    (64, 2, synth.tiny().specs),
    (128, 3, [(9, 37, 5), (4, 128, 3), (0, 2, 127)]),
    (128, 1, [(3, 1, 1)]),
])
def test_rope_within_one_ulp(cuda_lib, d, heads, specs):
    mf = cuda_lib
    cu, pos = mf.pack(specs)
    _, pos_ref = oracle.pack(specs)
    T = pos_ref.shape[0]
    q = synth.normal_bf16_bits(7, synth.STREAM_Q, (T, heads, d))
    k = synth.normal_bf16_bits(7, synth.STREAM_K, (T, heads, d))
    qr, kr = mf.rope2d_qk(dev(q), dev(k), pos)
    for got, x in ((qr, q), (kr, k)):
        xf = synth.bf16_bits_to_f64(x)
        ref = oracle.rope2d(xf, pos_ref)
        err = np.abs(f64(got) - ref)
        # 1 bf16 ulp of the exact value, plus the fp32 evaluation error of the
        # rotation, bounded by 2^-20 of the pair's norm (sin/cos to ~2^-22
        # relative, two products): it only matters where x cos - y sin nearly
        # cancels to a value far below the pair's magnitude.
        norm = np.sqrt(xf[..., 0::2] ** 2 + xf[..., 1::2] ** 2).repeat(2, axis=-1)
        bound = bf16_ulp(ref) + 2.0 ** -20 * norm
        assert (err <= bound).all(), f"max err/bound {(err / bound).max()}"
        assert (err <= bf16_ulp(ref)).mean() > 0.999


def test_rope_in_place_and_single(cuda_lib):
    mf = cuda_lib
    specs = [(2, 5, 9), (1, 3, 3)]
    cu, pos = mf.pack(specs)
    _, pos_ref = oracle.pack(specs)
    T = pos_ref.shape[0]
    k = synth.normal_bf16_bits(3, synth.STREAM_K, (T, 4, 128))
    kd = dev(k)
    _, out = mf.rope2d_qk(None, kd.clone(), pos)
    _, same = mf.rope2d_qk(None, kd, pos, k_out=kd)  # in place
    torch.cuda.synchronize()
    assert torch.equal(out, same) and same.data_ptr() == kd.data_ptr()


def test_rope_text_tokens_unrotated(cuda_lib):
    mf = cuda_lib
    specs = [(11, 0, 0), (3, 0, 0)]
    cu, pos = mf.pack(specs)
    x = dev(synth.normal_bf16_bits(1, synth.STREAM_Q, (14, 2, 64)))
    y, _ = mf.rope2d_qk(x, None, pos)
    torch.cuda.synchronize()
    assert torch.equal(x, y)
