"""GPU parity of the 8-bit (E4M3) forward variant and its operand quantisation
against the oracle of the same steps (oracle.quant_e4m3, oracle.attn_fwd_e4m3),
through the C-ABI binding.

Tolerances.  Every scale is a power of two, so dividing by it is exact on both
sides: codes of values that are not rotated (V, text tokens, no-RoPE calls) are
bit-exact.  A rotated value is formed in fp32 by the kernel and in fp64 by the
oracle: there the codes agree except where the exact value sits within fp32
rounding of a rounding midpoint, where the two sides may pick the two neighbours.  The attention then differs by (i) the bf16 rounding of
O (2^-9 relative), (ii) fp32 logits and the hardware exp2 (about 2^-22 relative),
and (iii) the rare E4M3 roundings of P that (ii) tips over a midpoint, each of
which moves O by at most 2^-4 of that key's weight.  The checks are the bf16
path's: O max |d| <= 2e-2 and mean |d| <= 2e-3, LSE max |d| <= 1e-2, here against
the 8-bit oracle.

The 8-bit oracle follows the variant's own steps (128-key tiles from the sample's
first key, a running maximum raised past a margin of 8), so a step that the kernel
and that oracle got wrong in the same way would pass the comparison above.  Every
forward test therefore also gates the GPU's O and LSE against the EXACT attention
of the un-rounded operands (oracle.attn_fwd, the joint attention of paperlayer.ai
3.2.1), within the rigorous per-row bounds of e4m3_bound, which hold for any tiling
and any margin, plus the tie allowance between the kernel and exact arithmetic
on the same rounding decisions: the bf16 rounding of O (2^-9 relative, doubled to
cover fp32 accumulation and the hardware exp2) and 1e-5 absolute on O and LSE for
the fp32 arithmetic of logits, sums and logarithms.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from e4m3_bound import e4m3_attention_bounds
from gpu_util import check_lse, check_o, dev, f64, random_inputs

# tie allowance between the kernel and exact arithmetic on the same roundings
TIE_O_REL, TIE_ABS = 2.0 ** -8, 1e-5
# Statistical gates on pairs of at least 64 tokens.  The rigorous bound is loose
# (it adds every rounding's worst case), so on top of it: rounding to nearest
# leaves no systematic error, so the regression coefficient of the error on the
# exact O, alpha = <dO, O> / <O, O>, stays near zero (measured on the 8-bit
# oracle: |alpha| <= 7e-3 on the packs of this file, a slight shrinkage), and the
# relative RMS error stays near 5 % (3-9 % measured).  A 2 % scale error of O
# fails the first.
ALPHA_MAX, REL_RMS_MAX = 1.5e-2, 0.15


def check_exact_bounds(og, lg, qf, kf, vf, cu_r, pos_r, scale=None, pairs=None):
    """GPU O [T, h, d] and LSE [h, T] against the exact attention, within the
    rigorous bounds of the 8-bit steps plus the tie allowance, for every (sample,
    head) pair or the given ones.  The K and V scales are the whole head's, so the
    rotation and quant_e4m3 run on full heads (one head at a time)."""
    T, h, d = qf.shape
    sc = 1.0 / np.sqrt(d) if scale is None else scale
    if pairs is None:
        pairs = [(i, a) for i in range(len(cu_r) - 1) for a in range(h)]
    heads = {}

    def head(a):
        if a not in heads:
            qa, ka, va = qf[:, a:a + 1], kf[:, a:a + 1], vf[:, a:a + 1]
            if pos_r is None:
                qr, kr = qa, ka
            elif pos_r.shape[1] == 3:
                qr, kr = oracle.rope3d(qa, pos_r), oracle.rope3d(ka, pos_r)
            else:
                qr, kr = oracle.rope2d(qa, pos_r), oracle.rope2d(ka, pos_r)
            _, sq, _, sk, _, sv = oracle.quant_e4m3(qa, ka, va, pos_r)
            heads[a] = (qr, kr, sq, sk, sv)
        return heads[a]

    worst = 0.0
    for i, a in pairs:
        s0, s1 = int(cu_r[i]), int(cu_r[i + 1])
        if s1 == s0:
            continue
        qr, kr, sq, sk, sv = head(a)
        sl = slice(s0, s1)
        o_ex, l_ex = oracle.attn_fwd(qr[sl], kr[sl], vf[sl, a:a + 1], np.array([0, s1 - s0]), None,
                                     scale=sc)
        delta, bound = e4m3_attention_bounds(qr[sl, 0], kr[sl, 0], vf[sl, a], sq[sl, 0], sk[0],
                                             sv[0], sc, l_ex[0])
        dl = np.abs(lg[a, sl] - l_ex[0])
        assert np.all(dl <= delta + TIE_ABS + 2.0 ** -20 * np.abs(l_ex[0])), \
            f"LSE sample {i} head {a}: {dl.max():.3e} over the bound"
        do = np.abs(og[sl, a] - o_ex[:, 0])
        allow = bound + TIE_O_REL * (np.abs(o_ex[:, 0]) + bound) + TIE_ABS
        assert np.all(do <= allow), \
            f"O sample {i} head {a}: {(do - allow).max():.3e} over the bound"
        worst = max(worst, float((do / allow).max()))
        if s1 - s0 >= 64:
            e, x = og[sl, a] - o_ex[:, 0], o_ex[:, 0]
            alpha = float((e * x).sum() / (x * x).sum())
            rel = float(np.sqrt((e * e).mean() / (x * x).mean()))
            assert abs(alpha) <= ALPHA_MAX, f"O sample {i} head {a}: systematic error {alpha:+.3e}"
            assert rel <= REL_RMS_MAX, f"O sample {i} head {a}: relative RMS error {rel:.3f}"
    return worst


pytestmark = pytest.mark.gpu

SPECS = [(1, 0, 0), (7, 8, 15), (0, 8, 16), (1, 8, 16), (15, 16, 15), (1, 16, 16),
         (0, 0, 0), (40, 24, 40), (3, 1, 1)]


def _codes(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _check_codes(gpu, ref, exact, what, rotated):
    """Codes equal, or (rotated operands only) neighbours around a midpoint that
    the exact value nearly hits.  A rotated component carries an fp32 error
    relative to its pair's norm (at most 448 sqrt(2) in code units), not to itself:
    near-zero components of large pairs get that absolute allowance."""
    bad = gpu != ref
    if not rotated:
        assert not bad.any(), f"{what}: {bad.mean():.2e} of codes differ"
        return
    frac = bad.mean() if bad.size else 0.0
    assert frac <= 1e-3, f"{what}: {frac:.2e} of codes differ"
    if bad.any():
        mid = (gpu[bad] + ref[bad]) / 2
        tol = 2.0 ** -20 * (np.abs(exact[bad]) + (448 * np.sqrt(2) if what in "qk" else 0.0))
        assert np.all(np.abs(exact[bad] - mid) <= tol + 1e-30), what
        assert np.all(oracle.e4m3(mid) != mid), what  # the two are neighbours


@pytest.mark.parametrize("axes", [0, 2, 3])
def test_quant_matches_oracle(cuda_lib, axes):
    mf = cuda_lib
    specs5 = [(s[0], s[1], s[2], s[1], s[2]) for s in SPECS]
    if axes == 3:
        cu, pos = mf.pack3d(specs5)
        cu_r, pos_r = oracle.pack3d(specs5)
    else:
        cu, pos = mf.pack(SPECS)
        cu_r, pos_r = oracle.pack(SPECS)
    if axes == 0:
        pos, pos_r = None, None
    T = int(cu_r[-1])
    q, k, v, _ = random_inputs(T, 3, 128, seed=70 + axes, with_do=False)
    f = synth.bf16_bits_to_f64
    q8, k8, v8, qscale, kv_max2 = mf.quant_e4m3(dev(q), dev(k), dev(v), pos)
    torch.cuda.synchronize()
    qh, sq, kh, sk, vh, sv = oracle.quant_e4m3(f(q), f(k), f(v), pos_r)
    xq, _, xk, _, xv, _ = oracle.quant_e4m3(f(q), f(k), f(v), pos_r, round=False)
    assert np.array_equal(qscale.cpu().numpy().astype(np.float64), sq)
    mx = np.sqrt(kv_max2.cpu().numpy().astype(np.float64))
    # the scales' inputs: K's largest pair norm (fp32 sums of squares) and V's max |v|
    kmax = np.sqrt(f(k)[..., 0::2] ** 2 + f(k)[..., 1::2] ** 2).max(axis=(0, 2))
    assert np.allclose(mx[0], kmax, rtol=2e-7)
    assert np.array_equal(mx[1], np.abs(f(v)).max(axis=(0, 2)))
    for name, g, r, x in (("q", q8, qh, xq), ("k", k8, kh, xk), ("v", v8, vh, xv)):
        _check_codes(_codes(g), r, x, name, rotated=(axes != 0 and name != "v"))


def _fwd_compare(mf, specs, heads, seed, rope=True, head_scales=None, zero_rows=0, scale=0.0):
    cu, pos = mf.pack(specs)
    T, max_len = mf.pack_size(specs)
    cu_r, pos_r = oracle.pack(specs)
    q, k, v, _ = random_inputs(T, heads, 128, seed, with_do=False)
    f = synth.bf16_bits_to_f64
    qf, kf, vf = f(q), f(k), f(v)
    if head_scales is not None:
        # per-head scales on Q, K, V, the products rounded back to bf16
        qf, kf, vf = (x * s[None, :, None] for x, s in zip((qf, kf, vf), head_scales))
        q, k, v = (synth.torch_to_bits(torch.from_numpy(x).to(torch.bfloat16)) for x in (qf, kf, vf))
        qf, kf, vf = f(q), f(k), f(v)
    if zero_rows:
        rows = np.random.default_rng(seed).choice(T, zero_rows, replace=False)
        qf[rows] = 0.0
        q = synth.torch_to_bits(torch.from_numpy(qf).to(torch.bfloat16))
    ws = mf.workspace(T, len(specs), heads, 128, False)
    o, lse = mf.varlen_attn_fwd_fp8(dev(q), dev(k), dev(v), cu, pos if rope else None, max_len,
                                    scale, ws=ws)
    mf.get_status(ws)
    torch.cuda.synchronize()
    sc = None if scale <= 0 else scale
    o8, l8 = oracle.attn_fwd_e4m3(qf, kf, vf, cu_r, pos_r if rope else None, scale=sc)
    og, lg = f64(o), lse.cpu().numpy()
    res = check_o(og, o8, "O vs 8-bit oracle"), check_lse(lg, l8)
    o_ex, _ = oracle.attn_fwd(qf, kf, vf, cu_r, pos_r if rope else None, scale=sc)
    worst = check_exact_bounds(og, lg, qf, kf, vf, cu_r, pos_r if rope else None, scale=sc)
    print(f"vs 8-bit oracle: O max/mean {res[0][0]:.2e}/{res[0][1]:.2e}, LSE {res[1]:.2e}; "
          f"vs exact: O max/mean {np.abs(og - o_ex).max():.2e}/{np.abs(og - o_ex).mean():.2e}, "
          f"largest error / bound {worst:.2f}")
    return og, o8


def test_fwd_ragged_multi_tile(cuda_lib):
    _fwd_compare(cuda_lib, SPECS, heads=2, seed=71)


def test_fwd_no_rotation_and_explicit_scale(cuda_lib):
    _fwd_compare(cuda_lib, SPECS[:6], heads=2, seed=72, rope=False, scale=0.05)


def test_fwd_large_logits_and_zero_rows(cuda_lib):
    """Per-head scales on Q, K and V from {0.5, 1, 1.5, 2} (logit std up to 4) and
    all-zero Q rows (scale 0: uniform attention over the sample)."""
    rng = np.random.default_rng(73)
    hs = [rng.choice([0.5, 1.0, 1.5, 2.0], 3) for _ in range(3)]
    _fwd_compare(cuda_lib, [(64, 16, 16), (100, 8, 40), (0, 20, 20)], heads=3, seed=74,
                 head_scales=hs, zero_rows=25)


def test_fwd_3d_editing_pack(cuda_lib):
    mf = cuda_lib
    specs = [(12, 8, 8, 8, 8), (0, 16, 12, 12, 16), (30, 1, 5, 1, 5)]
    cu, pos = mf.pack3d(specs)
    T, max_len = mf.pack3d_size(specs)
    cu_r, pos_r = oracle.pack3d(specs)
    q, k, v, _ = random_inputs(T, 2, 128, seed=75, with_do=False)
    f = synth.bf16_bits_to_f64
    o, lse = mf.varlen_attn_fwd_fp8(dev(q), dev(k), dev(v), cu, pos, max_len)
    torch.cuda.synchronize()
    o8, l8 = oracle.attn_fwd_e4m3(f(q), f(k), f(v), cu_r, pos_r)
    check_o(f64(o), o8)
    check_lse(lse.cpu().numpy(), l8)
    check_exact_bounds(f64(o), lse.cpu().numpy(), f(q), f(k), f(v), cu_r, pos_r)


def test_fwd_empty_pack(cuda_lib):
    mf = cuda_lib
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    e = torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = mf.varlen_attn_fwd_fp8(e, e, e, cu, None, 0)
    torch.cuda.synchronize()
    assert o.numel() == 0 and lse.numel() == 0


@pytest.mark.parametrize("name", ["mixed_50k", "edit_50k"])
def test_fwd_full_size_sampled_pairs(cuda_lib, name):
    """The 50k packs at full size (the mixed pack the benchmark times, T = 48,019,
    and the editing pack with 3D positions, T = 48,230; 24 heads x 128), in the
    benchmark's call: (sample, head) pairs checked against the oracle, whose
    per-head scales come from quantising the whole head."""
    mf = cuda_lib
    wl = synth.workload(name, 0)
    q, k, v = synth.make_inputs(wl, with_do=False)[:3]
    if wl.edit:
        cu, pos = mf.pack3d(wl.specs)
        cu_r, pos_r = oracle.pack3d(wl.specs)
    else:
        cu, pos = mf.pack(wl.specs)
        cu_r, pos_r = oracle.pack(wl.specs)
    T, max_len = wl.total, wl.max_len
    ws = mf.workspace(T, len(wl.specs), wl.heads, 128, True)
    o, lse = mf.varlen_attn_fwd_fp8(dev(q), dev(k), dev(v), cu, pos, max_len, ws=ws)
    mf.get_status(ws)
    torch.cuda.synchronize()
    og, lg = f64(o), lse.cpu().numpy()
    f = synth.bf16_bits_to_f64
    lens = np.diff(cu_r)
    picks = [(int(np.argmax(lens)), 0), (int(np.argmin(lens)), 7), (3, 23)]
    for i, a in picks:
        qh, sq, kh, sk, vh, sv = oracle.quant_e4m3(f(q[:, a:a + 1]), f(k[:, a:a + 1]),
                                                   f(v[:, a:a + 1]), pos_r)
        s0, s1 = int(cu_r[i]), int(cu_r[i + 1])
        sl = slice(s0, s1)
        o8, l8 = oracle.attn_fwd_e4m3_quantized(qh[sl], sq[sl], kh[sl], sk, vh[sl], sv,
                                                np.array([0, s1 - s0]))
        check_o(og[sl, a], o8[:, 0], f"O sample {i} head {a}")
        check_lse(lg[a, sl], l8[0])
    # the same pairs against the exact attention, within the rigorous bounds
    check_exact_bounds(og, lg, f(q), f(k), f(v), cu_r, pos_r, pairs=picks)
