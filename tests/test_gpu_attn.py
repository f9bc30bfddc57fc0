"""GPU parity of the varlen attention forward and backward against the FP64
oracle, through the C-ABI binding: small packs element by element (several tiles
and ragged tails), the five workloads at full size on sampled rows / (sample,
head) pairs, invariants and edge cases."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (bf16_ulp, check_grad, check_lse, check_o, dev, f64, oracle_pairs_fwd,
                      random_inputs, run_gpu)

pytestmark = pytest.mark.gpu

# lengths 1, 127, 128, 129, 255, 256, 257, 384, 513 and a 1000-token image
RAGGED_SPECS = [(1, 0, 0), (7, 8, 15), (0, 8, 16), (1, 8, 16), (15, 16, 15), (0, 16, 16),
                (1, 16, 16), (0, 12, 32), (1, 16, 32), (40, 24, 40)]


def _close_ulp(x, y):
    """dQ is summed over key tiles with fp32 atomics, whose order varies from run
    to run: two runs agree to one bf16 ulp plus fp32 reordering noise (2^-20 of
    the tensor's largest value, which covers rows that cancel to near zero), not
    bit for bit."""
    a, b = f64(x), f64(y)
    tol = bf16_ulp(np.maximum(np.abs(a), np.abs(b))) + 2.0 ** -20 * np.abs(a).max()
    assert (np.abs(a - b) <= tol).all()


def _full_compare(specs, heads, d, seed, rope=True, bwd=True, scale=0.0):
    import packed_resolution_diffusion_pack_b300 as mf
    cu_ref, pos_ref = oracle.pack(specs)
    T = int(cu_ref[-1])
    q, k, v, do = random_inputs(T, heads, d, seed, with_do=bwd)
    out = run_gpu(mf, specs, q, k, v, do if bwd else None, rope=rope, scale=scale)
    f = synth.bf16_bits_to_f64
    sc = None if scale <= 0 else scale
    o_ref, lse_ref = oracle.attn_fwd(f(q), f(k), f(v), cu_ref, pos_ref if rope else None, scale=sc)
    res = {"o": check_o(f64(out["o"]), o_ref),
           "lse": check_lse(out["lse"].cpu().numpy(), lse_ref)}
    if bwd:
        g_ref = oracle.attn_bwd(f(q), f(k), f(v), f(do), cu_ref, pos_ref if rope else None, scale=sc)
        for name, g in zip(("dq", "dk", "dv"), g_ref):
            res[name] = check_grad(f64(out[name]), g, name)
    return res


def test_tiny_workload_fwd_bwd(cuda_lib):
    wl = synth.tiny()
    q, k, v, do = synth.make_inputs(wl)
    out = run_gpu(cuda_lib, wl.specs, q, k, v, do)
    f = synth.bf16_bits_to_f64
    cu, pos = oracle.pack(wl.specs)
    o_ref, lse_ref = oracle.attn_fwd(f(q), f(k), f(v), cu, pos)
    check_o(f64(out["o"]), o_ref)
    check_lse(out["lse"].cpu().numpy(), lse_ref)
    for name, g in zip(("dq", "dk", "dv"), oracle.attn_bwd(f(q), f(k), f(v), f(do), cu, pos)):
        check_grad(f64(out[name]), g, name)


@pytest.mark.parametrize("d", [64, 128])
def test_ragged_multi_tile(cuda_lib, d):
    _full_compare(RAGGED_SPECS, heads=2, d=d, seed=11)


def test_no_rotation_path(cuda_lib):
    _full_compare(RAGGED_SPECS[:6], heads=2, d=128, seed=12, rope=False)


def test_explicit_scale(cuda_lib):
    _full_compare(RAGGED_SPECS[:5], heads=1, d=64, seed=13, scale=0.3)


def test_large_logits(cuda_lib):
    """Per-head scales up to 2 on Q, K and V (logit std up to 4), as in the
    extreme-aspect workload, on a small pack."""
    import packed_resolution_diffusion_pack_b300 as mf
    specs = [(64, 16, 16), (100, 8, 40)]
    cu_ref, pos_ref = oracle.pack(specs)
    T = int(cu_ref[-1])
    s = np.array([0.5, 2.0, 1.3])
    q = synth.normal_bf16_bits(5, 2, (T, 3, 128), s)
    k = synth.normal_bf16_bits(5, 3, (T, 3, 128), s[::-1].copy())
    v = synth.normal_bf16_bits(5, 4, (T, 3, 128), s)
    do = synth.normal_bf16_bits(5, 5, (T, 3, 128))
    out = run_gpu(mf, specs, q, k, v, do)
    f = synth.bf16_bits_to_f64
    o_ref, lse_ref = oracle.attn_fwd(f(q), f(k), f(v), cu_ref, pos_ref)
    check_o(f64(out["o"]), o_ref)
    check_lse(out["lse"].cpu().numpy(), lse_ref)
    for name, g in zip(("dq", "dk", "dv"), oracle.attn_bwd(f(q), f(k), f(v), f(do), cu_ref, pos_ref)):
        check_grad(f64(out[name]), g, name)


def test_cross_sample_independence_bit_exact(cuda_lib):
    mf = cuda_lib
    specs = RAGGED_SPECS
    cu_ref, _ = oracle.pack(specs)
    T = int(cu_ref[-1])
    q, k, v, do = random_inputs(T, 2, 128, 21)
    a = run_gpu(mf, specs, q, k, v, do)
    s, e = int(cu_ref[4]), int(cu_ref[5])
    q2, k2, v2, do2 = (x.copy() for x in (q, k, v, do))
    rng = np.random.default_rng(0)
    for x in (q2, k2, v2, do2):
        x[s:e] = rng.integers(0, 2 ** 16, size=x[s:e].shape, dtype=np.uint16) & 0x3FFF
    b = run_gpu(mf, specs, q2, k2, v2, do2)
    keep = torch.ones(T, dtype=torch.bool)
    keep[s:e] = False
    keep = keep.cuda()
    for name in ("o", "dk", "dv"):
        assert torch.equal(a[name][keep], b[name][keep]), name
    assert torch.equal(a["lse"][:, keep], b["lse"][:, keep])
    _close_ulp(a["dq"][keep], b["dq"][keep])


def test_value_shift_invariance(cuda_lib):
    """V -> V + c (one vector per sample) moves O by c within tolerance."""
    mf = cuda_lib
    specs = RAGGED_SPECS[:6]
    cu_ref, pos_ref = oracle.pack(specs)
    T = int(cu_ref[-1])
    q, k, v, _ = random_inputs(T, 2, 64, 22, with_do=False)
    a = run_gpu(mf, specs, q, k, v)
    vf = synth.bf16_bits_to_f64(v)
    c = np.round(np.random.default_rng(1).standard_normal((len(specs), 2, 64)) * 4) / 4
    for i in range(len(specs)):
        vf[cu_ref[i]:cu_ref[i + 1]] += c[i]
    v2 = synth.torch_to_bits(torch.from_numpy(vf).to(torch.bfloat16))
    b = run_gpu(mf, specs, q, k, v2)
    diff = f64(b["o"]) - f64(a["o"])
    for i in range(len(specs)):
        check_o(diff[cu_ref[i]:cu_ref[i + 1]], np.broadcast_to(c[i], diff[cu_ref[i]:cu_ref[i + 1]].shape),
                "O shift")


def test_text_only_pack_rotation_is_identity(cuda_lib):
    mf = cuda_lib
    specs = [(300, 0, 0), (45, 0, 0)]
    q, k, v, do = random_inputs(345, 2, 128, 23)
    a = run_gpu(mf, specs, q, k, v, do, rope=True)
    b = run_gpu(mf, specs, q, k, v, do, rope=False)
    for name in ("o", "lse", "dk", "dv"):
        assert torch.equal(a[name], b[name]), name
    _close_ulp(a["dq"], b["dq"])


def test_small_gradients_keep_precision(cuda_lib):
    """dO scaled by 2^-24 (gradient sizes of real training): the fp16 staging of dS
    is rescaled per head, so the gradients match the oracle at the same relative
    tolerance instead of underflowing."""
    import packed_resolution_diffusion_pack_b300 as mf
    specs = RAGGED_SPECS[3:7]
    cu_ref, pos_ref = oracle.pack(specs)
    T = int(cu_ref[-1])
    q, k, v, do = random_inputs(T, 2, 128, 25)
    dof = synth.bf16_bits_to_f64(do) * 2.0 ** -24  # exact: a power of two
    do_small = synth.torch_to_bits(torch.from_numpy(dof).to(torch.bfloat16))
    out = run_gpu(mf, specs, q, k, v, do_small)
    f = synth.bf16_bits_to_f64
    g_ref = oracle.attn_bwd(f(q), f(k), f(v), dof, cu_ref, pos_ref)
    for name, g in zip(("dq", "dk", "dv"), g_ref):
        check_grad(f64(out[name]), g, name)


def test_fp16_range_flagged(cuda_lib):
    """Q values beyond the fp16 range of the internal operands are reported as
    MF_ERR_OVERFLOW by mf_get_status, never passed on silently."""
    mf = cuda_lib
    specs = [(10, 2, 3)]
    T = 16
    q = synth.bf16_bits_to_f64(synth.normal_bf16_bits(0, 2, (T, 1, 64)))
    q[3, 0, 5] = 1.0e5
    qd = synth.bits_to_torch(synth.torch_to_bits(torch.from_numpy(q).to(torch.bfloat16))).cuda()
    cu, pos = mf.pack(specs)
    ws = mf.workspace(T, 1, 1, 64, False)
    mf.varlen_attn_fwd(qd, qd, qd, cu, pos, T, ws=ws)
    with pytest.raises(mf.MFError) as ei:
        mf.get_status(ws)
    assert ei.value.status == 3


def test_zero_length_samples_and_single_tokens(cuda_lib):
    specs = [(0, 0, 0), (1, 0, 0), (0, 0, 0), (0, 1, 1), (2, 0, 0), (0, 0, 0), (130, 0, 0), (0, 0, 0)]
    _full_compare(specs, heads=3, d=64, seed=24)


def test_empty_pack(cuda_lib):
    mf = cuda_lib
    cu, pos = mf.pack([])
    z = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    ws = mf.workspace(0, 0, 2, 64, True)
    o, lse = mf.varlen_attn_fwd(z, z, z, cu, pos, 0, ws=ws)
    mf.get_status(ws)
    dq, dk, dv = mf.varlen_attn_bwd(z, z, z, o, lse, z, cu, pos, 0, ws=ws)
    mf.get_status(ws)
    assert o.shape == (0, 2, 64) and dq.shape == (0, 2, 64)


def test_bad_seqlens_reported(cuda_lib):
    mf = cuda_lib
    T = 64
    q = dev(synth.normal_bf16_bits(0, 2, (T, 1, 64)))
    ws = mf.workspace(T, 2, 1, 64, False)
    for bad in ([0, 40, 30], [0, 30, 63], [1, 30, 64]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        mf.varlen_attn_fwd(q, q, q, cu, None, 64, ws=ws)
        with pytest.raises(mf.MFError) as ei:
            mf.get_status(ws)
        assert ei.value.status == 6
    cu = torch.tensor([0, 40, 64], dtype=torch.int32, device="cuda")
    mf.varlen_attn_fwd(q, q, q, cu, None, 39, ws=ws)  # max_len too small
    with pytest.raises(mf.MFError):
        mf.get_status(ws)
    mf.varlen_attn_fwd(q, q, q, cu, None, 40, ws=ws)
    mf.get_status(ws)


# ------------------------------------------------- the workloads at full size
def _full_size(name, fwd_rows=48, bwd_pairs=()):
    """Full workload on the GPU (the launch configuration the benchmark times);
    oracle on sampled query rows of the longest, shortest and a middle sample for
    two heads, and the full backward of the given (sample, head) pairs."""
    import packed_resolution_diffusion_pack_b300 as mf
    wl = synth.workload(name)
    q, k, v, do = synth.make_inputs(wl)
    out = run_gpu(mf, wl.specs, q, k, v, do)
    cu, pos = oracle.pack(wl.specs)
    L = np.diff(cu)
    order = np.argsort(L)
    picks = sorted({int(order[-1]), int(order[0]), int(order[len(order) // 2])})
    heads = [0, wl.heads - 1]
    o_gpu = out["o"]
    lse_gpu = out["lse"]
    for (i, a, local, o_r, l_r) in oracle_pairs_fwd(q, k, v, cu, pos,
                                                     [(i, a) for i in picks for a in heads],
                                                     rows_per_pair=fwd_rows, seed=5):
        rows = torch.from_numpy(int(cu[i]) + local).cuda()
        check_o(f64(o_gpu[rows, a]), o_r, f"O sample {i} head {a}")
        check_lse(lse_gpu[a, rows].cpu().numpy(), l_r)
    f = synth.bf16_bits_to_f64
    for (i, a) in bwd_pairs:
        s, e = int(cu[i]), int(cu[i + 1])
        sl = lambda x: f(x[s:e, a:a + 1])  # noqa: E731
        g_ref = oracle.attn_bwd(sl(q), sl(k), sl(v), sl(do), np.array([0, e - s]), pos[s:e])
        for name, g in zip(("dq", "dk", "dv"), g_ref):
            check_grad(f64(out[name][s:e, a:a + 1]), g, f"{name} sample {i} head {a}")


def test_full_single_1024(cuda_lib):
    _full_size("single_1024")


def test_full_cfg_2048(cuda_lib):
    _full_size("cfg_2048", fwd_rows=24)


def test_full_mixed_50k(cuda_lib):
    """The benchmarked pack: the backward of its longest sample (4,291 tokens, 34
    key blocks whose dQ contributions are summed into each query row) and of its
    shortest, against the oracle's full backward of those (sample, head) pairs."""
    wl = synth.mixed_50k()
    L = np.array(wl.lengths)
    small, large = int(np.argmin(L)), int(np.argmax(L))
    _full_size("mixed_50k", bwd_pairs=[(large, 0), (large, wl.heads - 1), (small, 0),
                                       (small, wl.heads - 1)])


def test_full_extreme_aspect(cuda_lib):
    """The 128x128 sample (about 16.5k tokens, 130 key blocks) under the per-head
    scales of this workload, and the last 64x64 filler."""
    wl = synth.extreme_aspect()
    big = int(np.argmax(np.array(wl.lengths)))
    _full_size("extreme_aspect", fwd_rows=32, bwd_pairs=[(big, 5), (len(wl.specs) - 1, 5)])


@pytest.mark.parametrize("edit", [False, True])
def test_bwd_after_fwd_reuses_rotated_operands(cuda_lib, edit):
    """One workspace for forward and backward with the backward's rotation pre-pass
    skipped gives the regular backward's results (dK, dV bit for bit; dQ up to its
    atomic summation order)."""
    mf = cuda_lib
    if edit:
        specs = [(7, 8, 16, 8, 16), (1, 16, 16, 12, 20), (3, 5, 7, 5, 7)]
        cu, pos = mf.pack3d(specs)
        T, max_len = mf.pack3d_size(specs)
    else:
        specs = RAGGED_SPECS
        cu, pos = mf.pack(specs)
        T, max_len = mf.pack_size(specs)
    q, k, v, do = (dev(x) for x in random_inputs(T, 2, 128, 31))
    n = len(specs)
    o, lse = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len, ws=mf.workspace(T, n, 2, 128, False))
    ref = mf.varlen_attn_bwd(q, k, v, o, lse, do, cu, pos, max_len, ws=mf.workspace(T, n, 2, 128, True))
    ws = mf.workspace(T, n, 2, 128, True)
    o2, lse2 = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len, ws=ws)
    got = mf.varlen_attn_bwd(q, k, v, o2, lse2, do, cu, pos, max_len, ws=ws, after_fwd=True)
    mf.get_status(ws)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert torch.equal(ref[1], got[1]) and torch.equal(ref[2], got[2])
    _close_ulp(ref[0], got[0])
