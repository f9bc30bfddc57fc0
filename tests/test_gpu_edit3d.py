"""GPU parity of the editing-pack path (frame-aware 3D positions) through the
C-ABI binding: mf_pack3d bit-exact, mf_rope3d_qk within 1 bf16 ulp, and the 3D
attention forward / backward against the FP64 oracle under the same tolerances
as the 2D path (O max 2e-2, mean 2e-3; LSE 1e-2; dQ/dK/dV max|err|/max|ref| 5e-2)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_ulp, check_grad, check_lse, check_o, dev, f64, random_inputs

pytestmark = pytest.mark.gpu

EDGE_SPECS = {
    "zero_length_and_empty_pieces": [(0, 0, 0, 0, 0), (3, 0, 4, 2, 2), (0, 2, 2, 0, 0),
                                     (1, 1, 1, 1, 1), (0, 0, 0, 0, 0)],
    "different_grids": [(7, 8, 16, 16, 8), (0, 3, 5, 7, 2)],
    "many_samples": [(i % 4, (i * 3) % 5, (i * 5) % 4, (i * 7) % 3, (i * 2) % 5) for i in range(300)],
}

# ragged editing pack: lengths 2, 263, 1185, ... spanning several 128-tiles
RAGGED_EDIT = [(7, 8, 16, 8, 16), (1, 16, 16, 12, 20), (0, 1, 1, 1, 1), (40, 24, 40, 24, 40)]


@pytest.mark.parametrize("name", list(EDGE_SPECS) + ["edit_tiny", "edit_50k"])
def test_pack3d_bit_exact(cuda_lib, name):
    mf = cuda_lib
    specs = EDGE_SPECS[name] if name in EDGE_SPECS else synth.workload(name).specs
    cu, pos = mf.pack3d(specs)
    cu_ref, pos_ref = oracle.pack3d(specs)
    assert np.array_equal(cu.cpu().numpy().astype(np.int64), cu_ref)
    assert np.array_equal(pos.cpu().numpy().astype(np.int64), pos_ref)
    assert mf.pack3d_size(specs) == (int(cu_ref[-1]), int(np.diff(cu_ref).max(initial=0)))


@pytest.mark.parametrize("d", [64, 128])
def test_rope3d_within_one_ulp(cuda_lib, d):
    mf = cuda_lib
    specs = RAGGED_EDIT
    cu, pos = mf.pack3d(specs)
    T = int(cu[-1])
    q, k, _, _ = random_inputs(T, 3, d, 41, with_do=False)
    qo, ko = mf.rope3d_qk(dev(q), dev(k), pos)
    torch.cuda.synchronize()
    p = pos.cpu().numpy().astype(np.int64)
    for x, y in ((q, qo), (k, ko)):
        xf = synth.bf16_bits_to_f64(x)
        ref = oracle.rope3d(xf, p)
        pair = np.repeat(np.hypot(xf[..., 0::2], xf[..., 1::2]), 2, axis=-1)
        err = np.abs(f64(y) - ref)
        assert np.all(err <= bf16_ulp(ref) + 2.0 ** -20 * pair), err.max()


def run_gpu3d(mf, specs, q, k, v, do=None):
    cu, pos = mf.pack3d(specs)
    T, max_len = mf.pack3d_size(specs)
    h, d = q.shape[1], q.shape[2]
    qd, kd, vd = dev(q), dev(k), dev(v)
    ws_f = mf.workspace(T, len(specs), h, d, False)
    o, lse = mf.varlen_attn_fwd(qd, kd, vd, cu, pos, max_len, ws=ws_f)
    mf.get_status(ws_f)
    out = {"o": o, "lse": lse, "pos": pos}
    if do is not None:
        ws_b = mf.workspace(T, len(specs), h, d, True)
        dq, dk, dv = mf.varlen_attn_bwd(qd, kd, vd, o, lse, dev(do), cu, pos, max_len, ws=ws_b)
        mf.get_status(ws_b)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    return out


def _full_compare3d(specs, heads, d, seed):
    import packed_resolution_diffusion_pack_b300 as mf
    cu_ref, pos_ref = oracle.pack3d(specs)
    T = int(cu_ref[-1])
    q, k, v, do = random_inputs(T, heads, d, seed)
    out = run_gpu3d(mf, specs, q, k, v, do)
    f = synth.bf16_bits_to_f64
    o_ref, lse_ref = oracle.attn_fwd3d(f(q), f(k), f(v), cu_ref, pos_ref)
    check_o(f64(out["o"]), o_ref)
    check_lse(out["lse"].cpu().numpy(), lse_ref)
    g_ref = oracle.attn_bwd3d(f(q), f(k), f(v), f(do), cu_ref, pos_ref)
    for name, g in zip(("dq", "dk", "dv"), g_ref):
        check_grad(f64(out[name]), g, name)


@pytest.mark.parametrize("d", [64, 128])
def test_ragged_editing_pack(cuda_lib, d):
    _full_compare3d(RAGGED_EDIT, heads=2, d=d, seed=42)


def test_edit_tiny_workload(cuda_lib):
    wl = synth.edit_tiny()
    _full_compare3d(wl.specs, wl.heads, wl.head_dim, seed=43)


def test_frame_changes_the_result(cuda_lib):
    """The same tokens with the target's frame coordinate at 1 (3D) and with the
    plain 2D positions give different outputs: the frame axis is not ignored."""
    mf = cuda_lib
    specs = [(2, 4, 4, 4, 4)]
    cu, pos3 = mf.pack3d(specs)
    T = int(cu[-1])
    q, k, v, _ = random_inputs(T, 1, 64, 44, with_do=False)
    a = mf.rope3d_qk(dev(q), None, pos3)[0]
    pos0 = pos3.clone()
    pos0[:, 0] = 0
    b = mf.rope3d_qk(dev(q), None, pos0)[0]
    src_end = 2 + 16
    assert torch.equal(a[:src_end], b[:src_end])
    assert not torch.equal(a[src_end:], b[src_end:])


def test_full_edit_50k(cuda_lib):
    """The 50k editing pack at full size: sampled query rows of three samples and
    two heads against the oracle, and the full backward of the smallest sample for
    two heads."""
    mf = cuda_lib
    wl = synth.edit_50k()
    q, k, v, do = synth.make_inputs(wl)
    out = run_gpu3d(mf, wl.specs, q, k, v, do)
    cu, pos = oracle.pack3d(wl.specs)
    L = np.diff(cu)
    order = np.argsort(L)
    f = synth.bf16_bits_to_f64
    rng = np.random.default_rng(7)
    for i in sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])}):
        s, e = int(cu[i]), int(cu[i + 1])
        for a in (0, wl.heads - 1):
            sl = lambda x: oracle.rope3d(f(x[s:e, a:a + 1]), pos[s:e])  # noqa: E731
            local = np.sort(rng.choice(e - s, min(40, e - s), replace=False))
            rows = np.stack([local, np.zeros_like(local)], 1)
            o_r, l_r = oracle.attn_fwd_rows(sl(q), sl(k), f(v[s:e, a:a + 1]), np.array([0, e - s]),
                                            None, rows)
            idx = torch.from_numpy(s + local).cuda()
            check_o(f64(out["o"][idx, a]), o_r, f"O sample {i} head {a}")
            check_lse(out["lse"][a, idx].cpu().numpy(), l_r)
    i = int(order[0])
    s, e = int(cu[i]), int(cu[i + 1])
    for a in (0, wl.heads - 1):
        sl = lambda x: f(x[s:e, a:a + 1])  # noqa: E731
        g_ref = oracle.attn_bwd3d(sl(q), sl(k), sl(v), sl(do), np.array([0, e - s]), pos[s:e])
        for name, g in zip(("dq", "dk", "dv"), g_ref):
            check_grad(f64(out[name][s:e, a:a + 1]), g, f"{name} sample {i} head {a}")
