"""Run-to-run determinism.  The persistent kernels hand out work items through
atomic counters, so which CTA computes an item changes from run to run; every
item's result depends only on its own (sample, head, tile), so the outputs must
not.  The forward (16-bit, 8-bit, rotate-on-load) and both backward forms are
run three times on the full mixed 50k-token pack (24 heads x 128, seeded N(0, 1)
bf16 inputs made on the device) and compared bit for bit; a fourth forward runs
on a workspace reused after a backward."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _inputs(wl, seed):
    T = int(sum(wl.lengths))
    g = torch.Generator(device="cuda").manual_seed(seed)
    shape = (T, wl.heads, wl.head_dim)
    return [torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16) for _ in range(4)]


def test_forward_variants_bit_identical_across_runs(cuda_lib):
    mf = cuda_lib
    wl = synth.workload("mixed_50k")
    q, k, v, _ = _inputs(wl, 11)
    cu, pos = mf.pack(wl.specs)
    T, max_len = mf.pack_size(wl.specs)
    n, h, d = len(wl.specs), wl.heads, wl.head_dim
    ws = mf.workspace(T, n, h, d, False)
    for fn in (mf.varlen_attn_fwd, mf.varlen_attn_fwd_fp8, mf.varlen_attn_fwd_fused_rope):
        runs = []
        for _ in range(3):
            o, lse = fn(q, k, v, cu, pos, max_len, ws=ws)
            mf.get_status(ws)
            runs.append((o.clone(), lse.clone()))
        for o, lse in runs[1:]:
            assert torch.equal(o, runs[0][0]), fn.__name__
            assert torch.equal(lse, runs[0][1]), fn.__name__


@pytest.mark.parametrize("stored_ds", [True, False])
def test_backward_bit_identical_across_runs(cuda_lib, stored_ds):
    mf = cuda_lib
    wl = synth.workload("mixed_50k")
    q, k, v, do = _inputs(wl, 12)
    cu, pos = mf.pack(wl.specs)
    T, max_len = mf.pack_size(wl.specs)
    n, h, d = len(wl.specs), wl.heads, wl.head_dim
    ws = mf.workspace(T, n, h, d, True, store_ds_max_len=max_len if stored_ds else None)
    o, lse = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len, ws=ws)
    mf.get_status(ws)
    o0, lse0 = o.clone(), lse.clone()
    runs = []
    for _ in range(3):
        grads = mf.varlen_attn_bwd(q, k, v, o, lse, do, cu, pos, max_len, ws=ws, after_fwd=True)
        mf.get_status(ws)
        runs.append([g.clone() for g in grads])
    for r in runs[1:]:
        for name, a, b in zip(("dq", "dk", "dv"), r, runs[0]):
            assert torch.equal(a, b), name
    # the same workspace, after the backwards, serves the forward again unchanged
    o2, lse2 = mf.varlen_attn_fwd(q, k, v, cu, pos, max_len, ws=ws)
    mf.get_status(ws)
    assert torch.equal(o2, o0) and torch.equal(lse2, lse0)
