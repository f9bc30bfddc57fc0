"""Packs of thousands of short samples (paperlayer.ai summary 3.2.1: many samples of
mixed sizes in one packed update).  Above 4,096 samples the schedule keeps pack
order instead of ranking by length; either way each CTA of the forward and of
the dK / dV kernel claims hundreds of work items through its atomic counter and
cycles its item ring many times.  The forward and both backward forms against
the FP64 oracle; dK and dV of the two backward forms bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import check_grad, check_lse, check_o, dev, f64, random_inputs

pytestmark = pytest.mark.gpu


def _specs(n, seed, long_at=None):
    """n samples: text-only (1-23 tokens), small images with a caption (1-4 x 1-4
    latents, 0-5 text tokens) and zero-length samples; optionally one 1,280-token
    image at position long_at."""
    rng = np.random.default_rng(seed)
    specs = []
    for _ in range(n):
        kind = int(rng.integers(0, 5))
        if kind < 2:
            specs.append((int(rng.integers(1, 24)), 0, 0))
        elif kind < 4:
            specs.append((int(rng.integers(0, 6)), int(rng.integers(1, 5)), int(rng.integers(1, 5))))
        else:
            specs.append((0, 0, 0))
    if long_at is not None:
        specs[long_at] = (0, 32, 40)
    return specs


def _run(mf, specs, d, seed):
    cu_r, pos_r = oracle.pack(specs)
    T = int(cu_r[-1])
    h = 2
    q, k, v, do = random_inputs(T, h, d, seed)
    cu, pos = mf.pack(specs)
    _, max_len = mf.pack_size(specs)
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    o, lse = mf.varlen_attn_fwd(qd, kd, vd, cu, pos, max_len)
    ws_r = mf.workspace(T, len(specs), h, d, True)
    ws_s = mf.workspace(T, len(specs), h, d, True, store_ds_max_len=max_len)
    rec = mf.varlen_attn_bwd(qd, kd, vd, o, lse, dod, cu, pos, max_len, ws=ws_r)
    mf.get_status(ws_r)
    sto = mf.varlen_attn_bwd(qd, kd, vd, o, lse, dod, cu, pos, max_len, ws=ws_s)
    mf.get_status(ws_s)
    torch.cuda.synchronize()
    f = synth.bf16_bits_to_f64
    o_ref, lse_ref = oracle.attn_fwd(f(q), f(k), f(v), cu_r, pos_r)
    check_o(f64(o), o_ref)
    check_lse(lse.cpu().numpy(), lse_ref)
    g_ref = oracle.attn_bwd(f(q), f(k), f(v), f(do), cu_r, pos_r)
    for name, g, r in zip(("dq", "dk", "dv"), sto, g_ref):
        check_grad(f64(g), r, name)
    check_grad(f64(rec[0]), g_ref[0], "dq (recompute form)")
    assert torch.equal(rec[1], sto[1]) and torch.equal(rec[2], sto[2])


@pytest.mark.parametrize("d", [64, 128])
def test_beyond_rank_limit_pack_order(cuda_lib, d):
    """4,500 samples (pack order), one long image in the middle of the list."""
    _run(cuda_lib, _specs(4500, 91, long_at=2000), d, 92)


def test_ranked_many_samples(cuda_lib):
    """3,000 samples (ranked longest first), one long image at the end."""
    _run(cuda_lib, _specs(3000, 93, long_at=2999), 64, 94)
