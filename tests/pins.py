"""Pins of the FP64 oracle against things other than itself.

Each ``pin_*`` function raises AssertionError when the oracle (``so`` selects a
build of it) disagrees with a hand-computed table, a closed form, a library
routine on a special case, an invariant of the definition, or finite
differences.  ``tests/test_oracle_pins.py`` runs them on the real oracle;
``tests/test_oracle_mutants.py`` plants plausible mistakes in copies of the
oracle source and checks that some pin fails for each.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _tiny_inputs(seed=0):
    wl = synth.tiny(seed)
    q, k, v, do = synth.make_inputs(wl, with_do=True)
    f = synth.bf16_bits_to_f64
    return wl, f(q), f(k), f(v), f(do)


# ------------------------------------------------------------------ packing
def pin_pack_golden(so=None):
    for case in _golden("pack_cases.json")["cases"]:
        cu, pos = oracle.pack(case["specs"], so=so)
        assert cu.tolist() == case["cu"], (case["specs"], cu)
        if "pos" in case:
            assert pos.tolist() == case["pos"], (case["specs"], pos)
        for t, rc in case.get("pos_spot", {}).items():
            assert pos[int(t)].tolist() == rc, (t, pos[int(t)], rc)


# --------------------------------------------------------------------- RoPE
def pin_rope_golden(so=None):
    fn = {"cos": math.cos, "sin": math.sin, "-sin": lambda a: -math.sin(a)}
    for case in _golden("rope_d8.json")["cases"]:
        x = np.zeros((1, 1, 8))
        x[0, 0, case["unit"]] = 1.0
        y = oracle.rope2d(x, np.array([case["pos"]]), so=so)[0, 0]
        want = np.zeros(8)
        for dim, (kind, ang) in case["out"].items():
            want[int(dim)] = fn[kind](ang)
        np.testing.assert_allclose(y, want, atol=1e-15, err_msg=str(case))


def pin_rope_frequencies_d128(so=None):
    """d = 128: pair j of the row half turns by r * 10000^(-j/32) (closed form
    of 10000^(-2j/(d/2)) at d/2 = 64); checked at j = 0, 16 (10000^-0.5 = 0.01)
    and 31, for r = 1, and for the column half with c = 1."""
    for half, pos in ((0, [1, 0]), (1, [0, 1])):
        for j, omega in ((0, 1.0), (16, 0.01), (31, 10000.0 ** (-31 / 32))):
            x = np.zeros((1, 1, 128))
            x[0, 0, 64 * half + 2 * j] = 1.0
            y = oracle.rope2d(x, np.array([pos]), so=so)[0, 0]
            assert abs(y[64 * half + 2 * j] - math.cos(omega)) < 1e-14
            assert abs(y[64 * half + 2 * j + 1] - math.sin(omega)) < 1e-14
            y[64 * half + 2 * j: 64 * half + 2 * j + 2] = 0
            assert np.abs(y).max() == 0.0


def pin_rope_identity_and_norm(so=None):
    r = _rng(1)
    x = r.standard_normal((50, 3, 64))
    pos = np.zeros((50, 2), dtype=np.int64)
    np.testing.assert_array_equal(oracle.rope2d(x, pos, so=so), x)
    pos = r.integers(0, 128, size=(50, 2))
    y = oracle.rope2d(x, pos, so=so)
    nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(ny, nx, rtol=0, atol=1e-12)
    back = oracle.rope2d(y, pos, inverse=True, so=so)
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-12)


def pin_rope_relative(so=None):
    """<R(p1) q, R(p2) k> depends only on p1 - p2: shifting both positions by the
    same (dr, dc) leaves the dot product unchanged."""
    r = _rng(2)
    for d in (64, 128):
        q = r.standard_normal((20, 1, d))
        k = r.standard_normal((20, 1, d))
        p1 = r.integers(0, 100, size=(20, 2))
        p2 = r.integers(0, 100, size=(20, 2))
        shift = r.integers(-20, 20, size=(20, 2))
        shift = np.maximum(shift, -np.minimum(p1, p2))
        a = (oracle.rope2d(q, p1, so=so) * oracle.rope2d(k, p2, so=so)).sum(-1)
        b = (oracle.rope2d(q, p1 + shift, so=so) * oracle.rope2d(k, p2 + shift, so=so)).sum(-1)
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)
        # and it does depend on the offset (a rotation that ignored positions passes
        # the shift test trivially)
        c = (oracle.rope2d(q, p1 + 1, so=so) * oracle.rope2d(k, p2, so=so)).sum(-1)
        assert np.abs(a - c).max() > 1e-3


# ---------------------------------------------------------------- attention
def _sdpa_per_sample(q, k, v, cu):
    """torch.nn.functional.scaled_dot_product_attention (a library routine) run
    on each sample alone, fp64 on the CPU; LSE from torch.logsumexp."""
    T, h, d = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((h, T))
    for i in range(len(cu) - 1):
        s, e = int(cu[i]), int(cu[i + 1])
        if e == s:
            continue
        Q = torch.from_numpy(q[s:e]).permute(1, 0, 2)
        K = torch.from_numpy(k[s:e]).permute(1, 0, 2)
        V = torch.from_numpy(v[s:e]).permute(1, 0, 2)
        o[s:e] = torch.nn.functional.scaled_dot_product_attention(Q, K, V).permute(1, 0, 2).numpy()
        lse[:, s:e] = torch.logsumexp(torch.einsum("hqd,hkd->hqk", Q, K) / math.sqrt(d), -1).numpy()
    return o, lse


def pin_attn_vs_library(so=None):
    """No rotation: the oracle equals per-sample torch SDPA; with rotation it equals
    SDPA on the rotated inputs (RoPE itself pinned above)."""
    wl, q, k, v, _ = _tiny_inputs()
    cu, pos = oracle.pack(wl.specs)
    o, lse = oracle.attn_fwd(q, k, v, cu, None, so=so)
    o_ref, lse_ref = _sdpa_per_sample(q, k, v, cu)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    o, lse = oracle.attn_fwd(q, k, v, cu, pos, so=so)
    qr, kr = oracle.rope2d(q, pos), oracle.rope2d(k, pos)
    o_ref, lse_ref = _sdpa_per_sample(qr, kr, v, cu)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def pin_attn_packed_equals_unpacked(so=None):
    wl, q, k, v, _ = _tiny_inputs()
    cu, pos = oracle.pack(wl.specs, so=so)
    o, lse = oracle.attn_fwd(q, k, v, cu, pos, so=so)
    for i in range(len(cu) - 1):
        s, e = int(cu[i]), int(cu[i + 1])
        oi, li = oracle.attn_fwd(q[s:e], k[s:e], v[s:e], np.array([0, e - s]), pos[s:e], so=so)
        np.testing.assert_allclose(o[s:e], oi, rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[:, s:e], li, rtol=0, atol=1e-15)


def pin_attn_cross_sample_independence(so=None):
    wl, q, k, v, _ = _tiny_inputs()
    cu, pos = oracle.pack(wl.specs, so=so)
    o, lse = oracle.attn_fwd(q, k, v, cu, pos, so=so)
    s, e = int(cu[1]), int(cu[2])
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    r = _rng(3)
    for x in (q2, k2, v2):
        x[s:e] = r.standard_normal(x[s:e].shape) * 3
    o2, lse2 = oracle.attn_fwd(q2, k2, v2, cu, pos, so=so)
    keep = np.r_[0:s, e:len(q)]
    assert np.array_equal(o[keep], o2[keep])
    assert np.array_equal(lse[:, keep], lse2[:, keep])
    assert np.abs(o[s:e] - o2[s:e]).max() > 1e-3


def pin_attn_closed_forms(so=None):
    wl, q, k, v, _ = _tiny_inputs()
    cu, pos = oracle.pack(wl.specs, so=so)
    T, h, d = q.shape
    # V -> V + c_i (a constant vector per sample) gives O -> O + c_i
    c = _rng(4).standard_normal((len(cu) - 1, h, d))
    v2 = v.copy()
    for i in range(len(cu) - 1):
        v2[cu[i]:cu[i + 1]] += c[i]
    o, _ = oracle.attn_fwd(q, k, v, cu, pos, so=so)
    o2, _ = oracle.attn_fwd(q, k, v2, cu, pos, so=so)
    for i in range(len(cu) - 1):
        np.testing.assert_allclose(o2[cu[i]:cu[i + 1]] - o[cu[i]:cu[i + 1]],
                                   np.broadcast_to(c[i], o[cu[i]:cu[i + 1]].shape), atol=1e-12)
    # Q = 0: uniform weights, O = per-sample mean of V, LSE = ln L
    o0, lse0 = oracle.attn_fwd(np.zeros_like(q), k, v, cu, pos, so=so)
    for i in range(len(cu) - 1):
        s, e = int(cu[i]), int(cu[i + 1])
        np.testing.assert_allclose(o0[s:e], np.broadcast_to(v[s:e].mean(0), o0[s:e].shape), atol=1e-13)
        np.testing.assert_allclose(lse0[:, s:e], math.log(e - s), atol=1e-13)
    # L = 1 samples: O = V, LSE = <q, k> / sqrt(d) (one rotation on both sides)
    specs = [(1, 0, 0), (0, 1, 1), (0, 3, 3)]
    cu1, pos1 = oracle.pack(specs, so=so)
    r = _rng(5)
    q1, k1, v1 = (r.standard_normal((int(cu1[-1]), 2, 64)) for _ in range(3))
    pos1 = pos1 + np.array([[5, 7], [2, 9]] + [[3, 4]] * 9)
    o1, l1 = oracle.attn_fwd(q1, k1, v1, cu1, pos1, so=so)
    for t in (0, 1):
        np.testing.assert_allclose(o1[t], v1[t], atol=1e-15)
        np.testing.assert_allclose(l1[:, t], (q1[t] * k1[t]).sum(-1) / 8.0, atol=1e-13)


# ----------------------------------------------------------------- backward
def pin_bwd_finite_differences(so=None, ncoord=240):
    """Central differences of f = <dO, O(q, k, v)> (step 1e-6) at >= 200 random
    coordinates of q, k and v, with rotation, on the tiny workload."""
    wl, q, k, v, do = _tiny_inputs()
    cu, pos = oracle.pack(wl.specs)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, cu, pos, so=so)
    grads = {"q": dq, "k": dk, "v": dv}
    base = {"q": q, "k": k, "v": v}

    def f(xs):
        o, _ = oracle.attn_fwd(xs["q"], xs["k"], xs["v"], cu, pos, so=so)
        return float((o * do).sum())

    r = _rng(6)
    eps = 1e-6
    worst = 0.0
    for it in range(ncoord):
        name = "qkv"[it % 3]
        idx = tuple(int(r.integers(0, s)) for s in q.shape)
        xs = {n: base[n] for n in base}
        xp = base[name].copy(); xp[idx] += eps
        xm = base[name].copy(); xm[idx] -= eps
        xs[name] = xp; fp = f(xs)
        xs[name] = xm; fm = f(xs)
        fd = (fp - fm) / (2 * eps)
        g = grads[name][idx]
        err = abs(fd - g) / max(1.0, abs(g))
        worst = max(worst, err)
        assert err < 1e-6, (name, idx, fd, g)
    return worst


def pin_bwd_vs_library(so=None):
    """No rotation: the oracle's gradients equal torch autograd through per-sample
    SDPA in fp64."""
    wl, q, k, v, do = _tiny_inputs()
    cu, _ = oracle.pack(wl.specs)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, cu, None, so=so)
    for i in range(len(cu) - 1):
        s, e = int(cu[i]), int(cu[i + 1])
        Q, K, V = (torch.from_numpy(x[s:e].copy()).permute(1, 0, 2).requires_grad_() for x in (q, k, v))
        O = torch.nn.functional.scaled_dot_product_attention(Q, K, V)
        O.backward(torch.from_numpy(do[s:e]).permute(1, 0, 2))
        for g, t in ((dq, Q), (dk, K), (dv, V)):
            np.testing.assert_allclose(g[s:e], t.grad.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def pin_bwd_invariants(so=None):
    """Two consequences of the definition.  (1) Rows of P sum to one, so
    sum_k dV_k = sum_j dO_j within each sample.  (2) Rows of dS sum to zero: in a
    text-only sample (every token at (0,0), so no rotation), adding one vector c
    to every key shifts each logit row by a constant; P, O, dV and dK are
    unchanged and dQ moves by scale * c * sum_k dS_jk = 0."""
    wl, q, k, v, do = _tiny_inputs()
    cu, pos = oracle.pack(wl.specs)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, cu, pos, so=so)
    for i in range(len(cu) - 1):
        s, e = int(cu[i]), int(cu[i + 1])
        np.testing.assert_allclose(dv[s:e].sum(0), do[s:e].sum(0), atol=1e-11)
    r = _rng(7)
    L, h, d = 40, 2, 64
    cu1 = np.array([0, L]); pos1 = np.zeros((L, 2), dtype=np.int64)
    q1, k1, v1, do1 = (r.standard_normal((L, h, d)) for _ in range(4))
    g1 = oracle.attn_bwd(q1, k1, v1, do1, cu1, pos1, so=so)
    g2 = oracle.attn_bwd(q1, k1 + r.standard_normal((1, h, d)), v1, do1, cu1, pos1, so=so)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, atol=1e-11)


def pin_fwd_rows_match_full(so=None):
    """The row-subset entry gives the same rows as the full forward (it is the
    same definition restricted to those rows)."""
    wl, q, k, v, _ = _tiny_inputs()
    cu, pos = oracle.pack(wl.specs)
    o, lse = oracle.attn_fwd(q, k, v, cu, pos, so=so)
    rows = [(0, 0), (28, 1), (29, 0), (99, 1), (134, 0), (100, 1)]
    orow, lrow = oracle.attn_fwd_rows(q, k, v, cu, pos, rows, so=so)
    for r, (t, a) in enumerate(rows):
        np.testing.assert_array_equal(orow[r], o[t, a])
        assert lrow[r] == lse[a, t]


# ------------------------------------------------- packed CFG + Euler step
def pin_cfg_euler_golden(so=None):
    for case in _golden("cfg_euler.json")["cases"]:
        out = oracle.cfg_euler(np.array(case["v"], float), case["specs"], case["g"], case["dt"],
                               np.array(case["z"], float), so=so)
        assert np.array_equal(out, np.array(case["z_out"])), out


def _cfg_pack(rng, grids, texts, C):
    specs = []
    for (H, W), (tc, tu) in zip(grids, texts):
        specs += [(tc, H, W), (tu, H, W)]
    cu, _ = oracle.pack(specs)
    return specs, cu, rng.standard_normal((int(cu[-1]), C))


def pin_cfg_euler_straight_line(so=None):
    """On a straight rectified-flow path z_t = (1 - t) z0 + t eps with both branches
    predicting the exact velocity z0 - eps, one Euler step from t to t - dt lands
    exactly on z_{t-dt} for any guidance scale (pins the step's sign and the velocity
    convention against the pages' objective)."""
    rng = _rng(11)
    C = 8
    specs, cu, v = _cfg_pack(rng, [(3, 5), (2, 2)], [(4, 1), (0, 6)], C)
    N = 15 + 4
    z0, eps = rng.standard_normal((N, C)), rng.standard_normal((N, C))
    vel = z0 - eps
    row = 0
    for p in range(2):
        tc, H, W = specs[2 * p]
        tu = specs[2 * p + 1][0]
        n = H * W
        v[cu[2 * p] + tc: cu[2 * p] + tc + n] = vel[row:row + n]
        v[cu[2 * p + 1] + tu: cu[2 * p + 1] + tu + n] = vel[row:row + n]
        row += n
    t, dt = 0.7, 0.25
    for g in (0.0, 1.0, 4.5):
        out = oracle.cfg_euler(v, specs, g, dt, (1 - t) * z0 + t * eps, so=so)
        want = (1 - (t - dt)) * z0 + (t - dt) * eps
        assert np.abs(out - want).max() < 1e-12, (g, np.abs(out - want).max())


def pin_cfg_euler_branch_limits(so=None):
    """g = 0 follows the unconditional branch and g = 1 the conditional one, each
    read from its own sample's image rows (past its own text)."""
    rng = _rng(12)
    C = 4
    specs, cu, v = _cfg_pack(rng, [(2, 3)], [(5, 2)], C)
    z = rng.standard_normal((6, C))
    dt = 0.125
    vc = v[cu[0] + 5: cu[0] + 11]
    vu = v[cu[1] + 2: cu[1] + 8]
    # vu + (vc - vu) is vc up to one rounding of each operation
    assert np.abs(oracle.cfg_euler(v, specs, 1.0, dt, z, so=so) - (z + dt * vc)).max() < 1e-14
    assert np.array_equal(oracle.cfg_euler(v, specs, 0.0, dt, z, so=so), z + dt * vu)
    assert np.array_equal(oracle.cfg_euler(v, specs, 2.0, 0.0, z, so=so), z)


def pin_cfg_euler_pairs_independent(so=None):
    rng = _rng(13)
    C = 4
    specs, cu, v = _cfg_pack(rng, [(2, 3), (4, 1), (1, 1)], [(5, 2), (0, 3), (2, 2)], C)
    z = rng.standard_normal((6 + 4 + 1, C))
    full = oracle.cfg_euler(v, specs, 2.5, 0.3, z, so=so)
    row = 0
    for p in range(3):
        H, W = specs[2 * p][1], specs[2 * p][2]
        part = oracle.cfg_euler(v[cu[2 * p]:cu[2 * p + 2]], specs[2 * p:2 * p + 2], 2.5, 0.3,
                                z[row:row + H * W], so=so)
        assert np.array_equal(part, full[row:row + H * W]), p
        row += H * W


# ------------------------------------------ adaptive LayerNorm, gated residual
def _adaln_pack(rng, lens, Dm):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return cu, rng.standard_normal((int(cu[-1]), Dm)) * 3.0 + 0.5


def pin_adaln_vs_library(so=None):
    """With zero modulation the block is plain LayerNorm without affine parameters:
    torch's layer_norm in float64."""
    rng = _rng(21)
    Dm, eps = 48, 1e-6
    cu, x = _adaln_pack(rng, [3, 0, 7, 1], Dm)
    z = np.zeros((4, Dm))
    y = oracle.adaln(x, cu, z, z, eps, so=so)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (Dm,), eps=eps).numpy()
    assert np.abs(y - ref).max() < 1e-12, np.abs(y - ref).max()


def pin_adaln_variance_closed_form(so=None):
    """Each normalised row has mean 0 and variance var / (var + eps)."""
    rng = _rng(22)
    Dm, eps = 64, 0.25
    cu, x = _adaln_pack(rng, [5, 3], Dm)
    z = np.zeros((2, Dm))
    y = oracle.adaln(x, cu, z, z, eps, so=so)
    var = x.var(axis=1)
    assert np.abs(y.mean(axis=1)).max() < 1e-12
    assert np.abs(y.var(axis=1) - var / (var + eps)).max() < 1e-12


def pin_adaln_modulation_per_sample(so=None):
    """A constant row (small dyadic values, so its sum and mean are exact)
    normalises to exactly 0, so its output is its own sample's shift; a row with a
    +1/-1 pattern gets (1 + scale) times it."""
    rng = _rng(23)
    Dm = 16
    cu = np.array([0, 2, 2, 5], dtype=np.int64)
    x = np.repeat(rng.integers(-16, 16, size=(5, 1)) / 4.0, Dm, axis=1)
    shift, scale = rng.standard_normal((3, Dm)), rng.standard_normal((3, Dm))
    y = oracle.adaln(x, cu, shift, scale, 1e-6, so=so)
    for s in range(3):
        for t in range(cu[s], cu[s + 1]):
            assert np.array_equal(y[t], shift[s]), (s, t)
    alt = np.tile([1.0, -1.0], Dm // 2)[None, :].repeat(5, 0)
    y = oracle.adaln(alt, cu, np.zeros((3, Dm)), scale, 0.0, so=so)
    for s in range(3):
        for t in range(cu[s], cu[s + 1]):
            assert np.abs(y[t] - alt[t] * (1 + scale[s])).max() < 1e-15, (s, t)


def pin_gated_residual(so=None):
    rng = _rng(24)
    Dm = 8
    cu, x = _adaln_pack(rng, [2, 4, 1], Dm)
    h = rng.standard_normal(x.shape)
    zero = np.zeros((3, Dm))
    assert np.array_equal(oracle.gated_residual(x, h, cu, zero, so=so), x)
    gate = rng.standard_normal((3, Dm))
    out = oracle.gated_residual(x, np.ones_like(x), cu, gate, so=so)
    for s in range(3):
        for t in range(cu[s], cu[s + 1]):
            assert np.array_equal(out[t], x[t] + gate[s]), (s, t)


# ------------------------------------------- frame-aware 3D RoPE (editing)
def pin_pack3d_golden(so=None):
    for case in _golden("pack3d_cases.json")["cases"]:
        cu, pos = oracle.pack3d(case["specs"], so=so)
        assert cu.tolist() == case["cu"], (case["specs"], cu)
        assert pos.tolist() == case["pos"], (case["specs"], pos)


def pin_rope3d_golden(so=None):
    fn = {"cos": math.cos, "sin": math.sin, "-sin": lambda a: -math.sin(a)}
    for case in _golden("rope3d_d16.json")["cases"]:
        x = np.zeros((1, 1, 16))
        x[0, 0, case["unit"]] = 1.0
        y = oracle.rope3d(x, np.array([case["pos"]]), so=so)[0, 0]
        want = np.zeros(16)
        for dim, (kind, ang) in case["out"].items():
            want[int(dim)] = fn[kind](ang)
        assert np.abs(y - want).max() < 1e-14, (case, y)


def pin_rope3d_norm_identity_inverse(so=None):
    rng = _rng(31)
    x = rng.standard_normal((7, 3, 64))
    pos = rng.integers(0, 100, size=(7, 3))
    y = oracle.rope3d(x, pos, so=so)
    pairs = lambda a: np.hypot(a[..., 0::2], a[..., 1::2])  # noqa: E731
    assert np.abs(pairs(y) - pairs(x)).max() < 1e-12
    assert np.abs(oracle.rope3d(y, pos, inverse=True, so=so) - x).max() < 1e-12
    assert np.array_equal(oracle.rope3d(x, np.zeros((7, 3), dtype=np.int64), so=so), x)


def pin_rope3d_relative(so=None):
    """<R(p1) q, R(p2) k> depends only on p1 - p2 along all three axes, and does
    depend on the frame offset (source and target tokens at one grid position are
    told apart)."""
    rng = _rng(32)
    q, k = rng.standard_normal((1, 1, 32)), rng.standard_normal((1, 1, 32))
    dot = lambda p1, p2: float((oracle.rope3d(q, np.array([p1]), so=so) *  # noqa: E731
                                oracle.rope3d(k, np.array([p2]), so=so)).sum())
    base = dot([1, 5, 9], [0, 2, 4])
    for sh in ([0, 3, 1], [2, 0, 0], [5, 7, 11]):
        s = np.array(sh)
        assert abs(dot(np.array([1, 5, 9]) + s, np.array([0, 2, 4]) + s) - base) < 1e-12, sh
    assert abs(dot([1, 3, 3], [0, 3, 3]) - dot([0, 3, 3], [0, 3, 3])) > 1e-3


def pin_attn3d_bwd_finite_differences(so=None):
    """Central differences of <dO, O(q, k, v)> for an editing pack with 3D rotation
    (relative error < 1e-6 at sampled coordinates of q, k and v)."""
    rng = _rng(33)
    specs = [(3, 2, 3, 2, 3), (2, 1, 4, 2, 2)]
    cu, pos = oracle.pack3d(specs, so=so)
    T, h, d = int(cu[-1]), 2, 16
    q, k, v, do = (rng.standard_normal((T, h, d)) for _ in range(4))
    dq, dk, dv = oracle.attn_bwd3d(q, k, v, do, cu, pos, so=so)
    f = lambda q_, k_, v_: float((oracle.attn_fwd3d(q_, k_, v_, cu, pos, so=so)[0] * do).sum())  # noqa: E731
    eps = 1e-6
    for which, g in ((0, dq), (1, dk), (2, dv)):
        for _ in range(20):
            idx = (int(rng.integers(T)), int(rng.integers(h)), int(rng.integers(d)))
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += eps
            args_m[which][idx] -= eps
            num = (f(*args_p) - f(*args_m)) / (2 * eps)
            assert abs(num - g[idx]) <= 1e-6 * max(1.0, abs(num)), (which, idx, num, g[idx])


# ------------------------------------------------------- e4m3 forward variant
def _e4m3_table():
    """Every E4M3 code decoded from its bit fields (OCP 8-bit floating point:
    sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 15 with mantissa 7
    is NaN, no infinities): {code: value}, NaN codes left out."""
    out = {}
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        out[code] = -mag if s else mag
    return out


def pin_e4m3_code_table(so=None):
    """Representable values map to themselves; every midpoint between neighbours
    goes to the neighbour with the even mantissa; a nudge off the midpoint goes to
    the nearer one; beyond the largest finite value (448) the result saturates."""
    table = _e4m3_table()
    assert len(table) == 254 and max(table.values()) == 448.0
    vals = np.array(sorted(set(table.values())))
    assert np.array_equal(oracle.e4m3(vals, so=so), vals)
    pos = vals[vals >= 0]
    code_of = {v: c for c, v in table.items() if c < 128}
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2
    even = np.where(np.array([code_of[v] & 1 for v in lo]) == 0, lo, hi)
    assert np.array_equal(oracle.e4m3(mid, so=so), even)
    assert np.array_equal(oracle.e4m3(-mid, so=so), -even)
    assert np.array_equal(oracle.e4m3(np.nextafter(mid, np.inf), so=so), hi)
    assert np.array_equal(oracle.e4m3(np.nextafter(mid, -np.inf), so=so), lo)
    big = np.array([448.0, 449.0, 464.0, 1e4, 1e300])
    assert np.array_equal(oracle.e4m3(big, so=so), np.full(5, 448.0))
    assert np.array_equal(oracle.e4m3(-big, so=so), np.full(5, -448.0))


def pin_e4m3_vs_library(so=None):
    """torch's float32 -> float8_e4m3fn conversion (round to nearest even) on
    200,000 in-range values spread over 21 binades, subnormals included."""
    rng = _rng(40)
    x = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-12, 9, 200_000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3(x.astype(np.float64), so=so), ref)


def _e4m3_inputs(seed, specs, h, d, scales=None):
    rng = _rng(seed)
    cu, pos = oracle.pack(specs, so=None)
    T = int(cu[-1])
    q, k, v = (rng.standard_normal((T, h, d)) for _ in range(3))
    if scales is not None:
        q, k, v = q * scales[0][None, :, None], k * scales[1][None, :, None], v * scales[2][None, :, None]
    return cu, pos, q, k, v


def pin_quant_e4m3(so=None):
    """Quantised operands: every scale is a power of two, the smallest that brings
    the block's largest magnitude to at most 448 (so that largest magnitude lands in
    (224, 448]); every value is an e4m3 value; every rotated K component stays
    within 448 at every position; dequantised values are within half an e4m3
    quantum of the exact rotated operands (2^-4 relative in the normal range, 2^-10
    of the scale below it)."""
    rng = _rng(41)
    specs = [(7, 9, 13), (3, 16, 4), (0, 5, 31)]
    scales = [rng.uniform(0.5, 2, 3) for _ in range(3)]
    cu, pos, q, k, v = _e4m3_inputs(42, specs, 3, 64, scales)
    qh, sq, kh, sk, vh, sv = oracle.quant_e4m3(q, k, v, pos, so=so)
    qr, kr = oracle.rope2d(q, pos), oracle.rope2d(k, pos)
    for a in (qh, kh, vh):
        assert np.array_equal(oracle.e4m3(a), a)
    for s_, amax in ((sq, np.abs(qr).max(axis=2)), (sv, np.abs(v).max(axis=(0, 2))),
                     (sk, np.sqrt(k[..., 0::2] ** 2 + k[..., 1::2] ** 2).max(axis=(0, 2)))):
        assert np.all(np.exp2(np.round(np.log2(s_))) == s_)
        assert np.all((amax / s_ > 224.0) & (amax / s_ <= 448.0))
    assert np.all(np.abs(qh).max(axis=2) >= 224.0) and np.all(np.abs(vh).max(axis=(0, 2)) >= 224.0)
    assert np.abs(kh).max() <= 448.0
    for hat, s, ref in ((qh, sq[:, :, None], qr), (kh, sk[None, :, None], kr),
                        (vh, sv[None, :, None], v)):
        err = np.abs(hat * s - ref)
        assert np.all(err <= 2.0 ** -4 * np.abs(ref) + 2.0 ** -10 * s + 1e-15)
    assert np.all(sk * 448.0 >= np.abs(kr).max(axis=(0, 2)) - 1e-12)


def pin_attn_e4m3_exact_limit(so=None):
    """With rounding switched off the variant's tiled steps (running maximum raised
    only past a margin, rescaling of l and the accumulator) are exact: O and
    LSE equal the plain attention of the same operands to 1e-12, on a tiny pack and
    on samples of several 128-key tiles whose logits rise along the keys, so that
    later tiles raise the maximum and rescale."""
    wl, q, k, v, _ = _tiny_inputs(0)
    cu, pos = oracle.pack(wl.specs)
    o8, l8 = oracle.attn_fwd_e4m3(q, k, v, cu, pos, round=False, so=so)
    o, l = oracle.attn_fwd(q, k, v, cu, pos)
    assert np.abs(o8 - o).max() < 1e-12 and np.abs(l8 - l).max() < 1e-12
    rng = _rng(43)
    specs = [(0, 10, 40), (5, 3, 100), (2, 1, 129)]
    cu2, _ = oracle.pack(specs)
    T, h, d = int(cu2[-1]), 2, 32
    u = rng.standard_normal(d)
    q2 = np.tile(3.0 * u, (T, h, 1))
    ramp = np.concatenate([np.arange(cu2[i + 1] - cu2[i]) for i in range(len(specs))]) / 20.0
    k2 = ramp[:, None, None] * u[None, None, :] + 0.1 * rng.standard_normal((T, h, d))
    v2 = rng.standard_normal((T, h, d))
    o8, l8 = oracle.attn_fwd_e4m3(q2, k2, v2, cu2, None, round=False, so=so)
    o, l = oracle.attn_fwd(q2, k2, v2, cu2, None)
    assert np.abs(o8 - o).max() < 1e-12 * max(1.0, np.abs(o).max())
    assert np.abs(l8 - l).max() < 1e-10


def pin_attn_e4m3_error_bounds(so=None):
    """Against the exact attention of the un-rounded operands, with rounding on,
    the 8-bit oracle lies within the rigorous per-row bounds of e4m3_bound (LSE
    within the largest logit change the operand rounding permits; O within the
    sum of the probability-rounding, V-rounding and softmax-response terms).
    On this data (per-head scales up to 2 on q, k and v) the mean error is about 6 %
    of the mean |O|; the last check allows 10 %."""
    from e4m3_bound import e4m3_attention_bounds
    rng = _rng(44)
    specs = [(9, 6, 11), (4, 20, 9), (1, 1, 1)]
    scales = [rng.uniform(0.5, 2, 2) for _ in range(3)]
    cu, pos, q, k, v = _e4m3_inputs(45, specs, 2, 32, scales)
    T, h, d = q.shape
    sc = 1.0 / math.sqrt(d)
    o8, l8 = oracle.attn_fwd_e4m3(q, k, v, cu, pos, so=so)
    o, l = oracle.attn_fwd(q, k, v, cu, pos)
    qr, kr = oracle.rope2d(q, pos), oracle.rope2d(k, pos)
    qh, sq, kh, sk, vh, sv = oracle.quant_e4m3(q, k, v, pos)
    for i in range(len(specs)):
        s0, s1 = int(cu[i]), int(cu[i + 1])
        for a in range(h):
            delta, bound = e4m3_attention_bounds(qr[s0:s1, a], kr[s0:s1, a], v[s0:s1, a],
                                                 sq[s0:s1, a], sk[a], sv[a], sc, l[a, s0:s1])
            assert np.all(np.abs(l8[a, s0:s1] - l[a, s0:s1]) <= delta + 1e-9)
            assert np.all(np.abs(o8[s0:s1, a] - o[s0:s1, a]) <= bound + 1e-12)
    assert np.abs(o8 - o).mean() < 0.1 * np.abs(o).mean()
