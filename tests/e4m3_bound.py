"""Rigorous per-row error bounds of the 8-bit (E4M3) attention forward against the
exact attention of the un-rounded operands (test helper, CPU, numpy).

The 8-bit variant rounds Q' (one power-of-two scale sq per row), K' (one scale sk
per head) and V (one scale sv per head) to E4M3, and each probability before it
weights V.  A value x rounded to E4M3 after division by its scale s moves by at
most half a quantum: |x~ - x| <= b(x) = 2^-4 |x| + 2^-10 s (the first term for
normal codes, three mantissa bits; the second for E4M3's subnormal range, whose
quantum is 2^-9 s).  From that, for query row j of one (sample, head):

  LSE: the rounded logits z~ = scale <q~, k~> differ from z = scale <q', k'> by at
       most delta_j = scale max_k sum_e (|q'_e| bk_e + bq_e |k'_e| + bq_e bk_e), so
       |LSE~_j - LSE_j| <= delta_j.
  O:   |O~_je - O_je| <= the sum of
       probability rounding   2^-4 g sum_k P_k |v~_ke| + 2^-10 sum_k |v~_ke| / l_lb,
       V rounding             g sum_k P_k (2^-4 |v_ke| + 2^-10 sv),
       the logits' change     (g - 1) sum_k P_k |v_ke|,
       with P the exact probabilities, g = e^(2 delta_j), |v~| <= (1 + 2^-4)|v| +
       2^-10 sv, and l_lb = sum_k exp(z_k - max_k z - 2 delta_j) a lower bound of the
       variant's normaliser (its running maximum never exceeds the largest rounded
       logit, and every rounded logit is within delta_j of the exact one).

The bounds do not depend on the order in which the variant visits the keys, on
its tile size or on how often its running maximum is raised: any implementation
of the steps above, tiled or not, satisfies them.
"""
from __future__ import annotations

import numpy as np


def e4m3_attention_bounds(Q, K, V, sq_rows, sk, sv, scale, lse_exact, block=512):
    """Q, K: the rotated operands of one (sample, head) [L, d]; V [L, d]; sq_rows
    [L] the Q row scales; sk, sv the head's K and V scales; lse_exact [L] the exact
    LSE.  Returns (delta [L], o_bound [L, d]).  Rows in blocks of `block`."""
    Q, K, V = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
    L = Q.shape[0]
    bk = 2.0 ** -4 * np.abs(K) + 2.0 ** -10 * sk
    aK = np.abs(K)
    aV = np.abs(V)
    vt = (1 + 2.0 ** -4) * aV + 2.0 ** -10 * sv
    vt_sum = vt.sum(axis=0)
    vr = 2.0 ** -4 * aV + 2.0 ** -10 * sv
    delta = np.empty(L)
    bound = np.empty_like(Q)
    for r0 in range(0, L, block):
        r1 = min(L, r0 + block)
        Qb = Q[r0:r1]
        bq = 2.0 ** -4 * np.abs(Qb) + 2.0 ** -10 * np.asarray(sq_rows[r0:r1])[:, None]
        dl = scale * (np.abs(Qb) @ bk.T + bq @ aK.T + bq @ bk.T).max(axis=1)
        z = scale * Qb @ K.T
        P = np.exp(z - np.asarray(lse_exact[r0:r1])[:, None])
        g = np.exp(2 * dl)[:, None]
        l_lb = np.exp(z - z.max(axis=1, keepdims=True) - 2 * dl[:, None]).sum(axis=1)
        bound[r0:r1] = (2.0 ** -4 * g * (P @ vt) + 2.0 ** -10 * vt_sum[None, :] / l_lb[:, None]
                        + g * (P @ vr) + (g - 1) * (P @ aV))
        delta[r0:r1] = dl
    return delta, bound
