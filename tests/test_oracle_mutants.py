"""Plant plausible mistakes in copies of the oracle source (CPU only) and check
that at least one pin fails for each: the pins would catch such a slip in the
oracle itself."""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mf_oracle.c")

# (name, exact source fragment, replacement)
MUTANTS = [
    ("rope_sign", "out[h * half + 2 * j] = x * cos(theta) - y * sin(theta);",
     "out[h * half + 2 * j] = x * cos(theta) + y * sin(theta);"),
    ("rope_freq_exponent", "pow(base, -2.0 * (double)j / (double)half)",
     "pow(base, -1.0 * (double)j / (double)half)"),
    ("rope_rows_cols_swapped", "double p = (h == 0) ? (double)r : (double)c;",
     "double p = (h == 0) ? (double)c : (double)r;"),
    ("pack_col_major_flatten", "pos[2 * (cu[i] + t + k) + 1] = k % W;",
     "pos[2 * (cu[i] + t + k) + 1] = k / (H > 0 ? H : 1);"),
    ("pack_one_based_rows", "pos[2 * (cu[i] + t + k)] = k / W;",
     "pos[2 * (cu[i] + t + k)] = k / W + 1;"),
    ("attn_no_scale", "srow[kk] = scale * acc;", "srow[kk] = acc;"),
    ("attn_lse_without_max", "double lj = m + log(l);", "double lj = log(l);"),
    ("attn_unnormalised", "double p = exp(srow[kk] - lj);", "double p = exp(srow[kk] - m);"),
    ("bwd_missing_D", "const double ds = p * (dp - Dj);", "const double ds = p * dp;"),
    ("bwd_missing_D_key_pass", "const double dsk = pk * (dp - D[a * T + tq]);",
     "const double dsk = pk * dp;"),
    ("bwd_dk_forward_rotation", "oracle_rope2d(dkr, pos, T, heads, d, base, -1, dk);",
     "oracle_rope2d(dkr, pos, T, heads, d, base, +1, dk);"),
    ("bwd_dq_forward_rotation", "oracle_rope2d(dqr, pos, T, heads, d, base, -1, dq);",
     "oracle_rope2d(dqr, pos, T, heads, d, base, +1, dq);"),
    ("bwd_dv_own_row", "dvk[e] += pk * d_o[rq + e];", "dvk[e] += pk * d_o[r * d + e];"),
    ("bwd_dk_missing_scale", "dkk[e] += scale * dsk * qr[rq + e];", "dkk[e] += dsk * qr[rq + e];"),
    ("bwd_dq_unrotated_keys", "dqj[e] += scale * ds * kr[rk + e];",
     "dqj[e] += scale * ds * k[rk + e];"),
    ("bwd_key_pass_wrong_lse", "const double pk = exp(scale * acc - lse[a * T + tq]);",
     "const double pk = exp(scale * acc - lse[a * T + tk]);"),
    ("cfg_branches_swapped", "const double vg = vu + g * (vc - vu);",
     "const double vg = vc + g * (vu - vc);"),
    ("cfg_no_text_offset", "const int64_t img_c = start + sc[0];",
     "const int64_t img_c = start;"),
    ("cfg_step_sign", "z_in[(zrow + k) * C + e] + dt * vg;", "z_in[(zrow + k) * C + e] - dt * vg;"),
    ("adaln_unbiased_variance", "var /= (double)Dm;", "var /= (double)(Dm - 1);"),
    ("adaln_scale_without_one", "* (1.0 + scale[s * Dm + e]) + shift[s * Dm + e];",
     "* scale[s * Dm + e] + shift[s * Dm + e];"),
    ("adaln_first_sample_shift", "* (1.0 + scale[s * Dm + e]) + shift[s * Dm + e];",
     "* (1.0 + scale[s * Dm + e]) + shift[e];"),
    ("pack3d_target_frame_zero", "        pos[3 * tok] = 1;", "        pos[3 * tok] = 0;"),
    ("pack3d_source_col_major", "pos[3 * tok + 2] = k % Ws;", "pos[3 * tok + 2] = k / (Hs > 0 ? Hs : 1);"),
    ("rope3d_frame_slice_d8", "const int64_t width[3] = {d / 4, 3 * d / 8, 3 * d / 8};",
     "const int64_t width[3] = {d / 8, 7 * d / 16, 7 * d / 16};"),
    ("rope3d_freq_over_d", "pow(base, -2.0 * (double)j / (double)width[a])",
     "pow(base, -2.0 * (double)j / (double)d)"),
    ("rope3d_sign", "out[off + 2 * j] = x * cos(theta) - y * sin(theta);",
     "out[off + 2 * j] = x * cos(theta) + y * sin(theta);"),
    ("gated_first_sample_gate", "out[t * Dm + e] = x[t * Dm + e] + gate[s * Dm + e] * h[t * Dm + e];",
     "out[t * Dm + e] = x[t * Dm + e] + gate[e] * h[t * Dm + e];"),
    ("e4m3_truncates", "nearbyint(a / quantum) * quantum", "floor(a / quantum) * quantum"),
    ("e4m3_no_subnormal_floor", "if (e < -6) e = -6;", "if (e < -9) e = -9;"),
    ("e4m3_two_mantissa_bits", "ldexp(1.0, e - 3)", "ldexp(1.0, e - 2)"),
    ("e4m3_scale_threshold", "(2.0 * f > 1.75 ? 1 : 0)", "(2.0 * f > 1.5 ? 1 : 0)"),
    ("e4m3_scale_not_power_of_two", "  if (!(A > 0.0)) return 0.0;\n  int ex;",
     "  if (!(A > 0.0)) return 0.0;\n  if (A > 0.0) return A / 448.0;\n  int ex;"),
    ("quant_k_scale_from_max_abs", "const double nrm = sqrt(kk[e] * kk[e] + kk[e + 1] * kk[e + 1]);",
     "const double nrm = fabs(kk[e]) > fabs(kk[e + 1]) ? fabs(kk[e]) : fabs(kk[e + 1]);"),
    ("quant_q_scale_per_head", "if (fabs(qr[row + e]) > qmax) qmax = fabs(qr[row + e]);",
     "if (fabs(qr[e]) > qmax) qmax = fabs(qr[e]);"),
    ("attn_e4m3_lse_natural_log_of_l", "lse[a * T + j] = (m + log2(l)) * 0.69314718055994530942;",
     "lse[a * T + j] = (m + log(l)) * 0.69314718055994530942;"),
    ("attn_e4m3_l_not_rescaled", "          l *= f;\n", "\n"),
    ("attn_e4m3_rescale_inverted", "const double f = exp2(m - M);", "const double f = exp2(M - m);"),
    ("attn_e4m3_missing_v_scale", "o[(j * heads + a) * d + e] = sv[a] * acc[e] / l;",
     "o[(j * heads + a) * d + e] = acc[e] / l;"),
    ("attn_e4m3_missing_k_scale", "const double c = log2e * scale * sq[j * heads + a] * sk[a];",
     "const double c = log2e * scale * sq[j * heads + a];"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"fragment for {name} not found exactly once"
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_source(str(path), str(tmp_path / f"lib_{name}.so"))
    failed = []
    for pin in [n for n in dir(pins) if n.startswith("pin_")]:
        try:
            getattr(pins, pin)(so=so)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin)
    assert failed, f"planted mistake {name} passed every pin"
