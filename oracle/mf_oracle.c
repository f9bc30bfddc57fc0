/*
 * FP64 CPU oracle for packed native-resolution 2D-RoPE varlen attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg load this library.  It shares no code, header,
 * table or helper with the CUDA library and never calls it.
 *
 * What it computes, and where the pages define it:
 *  - Packing: Mage-Flow (arXiv 2607.19064), rcap.io post, training-step listing
 *    "native-resolution packed step" (pack(text_tokens + tokens, budget=50_000));
 *    paperlayer.ai summary §3.2.1 "Model Architecture and Native Packing" (variable
 *    length text and image sequences packed under a fixed token budget, each image
 *    keeping its native latent grid, no padding, no buckets).
 *  - Per-sample 2D RoPE: rcap.io post, same listing (per_sample_2d_rope(packed),
 *    "native positions"); ai.thesatyajit.com explainer, "A backbone that doesn't
 *    crop" (per-sample 2D rotary embeddings preserving each image's native layout).
 *    The pages give no formula; the problem statement fixes it: image token k of an
 *    H x W grid sits at (r, c) = (k div W, k mod W); text tokens at (0, 0); the first
 *    half of head_dim rotates by r, the second half by c; within a half, the pair
 *    (2j, 2j+1) rotates by theta = p * 10000^(-2j/(d/2)), j < d/4, with the usual
 *    rotary sign (x, y) -> (x cos - y sin, x sin + y cos).
 *  - Joint attention within a sample: paperlayer.ai §3.2.1 (concatenated text and
 *    image tokens use joint self-attention; cross-modal interaction through
 *    self-attention over the combined sequence), realised with variable-length
 *    kernels (rcap.io post, "Native-resolution packing"): non-causal softmax
 *    attention restricted to each sample's own tokens, scale 1/sqrt(d), sequence
 *    order [text; image].  LSE is the natural-log logsumexp of the scaled logits.
 *  - Backward: the training step of the rcap.io listing differentiates through
 *    the attention; the gradient is the exact derivative of the definitions above
 *    (softmax Jacobian and the transpose of the rotation, which is its inverse).
 *
 * Every loop follows the definition directly, one row at a time, in double: the
 * forward one query row at a time, the backward in two passes (one query row at a
 * time for dQ, one key row at a time for dK and dV, each recomputing the row's
 * probabilities from the LSE), OpenMP across rows.  No blocking, no fusion, no
 * online softmax.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_OK = 0, ORACLE_ERR = 1 };

/* ---------------------------------------------------------------- packing */
/*
 * specs[i] = {text_len, H, W}.  cu[0] = 0, cu[i+1] = cu[i] + text_len + H*W.
 * Within sample i, tokens [cu[i], cu[i]+text_len) are text at (0,0); token
 * cu[i]+text_len+k, 0 <= k < H*W, is image token k at (k div W, k mod W).
 * pos is [T][2] = (r, c).  pos may be NULL (sizes only).
 */
int oracle_pack(const int64_t* specs, int64_t n, int64_t* cu, int64_t* pos) {
  cu[0] = 0;
  for (int64_t i = 0; i < n; ++i) {
    int64_t t = specs[3 * i], H = specs[3 * i + 1], W = specs[3 * i + 2];
    if (t < 0 || H < 0 || W < 0) return ORACLE_ERR;
    int64_t L = t + H * W;
    if (pos) {
      for (int64_t k = 0; k < t; ++k) {
        pos[2 * (cu[i] + k)] = 0;
        pos[2 * (cu[i] + k) + 1] = 0;
      }
      for (int64_t k = 0; k < H * W; ++k) {
        pos[2 * (cu[i] + t + k)] = k / W;
        pos[2 * (cu[i] + t + k) + 1] = k % W;
      }
    }
    cu[i + 1] = cu[i] + L;
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------- RoPE */
/*
 * Rotate one head vector v[d] of a token at position (r, c) by +theta
 * (sign = +1) or -theta (sign = -1), writing out[d].
 */
static void rope_vec(const double* v, int64_t r, int64_t c, int64_t d, double base, int sign,
                     double* out) {
  int64_t half = d / 2, nfreq = d / 4;
  for (int64_t h = 0; h < 2; ++h) {
    double p = (h == 0) ? (double)r : (double)c;
    for (int64_t j = 0; j < nfreq; ++j) {
      double omega = pow(base, -2.0 * (double)j / (double)half);
      double theta = sign * p * omega;
      double x = v[h * half + 2 * j], y = v[h * half + 2 * j + 1];
      out[h * half + 2 * j] = x * cos(theta) - y * sin(theta);
      out[h * half + 2 * j + 1] = x * sin(theta) + y * cos(theta);
    }
  }
}

/* x, y: [T][heads][d]; pos [T][2]; sign +1 forward rotation, -1 inverse. */
int oracle_rope2d(const double* x, const int64_t* pos, int64_t T, int64_t heads, int64_t d,
                  double base, int sign, double* y) {
  if (d % 4 != 0) return ORACLE_ERR;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t a = 0; a < heads; ++a)
      rope_vec(x + (t * heads + a) * d, pos[2 * t], pos[2 * t + 1], d, base, sign,
               y + (t * heads + a) * d);
  return ORACLE_OK;
}

/* ------------------------------------------------------ attention forward */
/*
 * One query row (token tj, head a) of sample [s0, s0+L), rotated inputs qr, kr:
 *   S_k = scale * <q'_j, k'_k> over the keys k of the sample only,
 *   m = max_k S_k, LSE = m + ln sum_k exp(S_k - m),  O_j = sum_k exp(S_k - LSE) v_k.
 * srow is scratch of length L.
 */
static void attn_row(const double* qr, const double* kr, const double* v, int64_t s0, int64_t L,
                     int64_t tj, int64_t a, int64_t heads, int64_t d, double scale, double* srow,
                     double* oj, double* lse_j) {
  const double* qj = qr + (tj * heads + a) * d;
  double m = -INFINITY;
  for (int64_t kk = 0; kk < L; ++kk) {
    const double* kv = kr + ((s0 + kk) * heads + a) * d;
    double acc = 0.0;
    for (int64_t e = 0; e < d; ++e) acc += qj[e] * kv[e];
    srow[kk] = scale * acc;
    if (srow[kk] > m) m = srow[kk];
  }
  double l = 0.0;
  for (int64_t kk = 0; kk < L; ++kk) l += exp(srow[kk] - m);
  double lj = m + log(l);
  *lse_j = lj;
  for (int64_t e = 0; e < d; ++e) oj[e] = 0.0;
  for (int64_t kk = 0; kk < L; ++kk) {
    double p = exp(srow[kk] - lj);
    const double* vk = v + ((s0 + kk) * heads + a) * d;
    for (int64_t e = 0; e < d; ++e) oj[e] += p * vk[e];
  }
}

/* Index of the sample holding each token: samp[t] = i for cu[i] <= t < cu[i+1]
 * (zero-length samples hold no token).  Returns a malloc'd int64[T] or NULL. */
static int64_t* sample_of_tokens(const int64_t* cu, int64_t n, int64_t T) {
  int64_t* samp = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T + 1));
  if (!samp) return NULL;
  for (int64_t i = 0; i < n; ++i)
    for (int64_t t = cu[i]; t < cu[i + 1]; ++t) samp[t] = i;
  return samp;
}

static int rotate_qk(const double* q, const double* k, const int64_t* pos, int64_t T,
                     int64_t heads, int64_t d, double base, double** qr, double** kr) {
  *qr = (double*)malloc(sizeof(double) * (size_t)(T * heads * d + 1));
  *kr = (double*)malloc(sizeof(double) * (size_t)(T * heads * d + 1));
  if (!*qr || !*kr) { free(*qr); free(*kr); return ORACLE_ERR; }
  if (pos) {
    oracle_rope2d(q, pos, T, heads, d, base, +1, *qr);
    oracle_rope2d(k, pos, T, heads, d, base, +1, *kr);
  } else {
    memcpy(*qr, q, sizeof(double) * (size_t)(T * heads * d));
    memcpy(*kr, k, sizeof(double) * (size_t)(T * heads * d));
  }
  return ORACLE_OK;
}

/*
 * Inputs un-rotated q, k, v [T][heads][d]; cu [n+1]; pos [T][2] or NULL (no
 * rotation).  Outputs o [T][heads][d], lse [heads][T]: every row of every sample
 * and head, each by attn_row.  q' = R(theta) q and k' = R(theta) k are formed
 * first, exactly as defined above.
 */
int oracle_attn_fwd(const double* q, const double* k, const double* v, const int64_t* cu,
                    int64_t n, const int64_t* pos, int64_t T, int64_t heads, int64_t d,
                    double scale, double base, double* o, double* lse) {
  double *qr, *kr;
  if (rotate_qk(q, k, pos, T, heads, d, base, &qr, &kr) != ORACLE_OK) return ORACLE_ERR;
  int64_t* samp = sample_of_tokens(cu, n, T);
  if (!samp) { free(qr); free(kr); return ORACLE_ERR; }
  /* every (token, head) row on its own: row r is token r / heads, head r % heads */
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t r = 0; r < T * heads; ++r) {
    int64_t tj = r / heads, a = r % heads, i = samp[tj];
    int64_t s0 = cu[i], L = cu[i + 1] - cu[i];
    double* srow = (double*)malloc(sizeof(double) * (size_t)L);
    attn_row(qr, kr, v, s0, L, tj, a, heads, d, scale, srow, o + r * d, lse + a * T + tj);
    free(srow);
  }
  free(samp);
  free(qr);
  free(kr);
  return ORACLE_OK;
}

/*
 * The same definition restricted to m requested rows: rows[r] = (token, head).
 * Writes o_rows [m][d] and lse_rows [m].  Rotation of q and k is applied to the
 * whole input (as above) before the rows are evaluated.
 */
int oracle_attn_fwd_rows(const double* q, const double* k, const double* v, const int64_t* cu,
                         int64_t n, const int64_t* pos, int64_t T, int64_t heads, int64_t d,
                         double scale, double base, const int64_t* rows, int64_t m,
                         double* o_rows, double* lse_rows) {
  double *qr, *kr;
  if (rotate_qk(q, k, pos, T, heads, d, base, &qr, &kr) != ORACLE_OK) return ORACLE_ERR;
  int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < m; ++r) {
    int64_t tj = rows[2 * r], a = rows[2 * r + 1];
    int64_t i = 0;
    while (i < n && cu[i + 1] <= tj) ++i; /* the sample holding token tj */
    if (i >= n || tj < 0 || a < 0 || a >= heads) { err = ORACLE_ERR; continue; }
    int64_t s0 = cu[i], L = cu[i + 1] - cu[i];
    double* srow = (double*)malloc(sizeof(double) * (size_t)L);
    attn_row(qr, kr, v, s0, L, tj, a, heads, d, scale, srow, o_rows + r * d, lse_rows + r);
    free(srow);
  }
  free(qr);
  free(kr);
  return err;
}

/* ----------------------------------------------------- attention backward */
/*
 * Gradients of the forward above with respect to the un-rotated q, k and v, for
 * the upstream gradient d_o [T][heads][d].  Per sample and head:
 *   O, LSE recomputed as in the forward;  D_j = <dO_j, O_j>;
 *   P_jk = exp(S_jk - LSE_j);  dV_k = sum_j P_jk dO_j;
 *   dP_jk = <dO_j, v_k>;  dS_jk = P_jk (dP_jk - D_j);
 *   dQ'_j = scale sum_k dS_jk k'_k;  dK'_k = scale sum_j dS_jk q'_j;
 *   dQ = R(-theta) dQ',  dK = R(-theta) dK'  (R is orthogonal: R^T = R(-theta)).
 */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* d_o,
                    const int64_t* cu, int64_t n, const int64_t* pos, int64_t T, int64_t heads,
                    int64_t d, double scale, double base, double* dq, double* dk, double* dv) {
  size_t N = (size_t)(T * heads * d);
  double *qr = NULL, *kr = NULL;
  if (rotate_qk(q, k, pos, T, heads, d, base, &qr, &kr) != ORACLE_OK) return ORACLE_ERR;
  double* o = (double*)malloc(sizeof(double) * (N + 1));
  double* lse = (double*)malloc(sizeof(double) * (size_t)(heads * T + 1));
  double* D = (double*)malloc(sizeof(double) * (size_t)(heads * T + 1));
  double* dqr = (double*)calloc(N + 1, sizeof(double));
  double* dkr = (double*)calloc(N + 1, sizeof(double));
  int64_t* samp = sample_of_tokens(cu, n, T);
  if (!qr || !kr || !o || !lse || !D || !dqr || !dkr || !samp) {
    free(qr); free(kr); free(o); free(lse); free(D); free(dqr); free(dkr); free(samp);
    return ORACLE_ERR;
  }
  oracle_attn_fwd(q, k, v, cu, n, pos, T, heads, d, scale, base, o, lse);
  memset(dv, 0, sizeof(double) * N);
  /* D_j = <dO_j, O_j> of every (token, head) row r (token r / heads, head r % heads) */
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < T * heads; ++r) {
    double acc = 0.0;
    for (int64_t e = 0; e < d; ++e) acc += d_o[r * d + e] * o[r * d + e];
    D[(r % heads) * T + r / heads] = acc;
  }
  /* Pass 1, one query row j at a time: over the keys k of its sample,
   * P_jk = exp(S_jk - LSE_j), dP_jk = <dO_j, v_k>, dS_jk = P_jk (dP_jk - D_j), and
   * dQ'_j = scale sum_k dS_jk k'_k. */
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t r = 0; r < T * heads; ++r) {
    int64_t tj = r / heads, a = r % heads, i = samp[tj];
    int64_t s0 = cu[i], L = cu[i + 1] - cu[i];
    const double* qj = qr + r * d;
    const double* doj = d_o + r * d;
    double* dqj = dqr + r * d;
    const double lj = lse[a * T + tj], Dj = D[a * T + tj];
    for (int64_t kk = 0; kk < L; ++kk) {
      int64_t rk = ((s0 + kk) * heads + a) * d;
      double acc = 0.0, dp = 0.0;
      for (int64_t e = 0; e < d; ++e) {
        acc += qj[e] * kr[rk + e];
        dp += doj[e] * v[rk + e];
      }
      const double p = exp(scale * acc - lj);
      const double ds = p * (dp - Dj);
      for (int64_t e = 0; e < d; ++e) dqj[e] += scale * ds * kr[rk + e];
    }
  }
  /* Pass 2, one key row k at a time: over the queries j of its sample, the same
   * P_jk and dS_jk, and dV_k = sum_j P_jk dO_j, dK'_k = scale sum_j dS_jk q'_j. */
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t r = 0; r < T * heads; ++r) {
    int64_t tk = r / heads, a = r % heads, i = samp[tk];
    int64_t s0 = cu[i], L = cu[i + 1] - cu[i];
    const double* kk_r = kr + r * d;
    const double* vk = v + r * d;
    double* dvk = dv + r * d;
    double* dkk = dkr + r * d;
    for (int64_t jj = 0; jj < L; ++jj) {
      int64_t tq = s0 + jj, rq = (tq * heads + a) * d;
      double acc = 0.0, dp = 0.0;
      for (int64_t e = 0; e < d; ++e) {
        acc += qr[rq + e] * kk_r[e];
        dp += d_o[rq + e] * vk[e];
      }
      const double pk = exp(scale * acc - lse[a * T + tq]);
      const double dsk = pk * (dp - D[a * T + tq]);
      for (int64_t e = 0; e < d; ++e) {
        dvk[e] += pk * d_o[rq + e];
        dkk[e] += scale * dsk * qr[rq + e];
      }
    }
  }
  if (pos) {
    oracle_rope2d(dqr, pos, T, heads, d, base, -1, dq);
    oracle_rope2d(dkr, pos, T, heads, d, base, -1, dk);
  } else {
    memcpy(dq, dqr, sizeof(double) * N);
    memcpy(dk, dkr, sizeof(double) * N);
  }
  free(qr); free(kr); free(o); free(lse); free(D); free(dqr); free(dkr); free(samp);
  return ORACLE_OK;
}

/* ------------------------------------------------ packed CFG + Euler step */
/*
 * Packed classifier-free guidance (paperlayer.ai summary section 3.2.1 and
 * hyper.ai "Experiment": the conditional and unconditional branches are two
 * samples of one packed forward pass, which leaves the denoising trajectory
 * unchanged) followed by one step of the rectified-flow sampler.  The pages give
 * the flow-matching objective (hyper.ai "Method": z_t = (1 - t) z + t eps, the
 * network regresses z - eps), so dz_t/dt = -(z - eps) = -v and a step from t to
 * t - dt is z <- z + dt * v.  They print no guidance formula; the standard
 * combination v = v_u + g (v_c - v_u) is taken.
 *
 * specs[2p], specs[2p+1] = {text_len, H, W} of pair p's conditional and
 * unconditional samples (same H, W); the pack is all 2*pairs samples in that
 * order.  v: [T][C] model output of the packed batch.  z_in, z_out: [N][C] with
 * N = sum_p H_p W_p, pair p's image latent rows in pair order.
 */
int oracle_cfg_euler(const double* v, const int64_t* specs, int64_t pairs, int64_t C, double g,
                     double dt, const double* z_in, double* z_out) {
  int64_t start = 0, zrow = 0;
  for (int64_t p = 0; p < pairs; ++p) {
    const int64_t* sc = specs + 6 * p;
    const int64_t* su = sc + 3;
    if (sc[1] != su[1] || sc[2] != su[2]) return ORACLE_ERR;
    const int64_t Lc = sc[0] + sc[1] * sc[2], Lu = su[0] + su[1] * su[2];
    const int64_t img_c = start + sc[0];        /* first image token of the cond sample */
    const int64_t img_u = start + Lc + su[0];   /* first image token of the uncond sample */
    const int64_t n_img = sc[1] * sc[2];
    for (int64_t k = 0; k < n_img; ++k) {
      for (int64_t e = 0; e < C; ++e) {
        const double vc = v[(img_c + k) * C + e];
        const double vu = v[(img_u + k) * C + e];
        const double vg = vu + g * (vc - vu);
        z_out[(zrow + k) * C + e] = z_in[(zrow + k) * C + e] + dt * vg;
      }
    }
    start += Lc + Lu;
    zrow += n_img;
  }
  return ORACLE_OK;
}

/* ----------------------------------- adaptive LayerNorm and gated residual */
/*
 * The Transformer-side fused chain around the packed attention (paperlayer.ai
 * summary section 3.3 "Training Infrastructure": adaptive normalization, rotary
 * embeddings and gated residual updates are fused).  The pages print no formula;
 * the reading is the DiT-style block: per sample s, conditioning vectors shift_s,
 * scale_s, gate_s of width Dm; for every token t of sample s (from cu_seqlens)
 *   y_t = LN(x_t) * (1 + scale_s) + shift_s,   LN(x) = (x - mean) / sqrt(var + eps)
 * with the biased variance over the Dm features and no affine parameters, and
 *   out_t = x_t + gate_s * h_t
 * for the block branch output h.  x, h, y, out: [T][Dm]; shift, scale, gate: [n][Dm].
 */
int oracle_adaln(const double* x, const int64_t* cu, int64_t n, int64_t Dm, const double* shift,
                 const double* scale, double eps, double* y) {
  for (int64_t s = 0; s < n; ++s) {
    for (int64_t t = cu[s]; t < cu[s + 1]; ++t) {
      const double* xr = x + t * Dm;
      double mean = 0.0;
      for (int64_t e = 0; e < Dm; ++e) mean += xr[e];
      mean /= (double)Dm;
      double var = 0.0;
      for (int64_t e = 0; e < Dm; ++e) var += (xr[e] - mean) * (xr[e] - mean);
      var /= (double)Dm;
      const double rstd = 1.0 / sqrt(var + eps);
      for (int64_t e = 0; e < Dm; ++e)
        y[t * Dm + e] = (xr[e] - mean) * rstd * (1.0 + scale[s * Dm + e]) + shift[s * Dm + e];
    }
  }
  return ORACLE_OK;
}

int oracle_gated_residual(const double* x, const double* h, const int64_t* cu, int64_t n,
                          int64_t Dm, const double* gate, double* out) {
  for (int64_t s = 0; s < n; ++s)
    for (int64_t t = cu[s]; t < cu[s + 1]; ++t)
      for (int64_t e = 0; e < Dm; ++e)
        out[t * Dm + e] = x[t * Dm + e] + gate[s * Dm + e] * h[t * Dm + e];
  return ORACLE_OK;
}

/* ------------------------------------ frame-aware 3D packing and RoPE */
/*
 * Editing packs (hyper.ai summary "Method": for editing the 2D rotary embedding is
 * extended with a frame dimension that tells source and target visual tokens
 * apart; paperlayer.ai summary 3.2.2: editing concatenates the text conditioning
 * with the source-image latents and the noisy target latents).  Reading taken
 * (the pages give no layout or frequencies): sample i is [text; source grid;
 * target grid], specs[i] = {text_len, Hs, Ws, Ht, Wt}; pos is [T][3] = (f, r, c):
 * text (0, 0, 0), source token k at (0, k div Ws, k mod Ws), target token k at
 * (1, k div Wt, k mod Wt).
 */
int oracle_pack3d(const int64_t* specs, int64_t n, int64_t* cu, int64_t* pos) {
  cu[0] = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t* s = specs + 5 * i;
    for (int q = 0; q < 5; ++q)
      if (s[q] < 0) return ORACLE_ERR;
    const int64_t t = s[0], Hs = s[1], Ws = s[2], Ht = s[3], Wt = s[4];
    const int64_t L = t + Hs * Ws + Ht * Wt;
    if (pos) {
      int64_t tok = cu[i];
      for (int64_t k = 0; k < t; ++k, ++tok) {
        pos[3 * tok] = 0;
        pos[3 * tok + 1] = 0;
        pos[3 * tok + 2] = 0;
      }
      for (int64_t k = 0; k < Hs * Ws; ++k, ++tok) {
        pos[3 * tok] = 0;
        pos[3 * tok + 1] = k / Ws;
        pos[3 * tok + 2] = k % Ws;
      }
      for (int64_t k = 0; k < Ht * Wt; ++k, ++tok) {
        pos[3 * tok] = 1;
        pos[3 * tok + 1] = k / Wt;
        pos[3 * tok + 2] = k % Wt;
      }
    }
    cu[i + 1] = cu[i] + L;
  }
  return ORACLE_OK;
}

/*
 * 3D rotation of one head vector.  Reading taken: head_dim is split into three
 * contiguous slices, frame [0, d/4), row [d/4, 5d/8), column [5d/8, d) (for
 * d = 128: 16, 24 and 24 rotary pairs); within a slice of width w, the pair
 * (2j, 2j+1) of the slice rotates by p * base^(-2j / w), p the token's
 * coordinate on that axis -- the per-axis rule of the 2D embedding with the slice
 * width in place of d/2.
 */
static void rope3_vec(const double* v, const int64_t* p3, int64_t d, double base, int sign,
                      double* out) {
  const int64_t width[3] = {d / 4, 3 * d / 8, 3 * d / 8};
  int64_t off = 0;
  for (int a = 0; a < 3; ++a) {
    const double p = (double)p3[a];
    for (int64_t j = 0; j < width[a] / 2; ++j) {
      const double omega = pow(base, -2.0 * (double)j / (double)width[a]);
      const double theta = sign * p * omega;
      const double x = v[off + 2 * j], y = v[off + 2 * j + 1];
      out[off + 2 * j] = x * cos(theta) - y * sin(theta);
      out[off + 2 * j + 1] = x * sin(theta) + y * cos(theta);
    }
    off += width[a];
  }
}

/* x, y: [T][heads][d] with d a multiple of 16; pos [T][3]; sign +1 / -1. */
int oracle_rope3d(const double* x, const int64_t* pos, int64_t T, int64_t heads, int64_t d,
                  double base, int sign, double* y) {
  if (d % 16 != 0) return ORACLE_ERR;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t a = 0; a < heads; ++a)
      rope3_vec(x + (t * heads + a) * d, pos + 3 * t, d, base, sign, y + (t * heads + a) * d);
  return ORACLE_OK;
}

/* ------------------------------------------------- e4m3 forward variant */
/*
 * The 8-bit variant of the attention forward.  The pages give no low-precision
 * recipe (it is an engineering variant of the same attention); every step below
 * is this variant's own definition, written in the order the variant takes it.
 *
 * E4M3 is the OCP 8-bit floating-point format: a sign bit, 4 exponent bits with
 * bias 7 and 3 mantissa bits; normals (1 + m/8) 2^(e-7) for e = 1..15, except that
 * e = 15 with m = 7 is NaN, so the largest finite value is 448; subnormals
 * (m/8) 2^-6; no infinities.  oracle_e4m3 rounds a double to the nearest such
 * value, ties to the even mantissa, and saturates beyond +-448 (the
 * "satfinite" conversion).
 */
double oracle_e4m3(double x) {
  if (x != x) return x;
  const double a = fabs(x);
  if (a >= 448.0) return x < 0 ? -448.0 : 448.0;
  if (a == 0.0) return x;
  int ex;
  frexp(a, &ex);             /* a = f 2^ex, f in [0.5, 1): binade [2^(ex-1), 2^ex) */
  int e = ex - 1;
  if (e < -6) e = -6;        /* subnormals share the quantum of the lowest binade */
  const double quantum = ldexp(1.0, e - 3);
  const double r = nearbyint(a / quantum) * quantum; /* default mode: ties to even */
  const double out = r > 448.0 ? 448.0 : r;
  return x < 0 ? -out : out;
}

/*
 * Scale of a block whose largest magnitude is A: the smallest power of two s with
 * A / s <= 448 (0 when A = 0).  A power of two makes x / s exact, so the rounding
 * to e4m3 is the only rounding of the operands.  With A = m 2^p, m in [1, 2):
 * s = 2^(p - 8) when m <= 1.75 (A / s = 256 m <= 448), else 2^(p - 7).
 */
static double e4m3_scale(double A) {
  if (!(A > 0.0)) return 0.0;
  int ex;
  const double f = frexp(A, &ex); /* A = f 2^ex, f in [0.5, 1): m = 2f, p = ex - 1 */
  return ldexp(1.0, (ex - 1) - 8 + (2.0 * f > 1.75 ? 1 : 0));
}

/*
 * Quantisation of the operands (their values as doubles; the codes are these
 * values' e4m3 encodings).  Inputs: the rotated qr, kr, the un-rotated k and v,
 * all [T][heads][d].  round = 0 replaces e4m3 rounding by the identity.
 *  Q: per (token, head) row, sq = e4m3_scale(max_e |q'_e|), qh = e4m3(q' / sq)
 *     (0 where sq = 0).
 *  K: per head, sk = e4m3_scale of the largest pair norm
 *     sqrt(k_2P^2 + k_2P+1^2) of the UN-rotated k over the head's tokens and
 *     rotary pairs (2P, 2P+1).  A rotation keeps each pair's norm, so the norm
 *     bounds every rotated component at every position: kh = e4m3(k' / sk).
 *  V: per head, sv = e4m3_scale(max |v|), vh = e4m3(v / sv).
 * Outputs qh, kh, vh [T][heads][d]; sq [T][heads]; sk, sv [heads].
 */
int oracle_quant_e4m3(const double* qr, const double* k, const double* kr, const double* v,
                      int64_t T, int64_t heads, int64_t d, int round, double* qh, double* sq,
                      double* kh, double* sk, double* vh, double* sv) {
  if (d % 2 != 0) return ORACLE_ERR;
  for (int64_t a = 0; a < heads; ++a) {
    double kmax = 0.0, vmax = 0.0;
    for (int64_t t = 0; t < T; ++t) {
      const double* kk = k + (t * heads + a) * d;
      const double* vv = v + (t * heads + a) * d;
      for (int64_t e = 0; e < d; e += 2) {
        const double nrm = sqrt(kk[e] * kk[e] + kk[e + 1] * kk[e + 1]);
        if (nrm > kmax) kmax = nrm;
      }
      for (int64_t e = 0; e < d; ++e)
        if (fabs(vv[e]) > vmax) vmax = fabs(vv[e]);
    }
    sk[a] = e4m3_scale(kmax);
    sv[a] = e4m3_scale(vmax);
  }
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t a = 0; a < heads; ++a) {
      const int64_t row = (t * heads + a) * d;
      double qmax = 0.0;
      for (int64_t e = 0; e < d; ++e)
        if (fabs(qr[row + e]) > qmax) qmax = fabs(qr[row + e]);
      const double s = e4m3_scale(qmax);
      sq[t * heads + a] = s;
      for (int64_t e = 0; e < d; ++e) {
        const double xq = s > 0 ? qr[row + e] / s : 0.0;
        const double xk = sk[a] > 0 ? kr[row + e] / sk[a] : 0.0;
        const double xv = sv[a] > 0 ? v[row + e] / sv[a] : 0.0;
        qh[row + e] = round ? oracle_e4m3(xq) : xq;
        kh[row + e] = round ? oracle_e4m3(xk) : xk;
        vh[row + e] = round ? oracle_e4m3(xv) : xv;
      }
    }
  return ORACLE_OK;
}

/*
 * Attention of one sample from the quantised operands, one query row at a time,
 * with the probabilities themselves rounded to e4m3 before they weight V.  The
 * rounding of a probability depends on the reference it is taken against, so the
 * row follows the variant's steps over keys in tiles of 128 from the sample's
 * first key (base-2 logits and a running maximum that lags by at most 8):
 *   x_k   = log2(e) * scale * sq_j * sk * <qh_j, kh_k>          (all keys of the tile)
 *   tile 0 sets m = max_k x_k;  a later tile replaces m by its own maximum M only
 *         when M > m + 8, and then multiplies l and the accumulator by 2^(m - M);
 *   p_k   = 2^(x_k - m)           (at most 2^8 < 448: no saturation)
 *   l    += p_k;   acc += e4m3(p_k) * vh_k
 * and at the end O_j = sv * acc / l, LSE_j = ln(2) * (m + log2 l).
 * With round = 0 nothing is rounded and O, LSE are the exact attention of the
 * (unrounded) scaled operands.
 */
int oracle_attn_fwd_e4m3(const double* qh, const double* sq, const double* kh, const double* sk,
                         const double* vh, const double* sv, const int64_t* cu, int64_t n,
                         int64_t T, int64_t heads, int64_t d, double scale, int round, double* o,
                         double* lse) {
  const double log2e = 1.4426950408889634074;
  const int64_t tile = 128;
  int64_t npairs = n * heads;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t pr = 0; pr < npairs; ++pr) {
    const int64_t i = pr / heads, a = pr % heads;
    const int64_t s0 = cu[i], L = cu[i + 1] - cu[i];
    if (L <= 0) continue;
    double* x = (double*)malloc(sizeof(double) * (size_t)tile);
    double* acc = (double*)malloc(sizeof(double) * (size_t)d);
    for (int64_t j = s0; j < s0 + L; ++j) {
      const double* qj = qh + (j * heads + a) * d;
      const double c = log2e * scale * sq[j * heads + a] * sk[a];
      double m = 0.0, l = 0.0;
      for (int64_t e = 0; e < d; ++e) acc[e] = 0.0;
      for (int64_t t0 = 0; t0 < L; t0 += tile) {
        const int64_t nk = L - t0 < tile ? L - t0 : tile;
        double M = -INFINITY;
        for (int64_t kk = 0; kk < nk; ++kk) {
          const double* kv = kh + ((s0 + t0 + kk) * heads + a) * d;
          double dot = 0.0;
          for (int64_t e = 0; e < d; ++e) dot += qj[e] * kv[e];
          x[kk] = c * dot;
          if (x[kk] > M) M = x[kk];
        }
        if (t0 == 0) {
          m = M;
        } else if (M > m + 8.0) {
          const double f = exp2(m - M);
          l *= f;
          for (int64_t e = 0; e < d; ++e) acc[e] *= f;
          m = M;
        }
        for (int64_t kk = 0; kk < nk; ++kk) {
          const double p = exp2(x[kk] - m);
          const double pr8 = round ? oracle_e4m3(p) : p;
          const double* vk = vh + ((s0 + t0 + kk) * heads + a) * d;
          l += p;
          for (int64_t e = 0; e < d; ++e) acc[e] += pr8 * vk[e];
        }
      }
      for (int64_t e = 0; e < d; ++e) o[(j * heads + a) * d + e] = sv[a] * acc[e] / l;
      lse[a * T + j] = (m + log2(l)) * 0.69314718055994530942;
    }
    free(x);
    free(acc);
  }
  return ORACLE_OK;
}

/* oracle_e4m3 applied to n values. */
int oracle_e4m3_array(const double* x, int64_t n, double* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_e4m3(x[i]);
  return ORACLE_OK;
}
