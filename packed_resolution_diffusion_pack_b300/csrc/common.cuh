// Shared internal definitions of the CUDA library: workspace layout, kernel
// launch declarations and host helpers.  Not part of the public ABI (mf.h).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mf.h"

namespace mf {

constexpr double kRopeBase = 10000.0;
constexpr int kMaxPairs = 64;  // rotary pairs (d/2) for head_dim 128

// Rotary angle of every pair of a head vector: pair P (dims 2P, 2P+1) rotates by
// theta = pos[axis[P]] * omega[P], pos being the token's naxes coordinates.  omega
// is computed on the host in double and split into fp32 hi + lo parts, so a kernel
// can form theta to ~2^-40 relative before taking sin/cos.
//  naxes = 2 (native-resolution packs): pos = (r, c); pairs [0, d/4) rotate by r,
//    [d/4, d/2) by c, pair j of a half with omega = base^(-2j/(d/2)).
//  naxes = 3 (editing packs): pos = (f, r, c); the frame, row and column slices
//    are d/4, 3d/8 and 3d/8 dims wide; pair j of a slice of width w has
//    omega = base^(-2j/w).
struct RopeFreqs {
  float omega[kMaxPairs];
  float omega_lo[kMaxPairs];
  int8_t axis[kMaxPairs];
  int32_t naxes;
};
RopeFreqs make_rope_freqs(int head_dim, int naxes);

// sin and cos of theta = sign * p * omega (p a small integer as float): the fp32
// product's rounding error is recovered exactly with an FMA and added, together
// with p * omega_lo, as a first-order correction to sincosf(theta_hi).
__device__ __forceinline__ void rope_sincos(float p, float w_hi, float w_lo, float sign,
                                            float* s, float* c) {
  const float th = p * w_hi;
  const float err = fmaf(p, w_hi, -th) + p * w_lo;
  float s0, c0;
  sincosf(sign * th, &s0, &c0);
  const float e = sign * err;
  *s = fmaf(e, c0, s0);
  *c = fmaf(-e, s0, c0);
}

// The same angle with a cheaper evaluation, for epilogues that rotate many
// values per thread: theta = p * omega as above (hi part + first-order error),
// Cody-Waite reduction of the hi part by pi/2 with a three-part constant (the
// first two parts carry 12 trailing zero bits, so k * part is exact for
// |k| < 2^12), then the hardware sine / cosine approximations on
// |r| <= pi/4 (absolute error ~2^-21 there) and the quadrant's sign swap.
__device__ __forceinline__ void rope_sincos_fast(float p, float w_hi, float w_lo, float sign,
                                                 float* s, float* c) {
  constexpr float kPio2Hi = 1.5703125f;                 // 0x1.92p+0
  constexpr float kPio2Mid = 4.837512969970703e-04f;    // 0x1.fb4p-12
  constexpr float kPio2Lo = 7.549790126404332e-08f;     // 0x1.4442d2p-24
  constexpr float kTwoOverPi = 0.6366197466850281f;
  const float th = p * w_hi;
  const float err = fmaf(p, w_hi, -th) + p * w_lo;
  const float k = rintf(th * kTwoOverPi);
  float r = fmaf(-k, kPio2Hi, th);
  r = fmaf(-k, kPio2Mid, r);
  r = fmaf(-k, kPio2Lo, r);
  r += err;
  const float s0 = __sinf(r), c0 = __cosf(r);
  const int q = static_cast<int>(k) & 3;
  float ss = (q & 1) ? c0 : s0;
  float cc = (q & 1) ? s0 : c0;
  if (q == 1 || q == 2) cc = -cc;
  if (q >= 2) ss = -ss;
  *s = sign * ss;
  *c = cc;
}

// Scale of an E4M3 block whose largest magnitude is A: the smallest power of two s
// with A / s <= 448.  With A = m 2^p, m in [1, 2): s = 2^(p - 8) when m <= 1.75
// (then A / s = 256 m <= 448), else 2^(p - 7).  Worked on the bits, so s and 1 / s
// are exact and x / s = x * (1 / s) rounds nowhere; s is clamped to the normal
// range (A below 2^-118 gets 2^-126).  A = 0 gives s = 1 / s = 0.
struct E4m3Scale {
  float s, inv;
};
__device__ __forceinline__ E4m3Scale e4m3_scale(float A) {
  if (!(A > 0.f)) return {0.f, 0.f};
  const uint32_t b = __float_as_uint(A);
  int e = static_cast<int>(b >> 23) - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  e = e < -126 ? -126 : (e > 126 ? 126 : e);
  return {__uint_as_float(static_cast<uint32_t>(127 + e) << 23),
          __uint_as_float(static_cast<uint32_t>(127 - e) << 23)};
}

// --------------------------------------------------------- workspace layout
// [0, 256)            device status word (uint32, flags kFlag*); words 1-3 the work-item
//                      counters of the forward, the dK / dV kernel and the recompute
//                      form's dQ kernel
// [256, +sched)       schedule: int32 order[n], int32 prefix[n+1]
// then 1024-aligned:  q16, k16  fp16 [T][h][d]  (rotated Q', K')
// fwd only:           v16 fp16 [T][h][d]
// rotate-on-load fwd:  rtab fp32 [R][d/2][2] from q16's offset, R <= T rows
//                      (4 T d bytes, inside the 6 T h d of q16, k16, v16)
// e4m3 fwd (inside the same total): q8, k8, v8 E4M3 [T][h][d] from q16's offset,
//                     qscale fp32 [T][h], amax2 uint32 [2][h]
// bwd only:           hmax fp32 [2][h] (per-head max ||dO_j||, max ||v_k||),
//                     pad fp32 [256] (128 x -inf, 128 x 0: -LSE log2 e / D of rows
//                     past a sample), nlse2 fp32 [h][T] (-LSE * log2 e), delta fp32 [h][T]
struct WsLayout {
  size_t status = 0;
  size_t order = 0, prefix = 0;
  size_t q16 = 0, k16 = 0, v16 = 0;
  size_t q8 = 0, k8 = 0, v8 = 0, qscale = 0, amax2 = 0;
  size_t hmax = 0, pad = 0, nlse2 = 0, delta = 0;
  size_t total = 0;
};
WsLayout ws_layout(int64_t T, int64_t n, int64_t heads, int64_t head_dim, bool bwd);

// ---------------------------------------------------------------- launches
cudaError_t launch_pack(const int32_t* specs, int32_t n, int32_t* d_cu, int32_t* d_pos,
                        cudaStream_t s);
// Editing packs: specs [n][5] = {text, Hs, Ws, Ht, Wt}; pos [T][3] = (f, r, c).
cudaError_t launch_pack3d(const int32_t* specs, int32_t n, int32_t* d_cu, int32_t* d_pos,
                          cudaStream_t s);
// bf16 in, bf16 out (the standalone mf_rope2d_qk / mf_rope3d_qk); pos has naxes
// coordinates per token.
cudaError_t launch_rope(const uint16_t* q, const uint16_t* k, uint16_t* q_out, uint16_t* k_out,
                        const int32_t* d_pos, int32_t naxes, int32_t T, int32_t heads,
                        int32_t head_dim, float sign, cudaStream_t s);
// bf16 in, fp16 out: the attention's operands Q' = R q, K' = R k (R the identity
// when d_pos is null) and, when v is given, V' = v converted.  fp16 carries 3 more
// mantissa bits than bf16 at the same tensor-core rate.  Sets kFlagFp16Range in
// *status if a value leaves the fp16 range.  Any of q/k/v may be null.
cudaError_t launch_prep_f16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            uint16_t* q_out, uint16_t* k_out, uint16_t* v_out,
                            const int32_t* d_pos, int32_t naxes, int32_t T, int32_t heads,
                            int32_t head_dim, uint32_t* status, cudaStream_t s);
// bf16 in, E4M3 out: the 8-bit forward's operands (head_dim 128 only).  Q' = R q
// scaled per (token, head) row to a largest magnitude of 448 (the scale, largest
// |q'| / 448, in qscale [T][heads]); K' = R k and V scaled per head from the maxima
// that the first pass gathers in amax2 [2][heads] (squared largest pair norm of k,
// squared largest |v|; zero on entry).
cudaError_t launch_prep_e4m3(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             uint8_t* q8, uint8_t* k8, uint8_t* v8, float* qscale,
                             uint32_t* amax2, const int32_t* d_pos, int32_t naxes, int32_t T,
                             int32_t heads, int32_t head_dim, cudaStream_t s);
// Builds the longest-first work list (items of `blk` rows per sample and head)
// and validates cu_seqlens; zeroes the status word and the work-item counters
// after it (words 1-7) first, and `nzero` floats at
// `zero` (may be null).
cudaError_t launch_schedule(const int32_t* d_cu, int32_t n, int32_t T, int32_t max_len,
                            int32_t heads, int32_t blk, uint32_t* status, int32_t* order,
                            int32_t* prefix, float* zero, int32_t nzero, cudaStream_t s);

struct AttnFwdArgs {
  const uint16_t* q;  // fp16 Q' (rotated); E4M3 bytes when f8
  const uint16_t* k;  // fp16 K' (rotated); E4M3 bytes when f8
  const uint16_t* v;  // fp16 V'; E4M3 bytes when f8
  bool f8 = false;    // the 8-bit variant (head_dim 128)
  const float* qscale = nullptr;     // f8: [T][heads] Q row scales
  const uint32_t* amax2 = nullptr;   // f8: [2][heads] squared K pair-norm and V maxima
  const int32_t* cu;
  const int32_t* order;
  const int32_t* prefix;
  uint32_t* status;
  uint16_t* o;  // bf16
  float* lse;
  int32_t n, T, heads, head_dim;
  float scale;
  uint32_t stall_us = 0;  // test hook: see mf_test_varlen_attn_fwd_stalled
  // rotate-on-load form: q, k, v are the caller's bf16 tensors; the kernel rotates
  // Q and K (2D positions `pos`, may be null) and converts V in shared memory,
  // reading (cos, sin) from rtab [rtab_rows][head_dim / 2]
  bool rot = false;
  const int32_t* pos = nullptr;
  const float* rtab = nullptr;
  int32_t rtab_rows = 0;
};
cudaError_t launch_attn_fwd(const AttnFwdArgs& a, cudaStream_t s);
// Multiprocessor count of the current device (the persistent kernels' grid).
int device_sm_count();
// The rotate-on-load forward's table: (cos, sin) of v * omega_P (2D frequencies)
// for v in [0, rows), as [rows][head_dim / 2] float pairs.
cudaError_t launch_rope_table(int32_t head_dim, int32_t rows, float* tab, cudaStream_t s);

struct AttnBwdArgs {
  const uint16_t* q;    // fp16 Q' (rotated)
  const uint16_t* k;    // fp16 K' (rotated)
  const uint16_t* v;    // bf16 (caller's)
  const uint16_t* o;    // bf16
  const uint16_t* d_o;  // bf16
  const float* lse;
  const int32_t* cu;
  const int32_t* pos;  // may be null; naxes coordinates per token
  int32_t naxes;       // 2 or 3
  const int32_t* order;
  const int32_t* prefix;
  uint32_t* status;
  float* hmax;    // [2][h]: max ||dO_j||, max ||v_k|| per head (zeroed by the schedule)
  float* pad;     // [256]: 128 x -inf then 128 x 0 (written by the preprocess)
  float* nlse2;   // [h][T]: -LSE * log2 e (written by the preprocess)
  float* delta;   // [h][T]
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  int32_t n, T, heads, head_dim;
  float scale;
  uint32_t stall_us = 0;  // test hook: see mf_test_varlen_attn_bwd_stalled
  // stored-dS form (null: the dQ kernel recomputes S and dP): the dK / dV kernel
  // writes every (sample, head)'s scaled fp16 dS^T and a streaming kernel forms
  // dQ = dS K' from it (layout: ds_layout_bytes)
  uint16_t* ds = nullptr;
  int64_t ds_cols = 0;
};
// Bytes of the stored-dS region for these sizes: heads (ceil(T / 128) + n) tiles of
// 128 keys x cols queries in fp16, cols = max_len rounded up to 128; each tile is
// [cols / 8 units of 8 queries][128 keys][8].  (Sample i, head a) owns the tiles
// from heads (ceil(cu[i] / 128) + i) + a a_i / 128, a_i = L_i rounded up to 128.
size_t ds_layout_bytes(int64_t T, int64_t n, int64_t heads, int64_t max_len, int64_t* cols);
cudaError_t launch_attn_bwd(const AttnBwdArgs& a, cudaStream_t s);

// Neighbours of the attention (neighbors.cu).  specs: host [2 * pairs][3].
cudaError_t launch_cfg_euler(const uint16_t* v, const int32_t* specs, int32_t pairs, int32_t C,
                             float g, float dt, float* z, cudaStream_t s);
cudaError_t launch_adaln(const uint16_t* x, const int32_t* cu, int32_t n, int32_t T, int32_t Dm,
                         const uint16_t* shift, const uint16_t* scale, float eps, uint16_t* y,
                         cudaStream_t s);
cudaError_t launch_gated_residual(const uint16_t* x, const uint16_t* h, const int32_t* cu,
                                  int32_t n, int32_t T, int32_t Dm, const uint16_t* gate,
                                  uint16_t* out, cudaStream_t s);

// RAII bracket of one kernel launch for the opt-in timing (mf_timing_*): records
// an event on `s` when built and another when destroyed; no-op when disabled.
class KernelTimer {
 public:
  KernelTimer(int id, cudaStream_t s);
  ~KernelTimer();
  KernelTimer(const KernelTimer&) = delete;
  KernelTimer& operator=(const KernelTimer&) = delete;

 private:
  int id_;
  cudaStream_t s_;
  void* a_ = nullptr;
};

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
// Element type bf16, or fp16 when `f16` (same size and layout).
bool make_tmap_thd(CUtensorMap* map, const void* base, int64_t T, int64_t heads,
                   int64_t head_dim, int box_rows, bool f16 = false);
// One-byte elements [T][heads][128] with a {128, 1, box_rows} box, 128-byte swizzle.
bool make_tmap_thd_u8(CUtensorMap* map, const void* base, int64_t T, int64_t heads,
                      int box_rows);
// fp32 [T][heads][head_dim] map with a {head_dim, 1, box_rows} box, no swizzle
// (the target of tiled reduce-adds).
bool make_tmap_f32_thd(CUtensorMap* map, const void* base, int64_t T, int64_t heads,
                       int64_t head_dim, int box_rows);

}  // namespace mf
