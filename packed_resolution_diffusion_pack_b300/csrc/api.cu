// C ABI (include/mf.h): argument validation, workspace layout and launch order.
// The arithmetic is in the kernels of pack_rope.cu, attn_fwd.cu and attn_bwd.cu.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "../../include/mf.h"
#include "common.cuh"
#include "ptx.cuh"

namespace mf {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WsLayout ws_layout(int64_t T, int64_t n, int64_t heads, int64_t head_dim, bool bwd) {
  WsLayout L;
  size_t off = 0;
  L.status = off;
  off += 256;
  L.order = off;
  off += align_up(sizeof(int32_t) * static_cast<size_t>(n > 0 ? n : 1), 256);
  L.prefix = off;
  off += align_up(sizeof(int32_t) * static_cast<size_t>(n + 1), 256);
  off = align_up(off, 1024);
  const size_t elems = static_cast<size_t>(T) * heads * head_dim;
  L.q16 = off;
  off = align_up(off + 2 * elems, 1024);
  L.k16 = off;
  off = align_up(off + 2 * elems, 1024);
  if (!bwd) {
    L.v16 = off;
    off = align_up(off + 2 * elems, 1024);
    // the 8-bit forward's operands and scales reuse the 16-bit operand space
    size_t o8 = L.q16;
    L.q8 = o8;
    o8 = align_up(o8 + elems, 1024);
    L.k8 = o8;
    o8 = align_up(o8 + elems, 1024);
    L.v8 = o8;
    o8 = align_up(o8 + elems, 1024);
    L.qscale = o8;
    o8 = align_up(o8 + 4 * static_cast<size_t>(heads) * T, 256);
    L.amax2 = o8;
    o8 = align_up(o8 + 8 * static_cast<size_t>(heads), 1024);
    if (o8 > off) off = o8;
  } else {
    L.hmax = off;
    off = align_up(off + 8 * static_cast<size_t>(heads), 256);
    L.pad = off;
    off = align_up(off + 4 * 256, 1024);
    L.nlse2 = off;
    off = align_up(off + 4 * static_cast<size_t>(heads) * T, 1024);
    L.delta = off;
    off = align_up(off + 4 * static_cast<size_t>(heads) * T, 1024);
  }
  L.total = off;
  // a backward workspace also serves the forward of the same call sizes (the
  // training step shares one: mf_varlen_attn_bwd_after_fwd), so it is never
  // smaller than the forward's
  if (bwd) {
    const size_t fwd_total = ws_layout(T, n, heads, head_dim, false).total;
    if (fwd_total > L.total) L.total = fwd_total;
  }
  return L;
}

size_t ds_layout_bytes(int64_t T, int64_t n, int64_t heads, int64_t max_len, int64_t* cols) {
  const int64_t A = (max_len > 0 ? (max_len + 127) / 128 : 1) * 128;
  const int64_t tiles = heads * ((T + 127) / 128 + n);  // 128-key tiles, see ds_tile_base
  if (T < 0 || n < 0 || heads < 1 || A > INT32_MAX || tiles > (INT64_MAX / 256) / A) return 0;
  if (cols) *cols = A;
  return static_cast<size_t>(tiles) * 128 * static_cast<size_t>(A) * 2;
}

static bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Shared validation of the attention calls.
static mf_status check_attn(const void* const* ptrs, int nptr, const int32_t* cu, int32_t n,
                            int32_t T, int32_t max_len, int32_t heads, int32_t head_dim,
                            const void* ws, size_t ws_bytes, bool bwd) {
  if (n < 0 || T < 0 || max_len < 0 || heads < 1 || cu == nullptr || ws == nullptr)
    return MF_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  const int64_t items = (static_cast<int64_t>(T) / 128 + 1 + n) * heads;
  if (items > INT32_MAX || static_cast<int64_t>(heads) * T > INT32_MAX) return MF_ERR_OVERFLOW;
  for (int i = 0; i < nptr; ++i) {
    if (T > 0 && ptrs[i] == nullptr) return MF_ERR_INVALID_ARG;
    if (!aligned(ptrs[i], 16)) return MF_ERR_UNSUPPORTED;
  }
  if (!aligned(ws, 256)) return MF_ERR_UNSUPPORTED;
  if (ws_bytes < ws_layout(T, n, heads, head_dim, bwd).total) return MF_ERR_INVALID_ARG;
  return MF_OK;
}

static mf_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MF_OK : MF_ERR_CUDA; }

}  // namespace mf

using namespace mf;

extern "C" {

const char* mf_status_string(mf_status s) {
  switch (s) {
    case MF_OK: return "MF_OK";
    case MF_ERR_INVALID_ARG: return "MF_ERR_INVALID_ARG";
    case MF_ERR_UNSUPPORTED: return "MF_ERR_UNSUPPORTED";
    case MF_ERR_OVERFLOW: return "MF_ERR_OVERFLOW";
    case MF_ERR_CUDA: return "MF_ERR_CUDA";
    case MF_ERR_TIMEOUT: return "MF_ERR_TIMEOUT";
    case MF_ERR_BAD_SEQLENS: return "MF_ERR_BAD_SEQLENS";
  }
  return "MF_ERR_UNKNOWN";
}

int32_t mf_version(void) { return 10000; }

mf_status mf_pack_size(const int32_t* specs, int32_t n, int32_t* total, int32_t* max_len) {
  if (n < 0 || (n > 0 && specs == nullptr)) return MF_ERR_INVALID_ARG;
  int64_t T = 0, mx = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t t = specs[3 * i], H = specs[3 * i + 1], W = specs[3 * i + 2];
    if (t < 0 || H < 0 || W < 0) return MF_ERR_INVALID_ARG;
    const int64_t L = t + H * W;
    if (H * W > INT32_MAX || L > INT32_MAX) return MF_ERR_OVERFLOW;
    T += L;
    if (T > INT32_MAX) return MF_ERR_OVERFLOW;
    if (L > mx) mx = L;
  }
  if (total) *total = static_cast<int32_t>(T);
  if (max_len) *max_len = static_cast<int32_t>(mx);
  return MF_OK;
}

mf_status mf_pack(const int32_t* specs, int32_t n, int32_t* d_cu_seqlens, int32_t* d_pos,
                  mf_stream stream) {
  int32_t T = 0;
  const mf_status st = mf_pack_size(specs, n, &T, nullptr);
  if (st != MF_OK) return st;
  if (d_cu_seqlens == nullptr) return MF_ERR_INVALID_ARG;
  if (d_pos != nullptr && !aligned(d_pos, 8)) return MF_ERR_UNSUPPORTED;
  return cuda_status(
      launch_pack(specs, n, d_cu_seqlens, d_pos, static_cast<cudaStream_t>(stream)));
}

mf_status mf_rope2d_qk(const mf_bf16* q, const mf_bf16* k, mf_bf16* q_out, mf_bf16* k_out,
                       const int32_t* d_pos, int32_t T, int32_t heads, int32_t head_dim,
                       mf_stream stream) {
  if (T < 0 || heads < 1) return MF_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(heads) * head_dim * T / 8 > INT64_MAX / 2) return MF_ERR_OVERFLOW;
  if (T == 0) return MF_OK;
  if (d_pos == nullptr || (q == nullptr && k == nullptr)) return MF_ERR_INVALID_ARG;
  if ((q == nullptr) != (q_out == nullptr) || (k == nullptr) != (k_out == nullptr))
    return MF_ERR_INVALID_ARG;
  const void* ps[4] = {q, k, q_out, k_out};
  for (const void* ptr : ps)
    if (ptr != nullptr && !aligned(ptr, 16)) return MF_ERR_UNSUPPORTED;
  if (!aligned(d_pos, 8)) return MF_ERR_UNSUPPORTED;
  return cuda_status(launch_rope(q, k, q_out, k_out, d_pos, 2, T, heads, head_dim, 1.0f,
                                 static_cast<cudaStream_t>(stream)));
}

size_t mf_attn_workspace_bytes(int32_t T, int32_t n, int32_t heads, int32_t head_dim,
                               int32_t bwd) {
  if (T < 0 || n < 0 || heads < 1 || (head_dim != 64 && head_dim != 128)) return 0;
  return ws_layout(T, n, heads, head_dim, bwd != 0).total;
}

size_t mf_attn_workspace_bytes_ds(int32_t T, int32_t n, int32_t heads, int32_t head_dim,
                                  int32_t max_len) {
  if (T < 0 || n < 0 || heads < 1 || max_len < 0 || (head_dim != 64 && head_dim != 128)) return 0;
  const size_t dsb = ds_layout_bytes(T, n, heads, max_len, nullptr);
  if (dsb == 0) return 0;
  return align_up(ws_layout(T, n, heads, head_dim, true).total, 1024) + dsb;
}

}  // extern "C"

namespace mf {

// The forward for positions of `naxes` coordinates per token (2: native-resolution
// packs, 3: editing packs); only the fp16 rotation pre-pass depends on it.
static mf_status attn_fwd_impl(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                               const int32_t* d_cu_seqlens, const int32_t* d_pos, int32_t naxes,
                               int32_t n, int32_t T, int32_t max_len, int32_t heads,
                               int32_t head_dim, float softmax_scale, mf_bf16* o, float* lse,
                               void* ws, size_t ws_bytes, mf_stream stream,
                               uint32_t stall_us = 0) {
  const void* ptrs[5] = {q, k, v, o, lse};
  mf_status st = check_attn(ptrs, 5, d_cu_seqlens, n, T, max_len, heads, head_dim, ws, ws_bytes,
                            false);
  if (st != MF_OK) return st;
  if (d_pos != nullptr && !aligned(d_pos, 4)) return MF_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(T, n, heads, head_dim, false);
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto* status = reinterpret_cast<uint32_t*>(w + L.status);
  auto* order = reinterpret_cast<int32_t*>(w + L.order);
  auto* prefix = reinterpret_cast<int32_t*>(w + L.prefix);
  cudaError_t e =
      launch_schedule(d_cu_seqlens, n, T, max_len, heads, 256, status, order, prefix, nullptr, 0, s);
  if (e != cudaSuccess) return MF_ERR_CUDA;
  if (T == 0) return MF_OK;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  // Q' = R q, K' = R k (R = I without positions) and V' = v, all fp16
  auto* q16 = reinterpret_cast<uint16_t*>(w + L.q16);
  auto* k16 = reinterpret_cast<uint16_t*>(w + L.k16);
  auto* v16 = reinterpret_cast<uint16_t*>(w + L.v16);
  e = launch_prep_f16(q, k, v, q16, k16, v16, d_pos, naxes, T, heads, head_dim, status, s);
  if (e != cudaSuccess) return MF_ERR_CUDA;
  AttnFwdArgs a;
  a.q = q16;
  a.k = k16;
  a.v = v16;
  a.cu = d_cu_seqlens;
  a.order = order;
  a.prefix = prefix;
  a.status = status;
  a.o = o;
  a.lse = lse;
  a.n = n;
  a.T = T;
  a.heads = heads;
  a.head_dim = head_dim;
  a.scale = scale;
  a.stall_us = stall_us;
  return cuda_status(launch_attn_fwd(a, s));
}

// The forward with the rotation applied on the tile load: schedule, the (cos, sin)
// table, and the attention kernel on the caller's bf16 q, k, v.
static mf_status attn_fwd_rot_impl(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                   const int32_t* d_cu_seqlens, const int32_t* d_pos, int32_t n,
                                   int32_t T, int32_t max_len, int32_t heads, int32_t head_dim,
                                   float softmax_scale, mf_bf16* o, float* lse, void* ws,
                                   size_t ws_bytes, mf_stream stream) {
  const void* ptrs[5] = {q, k, v, o, lse};
  mf_status st = check_attn(ptrs, 5, d_cu_seqlens, n, T, max_len, heads, head_dim, ws, ws_bytes,
                            false);
  if (st != MF_OK) return st;
  if (d_pos != nullptr && !aligned(d_pos, 8)) return MF_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(T, n, heads, head_dim, false);
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto* status = reinterpret_cast<uint32_t*>(w + L.status);
  auto* order = reinterpret_cast<int32_t*>(w + L.order);
  auto* prefix = reinterpret_cast<int32_t*>(w + L.prefix);
  cudaError_t e =
      launch_schedule(d_cu_seqlens, n, T, max_len, heads, 256, status, order, prefix, nullptr, 0, s);
  if (e != cudaSuccess) return MF_ERR_CUDA;
  if (T == 0) return MF_OK;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  // table rows: every coordinate of a valid pack is below max(H, W) <= L_i <= max_len
  // (and below T); 4 T head_dim bytes at most, inside the operand region
  const int32_t rows = max_len < T ? (max_len > 0 ? max_len : 1) : T;
  auto* rtab = reinterpret_cast<float*>(w + L.q16);
  if (d_pos != nullptr) {
    e = launch_rope_table(head_dim, rows, rtab, s);
    if (e != cudaSuccess) return MF_ERR_CUDA;
  }
  AttnFwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.rot = true;
  a.pos = d_pos;
  a.rtab = rtab;
  a.rtab_rows = rows;
  a.cu = d_cu_seqlens;
  a.order = order;
  a.prefix = prefix;
  a.status = status;
  a.o = o;
  a.lse = lse;
  a.n = n;
  a.T = T;
  a.heads = heads;
  a.head_dim = head_dim;
  a.scale = scale;
  return cuda_status(launch_attn_fwd(a, s));
}

// The 8-bit variant of the forward: E4M3 operands with per-row Q and per-head K,
// V scales, E4M3 probabilities, fp32 accumulation; head_dim 128.
static mf_status attn_fwd_e4m3_impl(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                    const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                    int32_t naxes, int32_t n, int32_t T, int32_t max_len,
                                    int32_t heads, int32_t head_dim, float softmax_scale,
                                    mf_bf16* o, float* lse, void* ws, size_t ws_bytes,
                                    mf_stream stream) {
  const void* ptrs[5] = {q, k, v, o, lse};
  mf_status st = check_attn(ptrs, 5, d_cu_seqlens, n, T, max_len, heads, head_dim, ws, ws_bytes,
                            false);
  if (st != MF_OK) return st;
  if (head_dim != 128) return MF_ERR_UNSUPPORTED;
  if (d_pos != nullptr && !aligned(d_pos, 4)) return MF_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(T, n, heads, head_dim, false);
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto* status = reinterpret_cast<uint32_t*>(w + L.status);
  auto* order = reinterpret_cast<int32_t*>(w + L.order);
  auto* prefix = reinterpret_cast<int32_t*>(w + L.prefix);
  auto* amax2 = reinterpret_cast<uint32_t*>(w + L.amax2);
  // the schedule also zeroes the per-head maxima
  cudaError_t e = launch_schedule(d_cu_seqlens, n, T, max_len, heads, 256, status, order, prefix,
                                  reinterpret_cast<float*>(amax2), 2 * heads, s);
  if (e != cudaSuccess) return MF_ERR_CUDA;
  if (T == 0) return MF_OK;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  auto* q8 = w + L.q8;
  auto* k8 = w + L.k8;
  auto* v8 = w + L.v8;
  auto* qscale = reinterpret_cast<float*>(w + L.qscale);
  e = launch_prep_e4m3(q, k, v, q8, k8, v8, qscale, amax2, d_pos, naxes, T, heads, head_dim, s);
  if (e != cudaSuccess) return MF_ERR_CUDA;
  AttnFwdArgs a;
  a.q = reinterpret_cast<const uint16_t*>(q8);
  a.k = reinterpret_cast<const uint16_t*>(k8);
  a.v = reinterpret_cast<const uint16_t*>(v8);
  a.f8 = true;
  a.qscale = qscale;
  a.amax2 = amax2;
  a.cu = d_cu_seqlens;
  a.order = order;
  a.prefix = prefix;
  a.status = status;
  a.o = o;
  a.lse = lse;
  a.n = n;
  a.T = T;
  a.heads = heads;
  a.head_dim = head_dim;
  a.scale = scale;
  return cuda_status(launch_attn_fwd(a, s));
}

static mf_status attn_bwd_impl(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                               const mf_bf16* o, const float* lse, const mf_bf16* d_o,
                               const int32_t* d_cu_seqlens, const int32_t* d_pos, int32_t naxes,
                               int32_t n, int32_t T, int32_t max_len, int32_t heads,
                               int32_t head_dim, float softmax_scale, mf_bf16* dq, mf_bf16* dk,
                               mf_bf16* dv, void* ws, size_t ws_bytes, mf_stream stream,
                               bool reuse_rotated = false, uint32_t stall_us = 0) {
  const void* ptrs[9] = {q, k, v, o, lse, d_o, dq, dk, dv};
  mf_status st = check_attn(ptrs, 9, d_cu_seqlens, n, T, max_len, heads, head_dim, ws, ws_bytes,
                            true);
  if (st != MF_OK) return st;
  if (d_pos != nullptr && !aligned(d_pos, 4)) return MF_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(T, n, heads, head_dim, true);
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto* status = reinterpret_cast<uint32_t*>(w + L.status);
  auto* order = reinterpret_cast<int32_t*>(w + L.order);
  auto* prefix = reinterpret_cast<int32_t*>(w + L.prefix);
  auto* hmax = reinterpret_cast<float*>(w + L.hmax);
  cudaError_t e = launch_schedule(d_cu_seqlens, n, T, max_len, heads, 128, status, order, prefix,
                                  hmax, 2 * heads, s);
  if (e != cudaSuccess) return MF_ERR_CUDA;
  if (T == 0) return MF_OK;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  // Q' = R q, K' = R k in fp16, as in the forward (same logits as the LSE came from)
  auto* q16 = reinterpret_cast<uint16_t*>(w + L.q16);
  auto* k16 = reinterpret_cast<uint16_t*>(w + L.k16);
  if (!reuse_rotated) {
    e = launch_prep_f16(q, k, nullptr, q16, k16, nullptr, d_pos, naxes, T, heads, head_dim, status,
                        s);
    if (e != cudaSuccess) return MF_ERR_CUDA;
  }
  AttnBwdArgs a;
  // a workspace sized by mf_attn_workspace_bytes_ds selects the stored-dS form
  int64_t ds_cols = 0;
  const size_t dsb = ds_layout_bytes(T, n, heads, max_len, &ds_cols);
  const size_t ds_off = align_up(L.total, 1024);
  if (dsb > 0 && ws_bytes >= ds_off + dsb) {
    a.ds = reinterpret_cast<uint16_t*>(w + ds_off);
    a.ds_cols = ds_cols;
  }
  a.q = q16;
  a.k = k16;
  a.v = v;
  a.hmax = hmax;
  a.o = o;
  a.d_o = d_o;
  a.lse = lse;
  a.cu = d_cu_seqlens;
  a.pos = d_pos;
  a.naxes = naxes;
  a.order = order;
  a.prefix = prefix;
  a.status = status;
  a.pad = reinterpret_cast<float*>(w + L.pad);
  a.nlse2 = reinterpret_cast<float*>(w + L.nlse2);
  a.delta = reinterpret_cast<float*>(w + L.delta);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.n = n;
  a.T = T;
  a.heads = heads;
  a.head_dim = head_dim;
  a.scale = scale;
  a.stall_us = stall_us;
  return cuda_status(launch_attn_bwd(a, s));
}

}  // namespace mf

extern "C" {

mf_status mf_varlen_attn_fwd(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                             const int32_t* d_cu_seqlens, const int32_t* d_pos, int32_t n,
                             int32_t T, int32_t max_len, int32_t heads, int32_t head_dim,
                             float softmax_scale, mf_bf16* o, float* lse, void* ws,
                             size_t ws_bytes, mf_stream stream) {
  return attn_fwd_impl(q, k, v, d_cu_seqlens, d_pos, 2, n, T, max_len, heads, head_dim,
                       softmax_scale, o, lse, ws, ws_bytes, stream);
}

mf_status mf_varlen_attn_fwd_fused_rope(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                        const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                        int32_t n, int32_t T, int32_t max_len, int32_t heads,
                                        int32_t head_dim, float softmax_scale, mf_bf16* o,
                                        float* lse, void* ws, size_t ws_bytes, mf_stream stream) {
  return attn_fwd_rot_impl(q, k, v, d_cu_seqlens, d_pos, n, T, max_len, heads, head_dim,
                           softmax_scale, o, lse, ws, ws_bytes, stream);
}

mf_status mf_test_varlen_attn_fwd_stalled(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                          const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                          int32_t n, int32_t T, int32_t max_len, int32_t heads,
                                          int32_t head_dim, float softmax_scale, mf_bf16* o,
                                          float* lse, void* ws, size_t ws_bytes,
                                          int32_t stall_us, mf_stream stream) {
  if (stall_us < 1 || stall_us > 1000000) return MF_ERR_INVALID_ARG;
  return attn_fwd_impl(q, k, v, d_cu_seqlens, d_pos, 2, n, T, max_len, heads, head_dim,
                       softmax_scale, o, lse, ws, ws_bytes, stream,
                       static_cast<uint32_t>(stall_us));
}

mf_status mf_test_varlen_attn_bwd_stalled(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                          const mf_bf16* o, const float* lse, const mf_bf16* d_o,
                                          const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                          int32_t n, int32_t T, int32_t max_len, int32_t heads,
                                          int32_t head_dim, float softmax_scale, mf_bf16* dq,
                                          mf_bf16* dk, mf_bf16* dv, void* ws, size_t ws_bytes,
                                          int32_t stall_us, mf_stream stream) {
  if (stall_us < 1 || stall_us > 1000000) return MF_ERR_INVALID_ARG;
  return attn_bwd_impl(q, k, v, o, lse, d_o, d_cu_seqlens, d_pos, 2, n, T, max_len, heads,
                       head_dim, softmax_scale, dq, dk, dv, ws, ws_bytes, stream, false,
                       static_cast<uint32_t>(stall_us));
}

mf_status mf_varlen_attn_bwd(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                             const mf_bf16* o, const float* lse, const mf_bf16* d_o,
                             const int32_t* d_cu_seqlens, const int32_t* d_pos, int32_t n,
                             int32_t T, int32_t max_len, int32_t heads, int32_t head_dim,
                             float softmax_scale, mf_bf16* dq, mf_bf16* dk, mf_bf16* dv,
                             void* ws, size_t ws_bytes, mf_stream stream) {
  return attn_bwd_impl(q, k, v, o, lse, d_o, d_cu_seqlens, d_pos, 2, n, T, max_len, heads,
                       head_dim, softmax_scale, dq, dk, dv, ws, ws_bytes, stream);
}

mf_status mf_varlen_attn_bwd_after_fwd(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                       const mf_bf16* o, const float* lse, const mf_bf16* d_o,
                                       const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                       int32_t pos_axes, int32_t n, int32_t T, int32_t max_len,
                                       int32_t heads, int32_t head_dim, float softmax_scale,
                                       mf_bf16* dq, mf_bf16* dk, mf_bf16* dv, void* ws,
                                       size_t ws_bytes, mf_stream stream) {
  if (pos_axes != 2 && pos_axes != 3) return MF_ERR_INVALID_ARG;
  return attn_bwd_impl(q, k, v, o, lse, d_o, d_cu_seqlens, d_pos, pos_axes, n, T, max_len, heads,
                       head_dim, softmax_scale, dq, dk, dv, ws, ws_bytes, stream, true);
}

mf_status mf_varlen_attn_fwd_fp8(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                 const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                 int32_t pos_axes, int32_t n, int32_t T, int32_t max_len,
                                 int32_t heads, int32_t head_dim, float softmax_scale, mf_bf16* o,
                                 float* lse, void* ws, size_t ws_bytes, mf_stream stream) {
  if (d_pos != nullptr && pos_axes != 2 && pos_axes != 3) return MF_ERR_INVALID_ARG;
  return attn_fwd_e4m3_impl(q, k, v, d_cu_seqlens, d_pos, d_pos ? pos_axes : 2, n, T, max_len,
                            heads, head_dim, softmax_scale, o, lse, ws, ws_bytes, stream);
}

mf_status mf_quant_e4m3(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                        const int32_t* d_pos, int32_t pos_axes, int32_t T, int32_t heads,
                        int32_t head_dim, uint8_t* q8, uint8_t* k8, uint8_t* v8, float* qscale,
                        float* kv_max2, mf_stream stream) {
  if (T < 0 || heads < 1) return MF_ERR_INVALID_ARG;
  if (head_dim != 128) return MF_ERR_UNSUPPORTED;
  if (d_pos != nullptr && pos_axes != 2 && pos_axes != 3) return MF_ERR_INVALID_ARG;
  if (static_cast<int64_t>(heads) * T > INT32_MAX) return MF_ERR_OVERFLOW;
  const void* ps[9] = {q, k, v, q8, k8, v8, qscale, kv_max2, d_pos};
  for (int i = 0; i < 8; ++i)
    if (ps[i] == nullptr) return MF_ERR_INVALID_ARG;
  for (int i = 0; i < 6; ++i)
    if (!aligned(ps[i], 16)) return MF_ERR_UNSUPPORTED;
  if (!aligned(qscale, 4) || !aligned(kv_max2, 4) || (d_pos && !aligned(d_pos, 4)))
    return MF_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(kv_max2, 0, 8 * static_cast<size_t>(heads), s) != cudaSuccess)
    return MF_ERR_CUDA;
  if (T == 0) return MF_OK;
  return cuda_status(launch_prep_e4m3(q, k, v, q8, k8, v8, qscale,
                                      reinterpret_cast<uint32_t*>(kv_max2), d_pos,
                                      d_pos ? pos_axes : 2, T, heads, head_dim, s));
}

mf_status mf_varlen_attn_fwd_3d(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                const int32_t* d_cu_seqlens, const int32_t* d_pos3, int32_t n,
                                int32_t T, int32_t max_len, int32_t heads, int32_t head_dim,
                                float softmax_scale, mf_bf16* o, float* lse, void* ws,
                                size_t ws_bytes, mf_stream stream) {
  if (d_pos3 == nullptr) return MF_ERR_INVALID_ARG;
  return attn_fwd_impl(q, k, v, d_cu_seqlens, d_pos3, 3, n, T, max_len, heads, head_dim,
                       softmax_scale, o, lse, ws, ws_bytes, stream);
}

mf_status mf_varlen_attn_bwd_3d(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                const mf_bf16* o, const float* lse, const mf_bf16* d_o,
                                const int32_t* d_cu_seqlens, const int32_t* d_pos3, int32_t n,
                                int32_t T, int32_t max_len, int32_t heads, int32_t head_dim,
                                float softmax_scale, mf_bf16* dq, mf_bf16* dk, mf_bf16* dv,
                                void* ws, size_t ws_bytes, mf_stream stream) {
  if (d_pos3 == nullptr) return MF_ERR_INVALID_ARG;
  return attn_bwd_impl(q, k, v, o, lse, d_o, d_cu_seqlens, d_pos3, 3, n, T, max_len, heads,
                       head_dim, softmax_scale, dq, dk, dv, ws, ws_bytes, stream);
}

mf_status mf_pack3d_size(const int32_t* specs, int32_t n, int32_t* total, int32_t* max_len) {
  if (n < 0 || (n > 0 && specs == nullptr)) return MF_ERR_INVALID_ARG;
  int64_t T = 0, mx = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t* sp = specs + 5 * i;
    for (int q = 0; q < 5; ++q)
      if (sp[q] < 0) return MF_ERR_INVALID_ARG;
    const int64_t src = static_cast<int64_t>(sp[1]) * sp[2];
    const int64_t tgt = static_cast<int64_t>(sp[3]) * sp[4];
    const int64_t L = sp[0] + src + tgt;
    if (src > INT32_MAX || tgt > INT32_MAX || L > INT32_MAX) return MF_ERR_OVERFLOW;
    T += L;
    if (T > INT32_MAX) return MF_ERR_OVERFLOW;
    if (L > mx) mx = L;
  }
  if (total) *total = static_cast<int32_t>(T);
  if (max_len) *max_len = static_cast<int32_t>(mx);
  return MF_OK;
}

mf_status mf_pack3d(const int32_t* specs, int32_t n, int32_t* d_cu_seqlens, int32_t* d_pos3,
                    mf_stream stream) {
  const mf_status st = mf_pack3d_size(specs, n, nullptr, nullptr);
  if (st != MF_OK) return st;
  if (d_cu_seqlens == nullptr) return MF_ERR_INVALID_ARG;
  if (d_pos3 != nullptr && !aligned(d_pos3, 4)) return MF_ERR_UNSUPPORTED;
  return cuda_status(
      launch_pack3d(specs, n, d_cu_seqlens, d_pos3, static_cast<cudaStream_t>(stream)));
}

mf_status mf_rope3d_qk(const mf_bf16* q, const mf_bf16* k, mf_bf16* q_out, mf_bf16* k_out,
                       const int32_t* d_pos3, int32_t T, int32_t heads, int32_t head_dim,
                       mf_stream stream) {
  if (T < 0 || heads < 1) return MF_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  if (T == 0) return MF_OK;
  if (d_pos3 == nullptr || (q == nullptr && k == nullptr)) return MF_ERR_INVALID_ARG;
  if ((q == nullptr) != (q_out == nullptr) || (k == nullptr) != (k_out == nullptr))
    return MF_ERR_INVALID_ARG;
  const void* ps[4] = {q, k, q_out, k_out};
  for (const void* ptr : ps)
    if (ptr != nullptr && !aligned(ptr, 16)) return MF_ERR_UNSUPPORTED;
  if (!aligned(d_pos3, 4)) return MF_ERR_UNSUPPORTED;
  return cuda_status(launch_rope(q, k, q_out, k_out, d_pos3, 3, T, heads, head_dim, 1.0f,
                                 static_cast<cudaStream_t>(stream)));
}

mf_status mf_cfg_euler_step(const mf_bf16* v, const int32_t* specs, int32_t pairs, int32_t C,
                            float guidance, float dt, float* z, mf_stream stream) {
  if (pairs < 0 || C <= 0 || (pairs > 0 && specs == nullptr)) return MF_ERR_INVALID_ARG;
  if (C % 8 != 0) return MF_ERR_UNSUPPORTED;
  int64_t T = 0, N = 0;
  for (int32_t p = 0; p < pairs; ++p) {
    const int32_t* sc = specs + 6 * p;
    const int32_t* su = sc + 3;
    for (int i = 0; i < 6; ++i)
      if (sc[i] < 0) return MF_ERR_INVALID_ARG;
    if (sc[1] != su[1] || sc[2] != su[2]) return MF_ERR_INVALID_ARG;
    const int64_t n_img = static_cast<int64_t>(sc[1]) * sc[2];
    T += static_cast<int64_t>(sc[0]) + su[0] + 2 * n_img;
    N += n_img;
  }
  if (T > INT32_MAX || N > INT32_MAX || T * (C / 8) > INT64_MAX / 16) return MF_ERR_OVERFLOW;
  if (N == 0) return MF_OK;
  if (v == nullptr || z == nullptr) return MF_ERR_INVALID_ARG;
  if (!aligned(v, 16) || !aligned(z, 16)) return MF_ERR_UNSUPPORTED;
  return cuda_status(launch_cfg_euler(v, specs, pairs, C, guidance, dt, z,
                                      static_cast<cudaStream_t>(stream)));
}

// Shared checks of the row-wise packed neighbours.
static mf_status check_rows(const void* const* ptrs, int nptr, const int32_t* cu, int32_t n,
                            int32_t T, int32_t Dm, int32_t max_dm) {
  if (n < 0 || T < 0 || Dm <= 0 || (T > 0 && n == 0)) return MF_ERR_INVALID_ARG;
  if (Dm % 8 != 0 || Dm > max_dm) return MF_ERR_UNSUPPORTED;
  if (T == 0) return MF_OK;
  if (cu == nullptr) return MF_ERR_INVALID_ARG;
  for (int i = 0; i < nptr; ++i) {
    if (ptrs[i] == nullptr) return MF_ERR_INVALID_ARG;
    if (!aligned(ptrs[i], 16)) return MF_ERR_UNSUPPORTED;
  }
  return MF_OK;
}

mf_status mf_adaln_modulate(const mf_bf16* x, const int32_t* d_cu_seqlens, int32_t n, int32_t T,
                            int32_t Dm, const mf_bf16* shift, const mf_bf16* scale, float eps,
                            mf_bf16* y, mf_stream stream) {
  const void* ptrs[4] = {x, shift, scale, y};
  const mf_status st = check_rows(ptrs, 4, d_cu_seqlens, n, T, Dm, INT32_MAX);
  if (st != MF_OK) return st;
  if (!(eps >= 0.f)) return MF_ERR_INVALID_ARG;
  return cuda_status(launch_adaln(x, d_cu_seqlens, n, T, Dm, shift, scale, eps, y,
                                  static_cast<cudaStream_t>(stream)));
}

mf_status mf_gated_residual(const mf_bf16* x, const mf_bf16* h, const int32_t* d_cu_seqlens,
                            int32_t n, int32_t T, int32_t Dm, const mf_bf16* gate, mf_bf16* out,
                            mf_stream stream) {
  const void* ptrs[4] = {x, h, gate, out};
  const mf_status st = check_rows(ptrs, 4, d_cu_seqlens, n, T, Dm, INT32_MAX);
  if (st != MF_OK) return st;
  return cuda_status(launch_gated_residual(x, h, d_cu_seqlens, n, T, Dm, gate, out,
                                           static_cast<cudaStream_t>(stream)));
}

mf_status mf_get_status(void* ws, mf_stream stream) {
  if (ws == nullptr) return MF_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MF_ERR_CUDA;
  uint32_t flags = 0;
  if (cudaMemcpy(&flags, ws, sizeof(flags), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MF_ERR_CUDA;
  if (flags & kFlagBadSeqlens) return MF_ERR_BAD_SEQLENS;
  if (flags & kFlagTimeout) return MF_ERR_TIMEOUT;
  if (flags & kFlagFp16Range) return MF_ERR_OVERFLOW;
  if (flags & kFlagSmemAlign) return MF_ERR_CUDA;
  if (flags & kFlagPosRange) return MF_ERR_INVALID_ARG;
  return MF_OK;
}

}  // extern "C"
