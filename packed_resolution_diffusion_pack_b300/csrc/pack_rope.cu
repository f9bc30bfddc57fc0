// Packing tables and the standalone 2D RoPE: memory-bound kernels.
//
// Packing (Mage-Flow, rcap.io post, training-step listing "native-resolution
// packed step"; paperlayer.ai summary 3.2.1): samples [text; image] are laid end
// to end; image token m of an H x W latent grid sits at (m div W, m mod W), text
// tokens at (0, 0).
// 2D RoPE (rcap.io post, per_sample_2d_rope; ai.thesatyajit.com explainer "A
// backbone that doesn't crop"): dims [0, d/2) rotate by the row, [d/2, d) by the
// column; pair (2j, 2j+1) of a half by p * 10000^(-2j/(d/2)).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace mf {

RopeFreqs make_rope_freqs(int head_dim, int naxes) {
  RopeFreqs f{};
  f.naxes = naxes;
  // slice widths (dims) per axis
  int width[3] = {head_dim / 2, head_dim / 2, 0};
  if (naxes == 3) {
    width[0] = head_dim / 4;
    width[1] = 3 * head_dim / 8;
    width[2] = 3 * head_dim / 8;
  }
  int P = 0;
  for (int a = 0; a < naxes; ++a) {
    for (int j = 0; j < width[a] / 2 && P < kMaxPairs; ++j, ++P) {
      const double w = std::pow(kRopeBase, -2.0 * j / static_cast<double>(width[a]));
      f.omega[P] = static_cast<float>(w);
      f.omega_lo[P] = static_cast<float>(w - static_cast<double>(f.omega[P]));
      f.axis[P] = static_cast<int8_t>(a);
    }
  }
  return f;
}

// ------------------------------------------------------------------ packing
constexpr int kPackChunk = 256;  // samples per launch (kernel parameter space)

struct PackChunk {
  int32_t first;      // global index of the chunk's first sample
  int32_t count;      // samples in the chunk
  int32_t tok_begin;  // first token of the chunk
  int32_t tok_end;    // one past its last token
  int32_t last;       // 1 if this chunk holds sample n-1 (writes cu[n])
  int32_t start[kPackChunk];
  int32_t text[kPackChunk];
  int32_t width[kPackChunk];
};

__global__ void __launch_bounds__(256) pack_kernel(const __grid_constant__ PackChunk c,
                                                   int32_t* __restrict__ cu,
                                                   int2* __restrict__ pos) {
  __shared__ int32_t s_start[kPackChunk], s_text[kPackChunk], s_width[kPackChunk];
  for (int i = threadIdx.x; i < c.count; i += blockDim.x) {
    s_start[i] = c.start[i];
    s_text[i] = c.text[i];
    s_width[i] = c.width[i];
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < c.count; i += blockDim.x) cu[c.first + i] = s_start[i];
    if (c.last && threadIdx.x == 0) cu[c.first + c.count] = c.tok_end;
  }
  if (pos == nullptr) return;
  const int64_t t = static_cast<int64_t>(c.tok_begin) + blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= c.tok_end) return;
  // last sample whose start <= t (zero-length samples share a start; the last of
  // them is the one holding t)
  int lo = 0, hi = c.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int32_t k = static_cast<int32_t>(t) - s_start[lo];
  int2 p = make_int2(0, 0);
  if (k >= s_text[lo]) {
    const int32_t m = k - s_text[lo], W = s_width[lo];
    p = make_int2(m / W, m - (m / W) * W);
  }
  pos[t] = p;
}

cudaError_t launch_pack(const int32_t* specs, int32_t n, int32_t* d_cu, int32_t* d_pos,
                        cudaStream_t s) {
  int64_t start = 0;
  for (int32_t first = 0; first < n || (n == 0 && first == 0); first += kPackChunk) {
    PackChunk c{};
    c.first = first;
    c.count = n - first < kPackChunk ? n - first : kPackChunk;
    c.tok_begin = static_cast<int32_t>(start);
    for (int i = 0; i < c.count; ++i) {
      const int32_t* sp = specs + 3 * (first + i);
      c.start[i] = static_cast<int32_t>(start);
      c.text[i] = sp[0];
      c.width[i] = sp[2];
      start += static_cast<int64_t>(sp[0]) + static_cast<int64_t>(sp[1]) * sp[2];
    }
    c.tok_end = static_cast<int32_t>(start);
    c.last = (first + c.count >= n) ? 1 : 0;
    const int64_t ntok = c.tok_end - c.tok_begin;
    const int blocks = static_cast<int>(ntok > 0 ? (ntok + 255) / 256 : 1);
    {
      KernelTimer kt(MF_K_PACK, s);
      pack_kernel<<<blocks, 256, 0, s>>>(c, d_cu, reinterpret_cast<int2*>(d_pos));
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (n == 0) break;
  }
  return cudaSuccess;
}

// ------------------------------------------------------- editing packs (3D)
// Sample i is [text; source grid; target grid] (specs {text, Hs, Ws, Ht, Wt}):
// text tokens at (0, 0, 0), source token m at (0, m div Ws, m mod Ws), target
// token m at (1, m div Wt, m mod Wt).
struct Pack3Chunk {
  int32_t first, count, tok_begin, tok_end, last;
  int32_t start[kPackChunk];
  int32_t text[kPackChunk];
  int32_t src_n[kPackChunk];   // Hs * Ws
  int32_t src_w[kPackChunk];
  int32_t tgt_w[kPackChunk];
};

__global__ void __launch_bounds__(256) pack3_kernel(const __grid_constant__ Pack3Chunk c,
                                                    int32_t* __restrict__ cu,
                                                    int32_t* __restrict__ pos) {
  __shared__ int32_t s_start[kPackChunk];
  for (int i = threadIdx.x; i < c.count; i += blockDim.x) s_start[i] = c.start[i];
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < c.count; i += blockDim.x) cu[c.first + i] = s_start[i];
    if (c.last && threadIdx.x == 0) cu[c.first + c.count] = c.tok_end;
  }
  if (pos == nullptr) return;
  const int64_t t = static_cast<int64_t>(c.tok_begin) + blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= c.tok_end) return;
  int lo = 0, hi = c.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int32_t k = static_cast<int32_t>(t) - s_start[lo];
  int32_t f = 0, r = 0, col = 0;
  if (k >= c.text[lo]) {
    int32_t m = k - c.text[lo];
    int32_t W = c.src_w[lo];
    if (m >= c.src_n[lo]) {
      m -= c.src_n[lo];
      W = c.tgt_w[lo];
      f = 1;
    }
    r = m / W;
    col = m - r * W;
  }
  pos[3 * t] = f;
  pos[3 * t + 1] = r;
  pos[3 * t + 2] = col;
}

cudaError_t launch_pack3d(const int32_t* specs, int32_t n, int32_t* d_cu, int32_t* d_pos,
                          cudaStream_t s) {
  int64_t start = 0;
  for (int32_t first = 0; first < n || (n == 0 && first == 0); first += kPackChunk) {
    Pack3Chunk c{};
    c.first = first;
    c.count = n - first < kPackChunk ? n - first : kPackChunk;
    c.tok_begin = static_cast<int32_t>(start);
    for (int i = 0; i < c.count; ++i) {
      const int32_t* sp = specs + 5 * (first + i);
      c.start[i] = static_cast<int32_t>(start);
      c.text[i] = sp[0];
      c.src_n[i] = sp[1] * sp[2];
      c.src_w[i] = sp[2];
      c.tgt_w[i] = sp[4];
      start += static_cast<int64_t>(sp[0]) + static_cast<int64_t>(sp[1]) * sp[2] +
               static_cast<int64_t>(sp[3]) * sp[4];
    }
    c.tok_end = static_cast<int32_t>(start);
    c.last = (first + c.count >= n) ? 1 : 0;
    const int64_t ntok = c.tok_end - c.tok_begin;
    const int blocks = static_cast<int>(ntok > 0 ? (ntok + 255) / 256 : 1);
    {
      KernelTimer kt(MF_K_PACK, s);
      pack3_kernel<<<blocks, 256, 0, s>>>(c, d_cu, d_pos);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (n == 0) break;
  }
  return cudaSuccess;
}

// --------------------------------------------------------------------- RoPE
// One block handles kRopeTok tokens: all heads of q and k (rotated) and of v
// (converted only).  Phase 1 builds the (cos, sin) of every rotary pair of those
// tokens in shared memory (shared by all heads and by q and k; the identity when
// pos is null); phase 2 streams 16-byte chunks (4 pairs) through it, four loads
// in flight per thread (with one, the pass was bound by loads in flight: 0.90 of
// the copy bandwidth on the 50k pack, against 1.03 with four; 8 or 16 tokens per
// block measured 1.00 and 0.95).
constexpr int kRopeTok = 4;

// F16_OUT: write fp16 (the attention's internal Q', K', V') instead of bf16, and
// flag values outside the fp16 range in *status.
template <int D, bool F16_OUT>
__global__ void __launch_bounds__(256) rope_kernel(const uint4* __restrict__ q,
                                                   const uint4* __restrict__ k,
                                                   const uint4* __restrict__ v,
                                                   uint4* __restrict__ q_out,
                                                   uint4* __restrict__ k_out,
                                                   uint4* __restrict__ v_out,
                                                   const int32_t* __restrict__ pos, int32_t T,
                                                   int32_t heads,
                                                   const __grid_constant__ RopeFreqs f,
                                                   float sign, uint32_t* status) {
  constexpr int NP = D / 2;  // rotary pairs per head vector
  __shared__ float2 cs[kRopeTok][NP];
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kRopeTok;
  for (int i = threadIdx.x; i < kRopeTok * NP; i += blockDim.x) {
    const int tt = i / NP, P = i % NP;
    float c = 1.f, s = 0.f;
    if (t0 + tt < T && pos != nullptr) {
      const float pp = static_cast<float>(pos[(t0 + tt) * f.naxes + f.axis[P]]);
      rope_sincos(pp, f.omega[P], f.omega_lo[P], sign, &s, &c);
    }
    cs[tt][P] = make_float2(c, s);
  }
  __syncthreads();
  float vmax = 0.f;
  constexpr int CPR = D / 8;  // 16-byte chunks per head vector
  const int per_tok = heads * CPR;
  const int ntok = static_cast<int>(T - t0 < kRopeTok ? T - t0 : kRopeTok);
  const int total = ntok * per_tok;  // chunks of one tensor in this block's tokens
  constexpr int U = 4;               // chunks in flight per thread
  // q, k, v in turn; the block's tokens are contiguous, so chunk i of a tensor sits
  // at t0 per_tok + i, its token at i / per_tok and its pairs at (i % CPR) * 4
  for (int which = 0; which < 3; ++which) {
    const uint4* src = which == 0 ? q : which == 1 ? k : v;
    uint4* dst = which == 0 ? q_out : which == 1 ? k_out : v_out;
    if (src == nullptr) continue;
    const int64_t base = t0 * per_tok;
    for (int i0 = threadIdx.x; i0 < total; i0 += U * blockDim.x) {
      uint4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * static_cast<int>(blockDim.x);
        if (i < total) x[u] = src[base + i];
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * static_cast<int>(blockDim.x);
        if (i >= total) continue;
        const int tt = i / per_tok, P0 = (i % CPR) * 4;
        uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = __uint_as_float(w[e] << 16);
          const float b = __uint_as_float(w[e] & 0xFFFF0000u);
          float ya = a, yb = b;
          if (which < 2) {
            const float2 r = cs[tt][P0 + e];
            ya = fmaf(a, r.x, -b * r.y);
            yb = fmaf(a, r.y, b * r.x);
          }
          if (F16_OUT) {
            vmax = fmaxf(vmax, fmaxf(fabsf(ya), fabsf(yb)));
            w[e] = pack_f16x2(ya, yb);
          } else {
            w[e] = pack_bf16x2(ya, yb);
          }
        }
        dst[base + i] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  if (F16_OUT && !(vmax <= 65504.f)) atomicOr(status, kFlagFp16Range);
}

// ---------------------------------------------------- e4m3 operands
// Operands of the 8-bit forward variant, in two passes over bf16 q, k, v.  In both
// passes a warp works on one token at a time: a half-warp covers one row (token,
// head) of D = 128 with 16-byte chunks of 8 elements (lane l of the half: elements
// [8l, 8l + 8) = rotary pairs [4l, 4l + 4)), and a warp keeps kF8Unroll pairs of
// rows (consecutive heads) in flight, every load issued before any is used.
constexpr int kF8Unroll = 4;
constexpr int kF8Warps = 8;  // warps per block (256 threads)

// Pass 1 (f8_amax_kernel): per-head maxima for the K and V scales.
//   amax2[h]         = max over the head's tokens and rotary pairs of
//                      k_2P^2 + k_2P+1^2, the squared norm of the un-rotated pair.
//                      A rotation keeps a pair's norm, so its root bounds every
//                      rotated component at every position.
//   amax2[heads + h] = max v^2.
// The values are non-negative floats, whose bit patterns order like unsigned
// integers, so atomicMax on the bits takes the maximum; amax2 is zero on entry.
// Each half-warp reduces its row with shuffles, then one lane per row merges it
// into the block's per-head maxima in shared memory, flushed to amax2 at the end.
// Warps stride over tokens (one wave of resident blocks).
template <int D>
__global__ void __launch_bounds__(256) f8_amax_kernel(const uint4* __restrict__ k,
                                                      const uint4* __restrict__ v, int32_t T,
                                                      int32_t heads, bool smem_heads,
                                                      uint32_t* __restrict__ amax2) {
  extern __shared__ uint32_t s_max[];  // [2][heads] when smem_heads
  constexpr int CPR = D / 8;           // 16-byte chunks per row
  static_assert(CPR == 16, "a half-warp covers one row");
  if (smem_heads)
    for (int i = threadIdx.x; i < 2 * heads; i += blockDim.x) s_max[i] = 0u;
  __syncthreads();
  uint32_t* tgt = smem_heads ? s_max : amax2;
  const int lane = threadIdx.x & 31, hl = lane >> 4, l16 = lane & 15;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kF8Warps;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kF8Warps + (threadIdx.x >> 5); t < T;
       t += nw) {
    const uint4* kt = k + t * heads * CPR + l16;
    const uint4* vt = v + t * heads * CPR + l16;
    for (int hb = 0; hb < heads; hb += 2 * kF8Unroll) {
      uint4 x[2 * kF8Unroll];  // K rows, then V rows of the same heads
#pragma unroll
      for (int u = 0; u < 2 * kF8Unroll; ++u) {
        const int h = hb + 2 * (u % kF8Unroll) + hl;
        x[u] = h < heads ? (u < kF8Unroll ? kt : vt)[h * CPR] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 2 * kF8Unroll; ++u) {
        const bool is_v = u >= kF8Unroll;
        const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
        float mx = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = __uint_as_float(w[e] << 16);
          const float b = __uint_as_float(w[e] & 0xFFFF0000u);
          mx = is_v ? fmaxf(mx, fmaxf(a * a, b * b)) : fmaxf(mx, fmaf(a, a, b * b));
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1)
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const int h = hb + 2 * (u % kF8Unroll) + hl;
        if (h < heads && l16 == 0) atomicMax(tgt + (is_v ? heads : 0) + h, __float_as_uint(mx));
      }
    }
  }
  if (smem_heads) {
    __syncthreads();
    for (int i = threadIdx.x; i < 2 * heads; i += blockDim.x)
      if (s_max[i] != 0u) atomicMax(amax2 + i, s_max[i]);
  }
}

// Pass 2 (f8_quant_kernel): one warp per token, all heads of Q, then K, then V.
// Each block's scale s is the power of two of e4m3_scale, so x / s is exact:
//   Q: rotated; s from the row's largest |q'|, written to qscale[token][head];
//   K: rotated; s from sqrt(amax2[h]), the head's largest pair norm;
//   V: s from sqrt(amax2[heads + h]), the head's largest |v|;
// each x / s rounded to E4M3 (nearest even, saturating) into [T][heads][D] bytes.
// The warp's first loads are issued before it builds its token's (cos, sin)
// table, and each later batch while the previous batch is converted.
template <int D>
__global__ void __launch_bounds__(256) f8_quant_kernel(const uint4* __restrict__ q,
                                                       const uint4* __restrict__ k,
                                                       const uint4* __restrict__ v,
                                                       uint2* __restrict__ q8,
                                                       uint2* __restrict__ k8,
                                                       uint2* __restrict__ v8,
                                                       float* __restrict__ qscale,
                                                       const uint32_t* __restrict__ amax2,
                                                       const int32_t* __restrict__ pos, int32_t T,
                                                       int32_t heads,
                                                       const __grid_constant__ RopeFreqs f) {
  constexpr int NP = D / 2;
  constexpr int CPR = D / 8;
  static_assert(CPR == 16 && NP == 64, "a half-warp covers one row");
  __shared__ float2 cs_all[kF8Warps][NP];
  const int wid = threadIdx.x >> 5;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kF8Warps + wid;
  if (t >= T) return;  // warp-uniform; no block-wide barrier follows
  float2* cs = cs_all[wid];
  const int lane = threadIdx.x & 31, hl = lane >> 4, l16 = lane & 15;
  const int nh = (heads + 2 * kF8Unroll - 1) / (2 * kF8Unroll);  // batches per operand
  const int nit = 3 * nh;
  const int64_t row0 = t * heads;
  auto load_batch = [&](int it, uint4 (&x)[kF8Unroll]) {
    const int which = it / nh;
    const int hb = (it - which * nh) * 2 * kF8Unroll;
    const uint4* src = which == 0 ? q : which == 1 ? k : v;
#pragma unroll
    for (int u = 0; u < kF8Unroll; ++u) {
      const int h = hb + 2 * u + hl;
      x[u] = (it < nit && h < heads) ? src[(row0 + h) * CPR + l16] : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  uint4 x[kF8Unroll];
  load_batch(0, x);
  for (int P = lane; P < NP; P += 32) {
    float c = 1.f, s = 0.f;
    if (pos != nullptr) {
      const float pp = static_cast<float>(pos[t * f.naxes + f.axis[P]]);
      rope_sincos(pp, f.omega[P], f.omega_lo[P], 1.f, &s, &c);
    }
    cs[P] = make_float2(c, s);
  }
  __syncwarp();
  for (int it = 0; it < nit; ++it) {
    uint4 xn[kF8Unroll];
    load_batch(it + 1, xn);
    const int which = it / nh;
    const int hb = (it - which * nh) * 2 * kF8Unroll;
    uint2* dst = which == 0 ? q8 : which == 1 ? k8 : v8;
#pragma unroll
    for (int u = 0; u < kF8Unroll; ++u) {
      const int h = hb + 2 * u + hl;
      const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
      float y[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = __uint_as_float(w[e] << 16);
        const float b = __uint_as_float(w[e] & 0xFFFF0000u);
        if (which < 2) {
          const float2 r = cs[l16 * 4 + e];
          y[2 * e] = fmaf(a, r.x, -b * r.y);
          y[2 * e + 1] = fmaf(a, r.y, b * r.x);
        } else {
          y[2 * e] = a;
          y[2 * e + 1] = b;
        }
      }
      float ref;
      if (which == 0) {  // warp-uniform branch: the row maximum of Q'
        ref = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ref = fmaxf(ref, fabsf(y[e]));
#pragma unroll
        for (int off = 8; off > 0; off >>= 1)
          ref = fmaxf(ref, __shfl_xor_sync(0xffffffffu, ref, off));
      } else {
        ref = h < heads ? sqrtf(__uint_as_float(amax2[(which - 1) * heads + h])) : 0.f;
      }
      if (h < heads) {
        const E4m3Scale sc = e4m3_scale(ref);
        if (which == 0 && l16 == 0) qscale[row0 + h] = sc.s;
        const float inv = sc.inv;
        dst[(row0 + h) * CPR + l16] =
            make_uint2(pack_e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv),
                       pack_e4m3x4(y[4] * inv, y[5] * inv, y[6] * inv, y[7] * inv));
      }
    }
#pragma unroll
    for (int u = 0; u < kF8Unroll; ++u) x[u] = xn[u];
  }
}

cudaError_t launch_prep_e4m3(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             uint8_t* q8, uint8_t* k8, uint8_t* v8, float* qscale,
                             uint32_t* amax2, const int32_t* d_pos, int32_t naxes, int32_t T,
                             int32_t heads, int32_t head_dim, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (head_dim != 128) return cudaErrorInvalidValue;
  const bool smem_heads = heads <= 4096;
  // one wave of resident blocks (each loops over the chunks)
  static int per_sm = 0, sms = 0;
  if (per_sm == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f8_amax_kernel<128>, 256,
                                                      8 * 4096) != cudaSuccess || per_sm < 1) {
      per_sm = 1;
      sms = sms > 0 ? sms : 148;
    }
  }
  const int amax_blocks = static_cast<int>(std::max<int64_t>(
      1, std::min<int64_t>((T + kF8Warps - 1) / kF8Warps, static_cast<int64_t>(per_sm) * sms)));
  {
    KernelTimer kt(MF_K_F8_AMAX, s);
    f8_amax_kernel<128><<<amax_blocks, 256, smem_heads ? 8 * heads : 0, s>>>(
        reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), T, heads,
        smem_heads, amax2);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const RopeFreqs f = make_rope_freqs(head_dim, naxes);
  const int blocks = (T + kF8Warps - 1) / kF8Warps;
  {
    KernelTimer kt(MF_K_F8_QUANT, s);
    f8_quant_kernel<128><<<blocks, 256, 0, s>>>(
        reinterpret_cast<const uint4*>(q), reinterpret_cast<const uint4*>(k),
        reinterpret_cast<const uint4*>(v), reinterpret_cast<uint2*>(q8),
        reinterpret_cast<uint2*>(k8), reinterpret_cast<uint2*>(v8), qscale, amax2, d_pos, T,
        heads, f);
  }
  return cudaGetLastError();
}

template <bool F16_OUT>
static cudaError_t launch_rope_t(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 uint16_t* q_out, uint16_t* k_out, uint16_t* v_out,
                                 const int32_t* d_pos, int32_t naxes, int32_t T, int32_t heads,
                                 int32_t head_dim, float sign, uint32_t* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const RopeFreqs f = make_rope_freqs(head_dim, naxes);
  const int blocks = (T + kRopeTok - 1) / kRopeTok;
  auto in = [](const uint16_t* x) { return reinterpret_cast<const uint4*>(x); };
  auto out = [](uint16_t* x) { return reinterpret_cast<uint4*>(x); };
  const int32_t* p = d_pos;
  KernelTimer kt(MF_K_ROPE, s);
  if (head_dim == 128)
    rope_kernel<128, F16_OUT><<<blocks, 256, 0, s>>>(in(q), in(k), in(v), out(q_out), out(k_out),
                                                     out(v_out), p, T, heads, f, sign, status);
  else
    rope_kernel<64, F16_OUT><<<blocks, 256, 0, s>>>(in(q), in(k), in(v), out(q_out), out(k_out),
                                                    out(v_out), p, T, heads, f, sign, status);
  return cudaGetLastError();
}

cudaError_t launch_rope(const uint16_t* q, const uint16_t* k, uint16_t* q_out, uint16_t* k_out,
                        const int32_t* d_pos, int32_t naxes, int32_t T, int32_t heads,
                        int32_t head_dim, float sign, cudaStream_t s) {
  return launch_rope_t<false>(q, k, nullptr, q_out, k_out, nullptr, d_pos, naxes, T, heads,
                              head_dim, sign, nullptr, s);
}

cudaError_t launch_prep_f16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            uint16_t* q_out, uint16_t* k_out, uint16_t* v_out,
                            const int32_t* d_pos, int32_t naxes, int32_t T, int32_t heads,
                            int32_t head_dim, uint32_t* status, cudaStream_t s) {
  return launch_rope_t<true>(q, k, v, q_out, k_out, v_out, d_pos, naxes, T, heads, head_dim,
                             1.0f, status, s);
}

}  // namespace mf
