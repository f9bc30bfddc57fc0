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
// pos is null); phase 2 streams 16-byte chunks (4 pairs) through it.
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
  const int total = 3 * ntok * per_tok;
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int which = i / (ntok * per_tok);  // 0: q, 1: k, 2: v
    const int rem = i - which * ntok * per_tok;
    const int tt = rem / per_tok, ch = rem % per_tok;
    const uint4* src = which == 0 ? q : which == 1 ? k : v;
    uint4* dst = which == 0 ? q_out : which == 1 ? k_out : v_out;
    if (src == nullptr) continue;
    const int64_t idx = (t0 + tt) * per_tok + ch;
    uint4 x = src[idx];
    const int P0 = (ch % CPR) * 4;
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float a = __uint_as_float(w[u] << 16);
      const float b = __uint_as_float(w[u] & 0xFFFF0000u);
      float ya = a, yb = b;
      if (which < 2) {
        const float2 r = cs[tt][P0 + u];
        ya = fmaf(a, r.x, -b * r.y);
        yb = fmaf(a, r.y, b * r.x);
      }
      if (F16_OUT) {
        vmax = fmaxf(vmax, fmaxf(fabsf(ya), fabsf(yb)));
        w[u] = pack_f16x2(ya, yb);
      } else {
        w[u] = pack_bf16x2(ya, yb);
      }
    }
    dst[idx] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (F16_OUT && !(vmax <= 65504.f)) atomicOr(status, kFlagFp16Range);
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
