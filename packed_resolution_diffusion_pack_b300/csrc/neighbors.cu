// Memory-bound neighbours of the packed attention: the packed-CFG rectified-flow
// Euler step, the adaptive LayerNorm modulation that feeds the QKV projection and
// the gated residual after the attention's output projection.
//
// Packed CFG (paperlayer.ai summary 3.2.1; hyper.ai "Experiment"): the
// conditional and unconditional branches are two samples of one packed pass; per
// pair, v = v_u + g (v_c - v_u) over the image rows, then one rectified-flow Euler
// step z <- z + dt v (hyper.ai "Method": z_t = (1 - t) z + t eps, the network
// regresses z - eps).
// Adaptive LayerNorm and gated residual (paperlayer.ai summary 3.3: the
// Transformer-side fused chain of adaptive normalization, rotary embeddings and
// gated residual updates): per sample s, y = LN(x) (1 + scale_s) + shift_s and
// out = x + gate_s h, every token using its own sample's vectors (cu_seqlens).
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mf {

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// Sample holding row t: the last s in [0, n) with cu[s] <= t (zero-length samples
// share a start; the last of them is the one that holds t).  Always in [0, n).
__device__ __forceinline__ int32_t sample_of(const int32_t* __restrict__ cu, int32_t n, int32_t t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------- CFG Euler step
constexpr int kCfgChunk = 256;  // pairs per launch (kernel parameter space)

struct CfgChunk {
  int32_t count;
  int32_t z_begin;                // first latent row of the chunk
  int32_t z_end;                  // one past its last latent row
  int32_t z_start[kCfgChunk];     // first latent row of each pair
  int32_t img_c[kCfgChunk];       // first image token of the conditional sample
  int32_t img_u[kCfgChunk];       // first image token of the unconditional sample
};

// One thread = 8 channels of one latent row.
__global__ void __launch_bounds__(256) cfg_euler_kernel(const __grid_constant__ CfgChunk c,
                                                        const uint4* __restrict__ v,
                                                        float4* __restrict__ z, int32_t C8,
                                                        float g, float dt) {
  __shared__ int32_t s_zs[kCfgChunk];
  for (int i = threadIdx.x; i < c.count; i += blockDim.x) s_zs[i] = c.z_start[i];
  __syncthreads();
  const int64_t nrow = c.z_end - c.z_begin;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       idx < nrow * C8; idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t row = c.z_begin + static_cast<int32_t>(idx / C8);
    const int32_t grp = static_cast<int32_t>(idx % C8);
    int lo = 0, hi = c.count - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_zs[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const int32_t k = row - s_zs[lo];
    float vc[8], vu[8];
    bf16x8_to_f32(v[static_cast<int64_t>(c.img_c[lo] + k) * C8 + grp], vc);
    bf16x8_to_f32(v[static_cast<int64_t>(c.img_u[lo] + k) * C8 + grp], vu);
    float4* zp = z + (static_cast<int64_t>(row) * C8 + grp) * 2;
    float4 a = zp[0], b = zp[1];
    float zz[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) zz[e] = fmaf(dt, fmaf(g, vc[e] - vu[e], vu[e]), zz[e]);
    zp[0] = make_float4(zz[0], zz[1], zz[2], zz[3]);
    zp[1] = make_float4(zz[4], zz[5], zz[6], zz[7]);
  }
}

cudaError_t launch_cfg_euler(const uint16_t* v, const int32_t* specs, int32_t pairs, int32_t C,
                             float g, float dt, float* z, cudaStream_t s) {
  int64_t tok = 0, zrow = 0;
  for (int32_t first = 0; first < pairs; first += kCfgChunk) {
    CfgChunk c{};
    c.count = pairs - first < kCfgChunk ? pairs - first : kCfgChunk;
    c.z_begin = static_cast<int32_t>(zrow);
    for (int i = 0; i < c.count; ++i) {
      const int32_t* sc = specs + 6 * (first + i);
      const int32_t* su = sc + 3;
      const int64_t n_img = static_cast<int64_t>(sc[1]) * sc[2];
      c.z_start[i] = static_cast<int32_t>(zrow);
      c.img_c[i] = static_cast<int32_t>(tok + sc[0]);
      const int64_t Lc = sc[0] + n_img;
      c.img_u[i] = static_cast<int32_t>(tok + Lc + su[0]);
      tok += Lc + su[0] + n_img;
      zrow += n_img;
    }
    c.z_end = static_cast<int32_t>(zrow);
    const int64_t work = static_cast<int64_t>(c.z_end - c.z_begin) * (C / 8);
    if (work == 0) continue;
    const int64_t want = (work + 255) / 256;
    const int blocks = static_cast<int>(want < 148 * 16 ? want : 148 * 16);
    KernelTimer kt(MF_K_CFG_EULER, s);
    cfg_euler_kernel<<<blocks, 256, 0, s>>>(c, reinterpret_cast<const uint4*>(v),
                                            reinterpret_cast<float4*>(z), C / 8, g, dt);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// --------------------------------------------- adaptive LayerNorm, residual
constexpr int kRowWarps = 8;        // rows (warps) per block
constexpr int kCuSmem = 2048;       // cu_seqlens entries cached in shared memory

// Sample of row t from the block's cached cu_seqlens (or global memory when the
// pack has more samples than the cache holds).
struct CuView {
  const int32_t* g;
  const int32_t* s;  // shared copy, or null
  int32_t n;
  __device__ __forceinline__ int32_t sample(int32_t t) const {
    if (s == nullptr) return sample_of(g, n, t);
    int lo = 0, hi = n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
  }
};
__device__ __forceinline__ CuView cache_cu(const int32_t* __restrict__ cu, int32_t n,
                                           int32_t* smem) {
  const bool fits = n + 1 <= kCuSmem;
  if (fits)
    for (int i = threadIdx.x; i <= n; i += blockDim.x) smem[i] = cu[i];
  __syncthreads();
  return CuView{cu, fits ? smem : nullptr, n};
}

// The two bf16 values of a 32-bit word as a packed fp32 pair (low half first).
__device__ __forceinline__ uint64_t bf16x2_pair(uint32_t w) {
  return f32x2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// Sum over the warp's lanes.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Running mean / sum of squared deviations (count n) merged with another
// partial (Chan, Golub and LeVeque's pairwise update; stable in fp32).
__device__ __forceinline__ void merge_stats(float& n, float& mean, float& m2, float nb,
                                            float meanb, float m2b) {
  const float nn = n + nb;
  if (nb > 0.f) {
    const float d = meanb - mean;
    const float w = nb / nn;
    mean = fmaf(d, w, mean);
    m2 = m2 + m2b + d * d * n * w;
    n = nn;
  }
}

// One warp = one row.  Pass 1 streams the row once: every 16-byte chunk's exact
// mean and sum of squared deviations are merged into the lane's running
// statistics, then the 32 lanes merge theirs with shuffles.  Pass 2 reads the row
// again (from L1 / L2: HBM sees it once) and writes the modulated result.  Few
// registers per thread keep many rows in flight.
__global__ void __launch_bounds__(32 * kRowWarps) adaln_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ cu, int32_t n, int32_t T,
    int32_t D8, const uint4* __restrict__ shift, const uint4* __restrict__ scale, float eps,
    uint4* __restrict__ y) {
  __shared__ int32_t s_cu[kCuSmem];
  const CuView cv = cache_cu(cu, n, s_cu);
  const int lane = threadIdx.x & 31;
  const float inv_dm = 1.f / static_cast<float>(D8 * 8);
  for (int32_t t = blockIdx.x * kRowWarps + (threadIdx.x >> 5); t < T;
       t += gridDim.x * kRowWarps) {
    const int64_t base = static_cast<int64_t>(t) * D8;
    const int64_t mbase = static_cast<int64_t>(cv.sample(t)) * D8;
    float cnt = 0.f, mean = 0.f, m2 = 0.f;
#pragma unroll 4
    for (int ch = lane; ch < D8; ch += 32) {
      float f[8];
      bf16x8_to_f32(__ldg(x + base + ch), f);
      const float cm = (((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7]))) * 0.125f;
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        a = fmaf(f[e] - cm, f[e] - cm, a);
        b = fmaf(f[e + 1] - cm, f[e + 1] - cm, b);
      }
      merge_stats(cnt, mean, m2, 8.f, cm, a + b);
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
      const float nb = __shfl_xor_sync(0xffffffffu, cnt, m);
      const float mb = __shfl_xor_sync(0xffffffffu, mean, m);
      const float qb = __shfl_xor_sync(0xffffffffu, m2, m);
      if (cnt == 0.f) {
        cnt = nb;
        mean = mb;
        m2 = qb;
      } else {
        merge_stats(cnt, mean, m2, nb, mb, qb);
      }
    }
    const float rstd = rsqrtf(m2 * inv_dm + eps);
#pragma unroll 4
    for (int ch = lane; ch < D8; ch += 32) {
      float f[8], sh[8], sc[8];
      bf16x8_to_f32(__ldg(x + base + ch), f);
      bf16x8_to_f32(__ldg(shift + mbase + ch), sh);
      bf16x8_to_f32(__ldg(scale + mbase + ch), sc);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = fmaf((f[e] - mean) * rstd, 1.f + sc[e], sh[e]);
      y[base + ch] = f32_to_bf16x8(f);
    }
  }
}

// The same modulation with the rows streamed through shared memory: one block
// per SM owns a contiguous run of rows; a producer thread keeps up to kRingSlots
// rows in flight with bulk copies into a ring, and kRingWarps consumer warps take
// the rows in turn (statistics from shared memory, then the modulated row written
// straight to global memory).  Loads never wait on a row's reduction.  Measured
// on the 50k pack at Dm = 3072: 0.69 of the copy bandwidth for adaln_kernel (a
// warp per row serialises load, reduce and store); 0.62 / 0.75 / 0.77 for this
// ring with 8 / 16 / 24 consumer warps merging per-chunk statistics pairwise, when
// the consumers were issue bound (70 % issue active, a division per merge); 0.85
// with the two-pass statistics and packed arithmetic below.  More slots than
// consumers (32, 36) changed nothing.  Rows of at most kRingRowBytes; wider rows
// take adaln_kernel.
constexpr int kRingWarps = 24;                     // consumer warps (800 threads a block)
constexpr int kRingSlots = 24;                     // rows in flight per block (at most)
constexpr int kRingBytes = 196608;                 // ring size
constexpr int kRingRowBytes = kRingBytes / 2;      // at least two slots
__global__ void __launch_bounds__(32 * (kRingWarps + 1), 1) adaln_ring_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ cu, int32_t n, int32_t T,
    int32_t D8, const uint4* __restrict__ shift, const uint4* __restrict__ scale, float eps,
    uint4* __restrict__ y, int32_t nslot) {
  extern __shared__ __align__(128) uint8_t ring[];
  const uint32_t rowbytes = static_cast<uint32_t>(D8) * 16u;
  const uint32_t sring = smem_u32(ring);
  const uint32_t bar_full = sring + nslot * rowbytes;  // [nslot]
  const uint32_t bar_empty = bar_full + 8 * nslot;     // [nslot]
  __shared__ uint32_t s_abort;
  const int32_t per = (T + gridDim.x - 1) / gridDim.x;
  const int32_t t0 = blockIdx.x * per;
  const int32_t rows = max(0, min(T, t0 + per) - t0);
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < nslot; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kRingWarps) {
    // producer: row i into slot i % nslot once its previous row was consumed
    if (lane == 0) {
      int32_t issued = 0;
      for (int32_t i = 0; i < rows; ++i) {
        const int32_t slot = i % nslot, use = i / nslot;
        if (use > 0 && !mbar_wait_bk(bar_empty + 8 * slot, (use - 1) & 1, &s_abort)) {
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(bar_full + 8 * slot, rowbytes);
        bulk_load(sring + slot * rowbytes, x + static_cast<int64_t>(t0 + i) * D8, rowbytes,
                  bar_full + 8 * slot);
        ++issued;
      }
      // every issued copy lands before the block exits
      for (int32_t c = (issued > nslot ? issued - nslot : 0); c < issued; ++c)
        mbar_wait_drain(bar_full + 8 * (c % nslot), (c / nslot) & 1);
    }
  } else {
    const float inv_dm = 1.f / static_cast<float>(D8 * 8);
    int32_t s = 0, s_end = -1;  // sample of the current row and its end
    for (int32_t i = static_cast<int32_t>(warp); i < rows; i += kRingWarps) {
      const int32_t slot = i % nslot, t = t0 + i;
      if (!__all_sync(0xffffffffu, mbar_wait_bk(bar_full + 8 * slot, (i / nslot) & 1, &s_abort))) {
        s_abort = 1;
        break;
      }
      if (t >= s_end) {
        s = sample_of(cu, n, t);
        s_end = __ldg(cu + s + 1);
      }
      const uint4* row = reinterpret_cast<const uint4*>(ring + slot * rowbytes);
      // Two passes over the row in shared memory: the exact mean (fp32 sum), then the
      // sum of squared deviations about it, both with packed two-lane arithmetic; the
      // classic two-pass variance, as accurate as the pairwise merges it replaces at
      // a fraction of their instructions (this loop is issue bound).
      uint64_t s2a = 0, s2b = 0;  // two packed accumulators (0 bits = +0.0f pairs)
      for (int ch = lane; ch < D8; ch += 32) {
        const uint4 u = row[ch];
        s2a = f32x2_add(s2a, bf16x2_pair(u.x));
        s2b = f32x2_add(s2b, bf16x2_pair(u.y));
        s2a = f32x2_add(s2a, bf16x2_pair(u.z));
        s2b = f32x2_add(s2b, bf16x2_pair(u.w));
      }
      float sa, sb, sc_, sd;
      f32x2_unpack(s2a, sa, sb);
      f32x2_unpack(s2b, sc_, sd);
      const float mean = warp_sum((sa + sb) + (sc_ + sd)) * inv_dm;
      const uint64_t nmean2 = f32x2_pack(-mean, -mean);
      uint64_t q2a = 0, q2b = 0;
      for (int ch = lane; ch < D8; ch += 32) {
        const uint4 u = row[ch];
        const uint64_t d0 = f32x2_add(bf16x2_pair(u.x), nmean2), d1 = f32x2_add(bf16x2_pair(u.y), nmean2);
        const uint64_t d2 = f32x2_add(bf16x2_pair(u.z), nmean2), d3 = f32x2_add(bf16x2_pair(u.w), nmean2);
        q2a = f32x2_fma(d0, d0, q2a);
        q2b = f32x2_fma(d1, d1, q2b);
        q2a = f32x2_fma(d2, d2, q2a);
        q2b = f32x2_fma(d3, d3, q2b);
      }
      f32x2_unpack(q2a, sa, sb);
      f32x2_unpack(q2b, sc_, sd);
      const float m2 = warp_sum((sa + sb) + (sc_ + sd));
      const float rstd = rsqrtf(m2 * inv_dm + eps);
      const int64_t base = static_cast<int64_t>(t) * D8, mbase = static_cast<int64_t>(s) * D8;
      // y = ((x - mean) rstd)(1 + scale) + shift: (x - mean) rstd as x rstd - mean rstd
      const uint64_t rstd2 = f32x2_pack(rstd, rstd), nmr2 = f32x2_pack(-mean * rstd, -mean * rstd);
      const uint64_t one2 = f32x2_pack(1.f, 1.f);
      for (int ch = lane; ch < D8; ch += 32) {
        const uint4 u = row[ch], sh = __ldg(shift + mbase + ch), sc = __ldg(scale + mbase + ch);
        const uint32_t xw[4] = {u.x, u.y, u.z, u.w}, hw[4] = {sh.x, sh.y, sh.z, sh.w};
        const uint32_t cw[4] = {sc.x, sc.y, sc.z, sc.w};
        uint32_t ow[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t a2 = f32x2_fma(bf16x2_pair(xw[k]), rstd2, nmr2);
          const uint64_t y2 = f32x2_fma(a2, f32x2_add(bf16x2_pair(cw[k]), one2), bf16x2_pair(hw[k]));
          float y0, y1;
          f32x2_unpack(y2, y0, y1);
          ow[k] = pack_bf16x2(y0, y1);
        }
        y[base + ch] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      }
      __syncwarp();  // every lane's reads of the slot are done
      if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
    }
  }
}

__global__ void __launch_bounds__(32 * kRowWarps) gated_residual_kernel(
    const uint4* __restrict__ x, const uint4* __restrict__ h, const int32_t* __restrict__ cu,
    int32_t n, int32_t T, int32_t D8, const uint4* __restrict__ gate, uint4* __restrict__ out) {
  __shared__ int32_t s_cu[kCuSmem];
  const CuView cv = cache_cu(cu, n, s_cu);
  const int lane = threadIdx.x & 31;
  for (int32_t t = blockIdx.x * kRowWarps + (threadIdx.x >> 5); t < T;
       t += gridDim.x * kRowWarps) {
    const int64_t base = static_cast<int64_t>(t) * D8;
    const int64_t gbase = static_cast<int64_t>(cv.sample(t)) * D8;
    for (int ch = lane; ch < D8; ch += 32) {
      float a[8], b[8], gg[8];
      bf16x8_to_f32(x[base + ch], a);
      bf16x8_to_f32(h[base + ch], b);
      bf16x8_to_f32(__ldg(gate + gbase + ch), gg);
#pragma unroll
      for (int e = 0; e < 8; ++e) a[e] = fmaf(gg[e], b[e], a[e]);
      out[base + ch] = f32_to_bf16x8(a);
    }
  }
}

// Grid of a row kernel: every block resident at once (SMs x blocks per SM from
// the occupancy calculator), each striding over rows, capped by the row count.
template <typename K>
static int row_blocks(K kernel, int32_t T) {
  int dev = 0, sms = 148, per_sm = 1;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32 * kRowWarps, 0) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (static_cast<int64_t>(T) + kRowWarps - 1) / kRowWarps;
  const int64_t full = static_cast<int64_t>(sms) * per_sm;
  return static_cast<int>(want < full ? want : full);
}

cudaError_t launch_adaln(const uint16_t* x, const int32_t* cu, int32_t n, int32_t T, int32_t Dm,
                         const uint16_t* shift, const uint16_t* scale, float eps, uint16_t* y,
                         cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int64_t rowbytes = static_cast<int64_t>(Dm) * 2;
  if (rowbytes <= kRingRowBytes) {
    // rows through a shared-memory ring (see adaln_ring_kernel)
    static bool attr_done = false;
    if (!attr_done) {
      cudaError_t e = cudaFuncSetAttribute(adaln_ring_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kRingBytes + 16 * kRingSlots);
      if (e != cudaSuccess) return e;
      attr_done = true;
    }
    const int nslot = static_cast<int>(kRingBytes / rowbytes < kRingSlots ? kRingBytes / rowbytes
                                                                           : kRingSlots);
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int blocks = static_cast<int>(T < sms ? T : sms);
    KernelTimer kt(MF_K_ADALN, s);
    adaln_ring_kernel<<<blocks, 32 * (kRingWarps + 1),
                        static_cast<size_t>(nslot) * rowbytes + 16 * nslot, s>>>(
        reinterpret_cast<const uint4*>(x), cu, n, T, Dm / 8,
        reinterpret_cast<const uint4*>(shift), reinterpret_cast<const uint4*>(scale), eps,
        reinterpret_cast<uint4*>(y), nslot);
    return cudaGetLastError();
  }
  KernelTimer kt(MF_K_ADALN, s);
  adaln_kernel<<<row_blocks(adaln_kernel, T), 32 * kRowWarps, 0, s>>>(
      reinterpret_cast<const uint4*>(x), cu, n, T, Dm / 8, reinterpret_cast<const uint4*>(shift),
      reinterpret_cast<const uint4*>(scale), eps, reinterpret_cast<uint4*>(y));
  return cudaGetLastError();
}

cudaError_t launch_gated_residual(const uint16_t* x, const uint16_t* h, const int32_t* cu,
                                  int32_t n, int32_t T, int32_t Dm, const uint16_t* gate,
                                  uint16_t* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  KernelTimer kt(MF_K_GATED_RESIDUAL, s);
  const int64_t want = (static_cast<int64_t>(T) + kRowWarps - 1) / kRowWarps;
  gated_residual_kernel<<<static_cast<unsigned>(want < 148 * 32 ? want : 148 * 32), 32 * kRowWarps,
                          0, s>>>(
      reinterpret_cast<const uint4*>(x), reinterpret_cast<const uint4*>(h), cu, n, T, Dm / 8,
      reinterpret_cast<const uint4*>(gate), reinterpret_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace mf
