// Block-diagonal attention backward with the RoPE transpose folded in, on
// tcgen05 / TMEM / TMA.
//
// Gradient of the forward (Mage-Flow training step, rcap.io post listing:
// the loss is back-propagated through the packed attention).  Per sample, head:
//   D_j = <dO_j, O_j>,  P = exp(S - LSE),  dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - D),  dQ' = scale dS K',  dK' = scale dS^T Q',
//   dQ = R(-theta) dQ',  dK = R(-theta) dK'   (R orthogonal, R^T = R(-theta)).
//
// Kernels:
//   bwd_pre_kernel   D = rowsum(dO o O) in fp32 ([h][T]); zeroes the fp32 dQ
//                    accumulator rows.
//   attn_bwd_kernel  one CTA = one sample, one head, one 128-key tile (K_j, V_j
//                    resident in smem); loops over the sample's 128-row Q tiles:
//       warp 8     TMA: K, V once; (Q_i, dO_i) through a 2-stage ring.
//       warp 9     MMA (one thread): S^T = K Q_i^T, dP^T = V dO_i^T (SS);
//                  dV += P^T dO_i (P^T from TMEM, TS); dK += dS^T Q_i and
//                  dQ_i = dS K (SS, dS^T staged in smem, read K- and MN-major).
//       warps 0-3  thread = key row: P^T = exp2(S^T scale log2e - LSE log2e),
//                  P^T -> TMEM (bf16), dS^T = P^T (dP^T - D) -> smem (bf16);
//                  epilogue dV -> bf16, dK -> scale, R(-theta), bf16.
//       warps 4-7  thread = query row: dQ_i from TMEM, scaled, added into the
//                  fp32 accumulator with vector atomics.
//   dq_post_kernel   dQ = R(-theta) dq_acc -> bf16.
// TMEM: S^T [0,128) (P^T bf16 over its first 64 columns), dP^T [128,256) reused
// for dQ_i, dV [256,256+D), dK [256+D,256+2D).
#include <cuda_bf16.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace mf {

struct WorkItemB {
  int32_t sample, head, blk, start, len;
};
// Per-CTA scalars kept in the dynamic shared-memory region.
struct CtaMiscB {
  WorkItemB w;
  int valid;
  uint32_t tmem;
  uint32_t abort;
};
__device__ __forceinline__ bool find_item_b(const int32_t* __restrict__ cu,
                                            const int32_t* __restrict__ order,
                                            const int32_t* __restrict__ prefix, int32_t n,
                                            int32_t blk_rows, int32_t idx, WorkItemB& w) {
  if (n <= 0 || idx >= prefix[n]) return false;
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  w.sample = order[lo];
  w.start = cu[w.sample];
  w.len = cu[w.sample + 1] - w.start;
  const int32_t nb = (w.len + blk_rows - 1) / blk_rows;
  const int32_t local = idx - prefix[lo];
  w.head = local / nb;
  w.blk = local - w.head * nb;
  return true;
}

// ------------------------------------------------------------- preprocess
// Rows are (token, head) pairs in THD order; 8 lanes per row, each covering D/8
// elements.  Per row: D = <dO, O> -> delta[h][t]; -LSE * log2 e -> nlse2[h][t]; the
// row of the fp32 dQ accumulator zeroed; ||dO|| and ||v|| folded into per-head
// maxima (shared memory per block, then one atomicMax per head: non-negative
// floats order like their bit patterns).  Block 0 also writes the pad rows
// (64 x -inf as -LSE log2 e, 64 x 0 as D) that stand in for query rows past a
// sample (they make P = 0 there).
constexpr int kPreRowsPerBlock = 512;
constexpr int kPreMaxHeads = 256;

__device__ __forceinline__ void bf16x8_dot(const uint4& a, const uint4& b, float& acc) {
  const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    acc = fmaf(__uint_as_float(wa[e] << 16), __uint_as_float(wb[e] << 16), acc);
    acc = fmaf(__uint_as_float(wa[e] & 0xFFFF0000u), __uint_as_float(wb[e] & 0xFFFF0000u), acc);
  }
}

template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint4* __restrict__ o,
                                                      const uint4* __restrict__ d_o,
                                                      const uint4* __restrict__ v,
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ nlse2,
                                                      float* __restrict__ delta,
                                                      float* __restrict__ pad,
                                                      float4* __restrict__ dq_acc,
                                                      float* __restrict__ hmax, int64_t rows,
                                                      int32_t T, int32_t heads) {
  constexpr int V = D / 64;  // uint4 (8 bf16) per lane
  __shared__ float s_max[2 * kPreMaxHeads];
  const bool smem_max = heads <= kPreMaxHeads;
  for (int i = threadIdx.x; i < 2 * kPreMaxHeads; i += blockDim.x) s_max[i] = 0.f;
  if (blockIdx.x == 0 && threadIdx.x < 128) pad[threadIdx.x] = threadIdx.x < 64 ? -INFINITY : 0.f;
  __syncthreads();
  const int sub = threadIdx.x & 7;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kPreRowsPerBlock;
  for (int it = 0; it < kPreRowsPerBlock; it += 32) {
    const int64_t row = row0 + it + (threadIdx.x >> 3);
    const bool ok = row < rows;
    float acc = 0.f, ndo = 0.f, nv = 0.f;
    if (ok) {
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const int64_t idx = row * (D / 8) + sub * V + u;
        const uint4 a = o[idx], b = d_o[idx], c = v[idx];
        bf16x8_dot(a, b, acc);
        bf16x8_dot(b, b, ndo);
        bf16x8_dot(c, c, nv);
      }
#pragma unroll
      for (int u = 0; u < 2 * V; ++u)
        dq_acc[row * (D / 4) + sub * 2 * V + u] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
      acc += __shfl_xor_sync(0xffffffffu, acc, m);
      ndo += __shfl_xor_sync(0xffffffffu, ndo, m);
      nv += __shfl_xor_sync(0xffffffffu, nv, m);
    }
    if (ok && sub == 0) {
      const int64_t t = row / heads;
      const int32_t a = static_cast<int32_t>(row - t * heads);
      const int64_t g = static_cast<int64_t>(a) * T + t;
      delta[g] = acc;
      nlse2[g] = lse[g] * -1.4426950408889634f;
      const unsigned bdo = __float_as_uint(sqrtf(ndo)), bv = __float_as_uint(sqrtf(nv));
      if (smem_max) {
        atomicMax(reinterpret_cast<unsigned*>(&s_max[a]), bdo);
        atomicMax(reinterpret_cast<unsigned*>(&s_max[kPreMaxHeads + a]), bv);
      } else {
        atomicMax(reinterpret_cast<unsigned*>(&hmax[a]), bdo);
        atomicMax(reinterpret_cast<unsigned*>(&hmax[heads + a]), bv);
      }
    }
  }
  __syncthreads();
  if (smem_max) {
    for (int i = threadIdx.x; i < heads; i += blockDim.x) {
      if (s_max[i] > 0.f) atomicMax(reinterpret_cast<unsigned*>(&hmax[i]), __float_as_uint(s_max[i]));
      if (s_max[kPreMaxHeads + i] > 0.f)
        atomicMax(reinterpret_cast<unsigned*>(&hmax[heads + i]),
                  __float_as_uint(s_max[kPreMaxHeads + i]));
    }
  }
}

// --------------------------------------------------------- dQ post-process
// dq[t][a][:] = R(-theta(pos_t)) dq_acc[t][a][:] (a plain cast without pos).  One
// block handles kPostTok tokens: their (cos, sin) per rotary pair are formed once
// in shared memory and shared by all heads; then 16-byte fp32 chunks (2 pairs) of
// every head stream through it.
constexpr int kPostTok = 4;

template <int D>
__global__ void __launch_bounds__(256) dq_post_kernel(const float4* __restrict__ acc,
                                                      uint2* __restrict__ dq,
                                                      const int32_t* __restrict__ pos, int32_t T,
                                                      int32_t heads,
                                                      const __grid_constant__ RopeFreqs f) {
  constexpr int NP = D / 2;
  __shared__ float2 cs[kPostTok][NP];
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kPostTok;
  for (int i = threadIdx.x; i < kPostTok * NP; i += blockDim.x) {
    const int tt = i / NP, P = i % NP;
    float c = 1.f, sn = 0.f;
    if (t0 + tt < T && pos != nullptr) {
      const float pp = static_cast<float>(pos[(t0 + tt) * f.naxes + f.axis[P]]);
      rope_sincos(pp, f.omega[P], f.omega_lo[P], -1.f, &sn, &c);
    }
    cs[tt][P] = make_float2(c, sn);
  }
  __syncthreads();
  constexpr int CPR = D / 4;  // float4 chunks per head vector
  const int per_tok = heads * CPR;
  const int ntok = static_cast<int>(T - t0 < kPostTok ? T - t0 : kPostTok);
  for (int i = threadIdx.x; i < ntok * per_tok; i += blockDim.x) {
    const int tt = i / per_tok, ch = i % per_tok;
    const int64_t idx = (t0 + tt) * per_tok + ch;
    const float4 x = acc[idx];
    const int P0 = (ch % CPR) * 2;
    const float2 r0 = cs[tt][P0], r1 = cs[tt][P0 + 1];
    dq[idx] = make_uint2(pack_bf16x2(fmaf(x.x, r0.x, -x.y * r0.y), fmaf(x.x, r0.y, x.y * r0.x)),
                         pack_bf16x2(fmaf(x.z, r1.x, -x.w * r1.y), fmaf(x.z, r1.y, x.w * r1.x)));
  }
}

// --------------------------------------------------------------- main kernel
// One CTA = one sample, one head, one 128-key tile (K', V resident in smem); it
// walks the sample's queries in 64-row tiles i.  Per tile (b = i % 2):
//   S^T_i  = K' Q'_i^T        M=128 keys, N=64, K=d   SS fp16   -> TMEM ST[b]
//   dP^T_i = V dO_i^T         M=128 keys, N=64, K=d   SS bf16   -> TMEM DPT
//   P^T_i  = exp2(S^T scale log2e - LSE log2e) (bf16 -> ST[b] columns [0,32))
//            (the preprocess stores -LSE log2e, so this is one packed FMA per pair)
//   dS^T_i = P^T (dP^T - D) * ds_mul           (fp16 -> smem DS[b])
//   dV    += P^T_i dO_i       M=128 keys, N=d, K=64   TS bf16
//   dK    += dS^T_i Q'_i      M=128 keys, N=d, K=64   SS fp16
//   dQ^T_i = K'^T dS^T_i      M=128 (d),  N=64, K=128 SS fp16   -> TMEM DQT
// dQ is produced transposed (TMEM lane = head-dim index, column = query): the
// warps that drain it write a [query][d] fp32 tile to shared memory with
// conflict-free stores, and one thread adds the tile into the fp32 accumulator
// with a TMA reduce-add (rows past the sample are zero, so they add nothing).
// S^T is double-buffered; the (Q', dO) stage of tile i is released as soon as
// dV_i and dK_i (its last readers) are issued, and dP^T_{i+1} and S^T_{i+2} are
// issued ahead of the GEMMs that need the P/dS warpgroup, so that warpgroup's
// exp/dS work overlaps the tensor core.
//   warp 8     TMA: K', V once; (Q'_i, dO_i) through an NST-stage ring; the
//              lanes copy the tile's -LSE * log2 e and D rows beside them with
//              cp.async (pad rows past the sample), all on the stage barrier.
//   warp 9     MMA issuer (one thread).
//   warps 0-3  thread = key row: P^T, dS^T; epilogue dV, dK (scale, R(-theta)).
//   warps 4-7  thread = head-dim row of dQ^T: smem tile + TMA reduce-add.
// At d = 64 the dQ^T GEMM is padded to M = 128 with a zero smem chunk (its rows
// 64-127 are ignored).
template <int D>
struct BwdCfg {
  static constexpr int BK = 128;                // keys per CTA
  static constexpr int BQ = 64;                 // queries per tile
  static constexpr int NST = 3;                 // (Q', dO) stages
  static constexpr int KCHUNK = 128 * 128;      // 64-column chunk of a 128-row tile
  static constexpr int QCHUNK = 64 * 128;       // 64-column chunk of a 64-row tile
  static constexpr int KTILE = 128 * D * 2;     // K' or V tile
  static constexpr int QTILE = 64 * D * 2;      // Q' or dO tile
  static constexpr int DSTILE = 128 * 64 * 2;   // dS^T tile (one chunk)
  static constexpr int DQTILE = BQ * D * 4;     // fp32 dQ staging tile [query][d]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KTILE;
  static constexpr int OFF_Z = 2 * KTILE;                         // zero chunk (d = 64)
  static constexpr int OFF_Q = OFF_Z + (D == 64 ? KCHUNK : 0);    // [NST]
  static constexpr int OFF_DO = OFF_Q + NST * QTILE;              // [NST]
  static constexpr int OFF_DS = OFF_DO + NST * QTILE;             // [2]
  static constexpr int OFF_DQ = OFF_DS + 2 * DSTILE;
  static constexpr int OFF_VEC = OFF_DQ + DQTILE;                 // [NST] x (-LSE log2e, D) x 64
  static constexpr int OFF_BAR = OFF_VEC + NST * 512;
  static constexpr int OFF_MISC = OFF_BAR + 256;
  static constexpr int SMEM = OFF_MISC + 64;
  static constexpr uint32_t COL_ST0 = 0, COL_ST1 = 64, COL_DPT = 128, COL_DQT = 192;
  static constexpr uint32_t COL_DV = 256, COL_DK = 256 + D;
  // fp16 where Q', K' and the scaled dS meet; bf16 where the caller's V and dO do
  // (gradient-sized values keep bf16's range there).
  static constexpr uint32_t IDESC_S = idesc_f32acc(128, 64, kF16, 0, 0);     // S^T
  static constexpr uint32_t IDESC_DP = idesc_f32acc(128, 64, kBF16, 0, 0);   // dP^T
  static constexpr uint32_t IDESC_DV = idesc_f32acc(128, D, kBF16, 0, 1);    // dV
  static constexpr uint32_t IDESC_DK = idesc_f32acc(128, D, kF16, 0, 1);     // dK
  static constexpr uint32_t IDESC_DQ = idesc_f32acc(128, 64, kF16, 1, 1);    // dQ^T
};
static_assert(BwdCfg<128>::SMEM <= 232448, "backward shared memory over the per-CTA limit");

struct BwdParams {
  const int32_t* cu;
  const int32_t* order;
  const int32_t* prefix;
  const int32_t* pos;
  const float* nlse2;
  const float* delta;
  const float* pad;
  uint32_t* status;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int32_t n, T, heads;
  float scale, scale_log2;
  RopeFreqs f;
  // per-head max ||dO_j|| at [a], max ||v_k|| at [heads + a]: they bound
  // |dS| <= |dP| + |D| <= 2 max||dO|| max||v||, which sets the power-of-two
  // scale under which dS is staged in fp16 (undone in the dK / dQ epilogues)
  const float* hmax;
};

// 2^e with e = floor(log2(2^15 / bound)) clamped to [-64, 64]: scaled |dS| stays
// below 2^15 (fp16 max 65504) and small gradients keep fp16's precision.
__device__ __forceinline__ float ds_scale_for(float max_do, float max_v) {
  const float bound = 2.f * max_do * max_v;
  if (!(bound > 0.f) || !(bound < 3.0e38f)) return 1.f;
  int e = static_cast<int>(floorf(log2f(32768.f / bound)));
  e = max(-64, min(64, e));
  return exp2f(static_cast<float>(e));
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D>;
  // All shared memory is dynamic (no static __shared__), so its base is the
  // start of the CTA's window: 1024-byte aligned, as the 128B-swizzled tiles need.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  uint8_t* gbase = smem_raw;
  CtaMiscB& misc = *reinterpret_cast<CtaMiscB*>(smem_raw + C::OFF_MISC);
  WorkItemB& s_w = misc.w;
  int& s_valid = misc.valid;
  uint32_t& s_tmem = misc.tmem;
  volatile uint32_t& s_abort = misc.abort;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kFlagSmemAlign);
    return;
  }
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sZ = sbase + C::OFF_Z;
  const uint32_t sQ = sbase + C::OFF_Q, sDO = sbase + C::OFF_DO, sDS = sbase + C::OFF_DS;
  const uint32_t sDQ = sbase + C::OFF_DQ, sVEC = sbase + C::OFF_VEC;
  // per stage: -LSE log2 e at [st*128, +64), D at [st*128+64, +64)
  const float* vec = reinterpret_cast<const float*>(gbase + C::OFF_VEC);
  const uint32_t bars = sbase + C::OFF_BAR;
  const uint32_t bar_kv = bars;
  const uint32_t bar_full = bars + 8;                // [NST]
  const uint32_t bar_empty = bar_full + 8 * C::NST;  // [NST]
  const uint32_t bar_st = bar_empty + 8 * C::NST;    // [2]
  const uint32_t bar_dp = bar_st + 16;
  const uint32_t bar_ds = bar_dp + 8;
  const uint32_t bar_dq = bar_ds + 8;
  const uint32_t bar_dq_empty = bar_dq + 8;
  const uint32_t bar_done = bar_dq_empty + 8;
  const uint32_t bar_drain = bar_done + 8;

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_valid = ((*p.status & kFlagBadSeqlens) == 0) &&
              find_item_b(p.cu, p.order, p.prefix, p.n, C::BK, blockIdx.x, s_w);
    if (s_valid) {
      mbar_init(bar_kv, 1);
      for (int i = 0; i < C::NST; ++i) {
        // 32 cp.async arrivals (LSE / D rows) + the TMA issuer's expect-tx arrival
        mbar_init(bar_full + 8 * i, 33);
        mbar_init(bar_empty + 8 * i, 1);
      }
      mbar_init(bar_st, 1);
      mbar_init(bar_st + 8, 1);
      mbar_init(bar_dp, 1);
      mbar_init(bar_ds, 128);
      mbar_init(bar_dq, 1);
      mbar_init(bar_dq_empty, 128);
      mbar_init(bar_done, 1);
      mbar_init(bar_drain, 1);
      fence_mbar_init();
    }
  }
  if (D == 64) {  // zero chunk padding the dQ^T GEMM to M = 128
    uint4* z = reinterpret_cast<uint4*>(gbase + C::OFF_Z);
    for (int i = threadIdx.x; i < C::KCHUNK / 16; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (!s_valid) return;
  if (warp == 9) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const WorkItemB w = s_w;
  const int32_t k0 = w.blk * C::BK;                // first key (in sample)
  const int32_t nq = (w.len + C::BQ - 1) / C::BQ;  // query tiles

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar_kv, 2 * C::KTILE);
      for (int ch = 0; ch < D / 64; ++ch) {
        tma_load_3d(sK + ch * C::KCHUNK, &tm_k, bar_kv, ch * 64, w.head, w.start + k0);
        tma_load_3d(sV + ch * C::KCHUNK, &tm_v, bar_kv, ch * 64, w.head, w.start + k0);
      }
    }
    __syncwarp();
    const int64_t gbase_row = static_cast<int64_t>(w.head) * p.T + w.start;
    int32_t issued = 0;
    for (int32_t i = 0; i < nq; ++i) {
      const int32_t st = i % C::NST, use = i / C::NST;
      if (use > 0 &&
          !__all_sync(0xffffffffu, mbar_wait(bar_empty + 8 * st, (use - 1) & 1, &s_abort))) {
        s_abort = 1;
        if (lane == 0) atomicOr(p.status, kFlagTimeout);
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_full + 8 * st, 2 * C::QTILE);
        for (int ch = 0; ch < D / 64; ++ch) {
          tma_load_3d(sQ + st * C::QTILE + ch * C::QCHUNK, &tm_q, bar_full + 8 * st, ch * 64,
                      w.head, w.start + i * C::BQ);
          tma_load_3d(sDO + st * C::QTILE + ch * C::QCHUNK, &tm_do, bar_full + 8 * st, ch * 64,
                      w.head, w.start + i * C::BQ);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = static_cast<int>(lane) * 2 + u;
        const int32_t qi = i * C::BQ + q;
        const bool q_ok = qi < w.len;
        cp_async_4(sVEC + st * 512 + q * 4, q_ok ? p.nlse2 + gbase_row + qi : p.pad + q);
        cp_async_4(sVEC + st * 512 + 256 + q * 4, q_ok ? p.delta + gbase_row + qi : p.pad + 64 + q);
      }
      cp_async_arrive_noinc(bar_full + 8 * st);
      ++issued;
    }
    if (lane == 0) {
      mbar_wait_drain(bar_kv, 0);
      for (int32_t c = (issued > C::NST ? issued - C::NST : 0); c < issued; ++c)
        mbar_wait_drain(bar_full + 8 * (c % C::NST), (c / C::NST) & 1);
    }
  } else if (warp == 9) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        const bool r = mbar_wait(bar, parity, &s_abort);
        tc_fence_after();
        return r;
      };
      // Shared-memory descriptors: one base per operand buffer, then the start
      // address field (16-byte units, bits 0-13) advanced by a small offset.
      // K-major operand, K-step kk of 16 elements; `chunk` = bytes per 64-col chunk
      auto kofs = [](int kk, uint32_t chunk) -> uint64_t {
        return ((kk >> 2) * chunk + (kk & 3) * 32) >> 4;
      };
      // MN-major operand, K-step kk of 16 rows
      auto mofs = [](int kk) -> uint64_t { return (kk * 2048) >> 4; };
      const uint32_t lbo_a = D == 128 ? static_cast<uint32_t>(C::KCHUNK) : (sZ - sK);
      const uint64_t dK_k = sdesc_sw128(sK, 16, 1024), dV_k = sdesc_sw128(sV, 16, 1024);
      const uint64_t dK_m = sdesc_sw128(sK, lbo_a, 1024);
      const uint64_t dQ_k0 = sdesc_sw128(sQ, 16, 1024), dQ_m0 = sdesc_sw128(sQ, C::QCHUNK, 1024);
      const uint64_t dO_k0 = sdesc_sw128(sDO, 16, 1024), dO_m0 = sdesc_sw128(sDO, C::QCHUNK, 1024);
      const uint64_t dS_k0 = sdesc_sw128(sDS, 16, 1024), dS_m0 = sdesc_sw128(sDS, C::DSTILE, 1024);
      constexpr uint64_t kStage = C::QTILE >> 4, kDsBuf = C::DSTILE >> 4;
      auto full = [&](int32_t i) {
        return wait(bar_full + 8 * (i % C::NST), (i / C::NST) & 1);
      };
      auto issue_st = [&](int32_t i) {  // S^T_i = K' Q'_i^T -> ST[i % 2]
        const uint64_t q = dQ_k0 + (i % C::NST) * kStage;
        const uint32_t d = tmem + ((i & 1) ? C::COL_ST1 : C::COL_ST0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(d, dK_k + kofs(kk, C::KCHUNK), q + kofs(kk, C::QCHUNK), C::IDESC_S, kk > 0);
        mma_commit(bar_st + 8 * (i & 1));
      };
      auto issue_dp = [&](int32_t i) {  // dP^T_i = V dO_i^T -> DPT
        const uint64_t o = dO_k0 + (i % C::NST) * kStage;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::COL_DPT, dV_k + kofs(kk, C::KCHUNK), o + kofs(kk, C::QCHUNK),
                 C::IDESC_DP, kk > 0);
        mma_commit(bar_dp);
      };
      bool ok = wait(bar_kv, 0) && full(0);
      if (ok) {
        issue_st(0);
        issue_dp(0);
        if (nq > 1) {
          ok = full(1);
          if (ok) issue_st(1);
        }
      }
      for (int32_t i = 0; i < nq && ok; ++i) {
        const int32_t st = i % C::NST;
        const uint64_t q_m = dQ_m0 + st * kStage, o_m = dO_m0 + st * kStage;
        const uint64_t ds_k = dS_k0 + (i & 1) * kDsBuf, ds_m = dS_m0 + (i & 1) * kDsBuf;
        const uint32_t stb = tmem + ((i & 1) ? C::COL_ST1 : C::COL_ST0);
        if (!(ok = wait(bar_ds, i & 1))) break;  // P^T_i in TMEM, dS^T_i in smem
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)  // dV += P^T_i dO_i
          mma_ts(tmem + C::COL_DV, stb + kk * 8, o_m + mofs(kk), C::IDESC_DV,
                 (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)  // dK += dS^T_i Q'_i
          mma_ss(tmem + C::COL_DK, ds_k + kofs(kk, C::DSTILE), q_m + mofs(kk), C::IDESC_DK,
                 (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar_empty + 8 * st);  // Q'_i, dO_i no longer read
        if (i + 1 < nq) issue_dp(i + 1);  // DPT was read before bar_ds(i); stage i+1 landed
        if (i > 0 && !(ok = wait(bar_dq_empty, (i - 1) & 1))) break;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk)  // dQ^T_i = K'^T dS^T_i
          mma_ss(tmem + C::COL_DQT, dK_m + mofs(kk), ds_m + mofs(kk), C::IDESC_DQ, kk > 0);
        mma_commit(bar_dq);
        if (i + 2 < nq) {  // ST[i % 2] is free once dV_i (issued above) has read P^T_i
          if (!(ok = full(i + 2))) break;
          issue_st(i + 2);
        }
      }
      if (ok) {
        mma_commit(bar_done);
      } else {
        s_abort = 1;
        atomicOr(p.status, kFlagTimeout);
      }
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------ P / dS warpgroup (keys)
    const uint32_t row = threadIdx.x;  // key row in the tile = TMEM lane
    const uint32_t lane_off = ((warp & 3) * 32) << 16;
    const uint32_t tDPT = tmem + lane_off + C::COL_DPT;
    const bool key_ok = k0 + static_cast<int32_t>(row) < w.len;
    const float sl2 = p.scale_log2;
    // dS is staged in fp16 as ds_mul * dS (a power of two; see ds_scale_for)
    const float ds_mul = ds_scale_for(p.hmax[w.head], p.hmax[p.heads + w.head]);
    float dsmax = 0.f;  // scaled |dS|: flag values outside the fp16 range
    bool ok = true;
    for (int32_t i = 0; i < nq; ++i) {
      const int32_t st = i % C::NST;
      const uint32_t tST = tmem + lane_off + ((i & 1) ? C::COL_ST1 : C::COL_ST0);
      uint8_t* gds = gbase + C::OFF_DS + (i & 1) * C::DSTILE;
      ok = __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * st, (i / C::NST) & 1, &s_abort) &&
                                       mbar_wait(bar_st + 8 * (i & 1), (i >> 1) & 1, &s_abort));
      if (!ok) break;
      tc_fence_after();
      const float4* vl4 = reinterpret_cast<const float4*>(vec + st * 128);  // -LSE log2 e
      const float4* vd4 = vl4 + 16;                                           // D
      // P^T: 64 queries, two per packed FMA; bf16 into ST columns [0, 32) (S^T
      // values already read).  Key rows past the sample get P = 0 (their S^T
      // holds another sample's keys).
      uint64_t pr2[32];
      {
        uint32_t r[64];
        {
          uint32_t r0[32], r1[32];
          tmem_ld32(tST, r0);
          tmem_ld32(tST + 32, r1);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            r[c] = r0[c];
            r[32 + c] = r1[c];
          }
        }
        const uint64_t sl2x2 = f32x2_pack(sl2, sl2);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l = vl4[c4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint64_t x = f32x2_fma(f32x2_pack(__uint_as_float(r[4 * c4 + 2 * h]),
                                                    __uint_as_float(r[4 * c4 + 2 * h + 1])),
                                         sl2x2, h ? f32x2_pack(l.z, l.w) : f32x2_pack(l.x, l.y));
            float x0, x1;
            f32x2_unpack(x, x0, x1);
            pr2[2 * c4 + h] = key_ok ? f32x2_pack(ex2_approx(x0), ex2_approx(x1)) : 0ull;
          }
        }
        uint32_t pk[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          float a, b;
          f32x2_unpack(pr2[u], a, b);
          pk[u] = pack_bf16x2(a, b);
        }
        tmem_st32(tST, pk);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar_dp, i & 1, &s_abort));
      if (!ok) break;
      tc_fence_after();
      // dS^T = P^T (dP^T - D) ds_mul, two queries per packed op; row -> smem
      // DS[i % 2], 128B-swizzled K-major [key][query]: 16-byte unit u (queries
      // 8u..8u+7) stored at u ^ (row % 8)
      const uint64_t dsm2 = f32x2_pack(ds_mul, ds_mul);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t rd[32];
        tmem_ld32(tDPT + c * 32, rd);
        tmem_wait_ld();
        uint32_t pd[16];
#pragma unroll
        for (int u4 = 0; u4 < 8; ++u4) {
          const float4 dd = vd4[c * 8 + u4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint64_t t2 = f32x2_sub(f32x2_pack(__uint_as_float(rd[u4 * 4 + 2 * h]),
                                                     __uint_as_float(rd[u4 * 4 + 2 * h + 1])),
                                          h ? f32x2_pack(dd.z, dd.w) : f32x2_pack(dd.x, dd.y));
            const uint64_t ds2 = f32x2_mul(f32x2_mul(pr2[c * 16 + u4 * 2 + h], dsm2), t2);
            float ds0, ds1;
            f32x2_unpack(ds2, ds0, ds1);
            dsmax = fmax3(dsmax, fabsf(ds0), fabsf(ds1));
            pd[u4 * 2 + h] = pack_f16x2(ds0, ds1);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = c * 4 + u;
          uint4* dst = reinterpret_cast<uint4*>(gds + row * 128 + ((unit ^ (row & 7)) << 4));
          *dst = make_uint4(pd[4 * u], pd[4 * u + 1], pd[4 * u + 2], pd[4 * u + 3]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_ds);
    }
    if (!(dsmax <= 65504.f)) atomicOr(p.status, kFlagFp16Range);
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_done, 0, &s_abort));
    // the four warps agree (a warp whose wait ran out skips the epilogue, and so
    // must every other: the epilogue has a barrier among them)
    const bool all_ok = !named_bar_or(2, 128, !ok);
    if (all_ok) {
      tc_fence_after();
      // dV and dK rows (bf16) are staged in the (now idle) Q' / dO stage buffers
      // as [128 keys][D] with 16-byte units XOR-swizzled by row, then written
      // out by all four warps with coalesced row stores.
      constexpr int UNITS = D / 8;  // 16-byte units per row
      uint8_t* sdv = gbase + C::OFF_Q;
      uint8_t* sdk = gbase + C::OFF_DO;
      auto put = [&](uint8_t* base, int unit, uint4 val) {
        *reinterpret_cast<uint4*>(base + row * (D * 2) + ((unit ^ (row % UNITS)) << 4)) = val;
      };
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::COL_DV + cc * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 4; ++u)
          put(sdv, cc * 4 + u,
              make_uint4(pack_bf16x2(__uint_as_float(r[8 * u]), __uint_as_float(r[8 * u + 1])),
                         pack_bf16x2(__uint_as_float(r[8 * u + 2]), __uint_as_float(r[8 * u + 3])),
                         pack_bf16x2(__uint_as_float(r[8 * u + 4]), __uint_as_float(r[8 * u + 5])),
                         pack_bf16x2(__uint_as_float(r[8 * u + 6]), __uint_as_float(r[8 * u + 7]))));
      }
      const float dk_mul = p.scale / ds_mul;  // exact: ds_mul is a power of two
      // the key row's position coordinates (2 or 3 of them)
      float pv0 = 0.f, pv1 = 0.f, pv2 = 0.f;
      if (key_ok && p.pos != nullptr) {
        const int32_t* pp = p.pos + static_cast<int64_t>(w.start + k0 + row) * p.f.naxes;
        pv0 = static_cast<float>(pp[0]);
        pv1 = static_cast<float>(pp[1]);
        if (p.f.naxes == 3) pv2 = static_cast<float>(pp[2]);
      }
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::COL_DK + cc * 32, r);
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) v[u] = __uint_as_float(r[u]) * dk_mul;
        if (p.pos != nullptr) {
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int P = cc * 16 + u;  // pair index
            float sn, cs;
            const int ax = p.f.axis[P];
            rope_sincos_fast(ax == 0 ? pv0 : ax == 1 ? pv1 : pv2, p.f.omega[P],
                             p.f.omega_lo[P], -1.f, &sn, &cs);
            const float a = v[2 * u], b = v[2 * u + 1];
            v[2 * u] = fmaf(a, cs, -b * sn);
            v[2 * u + 1] = fmaf(a, sn, b * cs);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          put(sdk, cc * 4 + u,
              make_uint4(pack_bf16x2(v[8 * u], v[8 * u + 1]), pack_bf16x2(v[8 * u + 2], v[8 * u + 3]),
                         pack_bf16x2(v[8 * u + 4], v[8 * u + 5]),
                         pack_bf16x2(v[8 * u + 6], v[8 * u + 7])));
      }
      named_bar_sync(2, 128);
      const int32_t nrows = min(C::BK, w.len - k0);
      const int u = static_cast<int>(row) % UNITS;
      for (int r = static_cast<int>(row) / UNITS; r < nrows; r += 128 / UNITS) {
        const int64_t g = ((static_cast<int64_t>(w.start) + k0 + r) * p.heads + w.head) * D + u * 8;
        const int off = r * (D * 2) + ((u ^ (r % UNITS)) << 4);
        *reinterpret_cast<uint4*>(p.dv + g) = *reinterpret_cast<const uint4*>(sdv + off);
        *reinterpret_cast<uint4*>(p.dk + g) = *reinterpret_cast<const uint4*>(sdk + off);
      }
    } else {
      s_abort = 1;
      atomicOr(p.status, kFlagTimeout);
    }
  } else {
    // ------------------------------------------ dQ^T warpgroup (head-dim rows)
    // Per tile: dQ^T from TMEM (thread e = head-dim index), scaled, written as
    // a [query][d] fp32 tile (rows past the sample = 0) to the staging buffer;
    // one thread adds the tile into the accumulator with a TMA reduce-add.  The
    // four warps agree on every step with a barrier-reduction, so a wait that
    // ran out in one of them stops all of them at the same point.
    const uint32_t e = threadIdx.x & 127;  // head-dim index = TMEM lane of dQ^T
    const uint32_t lane_off = ((warp & 3) * 32) << 16;
    const bool e_ok = e < static_cast<uint32_t>(D);
    const bool leader = threadIdx.x == 128;
    // softmax scale over the power-of-two dS staging scale (exact division)
    const float dq_mul = p.scale / ds_scale_for(p.hmax[w.head], p.hmax[p.heads + w.head]);
    float* stage = reinterpret_cast<float*>(gbase + C::OFF_DQ);
    if (leader) tma_prefetch_desc(&tm_dq);
    for (int32_t i = 0; i < nq; ++i) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_dq, i & 1, &s_abort));
      uint32_t r0[32], r1[32];
      if (ok) {
        tc_fence_after();
        tmem_ld32(tmem + lane_off + C::COL_DQT, r0);
        tmem_ld32(tmem + lane_off + C::COL_DQT + 32, r1);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar_dq_empty);
      }
      if (leader) bulk_wait_read_all();  // the previous tile's reduce has read the buffer
      if (named_bar_or(1, 128, !ok)) {
        s_abort = 1;
        if (lane == 0) atomicOr(p.status, kFlagTimeout);
        break;
      }
      const int32_t nvalid = min(C::BQ, w.len - i * C::BQ);
      if (e_ok) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          stage[c * D + e] = c < nvalid ? __uint_as_float(r0[c]) * dq_mul : 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          stage[(32 + c) * D + e] = 32 + c < nvalid ? __uint_as_float(r1[c]) * dq_mul : 0.f;
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (leader) {
        tma_reduce_add_3d(&tm_dq, sDQ, 0, w.head, w.start + i * C::BQ);
        bulk_commit_group();
      }
    }
    if (leader) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
static cudaError_t launch_bwd_d(const AttnBwdArgs& a, cudaStream_t s) {
  using C = BwdCfg<D>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int64_t rows = static_cast<int64_t>(a.T) * a.heads;
  const RopeFreqs f = make_rope_freqs(D, a.naxes);
  if (rows > 0) {
    const int64_t blocks = (rows + kPreRowsPerBlock - 1) / kPreRowsPerBlock;
    KernelTimer kt(MF_K_BWD_PRE, s);
    bwd_pre_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(a.o), reinterpret_cast<const uint4*>(a.d_o),
        reinterpret_cast<const uint4*>(a.v), a.lse, a.nlse2, a.delta, a.pad,
        reinterpret_cast<float4*>(a.dq_acc), a.hmax, rows, a.T, a.heads);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_tmap_thd(&tq, a.q, a.T, a.heads, D, C::BQ, true) ||
      !make_tmap_thd(&tk, a.k, a.T, a.heads, D, C::BK, true) ||
      !make_tmap_thd(&tv, a.v, a.T, a.heads, D, C::BK) ||
      !make_tmap_thd(&tdo, a.d_o, a.T, a.heads, D, C::BQ) ||
      !make_tmap_f32_thd(&tdq, a.dq_acc, a.T, a.heads, D, C::BQ))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.cu = a.cu;
  p.order = a.order;
  p.prefix = a.prefix;
  p.pos = a.pos;
  p.nlse2 = a.nlse2;
  p.delta = a.delta;
  p.pad = a.pad;
  p.status = a.status;
  p.dk = reinterpret_cast<__nv_bfloat16*>(a.dk);
  p.dv = reinterpret_cast<__nv_bfloat16*>(a.dv);
  p.n = a.n;
  p.T = a.T;
  p.heads = a.heads;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.f = f;
  p.hmax = a.hmax;
  const int64_t blocks = (static_cast<int64_t>(a.T + C::BK - 1) / C::BK + a.n) * a.heads;
  if (blocks > 0) {
    {
      KernelTimer kt(MF_K_ATTN_BWD, s);
      attn_bwd_kernel<D><<<static_cast<unsigned>(blocks), 320, C::SMEM, s>>>(tq, tk, tv, tdo, tdq, p);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (rows > 0) {
    KernelTimer kt(MF_K_DQ_POST, s);
    dq_post_kernel<D><<<static_cast<unsigned>((a.T + kPostTok - 1) / kPostTok), 256, 0, s>>>(
        reinterpret_cast<const float4*>(a.dq_acc), reinterpret_cast<uint2*>(a.dq),
        a.pos, a.T, a.heads, f);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

cudaError_t launch_attn_bwd(const AttnBwdArgs& a, cudaStream_t s) {
  return a.head_dim == 128 ? launch_bwd_d<128>(a, s) : launch_bwd_d<64>(a, s);
}

}  // namespace mf
