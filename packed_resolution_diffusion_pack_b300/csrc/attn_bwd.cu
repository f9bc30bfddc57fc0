// Block-diagonal attention backward with the RoPE transpose folded in, on
// tcgen05 / TMEM / TMA.
//
// Gradient of the forward (Mage-Flow training step, rcap.io post listing:
// the loss is back-propagated through the packed attention).  Per sample, head:
//   D_j = <dO_j, O_j>,  P = exp(S - LSE),  dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - D),  dQ' = scale dS K',  dK' = scale dS^T Q',
//   dQ = R(-theta) dQ',  dK = R(-theta) dK'   (R orthogonal, R^T = R(-theta)).
//
// Kernels (the attention ones persistent, one CTA per SM, over work items of one
// sample, head and 128-row tile, longest samples first):
//   bwd_pre_kernel      D = rowsum(dO o O) and -LSE log2 e in fp32 ([h][T]);
//                       per-head maxima of ||dO|| and ||v||.
//   attn_bwd_kv_kernel  dK, dV per 128-key tile (CTAs claim items through an
//                       atomic counter); in the stored-dS form also writes dS^T.
//   attn_bwd_dq_kernel  dQ per 128-query tile as one streaming GEMM over the
//                       stored dS^T (CTAs stride over the list).
//   attn_bwd_q_kernel   dQ per 128-query tile recomputing S and dP (the recompute
//                       form; CTAs claim items through an atomic counter).
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
  // dK / dV kernel: the work items its producer has claimed, ring slot k % 4 for
  // the CTA's k-th item (sample < 0: no more items)
  WorkItemB ring[4];
};
static_assert(sizeof(CtaMiscB) <= 128, "per-CTA scalars: 128 bytes in each kernel's layout");
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
// elements.  Per row: D = <dO, O> -> delta[h][t]; -LSE * log2 e -> nlse2[h][t];
// ||dO|| and ||v|| folded into per-head
// maxima (shared memory per block, then one atomicMax per head: non-negative
// floats order like their bit patterns).  Block 0 also writes the pad rows
// (128 x -inf as -LSE log2 e, 128 x 0 as D) that stand in for query rows past a
// sample (they make P = 0 there).
constexpr int kPreRowsPerBlock = 128;
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
                                                      float* __restrict__ hmax, int64_t rows,
                                                      int32_t T, int32_t heads) {
  constexpr int V = D / 64;  // uint4 (8 bf16) per lane
  __shared__ float s_max[2 * kPreMaxHeads];
  const bool smem_max = heads <= kPreMaxHeads;
  for (int i = threadIdx.x; i < 2 * kPreMaxHeads; i += blockDim.x) s_max[i] = 0.f;
  if (blockIdx.x == 0) pad[threadIdx.x] = threadIdx.x < 128 ? -INFINITY : 0.f;  // 256 threads
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

// ------------------------------------------------------------ main kernels
// The backward runs as two kernels that need no atomics on the data: each output
// row is written by exactly one work item.
//  attn_bwd_kv_kernel  one item = one sample, one head, one 128-key tile (K', V
//    resident): over the sample's 128-row query tiles i it accumulates
//      S^T_i  = K' Q'_i^T      M=128 keys, N=128, K=d    SS fp16  -> TMEM ST
//      P^T_i  = exp2(S^T scale log2e - LSE log2e)  (bf16, back into ST)
//      dP^T_i = V dO_i^T       M=128 keys, N=128, K=d    SS bf16  -> TMEM DPT
//      dS^T_i = P^T (dP^T - D) * ds_mul            (fp16, back into DPT)
//      dV    += P^T_i dO_i     M=128 keys, N=d,   K=128  TS bf16 (P^T from TMEM)
//      dK    += dS^T_i Q'_i    M=128 keys, N=d,   K=128  TS fp16 (dS^T from TMEM)
//    and writes dV and R(-theta) scale dK / ds_mul.
//  attn_bwd_q_kernel   one item = one sample, one head, one 128-query tile (Q',
//    dO resident): over the sample's 128-key tiles j it recomputes
//      S_j  = Q' K'_j^T        M=128 queries, N=128, K=d  SS fp16  -> TMEM S
//      dP_j = dO V_j^T         M=128 queries, N=128, K=d  SS bf16  -> TMEM DP[j % 2]
//      dS_j = P (dP - D) * ds_mul, P = exp2(S scale log2e - LSE log2e)
//                              (fp16, back into DP[j % 2])
//      dQ  += dS_j K'_j        M=128 queries, N=d, K=128  TS fp16 (dS from TMEM)
//    and writes dQ = R(-theta) scale dQ' / ds_mul in bf16.
// Splitting the work this way recomputes S and dP for dQ (7 GEMMs instead of
// 5), but a single kernel would have to add every key tile's dQ contribution
// into a global fp32 accumulator, and those additions (one fp32 add per key
// tile, query and head-dim element, 15 GB at the 50k pack) are limited by the L2
// reduction throughput (about 2.4 TB/s measured, with both bulk tensor
// reduce-adds and per-element reductions): slower than the extra GEMMs.
// Both kernels: warps 0-7 are two elementwise warpgroups, each covering 64 of the
// 128 columns of a tile (thread = TMEM lane = the tile's row); warp 8 issues TMA;
// warp 9 is the single MMA-issuing thread; warps 10-11 idle.  Every GEMM runs at
// N = 128 or N = d.
template <int D>
struct BwdCfg {
  static constexpr int BK = 128, BQ = 128;      // keys / queries per tile
  static constexpr int CHUNK = 128 * 128;       // 64-column (128-byte) chunk of a 128-row tile
  static constexpr int TILE = 128 * D * 2;      // any 128-row 16-bit operand tile
  static constexpr int VEC = 2 * BQ * 4;        // per stage: -LSE log2 e, D of BQ queries
  // kv kernel: K', V resident; (Q'_i, dO_i) through NST stages
  static constexpr int NST = D == 128 ? 2 : 3;
  static constexpr int KV_OFF_K = 0, KV_OFF_V = TILE, KV_OFF_Q = 2 * TILE;
  static constexpr int KV_OFF_DO = KV_OFF_Q + NST * TILE;
  static constexpr int KV_OFF_VEC = KV_OFF_DO + NST * TILE;
  static constexpr int KV_OFF_BAR = KV_OFF_VEC + NST * VEC;
  static constexpr int KV_OFF_MISC = KV_OFF_BAR + 256;
  static constexpr int KV_SMEM = KV_OFF_MISC + 128;
  // q kernel: Q', dO resident; K'_j through a ring of KSLOT tiles, V_j of VSLOT
  static constexpr int KSLOT = 3, VSLOT = 2;
  static constexpr int Q_OFF_Q = 0, Q_OFF_DO = TILE, Q_OFF_K = 2 * TILE;
  static constexpr int Q_OFF_V = Q_OFF_K + KSLOT * TILE;
  static constexpr int Q_OFF_BAR = Q_OFF_V + VSLOT * TILE;
  static constexpr int Q_OFF_MISC = Q_OFF_BAR + 256;
  static constexpr int Q_SMEM = Q_OFF_MISC + 128;
  // dQ-from-stored-dS kernel: (dS^T tile, K' tile) per stage, DQ_NS stages
  static constexpr int DS_TILE = 128 * 128 * 2;
  static constexpr int DQ_STAGE = DS_TILE + TILE;
  static constexpr int DQ_NS = D == 128 ? 3 : 4;
  static constexpr int DQ_OFF_BAR = DQ_NS * DQ_STAGE;
  static constexpr int DQ_OFF_MISC = DQ_OFF_BAR + 256;
  static constexpr int DQ_SMEM = DQ_OFF_MISC + 128;
  // TMEM columns
  static constexpr uint32_t KV_ST = 0, KV_DPT = 128, KV_DV = 256, KV_DK = 256 + D;
  static constexpr uint32_t Q_S = 0, Q_DP = 128, Q_DQ = 384;  // DP: two buffers
  // fp16 where Q', K' and the scaled dS meet; bf16 where the caller's V and dO do
  // (gradient-sized values keep bf16's range there).
  static constexpr uint32_t IDESC_S = idesc_f32acc(128, 128, kF16, 0, 0);   // S^T and S
  static constexpr uint32_t IDESC_DP = idesc_f32acc(128, 128, kBF16, 0, 0); // dP^T and dP
  static constexpr uint32_t IDESC_DV = idesc_f32acc(128, D, kBF16, 0, 1);   // dV (TS)
  static constexpr uint32_t IDESC_DKQ = idesc_f32acc(128, D, kF16, 0, 1);   // dK, dQ (TS)
  // dQ = dS K' with both operands MN-major in shared memory (dS^T rows are keys)
  static constexpr uint32_t IDESC_DQS = idesc_f32acc(128, D, kF16, 1, 1);
  static_assert(KV_OFF_Q % 1024 == 0 && KV_OFF_DO % 1024 == 0 && Q_OFF_K % 1024 == 0,
                "swizzled tiles start on 1024-byte boundaries");
  static_assert(KV_SMEM <= 232448 && Q_SMEM <= 232448 && DQ_SMEM <= 232448,
                "shared memory over the per-CTA limit");
  static_assert(DQ_STAGE % 1024 == 0 && DS_TILE % 1024 == 0, "dS / K' tiles on 1024-byte boundaries");
  static_assert(8 * (2 + 2 * NST + 17) <= 256 && 8 * (2 + 2 * (KSLOT + VSLOT) + 20) <= 256,
                "barrier areas");
};

// 384 threads: 170 registers each at launch (65,536 / 384), no reallocation.
constexpr int kBwdThreads = 384;

struct BwdParams {
  const int32_t* cu;
  const int32_t* order;
  const int32_t* prefix;
  const int32_t* pos;
  const float* nlse2;
  const float* delta;
  const float* pad;
  uint32_t* status;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int32_t n, T, heads;
  float scale, scale_log2;
  RopeFreqs f;
  // per-head max ||dO_j|| at [a], max ||v_k|| at [heads + a]: they bound
  // |dS| <= |dP| + |D| <= 2 max||dO|| max||v||, which sets the power-of-two
  // scale under which dS is staged in fp16 (undone in the dK / dQ epilogues)
  const float* hmax;
  // test hook (0 = off): the MMA thread first waits, at most this many
  // microseconds, on a barrier that nothing arrives on (failure-detection tests)
  uint32_t stall_us;
  // stored-dS form: scaled fp16 dS^T in 128-key tiles of ds_cols / 8 units of 8
  // queries (null: dQ recomputes); see ds_tile_base
  uint16_t* ds;
  int64_t ds_cols;
  // work-item counters, zeroed by the schedule kernel: the dK / dV kernel's at
  // next_item[0], the recompute form's dQ kernel's at next_item[1]; each CTA
  // claims its next item (an index into the ranked list) with an atomic add
  uint32_t* next_item;
};

// The stored-dS array holds 128-key tiles, each [ds_cols / 8 units][128 keys][8
// queries] (2 KB a unit), so a tile's 16-unit query block is 32 contiguous KB and
// 32 consecutive keys of one unit are 512 contiguous bytes.  First tile of (sample,
// head)'s block: heads (ceil(cu[i] / 128) + i) + head a_i / 128, a_i = L_i rounded
// up to 128.  The blocks never overlap: a sample's heads a_i / 128 tiles end at or
// before heads (ceil(cu[i + 1] / 128) + i + 1), the next sample's first tile.
__device__ __forceinline__ int64_t ds_tile_base(int32_t heads, int32_t start, int32_t sample,
                                                int32_t head, int32_t padded_len) {
  return static_cast<int64_t>(heads) * ((static_cast<int64_t>(start) + 127) / 128 + sample) +
         static_cast<int64_t>(head) * (padded_len / 128);
}

// 2^e with e = floor(log2(2^15 / bound)) clamped to [-64, 64]: scaled |dS| stays
// below 2^15 (fp16 max 65504) and small gradients keep fp16's precision.
__device__ __forceinline__ float ds_scale_for(float max_do, float max_v) {
  const float bound = 2.f * max_do * max_v;
  if (!(bound > 0.f) || !(bound < 3.0e38f)) return 1.f;
  int e = static_cast<int>(floorf(log2f(32768.f / bound)));
  e = max(-64, min(64, e));
  return exp2f(static_cast<float>(e));
}

// MMA-operand offsets in a 128B-swizzled tile, in the 16-byte units of a
// descriptor's start-address field.  K-major operand: K-step kk of 16 elements
// is 32 bytes into the 128-byte rows, the next 64-column chunk every 4 steps.
template <int D>
__device__ __forceinline__ uint64_t kofs(int kk) {
  return ((kk >> 2) * BwdCfg<D>::CHUNK + (kk & 3) * 32) >> 4;
}
// MN-major operand: K-step kk of 16 rows of 128 bytes.
__device__ __forceinline__ uint64_t mofs(int kk) { return (kk * 2048) >> 4; }

// TMEM column of K-step kk (16 elements = 8 columns) of a 16-bit operand that the
// two elementwise warpgroups packed into columns [0, 32) and [64, 96) of a
// 128-column region (warpgroup h holds elements [64h, 64h + 64)).
__device__ __forceinline__ uint32_t packed_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// 32 consecutive values (columns [32 cc, 32 cc + 32)) of one output row: times
// mul, rotated by R(-theta) at the row's position coordinates pv when rotating,
// converted to bf16 and stored at dst (the row's first element) as four 16-byte
// stores.
__device__ __forceinline__ void store_row_chunk(__nv_bfloat16* dst, int cc,
                                                const uint32_t (&r)[32], float mul, bool rotate,
                                                const float (&pv)[3], const RopeFreqs& f) {
  float v[32];
#pragma unroll
  for (int u = 0; u < 32; ++u) v[u] = __uint_as_float(r[u]) * mul;
  if (rotate) {
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int P = cc * 16 + u;  // pair index
      float sn, cs;
      const int ax = f.axis[P];
      rope_sincos_fast(ax == 0 ? pv[0] : ax == 1 ? pv[1] : pv[2], f.omega[P], f.omega_lo[P], -1.f,
                       &sn, &cs);
      const float a = v[2 * u], b = v[2 * u + 1];
      v[2 * u] = fmaf(a, cs, -b * sn);
      v[2 * u + 1] = fmaf(a, sn, b * cs);
    }
  }
  uint4* out = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
  for (int u = 0; u < 4; ++u)
    out[u] = make_uint4(pack_bf16x2(v[8 * u], v[8 * u + 1]), pack_bf16x2(v[8 * u + 2], v[8 * u + 3]),
                        pack_bf16x2(v[8 * u + 4], v[8 * u + 5]),
                        pack_bf16x2(v[8 * u + 6], v[8 * u + 7]));
}

// Position coordinates (up to 3) of token t as floats; zeros without positions.
__device__ __forceinline__ void token_pos(const BwdParams& p, int64_t t, bool ok, float (&pv)[3]) {
  pv[0] = pv[1] = pv[2] = 0.f;
  if (ok && p.pos != nullptr) {
    const int32_t* pp = p.pos + t * p.f.naxes;
    pv[0] = static_cast<float>(pp[0]);
    pv[1] = static_cast<float>(pp[1]);
    if (p.f.naxes == 3) pv[2] = static_cast<float>(pp[2]);
  }
}

// The CTA's k-th work item (static striding over the longest-first list).
__device__ __forceinline__ bool cta_item(const BwdParams& p, int32_t k, WorkItemB& w) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(k) * gridDim.x;
  if (idx > INT32_MAX) return false;
  return find_item_b(p.cu, p.order, p.prefix, p.n, 128, static_cast<int32_t>(idx), w);
}

// ------------------------------------------------------------- dK, dV kernel
// Persistent: one CTA per SM claims (sample, head, key tile) items from the
// longest-first list through an atomic counter.  Per item: K', V loaded once (as
// soon as the previous item's last S^T and dP^T have read theirs), (Q'_i, dO_i)
// through the stage ring that runs on across items, the dV / dK accumulators
// freed for the next item as soon as the elementwise warps have loaded them; the
// epilogue's conversion and stores then overlap the next item's first GEMMs.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using C = BwdCfg<D>;
  // All shared memory is dynamic (no static __shared__), so its base is the
  // start of the CTA's window: 1024-byte aligned, as the 128B-swizzled tiles need.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  uint8_t* gbase = smem_raw;
  CtaMiscB& misc = *reinterpret_cast<CtaMiscB*>(smem_raw + C::KV_OFF_MISC);
  uint32_t& s_tmem = misc.tmem;
  volatile uint32_t& s_abort = misc.abort;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kFlagSmemAlign);
    return;
  }
  if ((*p.status & kFlagBadSeqlens) != 0) return;  // the schedule listed no work
  const uint32_t sK = sbase + C::KV_OFF_K, sV = sbase + C::KV_OFF_V;
  const uint32_t sQ = sbase + C::KV_OFF_Q, sDO = sbase + C::KV_OFF_DO;
  const uint32_t sVEC = sbase + C::KV_OFF_VEC;
  // per stage: -LSE log2 e of the tile's queries at [st * 2BQ, +BQ), D at [+BQ, +2BQ)
  const float* vec = reinterpret_cast<const float*>(gbase + C::KV_OFF_VEC);
  const uint32_t bars = sbase + C::KV_OFF_BAR;
  const uint32_t bar_kv = bars;                      // K', V of an item loaded
  const uint32_t bar_kv_free = bars + 8;             // ... and no longer read
  const uint32_t bar_full = bars + 16;               // [NST]
  const uint32_t bar_empty = bar_full + 8 * C::NST;  // [NST]
  const uint32_t bar_st = bar_empty + 8 * C::NST;    // S^T in TMEM
  const uint32_t bar_p = bar_st + 8;                 // P^T in TMEM (256 arrivals)
  const uint32_t bar_dp = bar_p + 8;                 // dP^T in TMEM
  const uint32_t bar_ds = bar_dp + 8;                // dS^T in TMEM (256 arrivals)
  const uint32_t bar_done = bar_ds + 8;              // an item's dV, dK complete
  const uint32_t bar_acc_free = bar_done + 8;        // ... and loaded (256 arrivals)
  const uint32_t bar_drain = bar_acc_free + 8;
  const uint32_t bar_stall = bar_drain + 8;          // test hook: never arrived on
  // work-item ring: slot published by the producer / read by the MMA thread and the
  // 8 elementwise warps
  const uint32_t bar_ifull = bar_stall + 8;          // [4]
  const uint32_t bar_iempty = bar_ifull + 32;        // [4]
  volatile WorkItemB* ring = misc.ring;

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar_ifull + 8 * i, 1);
      mbar_init(bar_iempty + 8 * i, 9);
    }
    mbar_init(bar_kv, 1);
    mbar_init(bar_kv_free, 1);
    for (int i = 0; i < C::NST; ++i) {
      // 32 cp.async arrivals (LSE / D rows) + the TMA issuer's expect-tx arrival
      mbar_init(bar_full + 8 * i, 33);
      mbar_init(bar_empty + 8 * i, 1);
    }
    mbar_init(bar_st, 1);
    mbar_init(bar_p, 256);
    mbar_init(bar_dp, 1);
    mbar_init(bar_ds, 256);
    mbar_init(bar_done, 1);
    mbar_init(bar_acc_free, 256);
    mbar_init(bar_drain, 1);
    mbar_init(bar_stall, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 9) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 8) {
    // -------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
    }
    // Lane 0 claims the CTA's items from the ranked list with an atomic counter (a
    // CTA that finishes early takes more) and publishes each in ring slot k % 4 once
    // its readers are done with the item four before; item k + 1 is claimed while
    // item k's tiles stream.
    auto publish = [&](int32_t k, uint32_t idx) -> bool {
      const int32_t slot = k & 3;
      if (k >= 4 && !mbar_wait_bk(bar_iempty + 8 * slot, ((k >> 2) - 1) & 1, &s_abort))
        return false;
      WorkItemB wi{-1, 0, 0, 0, 0};
      const bool valid =
          idx <= static_cast<uint32_t>(INT32_MAX) &&
          find_item_b(p.cu, p.order, p.prefix, p.n, 128, static_cast<int32_t>(idx), wi);
      ring[slot].sample = valid ? wi.sample : -1;
      ring[slot].head = wi.head;
      ring[slot].blk = wi.blk;
      ring[slot].start = wi.start;
      ring[slot].len = wi.len;
      mbar_arrive(bar_ifull + 8 * slot);  // (release: the record is visible to its waiters)
      return true;
    };
    bool ok = true;
    if (lane == 0) ok = publish(0, atomicAdd(p.next_item, 1u));
    ok = __shfl_sync(0xffffffffu, ok, 0);
    int32_t gt = 0, items = 0;  // tiles issued (all items), items started
    for (int32_t k = 0; ok; ++k) {
      __syncwarp();  // lane 0's record for item k is in place
      const WorkItemB w{ring[k & 3].sample, ring[k & 3].head, ring[k & 3].blk, ring[k & 3].start,
                        ring[k & 3].len};
      if (w.sample < 0) break;  // no more items
      const int32_t k0 = w.blk * C::BK, nq = (w.len + C::BQ - 1) / C::BQ;
      if (k > 0 &&
          !__all_sync(0xffffffffu, mbar_wait_bk(bar_kv_free, (k - 1) & 1, &s_abort))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_kv, 2 * C::TILE);
        for (int ch = 0; ch < D / 64; ++ch) {
          tma_load_3d(sK + ch * C::CHUNK, &tm_k, bar_kv, ch * 64, w.head, w.start + k0);
          tma_load_3d(sV + ch * C::CHUNK, &tm_v, bar_kv, ch * 64, w.head, w.start + k0);
        }
      }
      ++items;
      const uint32_t idx_next = lane == 0 ? atomicAdd(p.next_item, 1u) : 0u;  // the next item
      const int64_t gbase_row = static_cast<int64_t>(w.head) * p.T + w.start;
      for (int32_t i = 0; i < nq; ++i, ++gt) {
        const int32_t st = gt % C::NST, use = gt / C::NST;
        if (use > 0 &&
            !__all_sync(0xffffffffu, mbar_wait_bk(bar_empty + 8 * st, (use - 1) & 1, &s_abort))) {
          ok = false;
          break;
        }
        const int32_t q0 = i * C::BQ;  // first query of the tile (in sample)
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_full + 8 * st, 2 * C::TILE);
          for (int ch = 0; ch < D / 64; ++ch) {
            tma_load_3d(sQ + st * C::TILE + ch * C::CHUNK, &tm_q, bar_full + 8 * st, ch * 64,
                        w.head, w.start + q0);
            tma_load_3d(sDO + st * C::TILE + ch * C::CHUNK, &tm_do, bar_full + 8 * st, ch * 64,
                        w.head, w.start + q0);
          }
        }
#pragma unroll
        for (int u = 0; u < C::BQ / 32; ++u) {
          const int q = u * 32 + static_cast<int>(lane);  // consecutive lanes, consecutive words
          const int32_t qi = q0 + q;
          const bool q_ok = qi < w.len;
          cp_async_4(sVEC + st * C::VEC + q * 4, q_ok ? p.nlse2 + gbase_row + qi : p.pad + q);
          cp_async_4(sVEC + st * C::VEC + C::BQ * 4 + q * 4,
                     q_ok ? p.delta + gbase_row + qi : p.pad + C::BQ + q);
        }
        cp_async_arrive_noinc(bar_full + 8 * st);
      }
      if (ok) {  // the next item, once this one's tiles are issued
        if (lane == 0) ok = publish(k + 1, idx_next);
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
    if (!ok) {
      s_abort = 1;
      if (lane == 0) atomicOr(p.status, kFlagTimeout);
    }
    // let every issued copy land before the CTA can exit
    if (lane == 0) {
      if (items > 0) mbar_wait_drain(bar_kv, (items - 1) & 1);
      for (int32_t c = (gt > C::NST ? gt - C::NST : 0); c < gt; ++c)
        mbar_wait_drain(bar_full + 8 * (c % C::NST), (c / C::NST) & 1);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        const bool r = mbar_wait(bar, parity, &s_abort);
        tc_fence_after();
        return r;
      };
      // descriptors: one base per operand buffer, advanced by constant offsets
      const uint64_t dK_k = sdesc_sw128(sK, 16, 1024), dV_k = sdesc_sw128(sV, 16, 1024);
      const uint64_t dQ_k0 = sdesc_sw128(sQ, 16, 1024), dQ_m0 = sdesc_sw128(sQ, C::CHUNK, 1024);
      const uint64_t dO_k0 = sdesc_sw128(sDO, 16, 1024), dO_m0 = sdesc_sw128(sDO, C::CHUNK, 1024);
      constexpr uint64_t kStage = C::TILE >> 4;
      auto full = [&](int32_t g) {
        return wait(bar_full + 8 * (g % C::NST), (g / C::NST) & 1);
      };
      auto issue_st = [&](int32_t g) {  // S^T = K' Q'_g^T -> ST
        const uint64_t q = dQ_k0 + (g % C::NST) * kStage;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::KV_ST, dK_k + kofs<D>(kk), q + kofs<D>(kk), C::IDESC_S, kk > 0);
        mma_commit(bar_st);
      };
      auto issue_dp = [&](int32_t g) {  // dP^T = V dO_g^T -> DPT
        const uint64_t o = dO_k0 + (g % C::NST) * kStage;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::KV_DPT, dV_k + kofs<D>(kk), o + kofs<D>(kk), C::IDESC_DP, kk > 0);
        mma_commit(bar_dp);
      };
      bool ok = p.stall_us == 0 ||
                mbar_wait_for(bar_stall, 0, &s_abort, static_cast<uint64_t>(p.stall_us) * 1000u);
      int32_t gt = 0;  // tiles of earlier items
      for (int32_t k = 0; ok; ++k) {
        if (!(ok = mbar_wait(bar_ifull + 8 * (k & 3), (k >> 2) & 1, &s_abort))) break;
        const int32_t sample = ring[k & 3].sample, len = ring[k & 3].len;
        mbar_arrive(bar_iempty + 8 * (k & 3));
        if (sample < 0) break;  // no more items
        const int32_t nq = (len + C::BQ - 1) / C::BQ;
        if (!(ok = wait(bar_kv, k & 1) && full(gt))) break;
        issue_st(gt);
        issue_dp(gt);
        for (int32_t i = 0; i < nq; ++i) {
          const int32_t g = gt + i, st = g % C::NST;
          const uint64_t q_m = dQ_m0 + st * kStage, o_m = dO_m0 + st * kStage;
          if (!(ok = wait(bar_p, g & 1))) break;  // P^T in ST (both halves)
          // the previous item's accumulators must have been loaded
          if (i == 0 && k > 0 && !(ok = wait(bar_acc_free, (k - 1) & 1))) break;
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)  // dV += P^T dO
            mma_ts(tmem + C::KV_DV, tmem + C::KV_ST + packed_col(kk), o_m + mofs(kk),
                   C::IDESC_DV, (i > 0 || kk > 0) ? 1u : 0u);
          if (i + 1 < nq) {  // ST is free once dV (issued above) has read P^T
            if (!(ok = full(g + 1))) break;
            issue_st(g + 1);
          } else {
            mma_commit(bar_kv_free);  // the item's last S^T and dP^T are issued
          }
          if (!(ok = wait(bar_ds, g & 1))) break;  // dS^T in DPT (both halves)
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)  // dK += dS^T Q'
            mma_ts(tmem + C::KV_DK, tmem + C::KV_DPT + packed_col(kk), q_m + mofs(kk),
                   C::IDESC_DKQ, (i > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar_empty + 8 * st);  // Q'_g, dO_g no longer read
          if (i + 1 < nq) issue_dp(g + 1);  // DPT is free once dK has read dS^T
        }
        if (!ok) break;
        mma_commit(bar_done);
        gt += nq;
      }
      if (!ok) {
        s_abort = 1;
        atomicOr(p.status, kFlagTimeout);
      }
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else if (warp < 8) {
    // ------------------------------------------ P / dS warpgroups (key rows), x 2
    const int h = warp >> 2;                 // query half: columns [64h, 64h + 64)
    const uint32_t row = threadIdx.x & 127;  // key row in the tile = TMEM lane
    const uint32_t lane_off = ((warp & 3) * 32) << 16;
    const uint32_t tST = tmem + lane_off + C::KV_ST + 64 * h;
    const uint32_t tDPT = tmem + lane_off + C::KV_DPT + 64 * h;
    const float sl2 = p.scale_log2;
    float dsmax = 0.f;  // scaled |dS|: flag values outside the fp16 range
    bool ok = true;
    int32_t gt = 0;
    for (int32_t k = 0; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_ifull + 8 * (k & 3), (k >> 2) & 1,
                                                      &s_abort))))
        break;
      const WorkItemB w{ring[k & 3].sample, ring[k & 3].head, ring[k & 3].blk, ring[k & 3].start,
                        ring[k & 3].len};
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_iempty + 8 * (k & 3));
      if (w.sample < 0) break;  // no more items
      const int32_t k0 = w.blk * C::BK, nq = (w.len + C::BQ - 1) / C::BQ;
      const bool key_ok = k0 + static_cast<int32_t>(row) < w.len;
      // dS is staged in fp16 as ds_mul * dS (a power of two; see ds_scale_for)
      const float ds_mul = ds_scale_for(p.hmax[w.head], p.hmax[p.heads + w.head]);
      const uint64_t dsm2 = f32x2_pack(ds_mul, ds_mul);
      // stored-dS form: this thread's key row in its 128-key tile; its 8-query unit
      // g sits at ds_row + g 1024 (consecutive rows adjacent)
      uint16_t* ds_row = nullptr;
      if (p.ds != nullptr)
        ds_row = p.ds + ((ds_tile_base(p.heads, w.start, w.sample, w.head, nq * C::BQ) + w.blk) *
                             (p.ds_cols / 8) * 128 + row) * 8;
      for (int32_t i = 0; i < nq; ++i) {
        const int32_t g = gt + i, st = g % C::NST;
        ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_full + 8 * st, (g / C::NST) & 1, &s_abort) &&
                                         mbar_wait_bk(bar_st, g & 1, &s_abort));
        if (!ok) break;
        tc_fence_after();
        const float4* vl4 = reinterpret_cast<const float4*>(vec + st * 2 * C::BQ + 64 * h);
        const float4* vd4 = reinterpret_cast<const float4*>(vec + st * 2 * C::BQ + C::BQ + 64 * h);
        // P^T: 64 queries, two per packed FMA; bf16 into ST columns [64h, 64h + 32)
        // (this half's S^T values already read).  Key rows past the sample get
        // P = 0 (their S^T holds another sample's keys).
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
            for (int hh = 0; hh < 2; ++hh) {
              const uint64_t x = f32x2_fma(f32x2_pack(__uint_as_float(r[4 * c4 + 2 * hh]),
                                                      __uint_as_float(r[4 * c4 + 2 * hh + 1])),
                                           sl2x2, hh ? f32x2_pack(l.z, l.w) : f32x2_pack(l.x, l.y));
              float x0, x1;
              f32x2_unpack(x, x0, x1);
              pr2[2 * c4 + hh] = key_ok ? f32x2_pack(ex2_approx(x0), ex2_approx(x1)) : 0ull;
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
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_p);
        ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_dp, g & 1, &s_abort));
        if (!ok) break;
        tc_fence_after();
        // dS^T = P^T (dP^T - D) ds_mul, two queries per packed op; fp16 into DPT
        // columns [64h, 64h + 32) (each 32-column load is complete before the
        // columns it overlaps are rewritten)
        uint32_t xs[2][16];  // stored-dS form: this row's dS^T values, both chunks
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
            for (int hh = 0; hh < 2; ++hh) {
              const uint64_t t2 = f32x2_sub(f32x2_pack(__uint_as_float(rd[u4 * 4 + 2 * hh]),
                                                       __uint_as_float(rd[u4 * 4 + 2 * hh + 1])),
                                            hh ? f32x2_pack(dd.z, dd.w) : f32x2_pack(dd.x, dd.y));
              const uint64_t ds2 = f32x2_mul(f32x2_mul(pr2[c * 16 + u4 * 2 + hh], dsm2), t2);
              float ds0, ds1;
              f32x2_unpack(ds2, ds0, ds1);
              dsmax = fmax3(dsmax, fabsf(ds0), fabsf(ds1));
              pd[u4 * 2 + hh] = pack_f16x2(ds0, ds1);
            }
          }
          tmem_st16(tDPT + c * 16, pd);
#pragma unroll
          for (int e = 0; e < 16; ++e) xs[c][e] = pd[e];
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_ds);
        if (ds_row != nullptr) {
          // After the release (the tensor core runs dK meanwhile): queries
          // [i BQ + 64h + 32c + 8u, +8) of the key row, as unit
          // g = 16 i + 8h + 4c + u.  The 32 lanes of a warp hold consecutive key
          // rows, so each store writes 512 contiguous bytes; streaming stores (read
          // once, much later) leave L2 to the Q' / dO tiles the CTAs re-read.
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int u = 0; u < 4; ++u)
              __stcs(reinterpret_cast<uint4*>(ds_row + (i * 16 + 8 * h + 4 * c + u) * 1024),
                     make_uint4(xs[c][4 * u], xs[c][4 * u + 1], xs[c][4 * u + 2], xs[c][4 * u + 3]));
        }
      }
      if (!ok) break;
      // epilogue: this warpgroup's columns [h D/2, (h + 1) D/2) of dV and dK into
      // registers, the accumulators released, then dV and R(-theta) scale dK /
      // ds_mul stored straight to the key row
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_done, k & 1, &s_abort)))) break;
      tc_fence_after();
      uint32_t rv[D / 64][32], rk[D / 64][32];
#pragma unroll
      for (int c2 = 0; c2 < D / 64; ++c2) {
        const int cc = h * (D / 64) + c2;  // 32-column chunk
        tmem_ld32(tmem + lane_off + C::KV_DV + cc * 32, rv[c2]);
        tmem_ld32(tmem + lane_off + C::KV_DK + cc * 32, rk[c2]);
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar_acc_free);
      if (key_ok) {
        float pv[3];
        token_pos(p, static_cast<int64_t>(w.start) + k0 + row, true, pv);
        const int64_t off = ((static_cast<int64_t>(w.start) + k0 + row) * p.heads + w.head) * D;
        const float dk_mul = p.scale / ds_mul;  // exact: ds_mul is a power of two
#pragma unroll
        for (int c2 = 0; c2 < D / 64; ++c2) {
          const int cc = h * (D / 64) + c2;
          store_row_chunk(p.dv + off, cc, rv[c2], 1.f, false, pv, p.f);
          store_row_chunk(p.dk + off, cc, rk[c2], dk_mul, p.pos != nullptr, pv, p.f);
        }
      }
      gt += nq;
    }
    if (!(dsmax <= 65504.f)) atomicOr(p.status, kFlagFp16Range);
    if (!ok) {
      s_abort = 1;
      atomicOr(p.status, kFlagTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------- dQ kernel
// Persistent like the dK / dV kernel: per (sample, head, query tile) item, Q' and
// dO are loaded once (as soon as the previous item's last S and dP have read
// theirs) and the dQ accumulator is freed for the next item as soon as the
// elementwise warps have loaded it.  Per global step g (key tile j of an item):
//   S_g  -> TMEM S (one buffer: the elementwise warps copy it to registers and
//           release it at once, so S_{g+1} follows as soon as they have)
//   dP_g -> TMEM DP[g % 2], issued two steps ahead
//   dS_g = P (dP - D) ds_mul, written over dP_g in DP[g % 2]
//   dQ  += dS_g K'_g (TS, dS from TMEM)
// MMA order per step: S_{g+1}, dQ_g, dP_{g+2}: the dS of step g+1 is computed
// while the tensor core runs step g's GEMMs.  K'_j goes through a 3-slot ring
// (read by S_j and dQ_j), V_j through a 2-slot ring (read by dP_j only).
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_q_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  CtaMiscB& misc = *reinterpret_cast<CtaMiscB*>(smem_raw + C::Q_OFF_MISC);
  uint32_t& s_tmem = misc.tmem;
  volatile uint32_t& s_abort = misc.abort;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kFlagSmemAlign);
    return;
  }
  if ((*p.status & kFlagBadSeqlens) != 0) return;  // the schedule listed no work
  const uint32_t sQ = sbase + C::Q_OFF_Q, sDO = sbase + C::Q_OFF_DO;
  const uint32_t sK = sbase + C::Q_OFF_K, sV = sbase + C::Q_OFF_V;
  const uint32_t bars = sbase + C::Q_OFF_BAR;
  const uint32_t bar_q = bars;                          // Q', dO of an item loaded
  const uint32_t bar_q_free = bars + 8;                 // ... and no longer read
  const uint32_t bar_kfull = bars + 16;                 // [KSLOT]
  const uint32_t bar_kempty = bar_kfull + 8 * C::KSLOT;  // [KSLOT]
  const uint32_t bar_vfull = bar_kempty + 8 * C::KSLOT;  // [VSLOT]
  const uint32_t bar_vempty = bar_vfull + 8 * C::VSLOT;  // [VSLOT]
  const uint32_t bar_s = bar_vempty + 8 * C::VSLOT;      // S in TMEM
  const uint32_t bar_s_free = bar_s + 8;                 // ... copied out (256 arrivals)
  const uint32_t bar_dp = bar_s_free + 8;                // [2] dP in DP[g % 2]
  const uint32_t bar_ds = bar_dp + 16;                   // [2] dS in DP[g % 2] (256 arrivals)
  const uint32_t bar_o = bar_ds + 16;                    // an item's dQ complete
  const uint32_t bar_acc_free = bar_o + 8;               // ... and loaded (256 arrivals)
  const uint32_t bar_drain = bar_acc_free + 8;
  const uint32_t bar_stall = bar_drain + 8;              // test hook: never arrived on
  // work-item ring: slot published by the producer / read by the MMA thread and the
  // 8 elementwise warps
  const uint32_t bar_ifull = bar_stall + 8;              // [4]
  const uint32_t bar_iempty = bar_ifull + 32;            // [4]
  volatile WorkItemB* ring = misc.ring;

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar_ifull + 8 * i, 1);
      mbar_init(bar_iempty + 8 * i, 9);
    }
    mbar_init(bar_q, 1);
    mbar_init(bar_q_free, 1);
    for (int i = 0; i < C::KSLOT; ++i) {
      mbar_init(bar_kfull + 8 * i, 1);
      mbar_init(bar_kempty + 8 * i, 1);
    }
    for (int i = 0; i < C::VSLOT; ++i) {
      mbar_init(bar_vfull + 8 * i, 1);
      mbar_init(bar_vempty + 8 * i, 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_s_free, 256);
    mbar_init(bar_dp, 1);
    mbar_init(bar_dp + 8, 1);
    mbar_init(bar_ds, 256);
    mbar_init(bar_ds + 8, 256);
    mbar_init(bar_o, 1);
    mbar_init(bar_acc_free, 256);
    mbar_init(bar_drain, 1);
    mbar_init(bar_stall, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 9) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 8) {
    // -------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      // The CTA's items are claimed from the ranked list with an atomic counter (a
      // CTA that finishes early takes more) and published in ring slot k % 4 once
      // their readers are done with the item four before; item k + 1 is claimed
      // while item k's tiles stream.
      uint32_t* const counter = p.next_item + 1;
      auto publish = [&](int32_t k, uint32_t idx, WorkItemB& wi, bool& valid) -> bool {
        const int32_t slot = k & 3;
        if (k >= 4 && !mbar_wait_bk(bar_iempty + 8 * slot, ((k >> 2) - 1) & 1, &s_abort))
          return false;
        wi = WorkItemB{-1, 0, 0, 0, 0};
        valid = idx <= static_cast<uint32_t>(INT32_MAX) &&
                find_item_b(p.cu, p.order, p.prefix, p.n, 128, static_cast<int32_t>(idx), wi);
        ring[slot].sample = valid ? wi.sample : -1;
        ring[slot].head = wi.head;
        ring[slot].blk = wi.blk;
        ring[slot].start = wi.start;
        ring[slot].len = wi.len;
        mbar_arrive(bar_ifull + 8 * slot);  // (release: the record is visible to its waiters)
        return true;
      };
      int32_t gs = 0, items = 0;  // steps (K', V copies) of earlier items, items started
      WorkItemB wn;
      bool more = false;
      bool ok = publish(0, atomicAdd(counter, 1u), wn, more);
      for (int32_t k = 0; ok && more; ++k) {
        const WorkItemB w = wn;
        const int32_t q0 = w.blk * C::BQ, nk = (w.len + C::BK - 1) / C::BK;
        if (k > 0 && !mbar_wait_bk(bar_q_free, (k - 1) & 1, &s_abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar_q, 2 * C::TILE);
        for (int ch = 0; ch < D / 64; ++ch) {
          tma_load_3d(sQ + ch * C::CHUNK, &tm_q, bar_q, ch * 64, w.head, w.start + q0);
          tma_load_3d(sDO + ch * C::CHUNK, &tm_do, bar_q, ch * 64, w.head, w.start + q0);
        }
        ++items;
        const uint32_t idx_next = atomicAdd(counter, 1u);  // read once the K', V loads are issued
        for (int32_t j = 0; j < nk; ++j) {
          const int32_t g = gs + j;
          const int32_t ks = g % C::KSLOT, ku = g / C::KSLOT;
          if (ku > 0 && !mbar_wait_bk(bar_kempty + 8 * ks, (ku - 1) & 1, &s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_kfull + 8 * ks, C::TILE);
          for (int ch = 0; ch < D / 64; ++ch)
            tma_load_3d(sK + ks * C::TILE + ch * C::CHUNK, &tm_k, bar_kfull + 8 * ks, ch * 64,
                        w.head, w.start + j * C::BK);
          const int32_t vs = g % C::VSLOT, vu = g / C::VSLOT;
          if (vu > 0 && !mbar_wait_bk(bar_vempty + 8 * vs, (vu - 1) & 1, &s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_vfull + 8 * vs, C::TILE);
          for (int ch = 0; ch < D / 64; ++ch)
            tma_load_3d(sV + vs * C::TILE + ch * C::CHUNK, &tm_v, bar_vfull + 8 * vs, ch * 64,
                        w.head, w.start + j * C::BK);
        }
        gs += nk;
        if (ok) ok = publish(k + 1, idx_next, wn, more);
      }
      if (!ok) {
        s_abort = 1;
        atomicOr(p.status, kFlagTimeout);
      }
      // every issued copy lands before the CTA exits: at most one per slot is in
      // flight (a slot is reloaded only after its previous copy was consumed)
      if (items > 0) mbar_wait_drain(bar_q, (items - 1) & 1);
      for (int32_t g = (gs > C::KSLOT ? gs - C::KSLOT : 0); g < gs; ++g)
        mbar_wait_drain(bar_kfull + 8 * (g % C::KSLOT), (g / C::KSLOT) & 1);
      for (int32_t g = (gs > C::VSLOT ? gs - C::VSLOT : 0); g < gs; ++g)
        mbar_wait_drain(bar_vfull + 8 * (g % C::VSLOT), (g / C::VSLOT) & 1);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        const bool r = mbar_wait(bar, parity, &s_abort);
        tc_fence_after();
        return r;
      };
      const uint64_t dQ_k = sdesc_sw128(sQ, 16, 1024), dO_k = sdesc_sw128(sDO, 16, 1024);
      const uint64_t k_k = sdesc_sw128(sK, 16, 1024);        // K' as K-major B (S)
      const uint64_t k_m = sdesc_sw128(sK, C::CHUNK, 1024);  // K' as MN-major B (dQ)
      const uint64_t v_k = sdesc_sw128(sV, 16, 1024);        // V as K-major B (dP)
      constexpr uint64_t kTile = C::TILE >> 4;
      auto issue_s = [&](int32_t g) {  // S_g = Q' K'_g^T -> S
        if (!wait(bar_kfull + 8 * (g % C::KSLOT), (g / C::KSLOT) & 1)) return false;
        const uint64_t b = k_k + (g % C::KSLOT) * kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::Q_S, dQ_k + kofs<D>(kk), b + kofs<D>(kk), C::IDESC_S, kk > 0);
        mma_commit(bar_s);
        return true;
      };
      auto issue_dp = [&](int32_t g) {  // dP_g = dO V_g^T -> DP[g % 2]; V_g then released
        if (!wait(bar_vfull + 8 * (g % C::VSLOT), (g / C::VSLOT) & 1)) return false;
        const uint64_t b = v_k + (g % C::VSLOT) * kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::Q_DP + (g & 1) * 128, dO_k + kofs<D>(kk), b + kofs<D>(kk),
                 C::IDESC_DP, kk > 0);
        mma_commit(bar_dp + 8 * (g & 1));
        mma_commit(bar_vempty + 8 * (g % C::VSLOT));
        return true;
      };
      bool ok = p.stall_us == 0 ||
                mbar_wait_for(bar_stall, 0, &s_abort, static_cast<uint64_t>(p.stall_us) * 1000u);
      int32_t gs = 0;  // steps of earlier items
      for (int32_t k = 0; ok; ++k) {
        if (!(ok = mbar_wait(bar_ifull + 8 * (k & 3), (k >> 2) & 1, &s_abort))) break;
        const int32_t sample = ring[k & 3].sample, len = ring[k & 3].len;
        mbar_arrive(bar_iempty + 8 * (k & 3));
        if (sample < 0) break;  // no more items
        const int32_t nk = (len + C::BK - 1) / C::BK;
        if (!(ok = wait(bar_q, k & 1))) break;
        // S is free once the elementwise warps have copied out the previous step's
        if (gs > 0 && !(ok = wait(bar_s_free, (gs - 1) & 1))) break;
        if (!(ok = issue_s(gs) && issue_dp(gs))) break;
        if (nk > 1 && !(ok = issue_dp(gs + 1))) break;
        for (int32_t j = 0; j < nk; ++j) {
          const int32_t g = gs + j;
          if (j == nk - 1) mma_commit(bar_q_free);  // the item's last S and dP are issued
          if (j + 1 < nk) {  // S_{g+1} once S_g is copied out
            if (!(ok = wait(bar_s_free, g & 1) && issue_s(g + 1))) break;
          }
          if (!(ok = wait(bar_ds + 8 * (g & 1), (g >> 1) & 1))) break;  // dS_g in DP[g % 2]
          // the previous item's accumulator must have been loaded
          if (j == 0 && k > 0 && !(ok = wait(bar_acc_free, (k - 1) & 1))) break;
          const uint64_t kb = k_m + (g % C::KSLOT) * kTile;
          const uint32_t da = tmem + C::Q_DP + (g & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk)  // dQ += dS K'_g
            mma_ts(tmem + C::Q_DQ, da + packed_col(kk), kb + mofs(kk), C::IDESC_DKQ,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar_kempty + 8 * (g % C::KSLOT));  // K'_g read by S_g and dQ
          // DP[g % 2] is free once dQ (issued above) has read dS_g
          if (j + 2 < nk && !(ok = issue_dp(g + 2))) break;
        }
        if (!ok) break;
        mma_commit(bar_o);
        gs += nk;
      }
      if (!ok) {
        s_abort = 1;
        atomicOr(p.status, kFlagTimeout);
      }
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else if (warp < 8) {
    // -------------------------------------- P / dS warpgroups (query rows), x 2
    const int h = warp >> 2;                 // key half: columns [64h, 64h + 64)
    const uint32_t row = threadIdx.x & 127;  // query row in the tile = TMEM lane
    const uint32_t lane_off = ((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::Q_S + 64 * h;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f32x2_pack(sl2, sl2);
    float dsmax = 0.f;
    bool ok = true;
    int32_t gs = 0;
    for (int32_t k = 0; ok; ++k) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_ifull + 8 * (k & 3), (k >> 2) & 1,
                                                      &s_abort))))
        break;
      const WorkItemB w{ring[k & 3].sample, ring[k & 3].head, ring[k & 3].blk, ring[k & 3].start,
                        ring[k & 3].len};
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_iempty + 8 * (k & 3));
      if (w.sample < 0) break;  // no more items
      const int32_t q0 = w.blk * C::BQ, nk = (w.len + C::BK - 1) / C::BK;
      const int32_t qrow = q0 + static_cast<int32_t>(row);
      const bool row_ok = qrow < w.len;
      const int64_t gidx = static_cast<int64_t>(w.head) * p.T + w.start + qrow;
      // rows past the sample: -inf makes P = 0 there
      const float nl2 = row_ok ? p.nlse2[gidx] : -INFINITY;
      const float drow = row_ok ? p.delta[gidx] : 0.f;
      const float ds_mul = ds_scale_for(p.hmax[w.head], p.hmax[p.heads + w.head]);
      const uint64_t nl2x2 = f32x2_pack(nl2, nl2);
      const uint64_t dsm2 = f32x2_pack(ds_mul, ds_mul), d2 = f32x2_pack(drow, drow);
      for (int32_t j = 0; j < nk; ++j) {
        const int32_t g = gs + j;
        const uint32_t tDP = tmem + lane_off + C::Q_DP + (g & 1) * 128 + 64 * h;
        ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_s, g & 1, &s_abort));
        if (!ok) break;
        tc_fence_after();
        // S to registers, released at once
        uint32_t r[64];
        {
          uint32_t r0[32], r1[32];
          tmem_ld32(tS, r0);
          tmem_ld32(tS + 32, r1);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            r[c] = r0[c];
            r[32 + c] = r1[c];
          }
        }
        tc_fence_before();
        mbar_arrive(bar_s_free);
        // P = exp2(S scale log2e - LSE log2e) over this half's 64 keys; keys past
        // the sample end get P = 0
        const int32_t nvalid = w.len - j * C::BK - 64 * h;
        uint64_t pr2[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const uint64_t x = f32x2_fma(
              f32x2_pack(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1])), sl2x2, nl2x2);
          float x0, x1;
          f32x2_unpack(x, x0, x1);
          pr2[u] = f32x2_pack(2 * u < nvalid ? ex2_approx(x0) : 0.f,
                              2 * u + 1 < nvalid ? ex2_approx(x1) : 0.f);
        }
        ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_dp + 8 * (g & 1), (g >> 1) & 1, &s_abort));
        if (!ok) break;
        tc_fence_after();
        // dS = P (dP - D) ds_mul, fp16 over dP in DP[g % 2] columns [64h, 64h + 32)
        // (each 32-column load is complete before the columns it overlaps are
        // rewritten)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t rd[32];
          tmem_ld32(tDP + c * 32, rd);
          tmem_wait_ld();
          uint32_t pd[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const uint64_t t2 = f32x2_sub(
                f32x2_pack(__uint_as_float(rd[2 * u]), __uint_as_float(rd[2 * u + 1])), d2);
            const uint64_t ds2 = f32x2_mul(f32x2_mul(pr2[c * 16 + u], dsm2), t2);
            float ds0, ds1;
            f32x2_unpack(ds2, ds0, ds1);
            dsmax = fmax3(dsmax, fabsf(ds0), fabsf(ds1));
            pd[u] = pack_f16x2(ds0, ds1);
          }
          tmem_st16(tDP + c * 16, pd);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_ds + 8 * (g & 1));
      }
      if (!ok) break;
      // epilogue: this warpgroup's columns [h D/2, (h + 1) D/2) of dQ into
      // registers, the accumulator released, then R(-theta) scale dQ' / ds_mul
      // stored straight to the query row
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_o, k & 1, &s_abort)))) break;
      tc_fence_after();
      uint32_t rq[D / 64][32];
#pragma unroll
      for (int c2 = 0; c2 < D / 64; ++c2)
        tmem_ld32(tmem + lane_off + C::Q_DQ + (h * (D / 64) + c2) * 32, rq[c2]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar_acc_free);
      if (row_ok) {
        float pv[3];
        token_pos(p, static_cast<int64_t>(w.start) + qrow, true, pv);
        const int64_t off = ((static_cast<int64_t>(w.start) + qrow) * p.heads + w.head) * D;
        const float dq_mul = p.scale / ds_mul;  // exact: ds_mul is a power of two
#pragma unroll
        for (int c2 = 0; c2 < D / 64; ++c2)
          store_row_chunk(p.dq + off, h * (D / 64) + c2, rq[c2], dq_mul, p.pos != nullptr, pv,
                          p.f);
      }
      gs += nk;
    }
    if (!(dsmax <= 65504.f)) atomicOr(p.status, kFlagFp16Range);
    if (!ok) {
      s_abort = 1;
      atomicOr(p.status, kFlagTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------- dQ from stored dS
// The stored-dS form's second kernel: dQ' = dS K' with the dK / dV kernel's scaled
// fp16 dS^T read back from memory instead of recomputing S and dP.  Persistent,
// one item per (sample, head, 128-query tile) as in attn_bwd_q_kernel.  Per key
// tile j the TMA warp copies the dS^T block [keys of j][queries of the item] --
// 32 contiguous KB, 16 units of 128 keys x 8 queries, which land as the
// unswizzled MN-major core-matrix layout (8 keys x 8 queries per 128 bytes) --
// and K'_j into one of DQ_NS stages; the MMA thread issues dQ += dS K'_j (both
// operands MN-major: dS^T rows are keys, K' rows are keys) into one of two TMEM
// accumulators, so that one item's epilogue overlaps the next item's GEMMs; the
// two elementwise warpgroups store R(-theta) scale dQ' / ds_mul in bf16.  Rows
// and columns of dS^T past the sample end hold zeros (P = 0 there), so the
// next sample's keys in a last tile add nothing.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_k, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  CtaMiscB& misc = *reinterpret_cast<CtaMiscB*>(smem_raw + C::DQ_OFF_MISC);
  uint32_t& s_tmem = misc.tmem;
  volatile uint32_t& s_abort = misc.abort;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kFlagSmemAlign);
    return;
  }
  if ((*p.status & kFlagBadSeqlens) != 0) return;  // the schedule listed no work
  const uint32_t bars = sbase + C::DQ_OFF_BAR;
  const uint32_t bar_full = bars;                        // [DQ_NS]
  const uint32_t bar_empty = bar_full + 8 * C::DQ_NS;    // [DQ_NS]
  const uint32_t bar_acc = bar_empty + 8 * C::DQ_NS;     // [2] an item's dQ complete
  const uint32_t bar_acc_free = bar_acc + 16;            // [2] ... loaded (256 arrivals)
  const uint32_t bar_drain = bar_acc_free + 16;
  const uint32_t bar_stall = bar_drain + 8;              // test hook: never arrived on
  static_assert(8 * (2 * C::DQ_NS + 6) <= 256, "barrier area");

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < C::DQ_NS; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, 1);
    }
    mbar_init(bar_acc, 1);
    mbar_init(bar_acc + 8, 1);
    mbar_init(bar_acc_free, 256);
    mbar_init(bar_acc_free + 8, 256);
    mbar_init(bar_drain, 1);
    mbar_init(bar_stall, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 9) {
    tmem_alloc(smem_u32(&s_tmem), 2 * D < 32 ? 32 : 2 * D);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 8) {
    // -------------------------------------------------------------- TMA producer
    // lane 0 paces the ring; lanes 0-15 each copy one 8-query unit of a dS^T block
    {
      if (lane == 0) tma_prefetch_desc(&tm_k);
      bool ok = true;
      int32_t gs = 0, issued = 0;  // steps of earlier items; stage fills issued
      WorkItemB w;
      for (int32_t k = 0; ok && cta_item(p, k, w); ++k) {
        const int32_t q0 = w.blk * C::BQ, nk = (w.len + C::BK - 1) / C::BK;
        const int64_t tile0 = ds_tile_base(p.heads, w.start, w.sample, w.head, nk * C::BK);
        for (int32_t j = 0; j < nk; ++j) {
          const int32_t g = gs + j, st = g % C::DQ_NS, use = g / C::DQ_NS;
          if (use > 0 &&
              !__all_sync(0xffffffffu,
                          mbar_wait_bk(bar_empty + 8 * st, (use - 1) & 1, &s_abort))) {
            ok = false;
            break;
          }
          const uint32_t sds = sbase + st * C::DQ_STAGE, sk = sds + C::DS_TILE;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar_full + 8 * st, C::DQ_STAGE);
            for (int ch = 0; ch < D / 64; ++ch)
              tma_load_3d(sk + ch * C::CHUNK, &tm_k, bar_full + 8 * st, ch * 64, w.head,
                          w.start + j * C::BK);
          }
          __syncwarp();  // the byte count is posted before any copy can complete
          if (lane < 2) {  // units q0 / 8 + 8 lane .. + 7 of key tile j: 16 contiguous KB
            const uint16_t* src =
                p.ds + ((tile0 + j) * (p.ds_cols / 8) + q0 / 8 + 8 * static_cast<int>(lane)) * 1024;
            bulk_load(sds + lane * 16384, src, 16384, bar_full + 8 * st);
          }
          issued = g + 1;
        }
        gs += nk;
      }
      if (!ok && lane == 0) {
        s_abort = 1;
        atomicOr(p.status, kFlagTimeout);
      }
      // every issued copy lands before the CTA exits (at most one per stage)
      if (lane == 0)
        for (int32_t g = (issued > C::DQ_NS ? issued - C::DQ_NS : 0); g < issued; ++g)
          mbar_wait_drain(bar_full + 8 * (g % C::DQ_NS), (g / C::DQ_NS) & 1);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        const bool r = mbar_wait(bar, parity, &s_abort);
        tc_fence_after();
        return r;
      };
      // dS: unswizzled MN-major, 8-key groups 128 bytes apart (leading offset),
      // 8-query core-matrix columns 2 KB apart (stride offset); a K-step of 16
      // keys advances 256 bytes
      const uint64_t a_m = sdesc_noswz(sbase, 128, 2048);
      const uint64_t b_m = sdesc_sw128(sbase + C::DS_TILE, C::CHUNK, 1024);  // K' (MN-major)
      constexpr uint64_t kStage = C::DQ_STAGE >> 4;
      bool ok = p.stall_us == 0 ||
                mbar_wait_for(bar_stall, 0, &s_abort, static_cast<uint64_t>(p.stall_us) * 1000u);
      int32_t gs = 0;
      WorkItemB w;
      for (int32_t k = 0; ok && cta_item(p, k, w); ++k) {
        const int32_t nk = (w.len + C::BK - 1) / C::BK, buf = k & 1;
        // the accumulator's previous item (k - 2) must have been loaded
        if (k >= 2 && !(ok = wait(bar_acc_free + 8 * buf, ((k >> 1) - 1) & 1))) break;
        for (int32_t j = 0; j < nk; ++j) {
          const int32_t g = gs + j, st = g % C::DQ_NS;
          if (!(ok = wait(bar_full + 8 * st, (g / C::DQ_NS) & 1))) break;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk)  // dQ += dS K'_j, keys kk*16 .. +16
            mma_ss(tmem + buf * D, a_m + st * kStage + ((kk * 256) >> 4),
                   b_m + st * kStage + mofs(kk), C::IDESC_DQS, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar_empty + 8 * st);
        }
        if (!ok) break;
        mma_commit(bar_acc + 8 * buf);
        gs += nk;
      }
      if (!ok) {
        s_abort = 1;
        atomicOr(p.status, kFlagTimeout);
      }
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else if (warp < 8) {
    // ------------------------------------------ epilogue warpgroups (query rows)
    const int h = warp >> 2;                 // columns [h D/2, (h + 1) D/2) of dQ
    const uint32_t row = threadIdx.x & 127;  // query row in the tile = TMEM lane
    const uint32_t lane_off = ((warp & 3) * 32) << 16;
    bool ok = true;
    WorkItemB w;
    for (int32_t k = 0; ok && cta_item(p, k, w); ++k) {
      const int32_t buf = k & 1;
      const int32_t qrow = w.blk * C::BQ + static_cast<int32_t>(row);
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_acc + 8 * buf, (k >> 1) & 1, &s_abort))))
        break;
      tc_fence_after();
      uint32_t rq[D / 64][32];
#pragma unroll
      for (int c2 = 0; c2 < D / 64; ++c2)
        tmem_ld32(tmem + lane_off + buf * D + (h * (D / 64) + c2) * 32, rq[c2]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar_acc_free + 8 * buf);
      if (qrow < w.len) {
        const float ds_mul = ds_scale_for(p.hmax[w.head], p.hmax[p.heads + w.head]);
        float pv[3];
        token_pos(p, static_cast<int64_t>(w.start) + qrow, true, pv);
        const int64_t off = ((static_cast<int64_t>(w.start) + qrow) * p.heads + w.head) * D;
        const float dq_mul = p.scale / ds_mul;  // exact: ds_mul is a power of two
#pragma unroll
        for (int c2 = 0; c2 < D / 64; ++c2)
          store_row_chunk(p.dq + off, h * (D / 64) + c2, rq[c2], dq_mul, p.pos != nullptr, pv,
                          p.f);
      }
    }
    if (!ok) {
      s_abort = 1;
      atomicOr(p.status, kFlagTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * D < 32 ? 32 : 2 * D);
  }
}

// Multiprocessor count of the current device (cached per device).
int device_sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int D>
static cudaError_t launch_bwd_d(const AttnBwdArgs& a, cudaStream_t s) {
  using C = BwdCfg<D>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kv_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::KV_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_q_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::Q_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::DQ_SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int64_t rows = static_cast<int64_t>(a.T) * a.heads;
  if (rows > 0) {
    const int64_t blocks = (rows + kPreRowsPerBlock - 1) / kPreRowsPerBlock;
    KernelTimer kt(MF_K_BWD_PRE, s);
    bwd_pre_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(a.o), reinterpret_cast<const uint4*>(a.d_o),
        reinterpret_cast<const uint4*>(a.v), a.lse, a.nlse2, a.delta, a.pad, a.hmax, rows, a.T,
        a.heads);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_thd(&tq, a.q, a.T, a.heads, D, 128, true) ||
      !make_tmap_thd(&tk, a.k, a.T, a.heads, D, 128, true) ||
      !make_tmap_thd(&tv, a.v, a.T, a.heads, D, 128) ||
      !make_tmap_thd(&tdo, a.d_o, a.T, a.heads, D, 128))
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
  p.dq = reinterpret_cast<__nv_bfloat16*>(a.dq);
  p.dk = reinterpret_cast<__nv_bfloat16*>(a.dk);
  p.dv = reinterpret_cast<__nv_bfloat16*>(a.dv);
  p.n = a.n;
  p.T = a.T;
  p.heads = a.heads;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.f = make_rope_freqs(D, a.naxes);
  p.hmax = a.hmax;
  p.stall_us = a.stall_us;
  p.ds = a.ds;
  p.ds_cols = a.ds_cols;
  p.next_item = a.status + 2;  // (the status block's words 2-3; see launch_schedule)
  // both kernels: one item per (sample, head, 128-row tile), longest samples
  // first; one persistent CTA per SM (at most one per item)
  const int64_t items = (static_cast<int64_t>(a.T + 127) / 128 + a.n) * a.heads;
  if (items > 0) {
    const unsigned grid = static_cast<unsigned>(items < device_sm_count() ? items : device_sm_count());
    {
      KernelTimer kt(MF_K_ATTN_BWD, s);
      attn_bwd_kv_kernel<D><<<grid, kBwdThreads, C::KV_SMEM, s>>>(tq, tk, tv, tdo, p);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.ds != nullptr) {
      KernelTimer kt(MF_K_ATTN_BWD_DQ, s);
      attn_bwd_dq_kernel<D><<<grid, kBwdThreads, C::DQ_SMEM, s>>>(tk, p);
    } else {
      KernelTimer kt(MF_K_ATTN_BWD_Q, s);
      attn_bwd_q_kernel<D><<<grid, kBwdThreads, C::Q_SMEM, s>>>(tq, tk, tv, tdo, p);
    }
    return cudaGetLastError();
  }
  return cudaSuccess;
}

cudaError_t launch_attn_bwd(const AttnBwdArgs& a, cudaStream_t s) {
  return a.head_dim == 128 ? launch_bwd_d<128>(a, s) : launch_bwd_d<64>(a, s);
}

}  // namespace mf
