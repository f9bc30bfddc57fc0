// Block-diagonal (per-sample) non-causal attention forward on tcgen05 / TMEM / TMA.
//
// Operation: Mage-Flow joint self-attention over each packed sample (paperlayer.ai
// summary 3.2.1 "Model Architecture and Native Packing"; rcap.io post, varlen
// attention over the packed stream).  For each sample i, head a, query row j:
//   O_j = sum_k softmax_k(scale <q'_j, k'_k>) v_k over the keys of sample i only,
//   LSE_j = ln sum_k exp(scale <q'_j, k'_k>).
//
// Design: a work item is one sample, one head and 256 query rows (two 128-row Q
// tiles).  Persistent CTAs, one per SM, claim items from the longest-first list
// through an atomic counter and keep TMEM and their barriers across items.  Three
// warpgroups, registers moved from the third to the first two:
//   warp 8      TMA producer: claims the items and publishes them to the other
//               roles in a four-slot ring; per item the Q tiles, then K_j, V_j
//               tiles through a ring of shared-memory slots (128B-swizzled,
//               64-column chunks) that runs on across items.  The next item's Q
//               tiles load once the current item's last S GEMMs are done.
//   warp 9      MMA issuer (one thread): S_t = Q'_t K'_j^T (SS, into TMEM), then
//               O_t += P_t V'_j with P_t read from TMEM (TS).  Q', K', V', P are
//               fp16 (11 significant bits), accumulation fp32.  The two Q tiles
//               ping-pong so the tensor core works on one while the other's
//               softmax runs; an item's first S GEMMs run during the previous
//               item's epilogue.
//   warps 10-11 idle (they complete the third warpgroup), except in the
//               rotate-on-load form (ROT): there they apply the 2D rotation to
//               the bf16 Q and K tiles in shared memory as soon as TMA has
//               landed them, and convert the V tiles to fp16, in place (see
//               rot_tile below), before the MMA issuer may read them.
//   warps 0-7   two softmax warpgroups, one per Q tile; thread = query row =
//               TMEM lane.  Online softmax in base 2: row max by a tree of
//               three-input maxima, packed two-lane FMAs and adds around the
//               exponentials, a lazy rescale
//               of O (only when the running max grows by more than 2^8), P
//               written back to TMEM as fp16 over the S columns.  Epilogue: O / l
//               in bf16 through a per-warp staging chunk, written out as 64-byte
//               row pieces; LSE.
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D, 256+2D).
// Tiles never cross a sample: K/V tiles start at the sample's first token, key
// columns past the sample end are masked to -inf, query rows past it not stored.
// Every wait is bounded; a CTA that gives up records kFlagTimeout, lets its
// in-flight copies and MMAs land, frees TMEM and exits.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace mf {

// ----------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (encode == nullptr) {
    cudaDriverEntryPointQueryResult qres;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qres) != cudaSuccess ||
        qres != cudaDriverEntryPointSuccess || fn == nullptr)
      return nullptr;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}

bool make_tmap_thd(CUtensorMap* map, const void* base, int64_t T, int64_t heads,
                   int64_t head_dim, int box_rows, bool f16) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (encode == nullptr) return false;
  const int64_t rows = T > 0 ? T : 1;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim * 2),
                           static_cast<cuuint64_t>(heads * head_dim * 2)};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      3, const_cast<void*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_thd_u8(CUtensorMap* map, const void* base, int64_t T, int64_t heads,
                      int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (encode == nullptr) return false;
  const int64_t rows = T > 0 ? T : 1;
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(heads * 128)};
  cuuint32_t box[3] = {128, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_f32_thd(CUtensorMap* map, const void* base, int64_t T, int64_t heads,
                       int64_t head_dim, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (encode == nullptr) return false;
  const int64_t rows = T > 0 ? T : 1;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim * 4),
                           static_cast<cuuint64_t>(heads * head_dim * 4)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(head_dim), 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------- scheduling
// One block.  Validates cu_seqlens (cu[0] = 0, non-decreasing, cu[n] = T, every
// L_i <= max_len), zeroes the status word, ranks samples longest first and writes
// prefix[r] = work items of ranks < r, where a sample holds ceil(L/blk) * heads
// items.  On a malformed cu_seqlens it records kFlagBadSeqlens and schedules no
// work at all.
constexpr int kRankLimit = 4096;  // larger n keeps pack order (no LPT ranking)

__global__ void __launch_bounds__(1024) schedule_kernel(const int32_t* __restrict__ cu,
                                                        int32_t n, int32_t T, int32_t max_len,
                                                        int32_t heads, int32_t blk,
                                                        uint32_t* __restrict__ status,
                                                        int32_t* __restrict__ order,
                                                        int32_t* __restrict__ prefix,
                                                        float* __restrict__ zero, int32_t nzero) {
  __shared__ int s_bad;
  __shared__ int64_t s_part[1024];
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int i = tid; i < nzero; i += nt) zero[i] = 0.f;
  // words 1-7 of the status block: the attention kernels' work-item counters
  if (tid >= 1 && tid < 8) status[tid] = 0u;
  if (tid == 0) s_bad = (cu[0] != 0 || cu[n] != T) ? 1 : 0;
  __syncthreads();
  for (int i = tid; i < n; i += nt) {
    const int32_t L = cu[i + 1] - cu[i];
    if (L < 0 || L > max_len) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    for (int i = tid; i <= n; i += nt) prefix[i] = 0;
    if (tid == 0) *status = kFlagBadSeqlens;
    return;
  }
  if (tid == 0) *status = 0u;
  if (n <= kRankLimit) {
    for (int i = tid; i < n; i += nt) {
      const int32_t Li = cu[i + 1] - cu[i];
      int rank = 0;
      for (int k = 0; k < n; ++k) {
        const int32_t Lk = cu[k + 1] - cu[k];
        rank += (Lk > Li) || (Lk == Li && k < i);
      }
      order[rank] = i;
    }
  } else {
    for (int i = tid; i < n; i += nt) order[i] = i;
  }
  __syncthreads();
  // chunked exclusive scan of items over ranks
  const int per = (n + nt - 1) / nt;
  const int b = tid * per, e = min(n, b + per);
  int64_t sum = 0;
  for (int r = b; r < e; ++r) {
    const int i = order[r];
    sum += static_cast<int64_t>((cu[i + 1] - cu[i] + blk - 1) / blk) * heads;
  }
  s_part[tid] = sum;
  __syncthreads();
  if (tid == 0) {
    int64_t acc = 0;
    for (int t = 0; t < nt; ++t) {
      const int64_t v = s_part[t];
      s_part[t] = acc;
      acc += v;
    }
    prefix[n] = static_cast<int32_t>(acc);
  }
  __syncthreads();
  int64_t acc = s_part[tid];
  for (int r = b; r < e; ++r) {
    prefix[r] = static_cast<int32_t>(acc);
    const int i = order[r];
    acc += static_cast<int64_t>((cu[i + 1] - cu[i] + blk - 1) / blk) * heads;
  }
}

cudaError_t launch_schedule(const int32_t* d_cu, int32_t n, int32_t T, int32_t max_len,
                            int32_t heads, int32_t blk, uint32_t* status, int32_t* order,
                            int32_t* prefix, float* zero, int32_t nzero, cudaStream_t s) {
  KernelTimer kt(MF_K_SCHEDULE, s);
  schedule_kernel<<<1, 1024, 0, s>>>(d_cu, n, T, max_len, heads, blk, status, order, prefix, zero,
                                     nzero);
  return cudaGetLastError();
}

// Resolve the work item of this CTA: rank r with prefix[r] <= idx < prefix[r+1].
struct WorkItem {
  int32_t sample, head, blk, start, len;
};
// Per-CTA scalars kept in the dynamic shared-memory region.
struct CtaMisc {
  uint32_t tmem;
  uint32_t abort;
  // each softmax warp's counters (item index, S steps and items of its Q tile so
  // far), read back from shared memory where used: kept out of the registers its
  // score row needs
  int32_t cnt[8][4];
  // forward: the work items the producer has claimed, ring slot k % 4 for the
  // CTA's k-th item (sample < 0: no more items)
  WorkItem ring[4];
};
__device__ __forceinline__ bool find_item(const int32_t* __restrict__ cu,
                                          const int32_t* __restrict__ order,
                                          const int32_t* __restrict__ prefix, int32_t n,
                                          int32_t blk_rows, int32_t idx, WorkItem& w) {
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

// ------------------------------------------------------------------ forward
// Three warpgroups: softmax (warps 0-3, 4-7) and producer / MMA / idle (8-11).
// Launched at 168 registers a thread (384 x 168 = 64,512); the third warpgroup
// drops to 88 and the softmax warpgroups rise to 208: 128 x 88 + 256 x 208 =
// 64,512, exactly the launch total.
constexpr int kFwdThreads = 384;
constexpr uint32_t kFwdRegsLow = 88, kFwdRegsHigh = 208;
static_assert(128 * kFwdRegsLow + 256 * kFwdRegsHigh <= kFwdThreads * 168,
              "forward register split exceeds the launch total");

// F8: the 8-bit variant (E4M3 operands and probabilities, head_dim 128); ROT: the
// rotate-on-load form (a larger barrier region and the staged positions).
template <int D, bool F8, bool ROT = false>
struct FwdCfg {
  static constexpr int BM = 128;                  // query rows per Q tile
  static constexpr int BN = 128;                  // keys per K/V tile
  static constexpr int EB = F8 ? 1 : 2;           // bytes per operand element
  static constexpr int KSTEP = F8 ? 32 : 16;      // K elements per MMA (32 bytes either way)
  static constexpr int CHUNK = 128 * 128;         // one 128-byte-wide column chunk of a 128-row tile
  static constexpr int TILE = BM * D * EB;        // bytes of one 128 x D operand tile
  static constexpr int NCH = TILE / CHUNK;        // TMA boxes per tile
  static constexpr int NSLOT = F8 ? 8 : (D == 128 ? 4 : 8);  // K/V ring slots
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = 2 * TILE;
  // bf16 O staging of the epilogue: 32 rows x 64 bytes per softmax warp (one
  // 32-column chunk of its rows at a time), apart from the Q buffers, which the
  // next item's Q tiles take as soon as this item's last S GEMMs are done
  static constexpr int OFF_STG = OFF_KV + NSLOT * TILE;
  static constexpr int STG = 8 * 32 * 64;
  static constexpr int OFF_BAR = OFF_STG + STG;
  static constexpr int OFF_MISC = OFF_BAR + 512;
  // rotate-on-load form: token positions staged per transform warp, int2 [2][192]
  // (its rows of Q tile 0, Q tile 1 and the current K tile)
  static constexpr int OFF_POS = OFF_MISC + 384;
  static constexpr int SMEM = OFF_POS + (ROT ? 2 * 192 * 8 : 0);
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL0 = 256, O_COL1 = 256 + D;
  // S = Q'K'^T and O += P V' (V' MN-major); operand format code 0 is fp16 under
  // kind::f16 and E4M3 under kind::f8f6f4
  static constexpr uint32_t IDESC_S = idesc_f32acc(128, 128, kF16, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_f32acc(128, D, kF16, 0, 1);
  // Online softmax in base 2: the running maximum m is raised only when a tile's
  // maximum exceeds it by more than TAU, so P = 2^(x - m) <= 2^TAU = 256, within
  // fp16 and within E4M3's largest finite value 448.
  static constexpr float TAU = 8.f;
  static_assert(!F8 || D == 128, "the 8-bit variant holds a 128-element row in one 128-byte chunk");
  static_assert(SMEM <= 232448, "dynamic shared memory over the 227 KB limit");
};

struct FwdParams {
  const int32_t* cu;
  const int32_t* order;
  const int32_t* prefix;
  uint32_t* status;
  __nv_bfloat16* o;
  float* lse;
  const float* qscale;    // 8-bit variant: [T][heads] Q row scales
  const uint32_t* amax2;  // 8-bit variant: [2][heads] squared K pair-norm / V maxima
  int32_t n, T, heads;
  float scale_log2;
  // test hook (0 = off): the MMA thread first waits, at most this many
  // microseconds, on a barrier that nothing arrives on, so the CTA takes its
  // time-out path (failure-detection tests; never set by the product calls)
  uint32_t stall_us;
  // rotate-on-load form only: (r, c) per token (null: no rotation), and the
  // (cos, sin) table of angle v * omega_P for v in [0, rtab_rows), [v][D/2]
  const int32_t* pos;
  const float4* rtab;
  int32_t rtab_rows;
  // work-item counter, zeroed by the schedule kernel: each CTA claims its next
  // item (an index into the ranked list) with an atomic add
  uint32_t* next_item;
};

// ------------------------------------------------------ rotation on load
// One bf16 tile of 128 token rows x D in shared memory, as TMA lands it (64-column
// chunks of 128 rows x 128 bytes, the 16-byte units of row r XOR-swizzled by
// r % 8), rewritten in place as the fp16 operand the 16-bit forward's pre-pass
// would have produced for those rows: with ROTATE, pair P = (2P, 2P + 1) of the
// row of token t turned by the angle pos[t][axis_P] * omega_P,
//   y0 = x0 cos - x1 sin,  y1 = x0 sin + x1 cos   (fp32: a product, then one FMA),
// the first D/4 pairs by the row coordinate r and the rest by the column c
// (paperlayer.ai summary 3.2.1, per-sample 2D rotary positions); without, the
// bf16 values converted.  Same fp32 operations and roundings as the pre-pass, so
// the operands, and hence O and LSE, are bit-identical to the two-pass forward's.
// Rows past the pack (zero-filled by TMA) are left unrotated.  vmax collects the
// largest |y| (fp16 range check); a position outside [0, rtab_rows) sets `bad`
// and is read as 0.
//
// The 64 threads of warps 10-11 share a tile.  Thread tid owns the 16-byte unit
// column tid % 8 of rows tid / 8 + 8 i (i < 16) in every chunk: 8 consecutive
// lanes cover one 128-byte row chunk (conflict-free), and since r % 8 is the same
// for all of a thread's rows, so is its logical unit, hence its 4 pairs.  A warp's
// rows are those with (r / 4) % 2 = its index; their positions come staged in
// shared memory (spos[m] for row (m % 4) + 8 (m / 4) + 4 warp, see pos_row), and
// rows are taken RB at a time with every load of the batch issued before any
// use (the loop is bound by load latency otherwise).
__device__ __forceinline__ int pos_row(int m, int wi) { return (m & 3) + 8 * (m >> 2) + 4 * wi; }

template <int D>
__device__ __forceinline__ void rot_tile_qk(uint8_t* tile, int64_t row0, int32_t T, bool has_pos,
                                            const int2* spos, const float4* __restrict__ rtab,
                                            int32_t rtab_rows, uint32_t tid, float& vmax,
                                            uint32_t& bad) {
  constexpr int NP = D / 2, NCH = D / 64;
  constexpr int RB = 2;  // rows per batch (register limit of the 88-register warps)
  const int up = tid & 7, rr = tid >> 3, ul = up ^ rr;
  uint8_t* base = tile + rr * 128 + up * 16;
#pragma unroll 1
  for (int ib = 0; ib < 16; ib += RB) {
    int2 pv[RB];
    bool rot[RB];
#pragma unroll
    for (int u = 0; u < RB; ++u) {
      const int64_t t = row0 + rr + 8 * (ib + u);
      rot[u] = has_pos && t < T;
      pv[u] = spos[(rr & 3) + 4 * (ib + u)];
    }
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      const int P0 = ch * 32 + ul * 4;  // first of the unit's 4 pairs
      const bool col = P0 >= NP / 2;    // pairs of the column coordinate
      uint4 x[RB];
      float4 ta[RB], tb[RB];
#pragma unroll
      for (int u = 0; u < RB; ++u)
        x[u] = *reinterpret_cast<const uint4*>(base + ch * (128 * 128) + (ib + u) * 1024);
#pragma unroll
      for (int u = 0; u < RB; ++u) {
        int32_t v = col ? pv[u].y : pv[u].x;
        if (v < 0 || v >= rtab_rows) {
          bad |= rot[u] ? 1u : 0u;
          v = 0;
        }
        const float4* e = rtab + ((static_cast<int64_t>(v) * NP + P0) >> 1);
        if (rot[u]) {
          ta[u] = __ldg(e);
          tb[u] = __ldg(e + 1);
        } else {
          ta[u] = make_float4(1.f, 0.f, 1.f, 0.f);
          tb[u] = ta[u];
        }
      }
#pragma unroll
      for (int u = 0; u < RB; ++u) {
        const uint32_t wv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
        const float cs[4] = {ta[u].x, ta[u].z, tb[u].x, tb[u].z};
        const float sn[4] = {ta[u].y, ta[u].w, tb[u].y, tb[u].w};
        uint32_t yv[4];
#pragma unroll
        for (int k2 = 0; k2 < 4; k2 += 2) {
          // two pairs per packed op: (a0, b0) the even elements, (a1, b1) the odd
          const uint64_t x0 = f32x2_pack(__uint_as_float(wv[k2] << 16),
                                         __uint_as_float(wv[k2 + 1] << 16));
          const uint64_t x1 = f32x2_pack(__uint_as_float(wv[k2] & 0xFFFF0000u),
                                         __uint_as_float(wv[k2 + 1] & 0xFFFF0000u));
          const uint64_t nx1 = f32x2_pack(__uint_as_float((wv[k2] & 0xFFFF0000u) ^ 0x80000000u),
                                          __uint_as_float((wv[k2 + 1] & 0xFFFF0000u) ^ 0x80000000u));
          const uint64_t c2 = f32x2_pack(cs[k2], cs[k2 + 1]), s2 = f32x2_pack(sn[k2], sn[k2 + 1]);
          const uint64_t y0 = f32x2_fma(x0, c2, f32x2_mul(nx1, s2));  // x0 c + (-x1) s
          const uint64_t y1 = f32x2_fma(x0, s2, f32x2_mul(x1, c2));   // x0 s + x1 c
          float y00, y01, y10, y11;
          f32x2_unpack(y0, y00, y01);
          f32x2_unpack(y1, y10, y11);
          vmax = fmax3(vmax, fabsf(y00), fabsf(y10));
          vmax = fmax3(vmax, fabsf(y01), fabsf(y11));
          yv[k2] = pack_f16x2(y00, y10);
          yv[k2 + 1] = pack_f16x2(y01, y11);
        }
        *reinterpret_cast<uint4*>(base + ch * (128 * 128) + (ib + u) * 1024) =
            make_uint4(yv[0], yv[1], yv[2], yv[3]);
      }
    }
  }
}

// The V tile: bf16 to fp16 in place (the pre-pass's V' = v), eight units per
// batch; same unit ownership as rot_tile_qk.
template <int D>
__device__ __forceinline__ void cvt_tile_v(uint8_t* tile, uint32_t tid, float& vmax) {
  constexpr int NCH = D / 64;
  uint8_t* base = tile + (tid >> 3) * 128 + (tid & 7) * 16;
#pragma unroll 1
  for (int b = 0; b < 16 * NCH; b += 8) {
    uint4 x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = b + u;  // chunk i / 16, row tid / 8 + 8 (i % 16)
      x[u] = *reinterpret_cast<const uint4*>(base + (i >> 4) * (128 * 128) + (i & 15) * 1024);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = b + u;
      const uint32_t wv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
      uint32_t yv[4];
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        const float a0 = __uint_as_float(wv[k2] << 16), a1 = __uint_as_float(wv[k2] & 0xFFFF0000u);
        vmax = fmax3(vmax, fabsf(a0), fabsf(a1));
        yv[k2] = pack_f16x2(a0, a1);
      }
      *reinterpret_cast<uint4*>(base + (i >> 4) * (128 * 128) + (i & 15) * 1024) =
          make_uint4(yv[0], yv[1], yv[2], yv[3]);
    }
  }
}

template <int D, bool F8, bool ROT>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D, F8, ROT>;
  // All shared memory is dynamic (no static __shared__), so its base is the
  // start of the CTA's window: 1024-byte aligned, as the 128B-swizzled tiles need.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  CtaMisc& misc = *reinterpret_cast<CtaMisc*>(smem_raw + C::OFF_MISC);
  static_assert(sizeof(CtaMisc) <= 384, "per-CTA scalars");
  uint32_t& s_tmem = misc.tmem;
  volatile uint32_t& s_abort = misc.abort;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kFlagSmemAlign);
    return;
  }
  if ((*p.status & kFlagBadSeqlens) != 0) return;  // the schedule listed no work
  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sKV = sbase + C::OFF_KV;
  const uint32_t bars = sbase + C::OFF_BAR;
  // barrier addresses (8 bytes each)
  const uint32_t bar_q = bars;                            // an item's Q tiles loaded
  const uint32_t bar_qfree = bars + 8;                    // ... and read by its last S GEMMs
  const uint32_t bar_full = bars + 16;                    // [NSLOT]
  const uint32_t bar_empty = bar_full + 8 * C::NSLOT;     // [NSLOT]
  const uint32_t bar_s = bar_empty + 8 * C::NSLOT;        // [2]
  const uint32_t bar_p = bar_s + 16;                      // [2]
  const uint32_t bar_o = bar_p + 16;                      // [2]
  const uint32_t bar_drain = bar_o + 16;
  const uint32_t bar_stall = bar_drain + 8;  // test hook: never arrived on
  // work-item ring: slot published by the producer / read by every role
  const uint32_t bar_ifull = bar_stall + 8;  // [4]
  const uint32_t bar_iempty = bar_ifull + 32;  // [4]
  // rotate-on-load form: Q tile t / ring slot rewritten in place and fenced
  const uint32_t bar_qr = bar_iempty + 32;   // [2]
  const uint32_t bar_rdy = bar_qr + 16;      // [NSLOT]
  static_assert(!ROT || !F8, "the rotate-on-load form is a 16-bit forward");
  static_assert(8 * (ROT ? 19 + 3 * C::NSLOT : 17 + 2 * C::NSLOT) <= C::OFF_MISC - C::OFF_BAR,
                "barrier region too small");
  // readers of each work item: the MMA thread, the 8 softmax warps, the 2 rotation warps
  constexpr uint32_t kTakers = ROT ? 11 : 9;

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(bar_q, 1);
    mbar_init(bar_qfree, 1);
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_s + 8, 1);
    mbar_init(bar_p, 128);
    mbar_init(bar_p + 8, 128);
    mbar_init(bar_o, 1);
    mbar_init(bar_o + 8, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_stall, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar_ifull + 8 * i, 1);
      mbar_init(bar_iempty + 8 * i, kTakers);
    }
    if (ROT) {
      mbar_init(bar_qr, 64);
      mbar_init(bar_qr + 8, 64);
      for (int i = 0; i < C::NSLOT; ++i) mbar_init(bar_rdy + 8 * i, 64);
    }
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

  // Persistent: each CTA claims work items from the ranked list (longest samples
  // first) with an atomic counter, so that a CTA that finishes early takes more.
  // The producer claims item k + 1 while item k's tiles stream and publishes it in
  // ring slot (k + 1) % 4; every other role reads its items from the ring.  Ring
  // position c counts the K and V tiles across items (K_j of an item whose first
  // tile is c0 at c0 + 2j, V_j at c0 + 2j + 1).
  volatile WorkItem* ring = misc.ring;

  if (warp >= 8) {
    warpgroup_reg_dealloc<kFwdRegsLow>();
    if (warp == 8) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        // publishes the CTA's k-th item, list index idx (claimed earlier), in ring slot
        // k % 4 once its last reader is done with the item four before; false on a
        // time-out
        auto publish = [&](int32_t k, uint32_t idx, WorkItem& w, bool& valid) -> bool {
          const int32_t slot = k & 3;
          if (k >= 4 && !mbar_wait_bk(bar_iempty + 8 * slot, ((k >> 2) - 1) & 1, &s_abort))
            return false;
          w = WorkItem{-1, 0, 0, 0, 0};
          valid = idx <= static_cast<uint32_t>(INT32_MAX) &&
                  find_item(p.cu, p.order, p.prefix, p.n, 2 * C::BM, static_cast<int32_t>(idx), w);
          ring[slot].sample = valid ? w.sample : -1;
          ring[slot].head = w.head;
          ring[slot].blk = w.blk;
          ring[slot].start = w.start;
          ring[slot].len = w.len;
          mbar_arrive(bar_ifull + 8 * slot);  // (release: the record is visible to its waiters)
          return true;
        };
        int32_t c = 0, items = 0;
        WorkItem wn;
        bool more = false;
        bool ok = publish(0, atomicAdd(p.next_item, 1u), wn, more);
        for (int32_t k = 0; ok && more; ++k) {
          const WorkItem w = wn;
          const int32_t q0 = w.blk * 2 * C::BM;
          const bool has1 = q0 + C::BM < w.len;
          const int32_t nkv = (w.len + C::BN - 1) / C::BN;
          // the Q buffers are free once the previous item's last S GEMMs are done
          if (k > 0 && !(ok = mbar_wait_bk(bar_qfree, (k - 1) & 1, &s_abort))) break;
          mbar_arrive_expect_tx(bar_q, (has1 ? 2 : 1) * C::TILE);
          for (int t = 0; t < (has1 ? 2 : 1); ++t)
            for (int ch = 0; ch < C::NCH; ++ch)
              tma_load_3d(sQ + t * C::TILE + ch * C::CHUNK, &tm_q, bar_q, ch * (128 / C::EB),
                          w.head, w.start + q0 + t * C::BM);
          ++items;
          // claim the next item now; the 16-bit forms read its index (and publish the
          // item) once this item's K / V loads are issued, so the atomic's latency is
          // hidden; the 8-bit form, whose steps are shorter, publishes it at once
          // (each measured the faster on the 50k pack)
          const uint32_t idx_next = atomicAdd(p.next_item, 1u);
          if constexpr (F8) {
            if (!(ok = publish(k + 1, idx_next, wn, more))) break;
          }
          for (int32_t j = 0; j < nkv && ok; ++j) {
            for (int kv = 0; kv < 2; ++kv, ++c) {
              const int32_t slot = c % C::NSLOT, use = c / C::NSLOT;
              if (use > 0 && !mbar_wait_bk(bar_empty + 8 * slot, (use - 1) & 1, &s_abort)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(bar_full + 8 * slot, C::TILE);
              for (int ch = 0; ch < C::NCH; ++ch)
                tma_load_3d(sKV + slot * C::TILE + ch * C::CHUNK, kv ? &tm_v : &tm_k,
                            bar_full + 8 * slot, ch * (128 / C::EB), w.head, w.start + j * C::BN);
            }
          }
          if (!F8 && ok) ok = publish(k + 1, idx_next, wn, more);
        }
        if (!ok) {
          s_abort = 1;
          atomicOr(p.status, kFlagTimeout);
        }
        // let every issued copy land before the CTA can exit
        if (items > 0) mbar_wait_drain(bar_q, (items - 1) & 1);
        for (int32_t i = (c > C::NSLOT ? c - C::NSLOT : 0); i < c; ++i)
          mbar_wait_drain(bar_full + 8 * (i % C::NSLOT), (i / C::NSLOT) & 1);
      }
    } else if (warp == 9) {
      // -------------------------------------------------------------- MMA issuer
      if (lane == 0) {
        bool ok = p.stall_us == 0 ||
                  mbar_wait_for(bar_stall, 0, &s_abort, static_cast<uint64_t>(p.stall_us) * 1000u);
        auto kv_wait = [&](int32_t c) -> bool {
          const bool r = mbar_wait((ROT ? bar_rdy : bar_full) + 8 * (c % C::NSLOT),
                                   (c / C::NSLOT) & 1, &s_abort);
          tc_fence_after();
          return r;
        };
        // Shared-memory descriptors: one base per buffer, then the start-address
        // field (16-byte units, low word) advanced by constant offsets.  The high
        // word (stride 1024 bytes, version, 128B swizzle) is the same for all three.
        const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
        const uint64_t dkv_k = sdesc_sw128(sKV, 16, 1024);          // K-major (K tiles)
        const uint64_t dkv_m = sdesc_sw128(sKV, C::CHUNK, 1024);    // MN-major (V tiles)
        const uint32_t hi = static_cast<uint32_t>(dq0 >> 32);
        const uint32_t q_lo = static_cast<uint32_t>(dq0), k_lo = static_cast<uint32_t>(dkv_k),
                       v_lo = static_cast<uint32_t>(dkv_m);
        constexpr uint32_t kTile = C::TILE >> 4;
        auto issue_s = [&](int t, int32_t c) {  // S_t = Q_t K^T, K at ring position c
          const uint32_t a0 = q_lo + t * kTile;
          const uint32_t b0 = k_lo + (c % C::NSLOT) * kTile;
          const uint32_t d = tmem + (t ? C::S_COL1 : C::S_COL0);
          // K step kk starts kk * 32 bytes into the 128-byte rows (next chunk every 4)
#pragma unroll
          for (int kk = 0; kk < D / C::KSTEP; ++kk) {
            const uint32_t o = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
            mma_ss_w<F8>(d, a0 + o, hi, b0 + o, hi, C::IDESC_S, kk > 0);
          }
          mma_commit(bar_s + 8 * t);
        };
        auto issue_pv = [&](int t, int32_t c, bool first) {  // O_t += P_t V, V at c
          const uint32_t b0 = v_lo + (c % C::NSLOT) * kTile;
          const uint32_t d = tmem + (t ? C::O_COL1 : C::O_COL0);
          const uint32_t a = tmem + (t ? C::S_COL1 : C::S_COL0);
          // P step kk: 32 bytes of each TMEM lane (8 columns); V rows kk * KSTEP on
#pragma unroll
          for (int kk = 0; kk < C::BN / C::KSTEP; ++kk)
            mma_ts_w<F8>(d, a + kk * 8, b0 + ((kk * C::KSTEP * 128) >> 4), hi, C::IDESC_PV,
                         (!first || kk > 0) ? 1u : 0u);
        };
        // parities: n0 / n1 S steps of Q tile 0 / 1 so far, i1 items with a tile 1
        int32_t c0 = 0, n0 = 0, n1 = 0, i1 = 0;
        for (int32_t k = 0; ok; ++k) {
          if (!(ok = mbar_wait(bar_ifull + 8 * (k & 3), (k >> 2) & 1, &s_abort))) break;
          const int32_t sample = ring[k & 3].sample, blk = ring[k & 3].blk, len = ring[k & 3].len;
          mbar_arrive(bar_iempty + 8 * (k & 3));
          if (sample < 0) break;  // no more items
          const int32_t q0 = blk * 2 * C::BM;
          const bool has1 = q0 + C::BM < len;
          const int32_t nkv = (len + C::BN - 1) / C::BN;
          ok = mbar_wait(ROT ? bar_qr : bar_q, k & 1, &s_abort);
          tc_fence_after();
          // The first S GEMM of this item overwrites S_0, and its first P V (no
          // accumulate) O_0, while the previous item may still be in its epilogue:
          // S_0 held that item's last P, already read by its last P V (issued
          // earlier, and MMAs run in order); O_0 is overwritten only after the
          // softmax warpgroup has arrived on bar_p for this item, which it does
          // after loading the previous item's O.
          if (ok) ok = kv_wait(c0);
          if (ok) {
            issue_s(0, c0);
            if (ROT && has1) {
              ok = mbar_wait(bar_qr + 8, i1 & 1, &s_abort);
              tc_fence_after();
            }
          }
          if (ok) {
            if (has1) issue_s(1, c0);
            if (nkv == 1) mma_commit(bar_qfree);
            mma_commit(bar_empty + 8 * (c0 % C::NSLOT));
          }
          for (int32_t j = 0; j < nkv && ok; ++j) {
            const int32_t ck = c0 + 2 * j;  // K_j; V_j at ck + 1
            ok = mbar_wait(bar_p, (n0 + j) & 1, &s_abort) && kv_wait(ck + 1);
            if (!ok) break;
            issue_pv(0, ck + 1, j == 0);
            const bool more = j + 1 < nkv;
            if (more) {
              if (!(ok = kv_wait(ck + 2))) break;
              issue_s(0, ck + 2);
            } else {
              // O_0 is final once this P V is done: tile 0's epilogue need not wait
              // for tile 1's last softmax and P V
              mma_commit(bar_o);
            }
            if (has1) {
              if (!(ok = mbar_wait(bar_p + 8, (n1 + j) & 1, &s_abort))) break;
              tc_fence_after();
              issue_pv(1, ck + 1, j == 0);
            }
            mma_commit(bar_empty + 8 * ((ck + 1) % C::NSLOT));
            if (more) {
              if (has1) issue_s(1, ck + 2);
              if (j + 2 == nkv) mma_commit(bar_qfree);  // the item's last S GEMMs
              mma_commit(bar_empty + 8 * ((ck + 2) % C::NSLOT));
            }
          }
          if (!ok) break;
          if (has1) mma_commit(bar_o + 8);
          c0 += 2 * nkv;
          n0 += nkv;
          if (has1) {
            n1 += nkv;
            ++i1;
          }
        }
        if (!ok) {
          s_abort = 1;
          atomicOr(p.status, kFlagTimeout);
        }
        // every MMA issued so far must finish before TMEM is released
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0);
      }
    } else if (ROT) {
      // ------------------------------------------- rotation on load (warps 10-11)
      // Tiles in the order the MMA issuer consumes them: Q_0, K_0, Q_1, V_0, K_1,
      // V_1, ...; each one rewritten in place, fenced for the tensor core's
      // (async-proxy) reads and released on its own barrier.
      const uint32_t tid = threadIdx.x - 320;
      float vmax = 0.f;
      uint32_t bad = 0;
      const int2* pos2 = reinterpret_cast<const int2*>(p.pos);
      const bool has_pos = pos2 != nullptr;
      const int wi = static_cast<int>(warp) - 10;
      int2* sp = reinterpret_cast<int2*>(smem_raw + C::OFF_POS) + 192 * wi;  // Q0, Q1, K
      // this lane's two rows (m = lane, lane + 32) of the warp's share of a tile
      auto pos_ld = [&](int64_t row0, int m) -> int2 {
        const int64_t t = row0 + pos_row(m, wi);
        return has_pos && t < p.T ? pos2[t] : make_int2(0, 0);
      };
      auto release = [&](uint32_t bar) {
        fence_proxy_async_smem();
        mbar_arrive(bar);
      };
      bool ok = true;
      int32_t c0 = 0;
      for (int32_t k = 0; ok; ++k) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_ifull + 8 * (k & 3), (k >> 2) & 1,
                                                        &s_abort))))
          break;
        const WorkItem w{ring[k & 3].sample, ring[k & 3].head, ring[k & 3].blk, ring[k & 3].start,
                         ring[k & 3].len};
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_iempty + 8 * (k & 3));
        if (w.sample < 0) break;  // no more items
        const int32_t q0 = w.blk * 2 * C::BM;
        const bool has1 = q0 + C::BM < w.len;
        const int32_t nkv = (w.len + C::BN - 1) / C::BN;
        const int64_t qrow0 = static_cast<int64_t>(w.start) + q0;
        // (the previous item's positions are no longer read: its tiles are done)
        __syncwarp();
        sp[lane] = pos_ld(qrow0, lane);
        sp[lane + 32] = pos_ld(qrow0, lane + 32);
        sp[64 + lane] = pos_ld(qrow0 + C::BM, lane);
        sp[96 + lane] = pos_ld(qrow0 + C::BM, lane + 32);
        int2 ka = pos_ld(w.start, lane), kb = pos_ld(w.start, lane + 32);  // next K tile's
        __syncwarp();
        ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_q, k & 1, &s_abort));
        if (!ok) break;
        rot_tile_qk<D>(smem_raw + C::OFF_Q, qrow0, p.T, has_pos, sp, p.rtab, p.rtab_rows, tid,
                       vmax, bad);
        release(bar_qr);
        for (int32_t cc = 0; ok && cc < 2 * nkv; ++cc) {
          const int32_t c = c0 + cc, slot = c % C::NSLOT;
          ok = __all_sync(0xffffffffu,
                          mbar_wait_bk(bar_full + 8 * slot, (c / C::NSLOT) & 1, &s_abort));
          if (!ok) break;
          uint8_t* tile = smem_raw + C::OFF_KV + slot * C::TILE;
          const int64_t krow0 = static_cast<int64_t>(w.start) + (cc >> 1) * C::BN;
          if (cc & 1) {
            cvt_tile_v<D>(tile, tid, vmax);
          } else {
            // stage this K tile's positions, then prefetch the next tile's
            __syncwarp();
            sp[128 + lane] = ka;
            sp[160 + lane] = kb;
            __syncwarp();
            if ((cc >> 1) + 1 < nkv) {
              ka = pos_ld(krow0 + C::BN, lane);
              kb = pos_ld(krow0 + C::BN, lane + 32);
            }
            rot_tile_qk<D>(tile, krow0, p.T, has_pos, sp + 128, p.rtab, p.rtab_rows, tid, vmax,
                           bad);
          }
          release(bar_rdy + 8 * slot);
          if (cc == 0 && has1) {
            rot_tile_qk<D>(smem_raw + C::OFF_Q + C::TILE, qrow0 + C::BM, p.T, has_pos, sp + 64,
                           p.rtab, p.rtab_rows, tid, vmax, bad);
            release(bar_qr + 8);
          }
        }
        c0 += 2 * nkv;
      }
      if (!ok) {
        s_abort = 1;
        atomicOr(p.status, kFlagTimeout);
      }
      if (!(vmax <= 65504.f)) atomicOr(p.status, kFlagFp16Range);
      if (bad) atomicOr(p.status, kFlagPosRange);
    }
  } else {
    warpgroup_reg_alloc<kFwdRegsHigh>();
    // ---------------------------------------------------- softmax warpgroups
    const int t = warp >> 2;  // Q tile of this warpgroup
    const uint32_t row = threadIdx.x & 127;
    const uint32_t lane_off = ((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + (t ? C::S_COL1 : C::S_COL0);
    // this warp's O staging: 32 rows x 64 bytes (one 32-column chunk at a time)
    uint8_t* so = smem_raw + C::OFF_STG + warp * (32 * 64);
    bool ok = true;
    // the CTA's item index k; S steps, items of this Q tile so far (parities)
    volatile int32_t* cnt = misc.cnt[warp];
    if (lane == 0) {
      cnt[0] = 0;
      cnt[1] = 0;
      cnt[2] = 0;
    }
    __syncwarp();
    // the current item is read from its ring slot, released once the epilogue is done
    auto release_item = [&]() {
      __syncwarp();  // every lane done with the item's fields
      if (lane == 0) {
        const int32_t k = cnt[0];
        mbar_arrive(bar_iempty + 8 * (k & 3));
        cnt[0] = k + 1;
      }
      __syncwarp();
    };
    while (ok) {
      const int32_t k = cnt[0];
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_ifull + 8 * (k & 3), (k >> 2) & 1,
                                                      &s_abort))))
        break;
      volatile WorkItem& w = ring[k & 3];
      if (w.sample < 0) break;  // no more items
      const int32_t q0 = w.blk * 2 * C::BM;
      const bool has1 = q0 + C::BM < w.len;
      if (t == 1 && !has1) {
        release_item();
        continue;
      }
      const int32_t nkv = (w.len + C::BN - 1) / C::BN;
      // logit scale in base 2; the 8-bit variant folds in the row's Q scale and the
      // head's K scale (kept positive, so that masked -inf columns stay -inf)
      float sl2 = p.scale_log2;
      if constexpr (F8) {
        const float sk = e4m3_scale(sqrtf(__uint_as_float(p.amax2[w.head]))).s;
        const float sq =
            q0 + t * C::BM + static_cast<int32_t>(row) < w.len
                ? p.qscale[(static_cast<int64_t>(w.start) + q0 + t * C::BM + row) * p.heads + w.head]
                : 0.f;
        sl2 = fmaxf(sl2 * sq * sk, 1e-30f);
      }
      float m = -INFINITY, l = 0.f;
      const int32_t par0 = cnt[1], len = w.len;
      for (int32_t j = 0; j < nkv; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_s + 8 * t, (par0 + j) & 1, &s_abort));
        if (!ok) break;
        tc_fence_after();
        uint32_t s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tS + c * 32, r);
#pragma unroll
          for (int u = 0; u < 32; ++u) s[c * 32 + u] = r[u];
        }
        tmem_wait_ld();
        const int32_t nvalid = len - j * C::BN;
        if (nvalid < C::BN) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= nvalid) s[c] = __float_as_uint(-INFINITY);
        }
        // row max: a tree of three-input maxima (depth 4 instead of a 127-long chain)
        float mx;
        {
          float m0[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t* v = s + 8 * i;
            m0[i] = fmax3(fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2])),
                          fmax3(__uint_as_float(v[3]), __uint_as_float(v[4]), __uint_as_float(v[5])),
                          fmaxf(__uint_as_float(v[6]), __uint_as_float(v[7])));
          }
          mx = fmax3(fmax3(fmax3(m0[0], m0[1], m0[2]), fmax3(m0[3], m0[4], m0[5]),
                           fmax3(m0[6], m0[7], m0[8])),
                     fmax3(m0[9], m0[10], m0[11]), fmax3(m0[12], m0[13], fmaxf(m0[14], m0[15])));
        }
        const float m_new = fmaxf(m, mx * sl2);
        if (j == 0) {
          m = m_new;
        } else {
          const bool need = m_new > m + C::TAU;
          if (__any_sync(0xffffffffu, need)) {
            const float f = need ? ex2_approx(m - m_new) : 1.f;
            if (need) {
              l *= f;
              m = m_new;
            }
            // (16 columns at a time: the score row is live here)
            const uint32_t tO = tmem + lane_off + (t ? C::O_COL1 : C::O_COL0);
#pragma unroll
            for (int cc = 0; cc < D / 16; ++cc) {
              uint32_t r[16];
              tmem_ld16(tO + cc * 16, r);
              tmem_wait_ld();
#pragma unroll
              for (int u = 0; u < 16; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * f);
              tmem_st16(tO + cc * 16, r);
            }
            tmem_wait_st();
          }
        }
        // P = 2^(s scale log2e - m), two columns per packed FMA; two packed sums
        const uint64_t sl2x2 = f32x2_pack(sl2, sl2), negm2 = f32x2_pack(-m, -m);
        uint64_t sum2[2] = {f32x2_pack(0.f, 0.f), f32x2_pack(0.f, 0.f)};
        if constexpr (F8) {
          // E4M3 P: four columns per 32-bit TMEM column, 32 columns in all
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
            uint32_t pk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int c0 = hh * 32 + 4 * u;
              const uint64_t xa = f32x2_fma(
                  f32x2_pack(__uint_as_float(s[c0]), __uint_as_float(s[c0 + 1])), sl2x2, negm2);
              const uint64_t xb = f32x2_fma(
                  f32x2_pack(__uint_as_float(s[c0 + 2]), __uint_as_float(s[c0 + 3])), sl2x2, negm2);
              float x0, x1, x2, x3;
              f32x2_unpack(xa, x0, x1);
              f32x2_unpack(xb, x2, x3);
              const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
              sum2[0] = f32x2_add(sum2[0], f32x2_pack(p0, p1));
              sum2[1] = f32x2_add(sum2[1], f32x2_pack(p2, p3));
              pk[u] = pack_e4m3x4(p0, p1, p2, p3);
            }
            tmem_st8(tS + hh * 8, pk);
          }
        } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const uint64_t x = f32x2_fma(f32x2_pack(__uint_as_float(s[c * 32 + 2 * u]),
                                                    __uint_as_float(s[c * 32 + 2 * u + 1])),
                                         sl2x2, negm2);
            float x0, x1;
            f32x2_unpack(x, x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            sum2[u & 1] = f32x2_add(sum2[u & 1], f32x2_pack(p0, p1));
            pk[u] = pack_f16x2(p0, p1);
          }
          tmem_st16(tS + c * 16, pk);
        }
        }
        float sa, sb, sc, sd;
        f32x2_unpack(sum2[0], sa, sb);
        f32x2_unpack(sum2[1], sc, sd);
        const float sum = (sa + sb) + (sc + sd);
        l += sum;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_p + 8 * t);
      }
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bk(bar_o + 8 * t, cnt[2] & 1, &s_abort));
      // the warpgroup's four warps agree before they leave the item
      if (t ? named_bar_or(2, 128, !ok) : named_bar_or(1, 128, !ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Epilogue: O / l in bf16, one 32-column chunk at a time through the warp's
      // staging (16-byte units of row r XOR-swizzled by (r / 2) % 4: conflict-free
      // both ways), then out as 64-byte row pieces, 8 rows a store.  O is loaded
      // from TMEM before this warpgroup's next arrival on bar_p, which is what
      // lets the next item's first P V overwrite it.
      {
        // the 8-bit variant's head V scale
        const float sv = F8 ? e4m3_scale(sqrtf(__uint_as_float(p.amax2[p.heads + w.head]))).s : 1.f;
        const float inv = sv / l;
        const int32_t tile0 = w.blk * 2 * C::BM + t * C::BM;  // first row of the Q tile (in sample)
        const int32_t wrow0 = tile0 + static_cast<int32_t>(warp & 3) * 32;
        const uint32_t tO = tmem + lane_off + (t ? C::O_COL1 : C::O_COL0);
        const int rr0 = static_cast<int>(lane >> 2), un = static_cast<int>(lane & 3);
        // the row's whole O in one round of TMEM loads (the score row is dead here)
        uint32_t r[D];
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc)
          tmem_ld32(tO + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(r + cc * 32));
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t* v = r + cc * 32 + 8 * u;
            const uint4 val = make_uint4(
                pack_bf16x2(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                pack_bf16x2(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                pack_bf16x2(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                pack_bf16x2(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
            *reinterpret_cast<uint4*>(so + lane * 64 + ((u ^ ((lane >> 1) & 3)) << 4)) = val;
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rr = rr0 + 8 * i;
            const uint4 val =
                *reinterpret_cast<const uint4*>(so + rr * 64 + ((un ^ ((rr >> 1) & 3)) << 4));
            if (wrow0 + rr < w.len) {
              const int64_t g =
                  ((static_cast<int64_t>(w.start) + wrow0 + rr) * p.heads + w.head) * D + cc * 32 +
                  un * 8;
              *reinterpret_cast<uint4*>(p.o + g) = val;
            }
          }
          __syncwarp();
        }
        if (tile0 + static_cast<int32_t>(row) < w.len)
          p.lse[static_cast<int64_t>(w.head) * p.T + w.start + tile0 + row] =
              (m + log2f(l)) * 0.69314718055994530942f;
      }
      __syncwarp();
      if (lane == 0) {
        cnt[1] = cnt[1] + nkv;
        cnt[2] = cnt[2] + 1;
      }
      release_item();
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
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool F8, bool ROT>
static cudaError_t launch_fwd_d(const AttnFwdArgs& a, cudaStream_t s) {
  using C = FwdCfg<D, F8, ROT>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, F8, ROT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  CUtensorMap tq, tk, tv;
  if (F8) {
    if (!make_tmap_thd_u8(&tq, a.q, a.T, a.heads, 128) ||
        !make_tmap_thd_u8(&tk, a.k, a.T, a.heads, 128) ||
        !make_tmap_thd_u8(&tv, a.v, a.T, a.heads, 128))
      return cudaErrorInvalidValue;
  } else if (!make_tmap_thd(&tq, a.q, a.T, a.heads, D, 128, !ROT) ||
             !make_tmap_thd(&tk, a.k, a.T, a.heads, D, 128, !ROT) ||
             !make_tmap_thd(&tv, a.v, a.T, a.heads, D, 128, !ROT)) {
    return cudaErrorInvalidValue;  // the rotate-on-load form maps the caller's bf16
  }
  FwdParams p;
  p.cu = a.cu;
  p.order = a.order;
  p.prefix = a.prefix;
  p.status = a.status;
  p.o = reinterpret_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.qscale = a.qscale;
  p.amax2 = a.amax2;
  p.n = a.n;
  p.T = a.T;
  p.heads = a.heads;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.stall_us = a.stall_us;
  p.pos = a.pos;
  p.rtab = reinterpret_cast<const float4*>(a.rtab);
  p.rtab_rows = a.rtab_rows;
  p.next_item = a.status + 1;  // (the status block's second word; see launch_schedule)
  // an upper bound on the items (256-row query blocks of every (sample, head));
  // persistent grid: one CTA per SM at most
  const int64_t items = (static_cast<int64_t>(a.T + 2 * C::BM - 1) / (2 * C::BM) + a.n) * a.heads;
  if (items <= 0) return cudaSuccess;
  const int64_t blocks = items < device_sm_count() ? items : device_sm_count();
  {
    KernelTimer kt(F8 ? MF_K_ATTN_FWD_F8 : ROT ? MF_K_ATTN_FWD_ROT : MF_K_ATTN_FWD, s);
    attn_fwd_kernel<D, F8, ROT>
        <<<static_cast<unsigned>(blocks), kFwdThreads, C::SMEM, s>>>(tq, tk, tv, p);
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const AttnFwdArgs& a, cudaStream_t s) {
  if (a.f8) return a.head_dim == 128 ? launch_fwd_d<128, true, false>(a, s) : cudaErrorInvalidValue;
  if (a.rot)
    return a.head_dim == 128 ? launch_fwd_d<128, false, true>(a, s)
                             : launch_fwd_d<64, false, true>(a, s);
  return a.head_dim == 128 ? launch_fwd_d<128, false, false>(a, s)
                           : launch_fwd_d<64, false, false>(a, s);
}

// (cos, sin) of v * omega_P for v in [0, rows), P in [0, head_dim / 2): the table
// the rotate-on-load forward reads, computed with the pre-pass's own angle
// evaluation (rope_sincos of float(v)), so both forms turn a pair identically.
template <int D>
__global__ void __launch_bounds__(256) rope_table_kernel(const __grid_constant__ RopeFreqs f,
                                                         int32_t rows, float2* __restrict__ tab) {
  constexpr int NP = D / 2;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(rows) * NP) return;
  const int P = static_cast<int>(i % NP);
  float sn, cs;
  rope_sincos(static_cast<float>(i / NP), f.omega[P], f.omega_lo[P], 1.0f, &sn, &cs);
  tab[i] = make_float2(cs, sn);
}

cudaError_t launch_rope_table(int32_t head_dim, int32_t rows, float* tab, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const RopeFreqs f = make_rope_freqs(head_dim, 2);
  const int64_t n = static_cast<int64_t>(rows) * (head_dim / 2);
  const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
  KernelTimer kt(MF_K_ROPE_TABLE, s);
  if (head_dim == 128)
    rope_table_kernel<128><<<blocks, 256, 0, s>>>(f, rows, reinterpret_cast<float2*>(tab));
  else
    rope_table_kernel<64><<<blocks, 256, 0, s>>>(f, rows, reinterpret_cast<float2*>(tab));
  return cudaGetLastError();
}

}  // namespace mf
