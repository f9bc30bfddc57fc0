// mf_varlen_attn_fwd_noalloc: the attention forward for callers that cannot
// allocate device memory.  Some callers are handed only their inputs and outputs
// and may not call cudaMalloc themselves: a plugin inside a framework that owns
// the device allocator, or a latency-critical loop where cudaMalloc/cudaFree
// (which can synchronise the device) are not allowed.  This entry point needs no
// workspace from them: its scratch is one file-scope device array of fixed size,
// which every GPU that loads this library holds until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/mf.h"
#include "common.cuh"

namespace mf {
namespace {

constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The forward's workspace for the largest accepted problem (see ws_layout):
// status word, the work list of up to MF_NOALLOC_MAX_SAMPLES samples, and three
// fp16 [T][heads][head_dim] operand copies of up to MF_NOALLOC_MAX_ELEMS elements.
constexpr size_t kScratchBytes =
    round_up(256 + round_up(4 * static_cast<size_t>(MF_NOALLOC_MAX_SAMPLES), 256) +
                 round_up(4 * (static_cast<size_t>(MF_NOALLOC_MAX_SAMPLES) + 1), 256),
             1024) +
    3 * round_up(2 * static_cast<size_t>(MF_NOALLOC_MAX_ELEMS), 1024);
static_assert(kScratchBytes == MF_NOALLOC_SCRATCH_BYTES, "mf.h states the scratch size");

// The scratch itself.  Host code must not pass this name to a kernel: on the host
// it is only a stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device
// (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace mf

extern "C" mf_status mf_varlen_attn_fwd_noalloc(const mf_bf16* q, const mf_bf16* k,
                                                const mf_bf16* v, const int32_t* d_cu_seqlens,
                                                const int32_t* d_pos, int32_t n, int32_t T,
                                                int32_t max_len, int32_t heads, int32_t head_dim,
                                                float softmax_scale, mf_bf16* o, float* lse,
                                                mf_stream stream) {
  if (n < 0 || T < 0 || heads < 1) return MF_ERR_INVALID_ARG;
  if (n > MF_NOALLOC_MAX_SAMPLES ||
      static_cast<int64_t>(T) * heads * head_dim > MF_NOALLOC_MAX_ELEMS)
    return MF_ERR_UNSUPPORTED;  // beyond the fixed scratch: use mf_varlen_attn_fwd
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  const size_t need = mf::ws_layout(T, n, heads, head_dim, false).total;
  if (need > mf::kScratchBytes) return MF_ERR_UNSUPPORTED;
  void* ws = nullptr;
  if (mf::scratch_address(&ws) != cudaSuccess) return MF_ERR_CUDA;
  return mf_varlen_attn_fwd(q, k, v, d_cu_seqlens, d_pos, n, T, max_len, heads, head_dim,
                            softmax_scale, o, lse, ws, mf::kScratchBytes, stream);
}
