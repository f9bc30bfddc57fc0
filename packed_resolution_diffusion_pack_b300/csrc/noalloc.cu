// mf_varlen_attn_fwd_noalloc: the attention forward for callers that cannot
// allocate device memory.  Some callers are handed only their inputs and outputs
// and may not call cudaMalloc themselves: a plugin inside a framework that owns
// the device allocator, or a latency-critical loop where cudaMalloc/cudaFree
// (which can synchronise the device) are not allowed.  This entry point needs no
// workspace from them: its scratch is one file-scope device array of fixed size,
// which every GPU that loads this library holds until the process exits.
#include <cuda.h>
#include <cudaTypedefs.h>
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
struct Cached {
  void* addr = nullptr;
  unsigned long long ctx_id = 0;  // unique id of the context the address belongs to
};
Cached g_cache[kMaxDevices];

// Unique id of the calling thread's current context (driver entry points through
// the runtime, so the library needs no -lcuda).  A device reset or a new primary
// context gets a new id; ids are never reused within a process.
cudaError_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  if (get_current == nullptr || get_id == nullptr) {
    cudaDriverEntryPointQueryResult q1, q2;
    void *f1 = nullptr, *f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return cudaErrorNotSupported;
    get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
    get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

// Device address of g_scratch on the current device, looked up once per device
// and context (with that device current) and cached.  The cache is keyed on the
// context's unique id: after cudaDeviceReset the module is loaded again in a new
// context, and the address is looked up afresh on the next call.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long id = 0;
  if (current_context_id(&id) != cudaSuccess) {
    // no context current yet: cudaSetDevice initialises the device's primary one
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    e = current_context_id(&id);
    if (e != cudaSuccess) return e;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  Cached& c = g_cache[dev];
  if (c.addr == nullptr || c.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    c.addr = p;
    c.ctx_id = id;
  }
  *out = c.addr;
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

// The status word of the last allocation-free forward on the current device: it
// sits at offset 0 of the scratch array, where mf_get_status reads it for a
// caller workspace.
extern "C" mf_status mf_noalloc_get_status(mf_stream stream) {
  void* ws = nullptr;
  if (mf::scratch_address(&ws) != cudaSuccess) return MF_ERR_CUDA;
  return mf_get_status(ws, stream);
}
