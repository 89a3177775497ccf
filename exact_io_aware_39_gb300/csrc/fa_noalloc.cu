// Backward pass without any device allocation by the caller or the library.
//
// flash_attn_bwd needs a device workspace (the fp32 dQ accumulator and two
// fp32 row vectors). Some callers cannot hand one over: code running as a
// plug-in inside another runtime's execute callback, where allocating device
// memory is not allowed; serving loops that must never call cudaMalloc on the
// request path, because it synchronises the device and can stall every
// stream; and programs whose device memory is owned entirely by a pool that
// does not give out raw buffers. flash_attn_bwd_noalloc serves them with a
// fixed scratch array that lives in this file as a device global, so nothing
// is allocated at call time. It runs the same launch sequence as
// flash_attn_bwd (one shared host function), over that array.
//
// Costs and rules of that choice:
//   * every GPU that loads the library holds the array (kScratchBytes) until
//     the process exits. Under CUDA's lazy module loading (the default) the
//     array is reserved when this file's module is first loaded on a device,
//     which is the first call of this entry point there: make that first call
//     outside any context that forbids allocation (or set
//     CUDA_MODULE_LOADING=EAGER, which loads it with the context); a call that
//     is refused for its shape after the address lookup also serves as such a
//     warm-up, since the lookup comes first;
//   * shapes whose workspace exceeds kScratchBytes are rejected;
//   * all calls share the one array: two calls whose kernels overlap on the
//     GPU (different streams, or the same stream from several threads without
//     ordering) race on it and give wrong results. Calls ordered on one stream
//     are fine. Everything the kernels read from it is written first within the
//     same call (the dQ accumulator is zeroed, the row vectors recomputed, the
//     work counter reset), so what a previous call left behind never matters;
//   * the first call on a device looks up the array's device address (the
//     host-side name of a __device__ array is not a device address) with that
//     device current; make that first call before any stream capture begins.
// There is no counterpart of this entry point on the pages describing the
// method; it is an interface convenience.
#include "flash_attn.h"
#include "fa_common.cuh"

#include <mutex>

namespace fa {
namespace {

constexpr size_t kScratchBytes = FA_BWD_NOALLOC_SCRATCH_BYTES;   // 64 MiB per device

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (looked up once per
// device, with that device current).
fa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" fa_status flash_attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                            const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                                            int B, int H, int N, int d, float scale, int causal,
                                            const int32_t* kv_len, const uint8_t* block_mask, void* stream) {
  const BwdArgs a{Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal, kv_len, block_mask};
  fa_status st = static_cast<fa_status>(internal_bwd_validate(a, nullptr));
  if (st != FA_OK) return st;
  void* scratch = nullptr;   // looked up before the size check, so that a refused call still loads the array
  if ((st = scratch_address(&scratch)) != FA_OK) return st;
  if (bwd_workspace_layout(B, H, N, d).total > kScratchBytes) return FA_ERR_SCRATCH_LIMIT;
  return static_cast<fa_status>(internal_bwd_run(a, nullptr, scratch, stream));
}
