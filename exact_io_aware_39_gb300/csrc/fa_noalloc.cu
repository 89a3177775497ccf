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
// is allocated at call time.
//
// Costs and rules of that choice:
//   * every GPU that loads the library holds the array (kScratchBytes) until
//     the process exits;
//   * shapes whose workspace exceeds kScratchBytes are rejected;
//   * all calls share the one array: two calls whose kernels overlap on the
//     GPU (different streams, or the same stream from several threads without
//     ordering) race on it and give wrong results. Calls ordered on one stream
//     are fine. Everything the kernels read from it is written first within the
//     same call (the dQ accumulator is zeroed, the row vectors recomputed), so
//     what a previous call left behind never matters;
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
  fa_status st = static_cast<fa_status>(internal_check_shape(B, H, N, d, scale, causal));
  if (st != FA_OK) return st;
  const void* ptrs[] = {Q, K, V, O, dO, LSE, dQ, dK, dV};
  for (const void* q : ptrs)
    if (q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u) != 0) return FA_ERR_INVALID_ARG;
  const BwdWorkspace w = bwd_workspace_layout(B, H, N, d);
  if (w.total > kScratchBytes) return FA_ERR_SCRATCH_LIMIT;
  unsigned int* err = nullptr;
  if ((st = static_cast<fa_status>(internal_device_error_word(&err))) != FA_OK) return st;
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != FA_OK) return st;

  const int BH = B * H;
  const int nT = (N + kTile - 1) / kTile;
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  float* dq_acc = reinterpret_cast<float*>(ws + w.dq_off);
  float* lse2 = reinterpret_cast<float*>(ws + w.lse2_off);
  float* delta = reinterpret_cast<float*>(ws + w.delta_off);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  if (internal_make_map(&tq, Q, BH, N, d) || internal_make_map(&tk, K, BH, N, d) ||
      internal_make_map(&tv, V, BH, N, d) || internal_make_map(&tdo, dO, BH, N, d) ||
      internal_make_map(&tdk, dK, BH, N, d) || internal_make_map(&tdv, dV, BH, N, d))
    return FA_ERR_CUDA;
  CUtensorMap tdq;
  if (internal_make_dq_map(&tdq, dq_acc, BH, nT * kTile, d)) return FA_ERR_CUDA;
  // the pre-pass zeroes the dQ accumulator and rewrites both row vectors
  unsigned int* sched = reinterpret_cast<unsigned int*>(ws + w.sched_off);
  if (launch_bwd_pre(false, O, dO, LSE, dq_acc, lse2, delta, sched, BH, N, nT, d, s) != cudaSuccess)
    return FA_ERR_CUDA;
  BwdParams p{};
  p.kv_len = kv_len;
  p.block_mask = block_mask;
  p.dq_acc = dq_acc;
  p.lse2 = lse2;
  p.delta = delta;
  p.sched = sched;
  p.err = err;
  p.B = B;
  p.H = H;
  p.N = N;
  p.nT = nT;
  p.causal = causal;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.d = d;
  if (launch_bwd_main(d, false, tq, tk, tv, tdo, tdk, tdv, tdq, p, s) != cudaSuccess) return FA_ERR_CUDA;
  if (launch_bwd_dq(false, dq_acc, dQ, scale, BH, N, nT, d, s) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}
