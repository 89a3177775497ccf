// C ABI of the attention library: argument validation, TMA tensor-map
// construction, launches, the tile classifier export and the device error
// word. Declarations and the contract of every call are in flash_attn.h.
#include "flash_attn.h"
#include "fa_common.cuh"

#include <cmath>
#include <cstddef>
#include <cstring>
#include <mutex>

namespace fa {

// Device error word: {code, site, block, thread}. One copy per device that
// loads the library; kernels receive its address.
__device__ unsigned int g_fa_err[4];

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool ready = false;
  bool supported = false;
  unsigned int* err = nullptr;
};

// events recorded around the dominant kernel of the next call of this thread
thread_local cudaEvent_t t_prof_start = nullptr;
thread_local cudaEvent_t t_prof_stop = nullptr;

struct ProfileScope {
  cudaEvent_t a, b;
  cudaStream_t s;
  explicit ProfileScope(cudaStream_t st) : a(t_prof_start), b(t_prof_stop), s(st) {
    t_prof_start = t_prof_stop = nullptr;
  }
  void before() const { if (a) cudaEventRecord(a, s); }
  void after() const { if (b) cudaEventRecord(b, s); }
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

// Per-device set-up: checks for a compute capability 10.3 device and looks up
// the address of the error word on it.
fa_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    st.supported = (major == 10 && minor == 3);
    if (st.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_fa_err) != cudaSuccess) return FA_ERR_CUDA;
      st.err = static_cast<unsigned int*>(p);
    }
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return FA_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    st.ready = true;
  }
  if (!st.supported) return FA_ERR_UNSUPPORTED;
  *out = &st;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D view [BH, N, d] of a bf16 (or fp16) tensor, box 64 x rows x 1, 128-byte
// swizzle; rows past N read as zeros and are not written by stores. Loads use
// 128-row boxes (a whole tile); the outputs are stored by each warp for its
// own 32 rows.
fa_status make_map(CUtensorMap* m, const void* base, int BH, int N, int d, bool f16, int rows = kTile) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 3-D view [BH, Np, d] of the fp32 dQ accumulator, box 32 x rows x 1 (one
// 128-byte row per box row), 128-byte swizzle: whole 128-row tiles for the
// narrow backward, 32 rows (each warp its own) for the wide one.
fa_status make_dq_map(CUtensorMap* m, const float* base, int BH, int Np, int d, int rows) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Np, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)Np * d * 4};
  cuuint32_t box[3] = {32, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

struct Options {
  bool f16 = false;
  DropoutParams drop{0u, 0u, 0u, 1.0f};
  CheckParams chk{nullptr, 2000000u, 0u};   // 2 s per wait
};

// Reads the caller's options (NULL = defaults). Fields beyond the caller's
// declared size keep their defaults, so older callers of a grown struct work.
fa_status read_options(const fa_options* opt, Options* out) {
  *out = Options{};
  if (opt == nullptr) return FA_OK;
  if (opt->size < sizeof(uint32_t) + sizeof(int32_t)) return FA_ERR_INVALID_ARG;
  if (opt->dtype != FA_DTYPE_BF16 && opt->dtype != FA_DTYPE_F16) return FA_ERR_UNSUPPORTED;
  out->f16 = opt->dtype == FA_DTYPE_F16;
  if (opt->size >= offsetof(fa_options, seed) + sizeof(uint64_t)) {
    const float p = opt->p_drop;
    if (!std::isfinite(p) || p < 0.f || p >= 1.f) return FA_ERR_INVALID_ARG;
    const uint32_t t = (uint32_t)std::floor((double)p * 256.0 + 0.5);
    if (t > 255u) return FA_ERR_INVALID_ARG;
    out->drop.t = t;
    out->drop.keep_scale = (float)(256.0 / (256.0 - (double)t));
    out->drop.seed_lo = (uint32_t)(opt->seed & 0xFFFFFFFFull);
    out->drop.seed_hi = (uint32_t)(opt->seed >> 32);
  }
  if (opt->size >= offsetof(fa_options, tile_record) + sizeof(uint8_t*)) out->chk.rec = opt->tile_record;
  if (opt->size >= offsetof(fa_options, wait_limit_us) + sizeof(uint32_t) && opt->wait_limit_us != 0u)
    out->chk.wait_us = opt->wait_limit_us;
  if (opt->size >= offsetof(fa_options, test_stall) + sizeof(uint32_t)) {
    if (opt->test_stall > 1u) return FA_ERR_INVALID_ARG;
    out->chk.stall = opt->test_stall;
  }
  return FA_OK;
}

fa_status check_shape(int B, int H, int N, int d, float scale, int causal) {
  if (B < 1 || H < 1 || N < 1 || !std::isfinite(scale) || (causal != 0 && causal != 1))
    return FA_ERR_INVALID_ARG;
  if (d < 8 || d > kMaxHeadDim || (d % 8) != 0) return FA_ERR_UNSUPPORTED;
  if (N > kMaxN) return FA_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  const long long nT = (N + kTile - 1) / kTile;
  if (BH * nT > 0x7FFFFFFFll) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

__global__ void tile_map_kernel(int B, int N, int nT, int causal, const int32_t* kv_len, const uint8_t* bm,
                                uint8_t* out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)B * nT * nT;
  if (idx >= total) return;
  const int b = (int)(idx / ((long long)nT * nT));
  const int rem = (int)(idx % ((long long)nT * nT));
  const int qi = rem / nT, kj = rem % nT;
  out[idx] = (uint8_t)tile_state(qi, kj, effective_kv_len(kv_len, b, N), nT, causal, bm);
}

}  // namespace

// Internal accessors for other translation units of the library.
int internal_check_shape(int B, int H, int N, int d, float scale, int causal) {
  return check_shape(B, H, N, d, scale, causal);
}

int internal_device_error_word(unsigned int** err) {
  DeviceState* ds = nullptr;
  const fa_status st = device_state(&ds);
  if (st == FA_OK) *err = ds->err;
  return st;
}

int internal_read_options(const void* options, bool* f16, bool* flash_only) {
  Options o;
  const fa_status st = read_options(static_cast<const fa_options*>(options), &o);
  if (st == FA_OK) {
    *f16 = o.f16;
    *flash_only = o.drop.t != 0u || o.chk.rec != nullptr || o.chk.stall != 0u;
  }
  return st;
}

int internal_bwd_validate(const BwdArgs& a, const void* options) {
  fa_status st = check_shape(a.B, a.H, a.N, a.d, a.scale, a.causal);
  if (st != FA_OK) return st;
  Options o;
  if ((st = read_options(static_cast<const fa_options*>(options), &o)) != FA_OK) return st;
  if (o.drop.t != 0u && a.d > 128) return FA_ERR_UNSUPPORTED;   // no dropout in the wide kernels
  const void* ptrs[] = {a.Q, a.K, a.V, a.O, a.dO, a.LSE, a.dQ, a.dK, a.dV};
  for (const void* q : ptrs)
    if (q == nullptr || !aligned16(q)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// The backward launch sequence over a workspace of at least
// bwd_workspace_layout(...).total bytes (256-byte aligned): the pre-pass
// (row statistics, zeroed dQ accumulator and work counter), the main kernel
// (with the caller's profile events around it) and the dQ conversion.
int internal_bwd_run(const BwdArgs& a, const void* options, void* workspace, void* stream) {
  Options o;
  fa_status st = read_options(static_cast<const fa_options*>(options), &o);
  if (st != FA_OK) return st;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;
  const int B = a.B, H = a.H, N = a.N, d = a.d;
  const BwdWorkspace w = bwd_workspace_layout(B, H, N, d);
  const int BH = B * H;
  const int nT = (N + kTile - 1) / kTile;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(ws + w.dq_off);
  float* lse2 = reinterpret_cast<float*>(ws + w.lse2_off);
  float* delta = reinterpret_cast<float*>(ws + w.delta_off);
  unsigned int* sched = reinterpret_cast<unsigned int*>(ws + w.sched_off);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
  const int kd = kernel_head_dim(d);
  const int qrows = kd == 256 ? 64 : kTile;    // the wide backward takes 64 queries at a time
  // the narrow kernels store dK and dV a whole tile at a time, the wide one per
  // warp (32 rows); the dQ partials are added per warp (32 rows) except by the
  // 64-column kernel, which adds whole 128-row tiles
  const int srows = kd == 256 ? 32 : kTile;
  const int dqrows = kd == 64 ? kTile : 32;
  if (make_map(&tq, a.Q, BH, N, d, o.f16, qrows) || make_map(&tk, a.K, BH, N, d, o.f16) ||
      make_map(&tv, a.V, BH, N, d, o.f16) || make_map(&tdo, a.dO, BH, N, d, o.f16, qrows) ||
      make_map(&tdk, a.dK, BH, N, d, o.f16, srows) || make_map(&tdv, a.dV, BH, N, d, o.f16, srows) ||
      make_dq_map(&tdq, dq_acc, BH, nT * kTile, d, dqrows))
    return FA_ERR_CUDA;
  if (launch_bwd_pre(o.f16, a.O, a.dO, a.LSE, dq_acc, lse2, delta, sched, BH, N, nT, d, s) != cudaSuccess)
    return FA_ERR_CUDA;
  BwdParams p{};
  p.kv_len = a.kv_len;
  p.block_mask = a.block_mask;
  p.dq_acc = dq_acc;
  p.lse2 = lse2;
  p.delta = delta;
  p.sched = sched;
  p.err = ds->err;
  p.B = B;
  p.H = H;
  p.N = N;
  p.nT = nT;
  p.causal = a.causal;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.drop = o.drop;
  p.chk = o.chk;
  p.d = d;
  const ProfileScope prof(s);
  prof.before();
  const cudaError_t e = launch_bwd_main(d, o.f16, tq, tk, tv, tdo, tdk, tdv, tdq, p, s);
  prof.after();
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (launch_bwd_dq(o.f16, dq_acc, a.dQ, a.scale, BH, N, nT, d, s) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

cudaError_t launch_tile_map(int B, int N, int nT, int causal, const int32_t* kv_len, const uint8_t* block_mask,
                            uint8_t* out, cudaStream_t s) {
  const long long total = (long long)B * nT * nT;
  const unsigned grid = (unsigned)((total + 255) / 256);
  tile_map_kernel<<<grid, 256, 0, s>>>(B, N, nT, causal, kv_len, block_mask, out);
  return cudaGetLastError();
}

}  // namespace fa

using namespace fa;

extern "C" {

fa_status flash_attn_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                            int N, int d, float scale, int causal, const int32_t* kv_len,
                            const uint8_t* block_mask, const fa_options* options, void* stream) {
  fa_status st = check_shape(B, H, N, d, scale, causal);
  if (st != FA_OK) return st;
  Options o;
  if ((st = read_options(options, &o)) != FA_OK) return st;
  if (o.drop.t != 0u && d > 128) return FA_ERR_UNSUPPORTED;   // no dropout in the wide kernels
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return FA_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv, to;
  if (make_map(&tq, Q, BH, N, d, o.f16) || make_map(&tk, K, BH, N, d, o.f16) ||
      make_map(&tv, V, BH, N, d, o.f16) || make_map(&to, O, BH, N, d, o.f16, 32))
    return FA_ERR_CUDA;
  FwdParams p{};
  p.lse = LSE;
  p.kv_len = kv_len;
  p.block_mask = block_mask;
  p.err = ds->err;
  p.B = B;
  p.H = H;
  p.N = N;
  p.nT = (N + kTile - 1) / kTile;
  p.causal = causal;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.drop = o.drop;
  p.chk = o.chk;
  p.d = d;
  const ProfileScope prof(static_cast<cudaStream_t>(stream));
  prof.before();
  const cudaError_t e = launch_fwd(d, o.f16, tq, tk, tv, to, p, static_cast<cudaStream_t>(stream));
  prof.after();
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status flash_attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                         int d, float scale, int causal, const int32_t* kv_len, const uint8_t* block_mask,
                         void* stream) {
  return flash_attn_fwd_ex(Q, K, V, O, LSE, B, H, N, d, scale, causal, kv_len, block_mask, nullptr, stream);
}

size_t flash_attn_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d, 1.0f, 0) != FA_OK) return 0;
  return bwd_workspace_layout(B, H, N, d).total;
}

fa_status flash_attn_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                            const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                            float scale, int causal, const int32_t* kv_len, const uint8_t* block_mask,
                            const fa_options* options, void* workspace, size_t workspace_bytes, void* stream) {
  const BwdArgs a{Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal, kv_len, block_mask};
  fa_status st = static_cast<fa_status>(internal_bwd_validate(a, options));
  if (st != FA_OK) return st;
  const BwdWorkspace w = bwd_workspace_layout(B, H, N, d);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < w.total)
    return FA_ERR_WORKSPACE;
  return static_cast<fa_status>(internal_bwd_run(a, options, workspace, stream));
}

fa_status flash_attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                         const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int N, int d, float scale,
                         int causal, const int32_t* kv_len, const uint8_t* block_mask, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return flash_attn_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal, kv_len, block_mask,
                           nullptr, workspace, workspace_bytes, stream);
}

fa_status flash_attn_tile_map(int B, int N, int causal, const int32_t* kv_len, const uint8_t* block_mask,
                              uint8_t* out, void* stream) {
  if (B < 1 || N < 1 || N > kMaxN || (causal != 0 && causal != 1) || out == nullptr) return FA_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  fa_status st = device_state(&ds);
  if (st != FA_OK) return st;
  const int nT = (N + kTile - 1) / kTile;
  return launch_tile_map(B, N, nT, causal, kv_len, block_mask, out, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status flash_attn_get_device_error(uint32_t* detail) {
  DeviceState* ds = nullptr;
  fa_status st = device_state(&ds);
  if (st != FA_OK) return st;
  unsigned int h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, ds->err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  const unsigned int zero[4] = {0, 0, 0, 0};
  if (cudaMemcpy(ds->err, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  if (detail) std::memcpy(detail, h, sizeof(h));
  if (h[0] == 0) return FA_OK;
  if (h[0] == kErrTimeout) return FA_ERR_DEVICE_TIMEOUT;
  return FA_ERR_DEVICE_INTERNAL;
}

fa_status flash_attn_set_profile_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return FA_ERR_INVALID_ARG;
  t_prof_start = static_cast<cudaEvent_t>(start_event);
  t_prof_stop = static_cast<cudaEvent_t>(stop_event);
  return FA_OK;
}

const char* flash_attn_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported shape or device";
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case FA_ERR_DEVICE_INTERNAL: return "device internal error";
    case FA_ERR_SCRATCH_LIMIT: return "shape needs more scratch than the fixed no-alloc scratch array";
  }
  return "unknown status";
}

int flash_attn_version(void) { return 100; }

}  // extern "C"
