// Standard (materialising) attention: the baseline of the IO comparison
// (FlashAttention milestone page (nlp-lineage), "The notation" and "What it
// showed"). The score matrix S and the probabilities P live in device memory;
// the six matrix products are cuBLAS strided-batched GEMMs, the masked row
// softmax and the dS rows are the two kernels below. The contract of the
// entry points is in standard_attn.h.
#include "standard_attn.h"
#include "fa_common.cuh"

#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>

namespace fa {
namespace {

constexpr int kRowThreads = 256;
constexpr int kStdMaxN = 65536;

template <bool F16>
__device__ __forceinline__ float load16(uint32_t v) {   // the low 16 bits hold the value
  if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)v));
  else return __bfloat162float(__ushort_as_bfloat16((unsigned short)v));
}

template <bool F16>
__device__ __forceinline__ uint16_t to16(float x) {
  if constexpr (F16) return __half_as_ushort(__float2half_rn(x));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

constexpr int kRowsPerCta = kRowThreads / 32;   // one warp per row

// Element e (and e .. e + 3, 16-byte / 8-byte aligned for rows with N a
// multiple of 4) of a stored score-like matrix: fp32, or the 16-bit input type.
template <bool F16, bool S16>
__device__ __forceinline__ float4 row_load4(const void* base, size_t e) {
  if constexpr (S16) {
    const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + e);
    return make_float4(load16<F16>(v.x & 0xFFFFu), load16<F16>(v.x >> 16), load16<F16>(v.y & 0xFFFFu),
                       load16<F16>(v.y >> 16));
  } else {
    return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + e);
  }
}

template <bool F16, bool S16>
__device__ __forceinline__ float row_load1(const void* base, size_t e) {
  if constexpr (S16) return load16<F16>(static_cast<const uint16_t*>(base)[e]);
  else return static_cast<const float*>(base)[e];
}

// Warp-wide combination of per-lane (max, sum of exp(x - max)) pairs.
__device__ __forceinline__ void warp_max_sum(float& m, float& l) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l, o);
    const float mn = fmaxf(m, m2);
    l = (mn == -INFINITY) ? 0.f : l * expf(m - mn) + l2 * expf(m2 - mn);
    m = mn;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ void online_add(float x, float& m, float& l) {
  if (x > m) {
    l = l * expf(m - x) + 1.f;
    m = x;
  } else {
    l += expf(x - m);
  }
}

// One warp per row i of one (batch, head): masked softmax of the (already
// scaled) scores. P_ij = exp(S_ij - LSE_i) on allowed keys, 0 elsewhere;
// LSE_i = max + ln(sum exp(S_ij - max)), -inf for a row with no allowed key.
// Rows with N a multiple of 4 are read as float4 (16-byte aligned rows).
template <bool F16, bool S16>
__global__ void __launch_bounds__(kRowThreads) std_softmax_kernel(const void* __restrict__ Sv,
                                                                  uint16_t* __restrict__ P, float* __restrict__ lse,
                                                                  long long rows, int H, int N, int nT, int causal,
                                                                  const int32_t* kv_len, const uint8_t* bm) {
  const long long row = (long long)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const int i = (int)(row % N);
  const int b = (int)(row / N) / H;
  const int kvl = effective_kv_len(kv_len, b, N);
  const int jmax = causal ? min(kvl, i + 1) : kvl;          // allowed keys are j < jmax ...
  uint16_t* p = P + (size_t)row * N;
  const uint8_t* bmrow = bm ? bm + (size_t)(i / kTile) * nT : nullptr;
  auto allowed = [&](int j) -> bool {                        // ... and not in a masked block
    return j < jmax && (bmrow == nullptr || bmrow[j / kTile] != 0);
  };
  float m = -INFINITY, l = 0.f;
  const bool vec = (N & 3) == 0;
  auto load4 = [&](int j) -> float4 { return row_load4<F16, S16>(Sv, (size_t)row * N + j); };
  auto load1 = [&](int j) -> float { return row_load1<F16, S16>(Sv, (size_t)row * N + j); };
  if (vec) {
    for (int j = 4 * lane; j < N; j += 128) {
      const float4 x = load4(j);
      if (allowed(j)) online_add(x.x, m, l);
      if (allowed(j + 1)) online_add(x.y, m, l);
      if (allowed(j + 2)) online_add(x.z, m, l);
      if (allowed(j + 3)) online_add(x.w, m, l);
    }
  } else {
    for (int j = lane; j < N; j += 32)
      if (allowed(j)) online_add(load1(j), m, l);
  }
  warp_max_sum(m, l);
  const float L = (m == -INFINITY) ? -INFINITY : m + logf(l);
  if (vec) {
    for (int j = 4 * lane; j < N; j += 128) {
      const float4 x = load4(j);
      const uint32_t a = (uint32_t)to16<F16>(allowed(j) ? expf(x.x - L) : 0.f) |
                         ((uint32_t)to16<F16>(allowed(j + 1) ? expf(x.y - L) : 0.f) << 16);
      const uint32_t c = (uint32_t)to16<F16>(allowed(j + 2) ? expf(x.z - L) : 0.f) |
                         ((uint32_t)to16<F16>(allowed(j + 3) ? expf(x.w - L) : 0.f) << 16);
      *reinterpret_cast<uint2*>(p + j) = make_uint2(a, c);
    }
  } else {
    for (int j = lane; j < N; j += 32) p[j] = to16<F16>(allowed(j) ? expf(load1(j) - L) : 0.f);
  }
  if (lane == 0) lse[row] = L;
}

// One warp per row: D_i = sum_j P_ij dP_ij, then dS_ij = P_ij (dP_ij - D_i)
// written over P (the gradient of the softmax, as autograd forms it).
template <bool F16, bool S16>
__global__ void __launch_bounds__(kRowThreads) std_ds_kernel(const void* __restrict__ dPv, uint16_t* PdS,
                                                             long long rows, int N) {
  const long long row = (long long)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  uint16_t* p = PdS + (size_t)row * N;
  const bool vec = (N & 3) == 0;
  auto load4 = [&](int j) -> float4 { return row_load4<F16, S16>(dPv, (size_t)row * N + j); };
  auto load1 = [&](int j) -> float { return row_load1<F16, S16>(dPv, (size_t)row * N + j); };
  float acc = 0.f;
  if (vec) {
    for (int j = 4 * lane; j < N; j += 128) {
      const float4 x = load4(j);
      const uint2 pp = *reinterpret_cast<const uint2*>(p + j);
      acc += load16<F16>(pp.x & 0xFFFFu) * x.x + load16<F16>(pp.x >> 16) * x.y +
             load16<F16>(pp.y & 0xFFFFu) * x.z + load16<F16>(pp.y >> 16) * x.w;
    }
  } else {
    for (int j = lane; j < N; j += 32) acc += load16<F16>(p[j]) * load1(j);
  }
  const float D = warp_sum(acc);
  if (vec) {
    for (int j = 4 * lane; j < N; j += 128) {
      const float4 x = load4(j);
      const uint2 pp = *reinterpret_cast<const uint2*>(p + j);
      const uint32_t a = (uint32_t)to16<F16>(load16<F16>(pp.x & 0xFFFFu) * (x.x - D)) |
                         ((uint32_t)to16<F16>(load16<F16>(pp.x >> 16) * (x.y - D)) << 16);
      const uint32_t c = (uint32_t)to16<F16>(load16<F16>(pp.y & 0xFFFFu) * (x.z - D)) |
                         ((uint32_t)to16<F16>(load16<F16>(pp.y >> 16) * (x.w - D)) << 16);
      *reinterpret_cast<uint2*>(p + j) = make_uint2(a, c);
    }
  } else {
    for (int j = lane; j < N; j += 32) p[j] = to16<F16>(load16<F16>(p[j]) * (load1(j) - D));
  }
}

struct Handle {
  bool ready = false;
  cublasHandle_t h = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
Handle g_handles[kMaxDevices];

// cuBLAS handle of the current device (created on first use); the caller
// holds g_mu while it uses it, since the stream is set per call.
fa_status cublas_handle(cublasHandle_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  Handle& hd = g_handles[dev];
  if (!hd.ready) {
    if (cublasCreate(&hd.h) != CUBLAS_STATUS_SUCCESS) return FA_ERR_CUDA;
    hd.ready = true;
  }
  *out = hd.h;
  return FA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool ws_layout(int B, int H, int N, size_t* s_bytes, size_t* total) {
  if (B < 1 || H < 1 || N < 1 || N > kStdMaxN) return false;
  const unsigned long long BH = (unsigned long long)B * (unsigned long long)H;
  const unsigned long long nn = (unsigned long long)N * (unsigned long long)N;
  if (BH > (1ull << 40) / nn) return false;   // keeps every product below 2^43 bytes
  *s_bytes = align256((size_t)(BH * nn * 4ull));
  *total = *s_bytes + align256((size_t)(BH * nn * 2ull));
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_common(int B, int H, int N, int d, float scale, const fa_options* options, bool* f16,
                       void* workspace, size_t workspace_bytes, size_t* s_bytes) {
  if (B < 1 || H < 1 || N < 1 || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (N > kStdMaxN || d < 8 || d > 256 || (d % 8) != 0) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H * N > 0x7FFFFFFFll) return FA_ERR_UNSUPPORTED;   // one warp per row
  bool flash_only = false;   // dropout, tile record and test stall belong to the flash kernels
  const int so = internal_read_options(options, f16, &flash_only);
  if (so != FA_OK) return (fa_status)so;
  if (flash_only) return FA_ERR_UNSUPPORTED;
  size_t total = 0;
  if (!ws_layout(B, H, N, s_bytes, &total)) return FA_ERR_UNSUPPORTED;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < total)
    return FA_ERR_WORKSPACE;
  unsigned int* err = nullptr;   // device check (sm_103a) and per-device set-up
  return (fa_status)internal_device_error_word(&err);
}

// Row-major C[BH][rows_c][cols_c] products through cuBLAS's column-major
// GEMM: a row-major matrix is the column-major matrix of its transpose.
cublasStatus_t gemm(cublasHandle_t h, cublasOperation_t ta, cublasOperation_t tb, int m, int n, int k, float alpha,
                    const void* A, cudaDataType at, int lda, long long sa, const void* Bm, cudaDataType bt, int ldb,
                    long long sb, void* C, cudaDataType ct, int ldc, long long sc, int batch) {
  const float beta = 0.f;
  return cublasGemmStridedBatchedEx(h, ta, tb, m, n, k, &alpha, A, at, lda, sa, Bm, bt, ldb, sb, &beta, C, ct, ldc,
                                    sc, batch, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

size_t standard_attn_workspace_size(int B, int H, int N) {
  size_t s_bytes = 0, total = 0;
  return ws_layout(B, H, N, &s_bytes, &total) ? total : 0;
}

fa_status standard_attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                            int d, float scale, int causal, const int32_t* kv_len, const uint8_t* block_mask,
                            const fa_options* options, int flags, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!Q || !K || !V || !O || !LSE || !aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
      !aligned16(LSE) || (causal != 0 && causal != 1) || (flags & ~STANDARD_ATTN_S16) != 0)
    return FA_ERR_INVALID_ARG;
  const bool s16 = (flags & STANDARD_ATTN_S16) != 0;
  bool f16 = false;
  size_t s_bytes = 0;
  fa_status st = check_common(B, H, N, d, scale, options, &f16, workspace, workspace_bytes, &s_bytes);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* S = workspace;
  uint16_t* P = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + s_bytes);
  const cudaDataType t16 = f16 ? CUDA_R_16F : CUDA_R_16BF;
  const cudaDataType ts = s16 ? t16 : CUDA_R_32F;
  const int BH = B * H;
  const long long nd = (long long)N * d, nn = (long long)N * N;
  std::lock_guard<std::mutex> lk(g_mu);
  cublasHandle_t h = nullptr;
  if ((st = cublas_handle(&h)) != FA_OK) return st;
  if (cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return FA_ERR_CUDA;
  // S = scale * Q K^T  (column-major: S^T = K Q^T)
  if (gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, N, N, d, scale, K, t16, d, nd, Q, t16, d, nd, S, ts, N, nn, BH) !=
      CUBLAS_STATUS_SUCCESS)
    return FA_ERR_CUDA;
  const int nT = (N + kTile - 1) / kTile;
  const long long rows = (long long)BH * N;
  const unsigned grid = (unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta);
#define STD_SOFTMAX(FF, SS) \
  std_softmax_kernel<FF, SS><<<grid, kRowThreads, 0, s>>>(S, P, LSE, rows, H, N, nT, causal, kv_len, block_mask)
  if (f16) {
    if (s16) STD_SOFTMAX(true, true); else STD_SOFTMAX(true, false);
  } else {
    if (s16) STD_SOFTMAX(false, true); else STD_SOFTMAX(false, false);
  }
#undef STD_SOFTMAX
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  // O = P V  (column-major: O^T = V^T P^T)
  if (gemm(h, CUBLAS_OP_N, CUBLAS_OP_N, d, N, N, 1.f, V, t16, d, nd, P, t16, N, nn, O, t16, d, nd, BH) !=
      CUBLAS_STATUS_SUCCESS)
    return FA_ERR_CUDA;
  return FA_OK;
}

fa_status standard_attn_bwd(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK,
                            void* dV, int B, int H, int N, int d, float scale, const fa_options* options,
                            int flags, void* workspace, size_t workspace_bytes, void* stream) {
  if (!Q || !K || !V || !dO || !dQ || !dK || !dV || !aligned16(Q) || !aligned16(K) || !aligned16(V) ||
      !aligned16(dO) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV) || (flags & ~STANDARD_ATTN_S16) != 0)
    return FA_ERR_INVALID_ARG;
  const bool s16 = (flags & STANDARD_ATTN_S16) != 0;
  bool f16 = false;
  size_t s_bytes = 0;
  fa_status st = check_common(B, H, N, d, scale, options, &f16, workspace, workspace_bytes, &s_bytes);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* dP = workspace;
  uint16_t* P = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + s_bytes);
  const cudaDataType t16 = f16 ? CUDA_R_16F : CUDA_R_16BF;
  const cudaDataType ts = s16 ? t16 : CUDA_R_32F;
  const int BH = B * H;
  const long long nd = (long long)N * d, nn = (long long)N * N;
  std::lock_guard<std::mutex> lk(g_mu);
  cublasHandle_t h = nullptr;
  if ((st = cublas_handle(&h)) != FA_OK) return st;
  if (cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return FA_ERR_CUDA;
  // dV = P^T dO  (column-major: dV^T = dO^T P)
  if (gemm(h, CUBLAS_OP_N, CUBLAS_OP_T, d, N, N, 1.f, dO, t16, d, nd, P, t16, N, nn, dV, t16, d, nd, BH) !=
      CUBLAS_STATUS_SUCCESS)
    return FA_ERR_CUDA;
  // dP = dO V^T  (column-major: dP^T = V dO^T)
  if (gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, N, N, d, 1.f, V, t16, d, nd, dO, t16, d, nd, dP, ts, N, nn, BH) !=
      CUBLAS_STATUS_SUCCESS)
    return FA_ERR_CUDA;
  const long long rows = (long long)BH * N;
  const unsigned grid = (unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta);
  if (f16) {
    if (s16) std_ds_kernel<true, true><<<grid, kRowThreads, 0, s>>>(dP, P, rows, N);
    else std_ds_kernel<true, false><<<grid, kRowThreads, 0, s>>>(dP, P, rows, N);
  } else {
    if (s16) std_ds_kernel<false, true><<<grid, kRowThreads, 0, s>>>(dP, P, rows, N);
    else std_ds_kernel<false, false><<<grid, kRowThreads, 0, s>>>(dP, P, rows, N);
  }
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  const uint16_t* dS = P;
  // dQ = scale * dS K  (column-major: dQ^T = K^T dS^T)
  if (gemm(h, CUBLAS_OP_N, CUBLAS_OP_N, d, N, N, scale, K, t16, d, nd, dS, t16, N, nn, dQ, t16, d, nd, BH) !=
      CUBLAS_STATUS_SUCCESS)
    return FA_ERR_CUDA;
  // dK = scale * dS^T Q  (column-major: dK^T = Q^T dS)
  if (gemm(h, CUBLAS_OP_N, CUBLAS_OP_T, d, N, N, scale, Q, t16, d, nd, dS, t16, N, nn, dK, t16, d, nd, BH) !=
      CUBLAS_STATUS_SUCCESS)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"
