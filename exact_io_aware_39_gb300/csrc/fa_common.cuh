// Shared definitions of the attention kernels: tile size, the tile
// classifier, kernel parameter blocks and the internal launcher interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

constexpr int kTile = 128;            // rows of a Q tile and of a K/V tile
constexpr int kMaxN = 131072;         // longest supported sequence
constexpr int kMaxDevices = 64;       // device ordinals with per-device library state

enum TileState : int { kSkip = 0, kFull = 1, kPartial = 2 };

// Device error word layout: [0] = first error code (0 = none), [1] = site id,
// [2] = blockIdx.x of the reporting CTA, [3] = threadIdx.x.
enum DeviceErr : uint32_t { kErrNone = 0, kErrTimeout = 5, kErrSmemAlign = 6 };

// State of the (query tile qi, key tile kj) pair. kvl is the effective key
// length of the batch entry, already clamped to [0, N]; bm is the block mask
// (nT x nT, row = query tile) or null. Masks combine by AND: a tile is skipped
// when its block is masked off, when it lies above the diagonal under the
// causal mask, or when all its keys are at or past kvl; it is partial when it
// straddles the diagonal or the key limit (keys past N always count as
// masked, so the ragged last key tile is partial), and full otherwise.
__host__ __device__ __forceinline__ int tile_state(int qi, int kj, int kvl, int nT, int causal,
                                                   const uint8_t* bm) {
  if (bm != nullptr && bm[qi * nT + kj] == 0) return kSkip;
  if (causal && kj > qi) return kSkip;
  if (kj * kTile >= kvl) return kSkip;
  if ((causal && kj == qi) || (kj + 1) * kTile > kvl) return kPartial;
  return kFull;
}

__host__ __device__ __forceinline__ int effective_kv_len(const int32_t* kv_len, int b, int N) {
  if (kv_len == nullptr) return N;
  int v = kv_len[b];
  return v < 0 ? 0 : (v > N ? N : v);
}

// Dropout on P. The keep decision of (batch-head bh, query i, key j) is the
// byte 4 (i mod 4) + (j mod 4) of Philox4x32-10 with counter
// (i / 4, j / 4, bh, 0) and key (seed_lo, seed_hi), compared with t: kept when
// >= t, a kept value is multiplied by keep_scale = 256 / (256 - t).
struct DropoutParams {
  uint32_t seed_lo, seed_hi;
  uint32_t t;          // 0..255; 0 keeps everything
  float keep_scale;
};

struct FwdParams {
  float* lse;                 // [BH, N] fp32
  const int32_t* kv_len;      // [B] or null
  const uint8_t* block_mask;  // [nT, nT] or null
  unsigned int* err;          // device error word
  int B, H, N, nT;
  int causal;
  float scale_log2;           // scale * log2(e)
  DropoutParams drop;
};

struct BwdParams {
  const int32_t* kv_len;
  const uint8_t* block_mask;
  float* dq_acc;              // [BH, nT*128, d] fp32 workspace
  const float* lse2;          // [BH, nT*128] fp32 workspace: LSE * log2(e), +inf on padding
  const float* delta;         // [BH, nT*128] fp32 workspace: rowsum(dO * O)
  unsigned int* sched;        // workspace word: next work item of the persistent main kernel (zeroed by the pre-pass)
  unsigned int* err;
  int B, H, N, nT;
  int causal;
  float scale_log2;
  DropoutParams drop;
  int d;                      // head dimension of the tensors (<= the kernel's tile width)
};

// Head dimension of the kernel that serves a head dimension d (a multiple of
// 8 up to 128): tiles are 64 or 128 columns wide; columns past d are zeros on
// load (TMA out-of-bounds fill) and are not written on store.
__host__ __device__ __forceinline__ int kernel_head_dim(int d) { return d <= 64 ? 64 : 128; }

// Launchers (host). Tensor maps are 3-D [BH, N, d] bf16 views, box 64 x 128 x 1,
// 128-byte swizzle. d is the tensors' head dimension; the kernel instance is
// chosen by kernel_head_dim(d). Return the cudaError_t of the launch.
// f16 selects fp16 elements (else bf16) for Q, K, V, O, dO, dQ, dK, dV.
// dropout is applied when p.drop.t > 0.
cudaError_t launch_fwd(int d, bool f16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, cudaStream_t s);

cudaError_t launch_bwd_pre(bool f16, const void* o, const void* dout, const float* lse, float* dq_acc,
                           float* lse2, float* delta, unsigned int* sched, int BH, int N, int nT, int d,
                           cudaStream_t s);

// tdq is the fp32 dQ accumulator seen as [BH, nT*128, d], box 32 x 128 x 1,
// 128-byte swizzle (internal_make_dq_map); partial dQ tiles are added into it
// with TMA reduce-add.
cudaError_t launch_bwd_main(int d, bool f16, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tdk, const CUtensorMap& tdv, const CUtensorMap& tdq,
                            const BwdParams& p, cudaStream_t s);

cudaError_t launch_bwd_dq(bool f16, const float* dq_acc, void* dq, float scale, int BH, int N, int nT, int d,
                          cudaStream_t s);

cudaError_t launch_tile_map(int B, int N, int nT, int causal, const int32_t* kv_len,
                            const uint8_t* block_mask, uint8_t* out, cudaStream_t s);

// Host helpers defined with the C ABI (return fa_status values).
int internal_check_shape(int B, int H, int N, int d, float scale, int causal);
int internal_device_error_word(unsigned int** err);   // current device; runs its set-up once
int internal_read_options(const void* options, bool* f16, bool* dropout);   // options: const fa_options*
int internal_make_map(CUtensorMap* m, const void* base, int BH, int N, int d);   // bf16
int internal_make_dq_map(CUtensorMap* m, const float* dq_acc, int BH, int Np, int d);

// Workspace layout of the backward pass (byte offsets, 256-aligned sections).
struct BwdWorkspace {
  size_t dq_off, lse2_off, delta_off, sched_off, total;
};

inline BwdWorkspace bwd_workspace_layout(int B, int H, int N, int d) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t BH = (size_t)B * H;
  const size_t Np = (size_t)((N + kTile - 1) / kTile) * kTile;
  BwdWorkspace w;
  w.dq_off = 0;
  w.lse2_off = al(w.dq_off + BH * Np * d * sizeof(float));
  w.delta_off = al(w.lse2_off + BH * Np * sizeof(float));
  w.sched_off = al(w.delta_off + BH * Np * sizeof(float));   // work counter of the main kernel
  w.total = w.sched_off + 256;
  return w;
}

}  // namespace fa
