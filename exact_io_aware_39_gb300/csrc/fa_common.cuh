// Shared definitions of the attention kernels: tile size, the tile
// classifier, kernel parameter blocks and the internal launcher interface.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

constexpr int kTile = 128;            // rows of a Q tile and of a K/V tile
constexpr int kMaxN = 131072;         // longest supported sequence
constexpr int kMaxDevices = 64;       // device ordinals with per-device library state

enum TileState : int { kSkip = 0, kFull = 1, kPartial = 2 };

// Device error word layout: [0] = first error code (0 = none), [1] = site id,
// [2] = blockIdx.x of the reporting CTA, [3] = threadIdx.x.
enum DeviceErr : uint32_t { kErrNone = 0, kErrTimeout = 5, kErrSmemAlign = 6, kErrInternal = 6 };

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

// Run-time checks shared by the kernels. rec, when not null, is the caller's
// uint8 [BH, nT, nT] record of the tiles a kernel computed: the thread that
// decides whether a tile needs element masking adds 1 (no masking) or 2
// (masking) to the tile's byte, so that a tile computed twice would show as a
// larger value. wait_us bounds every mbarrier wait. stall (test only, 0 in
// normal use) makes a producer stop loading after its first tile, so that a
// consumer's bounded wait runs out and the kernel reports a timeout.
struct CheckParams {
  uint8_t* rec;
  uint32_t wait_us;
  uint32_t stall;
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
  CheckParams chk;
  int d;                      // head dimension of the tensors (<= the kernel's tile width)
  int group;                  // heads per group of the CTA order (set by the launcher)
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
  CheckParams chk;
  int d;                      // head dimension of the tensors (<= the kernel's tile width)
  int group;                  // heads per group of the work-item order (set by the launcher)
};

// Adds 1 (no element mask) or 2 (masked) to the record byte of tile (qi, kj)
// of batch-head bh. Out of line: it runs only when a caller asks for the
// record, and keeps its address arithmetic out of the hot loops' registers.
__device__ __noinline__ inline void record_tile(uint8_t* rec, int bh, int qi, int kj, int nT, bool partial) {
  uint8_t* rc = rec + ((size_t)bh * nT + qi) * nT + kj;
  *rc = (uint8_t)(*rc + (partial ? 2 : 1));
}

// Heads per group when the work of a launch is ordered group by group so that
// the data one group touches stays in L2 (~126 MB): bytes_per_head is what a
// head keeps re-reading while its items run; groups get a 32 MB share, since
// the items in flight can span two neighbouring groups and the rest of L2
// holds streamed data.
inline int l2_head_group(double bytes_per_head, int BH) {
  const double budget = 32.0 * 1024 * 1024;
  int g = (int)(budget / (bytes_per_head > 1.0 ? bytes_per_head : 1.0));
  return g < 1 ? 1 : (g > BH ? BH : g);
}

// Splits a work index of an order that walks groups of `group` heads, within
// a group `inner` steps (inner-major) over the group's heads (the last group
// may have fewer heads): returns the inner step and sets bh.
__host__ __device__ __forceinline__ int split_grouped(int index, int group, int inner, int BH, int* bh) {
  const int full = BH / group;              // groups of `group` heads
  const int per = inner * group;
  const int gi = index / per;
  if (gi < full) {
    const int rem = index - gi * per;
    *bh = gi * group + rem % group;
    return rem / group;
  }
  const int last = BH - full * group;       // heads of the last, smaller group
  const int rem = index - full * per;
  *bh = full * group + rem % last;
  return rem / last;
}

// Calls f() once per device for a setting that belongs to each device's copy
// of a kernel (its shared-memory limit); safe under concurrent callers.
struct PerDeviceOnce {
  std::atomic<bool> done[kMaxDevices];
  std::mutex mu;
};

template <typename F>
cudaError_t once_per_device(PerDeviceOnce& o, int dev, F&& f) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (o.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lk(o.mu);
  if (o.done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = f();
  if (e == cudaSuccess) o.done[dev].store(true, std::memory_order_release);
  return e;
}

// Launches a kernel, with programmatic stream serialization when pdl is set:
// it may then be scheduled while the previous kernel in the stream is still
// running (once that one allows it, or when its blocks exit), overlapping its
// launch and set-up with the other's tail. Every kernel waits
// (griddepcontrol.wait, a no-op without the attribute) before it touches
// global memory. Measured on the four-kernel step: with the attribute on the
// forward and backward main kernels only, 0-2 % faster on the short
// workloads; on all four launches the short non-causal ones lost 1-3 %.
template <typename... Exp, typename... Act>
cudaError_t launch_pdl(bool pdl, void (*kern)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Act>(args)...);
}

// Head dimension of the kernel that serves a head dimension d (a multiple of
// 8 up to 256): tiles are 64, 128 or 256 columns wide; columns past d are
// zeros on load (TMA out-of-bounds fill) and are not written on store.
__host__ __device__ __forceinline__ int kernel_head_dim(int d) { return d <= 64 ? 64 : (d <= 128 ? 128 : 256); }
constexpr int kMaxHeadDim = 256;

// Launchers (host). Tensor maps are 3-D [BH, N, d] bf16 views, box 64 x 128 x 1
// for loads and 64 x 32 x 1 for the stores of O, dK and dV (one box per warp),
// 128-byte swizzle. d is the tensors' head dimension; the kernel instance is
// chosen by kernel_head_dim(d). Return the cudaError_t of the launch.
// f16 selects fp16 elements (else bf16) for Q, K, V, O, dO, dQ, dK, dV.
// dropout is applied when p.drop.t > 0.
cudaError_t launch_fwd(int d, bool f16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, cudaStream_t s);

cudaError_t launch_bwd_pre(bool f16, const void* o, const void* dout, const float* lse, float* dq_acc,
                           float* lse2, float* delta, unsigned int* sched, int BH, int N, int nT, int d,
                           cudaStream_t s);

// tdq is the fp32 dQ accumulator seen as [BH, nT*128, d], box 32 x 128 x 1
// (32 x 32 x 1 for the wide kernel), 128-byte swizzle; partial dQ tiles are
// added into it with TMA reduce-add.
cudaError_t launch_bwd_main(int d, bool f16, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tdk, const CUtensorMap& tdv, const CUtensorMap& tdq,
                            const BwdParams& p, cudaStream_t s);

// The kernels for 128 < d <= 256 (fa_wide.cu; no dropout). The backward's
// tq and tdo are views with 64-row boxes (queries are taken 64 at a time).
// The one-Q-tile forward (S double-buffered in TMEM, K/V streamed in units of
// up to 128 columns) for a kernel head dimension kd of 64, 128 or 256.
cudaError_t launch_fwd_single(int kd, bool f16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, const FwdParams& p, cudaStream_t s);
cudaError_t launch_bwd_wide(bool f16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const CUtensorMap& tdq, const BwdParams& p, cudaStream_t s);

cudaError_t launch_bwd_dq(bool f16, const float* dq_acc, void* dq, float scale, int BH, int N, int nT, int d,
                          cudaStream_t s);

cudaError_t launch_tile_map(int B, int N, int nT, int causal, const int32_t* kv_len,
                            const uint8_t* block_mask, uint8_t* out, cudaStream_t s);

// Host helpers defined with the C ABI (return fa_status values).
int internal_check_shape(int B, int H, int N, int d, float scale, int causal);
int internal_device_error_word(unsigned int** err);   // current device; runs its set-up once
// options: const fa_options* or null. flash_only: an option only the flash
// kernels implement is set (dropout, tile record, test stall).
int internal_read_options(const void* options, bool* f16, bool* flash_only);

// Arguments of a backward call (the flash_attn_bwd signature without the
// workspace and the stream).
struct BwdArgs {
  const void *Q, *K, *V, *O, *dO;
  const float* LSE;
  void *dQ, *dK, *dV;
  int B, H, N, d;
  float scale;
  int causal;
  const int32_t* kv_len;
  const uint8_t* block_mask;
};
// Shape, pointer and option checks of a backward call (nothing launched).
int internal_bwd_validate(const BwdArgs& a, const void* options);
// The backward launch sequence over a validated call and a workspace of
// bwd_workspace_layout(...).total bytes, 256-byte aligned.
int internal_bwd_run(const BwdArgs& a, const void* options, void* workspace, void* stream);

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
