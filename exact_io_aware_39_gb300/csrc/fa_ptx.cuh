// Hand-written inline-PTX primitives for sm_103a: mbarriers with bounded
// waits, TMA (cp.async.bulk.tensor) loads and stores, and the tcgen05 tensor
// core family (TMEM allocation, MMA, commit, TMEM loads and stores).
//
// Every wait on an mbarrier is bounded by a wall-clock limit read from
// %globaltimer; on expiry the waiting thread records a code in the device
// error word, raises the CTA's abort flag and returns false, so that a lost
// arrival ends the kernel with an error status instead of a hang.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "fa_common.cuh"

namespace fa {

// ---------------------------------------------------------------------------
// error reporting
// ---------------------------------------------------------------------------

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: default bound of a wait, and of every drain wait

// The wait limit is kept in shared memory next to the abort flag (read only
// on the slow path of a wait), so that it holds no register in the roles.
struct Ctl {
  unsigned int* err;          // global error word (4 x u32)
  volatile uint32_t* abort;   // [0] abort flag of this CTA, [2] bound of one mbarrier wait in microseconds
};

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report_error(const Ctl& c, uint32_t code, uint32_t site) {
  *c.abort = 1u;
  if (atomicCAS(c.err, 0u, code) == 0u) {
    c.err[1] = site;
    c.err[2] = blockIdx.x;
    c.err[3] = threadIdx.x;
  }
}

// ---------------------------------------------------------------------------
// shared-memory addresses, fences, named barriers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// Named barrier with an AND-reduction: every one of the nthreads threads
// arrives with a flag and all receive the AND of them. A group of warps that
// decides with this before a group-wide barrier takes the same branch
// everywhere, so that no warp can wait at a barrier that another has left.
__device__ __forceinline__ bool group_all(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r) : "r"(v ? 1u : 0u), "r"(id), "r"(nthreads) : "memory");
  return r != 0;
}

// Programmatic dependent launch: wait until the grid this one depends on (the
// previous kernel in the stream) has completed and its writes are visible;
// allow the next grid to be scheduled. Both are no-ops for a kernel launched
// without the programmatic-serialization attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}

// One arrival per warp: the warp's lanes synchronise (which orders their
// earlier memory and, after tcgen05.fence::before_thread_sync, TMEM accesses)
// and lane 0 arrives. Barriers signalled this way count warps, not threads.
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31u) == 0u) mbar_arrive(bar);
}

// Non-blocking test of phase completion.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Potentially blocking (for a hardware-chosen time) test of phase completion.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity. Returns false (after
// reporting) on timeout or when another thread of the CTA has aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  uint32_t n = 0;
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if ((++n & 15u) == 0u) {
      if (*c.abort) return false;
      if (globaltimer() - t0 > 1000ull * c.abort[2]) {
        report_error(c, kErrTimeout, site);
        return false;
      }
    }
  }
}

// Warp-collective bounded wait: every lane polls, and the result is the AND
// over the warp, so that the warp-collective tcgen05.ld/st that follow are
// executed by all lanes or by none.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
  const bool ok = mbar_wait(bar, parity, c, site);
  return __all_sync(0xFFFFFFFFu, ok);
}

template <bool W>
__device__ __forceinline__ bool mbar_wait_t(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
  if constexpr (W) return mbar_wait_warp(bar, parity, c, site);
  else return mbar_wait(bar, parity, c, site);
}

// Bounded wait that ignores the abort flag: used on exit paths to let copies
// and MMAs that were already issued finish before shared memory or TMEM is
// released.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

// ---------------------------------------------------------------------------
// TMA (tensor) copies
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src,
                                             int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
      :: "l"(reinterpret_cast<uint64_t>(m)), "r"(src), "r"(c0), "r"(c1), "r"(c2) : "memory");
}

// Element-wise reduce-add of a shared-memory box into global memory through
// the tensor map (fp32 add performed in L2 by the TMA unit).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, uint32_t src,
                                                  int c0, int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
      :: "l"(reinterpret_cast<uint64_t>(m)), "r"(src), "r"(c0), "r"(c1), "r"(c2) : "memory");
}

// Wait until the shared-memory sources of all committed bulk groups have
// been read (the buffers may be rewritten; the global writes may still be
// in flight).
__device__ __forceinline__ void bulk_wait_group_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_group_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Plain (non-tensor) bulk copy global -> shared; 16-byte aligned, size % 16 == 0.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar) : "memory");
}

// ---------------------------------------------------------------------------
// Cluster launch control: a running CTA cancels a CTA of its own grid that
// has not started yet and takes over its work. The 16-byte answer is written
// into shared memory and completes a transaction count on the mbarrier.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void clc_try_cancel(uint32_t answer_smem, uint32_t bar) {
  asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];"
               :: "r"(answer_smem), "r"(bar) : "memory");
}

// x index of the first CTA the answer cancelled, or -1 when nothing was left
// to cancel (read after the mbarrier phase has completed).
__device__ __forceinline__ int clc_first_ctaid_x(uint32_t answer_smem) {
  uint32_t x, ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b128 h;\n\t"
      "ld.shared.b128 h, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, h;\n\t"
      "selp.u32 %1, 1, 0, p;\n\t"
      "mov.u32 %0, 0;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %0, h;\n\t}"
      : "=r"(x), "=r"(ok) : "r"(answer_smem) : "memory");
  return ok ? (int)x : -1;
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor core
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]. The MMA touches no memory the
// compiler tracks, so the statement carries no memory clobber (a clobber
// would force reloads around every MMA on the single issuing thread); volatile
// asm statements keep their order relative to the barrier and commit ones.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Arrive once on the mbarrier when every tcgen05 operation this thread has
// issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}

// Warp-wide forms of the three calls above: every lane of the warp executes
// the call (with the same operands), and elect.sync picks the one lane that
// issues the instruction. Running the issuing loop convergently on the whole
// warp, rather than on one lane under a lane-dependent branch, keeps the
// issue cost per instruction below the tensor pipe's time for an N = 64
// product (measured on GB300: a stream of S and P V products at d = 64 took
// 1312 cycles per entry issued from one lane, 1037 warp-wide, against 1024
// cycles of tensor work).
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
      :: "r"(bar) : "memory");
}

// The same calls with the issuing form chosen at compile time: the whole
// warp (W = true, the _w forms and warp-collective waits) or one lane.
template <bool W>
__device__ __forceinline__ void mma_ss_t(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  if constexpr (W) mma_ss_w(d_tmem, a_desc, b_desc, idesc, accumulate);
  else mma_ss(d_tmem, a_desc, b_desc, idesc, accumulate);
}
template <bool W>
__device__ __forceinline__ void mma_ts_t(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  if constexpr (W) mma_ts_w(d_tmem, a_tmem, b_desc, idesc, accumulate);
  else mma_ts(d_tmem, a_tmem, b_desc, idesc, accumulate);
}
template <bool W>
__device__ __forceinline__ void mma_commit_t(uint32_t bar) {
  if constexpr (W) mma_commit_w(bar);
  else mma_commit(bar);
}

// Instruction descriptor of kind::f16 with bf16 A and B and an fp32
// accumulator. Bit fields: [4,6) D format (1 = f32), [7,10) A format
// (1 = bf16), [10,13) B format (1 = bf16), bit 15 A major (1 = MN-major),
// bit 16 B major, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The same with A and B of one 16-bit type: bf16 (format 1) or fp16 (format 0).
template <bool F16>
__host__ __device__ constexpr uint32_t idesc_16(int M, int N, bool a_mn, bool b_mn) {
  return F16 ? (idesc_bf16(M, N, a_mn, b_mn) & ~((7u << 7) | (7u << 10))) : idesc_bf16(M, N, a_mn, b_mn);
}

// Shared-memory matrix descriptor, 128-byte swizzle. Fields: [0,14) start
// address >> 4, [16,30) leading byte offset >> 4, [32,46) stride byte offset
// >> 4, [46,48) = 1 (descriptor version), [49,52) base offset (0: every
// swizzle atom here is 1024-byte aligned), [61,64) layout (2 = 128B swizzle).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Operand tiles here are always 128 rows (or 128 K-rows) with the inner
// dimension split in 64-element (128-byte) swizzle atoms stored 16 KB apart,
// exactly as TMA writes a [128 x 64] bf16 box with 128-byte swizzling.
//
// K-major operand (K contiguous): the k-th 16-element step lives in atom
// k / 4 at byte offset 32 * (k % 4); 8-row groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kstep) {
  return sdesc_sw128(tile + (uint32_t)(kstep >> 2) * 16384u + (uint32_t)(kstep & 3) * 32u, 16u, 1024u);
}

// MN-major operand (M or N contiguous, K-rows 128 bytes apart): the k-th
// 16-row step starts 2048 bytes further; 64-wide MN chunks are 16 KB apart
// (leading byte offset), 8-row K groups 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kstep) {
  return sdesc_sw128(tile + (uint32_t)kstep * 2048u, 16384u, 1024u);
}

// The same two layouts for tiles whose 64-element atoms are `atom` bytes
// apart (8 KB for a 64-row tile as TMA writes a [64 x 64] box): K-major with
// the k-th step in atom k / 4; MN-major with 64-wide MN chunks `atom` apart.
__device__ __forceinline__ uint64_t desc_kmajor_at(uint32_t tile, int kstep, uint32_t atom) {
  return sdesc_sw128(tile + (uint32_t)(kstep >> 2) * atom + (uint32_t)(kstep & 3) * 32u, 16u, 1024u);
}
__device__ __forceinline__ uint64_t desc_mnmajor_at(uint32_t tile, int kstep, uint32_t atom) {
  return sdesc_sw128(tile + (uint32_t)kstep * 2048u, atom, 1024u);
}

// Per-step descriptor increments (in the 16-byte units of the address
// field) for the layouts above, so that a loop can add a constant to a base
// descriptor computed once: K-major step k -> atom k / 4 (16 KB) plus 32 bytes
// per step inside the atom; MN-major step k -> 2048 bytes.
__host__ __device__ constexpr uint64_t kmajor_step(int kstep) {
  return (uint64_t)((kstep >> 2) * 1024 + (kstep & 3) * 2);
}
__host__ __device__ constexpr uint64_t mnmajor_step(int kstep) { return (uint64_t)(kstep * 128); }

// TMEM loads/stores: 32 lanes x 32 bits, 32 consecutive columns per thread.
#define FA_R32(a) a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7], a[8], a[9], a[10], a[11], \
  a[12], a[13], a[14], a[15], a[16], a[17], a[18], a[19], a[20], a[21], a[22], a[23], a[24], \
  a[25], a[26], a[27], a[28], a[29], a[30], a[31]

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Wait for this thread's outstanding TMEM loads. The registers are passed
// through so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :: "memory");
}

__device__ __forceinline__ void tmem_ld_wait_only() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
         "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
         "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
         "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
         "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
         "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
         "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Warpgroup register reallocation: every warp of a warpgroup executes the
// same one. The counts of a kernel must add up to at most the registers it
// was launched with (threads x registers per thread at launch).
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(N));
}

// ---------------------------------------------------------------------------
// arithmetic helpers
// ---------------------------------------------------------------------------

// max of three (the three-input form of PTX max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two floats -> one 32-bit word of the kernel's 16-bit element type (low half
// = first element), round to nearest even.
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return F16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

// One 32-bit word of two 16-bit elements -> two floats (exact).
template <bool F16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if (F16) {
    float2 r;
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(r.x), "=f"(r.y) : "r"(w));
    return r;
  }
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers:
// as easy as 1, 2, 3", SC 2011): ten rounds of
//   (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2,
//   c <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0),
// the key growing by (W0, W1) before every round but the first.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return make_uint4(c0, c1, c2, c3);
}

// 4 x 4 transpose of 32-bit words across the four lanes of a lane quad (lane
// index s = lane mod 4): lane s holds x[j] = M[s][j] on entry and
// x[j] = M[j][s] on exit. Two butterfly rounds (lane distance 1, then 2), in
// each of which a lane swaps the two words whose index differs from its own in
// that bit. Every lane of the warp must take part.
__device__ __forceinline__ void quad_transpose(uint32_t (&x)[4], uint32_t s) {
  const bool h1 = (s & 1u) != 0u;
  uint32_t v0 = h1 ? x[0] : x[1], v1 = h1 ? x[2] : x[3];
  v0 = __shfl_xor_sync(0xFFFFFFFFu, v0, 1);
  v1 = __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
  if (h1) { x[0] = v0; x[2] = v1; } else { x[1] = v0; x[3] = v1; }
  const bool h2 = (s & 2u) != 0u;
  v0 = h2 ? x[0] : x[2];
  v1 = h2 ? x[1] : x[3];
  v0 = __shfl_xor_sync(0xFFFFFFFFu, v0, 2);
  v1 = __shfl_xor_sync(0xFFFFFFFFu, v1, 2);
  if (h2) { x[0] = v0; x[1] = v1; } else { x[2] = v0; x[3] = v1; }
}

// Byte permute (PTX prmt.b32, default mode): byte n of the result is chosen
// by nibble n of sel from the eight bytes of {b, a} (0-3: a, 4-7: b); when the
// nibble's top bit is set the chosen byte's bit 7 is copied to all 8 bits.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Keep flags of the four bytes of w, in bit 7 of each byte: set where the byte
// is >= t (1 <= t <= 255), unsigned, given c4 = (256 - t) repeated in all four
// bytes. b >= t exactly when b + (256 - t) carries out of the byte. Added
// without the top bits, the bytes cannot carry into one another, and bit 7
// of each sum byte is the carry out of the low seven bits; the carry out of
// the byte is then the majority of that carry and the two top bits.
__device__ __forceinline__ uint32_t bytes_ge_flags(uint32_t w, uint32_t c4) {
  const uint32_t s = (w & 0x7F7F7F7Fu) + (c4 & 0x7F7F7F7Fu);
  return ((w & c4) | ((w | c4) & s)) & 0x80808080u;
}

__device__ __forceinline__ void red_add_v4(float* gptr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
               :: "l"(gptr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

}  // namespace fa
