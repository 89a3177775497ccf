// Backward pass of exact attention by recomputation, for sm_103a.
//
// The method (FlashAttention milestone page (nlp-lineage), "The idea --
// Recomputation"; FlashAttention proof-of-work page, "Activation Gradient
// Recomputation"; pixelation.org article, "The Recomputation Trade-off"): keep
// only O and the per-row softmax statistics from the forward pass and
// recompute the attention blocks on chip, never storing the N x N matrix.
// The gradient algebra is the textbook one for L = sum(dO * O):
//   P = exp(scale * Q K^T - LSE), dV = P^T dO, dP = dO V^T,
//   D = rowsum(dO * O), dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q.
//
// Three launches on one stream:
//   1. fa_bwd_pre:  D = rowsum(dO * O) in fp32, LSE2 = LSE * log2(e) (+inf on
//      rows past N and on fully masked rows), dQ accumulator zeroed;
//   2. fa_bwd_main: persistent, one CTA per SM. The (128-key tile,
//      batch-head) items are handed out in order (key tiles with the most live
//      query tiles first) from a grid-wide counter, each to the first CTA
//      ready for one; a CTA loops over the live 128-query tiles of each. The Q/dO
//      ring and every barrier phase run on across items; K and V are double
//      buffered at d = 64, so that the next item's key tile loads while this
//      one's dV and dK are stored through the other buffer. TMEM holds dV and
//      dK (accumulated over the item's loop), S^T, then P^T as packed bf16 in
//      place, and dP^T, which is then reused for the dQ partial of the tile.
//      Five tcgen05 MMAs per tile pair:
//        S^T  = K Q^T          (A = K, B = Q,   both K-major)
//        dP^T = V dO^T         (A = V, B = dO,  both K-major)
//        dV  += P^T dO         (A = P^T from TMEM, B = dO MN-major)
//        dK  += dS^T Q         (A = dS^T from TMEM, B = Q MN-major)
//        dQ_i = dS K           (A = the same dS^T buffer read MN-major, B = K MN-major)
//      At d = 128 without dropout, dQ is issued as soon as dS is complete,
//      between the two halves of dK, and S^T of the next query tile after dK,
//      which leaves its Q load the longest window (the dQ partial reuses the
//      dP^T columns, so the next dP^T waits for its drain; S^T runs
//      meanwhile). At d = 64 the dQ partial has TMEM columns of its own and
//      S^T of the next tile follows dV directly, so that P of the next tile
//      is recomputed while dK, dQ and the next dP^T run; with dropout the
//      same early S^T is used at d = 128 too (dS^T then packed over the
//      consumed dP^T columns).
//      Each dQ partial is drained from TMEM into shared memory (the dO ring
//      slot of its own query tile, dead once dQ is issued, in two rounds) and
//      added into the fp32 workspace with TMA reduce-add, so L2 receives whole
//      128-byte lines. Q and the row statistics have their own barrier and are
//      refilled as soon as dK has read Q; dO only after the reductions have
//      read the slot.
//      Warps (BwdWarps): without dropout 0-3 and 4-7 recompute P and dS for
//      query columns 0-63 and 64-127 (thread = key row), 8-11 drain dQ from
//      TMEM into the workspace (thread = query row), 12 TMA producer, 13 MMA,
//      14-15 idle (their warpgroup hands its registers to the others); with
//      dropout four P/dS warpgroups of 32 query columns (warps 0-15), then
//      the drain (16-19), the producer (20), MMA (21) and two idle warps.
//   3. fa_bwd_dq:   dQ = bf16(scale * dQ_acc).
#include "fa_common.cuh"
#include "fa_ptx.cuh"

#include <cuda_bf16.h>

namespace fa {

namespace {

// Warp roles of the main kernel. kGroups P/dS warpgroups split each tile's
// 128 query columns (kCols each), then one warpgroup drains dQ and one holds
// the TMA producer, the MMA warp and two idle warps. Four groups of 32
// queries with dropout, where the keep bits (generator rounds) make the P/dS
// work the bound (measured on the backward main kernel: +8 % at d = 128,
// +10 % at d = 64; without dropout -6 % at d = 128 and -5 % to +1 % at
// d = 64, where two groups of more registers each do better). The registers after
// reallocation add up to what the CTA is launched with (setmaxnreg.inc
// draws on that, not on the SM): 2 groups, 512 threads launched at 128:
// 2 x 128 x 160 + 128 x 96 + 128 x 96 = 512 x 128; 4 groups, 768 threads
// launched at 80: 4 x 128 x 88 + 128 x 72 + 128 x 56 = 768 x 80.
template <int D, bool DROP>
struct BwdWarps {
  static constexpr int kGroups = DROP ? 4 : 2;
  static constexpr int kCols = kTile / kGroups;
  static constexpr int kThreads = 128 * (kGroups + 2);
  static constexpr int kDrainWarp0 = 4 * kGroups;
  static constexpr int kProducerWarp = kDrainWarp0 + 4;
  static constexpr int kMmaWarp = kProducerWarp + 1;
  static constexpr int kComputeRegs = kGroups == 2 ? 160 : 88;
  static constexpr int kDrainRegs = kGroups == 2 ? 96 : 72;
  static constexpr int kOtherRegs = kGroups == 2 ? 96 : 56;
  static_assert(128 * (kGroups * kComputeRegs + kDrainRegs + kOtherRegs) ==
                    kThreads * (kGroups == 2 ? 128 : 80),
                "the reallocated registers must add up to the launch allocation");
};

template <int D>
struct BwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kHalves = D / 64;
  static constexpr int kStages = (D == 64) ? 3 : 2;   // Q/dO ring depth (smem-limited at d = 128)
  static constexpr int kKV = (D == 64) ? 2 : 1;        // K/V buffers (a second one fits at d = 64)
  static constexpr int kKVBytes = 2 * kTileBytes;
  static constexpr int kK = 0;                                // [kKV] buffers of K then V
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kKV * kKVBytes;                   // [stages]
  static constexpr int kdO = kQ + kStages * kTileBytes;       // [stages]
  static constexpr int kdS = kdO + kStages * kTileBytes;      // 128 x 128 bf16
  static constexpr int kRow = kdS + kTile * kTile * 2;        // [stages] x (LSE2[128], D[128])
  static constexpr int kBar = kRow + kStages * 2 * kTile * 4;
  static constexpr int bKV = 0;                            // [kKV]
  static constexpr int bQFull = bKV + kKV;
  static constexpr int bQEmpty = bQFull + kStages;
  static constexpr int bdOFull = bQEmpty + kStages;        // [stages]
  static constexpr int bdOFree = bdOFull + kStages;        // [stages]: dQ staging read by TMA (1 arrival, 4 per warp at d = 128)
  static constexpr int bSFull = bdOFree + kStages;
  static constexpr int bPFull = bSFull + 1;
  static constexpr int bdPFull = bPFull + 1;
  static constexpr int bdSFull = bdPFull + 1;
  static constexpr int bdSEmpty = bdSFull + 1;
  static constexpr int bdQFull = bdSEmpty + 1;
  static constexpr int bdQFree = bdQFull + 1;
  static constexpr int bFinal = bdQFree + 1;
  static constexpr int bDrain = bFinal + 1;
  static constexpr int bKVFree = bDrain + 1;   // [kKV]: the epilogue's staging has been read (2 arrivals)
  // work items reach the other roles through a ring filled by the producer
  static constexpr int kItemRing = 4;
  static constexpr int bItemFull = bKVFree + kKV;            // [kItemRing]
  static constexpr int bItemEmpty = bItemFull + kItemRing;   // [kItemRing]: MMA warp, compute and drain warps
  static constexpr int bdSHalf = bItemEmpty + kItemRing;     // the first 32 dS^T columns of each warpgroup
  static constexpr int kNumBars = bdSHalf + 1;
  static constexpr int kMisc = kBar + 8 * kNumBars;   // tmem slot, abort flag, -, wait limit
  static constexpr int kRing = kMisc + 16;                    // [kItemRing] x {key tile, batch-head, key length, -}
  static constexpr int kSmemBytes = kRing + 16 * kItemRing;
  // the dQ partial is drained per warp (each warp adds its own 32 rows) at
  // d = 128 and by the four warps together (whole 128-row boxes) at d = 64:
  // measured, each is the faster one at its width
  static constexpr bool kGroupDrain = (D == 64);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

__device__ __forceinline__ uint32_t swz_off(int r, int col) {
  // byte offset of bf16 element (row r, column col) in a 128-row tile stored
  // as 64-column halves 16 KB apart with 128-byte swizzling
  const int h = col >> 6;
  const int chunk = (col & 63) >> 3;
  return (uint32_t)(h * 16384 + (r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ (r & 7)) << 4) + ((col & 7) << 1));
}

template <int D, bool F16, bool DROP>
__global__ void __launch_bounds__(BwdWarps<D, DROP>::kThreads, 1)
fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                   const __grid_constant__ CUtensorMap tdq, const BwdParams p, const float scale) {
  using L = BwdLayout<D>;
  using W = BwdWarps<D, DROP>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int BH = p.B * p.H;
  const int Np = p.nT * kTile;
  // Work items are (key tile, batch-head) pairs, ordered group by group of
  // p.group heads (whose Q, dO and dQ accumulator fit in L2 together) and,
  // within a group, low key tiles (the most live query tiles) first. A CTA
  // starts with item blockIdx.x and then takes the next unclaimed one from a
  // grid-wide counter (zeroed by the pre-pass), so that items are handed out
  // in order, each to the first CTA that is ready for one. The producer
  // decodes each item once and hands it to the other roles through the ring.
  const int total = p.nT * BH;
  struct Item {
    int kj, bh, kvl;   // key tile, batch-head, key length of the batch entry
  };
  auto item_at = [&](int item) -> Item {
    Item w;
    w.kj = split_grouped(item, p.group, p.nT, BH, &w.bh);
    w.kvl = effective_kv_len(p.kv_len, w.bh / p.H, p.N);
    return w;
  };

  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * (uint32_t)i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = misc + 1;
  // live query tiles of an item's key tile, visited in ascending order by every role
  auto next_live = [&](const Item& w, int i) -> int {
    while (i < p.nT && tile_state(i, w.kj, w.kvl, p.nT, p.causal, p.block_mask) == kSkip) ++i;
    return i;
  };
  Ctl ctl{p.err, abort_flag};
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::kRing);
  // item k of this CTA from the ring; kj < 0 when none is left or a wait
  // failed (then ok is false too)
  auto take_item = [&](int k, bool warp_wide, bool& ok) -> Item {
    const int rs = k % L::kItemRing;
    const uint32_t ph = (uint32_t)(k / L::kItemRing) & 1u;
    ok = warp_wide ? mbar_wait_warp(bar(L::bItemFull + rs), ph, ctl, 105)
                   : mbar_wait(bar(L::bItemFull + rs), ph, ctl, 105);
    if (!ok) return Item{-1, 0, 0};
    const Item w{ring[4 * rs], ring[4 * rs + 1], ring[4 * rs + 2]};
    if (warp_wide)
      mbar_arrive_warp(bar(L::bItemEmpty + rs));
    else
      mbar_arrive(bar(L::bItemEmpty + rs));
    return w;
  };

  if ((sbase & 1023u) != 0u) {   // uniform across the CTA: nothing has started yet
    if (tid == 0) {
      uint32_t dummy = 0;   // report_error writes only the abort flag
      Ctl c0{p.err, &dummy};
      report_error(c0, kErrSmemAlign, 100);
    }
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < L::kNumBars; ++i)
      mbar_init(bar(i), (i == L::bPFull || i == L::bdSFull || i == L::bdSHalf) ? (uint32_t)(4 * W::kGroups)
                        : i == L::bdQFree ? 4u                                       // the four drain warps
                        : (i >= L::bKVFree && i < L::bKVFree + L::kKV) ? (uint32_t)W::kGroups   // one thread per compute group
                        : (!L::kGroupDrain && i >= L::bdOFree && i < L::bdOFree + L::kStages) ? 4u   // the drain warps
                        : (i >= L::bItemEmpty && i < L::bItemEmpty + L::kItemRing)
                            ? (uint32_t)(1 + 4 * W::kGroups + 4) : 1u);   // arrivals: MMA, compute and drain warps
    abort_flag[0] = 0u;
    abort_flag[2] = p.chk.wait_us;   // the wait limit, read by the slow path of every wait
    fence_mbar_init();
  }
  if (warp == W::kMmaWarp) {
    tmem_alloc(smem_u32(misc), 512);
    tmem_relinquish();
  }
  // global memory is read and written only from here on: what the pre-pass
  // wrote (row statistics, zeroed accumulator and work counter) is visible
  grid_dep_wait();
  grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = misc[0];
  const uint32_t tdV = tmem;
  const uint32_t tdK = tmem + (uint32_t)D;
  const uint32_t tS = tmem + 2u * D;
  const uint32_t tP = tmem + 2u * D + 128u;   // dP^T (and at d = 128 then the dQ partial)
  // At d = 64 the dQ partial has 64 columns of its own (2d + 256 + d <= 512),
  // which allows a schedule where nothing waits for its drain (see the MMA
  // issuer); at d = 128 it reuses the dP^T columns.
  constexpr bool kOwnDQ = (D == 64);
  constexpr bool kSplitDS = (D == 128) && W::kGroups == 2;   // dS^T handed to dK in two halves
  const uint32_t tQ = kOwnDQ ? tmem + 2u * D + 256u : tP;
  // S^T of the next tile right behind dV (before dK) at d = 64, and at d = 128
  // with dropout, where the P/dS warps bound the kernel and the next P then
  // overlaps dK and dQ (measured: +2 % there, -2.5 % at d = 128 without
  // dropout, where the dQ drain then sits in front of the next dP^T)
  constexpr bool kEarlyS = kOwnDQ || DROP;
  // dS^T for dK: packed over the consumed dP^T columns when the next S^T is
  // issued before dK (dQ, which reuses those columns at d = 128, is issued
  // after dK, and the tensor pipe runs in issue order), else into the S
  // columns next to P^T
  const uint32_t tDS = kEarlyS ? tP : tS + (uint32_t)(W::kCols / 2);
  // TMEM column of K step ks (16 queries) of the packed P^T / dS^T: each
  // warpgroup packs its kCols queries into the first kCols / 2 of its own
  // kCols S (or dP^T) columns
  auto packed_col = [](int ks) -> uint32_t {
    constexpr int kSteps = W::kCols / 16;   // K steps per warpgroup
    return (uint32_t)(W::kCols * (ks / kSteps) + 8 * (ks % kSteps));
  };

  // Every role walks the same items in the same order and counts the live
  // query tiles it has passed over all of them (g): ring slots and barrier
  // phases follow g, so the pipeline runs on across item boundaries.
  if (warp >= W::kProducerWarp) regs_dec<W::kOtherRegs>();
  if (warp == W::kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tq);
      tma_prefetch_map(&tk);
      tma_prefetch_map(&tv);
      tma_prefetch_map(&tdo);
      int nq = 0, nd = 0, nkv = 0;
      // K and V of item k into buffer k % kKV, once the epilogue of the item
      // that used the buffer before has been read out of it; a key tile with
      // no live query tile loads nothing (its epilogue stores zeros)
      auto load_kv = [&](int k, const Item& w, bool live) -> bool {
        const int kb = k % L::kKV;
        if (k >= L::kKV && !mbar_wait(bar(L::bKVFree + kb), (uint32_t)(k / L::kKV - 1) & 1u, ctl, 103)) return false;
        if (live) {
          mbar_arrive_expect_tx(bar(L::bKV + kb), 2u * L::kTileBytes);
          for (int h = 0; h < L::kHalves; ++h) {
            tma_load_3d(sbase + L::kK + kb * L::kKVBytes + h * 16384, &tk, bar(L::bKV + kb), 64 * h, kTile * w.kj, w.bh);
            tma_load_3d(sbase + L::kV + kb * L::kKVBytes + h * 16384, &tv, bar(L::bKV + kb), 64 * h, kTile * w.kj, w.bh);
          }
        } else {
          mbar_arrive(bar(L::bKV + kb));
        }
        ++nkv;
        return true;
      };
      bool ok = true;
      int g = 0;
      for (int k = 0; ok; ++k) {
        // claim the next item and hand it to the other roles
        const int rs = k % L::kItemRing;
        if (k >= L::kItemRing &&
            !(ok = mbar_wait(bar(L::bItemEmpty + rs), (uint32_t)(k / L::kItemRing - 1) & 1u, ctl, 104)))
          break;
        const int item = k == 0 ? (int)blockIdx.x : (int)gridDim.x + (int)atomicAdd(p.sched, 1u);
        const bool more = item < total;
        const Item w = more ? item_at(item) : Item{-1, 0, 0};
        ring[4 * rs] = w.kj;
        ring[4 * rs + 1] = w.bh;
        ring[4 * rs + 2] = w.kvl;
        mbar_arrive(bar(L::bItemFull + rs));   // (release: the ring entry is visible to the waiters)
        if (!more) break;
        int i = next_live(w, 0);
        if (i >= p.nT) {
          ok = load_kv(k, w, false);
          continue;
        }
        for (int it = 0; i < p.nT; ++it, ++g, i = next_live(w, i + 1)) {
          if (p.chk.stall != 0u && g >= 1) { ok = false; break; }   // test of the timeout path: Q of tile 1 never comes
          const int s = g % L::kStages;
          const uint32_t n = (uint32_t)(g / L::kStages);
          // Q and the row statistics once dK has read the slot's Q; dO once the
          // dQ partial staged in the slot's dO buffer has been read
          if (g >= L::kStages && !(ok = mbar_wait(bar(L::bQEmpty + s), (n - 1) & 1u, ctl, 101))) break;
          mbar_arrive_expect_tx(bar(L::bQFull + s), L::kTileBytes + 2u * kTile * 4u);
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sbase + L::kQ + s * L::kTileBytes + h * 16384, &tq, bar(L::bQFull + s),
                        64 * h, kTile * i, w.bh);
          const size_t roff = (size_t)w.bh * Np + (size_t)kTile * i;
          bulk_load(sbase + L::kRow + s * 1024, p.lse2 + roff, kTile * 4, bar(L::bQFull + s));
          bulk_load(sbase + L::kRow + s * 1024 + 512, p.delta + roff, kTile * 4, bar(L::bQFull + s));
          ++nq;
          if (g >= L::kStages && !(ok = mbar_wait(bar(L::bdOFree + s), (n - 1) & 1u, ctl, 102))) break;
          mbar_arrive_expect_tx(bar(L::bdOFull + s), L::kTileBytes);
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sbase + L::kdO + s * L::kTileBytes + h * 16384, &tdo, bar(L::bdOFull + s),
                        64 * h, kTile * i, w.bh);
          ++nd;
          // K and V behind the first query tile of the item, whose loads only
          // wait for ring slots of the previous item
          if (it == 0 && !(ok = load_kv(k, w, true))) break;
        }
      }
      // every load issued has landed before the CTA exits
      for (int kb = 0; kb < L::kKV && kb < nkv; ++kb)
        drain_wait(bar(L::bKV + kb), (uint32_t)((nkv - 1 - kb) / L::kKV) & 1u);
      for (int s = 0; s < L::kStages; ++s) {
        if (s < nq) drain_wait(bar(L::bQFull + s), (uint32_t)((nq - 1 - s) / L::kStages) & 1u);
        if (s < nd) drain_wait(bar(L::bdOFull + s), (uint32_t)((nd - 1 - s) / L::kStages) & 1u);
      }
    }
  } else if (warp == W::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // At d = 128, and at d = 64 with dropout, the whole warp runs the schedule
    // and one elected lane issues each MMA and commit; at d = 64 without
    // dropout one lane runs it (measured: the warp-wide form is 1.5 % faster at
    // d = 128, 4 % faster at d = 64 with dropout, and between 4 % slower and
    // 1 % faster on the d = 64 workloads without dropout).
    constexpr bool kW = (D == 128) || DROP;
    if (kW || lane == 0) {
      constexpr uint32_t idSP = idesc_16<F16>(128, 128, false, false);
      constexpr uint32_t idV = idesc_16<F16>(128, D, false, true);
      constexpr uint32_t idK = idesc_16<F16>(128, D, false, true);
      constexpr uint32_t idQ = idesc_16<F16>(128, D, true, true);
      const uint32_t sdS = sbase + L::kdS;
      bool ok = true;
      int g = 0;
      // Shared-memory descriptors are built as a base plus a constant step per
      // K step wherever that keeps within the MMA thread's registers, so that
      // issuing an MMA costs the thread one 64-bit add.
      // S^T = K Q^T of running query tile g
      auto issue_s = [&](uint32_t sK, int g1) -> bool {
        const int s1 = g1 % L::kStages;
        if (!mbar_wait_t<kW>(bar(L::bQFull + s1), (uint32_t)(g1 / L::kStages) & 1u, ctl, 114)) return false;
        tc_fence_after();
        const uint64_t dK0 = desc_kmajor(sK, 0), dQ0 = desc_kmajor(sbase + L::kQ + s1 * L::kTileBytes, 0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss_t<kW>(tS, dK0 + kmajor_step(ks), dQ0 + kmajor_step(ks), idSP, ks > 0 ? 1u : 0u);
        mma_commit_t<kW>(bar(L::bSFull));
        return true;
      };
      for (int k = 0; ok; ++k) {
        const Item w = take_item(k, kW, ok);
        if (w.kj < 0) break;
        int i = next_live(w, 0);
        if (i >= p.nT) continue;
        const int kb = k % L::kKV;
        const uint32_t sK = sbase + L::kK + kb * L::kKVBytes, sV = sbase + L::kV + kb * L::kKVBytes;
        const uint64_t mK = desc_mnmajor(sK, 0);
        if (!(ok = mbar_wait_t<kW>(bar(L::bKV + kb), (uint32_t)(k / L::kKV) & 1u, ctl, 110))) break;
        if (!(ok = issue_s(sK, g))) break;
        for (int it = 0; i < p.nT; ++it, ++g) {
          const int inext = next_live(w, i + 1);
          const int s = g % L::kStages;
          const uint32_t sQ = sbase + L::kQ + s * L::kTileBytes;
          const uint32_t sdO = sbase + L::kdO + s * L::kTileBytes;
          // dP^T = V dO^T (at d = 128 the dQ partial of the previous tile must
          // have been read out of these columns)
          if (!kOwnDQ && g > 0 && !(ok = mbar_wait_t<kW>(bar(L::bdQFree), (uint32_t)(g - 1) & 1u, ctl, 112))) break;
          if (!(ok = mbar_wait_t<kW>(bar(L::bdOFull + s), (uint32_t)(g / L::kStages) & 1u, ctl, 116))) break;
          tc_fence_after();
          const uint64_t kdV = desc_kmajor(sV, 0), kdO = desc_kmajor(sdO, 0);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_ss_t<kW>(tP, kdV + kmajor_step(ks), kdO + kmajor_step(ks), idSP, ks > 0 ? 1u : 0u);
          mma_commit_t<kW>(bar(L::bdPFull));
          // dV += P^T dO (at it == 0 over the previous item's dV and dK, which
          // the compute warps have read out of TMEM before arriving on this P)
          if (!(ok = mbar_wait_t<kW>(bar(L::bPFull), (uint32_t)g & 1u, ctl, 113))) break;
          tc_fence_after();
          const uint64_t mdO = desc_mnmajor(sdO, 0);
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            // P of each warpgroup's queries packed in the first half of its own S columns
            mma_ts_t<kW>(tdV, tS + packed_col(ks), mdO + mnmajor_step(ks), idV,
                   (it > 0 || ks > 0) ? 1u : 0u);
          // next S^T of this item: early, right behind dV (the tensor pipe
          // runs in issue order, so dV has read P first), so that P of the
          // next tile is recomputed while dK, dQ and the next dP run; else
          // after dQ, which leaves the next Q load the longest window
          if (kEarlyS && inext < p.nT && !(ok = issue_s(sK, g + 1))) break;
          // dK += dS^T Q ; dQ_i = dS K. dS^T is packed like P (packed_col) from
          // tDS on; with two warpgroups, at d = 128 each
          // warpgroup hands over its first 32 queries (K steps 0, 1 and 4, 5)
          // before the rest (2, 3 and 6, 7), so half of dK runs while dS is
          // finished (measured: +1.5 % at d = 128, -0.4 to -1.2 % at d = 64)
          const uint64_t mQ = desc_mnmajor(sQ, 0);
          // dQ_i = dS K: with dS^T handed over in halves, dQ goes right after
          // dS is complete, in front of the second half of dK, so that its
          // drain overlaps that half
          auto issue_dq = [&]() {
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks)
              mma_ss_t<kW>(tQ, desc_mnmajor(sdS, ks), mK + mnmajor_step(ks), idQ, ks > 0 ? 1u : 0u);
            mma_commit_t<kW>(bar(L::bdQFull));
          };
#pragma unroll
          for (int half = kSplitDS ? 0 : 1; half < 2; ++half) {
            if (!(ok = mbar_wait_t<kW>(bar(half == 0 ? L::bdSHalf : L::bdSFull), (uint32_t)g & 1u, ctl, 115)))
              break;
            tc_fence_after();
            if (kSplitDS && half == 1) issue_dq();
#pragma unroll
            for (int k4 = 0; k4 < (kSplitDS ? 4 : 8); ++k4) {
              const int ks = kSplitDS ? 2 * half + (k4 & 1) + 4 * (k4 >> 1) : k4;
              mma_ts_t<kW>(tdK, tDS + packed_col(ks), mQ + mnmajor_step(ks), idK,
                           (it > 0 || ks > 0) ? 1u : 0u);
            }
          }
          if (!ok) break;
          mma_commit_t<kW>(bar(L::bQEmpty + s));   // the slot's Q has been read for the last time
          if (!kSplitDS) {
            // at d = 64 the previous dQ partial must have been read out of its columns
            if (kOwnDQ && g > 0 && !(ok = mbar_wait_t<kW>(bar(L::bdQFree), (uint32_t)(g - 1) & 1u, ctl, 112))) break;
            tc_fence_after();
            issue_dq();
          }
          mma_commit_t<kW>(bar(L::bdSEmpty));      // dK and dQ have read dS
          if (!kEarlyS && inext < p.nT && !(ok = issue_s(sK, g + 1))) break;
          i = inext;
        }
        if (ok) mma_commit_t<kW>(bar(L::bFinal));   // dV and dK of the item are complete
      }
      mma_commit_t<kW>(bar(L::bDrain));
      drain_wait(bar(L::bDrain), 0);
    }
  } else if (warp < W::kDrainWarp0) {
    // ------------------------------------------------------------ P and dS (thread = key row)
    // warpgroup cw handles query columns kC cw .. kC cw + kC - 1 of each tile
    regs_inc<W::kComputeRegs>();
    constexpr int kC = W::kCols;
    const int cw = warp >> 2;
    const int cb = kC * cw;
    const int r = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g = 0, nf = 0;
    int pending = -1;   // K/V buffer whose epilogue store has not been waited for yet (thread r == 0)
    // the store out of buffer `pending` has read its staging: the buffer goes
    // back to the producer
    auto release_kv = [&]() {
      if (pending >= 0) {
        if (r == 0) {
          bulk_wait_group_read_all();
          mbar_arrive(bar(L::bKVFree + pending));
        }
        pending = -1;
      }
    };
    // The four warps of a group meet at a named barrier in each item's
    // epilogue; before it, and wherever one of them may have stopped (a wait
    // that ran out or saw the abort flag), they agree with group_all, so that
    // all of them take the same branch and none waits for one that has left.
    // Where two groups share a 64-column store box of dV or dK (d = 64 with
    // four groups), all the groups meet and agree together instead.
    constexpr int kAccGroups = W::kGroups / 2;   // warpgroups per accumulator
    constexpr int kAccCols = D / kAccGroups;       // columns each stores
    constexpr bool kJoint = kAccCols < 64;
    const uint32_t gbar = kJoint ? 1u : 1u + (uint32_t)cw;
    constexpr uint32_t kGThreads = kJoint ? 128u * W::kGroups : 128u;
    for (int k = 0; ok; ++k) {
      const Item w = take_item(k, true, ok);
      ok = group_all(gbar, kGThreads, ok);
      if (!ok || w.kj < 0) break;
      const int krow = kTile * w.kj + r;
      int i = next_live(w, 0);
      const bool live = i < p.nT;
      for (int it = 0; i < p.nT; ++it, ++g, i = next_live(w, i + 1)) {
        const bool partial = tile_state(i, w.kj, w.kvl, p.nT, p.causal, p.block_mask) == kPartial;
        // dropout: keep bits of this warpgroup's kC query columns, made before
        // the waits below so that the generator runs while the tensor pipe
        // computes S^T. One generator call (counter (query block, key block,
        // bh, 0)) covers 4 queries (word d: query d of the block) and 4 keys
        // (byte k: key k); a query is kept iff its byte is >= t. The four key
        // rows of a lane quad share their calls: lane s makes the calls of
        // query blocks 4 m4 + s and files the flags of call m4, word d in bit
        // 2 m4 + d / 2 of byte k of ev (d even) or od (d odd); bytes k of ev
        // and od go to key row k of the quad, by a 4 x 4 transpose across the
        // quad. Query column c = 16 m4 + 4 j + d is then bit
        // kbase(j) + 8 (d mod 2) + 2 m4 + d / 2 of keep[kword(j)]: the two
        // queries of a pair (d, d + 1) sit 8 bits apart (see pair_mask).
        auto kword = [](int j) { return kC == 64 ? (j >> 1) : 0; };
        auto kbase = [](int j) { return kC == 64 ? 16 * (j & 1) : 16 * (j >> 1) + 4 * (j & 1); };
        uint32_t keep[kC / 32];
#pragma unroll
        for (int q = 0; q < kC / 32; ++q) keep[q] = 0u;
        if constexpr (DROP) {
          const uint32_t qb0 = 32u * (uint32_t)i + (uint32_t)(cb >> 2);
          const uint32_t s4 = (uint32_t)lane & 3u;   // = key row mod 4
          const uint32_t c4 = (256u - p.drop.t) * 0x01010101u;
          uint32_t ev = 0u, od = 0u;
#pragma unroll
          for (int m4 = 0; m4 < kC / 16; ++m4) {
            const uint4 v = philox4x32_10(qb0 + 4u * (uint32_t)m4 + s4, (uint32_t)krow >> 2, (uint32_t)w.bh, 0u,
                                          p.drop.seed_lo, p.drop.seed_hi);
            ev |= (bytes_ge_flags(v.x, c4) >> (7 - 2 * m4)) | (bytes_ge_flags(v.z, c4) >> (6 - 2 * m4));
            od |= (bytes_ge_flags(v.y, c4) >> (7 - 2 * m4)) | (bytes_ge_flags(v.w, c4) >> (6 - 2 * m4));
          }
          uint32_t x4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) x4[k] = ((ev >> (8 * k)) & 0xFFu) | (((od >> (8 * k)) & 0xFFu) << 8);
          quad_transpose(x4, s4);
#pragma unroll
          for (int j = 0; j < 4; ++j) keep[kword(j)] |= x4[j] << (kC == 64 ? 16 * (j & 1) : 16 * (j >> 1) + 4 * (j & 1));
          // the bits are complete here: the compiler may not move the generator
          // past the waits
#pragma unroll
          for (int q = 0; q < kC / 32; ++q) asm volatile("" : "+r"(keep[q]));
        }
        const int s = g % L::kStages;
        if (!(ok = mbar_wait_warp(bar(L::bQFull + s), (uint32_t)(g / L::kStages) & 1u, ctl, 120))) break;
        if (!(ok = mbar_wait_warp(bar(L::bSFull), (uint32_t)g & 1u, ctl, 121))) break;
        tc_fence_after();
        if (p.chk.rec != nullptr && tid == 0) record_tile(p.chk.rec, w.bh, i, w.kj, p.nT, partial);   // as computed
        const float* lse2 = reinterpret_cast<const float*>(smem + L::kRow + s * 1024) + cb;
        const float* dlt = lse2 + kTile;
        float x[kC];
        {
          uint32_t u0[32], u1[32];
          tmem_ld32(tS + lane_off + (uint32_t)cb, u0);
          if constexpr (kC == 64) tmem_ld32(tS + lane_off + (uint32_t)cb + 32u, u1);
          tmem_ld_wait(u0);
          if constexpr (kC == 64) tmem_ld_wait(u1);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            x[c] = __uint_as_float(u0[c]);
            if constexpr (kC == 64) x[32 + c] = __uint_as_float(u1[c]);
          }
        }
        // P^T row: p[c] = exp2(s * scale * log2e - LSE2[query c])
#pragma unroll
        for (int c4 = 0; c4 < kC / 4; ++c4) {
          const float4 l = reinterpret_cast<const float4*>(lse2)[c4];   // one broadcast load per 4 queries
          x[4 * c4] = ex2(fmaf(x[4 * c4], sl2, -l.x));
          x[4 * c4 + 1] = ex2(fmaf(x[4 * c4 + 1], sl2, -l.y));
          x[4 * c4 + 2] = ex2(fmaf(x[4 * c4 + 2], sl2, -l.z));
          x[4 * c4 + 3] = ex2(fmaf(x[4 * c4 + 3], sl2, -l.w));
        }
        if (partial) {
          // key row krow is masked for query q0 + c when it lies past the
          // query (causal: c < krow - q0) or at or past the key length (every c)
          const int lim = krow >= w.kvl ? kC : (p.causal ? krow - (kTile * i + cb) : 0);
#pragma unroll
          for (int c = 0; c < kC; ++c)
            if (c < lim) x[c] = 0.f;
        }
        auto kept = [&](int c) -> bool {
          const int j = (c >> 2) & 3, d = c & 3;
          return (keep[kword(j)] >> (kbase(j) + 8 * (d & 1) + 2 * (c >> 4) + (d >> 1))) & 1u;
        };
        // masks of the two 16-bit halves of the packed pair of queries c0, c0 + 1
        // (c0 even): their bits, shifted to bit 7 of two bytes, are replicated
        // by prmt over the bytes of each half
        auto pair_mask = [&](int c0) -> uint32_t {
          const int j = (c0 >> 2) & 3, b0 = kbase(j) >> 3;
          const int pos = (kbase(j) & 7) + 2 * (c0 >> 4) + ((c0 & 3) >> 1);
          return prmt(keep[kword(j)] << (7 - pos), 0u, (uint32_t)((8 + b0) * 0x11 + (9 + b0) * 0x1100));
        };
        // the dV operand is the dropped P (P * Z; the keep scale, the same for
        // every kept term, is applied to dV in the epilogue), packed two
        // queries per TMEM column into the first half of this warpgroup's own
        // S columns (the other warpgroup may still be reading its half)
        {
          uint32_t pk[kC / 2];
#pragma unroll
          for (int c = 0; c < kC / 2; ++c) {
            pk[c] = pack2<F16>(x[2 * c], x[2 * c + 1]);
            if constexpr (DROP) pk[c] &= pair_mask(2 * c);
          }
          if constexpr (kC == 64) tmem_st32(tS + lane_off + (uint32_t)cb, pk);
          else tmem_st16(tS + lane_off + (uint32_t)cb, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(bar(L::bPFull));
        if (it == 0) release_kv();   // the previous item's store has had this tile's time to read its staging

        // dS^T row: ds[c] = p[c] * (dP[c] - D[query c]) -> 16-bit -> swizzled smem
        if (!(ok = mbar_wait_warp(bar(L::bdPFull), (uint32_t)g & 1u, ctl, 122))) break;
        if (g > 0 && !(ok = mbar_wait_warp(bar(L::bdSEmpty), (uint32_t)(g - 1) & 1u, ctl, 123))) break;
        tc_fence_after();
        // at d = 128 both 32-column halves of this warpgroup's dP^T are loaded
        // before the first wait, so their TMEM latencies overlap (measured:
        // +0.9 % on the backward at d = 128; at d = 64 the 32 extra live
        // registers spill and it lost 3.5 %)
        constexpr bool kBothHalves = (D == 128);
        uint32_t ud[kC / 32][32];
        if constexpr (kBothHalves) {
#pragma unroll
          for (int cc = 0; cc < kC / 32; ++cc) tmem_ld32(tP + lane_off + (uint32_t)cb + 32u * cc, ud[cc]);
#pragma unroll
          for (int cc = 0; cc < kC / 32; ++cc) tmem_ld_wait(ud[cc]);
        }
#pragma unroll
        for (int cc = 0; cc < kC / 32; ++cc) {
          if constexpr (!kBothHalves) {
            tmem_ld32(tP + lane_off + (uint32_t)cb + 32u * cc, ud[cc]);
            tmem_ld_wait(ud[cc]);
          }
          const uint32_t* u = ud[cc];
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int c0 = 32 * cc + 2 * c;
            float g0 = __uint_as_float(u[2 * c]), g1 = __uint_as_float(u[2 * c + 1]);
            const float2 dl = reinterpret_cast<const float2*>(dlt)[c0 >> 1];
            float d0, d1;
            if constexpr (DROP) {   // dP = (dO V^T) * Z * keep_scale
              g0 = kept(c0) ? g0 : 0.f;
              g1 = kept(c0 + 1) ? g1 : 0.f;
              d0 = x[c0] * fmaf(g0, p.drop.keep_scale, -dl.x);
              d1 = x[c0 + 1] * fmaf(g1, p.drop.keep_scale, -dl.y);
            } else {
              d0 = x[c0] * (g0 - dl.x);
              d1 = x[c0 + 1] * (g1 - dl.y);
            }
            pk[c] = pack2<F16>(d0, d1);
          }
          // dS^T also goes to TMEM (the A operand of dK), packed (tDS): over
          // this warpgroup's dP columns, which it has already read, or into the
          // second half of its S columns, after its P
          tmem_st16(tDS + lane_off + (uint32_t)cb + 16u * cc, pk);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            uint8_t* dst = smem + L::kdS + swz_off(r, cb + 32 * cc + 8 * k4);
            *reinterpret_cast<uint4*>(dst) =
                make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
          }
          if (kSplitDS && cc == 0) {   // the first 32 queries' dS^T is in TMEM: dK may start on them
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(bar(L::bdSHalf));
          }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive_warp(bar(L::bdSFull));
      }

      // epilogue: the first half of the warpgroups store dV, the second half
      // scale * dK (each its share of the columns), for every key row of the
      // tile (zeros when no query tile was live), staged in the item's V or K
      // buffer once every MMA has read it, and stored by TMA
      ok = group_all(gbar, kGThreads, ok);
      if (!ok) break;
      release_kv();   // the buffer of an earlier item without live query tiles
      const int kb = k % L::kKV;
      ok = mbar_wait_warp(bar(L::bKV + kb), (uint32_t)(k / L::kKV) & 1u, ctl, 124);
      if (ok && live) ok = mbar_wait_warp(bar(L::bFinal), (uint32_t)nf & 1u, ctl, 125);
      ok = group_all(gbar, kGThreads, ok);
      if (!ok) break;
      nf += live ? 1 : 0;
      tc_fence_after();
      const bool is_v = cw < kAccGroups;
      const int col0 = kAccCols * (cw % kAccGroups);
      const uint32_t tacc = (is_v ? tdV : tdK) + lane_off + (uint32_t)col0;
      const float mul = is_v ? (DROP ? p.drop.keep_scale : 1.f) : scale;
      const int stage_off = (is_v ? L::kV : L::kK) + kb * L::kKVBytes;
      uint8_t* stage = smem + stage_off;
#pragma unroll
      for (int cc = 0; cc < kAccCols / 32; ++cc) {
        uint32_t u[32];
        if (live) {
          tmem_ld32(tacc + 32u * cc, u);
          tmem_ld_wait(u);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) u[c] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack2<F16>(__uint_as_float(u[2 * c]) * mul, __uint_as_float(u[2 * c + 1]) * mul);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          uint8_t* dst = stage + swz_off(r, col0 + 32 * cc + 8 * k4);
          *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      named_bar_sync(gbar, kGThreads);
      if (r == 0 && col0 % 64 == 0) {   // a shared box: its first group stores it
        for (int h = col0 / 64; h < (col0 + (kJoint ? 64 : kAccCols)) / 64; ++h)
          tma_store_3d(is_v ? &tdv : &tdk, sbase + stage_off + h * 16384, 64 * h, kTile * w.kj, w.bh);
        bulk_commit_group();
      }
      pending = kb;
      // with one K/V buffer the next item's K and V wait for this store
      if (L::kKV == 1) release_kv();
    }
    if (r == 0) bulk_wait_group_read_all();   // the stores have read the staging; the grid's end makes them visible
  } else if (warp < W::kProducerWarp) {
    // ------------------------------------------------------------ dQ drain (thread = query row)
    // TMEM -> fp32 rows staged in this iteration's dO ring slot (dead once dQ
    // has completed) in two rounds of 32-column boxes, 128-byte swizzled ->
    // TMA reduce-add into the accumulator. The TMEM columns are released as
    // soon as they are all in registers or staged; the slot goes back to the
    // producer when its last round has been read.
    //   d = 128: each warp stages and adds its own 32 query rows (boxes of 32
    //            rows) and synchronises only within itself.
    //   d = 64:  the four warps stage whole 128-row boxes that one thread adds,
    //            meeting at named barriers; after each wait that one of them
    //            may fail they agree with group_all, so that they always take
    //            the same branch and none waits at a barrier another has left.
    regs_dec<W::kDrainRegs>();
    constexpr uint32_t kDrainBar = 1u + W::kGroups;   // named barrier of the drain warps (d = 64)
    constexpr int kBoxesPerRound = L::kTileBytes / 16384;    // 1 (d = 64) or 2 (d = 128)
    constexpr int kRounds = D / 32 / kBoxesPerRound;
    const int r = tid - 32 * W::kDrainWarp0;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t sw = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);
    const uint32_t wrow = L::kGroupDrain ? 0u : 4096u * (uint32_t)(warp & 3);   // this warp's rows in a box
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      const Item w = take_item(k, true, ok);
      if constexpr (L::kGroupDrain) ok = group_all(kDrainBar, 128, ok);
      if (!ok || w.kj < 0) break;
      for (int i = next_live(w, 0); i < p.nT; ++g, i = next_live(w, i + 1)) {
        const int s = g % L::kStages;
        const uint32_t stage = (uint32_t)(L::kdO + s * L::kTileBytes);
        ok = mbar_wait_warp(bar(L::bdQFull), (uint32_t)g & 1u, ctl, 130);
        if constexpr (L::kGroupDrain) ok = group_all(kDrainBar, 128, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t u[kBoxesPerRound][32];
#pragma unroll
        for (int b = 0; b < kBoxesPerRound; ++b) tmem_ld32(tQ + lane_off + 32u * b, u[b]);
#pragma unroll
        for (int b = 0; b < kBoxesPerRound; ++b) tmem_ld_wait(u[b]);
#pragma unroll
        for (int round = 0; round < kRounds; ++round) {
          if (round == kRounds - 1) {
            tc_fence_before();
            mbar_arrive_warp(bar(L::bdQFree));   // every dQ column is in registers or staged
          }
          if (round > 0) {              // the previous round has been read out of the slot
            if constexpr (L::kGroupDrain) {
              if (r == 0) bulk_wait_group_read_all();
              named_bar_sync(kDrainBar, 128);
            } else {
              if (lane == 0) bulk_wait_group_read_all();
              __syncwarp();
            }
          }
#pragma unroll
          for (int b = 0; b < kBoxesPerRound; ++b)
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {    // 8 chunks of 4 fp32 per 32-column box
              const uint32_t o = sw + (uint32_t)((k8 ^ (r & 7)) << 4);
              *reinterpret_cast<uint4*>(smem + stage + 16384 * b + o) =
                  make_uint4(u[b][4 * k8], u[b][4 * k8 + 1], u[b][4 * k8 + 2], u[b][4 * k8 + 3]);
            }
          fence_proxy_async_smem();
          if constexpr (L::kGroupDrain)
            named_bar_sync(kDrainBar, 128);
          else
            __syncwarp();
          if (L::kGroupDrain ? r == 0 : lane == 0) {
            const int row0 = kTile * i + (L::kGroupDrain ? 0 : 32 * (warp & 3));
#pragma unroll
            for (int b = 0; b < kBoxesPerRound; ++b)
              if (32 * (round * kBoxesPerRound + b) < p.d)   // boxes wholly past the head dimension hold zeros
                tma_reduce_add_3d(&tdq, sbase + stage + 16384u * b + wrow, 32 * (round * kBoxesPerRound + b),
                                  row0, w.bh);
            bulk_commit_group();
          }
          if (round + 1 < kRounds) {    // the next columns into registers while the round is read
#pragma unroll
            for (int b = 0; b < kBoxesPerRound; ++b)
              tmem_ld32(tQ + lane_off + 32u * ((round + 1) * kBoxesPerRound + b), u[b]);
#pragma unroll
            for (int b = 0; b < kBoxesPerRound; ++b) tmem_ld_wait(u[b]);
          }
        }
        if (L::kGroupDrain ? r == 0 : lane == 0) {
          bulk_wait_group_read_all();
          mbar_arrive(bar(L::bdOFree + s));
        }
      }
    }
    if (L::kGroupDrain ? r == 0 : lane == 0) bulk_wait_group_all();     // reductions complete before exit
  }

  tc_fence_before();
  __syncthreads();
  if (warp == W::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// D = rowsum(dO * O) (fp32), LSE2 = LSE * log2(e) with +inf for -inf and
// padding rows, dQ accumulator and the main kernel's work counter zeroed. A group of G threads per row (G the
// power of two >= d / 8); thread `part` owns columns 8 part .. 8 part + 7 when
// 8 part < d.
template <int G, bool F16>
__global__ void fa_bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                  const float* __restrict__ lse, float* __restrict__ dq_acc,
                                  float* __restrict__ lse2, float* __restrict__ delta,
                                  unsigned int* __restrict__ sched, int BH, int N, int Np, int d) {
  grid_dep_wait();   // O and LSE of the forward kernel are complete
  grid_dep_launch();
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid == 0) *sched = 0u;
  const long long row = gid / G;           // over BH * Np
  const int part = (int)(gid % G);
  if (row >= (long long)BH * Np) return;   // whole groups leave together (G divides the block)
  const int bh = (int)(row / Np);
  const int n = (int)(row % Np);
  const bool mine = 8 * part < d;
  float acc = 0.f;
  if (n < N && mine) {
    const size_t off = ((size_t)bh * N + n) * d + part * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(o + off);
    const uint4 g = *reinterpret_cast<const uint4*>(dout + off);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 af = unpack2<F16>(aw[k]);
      const float2 gf = unpack2<F16>(gw[k]);
      acc = fmaf(af.x, gf.x, acc);
      acc = fmaf(af.y, gf.y, acc);
    }
  }
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (mine) {
    float4* z = reinterpret_cast<float4*>(dq_acc + (size_t)row * d + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (part == 0) {
    delta[row] = acc;
    float v = INFINITY;
    if (n < N) {
      const float l = lse[(size_t)bh * N + n];
      v = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
    }
    lse2[row] = v;
  }
}

// dQ = 16-bit(scale * dQ accumulator), one thread per 8 columns.
template <bool F16>
__global__ void fa_bwd_dq_kernel(const float* __restrict__ dq_acc, uint16_t* __restrict__ dq, float scale,
                                 int BH, int N, int Np, int d) {
  grid_dep_wait();   // every partial of the main kernel has been added
  grid_dep_launch();
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int parts = d / 8;
  const long long total = (long long)BH * N * parts;
  if (gid >= total) return;
  const long long row = gid / parts;
  const int part = (int)(gid % parts);
  const int bh = (int)(row / N);
  const int n = (int)(row % N);
  const float4* src = reinterpret_cast<const float4*>(dq_acc + ((size_t)bh * Np + n) * d + part * 8);
  const float4 a = src[0], c = src[1];
  uint4 out;
  out.x = pack2<F16>(a.x * scale, a.y * scale);
  out.y = pack2<F16>(a.z * scale, a.w * scale);
  out.z = pack2<F16>(c.x * scale, c.y * scale);
  out.w = pack2<F16>(c.z * scale, c.w * scale);
  *reinterpret_cast<uint4*>(dq + (size_t)row * d + part * 8) = out;
}

template <int D, bool F16, bool DROP>
cudaError_t launch_bwd_main_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                              const CUtensorMap& tdq, const BwdParams& p, float scale, cudaStream_t s) {
  using L = BwdLayout<D>;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static PerDeviceOnce smem_set;
  e = once_per_device(smem_set, dev, [] {
    return cudaFuncSetAttribute(fa_bwd_main_kernel<D, F16, DROP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                L::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  BwdParams q = p;
  // a head's Q and dO (16-bit) and its fp32 dQ accumulator are re-read by
  // all of its key-tile items
  q.group = l2_head_group(8.0 * p.N * p.d, p.B * p.H);
  // persistent: at most one CTA per SM (the kernel holds all of TMEM), each
  // taking (key tile, batch-head) items from the work counter
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long items = (long long)p.nT * p.B * p.H;
  const dim3 grid((unsigned)(items < sms ? items : sms));
  return launch_pdl(true, fa_bwd_main_kernel<D, F16, DROP>, grid, dim3(BwdWarps<D, DROP>::kThreads), L::kSmemBytes, s, tq, tk, tv, tdo,
                    tdk, tdv, tdq, q, scale);
}

}  // namespace

cudaError_t launch_bwd_pre(bool f16, const void* o, const void* dout, const float* lse, float* dq_acc, float* lse2,
                           float* delta, unsigned int* sched, int BH, int N, int nT, int d, cudaStream_t s) {
  const int Np = nT * kTile;
  int G = 1;
  while (G < d / 8) G <<= 1;              // 1 .. 32: divides the block and the warp
  const long long threads = (long long)BH * Np * G;
  const int block = 256;
  const unsigned grid = (unsigned)((threads + block - 1) / block);
  const uint16_t* o16 = static_cast<const uint16_t*>(o);
  const uint16_t* g16 = static_cast<const uint16_t*>(dout);
#define FA_PRE_CASE(GG)                                                                                       \
  if (G == GG)                                                                                                \
    return launch_pdl(false, f16 ? fa_bwd_pre_kernel<GG, true> : fa_bwd_pre_kernel<GG, false>, dim3(grid), dim3(block), 0, \
                      s, o16, g16, lse, dq_acc, lse2, delta, sched, BH, N, Np, d);
  FA_PRE_CASE(1)
  FA_PRE_CASE(2)
  FA_PRE_CASE(4)
  FA_PRE_CASE(8)
  FA_PRE_CASE(16)
  FA_PRE_CASE(32)
#undef FA_PRE_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_main(int d, bool f16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const CUtensorMap& tdq, const BwdParams& p, cudaStream_t s) {
  const float scale = p.scale_log2 / 1.4426950408889634f;
  const bool drop = p.drop.t > 0;
  const int kd = kernel_head_dim(d);
  if (kd == 256) return drop ? cudaErrorInvalidValue : launch_bwd_wide(f16, tq, tk, tv, tdo, tdk, tdv, tdq, p, s);
#define FA_BWD_CASE(DD, FF, DR) \
  if (kd == DD && f16 == FF && drop == DR) \
    return launch_bwd_main_d<DD, FF, DR>(tq, tk, tv, tdo, tdk, tdv, tdq, p, scale, s);
  FA_BWD_CASE(64, false, false)
  FA_BWD_CASE(128, false, false)
  FA_BWD_CASE(64, true, false)
  FA_BWD_CASE(128, true, false)
  FA_BWD_CASE(64, false, true)
  FA_BWD_CASE(128, false, true)
  FA_BWD_CASE(64, true, true)
  FA_BWD_CASE(128, true, true)
#undef FA_BWD_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dq(bool f16, const float* dq_acc, void* dq, float scale, int BH, int N, int nT, int d,
                          cudaStream_t s) {
  const int Np = nT * kTile;
  if ((long long)BH * N == 0) return cudaSuccess;
  const long long threads = (long long)BH * N * (d / 8);
  const int block = 256;
  const unsigned grid = (unsigned)((threads + block - 1) / block);
  return launch_pdl(false, f16 ? fa_bwd_dq_kernel<true> : fa_bwd_dq_kernel<false>, dim3(grid), dim3(block), 0, s, dq_acc,
                    static_cast<uint16_t*>(dq), scale, BH, N, Np, d);
}

}  // namespace fa
