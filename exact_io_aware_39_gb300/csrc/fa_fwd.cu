// Forward pass of exact attention, tile by tile with online softmax, for
// sm_103a (tcgen05 tensor cores, TMEM accumulators, TMA staging).
//
// The method (FlashAttention milestone page (nlp-lineage), "The idea -- Tiling";
// FlashAttention proof-of-work page, "SRAM Block Tiling" and "Online Softmax
// Computation"): split Q, K and V into blocks that fit on chip, stream K/V
// blocks past a resident Q block, keep a running row max m and row sum l, and
// rescale the earlier partial output when m grows, so that the result equals
// standard attention exactly. Only O and one log-sum-exp per row leave the
// chip (milestone page, "The idea -- Recomputation").
//
// GB300 design (not the pages' A100 design):
//   * a work item is a pair of 128-row Q tiles of one (batch, head); a CTA
//     (one per SM) takes items one after another: its own, then CTAs of the
//     grid that have not started, cancelled through cluster launch control;
//     12 warps:
//       warps 0-3  softmax / correction / epilogue of Q tile 0 (TMEM lanes 0-127)
//       warps 4-7  the same for Q tile 1
//       warp  8    builds each item's list of live key tiles; TMA producer of
//                  Q and of the K ring; asks for the next item and, at d = 64
//                  (two Q buffers), sets it up while the current one runs
//       warp  9    TMEM allocator; runs the MMA schedule (one lane picked by
//                  elect.sync issues each tcgen05.mma)
//       warp 10    TMA producer of the V ring
//       warp 11    no role; the third warpgroup gives its registers to the
//                  softmax warpgroups (216 vs 72 per thread)
//   * S_t = Q_t K_j^T accumulates in TMEM (128 fp32 columns per Q tile); the
//     softmax warps write P_t as packed bf16 (over S_t at d = 128, into
//     columns of their own at d = 64), which the tensor core then reads
//     straight from TMEM for O_t += P_t V_j;
//   * O_t accumulates in TMEM over the item's K/V sweep and is written once;
//   * the two Q tiles share the tensor core: while one softmax group works on
//     its S, the tensor core runs the other tile's P V and next S;
//   * the MMA warp follows a fixed schedule over the union list of key
//     tiles live for either Q tile (causal, key-length and block-sparse
//     skipping are exact per tile), while K/V tiles are loaded once for the
//     pair;
//   * the running max is moved (and O rescaled) only when a new row max
//     exceeds it by more than 2^8; the final O / l and LSE use the same
//     reference max, so the result is unchanged;
//   * with P over S (d = 128), P of a tile's first 64 keys goes to the
//     tensor core before the rest is formed, so half of P V overlaps the
//     second half of the exponentials.
#include "fa_common.cuh"
#include "fa_ptx.cuh"

#include <cuda_bf16.h>

namespace fa {

namespace {

constexpr int kFwdThreads = 384;
constexpr int kSoftmaxRegs = 216;   // 2 x 128 x 216 + 128 x 72 = 384 x 168 registers
constexpr int kOtherRegs = 72;
constexpr int kListMax = kMaxN / kTile;   // union list capacity
constexpr float kRescaleThreshold = 8.0f; // log2 units
constexpr float kSpecSumLimit = 256.0f;    // 2^kRescaleThreshold

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kHalves = D / 64;
  // separate K and V rings; the K ring is the deeper one, since the S MMAs
  // that read K come first
  static constexpr int kStagesK = (D == 64) ? 5 : 3;
  static constexpr int kStagesV = (D == 64) ? 4 : 2;
  // Q buffers (each the two Q tiles of an item, and then the item's O
  // staging) and key-tile lists: at d = 64 two, so that the next item's list
  // is built and its Q and first K tiles are loaded while this item runs; at
  // d = 128 the shared memory holds one
  // At d = 64, S_0, S_1 (128 columns each) and O_0, O_1 (64 each) leave 128
  // TMEM columns, which give each Q tile's P columns of their own: S_t is then
  // free as soon as its softmax group has read it into registers, and the
  // next S_t is computed while that group works on this one. At d = 128 the
  // four regions fill TMEM and P is packed over S in place.
  static constexpr bool kOwnP = (D == 64);
  static constexpr int kQBuf = (D == 64) ? 2 : 1;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBuf * 2 * kTileBytes;
  static constexpr int kV = kK + kStagesK * kTileBytes;
  static constexpr int kBar = kV + kStagesV * kTileBytes;   // 8-byte mbarriers
  // barrier slots
  static constexpr int bQFull = 0;                    // [kQBuf]
  static constexpr int bKFull = bQFull + kQBuf;
  static constexpr int bKEmpty = bKFull + kStagesK;
  static constexpr int bVFull = bKEmpty + kStagesK;
  static constexpr int bVEmpty = bVFull + kStagesV;
  static constexpr int bSFull = bVEmpty + kStagesV;   // [2]
  static constexpr int bPFull = bSFull + 2;           // [2]
  static constexpr int bOFinal = bPFull + 2;          // [2]
  static constexpr int bSFree = bOFinal + 2;          // [2] S_t read into registers (own P columns only)
  static constexpr int bPVDone = bSFree + 2;          // [2] O_t += P_t V complete (own P columns only)
  static constexpr int bPHalf = bPVDone + 2;          // [2] P_t of the first 64 keys is in TMEM (P over S only)
  static constexpr int bClc = bPHalf + 2;             // the next item's cancellation answer has arrived
  static constexpr int bDrain = bClc + 1;
  static constexpr int kNumBars = bDrain + 1;
  // 32-bit words: tmem slot, abort flag, -, wait limit, -, -, next item, -;
  // then per buffer b at 8 + 4 b: list length, last list entry live for Q
  // tile 0 and for Q tile 1, -
  static constexpr int kMisc = kBar + 8 * kNumBars;
  static constexpr int kClc = (kMisc + 4 * (8 + 4 * kQBuf) + 15) & ~15;   // 16-byte answer of a launch cancellation
  static constexpr int kList = kClc + 16;                // uint16 entries, kListMax per buffer
  static constexpr int kSmemBytes = kList + kQBuf * 2 * kListMax;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// union-list entry: key tile j in bits 0-9 (j < 1024), live flags of the two
// Q tiles in bits 10-11, partial flags in bits 12-13
__device__ __forceinline__ int entry_j(uint32_t e) { return (int)(e & 0x3FFu); }
__device__ __forceinline__ uint32_t entry_live(uint32_t e, int t) { return (e >> (10 + t)) & 1u; }
__device__ __forceinline__ uint32_t entry_partial(uint32_t e, int t) { return (e >> (12 + t)) & 1u; }

template <int D, bool F16, bool DROP>
__global__ void __launch_bounds__(kFwdThreads, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
              const FwdParams p) {
  using L = FwdLayout<D>;
  // With P over S (d = 128) and without dropout, P of a tile's first 64 keys
  // goes to the tensor core before the rest is formed, and its half of P V
  // runs meanwhile; the softmax then always takes the row max first, since P
  // may not be formed again once half of it has been used (measured: forward
  // long_causal 1729 -> 1817 TFLOP/s; with dropout -1.7 %, not used there)
  constexpr bool kHalfP = !L::kOwnP && !DROP;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int BH = p.B * p.H;
  const int nC = (p.nT + 1) >> 1;

  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * (uint32_t)i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = misc + 1;
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::kList);
  Ctl ctl{p.err, abort_flag};

  if ((sbase & 1023u) != 0u) {   // uniform across the CTA: nothing has started yet
    if (tid == 0) {
      uint32_t dummy = 0;   // report_error writes only the abort flag
      Ctl c0{p.err, &dummy};
      report_error(c0, kErrSmemAlign, 0);
    }
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < L::kNumBars; ++i)
      mbar_init(bar(i), (i == L::bPFull || i == L::bPFull + 1 || i == L::bSFree || i == L::bSFree + 1 ||
                         i == L::bPHalf || i == L::bPHalf + 1) ? 4u
                                                                                                      : 1u);   // 4 = warps
    abort_flag[0] = 0u;
    abort_flag[2] = p.chk.wait_us;   // the wait limit, read by the slow path of every wait
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(misc), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();   // the barriers are initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // global memory is read and written only from here on: what the previous
  // kernel in the stream wrote is complete and visible
  grid_dep_wait();
  grid_dep_launch();

  // Persistent over items (pairs of Q tiles of one batch-head): the first is
  // this CTA's own, each further one is a CTA of this grid that has not
  // started yet, cancelled through cluster launch control (so items are
  // taken in launch order, each by the first CTA ready for one, and no
  // workspace counter is needed). The CTAs walk groups of p.group heads
  // whose K and V fit in L2 together; within a group the heaviest Q-tile
  // pairs come first. Every ring and barrier phase runs on across items:
  // eK / eV count the K / V ring entries of the items before this one, and
  // each role keeps its own running counts.
  int eK = 0, eV = 0;
  int nk = 0, nv = 0;                     // K / V loads issued (producer threads)
  bool clc_out = false;                   // a cancellation answer is outstanding (K producer)
  uint32_t ns[2] = {0u, 0u}, npv[2] = {0u, 0u};   // S and PV groups issued per Q tile (MMA warp)
  uint32_t nS = 0u, nOF = 0u;             // S tiles and final O read by this softmax group
  int item = (int)blockIdx.x;
  uint32_t kq = 0u;                       // items started: the phase of the Q barrier
  // The roles meet at a named barrier before each item (its list is in
  // shared memory) and after it (its O is stored, its products read out).
  auto item_sync = [&]() {
    tc_fence_before();
    named_bar_sync(1, kFwdThreads);
    tc_fence_after();
  };
  // after an item: the next one, or none (then every role leaves its loop)
  auto next_item = [&]() -> int {
    const int next = (int)misc[6];
    return abort_flag[0] != 0u ? -1 : next;
  };
  if (warp == 8) {
    regs_dec<kOtherRegs>();
    uint32_t nq[2] = {0u, 0u};   // Q loads issued into each buffer (lane 0)
    // Sets item `it` up in buffer qb: its Q tiles are loaded, the union list
    // of the key tiles live for either Q tile is built (ascending j) with its
    // length and the last entry live for each tile, and the K tiles of the
    // first ring's worth of entries are loaded (K ring entries base, base + 1,
    // ...), so that their loads overlap the rest of the set-up. Returns (on
    // lane 0) the K loads issued.
    auto setup = [&](int it, int qb, int base) -> int {
      int bh = 0;
      const int c = nC - 1 - split_grouped(it, p.group, nC, BH, &bh);
      const int qi0 = 2 * c;
      const bool has_t1 = (qi0 + 1) < p.nT;
      const int kvl = effective_kv_len(p.kv_len, bh / p.H, p.N);
      uint16_t* lst = list + qb * kListMax;
      if (lane == 0) {
        const uint32_t qbytes = (has_t1 ? 2u : 1u) * L::kTileBytes;
        mbar_arrive_expect_tx(bar(L::bQFull + qb), qbytes);
        for (int t = 0; t < (has_t1 ? 2 : 1); ++t)
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sbase + L::kQ + (2 * qb + t) * L::kTileBytes + h * 16384, &tq, bar(L::bQFull + qb),
                        64 * h, kTile * (qi0 + t), bh);
        ++nq[qb];
      }
      int count = 0;
      int last[2] = {-1, -1};
      for (int jb = 0; jb < p.nT; jb += 32) {
        const int j = jb + lane;
        uint32_t e = 0;
        if (j < p.nT) {
          const int s0 = tile_state(qi0, j, kvl, p.nT, p.causal, p.block_mask);
          const int s1 = has_t1 ? tile_state(qi0 + 1, j, kvl, p.nT, p.causal, p.block_mask) : kSkip;
          e = (uint32_t)j | ((s0 != kSkip) ? (1u << 10) : 0u) | ((s1 != kSkip) ? (1u << 11) : 0u) |
              ((s0 == kPartial) ? (1u << 12) : 0u) | ((s1 == kPartial) ? (1u << 13) : 0u);
        }
        const bool live = (e >> 10) & 3u;
        const uint32_t ball = __ballot_sync(0xFFFFFFFFu, live);
        if (live) lst[count + __popc(ball & ((1u << lane) - 1u))] = (uint16_t)e;
#pragma unroll
        for (int t = 0; t < 2; ++t) {   // list index of the last entry live for Q tile t so far
          const uint32_t bt = __ballot_sync(0xFFFFFFFFu, (e >> (10 + t)) & 1u);
          if (bt != 0u) last[t] = count + __popc(ball & ((1u << (31 - __clz(bt))) - 1u));
        }
        count += __popc(ball);
      }
      __syncwarp();
      int kpre = 0;
      if (lane == 0) {
        misc[8 + 4 * qb] = (uint32_t)count;
        misc[9 + 4 * qb] = (uint32_t)last[0];
        misc[10 + 4 * qb] = (uint32_t)last[1];
        // (a slot's previous user is an entry of this or an earlier item whose
        // S products free it)
        for (; kpre < count && kpre < L::kStagesK; ++kpre) {
          if (p.chk.stall != 0u && kpre >= 1) break;   // test of the timeout path: K of entry 1 never comes
          const int n = base + kpre;
          const int sk = n % L::kStagesK;
          if (n >= L::kStagesK && !mbar_wait(bar(L::bKEmpty + sk), (uint32_t)(n / L::kStagesK - 1) & 1u, ctl, 1))
            break;
          mbar_arrive_expect_tx(bar(L::bKFull + sk), L::kTileBytes);
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sbase + L::kK + sk * L::kTileBytes + h * 16384, &tk, bar(L::bKFull + sk), 64 * h,
                        kTile * entry_j(lst[kpre]), bh);
          ++nk;
        }
      }
      return kpre;
    };
    if (lane == 0) {
      tma_prefetch_map(&tq);
      tma_prefetch_map(&tk);
    }
    int kpre = setup(item, 0, 0);   // K loads of the current item issued during its set-up (lane 0)
    for (;; ++kq) {
      const int qb = (int)(kq % L::kQBuf);
      int bh = 0;
      (void)split_grouped(item, p.group, nC, BH, &bh);
      item_sync();
      const int len = (int)misc[8 + 4 * qb];
      const uint16_t* lst = list + qb * kListMax;
      // ------------------------------------------------------------ Q and K producer
      int next = -1;
      if (lane == 0) {
        // K of ring entry eK + e into slot (eK + e) mod S, once the MMAs of the
        // entry that used the slot before (of this item or an earlier one)
        // have read it
        bool ok = true;
        for (int e = kpre; e < len; ++e) {
          if (p.chk.stall != 0u && e >= 1) { ok = false; break; }   // test of the timeout path: K of entry 1 never comes
          const int n = eK + e;
          const int sk = n % L::kStagesK;
          if (n >= L::kStagesK && !(ok = mbar_wait(bar(L::bKEmpty + sk), (uint32_t)(n / L::kStagesK - 1) & 1u, ctl, 1)))
            break;
          mbar_arrive_expect_tx(bar(L::bKFull + sk), L::kTileBytes);
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sbase + L::kK + sk * L::kTileBytes + h * 16384, &tk, bar(L::bKFull + sk),
                        64 * h, kTile * entry_j(lst[e]), bh);
          ++nk;
        }
        // every K load of the item is issued: ask for the next item (the answer
        // lands while this one is computed)
        if (ok) {
          mbar_arrive_expect_tx(bar(L::bClc), 16u);
          clc_try_cancel(sbase + L::kClc, bar(L::bClc));
          clc_out = true;
          if (mbar_wait(bar(L::bClc), kq & 1u, ctl, 3)) {
            clc_out = false;
            next = clc_first_ctaid_x(sbase + L::kClc);
            if (next >= (int)gridDim.x) {   // not a CTA of this grid: stop rather than decode it
              report_error(ctl, kErrInternal, 9);
              next = -1;
            }
          }
        }
        misc[6] = (uint32_t)next;
      }
      // with two buffers the next item is set up while this one runs (the
      // other buffer's item has been stored and its list read: every role
      // has passed the barrier after it)
      next = __shfl_sync(0xFFFFFFFFu, next, 0);
      if (L::kQBuf == 2 && next >= 0) kpre = setup(next, qb ^ 1, eK + len);
      item_sync();
      item = next_item();
      if (item < 0) break;
      eK += len;
      if (L::kQBuf == 1) kpre = setup(item, 0, eK);
    }
    // every load and cancellation request issued has completed before the
    // CTA exits; loads were issued in ring order, so the last load into slot
    // s was number s + S * floor((n - 1 - s) / S)
    if (lane == 0) {
      for (int b = 0; b < L::kQBuf; ++b)
        if (nq[b] > 0u) drain_wait(bar(L::bQFull + b), (nq[b] - 1u) & 1u);
      for (int s = 0; s < L::kStagesK && s < nk; ++s)
        drain_wait(bar(L::bKFull + s), (uint32_t)((nk - 1 - s) / L::kStagesK) & 1u);
      if (clc_out) drain_wait(bar(L::bClc), kq & 1u);
    }
  } else if (warp == 10) {
    regs_dec<kOtherRegs>();
    for (;; ++kq) {
      const int qb = (int)(kq % L::kQBuf);
      int bh = 0;
      (void)split_grouped(item, p.group, nC, BH, &bh);
      item_sync();
      const int len = (int)misc[8 + 4 * qb];
      const uint16_t* lst = list + qb * kListMax;
      // ------------------------------------------------------------ V producer
      // (its own thread, so that the K ring can run ahead of the V ring)
      if (lane == 0) {
        if (kq == 0u) tma_prefetch_map(&tv);
        for (int e = 0; e < len; ++e) {
          const int n = eV + e;
          const int sv = n % L::kStagesV;
          if (n >= L::kStagesV && !mbar_wait(bar(L::bVEmpty + sv), (uint32_t)(n / L::kStagesV - 1) & 1u, ctl, 2))
            break;
          mbar_arrive_expect_tx(bar(L::bVFull + sv), L::kTileBytes);
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sbase + L::kV + sv * L::kTileBytes + h * 16384, &tv, bar(L::bVFull + sv),
                        64 * h, kTile * entry_j(lst[e]), bh);
          ++nv;
        }
      }
      item_sync();
      item = next_item();
      if (item < 0) break;
      eV += len;
    }
    if (lane == 0)
      for (int s = 0; s < L::kStagesV && s < nv; ++s)
        drain_wait(bar(L::bVFull + s), (uint32_t)((nv - 1 - s) / L::kStagesV) & 1u);
  } else if (warp == 9) {
    regs_dec<kOtherRegs>();
    for (;; ++kq) {
      const int qb = (int)(kq % L::kQBuf);
      item_sync();
      const int len = (int)misc[8 + 4 * qb];
      const uint16_t* lst = list + qb * kListMax;
      // ------------------------------------------------------------ MMA issuer
      // Fixed schedule over the union list: at entry e, for each Q tile t, first
      // the pending O_t += P_t V of t's previous live entry (waiting for P_t),
      // then S_t = Q_t K_e^T if t is live at e. For dense rows this is
      //   PV0(e-1), S0(e), PV1(e-1), S1(e), PV0(e), ...
      // so that while one softmax group works the tensor core runs the other
      // tile's products. A pending PV is issued at the very next entry, so each
      // V slot is released one entry after its load and the K slot of entry e
      // right after its S products.
      {   // the whole warp runs the schedule; one elected lane issues each MMA and commit
        constexpr uint32_t idS = idesc_16<F16>(128, 128, false, false);
        constexpr uint32_t idO = idesc_16<F16>(128, D, false, true);
        const uint32_t tS[2] = {tmem + 0u, tmem + 128u};
        const uint32_t tO[2] = {tmem + 256u, tmem + 256u + (uint32_t)D};
        // P_t: over S_t, or in columns of its own (after O_1)
        const uint32_t tP[2] = {L::kOwnP ? tmem + 256u + 2u * D : tS[0], L::kOwnP ? tmem + 320u + 2u * D : tS[1]};
        const uint64_t dQ[2] = {desc_kmajor(sbase + L::kQ + 2 * qb * L::kTileBytes, 0),
                                desc_kmajor(sbase + L::kQ + (2 * qb + 1) * L::kTileBytes, 0)};
        const uint64_t dK0 = desc_kmajor(sbase + L::kK, 0);
        const uint64_t dV0 = desc_mnmajor(sbase + L::kV, 0);
        constexpr uint64_t kSlotStep = (uint64_t)(L::kTileBytes >> 4);
        int prev[2] = {-1, -1};       // entry of the pending PV of each Q tile
        // the last entry live for each Q tile: its PV completes O_t, which the
        // softmax group may then read out while the other tile's products run
        const int lastE[2] = {(int)misc[9 + 4 * qb], (int)misc[10 + 4 * qb]};
        uint32_t npv_item[2] = {0u, 0u};   // PV groups of this item per Q tile
        bool ok = mbar_wait_warp(bar(L::bQFull + qb), (kq / L::kQBuf) & 1u, ctl, 4);
        tc_fence_after();

        // O_t += P_t V_{entry pe}
        auto issue_pv = [&](int t, int pe) -> bool {
          const int nvp = eV + pe;
          const int sv = nvp % L::kStagesV;
          if (!mbar_wait_warp(bar((kHalfP ? L::bPHalf : L::bPFull) + t), npv[t] & 1u, ctl, 5)) return false;
          if (!mbar_wait_warp(bar(L::bVFull + sv), (uint32_t)(nvp / L::kStagesV) & 1u, ctl, 6)) return false;
          tc_fence_after();
          const uint64_t dV = dV0 + (uint64_t)sv * kSlotStep;
          const uint32_t acc0 = npv_item[t] > 0 ? 1u : 0u;
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) {
            if (kHalfP && ks == kTile / 32) {   // the second half of P
              if (!mbar_wait_warp(bar(L::bPFull + t), npv[t] & 1u, ctl, 5)) return false;
              tc_fence_after();
            }
            mma_ts_w(tO[t], tP[t] + (uint32_t)ks * 8u, dV + mnmajor_step(ks), idO, ks > 0 ? 1u : acc0);
          }
          if constexpr (L::kOwnP) mma_commit_w(bar(L::bPVDone + t));   // P_t may be rewritten, O_t rescaled
          if (pe == lastE[t]) mma_commit_w(bar(L::bOFinal + t));       // O_t is complete
          ++npv[t];
          ++npv_item[t];
          return true;
        };

        if constexpr (L::kOwnP) {
          // Own P columns: at entry e, first S_t(e) for each live tile, each as
          // soon as group t has read its previous S_t into registers, then the
          // PVs of entry e - 1. For dense rows:
          //   S0(e), S1(e), PV0(e-1), PV1(e-1), S0(e+1), ...
          // so S_t(e+1) is computed while group t still works on S_t(e).
          for (int e = 0; e < len && ok; ++e) {
            const uint32_t ent = lst[e];
            const int sk = (eK + e) % L::kStagesK;
            bool k_ready = false;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (!ok || !entry_live(ent, t)) continue;
              if (ns[t] > 0 && !(ok = mbar_wait_warp(bar(L::bSFree + t), (ns[t] - 1u) & 1u, ctl, 8))) break;
              if (!k_ready) {
                ok = mbar_wait_warp(bar(L::bKFull + sk), (uint32_t)((eK + e) / L::kStagesK) & 1u, ctl, 7);
                if (!ok) break;
                tc_fence_after();
                k_ready = true;
              }
              const uint64_t dK = dK0 + (uint64_t)sk * kSlotStep;
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks)
                mma_ss_w(tS[t], dQ[t] + kmajor_step(ks), dK + kmajor_step(ks), idS, ks > 0 ? 1u : 0u);
              mma_commit_w(bar(L::bSFull + t));
              ++ns[t];
            }
            if (!ok) break;
            mma_commit_w(bar(L::bKEmpty + sk));   // K_e is no longer needed
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (ok && prev[t] >= 0) ok = issue_pv(t, prev[t]);
              prev[t] = entry_live(ent, t) ? e : -1;
            }
            if (!ok) break;
            if (e > 0) mma_commit_w(bar(L::bVEmpty + (eV + e - 1) % L::kStagesV));   // both PVs of entry e-1 issued
          }
        } else {
          for (int e = 0; e < len && ok; ++e) {
            const uint32_t ent = lst[e];
            const int sk = (eK + e) % L::kStagesK;
            bool k_ready = false;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (!ok) break;
              if (prev[t] >= 0) {
                ok = issue_pv(t, prev[t]);
                prev[t] = -1;
                if (!ok) break;
              }
              if (entry_live(ent, t)) {
                if (!k_ready) {
                  ok = mbar_wait_warp(bar(L::bKFull + sk), (uint32_t)((eK + e) / L::kStagesK) & 1u, ctl, 7);
                  if (!ok) break;
                  tc_fence_after();
                  k_ready = true;
                }
                const uint64_t dK = dK0 + (uint64_t)sk * kSlotStep;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                  mma_ss_w(tS[t], dQ[t] + kmajor_step(ks), dK + kmajor_step(ks), idS, ks > 0 ? 1u : 0u);
                mma_commit_w(bar(L::bSFull + t));
                prev[t] = e;
              }
            }
            if (!ok) break;
            mma_commit_w(bar(L::bKEmpty + sk));                       // K_e is no longer needed
            if (e > 0) mma_commit_w(bar(L::bVEmpty + (eV + e - 1) % L::kStagesV));   // both PVs of entry e-1 issued
          }
        }
        if (ok) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (ok && prev[t] >= 0) ok = issue_pv(t, prev[t]);   // (commits O_t's completion)
          }
          // the last entry's V slot goes back to the producer
          if (ok && len > 0) mma_commit_w(bar(L::bVEmpty + (eV + len - 1) % L::kStagesV));
        }
      }
      item_sync();
      item = next_item();
      if (item < 0) break;
      eK += len;
      eV += len;
    }
    // every MMA issued has completed before TMEM is freed
    mma_commit_w(bar(L::bDrain));
    drain_wait(bar(L::bDrain), 0);
  } else if (warp < 8) {
    regs_inc<kSoftmaxRegs>();
    for (;; ++kq) {
      int bh = 0;
      const int c = nC - 1 - split_grouped(item, p.group, nC, BH, &bh);
      const int qi0 = 2 * c;
      const int kvl = effective_kv_len(p.kv_len, bh / p.H, p.N);
      item_sync();
      const int qb = (int)(kq % L::kQBuf);
      const int len = (int)misc[8 + 4 * qb];
      const uint16_t* lst = list + qb * kListMax;
      // ------------------------------------------------------------ softmax groups
      const int t = warp >> 2;                 // Q tile of this warpgroup
      const int r = tid & 127;                 // row within the tile = TMEM lane
      const int qi = qi0 + t;
      const int row = kTile * qi + r;          // query index within the head
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t tS = tmem + (uint32_t)(t * 128) + lane_off;
      const uint32_t tO = tmem + 256u + (uint32_t)(t * D) + lane_off;
      const uint32_t tP = L::kOwnP ? tmem + 256u + 2u * D + 64u * (uint32_t)t + lane_off : tS;
      const float sl2 = p.scale_log2;

      float m_ref = -INFINITY;
      float l = 0.f;
      uint32_t n = 0;   // S tiles of this item (nS: of all items)
      bool ok = (qi < p.nT);
      for (int e = 0; e < len && ok; ++e) {
        const uint32_t ent = lst[e];
        if (!entry_live(ent, t)) continue;
        // dropout: keep bits of this row for the entry's 128 keys, made before S
        // is awaited, so that the generator runs while the tensor pipe computes
        // S. Keep bytes of keys 4b .. 4b + 3 of a row come from one generator
        // call, counter (row / 4, key block b, bh, 0), word row mod 4; a key is
        // kept iff its byte is >= t. The four rows of a lane quad share their
        // calls: for keys 16m .. 16m + 15 lane s of the quad makes the call of
        // key block 4m + s and files the flags of word d (row d of the quad) in
        // bits 8k + m of word d (k: key of the block); a 4 x 4 transpose across
        // the quad then hands every row its four words. keep[s] bit 8k + m:
        // key 16m + 4s + k of the entry.
        uint32_t keep[4] = {0u, 0u, 0u, 0u};
        if constexpr (DROP) {
          const uint32_t kb0 = 32u * (uint32_t)entry_j(ent);
          const uint32_t s4 = (uint32_t)lane & 3u;   // = row mod 4
          const uint32_t c4 = (256u - p.drop.t) * 0x01010101u;
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const uint4 v = philox4x32_10((uint32_t)row >> 2, kb0 + 4u * (uint32_t)m + s4, (uint32_t)bh, 0u,
                                          p.drop.seed_lo, p.drop.seed_hi);
            keep[0] |= bytes_ge_flags(v.x, c4) >> (7 - m);
            keep[1] |= bytes_ge_flags(v.y, c4) >> (7 - m);
            keep[2] |= bytes_ge_flags(v.z, c4) >> (7 - m);
            keep[3] |= bytes_ge_flags(v.w, c4) >> (7 - m);
          }
          quad_transpose(keep, s4);
          // the bits are complete here: the compiler may not move the generator
          // past the wait into the exponential loop
          asm volatile("" : "+r"(keep[0]), "+r"(keep[1]), "+r"(keep[2]), "+r"(keep[3]));
        }
        if (!mbar_wait_warp(bar(L::bSFull + t), nS & 1u, ctl, 10 + t)) { ok = false; break; }
        tc_fence_after();
        if (p.chk.rec != nullptr && r == 0) {   // the tile as this kernel computes it
          uint8_t* rc = p.chk.rec + ((size_t)bh * p.nT + qi) * p.nT + entry_j(ent);
          *rc = (uint8_t)(*rc + (entry_partial(ent, t) ? 2 : 1));
        }
        float x[128];
        {
          uint32_t u0[32], u1[32], u2[32], u3[32];
          tmem_ld32(tS + 0u, u0);
          tmem_ld32(tS + 32u, u1);
          tmem_ld32(tS + 64u, u2);
          tmem_ld32(tS + 96u, u3);
          tmem_ld_wait(u0);
          tmem_ld_wait(u1);
          tmem_ld_wait(u2);
          tmem_ld_wait(u3);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            x[i] = __uint_as_float(u0[i]);
            x[32 + i] = __uint_as_float(u1[i]);
            x[64 + i] = __uint_as_float(u2[i]);
            x[96 + i] = __uint_as_float(u3[i]);
          }
        }
        if constexpr (L::kOwnP) {   // S_t is in registers: the next S_t may be computed
          tc_fence_before();
          mbar_arrive_warp(bar(L::bSFree + t));
        }
        if (entry_partial(ent, t)) {
          // a key is masked when it lies past the row (causal) or at or past the
          // key length: key >= min(row + 1, key length), i.e. column i >= lim
          const int lim = (p.causal ? min(row + 1, kvl) : kvl) - kTile * entry_j(ent);
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim) x[i] = -INFINITY;
        }
        if (L::kOwnP && nS > 0) {
          // the previous O_t += P_t V has completed (of this item or the last
          // one): O_t may be rescaled and the P_t columns rewritten
          if (!mbar_wait_warp(bar(L::bPVDone + t), (nS - 1u) & 1u, ctl, 16 + t)) { ok = false; break; }
          tc_fence_after();
        }
        // Two passes at most (at d = 64 without dropout; otherwise only pass 1).
        // Pass 0 (not for a row block's first tile) takes the
        // exponentials with the current reference max: if every row of the warp
        // then sums to less than 2^8, no score exceeds the reference by the
        // rescale threshold, so the row max would not have moved it and P is
        // exactly what pass 1 would give. Otherwise pass 1 takes the row max,
        // moves the reference (rescaling O) where it grew past the threshold,
        // and redoes the exponentials (the whole warp: the TMEM stores are
        // warp-collective). This saves the row max on most tiles.
        float s_row = 0.f;
        // (with dropout, and when half of P goes ahead: always the row max)
        for (int pass = (n == 0 || DROP || kHalfP) ? 1 : 0; pass < 2; ++pass) {
          if (pass == 1) {
            // row max with three-input max: 8 independent chains over 128 scores
            float mx8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx8[k] = x[k];
#pragma unroll
            for (int i = 8; i < 120; i += 16)
#pragma unroll
              for (int k = 0; k < 8; ++k) mx8[k] = fmax3(mx8[k], x[i + k], x[i + 8 + k]);
#pragma unroll
            for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(mx8[k], x[120 + k]);
            const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
            const float m_new = mx * sl2;
            // move the reference max only when the row max grew by more than the
            // threshold; the O rescale is warp-collective (tcgen05.ld/st), so a
            // warp rescales when any of its rows needs it (alpha = 1 for the rest)
            const bool move = (n == 0) || (m_new > m_ref + kRescaleThreshold);
            float alpha = 1.f;
            if (move) {
              alpha = (n == 0 || m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
              l *= alpha;
              m_ref = m_new;
            }
            if (n > 0 && __any_sync(0xFFFFFFFFu, move)) {
              uint32_t u[32];
#pragma unroll
              for (int cc = 0; cc < D / 32; ++cc) {
                tmem_ld32(tO + 32u * cc, u);
                tmem_ld_wait(u);
#pragma unroll
                for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
                tmem_st32(tO + 32u * cc, u);
              }
              tmem_st_wait();
            }
          }
          const float ref = (m_ref == -INFINITY) ? 0.f : m_ref;
          // packed fp32 pairs (one f32x2 instruction per two keys) for the
          // exponent arguments and the row sum: the softmax is issue-bound
          const float2 sl2x2 = make_float2(sl2, sl2);
          const float2 nref2 = make_float2(-ref, -ref);
          float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float2 a = __ffma2_rn(make_float2(x[64 * hh + 2 * i], x[64 * hh + 2 * i + 1]), sl2x2, nref2);
              const float p0 = ex2(a.x);
              const float p1 = ex2(a.y);
              sum4[i & 3] = __fadd2_rn(sum4[i & 3], make_float2(p0, p1));   // statistics use the undropped P
              pk[i] = pack2<F16>(p0, p1);
              if constexpr (DROP) {
                // keys 64 hh + 2 i and + 1 are bits 8k + m and 8k + 8 + m of
                // keep[(i / 2) mod 4] (m = 4 hh + i / 8, k = 2 (i mod 2)): shifted
                // to bit 7 of bytes k and k + 1, they become the masks of the
                // two 16-bit halves by sign replication. The keep scale is
                // applied to O in the epilogue (the same factor for every kept term).
                const int m = 4 * hh + (i >> 3), k = 2 * (i & 1);
                const uint32_t kw = keep[(i >> 1) & 3] << (7 - m);
                pk[i] &= prmt(kw, 0u, (uint32_t)((8 + k) * 0x11 + (9 + k) * 0x1100));
              }
            }
            tmem_st32(tP + 32u * hh, pk);
            if (kHalfP && hh == 0) {   // the first 64 keys' P: its half of P V may start
              tmem_st_wait();
              tc_fence_before();
              mbar_arrive_warp(bar(L::bPHalf + t));
            }
          }
          tmem_st_wait();
          const float2 s01 = __fadd2_rn(sum4[0], sum4[1]), s23 = __fadd2_rn(sum4[2], sum4[3]);
          const float2 s4 = __fadd2_rn(s01, s23);
          s_row = s4.x + s4.y;
          // (a row whose reference is still -inf, every earlier key masked,
          // always takes the row max)
          if (pass == 0 && __all_sync(0xFFFFFFFFu, s_row < kSpecSumLimit && m_ref != -INFINITY)) break;
        }
        l += s_row;
        tc_fence_before();
        mbar_arrive_warp(bar(L::bPFull + t));
        ++n;
        ++nS;
      }

      if (qi < p.nT) {
        // all MMAs that read Q_t have completed (or never ran); make sure the
        // Q load itself has landed before its buffer is reused for staging O
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (ok) ok = mbar_wait_warp(bar(L::bQFull + qb), (kq / L::kQBuf) & 1u, ctl, 12 + t);
        if (ok && n > 0) ok = mbar_wait_warp(bar(L::bOFinal + t), nOF & 1u, ctl, 14 + t);
        if (n > 0) ++nOF;
        if (!ok) drain_wait(bar(L::bQFull + qb), (kq / L::kQBuf) & 1u);   // after an abort: the Q load (always issued) lands before its buffer is rewritten
        tc_fence_after();
        uint8_t* stage = smem + L::kQ + (2 * qb + t) * L::kTileBytes;
        const float inv_l = (n > 0 && l > 0.f) ? (DROP ? p.drop.keep_scale : 1.f) / l : 0.f;
        const bool have_o = ok && n > 0;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t u[32];
          if (have_o) {
            tmem_ld32(tO + 32u * cc, u);
            tmem_ld_wait(u);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack2<F16>(__uint_as_float(u[2 * i]) * inv_l, __uint_as_float(u[2 * i + 1]) * inv_l);
          // 32 columns = 4 chunks of 16 bytes, 128B-swizzled rows
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int col = 32 * cc + 8 * k;           // first column of the chunk
            const int h = col >> 6;                    // 64-column half
            const int chunk = (col & 63) >> 3;         // chunk within the 128-byte row
            uint8_t* dst = stage + h * 16384 + (r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
          }
        }
        if (row < p.N) {
          float lse = -INFINITY;
          if (have_o && l > 0.f) lse = (m_ref + log2f(l)) * 0.69314718055994531f;
          p.lse[(size_t)bh * p.N + row] = lse;
        }
        // each warp stores its own 32 rows (boxes of 32 rows), so that no warp
        // ever waits for another at a group-wide barrier
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int row0 = kTile * qi + 32 * (warp & 3);
          if (row0 < p.N)
            for (int h = 0; h < L::kHalves; ++h)
              tma_store_3d(&to, smem_u32(stage) + h * 16384 + 4096 * (warp & 3), 64 * h, row0, bh);
          bulk_commit_group();
          bulk_wait_group_read_all();   // the store has read the staging; the grid's end makes it visible
        }
      }
      item_sync();
      item = next_item();
      if (item < 0) break;
    }
  } else {
    regs_dec<kOtherRegs>();   // warp 11: no role of its own, it only keeps the item barriers
    for (;; ++kq) {
      item_sync();
      item_sync();
      item = next_item();
      if (item < 0) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool F16, bool DROP>
cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const FwdParams& p, cudaStream_t s) {
  using L = FwdLayout<D>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static PerDeviceOnce smem_set;
  e = once_per_device(smem_set, dev, [] {
    return cudaFuncSetAttribute(fa_fwd_kernel<D, F16, DROP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                L::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  FwdParams q = p;
  // a head's K and V (2 N d 16-bit elements) are re-read by all of its CTAs
  q.group = l2_head_group(4.0 * p.N * p.d, p.B * p.H);
  const int nC = (p.nT + 1) / 2;
  const dim3 grid((unsigned)(nC * p.B * p.H));
  return launch_pdl(true, fa_fwd_kernel<D, F16, DROP>, grid, dim3(kFwdThreads), L::kSmemBytes, s, tq, tk, tv, to, q);
}

}  // namespace

cudaError_t launch_fwd(int d, bool f16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, cudaStream_t s) {
  const bool drop = p.drop.t > 0;
  const int kd = kernel_head_dim(d);
  if (kd == 256) return drop ? cudaErrorInvalidValue : launch_fwd_single(kd, f16, tq, tk, tv, to, p, s);
#define FA_FWD_CASE(DD, FF, DR) \
  if (kd == DD && f16 == FF && drop == DR) return launch_fwd_d<DD, FF, DR>(tq, tk, tv, to, p, s);
  FA_FWD_CASE(64, false, false)
  FA_FWD_CASE(128, false, false)
  FA_FWD_CASE(64, true, false)
  FA_FWD_CASE(128, true, false)
  FA_FWD_CASE(64, false, true)
  FA_FWD_CASE(128, false, true)
  FA_FWD_CASE(64, true, true)
  FA_FWD_CASE(128, true, true)
#undef FA_FWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa
