// Forward and backward kernels for head dimensions above 128 (up to 256), for
// sm_103a. Same method and arithmetic as fa_fwd.cu / fa_bwd.cu (FlashAttention
// milestone page (nlp-lineage), "The idea -- Tiling" and "Recomputation";
// "The notation" gives d of 64 to 128 as typical, so these are the wider
// variants), with tiles 256 columns wide (columns past d are zero on load and
// are not stored).
//
// At d = 256 a 128-row tile of Q, K or V is 64 KB and an fp32 accumulator of
// width d fills half of the 512 TMEM columns, so both kernels are laid out
// differently from the narrower ones:
//
// Forward (fa_fwd_wide_kernel<256>): one 128-row Q tile per CTA (64 KB,
// resident); K and V stream through a ring of five 32 KB half tiles (128 keys
// x 128 columns) in the order the tensor core reads them (the kernel is
// written for any tile width of 64, 128 or 256 columns, in ring units of up to
// 128 columns). TMEM: S twice (2 x 128
// fp32 columns, so that S of the next key tile is computed while the softmax
// works on this one) and O (256 columns). Schedule of the single MMA thread:
//   S(0), S(1), PV(0), S(2), PV(1), ...   (PV(e) once P(e) is in TMEM)
// Because S(e+1) completes before PV(e) may have run, a softmax step that has
// to rescale O first waits for the previous PV (two alternating barriers, so
// that a waiter never falls two phases behind). Warps: 0-3 softmax (thread =
// row), 4 TMA producer, 5 TMEM allocator and MMA issuer.
//
// Backward (fa_bwd_wide_kernel): persistent like the narrow backward, over
// items (128-key tile, batch-head, half of the head dimension): two CTAs share
// a key tile, each recomputing S^T and dP^T over the full d and accumulating
// dV, dK and dQ for its 128 columns only, so that the accumulators fit in TMEM.
// Queries are taken 64 at a time (a 64 x 256 tile is 32 KB), which leaves
// shared memory for K and V (64 KB each, resident for the item):
//   S^T  = K Q^T             M = 128 keys, N = 64 queries, K = d
//   dP^T = V dO^T            the same shapes
//   dV_h += P^T dO_h         A = P^T packed in TMEM, B = dO columns of half h
//   dK_h += dS^T Q_h         A = dS^T packed in TMEM, B = Q columns of half h
//   dQ_h^T = K_h^T dS^T      M = 128 columns of half h, N = 64 queries, K = 128
//                            keys (A = K read MN-major, B = dS^T in smem)
// The dQ partial is computed transposed so that every product keeps M = 128;
// the drain warps (thread = head-dimension column) stage it as query rows and
// add it into the fp32 accumulator with TMA reduce-add. TMEM: S^T 64, dP^T 64,
// dQ^T 64, dV 128, dK 128 columns. Warps: 0-3 and 4-7 recompute P and dS for
// query columns 0-31 and 32-63 (thread = key row), 8-11 drain dQ, 12 TMA
// producer, 13 TMEM allocator and MMA issuer.
//
// Dropout is not offered at these widths (the call reports unsupported).
#include "fa_common.cuh"
#include "fa_ptx.cuh"

namespace fa {

namespace {

constexpr int kWListMax = kMaxN / kTile;
constexpr float kWRescaleThreshold = 8.0f;   // log2 units, as in the narrow forward

// --------------------------------------------------------------------------
// forward
// --------------------------------------------------------------------------

// Layout of the one-Q-tile forward for a tile width D (64, 128 or 256): K and
// V stream through a ring of units of 128 keys x U columns (U = min(D, 128)),
// D / U units per tile, in the order the MMA thread reads them.
template <int D>
struct WFwdLayout {
  static constexpr int kU = D < 128 ? D : 128;          // columns per ring unit
  static constexpr int kUnits = D / kU;                  // units per K or V tile
  static constexpr int kAtomsPerUnit = kU / 64;
  static constexpr int kUnitBytes = kTile * kU * 2;
  static constexpr int kSlots = D == 64 ? 12 : (D == 128 ? 6 : 5);
  static constexpr int kQ = 0;                           // 128 x D: D / 64 atoms of 16 KB
  static constexpr int kRing = kQ + (D / 64) * 16384;    // [kSlots] units
  static constexpr int kBar = kRing + kSlots * kUnitBytes;
  static constexpr int bQFull = 0;
  static constexpr int bFull = 1;                      // [kSlots]
  static constexpr int bEmpty = bFull + kSlots;        // [kSlots]
  static constexpr int bSFull = bEmpty + kSlots;       // [2]
  static constexpr int bPFull = bSFull + 2;            // [2], 4 arrivals (warps)
  static constexpr int bPV = bPFull + 2;               // [2]
  static constexpr int bOFinal = bPV + 2;
  static constexpr int bDrain = bOFinal + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kMisc = kBar + 8 * kNumBars;    // tmem slot, abort flag, list length, wait limit
  static constexpr int kList = kMisc + 16;             // uint16 entries
  static constexpr int kSmemBytes = kList + 2 * kWListMax;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

constexpr int kWFwdThreads = 192;

// list entry: key tile in bits 0-9, partial flag in bit 10
__device__ __forceinline__ int wentry_j(uint32_t e) { return (int)(e & 0x3FFu); }
__device__ __forceinline__ bool wentry_partial(uint32_t e) { return (e >> 10) & 1u; }

template <int D, bool F16>
__global__ void __launch_bounds__(kWFwdThreads, 1)
fa_fwd_wide_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                   const FwdParams p) {
  using L = WFwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int BH = p.B * p.H;
  int bh = 0;
  // groups of p.group heads whose K and V fit in L2 together; heaviest Q tiles first
  const int qi = p.nT - 1 - split_grouped((int)blockIdx.x, p.group, p.nT, BH, &bh);

  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * (uint32_t)i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = misc + 1;
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::kList);
  Ctl ctl{p.err, abort_flag};

  if ((sbase & 1023u) != 0u) {
    if (tid == 0) {
      uint32_t dummy = 0;   // report_error writes only the abort flag
      Ctl c0{p.err, &dummy};
      report_error(c0, kErrSmemAlign, 40);
    }
    return;
  }
  if (tid == 0) {
    for (int i = 0; i < L::kNumBars; ++i) mbar_init(bar(i), (i == L::bPFull || i == L::bPFull + 1) ? 4u : 1u);
    abort_flag[0] = 0u;
    abort_flag[2] = p.chk.wait_us;   // the wait limit, read by the slow path of every wait
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(misc), 512);
    tmem_relinquish();
  }
  grid_dep_wait();   // global memory only from here on (programmatic dependent launch)
  grid_dep_launch();
  const int kvl = effective_kv_len(p.kv_len, bh / p.H, p.N);
  if (warp == 4) {
    // live key tiles of this Q tile, ascending
    int count = 0;
    for (int base = 0; base < p.nT; base += 32) {
      const int j = base + lane;
      const int st = j < p.nT ? tile_state(qi, j, kvl, p.nT, p.causal, p.block_mask) : kSkip;
      const bool live = st != kSkip;
      const uint32_t ball = __ballot_sync(0xFFFFFFFFu, live);
      if (live) list[count + __popc(ball & ((1u << lane) - 1u))] = (uint16_t)(j | (st == kPartial ? 1024 : 0));
      count += __popc(ball);
    }
    if (lane == 0) misc[2] = (uint32_t)count;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const int len = (int)misc[2];

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tq);
      tma_prefetch_map(&tk);
      tma_prefetch_map(&tv);
      mbar_arrive_expect_tx(bar(L::bQFull), (uint32_t)(D / 64) * 16384u);
      for (int a = 0; a < D / 64; ++a) tma_load_3d(sbase + L::kQ + a * 16384, &tq, bar(L::bQFull), 64 * a, kTile * qi, bh);
      int u = 0;   // units issued, in the order the MMA thread reads them: K(0), then K(e+1), V(e) per entry
      auto load_unit = [&](const CUtensorMap* m, int j, int unit) -> bool {
        const int s = u % L::kSlots;
        const uint32_t n = (uint32_t)(u / L::kSlots);
        if (u >= L::kSlots && !mbar_wait(bar(L::bEmpty + s), (n - 1) & 1u, ctl, 41)) return false;
        mbar_arrive_expect_tx(bar(L::bFull + s), (uint32_t)L::kUnitBytes);
        for (int a = 0; a < L::kAtomsPerUnit; ++a)
          tma_load_3d(sbase + L::kRing + s * L::kUnitBytes + a * 16384, m, bar(L::bFull + s), L::kU * unit + 64 * a,
                      kTile * j, bh);
        ++u;
        return true;
      };
      auto load_tile = [&](const CUtensorMap* m, int j) -> bool {
        for (int unit = 0; unit < L::kUnits; ++unit)
          if (!load_unit(m, j, unit)) return false;
        return true;
      };
      if (len > 0) {
        bool ok = load_tile(&tk, wentry_j(list[0]));
        for (int e = 0; e < len && ok; ++e) {
          if (p.chk.stall != 0u) break;   // test of the timeout path: nothing after K of entry 0
          if (e + 1 < len && !(ok = load_tile(&tk, wentry_j(list[e + 1])))) break;
          ok = load_tile(&tv, wentry_j(list[e]));
        }
      }
      drain_wait(bar(L::bQFull), 0);
      for (int s = 0; s < L::kSlots && s < u; ++s)
        drain_wait(bar(L::bFull + s), (uint32_t)((u - 1 - s) / L::kSlots) & 1u);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    {   // the whole warp runs the schedule; one elected lane issues each MMA and commit
      constexpr uint32_t idS = idesc_16<F16>(128, 128, false, false);
      constexpr uint32_t idO = idesc_16<F16>(128, L::kU, false, true);
      constexpr int kStepsPerUnit = L::kU / 16;
      const uint32_t tS[2] = {tmem, tmem + 128u};
      const uint32_t tO = tmem + 256u;
      const uint64_t dQ0 = desc_kmajor(sbase + L::kQ, 0);
      bool ok = mbar_wait_warp(bar(L::bQFull), 0, ctl, 44);
      tc_fence_after();
      int u = 0;
      auto slot = [&](int uu) -> uint32_t { return sbase + L::kRing + (uint32_t)(uu % L::kSlots) * L::kUnitBytes; };
      auto wait_units = [&](uint32_t site) -> bool {
        for (int unit = 0; unit < L::kUnits; ++unit)
          if (!mbar_wait_warp(bar(L::bFull + (u + unit) % L::kSlots), (uint32_t)((u + unit) / L::kSlots) & 1u, ctl, site))
            return false;
        return true;
      };
      auto release_units = [&]() {
        for (int unit = 0; unit < L::kUnits; ++unit) mma_commit_w(bar(L::bEmpty + (u + unit) % L::kSlots));
        u += L::kUnits;
      };
      // S(e) = Q K_e^T into buffer e mod 2 (K in units u ..)
      auto issue_s = [&](int e) -> bool {
        if (!wait_units(45)) return false;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss_w(tS[e & 1], dQ0 + kmajor_step(ks), desc_kmajor(slot(u + ks / kStepsPerUnit), ks % kStepsPerUnit), idS,
                 ks > 0 ? 1u : 0u);
        release_units();
        mma_commit_w(bar(L::bSFull + (e & 1)));
        return true;
      };
      // O += P(e) V_e (V in units u ..: output columns kU h .. kU h + kU - 1)
      auto issue_pv = [&](int e) -> bool {
        if (!mbar_wait_warp(bar(L::bPFull + (e & 1)), (uint32_t)(e >> 1) & 1u, ctl, 46)) return false;
        if (!wait_units(47)) return false;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < L::kUnits; ++h)
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            mma_ts_w(tO + (uint32_t)(L::kU * h), tS[e & 1] + (uint32_t)ks * 8u, desc_mnmajor(slot(u + h), ks), idO,
                   (e > 0 || ks > 0) ? 1u : 0u);
        release_units();
        mma_commit_w(bar(L::bPV + (e & 1)));
        return true;
      };
      if (len > 0 && ok) {
        ok = issue_s(0);
        for (int e = 0; e < len && ok; ++e) {
          if (e + 1 < len && !(ok = issue_s(e + 1))) break;
          ok = issue_pv(e);
        }
        if (ok) mma_commit_w(bar(L::bOFinal));
      }
      mma_commit_w(bar(L::bDrain));
      drain_wait(bar(L::bDrain), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax (thread = row)
    const int r = tid;
    const int row = kTile * qi + r;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    uint32_t n = 0;
    bool ok = true;
    for (int e = 0; e < len; ++e) {
      const uint32_t ent = list[e];
      const uint32_t tSe = tmem + 128u * (uint32_t)(e & 1) + lane_off;
      if (!(ok = mbar_wait_warp(bar(L::bSFull + (e & 1)), (uint32_t)(e >> 1) & 1u, ctl, 50))) break;
      tc_fence_after();
      if (p.chk.rec != nullptr && r == 0)   // the tile as this kernel computes it
        record_tile(p.chk.rec, bh, qi, wentry_j(ent), p.nT, wentry_partial(ent));
      float x[128];
      {
        uint32_t u0[32], u1[32], u2[32], u3[32];
        tmem_ld32(tSe + 0u, u0);
        tmem_ld32(tSe + 32u, u1);
        tmem_ld32(tSe + 64u, u2);
        tmem_ld32(tSe + 96u, u3);
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
      if (wentry_partial(ent)) {
        const int key0 = kTile * wentry_j(ent);
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          const int key = key0 + i;
          if ((p.causal && key > row) || key >= kvl) x[i] = -INFINITY;
        }
      }
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
      const bool move = (n == 0) || (m_new > m_ref + kWRescaleThreshold);
      float alpha = 1.f;
      if (move) {
        alpha = (n == 0 || m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
        l *= alpha;
        m_ref = m_new;
      }
      if (n > 0 && __any_sync(0xFFFFFFFFu, move)) {
        // O holds the products through entry e - 1 only once PV(e - 1) has
        // completed: S(e) may have finished before it ran
        if (!(ok = mbar_wait_warp(bar(L::bPV + ((e - 1) & 1)), (uint32_t)((e - 1) >> 1) & 1u, ctl, 51))) break;
        tc_fence_after();
        const uint32_t tO = tmem + 256u + lane_off;
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
      const float ref = (m_ref == -INFINITY) ? 0.f : m_ref;
      const float2 sl2x2 = make_float2(sl2, sl2);
      const float2 nref2 = make_float2(-ref, -ref);
      float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 a = __ffma2_rn(make_float2(x[64 * hh + 2 * i], x[64 * hh + 2 * i + 1]), sl2x2, nref2);
          const float p0 = ex2(a.x), p1 = ex2(a.y);
          sum4[i & 3] = __fadd2_rn(sum4[i & 3], make_float2(p0, p1));
          pk[i] = pack2<F16>(p0, p1);
        }
        tmem_st32(tSe + 32u * hh, pk);
      }
      tmem_st_wait();
      const float2 s4 = __fadd2_rn(__fadd2_rn(sum4[0], sum4[1]), __fadd2_rn(sum4[2], sum4[3]));
      l += s4.x + s4.y;
      tc_fence_before();
      mbar_arrive_warp(bar(L::bPFull + (e & 1)));
      ++n;
    }
    // epilogue: O / l -> 16-bit, staged in the Q buffer (free once every MMA
    // has completed), each warp storing its own 32 rows
    ok = __all_sync(0xFFFFFFFFu, ok);
    // the Q load (issued even when no key tile is live) must have landed
    // before its buffer is rewritten, and every MMA that read it completed
    if (ok) ok = mbar_wait_warp(bar(L::bQFull), 0, ctl, 53);
    if (ok && n > 0) ok = mbar_wait_warp(bar(L::bOFinal), 0, ctl, 52);
    if (!ok) drain_wait(bar(L::bQFull), 0);
    tc_fence_after();
    const bool have_o = ok && n > 0;
    const float inv_l = (have_o && l > 0.f) ? 1.f / l : 0.f;
    uint8_t* stage = smem + L::kQ;
#pragma unroll 1
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t u[32];
      if (have_o) {
        tmem_ld32(tmem + 256u + lane_off + 32u * cc, u);
        tmem_ld_wait(u);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) u[i] = 0u;
      }
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pk[i] = pack2<F16>(__uint_as_float(u[2 * i]) * inv_l, __uint_as_float(u[2 * i + 1]) * inv_l);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int col = 32 * cc + 8 * k;
        const int a = col >> 6;
        const int chunk = (col & 63) >> 3;
        uint8_t* dst = stage + a * 16384 + (r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
    }
    if (row < p.N) {
      float lse = -INFINITY;
      if (have_o && l > 0.f) lse = (m_ref + log2f(l)) * 0.69314718055994531f;
      p.lse[(size_t)bh * p.N + row] = lse;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const int row0 = kTile * qi + 32 * warp;
      if (row0 < p.N)
        for (int a = 0; a < D / 64; ++a)
          if (64 * a < p.d) tma_store_3d(&to, sbase + L::kQ + a * 16384 + 4096 * warp, 64 * a, row0, bh);
      bulk_commit_group();
      bulk_wait_group_read_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// --------------------------------------------------------------------------
// backward
// --------------------------------------------------------------------------

struct WBwdLayout {
  static constexpr int kK = 0;                 // 128 keys x 256: four 16 KB atoms
  static constexpr int kV = kK + 65536;
  static constexpr int kQ = kV + 65536;        // 64 queries x 256: four 8 KB atoms
  static constexpr int kdO = kQ + 32768;
  static constexpr int kdS = kdO + 32768;      // dS^T: 128 keys x 64 queries, 16-bit, one 16 KB atom
  static constexpr int kdQ = kdS + 16384;      // dQ staging: 4 warps x [32 queries x 32 fp32]
  static constexpr int kRow = kdQ + 16384;     // LSE2[64], D[64]
  static constexpr int kBar = kRow + 512;
  static constexpr int bKV = 0;
  static constexpr int bKVFree = 1;            // 8 arrivals: the epilogue's stores have read their staging
  static constexpr int bQFull = 2;
  static constexpr int bQEmpty = 3;
  static constexpr int bdOFull = 4;
  static constexpr int bdOEmpty = 5;
  static constexpr int bSFull = 6;
  static constexpr int bPFull = 7;             // 8 arrivals
  static constexpr int bdPFull = 8;
  static constexpr int bdSFull = 9;            // 8 arrivals
  static constexpr int bdSEmpty = 10;
  static constexpr int bdQFull = 11;
  static constexpr int bdQFree = 12;           // 4 arrivals
  static constexpr int bFinal = 13;
  static constexpr int bDrain = 14;
  static constexpr int kItemRing = 4;
  static constexpr int bItemFull = 15;                       // [kItemRing]
  static constexpr int bItemEmpty = bItemFull + kItemRing;   // [kItemRing], 13 arrivals
  static constexpr int kNumBars = bItemEmpty + kItemRing;
  static constexpr int kMisc = kBar + 8 * kNumBars;   // tmem slot, abort flag, -, wait limit
  static constexpr int kRing = kMisc + 16;
  static constexpr int kSmemBytes = kRing + 4 * kItemRing;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

constexpr int kWBwdThreads = 448;   // 14 warps

template <bool F16>
__global__ void __launch_bounds__(kWBwdThreads, 1)
fa_bwd_wide_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                   const __grid_constant__ CUtensorMap tdq, const BwdParams p, const float scale) {
  using L = WBwdLayout;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int BH = p.B * p.H;
  const int VH = 2 * BH;   // (batch-head, half of the head dimension)
  const int Np = p.nT * kTile;
  const int total = p.nT * VH;
  struct Item {
    int kj, bh, hd, kvl;
  };
  // items: groups of p.group heads (both halves of each), within a group low
  // key tiles first; handed out in order from the work counter
  auto item_at = [&](int item) -> Item {
    Item w;
    int vh = 0;
    w.kj = split_grouped(item, 2 * p.group, p.nT, VH, &vh);
    w.bh = vh >> 1;
    w.hd = vh & 1;
    w.kvl = effective_kv_len(p.kv_len, w.bh / p.H, p.N);
    return w;
  };
  auto next_live = [&](const Item& w, int i) -> int {
    while (i < p.nT && tile_state(i, w.kj, w.kvl, p.nT, p.causal, p.block_mask) == kSkip) ++i;
    return i;
  };
  // the 64-query sub-tiles of an item: (i, 0) and, unless it starts past N, (i, 1)
  auto advance = [&](const Item& w, int& i, int& sub) {
    if (sub == 0 && kTile * i + 64 < p.N) {
      sub = 1;
    } else {
      i = next_live(w, i + 1);
      sub = 0;
    }
  };

  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * (uint32_t)i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = misc + 1;
  Ctl ctl{p.err, abort_flag};
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::kRing);
  auto take_item = [&](int k, bool warp_wide, bool& ok) -> int {
    const int rs = k % L::kItemRing;
    const uint32_t ph = (uint32_t)(k / L::kItemRing) & 1u;
    ok = warp_wide ? mbar_wait_warp(bar(L::bItemFull + rs), ph, ctl, 155)
                   : mbar_wait(bar(L::bItemFull + rs), ph, ctl, 155);
    if (!ok) return -1;
    const int item = ring[rs];
    if (warp_wide)
      mbar_arrive_warp(bar(L::bItemEmpty + rs));
    else
      mbar_arrive(bar(L::bItemEmpty + rs));
    return item;
  };

  if ((sbase & 1023u) != 0u) {
    if (tid == 0) {
      uint32_t dummy = 0;   // report_error writes only the abort flag
      Ctl c0{p.err, &dummy};
      report_error(c0, kErrSmemAlign, 150);
    }
    return;
  }
  if (tid == 0) {
    for (int i = 0; i < L::kNumBars; ++i)
      mbar_init(bar(i), (i == L::bPFull || i == L::bdSFull || i == L::bKVFree) ? 8u
                        : i == L::bdQFree ? 4u
                        : i >= L::bItemEmpty ? 13u : 1u);
    abort_flag[0] = 0u;
    abort_flag[2] = p.chk.wait_us;   // the wait limit, read by the slow path of every wait
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(misc), 512);
    tmem_relinquish();
  }
  grid_dep_wait();   // global memory only from here on (programmatic dependent launch)
  grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint32_t tS = tmem;           // S^T, then P^T (cols +0..15 per warpgroup) and dS^T (+16..31)
  const uint32_t tP = tmem + 64u;     // dP^T
  const uint32_t tQ = tmem + 128u;    // dQ^T of the half
  const uint32_t tdV = tmem + 192u;
  const uint32_t tdK = tmem + 320u;

  if (warp == 12) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tq);
      tma_prefetch_map(&tk);
      tma_prefetch_map(&tv);
      tma_prefetch_map(&tdo);
      int nq = 0, nd = 0, nkv = 0, g = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int rs = k % L::kItemRing;
        if (k >= L::kItemRing &&
            !(ok = mbar_wait(bar(L::bItemEmpty + rs), (uint32_t)(k / L::kItemRing - 1) & 1u, ctl, 154)))
          break;
        const int item = k == 0 ? (int)blockIdx.x : (int)gridDim.x + (int)atomicAdd(p.sched, 1u);
        ring[rs] = item < total ? item : -1;
        mbar_arrive(bar(L::bItemFull + rs));
        if (item >= total) break;
        const Item w = item_at(item);
        int i = next_live(w, 0), sub = 0;
        // K and V of the item once the previous item's stores have read their staging
        if (k >= 1 && !(ok = mbar_wait(bar(L::bKVFree), (uint32_t)(k - 1) & 1u, ctl, 153))) break;
        if (i < p.nT) {
          mbar_arrive_expect_tx(bar(L::bKV), 2u * 65536u);
          for (int a = 0; a < 4; ++a) {
            tma_load_3d(sbase + L::kK + a * 16384, &tk, bar(L::bKV), 64 * a, kTile * w.kj, w.bh);
            tma_load_3d(sbase + L::kV + a * 16384, &tv, bar(L::bKV), 64 * a, kTile * w.kj, w.bh);
          }
        } else {
          mbar_arrive(bar(L::bKV));
        }
        ++nkv;
        for (; i < p.nT; advance(w, i, sub), ++g) {
          if (p.chk.stall != 0u && g >= 1) { ok = false; break; }   // test of the timeout path
          const int q0 = kTile * i + 64 * sub;
          if (g >= 1 && !(ok = mbar_wait(bar(L::bQEmpty), (uint32_t)(g - 1) & 1u, ctl, 151))) break;
          mbar_arrive_expect_tx(bar(L::bQFull), 32768u + 512u);
          for (int a = 0; a < 4; ++a) tma_load_3d(sbase + L::kQ + a * 8192, &tq, bar(L::bQFull), 64 * a, q0, w.bh);
          const size_t roff = (size_t)w.bh * Np + (size_t)q0;
          bulk_load(sbase + L::kRow, p.lse2 + roff, 256, bar(L::bQFull));
          bulk_load(sbase + L::kRow + 256, p.delta + roff, 256, bar(L::bQFull));
          ++nq;
          if (g >= 1 && !(ok = mbar_wait(bar(L::bdOEmpty), (uint32_t)(g - 1) & 1u, ctl, 152))) break;
          mbar_arrive_expect_tx(bar(L::bdOFull), 32768u);
          for (int a = 0; a < 4; ++a) tma_load_3d(sbase + L::kdO + a * 8192, &tdo, bar(L::bdOFull), 64 * a, q0, w.bh);
          ++nd;
        }
      }
      if (nkv > 0) drain_wait(bar(L::bKV), (uint32_t)(nkv - 1) & 1u);
      if (nq > 0) drain_wait(bar(L::bQFull), (uint32_t)(nq - 1) & 1u);
      if (nd > 0) drain_wait(bar(L::bdOFull), (uint32_t)(nd - 1) & 1u);
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_16<F16>(128, 64, false, false);
      constexpr uint32_t idA = idesc_16<F16>(128, 128, false, true);
      constexpr uint32_t idQ = idesc_16<F16>(128, 64, true, true);
      const uint32_t sK = sbase + L::kK, sV = sbase + L::kV, sQ = sbase + L::kQ, sdO = sbase + L::kdO;
      const uint32_t sdS = sbase + L::kdS;
      bool ok = true;
      int g = 0;
      for (int k = 0; ok; ++k) {
        const int item = take_item(k, false, ok);
        if (item < 0) break;
        const Item w = item_at(item);
        int i = next_live(w, 0), sub = 0;
        if (i >= p.nT) continue;
        if (!(ok = mbar_wait(bar(L::bKV), (uint32_t)k & 1u, ctl, 160))) break;
        const uint32_t hq = (uint32_t)w.hd * 2u * 8192u;     // columns of half hd in a 64-row tile
        const uint32_t hk = (uint32_t)w.hd * 2u * 16384u;    // ... in a 128-row tile
        for (int it = 0; i < p.nT; advance(w, i, sub), ++it, ++g) {
          // S^T = K Q^T
          if (!(ok = mbar_wait(bar(L::bQFull), (uint32_t)g & 1u, ctl, 161))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 16; ++ks)
            mma_ss(tS, desc_kmajor(sK, ks), desc_kmajor_at(sQ, ks, 8192u), idS, ks > 0 ? 1u : 0u);
          mma_commit(bar(L::bSFull));
          // dP^T = V dO^T
          if (!(ok = mbar_wait(bar(L::bdOFull), (uint32_t)g & 1u, ctl, 162))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 16; ++ks)
            mma_ss(tP, desc_kmajor(sV, ks), desc_kmajor_at(sdO, ks, 8192u), idS, ks > 0 ? 1u : 0u);
          mma_commit(bar(L::bdPFull));
          // dV_h += P^T dO_h (P^T of queries 0-31 packed in S columns 0-15, of 32-63 in 32-47)
          if (!(ok = mbar_wait(bar(L::bPFull), (uint32_t)g & 1u, ctl, 163))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts(tdV, tS + 32u * (uint32_t)(ks >> 1) + 8u * (uint32_t)(ks & 1), desc_mnmajor_at(sdO + hq, ks, 8192u),
                   idA, (it > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar(L::bdOEmpty));   // dO read by dP^T and dV
          // dK_h += dS^T Q_h (dS^T packed in S columns 16-31 and 48-63)
          if (!(ok = mbar_wait(bar(L::bdSFull), (uint32_t)g & 1u, ctl, 164))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts(tdK, tS + 16u + 32u * (uint32_t)(ks >> 1) + 8u * (uint32_t)(ks & 1),
                   desc_mnmajor_at(sQ + hq, ks, 8192u), idA, (it > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar(L::bQEmpty));    // Q (and its row statistics) read for the last time
          // dQ_h^T = K_h^T dS^T, once the previous partial has left its columns
          if (g > 0 && !(ok = mbar_wait(bar(L::bdQFree), (uint32_t)(g - 1) & 1u, ctl, 165))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            mma_ss(tQ, desc_mnmajor(sK + hk, ks), desc_mnmajor(sdS, ks), idQ, ks > 0 ? 1u : 0u);
          mma_commit(bar(L::bdQFull));
          mma_commit(bar(L::bdSEmpty));
        }
        if (ok) mma_commit(bar(L::bFinal));
      }
      mma_commit(bar(L::bDrain));
      drain_wait(bar(L::bDrain), 0);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ P and dS (thread = key row)
    const int cw = warp >> 2;
    const int cb = 32 * cw;   // query columns of this warpgroup
    const int r = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g = 0, nf = 0;
    for (int k = 0; ok; ++k) {
      const int item = take_item(k, true, ok);
      if (item < 0) break;
      const Item w = item_at(item);
      const int krow = kTile * w.kj + r;
      int i = next_live(w, 0), sub = 0;
      const bool live = i < p.nT;
      for (; i < p.nT; advance(w, i, sub), ++g) {
        const bool partial = tile_state(i, w.kj, w.kvl, p.nT, p.causal, p.block_mask) == kPartial;
        if (!(ok = mbar_wait_warp(bar(L::bQFull), (uint32_t)g & 1u, ctl, 170))) break;
        if (!(ok = mbar_wait_warp(bar(L::bSFull), (uint32_t)g & 1u, ctl, 171))) break;
        tc_fence_after();
        if (p.chk.rec != nullptr && tid == 0 && w.hd == 0 && sub == 0)   // the tile as this kernel computes it
          record_tile(p.chk.rec, w.bh, i, w.kj, p.nT, partial);
        const float* lse2 = reinterpret_cast<const float*>(smem + L::kRow) + cb;
        const float* dlt = lse2 + 64;
        float x[32];
        {
          uint32_t u[32];
          tmem_ld32(tS + lane_off + (uint32_t)cb, u);
          tmem_ld_wait(u);
#pragma unroll
          for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(u[c]);
        }
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 lq = reinterpret_cast<const float4*>(lse2)[c4];
          x[4 * c4] = ex2(fmaf(x[4 * c4], sl2, -lq.x));
          x[4 * c4 + 1] = ex2(fmaf(x[4 * c4 + 1], sl2, -lq.y));
          x[4 * c4 + 2] = ex2(fmaf(x[4 * c4 + 2], sl2, -lq.z));
          x[4 * c4 + 3] = ex2(fmaf(x[4 * c4 + 3], sl2, -lq.w));
        }
        if (partial) {
          const int q0 = kTile * i + 64 * sub + cb;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if ((p.causal && krow > q0 + c) || krow >= w.kvl) x[c] = 0.f;
        }
        {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = pack2<F16>(x[2 * c], x[2 * c + 1]);
          tmem_st16(tS + lane_off + (uint32_t)cb, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(bar(L::bPFull));
        if (!(ok = mbar_wait_warp(bar(L::bdPFull), (uint32_t)g & 1u, ctl, 172))) break;
        if (g > 0 && !(ok = mbar_wait_warp(bar(L::bdSEmpty), (uint32_t)(g - 1) & 1u, ctl, 173))) break;
        tc_fence_after();
        {
          uint32_t u[32];
          tmem_ld32(tP + lane_off + (uint32_t)cb, u);
          tmem_ld_wait(u);
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float2 dl = reinterpret_cast<const float2*>(dlt)[c];
            pk[c] = pack2<F16>(x[2 * c] * (__uint_as_float(u[2 * c]) - dl.x),
                               x[2 * c + 1] * (__uint_as_float(u[2 * c + 1]) - dl.y));
          }
          tmem_st16(tS + lane_off + (uint32_t)cb + 16u, pk);
          // the same dS^T row into the swizzled smem tile read by dQ^T
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int col = cb + 8 * k4;
            uint8_t* dst = smem + L::kdS + (r >> 3) * 1024 + (r & 7) * 128 + (((col >> 3) ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
          }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive_warp(bar(L::bdSFull));
      }
      // epilogue: warpgroup 0 stores dV, warpgroup 1 scale * dK, the item's
      // 128 columns, staged in the V or K buffer once every MMA has read it;
      // each warp stores its own 32 key rows
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      if (!(ok = mbar_wait_warp(bar(L::bKV), (uint32_t)k & 1u, ctl, 174))) break;
      if (live && !(ok = mbar_wait_warp(bar(L::bFinal), (uint32_t)nf & 1u, ctl, 175))) break;
      nf += live ? 1 : 0;
      tc_fence_after();
      const uint32_t tacc = (cw == 0 ? tdV : tdK) + lane_off;
      const float mul = (cw == 0) ? 1.f : scale;
      const int stage_off = cw == 0 ? L::kV : L::kK;
      uint8_t* stage = smem + stage_off;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
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
          const int col = 32 * cc + 8 * k4;
          uint8_t* dst = stage + (col >> 6) * 16384 + (r >> 3) * 1024 + (r & 7) * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int row0 = kTile * w.kj + 32 * (warp & 3);
        if (row0 < p.N)
          for (int a = 0; a < 2; ++a) {
            const int x0 = 128 * w.hd + 64 * a;
            if (x0 < p.d)
              tma_store_3d(cw == 0 ? &tdv : &tdk, sbase + stage_off + a * 16384 + 4096 * (warp & 3), x0, row0, w.bh);
          }
        bulk_commit_group();
        bulk_wait_group_read_all();   // one K/V buffer: the next item's loads wait for this
        mbar_arrive(bar(L::bKVFree));
      }
    }
    if (lane == 0) bulk_wait_group_read_all();
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ drain (thread = head-dimension column)
    // dQ_h^T in TMEM (lane = column c of the half, 64 query columns) -> two
    // rounds of 32 queries, each warp staging [32 query rows x its 32 fp32
    // columns] (128-byte swizzled) and adding it into the accumulator with TMA
    // reduce-add
    const int dw = warp - 8;
    const uint32_t lane_off = (uint32_t)(dw * 32) << 16;
    uint8_t* stage = smem + L::kdQ + 4096 * dw;
    bool ok = true;
    int g = 0;
    bool pending = false;   // this warp has a reduction whose staging may still be read
    for (int k = 0; ok; ++k) {
      const int item = take_item(k, true, ok);
      if (item < 0) break;
      const Item w = item_at(item);
      int i = next_live(w, 0), sub = 0;
      for (; i < p.nT; advance(w, i, sub), ++g) {
        if (!(ok = mbar_wait_warp(bar(L::bdQFull), (uint32_t)g & 1u, ctl, 180))) break;
        tc_fence_after();
        uint32_t u0[32], u1[32];
        tmem_ld32(tQ + lane_off, u0);
        tmem_ld32(tQ + lane_off + 32u, u1);
        tmem_ld_wait(u0);
        tmem_ld_wait(u1);
        tc_fence_before();
        mbar_arrive_warp(bar(L::bdQFree));
#pragma unroll
        for (int round = 0; round < 2; ++round) {
          if (pending) {
            if (lane == 0) bulk_wait_group_read_all();
            __syncwarp();
          }
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const uint32_t v = round == 0 ? u0[q] : u1[q];
            *reinterpret_cast<uint32_t*>(stage + q * 128 + ((((lane >> 2) ^ (q & 7)) << 4) | ((lane & 3) << 2))) = v;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int x0 = 128 * w.hd + 32 * dw;
            if (x0 < p.d) tma_reduce_add_3d(&tdq, smem_u32(stage), x0, kTile * i + 64 * sub + 32 * round, w.bh);
            bulk_commit_group();
          }
          pending = true;
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D>
cudaError_t launch_fwd_single_d(bool f16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, const FwdParams& p, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static PerDeviceOnce smem_set[2];
  auto kern = f16 ? fa_fwd_wide_kernel<D, true> : fa_fwd_wide_kernel<D, false>;
  e = once_per_device(smem_set[f16 ? 1 : 0], dev, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, WFwdLayout<D>::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  FwdParams q = p;
  q.group = l2_head_group(4.0 * p.N * p.d, p.B * p.H);
  const dim3 grid((unsigned)(p.nT * p.B * p.H));
  return launch_pdl(true, kern, grid, dim3(kWFwdThreads), WFwdLayout<D>::kSmemBytes, s, tq, tk, tv, to, q);
}

// Only the 256-column instance is used: at 64 and 128 columns the two-Q-tile
// kernel of fa_fwd.cu was measured faster (per-CTA set-up and epilogue are
// paid twice as often with one Q tile per CTA).
cudaError_t launch_fwd_single(int kd, bool f16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, const FwdParams& p, cudaStream_t s) {
  if (kd == 256) return launch_fwd_single_d<256>(f16, tq, tk, tv, to, p, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_wide(bool f16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const CUtensorMap& tdq, const BwdParams& p, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static PerDeviceOnce smem_set[2];
  auto kern = f16 ? fa_bwd_wide_kernel<true> : fa_bwd_wide_kernel<false>;
  e = once_per_device(smem_set[f16 ? 1 : 0], dev, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, WBwdLayout::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  BwdParams q = p;
  q.group = l2_head_group(8.0 * p.N * p.d, p.B * p.H);
  const long long items = 2LL * p.nT * p.B * p.H;
  const dim3 grid((unsigned)(items < sms ? items : sms));
  const float scale = p.scale_log2 / 1.4426950408889634f;
  return launch_pdl(true, kern, grid, dim3(kWBwdThreads), WBwdLayout::kSmemBytes, s, tq, tk, tv, tdo, tdk, tdv, tdq, q, scale);
}

}  // namespace fa
