// Pair variant of the attention forward for d = 128: clusters of two CTAs on
// two SMs issue tcgen05 MMAs with cta_group::2 (M = 256).
//
// Each CTA keeps its own two 128-row query tiles (a work unit is 512 query
// rows of one (b,h): rows rank*256 .. rank*256+255 of it belong to CTA
// `rank`).  For S = Q K^T the 128-key tile is split by keys: CTA r loads keys
// 64r .. 64r+63 of it; for O += P V the value tile is split by columns: CTA r
// loads value columns 64r .. 64r+63 of all 128 keys.  One thread of the
// leader CTA (rank 0) issues every MMA; each MMA reads both CTAs' shared
// memory at the same offsets and writes each CTA's own TMEM rows.  Compared
// with one CTA per tile, every SM fetches half of the B operand per MMA and
// half of the K/V bytes per key tile, which lets the MMAs run at the full
// tensor rate.
//
// Hand-offs: TMA loads of both CTAs complete on the leader's "full" barriers
// (the leader's producer posts the byte count of both halves); MMA completion
// is multicast to the barriers of both CTAs; each softmax warp reports P-ready
// on the leader's barrier.  Every wait is bounded like the single-CTA kernel's.
//
// kQK8 selects e4m3 queries and keys: S = Q K^T runs as kind::f8f6f4 MMAs (32
// bytes of K per instruction, half the tensor time of bf16 for the same
// product), with the per-tensor dequantisation scales folded into the softmax
// scale.  P and V stay bf16, so the second product and the softmax are
// unchanged.  A query tile and a key half are one 128-byte-wide box each; the
// shared memory this frees over bf16 holds two more pipeline stages.
//
// kPV8 (with kQK8) also takes e4m3 values: P is rounded to e4m3 in the softmax
// (four keys per TMEM column, so P takes 16 of a half-row's 64 S columns) and
// O += P V runs as kind::f8f6f4 with V's 128 keys x 64 columns per CTA in a
// 64-byte-swizzled half.  Probabilities carry an offset of 2^3 against the
// running max and the lazy rescale threshold is 5, so every stored p is at
// most 448 (e4m3's largest finite value; 2^8 after a max pass) and at least
// 2^-6 (its smallest normal) unless it is under 2^-9 of the row's largest.
// The row sum adds the fp32 probabilities before their rounding (two paired
// adds per four keys; summing the rounded values through an f16 widening took
// 10% more cycles), so every weight carries only its own rounding error.  The
// per-tensor value scale is applied with 1/l in the epilogue.
#pragma once

namespace dit {

// Warp roles of the pair kernel (640 threads, five warpgroups): warps 0-7
// run the softmax of query tile 0 and warps 8-15 that of tile 1, so the two
// warps of a tile on an SM sub-partition have two partners working on the
// other tile while they wait; warp 16 issues the MMAs (leader CTA) and owns
// TMEM, warp 17 loads, warps 18-19 only complete the fifth warpgroup.
// Registers: launched at 96 per thread (640 x 96 = 61440); the four softmax
// warpgroups raise to 112 and the fifth drops to 32: 512 x 112 + 128 x 32 =
// 61440.
constexpr int kPairThreads = 640;
constexpr int kPairMmaWarp = 16;
constexpr int kPairLoadWarp = 17;
constexpr int kPairRegsSoftmax = 112;
constexpr int kPairRegsOther = 32;

// e4m3 probabilities: p = 2^(x - m + kProbOffsetE4M3) with the lazy rescale at
// kRescaleThresholdE4M3, so p <= 2^8 after a max pass; an optimistic pass is
// kept while the sum of each thread's 64 values stays below 448 (no value
// saturated).  With RMS-normalised logits the half-row sum of a key tile is
// about 2^6 at this offset, so the optimistic pass holds; testing the whole
// row's sum instead sent 4% more SM cycles into needless max passes, and at
// an offset of 2^4 the row sum would exceed 448 on most warp steps.
constexpr float kProbOffsetE4M3 = 3.0f;
constexpr float kRescaleThresholdE4M3 = 5.0f;
constexpr float kOptimisticSumLimitE4M3 = 448.0f;

template <bool kQK8, bool kPV8 = false>
struct PairTraitsT {
  static_assert(kQK8 || !kPV8, "e4m3 values come with e4m3 queries and keys");
  static constexpr bool kP8 = kPV8;
  static constexpr int D = 128;
  static constexpr int kBoxCols = 64;                       // bf16 columns in a 128-byte box row
  static constexpr int kQKBoxes = kQK8 ? 1 : 2;             // 128-byte boxes across d for Q, K
  static constexpr uint32_t kQBoxBytes = 128u * 128u;       // 128 rows x 128 bytes
  static constexpr uint32_t kQTileBytes = kQKBoxes * kQBoxBytes;   // one 128-row query tile
  static constexpr uint32_t kKBoxBytes = 64u * 128u;        // 64 keys x 128 bytes
  static constexpr uint32_t kKHalfBytes = kQKBoxes * kKBoxBytes;   // one K half
  static constexpr uint32_t kVHalfBytes = kPV8 ? 128u * 64u : 128u * 128u;  // 128 keys x 64 columns
  // A ring slot holds what one key-tile iteration of the MMA warp reads:
  // V(j) for P.V and K(j+1) for the next Q K^T (the first slot of a work
  // item holds K(0) alone, its last slot V(n-1) alone).  K at offset 0, V
  // after it.
  static constexpr uint32_t kSlotBytes = kKHalfBytes + kVHalfBytes;
  static constexpr int kStages = kPV8 ? 10 : (kQK8 ? 6 : 4);   // ring slots
  __host__ __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + 128u * t; }
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKV = 2 * kQTileBytes;
  static constexpr uint32_t kOffBar = kOffKV + kStages * kSlotBytes;
  static constexpr int kBarFull = 0;                 // leader: both CTAs' copies of a slot landed
  static constexpr int kBarEmpty = kStages;          // both: the slot may be refilled
  static constexpr int kBarQFull = 2 * kStages;      // leader: both CTAs' query tile t landed
  static constexpr int kBarQEmpty = kBarQFull + 2;   // both
  static constexpr int kBarSFull = kBarQEmpty + 2;   // both
  static constexpr int kBarPFull = kBarSFull + 2;    // leader: 16 warp arrivals
  static constexpr int kBarOFull = kBarPFull + 2;    // both
  static constexpr int kBarDrain = kBarOFull + 2;    // leader
  static constexpr int kBarProdDone = kBarDrain + 1; // leader: both producers reported
  static constexpr int kNumBars = kBarProdDone + 1;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = 1024 + kOffMisc + kMiscWords * 4;
  static constexpr uint32_t kPFullArrivals = 16;     // 8 softmax warps x 2 CTAs
};
using PairTraits = PairTraitsT<false>;

// ----------------------------------------------------------------- producer (both CTAs)
template <bool kQK8, bool kPV8>
__device__ void pair_load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                               const CUtensorMap* tmV, const Params& p, const Shared& sh) {
  using T = PairTraitsT<kQK8, kPV8>;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint64_t pol_kv = policy_evict_last();
  const uint64_t pol_q = policy_evict_first();
  const uint32_t full0_leader = mapa_shared(sh.bar(T::kBarFull), 0);
  const uint32_t qfull0_leader = mapa_shared(sh.bar(T::kBarQFull), 0);
  // fills: slot fills issued so far (slot = fills mod kStages); each fill's
  // byte count (this CTA's share) is kept per slot in the misc words;
  // q_loads0/1: query-tile-0/1 copies issued so far.  All are left in shared
  // memory for the teardown drain.
  uint32_t stage = 0, phase = 0, fills = 0, it = 0, q_loads0 = 0, q_loads1 = 0;
  bool ok = true;
  const int n_kv = (p.Lk + kBN - 1) / kBN;

  auto load_q = [&](int t, int bh, int row0) -> bool {
    if (!mbar_wait(sh.bar(T::kBarQEmpty + t), (it & 1u) ^ 1u, kWaitLimitNs, sh.abort)) return false;
    const uint32_t dst = sh.base + T::kOffQ + t * T::kQTileBytes;
    if (leader) mbar_arrive_expect_tx(sh.bar(T::kBarQFull + t), 2 * T::kQTileBytes);
    for (int b = 0; b < T::kQKBoxes; ++b)
      tma_load_3d_pair(dst + b * T::kQBoxBytes, tmQ, qfull0_leader + 8u * t, b * T::kBoxCols,
                       row0 + t * kBM, bh, pol_q);
    if (t == 0) ++q_loads0;
    else ++q_loads1;
    return true;
  };
  auto take_empty = [&](uint32_t bytes) -> bool {   // bytes: this CTA's copies into the slot
    if (!mbar_wait(sh.bar(T::kBarEmpty + stage), phase ^ 1u, kWaitLimitNs, sh.abort)) return false;
    if (leader) mbar_arrive_expect_tx(sh.bar(T::kBarFull + stage), 2 * bytes);
    st_shared_u32(sh.misc_word(kMiscSlotBytes + static_cast<int>(stage)), bytes);
    return true;
  };
  auto slot_base = [&]() { return sh.base + T::kOffKV + stage * T::kSlotBytes; };
  auto load_k = [&](int j, int bh) {   // keys j*128 + 64*rank .. +63, all d columns
    for (int b = 0; b < T::kQKBoxes; ++b)
      tma_load_3d_pair(slot_base() + b * T::kKBoxBytes, tmK, full0_leader + 8u * stage,
                       b * T::kBoxCols, j * kBN + static_cast<int>(rank) * 64, bh, pol_kv);
  };
  auto load_v = [&](int j, int bh) {   // keys j*128 .. +127, columns 64*rank .. +63
    tma_load_3d_pair(slot_base() + T::kKHalfBytes, tmV, full0_leader + 8u * stage,
                     static_cast<int>(rank) * 64, j * kBN, bh, pol_kv);
  };
  auto advance = [&]() {
    ++fills;
    if (++stage == T::kStages) { stage = 0; phase ^= 1u; }
  };

  for (int i = static_cast<int>(cluster_id_x()); i < p.num_items && ok;
       i += static_cast<int>(num_clusters_x()), ++it) {
    const WorkItem w = work_item(i, p, n_kv);
    const int bh = w.bh;
    const int row0 = w.qblock * (2 * kUnitRows) + static_cast<int>(rank) * kUnitRows;
    ok = load_q(0, bh, row0) && take_empty(T::kKHalfBytes);
    if (!ok) break;
    load_k(w.j0, bh);   // the item's first slot: K(j0)
    advance();
    ok = load_q(1, bh, row0);
    for (int j = w.j0; j < w.j1 && ok; ++j) {
      const bool more = j + 1 < w.j1;
      ok = take_empty(T::kVHalfBytes + (more ? T::kKHalfBytes : 0u));
      if (!ok) break;
      load_v(j, bh);
      if (more) load_k(j + 1, bh);
      advance();
    }
  }
  if (!ok) record_timeout<true>(sh);
  // Report the copies issued to the leader (for the teardown drain).
  if (leader) {
    st_shared_u32(sh.misc_word(kMiscFills), fills);
    st_shared_u32(sh.misc_word(kMiscQLoads), q_loads0);
    st_shared_u32(sh.misc_word(kMiscQLoads + 1), q_loads1);
    mbar_arrive(sh.bar(T::kBarProdDone));
  } else {
    st_shared_cluster_u32(mapa_shared(sh.misc_word(kMiscPeerFills), 0), fills);
    st_shared_cluster_u32(mapa_shared(sh.misc_word(kMiscPeerQLoads), 0), q_loads0);
    st_shared_cluster_u32(mapa_shared(sh.misc_word(kMiscPeerQLoads + 1), 0), q_loads1);
    mbar_arrive_release_cluster(mapa_shared(sh.bar(T::kBarProdDone), 0));
  }
}

// Teardown after a bounded wait gave up (one thread of the leader CTA, once
// its own role has returned): every copy either CTA issued must land before
// the CTAs' shared memory goes away.  Both producers report how many copies
// they issued and arrive on the leader's producer-done barrier.  All copies
// complete on the leader's barriers, and a barrier phase only completes when
// the leader armed it for both CTAs' shares and both landed, but the two
// producers may have stopped at different points.  For each of the last
// kStages slot fills and each query tile's last load, the leader balances the
// phase: where only the leader issued the fill it retires the peer's share of
// the bytes itself (mbarrier.complete_tx), where only the peer did it arms the
// phase for the peer's share alone; then it waits (bounded) for the phase.
template <class T>
__device__ void pair_teardown_drain(const Shared& sh) {
  const volatile int no_abort = 0;
  if (!mbar_wait_acquire_cluster(sh.bar(T::kBarProdDone), 0, kWaitLimitNs)) return;
  auto word = [&](int i) { return ld_shared_u32(sh.misc_word(i)); };
  auto balance_and_wait = [&](uint32_t bar, bool by_leader, bool by_peer, uint32_t half_bytes,
                              uint32_t parity) {
    if (by_leader && !by_peer) mbar_complete_tx(bar, half_bytes);
    if (by_peer && !by_leader) mbar_arrive_expect_tx(bar, half_bytes);
    mbar_wait(bar, parity, kWaitLimitNs, &no_abort);
  };
  // fill counts of the two producers differ by at most kStages (each waits
  // for the consumption of the fill kStages back, which needs both halves);
  // each CTA keeps its share of every slot's bytes, the peer's read remotely
  const uint32_t fl = word(kMiscFills), fp = word(kMiscPeerFills);
  const uint32_t last = static_cast<int32_t>(fp - fl) > 0 ? fp : fl;
  const uint32_t window = last < static_cast<uint32_t>(T::kStages) ? last : T::kStages;
  for (uint32_t k = 1; k <= window; ++k) {
    const uint32_t f = last - k;
    const int slot = static_cast<int>(f % T::kStages);
    const bool by_leader = static_cast<int32_t>(f - fl) < 0, by_peer = static_cast<int32_t>(f - fp) < 0;
    const uint32_t bytes =
        by_leader ? word(kMiscSlotBytes + slot)
                  : ld_shared_cluster_u32(mapa_shared(sh.misc_word(kMiscSlotBytes + slot), 1u));
    balance_and_wait(sh.bar(T::kBarFull + slot), by_leader, by_peer, bytes, (f / T::kStages) & 1u);
  }
  // query tiles: the two producers' load counts differ by at most one
  for (int t = 0; t < 2; ++t) {
    const uint32_t ql = word(kMiscQLoads + t), qp = word(kMiscPeerQLoads + t);
    const uint32_t q_last = static_cast<int32_t>(qp - ql) > 0 ? qp : ql;
    if (q_last == 0) continue;
    balance_and_wait(sh.bar(T::kBarQFull + t), ql == q_last, qp == q_last, T::kQTileBytes,
                     (q_last - 1u) & 1u);
  }
}

// ----------------------------------------------------------------- MMA issuer (leader CTA)
template <bool kQK8>
__device__ __forceinline__ void pair_issue_qk(uint32_t d_tmem, uint32_t q_lo, uint32_t k_lo) {
  using T = PairTraitsT<kQK8, false>;
  constexpr uint32_t hi = desc_hi_sw128(1024);
  if constexpr (kQK8) {
    // one 128-byte box row holds all of d; each instruction takes 32 bytes of it
    constexpr uint32_t idesc = idesc_e4m3_f32(2 * kBM, kBN);
#pragma unroll
    for (int k = 0; k < T::D / 32; ++k)
      mma_ss_lo_pair_f8(d_tmem, q_lo + ((k * 32) >> 4), k_lo + ((k * 32) >> 4), hi, idesc,
                        k > 0 ? 1u : 0u);
  } else {
    constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, kBN, 0, 0);
#pragma unroll
    for (int k = 0; k < T::D / 16; ++k) {
      const uint32_t a_off = ((k / 4) * T::kQBoxBytes + (k % 4) * 32) >> 4;
      const uint32_t b_off = ((k / 4) * T::kKBoxBytes + (k % 4) * 32) >> 4;
      mma_ss_lo_pair(d_tmem, q_lo + a_off, k_lo + b_off, hi, idesc, k > 0 ? 1u : 0u);
    }
  }
}

template <bool kPV8>
__device__ __forceinline__ void pair_issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_lo,
                                              bool accumulate) {
  if constexpr (kPV8) {
    // e4m3 P of keys [64h, 64h+64) is in S columns [64h, 64h+16); V rows are
    // 64 bytes, so 32 keys (one instruction) span 2048 bytes
    constexpr uint32_t idesc = idesc_e4m3_f32(2 * kBM, PairTraits::D, 0, 1);
    constexpr uint32_t hi = desc_hi_sw64(512);
#pragma unroll
    for (int k = 0; k < kBN / 32; ++k)
      mma_ts_lo_pair_f8(d_tmem, p_tmem + (k / 2) * 64 + (k % 2) * 8,
                        v_lo + ((k * 32 * 64) >> 4), hi, idesc, (accumulate || k > 0) ? 1u : 0u);
  } else {
    constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, PairTraits::D, 0, 1);
    constexpr uint32_t hi = desc_hi_sw128(1024);
#pragma unroll
    for (int k = 0; k < kBN / 16; ++k)   // P of keys [64h, 64h+64) is in S columns [64h, 64h+32)
      mma_ts_lo_pair(d_tmem, p_tmem + (k / 4) * 64 + (k % 4) * 8, v_lo + ((k * 16 * 128) >> 4),
                     hi, idesc, (accumulate || k > 0) ? 1u : 0u);
  }
}

template <bool kQK8, bool kPV8>
__device__ void pair_mma_role(const Params& p, const Shared& sh, uint32_t tmem) {
  using T = PairTraitsT<kQK8, kPV8>;
  constexpr uint16_t kBoth = 3;
  const bool issuer = (threadIdx.x & 31) == 0;
  uint32_t stage = 0, phase = 0, g = 0, it = 0;
  bool ok = true;
  const int n_kv = (p.Lk + kBN - 1) / kBN;
  const uint32_t q_lo0 = desc_lo_sw128(sh.base + T::kOffQ, 16);
  const uint32_t q_lo1 = desc_lo_sw128(sh.base + T::kOffQ + T::kQTileBytes, 16);
  const uint32_t kv_lo0 = desc_lo_sw128(sh.base + T::kOffKV, 16);
  auto k_lo = [&](uint32_t s) { return kv_lo0 + s * (T::kSlotBytes >> 4); };
  auto v_lo = [&](uint32_t s) { return k_lo(s) + (T::kKHalfBytes >> 4); };
  auto wait = [&](int bar, uint32_t parity) -> bool {
    const bool got = mbar_wait(sh.bar(bar), parity, kWaitLimitNs, sh.abort);
    return __all_sync(0xffffffffu, got);
  };
  auto take_slot = [&](uint32_t& s_out) -> bool {
    s_out = stage;
    if (!wait(T::kBarFull + stage, phase)) return false;
    if (++stage == T::kStages) { stage = 0; phase ^= 1u; }
    return true;
  };

  // One slot per key tile: iteration j reads V(j) and K(j+1) from the slot
  // taken while the warp would wait for P_1 of the iteration before, and
  // releases it with one commit.  Commits follow the MMA block they track (a
  // commit between MMAs stalls the issuing thread).
  for (int i = static_cast<int>(cluster_id_x()); i < p.num_items && ok;
       i += static_cast<int>(num_clusters_x()), ++it) {
    int n = n_kv;                // key tiles of this item
    if (i >= p.split_base) {
      const int s = (i - p.split_base) % p.splits;
      n = (s + 1) * n_kv / p.splits - s * n_kv / p.splits;
    }
    uint32_t s0 = 0, sCur = 0, sNext = 0;
    ok = wait(T::kBarQFull + 0, it & 1u) && take_slot(s0);   // K(0)
    if (!ok) break;
    tc_fence_after();
    if (issuer) {
      pair_issue_qk<kQK8>(tmem + T::col_s(0), q_lo0, k_lo(s0));
      mma_commit_pair(sh.bar(T::kBarSFull + 0), kBoth);
      if (n == 1) mma_commit_pair(sh.bar(T::kBarQEmpty + 0), kBoth);
    }
    __syncwarp();
    ok = wait(T::kBarQFull + 1, it & 1u) && take_slot(sCur);   // V(0), K(1)
    if (!ok) break;
    tc_fence_after();
    if (issuer) {
      pair_issue_qk<kQK8>(tmem + T::col_s(1), q_lo1, k_lo(s0));
      mma_commit_pair(sh.bar(T::kBarSFull + 1), kBoth);
      if (n == 1) mma_commit_pair(sh.bar(T::kBarQEmpty + 1), kBoth);
      mma_commit_pair(sh.bar(T::kBarEmpty + s0), kBoth);
    }
    __syncwarp();

    for (int j = 0; j < n && ok; ++j, ++g) {   // j: tile index within the item
      // held: sCur = V(j) (and K(j+1) when j+1 < n)
      const bool more = j + 1 < n;
      ok = wait(T::kBarPFull + 0, g & 1u);
      if (!ok) break;
      tc_fence_after();
      if (issuer) {
        pair_issue_pv<kPV8>(tmem + T::col_o(0), tmem + T::col_s(0), v_lo(sCur), j > 0);
        if (more) {
          pair_issue_qk<kQK8>(tmem + T::col_s(0), q_lo0, k_lo(sCur));
          mma_commit_pair(sh.bar(T::kBarSFull + 0), kBoth);
          if (j + 2 == n) mma_commit_pair(sh.bar(T::kBarQEmpty + 0), kBoth);
        } else {
          mma_commit_pair(sh.bar(T::kBarOFull + 0), kBoth);
        }
      }
      __syncwarp();
      if (more) ok = take_slot(sNext);   // V(j+1), K(j+2)
      ok = ok && wait(T::kBarPFull + 1, g & 1u);
      if (!ok) break;
      tc_fence_after();
      if (issuer) {
        pair_issue_pv<kPV8>(tmem + T::col_o(1), tmem + T::col_s(1), v_lo(sCur), j > 0);
        if (more) {
          pair_issue_qk<kQK8>(tmem + T::col_s(1), q_lo1, k_lo(sCur));
          mma_commit_pair(sh.bar(T::kBarSFull + 1), kBoth);
          if (j + 2 == n) mma_commit_pair(sh.bar(T::kBarQEmpty + 1), kBoth);
          mma_commit_pair(sh.bar(T::kBarEmpty + sCur), kBoth);
        } else {
          mma_commit_pair(sh.bar(T::kBarEmpty + sCur), kBoth);
          mma_commit_pair(sh.bar(T::kBarOFull + 1), kBoth);
        }
      }
      __syncwarp();
      sCur = sNext;
    }
  }
  if (!ok && issuer) record_timeout<true>(sh);
  if (issuer) {
    mma_commit_pair(sh.bar(T::kBarDrain), 1);
    const volatile int no_abort = 0;
    mbar_wait(sh.bar(T::kBarDrain), 0, kWaitLimitNs, &no_abort);
  }
  __syncwarp();
}

// ----------------------------------------------------------------- softmax (pair kernel)
// Largest scaled logit s * scale_log2 of 32 logits, keys at or beyond `valid`
// excluded (-inf when all are).  Scaling is monotone, so this is scale_log2
// times the largest raw logit when scale_log2 >= 0 and times the smallest
// when it is negative; the sign is the same for the whole launch.
template <bool kMasked>
__device__ __forceinline__ float rowmax_chunk(const uint32_t (&sr)[32], int key0, int valid,
                                              float scale_log2) {
  const bool neg = scale_log2 < 0.f;
  const float sentinel = neg ? INFINITY : -INFINITY;
  float m[4] = {sentinel, sentinel, sentinel, sentinel};
  if (!neg) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float a = __uint_as_float(sr[i]), b = __uint_as_float(sr[i + 1]);
      if (kMasked) {
        a = (key0 + i < valid) ? a : -INFINITY;
        b = (key0 + i + 1 < valid) ? b : -INFINITY;
      }
      m[(i / 2) & 3] = fmax3(m[(i / 2) & 3], a, b);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float a = __uint_as_float(sr[i]), b = __uint_as_float(sr[i + 1]);
      if (kMasked) {
        a = (key0 + i < valid) ? a : INFINITY;
        b = (key0 + i + 1 < valid) ? b : INFINITY;
      }
      m[(i / 2) & 3] = fmin3(m[(i / 2) & 3], a, b);
    }
  }
  const float e = neg ? fminf(fminf(m[0], m[1]), fminf(m[2], m[3]))
                      : fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
  return e == sentinel ? -INFINITY : e * scale_log2;
}

// Probabilities of 32 logits rounded to e4m3, four keys per word (key order =
// byte order); their fp32 values, before the rounding, are added into acc.
template <bool kMasked>
__device__ __forceinline__ void probs_chunk_e4m3(const uint32_t (&sr)[32], float scale_log2,
                                                 float neg_m, int key0, int valid, uint32_t* pk,
                                                 float (&acc)[8]) {
  const float2 sl2 = make_float2(scale_log2, scale_log2);
  const float2 nm = make_float2(neg_m, neg_m);
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const float2 x01 =
        __ffma2_rn(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), sl2, nm);
    const float2 x23 =
        __ffma2_rn(make_float2(__uint_as_float(sr[i + 2]), __uint_as_float(sr[i + 3])), sl2, nm);
    float p0, p1, p2, p3;
    if ((kExp2FmaQuadsE4M3 >> (i / 4)) & 1u) {   // this quad's exp2 on the FMA pipe
      const float2 e01 = exp2_fma_pair<2>(x01), e23 = exp2_fma_pair<2>(x23);
      p0 = e01.x;
      p1 = e01.y;
      p2 = e23.x;
      p3 = e23.y;
    } else {
      p0 = ex2_approx(x01.x);
      p1 = ex2_approx(x01.y);
      p2 = ex2_approx(x23.x);
      p3 = ex2_approx(x23.y);
    }
    if (kMasked) {
      p0 = (key0 + i < valid) ? p0 : 0.f;
      p1 = (key0 + i + 1 < valid) ? p1 : 0.f;
      p2 = (key0 + i + 2 < valid) ? p2 : 0.f;
      p3 = (key0 + i + 3 < valid) ? p3 : 0.f;
    }
    pk[i / 4] = pack_e4m3x4(p0, p1, p2, p3);
    const float2 s = __fadd2_rn(make_float2(p0, p1), make_float2(p2, p3));
    const float2 a = __fadd2_rn(make_float2(acc[(i / 4) & 3], acc[4 + ((i / 4) & 3)]), s);
    acc[(i / 4) & 3] = a.x;
    acc[4 + ((i / 4) & 3)] = a.y;
  }
}

// One query tile's softmax step for this thread's half-row (keys key0 ..
// key0+63 of the tile) with a small register footprint: the logits are read
// from TMEM 32 columns at a time, and the probabilities of both chunks are
// stored once, at the end, over the half-row's first S columns (32 for bf16,
// 16 for e4m3), so that a recompute can read the logits again.  Otherwise as
// softmax_tile_half.
template <int D, bool kP8, class ORescale>
__device__ __forceinline__ void softmax_tile_lean(uint32_t taddr_s, int key0, bool first,
                                                  bool masked, int valid, float scale_log2,
                                                  float& m_used, float& l, ORescale&& o_rescale) {
  constexpr int kPWords = kP8 ? 8 : 16;   // packed probability words per 32 keys
  constexpr float kThreshold = kP8 ? kRescaleThresholdE4M3 : kRescaleThreshold;
  uint32_t sr[32];
  uint32_t pk[2 * kPWords];
  float acc[8];
  auto load = [&](int c) {
    tmem_ld16x2_32<64>(taddr_s + 32 * c, sr);
    tmem_wait_ld();
  };
  auto probs = [&](int c, float m) {
    if constexpr (kP8) {
      const float neg_m = kProbOffsetE4M3 - m;
      if (masked) probs_chunk_e4m3<true>(sr, scale_log2, neg_m, key0 + 32 * c, valid, &pk[8 * c], acc);
      else probs_chunk_e4m3<false>(sr, scale_log2, neg_m, key0 + 32 * c, kBN, &pk[8 * c], acc);
    } else {
      if (masked) probs_chunk<true>(sr, scale_log2, -m, key0 + 32 * c, valid, &pk[16 * c], acc);
      else probs_chunk<false>(sr, scale_log2, -m, key0 + 32 * c, kBN, &pk[16 * c], acc);
    }
  };
  auto chunk_max = [&](int c) -> float {   // largest scaled logit of chunk c
    return masked ? rowmax_chunk<true>(sr, key0 + 32 * c, valid, scale_log2)
                  : rowmax_chunk<false>(sr, key0 + 32 * c, kBN, scale_log2);
  };
  auto clear = [&]() {
#pragma unroll
    for (int a = 0; a < 8; ++a) acc[a] = 0.f;
  };
  // Row max over both halves, lazy rescale of l and O, then the probabilities
  // (sr holds chunk 1 after the max, so it goes first).
  auto max_pass = [&]() {
    load(0);
    float mx = chunk_max(0);
    load(1);
    mx = fmaxf(mx, chunk_max(1));
    const float m_tile = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    float factor = 1.f;
    if (m_tile > m_used + kThreshold) {
      factor = ex2_approx(m_used - m_tile);   // 0 on the first tile
      l *= factor;
      m_used = m_tile;
    }
    if (!first && __any_sync(0xffffffffu, factor != 1.f)) o_rescale(factor);
    clear();
    probs(1, m_used);
    load(0);
    probs(0, m_used);
  };
  clear();
  if (first) {
    max_pass();
  } else {
    // Optimistic pass against the running max; each thread tests the sum of
    // its own 64 probabilities.  A rounded half-row sum above 2^48 (or an
    // overflow) means some p > 2^42: raise the max (always by more than 8),
    // rescale l and O, recompute.  With e4m3 P a half-row sum (of the fp32
    // values) of 448 or more may hide a saturated value: take the max pass.
    // The vote makes the branch warp-uniform, so both halves of a row agree.
    load(0);
    probs(0, m_used);
    load(1);
    probs(1, m_used);
    const float half_sum = sum8(acc);
    const bool redo = kP8 ? !(half_sum < kOptimisticSumLimitE4M3)
                          : !(half_sum <= kOptimisticSumLimit);
    if (__any_sync(0xffffffffu, redo)) max_pass();
  }
  if constexpr (kP8) {
    tmem_st16x2_16<64>(taddr_s, &pk[0]);
  } else {
    tmem_st16x2_16<64>(taddr_s, &pk[0]);
    tmem_st16x2_16<64>(taddr_s + 16, &pk[16]);
  }
  l += sum8(acc);
}

// Softmax and epilogue of the pair kernel: warp w works on query tile w / 8
// and, with q = w mod 8, on TMEM lanes (rows) 32*(q%4) + 16*(q/4) .. +15, two
// threads per row (lanes 0-15 take keys 0-63, lanes 16-31 keys 64-127).
// Each warp arrives once per key tile on its tile's P-ready barrier of the
// leader CTA (8 warps x 2 CTAs).
template <int D, class T>
__device__ void softmax_role_pair(const Params& p, const Shared& sh, uint32_t tmem) {
  const int warp = threadIdx.x / 32;                 // 0..15
  const int lane = threadIdx.x & 31;
  const int t = warp >> 3;                           // query tile
  const int wq = warp & 7;
  const int half = lane >> 4;                        // keys [64*half, 64*half + 64) of a tile
  const int lane0 = (wq & 3) * 32 + (wq >> 2) * 16;  // warp % 4 == wq % 4: its TMEM sub-partition
  const int r = lane0 + (lane & 15);                 // row within the query tile
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(lane0) << 16);
  const uint32_t taddr_s = lane_addr + T::col_s(t);
  const uint32_t taddr_o = lane_addr + T::col_o(t);
  const float scale_log2 = p.scale_log2;
  const int n_kv = (p.Lk + kBN - 1) / kBN;
  const int tail = p.Lk - (n_kv - 1) * kBN;          // valid keys in the last tile, 1..128
  const int key0 = 64 * half;
  const int rank = static_cast<int>(cluster_ctarank());
  const uint32_t p_full_leader = mapa_shared(sh.bar(T::kBarPFull + t), 0);
  uint32_t g = 0, it = 0;
  bool ok = true;

  for (int i = static_cast<int>(cluster_id_x()); i < p.num_items && ok;
       i += static_cast<int>(num_clusters_x()), ++it) {
    const WorkItem w = work_item(i, p, n_kv);
    float m_used = -INFINITY;   // running max, in units of s*scale*log2(e)
    float l = 0.f;              // this half-row's share of the row sum
    for (int j = w.j0; j < w.j1 && ok; ++j, ++g) {
      const bool masked = (j == n_kv - 1) && (tail < kBN);
      const int valid = masked ? tail : kBN;
      const bool got = mbar_wait(sh.bar(T::kBarSFull + t), g & 1u, kWaitLimitNs, sh.abort);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
      // O_t is quiescent here: S_t's completion implies the previous P.V
      // product into O_t finished.
      softmax_tile_lean<D, T::kP8>(taddr_s, key0, j == w.j0, masked, valid, scale_log2, m_used,
                                   l, [&](float f) { rescale_o_half<D>(taddr_o, f); });
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(p_full_leader);
    }
    if (!ok) break;
    // Epilogue: O_t / l -> bf16 -> global, each thread its D/2 columns; a
    // chunk of a split unit stores O_t, its max and row sum unnormalised.
    const bool got = mbar_wait(sh.bar(T::kBarOFull + t), it & 1u, kWaitLimitNs, sh.abort);
    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
    tc_fence_after();
    const float l_row = l + __shfl_xor_sync(0xffffffffu, l, 16);
    const int prow = rank * kUnitRows + t * kBM + r;   // row within the 512-row unit
    // e4m3 values: out = v_scale * O / l; a partial row keeps O and l / v_scale
    if (w.chunk >= 0) {
      store_partial<D>(p, static_cast<int64_t>(w.chunk) * (2 * kUnitRows) + prow, half, taddr_o,
                       m_used, T::kP8 ? l_row * p.inv_v_scale : l_row);
      continue;
    }
    const float inv_l = T::kP8 ? p.v_scale / l_row : 1.f / l_row;
    const int row = w.qblock * (2 * kUnitRows) + prow;
    const bool row_ok = row < p.Lq;
    uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(w.bh) * p.Lq + row) * D +
                                          half * (D / 2));
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      uint32_t o[32];
      tmem_ld16x2_32<D / 2>(taddr_o + c * 32, o);
      tmem_wait_ld();
      uint32_t wv[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        wv[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l);
      if (row_ok) {
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[c * 4 + v] = make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
      }
    }
  }
  if (!ok) record_timeout<true>(sh);
}

// ----------------------------------------------------------------- kernel
// Launched with a cluster dimension of 2 (consecutive CTAs form a pair).
template <bool kQK8, bool kPV8>
__global__ void __launch_bounds__(kPairThreads, 1)
    fmha_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params p) {
  using T = PairTraitsT<kQK8, kPV8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint32_t* misc = reinterpret_cast<uint32_t*>(base_ptr + T::kOffMisc);
  Shared sh;
  sh.base = base;
  sh.bar0 = base + T::kOffBar;
  sh.abort = reinterpret_cast<volatile int*>(misc + kMiscAbort);
  sh.misc = base + T::kOffMisc;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const bool leader = cluster_ctarank() == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < T::kStages; ++s) {
      mbar_init(sh.bar(T::kBarFull + s), 1);
      mbar_init(sh.bar(T::kBarEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(sh.bar(T::kBarQFull + t), 1);
      mbar_init(sh.bar(T::kBarQEmpty + t), 1);
      mbar_init(sh.bar(T::kBarSFull + t), 1);
      mbar_init(sh.bar(T::kBarPFull + t), T::kPFullArrivals);
      mbar_init(sh.bar(T::kBarOFull + t), 1);
    }
    mbar_init(sh.bar(T::kBarDrain), 1);
    mbar_init(sh.bar(T::kBarProdDone), 2);
    *sh.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == kPairLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == kPairMmaWarp) {
    tmem_alloc_pair(smem_u32(misc + kMiscTmem), T::kTmemCols);
    tmem_relinquish_pair();
  }
  // Both CTAs' barriers and TMEM exist before either CTA touches the other's.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = misc[kMiscTmem];

  if (warp < kPairMmaWarp) {
    reg_alloc<kPairRegsSoftmax>();
    softmax_role_pair<T::D, T>(p, sh, tmem);
    if (leader && threadIdx.x == 0 && *sh.abort) pair_teardown_drain<T>(sh);
  } else if (warp == kPairMmaWarp) {
    reg_dealloc<kPairRegsOther>();
    if (leader) pair_mma_role<kQK8, kPV8>(p, sh, tmem);
  } else if (warp == kPairLoadWarp) {
    reg_dealloc<kPairRegsOther>();
    if (lane == 0) pair_load_role<kQK8, kPV8>(&tmQ, &tmK, &tmV, p, sh);
    __syncwarp();
  } else {
    reg_dealloc<kPairRegsOther>();
  }

  // The leader drained its MMAs and, after a give-up, every copy either CTA
  // issued; neither CTA leaves while the pair's MMAs or copies could still
  // touch its shared memory or TMEM.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == kPairMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, T::kTmemCols);
  }
}

}  // namespace dit
