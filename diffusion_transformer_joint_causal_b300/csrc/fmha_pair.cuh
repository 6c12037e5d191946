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
#pragma once

namespace dit {

template <bool kQK8>
struct PairTraitsT {
  static constexpr int D = 128;
  static constexpr int kBoxCols = 64;                       // bf16 columns in a 128-byte box row
  static constexpr int kQKBoxes = kQK8 ? 1 : 2;             // 128-byte boxes across d for Q, K
  static constexpr uint32_t kQBoxBytes = 128u * 128u;       // 128 rows x 128 bytes
  static constexpr uint32_t kQTileBytes = kQKBoxes * kQBoxBytes;   // one 128-row query tile
  static constexpr uint32_t kKBoxBytes = 64u * 128u;        // 64 keys x 128 bytes
  static constexpr uint32_t kKHalfBytes = kQKBoxes * kKBoxBytes;   // one K half
  static constexpr uint32_t kHalfBytes = 16384;             // a stage: one V half (or K half)
  static constexpr int kStages = kQK8 ? 10 : 8;
  __host__ __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + 128u * t; }
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKV = 2 * kQTileBytes;
  static constexpr uint32_t kOffBar = kOffKV + kStages * kHalfBytes;
  static constexpr int kBarFull = 0;                 // leader: both halves of a stage landed
  static constexpr int kBarEmpty = kStages;          // both: the stage may be refilled
  static constexpr int kBarQFull = 2 * kStages;      // leader: both CTAs' query tile t landed
  static constexpr int kBarQEmpty = kBarQFull + 2;   // both
  static constexpr int kBarSFull = kBarQEmpty + 2;   // both
  static constexpr int kBarPFull = kBarSFull + 2;    // leader: 16 warp arrivals
  static constexpr int kBarOFull = kBarPFull + 2;    // both
  static constexpr int kBarDrain = kBarOFull + 2;    // leader
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = 1024 + kOffMisc + 16;
  static constexpr uint32_t kPFullArrivals = 16;     // 8 softmax warps x 2 CTAs
};
using PairTraits = PairTraitsT<false>;

// ----------------------------------------------------------------- producer (both CTAs)
template <bool kQK8>
__device__ void pair_load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                               const CUtensorMap* tmV, const Params& p, const Shared& sh) {
  using T = PairTraitsT<kQK8>;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint64_t pol_kv = policy_evict_last();
  const uint64_t pol_q = policy_evict_first();
  const uint32_t full0_leader = mapa_shared(sh.bar(T::kBarFull), 0);
  const uint32_t qfull0_leader = mapa_shared(sh.bar(T::kBarQFull), 0);
  uint32_t stage = 0, phase = 0, n_fills = 0, q_fills = 0, q_parity = 0, it = 0;
  bool ok = true;
  const int n_kv = (p.Lk + kBN - 1) / kBN;

  auto load_q = [&](int t, int bh, int row0) -> bool {
    if (!mbar_wait(sh.bar(T::kBarQEmpty + t), (it & 1u) ^ 1u, kWaitLimitNs, sh.abort)) return false;
    if (leader) mbar_arrive_expect_tx(sh.bar(T::kBarQFull + t), 2 * T::kQTileBytes);
    const uint32_t dst = sh.base + T::kOffQ + t * T::kQTileBytes;
    for (int b = 0; b < T::kQKBoxes; ++b)
      tma_load_3d_pair(dst + b * T::kQBoxBytes, tmQ, qfull0_leader + 8u * t, b * T::kBoxCols,
                       row0 + t * kBM, bh, pol_q);
    q_fills |= 1u << t;
    q_parity = (q_parity & ~(1u << t)) | ((it & 1u) << t);
    return true;
  };
  auto take_empty = [&](uint32_t half_bytes) -> bool {
    if (!mbar_wait(sh.bar(T::kBarEmpty + stage), phase ^ 1u, kWaitLimitNs, sh.abort)) return false;
    if (leader) mbar_arrive_expect_tx(sh.bar(T::kBarFull + stage), 2 * half_bytes);
    return true;
  };
  auto advance = [&]() {
    if (n_fills < T::kStages) ++n_fills;
    if (++stage == T::kStages) { stage = 0; phase ^= 1u; }
  };

  for (int i = static_cast<int>(cluster_id_x()); i < p.num_items && ok;
       i += static_cast<int>(num_clusters_x()), ++it) {
    const WorkItem w = work_item(i, p, n_kv);
    const int bh = w.bh;
    const int row0 = w.qblock * (2 * kUnitRows) + static_cast<int>(rank) * kUnitRows;
    ok = load_q(0, bh, row0);
    for (int j = w.j0; j < w.j1 && ok; ++j) {
      // K half: keys j*128 + 64*rank .. +63, all d columns (128-byte boxes)
      ok = take_empty(T::kKHalfBytes);
      if (!ok) break;
      {
        const uint32_t dst = sh.base + T::kOffKV + stage * T::kHalfBytes;
        for (int b = 0; b < T::kQKBoxes; ++b)
          tma_load_3d_pair(dst + b * T::kKBoxBytes, tmK, full0_leader + 8u * stage, b * T::kBoxCols,
                           j * kBN + static_cast<int>(rank) * 64, bh, pol_kv);
      }
      advance();
      if (j == w.j0) {
        ok = load_q(1, bh, row0);
        if (!ok) break;
      }
      // V half: keys j*128 .. +127, columns 64*rank .. +63
      ok = take_empty(T::kHalfBytes);
      if (!ok) break;
      tma_load_3d_pair(sh.base + T::kOffKV + stage * T::kHalfBytes, tmV, full0_leader + 8u * stage,
                       static_cast<int>(rank) * T::kBoxCols, j * kBN, bh, pol_kv);
      advance();
    }
  }
  if (!ok) {
    record_timeout<true>(sh);
    // Let this CTA's copies in flight land before its shared memory goes away.
    // Their completion is counted on the leader's barriers, so the leader waits.
    if (leader) {
      const volatile int no_abort = 0;
      uint32_t s = stage, ph = phase;
      for (uint32_t f = 0; f < n_fills; ++f) {
        if (s == 0) { s = T::kStages - 1; ph ^= 1u; } else { --s; }
        mbar_wait(sh.bar(T::kBarFull + s), ph, kWaitLimitNs, &no_abort);
      }
      for (int t = 0; t < 2; ++t)
        if (q_fills & (1u << t))
          mbar_wait(sh.bar(T::kBarQFull + t), (q_parity >> t) & 1u, kWaitLimitNs, &no_abort);
    } else {
      // The peer cannot wait on the leader's barriers; a TMA copy lands within
      // microseconds, so give the last ones 200 us.
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 200000ull) {
      }
    }
  }
}

// ----------------------------------------------------------------- MMA issuer (leader CTA)
template <bool kQK8>
__device__ __forceinline__ void pair_issue_qk(uint32_t d_tmem, uint32_t q_lo, uint32_t k_lo) {
  using T = PairTraitsT<kQK8>;
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

__device__ __forceinline__ void pair_issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_lo,
                                              bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, PairTraits::D, 0, 1);
  constexpr uint32_t hi = desc_hi_sw128(1024);
#pragma unroll
  for (int k = 0; k < kBN / 16; ++k)   // P of keys [64h, 64h+64) is in S columns [64h, 64h+32)
    mma_ts_lo_pair(d_tmem, p_tmem + (k / 4) * 64 + (k % 4) * 8, v_lo + ((k * 16 * 128) >> 4), hi,
                   idesc, (accumulate || k > 0) ? 1u : 0u);
}

template <bool kQK8>
__device__ void pair_mma_role(const Params& p, const Shared& sh, uint32_t tmem) {
  using T = PairTraitsT<kQK8>;
  constexpr uint16_t kBoth = 3;
  const bool issuer = (threadIdx.x & 31) == 0;
  uint32_t stage = 0, phase = 0, g = 0, it = 0;
  bool ok = true;
  const int n_kv = (p.Lk + kBN - 1) / kBN;
  const uint32_t q_lo0 = desc_lo_sw128(sh.base + T::kOffQ, 16);
  const uint32_t q_lo1 = desc_lo_sw128(sh.base + T::kOffQ + T::kQTileBytes, 16);
  const uint32_t kv_lo0 = desc_lo_sw128(sh.base + T::kOffKV, 16);
  auto kv_lo = [&](uint32_t s) { return kv_lo0 + s * (T::kHalfBytes >> 4); };
  auto wait = [&](int bar, uint32_t parity) -> bool {
    const bool got = mbar_wait(sh.bar(bar), parity, kWaitLimitNs, sh.abort);
    return __all_sync(0xffffffffu, got);
  };
  auto take_stage = [&](uint32_t& s_out) -> bool {
    s_out = stage;
    if (!wait(T::kBarFull + stage, phase)) return false;
    if (++stage == T::kStages) { stage = 0; phase ^= 1u; }
    return true;
  };

  // Stage waits for the next key tile (its V and the following K) happen while
  // the warp waits for P_1 anyway, off the path from P-ready to the next MMA.
  // Commits follow the MMA block they track (a commit between MMAs stalls
  // the issuing thread).
  for (int i = static_cast<int>(cluster_id_x()); i < p.num_items && ok;
       i += static_cast<int>(num_clusters_x()), ++it) {
    int n = n_kv;                // key tiles of this item
    if (i >= p.split_base) {
      const int s = (i - p.split_base) % p.splits;
      n = (s + 1) * n_kv / p.splits - s * n_kv / p.splits;
    }
    uint32_t sK = 0, sV = 0, sK_next = 0, sV_next = 0;
    ok = wait(T::kBarQFull + 0, it & 1u) && take_stage(sK);
    if (!ok) break;
    tc_fence_after();
    if (issuer) {
      pair_issue_qk<kQK8>(tmem + T::col_s(0), q_lo0, kv_lo(sK));
      mma_commit_pair(sh.bar(T::kBarSFull + 0), kBoth);
      if (n == 1) mma_commit_pair(sh.bar(T::kBarQEmpty + 0), kBoth);
    }
    __syncwarp();
    ok = wait(T::kBarQFull + 1, it & 1u) && take_stage(sV) && (n == 1 || take_stage(sK_next));
    if (!ok) break;
    tc_fence_after();
    if (issuer) {
      pair_issue_qk<kQK8>(tmem + T::col_s(1), q_lo1, kv_lo(sK));
      mma_commit_pair(sh.bar(T::kBarSFull + 1), kBoth);
      if (n == 1) mma_commit_pair(sh.bar(T::kBarQEmpty + 1), kBoth);
      mma_commit_pair(sh.bar(T::kBarEmpty + sK), kBoth);
    }
    __syncwarp();

    for (int j = 0; j < n && ok; ++j, ++g) {   // j: tile index within the item
      // held: sV = V(j); sK_next = K(j+1) when j+1 < n
      const bool more = j + 1 < n;
      ok = wait(T::kBarPFull + 0, g & 1u);
      if (!ok) break;
      tc_fence_after();
      if (issuer) {
        pair_issue_pv(tmem + T::col_o(0), tmem + T::col_s(0), kv_lo(sV), j > 0);
        if (more) {
          pair_issue_qk<kQK8>(tmem + T::col_s(0), q_lo0, kv_lo(sK_next));
          mma_commit_pair(sh.bar(T::kBarSFull + 0), kBoth);
          if (j + 2 == n) mma_commit_pair(sh.bar(T::kBarQEmpty + 0), kBoth);
        } else {
          mma_commit_pair(sh.bar(T::kBarOFull + 0), kBoth);
        }
      }
      __syncwarp();
      if (more) ok = take_stage(sV_next) && (j + 2 >= n || take_stage(sK));
      ok = ok && wait(T::kBarPFull + 1, g & 1u);
      if (!ok) break;
      tc_fence_after();
      if (issuer) {
        pair_issue_pv(tmem + T::col_o(1), tmem + T::col_s(1), kv_lo(sV), j > 0);
        if (more) {
          pair_issue_qk<kQK8>(tmem + T::col_s(1), q_lo1, kv_lo(sK_next));
          mma_commit_pair(sh.bar(T::kBarEmpty + sV), kBoth);
          mma_commit_pair(sh.bar(T::kBarSFull + 1), kBoth);
          if (j + 2 == n) mma_commit_pair(sh.bar(T::kBarQEmpty + 1), kBoth);
          mma_commit_pair(sh.bar(T::kBarEmpty + sK_next), kBoth);
        } else {
          mma_commit_pair(sh.bar(T::kBarEmpty + sV), kBoth);
          mma_commit_pair(sh.bar(T::kBarOFull + 1), kBoth);
        }
      }
      __syncwarp();
      sV = sV_next;
      sK_next = sK;   // K(j+2), taken above when it exists
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

// ----------------------------------------------------------------- kernel
// Launched with a cluster dimension of 2 (consecutive CTAs form a pair).
template <bool kQK8>
__global__ void __launch_bounds__(kNumThreads, 1)
    fmha_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params p) {
  using T = PairTraitsT<kQK8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint32_t* misc = reinterpret_cast<uint32_t*>(base_ptr + T::kOffMisc);  // [0] TMEM, [1] abort
  Shared sh;
  sh.base = base;
  sh.bar0 = base + T::kOffBar;
  sh.abort = reinterpret_cast<volatile int*>(misc + 1);
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
    *sh.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_u32(misc), T::kTmemCols);
    tmem_relinquish_pair();
  }
  // Both CTAs' barriers and TMEM exist before either CTA touches the other's.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp < kMmaWarp) {
    reg_alloc<kRegsSoftmax>();
    softmax_role<T::D, T, true>(p, sh, tmem);
  } else if (warp == kMmaWarp) {
    reg_dealloc<kRegsOther>();
    if (leader) pair_mma_role<kQK8>(p, sh, tmem);
  } else if (warp == kLoadWarp) {
    reg_dealloc<kRegsOther>();
    if (lane == 0) pair_load_role<kQK8>(&tmQ, &tmK, &tmV, p, sh);
    __syncwarp();
  } else {
    reg_dealloc<kRegsOther>();
  }

  // The leader drained its MMAs; neither CTA leaves while the pair's MMAs or
  // copies could still touch its shared memory or TMEM.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, T::kTmemCols);
  }
}

}  // namespace dit
