// dit_attn: dense non-causal softmax attention forward for sm_103a (B300).
//
// Operation (standard attention, the "traditional BF16 attention" that "Speed
// Up Image Generation with FLUX 3 Image Klein on NVIDIA Blackwell GPUs", Key
// takeaways, second item, puts at about 60% of DiT kernel time at 2048x2048):
// o_i = sum_j softmax_j(scale * q_i . k_j) v_j for every (batch, head), over
// the joint text+image token sequence.
//
// This file holds the device pieces the kernels share (parameters, work
// items, bounded waits, the probability and row-sum helpers, the partial-row
// store), the single-CTA kernel that serves d = 64, and the host side of the
// C ABI.  d = 128 runs on CTA pairs (fmha_pair.cuh: bf16, e4m3 Q/K and e4m3
// Q/K/V variants); combine.cuh merges a split last wave; rmsnorm.cuh and
// quantize.cuh are the input prologues.
//
// Single-CTA kernel (d = 64; one persistent CTA per SM, 384 threads):
//   warps 0-7   softmax: query tile 0, then tile 1, of every key tile
//   warp  8     tcgen05 MMA issuer and TMEM allocator
//   warp  9     TMA producer
//   warps 10-11 idle (they complete the third warpgroup for setmaxnreg)
// A work unit is 2 x 128 query rows of one (b,h).  Q tiles stay in shared
// memory for the whole unit; K and V tiles of 128 keys stream through a ring
// of shared-memory stages.  For every key tile j the MMA warp computes
// S_t = Q_t K_j^T into TMEM; the softmax warps turn S_t into bf16
// probabilities P_t in place (the same TMEM columns), and the MMA warp then
// accumulates O_t += P_t V_j in TMEM; one tile's softmax overlaps the other
// tile's MMAs.
//
// Online softmax (base 2): x = s * scale*log2(e).  Probabilities are first
// computed against the running maximum m; only when a tile's row sum against
// it exceeds 2^48 (or overflows) does the row take the tile's maximum, and m
// rises only if that maximum exceeds it by more than 8 (a factor 256); l and
// O are then rescaled by exp2(m_old - m_new).  O / l is exact in exact
// arithmetic whatever m is.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/dit_attn.h"
#include "ptx.cuh"

namespace dit {

// Set (never cleared by kernels) when a bounded wait gives up.
__device__ int g_device_error = 0;

constexpr int kBM = 128;                 // query rows per tile (one TMEM lane each)
constexpr int kBN = 128;                 // keys per K/V tile
constexpr int kTilesPerUnit = 2;         // query tiles per work unit
constexpr int kUnitRows = kBM * kTilesPerUnit;
// The single-CTA kernel (d = 64) runs three full warpgroups (setmaxnreg
// works per warpgroup); the d = 128 CTA-pair kernel has its own constants.
constexpr int kNumThreads = 384;
// Register split of the single-CTA kernel: launched at 168 per thread
// (384 x 168 = 64512); the two softmax warpgroups raise to 208 and the
// MMA/TMA warpgroup drops to 88: 256 x 208 + 128 x 88 = 64512, exactly the
// launch's total.
constexpr int kRegsSoftmax = 208;
constexpr int kRegsOther = 88;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s per wait
constexpr float kRescaleThreshold = 8.0f;          // log2 units
// 2^48: a tile's row sum above it (or not finite) forces the max pass (the
// pair kernels test each thread's half-row sum against it instead).  Below
// it the stale max is kept even when the row's max has risen: O and l carry
// the same factor, which cancels in O / l, and p <= 2^48 keeps both far from
// fp32's range.  (At 2^16, rows whose keys include a few large outliers took
// the max pass on about 14% of warp steps.)
constexpr float kOptimisticSumLimit = 281474976710656.0f;
// Which exponentials of a 32-key chunk the softmax evaluates on the FMA pipe
// (exp2_fma_pair) instead of the MUFU unit: bit i of the bf16 mask is the key
// pair 2i, 2i+1 (degree-3 polynomial, below bf16's rounding); bit i of the
// e4m3 mask is the key quad 4i .. 4i+3 (degree 2, below e4m3's rounding).
constexpr uint32_t kExp2FmaPairsBf16 = 0x0000u;
constexpr uint32_t kExp2FmaQuadsE4M3 = 0x00u;

// Words of a kernel's small "misc" area in shared memory.
constexpr int kMiscTmem = 0;     // TMEM base address written by the allocation
constexpr int kMiscAbort = 1;    // non-zero once any role gave up
// Pair kernel, leader CTA only: the copies each producer issued (K/V fills,
// query tiles 0 and 1), the leader's own and the peer's, for the teardown drain.
constexpr int kMiscFills = 2;
constexpr int kMiscQLoads = 3;
constexpr int kMiscPeerFills = 5;
constexpr int kMiscPeerQLoads = 6;
constexpr int kMiscSlotBytes = 8;   // [8, 8 + ring slots): this CTA's bytes of each slot's last fill
constexpr int kMiscWords = 24;

template <int D>
struct Traits {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kBoxCols = 64;                         // one 128-byte swizzle span
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr uint32_t kBoxBytes = 128u * 128u;          // 128 rows x 128 bytes
  static constexpr uint32_t kTileBytes = kBoxBytes * kBoxes;  // one Q, K or V tile
  static constexpr int kStages = D == 128 ? 4 : 8;
  // TMEM columns (fp32): S0, S1, O0, O1.  P_t (bf16 pairs) reuses the first 32
  // of each half-row's 64 S_t columns.
  __host__ __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(D) * t; }
  static constexpr uint32_t kTmemCols = 512;
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKV = kTilesPerUnit * kTileBytes;
  static constexpr uint32_t kOffBar = kOffKV + kStages * kTileBytes;
  // barriers: full[S], empty[S], q_full[2], q_empty[2], s_full[2], p_full[2], o_full[2], drain
  static constexpr int kBarFull = 0;
  static constexpr int kBarEmpty = kStages;
  static constexpr int kBarQFull = 2 * kStages;
  static constexpr int kBarQEmpty = kBarQFull + 2;
  static constexpr int kBarSFull = kBarQEmpty + 2;
  static constexpr int kBarPFull = kBarSFull + 2;
  static constexpr int kBarOFull = kBarPFull + 2;
  static constexpr int kBarDrain = kBarOFull + 2;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = 1024 + kOffMisc + kMiscWords * 4;
};

struct Params {
  __nv_bfloat16* out;
  int Lq, Lk;
  int num_qblocks;   // query blocks (work units) per (b,h)
  int num_units;     // B*H*num_qblocks
  float scale_log2;  // scale * log2(e)
  // Split tail (pair kernel).  Work items [0, split_base) are whole units; each
  // unit in [split_base, num_units) is cut into `splits` key ranges, items
  // split_base + c for chunk c < (num_units - split_base) * splits, whose
  // unnormalised results go to part_o / part_ml for the combine kernel.
  int split_base;    // num_units when nothing is split
  int splits;        // 1 when nothing is split
  int num_items;     // split_base + (num_units - split_base) * splits
  float* part_o;     // [chunk][512 rows][D] fp32: sum_j p_j v_j against the chunk's max
  float* part_ml;    // [chunk][512 rows][2] fp32: running max (log2 units), row sum
  float v_scale;     // e4m3 values: dequantisation scale of v (1 otherwise)
  float inv_v_scale; // 1 / v_scale
};

// One work item: query block `qblock` of head `bh` against key tiles
// [j0, j1); chunk >= 0 marks a key range of a split unit.
struct WorkItem {
  int bh, qblock, j0, j1, chunk;
};

__device__ __forceinline__ WorkItem work_item(int i, const Params& p, int n_kv) {
  WorkItem w;
  int u = i, s = 0;
  w.chunk = -1;
  if (i >= p.split_base) {
    const int c = i - p.split_base;
    u = p.split_base + c / p.splits;
    s = c % p.splits;
    w.chunk = c;
  }
  w.bh = u / p.num_qblocks;
  w.qblock = u % p.num_qblocks;
  // s < splits <= 16 and n_kv < 2^24, so the products fit in 32 bits
  w.j0 = w.chunk < 0 ? 0 : s * n_kv / p.splits;
  w.j1 = w.chunk < 0 ? n_kv : (s + 1) * n_kv / p.splits;
  return w;
}

struct Shared {
  uint32_t base;          // shared-window address of the aligned base
  uint32_t bar0;          // address of barrier 0
  volatile int* abort;    // set when any role gives up
  uint32_t misc;          // shared-window address of the misc words (kMisc*)
  __device__ uint32_t bar(int i) const { return bar0 + 8u * static_cast<uint32_t>(i); }
  __device__ uint32_t misc_word(int i) const { return misc + 4u * static_cast<uint32_t>(i); }
};

// Give up: stop every role of this CTA (and, for a CTA pair, of the peer CTA)
// and record TIMEOUT in the device error word.
template <bool kPair = false>
__device__ __forceinline__ void record_timeout(const Shared& sh) {
  *sh.abort = 1;
  if (kPair) {
    const uint32_t local = smem_u32(const_cast<int*>(sh.abort));
    st_shared_cluster_u32(mapa_shared(local, cluster_ctarank() ^ 1u), 1u);
  }
  atomicExch(&g_device_error, DIT_ATTN_ERR_TIMEOUT);
}

// ----------------------------------------------------------------- producer
template <int D>
__device__ void load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                          const Params& p, const Shared& sh) {
  using T = Traits<D>;
  const uint64_t pol_kv = policy_evict_last();
  const uint64_t pol_q = policy_evict_first();
  uint32_t stage = 0, phase = 0;
  uint32_t n_fills = 0;                  // K/V fills issued (saturates at kStages)
  uint32_t q_fills = 0;                  // bit t: query tile t was ever loaded
  uint32_t q_parity = 0;                 // bit t: parity of tile t's last load
  bool ok = true;
  const int n_kv = (p.Lk + kBN - 1) / kBN;
  uint32_t it = 0;

  auto load_q = [&](int t, int bh, int row0) -> bool {
    if (!mbar_wait(sh.bar(T::kBarQEmpty + t), (it & 1u) ^ 1u, kWaitLimitNs, sh.abort)) return false;
    const uint32_t bar = sh.bar(T::kBarQFull + t);
    mbar_arrive_expect_tx(bar, T::kTileBytes);
    const uint32_t dst = sh.base + T::kOffQ + t * T::kTileBytes;
    for (int b = 0; b < T::kBoxes; ++b)
      tma_load_3d(dst + b * T::kBoxBytes, tmQ, bar, b * T::kBoxCols, row0 + t * kBM, bh, pol_q);
    q_fills |= 1u << t;
    q_parity = (q_parity & ~(1u << t)) | ((it & 1u) << t);
    return true;
  };
  auto load_kv = [&](const CUtensorMap* tm, int bh, int key0) -> bool {
    if (!mbar_wait(sh.bar(T::kBarEmpty + stage), phase ^ 1u, kWaitLimitNs, sh.abort)) return false;
    const uint32_t bar = sh.bar(T::kBarFull + stage);
    mbar_arrive_expect_tx(bar, T::kTileBytes);
    const uint32_t dst = sh.base + T::kOffKV + stage * T::kTileBytes;
    for (int b = 0; b < T::kBoxes; ++b)
      tma_load_3d(dst + b * T::kBoxBytes, tm, bar, b * T::kBoxCols, key0, bh, pol_kv);
    if (n_fills < T::kStages) ++n_fills;
    if (++stage == T::kStages) { stage = 0; phase ^= 1u; }
    return true;
  };

  for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++it) {
    const int bh = u / p.num_qblocks;
    const int row0 = (u % p.num_qblocks) * kUnitRows;
    ok = load_q(0, bh, row0);
    for (int j = 0; j < n_kv && ok; ++j) {
      ok = load_kv(tmK, bh, j * kBN);
      if (ok && j == 0) ok = load_q(1, bh, row0);
      if (ok) ok = load_kv(tmV, bh, j * kBN);
    }
  }
  if (!ok) {
    record_timeout(sh);
    // Let every copy already issued land before the CTA's shared memory goes away.
    const volatile int no_abort = 0;
    // The last n_fills fills went to the stages just before `stage`.
    uint32_t s = stage, ph = phase;
    for (uint32_t f = 0; f < n_fills; ++f) {
      if (s == 0) { s = T::kStages - 1; ph ^= 1u; } else { --s; }
      mbar_wait(sh.bar(T::kBarFull + s), ph, kWaitLimitNs, &no_abort);
    }
    for (int t = 0; t < 2; ++t)
      if (q_fills & (1u << t))
        mbar_wait(sh.bar(T::kBarQFull + t), (q_parity >> t) & 1u, kWaitLimitNs, &no_abort);
  }
}

// ----------------------------------------------------------------- MMA issuer
// Descriptor low words carry (address >> 4) in their 14-bit start field; the
// shared window is below 256 KB, so adding (bytes >> 4) to a low word advances
// the start address without touching the other fields.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_lo, uint32_t k_lo) {
  using T = Traits<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, 0, 0);
  constexpr uint32_t hi = desc_hi_sw128(1024);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    // K step k: 16 columns = 32 bytes into the 128-byte swizzle span of box k/4.
    const uint32_t off = ((k / 4) * T::kBoxBytes + (k % 4) * 32) >> 4;
    mma_ss_lo(d_tmem, q_lo + off, k_lo + off, hi, idesc, k > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_lo,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, D, 0, 1);
  constexpr uint32_t hi = desc_hi_sw128(1024);
#pragma unroll
  for (int k = 0; k < kBN / 16; ++k) {
    // K step k: 16 keys = 16 rows of 128 bytes.  P of keys [64h, 64h+64) is in
    // S columns [64h, 64h+32) as bf16 pairs.
    mma_ts_lo(d_tmem, p_tmem + (k / 4) * 64 + (k % 4) * 8, v_lo + ((k * 16 * 128) >> 4), hi, idesc,
              (accumulate || k > 0) ? 1u : 0u);
  }
}

// Run by the whole MMA warp so that barrier waits and descriptor arithmetic
// stay warp-uniform; lane 0 alone issues the MMAs and the commits that track them.
template <int D>
__device__ void mma_role(const Params& p, const Shared& sh, uint32_t tmem) {
  using T = Traits<D>;
  const bool leader = (threadIdx.x & 31) == 0;
  uint32_t stage = 0, phase = 0;
  uint32_t g = 0;    // key-tile iterations so far (P hand-offs per query tile)
  uint32_t it = 0;   // work units so far
  bool ok = true;
  const int n_kv = (p.Lk + kBN - 1) / kBN;
  // K-major Q/K tiles: LBO unused (16); V tiles (MN-major): LBO = one 64-column box.
  const uint32_t q_lo0 = desc_lo_sw128(sh.base + T::kOffQ, 16);
  const uint32_t q_lo1 = desc_lo_sw128(sh.base + T::kOffQ + T::kTileBytes, 16);
  const uint32_t kv_lo0 = desc_lo_sw128(sh.base + T::kOffKV, 16);
  const uint32_t v_lbo = ((T::kBoxBytes >> 4) << 16) - (1u << 16);   // LBO 16 -> one box
  auto k_lo = [&](uint32_t s) { return kv_lo0 + s * (T::kTileBytes >> 4); };
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

  for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++it) {
    uint32_t sK = 0, sV = 0;
    // S_t = Q_t K_0^T for both tiles
    ok = wait(T::kBarQFull + 0, it & 1u) && take_stage(sK);
    if (!ok) break;
    tc_fence_after();
    if (leader) {
      issue_qk<D>(tmem + T::col_s(0), q_lo0, k_lo(sK));
      mma_commit(sh.bar(T::kBarSFull + 0));
      if (n_kv == 1) mma_commit(sh.bar(T::kBarQEmpty + 0));
    }
    __syncwarp();
    ok = wait(T::kBarQFull + 1, it & 1u);
    if (!ok) break;
    tc_fence_after();
    if (leader) {
      issue_qk<D>(tmem + T::col_s(1), q_lo1, k_lo(sK));
      mma_commit(sh.bar(T::kBarSFull + 1));
      if (n_kv == 1) mma_commit(sh.bar(T::kBarQEmpty + 1));
      mma_commit(sh.bar(T::kBarEmpty + sK));
    }
    __syncwarp();

    for (int j = 0; j < n_kv && ok; ++j, ++g) {
      const bool more = j + 1 < n_kv;
      ok = take_stage(sV) && wait(T::kBarPFull + 0, g & 1u);
      if (more) ok = ok && take_stage(sK);
      if (!ok) break;
      tc_fence_after();
      if (leader) {
        issue_pv<D>(tmem + T::col_o(0), tmem + T::col_s(0), k_lo(sV) + v_lbo, j > 0);
        if (more) {
          issue_qk<D>(tmem + T::col_s(0), q_lo0, k_lo(sK));
          mma_commit(sh.bar(T::kBarSFull + 0));
          if (j + 2 == n_kv) mma_commit(sh.bar(T::kBarQEmpty + 0));
        } else {
          mma_commit(sh.bar(T::kBarOFull + 0));
        }
      }
      __syncwarp();
      ok = wait(T::kBarPFull + 1, g & 1u);
      if (!ok) break;
      tc_fence_after();
      if (leader) {
        issue_pv<D>(tmem + T::col_o(1), tmem + T::col_s(1), k_lo(sV) + v_lbo, j > 0);
        mma_commit(sh.bar(T::kBarEmpty + sV));
        if (more) {
          issue_qk<D>(tmem + T::col_s(1), q_lo1, k_lo(sK));
          mma_commit(sh.bar(T::kBarSFull + 1));
          if (j + 2 == n_kv) mma_commit(sh.bar(T::kBarQEmpty + 1));
          mma_commit(sh.bar(T::kBarEmpty + sK));
        } else {
          mma_commit(sh.bar(T::kBarOFull + 1));
        }
      }
      __syncwarp();
    }
  }
  if (!ok && leader) record_timeout(sh);
  // Drain: every MMA lane 0 issued completes before TMEM is released.
  if (leader) {
    mma_commit(sh.bar(T::kBarDrain));
    const volatile int no_abort = 0;
    mbar_wait(sh.bar(T::kBarDrain), 0, kWaitLimitNs, &no_abort);
  }
  __syncwarp();
}

// ----------------------------------------------------------------- softmax + epilogue
// Single-CTA kernel (d = 64): the eight softmax warps work on one query tile
// at a time, two threads per query row (TMEM shape 16x32bx2): warp w owns
// TMEM lanes 32*(w%4) + 16*(w/4) .. +15; lanes 0-15 of the warp take keys
// 0-63 of the tile and lanes 16-31 take keys 64-127 of the same rows.  A half-row's probabilities (32 packed
// bf16 pairs) go over the first 32 columns of its own 64 S columns, so the two
// halves never overwrite each other's logits.  Row max, row sum and the
// recompute decision are combined across the pair with one shuffle.

// O_t row-half rescale: the thread's D/2 output columns times factor.
template <int D>
__device__ __forceinline__ void rescale_o_half(uint32_t taddr_o, float factor) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t o[32];
    tmem_ld16x2_32<D / 2>(taddr_o + c * 32, o);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * factor);
    tmem_st16x2_32<D / 2>(taddr_o + c * 32, o);
  }
}

// exp2 of 32 keys of a half-row (first key index key0) into 16 packed bf16
// pairs (pk[i] holds keys key0+2i, key0+2i+1), accumulating into acc[8] the
// probabilities *as rounded to bf16*, so that the row sum l and the P.V
// product weigh every key identically (a row dominated by one key then
// returns that key's value row without a rounding-induced scale error); the
// sum uses mixed-precision f32 += bf16 adds on the packed halves.
// kMasked: keys at or beyond `valid` get probability 0.
template <bool kMasked>
__device__ __forceinline__ void probs_chunk(const uint32_t (&sr)[32], float scale_log2, float neg_m,
                                            int key0, int valid, uint32_t* pk, float (&acc)[8]) {
  const float2 sl2 = make_float2(scale_log2, scale_log2);
  const float2 nm = make_float2(neg_m, neg_m);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 x =
        __ffma2_rn(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), sl2, nm);
    float p0, p1;
    if ((kExp2FmaPairsBf16 >> (i / 2)) & 1u) {   // this pair's exp2 on the FMA pipe
      const float2 e = exp2_fma_pair<3>(x);
      p0 = e.x;
      p1 = e.y;
    } else {
      p0 = ex2_approx(x.x);
      p1 = ex2_approx(x.y);
    }
    if (kMasked) {
      p0 = (key0 + i < valid) ? p0 : 0.f;
      p1 = (key0 + i + 1 < valid) ? p1 : 0.f;
    }
    const uint32_t w = pack_bf16x2(p0, p1);
    pk[i / 2] = w;
    add_bf16x2_halves(acc[(i / 2) & 7], acc[((i / 2) + 4) & 7], w);
  }
}

__device__ __forceinline__ float sum8(const float (&acc)[8]) {
  return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}

// Largest scaled logit s * scale_log2 of a half-row's 64 logits, keys at or
// beyond `valid` excluded (-inf when all are): scale_log2 times the largest
// raw logit when scale_log2 >= 0, times the smallest when it is negative (the
// sign is the same for the whole launch).
template <bool kMasked>
__device__ __forceinline__ float rowmax_half(const uint32_t (&sr)[2][32], int key0, int valid,
                                             float scale_log2) {
  const bool neg = scale_log2 < 0.f;
  const float sentinel = neg ? INFINITY : -INFINITY;
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = sentinel;
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float a = __uint_as_float(sr[c][i]), b = __uint_as_float(sr[c][i + 1]);
      if (kMasked) {
        a = (key0 + c * 32 + i < valid) ? a : sentinel;
        b = (key0 + c * 32 + i + 1 < valid) ? b : sentinel;
      }
      m[(c * 16 + i / 2) & 7] = neg ? fmin3(m[(c * 16 + i / 2) & 7], a, b)
                                    : fmax3(m[(c * 16 + i / 2) & 7], a, b);
    }
  const float e = neg ? fminf(fmin3(m[0], m[1], m[2]), fmin3(m[3], m[4], fmin3(m[5], m[6], m[7])))
                      : fmaxf(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], fmax3(m[5], m[6], m[7])));
  return e == sentinel ? -INFINITY : e * scale_log2;
}

// One query tile's softmax step for this thread's half-row (keys key0 ..
// key0+63 of the tile): loads the logits from TMEM at taddr_s, updates the
// running max m_used and this half-row's share of the row sum l, calls
// o_rescale(factor) when the max rises (the hook must scale this thread's
// half of every O accumulator of the row, once no P.V product still writes
// them), and writes the packed bf16 probabilities over the half-row's first
// 32 S columns.  Returns after issuing the TMEM stores (the caller waits).
template <int D, class ORescale>
__device__ __forceinline__ void softmax_tile_half(uint32_t taddr_s, int key0, bool first,
                                                  bool masked, int valid, float scale_log2,
                                                  float& m_used, float& l, ORescale&& o_rescale) {
  // Logits stay in registers for the whole tile; the second chunk's TMEM
  // load and the first chunk's P store overlap with arithmetic.  A recompute
  // overwrites P before P-ready is signalled.
  uint32_t sr[2][32];
  uint32_t pk[32];
  float acc[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) acc[a] = 0.f;
  tmem_ld16x2_32<64>(taddr_s, sr[0]);
  tmem_wait_ld();
  tmem_ld16x2_32<64>(taddr_s + 32, sr[1]);
  // probabilities of chunk c against the running max m, packed and stored
  auto chunk = [&](int c, float m) {
    if (masked) probs_chunk<true>(sr[c], scale_log2, -m, key0 + 32 * c, valid, &pk[16 * c], acc);
    else probs_chunk<false>(sr[c], scale_log2, -m, key0 + 32 * c, kBN, &pk[16 * c], acc);
    tmem_st16x2_16<64>(taddr_s + 16 * c, &pk[16 * c]);
  };
  // Row max over both halves, lazy rescale of l and O, probabilities
  // (first tile, or a recompute).
  auto max_pass = [&]() {
    tmem_wait_st();   // earlier optimistic P stores land before they are overwritten
    const float mx = masked ? rowmax_half<true>(sr, key0, valid, scale_log2)
                            : rowmax_half<false>(sr, key0, kBN, scale_log2);
    const float m_tile = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    float factor = 1.f;
    if (m_tile > m_used + kRescaleThreshold) {
      factor = ex2_approx(m_used - m_tile);   // 0 on the first tile
      l *= factor;
      m_used = m_tile;
    }
    if (!first && __any_sync(0xffffffffu, factor != 1.f)) o_rescale(factor);
#pragma unroll
    for (int a = 0; a < 8; ++a) acc[a] = 0.f;
    chunk(0, m_used);
    chunk(1, m_used);
  };
  if (first) {
    tmem_wait_ld();
    max_pass();
  } else {
    // Optimistic pass against the running max.  If a row's rounded sum
    // exceeds 2^48 (or overflowed), some p > 2^41: the row raises its max
    // (always, since p > 2^8), rescales l and O and recomputes.  Warp-uniform
    // branch.
    chunk(0, m_used);
    tmem_wait_ld();
    chunk(1, m_used);
    const float half_sum = sum8(acc);
    const float row_sum = half_sum + __shfl_xor_sync(0xffffffffu, half_sum, 16);
    if (__any_sync(0xffffffffu, !(row_sum <= kOptimisticSumLimit))) max_pass();
  }
  l += sum8(acc);
}

// A chunk of a split unit: this thread's D/2 unnormalised output columns of
// partial row prow, and (from the first half) the row's running max and sum.
template <int D>
__device__ __forceinline__ void store_partial(const Params& p, int64_t prow, int half,
                                           uint32_t taddr_o, float m_used, float l_row) {
  float4* po = reinterpret_cast<float4*>(p.part_o + prow * D + half * (D / 2));
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t o[32];
    tmem_ld16x2_32<D / 2>(taddr_o + c * 32, o);
    tmem_wait_ld();
#pragma unroll
    for (int v = 0; v < 8; ++v)
      po[c * 8 + v] = make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                  __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
  }
  if (half == 0) reinterpret_cast<float2*>(p.part_ml)[prow] = make_float2(m_used, l_row);
}

// Softmax and epilogue of the single-CTA kernel: the eight softmax warps take
// query tile 0, then tile 1, of every key tile; each warp arrives once per
// tile on P-ready (after its TMEM stores completed).
template <int D, class T>
__device__ void softmax_role(const Params& p, const Shared& sh, uint32_t tmem) {
  const int warp = threadIdx.x / 32;                 // 0..7
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;                        // keys [64*half, 64*half + 64) of a tile
  const int lane0 = (warp & 3) * 32 + (warp >> 2) * 16;
  const int r = lane0 + (lane & 15);                 // row within a query tile
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(lane0) << 16);
  const float scale_log2 = p.scale_log2;
  const int n_kv = (p.Lk + kBN - 1) / kBN;
  const int tail = p.Lk - (n_kv - 1) * kBN;          // valid keys in the last tile, 1..128
  const int key0 = 64 * half;
  uint32_t g = 0, it = 0;
  bool ok = true;

  for (int u = static_cast<int>(blockIdx.x); u < p.num_units && ok;
       u += static_cast<int>(gridDim.x), ++it) {
    const int bh = u / p.num_qblocks;
    const int row_base = (u % p.num_qblocks) * kUnitRows + r;
    float m_used[2] = {-INFINITY, -INFINITY};   // running max, in units of s*scale*log2(e)
    float l[2] = {0.f, 0.f};                     // this half-row's share of the row sum
    for (int j = 0; j < n_kv && ok; ++j, ++g) {
      const bool masked = (j == n_kv - 1) && (tail < kBN);
      const int valid = masked ? tail : kBN;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const bool got = mbar_wait(sh.bar(T::kBarSFull + t), g & 1u, kWaitLimitNs, sh.abort);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        // O_t is quiescent here: S_t's completion implies the previous P.V
        // product into O_t finished.
        const uint32_t taddr_o = lane_addr + T::col_o(t);
        softmax_tile_half<D>(lane_addr + T::col_s(t), key0, j == 0, masked, valid, scale_log2,
                             m_used[t], l[t], [&](float f) { rescale_o_half<D>(taddr_o, f); });
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sh.bar(T::kBarPFull + t));
      }
    }
    if (!ok) break;
    // Epilogue: O_t / l -> bf16 -> global; each thread writes its D/2 columns.
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const bool got = mbar_wait(sh.bar(T::kBarOFull + t), it & 1u, kWaitLimitNs, sh.abort);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
      const float l_row = l[t] + __shfl_xor_sync(0xffffffffu, l[t], 16);
      const float inv_l = 1.f / l_row;
      const int row = row_base + t * kBM;
      const bool row_ok = row < p.Lq;
      uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(bh) * p.Lq + row) * D +
                                            half * (D / 2));
      const uint32_t taddr_o = lane_addr + T::col_o(t);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o[32];
        tmem_ld16x2_32<D / 2>(taddr_o + c * 32, o);
        tmem_wait_ld();
        uint32_t wv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          wv[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        if (row_ok) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[c * 4 + v] = make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
        }
      }
    }
  }
  if (!ok) record_timeout(sh);
}

// ----------------------------------------------------------------- kernel
template <int D>
__global__ void __launch_bounds__(kNumThreads, 1)
    fmha_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params p) {
  using T = Traits<D>;
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

  if (threadIdx.x == 0) {
    for (int s = 0; s < T::kStages; ++s) {
      mbar_init(sh.bar(T::kBarFull + s), 1);
      mbar_init(sh.bar(T::kBarEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(sh.bar(T::kBarQFull + t), 1);
      mbar_init(sh.bar(T::kBarQEmpty + t), 1);
      mbar_init(sh.bar(T::kBarSFull + t), 1);
      mbar_init(sh.bar(T::kBarPFull + t), 8);   // one arrival per softmax warp
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
    tmem_alloc(smem_u32(misc + kMiscTmem), T::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[kMiscTmem];

  if (warp < kMmaWarp) {
    reg_alloc<kRegsSoftmax>();
    softmax_role<D, Traits<D>>(p, sh, tmem);
  } else if (warp == kMmaWarp) {
    reg_dealloc<kRegsOther>();
    mma_role<D>(p, sh, tmem);
  } else if (warp == kLoadWarp) {
    reg_dealloc<kRegsOther>();
    if (lane == 0) load_role<D>(&tmQ, &tmK, &tmV, p, sh);
    __syncwarp();
  } else {
    reg_dealloc<kRegsOther>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, T::kTmemCols);
  }
}

// Self-test of the bounded-wait path: one thread waits on an mbarrier that
// nothing ever arrives on, gives up after limit_ns and records TIMEOUT in the
// device error word, exactly as an attention kernel role does when a
// hand-off never comes.  Nothing faults or hangs.
__global__ void wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbarrier_init();
    if (!mbar_wait(smem_u32(&bar), 0, limit_ns, &abort_flag))
      atomicExch(&g_device_error, DIT_ATTN_ERR_TIMEOUT);
  }
}

// Self-test of the FMA-pipe exp2: y_fma[i] = exp2_fma_pair of x[i] (degree 2
// or 3), y_mufu[i] = ex2.approx.ftz of x[i], one element per thread.
template <int kDeg>
__global__ void exp2_check_kernel(const float* __restrict__ x, float* __restrict__ y_fma,
                                  float* __restrict__ y_mufu, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float v = x[i];
  y_fma[i] = exp2_fma_pair<kDeg>(make_float2(v, v)).x;
  y_mufu[i] = ex2_approx(v);
}

// Read and clear the device error word in one atomic step, so that a TIMEOUT
// a kernel on another stream records meanwhile is never lost.
__device__ int g_error_taken = 0;
__global__ void take_device_error_kernel() { g_error_taken = atomicExch(&g_device_error, 0); }

}  // namespace dit

#include "fmha_pair.cuh"
#include "combine.cuh"
#include "rmsnorm.cuh"
#include "quantize.cuh"

// =================================================================== host side
namespace {

using dit::Traits;

// Scratch of dit_attn_forward_noalloc, a file-scope device array: room for the
// split tail's partial rows (512 x (128 + 2) fp32 per key-range chunk) of up
// to kScratchChunks chunks.  A split plan needs at most one chunk per CTA pair
// (74 on a 148-SM B300).  In host code g_scratch only names the array; its
// device address comes from cudaGetSymbolAddress in dit_attn_create.
constexpr int64_t kScratchChunks = 80;
constexpr int64_t kScratchBytes =
    kScratchChunks * 2 * dit::kUnitRows * (128 + 2) * static_cast<int64_t>(sizeof(float));
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int max_pairs = 0;       // co-resident clusters of two CTAs of the bf16 pair kernel
  int max_pairs_qk8 = 0;   // the same for the e4m3-QK pair kernel
  int max_pairs_fp8 = 0;   // the same for the e4m3 Q/K/V pair kernel
  void* scratch = nullptr; // device address of g_scratch on this device
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
std::mutex g_err_mu;   // serialises dit_attn_get_device_error
DeviceState g_state[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return DIT_ATTN_ERR_CUDA;
}

bool current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return *dev >= 0 && *dev < kMaxDevices;
}

// 3-D view [BH][L][d] of bf16 (elem_bytes 2) or e4m3 bytes (elem_bytes 1)
// with a box of one row segment of box_bytes (128 or 64) x box_rows rows,
// swizzled at the segment's width.  Rows beyond L inside one head read as
// zeros, never as the next head's rows.
int encode_map(CUtensorMap* map, const void* ptr, int64_t BH, int64_t L, int d,
               uint32_t box_rows = 128, int elem_bytes = 2, uint32_t box_bytes = 128) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t eb = static_cast<cuuint64_t>(elem_bytes);
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * eb,
                                 static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(d) * eb};
  const cuuint32_t box[3] = {box_bytes / static_cast<cuuint32_t>(elem_bytes), box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dtype =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUresult r = g_encode(map, dtype, 3, const_cast<void*>(ptr), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = static_cast<int>(r);
    return DIT_ATTN_ERR_CUDA;
  }
  return DIT_ATTN_OK;
}

bool overlaps(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

template <int D>
int launch(const void* q, const void* k, const void* v, void* out, int64_t BH, int Lq, int Lk,
           float scale, cudaStream_t stream, int num_sms) {
  CUtensorMap tq, tk, tv;
  int rc;
  if ((rc = encode_map(&tq, q, BH, Lq, D)) != DIT_ATTN_OK) return rc;
  if ((rc = encode_map(&tk, k, BH, Lk, D)) != DIT_ATTN_OK) return rc;
  if ((rc = encode_map(&tv, v, BH, Lk, D)) != DIT_ATTN_OK) return rc;
  dit::Params p;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.Lq = Lq;
  p.Lk = Lk;
  p.num_qblocks = (Lq + dit::kUnitRows - 1) / dit::kUnitRows;
  p.num_units = static_cast<int>(BH * p.num_qblocks);
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.split_base = p.num_units;
  p.splits = 1;
  p.num_items = p.num_units;
  p.part_o = nullptr;
  p.part_ml = nullptr;
  p.v_scale = 1.f;
  p.inv_v_scale = 1.f;
  const int grid = p.num_units < num_sms ? p.num_units : num_sms;
  dit::fmha_fwd_kernel<D><<<grid, dit::kNumThreads, Traits<D>::kSmemBytes, stream>>>(tq, tk, tv, p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return DIT_ATTN_OK;
}

cudaLaunchConfig_t pair_launch_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr,
                                      uint32_t smem_bytes = dit::PairTraits::kSmemBytes) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(dit::kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = 2;
  attr->val.clusterDim.y = 1;
  attr->val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Split tail of the pair kernel.  A persistent launch of P clusters runs the
// units in waves of P; when the last wave is partial (rem = units mod P > 0),
// its units are cut into `splits` key ranges so that the wave fills the GPU,
// each range at least kMinTilesPerChunk key tiles long (a chunk writes 260 KB
// of partial results, about one key tile's worth of time).
constexpr int kMinTilesPerChunk = 8;
constexpr int kMaxSplits = 16;
constexpr int kPairUnitRows = 2 * dit::kUnitRows;

struct SplitPlan {
  int split_base, splits, num_items;
  int64_t chunks;     // (num_units - split_base) * splits
  int64_t ws_bytes;   // partial O and (max, sum) of every chunk
};

SplitPlan plan_split(int64_t num_units, int n_kv, int max_pairs) {
  SplitPlan s = {static_cast<int>(num_units), 1, static_cast<int>(num_units), 0, 0};
  const int64_t rem = num_units % max_pairs;
  if (rem == 0) return s;
  int64_t splits = max_pairs / rem;
  if (splits > n_kv / kMinTilesPerChunk) splits = n_kv / kMinTilesPerChunk;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits < 2) return s;
  s.split_base = static_cast<int>(num_units - rem);
  s.splits = static_cast<int>(splits);
  s.chunks = rem * splits;
  s.num_items = static_cast<int>(s.split_base + s.chunks);
  s.ws_bytes = s.chunks * kPairUnitRows * (128 + 2) * static_cast<int64_t>(sizeof(float));
  return s;
}

// d = 128: clusters of two CTAs, one work unit = 512 query rows.  With kQK8,
// q and k hold e4m3 bytes and `scale` already includes their dequantisation
// scales; with kPV8, v holds e4m3 bytes too, dequantised by v_scale.  With a
// workspace of at least the plan's size the last, partial wave runs split,
// followed by the combine kernel on the same stream.
template <bool kQK8, bool kPV8>
int launch_pair(const void* q, const void* k, const void* v, void* out, int64_t BH, int Lq, int Lk,
                double scale, cudaStream_t stream, int max_pairs, void* ws, int64_t ws_bytes,
                float v_scale = 1.f) {
  CUtensorMap tq, tk, tv;
  int rc;
  const int qk_bytes = kQK8 ? 1 : 2;
  if ((rc = encode_map(&tq, q, BH, Lq, 128, 128, qk_bytes)) != DIT_ATTN_OK) return rc;
  if ((rc = encode_map(&tk, k, BH, Lk, 128, 64, qk_bytes)) != DIT_ATTN_OK) return rc;
  // a CTA's value half is 64 columns: 128 bytes of bf16 or 64 bytes of e4m3
  if ((rc = kPV8 ? encode_map(&tv, v, BH, Lk, 128, 128, 1, 64) : encode_map(&tv, v, BH, Lk, 128, 128))
      != DIT_ATTN_OK)
    return rc;
  dit::Params p;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.Lq = Lq;
  p.Lk = Lk;
  p.num_qblocks = (Lq + kPairUnitRows - 1) / kPairUnitRows;
  p.num_units = static_cast<int>(BH * p.num_qblocks);
  p.scale_log2 = static_cast<float>(scale * 1.4426950408889634);
  p.v_scale = v_scale;
  p.inv_v_scale = 1.f / v_scale;
  SplitPlan plan = plan_split(p.num_units, (Lk + dit::kBN - 1) / dit::kBN, max_pairs);
  if (plan.splits > 1 && (!ws || ws_bytes < plan.ws_bytes))
    plan = SplitPlan{p.num_units, 1, p.num_units, 0, 0};
  p.split_base = plan.split_base;
  p.splits = plan.splits;
  p.num_items = plan.num_items;
  p.part_o = plan.splits > 1 ? static_cast<float*>(ws) : nullptr;
  p.part_ml = plan.splits > 1 ? p.part_o + plan.chunks * kPairUnitRows * 128 : nullptr;
  const int pairs = p.num_items < max_pairs ? p.num_items : max_pairs;
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg =
      pair_launch_config(2 * pairs, stream, &attr, dit::PairTraitsT<kQK8, kPV8>::kSmemBytes);
  cudaError_t e = cudaLaunchKernelEx(&cfg, dit::fmha_fwd_pair_kernel<kQK8, kPV8>, tq, tk, tv, p);
  if (e != cudaSuccess) return cuda_fail(e);
  if (plan.splits > 1) {
    const int64_t rows = (plan.num_items - plan.split_base) / plan.splits * int64_t{kPairUnitRows};
    const int64_t blocks = (rows * 32 + 255) / 256;
    dit::combine_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        p.part_o, p.part_ml, p.out, p.split_base, p.splits, p.num_qblocks, p.Lq, rows);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return DIT_ATTN_OK;
}

// Shared memory and cluster attributes of a pair kernel; *pairs = clusters of
// two that fit on the device at once.
template <bool kQK8, bool kPV8>
int setup_pair_kernel(int num_sms, int* pairs) {
  const uint32_t smem = dit::PairTraitsT<kQK8, kPV8>::kSmemBytes;
  auto* kernel = dit::fmha_fwd_pair_kernel<kQK8, kPV8>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
  if (e != cudaSuccess) return cuda_fail(e);
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg = pair_launch_config(num_sms, nullptr, &attr, smem);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
  if (e != cudaSuccess) return cuda_fail(e);
  if (clusters < 1) return cuda_fail(cudaErrorInvalidConfiguration);
  *pairs = clusters;
  return DIT_ATTN_OK;
}

// A logit scale is usable when it is finite and scale * log2(e), the factor the
// kernels apply in fp32, is finite too (|scale| <= 2.35e38); any sign.
bool logit_scale_ok(double scale) {
  return std::isfinite(scale) && std::fabs(scale * 1.4426950408889634) <= FLT_MAX;
}

// Argument checks shared by the bf16 and e4m3 forwards (qk_bytes, v_bytes =
// bytes per element of q and k, of v).
int check_forward_args(const void* q, const void* k, const void* v, const void* out, int B, int H,
                       int Lq, int Lk, int d, float scale, int qk_bytes, int v_bytes = 2) {
  if (!q || !k || !v || !out) return DIT_ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Lq < 1 || Lk < 1) return DIT_ATTN_ERR_INVALID_ARG;
  if (!logit_scale_ok(scale)) return DIT_ATTN_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
  if (mis & 15u) return DIT_ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return DIT_ATTN_ERR_UNSUPPORTED;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t qblocks = (static_cast<int64_t>(Lq) + dit::kUnitRows - 1) / dit::kUnitRows;
  if (BH > INT_MAX || Lq > INT_MAX - 2 * dit::kUnitRows || Lk > INT_MAX - 2 * dit::kUnitRows ||
      BH * qblocks > INT_MAX)
    return DIT_ATTN_ERR_UNSUPPORTED;
  const int64_t o_bytes = BH * Lq * d * 2, v_all = BH * Lk * d * v_bytes;
  const int64_t q_bytes = BH * Lq * d * qk_bytes, k_bytes = BH * Lk * d * qk_bytes;
  if (overlaps(out, o_bytes, q, q_bytes) || overlaps(out, o_bytes, k, k_bytes) ||
      overlaps(out, o_bytes, v, v_all))
    return DIT_ATTN_ERR_INVALID_ARG;
  return DIT_ATTN_OK;
}

// The optional workspace of the split tail: 16-byte aligned, non-negative size,
// no overlap with the tensors (NULL with size 0 runs unsplit).
int check_workspace(const void* ws, long long ws_bytes, const void* q, const void* k,
                    const void* v, const void* out, int B, int H, int Lq, int Lk, int d,
                    int qk_bytes, int v_bytes = 2) {
  if (ws_bytes < 0 || (ws_bytes > 0 && !ws)) return DIT_ATTN_ERR_INVALID_ARG;
  if (!ws || ws_bytes == 0) return DIT_ATTN_OK;
  if (reinterpret_cast<uintptr_t>(ws) & 15u) return DIT_ATTN_ERR_INVALID_ARG;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t o_bytes = BH * Lq * d * 2, v_all = BH * Lk * d * v_bytes;
  const int64_t q_bytes = BH * Lq * d * qk_bytes, k_bytes = BH * Lk * d * qk_bytes;
  if (overlaps(ws, ws_bytes, q, q_bytes) || overlaps(ws, ws_bytes, k, k_bytes) ||
      overlaps(ws, ws_bytes, v, v_all) || overlaps(ws, ws_bytes, out, o_bytes))
    return DIT_ATTN_ERR_INVALID_ARG;
  return DIT_ATTN_OK;
}

}  // namespace

extern "C" {

int dit_attn_version(void) { return 100; }

const char* dit_attn_status_string(int status) {
  switch (status) {
    case DIT_ATTN_OK: return "ok";
    case DIT_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case DIT_ATTN_ERR_UNSUPPORTED: return "unsupported head dim or size";
    case DIT_ATTN_ERR_NOT_INITIALIZED: return "dit_attn_create() not called for this device";
    case DIT_ATTN_ERR_NO_DEVICE: return "no sm_103 CUDA device";
    case DIT_ATTN_ERR_CUDA: return "CUDA error";
    case DIT_ATTN_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int dit_attn_last_cuda_error(void) { return g_last_cuda_error; }

int dit_attn_create(void) {
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_state[dev].ready) return DIT_ATTN_OK;
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (prop.major != 10 || prop.minor != 3) return DIT_ATTN_ERR_NO_DEVICE;
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return cuda_fail(e);
    if (q != cudaDriverEntryPointSuccess || !fn) return cuda_fail(cudaErrorSymbolNotFound);
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  e = cudaFuncSetAttribute(dit::fmha_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Traits<64>::kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e);
  {
    int rc = DIT_ATTN_OK, bf16_pairs = 0, qk8_pairs = 0, fp8_pairs = 0;
    if ((rc = setup_pair_kernel<false, false>(prop.multiProcessorCount, &bf16_pairs)) != DIT_ATTN_OK)
      return rc;
    if ((rc = setup_pair_kernel<true, false>(prop.multiProcessorCount, &qk8_pairs)) != DIT_ATTN_OK)
      return rc;
    if ((rc = setup_pair_kernel<true, true>(prop.multiProcessorCount, &fp8_pairs)) != DIT_ATTN_OK)
      return rc;
    g_state[dev].max_pairs = bf16_pairs;
    g_state[dev].max_pairs_qk8 = qk8_pairs;
    g_state[dev].max_pairs_fp8 = fp8_pairs;
  }
  {
    // the no-allocation forward's scratch: its device address on this device
    void* scratch = nullptr;
    e = cudaGetSymbolAddress(&scratch, g_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_state[dev].scratch = scratch;
  }
  g_state[dev].num_sms = prop.multiProcessorCount;
  g_state[dev].ready = true;
  return DIT_ATTN_OK;
}

int dit_attn_destroy(void) {
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  g_state[dev] = DeviceState();
  return DIT_ATTN_OK;
}

int dit_attn_forward_ws(const void* q, const void* k, const void* v, void* out, int B, int H,
                        int Lq, int Lk, int d, float scale, void* workspace,
                        long long workspace_bytes, void* stream) {
  int rc = check_forward_args(q, k, v, out, B, H, Lq, Lk, d, scale, 2);
  if (rc != DIT_ATTN_OK) return rc;
  rc = check_workspace(workspace, workspace_bytes, q, k, v, out, B, H, Lq, Lk, d, 2);
  if (rc != DIT_ATTN_OK) return rc;
  const int64_t BH = static_cast<int64_t>(B) * H;
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  int num_sms, max_pairs;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_state[dev].ready) return DIT_ATTN_ERR_NOT_INITIALIZED;
    num_sms = g_state[dev].num_sms;
    max_pairs = g_state[dev].max_pairs;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return d == 64 ? launch<64>(q, k, v, out, BH, Lq, Lk, scale, s, num_sms)
                 : launch_pair<false, false>(q, k, v, out, BH, Lq, Lk, scale, s, max_pairs,
                                             workspace, workspace_bytes);
}

int dit_attn_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int Lq,
                     int Lk, int d, float scale, void* stream) {
  return dit_attn_forward_ws(q, k, v, out, B, H, Lq, Lk, d, scale, nullptr, 0, stream);
}

int dit_attn_forward_qk8_ws(const void* q8, const void* k8, const void* v, void* out, int B,
                            int H, int Lq, int Lk, int d, float scale, float q_scale,
                            float k_scale, void* workspace, long long workspace_bytes,
                            void* stream) {
  int rc = check_forward_args(q8, k8, v, out, B, H, Lq, Lk, d, scale, 1);
  if (rc != DIT_ATTN_OK) return rc;
  if (!std::isfinite(q_scale) || !std::isfinite(k_scale) || q_scale < 0.f || k_scale < 0.f)
    return DIT_ATTN_ERR_INVALID_ARG;
  const double logit_scale = static_cast<double>(scale) * q_scale * k_scale;
  if (!logit_scale_ok(logit_scale)) return DIT_ATTN_ERR_INVALID_ARG;
  if (d != 128) return DIT_ATTN_ERR_UNSUPPORTED;
  rc = check_workspace(workspace, workspace_bytes, q8, k8, v, out, B, H, Lq, Lk, d, 1);
  if (rc != DIT_ATTN_OK) return rc;
  const int64_t BH = static_cast<int64_t>(B) * H;
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  int max_pairs;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_state[dev].ready) return DIT_ATTN_ERR_NOT_INITIALIZED;
    max_pairs = g_state[dev].max_pairs_qk8;
  }
  return launch_pair<true, false>(q8, k8, v, out, BH, Lq, Lk, logit_scale,
                                  static_cast<cudaStream_t>(stream), max_pairs, workspace,
                                  workspace_bytes);
}

int dit_attn_forward_qk8(const void* q8, const void* k8, const void* v, void* out, int B, int H,
                         int Lq, int Lk, int d, float scale, float q_scale, float k_scale,
                         void* stream) {
  return dit_attn_forward_qk8_ws(q8, k8, v, out, B, H, Lq, Lk, d, scale, q_scale, k_scale,
                                 nullptr, 0, stream);
}

int dit_attn_forward_fp8_ws(const void* q8, const void* k8, const void* v8, void* out, int B,
                            int H, int Lq, int Lk, int d, float scale, float q_scale,
                            float k_scale, float v_scale, void* workspace,
                            long long workspace_bytes, void* stream) {
  int rc = check_forward_args(q8, k8, v8, out, B, H, Lq, Lk, d, scale, 1, 1);
  if (rc != DIT_ATTN_OK) return rc;
  if (!std::isfinite(q_scale) || !std::isfinite(k_scale) || q_scale < 0.f || k_scale < 0.f)
    return DIT_ATTN_ERR_INVALID_ARG;
  // 1/v_scale must be finite too: it scales the partial row sums of a split tail
  if (!std::isfinite(v_scale) || !(v_scale > 0.f) || !std::isfinite(1.f / v_scale))
    return DIT_ATTN_ERR_INVALID_ARG;
  const double logit_scale = static_cast<double>(scale) * q_scale * k_scale;
  if (!logit_scale_ok(logit_scale)) return DIT_ATTN_ERR_INVALID_ARG;
  if (d != 128) return DIT_ATTN_ERR_UNSUPPORTED;
  rc = check_workspace(workspace, workspace_bytes, q8, k8, v8, out, B, H, Lq, Lk, d, 1, 1);
  if (rc != DIT_ATTN_OK) return rc;
  const int64_t BH = static_cast<int64_t>(B) * H;
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  int max_pairs;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_state[dev].ready) return DIT_ATTN_ERR_NOT_INITIALIZED;
    max_pairs = g_state[dev].max_pairs_fp8;
  }
  return launch_pair<true, true>(q8, k8, v8, out, BH, Lq, Lk, logit_scale,
                                 static_cast<cudaStream_t>(stream), max_pairs, workspace,
                                 workspace_bytes, v_scale);
}

int dit_attn_forward_fp8(const void* q8, const void* k8, const void* v8, void* out, int B, int H,
                         int Lq, int Lk, int d, float scale, float q_scale, float k_scale,
                         float v_scale, void* stream) {
  return dit_attn_forward_fp8_ws(q8, k8, v8, out, B, H, Lq, Lk, d, scale, q_scale, k_scale,
                                 v_scale, nullptr, 0, stream);
}

}  // extern "C"

extern "C" {

int dit_attn_forward_noalloc(const void* q, const void* k, const void* v, void* out, int B, int H,
                             int Lq, int Lk, int d, float scale, void* stream) {
  const int rc = check_forward_args(q, k, v, out, B, H, Lq, Lk, d, scale, 2);
  if (rc != DIT_ATTN_OK) return rc;
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  void* scratch = nullptr;
  int max_pairs = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_state[dev].ready) return DIT_ATTN_ERR_NOT_INITIALIZED;
    scratch = g_state[dev].scratch;
    max_pairs = g_state[dev].max_pairs;
  }
  if (d == 128) {
    const int64_t units = static_cast<int64_t>(B) * H *
                          ((static_cast<int64_t>(Lq) + kPairUnitRows - 1) / kPairUnitRows);
    if (plan_split(units, (Lk + dit::kBN - 1) / dit::kBN, max_pairs).ws_bytes > kScratchBytes)
      return DIT_ATTN_ERR_UNSUPPORTED;
  }
  return dit_attn_forward_ws(q, k, v, out, B, H, Lq, Lk, d, scale, scratch, kScratchBytes, stream);
}

int dit_attn_workspace_size(int B, int H, int Lq, int Lk, int d, int variant, long long* bytes) {
  if (!bytes) return DIT_ATTN_ERR_INVALID_ARG;
  *bytes = 0;
  if (B < 1 || H < 1 || Lq < 1 || Lk < 1) return DIT_ATTN_ERR_INVALID_ARG;
  if (variant < 0 || variant > 2) return DIT_ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return DIT_ATTN_ERR_UNSUPPORTED;
  if (variant != 0 && d != 128) return DIT_ATTN_ERR_UNSUPPORTED;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t qblocks = (static_cast<int64_t>(Lq) + dit::kUnitRows - 1) / dit::kUnitRows;
  if (BH > INT_MAX || Lq > INT_MAX - 2 * dit::kUnitRows || Lk > INT_MAX - 2 * dit::kUnitRows ||
      BH * qblocks > INT_MAX)
    return DIT_ATTN_ERR_UNSUPPORTED;
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  int max_pairs;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_state[dev].ready) return DIT_ATTN_ERR_NOT_INITIALIZED;
    max_pairs = variant == 2   ? g_state[dev].max_pairs_fp8
                : variant == 1 ? g_state[dev].max_pairs_qk8
                               : g_state[dev].max_pairs;
  }
  if (d == 64) return DIT_ATTN_OK;   // the d = 64 kernel never splits
  const int64_t units = BH * ((static_cast<int64_t>(Lq) + kPairUnitRows - 1) / kPairUnitRows);
  *bytes = plan_split(units, (Lk + dit::kBN - 1) / dit::kBN, max_pairs).ws_bytes;
  return DIT_ATTN_OK;
}

int dit_attn_check_exp2(const void* x, void* y_fma, void* y_mufu, long long n, int degree,
                        void* stream) {
  if (!x || !y_fma || !y_mufu || n < 1 || n > (1ll << 40)) return DIT_ATTN_ERR_INVALID_ARG;
  if (degree != 2 && degree != 3) return DIT_ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y_fma) |
       reinterpret_cast<uintptr_t>(y_mufu)) & 3u)
    return DIT_ATTN_ERR_INVALID_ARG;
  const int64_t nb = static_cast<int64_t>(n) * 4;
  if (overlaps(x, nb, y_fma, nb) || overlaps(x, nb, y_mufu, nb) || overlaps(y_fma, nb, y_mufu, nb))
    return DIT_ATTN_ERR_INVALID_ARG;
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_state[dev].ready) return DIT_ATTN_ERR_NOT_INITIALIZED;
  }
  const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float* xf = static_cast<const float*>(x);
  float* yf = static_cast<float*>(y_fma);
  float* ym = static_cast<float*>(y_mufu);
  if (degree == 2) dit::exp2_check_kernel<2><<<blocks, 256, 0, s>>>(xf, yf, ym, n);
  else dit::exp2_check_kernel<3><<<blocks, 256, 0, s>>>(xf, yf, ym, n);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return DIT_ATTN_OK;
}

int dit_attn_check_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return DIT_ATTN_ERR_INVALID_ARG;
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_state[dev].ready) return DIT_ATTN_ERR_NOT_INITIALIZED;
  }
  dit::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(limit_us) * 1000ull);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return DIT_ATTN_OK;
}

}  // extern "C"

namespace {

// y_bytes = bytes per output element: 2 (bf16, y may equal x) or 1 (e4m3).
int rmsnorm_impl(const void* x, void* y, const void* weight, long long rows, int d, float eps,
                 float out_scale, int y_bytes, void* stream) {
  if (!x || !y) return DIT_ATTN_ERR_INVALID_ARG;
  if (rows < 1 || !std::isfinite(eps) || eps < 0.f) return DIT_ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(out_scale) || out_scale <= 0.f) return DIT_ATTN_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
                        reinterpret_cast<uintptr_t>(weight);
  if (mis & 15u) return DIT_ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return DIT_ATTN_ERR_UNSUPPORTED;
  if (rows > (static_cast<long long>(1) << 40)) return DIT_ATTN_ERR_UNSUPPORTED;
  const int64_t x_bytes = static_cast<int64_t>(rows) * d * 2;
  const int64_t out_bytes = static_cast<int64_t>(rows) * d * y_bytes;
  if (!(y_bytes == 2 && x == y) && overlaps(x, x_bytes, y, out_bytes)) return DIT_ATTN_ERR_INVALID_ARG;
  if (weight && (overlaps(weight, d * 2, y, out_bytes))) return DIT_ATTN_ERR_INVALID_ARG;
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  int num_sms;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_state[dev].ready) return DIT_ATTN_ERR_NOT_INITIALIZED;
    num_sms = g_state[dev].num_sms;
  }
  const int rows_per_block = 8 * (32 / (d / 8)) * 4;
  const int64_t want = (static_cast<int64_t>(rows) + rows_per_block - 1) / rows_per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint4* xv = static_cast<const uint4*>(x);
  const uint4* wv = static_cast<const uint4*>(weight);
  if (y_bytes == 2) {
    if (d == 64) dit::rmsnorm_kernel<64, false><<<grid, 256, 0, s>>>(xv, y, wv, rows, eps, 1.f);
    else dit::rmsnorm_kernel<128, false><<<grid, 256, 0, s>>>(xv, y, wv, rows, eps, 1.f);
  } else {
    if (d == 64) dit::rmsnorm_kernel<64, true><<<grid, 256, 0, s>>>(xv, y, wv, rows, eps, out_scale);
    else dit::rmsnorm_kernel<128, true><<<grid, 256, 0, s>>>(xv, y, wv, rows, eps, out_scale);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return DIT_ATTN_OK;
}

}  // namespace

extern "C" {

int dit_attn_rmsnorm(const void* x, void* y, const void* weight, long long rows, int d, float eps,
                     void* stream) {
  return rmsnorm_impl(x, y, weight, rows, d, eps, 1.f, 2, stream);
}

int dit_attn_rmsnorm_e4m3(const void* x, void* y8, const void* weight, long long rows, int d,
                          float eps, float out_scale, void* stream) {
  return rmsnorm_impl(x, y8, weight, rows, d, eps, out_scale, 1, stream);
}

int dit_attn_quantize_e4m3(const void* x, void* y8, long long n, float out_scale, void* stream) {
  if (!x || !y8 || n < 1) return DIT_ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(out_scale) || !(out_scale > 0.f)) return DIT_ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y8)) & 15u)
    return DIT_ATTN_ERR_INVALID_ARG;
  if (n > (static_cast<long long>(1) << 46)) return DIT_ATTN_ERR_UNSUPPORTED;
  if (overlaps(x, static_cast<int64_t>(n) * 2, y8, n)) return DIT_ATTN_ERR_INVALID_ARG;
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  int num_sms;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_state[dev].ready) return DIT_ATTN_ERR_NOT_INITIALIZED;
    num_sms = g_state[dev].num_sms;
  }
  const int64_t groups = n / 8;
  const int tail = static_cast<int>(n % 8);
  const int64_t per_block = 256 * dit::kQuantInFlight;
  const int64_t want = (groups + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
  dit::quantize_e4m3_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(x), static_cast<uint2*>(y8), groups,
      static_cast<const uint16_t*>(x) + groups * 8, static_cast<uint8_t*>(y8) + groups * 8, tail,
      out_scale);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return DIT_ATTN_OK;
}

int dit_attn_get_device_error(void* stream) {
  int dev = -1;
  if (!current_device(&dev)) return DIT_ATTN_ERR_NO_DEVICE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // one reader at a time: g_error_taken holds the word between the exchange
  // kernel and the copy
  std::lock_guard<std::mutex> lock(g_err_mu);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  dit::take_device_error_kernel<<<1, 1, 0, s>>>();
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  int word = 0;
  e = cudaMemcpyFromSymbolAsync(&word, dit::g_error_taken, sizeof(int), 0,
                                cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  return word != 0 ? word : DIT_ATTN_OK;
}

}  // extern "C"
