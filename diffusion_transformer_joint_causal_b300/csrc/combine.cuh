// Merge of the key-range chunks of split work units (the last, partial wave of
// a persistent launch).  Each chunk stores, per query row, its running max m_s
// (log2 units), its row sum l_s and its unnormalised output O_s, all against
// its own m_s.  The row's result is the same online-softmax merge the kernel
// does across key tiles:
//
//     M = max_s m_s,   o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,
//
// rounded to nearest-even bf16.  One warp per row, D/32 columns per lane;
// rows at or beyond Lq are not stored.
#pragma once

namespace dit {

template <int D>
__global__ void __launch_bounds__(256)
    combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                   __nv_bfloat16* out, int split_base, int splits, int num_qblocks, int Lq,
                   int64_t rows) {
  static_assert(D == 128, "the split tail runs on the d = 128 pair kernel");
  constexpr int kUnit = 2 * kUnitRows;   // query rows of a pair work unit
  const int64_t wrow = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (wrow >= rows) return;
  const int64_t su = wrow / kUnit;                 // split unit, counted from split_base
  const int prow = static_cast<int>(wrow % kUnit);
  const int64_t u = split_base + su;
  const int64_t bh = u / num_qblocks;
  const int row = static_cast<int>(u % num_qblocks) * kUnit + prow;
  if (row >= Lq) return;
  const float2* ml = reinterpret_cast<const float2*>(part_ml);
  float m_max = -INFINITY;
  for (int s = 0; s < splits; ++s) m_max = fmaxf(m_max, ml[(su * splits + s) * kUnit + prow].x);
  float l_sum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < splits; ++s) {
    const int64_t c = (su * splits + s) * kUnit + prow;
    const float2 v = ml[c];
    const float wgt = exp2f(v.x - m_max);
    l_sum = fmaf(wgt, v.y, l_sum);
    const float4 o = reinterpret_cast<const float4*>(part_o + c * D)[lane];
    acc.x = fmaf(wgt, o.x, acc.x);
    acc.y = fmaf(wgt, o.y, acc.y);
    acc.z = fmaf(wgt, o.z, acc.z);
    acc.w = fmaf(wgt, o.w, acc.w);
  }
  const float inv = 1.f / l_sum;
  reinterpret_cast<uint2*>(out + (bh * Lq + row) * D)[lane] =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

}  // namespace dit
