// RMS normalisation of queries or keys, per token and head, over the head
// dimension: y[r, :] = bf16(x[r, :] / sqrt(mean(x[r, :]^2) + eps) * w), with
// fp32 arithmetic.  The normalised workloads of the joint attention apply it
// to Q and K before the attention forward.  With kE4M3 the same value times
// out_scale is rounded to e4m3 (nearest even, saturating at +-448) instead:
// the quantising prologue of the e4m3-QK forward, one pass over the tensor.
//
// HBM-bound: every row is read once and written once.  A lane reads 16 bytes
// (8 bf16) per access; D/8 lanes cover a row, so one warp instruction reads
// 512 contiguous bytes; each lane group keeps kRowsInFlight rows in flight.
#pragma once

namespace dit {

template <int D, bool kE4M3>
__global__ void __launch_bounds__(256)
    rmsnorm_kernel(const uint4* x, void* y, const uint4* __restrict__ w, int64_t rows, float eps,
                   float out_scale) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  constexpr int kRowsInFlight = 4;
  constexpr int kRowsPerStep = kRowsPerWarp * kRowsInFlight;
  const int lane = threadIdx.x & 31;
  const int chunk = lane % kLanesPerRow;   // 8-column chunk of the row
  const int grp = lane / kLanesPerRow;     // row of the warp's group
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * blockDim.x / 32;

  float wf[8];
  if (w) {
    const uint4 wv = w[chunk];
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      wf[2 * i] = __uint_as_float(ww[i] << 16);
      wf[2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) wf[i] = 1.f;
  }

  for (int64_t base = warp * kRowsPerStep; base < rows; base += n_warps * kRowsPerStep) {
    uint4 v[kRowsInFlight];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int64_t r = base + u * kRowsPerWarp + grp;
      v[u] = r < rows ? x[r * kLanesPerRow + chunk] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const uint32_t vv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      float f[8];
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(vv[i] << 16);
        f[2 * i + 1] = __uint_as_float(vv[i] & 0xFFFF0000u);
        ss = fmaf(f[2 * i], f[2 * i], ss);
        ss = fmaf(f[2 * i + 1], f[2 * i + 1], ss);
      }
#pragma unroll
      for (int off = kLanesPerRow / 2; off > 0; off /= 2)
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float inv = rsqrtf(ss * (1.f / D) + eps);
      const int64_t r = base + u * kRowsPerWarp + grp;
      if constexpr (kE4M3) {
        float g[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) g[i] = f[i] * inv * wf[i] * out_scale;
        const uint2 o = make_uint2(pack_e4m3x4(g[0], g[1], g[2], g[3]),
                                   pack_e4m3x4(g[4], g[5], g[6], g[7]));
        if (r < rows) static_cast<uint2*>(y)[r * kLanesPerRow + chunk] = o;
      } else {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          o[i] = pack_bf16x2(f[2 * i] * inv * wf[2 * i], f[2 * i + 1] * inv * wf[2 * i + 1]);
        if (r < rows) static_cast<uint4*>(y)[r * kLanesPerRow + chunk] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

}  // namespace dit
