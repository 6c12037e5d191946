// Per-tensor e4m3 quantisation of a bf16 tensor: y[i] = e4m3(x[i] * out_scale),
// the product in fp32, rounded to nearest even and saturated at +-448 (a NaN
// stays NaN).  It produces the e4m3 values of the e4m3 Q/K/V forward (and any
// Q or K that is not RMS-normalised); out_scale is the inverse of the
// per-tensor dequantisation scale the forward is given.
//
// HBM-bound: 2 bytes read and 1 written per element.  A thread converts groups
// of eight elements (a 16-byte load, an 8-byte store) and keeps
// kQuantInFlight groups in flight; the grid strides over the groups.  The last
// n % 8 elements are done one by one by the first threads of block 0.
#pragma once

namespace dit {

constexpr int kQuantInFlight = 4;

__global__ void __launch_bounds__(256)
    quantize_e4m3_kernel(const uint4* __restrict__ x, uint2* __restrict__ y, int64_t groups,
                         const uint16_t* __restrict__ x_tail, uint8_t* __restrict__ y_tail,
                         int tail, float out_scale) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g0 = tid; g0 < groups; g0 += stride * kQuantInFlight) {
    uint4 v[kQuantInFlight];
#pragma unroll
    for (int u = 0; u < kQuantInFlight; ++u) {
      const int64_t g = g0 + u * stride;
      v[u] = g < groups ? x[g] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQuantInFlight; ++u) {
      const uint32_t vv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(vv[i] << 16) * out_scale;
        f[2 * i + 1] = __uint_as_float(vv[i] & 0xFFFF0000u) * out_scale;
      }
      const int64_t g = g0 + u * stride;
      if (g < groups)
        y[g] = make_uint2(pack_e4m3x4(f[0], f[1], f[2], f[3]), pack_e4m3x4(f[4], f[5], f[6], f[7]));
    }
  }
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail) {
    const float f = __uint_as_float(static_cast<uint32_t>(x_tail[threadIdx.x]) << 16) * out_scale;
    y_tail[threadIdx.x] = static_cast<uint8_t>(pack_e4m3x4(f, 0.f, 0.f, 0.f) & 0xFFu);
  }
}

}  // namespace dit
