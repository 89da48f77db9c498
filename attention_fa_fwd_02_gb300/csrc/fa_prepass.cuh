// fa_prepass.cuh -- memory-bound element-wise kernels that prepare tensor-core
// operands: bf16 -> fp16 copies (partner operands of the fp16 P / dS) and tf32
// hi / lo splits (optionally transposed) for the 3xTF32 fp32 path.
// Each translation unit gets its own (internal-linkage) copy.
#pragma once
#include <cstdint>
#include "ptx.cuh"

namespace fa {
namespace {

// bf16 -> fp16, exact for 2^-14 <= |x| <= 65504. 8 elements per 16-byte vector.
__global__ void cvt_bf16_to_f16_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                       size_t n8) {
  // four independent 16-byte loads in flight per thread, then the grid-stride tail
  auto cvt = [](uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16);
      const float hi = __uint_as_float(w[e] & 0xFFFF0000u);
      o[e] = ptx::pack_half2(lo, hi);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = in[i + u * stride];
#pragma unroll
    for (int u = 0; u < 4; ++u) out[i + u * stride] = cvt(v[u]);
  }
  for (; i < n8; i += stride) out[i] = cvt(in[i]);
}

// x = hi + lo with hi = x with its low 13 mantissa bits cleared (a tf32 value)
// and lo = x - hi (exact in fp32). `hi`/`lo` receive the pair in the input layout
// ([slabs][rows][D]); `hi_t`/`lo_t` (if non-null) receive it transposed per slab
// ([slabs][D][ld_t]).
__global__ void split_tf32_kernel(const float* __restrict__ in, float* __restrict__ hi,
                                  float* __restrict__ lo, float* __restrict__ hi_t,
                                  float* __restrict__ lo_t, int rows, int D, int ld_t,
                                  size_t n_slabs) {
  const size_t total = n_slabs * (size_t)rows * D;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const float x = in[idx];
    const float xh = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    const float xl = x - xh;
    if (hi) { hi[idx] = xh; lo[idx] = xl; }
    if (hi_t) {
      const size_t slab = idx / ((size_t)rows * D);
      const size_t rem = idx % ((size_t)rows * D);
      const size_t r = rem / D, d = rem % D;
      const size_t o = slab * (size_t)D * ld_t + d * ld_t + r;
      hi_t[o] = xh;
      lo_t[o] = xl;
    }
  }
}

}  // namespace
}  // namespace fa
