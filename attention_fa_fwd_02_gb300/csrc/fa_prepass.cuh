// fa_prepass.cuh -- memory-bound element-wise kernels that prepare tensor-core
// operands: bf16 -> fp16 copies (partner operands of the fp16 P / dS) and tf32
// hi / lo splits (optionally transposed) for the 3xTF32 fp32 path.
// Each translation unit gets its own (internal-linkage) copy.
#pragma once
#include <cstdint>
#include <initializer_list>
#include "ptx.cuh"
#include "fa_scale.cuh"

namespace fa {
namespace {

// bf16 -> fp16 copy with exponent 0 (exact for 2^-14 <= |x| <= 65504), 8 elements per
// 16-byte vector; block b also writes part[b], the largest |x| it read (fp32 bits),
// from which the scale kernel decides whether the copy must be redone scaled.
__global__ void cvt_bf16_to_f16_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                       size_t n8, uint32_t* __restrict__ part) {
  // the scale kernel launched after this one (a programmatic dependent) may be
  // scheduled as soon as SMs free up; it waits for this grid before reading part[]
  ptx::grid_launch_dependents();
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
  uint32_t m = 0;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = in[i + u * stride];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      out[i + u * stride] = cvt(v[u]);
      m = amax_acc(m, v[u]);
    }
  }
  for (; i < n8; i += stride) {
    const uint4 v = in[i];
    out[i] = cvt(v);
    m = amax_acc(m, v);
  }
  uint32_t mv[1] = {amax_bits(m)};
  block_max_store<1>(mv, part + blockIdx.x);
}

// x = hi + lo with hi = x with its low 13 mantissa bits cleared (a tf32 value)
// and lo = x - hi (exact in fp32). One tensor of a split launch: n_slabs x rows x D
// fp32 values at `in`; `hi` / `lo` (if hi is non-null) receive the pair in the same
// layout, `hi_t` / `lo_t` (if hi_t is non-null) receive it transposed per slab,
// [n_slabs][D][ld_t].
struct SplitJob {
  const float* in;
  float* hi;
  float* lo;
  float* hi_t;
  float* lo_t;
  int rows, ld_t, n_slabs;
};
constexpr int SPLIT_MAX_JOBS = 4, SPLIT_ROWS = 32, SPLIT_MAX_D = 64;
struct SplitJobs {
  SplitJob j[SPLIT_MAX_JOBS];
  int n, D;  // jobs, columns (a multiple of 16, at most SPLIT_MAX_D)
};

// All jobs of one launch as one list of tiles of SPLIT_ROWS rows (one slab each),
// jobs one after another, taken grid-stride by whole blocks. A tile is read with
// 16-byte loads and written back in the input layout with 16-byte stores; the
// transposed copy goes through a padded shared-memory tile so that each of its D
// rows leaves as SPLIT_ROWS consecutive floats (128 bytes).
__global__ void __launch_bounds__(256) split_tf32_kernel(const __grid_constant__ SplitJobs js) {
  __shared__ float th[SPLIT_MAX_D][SPLIT_ROWS + 1], tl[SPLIT_MAX_D][SPLIT_ROWS + 1];
  const int D = js.D, q4 = D / 4;
  long long total = 0;
  for (int k = 0; k < js.n; ++k)
    total += (long long)js.j[k].n_slabs * ((js.j[k].rows + SPLIT_ROWS - 1) / SPLIT_ROWS);
  for (long long t = blockIdx.x; t < total; t += gridDim.x) {
    int k = 0;
    long long u = t;  // tile index within job k
    for (; k < js.n - 1; ++k) {
      const long long tk =
          (long long)js.j[k].n_slabs * ((js.j[k].rows + SPLIT_ROWS - 1) / SPLIT_ROWS);
      if (u < tk) break;
      u -= tk;
    }
    const SplitJob& jb = js.j[k];
    const int tiles = (jb.rows + SPLIT_ROWS - 1) / SPLIT_ROWS;
    const long long slab = u / tiles;
    const int r0 = (int)(u - slab * tiles) * SPLIT_ROWS;
    const int nr = min(SPLIT_ROWS, jb.rows - r0);
    const size_t base = ((size_t)slab * jb.rows + r0) * D;
    for (int e = threadIdx.x; e < nr * q4; e += blockDim.x) {
      const int r = e / q4, c = (e - r * q4) * 4;
      const float4 x = *reinterpret_cast<const float4*>(jb.in + base + (size_t)r * D + c);
      const float xs[4] = {x.x, x.y, x.z, x.w};
      float h[4], l[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        h[v] = __uint_as_float(__float_as_uint(xs[v]) & 0xFFFFE000u);
        l[v] = xs[v] - h[v];
      }
      if (jb.hi) {
        *reinterpret_cast<float4*>(jb.hi + base + (size_t)r * D + c) = make_float4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<float4*>(jb.lo + base + (size_t)r * D + c) = make_float4(l[0], l[1], l[2], l[3]);
      }
      if (jb.hi_t) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          th[c + v][r] = h[v];
          tl[c + v][r] = l[v];
        }
      }
    }
    if (jb.hi_t) {  // (the same job, hence the same branch, for the whole block)
      __syncthreads();
      for (int e = threadIdx.x; e < D * SPLIT_ROWS; e += blockDim.x) {
        const int d = e / SPLIT_ROWS, r = e % SPLIT_ROWS;
        if (r < nr) {
          const size_t o = ((size_t)slab * D + d) * jb.ld_t + r0 + r;
          jb.hi_t[o] = th[d][r];
          jb.lo_t[o] = tl[d][r];
        }
      }
      __syncthreads();
    }
  }
}

// One launch for up to SPLIT_MAX_JOBS tensors of D <= SPLIT_MAX_D columns.
inline void launch_split_tf32(std::initializer_list<SplitJob> jobs, int D, int grid,
                              cudaStream_t stream) {
  SplitJobs js = {};
  js.n = 0;
  js.D = D;
  for (const SplitJob& jb : jobs) js.j[js.n++] = jb;
  split_tf32_kernel<<<grid, 256, 0, stream>>>(js);
}

}  // namespace
}  // namespace fa
