// fa_scale.cuh -- exact power-of-two scaling of the fp16 operand copies that the
// bf16 path feeds to the tensor cores next to the fp16 probabilities P and score
// gradients dS.
//
// bf16 has fp32's exponent range, fp16 does not (largest finite 65504, normal down
// to 2^-14, zero below 2^-25). Each copy is therefore x * 2^e with a per-tensor
// exponent e chosen from the tensor's largest magnitude, and every product of the
// scaled copies is brought back by the inverse power of two, folded into a
// multiplier the kernels apply anyway (the softmax scale, the epilogue scale). A
// power of two changes no significand, so the scaled copy of a bf16 value is exact
// whenever it lands in fp16's normal range, and the fp32 arithmetic on the products
// is the same up to that exponent shift. dS itself is formed from the scaled dP and
// the stored row term delta; its exponent comes from a bound on |dS|.
//
// The pre-pass kernels make the copies with e = 0 and record the largest magnitudes
// per block; a small kernel then reduces them, picks the exponents, and rewrites only
// the copies (and delta) whose exponent is not 0. For inputs of ordinary magnitude
// nothing is rewritten and the results are bit-identical to unscaled copies.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#if defined(__CUDACC__)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#endif

namespace fa {

// Exponent bookkeeping (host and device): floor(log2 x) of a non-negative float
// given by its bit pattern; -127 for subnormals, 128 for inf / NaN.
__host__ __device__ inline int flog2_bits(uint32_t b) { return (int)((b >> 23) & 0xFFu) - 127; }

constexpr int COPY_TOP = 14;    // a rescaled copy's largest magnitude lies in [2^14, 2^15)
constexpr int COPY_LO = -2;     // ... unless it already lies in [2^-2, 2^15): e = 0 stands
constexpr int DS_TOP = 15;      // |dS| bound after scaling: below 2^15 (fp16 max 65504)
constexpr int DS_LO = 8;        // bound exponent range [2^8, 2^15) in which e_dS = 0 stands
constexpr int EXP_LIMIT = 120;  // |e| cap: 2^e and its inverse stay normal fp32 numbers

__host__ __device__ inline int clamp_exp(int e) {
  return e < -EXP_LIMIT ? -EXP_LIMIT : (e > EXP_LIMIT ? EXP_LIMIT : e);
}

// Exponent of the fp16 copy of a tensor whose largest magnitude has bits `amax`:
// 0 for an all-zero or non-finite tensor or one already in [2^COPY_LO, 2^15);
// otherwise the e that moves its largest magnitude into [2^14, 2^15).
__host__ __device__ inline int copy_exponent(uint32_t amax) {
  if (amax == 0u) return 0;
  const int fl = flog2_bits(amax);
  if (fl >= 128) return 0;
  if (fl >= COPY_LO && fl <= COPY_TOP) return 0;
  return clamp_exp(COPY_TOP - fl);
}

// Exponent of dS = P (dP - delta). With P <= 1, |dP_ij| = |dO_i . V_j| <= Dv amax(dO)
// amax(V) and |delta_i| <= amax(delta):
//   |dS| < 2^U,  U = max(fl(dO) + fl(V) + dlog + 2, fl(delta) + 1) + 1,
// fl = floor(log2 amax), dlog = ceil(log2 Dv). e_dS = 0 if U is in [DS_LO, DS_TOP],
// else DS_TOP - U. `amax_*` are the unscaled tensors' largest magnitudes.
__host__ __device__ inline int ds_exponent(uint32_t amax_do, uint32_t amax_v,
                                           uint32_t amax_delta, int dlog) {
  if (amax_do == 0u || amax_v == 0u) return 0;  // dS = 0
  const int fg = flog2_bits(amax_do), fv = flog2_bits(amax_v);
  const int fd = amax_delta == 0u ? -127 : flog2_bits(amax_delta);
  if (fg >= 128 || fv >= 128 || fd >= 128) return 0;
  int u = fg + fv + dlog + 2;
  if (fd + 1 > u) u = fd + 1;
  u += 1;
  if (u >= DS_LO && u <= DS_TOP) return 0;
  return clamp_exp(DS_TOP - u);
}

// fp32 inputs carried as two scaled fp16 terms (x 2^e = hi + lo; the default fp32 path,
// the other being 3xTF32): the exponent always moves the
// largest magnitude into [2^14, 2^15), so that the lo terms of the elements stay as far
// above fp16's subnormal range as the tensor's range allows.
__host__ __device__ inline int x16_exponent(uint32_t amax) {
  if (amax == 0u) return 0;
  const int fl = flog2_bits(amax);
  if (fl >= 128) return 0;
  return clamp_exp(COPY_TOP - fl);
}
// ... and dS: the bound's exponent U always moves to DS_TOP (see ds_exponent)
__host__ __device__ inline int x16_ds_exponent(uint32_t amax_do, uint32_t amax_v,
                                               uint32_t amax_delta, int dlog) {
  if (amax_do == 0u || amax_v == 0u) return 0;
  const int fg = flog2_bits(amax_do), fv = flog2_bits(amax_v);
  const int fd = amax_delta == 0u ? -127 : flog2_bits(amax_delta);
  if (fg >= 128 || fv >= 128 || fd >= 128) return 0;
  int u = fg + fv + dlog + 2;
  if (fd + 1 > u) u = fd + 1;
  return clamp_exp(DS_TOP - (u + 1));
}

// Multipliers for the kernels, from the exponents of one call (written once per call
// by the scale kernel, read by every CTA of the attention kernels).
struct OperandScales {
  float sl2;     // score multiplier for the scaled copies: scale * log2(e) * 2^-(eQ + eK)
  float dp_mul;  // 2^(eD - eO - eV): dP from the scaled copies, in units of the stored delta
  float dq_mul;  // dQ epilogue: scale * 2^-(eD + eK)
  float dk_mul;  // dK epilogue: scale * 2^-(eD + eQ)
  float dv_mul;  // dV epilogue: 2^-eO
  float o_mul;   // forward O epilogue: 2^-eV
  int e[5];      // eQ, eK, eV, eO (of dO), eD (of dS)
  int pad;
};
enum { SC_Q = 0, SC_K = 1, SC_V = 2, SC_DO = 3, SC_DS = 4 };

#if defined(__CUDACC__)  // the rest is device code (the rules above also build as host C++)
// Largest |x| over packed bf16 pairs, kept as per-halfword maxima of the magnitude
// bits (bf16 magnitudes order like their bits, inf and NaN above every finite value).
__device__ __forceinline__ uint32_t amax_acc(uint32_t m, uint4 v) {
  m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
  m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
  m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
  m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
  return m;
}
// fp32 bit pattern of the larger of the two halfword maxima
__device__ __forceinline__ uint32_t amax_bits(uint32_t m) {
  const uint32_t lo = m & 0xFFFFu, hi = m >> 16;
  return (lo > hi ? lo : hi) << 16;
}

// Block-wide maximum of N words per thread; thread 0 writes them to out[0..N).
// Every thread of the block must call it (it synchronises the block).
template <int N>
__device__ __forceinline__ void block_max_store(uint32_t (&v)[N], uint32_t* out) {
  __shared__ uint32_t red[32][N];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < N; ++k) v[k] = __reduce_max_sync(0xffffffffu, v[k]);
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < N; ++k) red[wid][k] = v[k];
  __syncthreads();
  if (threadIdx.x < N) {
    uint32_t m = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = max(m, red[w][threadIdx.x]);
    out[threadIdx.x] = m;
  }
}

// Block-wide maximum of the n_part x N partial maxima; every thread gets the result.
template <int N>
__device__ __forceinline__ void reduce_partials(const uint32_t* part, int n_part,
                                                uint32_t (&m)[N]) {
  __shared__ uint32_t red[32][N];
  __shared__ uint32_t fin[N];
#pragma unroll
  for (int k = 0; k < N; ++k) m[k] = 0;
  for (int i = threadIdx.x; i < n_part; i += blockDim.x)
#pragma unroll
    for (int k = 0; k < N; ++k) m[k] = max(m[k], part[(size_t)i * N + k]);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < N; ++k) m[k] = __reduce_max_sync(0xffffffffu, m[k]);
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < N; ++k) red[wid][k] = m[k];
  __syncthreads();
  if (threadIdx.x < N) {
    uint32_t r = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = max(r, red[w][threadIdx.x]);
    fin[threadIdx.x] = r;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; ++k) m[k] = fin[k];
}

// Per-block largest |x| of up to 5 fp32 arrays (fp32 magnitudes order like their bits):
// block b writes part[N b + k] for array k. Grid-stride over 4-element vectors.
struct AmaxJobs {
  const float* a[5];
  size_t n4[5];  // 4-element vectors per array
  int n;         // arrays
};
namespace {  // (each translation unit gets its own copy of the kernel)
template <int N>
__global__ void __launch_bounds__(256) amax_f32_kernel(const __grid_constant__ AmaxJobs js,
                                                       uint32_t* __restrict__ part) {
  // (launched as a programmatic dependent after the delta pass: its arrays are read only
  // once that grid has completed; a plain launch returns from the wait at once)
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();
  uint32_t m[N];
  const size_t stride = (size_t)gridDim.x * blockDim.x;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    m[k] = 0;
    if (k >= js.n) continue;
    const uint4* p = reinterpret_cast<const uint4*>(js.a[k]);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < js.n4[k]; i += stride) {
      const uint4 v = p[i];
      m[k] = max(max(m[k], max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu)),
                 max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu));
    }
  }
  block_max_store<N>(m, part + (size_t)blockIdx.x * N);
}
}  // namespace

// x 2^e = hi + lo, hi = fp16(x 2^e), lo = fp16(x 2^e - hi), for n4 vectors of 4 fp32
// values; grid-stride.
__device__ __forceinline__ void split_x16(const float* __restrict__ x, __half* __restrict__ hi,
                                          __half* __restrict__ lo, size_t n4, int e) {
  const float f = __uint_as_float((uint32_t)(127 + e) << 23);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = reinterpret_cast<const float4*>(x)[i];
    const float y[4] = {v.x * f, v.y * f, v.z * f, v.w * f};
    uint32_t h[2], l[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const __half2 hh = __floats2half2_rn(y[2 * k], y[2 * k + 1]);
      const float2 hf = __half22float2(hh);
      const __half2 ll = __floats2half2_rn(y[2 * k] - hf.x, y[2 * k + 1] - hf.y);
      h[k] = *reinterpret_cast<const uint32_t*>(&hh);
      l[k] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    reinterpret_cast<uint2*>(hi)[i] = make_uint2(h[0], h[1]);
    reinterpret_cast<uint2*>(lo)[i] = make_uint2(l[0], l[1]);
  }
}

// 2^e as a float, |e| <= EXP_LIMIT (exact: a normal power of two).
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// Rewrites n8 groups of 8 values: dst = fp16(src * 2^e), src bf16. Grid-stride, four
// 16-byte loads in flight per thread.
__device__ __forceinline__ void rescale_copy(const __nv_bfloat16* __restrict__ src,
                                             __half* __restrict__ dst, size_t n8, int e) {
  const float f = pow2i(e);
  auto cvt = [f](uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 h = __floats2half2_rn(__uint_as_float(w[k] << 16) * f,
                                    __uint_as_float(w[k] & 0xFFFF0000u) * f);
      o[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
  const uint4* in = reinterpret_cast<const uint4*>(src);
  uint4* out = reinterpret_cast<uint4*>(dst);
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
#endif  // __CUDACC__

}  // namespace fa
