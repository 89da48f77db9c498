// fa_common.cuh -- tiling constants, tile-range arithmetic and host helpers shared
// by the forward and backward translation units of libfa.so.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include "fa.h"

namespace fa {

constexpr int BLOCK_M = 128;  // query rows per tile (tcgen05 M = 128, one TMEM lane per row)
constexpr int BLOCK_N = 128;  // key rows per tile
constexpr uint32_t SW128_ROW = 128;          // bytes per swizzled smem row
constexpr uint32_t SW128_ATOM = 1024;        // 8 rows x 128 bytes
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
// Rescale O only when the running max grows by more than this (log2 units): the
// unnormalised probabilities then stay below 2^8, well inside fp16 range.
constexpr float RESCALE_THRESHOLD = 8.0f;
// Short query sequences split each work item's keys into at most this many ranges
// (forward and dQ), whose partial results a combine kernel adds up, KEY_RANGE_GROUP
// ranges' loads in flight at a time.
constexpr int MAX_KEY_RANGES = 32;
constexpr int KEY_RANGE_GROUP = 16;

// Key tiles per range for a pass whose `base` work items (one persistent CTA per SM,
// `sms` of them) are fewer than the SMs: the split count s (ranges of at least 4 of
// the n_kt key tiles, at most MAX_KEY_RANGES) that minimises the estimated finish
// time ceil(base * s / sms) * (ceil(n_kt / s) + 2), i.e. rounds of equal items, each
// costing its key tiles plus about two tiles' worth of item overhead. n_kt: no split.
inline int key_range_tiles(int base, int n_kt, int sms) {
  if (base >= sms || n_kt < 8) return n_kt;
  int best_t = n_kt;
  long long best = -1;
  for (int s = 1; s <= MAX_KEY_RANGES && s <= n_kt / 4; ++s) {
    const int t = (n_kt + s - 1) / s, ns = (n_kt + t - 1) / t;
    const long long cost = ((long long)base * ns + sms - 1) / sms * (t + 2);
    if (best < 0 || cost < best) { best = cost; best_t = t; }
  }
  return best_t;
}

// bf16 inputs: whether P (forward and backward) and dS (backward) enter the
// accumulating products as two fp16 terms each. A dK / dV CTA walks rep * n_qt query
// chunks (the grouped heads' query tiles); with at most 8 of them that kernel is bound
// by its per-CTA set-up, not the tensor pipe, and short query sequences against long
// key sequences are where one key can take almost all of a row's weight, which one
// fp16 term of P / dS does not resolve to the 2e-2-of-RMS accuracy of the bf16 path.
// The forward follows the same rule, as its O enters the backward's D_i = dO_i . O_i.
inline bool split_operands(int rep, int n_qt) { return (long long)rep * n_qt <= 8; }

// Launch shape of the key-range combine kernels (one thread per 4 of a row's Dv
// columns): blockDim (Dv / 4, rows per block), about 64 threads; grid (row blocks,
// heads, at most 65535: the kernels loop over the rest).
inline void combine_launch_shape(int BH, int Sq, int Dv, dim3* grid, dim3* block) {
  const int q4 = Dv / 4, rpb = 64 / q4 > 1 ? 64 / q4 : 1;
  *block = dim3(q4, rpb);
  *grid = dim3((Sq + rpb - 1) / rpb, BH < 65535 ? BH : 65535);
}

// Operand tiles of 16-bit elements for head dim D: rows of min(2 D, 128) bytes, with
// the swizzle of that width (D = 32: 64-byte rows, so that the tensor cores do not
// work on padding columns).
constexpr int tile_row_bytes(int D) { return 2 * D < 128 ? 2 * D : 128; }

// Input precision of a kernel instantiation (the integer F32 template argument of the
// forward and backward kernels and their launchers): bf16 inputs; fp32 inputs as two
// scaled fp16 terms per operand (three kind::f16 products per GEMM); fp32 inputs as
// hi / lo tf32 splits (three kind::tf32 products per GEMM, head dims up to 64).
enum : int { IN_BF16 = 0, IN_F32_X16 = 1, IN_F32_TF32 = 2 };

// Status bits a kernel may set in its device status word.
enum : unsigned int {
  DEV_TIMEOUT = 1u,  // a barrier wait gave up
  DEV_LAYOUT = 2u,   // a kernel's shared-memory layout did not fit its allocation
};

// Half-open range [lo, hi) of key tiles that query rows [r0, r1] may attend to:
// key j is visible to row i iff j < Sk, (!causal || j <= i) and
// (window == 0 || j >= i - window + 1). Blocks wholly outside the band are
// skipped (forge flash_attn_fwd: kb limit for causal, tg_jmin for the window).
__host__ __device__ inline void kv_tile_range(int r0, int r1, int Sk, int causal, int window,
                                              int* lo, int* hi) {
  int jmax = Sk - 1;
  if (causal && r1 < jmax) jmax = r1;
  int jmin = 0;
  if (window > 0 && r0 - window + 1 > 0) jmin = r0 - window + 1;
  if (jmax < jmin) { *lo = 0; *hi = 0; return; }
  *lo = jmin / BLOCK_N;
  *hi = jmax / BLOCK_N + 1;
}

// Half-open range [lo, hi) of query tiles whose rows may see key rows [c0, c1]
// (the transpose of kv_tile_range; forge flash_attn_bwd_dv / _dk imin / imax).
__host__ __device__ inline void q_tile_range(int c0, int c1, int Sq, int causal, int window,
                                             int* lo, int* hi) {
  int imin = 0;
  if (causal) imin = c0;
  int imax = Sq - 1;
  if (window > 0) {
    long long lim = (long long)c1 + window - 1;
    if (lim < imax) imax = (int)lim;
  }
  if (imax < imin) { *lo = 0; *hi = 0; return; }
  *lo = imin / BLOCK_M;
  *hi = imax / BLOCK_M + 1;
}

// True if some (row, key) pair of the tile pair is invisible, i.e. the tile needs
// the per-element mask; interior tiles skip it (forge flash_attn_fwd: only the
// diagonal block pays the mask test).
__host__ __device__ inline bool tile_needs_mask(int r0, int r1, int c0, int c1, int Sk,
                                                int causal, int window) {
  if (c1 >= Sk) return true;
  if (causal && c1 > r0) return true;
  if (window > 0 && (long long)c0 < (long long)r1 - window + 1) return true;
  return false;
}

#if defined(__CUDACC__)
// x[c] = -inf for the columns c in [0, N) outside [lo, hi] (N a multiple of 32; an
// empty range when hi < lo). The kept columns become one bit mask per 32 columns and
// each element one bit test and select: about a third of the issue time of two
// comparisons per element.
template <int N>
__device__ __forceinline__ void mask_outside(float (&x)[N], int lo, int hi) {
  static_assert(N % 32 == 0, "32 columns per mask word");
#pragma unroll
  for (int w = 0; w < N / 32; ++w) {
    // (64-bit: lo and hi may sit near the ends of the int range)
    const int l = (int)min(max((long long)lo - 32 * w, 0ll), 32ll);
    const int h = (int)min(max((long long)hi - 32 * w + 1, 0ll), 32ll);
    const uint32_t below_h = h >= 32 ? 0xffffffffu : ((1u << h) - 1u);
    const uint32_t below_l = l >= 32 ? 0xffffffffu : ((1u << l) - 1u);
    const uint32_t keep = below_h & ~below_l;
#pragma unroll
    for (int b = 0; b < 32; ++b) x[32 * w + b] = ((keep >> b) & 1u) ? x[32 * w + b] : -INFINITY;
  }
}
#endif  // __CUDACC__

// ---------------------------------------------------------------- host side
namespace host {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
// A [outer][rows][inner] tensor whose rows are `row_stride` elements apart and whose
// outer slabs are rows * row_stride elements apart; box {box_inner, box_rows, 1},
// zero fill out of bounds; `swizzle_bytes` 128 (the default), 64 or 0 (none).
bool encode_tiled_3d(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base,
                     uint64_t inner, uint64_t rows, uint64_t outer, uint64_t row_stride,
                     uint32_t box_inner, uint32_t box_rows, int swizzle_bytes = 128);

// Stream-ordered scratch from a library-owned pool on the current device.
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s);
cudaError_t scratch_free(void* p, cudaStream_t s);

int sm_count();

// Largest dynamic shared-memory size a block of `kernel` may request on the current
// device (the per-block opt-in limit minus the kernel's static shared memory).
cudaError_t max_dynamic_smem(const void* kernel, int* bytes);

// Records a CUDA event pair around the launches made during its lifetime when
// kernel timing is enabled (fa_timing_enable); otherwise does nothing.
class KernelTimer {
 public:
  KernelTimer(const char* name, cudaStream_t s);
  ~KernelTimer();
  KernelTimer(const KernelTimer&) = delete;
  KernelTimer& operator=(const KernelTimer&) = delete;

 private:
  const char* name_;
  cudaStream_t stream_;
  cudaEvent_t start_ = nullptr;
};

}  // namespace host

// Launchers implemented by the kernel translation units.
fa_status launch_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     const fa_params& p, cudaStream_t stream);
fa_status launch_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* LSE, void* dQ, void* dK, void* dV, const fa_params& p,
                     cudaStream_t stream, bool dsmat);
fa_status launch_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE,
                             const fa_params& p, cudaStream_t stream);
fa_status launch_selftest_timeout(unsigned long long limit_ns, int* roles_done, cudaStream_t s);
unsigned int read_and_clear_fwd_status(cudaError_t* err);
unsigned int read_and_clear_bwd_status(cudaError_t* err);

// Launches `kernel` on `stream` (with `smem` bytes of dynamic shared memory) as a
// programmatic dependent of the grid launched before it there: its blocks may be
// scheduled once every block of that grid has signalled (griddepcontrol.launch_dependents)
// or exited, and the kernel must execute griddepcontrol.wait before it reads anything that
// grid writes -- and before it exits, so that it cannot complete before that grid (the
// kernels after it rely on the order).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_programmatic_smem(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                           size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same without dynamic shared memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_programmatic(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                      cudaStream_t stream, Args... args) {
  return launch_programmatic_smem(kernel, grid, block, 0, stream, args...);
}

// Default barrier-wait limit (ns) for the kernels.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

}  // namespace fa
