// fa_api.cu -- the extern "C" boundary of libfa.so (declared in include/fa.h):
// argument validation, the library's stream-ordered scratch pool, TMA descriptor
// encoding and the device status word. Kernels live in fa_fwd.cu / fa_bwd.cu.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>
#include <cudaTypedefs.h>
#include "fa_common.cuh"

namespace fa {
namespace host {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

constexpr int MAX_DEVICES = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pool[MAX_DEVICES] = {};
int g_sms[MAX_DEVICES] = {};
}  // namespace

bool encode_tiled_3d(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base,
                     uint64_t inner, uint64_t rows, uint64_t outer, uint64_t row_stride,
                     uint32_t box_inner, uint32_t box_rows, int swizzle_bytes) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {row_stride * esize, row_stride * esize * rows};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                        : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static cudaError_t pool_for_current_device(cudaMemPool_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_pool_mu);
  if (!g_pool[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;  // keep freed blocks for reuse instead of returning them
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    g_pool[dev] = pool;
  }
  *out = g_pool[dev];
  return cudaSuccess;
}

cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s) {
  cudaMemPool_t pool;
  cudaError_t e = pool_for_current_device(&pool);
  if (e != cudaSuccess) return e;
  return cudaMallocFromPoolAsync(p, bytes < 256 ? 256 : bytes, pool, s);
}

cudaError_t scratch_free(void* p, cudaStream_t s) {
  return p ? cudaFreeAsync(p, s) : cudaSuccess;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return 148;
  if (!g_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 148;
  }
  return g_sms[dev];
}

cudaError_t max_dynamic_smem(const void* kernel, int* bytes) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa_attr;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa_attr, kernel);
  if (e != cudaSuccess) return e;
  *bytes = optin - (int)fa_attr.sharedSizeBytes;
  return *bytes > 0 ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {
struct Pending {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_t_mu;
bool g_t_on = false;
std::vector<Pending> g_t_pending;
std::vector<cudaEvent_t> g_t_free;

cudaEvent_t take_event() {
  if (!g_t_free.empty()) {
    cudaEvent_t e = g_t_free.back();
    g_t_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

KernelTimer::KernelTimer(const char* name, cudaStream_t s) : name_(name), stream_(s) {
  std::lock_guard<std::mutex> lk(g_t_mu);
  if (!g_t_on) return;
  start_ = take_event();
  if (start_) cudaEventRecord(start_, stream_);
}

KernelTimer::~KernelTimer() {
  if (!start_) return;
  std::lock_guard<std::mutex> lk(g_t_mu);
  cudaEvent_t end = take_event();
  if (!end) { g_t_free.push_back(start_); return; }
  cudaEventRecord(end, stream_);
  g_t_pending.push_back({name_, start_, end});
}

}  // namespace host

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by fa_fwd and fa_bwd (see the field comments in fa.h).
fa_status validate(const fa_params* p) {
  if (!p) return FA_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || p->HKV < 1 || p->Sq < 0 || p->Sk < 0 || p->D < 1)
    return FA_ERR_INVALID_ARG;
  if (p->H % p->HKV != 0) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(p->scale) && p->scale > 0.f)) return FA_ERR_INVALID_ARG;
  if ((p->causal != 0 && p->causal != 1) || p->window < 0) return FA_ERR_INVALID_ARG;
  if ((p->in_dtype != FA_F32 && p->in_dtype != FA_BF16) ||
      (p->out_dtype != FA_F32 && p->out_dtype != FA_BF16) ||
      (p->f32_mma != FA_F32_MMA_F16X2 && p->f32_mma != FA_F32_MMA_TF32X3))
    return FA_ERR_INVALID_ARG;
  // Index arithmetic inside the kernels uses 32-bit row / head / grid counters.
  const long long bh = (long long)p->B * p->H;
  if (bh > (1ll << 30) || p->Sq > (1 << 30) || p->Sk > (1 << 30)) return FA_ERR_INVALID_ARG;
  if (bh * ((p->Sq + 255) / 256) > (1ll << 31) - 1) return FA_ERR_INVALID_ARG;
  // Every tensor's byte size (and the scratch sized from it) must be far from wrapping
  // a size_t: at most 2^50 bytes per tensor, in fp32, checked in double (no overflow).
  const double lim = 1125899906842624.0;  // 2^50
  if ((double)p->B * p->H * p->Sq * p->D * 4.0 > lim ||
      (double)p->B * p->HKV * p->Sk * p->D * 4.0 > lim)
    return FA_ERR_INVALID_ARG;
  // Head dims: multiples of 16 up to 128 (3xTF32: up to 64); each runs in the kernel
  // built for the next of 32 (bf16 in, fp32 out), 64 and 128, with the missing columns
  // read as zeros.
  const bool d16 = p->D % 16 == 0 && p->D >= 16;
  const bool ok_bf16 = p->in_dtype == FA_BF16 && d16 && p->D <= 128;
  const bool ok_f32 = p->in_dtype == FA_F32 && d16 &&
                      p->D <= (p->f32_mma == FA_F32_MMA_TF32X3 ? 64 : 128);
  if (!ok_bf16 && !ok_f32) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// A window of at least Sq keys excludes nothing (every key j >= 0 >= i - window + 1
// for i < Sq); dropping it keeps all kernel index arithmetic within 31 bits.
fa_params normalized(const fa_params& p) {
  fa_params q = p;
  if (q.window >= q.Sq) q.window = 0;
  return q;
}

fa_status check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* q : ptrs) {
    if (!q) return FA_ERR_INVALID_ARG;
    if (!aligned16(q)) return FA_ERR_ALIGNMENT;
  }
  return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

FA_API fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        const fa_params* p, fa_stream_t stream) {
  fa_status st = validate(p);
  if (st != FA_OK) return st;
  if (p->Sq == 0) return FA_OK;  // nothing to compute
  st = check_ptrs({O, LSE, Q});
  if (st != FA_OK) return st;
  if (p->Sk > 0) {
    st = check_ptrs({K, V});
    if (st != FA_OK) return st;
  }
  return launch_fwd(Q, K, V, O, LSE, normalized(*p), reinterpret_cast<cudaStream_t>(stream));
}

FA_API fa_status fa_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                const fa_params* p, fa_stream_t stream) {
  fa_status st = validate(p);
  if (st != FA_OK) return st;
  if (p->Sq == 0) return FA_OK;
  st = check_ptrs({O, LSE, Q});
  if (st != FA_OK) return st;
  if (p->Sk > 0) {
    st = check_ptrs({K, V});
    if (st != FA_OK) return st;
  }
  return launch_fwd_noalloc(Q, K, V, O, LSE, normalized(*p), reinterpret_cast<cudaStream_t>(stream));
}

namespace {
fa_status bwd_entry(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                    const float* LSE, void* dQ, void* dK, void* dV, const fa_params* p,
                    fa_stream_t stream, bool dsmat) {
  fa_status st = validate(p);
  if (st != FA_OK) return st;
  if (p->Sq > 0) {
    st = check_ptrs({Q, O, dO, LSE, dQ});
    if (st != FA_OK) return st;
  }
  if (p->Sk > 0) {
    st = check_ptrs({K, V, dK, dV});
    if (st != FA_OK) return st;
  }
  if (p->Sq == 0 && p->Sk == 0) return FA_OK;
  if (dsmat && p->in_dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  return launch_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, normalized(*p),
                    reinterpret_cast<cudaStream_t>(stream), dsmat);
}
}  // namespace

FA_API fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                        const fa_params* p, fa_stream_t stream) {
  return bwd_entry(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream, false);
}

FA_API fa_status fa_bwd_dsmat(const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                              const fa_params* p, fa_stream_t stream) {
  return bwd_entry(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream, true);
}

FA_API fa_status fa_device_status(fa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  cudaError_t e1 = cudaSuccess, e2 = cudaSuccess;
  const unsigned int v = read_and_clear_fwd_status(&e1) | read_and_clear_bwd_status(&e2);
  if (e1 != cudaSuccess || e2 != cudaSuccess) return FA_ERR_CUDA;
  if (v & DEV_LAYOUT) return FA_ERR_LAYOUT;
  return (v & DEV_TIMEOUT) ? FA_ERR_TIMEOUT : FA_OK;
}

FA_API const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "kernel barrier wait timed out";
    case FA_ERR_SCRATCH_LIMIT: return "problem needs more than the static scratch of fa_fwd_noalloc";
    case FA_ERR_LAYOUT: return "kernel shared-memory layout did not fit its allocation";
  }
  return "unknown status";
}

FA_API const char* fa_version(void) { return "fa-sm103a 0.1"; }

FA_API unsigned long long fa_noalloc_scratch_bytes(void) { return FA_NOALLOC_SCRATCH_BYTES; }

FA_API fa_status fa_selftest_timeout(unsigned long long limit_ns, int* roles_done,
                                     fa_stream_t stream) {
  if (!roles_done || limit_ns == 0 || limit_ns > 10000000000ull) return FA_ERR_INVALID_ARG;
  if (!aligned16(roles_done)) return FA_ERR_ALIGNMENT;
  return launch_selftest_timeout(limit_ns, roles_done, reinterpret_cast<cudaStream_t>(stream));
}

FA_API fa_status fa_timing_enable(int on) {
  using namespace fa::host;
  std::lock_guard<std::mutex> lk(g_t_mu);
  for (auto& p : g_t_pending) {
    cudaEventSynchronize(p.b);
    g_t_free.push_back(p.a);
    g_t_free.push_back(p.b);
  }
  g_t_pending.clear();
  g_t_on = on != 0;
  return FA_OK;
}

FA_API int fa_timing_read(fa_kernel_time* out, int max_entries) {
  using namespace fa::host;
  std::lock_guard<std::mutex> lk(g_t_mu);
  std::vector<fa_kernel_time> agg;
  bool fail = false;
  for (auto& p : g_t_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess)
      fail = true;
    size_t k = 0;
    while (k < agg.size() && std::strcmp(agg[k].name, p.name) != 0) ++k;
    if (k == agg.size()) agg.push_back({p.name, 0, 0.0});
    agg[k].launches += 1;
    agg[k].total_ms += ms;
    g_t_free.push_back(p.a);
    g_t_free.push_back(p.b);
  }
  g_t_pending.clear();
  if (fail) return -1;
  for (size_t k = 0; k < agg.size() && (int)k < max_entries; ++k)
    if (out) out[k] = agg[k];
  return (int)agg.size();
}

}  // extern "C"
