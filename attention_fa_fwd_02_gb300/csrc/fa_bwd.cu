// fa_bwd.cu -- backward attention kernels (placeholder until the kernels land).
#include "fa_common.cuh"

namespace fa {
static __device__ unsigned int g_bwd_status = 0;

fa_status launch_bwd(const void*, const void*, const void*, const void*, const void*, const float*,
                     void*, void*, void*, const fa_params&, cudaStream_t) {
  return FA_ERR_UNSUPPORTED;
}

unsigned int read_and_clear_bwd_status(cudaError_t* err) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_bwd_status, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(zero));
  if (err) *err = e;
  return v;
}
}  // namespace fa
