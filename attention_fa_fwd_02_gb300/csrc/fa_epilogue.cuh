// fa_epilogue.cuh -- writing a 128-row accumulator from TMEM to global memory.
//
// Each of the four epilogue warps owns 32 TMEM lanes = 32 output rows. A thread
// holds one whole row (tcgen05.ld 32x32b), so storing straight from registers
// would make every warp store touch 32 rows / 32 cache lines. Instead each warp
// stages its rows in shared memory as TMA boxes of 32 rows x 128 bytes in the
// 128-byte swizzled layout (16-byte chunk c of row r at chunk position c ^ (r % 8),
// which keeps the shared stores free of bank conflicts) and writes them out with
// tensor stores, which also drop rows past the tensor's end.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include "ptx.cuh"

namespace fa {

constexpr uint32_t EPI_BOX_BYTES = 32u * 128u;  // one box: 32 rows x 128 bytes

// Shared-memory bytes one warp needs to stage all its boxes at once.
template <int D, bool OUT_BF16>
constexpr uint32_t epi_warp_bytes() {
  return (uint32_t)(D * (OUT_BF16 ? 2 : 4) / 128) * EPI_BOX_BYTES;
}

// Rows r_base .. r_base + 31 of slab z: columns [0, D) of the fp32 accumulator at
// TMEM address t_addr (this warp's lane base), times mul, in the output type of
// the tensor map `tm` (fp32, or bf16 when OUT_BF16). `stage` (1024-byte aligned)
// holds BOXES boxes, used as a ring: each box is stored (its own bulk group) as soon
// as it is written, and a slot is refilled once the store that last used it has read
// it, so staging the next box overlaps the copy engine reading the previous ones (the
// reads complete in commit order; waiting until at most BOXES - 1 groups are unread
// frees the oldest slot, counting this thread's earlier groups too). have == false
// writes zeros (no accumulator). any_row == false skips the stores (all rows are
// past the tensor's end). With WAIT, the stores have read their shared-memory
// sources on return (the global writes complete on their own, before the kernel
// does); without, the caller issues bulk_wait_read_all() (lane 0) before the staging
// area is reused or the CTA exits.
// D is the number of columns this call stores: TMEM columns t_addr .. t_addr + D of
// the warp's lanes go to tensor columns x0 .. x0 + D. Boxes that would start at or
// beyond column x_end (the tensor's width, for head dims below the kernel's D) are not
// stored; the TMA store clips a box that crosses it.
template <int D, bool OUT_BF16, int BOXES, bool WAIT = true>
__device__ __forceinline__ void store_rows_tma(const CUtensorMap* tm, uint32_t t_addr, bool have,
                                               float mul, uint32_t stage, int r_base, bool any_row,
                                               int z, int x0 = 0, int x_end = 1 << 30) {
  using namespace ptx;
  constexpr int COLS = OUT_BF16 ? 64 : 32;  // output columns per 128-byte box row
  constexpr int NBOX = D / COLS;
  static_assert(BOXES >= 1 && D % COLS == 0, "epilogue staging");
  const uint32_t lane = lane_id();
  const uint32_t sw = lane & 7u;
#pragma unroll
  for (int b = 0; b < NBOX; ++b) {
    const int slot = b % BOXES;
    if (b >= BOXES) {
      if (lane == 0) bulk_wait_read<BOXES - 1>();
      __syncwarp();
    }
    const uint32_t row = stage + slot * EPI_BOX_BYTES + lane * 128u;
    if constexpr (!OUT_BF16) {
      uint32_t r[32];
      if (have) {
        tmem_ld32(t_addr + b * 32, r);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = 0u;
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(row + ((c ^ sw) << 4), __float_as_uint(__uint_as_float(r[4 * c]) * mul),
                     __float_as_uint(__uint_as_float(r[4 * c + 1]) * mul),
                     __float_as_uint(__uint_as_float(r[4 * c + 2]) * mul),
                     __float_as_uint(__uint_as_float(r[4 * c + 3]) * mul));
    } else {
      uint32_t r0[32], r1[32];
      if (have) {
        tmem_ld32x2(t_addr + b * 64, t_addr + b * 64 + 32, r0, r1);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r0[k] = r1[k] = 0u;
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = (c % 4) * 8 + 2 * e;
          const float x0 = __uint_as_float(c < 4 ? r0[k] : r1[k]) * mul;
          const float x1 = __uint_as_float(c < 4 ? r0[k + 1] : r1[k + 1]) * mul;
          __nv_bfloat162 v2 = __floats2bfloat162_rn(x0, x1);
          w[e] = *reinterpret_cast<uint32_t*>(&v2);
        }
        st_shared_v4(row + ((c ^ sw) << 4), w[0], w[1], w[2], w[3]);
      }
    }
    fence_async_shared();
    __syncwarp();
    if (lane == 0) {
      if (any_row && x0 + b * COLS < x_end)
        tma_store_3d(tm, stage + slot * EPI_BOX_BYTES, x0 + b * COLS, r_base, z);
      bulk_commit_group();  // (an empty group where nothing was stored keeps the count)
    }
  }
  if constexpr (WAIT) {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
  }
}

// The same rows written by the warp itself instead of by tensor stores: each 32 x
// 128-byte box is staged in `stage` (one box, 1024-byte aligned, this warp's alone) in
// the swizzled layout, read back four rows per instruction (thread t: row t / 8, 16-byte
// chunk t % 8) and written with coalesced 16-byte global stores, four whole 128-byte
// lines per instruction. Nothing waits on the copy engine: the box is free again once
// the warp's own shared loads returned. `out` is the [z][rows][x_end] tensor of the
// output type; rows at or past `rows` and columns at or past x_end are not written.
template <int D, bool OUT_BF16>
__device__ __forceinline__ void store_rows_direct(void* out, uint32_t t_addr, bool have, float mul,
                                                  uint32_t stage, int r_base, int rows, int z,
                                                  int x_end) {
  using namespace ptx;
  constexpr int COLS = OUT_BF16 ? 64 : 32;  // output columns per 128-byte box row
  constexpr int NBOX = D / COLS;
  constexpr int ESZ = OUT_BF16 ? 2 : 4;
  const uint32_t lane = lane_id();
  const uint32_t sw = lane & 7u;
  const uint32_t row = stage + lane * 128u;
  const int rr = (int)(lane >> 3), ch = (int)(lane & 7u);  // read-back: row rr + 4 i, chunk ch
#pragma unroll
  for (int b = 0; b < NBOX; ++b) {
    if (b * COLS >= x_end) break;
    if constexpr (!OUT_BF16) {
      uint32_t r[32];
      if (have) {
        tmem_ld32(t_addr + b * 32, r);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = 0u;
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(row + ((c ^ sw) << 4), __float_as_uint(__uint_as_float(r[4 * c]) * mul),
                     __float_as_uint(__uint_as_float(r[4 * c + 1]) * mul),
                     __float_as_uint(__uint_as_float(r[4 * c + 2]) * mul),
                     __float_as_uint(__uint_as_float(r[4 * c + 3]) * mul));
    } else {
      uint32_t r0[32], r1[32];
      if (have) {
        tmem_ld32x2(t_addr + b * 64, t_addr + b * 64 + 32, r0, r1);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r0[k] = r1[k] = 0u;
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = (c % 4) * 8 + 2 * e;
          const float x0 = __uint_as_float(c < 4 ? r0[k] : r1[k]) * mul;
          const float x1 = __uint_as_float(c < 4 ? r0[k + 1] : r1[k + 1]) * mul;
          __nv_bfloat162 v2 = __floats2bfloat162_rn(x0, x1);
          w[e] = *reinterpret_cast<uint32_t*>(&v2);
        }
        st_shared_v4(row + ((c ^ sw) << 4), w[0], w[1], w[2], w[3]);
      }
    }
    __syncwarp();
    const int col = b * COLS + ch * (16 / ESZ);  // first output column of this thread's chunk
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rl = rr + 4 * i;  // row of the box this thread reads
      const float4 v = ld_shared_v4(stage + (uint32_t)rl * 128u + (((uint32_t)ch ^ ((uint32_t)rl & 7u)) << 4));
      const int grow = r_base + rl;
      if (grow < rows && col < x_end) {
        char* dst = static_cast<char*>(out) + (((size_t)z * rows + grow) * x_end + col) * ESZ;
        *reinterpret_cast<float4*>(dst) = v;
      }
    }
    __syncwarp();  // the box is read back: the next one may overwrite it
  }
  // the staging writes ordered before later copy-engine writes into the same stage
  fence_async_shared();
}

}  // namespace fa
