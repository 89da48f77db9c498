// fa_bwd.cu -- backward attention on sm_103a (tcgen05 / TMEM / TMA).
//
// Follows forge "flash_attention.metal", backward section: D_i = dO_i . O_i is
// computed first (the FA2 identity, attention_bwd_d_f32 on that page); P is
// recomputed from the stored row statistic L ("recomputed, never stored");
// dS = P (dP - D); dQ = scale dS K; dK = scale dS^T Q; dV = P^T dO. As there, dK
// and dV are accumulated privately per key row, over all query heads of the kv
// group, without atomics (deterministic); dQ is accumulated per query row.
//
// Kernels:
//   preprocess   one warp per query row: D_i, the log2-domain LSE (+inf for rows
//                that saw no key, so their P is exactly 0), fp16 copies of Q, dO.
//   dkdv         one CTA per (batch, kv head, 128-key tile). It walks 64-query
//                chunks of every grouped query head that can see the tile:
//                S^T = K Q^T and dP^T = V dO^T into a double-buffered TMEM slot,
//                softmax warps turn them into P^T and dS^T (fp16, back into TMEM),
//                then dV += P^T dO and dK += dS^T Q accumulate in TMEM.
//   dq           one CTA per (batch, head, 128-query tile), 64-key chunks:
//                S = Q K^T, dP = dO V^T, dS = P (dP - D), dQ += dS K.
// While the softmax warps work on chunk c, the tensor core computes chunk c+1.
#include <cfloat>
#include <climits>
#include "fa_common.cuh"
#include "ptx.cuh"
#include "fa_prepass.cuh"

namespace fa {
using namespace ptx;

static __device__ unsigned int g_bwd_status = 0;

struct BwdArgs {
  void* dQ;
  void* dK;
  void* dV;
  const float* lse2;   // [B*H][ldq]: LSE * log2(e); +inf for empty rows and padding
  const float* delta;  // [B*H][ldq]: rowsum(dO * O); 0 for padding
  int H, HKV, Sq, Sk, ldq;
  float scale, scale_log2;
  int causal, window, out_bf16;
  int n_tiles;  // key tiles (dkdv) / query tiles (dq) per head
  int BHx;      // B*HKV (dkdv) / B*H (dq)
  int lpt;
  unsigned long long limit_ns;
};

template <int D_>
struct BwdCfg {
  static constexpr int D = D_;
  static constexpr int CH = 64;                        // rows per streamed chunk
  static constexpr int NCB = D / 64;                   // 128-byte column blocks (fp16)
  static constexpr uint32_t BIG_CB = 128u * 128u;      // column block of a 128-row tile
  static constexpr uint32_t SMALL_CB = 64u * 128u;     // column block of a 64-row chunk
  static constexpr uint32_t BIG_TILE = NCB * BIG_CB;
  static constexpr uint32_t SMALL_TILE = NCB * SMALL_CB;
  static constexpr int NST = 4;                        // chunk ring depth
  // dkdv smem: K | V | NST x (Q chunk, dO chunk) | NST x (lse2[64], delta[64])
  static constexpr uint32_t KV_CH_OFF = 2 * BIG_TILE;
  static constexpr uint32_t KV_VEC_OFF = KV_CH_OFF + NST * 2 * SMALL_TILE;
  static constexpr uint32_t KV_SMEM = KV_VEC_OFF + NST * 512 + 1024;
  // dq smem: Q | dO | NST x (K chunk, V chunk)
  static constexpr uint32_t Q_CH_OFF = 2 * BIG_TILE;
  static constexpr uint32_t Q_SMEM = Q_CH_OFF + NST * 2 * SMALL_TILE + 1024;
  static constexpr int THREADS = 192;  // 4 softmax warps, MMA warp, TMA warp
  static constexpr int MMA_WARP = 4, TMA_WARP = 5;
  static constexpr uint32_t TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t s_col(int b) { return 128u * b; }
  __host__ __device__ static constexpr uint32_t dp_col(int b) { return 128u * b + 64u; }
  static constexpr uint32_t ACC0 = 256;  // dV (dkdv) / dQ (dq)
  static constexpr uint32_t ACC1 = 256 + D;  // dK (dkdv)
  static_assert(KV_SMEM <= 227u * 1024u && Q_SMEM <= 227u * 1024u, "shared memory budget");
};

// S (+)= A[128 x D] * B[64 x D]^T, both K-major fp16 in 128B-swizzled smem.
template <class C>
__device__ __forceinline__ void issue_rowdot(uint32_t d_tmem, uint32_t sa, uint32_t sb) {
  constexpr uint32_t id = make_idesc(128, 64, FMT_F16, FMT_F16, false, false);
#pragma unroll
  for (int kk = 0; kk < C::D / 16; ++kk) {
    const uint32_t cb = kk * 16 / 64, in = (kk * 16 % 64) * 2;
    mma_f16_ss(d_tmem, make_sdesc(sa + cb * C::BIG_CB + in, 16, SW128_ATOM),
               make_sdesc(sb + cb * C::SMALL_CB + in, 16, SW128_ATOM), id, kk > 0);
  }
}

// ACC[128 x D] (+)= A(TMEM, fp16, 128 x 64) * B[64 x D] (smem, MN-major fp16 chunk).
template <class C>
__device__ __forceinline__ void issue_acc(uint32_t acc_tmem, uint32_t a_tmem, uint32_t sb,
                                          bool accumulate) {
  constexpr uint32_t id = make_idesc(128, C::D, FMT_F16, FMT_F16, false, true);
#pragma unroll
  for (int kk = 0; kk < C::CH / 16; ++kk)
    mma_f16_ts(acc_tmem, a_tmem + kk * 8, make_sdesc(sb + kk * 16 * 128, C::SMALL_CB, SW128_ATOM),
               id, (accumulate || kk > 0) ? 1u : 0u);
}

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit) return false;
  }
  return true;
}

// Store 32 consecutive fp32 values of one row (fp32 or bf16 destination).
__device__ __forceinline__ void store_row32(void* base, size_t elem_off, const uint32_t (&r)[32],
                                            float mul, int out_bf16) {
  if (!out_bf16) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + elem_off);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      dst[k] = make_float4(__uint_as_float(r[4 * k]) * mul, __uint_as_float(r[4 * k + 1]) * mul,
                           __uint_as_float(r[4 * k + 2]) * mul, __uint_as_float(r[4 * k + 3]) * mul);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + elem_off);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(r[8 * k + 2 * e]) * mul,
                                                  __uint_as_float(r[8 * k + 2 * e + 1]) * mul);
        w[e] = *reinterpret_cast<uint32_t*>(&v2);
      }
      dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// ------------------------------------------------------------------ dK / dV
template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmQc, const __grid_constant__ CUtensorMap tmdOc,
                       const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmDl,
                       const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_kv, bar_full[C::NST], bar_empty[C::NST], bar_sp[2],
      bar_ds[2], bar_done, bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = warp_id(), lane = lane_id();
  volatile int* abort_flag = &abort_sh;

  // Key tile 0 is seen by the most queries under a causal mask: schedule it first.
  const int jt = blockIdx.x / a.BHx;
  const int bg = blockIdx.x % a.BHx;
  const int b = bg / a.HKV, g = bg % a.HKV;
  const int rep = a.H / a.HKV;
  const int j0 = jt * BLOCK_N;
  int qc_lo, qc_hi;
  {
    int imin = a.causal ? j0 : 0;
    int imax = a.Sq - 1;
    if (a.window > 0) {
      const long long lim = (long long)j0 + BLOCK_N - 1 + a.window - 1;
      if (lim < imax) imax = (int)lim;
    }
    if (imax < imin) { qc_lo = 0; qc_hi = 0; }
    else { qc_lo = imin / C::CH; qc_hi = imax / C::CH + 1; }
  }
  const int ncq = qc_hi - qc_lo;
  const int nc = rep * ncq;

  if (threadIdx.x == 0) {
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < C::NST; ++s) { mbar_init(&bar_full[s], 1); mbar_init(&bar_empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&bar_sp[s], 1); mbar_init(&bar_ds[s], 128); }
    mbar_init(&bar_done, 1);
    mbar_init(&bar_drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) {
    __syncwarp();
    tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase, sV = sbase + C::BIG_TILE;
  auto sQc = [&](int st) { return sbase + C::KV_CH_OFF + st * 2 * C::SMALL_TILE; };
  auto sdOc = [&](int st) { return sbase + C::KV_CH_OFF + st * 2 * C::SMALL_TILE + C::SMALL_TILE; };
  float* vecs = reinterpret_cast<float*>(smem + C::KV_VEC_OFF);  // [NST][2][64]
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };
  auto chunk_rows = [&](int c, int* bh, int* i0) {
    const int r = c / ncq, qc = qc_lo + c % ncq;
    *bh = b * a.H + g * rep + r;
    *i0 = qc * C::CH;
  };

  if (warp == C::TMA_WARP) {
    if (lane == 0 && nc > 0) {
      tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmQc); tma_prefetch_desc(&tmdOc);
      mbar_arrive_expect_tx(&bar_kv, 2 * C::BIG_TILE);
      for (int cb = 0; cb < C::NCB; ++cb) {
        tma_load_3d(smem + cb * C::BIG_CB, &tmK, &bar_kv, cb * 64, j0, bg);
        tma_load_3d(smem + C::BIG_TILE + cb * C::BIG_CB, &tmV, &bar_kv, cb * 64, j0, bg);
      }
      int last[C::NST];
      for (int s = 0; s < C::NST; ++s) last[s] = -1;
      for (int c = 0; c < nc; ++c) {
        const int st = c % C::NST;
        if (!wait(&bar_empty[st], ((c / C::NST) & 1) ^ 1)) break;
        int bh, i0;
        chunk_rows(c, &bh, &i0);
        mbar_arrive_expect_tx(&bar_full[st], 2 * C::SMALL_TILE + 512);
        for (int cb = 0; cb < C::NCB; ++cb) {
          tma_load_3d(smem + (sQc(st) - sbase) + cb * C::SMALL_CB, &tmQc, &bar_full[st], cb * 64, i0, bh);
          tma_load_3d(smem + (sdOc(st) - sbase) + cb * C::SMALL_CB, &tmdOc, &bar_full[st], cb * 64, i0, bh);
        }
        tma_load_3d(vecs + st * 128, &tmL, &bar_full[st], i0, bh, 0);
        tma_load_3d(vecs + st * 128 + 64, &tmDl, &bar_full[st], i0, bh, 0);
        last[st] = c / C::NST;
      }
      drain_wait(&bar_kv, 0, a.limit_ns);
      for (int s = 0; s < C::NST; ++s)
        if (last[s] >= 0) drain_wait(&bar_full[s], last[s] & 1, a.limit_ns);
    }
  } else if (warp == C::MMA_WARP) {
    if (lane == 0 && nc > 0) {
      bool ok = wait(&bar_kv, 0);
      tc_fence_after();
      for (int c = 0; ok && c <= nc; ++c) {
        if (c < nc) {
          const int st = c % C::NST, bb = c & 1;
          if (!(ok = wait(&bar_full[st], (c / C::NST) & 1))) break;
          tc_fence_after();
          issue_rowdot<C>(tmem + C::s_col(bb), sK, sQc(st));    // S^T  = K Q^T
          issue_rowdot<C>(tmem + C::dp_col(bb), sV, sdOc(st));  // dP^T = V dO^T
          tc_commit(&bar_sp[bb]);
        }
        if (c >= 1) {
          const int pc = c - 1, pb = pc & 1, pst = pc % C::NST;
          if (!(ok = wait(&bar_ds[pb], (pc >> 1) & 1))) break;
          tc_fence_after();
          issue_acc<C>(tmem + C::ACC0, tmem + C::s_col(pb), sdOc(pst), pc > 0);  // dV += P^T dO
          issue_acc<C>(tmem + C::ACC1, tmem + C::dp_col(pb), sQc(pst), pc > 0); // dK += dS^T Q
          tc_commit(&bar_empty[pst]);
        }
      }
      if (ok) tc_commit(&bar_done);
      tc_commit(&bar_drain);
      drain_wait(&bar_drain, 0, a.limit_ns);
    }
  } else {
    // softmax warps: thread = one key row j = one TMEM lane
    const int wq = warp;  // 0..3
    const int r_in = wq * 32 + lane;
    const int j = j0 + r_in;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int c = 0; c < nc; ++c) {
      const int bb = c & 1, st = c % C::NST;
      int bh, i0;
      chunk_rows(c, &bh, &i0);
      ok = __all_sync(0xffffffffu, wait(&bar_sp[bb], (c >> 1) & 1) && wait(&bar_full[st], (c / C::NST) & 1));
      if (!ok) break;
      tc_fence_after();
      float s[64], dp[64];
      {
        uint32_t r[32];
        tmem_ld32(lane_addr + C::s_col(bb), r);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = __uint_as_float(r[k]);
        tmem_ld32(lane_addr + C::s_col(bb) + 32, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[32 + k] = __uint_as_float(r[k]);
        tmem_ld32(lane_addr + C::dp_col(bb), r);
#pragma unroll
        for (int k = 0; k < 32; ++k) dp[k] = __uint_as_float(r[k]);
        tmem_ld32(lane_addr + C::dp_col(bb) + 32, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) dp[32 + k] = __uint_as_float(r[k]);
      }
      // queries i = i0 + k; key j visible iff (!causal || j <= i) && (!window || j >= i-w+1)
      // && j < Sk && i < Sq
      if (tile_needs_mask(i0, i0 + C::CH - 1, j0, j0 + BLOCK_N - 1, a.Sk, a.causal, a.window) ||
          i0 + C::CH > a.Sq) {
        const int k_lo = a.causal ? j - i0 : INT_MIN / 2;                          // i >= j
        const int k_hi = min(a.window > 0 ? j + a.window - 1 - i0 : INT_MAX / 2,   // i <= j+w-1
                             a.Sq - 1 - i0);
        const bool row_dead = j >= a.Sk;
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (row_dead || k < k_lo || k > k_hi) s[k] = -INFINITY;
      }
      const float* lv = vecs + st * 128;
      uint32_t pk[32], dk[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float p0 = ex2(fmaf(s[2 * k], sl2, -lv[2 * k]));
        const float p1 = ex2(fmaf(s[2 * k + 1], sl2, -lv[2 * k + 1]));
        const float d0 = p0 * (dp[2 * k] - lv[64 + 2 * k]);
        const float d1 = p1 * (dp[2 * k + 1] - lv[64 + 2 * k + 1]);
        pk[k] = pack_half2(p0, p1);
        dk[k] = pack_half2(d0, d1);
      }
      tmem_st32(lane_addr + C::s_col(bb), pk);
      tmem_st32(lane_addr + C::dp_col(bb), dk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_ds[bb]);
    }
    if (ok && nc > 0) {
      ok = __all_sync(0xffffffffu, wait(&bar_done, 0));
      tc_fence_after();
    }
    if (ok) {
      const bool valid = j < a.Sk;
      const size_t row = (size_t)bg * a.Sk + (size_t)(valid ? j : 0);
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        void* dst = which == 0 ? a.dV : a.dK;
        const float mul = which == 0 ? 1.f : a.scale;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t r[32];
          if (nc > 0) {
            tmem_ld32(lane_addr + (which == 0 ? C::ACC0 : C::ACC1) + cc * 32, r);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = 0u;
          }
          if (valid) store_row32(dst, row * D + cc * 32, r, mul, a.out_bf16);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ----------------------------------------------------------------------- dQ
template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmKc, const __grid_constant__ CUtensorMap tmVc,
                     const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_q, bar_full[C::NST], bar_empty[C::NST], bar_sp[2], bar_ds[2],
      bar_done, bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = warp_id(), lane = lane_id();
  volatile int* abort_flag = &abort_sh;

  const int qt_lin = blockIdx.x / a.BHx;
  const int bh = blockIdx.x % a.BHx;
  const int qt = a.lpt ? (a.n_tiles - 1 - qt_lin) : qt_lin;
  const int b = bh / a.H, h = bh % a.H;
  const int bg = b * a.HKV + h / (a.H / a.HKV);
  const int i0 = qt * BLOCK_M;
  int kc_lo, kc_hi;
  {
    int jmax = a.Sk - 1;
    const int r1 = min(i0 + BLOCK_M - 1, a.Sq - 1);
    if (a.causal && r1 < jmax) jmax = r1;
    int jmin = 0;
    if (a.window > 0 && i0 - a.window + 1 > 0) jmin = i0 - a.window + 1;
    if (jmax < jmin) { kc_lo = 0; kc_hi = 0; }
    else { kc_lo = jmin / C::CH; kc_hi = jmax / C::CH + 1; }
  }
  const int nc = kc_hi - kc_lo;

  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < C::NST; ++s) { mbar_init(&bar_full[s], 1); mbar_init(&bar_empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&bar_sp[s], 1); mbar_init(&bar_ds[s], 128); }
    mbar_init(&bar_done, 1);
    mbar_init(&bar_drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) {
    __syncwarp();
    tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase, sdO = sbase + C::BIG_TILE;
  auto sKc = [&](int st) { return sbase + C::Q_CH_OFF + st * 2 * C::SMALL_TILE; };
  auto sVc = [&](int st) { return sbase + C::Q_CH_OFF + st * 2 * C::SMALL_TILE + C::SMALL_TILE; };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };

  if (warp == C::TMA_WARP) {
    if (lane == 0 && nc > 0) {
      tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmKc); tma_prefetch_desc(&tmVc);
      mbar_arrive_expect_tx(&bar_q, 2 * C::BIG_TILE);
      for (int cb = 0; cb < C::NCB; ++cb) {
        tma_load_3d(smem + cb * C::BIG_CB, &tmQ, &bar_q, cb * 64, i0, bh);
        tma_load_3d(smem + C::BIG_TILE + cb * C::BIG_CB, &tmdO, &bar_q, cb * 64, i0, bh);
      }
      int last[C::NST];
      for (int s = 0; s < C::NST; ++s) last[s] = -1;
      for (int c = 0; c < nc; ++c) {
        const int st = c % C::NST;
        if (!wait(&bar_empty[st], ((c / C::NST) & 1) ^ 1)) break;
        const int k0 = (kc_lo + c) * C::CH;
        mbar_arrive_expect_tx(&bar_full[st], 2 * C::SMALL_TILE);
        for (int cb = 0; cb < C::NCB; ++cb) {
          tma_load_3d(smem + (sKc(st) - sbase) + cb * C::SMALL_CB, &tmKc, &bar_full[st], cb * 64, k0, bg);
          tma_load_3d(smem + (sVc(st) - sbase) + cb * C::SMALL_CB, &tmVc, &bar_full[st], cb * 64, k0, bg);
        }
        last[st] = c / C::NST;
      }
      drain_wait(&bar_q, 0, a.limit_ns);
      for (int s = 0; s < C::NST; ++s)
        if (last[s] >= 0) drain_wait(&bar_full[s], last[s] & 1, a.limit_ns);
    }
  } else if (warp == C::MMA_WARP) {
    if (lane == 0 && nc > 0) {
      bool ok = wait(&bar_q, 0);
      tc_fence_after();
      for (int c = 0; ok && c <= nc; ++c) {
        if (c < nc) {
          const int st = c % C::NST, bb = c & 1;
          if (!(ok = wait(&bar_full[st], (c / C::NST) & 1))) break;
          tc_fence_after();
          issue_rowdot<C>(tmem + C::s_col(bb), sQ, sKc(st));    // S  = Q K^T
          issue_rowdot<C>(tmem + C::dp_col(bb), sdO, sVc(st));  // dP = dO V^T
          tc_commit(&bar_sp[bb]);
        }
        if (c >= 1) {
          const int pc = c - 1, pb = pc & 1, pst = pc % C::NST;
          if (!(ok = wait(&bar_ds[pb], (pc >> 1) & 1))) break;
          tc_fence_after();
          issue_acc<C>(tmem + C::ACC0, tmem + C::dp_col(pb), sKc(pst), pc > 0);  // dQ += dS K
          tc_commit(&bar_empty[pst]);
        }
      }
      if (ok) tc_commit(&bar_done);
      tc_commit(&bar_drain);
      drain_wait(&bar_drain, 0, a.limit_ns);
    }
  } else {
    const int wq = warp;
    const int r_in = wq * 32 + lane;
    const int i = i0 + r_in;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    const bool row_valid = i < a.Sq;
    const size_t vrow = (size_t)bh * a.ldq + (size_t)(row_valid ? i : 0);
    const float lse2 = row_valid ? a.lse2[vrow] : INFINITY;
    const float dl = row_valid ? a.delta[vrow] : 0.f;
    const int hi_i = a.causal ? min(i, a.Sk - 1) : a.Sk - 1;
    const int lo_i = a.window > 0 ? i - a.window + 1 : INT_MIN / 2;
    bool ok = true;
    for (int c = 0; c < nc; ++c) {
      const int bb = c & 1;
      const int k0 = (kc_lo + c) * C::CH;
      ok = __all_sync(0xffffffffu, wait(&bar_sp[bb], (c >> 1) & 1));
      if (!ok) break;
      tc_fence_after();
      float s[64], dp[64];
      {
        uint32_t r[32];
        tmem_ld32(lane_addr + C::s_col(bb), r);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = __uint_as_float(r[k]);
        tmem_ld32(lane_addr + C::s_col(bb) + 32, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[32 + k] = __uint_as_float(r[k]);
        tmem_ld32(lane_addr + C::dp_col(bb), r);
#pragma unroll
        for (int k = 0; k < 32; ++k) dp[k] = __uint_as_float(r[k]);
        tmem_ld32(lane_addr + C::dp_col(bb) + 32, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) dp[32 + k] = __uint_as_float(r[k]);
      }
      if (tile_needs_mask(i0, i0 + BLOCK_M - 1, k0, k0 + C::CH - 1, a.Sk, a.causal, a.window)) {
        const int rel_hi = hi_i - k0, rel_lo = lo_i - k0;
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (k > rel_hi || k < rel_lo) s[k] = -INFINITY;
      }
      const float nl = -lse2;
      uint32_t dk[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float p0 = ex2(fmaf(s[2 * k], sl2, nl));
        const float p1 = ex2(fmaf(s[2 * k + 1], sl2, nl));
        dk[k] = pack_half2(p0 * (dp[2 * k] - dl), p1 * (dp[2 * k + 1] - dl));
      }
      tmem_st32(lane_addr + C::dp_col(bb), dk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_ds[bb]);
    }
    if (ok && nc > 0) {
      ok = __all_sync(0xffffffffu, wait(&bar_done, 0));
      tc_fence_after();
    }
    if (ok) {
      const size_t row = (size_t)bh * a.Sq + (size_t)(row_valid ? i : 0);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t r[32];
        if (nc > 0) {
          tmem_ld32(lane_addr + C::ACC0 + cc * 32, r);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        if (row_valid) store_row32(a.dQ, row * D + cc * 32, r, a.scale, a.out_bf16);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// -------------------------------------------------------------- preprocess
// One warp per padded query row (bh, i), i < ldq:
//   delta[bh][i] = sum_d dO[i,d] * O[i,d];  lse2[bh][i] = LSE * log2(e) (+inf if -inf);
//   fp16 copies of the dO and Q rows. Rows i >= Sq get lse2 = +inf, delta = 0.
template <int D>
__global__ void bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ dO, const void* __restrict__ O,
                                      const float* __restrict__ LSE, const __nv_bfloat16* __restrict__ Q,
                                      __half* __restrict__ dO16, __half* __restrict__ Q16,
                                      float* __restrict__ lse2, float* __restrict__ delta, int Sq,
                                      int ldq, size_t n_rows_padded, int o_bf16) {
  const size_t warps = (size_t)gridDim.x * (blockDim.x / 32);
  const int lane = threadIdx.x & 31;
  for (size_t w = blockIdx.x * (size_t)(blockDim.x / 32) + threadIdx.x / 32; w < n_rows_padded;
       w += warps) {
    const size_t bh = w / ldq;
    const int i = (int)(w % ldq);
    if (i >= Sq) {
      if (lane == 0) { lse2[w] = INFINITY; delta[w] = 0.f; }
      continue;
    }
    const size_t row = bh * Sq + i;
    float acc = 0.f;
#pragma unroll
    for (int d0 = 0; d0 < D; d0 += 128) {
      const int d = d0 + lane * 4;
      if (d >= D) break;  // D = 64: lanes 16..31 have no columns
      const uint2 g = *reinterpret_cast<const uint2*>(dO + row * D + d);
      const uint2 qv = *reinterpret_cast<const uint2*>(Q + row * D + d);
      float gv[4] = {__uint_as_float(g.x << 16), __uint_as_float(g.x & 0xFFFF0000u),
                     __uint_as_float(g.y << 16), __uint_as_float(g.y & 0xFFFF0000u)};
      float ov[4];
      if (o_bf16) {
        const uint2 o = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(O) + row * D + d);
        ov[0] = __uint_as_float(o.x << 16); ov[1] = __uint_as_float(o.x & 0xFFFF0000u);
        ov[2] = __uint_as_float(o.y << 16); ov[3] = __uint_as_float(o.y & 0xFFFF0000u);
      } else {
        const float4 o = *reinterpret_cast<const float4*>(static_cast<const float*>(O) + row * D + d);
        ov[0] = o.x; ov[1] = o.y; ov[2] = o.z; ov[3] = o.w;
      }
      acc += gv[0] * ov[0] + gv[1] * ov[1] + gv[2] * ov[2] + gv[3] * ov[3];
      uint2 g16, q16;
      g16.x = pack_half2(gv[0], gv[1]);
      g16.y = pack_half2(gv[2], gv[3]);
      q16.x = pack_half2(__uint_as_float(qv.x << 16), __uint_as_float(qv.x & 0xFFFF0000u));
      q16.y = pack_half2(__uint_as_float(qv.y << 16), __uint_as_float(qv.y & 0xFFFF0000u));
      *reinterpret_cast<uint2*>(dO16 + row * D + d) = g16;
      *reinterpret_cast<uint2*>(Q16 + row * D + d) = q16;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const float L = LSE[row];
      lse2[w] = (L == -INFINITY) ? INFINITY : L * LOG2E;
      delta[w] = acc;
    }
  }
}

// Zero-fill outputs of an empty side (Sq == 0 or Sk == 0).
__global__ void zero_kernel(uint4* p, size_t n16) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = make_uint4(0, 0, 0, 0);
}

// ------------------------------------------------------------------ launcher
namespace {

template <int D>
fa_status run_bwd_bf16(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                       const float* LSE, void* dQ, void* dK, void* dV, const fa_params& p,
                       cudaStream_t stream) {
  using C = BwdCfg<D>;
  const size_t BH = (size_t)p.B * p.H, BHk = (size_t)p.B * p.HKV;
  const size_t nq = BH * p.Sq * D, nk = BHk * p.Sk * D;
  const int ldq = (p.Sq + 63) / 64 * 64;
  const size_t nvec = BH * ldq;
  const size_t bytes = (2 * nq + 2 * nk) * 2 + 2 * nvec * 4;
  void* ws = nullptr;
  if (host::scratch_alloc(&ws, bytes, stream) != cudaSuccess) return FA_ERR_CUDA;
  __half* q16 = static_cast<__half*>(ws);
  __half* do16 = q16 + nq;
  __half* k16 = do16 + nq;
  __half* v16 = k16 + nk;
  float* lse2 = reinterpret_cast<float*>(v16 + nk);
  float* delta = lse2 + nvec;
  const int grid_pp = 4 * host::sm_count();
  {
    host::KernelTimer kt("bwd_preprocess", stream);
    bwd_preprocess_kernel<D><<<grid_pp, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(dO), O, LSE, static_cast<const __nv_bfloat16*>(Q), do16,
        q16, lse2, delta, p.Sq, ldq, nvec, p.out_dtype == FA_BF16);
  }
  {
    host::KernelTimer kt("cvt_bf16_to_f16(K,V)", stream);
    cvt_bf16_to_f16_kernel<<<grid_pp, 256, 0, stream>>>(static_cast<const uint4*>(K),
                                                       reinterpret_cast<uint4*>(k16), nk / 8);
    cvt_bf16_to_f16_kernel<<<grid_pp, 256, 0, stream>>>(static_cast<const uint4*>(V),
                                                       reinterpret_cast<uint4*>(v16), nk / 8);
  }
  CUtensorMap mK, mV, mQc, mdOc, mL, mDl, mQ, mdO, mKc, mVc;
  const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const auto F32T = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  bool enc = true;
  enc &= host::encode_tiled_3d(&mK, F16, 2, k16, D, p.Sk, BHk, D, 64, 128);
  enc &= host::encode_tiled_3d(&mV, F16, 2, v16, D, p.Sk, BHk, D, 64, 128);
  enc &= host::encode_tiled_3d(&mKc, F16, 2, k16, D, p.Sk, BHk, D, 64, 64);
  enc &= host::encode_tiled_3d(&mVc, F16, 2, v16, D, p.Sk, BHk, D, 64, 64);
  enc &= host::encode_tiled_3d(&mQ, F16, 2, q16, D, p.Sq, BH, D, 64, 128);
  enc &= host::encode_tiled_3d(&mdO, F16, 2, do16, D, p.Sq, BH, D, 64, 128);
  enc &= host::encode_tiled_3d(&mQc, F16, 2, q16, D, p.Sq, BH, D, 64, 64);
  enc &= host::encode_tiled_3d(&mdOc, F16, 2, do16, D, p.Sq, BH, D, 64, 64);
  enc &= host::encode_tiled_3d(&mL, F32T, 4, lse2, ldq, BH, 1, ldq, 64, 1, false);
  enc &= host::encode_tiled_3d(&mDl, F32T, 4, delta, ldq, BH, 1, ldq, 64, 1, false);
  if (!enc) {
    host::scratch_free(ws, stream);
    return FA_ERR_CUDA;
  }
  BwdArgs a;
  a.dQ = dQ; a.dK = dK; a.dV = dV;
  a.lse2 = lse2; a.delta = delta;
  a.H = p.H; a.HKV = p.HKV; a.Sq = p.Sq; a.Sk = p.Sk; a.ldq = ldq;
  a.scale = p.scale; a.scale_log2 = p.scale * LOG2E;
  a.causal = p.causal; a.window = p.window; a.out_bf16 = p.out_dtype == FA_BF16;
  a.lpt = p.causal;
  a.limit_ns = WAIT_LIMIT_NS;
  cudaError_t e = cudaSuccess;
  if (p.Sk > 0) {
    BwdArgs ak = a;
    ak.n_tiles = (p.Sk + BLOCK_N - 1) / BLOCK_N;
    ak.BHx = (int)BHk;
    auto kern = fa_bwd_dkdv_kernel<D>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::KV_SMEM);
    if (e == cudaSuccess) {
      host::KernelTimer kt(D == 128 ? "fa_bwd_dkdv_kernel<128,bf16>" : "fa_bwd_dkdv_kernel<64,bf16>",
                           stream);
      kern<<<(unsigned)(BHk * ak.n_tiles), C::THREADS, C::KV_SMEM, stream>>>(mK, mV, mQc, mdOc, mL,
                                                                            mDl, ak);
      e = cudaGetLastError();
    }
  }
  if (e == cudaSuccess && p.Sq > 0) {
    BwdArgs aq = a;
    aq.n_tiles = (p.Sq + BLOCK_M - 1) / BLOCK_M;
    aq.BHx = (int)BH;
    auto kern = fa_bwd_dq_kernel<D>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::Q_SMEM);
    if (e == cudaSuccess) {
      host::KernelTimer kt(D == 128 ? "fa_bwd_dq_kernel<128,bf16>" : "fa_bwd_dq_kernel<64,bf16>",
                           stream);
      kern<<<(unsigned)(BH * aq.n_tiles), C::THREADS, C::Q_SMEM, stream>>>(mQ, mdO, mKc, mVc, aq);
      e = cudaGetLastError();
    }
  }
  const cudaError_t e2 = host::scratch_free(ws, stream);
  return (e == cudaSuccess && e2 == cudaSuccess) ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* LSE, void* dQ, void* dK, void* dV, const fa_params& p,
                     cudaStream_t stream) {
  const int grid_pp = 4 * host::sm_count();
  const size_t osz = p.out_dtype == FA_BF16 ? 2 : 4;
  if (p.Sq == 0 || p.Sk == 0) {
    // No query sees any key: every gradient is zero.
    if (p.Sq > 0)
      zero_kernel<<<grid_pp, 256, 0, stream>>>(static_cast<uint4*>(dQ),
                                               (size_t)p.B * p.H * p.Sq * p.D * osz / 16);
    if (p.Sk > 0) {
      const size_t n16 = (size_t)p.B * p.HKV * p.Sk * p.D * osz / 16;
      zero_kernel<<<grid_pp, 256, 0, stream>>>(static_cast<uint4*>(dK), n16);
      zero_kernel<<<grid_pp, 256, 0, stream>>>(static_cast<uint4*>(dV), n16);
    }
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }
  if (p.in_dtype == FA_BF16) {
    if (p.D == 128) return run_bwd_bf16<128>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream);
    if (p.D == 64) return run_bwd_bf16<64>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream);
  }
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
