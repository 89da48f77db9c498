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
//   preprocess   D_i, the log2-domain LSE (+inf for rows that saw no key, so their
//                P is exactly 0) and the tensor-core operand copies: fp16 for bf16
//                inputs; for fp32 inputs two scaled fp16 terms, or tf32 hi / lo
//                splits (plus transposed copies of Q, K, dO, since tf32 operands
//                must be K-major).
//   dkdv         per (batch, kv head, 128-key tile) -- for bf16 inputs a work item
//                of a persistent CTA, for fp32 inputs one CTA. It walks CH-query
//                chunks of every grouped query head that can see the tile:
//                S^T = K Q^T and dP^T = V dO^T into a double-buffered TMEM slot,
//                softmax warps turn them into P^T and dS^T (back into TMEM),
//                then dV += P^T dO and dK += dS^T Q accumulate in TMEM.
//   dq           per (batch, head, 128-query tile) -- for bf16 inputs a work item of
//                a persistent CTA, for fp32 inputs one CTA -- CH-key chunks:
//                S = Q K^T, dP = dO V^T, dS = P (dP - D), dQ += dS K.
// While the softmax warps work on chunk c, the tensor core computes chunk c+1.
// For fp32 inputs every product is the three-term sum a_hi b_hi + a_hi b_lo + a_lo b_hi,
// of fp16 terms (x 2^e = hi + lo) or of tf32 terms (3xTF32).
#include <cfloat>
#include <climits>
#include <algorithm>
#include <vector>
#include <type_traits>
#include "fa_common.cuh"
#include "ptx.cuh"
#include "fa_prepass.cuh"
#include "fa_epilogue.cuh"
#include "fa_decode_bwd.cuh"

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
  int Dv;      // head dim of the tensors (<= the kernel's D; missing columns read as 0)
  int* sched;  // dq (bf16 inputs): work-item counter, zero at launch
  int n_splits;  // dq (bf16 inputs): key ranges per query tile; > 1 writes partial dQ per range
  int tps;       // key tiles per range
  unsigned long long limit_ns;
  // bf16 inputs: multipliers that undo the power-of-two scaling of the fp16 operand
  // copies (written by bwd_scales_kernel before these kernels start)
  const OperandScales* sc;
  // materialised-dS backward: dS^T (scaled by 2^eD, fp16, hi and, with two-term
  // operands, lo) as [B*H][Sk][ldq], query index fastest
  __half* ds_hi;
  __half* ds_lo;
};

// Tensor maps of one kernel launch; index [split] selects the hi (0) / lo (1) copy.
// dK / dV / dQ: the outputs, stored by TMA in boxes of 32 rows x 128 bytes.
struct KVMaps {  // dkdv
  CUtensorMap K[2], V[2], Qc[2], dOc[2], Qt[2], dOt[2], L, Dl, dK, dV;
};
struct QMaps {  // dq
  CUtensorMap Q[2], dO[2], Kc[2], Vc[2], Kt[2], dQ;
};

template <int D_, int PREC>
struct BwdCfg {
  static constexpr int D = D_;
  static constexpr bool F32 = PREC != IN_BF16;
  // fp32 inputs: two scaled fp16 terms per operand (X16, x 2^e = hi + lo, three
  // kind::f16 products per GEMM; 16-bit B operands may be MN-major, so no transposed
  // copies), or 3xTF32 up to D = 64
  static constexpr bool X16 = PREC == IN_F32_X16;
  static constexpr bool TF32 = PREC == IN_F32_TF32;
  static_assert(!TF32 || D <= 64, "3xTF32 tiles up to D = 64");
  static constexpr int ESZ = TF32 ? 4 : 2;
  static constexpr int ROW = 128 / ESZ;                 // elements per 128-byte row
  static constexpr int NCB = D / ROW;                   // 128-byte column blocks per row
  // rows per streamed chunk: 32 where K and V hi / lo (resident) leave room for no more
  static constexpr int CH = (TF32 || (X16 && D > 64)) ? 32 : 64;
  static constexpr int NSPLIT = F32 ? 2 : 1;
  static constexpr uint32_t BIG_CB = 128u * 128u;       // column block of a 128-row tile
  static constexpr uint32_t SMALL_CB = CH * 128u;       // column block of a CH-row chunk
  static constexpr uint32_t BIG_TILE = NCB * BIG_CB;
  static constexpr uint32_t SMALL_TILE = NCB * SMALL_CB;
  static constexpr uint32_t T_TILE = TF32 ? D * 128u : 0u;  // transposed chunk: D rows x 32 fp32
  static constexpr uint32_t VEC_STAGE = 2 * CH * 4;        // lse2 + delta of one chunk
  // dkdv smem: K, V (hi[, lo]) | KV_NST x chunk (Q, dO [, Q^T, dO^T]) | KV_NST x vectors
  static constexpr int KV_NST = TF32 ? 1 : ((X16 && D > 64) ? 2 : 4);
  static constexpr uint32_t KV_RES = 2 * NSPLIT * BIG_TILE;
  static constexpr uint32_t KV_STAGE = NSPLIT * (2 * SMALL_TILE + 2 * T_TILE);
  static constexpr uint32_t KV_VEC_OFF = KV_RES + KV_NST * KV_STAGE;
  static constexpr uint32_t KV_SMEM = KV_VEC_OFF + KV_NST * VEC_STAGE + 1024;
  // dq smem: Q, dO (hi[, lo]) | Q_NST x chunk (K, V [, K^T])
  static constexpr int Q_NST = (TF32 || (X16 && D > 64)) ? 2 : 4;
  static constexpr uint32_t Q_RES = 2 * NSPLIT * BIG_TILE;
  static constexpr uint32_t Q_STAGE = NSPLIT * (2 * SMALL_TILE + T_TILE);
  static constexpr uint32_t Q_SMEM = Q_RES + Q_NST * Q_STAGE + 1024;
  // 4 softmax warps; a score-MMA issuer (also owns TMEM), an accumulate-MMA issuer,
  // the TMA producer and an idle warp. Separate issuers: after a burst of MMAs a
  // warp's next barrier operation waits for that burst, so one issuer alternating
  // score and accumulate bursts lets the tensor pipe drain at every switch.
  static constexpr int THREADS = 256;
  static constexpr int MMA_WARP = 4, ACC_WARP = 5, TMA_WARP = 6;
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM slots: S | dP | P_lo | dS_lo, CH columns each (3xTF32: fp32 P / dS hi
  // overwrite S / dP), or S | dP (X16: fp16 P / dS hi in the first CH/2 columns of
  // S / dP, lo in the other CH/2), CH columns each. A ring of slots
  // lets the tensor core score chunk c+1.. while the softmax works on chunk c:
  // dkdv has room for two slots next to its dV and dK accumulators, dq for three.
  static constexpr int KV_NSLOT = 2, Q_NSLOT = 3;
  __host__ __device__ static constexpr uint32_t s_col(int b) { return 128u * b; }
  __host__ __device__ static constexpr uint32_t dp_col(int b) { return 128u * b + CH; }
  __host__ __device__ static constexpr uint32_t plo_col(int b) {
    return X16 ? 128u * b + CH / 2 : 128u * b + 2 * CH;
  }
  __host__ __device__ static constexpr uint32_t dslo_col(int b) {
    return X16 ? 128u * b + CH + CH / 2 : 128u * b + 3 * CH;
  }
  static constexpr uint32_t KV_ACC0 = 128 * KV_NSLOT;      // dV (dkdv)
  static constexpr uint32_t KV_ACC1 = 128 * KV_NSLOT + D;  // dK (dkdv)
  static constexpr uint32_t Q_ACC = 128 * Q_NSLOT;         // dQ (dq)
  // (bf16 inputs use the Dkv16Cfg / Dq16Cfg kernels; these layouts are the fp32 kernels')
  static_assert(!F32 || (KV_SMEM <= 227u * 1024u && Q_SMEM <= 227u * 1024u), "shared memory budget");
  static_assert((TF32 ? 4 * CH : 2 * CH) <= 128, "TMEM slot width");
  static_assert(KV_ACC1 + D <= TMEM_COLS && Q_ACC + D <= TMEM_COLS, "TMEM budget");
  // Epilogues stage each warp's rows from the start of shared memory (every operand
  // buffer is spent by then): dV and dK side by side (dkdv), dQ (dq).
  static constexpr uint32_t EPI_WARP = epi_warp_bytes<D, false>();
  static_assert(!F32 || (4 * 2 * EPI_WARP <= KV_VEC_OFF && 4 * EPI_WARP <= Q_RES + Q_NST * Q_STAGE),
                "epilogue staging");
};

// S (+)= A[128 x D] * B[CH x D]^T, both K-major in 128B-swizzled smem.
template <class C>
__device__ __forceinline__ void issue_rowdot(uint32_t d, uint32_t a, uint32_t a_lo, uint32_t b,
                                             uint32_t b_lo) {
  if constexpr (!C::F32) {
    constexpr uint32_t id = make_idesc(128, C::CH, FMT_F16, FMT_F16, false, false);
#pragma unroll
    for (int kk = 0; kk < C::D / 16; ++kk) {
      const uint32_t cb = kk * 16 / 64, in = (kk * 16 % 64) * 2;
      mma_f16_ss(d, make_sdesc(a + cb * C::BIG_CB + in, 16, SW128_ATOM),
                 make_sdesc(b + cb * C::SMALL_CB + in, 16, SW128_ATOM), id, kk > 0);
    }
  } else if constexpr (C::X16) {
    constexpr uint32_t id = make_idesc(128, C::CH, FMT_F16, FMT_F16, false, false);
#pragma unroll
    for (int kk = 0; kk < C::D / 16; ++kk) {
      const uint32_t cb = kk * 16 / 64, in = (kk * 16 % 64) * 2;
      const uint64_t ah = make_sdesc(a + cb * C::BIG_CB + in, 16, SW128_ATOM);
      const uint64_t al = make_sdesc(a_lo + cb * C::BIG_CB + in, 16, SW128_ATOM);
      const uint64_t bh = make_sdesc(b + cb * C::SMALL_CB + in, 16, SW128_ATOM);
      const uint64_t bl = make_sdesc(b_lo + cb * C::SMALL_CB + in, 16, SW128_ATOM);
      mma_f16_ss(d, ah, bh, id, kk > 0);
      mma_f16_ss(d, ah, bl, id, 1);
      mma_f16_ss(d, al, bh, id, 1);
    }
  } else {
    constexpr uint32_t id = make_idesc(128, C::CH, FMT_TF32, FMT_TF32, false, false);
#pragma unroll
    for (int kk = 0; kk < C::D / 8; ++kk) {
      const uint32_t cb = kk * 8 / 32, in = (kk * 8 % 32) * 4;
      const uint64_t ah = make_sdesc(a + cb * C::BIG_CB + in, 16, SW128_ATOM);
      const uint64_t al = make_sdesc(a_lo + cb * C::BIG_CB + in, 16, SW128_ATOM);
      const uint64_t bh = make_sdesc(b + cb * C::SMALL_CB + in, 16, SW128_ATOM);
      const uint64_t bl = make_sdesc(b_lo + cb * C::SMALL_CB + in, 16, SW128_ATOM);
      mma_tf32_ss(d, ah, bh, id, kk > 0);
      mma_tf32_ss(d, ah, bl, id, 1);
      mma_tf32_ss(d, al, bh, id, 1);
    }
  }
}

// ACC[128 x D] (+)= A(TMEM, 128 x CH) * B[CH x D]. fp16: B is the MN-major chunk
// [CH rows][D]; tf32: B is the K-major transposed chunk [D rows][CH].
template <class C>
__device__ __forceinline__ void issue_acc(uint32_t acc, uint32_t a_tmem, uint32_t alo_tmem,
                                          uint32_t b, uint32_t b_lo, bool accumulate) {
  if constexpr (!C::F32) {
    constexpr uint32_t id = make_idesc(128, C::D, FMT_F16, FMT_F16, false, true);
#pragma unroll
    for (int kk = 0; kk < C::CH / 16; ++kk)
      mma_f16_ts(acc, a_tmem + kk * 8, make_sdesc(b + kk * 16 * 128, C::SMALL_CB, SW128_ATOM), id,
                 (accumulate || kk > 0) ? 1u : 0u);
  } else if constexpr (C::X16) {
    // A hi / lo: packed fp16 in TMEM (8 columns per 16 rows); B hi / lo: the MN-major chunk
    constexpr uint32_t id = make_idesc(128, C::D, FMT_F16, FMT_F16, false, true);
#pragma unroll
    for (int kk = 0; kk < C::CH / 16; ++kk) {
      const uint64_t bh = make_sdesc(b + kk * 16 * 128, C::SMALL_CB, SW128_ATOM);
      const uint64_t bl = make_sdesc(b_lo + kk * 16 * 128, C::SMALL_CB, SW128_ATOM);
      mma_f16_ts(acc, a_tmem + kk * 8, bh, id, (accumulate || kk > 0) ? 1u : 0u);
      mma_f16_ts(acc, a_tmem + kk * 8, bl, id, 1u);
      mma_f16_ts(acc, alo_tmem + kk * 8, bh, id, 1u);
    }
  } else {
    constexpr uint32_t id = make_idesc(128, C::D, FMT_TF32, FMT_TF32, false, false);
#pragma unroll
    for (int kk = 0; kk < C::CH / 8; ++kk) {
      const uint32_t in = (kk * 8 % 32) * 4;
      const uint64_t bh = make_sdesc(b + in, 16, SW128_ATOM);
      const uint64_t bl = make_sdesc(b_lo + in, 16, SW128_ATOM);
      mma_tf32_ts(acc, a_tmem + kk * 8, bh, id, (accumulate || kk > 0) ? 1u : 0u);
      mma_tf32_ts(acc, a_tmem + kk * 8, bl, id, 1);
      mma_tf32_ts(acc, alo_tmem + kk * 8, bh, id, 1);
    }
  }
}

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit) return false;
  }
  return true;
}

// Load CH fp32 columns at `sa` and CH at `da` of this thread's TMEM lane, with a
// single wait for all of them.
template <int CH>
__device__ __forceinline__ void tmem_ld_pair(uint32_t sa, uint32_t da, float (&x)[CH],
                                             float (&y)[CH]) {
  static_assert(CH == 32 || CH == 64, "chunk width");
  if constexpr (CH == 64) {
    uint32_t r0[32], r1[32], r2[32], r3[32];
    tmem_ld32x4(sa, sa + 32, da, da + 32, r0, r1, r2, r3);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      x[k] = __uint_as_float(r0[k]);
      x[32 + k] = __uint_as_float(r1[k]);
      y[k] = __uint_as_float(r2[k]);
      y[32 + k] = __uint_as_float(r3[k]);
    }
  } else {
    uint32_t r0[32], r1[32];
    tmem_ld32x2(sa, da, r0, r1);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      x[k] = __uint_as_float(r0[k]);
      y[k] = __uint_as_float(r1[k]);
    }
  }
}

// Write probabilities / score gradients back into TMEM as the A operand of the
// accumulating MMAs: fp16 pairs into the first CH/2 columns at `hi`, or tf32
// hi (at `hi`) and lo (at `lo`) parts, one column each.
template <class C>
__device__ __forceinline__ void tmem_st_operand(uint32_t hi, uint32_t lo, const float (&x)[C::CH]) {
  if constexpr (C::X16) {
    // fp16 pairs: hi = fp16(x) into CH / 2 columns at `hi`, lo = fp16(x - hi) at `lo`
    static_assert(C::CH % 32 == 0, "16 packed columns per store");
#pragma unroll
    for (int c = 0; c < C::CH / 32; ++c) {
      uint32_t ph[16], pl[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float x0 = x[c * 32 + 2 * k], x1 = x[c * 32 + 2 * k + 1];
        const __half2 h = __floats2half2_rn(x0, x1);
        const float2 hf = __half22float2(h);
        ph[k] = *reinterpret_cast<const uint32_t*>(&h);
        pl[k] = pack_half2(x0 - hf.x, x1 - hf.y);
      }
      tmem_st16(hi + c * 16, ph);
      tmem_st16(lo + c * 16, pl);
    }
  } else if constexpr (!C::F32) {
#pragma unroll
    for (int c = 0; c < C::CH / 64; ++c) {
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) pk[k] = pack_half2(x[c * 64 + 2 * k], x[c * 64 + 2 * k + 1]);
      tmem_st32(hi + c * 32, pk);
    }
  } else {
#pragma unroll
    for (int c = 0; c < C::CH / 32; ++c) {
      uint32_t ph[32], pl[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float v = x[c * 32 + k];
        const uint32_t hb = __float_as_uint(v) & 0xFFFFE000u;
        ph[k] = hb;
        pl[k] = __float_as_uint(v - __uint_as_float(hb));
      }
      tmem_st32(hi + c * 32, ph);
      tmem_st32(lo + c * 32, pl);
    }
  }
}

// ------------------------------------------------------------------ dK / dV
template <int D, int F32, bool QSPLIT = false>
__global__ void __launch_bounds__(BwdCfg<D, F32>::THREADS, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ KVMaps m, const BwdArgs a) {
  using C = BwdCfg<D, F32>;
  constexpr int CH = C::CH, NST = C::KV_NST;
  // A programmatic dependent of the kernel that wrote the operand copies: wait for it,
  // and only then let the dQ grid launched after this one start (it reads those copies
  // without a wait of its own, on the SMs this grid leaves free).
  grid_dependency_wait();
  grid_launch_dependents();
  // (fp32 inputs only: bf16 inputs use fa_bwd_dkdv16_kernel, whose accumulating MMAs
  // would read the score half of a stage, which this kernel releases early)
  static_assert(F32, "the 3xTF32 dK / dV kernel");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  // A stage has two halves with their own full / empty barriers: the score half (Q and
  // dO chunks, read by S^T and dP^T) is free once those MMAs completed, so the next
  // chunk's copy lands while the softmax and the accumulating MMAs of this one run;
  // the accumulate half (Q^T, dO^T chunks and the lse2 / delta vectors, read by dV, dK
  // and the softmax) once dV and dK completed.
  __shared__ __align__(8) uint64_t bar_kv, bar_sfull[NST], bar_sempty[NST], bar_afull[NST],
      bar_aempty[NST], bar_sp[2], bar_ds[2], bar_accdone[2], bar_done, bar_drain[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = warp_id(), lane = lane_id();
  volatile int* abort_flag = &abort_sh;

  // Key tile 0 is seen by the most queries under a causal mask: schedule it first.
  // QSPLIT (few items: short key sequences): each also takes query range kr of a.tps
  // query tiles, writing partial dK, dV to slab kr. (A template flag: as a runtime one it
  // cost the unsplit C5 kernel 2%.)
  const int kr = QSPLIT ? (int)(blockIdx.x % a.n_splits) : 0;
  const unsigned w_item = QSPLIT ? blockIdx.x / a.n_splits : blockIdx.x;  // (unsigned, as before)
  const int jt = w_item / a.BHx;
  const int bg = w_item % a.BHx;
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
    else { qc_lo = imin / CH; qc_hi = imax / CH + 1; }
    if constexpr (QSPLIT) {  // the range's chunks: query tiles [kr tps, (kr + 1) tps)
      constexpr int CPT = BLOCK_M / CH;
      qc_lo = max(qc_lo, kr * a.tps * CPT);
      qc_hi = min(qc_hi, (kr + 1) * a.tps * CPT);
      if (qc_hi < qc_lo) qc_hi = qc_lo;
    }
  }
  const int ncq = qc_hi - qc_lo;
  const int nc = rep * ncq;
  const int zkv = QSPLIT ? kr * a.BHx + bg : bg;  // dK / dV slab row block

  if (threadIdx.x == 0) {
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bar_sfull[s], 1);
      mbar_init(&bar_sempty[s], 1);
      mbar_init(&bar_afull[s], 1);
      mbar_init(&bar_aempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_sp[s], 1);
      mbar_init(&bar_ds[s], 128);
      mbar_init(&bar_accdone[s], 1);
      mbar_init(&bar_drain[s], 1);
    }
    mbar_init(&bar_done, 1);
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
  auto sK = [&](int sp) { return sbase + sp * C::BIG_TILE; };
  auto sV = [&](int sp) { return sbase + (C::NSPLIT + sp) * C::BIG_TILE; };
  auto stage = [&](int st) { return sbase + C::KV_RES + st * C::KV_STAGE; };
  auto sQc = [&](int st, int sp) { return stage(st) + sp * C::SMALL_TILE; };
  auto sdOc = [&](int st, int sp) { return stage(st) + (C::NSPLIT + sp) * C::SMALL_TILE; };
  auto sQt = [&](int st, int sp) { return stage(st) + 2 * C::NSPLIT * C::SMALL_TILE + sp * C::T_TILE; };
  auto sdOt = [&](int st, int sp) {
    return stage(st) + 2 * C::NSPLIT * C::SMALL_TILE + (C::NSPLIT + sp) * C::T_TILE;
  };
  float* vecs = reinterpret_cast<float*>(smem + C::KV_VEC_OFF);  // [NST][2][CH]
  auto gen = [&](uint32_t s) { return smem + (s - sbase); };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };
  // (the issuers poll: a suspending wait right after their own MMA burst returns only
  // once the burst has drained)
  auto poll = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait_poll(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };
  auto chunk_rows = [&](int c, int* bh, int* i0) {
    const int r = c / ncq, qc = qc_lo + c % ncq;
    *bh = b * a.H + g * rep + r;
    *i0 = qc * CH;
  };

  if (warp == C::TMA_WARP) {
    if (lane == 0 && nc > 0) {
      tma_prefetch_desc(&m.K[0]); tma_prefetch_desc(&m.Qc[0]); tma_prefetch_desc(&m.dOc[0]);
      mbar_arrive_expect_tx(&bar_kv, 2 * C::NSPLIT * C::BIG_TILE);
      for (int sp = 0; sp < C::NSPLIT; ++sp)
        for (int cb = 0; cb < C::NCB; ++cb) {
          tma_load_3d(gen(sK(sp)) + cb * C::BIG_CB, &m.K[sp], &bar_kv, cb * C::ROW, j0, bg);
          tma_load_3d(gen(sV(sp)) + cb * C::BIG_CB, &m.V[sp], &bar_kv, cb * C::ROW, j0, bg);
        }
      int last_s[NST], last_a[NST];
      for (int s = 0; s < NST; ++s) last_s[s] = last_a[s] = -1;
      for (int c = 0; c < nc; ++c) {
        const int st = c % NST;
        int bh, i0;
        chunk_rows(c, &bh, &i0);
        if (!wait(&bar_sempty[st], ((c / NST) & 1) ^ 1)) break;
        mbar_arrive_expect_tx(&bar_sfull[st], 2 * C::NSPLIT * C::SMALL_TILE);
        for (int sp = 0; sp < C::NSPLIT; ++sp) {
          for (int cb = 0; cb < C::NCB; ++cb) {
            tma_load_3d(gen(sQc(st, sp)) + cb * C::SMALL_CB, &m.Qc[sp], &bar_sfull[st], cb * C::ROW, i0, bh);
            tma_load_3d(gen(sdOc(st, sp)) + cb * C::SMALL_CB, &m.dOc[sp], &bar_sfull[st], cb * C::ROW, i0, bh);
          }
        }
        last_s[st] = c / NST;
        if (!wait(&bar_aempty[st], ((c / NST) & 1) ^ 1)) break;
        mbar_arrive_expect_tx(&bar_afull[st], 2 * C::NSPLIT * C::T_TILE + C::VEC_STAGE);
        if constexpr (C::TF32) {
          for (int sp = 0; sp < C::NSPLIT; ++sp) {
            tma_load_3d(gen(sQt(st, sp)), &m.Qt[sp], &bar_afull[st], i0, 0, bh);
            tma_load_3d(gen(sdOt(st, sp)), &m.dOt[sp], &bar_afull[st], i0, 0, bh);
          }
        }
        tma_load_3d(vecs + st * 2 * CH, &m.L, &bar_afull[st], i0, bh, 0);
        tma_load_3d(vecs + st * 2 * CH + CH, &m.Dl, &bar_afull[st], i0, bh, 0);
        last_a[st] = c / NST;
      }
      drain_wait(&bar_kv, 0, a.limit_ns);
      for (int s = 0; s < NST; ++s) {
        if (last_s[s] >= 0) drain_wait(&bar_sfull[s], last_s[s] & 1, a.limit_ns);
        if (last_a[s] >= 0) drain_wait(&bar_afull[s], last_a[s] & 1, a.limit_ns);
      }
    }
  } else if (warp == C::MMA_WARP) {
    // Score issuer: chunk c -> S^T = K Q^T and dP^T = V dO^T into TMEM slot c & 1,
    // once the slot's previous chunk (c - 2) has been accumulated.
    if (lane == 0 && nc > 0) {
      bool ok = wait(&bar_kv, 0);
      for (int c = 0; ok && c < nc; ++c) {
        const int st = c % NST, bb = c & 1;
        if (!(ok = poll(&bar_sfull[st], (c / NST) & 1))) break;
        if (c >= 2 && !(ok = poll(&bar_accdone[bb], ((c - 2) >> 1) & 1))) break;
        tc_fence_after();
        issue_rowdot<C>(tmem + C::s_col(bb), sK(0), sK(C::NSPLIT - 1), sQc(st, 0),
                        sQc(st, C::NSPLIT - 1));
        issue_rowdot<C>(tmem + C::dp_col(bb), sV(0), sV(C::NSPLIT - 1), sdOc(st, 0),
                        sdOc(st, C::NSPLIT - 1));
        tc_commit(&bar_sp[bb]);
        // the score half of the stage may take the next chunk (X16: not yet -- the
        // accumulating MMAs read the same Q / dO chunks; they release it)
        if constexpr (!C::X16) tc_commit(&bar_sempty[st]);
      }
      tc_commit(&bar_drain[0]);
      drain_wait(&bar_drain[0], 0, a.limit_ns);
    }
  } else if (warp == C::ACC_WARP) {
    // Accumulate issuer: chunk c -> dV += P^T dO, dK += dS^T Q once the softmax
    // wrote P^T / dS^T; then the chunk's smem stage and TMEM slot are free.
    if (lane == 0 && nc > 0) {
      bool ok = true;
      for (int c = 0; ok && c < nc; ++c) {
        const int pb = c & 1, pst = c % NST;
        if (!(ok = poll(&bar_ds[pb], (c >> 1) & 1))) break;
        // the accumulate half (its phase of chunk c cannot be passed before aempty(c))
        if (!(ok = poll(&bar_afull[pst], (c / NST) & 1))) break;
        tc_fence_after();
        if constexpr (C::X16) {  // B = the MN-major Q / dO chunks themselves
          issue_acc<C>(tmem + C::KV_ACC0, tmem + C::s_col(pb), tmem + C::plo_col(pb), sdOc(pst, 0),
                       sdOc(pst, 1), c > 0);
          issue_acc<C>(tmem + C::KV_ACC1, tmem + C::dp_col(pb), tmem + C::dslo_col(pb), sQc(pst, 0),
                       sQc(pst, 1), c > 0);
          tc_commit(&bar_sempty[pst]);
        } else {
          issue_acc<C>(tmem + C::KV_ACC0, tmem + C::s_col(pb), tmem + C::plo_col(pb), sdOt(pst, 0),
                       sdOt(pst, 1), c > 0);
          issue_acc<C>(tmem + C::KV_ACC1, tmem + C::dp_col(pb), tmem + C::dslo_col(pb), sQt(pst, 0),
                       sQt(pst, 1), c > 0);
        }
        tc_commit(&bar_aempty[pst]);
        tc_commit(&bar_accdone[pb]);
      }
      if (ok) tc_commit(&bar_done);
      tc_commit(&bar_drain[1]);
      drain_wait(&bar_drain[1], 0, a.limit_ns);
    }
  } else if (warp < C::MMA_WARP) {
    // softmax warps: thread = one key row j = one TMEM lane
    const int wq = warp;  // 0..3
    const int r_in = wq * 32 + lane;
    const int j = j0 + r_in;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    // X16: scores and dP^T from the scaled copies (multipliers as in the bf16 kernels)
    const float sl2 = C::X16 ? a.sc->sl2 : a.scale_log2;
    const float dp_mul = C::X16 ? a.sc->dp_mul : 1.f;
    bool ok = true;
    for (int c = 0; c < nc; ++c) {
      const int bb = c & 1, st = c % NST;
      int bh, i0;
      chunk_rows(c, &bh, &i0);
      ok = __all_sync(0xffffffffu, wait(&bar_sp[bb], (c >> 1) & 1) && wait(&bar_afull[st], (c / NST) & 1));
      if (!ok) break;
      tc_fence_after();
      float s[CH], dp[CH];
      tmem_ld_pair<CH>(lane_addr + C::s_col(bb), lane_addr + C::dp_col(bb), s, dp);
      // queries i = i0 + k; key j visible iff (!causal || j <= i) && (!window || j >= i-w+1)
      // && j < Sk && i < Sq
      if (tile_needs_mask(i0, i0 + CH - 1, j0, j0 + BLOCK_N - 1, a.Sk, a.causal, a.window) ||
          i0 + CH > a.Sq) {
        const int k_lo = a.causal ? j - i0 : INT_MIN / 2;                          // i >= j
        const int k_hi = min(a.window > 0 ? j + a.window - 1 - i0 : INT_MAX / 2,   // i <= j+w-1
                             a.Sq - 1 - i0);
        const bool row_dead = j >= a.Sk;
        mask_outside<CH>(s, row_dead ? INT_MAX / 2 : k_lo, k_hi);
      }
      const float* lv = vecs + st * 2 * CH;
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        const float p = ex2(fmaf(s[k], sl2, -lv[k]));
        dp[k] = p * (C::X16 ? fmaf(dp[k], dp_mul, -lv[CH + k]) : dp[k] - lv[CH + k]);
        s[k] = p;
      }
      tmem_st_operand<C>(lane_addr + C::s_col(bb), lane_addr + C::plo_col(bb), s);
      tmem_st_operand<C>(lane_addr + C::dp_col(bb), lane_addr + C::dslo_col(bb), dp);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_ds[bb]);
    }
    if (ok && nc > 0) {
      ok = __all_sync(0xffffffffu, wait(&bar_done, 0));
      tc_fence_after();
    }
    if (ok) {
      // bar_done: every MMA has completed, so all operand buffers are free.
      const uint32_t st_v = sbase + wq * 2 * C::EPI_WARP, st_k = st_v + C::EPI_WARP;
      const int r_base = j0 + wq * 32;
      const bool any = r_base < a.Sk;
      const float mul_v = C::X16 ? a.sc->dv_mul : 1.f, mul_k = C::X16 ? a.sc->dk_mul : a.scale;
      if (a.out_bf16) {
        store_rows_tma<D, true, D / 64, false>(&m.dV, lane_addr + C::KV_ACC0, nc > 0, mul_v, st_v,
                                               r_base, any, zkv, 0, a.Dv);
        store_rows_tma<D, true, D / 64, false>(&m.dK, lane_addr + C::KV_ACC1, nc > 0, mul_k, st_k,
                                               r_base, any, zkv, 0, a.Dv);
      } else {
        store_rows_tma<D, false, D / 32, false>(&m.dV, lane_addr + C::KV_ACC0, nc > 0, mul_v, st_v,
                                                r_base, any, zkv, 0, a.Dv);
        store_rows_tma<D, false, D / 32, false>(&m.dK, lane_addr + C::KV_ACC1, nc > 0, mul_k, st_k,
                                                r_base, any, zkv, 0, a.Dv);
      }
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
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
template <int D, int F32>
__global__ void __launch_bounds__(BwdCfg<D, F32>::THREADS, 1)
    fa_bwd_dq_kernel(const __grid_constant__ QMaps m, const BwdArgs a) {
  using C = BwdCfg<D, F32>;
  constexpr int CH = C::CH, NST = C::Q_NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int NSL = C::Q_NSLOT;
  __shared__ __align__(8) uint64_t bar_q, bar_full[NST], bar_empty[NST], bar_sp[NSL], bar_ds[NSL],
      bar_accdone[NSL], bar_done, bar_drain[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = warp_id(), lane = lane_id();
  volatile int* abort_flag = &abort_sh;

  // work item: (query tile, head) and, with the keys split into ranges (few query
  // tiles), key range kr of a.tps key tiles, whose partial dQ goes to slab kr
  const int kr = a.n_splits > 1 ? (int)(blockIdx.x % a.n_splits) : 0;
  const int w_item = a.n_splits > 1 ? (int)(blockIdx.x / a.n_splits) : (int)blockIdx.x;
  const int qt_lin = w_item / a.BHx;
  const int bh = w_item % a.BHx;
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
    else { kc_lo = jmin / CH; kc_hi = jmax / CH + 1; }
    if (a.n_splits > 1) {  // the range's chunks: key tiles [kr tps, (kr + 1) tps)
      constexpr int CPT = BLOCK_N / CH;
      kc_lo = max(kc_lo, kr * a.tps * CPT);
      kc_hi = min(kc_hi, (kr + 1) * a.tps * CPT);
      if (kc_hi < kc_lo) kc_hi = kc_lo;
    }
  }
  const int nc = kc_hi - kc_lo;
  const int zq = a.n_splits > 1 ? kr * a.BHx + bh : bh;  // dQ slab row block

  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < NST; ++s) { mbar_init(&bar_full[s], 1); mbar_init(&bar_empty[s], 1); }
    for (int s = 0; s < NSL; ++s) {
      mbar_init(&bar_sp[s], 1);
      mbar_init(&bar_ds[s], 128);
      mbar_init(&bar_accdone[s], 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(&bar_drain[s], 1);
    mbar_init(&bar_done, 1);
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
  auto sQ = [&](int sp) { return sbase + sp * C::BIG_TILE; };
  auto sdO = [&](int sp) { return sbase + (C::NSPLIT + sp) * C::BIG_TILE; };
  auto stage = [&](int st) { return sbase + C::Q_RES + st * C::Q_STAGE; };
  auto sKc = [&](int st, int sp) { return stage(st) + sp * C::SMALL_TILE; };
  auto sVc = [&](int st, int sp) { return stage(st) + (C::NSPLIT + sp) * C::SMALL_TILE; };
  auto sKt = [&](int st, int sp) { return stage(st) + 2 * C::NSPLIT * C::SMALL_TILE + sp * C::T_TILE; };
  auto gen = [&](uint32_t s) { return smem + (s - sbase); };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };
  // (the issuers poll: a suspending wait right after their own MMA burst returns only
  // once the burst has drained)
  auto poll = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait_poll(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };

  if (warp == C::TMA_WARP) {
    if (lane == 0 && nc > 0) {
      tma_prefetch_desc(&m.Q[0]); tma_prefetch_desc(&m.Kc[0]); tma_prefetch_desc(&m.Vc[0]);
      mbar_arrive_expect_tx(&bar_q, 2 * C::NSPLIT * C::BIG_TILE);
      for (int sp = 0; sp < C::NSPLIT; ++sp)
        for (int cb = 0; cb < C::NCB; ++cb) {
          tma_load_3d(gen(sQ(sp)) + cb * C::BIG_CB, &m.Q[sp], &bar_q, cb * C::ROW, i0, bh);
          tma_load_3d(gen(sdO(sp)) + cb * C::BIG_CB, &m.dO[sp], &bar_q, cb * C::ROW, i0, bh);
        }
      int last[NST];
      for (int s = 0; s < NST; ++s) last[s] = -1;
      for (int c = 0; c < nc; ++c) {
        const int st = c % NST;
        if (!wait(&bar_empty[st], ((c / NST) & 1) ^ 1)) break;
        const int k0 = (kc_lo + c) * CH;
        mbar_arrive_expect_tx(&bar_full[st], C::Q_STAGE);
        for (int sp = 0; sp < C::NSPLIT; ++sp) {
          for (int cb = 0; cb < C::NCB; ++cb) {
            tma_load_3d(gen(sKc(st, sp)) + cb * C::SMALL_CB, &m.Kc[sp], &bar_full[st], cb * C::ROW, k0, bg);
            tma_load_3d(gen(sVc(st, sp)) + cb * C::SMALL_CB, &m.Vc[sp], &bar_full[st], cb * C::ROW, k0, bg);
          }
          if constexpr (C::TF32) tma_load_3d(gen(sKt(st, sp)), &m.Kt[sp], &bar_full[st], k0, 0, bg);
        }
        last[st] = c / NST;
      }
      drain_wait(&bar_q, 0, a.limit_ns);
      for (int s = 0; s < NST; ++s)
        if (last[s] >= 0) drain_wait(&bar_full[s], last[s] & 1, a.limit_ns);
    }
  } else if (warp == C::MMA_WARP) {
    // Score issuer: chunk c -> S = Q K^T and dP = dO V^T into TMEM slot c % NSL,
    // once the slot's previous chunk (c - NSL) has been accumulated.
    if (lane == 0 && nc > 0) {
      bool ok = wait(&bar_q, 0);
      for (int c = 0; ok && c < nc; ++c) {
        const int st = c % NST, bb = c % NSL;
        if (!(ok = poll(&bar_full[st], (c / NST) & 1))) break;
        if (c >= NSL && !(ok = poll(&bar_accdone[bb], ((c / NSL) - 1) & 1))) break;
        tc_fence_after();
        issue_rowdot<C>(tmem + C::s_col(bb), sQ(0), sQ(C::NSPLIT - 1), sKc(st, 0),
                        sKc(st, C::NSPLIT - 1));
        issue_rowdot<C>(tmem + C::dp_col(bb), sdO(0), sdO(C::NSPLIT - 1), sVc(st, 0),
                        sVc(st, C::NSPLIT - 1));
        tc_commit(&bar_sp[bb]);
      }
      tc_commit(&bar_drain[0]);
      drain_wait(&bar_drain[0], 0, a.limit_ns);
    }
  } else if (warp == C::ACC_WARP) {
    // Accumulate issuer: chunk c -> dQ += dS K once the softmax wrote dS; then the
    // chunk's smem stage and TMEM slot are free.
    if (lane == 0 && nc > 0) {
      bool ok = true;
      for (int c = 0; ok && c < nc; ++c) {
        const int pb = c % NSL, pst = c % NST;
        if (!(ok = poll(&bar_ds[pb], (c / NSL) & 1))) break;
        tc_fence_after();
        if constexpr (!C::F32)
          issue_acc<C>(tmem + C::Q_ACC, tmem + C::dp_col(pb), 0, sKc(pst, 0), 0, c > 0);
        else if constexpr (C::X16)  // B = the MN-major K chunk itself
          issue_acc<C>(tmem + C::Q_ACC, tmem + C::dp_col(pb), tmem + C::dslo_col(pb), sKc(pst, 0),
                       sKc(pst, 1), c > 0);
        else
          issue_acc<C>(tmem + C::Q_ACC, tmem + C::dp_col(pb), tmem + C::dslo_col(pb), sKt(pst, 0),
                       sKt(pst, 1), c > 0);
        tc_commit(&bar_empty[pst]);
        tc_commit(&bar_accdone[pb]);
      }
      if (ok) tc_commit(&bar_done);
      tc_commit(&bar_drain[1]);
      drain_wait(&bar_drain[1], 0, a.limit_ns);
    }
  } else if (warp < C::MMA_WARP) {
    const int wq = warp;
    const int r_in = wq * 32 + lane;
    const int i = i0 + r_in;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = C::X16 ? a.sc->sl2 : a.scale_log2;
    const float dp_mul = C::X16 ? a.sc->dp_mul : 1.f;
    const bool row_valid = i < a.Sq;
    const size_t vrow = (size_t)bh * a.ldq + (size_t)(row_valid ? i : 0);
    const float lse2 = row_valid ? a.lse2[vrow] : INFINITY;
    const float dl = row_valid ? a.delta[vrow] : 0.f;
    const int hi_i = a.causal ? min(i, a.Sk - 1) : a.Sk - 1;
    const int lo_i = a.window > 0 ? i - a.window + 1 : INT_MIN / 2;
    bool ok = true;
    for (int c = 0; c < nc; ++c) {
      const int bb = c % NSL;
      const int k0 = (kc_lo + c) * CH;
      ok = __all_sync(0xffffffffu, wait(&bar_sp[bb], (c / NSL) & 1));
      if (!ok) break;
      tc_fence_after();
      float s[CH], dp[CH];
      tmem_ld_pair<CH>(lane_addr + C::s_col(bb), lane_addr + C::dp_col(bb), s, dp);
      if (tile_needs_mask(i0, i0 + BLOCK_M - 1, k0, k0 + CH - 1, a.Sk, a.causal, a.window)) {
        mask_outside<CH>(s, lo_i - k0, hi_i - k0);
      }
      const float nl = -lse2;
#pragma unroll
      for (int k = 0; k < CH; ++k)
        dp[k] = ex2(fmaf(s[k], sl2, nl)) * (C::X16 ? fmaf(dp[k], dp_mul, -dl) : dp[k] - dl);
      tmem_st_operand<C>(lane_addr + C::dp_col(bb), lane_addr + C::dslo_col(bb), dp);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_ds[bb]);
    }
    if (ok && nc > 0) {
      ok = __all_sync(0xffffffffu, wait(&bar_done, 0));
      tc_fence_after();
    }
    if (ok) {
      // bar_done: every MMA has completed, so all operand buffers are free.
      const uint32_t st_q = sbase + wq * C::EPI_WARP;
      const int r_base = i0 + wq * 32;
      const float mul_q = C::X16 ? a.sc->dq_mul : a.scale;
      if (a.out_bf16)
        store_rows_tma<D, true, D / 64>(&m.dQ, lane_addr + C::Q_ACC, nc > 0, mul_q, st_q, r_base,
                                        r_base < a.Sq, zq, 0, a.Dv);
      else
        store_rows_tma<D, false, D / 32>(&m.dQ, lane_addr + C::Q_ACC, nc > 0, mul_q, st_q,
                                         r_base, r_base < a.Sq, zq, 0, a.Dv);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // Launched as a programmatic dependent of the dK / dV grid (it reads nothing that grid
  // writes): this grid completes only after that one has.
  grid_dependency_wait();
}

// --------------------------------------------------------- dQ, fp16 operands
// bf16 inputs: work item = (batch, head, 128-query tile), 128-key chunks, so the
// score MMAs are 128 x 128 (a 128 x 64 MMA reads 3/4 of the shared-memory bytes of a
// 128 x 128 one for half the work, and the dq kernel is bound by those reads).
// TMEM: S slot [0, 128), dP slot [128, 256), two fp16 dS operand slots of 64
// columns at 256 / 320, dQ at 384. The S and dP slots are single: the softmax
// releases each as soon as it has loaded it, so chunk c+1's S = Q K^T runs while
// the softmax finishes chunk c. S, dP and dQ MMAs come from three issuing threads:
// an issuer stalls while the tensor pipe is full, so each stream gets its own. Eight softmax warps: warps w and w+4 share TMEM
// lanes 32*(w%4).., w < 4 taking keys [0, 64) of the chunk, w >= 4 keys [64, 128).
template <int D>
struct Dq16Cfg {
  // smem rows of RB bytes with the swizzle of that width (64 bytes at D = 32)
  static constexpr int RB = tile_row_bytes(D);
  static constexpr uint32_t SWZ = RB == 128 ? SWZ_128B : SWZ_64B;
  static constexpr uint32_t ATOM = 8u * RB;
  static constexpr int ROW = RB / 2;                     // elements per row
  static constexpr int NCB = D / ROW;                    // column blocks per row
  static constexpr uint32_t CB = 128u * RB;              // column block of a 128-row tile
  static constexpr uint32_t TILE = NCB * CB;
  static constexpr int KST = 3, VST = 2;                 // K is held until dQ += dS K
  static constexpr uint32_t Q_OFF = 0, DO_OFF = TILE, K_OFF = 2 * TILE;
  static constexpr uint32_t V_OFF = K_OFF + KST * TILE;
  static constexpr uint32_t SMEM = V_OFF + VST * TILE + 1024;
  static constexpr int SOFTMAX_WARPS = 8;
  static constexpr int MMA_WARP = 8, ACC_WARP = 9, TMA_WARP = 10, DP_WARP = 11;
  static constexpr int THREADS = 384;
  // work-item hand-out ring: the producer writes, the three issuers and the eight
  // softmax warps read every entry
  static constexpr int IRING = 4, ITEM_READERS = 3 + SOFTMAX_WARPS;
  static constexpr uint32_t REGS_SOFTMAX = 200, REGS_CONTROL = 96;
  static_assert(256 * REGS_SOFTMAX + 128 * REGS_CONTROL <= 384 * 168, "register split");
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DS_COL = 256, ACC = 384;
  static constexpr uint32_t EPI_WARP = epi_warp_bytes<D, false>();
  static_assert(SMEM <= 227u * 1024u, "shared memory budget");
  static_assert(4 * EPI_WARP <= VST * TILE, "epilogue staging (the V ring)");
};

template <int D>
__device__ __forceinline__ void issue_rowdot128(uint32_t d, uint32_t a, uint32_t b) {
  using L = Dq16Cfg<D>;  // (the tile layout of both backward kernels)
  constexpr uint32_t id = make_idesc(128, 128, FMT_F16, FMT_F16, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk * 16 / L::ROW) * L::CB + (kk * 16 % L::ROW) * 2;
    mma_f16_ss(d, make_sdesc(a + off, 16, L::ATOM, L::SWZ), make_sdesc(b + off, 16, L::ATOM, L::SWZ),
               id, kk > 0);
  }
}

// Epilogue piece of the persistent dQ kernel: NCOL accumulator columns of this
// warp's 32 rows, already in registers, times mul, go out through the 1024-byte
// aligned staging area `stage` (NCOL * 4 or * 2 bytes per row, as 128-byte boxes)
// with TMA stores to tensor columns x0 ..; lane 0 commits them as one bulk group.
template <int NCOL, bool OUT_BF16>
__device__ __forceinline__ void stage_store_rows(const uint32_t (&r)[NCOL], float mul,
                                                 uint32_t stage, const CUtensorMap* tm, int x0,
                                                 int r_base, bool any_row, int z, int x_end) {
  constexpr int COLS = OUT_BF16 ? 64 : 32;  // columns per 128-byte box row
  constexpr int NBOX = NCOL / COLS;
  static_assert(NCOL % COLS == 0, "whole boxes");
  const uint32_t lane = lane_id(), sw = lane & 7u;
#pragma unroll
  for (int bx = 0; bx < NBOX; ++bx) {
    const uint32_t row = stage + bx * EPI_BOX_BYTES + lane * 128u;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t w[4];
      if constexpr (!OUT_BF16) {
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = __float_as_uint(__uint_as_float(r[bx * 32 + 4 * c + e]) * mul);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = bx * 64 + 8 * c + 2 * e;
          __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(r[k]) * mul,
                                                    __uint_as_float(r[k + 1]) * mul);
          w[e] = *reinterpret_cast<uint32_t*>(&v2);
        }
      }
      st_shared_v4(row + ((c ^ sw) << 4), w[0], w[1], w[2], w[3]);
    }
  }
  fence_async_shared();
  __syncwarp();
  if (lane == 0) {
    if (any_row)
      for (int bx = 0; bx < NBOX; ++bx)
        if (x0 + bx * COLS < x_end)  // (boxes past the tensor's width are not stored)
          tma_store_3d(tm, stage + bx * EPI_BOX_BYTES, x0 + bx * COLS, r_base, z);
    bulk_commit_group();
  }
}

// Persistent: one CTA per SM walks (batch, head, query tile) work items, heaviest
// causal tiles first: its first item is blockIdx.x, the next ones come from a global
// counter (a CTA that starts late, e.g. while another kernel still holds SMs, takes
// fewer items). The TMA producer fetches them, one item ahead, and hands them to the
// other roles through a small shared ring. Every ring and hand-off barrier counts
// chunks across items (g), so the K / V ring streams the next item's first chunks
// while the current item's epilogue runs. Per item with keys (counted by j): Q_{j+1} (dO_{j+1}) is
// loaded as soon as the last S (dP) MMA of item j has completed (q_rel / do_rel),
// the epilogue stages dQ in the V ring, so item j+1's first V chunk waits until the
// epilogue has read that staging area (v_free), and the first dQ MMA of item j+1
// waits until the epilogue has read dQ out of TMEM (dq_free). Each of these
// per-item phases can only complete after every role has observed the one before
// (e.g. q_rel(j+1) follows S MMAs of item j+1, which need Q_{j+1}, loaded only after
// q_rel(j) was seen), so a parity wait never misses a phase. An item whose rows see
// no key (in its key range) touches none of these barriers and writes nothing: the
// launcher zeroes those dQ rows beforehand, or, with the keys split into ranges, the
// sum over the ranges leaves that range out. SPLIT: the keys are split into ranges (a
// separate instantiation, so the unsplit kernel's code is not touched by it).
template <int D, bool SPLIT>
__global__ void __launch_bounds__(Dq16Cfg<D>::THREADS, 1)
    fa_bwd_dq16_kernel(const __grid_constant__ QMaps m, const BwdArgs a) {
  using C = Dq16Cfg<D>;
  constexpr int KST = C::KST, VST = C::VST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_q, bar_do, bar_kfull[KST], bar_kempty[KST], bar_vfull[VST],
      bar_vempty[VST], bar_s, bar_dp, bar_sfree, bar_dpfree, bar_ds[2], bar_accdone[2], bar_done,
      bar_dqfree, bar_qrel, bar_dorel, bar_vfree, bar_drain[3], bar_ifull[C::IRING],
      bar_iempty[C::IRING];
  __shared__ int ring_w_sh[C::IRING];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = warp_id(), lane = lane_id();
  volatile int* abort_flag = &abort_sh;

  // Work item w = (qt_lin * BH + bh) * n_splits + sp: query tile, head and (SPLIT) key
  // range sp, key tiles [sp * tps, (sp + 1) * tps); dQ goes to slab zo = sp * BH + bh
  // (the partial sum over one key range when split, else dQ itself).
  const int n_items = a.n_tiles * a.BHx * (SPLIT ? a.n_splits : 1);
  struct Item { int bh, bg, i0, kt_lo, nc; };
  auto item = [&](int w) {
    Item it;
    const int wq = SPLIT ? w / a.n_splits : w;
    const int qt_lin = wq / a.BHx;
    it.bh = wq % a.BHx;
    const int qt = a.lpt ? (a.n_tiles - 1 - qt_lin) : qt_lin;
    const int b = it.bh / a.H, h = it.bh % a.H;
    it.bg = b * a.HKV + h / (a.H / a.HKV);
    it.i0 = qt * BLOCK_M;
    int hi;
    kv_tile_range(it.i0, min(it.i0 + BLOCK_M - 1, a.Sq - 1), a.Sk, a.causal, a.window, &it.kt_lo, &hi);
    if constexpr (SPLIT) {
      const int sp = w % a.n_splits;
      it.kt_lo = max(it.kt_lo, sp * a.tps);
      hi = min(hi, (sp + 1) * a.tps);
      if (hi < it.kt_lo) hi = it.kt_lo;
    }
    it.nc = hi - it.kt_lo;
    return it;
  };
  // work-item hand-out (see above): entry k of the ring holds this CTA's k-th item
  // (n_items or more: no further item)
  volatile int* ring_w = ring_w_sh;

  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_do, 1);
    for (int s = 0; s < KST; ++s) { mbar_init(&bar_kfull[s], 1); mbar_init(&bar_kempty[s], 1); }
    for (int s = 0; s < VST; ++s) { mbar_init(&bar_vfull[s], 1); mbar_init(&bar_vempty[s], 1); }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_sfree, 256);
    mbar_init(&bar_dpfree, 256);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_ds[s], 256);
      mbar_init(&bar_accdone[s], 1);
    }
    mbar_init(&bar_done, 1);
    mbar_init(&bar_dqfree, 256);
    mbar_init(&bar_qrel, 1);
    mbar_init(&bar_dorel, 1);
    mbar_init(&bar_vfree, 256);
    for (int s = 0; s < 3; ++s) mbar_init(&bar_drain[s], 1);
    for (int s = 0; s < C::IRING; ++s) {
      mbar_init(&bar_ifull[s], 1);
      mbar_init(&bar_iempty[s], C::ITEM_READERS);
    }
    abort_sh = 0;
    fence_mbar_init();
    if ((int)blockIdx.x < n_items && item(blockIdx.x).nc > 0) {
      // The first item's Q / dO tiles and first K / V chunk are issued here, before
      // the TMEM allocation and the CTA-wide sync, so their latency overlaps the setup.
      const Item it = item(blockIdx.x);
      const int k0 = it.kt_lo * BLOCK_N;
      mbar_arrive_expect_tx(&bar_q, C::TILE);
      mbar_arrive_expect_tx(&bar_do, C::TILE);
      mbar_arrive_expect_tx(&bar_kfull[0], C::TILE);
      mbar_arrive_expect_tx(&bar_vfull[0], C::TILE);
      for (int cb = 0; cb < C::NCB; ++cb) {
        tma_load_3d(smem + C::Q_OFF + cb * C::CB, &m.Q[0], &bar_q, cb * C::ROW, it.i0, it.bh);
        tma_load_3d(smem + C::DO_OFF + cb * C::CB, &m.dO[0], &bar_do, cb * C::ROW, it.i0, it.bh);
        tma_load_3d(smem + C::K_OFF + cb * C::CB, &m.Kc[0], &bar_kfull[0], cb * C::ROW, k0, it.bg);
        tma_load_3d(smem + C::V_OFF + cb * C::CB, &m.Vc[0], &bar_vfull[0], cb * C::ROW, k0, it.bg);
      }
    }
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
  auto sK = [&](int st) { return sbase + C::K_OFF + st * C::TILE; };
  auto sV = [&](int st) { return sbase + C::V_OFF + st * C::TILE; };
  auto gen = [&](uint32_t s) { return smem + (s - sbase); };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };
  auto poll = [&](uint64_t* bar, uint32_t parity) {  // (issuer waits on the softmax: no suspend)
    return mbar_wait_poll(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };
  // Reader side of the item ring: entry k, then release the entry (one arrival per
  // reading thread / warp). A failed wait reads as "no further item".
  auto take_thread = [&](int k) {
    const int s = k % C::IRING;
    if (!wait(&bar_ifull[s], (k / C::IRING) & 1)) return INT_MAX;
    const int w = ring_w[s];
    mbar_arrive(&bar_iempty[s]);
    return w;
  };
  auto take_warp = [&](int k) {
    const int s = k % C::IRING;
    if (!__all_sync(0xffffffffu, wait(&bar_ifull[s], (k / C::IRING) & 1))) return INT_MAX;
    const int w = ring_w[s];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar_iempty[s]);
    return w;
  };

  if (warp >= C::SOFTMAX_WARPS) {
  regs_decrease<C::REGS_CONTROL>();
  if (warp == C::TMA_WARP) {
    if (lane == 0) {
      const bool setup_issued = (int)blockIdx.x < n_items && item(blockIdx.x).nc > 0;
      int g = 0, j = 0;  // chunks, items with keys, issued so far
      int last_k[KST], last_v[VST], last_qd = setup_issued ? 0 : -1;
      for (int s = 0; s < KST; ++s) last_k[s] = -1;
      for (int s = 0; s < VST; ++s) last_v[s] = -1;
      auto load_k = [&](int g_, int k0, int bg) {
        const int ks = g_ % KST;
        if (!wait(&bar_kempty[ks], ((g_ / KST) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(&bar_kfull[ks], C::TILE);
        for (int cb = 0; cb < C::NCB; ++cb)
          tma_load_3d(gen(sK(ks)) + cb * C::CB, &m.Kc[0], &bar_kfull[ks], cb * C::ROW, k0, bg);
        last_k[ks] = g_ / KST;
        return true;
      };
      auto load_v = [&](int g_, int k0, int bg) {
        const int vs = g_ % VST;
        if (!wait(&bar_vempty[vs], ((g_ / VST) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(&bar_vfull[vs], C::TILE);
        for (int cb = 0; cb < C::NCB; ++cb)
          tma_load_3d(gen(sV(vs)) + cb * C::CB, &m.Vc[0], &bar_vfull[vs], cb * C::ROW, k0, bg);
        last_v[vs] = g_ / VST;
        return true;
      };
      // Q (dO) of item j once the last S (dP) MMA of item j-1 has read the buffer
      auto load_res = [&](const Item& it, bool is_q) {
        uint64_t* full = is_q ? &bar_q : &bar_do;
        if (j > 0 && !wait(is_q ? &bar_qrel : &bar_dorel, (j - 1) & 1)) return false;
        mbar_arrive_expect_tx(full, C::TILE);
        for (int cb = 0; cb < C::NCB; ++cb)
          tma_load_3d(gen(sbase + (is_q ? C::Q_OFF : C::DO_OFF)) + cb * C::CB, is_q ? &m.Q[0] : &m.dO[0],
                      full, cb * C::ROW, it.i0, it.bh);
        last_qd = j;
        return true;
      };
      // Writer side of the item ring: entry k once every reader released entry k - IRING.
      auto publish = [&](int k, int w) {
        const int s = k % C::IRING;
        if (!wait(&bar_iempty[s], ((k / C::IRING) & 1) ^ 1)) return false;
        ring_w[s] = w;
        mbar_arrive(&bar_ifull[s]);
        return true;
      };
      const int G = (int)gridDim.x;
      int w = blockIdx.x;  // the first item is fixed; the next is fetched one item early
      int w_next = n_items > G ? G + atomicAdd(a.sched, 1) : n_items;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (!(ok = publish(k, w)) || w >= n_items) break;
        const Item it = item(w);
        w = w_next;
        if (w_next < n_items) w_next = G + atomicAdd(a.sched, 1);
        if (it.nc == 0) continue;
        const bool pre = j == 0 && setup_issued;  // Q / dO and chunk 0 came with the setup
        for (int c = 0; c < it.nc; ++c, ++g) {
          const int k0 = (it.kt_lo + c) * BLOCK_N;
          if (c == 0) {
            if (pre) { last_k[0] = last_v[0] = 0; continue; }
            // Q, K_0, dO first; V_0 goes where the previous epilogue staged its dQ
            if (!(ok = load_res(it, true) && load_k(g, k0, it.bg) && load_res(it, false))) break;
            if (j > 0 && !(ok = wait(&bar_vfree, (j - 1) & 1))) break;
            if (!(ok = load_v(g, k0, it.bg))) break;
          } else if (!(ok = load_k(g, k0, it.bg) && load_v(g, k0, it.bg))) {
            break;
          }
        }
        ++j;
      }
      // Drain: every issued copy must land before the CTA may exit.
      for (int s = 0; s < KST; ++s)
        if (last_k[s] >= 0) drain_wait(&bar_kfull[s], last_k[s] & 1, a.limit_ns);
      for (int s = 0; s < VST; ++s)
        if (last_v[s] >= 0) drain_wait(&bar_vfull[s], last_v[s] & 1, a.limit_ns);
      if (last_qd >= 0) {
        drain_wait(&bar_q, last_qd & 1, a.limit_ns);
        drain_wait(&bar_do, last_qd & 1, a.limit_ns);
      }
    }
  } else if (warp == C::MMA_WARP || warp == C::DP_WARP) {
    // Score issuers (one thread each): S(g) = Q K_g^T once the softmax has loaded
    // S(g-1); dP(g) = dO V_g^T once it has loaded dP(g-1).
    const bool is_s = warp == C::MMA_WARP;
    if (lane == 0) {
      bool ok = true;
      int g = 0, j = 0;  // chunks and items with keys so far
      for (int k = 0, w = take_thread(0); ok && w < n_items; w = take_thread(++k)) {
        const Item it = item(w);
        if (it.nc == 0) continue;
        if (!(ok = poll(is_s ? &bar_q : &bar_do, j & 1))) break;  // S needs Q, dP needs dO
        ++j;
        for (int c = 0; c < it.nc; ++c, ++g) {
          if (is_s) {
            const int ks = g % KST;
            if (!(ok = poll(&bar_kfull[ks], (g / KST) & 1))) break;
            if (g > 0 && !(ok = poll(&bar_sfree, (g - 1) & 1))) break;
            tc_fence_after();
            issue_rowdot128<D>(tmem + C::S_COL, sbase + C::Q_OFF, sK(ks));
            tc_commit(&bar_s);
          } else {
            const int vs = g % VST;
            if (!(ok = poll(&bar_vfull[vs], (g / VST) & 1))) break;
            if (g > 0 && !(ok = poll(&bar_dpfree, (g - 1) & 1))) break;
            tc_fence_after();
            issue_rowdot128<D>(tmem + C::DP_COL, sbase + C::DO_OFF, sV(vs));
            tc_commit(&bar_dp);
            tc_commit(&bar_vempty[vs]);
          }
        }
        // the item's Q (dO) buffer is free once its last S (dP) MMA has completed
        if (ok) tc_commit(is_s ? &bar_qrel : &bar_dorel);
      }
      tc_commit(&bar_drain[is_s ? 0 : 2]);
      drain_wait(&bar_drain[is_s ? 0 : 2], 0, a.limit_ns);
    }
  } else if (warp == C::ACC_WARP) {
    // Accumulate issuer: dQ += dS(g) K_g once the softmax has written dS(g); the
    // first chunk of an item also waits until the previous dQ left TMEM.
    if (lane == 0) {
      constexpr uint32_t id = make_idesc(128, D, FMT_F16, FMT_F16, false, true);
      bool ok = true;
      int g = 0, j = 0;  // chunks and items with keys so far
      for (int k = 0, w = take_thread(0); ok && w < n_items; w = take_thread(++k)) {
        const Item it = item(w);
        if (it.nc == 0) continue;
        for (int c = 0; c < it.nc; ++c, ++g) {
          const int pb = g & 1, ks = g % KST;
          if (!(ok = poll(&bar_ds[pb], (g >> 1) & 1))) break;
          if (c == 0 && j > 0 && !(ok = poll(&bar_dqfree, (j - 1) & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BLOCK_N / 16; ++kk)
            mma_f16_ts(tmem + C::ACC, tmem + C::DS_COL + 64 * pb + kk * 8,
                       make_sdesc(sK(ks) + kk * 16 * C::RB, C::CB, C::ATOM, C::SWZ), id,
                       (c > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&bar_kempty[ks]);
          tc_commit(&bar_accdone[pb]);
        }
        if (ok) tc_commit(&bar_done);  // the item's dQ is complete (one phase per item)
        ++j;
      }
      tc_commit(&bar_drain[1]);
      drain_wait(&bar_drain[1], 0, a.limit_ns);
    }
  }  // the idle warp falls through
  } else {
    regs_increase<C::REGS_SOFTMAX>();
    const int wq = warp % 4, half = warp / 4;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    // scores and dP come from the scaled fp16 copies: sl2 and dp_mul bring them back
    // (dP into the stored delta's units, which makes dS = 2^eD dS), dq_mul undoes 2^eD 2^eK
    const float sl2 = a.sc->sl2, dp_mul = a.sc->dp_mul, dq_mul = a.sc->dq_mul;
    bool ok = true;
    int g = 0, j = 0;  // chunks and items with keys so far
    for (int k = 0, w = take_warp(0); ok && w < n_items; w = take_warp(++k)) {
      const Item it = item(w);
      const int i = it.i0 + wq * 32 + lane;
      if (it.nc == 0) continue;  // no key for any row of the tile: zeroed by the launcher
      const bool row_valid = i < a.Sq;
      const size_t vrow = (size_t)it.bh * a.ldq + (size_t)(row_valid ? i : 0);
      const float nl = row_valid ? -a.lse2[vrow] : -INFINITY;
      const float dl = row_valid ? a.delta[vrow] : 0.f;
      const int hi_i = a.causal ? min(i, a.Sk - 1) : a.Sk - 1;
      const int lo_i = a.window > 0 ? i - a.window + 1 : INT_MIN / 2;
      for (int c = 0; c < it.nc; ++c, ++g) {
        const int pb = g & 1;
        const int kc0 = (it.kt_lo + c) * BLOCK_N;
        const int k0 = kc0 + half * 64;
        float s[64], dp[64];
        ok = __all_sync(0xffffffffu, wait(&bar_s, g & 1));
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t r0[32], r1[32];
          tmem_ld32x2(lane_addr + C::S_COL + half * 64, lane_addr + C::S_COL + half * 64 + 32, r0, r1);
          tc_fence_before();
          mbar_arrive(&bar_sfree);
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) {
            s[kk] = __uint_as_float(r0[kk]);
            s[32 + kk] = __uint_as_float(r1[kk]);
          }
        }
        if (tile_needs_mask(it.i0, it.i0 + BLOCK_M - 1, kc0, kc0 + BLOCK_N - 1, a.Sk, a.causal,
                            a.window)) {
          mask_outside<64>(s, lo_i - k0, hi_i - k0);
        }
        {
          const float2 sl2x2 = make_float2(sl2, sl2), nlx2 = make_float2(nl, nl);
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) {  // exponent arguments on packed pairs
            const float2 x = fma2(make_float2(s[2 * kk], s[2 * kk + 1]), sl2x2, nlx2);
            s[2 * kk] = ex2(x.x);
            s[2 * kk + 1] = ex2(x.y);
          }
        }
        ok = __all_sync(0xffffffffu, wait(&bar_dp, g & 1));
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t r0[32], r1[32];
          tmem_ld32x2(lane_addr + C::DP_COL + half * 64, lane_addr + C::DP_COL + half * 64 + 32, r0, r1);
          tc_fence_before();
          mbar_arrive(&bar_dpfree);
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) {
            dp[kk] = __uint_as_float(r0[kk]);
            dp[32 + kk] = __uint_as_float(r1[kk]);
          }
        }
        uint32_t pk[32];
        const float2 ndl = make_float2(-dl, -dl), dpm = make_float2(dp_mul, dp_mul);
#pragma unroll
        for (int kk = 0; kk < 32; ++kk) {  // dS = P (dP - delta) on packed pairs
          const float2 u = mul2(make_float2(s[2 * kk], s[2 * kk + 1]),
                                fma2(make_float2(dp[2 * kk], dp[2 * kk + 1]), dpm, ndl));
          pk[kk] = pack_half2(u.x, u.y);
        }
        // the dS slot is free once dQ += dS(g-2) K has completed
        if (g >= 2) {
          ok = __all_sync(0xffffffffu, wait(&bar_accdone[pb], ((g >> 1) - 1) & 1));
          if (!ok) break;
          tc_fence_after();
        }
        tmem_st32(lane_addr + C::DS_COL + 64 * pb + half * 32, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_ds[pb]);
      }
      if (!ok) break;
      // ---- epilogue of the item: dQ * scale, rows i0 + 32 (w % 4) .., warps w < 4 and
      // w >= 4 taking halves of the columns (bf16 at D = 64: warps w < 4 all of them).
      ok = __all_sync(0xffffffffu, wait(&bar_done, j & 1));
      if (!ok) break;
      tc_fence_after();
      ++j;
      const int r_base = it.i0 + wq * 32;
      const bool any = r_base < a.Sq;
      auto epilogue = [&](auto out_bf16_tag) {
        constexpr bool BF = decltype(out_bf16_tag)::value;
        // a bf16 box is a whole 64-column row, an fp32 one 32 columns: then the first half
        // of the warps stores everything
        constexpr bool ONE_HALF = (BF && D == 64) || (!BF && D == 32);
        constexpr int NCOL = ONE_HALF ? D : D / 2;
        const bool mine = !ONE_HALF || half == 0;
        const int x0 = ONE_HALF ? 0 : half * (D / 2);
        uint32_t r[NCOL];
        if (mine) {
          if constexpr (NCOL == 64) tmem_ld32x2(lane_addr + C::ACC + x0, lane_addr + C::ACC + x0 + 32,
                                                *reinterpret_cast<uint32_t(*)[32]>(&r[0]),
                                                *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          else tmem_ld32(lane_addr + C::ACC + x0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        }
        tc_fence_before();
        mbar_arrive(&bar_dqfree);  // dQ has left TMEM: the next item may accumulate
        // staging: the V ring, one warp's boxes after another
        constexpr uint32_t STG = (uint32_t)(NCOL * (BF ? 2 : 4) / 128) * EPI_BOX_BYTES;
        static_assert(8 * STG <= C::VST * C::TILE || (ONE_HALF && 4 * STG <= C::VST * C::TILE),
                      "epilogue staging");
        if (mine)
          stage_store_rows<NCOL, BF>(r, dq_mul, sbase + C::V_OFF + warp * STG,
                                     &m.dQ, x0, r_base, any,
                                     SPLIT ? (w % a.n_splits) * a.BHx + it.bh : it.bh, a.Dv);
      };
      // (bf16 outputs only in the D >= 64 kernels: the host routes smaller head dims there)
      if constexpr (D >= 64) {
        if (a.out_bf16) epilogue(std::true_type{});
        else epilogue(std::false_type{});
      } else {
        epilogue(std::false_type{});
      }
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      mbar_arrive(&bar_vfree);  // the staging area (the V ring) may be refilled
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // Launched as a programmatic dependent of the dK / dV grid: this grid completes
  // only after that one has (nothing above reads its results).
  grid_dependency_wait();
}

// ------------------------------------------------------ dK / dV, fp16 operands
// bf16 inputs: work item = (batch, kv head, 128-key tile), walked by persistent CTAs
// (one per SM); an item takes the 128-query chunks of every grouped query head that can
// see the tile, so the score MMAs are 128 x 128.
// TMEM: S^T slot [0, 128), dP^T slot [128, 256), dV, dK accumulators after them.
// Three issuers (a thread's MMAs run in issue order; an issuer stalls while the
// tensor pipe is full, so independent streams get their own thread):
//   S issuer:  S^T(c) = K Q_c^T as soon as the softmax has loaded S^T(c-1);
//   dV issuer: dV += P^T(c) dO_c, P^T (fp16) written by the softmax to shared memory;
//   B issuer:  dP^T(c) = V dO_c^T, then dK += dS^T(c) Q_c with dS^T (fp16) written
//              by the softmax into the first half of each 64-column half of its
//              slot, so dP^T(c+1) may overwrite the slot right after dK(c) is issued.
// P^T lives in shared memory so that the next score tile can enter the tensor pipe
// while the softmax is still exponentiating (in the S^T slot, which would make dV a TS
// product, S^T(c + 1) had to wait for dV(c): 11% slower at C3).
//
// SPLIT (short query sequences, where a few keys can take almost all of a row's
// weight and this kernel is bound by per-CTA set-up rather than by the tensor pipe):
// P and dS enter the accumulating products as two fp16 terms each, x = hi + lo with
// hi = fp16(x), lo = fp16(x - hi), i.e. about 22 significant bits instead of 11. P^T
// hi / lo go into the S^T slot the softmax has just read (dV += P^T dO becomes two TS
// MMAs, and the slot is freed by their commit instead of by the softmax's load), dS^T
// lo into the half of its part's dP^T range that dS^T hi leaves free (two dK MMAs).
template <int D>
struct Dkv16Cfg {
  static constexpr int RB = Dq16Cfg<D>::RB;             // (the same tile layout as dQ's)
  static constexpr uint32_t SWZ = Dq16Cfg<D>::SWZ, ATOM = Dq16Cfg<D>::ATOM;
  static constexpr int ROW = Dq16Cfg<D>::ROW;
  static constexpr int NCB = D / ROW;
  static constexpr uint32_t CB = 128u * RB;
  static constexpr uint32_t PT_CB = 128u * 128u;        // column block of the P^T tile
  static constexpr uint32_t TILE = NCB * CB;            // 128 rows x D fp16
  static constexpr int NS = D == 128 ? 2 : 3;           // Q and dO ring depth
  static constexpr uint32_t K_OFF = 0, V_OFF = TILE, Q_OFF = 2 * TILE;
  static constexpr uint32_t DO_OFF = Q_OFF + NS * TILE;
  static constexpr uint32_t PT_OFF = DO_OFF + NS * TILE;  // P^T: 128 keys x 128 queries fp16
  static constexpr uint32_t VEC = 2 * 128 * 4;            // lse2 | delta of a chunk
  static constexpr uint32_t VEC_OFF = PT_OFF + 2 * PT_CB;
  static constexpr uint32_t LAYOUT = VEC_OFF + NS * VEC;  // bytes from the 1 KB-aligned base
  // NPART softmax warps share each TMEM lane quarter, each taking QC = 128 / NPART
  // of the chunk's queries: more warps per SM sub-partition hide more latency.
  static constexpr int NPART = 2, QC = 128 / NPART;
  static constexpr int SOFTMAX_WARPS = 4 * NPART;
  static constexpr int A_WARP = SOFTMAX_WARPS, B_WARP = A_WARP + 1, TMA_WARP = A_WARP + 2,
                       DV_WARP = A_WARP + 3;
  static constexpr int THREADS = 32 * (SOFTMAX_WARPS + 4);
  static constexpr int SM_THREADS = 32 * SOFTMAX_WARPS;
  // The softmax barriers take one arrival per warp (lane 0, after every lane's fence
  // and a warp sync): 32x fewer shared-memory atomics than one per thread.
  static constexpr int SM_ARRIVALS = SOFTMAX_WARPS;
  static constexpr uint32_t REGS_LAUNCH = (65536 / THREADS) / 8 * 8;
  static constexpr uint32_t REGS_SOFTMAX = NPART == 4 ? 104 : 200;
  static constexpr uint32_t REGS_CONTROL = NPART == 4 ? 64 : 96;
  static_assert(SM_THREADS * REGS_SOFTMAX + 128 * REGS_CONTROL <= THREADS * REGS_LAUNCH,
                "register split");
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DV = 256, DK = 256 + D;
  static constexpr uint32_t EPI_WARP = epi_warp_bytes<D, false>();
  // 227 KB per block minus the alignment of the base to 1 KB leaves 226 KB.
  static_assert(LAYOUT <= 226u * 1024u, "shared memory budget");
  static_assert(DK + D <= TMEM_COLS, "TMEM budget");
  static_assert(SOFTMAX_WARPS * (EPI_WARP * 2 / NPART) <= VEC_OFF, "epilogue staging");
  // fp16 dS^T column of k-step kk (16 queries): each part writes its QC / 2 packed
  // columns at the start of its own QC-column range of the dP^T slot.
  __host__ __device__ static constexpr uint32_t op_col(int kk) {
    return (kk / (QC / 16)) * QC + (kk % (QC / 16)) * 8;
  }
};

// ACC[128 x D] (+)= A(TMEM fp16, 128 x 128, halves at columns 0 / 64) * B[128 x D]
// (MN-major fp16 tile in smem).
template <int D>
__device__ __forceinline__ void issue_acc128(uint32_t acc, uint32_t a_tmem, uint32_t b,
                                             bool accumulate) {
  using L = Dkv16Cfg<D>;
  constexpr uint32_t id = make_idesc(128, D, FMT_F16, FMT_F16, false, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_f16_ts(acc, a_tmem + L::op_col(kk), make_sdesc(b + kk * 16 * L::RB, L::CB, L::ATOM, L::SWZ),
               id, (accumulate || kk > 0) ? 1u : 0u);
}

// ACC[128 x D] (+)= A[128 x 128] (K-major fp16 tile in smem) * B[128 x D] (MN-major).
template <int D>
__device__ __forceinline__ void issue_acc128_ss(uint32_t acc, uint32_t a, uint32_t b,
                                                bool accumulate) {
  using L = Dkv16Cfg<D>;
  constexpr uint32_t id = make_idesc(128, D, FMT_F16, FMT_F16, false, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    // A: the P^T tile (128-byte rows whatever D); B: the MN-major dO chunk
    const uint32_t off = (kk * 16 / 64) * L::PT_CB + (kk * 16 % 64) * 2;
    mma_f16_ss(acc, make_sdesc(a + off, 16, SW128_ATOM),
               make_sdesc(b + kk * 16 * L::RB, L::CB, L::ATOM, L::SWZ), id,
               (accumulate || kk > 0) ? 1u : 0u);
  }
}

// x = hi + lo for a pair of floats, both terms fp16 (packed as one 32-bit word each):
// hi = fp16(x), lo = fp16(x - hi)
__device__ __forceinline__ void split_half2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// MATDS (the materialised-dS backward): the softmax also stores every dS^T row it
// forms (this thread's key j, its part's QC queries: 2 QC bytes per term) to a.ds_hi
// (and a.ds_lo), from which dq_from_ds_kernel forms dQ = scale dS K as a GEMM instead
// of recomputing S and dP.
template <int D, bool SPLIT, bool MATDS, bool QSPLIT = false>
__global__ void __launch_bounds__(Dkv16Cfg<D>::THREADS, 1)
    fa_bwd_dkdv16_kernel(const __grid_constant__ KVMaps m, const BwdArgs a) {
  using C = Dkv16Cfg<D>;
  constexpr int NS = C::NS;
  static_assert(!SPLIT || C::QC == 64, "two-term operands: 32 packed columns per term and part");
  static_assert(!MATDS || C::QC == 64, "dS^T rows stored as 128-byte pieces");
  // A programmatic dependent of the kernel that fixed the operand copies' scales (and may
  // have rewritten the copies): wait for it first. The dQ grid launched after this one
  // reads those copies and nothing this grid writes: it may start once every block of
  // this grid has passed that wait (see the launcher).
  grid_dependency_wait();
  grid_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_kv, bar_kvfree, bar_qfull[NS], bar_qempty[NS], bar_dofull[NS],
      bar_doempty[NS], bar_s, bar_sfree, bar_p, bar_dvdone, bar_dp, bar_ds, bar_done, bar_drain[3];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  {
    // The layout needs LAYOUT bytes above the 1 KB-aligned base; the launch asks
    // for as much dynamic shared memory as the block may have.
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (smem_u32(smem) + C::LAYOUT > smem_u32(smem_raw) + dyn) {
      if (threadIdx.x == 0) atomicOr(&g_bwd_status, DEV_LAYOUT);
      return;
    }
  }
  const int warp = warp_id(), lane = lane_id();
  volatile int* abort_flag = &abort_sh;
  const int rep = a.H / a.HKV;

  // ---- work items: key tile jt of (batch, kv head) bg, w = jt * BHx + bg, so key
  // tile 0 -- which, under a causal mask, the most queries see -- comes first. Each
  // CTA walks items in rounds of gridDim.x, item c of even rounds and G - 1 - c of odd
  // ones (one round when the grid has a CTA per item). (A host-side longest-first
  // assignment to the least loaded CTA measured 1-3% slower than these rounds.)
  // QSPLIT (fewer (kv head, key tile) items than SMs: short key sequences): the queries
  // are also split into a.n_splits ranges of a.tps query tiles, item w = (jt * BHx + bg)
  // * n_splits + range, each writing partial dK, dV to slab range * BHx + bg (z). (A
  // template flag: the unsplit kernel stays exactly as it was, which a runtime flag did
  // not -- it cost the C3 dK / dV kernel 2%.)
  const int n_qs = QSPLIT ? a.n_splits : 1;
  const int n_items = a.n_tiles * a.BHx * n_qs;
  struct Item { int bg, b, g, j0, qt_lo, ncq, nc, z; };
  auto item = [&](int w) {
    Item it;
    int qs = 0, wk = w;
    if constexpr (QSPLIT) {
      qs = w % n_qs;
      wk = w / n_qs;
    }
    const int jt = wk / a.BHx;
    it.bg = wk % a.BHx;
    it.b = it.bg / a.HKV;
    it.g = it.bg % a.HKV;
    it.j0 = jt * BLOCK_N;
    int qt_hi;
    q_tile_range(it.j0, min(it.j0 + BLOCK_N - 1, a.Sk - 1), a.Sq, a.causal, a.window, &it.qt_lo, &qt_hi);
    if constexpr (QSPLIT) {
      it.qt_lo = max(it.qt_lo, qs * a.tps);
      qt_hi = min(qt_hi, (qs + 1) * a.tps);
      if (qt_hi < it.qt_lo) qt_hi = it.qt_lo;
    }
    it.ncq = qt_hi - it.qt_lo;
    it.nc = rep * it.ncq;
    it.z = QSPLIT ? qs * a.BHx + it.bg : it.bg;
    return it;
  };
  auto item_w = [&](int k) {
    const int G = gridDim.x, c = blockIdx.x;
    return k * G + ((k & 1) ? G - 1 - c : c);
  };
  auto chunk_rows = [&](const Item& it, int c, int* bh, int* i0) {
    const int r = c / it.ncq, qt = it.qt_lo + c % it.ncq;
    *bh = it.b * a.H + it.g * rep + r;
    *i0 = qt * BLOCK_M;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bar_kv, 1);
    mbar_init(&bar_kvfree, 2);  // the S and the B issuer: an item's last S^T / dP^T read K / V
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_qfull[s], 1);
      mbar_init(&bar_qempty[s], 2);   // S^T(c) (A) and dK(c) (B) have read Q_c
      mbar_init(&bar_dofull[s], 1);
      mbar_init(&bar_doempty[s], 2);  // dP^T(c) (B) and dV(c) (A) have read dO_c
    }
    mbar_init(&bar_s, 1);
    // the S^T slot is freed by the softmax's load, or (SPLIT) by the dV MMAs that read
    // P^T from it
    mbar_init(&bar_sfree, SPLIT ? 1 : C::SM_ARRIVALS);
    mbar_init(&bar_p, C::SM_ARRIVALS);
    mbar_init(&bar_dvdone, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_ds, C::SM_ARRIVALS);
    mbar_init(&bar_done, 2);  // dV issuer and B issuer, one phase per item with chunks
    for (int s = 0; s < 3; ++s) mbar_init(&bar_drain[s], 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == C::A_WARP) {
    __syncwarp();
    tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t sbase = smem_u32(smem);
  auto sQ = [&](int st) { return sbase + C::Q_OFF + st * C::TILE; };
  auto sdO = [&](int st) { return sbase + C::DO_OFF + st * C::TILE; };
  auto gen = [&](uint32_t s) { return smem + (s - sbase); };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };
  // (the issuers' waits for the softmax's hand-offs poll instead of suspending: they sit
  // on the per-chunk critical path)
  auto poll = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait_poll(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };
  // Chunk barriers count chunks across items (g); bar_kv, bar_kvfree and bar_done
  // count items with chunks (j). Every phase of a per-item barrier needs the previous
  // one observed first (K / V of item j load after kv_free(j - 1), whose commits follow
  // waits on bar_kv(j - 1); done(j) needs this item's P^T / dS^T, written after the
  // epilogue waited on done(j - 1)), so no parity wait can miss a phase. The first dV
  // and dK MMAs of an item overwrite the accumulators only after the softmax wrote that
  // item's first P^T / dS^T, i.e. after its epilogue read the previous item's out of
  // TMEM.

  if (warp >= C::SOFTMAX_WARPS) {
  regs_decrease<C::REGS_CONTROL>();
  if (warp == C::TMA_WARP) {
    if (lane == 0) {
      int last_q[NS], last_do[NS], last_kv = -1;
      for (int s = 0; s < NS; ++s) last_q[s] = last_do[s] = -1;
      bool ok = true;
      int g = 0, j = 0;
      for (int k = 0, w = item_w(0); ok && w < n_items; w = item_w(++k)) {
        const Item it = item(w);
        if (it.nc == 0) continue;
        // K / V of this item once the previous item's last S^T and dP^T have read them
        if (j > 0 && !(ok = wait(&bar_kvfree, (j - 1) & 1))) break;
        mbar_arrive_expect_tx(&bar_kv, 2 * C::TILE);
        for (int cb = 0; cb < C::NCB; ++cb) {
          tma_load_3d(smem + C::K_OFF + cb * C::CB, &m.K[0], &bar_kv, cb * C::ROW, it.j0, it.bg);
          tma_load_3d(smem + C::V_OFF + cb * C::CB, &m.V[0], &bar_kv, cb * C::ROW, it.j0, it.bg);
        }
        last_kv = j;
        for (int c = 0; c < it.nc; ++c, ++g) {
          const int st = g % NS;
          int bh, i0;
          chunk_rows(it, c, &bh, &i0);
          if (!(ok = wait(&bar_doempty[st], ((g / NS) & 1) ^ 1))) break;
          mbar_arrive_expect_tx(&bar_dofull[st], C::TILE);
          for (int cb = 0; cb < C::NCB; ++cb)
            tma_load_3d(gen(sdO(st)) + cb * C::CB, &m.dOc[0], &bar_dofull[st], cb * C::ROW, i0, bh);
          last_do[st] = g / NS;
          if (!(ok = wait(&bar_qempty[st], ((g / NS) & 1) ^ 1))) break;
          mbar_arrive_expect_tx(&bar_qfull[st], C::TILE + C::VEC);
          for (int cb = 0; cb < C::NCB; ++cb)
            tma_load_3d(gen(sQ(st)) + cb * C::CB, &m.Qc[0], &bar_qfull[st], cb * C::ROW, i0, bh);
          float* vec = reinterpret_cast<float*>(smem + C::VEC_OFF + st * C::VEC);
          tma_load_3d(vec, &m.L, &bar_qfull[st], i0, bh, 0);
          tma_load_3d(vec + 128, &m.Dl, &bar_qfull[st], i0, bh, 0);
          last_q[st] = g / NS;
        }
        ++j;
      }
      // Drain: every issued copy must land before the CTA may exit.
      if (last_kv >= 0) drain_wait(&bar_kv, last_kv & 1, a.limit_ns);
      for (int s = 0; s < NS; ++s) {
        if (last_q[s] >= 0) drain_wait(&bar_qfull[s], last_q[s] & 1, a.limit_ns);
        if (last_do[s] >= 0) drain_wait(&bar_dofull[s], last_do[s] & 1, a.limit_ns);
      }
    }
  } else if (warp == C::A_WARP) {
    // S issuer: S^T(c) once Q_c is in and the softmax has loaded S^T(c-1).
    if (lane == 0) {
      bool ok = true;
      int g = 0, j = 0;
      for (int k = 0, w = item_w(0); ok && w < n_items; w = item_w(++k)) {
        const Item it = item(w);
        if (it.nc == 0) continue;
        if (!(ok = wait(&bar_kv, j & 1))) break;
        for (int c = 0; c < it.nc; ++c, ++g) {
          const int st = g % NS;
          if (!(ok = poll(&bar_qfull[st], (g / NS) & 1))) break;
          if (g > 0 && !(ok = poll(&bar_sfree, (g - 1) & 1))) break;
          tc_fence_after();
          issue_rowdot128<D>(tmem + C::S_COL, sbase + C::K_OFF, sQ(st));
          tc_commit(&bar_s);
          tc_commit(&bar_qempty[st]);
        }
        tc_commit(&bar_kvfree);  // this item's S^T MMAs are done with K
        ++j;
      }
      tc_commit(&bar_drain[0]);
      drain_wait(&bar_drain[0], 0, a.limit_ns);
    }
  } else if (warp == C::DV_WARP) {
    // dV issuer: dV += P^T(c) dO_c once the softmax has written P^T(c); the softmax
    // observed dO_c land before that (an mbarrier wait here, right after this warp's
    // previous MMAs, would wait for them to drain: +4% kernel time).
    if (lane == 0) {
      bool ok = true;
      int g = 0;
      for (int k = 0, w = item_w(0); ok && w < n_items; w = item_w(++k)) {
        const Item it = item(w);
        if (it.nc == 0) continue;
        for (int c = 0; c < it.nc; ++c, ++g) {
          const int st = g % NS;
          if (!(ok = poll(&bar_p, g & 1))) break;
          tc_fence_after();
          if constexpr (SPLIT) {
            // P^T hi and lo from the S^T slot, which S^T(c + 1) may take once both are read
            issue_acc128<D>(tmem + C::DV, tmem + C::S_COL, sdO(st), c > 0);
            issue_acc128<D>(tmem + C::DV, tmem + C::S_COL + C::QC / 2, sdO(st), true);
            tc_commit(&bar_doempty[st]);
            tc_commit(&bar_sfree);
          } else {
            issue_acc128_ss<D>(tmem + C::DV, sbase + C::PT_OFF, sdO(st), c > 0);
            tc_commit(&bar_doempty[st]);
            tc_commit(&bar_dvdone);
          }
        }
        if (ok) tc_commit(&bar_done);
      }
      tc_commit(&bar_drain[2]);
      drain_wait(&bar_drain[2], 0, a.limit_ns);
    }
  } else if (warp == C::B_WARP) {
    // Chunk c: dP^T(c) = V dO^T, then dK += dS^T(c) Q once the softmax wrote dS^T(c).
    if (lane == 0) {
      bool ok = true;
      int g = 0, j = 0;
      for (int k = 0, w = item_w(0); ok && w < n_items; w = item_w(++k)) {
        const Item it = item(w);
        if (it.nc == 0) continue;
        if (!(ok = wait(&bar_kv, j & 1))) break;
        for (int c = 0; c < it.nc; ++c, ++g) {
          const int st = g % NS;
          if (!(ok = poll(&bar_dofull[st], (g / NS) & 1))) break;
          tc_fence_after();
          issue_rowdot128<D>(tmem + C::DP_COL, sbase + C::V_OFF, sdO(st));
          tc_commit(&bar_dp);
          tc_commit(&bar_doempty[st]);
          if (c + 1 == it.nc) tc_commit(&bar_kvfree);  // the item's last dP^T read V
          if (!(ok = poll(&bar_ds, g & 1))) break;
          tc_fence_after();
          issue_acc128<D>(tmem + C::DK, tmem + C::DP_COL, sQ(st), c > 0);
          if constexpr (SPLIT) issue_acc128<D>(tmem + C::DK, tmem + C::DP_COL + C::QC / 2, sQ(st), true);
          tc_commit(&bar_qempty[st]);
        }
        if (ok) tc_commit(&bar_done);
        ++j;
      }
      tc_commit(&bar_drain[1]);
      drain_wait(&bar_drain[1], 0, a.limit_ns);
    }
  }
  } else {
    regs_increase<C::REGS_SOFTMAX>();
    // thread = key row j = TMEM lane; warp w takes queries [QC p, QC p + QC), p = w / 4
    constexpr int QC = C::QC;
    const int wq = warp % 4, part = warp / 4;
    const int r_in = wq * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    // this thread's QC queries of row r_in of the swizzled P^T tile: column block
    // (QC p) / 64, 16-byte chunks from (QC p % 64) / 8
    const uint32_t pt_row = sbase + C::PT_OFF + (QC * part / 64) * C::PT_CB + r_in * 128;
    const uint32_t chunk0 = (uint32_t)((QC * part % 64) / 8);
    const uint32_t sw = (uint32_t)(r_in & 7);
    // scores and dP^T come from the scaled fp16 copies (see the dQ kernel)
    const float sl2 = a.sc->sl2, dp_mul = a.sc->dp_mul;
    auto ld_cols = [&](uint32_t addr, float (&x)[QC]) {
      if constexpr (QC == 64) {
        uint32_t r0[32], r1[32];
        tmem_ld32x2(addr, addr + 32, r0, r1);
#pragma unroll
        for (int k = 0; k < 32; ++k) { x[k] = __uint_as_float(r0[k]); x[32 + k] = __uint_as_float(r1[k]); }
      } else {
        uint32_t r0[32];
        tmem_ld32(addr, r0);
#pragma unroll
        for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(r0[k]);
      }
    };
    bool ok = true;
    int g = 0, jj = 0;  // chunks and items with chunks so far
    for (int k = 0, w = item_w(0); ok && w < n_items; w = item_w(++k)) {
      const Item it = item(w);
      const int j0 = it.j0;
      const int j = j0 + r_in;  // this thread's key row
      const bool row_dead = j >= a.Sk;
      for (int c = 0; c < it.nc; ++c, ++g) {
        const int st = g % NS;
        int bh, i0;
        chunk_rows(it, c, &bh, &i0);
        const int q0 = i0 + part * QC;  // first query of this thread's part
        float s[QC];
        // S^T(c) and chunk c's vectors; and dO_c, so that the dV MMA issued once P^T(c)
        // is written reads a landed tile (nothing else orders it after that copy)
        ok = __all_sync(0xffffffffu, wait(&bar_s, g & 1) && wait(&bar_qfull[st], (g / NS) & 1) &&
                                         wait(&bar_dofull[st], (g / NS) & 1));
        if (!ok) break;
        tc_fence_after();
        ld_cols(lane_addr + C::S_COL + part * QC, s);
        tc_fence_before();
        __syncwarp();
        if constexpr (!SPLIT)
          if (lane == 0) mbar_arrive(&bar_sfree);  // the S^T slot may take the next chunk
        // query i = q0 + k sees key j iff (!causal || j <= i) && (!window || j >= i-w+1)
        // && i < Sq && j < Sk
        if (tile_needs_mask(i0, i0 + BLOCK_M - 1, j0, j0 + BLOCK_N - 1, a.Sk, a.causal, a.window) ||
            i0 + BLOCK_M > a.Sq) {
          const int k_lo = a.causal ? j - q0 : INT_MIN / 2;
          const int k_hi = min(a.window > 0 ? j + a.window - 1 - q0 : INT_MAX / 2, a.Sq - 1 - q0);
          mask_outside<QC>(s, row_dead ? INT_MAX / 2 : k_lo, k_hi);
        }
        // lse2 / delta of the chunk's queries, read with explicit shared-space loads
        const uint32_t lv = sbase + C::VEC_OFF + st * C::VEC + part * QC * 4;
        const float2 sl2x2 = make_float2(sl2, sl2);
#pragma unroll
        for (int k4 = 0; k4 < QC / 4; ++k4) {  // exponent arguments on packed pairs
          const float4 l4 = ld_shared_v4(lv + 16 * k4);
          const float2 xa = fma2(make_float2(s[4 * k4], s[4 * k4 + 1]), sl2x2, make_float2(-l4.x, -l4.y));
          const float2 xb = fma2(make_float2(s[4 * k4 + 2], s[4 * k4 + 3]), sl2x2, make_float2(-l4.z, -l4.w));
          s[4 * k4] = ex2(xa.x);
          s[4 * k4 + 1] = ex2(xa.y);
          s[4 * k4 + 2] = ex2(xb.x);
          s[4 * k4 + 3] = ex2(xb.y);
        }
        if constexpr (SPLIT) {
          // P^T hi / lo over the S^T columns this thread has just read: hi in the first
          // QC / 2 packed columns of its part's range, lo in the other QC / 2
          uint32_t ph[QC / 2], pl[QC / 2];
#pragma unroll
          for (int kq = 0; kq < QC / 2; ++kq) split_half2(s[2 * kq], s[2 * kq + 1], ph[kq], pl[kq]);
          tmem_st32(lane_addr + C::S_COL + part * QC, ph);
          tmem_st32(lane_addr + C::S_COL + part * QC + QC / 2, pl);
          tmem_st_wait();
          tc_fence_before();
        } else {
          // P^T into shared memory once dV has consumed the previous chunk's
          if (g > 0) {
            ok = __all_sync(0xffffffffu, wait(&bar_dvdone, (g - 1) & 1));
            if (!ok) break;
          }
#pragma unroll
          for (int k8 = 0; k8 < QC / 8; ++k8)
            st_shared_v4(pt_row + (((chunk0 + (uint32_t)k8) ^ sw) << 4), pack_half2(s[8 * k8], s[8 * k8 + 1]),
                         pack_half2(s[8 * k8 + 2], s[8 * k8 + 3]), pack_half2(s[8 * k8 + 4], s[8 * k8 + 5]),
                         pack_half2(s[8 * k8 + 6], s[8 * k8 + 7]));
          fence_async_shared();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p);
        // dP^T(c) closes the per-chunk cycle (dS^T(c - 1) -> dK -> dP^T(c) -> dS^T(c)).
        // Two-term P: lane 0 polls, then every lane observes the completed phase (short
        // items, decode-shaped: -4% kernel time); one term: a suspending wait (polled,
        // +1.5% at long items, where the polls take issue slots from the issuers)
        {
          bool got = true;
          if (SPLIT && lane == 0) got = poll(&bar_dp, g & 1);
          got = __shfl_sync(0xffffffffu, got, 0) && wait(&bar_dp, g & 1);
          ok = __all_sync(0xffffffffu, got);
        }
        if (!ok) break;
        tc_fence_after();
        {
          float gd[QC];
          ld_cols(lane_addr + C::DP_COL + part * QC, gd);
          const uint32_t dv = lv + 128 * 4;
          const float2 dpm = make_float2(dp_mul, dp_mul);
          uint32_t pk[QC / 2], pl[SPLIT ? QC / 2 : 1];
#pragma unroll
          for (int k4 = 0; k4 < QC / 4; ++k4) {
            const float4 d4 = ld_shared_v4(dv + 16 * k4);
            const int kq = 4 * k4;
            // dS = P (dP - delta) on packed pairs
            const float2 ua = mul2(make_float2(s[kq], s[kq + 1]),
                                   fma2(make_float2(gd[kq], gd[kq + 1]), dpm, make_float2(-d4.x, -d4.y)));
            const float2 ub = mul2(make_float2(s[kq + 2], s[kq + 3]),
                                   fma2(make_float2(gd[kq + 2], gd[kq + 3]), dpm, make_float2(-d4.z, -d4.w)));
            if constexpr (SPLIT) {
              split_half2(ua.x, ua.y, pk[2 * k4], pl[2 * k4]);
              split_half2(ub.x, ub.y, pk[2 * k4 + 1], pl[2 * k4 + 1]);
            } else {
              pk[2 * k4] = pack_half2(ua.x, ua.y);
              pk[2 * k4 + 1] = pack_half2(ub.x, ub.y);
            }
          }
          // dS^T (fp16) into the first QC / 2 columns of this part's own dP^T range
          // (SPLIT: dS^T lo into the other QC / 2)
          if constexpr (QC == 64) tmem_st32(lane_addr + C::DP_COL + part * QC, pk);
          else tmem_st16(lane_addr + C::DP_COL + part * QC, pk);
          if constexpr (SPLIT) tmem_st32(lane_addr + C::DP_COL + part * QC + QC / 2, pl);
          if constexpr (MATDS) {
            // dS^T row j, queries q0 .. q0 + QC - 1 (padding queries carry P = 0, so 0)
            if (!row_dead) {
              const size_t off = ((size_t)bh * a.Sk + j) * a.ldq + q0;
              // QC halves = QC / 8 vectors of 16 bytes (4 packed pairs each)
              uint4* dh = reinterpret_cast<uint4*>(a.ds_hi + off);
#pragma unroll
              for (int v = 0; v < QC / 8; ++v)
                dh[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
              if constexpr (SPLIT) {
                uint4* dl = reinterpret_cast<uint4*>(a.ds_lo + off);
#pragma unroll
                for (int v = 0; v < QC / 8; ++v)
                  dl[v] = make_uint4(pl[4 * v], pl[4 * v + 1], pl[4 * v + 2], pl[4 * v + 3]);
              }
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_ds);
      }
      if (!ok) break;
      if (it.nc > 0) {
        ok = __all_sync(0xffffffffu, wait(&bar_done, jj & 1));
        if (!ok) break;
        tc_fence_after();
        ++jj;
      }
      // ---- epilogue of the item: every MMA of it has completed (an item without
      // chunks writes zeros). Parts 0 .. NPART/2-1 write dV, the others dK; each part D /
      // (NPART / 2) columns of rows j0 + 32 (w % 4) ... The stores are staged in the P^T
      // tile, one 32 x 128-byte box per warp at a time (the other buffers may already
      // hold the next item's tiles); it is free here (the item's dV MMAs are done) and
      // this thread writes the next P^T only after its stores have read it.
      constexpr int HP = C::NPART / 2;     // parts per output
      constexpr int DW = D / HP;           // columns per warp
      const int which = part / HP, cpart = part % HP;
      const int r_base = j0 + wq * 32;
      const bool any = r_base < a.Sk;
      const uint32_t acc = lane_addr + (which ? C::DK : C::DV) + cpart * DW;
      const CUtensorMap* tm = which ? &m.dK : &m.dV;
      const float mul = which ? a.sc->dk_mul : a.sc->dv_mul;  // scale 2^-(eD+eQ) / 2^-eO
      const uint32_t stage = sbase + C::PT_OFF + warp * EPI_BOX_BYTES;
      static_assert(C::SOFTMAX_WARPS * EPI_BOX_BYTES <= 2 * C::PT_CB, "epilogue staging");
      if (D >= 64 && a.out_bf16) {  // (bf16 outputs: D >= 64 kernels only)
        if constexpr (D >= 64) {
          if constexpr (DW % 64 == 0) {
            store_rows_tma<DW, true, 1>(tm, acc, it.nc > 0, mul, stage, r_base, any, it.z, cpart * DW,
                                        a.Dv);
          } else {
            // a bf16 box is a 64-column row: one warp per output does it
            if (cpart == 0)
              store_rows_tma<D, true, 1>(tm, lane_addr + (which ? C::DK : C::DV), it.nc > 0, mul, stage,
                                         r_base, any, it.z, 0, a.Dv);
          }
        }
      } else {
        store_rows_tma<DW, false, 1>(tm, acc, it.nc > 0, mul, stage, r_base, any, it.z, cpart * DW, a.Dv);
      }
      tc_fence_before();  // (the accumulator loads precede every later hand-off)
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::A_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------- dQ from the materialised dS
// The materialised-dS backward (metal-flash-attention README, backward pass: dS written
// to memory, so that dQ is a plain GEMM instead of a second recomputation of S and
// dP): dQ_i = scale sum_j dS_ij K_j over the key tiles query tile i can see, dS read
// from the [B*H][Sk][ldq] buffer the MATDS dK / dV kernel wrote (hi and, two-term, lo).
// One CTA per (head, 128-query tile) -- and key range: with fewer (head, query tile)
// items than SMs the keys are split into ranges of a.tps tiles, each CTA writing a
// partial dQ (fp32) that dq_range_sum_kernel adds up in range order, as for the
// recompute dQ kernel -- heaviest causal tiles first. Roles: warp 0 the
// TMA producer (a ring of NST stages, each the dS tile(s) and the K tile of one key
// tile), warp 1 the MMA issuer and TMEM owner, warps 2-5 the epilogue (one TMEM lane
// quarter each). The dS tile is stored key-major (queries fastest), which is the
// MN-major layout of the A operand [128 queries x 128 keys].
template <int D, bool SPLIT>
struct DqGemmCfg {
  static constexpr int NCB = D / 64;
  static constexpr uint32_t CB = 128u * 128u;  // 128 rows x 128 bytes
  static constexpr uint32_t A_TILE = 2 * CB;   // dS: 128 keys x 128 queries fp16
  static constexpr uint32_t B_TILE = NCB * CB; // K: 128 keys x D fp16
  static constexpr int NA = SPLIT ? 2 : 1;
  static constexpr uint32_t STAGE = NA * A_TILE + B_TILE;
  static constexpr int NST = (int)((200u * 1024u) / STAGE) < 4 ? (int)((200u * 1024u) / STAGE) : 4;
  static constexpr uint32_t SMEM = NST * STAGE + 1024;
  static constexpr int THREADS = 192;
  static constexpr int TMA_WARP = 0, MMA_WARP = 1;
  static constexpr uint32_t TMEM_COLS = D;  // the dQ accumulator
  static_assert(NST >= 2 && SMEM <= 227u * 1024u, "shared memory budget");
  static constexpr uint32_t EPI_WARP = epi_warp_bytes<D, false>();
  static_assert(4 * EPI_WARP <= NST * STAGE, "epilogue staging");
};

struct DsMaps {
  CUtensorMap ds_hi, ds_lo, K, dQ;
};

template <int D, bool SPLIT>
__global__ void __launch_bounds__(DqGemmCfg<D, SPLIT>::THREADS, 1)
    dq_from_ds_kernel(const __grid_constant__ DsMaps m, const BwdArgs a) {
  using C = DqGemmCfg<D, SPLIT>;
  constexpr int NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_full[NST], bar_empty[NST], bar_done, bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = warp_id(), lane = lane_id();
  volatile int* abort_flag = &abort_sh;

  const int sp = blockIdx.x % a.n_splits, w = blockIdx.x / a.n_splits;
  const int qt_lin = w / a.BHx, bh = w % a.BHx;
  const int qt = a.lpt ? a.n_tiles - 1 - qt_lin : qt_lin;
  const int i0 = qt * BLOCK_M;
  const int b = bh / a.H, h = bh % a.H;
  const int bg = b * a.HKV + h / (a.H / a.HKV);
  int kt_lo, kt_hi;
  kv_tile_range(i0, min(i0 + BLOCK_M - 1, a.Sq - 1), a.Sk, a.causal, a.window, &kt_lo, &kt_hi);
  if (a.n_splits > 1) {
    kt_lo = max(kt_lo, sp * a.tps);
    kt_hi = min(kt_hi, (sp + 1) * a.tps);
  }
  const int n = kt_hi > kt_lo ? kt_hi - kt_lo : 0;
  const int zo = sp * a.BHx + bh;  // output slab: dQ itself, or range sp's partial dQ

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
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
  auto stage = [&](int st) { return sbase + st * C::STAGE; };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait(bar, parity, abort_flag, &g_bwd_status, DEV_TIMEOUT, a.limit_ns);
  };

  if (warp == C::TMA_WARP) {
    if (lane == 0) {
      int loads[NST];
      for (int s = 0; s < NST; ++s) loads[s] = 0;
      for (int t = 0; t < n; ++t) {
        const int st = t % NST, k0 = (kt_lo + t) * BLOCK_N;
        if (t >= NST && !wait(&bar_empty[st], ((t / NST) - 1) & 1)) break;
        mbar_arrive_expect_tx(&bar_full[st], C::STAGE);
        uint8_t* dst = smem + st * C::STAGE;
        for (int blk = 0; blk < 2; ++blk) {  // the tile's two 64-query blocks
          tma_load_3d(dst + blk * C::CB, &m.ds_hi, &bar_full[st], i0 + 64 * blk, k0, bh);
          if constexpr (SPLIT)
            tma_load_3d(dst + C::A_TILE + blk * C::CB, &m.ds_lo, &bar_full[st], i0 + 64 * blk, k0, bh);
        }
        for (int cb = 0; cb < C::NCB; ++cb)
          tma_load_3d(dst + C::NA * C::A_TILE + cb * C::CB, &m.K, &bar_full[st], cb * 64, k0, bg);
        ++loads[st];
      }
      // every issued copy must land before the CTA may exit
      for (int s = 0; s < NST; ++s)
        if (loads[s] > 0) drain_wait(&bar_full[s], (loads[s] - 1) & 1, a.limit_ns);
    }
  } else if (warp == C::MMA_WARP) {
    if (lane == 0) {
      // A = dS [128 queries x 128 keys], MN-major (queries fastest); B = K [128 keys x D],
      // MN-major; 16 keys per MMA
      constexpr uint32_t id = make_idesc(128, D, FMT_F16, FMT_F16, true, true);
      bool ok = true;
      for (int t = 0; t < n; ++t) {
        const int st = t % NST;
        if (!(ok = wait(&bar_full[st], (t / NST) & 1))) break;
        tc_fence_after();
        const uint32_t sb = stage(st) + C::NA * C::A_TILE;
#pragma unroll
        for (int term = 0; term < C::NA; ++term) {
          const uint32_t sa = stage(st) + term * C::A_TILE;
#pragma unroll
          for (int kk = 0; kk < BLOCK_N / 16; ++kk)
            mma_f16_ss(tmem, make_sdesc(sa + kk * 16 * 128, C::CB, SW128_ATOM),
                       make_sdesc(sb + kk * 16 * 128, C::CB, SW128_ATOM), id,
                       (t > 0 || term > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&bar_empty[st]);
      }
      if (ok && n > 0) tc_commit(&bar_done);
      tc_commit(&bar_drain);
      drain_wait(&bar_drain, 0, a.limit_ns);
    }
  } else {
    // epilogue: dQ * dq_mul (scale, and 2^-(eD + eK) for the scaled copies); rows of a
    // tile that sees no key get 0. The ring is free once bar_done has completed (every
    // MMA, hence every load, is done), and stages the stores.
    const int wq = warp % 4;
    bool ok = true;
    if (n > 0) {
      ok = __all_sync(0xffffffffu, wait(&bar_done, 0));
      tc_fence_after();
    }
    if (ok) {
      const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
      const int r_base = i0 + wq * 32;
      const uint32_t st_w = sbase + wq * C::EPI_WARP;
      const float mul = a.sc->dq_mul;
      if (a.out_bf16)
        store_rows_tma<D, true, D / 64>(&m.dQ, lane_addr, n > 0, mul, st_w, r_base, r_base < a.Sq, zo,
                                        0, a.Dv);
      else
        store_rows_tma<D, false, D / 32>(&m.dQ, lane_addr, n > 0, mul, st_w, r_base, r_base < a.Sq, zo,
                                         0, a.Dv);
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
__device__ __forceinline__ void load4(const void* base, size_t off, int is_bf16, float (&v)[4]) {
  if (is_bf16) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + off);
    v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xFFFF0000u);
    v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xFFFF0000u);
  } else {
    const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  }
}

// One warp per padded query row (bh, i), i < ldq:
//   delta[bh][i] = sum_d dO[i,d] * O[i,d];  lse2[bh][i] = LSE * log2(e) (+inf if -inf);
//   for bf16 inputs also the fp16 copies of the dO and Q rows (dO16 / Q16 non-null).
// Rows i >= Sq get lse2 = +inf, delta = 0.
template <int D>
__global__ void bwd_preprocess_kernel(const void* __restrict__ dO, const void* __restrict__ O,
                                      const float* __restrict__ LSE, const void* __restrict__ Q,
                                      __half* __restrict__ dO16, __half* __restrict__ Q16,
                                      float* __restrict__ lse2, float* __restrict__ delta, int Sq,
                                      int ldq, size_t n_rows_padded, int in_bf16, int o_bf16,
                                      int Dv) {
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
      if (d >= Dv) break;  // rows of Dv <= D columns: the lanes past them have none
      float gv[4], ov[4];
      load4(dO, row * Dv + d, in_bf16, gv);
      load4(O, row * Dv + d, o_bf16, ov);
      acc += gv[0] * ov[0] + gv[1] * ov[1] + gv[2] * ov[2] + gv[3] * ov[3];
      if (dO16) {
        float qv[4];
        load4(Q, row * Dv + d, 1, qv);
        uint2 g16, q16;
        g16.x = pack_half2(gv[0], gv[1]);
        g16.y = pack_half2(gv[2], gv[3]);
        q16.x = pack_half2(qv[0], qv[1]);
        q16.y = pack_half2(qv[2], qv[3]);
        *reinterpret_cast<uint2*>(dO16 + row * Dv + d) = g16;
        *reinterpret_cast<uint2*>(Q16 + row * Dv + d) = q16;
      }
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

// bf16 inputs, one launch for every pre-pass of the backward:
//   rows (bh, i < ldq) of Q / dO / O:  delta[bh][i] = sum_d dO[i,d] * O[i,d],
//       lse2[bh][i] = LSE * log2(e) (+inf for LSE = -inf; rows i >= Sq get +inf / 0),
//       fp16 copies of the Q and dO rows;
//   rows of K / V (B*HKV*Sk of them): fp16 copies.
// The copies are made with exponent 0; block b writes part[5 b ..] = the largest |Q|,
// |K|, |V|, |dO| and |delta| it saw (fp32 bits), from which bwd_scales_kernel picks
// the exponents. D/8 threads per row, 8 elements (16 bytes of bf16) each, so a warp
// moves whole 256-byte rows with 16-byte accesses.
// (Launched as 8 blocks of 256 threads per SM, one wave: the bounds keep it at 32
// registers so that all 8 fit.) O_BF16: O is bf16 (else fp32).
template <int D, bool O_BF16>
__global__ void __launch_bounds__(256, 8)
    bwd_prepass16_kernel(const __nv_bfloat16* __restrict__ dO, const void* __restrict__ O,
                                     const float* __restrict__ LSE, const __nv_bfloat16* __restrict__ Q,
                                     const __nv_bfloat16* __restrict__ K,
                                     const __nv_bfloat16* __restrict__ V, __half* __restrict__ dO16,
                                     __half* __restrict__ Q16, __half* __restrict__ K16,
                                     __half* __restrict__ V16, float* __restrict__ lse2,
                                     float* __restrict__ delta, int Sq, int ldq, size_t q_rows,
                                     size_t kv_rows, int* __restrict__ sched, int Dv,
                                     uint32_t* __restrict__ part) {
  constexpr int TPR = D / 8;  // threads per row (rows have Dv <= D columns: the rest idle)
  grid_launch_dependents();  // bwd_scales_kernel waits for this grid before reading part[]
  if (blockIdx.x == 0 && threadIdx.x == 0) *sched = 0;  // the dQ kernel's work-item counter
  const int t = threadIdx.x % TPR;
  const bool cols = t * 8 < Dv;  // this thread's 8 columns exist
  const size_t rows_per_grid = (size_t)gridDim.x * (blockDim.x / TPR);
  auto cvt8 = [](uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = pack_half2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
  // Largest |Q|, |K|, |V|, |dO|, |delta| of the block (fp32 bits), folded in once per
  // warp and row group: nothing is carried across iterations in registers, which keeps
  // the kernel at 8 resident blocks per SM.
  __shared__ uint32_t amax_sh[5];
  if (threadIdx.x < 5) amax_sh[threadIdx.x] = 0;
  __syncthreads();
  auto fold = [&](int k, uint32_t v) {  // warp-uniform call sites only
    v = __reduce_max_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0 && v != 0) atomicMax(&amax_sh[k], v);
  };
  // The loop runs the same iterations in every thread of the block (rows past the end
  // do nothing), so the warp-wide reductions always see the whole warp; the Q-row /
  // KV-row branch is warp-uniform too (a warp's rows are consecutive and the Q rows
  // are a multiple of 128).
  const size_t rows = q_rows + kv_rows;
  for (size_t rb = blockIdx.x * (size_t)(blockDim.x / TPR); rb < rows; rb += rows_per_grid) {
    const size_t r = rb + threadIdx.x / TPR;
    if (r < q_rows) {
      const size_t bh = r / ldq;
      const int i = (int)(r % ldq);
      float acc = 0.f;
      uint32_t aq = 0, ag = 0;
      if (i < Sq && cols) {
        const size_t off = (bh * Sq + i) * Dv + t * 8;
        const uint4 g = *reinterpret_cast<const uint4*>(dO + off);
        const uint4 q = *reinterpret_cast<const uint4*>(Q + off);
        ag = amax_bits(amax_acc(0u, g));
        aq = amax_bits(amax_acc(0u, q));
        float ov[8];
        if constexpr (O_BF16) {
          const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(O) + off);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            ov[2 * e] = __uint_as_float(w[e] << 16);
            ov[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
          }
        } else {
          const float4 a4 = *reinterpret_cast<const float4*>(static_cast<const float*>(O) + off);
          const float4 b4 = *reinterpret_cast<const float4*>(static_cast<const float*>(O) + off + 4);
          ov[0] = a4.x; ov[1] = a4.y; ov[2] = a4.z; ov[3] = a4.w;
          ov[4] = b4.x; ov[5] = b4.y; ov[6] = b4.z; ov[7] = b4.w;
        }
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          acc += __uint_as_float(gw[e] << 16) * ov[2 * e] +
                 __uint_as_float(gw[e] & 0xFFFF0000u) * ov[2 * e + 1];
        *reinterpret_cast<uint4*>(dO16 + off) = cvt8(g);
        *reinterpret_cast<uint4*>(Q16 + off) = cvt8(q);
      }
#pragma unroll
      for (int w = TPR / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
      fold(0, aq);
      fold(3, ag);
      fold(4, i < Sq ? __float_as_uint(fabsf(acc)) : 0u);
      if (t == 0) {
        if (i < Sq) {
          const float L = LSE[bh * Sq + i];
          lse2[r] = (L == -INFINITY) ? INFINITY : L * LOG2E;
          delta[r] = acc;
        } else {
          lse2[r] = INFINITY;
          delta[r] = 0.f;
        }
      }
    } else {
      uint32_t ak = 0, av = 0;
      if (cols && r < rows) {
        const size_t off = (r - q_rows) * Dv + t * 8;
        const uint4 kx = *reinterpret_cast<const uint4*>(K + off);
        const uint4 vx = *reinterpret_cast<const uint4*>(V + off);
        *reinterpret_cast<uint4*>(K16 + off) = cvt8(kx);
        *reinterpret_cast<uint4*>(V16 + off) = cvt8(vx);
        ak = amax_bits(amax_acc(0u, kx));
        av = amax_bits(amax_acc(0u, vx));
      }
      fold(1, ak);
      fold(2, av);
    }
  }
  __syncthreads();
  if (threadIdx.x < 5) part[(size_t)blockIdx.x * 5 + threadIdx.x] = amax_sh[threadIdx.x];
}

// Exponents of the fp16 operand copies of one backward call (fa_scale.cuh): every block
// reduces the pre-pass blocks' partial maxima of |Q|, |K|, |V|, |dO| and |delta| and
// derives eQ, eK, eV, eO and eD; block 0 publishes the multipliers; then the grid
// rewrites every copy whose exponent is not 0 as fp16(x * 2^e), and delta as
// delta * 2^eD if eD is not 0. With all exponents 0 (inputs of ordinary magnitude)
// the blocks only reduce and return.
struct BwdScaleArgs {
  const uint32_t* part;
  int n_part;
  int dlog;  // ceil(log2 Dv)
  const __nv_bfloat16* src[4];  // Q, K, V, dO
  __half* dst[4];               // their fp16 copies
  size_t n8[4];                 // groups of 8 elements
  float* delta;
  size_t n_delta;
  float scale, scale_log2;
  OperandScales* out;
};

__global__ void __launch_bounds__(1024) bwd_scales_kernel(const __grid_constant__ BwdScaleArgs a) {
  // launched as a programmatic dependent of the pre-pass: wait until that grid has
  // completed and its writes (copies, delta, part[]) are visible
  grid_dependency_wait();
  uint32_t m[5];
  reduce_partials<5>(a.part, a.n_part, m);
  int e[5];
  for (int k = 0; k < 4; ++k) e[k] = copy_exponent(m[k]);
  e[SC_DS] = ds_exponent(m[3], m[2], m[4], a.dlog);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    OperandScales sc;
    sc.sl2 = ldexpf(a.scale_log2, -(e[SC_Q] + e[SC_K]));
    sc.dp_mul = ldexpf(1.f, e[SC_DS] - e[SC_DO] - e[SC_V]);
    sc.dq_mul = ldexpf(a.scale, -(e[SC_DS] + e[SC_K]));
    sc.dk_mul = ldexpf(a.scale, -(e[SC_DS] + e[SC_Q]));
    sc.dv_mul = ldexpf(1.f, -e[SC_DO]);
    sc.o_mul = 1.f;
    for (int k = 0; k < 5; ++k) sc.e[k] = e[k];
    sc.pad = 0;
    *a.out = sc;
  }
  for (int k = 0; k < 4; ++k)
    if (e[k] != 0) rescale_copy(a.src[k], a.dst[k], a.n8[k], e[k]);
  if (e[SC_DS] != 0) {
    const float f = pow2i(e[SC_DS]);
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < a.n_delta; i += stride)
      a.delta[i] *= f;
  }
}

// Key ranges of a query tile computed as separate dQ work items (few query tiles per
// SM): dQ = sum_s dQ_s over the ranges s that hold a key tile the query tile can see
// (exactly the ranges whose work items wrote their slab), summed in range order, so
// the result is deterministic; rows of a tile that sees no key get 0. Thread (x, y)
// of a block takes columns 4x.. of row blockIdx.x * blockDim.y + y of head blockIdx.y
// (+ multiples of gridDim.y); partial slab s holds rows (bh, i) of range s.
__global__ void dq_range_sum_kernel(const float* __restrict__ part, void* __restrict__ dQ,
                                    int tps, int BH, int Sq, int Sk, int causal, int window, int Dv,
                                    int out_bf16) {
  // a programmatic dependent of the kernel that wrote the partial dQ (every thread waits,
  // so this grid cannot complete before that one)
  grid_dependency_wait();
  const int i = blockIdx.x * blockDim.y + threadIdx.y;
  const int c = threadIdx.x * 4;
  if (i >= Sq || c >= Dv) return;
  const size_t slab = (size_t)BH * Sq * Dv;
  const int i0 = i / BLOCK_M * BLOCK_M;
  int lo, hi;
  kv_tile_range(i0, min(i0 + BLOCK_M - 1, Sq - 1), Sk, causal, window, &lo, &hi);
  // range s covers key tiles [s * tps, (s + 1) * tps): it meets [lo, hi) for s in
  // [lo / tps, (hi - 1) / tps]
  const int s_lo = lo / tps, n_s = hi > lo ? (hi - 1) / tps + 1 - s_lo : 0;
  constexpr int G = KEY_RANGE_GROUP;
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    const size_t r = (size_t)bh * Sq + i;
    const float* src = part + (size_t)s_lo * slab + r * Dv + c;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g0 = 0; g0 < n_s; g0 += G) {
      float4 v[G];  // a group's loads issued before any is used
#pragma unroll
      for (int k = 0; k < G; ++k)
        if (g0 + k < n_s) v[k] = *reinterpret_cast<const float4*>(src + (g0 + k) * slab);
#pragma unroll
      for (int k = 0; k < G; ++k) {
        if (g0 + k < n_s) {
          acc.x += v[k].x;
          acc.y += v[k].y;
          acc.z += v[k].z;
          acc.w += v[k].w;
        }
      }
    }
    if (out_bf16) {
      __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y), hi2 = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo2);
      u.y = *reinterpret_cast<uint32_t*>(&hi2);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(dQ) + r * Dv + c) = u;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(dQ) + r * Dv + c) = acc;
    }
  }
}

// fp32 inputs as two fp16 terms (X16): every block reduces the amax kernel's per-block maxima
// of |Q|, |K|, |V|, |dO| and |delta|, picks the exponents (x16_exponent for the
// copies, x16_ds_exponent for dS), and the grid writes x 2^e = hi + lo as fp16 pairs
// and delta 2^eD; block 0 publishes the multipliers (as bwd_scales_kernel does).
struct X16BwdArgs {
  const uint32_t* part;
  int n_part;
  int dlog;
  const float* src[4];  // Q, K, V, dO
  __half* hi[4];
  __half* lo[4];
  size_t n4[4];
  float* delta;
  size_t n_delta;
  float scale, scale_log2;
  OperandScales* out;
};
__global__ void __launch_bounds__(256) x16_bwd_split_kernel(const __grid_constant__ X16BwdArgs a) {
  // a programmatic dependent of the amax pass: its partial maxima once it has completed
  grid_launch_dependents();
  grid_dependency_wait();
  uint32_t m[5];
  reduce_partials<5>(a.part, a.n_part, m);
  int e[5];
  for (int k = 0; k < 4; ++k) e[k] = x16_exponent(m[k]);
  e[SC_DS] = x16_ds_exponent(m[3], m[2], m[4], a.dlog);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    OperandScales sc;
    sc.sl2 = ldexpf(a.scale_log2, -(e[SC_Q] + e[SC_K]));
    sc.dp_mul = ldexpf(1.f, e[SC_DS] - e[SC_DO] - e[SC_V]);
    sc.dq_mul = ldexpf(a.scale, -(e[SC_DS] + e[SC_K]));
    sc.dk_mul = ldexpf(a.scale, -(e[SC_DS] + e[SC_Q]));
    sc.dv_mul = ldexpf(1.f, -e[SC_DO]);
    sc.o_mul = 1.f;
    for (int k = 0; k < 5; ++k) sc.e[k] = e[k];
    sc.pad = 0;
    *a.out = sc;
  }
  for (int k = 0; k < 4; ++k) split_x16(a.src[k], a.hi[k], a.lo[k], a.n4[k], e[k]);
  if (e[SC_DS] != 0) {
    const float f = pow2i(e[SC_DS]);
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < a.n_delta; i += stride)
      a.delta[i] *= f;
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

// dsmat (bf16 inputs): the materialised-dS variant -- the dK / dV kernel also stores
// dS^T, and dQ is a GEMM over it (dq_from_ds_kernel) instead of the recompute kernel.
template <int D, int F32>
fa_status run_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* LSE, void* dQ, void* dK, void* dV, const fa_params& p,
                  cudaStream_t stream, bool dsmat) {
  using C = BwdCfg<D, F32>;
  if (F32 && dsmat) return FA_ERR_UNSUPPORTED;
  // Tensors have Dv = p.D <= D columns: loads past Dv read zeros, stores past it are
  // dropped, and the pre-passes work on Dv-element rows.
  const int Dv = p.D;
  const size_t BH = (size_t)p.B * p.H, BHk = (size_t)p.B * p.HKV;
  const size_t nq = BH * p.Sq * Dv, nk = BHk * p.Sk * Dv;
  const int ldq = (p.Sq + 127) / 128 * 128;  // lse2 / delta row pitch: whole 128-query chunks
  const size_t nvec = BH * ldq;
  const int ldqt = (p.Sq + 3) / 4 * 4, ldkt = (p.Sk + 3) / 4 * 4;  // transposed row pitch
  const size_t nqt = BH * Dv * ldqt, nkt = BHk * Dv * ldkt;
  size_t bytes = 2 * nvec * 4;
  if constexpr (!F32) bytes += (2 * nq + 2 * nk) * 2;
  else if constexpr (C::X16) bytes += (4 * nq + 4 * nk) * 2;  // Q,dO,K,V fp16 hi/lo
  else bytes += (4 * nq + 4 * nk + 4 * nqt + 2 * nkt) * 4;  // Q,dO,K,V hi/lo + Q^T,dO^T,K^T hi/lo
  const size_t sched_off = (bytes + 15) / 16 * 16;  // the dQ kernel's work-item counter
  bytes = sched_off + 16;
  // bf16 inputs: the call's OperandScales and the pre-pass blocks' partial maxima
  const int n_pre = 8 * host::sm_count();  // pre-pass blocks
  const size_t sc_off = (bytes + 255) / 256 * 256;
  if constexpr (!C::TF32) bytes = sc_off + 256 + (size_t)n_pre * 5 * 4;
  // Fewer query tiles than SMs (short query sequences): the dQ work items also split the
  // keys into ranges of tps tiles (key_range_tiles picks tps), each range writing a
  // partial dQ (fp32) that a sum kernel adds up afterwards. The fp32 dQ kernel is not
  // persistent (one CTA per item): it splits only below half the SMs, so that a grid
  // which nearly fills the GPU in one wave keeps that wave.
  const int sms = host::sm_count();
  const int n_qt = (p.Sq + BLOCK_M - 1) / BLOCK_M, n_kt = (p.Sk + BLOCK_N - 1) / BLOCK_N;
  int dq_tps = n_kt;
  if (F32 ? 2 * BH * n_qt <= (size_t)sms : BH * n_qt < (size_t)sms)
    dq_tps = key_range_tiles((int)BH * n_qt, n_kt, sms);
  const int dq_splits = (n_kt + dq_tps - 1) / dq_tps;
  const size_t part_off = (bytes + 255) / 256 * 256;  // partial dQ [splits][BH][Sq][Dv]
  if (dq_splits > 1) bytes = part_off + (size_t)dq_splits * nq * 4;
  // Fewer (kv head, key tile) items than SMs (short key sequences; for bf16 inputs the
  // plain recompute route, for fp32 -- whose kernel runs one CTA per item -- at most
  // half the SMs): the dK / dV items also split the queries into ranges of kv_qtps
  // tiles, each range writing partial dK and dV (fp32) that a sum kernel adds up.
  int kv_qtps = n_qt;
  if (F32 ? 2 * BHk * n_kt <= (size_t)sms
          : !dsmat && !split_operands(p.H / p.HKV, n_qt) && BHk * n_kt < (size_t)sms)
    kv_qtps = key_range_tiles((int)BHk * n_kt, n_qt, sms);
  const int kv_splits = (n_qt + kv_qtps - 1) / kv_qtps;
  const size_t kvp_off = (bytes + 255) / 256 * 256;  // partial dK then dV [splits][BHk][Sk][Dv]
  if (kv_splits > 1) bytes = kvp_off + 2 * (size_t)kv_splits * nk * 4;
  // two-term P / dS for short query sequences (see split_operands)
  const bool split = !F32 && split_operands(p.H / p.HKV, n_qt);
  // materialised dS^T: [B*H][Sk][ldq] fp16, one buffer per term
  const size_t ds_elems = BH * (size_t)p.Sk * ldq;
  const size_t ds_off = (bytes + 255) / 256 * 256;
  if (dsmat) bytes = ds_off + (split ? 2 : 1) * ds_elems * 2;
  void* ws = nullptr;
  if (host::scratch_alloc(&ws, bytes, stream) != cudaSuccess) return FA_ERR_CUDA;
  float* lse2 = static_cast<float*>(ws);
  float* delta = lse2 + nvec;
  int* sched = reinterpret_cast<int*>(static_cast<char*>(ws) + sched_off);
  OperandScales* sc =
      C::TF32 ? nullptr : reinterpret_cast<OperandScales*>(static_cast<char*>(ws) + sc_off);
  uint32_t* part = C::TF32 ? nullptr : reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + sc_off + 256);
  float* dq_part = dq_splits > 1 ? reinterpret_cast<float*>(static_cast<char*>(ws) + part_off) : nullptr;
  float* kv_part = kv_splits > 1 ? reinterpret_cast<float*>(static_cast<char*>(ws) + kvp_off) : nullptr;
  __half* ds_hi = dsmat ? reinterpret_cast<__half*>(static_cast<char*>(ws) + ds_off) : nullptr;
  __half* ds_lo = dsmat && split ? ds_hi + ds_elems : nullptr;
  const int grid_pp = 4 * sms;
  const auto F32T = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  KVMaps mk;
  QMaps mq;
  bool enc = true;
  const uint32_t qchunk = F32 ? C::CH : 128;  // query rows per dkdv chunk
  enc &= host::encode_tiled_3d(&mk.L, F32T, 4, lse2, ldq, BH, 1, ldq, qchunk, 1, 0);
  {
    const bool bf = p.out_dtype == FA_BF16;
    const auto odt = bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : F32T;
    const int oes = bf ? 2 : 4;
    if (kv_splits > 1) {
      const uint64_t zs = (uint64_t)kv_splits * BHk;
      enc &= host::encode_tiled_3d(&mk.dK, F32T, 4, kv_part, Dv, p.Sk, zs, Dv, 32, 32);
      enc &= host::encode_tiled_3d(&mk.dV, F32T, 4, kv_part + (size_t)kv_splits * nk, Dv, p.Sk, zs, Dv,
                                   32, 32);
    } else {
      enc &= host::encode_tiled_3d(&mk.dK, odt, oes, dK, Dv, p.Sk, BHk, Dv, 128 / oes, 32);
      enc &= host::encode_tiled_3d(&mk.dV, odt, oes, dV, Dv, p.Sk, BHk, Dv, 128 / oes, 32);
    }
    if (dq_splits > 1)
      enc &= host::encode_tiled_3d(&mq.dQ, F32T, 4, dq_part, Dv, p.Sq, (uint64_t)dq_splits * BH, Dv,
                                   32, 32);
    else
      enc &= host::encode_tiled_3d(&mq.dQ, odt, oes, dQ, Dv, p.Sq, BH, Dv, 128 / oes, 32);
  }
  enc &= host::encode_tiled_3d(&mk.Dl, F32T, 4, delta, ldq, BH, 1, ldq, qchunk, 1, 0);
  if constexpr (!F32) {
    __half* q16 = reinterpret_cast<__half*>(delta + nvec);
    __half* do16 = q16 + nq;
    __half* k16 = do16 + nq;
    __half* v16 = k16 + nk;
    {
      host::KernelTimer kt("bwd_prepass", stream);
      auto pre = p.out_dtype == FA_BF16 ? bwd_prepass16_kernel<D, true> : bwd_prepass16_kernel<D, false>;
      pre<<<n_pre, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(dO), O, LSE, static_cast<const __nv_bfloat16*>(Q),
          static_cast<const __nv_bfloat16*>(K), static_cast<const __nv_bfloat16*>(V), do16, q16, k16,
          v16, lse2, delta, p.Sq, ldq, nvec, BHk * p.Sk, sched, Dv, part);
    }
    {
      // exponents of the copies; rewrites the copies / delta whose exponent is not 0
      host::KernelTimer kt("bwd_scales", stream);
      BwdScaleArgs sa;
      sa.part = part;
      sa.n_part = n_pre;
      int dlog = 0;
      while ((1 << dlog) < Dv) ++dlog;
      sa.dlog = dlog;
      const __nv_bfloat16* srcs[4] = {static_cast<const __nv_bfloat16*>(Q),
                                      static_cast<const __nv_bfloat16*>(K),
                                      static_cast<const __nv_bfloat16*>(V),
                                      static_cast<const __nv_bfloat16*>(dO)};
      __half* dsts[4] = {q16, k16, v16, do16};
      const size_t n8s[4] = {nq / 8, nk / 8, nk / 8, nq / 8};
      for (int k = 0; k < 4; ++k) { sa.src[k] = srcs[k]; sa.dst[k] = dsts[k]; sa.n8[k] = n8s[k]; }
      sa.delta = delta;
      sa.n_delta = nvec;
      sa.scale = p.scale;
      sa.scale_log2 = p.scale * LOG2E;
      sa.out = sc;
      if (launch_programmatic(bwd_scales_kernel, dim3(sms), dim3(1024), stream, sa) != cudaSuccess) {
        host::scratch_free(ws, stream);
        return FA_ERR_CUDA;
      }
    }
    // Query tiles whose rows see no key (a window ending before the keys do: a suffix
    // of tiles) are skipped by the dQ kernel; their rows are zeroed here, before the
    // dK/dV launch (nothing may come between it and its dependent dQ launch). With
    // the keys split into ranges, the sum over the ranges writes them instead.
    if (dq_splits == 1 && !dsmat) {  // (the materialised-dS GEMM writes those rows itself)
      int t0 = n_qt;
      while (t0 > 0) {
        int lo, hi;
        kv_tile_range((t0 - 1) * BLOCK_M, std::min(t0 * BLOCK_M, p.Sq) - 1, p.Sk, p.causal,
                      p.window, &lo, &hi);
        if (hi > lo) break;
        --t0;
      }
      if (t0 < n_qt) {
        const size_t esz = p.out_dtype == FA_BF16 ? 2 : 4;
        const size_t row = (size_t)Dv * esz;
        if (cudaMemset2DAsync(static_cast<char*>(dQ) + (size_t)t0 * BLOCK_M * row, p.Sq * row, 0,
                              (size_t)(p.Sq - t0 * BLOCK_M) * row, BH, stream) != cudaSuccess) {
          host::scratch_free(ws, stream);
          return FA_ERR_CUDA;
        }
      }
    }
    const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // boxes of one tile row block: 64 elements (128-byte swizzle), 32 at D = 32 (64-byte)
    constexpr int ROWE = Dq16Cfg<D>::ROW, RBY = Dq16Cfg<D>::RB;
    enc &= host::encode_tiled_3d(&mk.K[0], F16, 2, k16, Dv, p.Sk, BHk, Dv, ROWE, 128, RBY);
    enc &= host::encode_tiled_3d(&mk.V[0], F16, 2, v16, Dv, p.Sk, BHk, Dv, ROWE, 128, RBY);
    enc &= host::encode_tiled_3d(&mk.Qc[0], F16, 2, q16, Dv, p.Sq, BH, Dv, ROWE, 128, RBY);
    enc &= host::encode_tiled_3d(&mk.dOc[0], F16, 2, do16, Dv, p.Sq, BH, Dv, ROWE, 128, RBY);
    enc &= host::encode_tiled_3d(&mq.Q[0], F16, 2, q16, Dv, p.Sq, BH, Dv, ROWE, 128, RBY);
    enc &= host::encode_tiled_3d(&mq.dO[0], F16, 2, do16, Dv, p.Sq, BH, Dv, ROWE, 128, RBY);
    enc &= host::encode_tiled_3d(&mq.Kc[0], F16, 2, k16, Dv, p.Sk, BHk, Dv, ROWE, 128, RBY);
    enc &= host::encode_tiled_3d(&mq.Vc[0], F16, 2, v16, Dv, p.Sk, BHk, Dv, ROWE, 128, RBY);
    mk.K[1] = mk.K[0]; mk.V[1] = mk.V[0]; mk.Qc[1] = mk.Qc[0]; mk.dOc[1] = mk.dOc[0];
    mk.Qt[0] = mk.Qt[1] = mk.Qc[0]; mk.dOt[0] = mk.dOt[1] = mk.dOc[0];
    mq.Q[1] = mq.Q[0]; mq.dO[1] = mq.dO[0]; mq.Kc[1] = mq.Kc[0]; mq.Vc[1] = mq.Vc[0];
    mq.Kt[0] = mq.Kt[1] = mq.Kc[0];
  } else if constexpr (C::X16) {
    __half* qh = reinterpret_cast<__half*>(delta + nvec);
    __half* ql = qh + nq;
    __half* doh = ql + nq;
    __half* dol = doh + nq;
    __half* kh = dol + nq;
    __half* kl = kh + nk;
    __half* vh = kl + nk;
    __half* vl = vh + nk;
    {
      host::KernelTimer kt("bwd_preprocess", stream);
      bwd_preprocess_kernel<D><<<grid_pp, 256, 0, stream>>>(dO, O, LSE, Q, nullptr, nullptr, lse2,
                                                           delta, p.Sq, ldq, nvec, 0,
                                                           p.out_dtype == FA_BF16, Dv);
    }
    AmaxJobs aj = {};
    aj.a[0] = static_cast<const float*>(Q);
    aj.a[1] = static_cast<const float*>(K);
    aj.a[2] = static_cast<const float*>(V);
    aj.a[3] = static_cast<const float*>(dO);
    aj.a[4] = delta;
    aj.n4[0] = aj.n4[3] = nq / 4;
    aj.n4[1] = aj.n4[2] = nk / 4;
    aj.n4[4] = nvec / 4;
    aj.n = 5;
    {
      host::KernelTimer kt("amax(Q,K,V,dO,delta)", stream);
      // programmatic dependents from here to dQ, each waiting for the grid before it
      if (launch_programmatic(amax_f32_kernel<5>, dim3(n_pre), dim3(256), stream, aj, part) !=
          cudaSuccess) {
        host::scratch_free(ws, stream);
        return FA_ERR_CUDA;
      }
    }
    X16BwdArgs xa;
    xa.part = part;
    xa.n_part = n_pre;
    int dlog = 0;
    while ((1 << dlog) < Dv) ++dlog;
    xa.dlog = dlog;
    __half* his[4] = {qh, kh, vh, doh};
    __half* los[4] = {ql, kl, vl, dol};
    for (int k = 0; k < 4; ++k) {
      xa.src[k] = aj.a[k];
      xa.hi[k] = his[k];
      xa.lo[k] = los[k];
      xa.n4[k] = aj.n4[k];
    }
    xa.delta = delta;
    xa.n_delta = nvec;
    xa.scale = p.scale;
    xa.scale_log2 = p.scale * LOG2E;
    xa.out = sc;
    {
      host::KernelTimer kt("x16_split(Q,K,V,dO)", stream);
      if (launch_programmatic(x16_bwd_split_kernel, dim3(n_pre), dim3(256), stream, xa) != cudaSuccess) {
        host::scratch_free(ws, stream);
        return FA_ERR_CUDA;
      }
    }
    const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    __half* hl_q[2] = {qh, ql};
    __half* hl_do[2] = {doh, dol};
    __half* hl_k[2] = {kh, kl};
    __half* hl_v[2] = {vh, vl};
    for (int sp = 0; sp < 2; ++sp) {
      enc &= host::encode_tiled_3d(&mk.K[sp], F16, 2, hl_k[sp], Dv, p.Sk, BHk, Dv, 64, 128);
      enc &= host::encode_tiled_3d(&mk.V[sp], F16, 2, hl_v[sp], Dv, p.Sk, BHk, Dv, 64, 128);
      enc &= host::encode_tiled_3d(&mk.Qc[sp], F16, 2, hl_q[sp], Dv, p.Sq, BH, Dv, 64, C::CH);
      enc &= host::encode_tiled_3d(&mk.dOc[sp], F16, 2, hl_do[sp], Dv, p.Sq, BH, Dv, 64, C::CH);
      enc &= host::encode_tiled_3d(&mq.Q[sp], F16, 2, hl_q[sp], Dv, p.Sq, BH, Dv, 64, 128);
      enc &= host::encode_tiled_3d(&mq.dO[sp], F16, 2, hl_do[sp], Dv, p.Sq, BH, Dv, 64, 128);
      enc &= host::encode_tiled_3d(&mq.Kc[sp], F16, 2, hl_k[sp], Dv, p.Sk, BHk, Dv, 64, C::CH);
      enc &= host::encode_tiled_3d(&mq.Vc[sp], F16, 2, hl_v[sp], Dv, p.Sk, BHk, Dv, 64, C::CH);
      mk.Qt[sp] = mk.Qc[sp];  // (no transposed copies: unused)
      mk.dOt[sp] = mk.dOc[sp];
      mq.Kt[sp] = mq.Kc[sp];
    }
  } else {
    float* qh = delta + nvec;
    float* ql = qh + nq;
    float* doh = ql + nq;
    float* dol = doh + nq;
    float* kh = dol + nq;
    float* kl = kh + nk;
    float* vh = kl + nk;
    float* vl = vh + nk;
    float* qth = vl + nk;
    float* qtl = qth + nqt;
    float* doth = qtl + nqt;
    float* dotl = doth + nqt;
    float* kth = dotl + nqt;
    float* ktl = kth + nkt;
    {
      host::KernelTimer kt("bwd_preprocess", stream);
      bwd_preprocess_kernel<D><<<grid_pp, 256, 0, stream>>>(dO, O, LSE, Q, nullptr, nullptr, lse2,
                                                           delta, p.Sq, ldq, nvec, 0,
                                                           p.out_dtype == FA_BF16, Dv);
    }
    {
      host::KernelTimer kt("split_tf32(Q,dO,K,V)", stream);
      launch_split_tf32({{static_cast<const float*>(Q), qh, ql, qth, qtl, p.Sq, ldqt, (int)BH},
                         {static_cast<const float*>(dO), doh, dol, doth, dotl, p.Sq, ldqt, (int)BH},
                         {static_cast<const float*>(K), kh, kl, kth, ktl, p.Sk, ldkt, (int)BHk},
                         {static_cast<const float*>(V), vh, vl, nullptr, nullptr, p.Sk, 0, (int)BHk}},
                        Dv, grid_pp, stream);
    }
    float* hl_q[2] = {qh, ql};
    float* hl_do[2] = {doh, dol};
    float* hl_k[2] = {kh, kl};
    float* hl_v[2] = {vh, vl};
    float* hl_qt[2] = {qth, qtl};
    float* hl_dot[2] = {doth, dotl};
    float* hl_kt[2] = {kth, ktl};
    for (int sp = 0; sp < 2; ++sp) {
      enc &= host::encode_tiled_3d(&mk.K[sp], F32T, 4, hl_k[sp], Dv, p.Sk, BHk, Dv, 32, 128);
      enc &= host::encode_tiled_3d(&mk.V[sp], F32T, 4, hl_v[sp], Dv, p.Sk, BHk, Dv, 32, 128);
      enc &= host::encode_tiled_3d(&mk.Qc[sp], F32T, 4, hl_q[sp], Dv, p.Sq, BH, Dv, 32, C::CH);
      enc &= host::encode_tiled_3d(&mk.dOc[sp], F32T, 4, hl_do[sp], Dv, p.Sq, BH, Dv, 32, C::CH);
      enc &= host::encode_tiled_3d(&mk.Qt[sp], F32T, 4, hl_qt[sp], p.Sq, Dv, BH, ldqt, 32, D);
      enc &= host::encode_tiled_3d(&mk.dOt[sp], F32T, 4, hl_dot[sp], p.Sq, Dv, BH, ldqt, 32, D);
      enc &= host::encode_tiled_3d(&mq.Q[sp], F32T, 4, hl_q[sp], Dv, p.Sq, BH, Dv, 32, 128);
      enc &= host::encode_tiled_3d(&mq.dO[sp], F32T, 4, hl_do[sp], Dv, p.Sq, BH, Dv, 32, 128);
      enc &= host::encode_tiled_3d(&mq.Kc[sp], F32T, 4, hl_k[sp], Dv, p.Sk, BHk, Dv, 32, C::CH);
      enc &= host::encode_tiled_3d(&mq.Vc[sp], F32T, 4, hl_v[sp], Dv, p.Sk, BHk, Dv, 32, C::CH);
      enc &= host::encode_tiled_3d(&mq.Kt[sp], F32T, 4, hl_kt[sp], p.Sk, Dv, BHk, ldkt, 32, D);
    }
  }
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
  a.Dv = Dv;
  a.sched = sched;
  a.n_splits = 1;
  a.tps = n_kt;
  a.limit_ns = WAIT_LIMIT_NS;
  a.sc = sc;
  a.ds_hi = ds_hi;
  a.ds_lo = ds_lo;
  cudaError_t e = cudaSuccess;
  {
    BwdArgs ak = a;
    ak.n_tiles = (p.Sk + BLOCK_N - 1) / BLOCK_N;
    ak.BHx = (int)BHk;
    ak.n_splits = kv_splits;  // query ranges of the dK / dV items
    ak.tps = kv_qtps;
    if (kv_splits > 1) ak.out_bf16 = 0;  // the partial sums are fp32
    if constexpr (F32) {
      auto kern = kv_splits > 1 ? fa_bwd_dkdv_kernel<D, F32, true> : fa_bwd_dkdv_kernel<D, F32>;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::KV_SMEM);
      if (e == cudaSuccess) {
        host::KernelTimer kt(C::TF32 ? "fa_bwd_dkdv_kernel<64,tf32>"
                             : (D == 128 ? "fa_bwd_dkdv_kernel<128,f32>" : "fa_bwd_dkdv_kernel<64,f32>"),
                             stream);
        e = launch_programmatic_smem(kern, dim3((unsigned)(BHk * ak.n_tiles * kv_splits)),
                                     dim3(C::THREADS), C::KV_SMEM, stream, mk, ak);
      }
    } else {
      using C16 = Dkv16Cfg<D>;
      auto kern = split ? fa_bwd_dkdv16_kernel<D, true, false> : fa_bwd_dkdv16_kernel<D, false, false>;
      if (kv_splits > 1) kern = fa_bwd_dkdv16_kernel<D, false, false, true>;  // (never with split)
      if constexpr (D >= 64)  // (the materialised-dS route runs in the D >= 64 kernels)
        if (dsmat) kern = split ? fa_bwd_dkdv16_kernel<D, true, true> : fa_bwd_dkdv16_kernel<D, false, true>;
      // all the dynamic shared memory a block may have: the layout fills it after
      // aligning its base to 1 KB (the kernel checks the fit)
      int dyn = 0;
      e = host::max_dynamic_smem(reinterpret_cast<const void*>(kern), &dyn);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
      if (e == cudaSuccess) {
        host::KernelTimer kt(D == 128 ? "fa_bwd_dkdv_kernel<128,bf16>"
                                      : (D == 64 ? "fa_bwd_dkdv_kernel<64,bf16>" : "fa_bwd_dkdv_kernel<32,bf16>"),
                             stream);
        // persistent: one CTA per SM (at most), walking the (key tile, kv head, query
        // range) items
        const unsigned grid = (unsigned)std::min<size_t>(BHk * ak.n_tiles * kv_splits, (size_t)sms);
        // a programmatic dependent of the scales kernel (it waits for it first)
        e = launch_programmatic_smem(kern, dim3(grid), dim3(C16::THREADS), (size_t)dyn, stream, mk, ak);
      }
    }
  }
  if (e == cudaSuccess) {
    BwdArgs aq = a;
    aq.n_tiles = n_qt;
    aq.BHx = (int)BH;
    aq.n_splits = dq_splits;
    aq.tps = dq_tps;
    if (dq_splits > 1) aq.out_bf16 = 0;  // the partial sums are fp32
    if constexpr (F32) {
      auto kern = fa_bwd_dq_kernel<D, F32>;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::Q_SMEM);
      if (e == cudaSuccess) {
        host::KernelTimer kt(C::TF32 ? "fa_bwd_dq_kernel<64,tf32>"
                             : (D == 128 ? "fa_bwd_dq_kernel<128,f32>" : "fa_bwd_dq_kernel<64,f32>"),
                             stream);
        // starts once every dK / dV block has, on the SMs that grid leaves free (it reads
        // nothing that grid writes; it waits for it before exiting)
        e = launch_programmatic_smem(kern, dim3((unsigned)(BH * aq.n_tiles * dq_splits)),
                                     dim3(C::THREADS), C::Q_SMEM, stream, mq, aq);
      }
      if (e == cudaSuccess && dq_splits > 1) {
        host::KernelTimer kt("dq_range_sum", stream);
        dim3 cg, cb;
        combine_launch_shape((int)BH, p.Sq, Dv, &cg, &cb);
        e = launch_programmatic(dq_range_sum_kernel, cg, cb, stream, (const float*)dq_part, dQ,
                                dq_tps, (int)BH, p.Sq, p.Sk, (int)p.causal, p.window, Dv,
                                (int)(p.out_dtype == FA_BF16));
      }
    } else if (D >= 64 && dsmat) {
      // dQ = scale dS K over the stored dS^T (an ordinary launch: it reads what the
      // dK / dV kernel wrote)
      if constexpr (D >= 64) {
      DsMaps md;
      const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
      bool enc2 = host::encode_tiled_3d(&md.ds_hi, F16, 2, ds_hi, ldq, p.Sk, BH, ldq, 64, 128);
      md.ds_lo = md.ds_hi;
      if (split) enc2 &= host::encode_tiled_3d(&md.ds_lo, F16, 2, ds_lo, ldq, p.Sk, BH, ldq, 64, 128);
      md.K = mq.Kc[0];
      md.dQ = mq.dQ;
      if (!enc2) e = cudaErrorInvalidValue;
      auto kern = split ? dq_from_ds_kernel<D, true> : dq_from_ds_kernel<D, false>;
      const uint32_t smem_b = split ? DqGemmCfg<D, true>::SMEM : DqGemmCfg<D, false>::SMEM;
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_b);
      if (e == cudaSuccess) {
        host::KernelTimer kt(D == 128 ? "dq_from_ds_kernel<128,bf16>" : "dq_from_ds_kernel<64,bf16>",
                             stream);
        kern<<<(unsigned)(BH * (size_t)n_qt * dq_splits), DqGemmCfg<D, false>::THREADS, smem_b,
               stream>>>(md, aq);
        e = cudaGetLastError();
      }
      if (e == cudaSuccess && dq_splits > 1) {
        host::KernelTimer kt("dq_range_sum", stream);
        dim3 cg, cb;
        combine_launch_shape((int)BH, p.Sq, Dv, &cg, &cb);
        e = launch_programmatic(dq_range_sum_kernel, cg, cb, stream, (const float*)dq_part, dQ,
                                dq_tps, (int)BH, p.Sq, p.Sk, (int)p.causal, p.window, Dv,
                                (int)(p.out_dtype == FA_BF16));
      }
      }
    } else {
      using C16 = Dq16Cfg<D>;
      auto kern = dq_splits > 1 ? fa_bwd_dq16_kernel<D, true> : fa_bwd_dq16_kernel<D, false>;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C16::SMEM);
      if (e == cudaSuccess) {
        host::KernelTimer kt(D == 128 ? "fa_bwd_dq_kernel<128,bf16>"
                                      : (D == 64 ? "fa_bwd_dq_kernel<64,bf16>" : "fa_bwd_dq_kernel<32,bf16>"),
                             stream);
        // Persistent: one CTA per SM (at most), work items handed out dynamically.
        // Launched as a programmatic dependent of the dK / dV kernel (which does not
        // write anything dQ reads): its blocks may start as soon as every dK / dV block
        // has started, on the SMs that dK / dV's last wave leaves idle, and each waits
        // for the dK / dV grid to complete before it exits, so the dQ grid's completion
        // (which the rest of the stream waits for) implies dK / dV's.
        const size_t n_items = BH * (size_t)aq.n_tiles * dq_splits;
        const unsigned grid = (unsigned)std::min<size_t>(n_items, (size_t)sms);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(C16::THREADS);
        cfg.dynamicSmemBytes = C16::SMEM;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, mq, aq);
        if (e == cudaSuccess) e = cudaGetLastError();
      }
      if (e == cudaSuccess && dq_splits > 1) {
        host::KernelTimer kt("dq_range_sum", stream);
        dim3 cg, cb;
        combine_launch_shape((int)BH, p.Sq, Dv, &cg, &cb);
        e = launch_programmatic(dq_range_sum_kernel, cg, cb, stream, (const float*)dq_part, dQ,
                                dq_tps, (int)BH, p.Sq, p.Sk, (int)p.causal, p.window, Dv,
                                (int)(p.out_dtype == FA_BF16));
      }
    }
  }
  if (e == cudaSuccess && kv_splits > 1) {
    // dK, dV = the sums of the query ranges' partial slabs, in a fixed order
    // (programmatic dependents of the launch before them, which completes after dK / dV)
    host::KernelTimer kt("dkv_range_sum", stream);
    const int q4 = Dv / 4;
    const int sg = std::max(1, std::min({256 / q4, kv_splits, DEC_SUM_GROUPS}));
    const size_t rows = BHk * (size_t)p.Sk;
    const dim3 cg((unsigned)std::min<size_t>(rows, 65535)), cb(q4, sg);
    const int obf = (int)(p.out_dtype == FA_BF16);
    e = launch_programmatic(dq_splits_sum_kernel, cg, cb, stream, (const float*)kv_part, dK, kv_splits,
                            (int)rows, Dv, obf);
    if (e == cudaSuccess)
      e = launch_programmatic(dq_splits_sum_kernel, cg, cb, stream,
                              (const float*)(kv_part + (size_t)kv_splits * nk), dV, kv_splits, (int)rows,
                              Dv, obf);
  }
  const cudaError_t e2 = host::scratch_free(ws, stream);
  return (e == cudaSuccess && e2 == cudaSuccess) ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

namespace {

// The decode backward (fa_decode_bwd.cuh): the keys of each (batch, kv head) split into
// ranges as for the decode forward, one wave of CTAs; with more than one range, partial
// dQ in scratch and the fixed-order range sum.
template <int DK, int ROWS, bool F32IN>
fa_status run_decode_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                         const float* LSE, void* dQ, void* dK, void* dV, const fa_params& p,
                         cudaStream_t stream) {
  DecodeBwdArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.O = O;
  a.dO = dO;
  a.LSE = LSE;
  a.dK = dK;
  a.dV = dV;
  a.B = p.B;
  a.H = p.H;
  a.HKV = p.HKV;
  a.Sq = p.Sq;
  a.Sk = p.Sk;
  a.Dv = p.D;
  a.rep = p.H / p.HKV;
  a.rows = a.rep * p.Sq;
  a.causal = p.causal;
  a.window = p.window;
  a.out_bf16 = p.out_dtype == FA_BF16;
  a.k_wide = reinterpret_cast<uintptr_t>(K) % 32 == 0;
  a.v_wide = reinterpret_cast<uintptr_t>(V) % 32 == 0;
  a.scale = p.scale;
  a.scale_log2 = p.scale * LOG2E;
  constexpr size_t smem = decode_bwd_smem_bytes<DK, ROWS, F32IN>();
  auto kern = fa_decode_bwd_kernel<DK, ROWS, F32IN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  // CTAs resident per SM (registers and shared memory), asked once per kernel
  static const int per_sm = [&] {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, DEC_WARPS * 32, smem) != cudaSuccess)
      o = 1;
    return std::max(o, 1);
  }();
  const long long groups = (long long)p.B * p.HKV;
  const int sms = host::sm_count();
  const int min_keys = DEC_WARPS * DEC_KEYS;
  long long n = ((long long)per_sm * sms + groups - 1) / groups;
  n = std::max(1ll, std::min(n, ((long long)p.Sk + min_keys - 1) / min_keys));
  int kps = (int)(((long long)p.Sk + n - 1) / n);
  kps = (kps + DEC_KEYS - 1) / DEC_KEYS * DEC_KEYS;
  a.keys_per_split = kps;
  a.n_splits = (p.Sk + kps - 1) / kps;
  const size_t rows_all = (size_t)p.B * p.H * p.Sq;
  void* pws = nullptr;
  if (a.n_splits > 1) {
    if (host::scratch_alloc(&pws, (size_t)a.n_splits * rows_all * p.D * 4, stream) != cudaSuccess)
      return FA_ERR_CUDA;
    a.dQ = pws;
  } else {
    a.dQ = dQ;
  }
  {
    host::KernelTimer kt("fa_decode_bwd_kernel", stream);
    kern<<<dim3((unsigned)groups, (unsigned)a.n_splits), DEC_WARPS * 32, smem, stream>>>(a);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess && a.n_splits > 1) {
    host::KernelTimer kt("dq_range_sum", stream);
    const int q4 = p.D / 4;
    const int sg = std::max(1, std::min({256 / q4, a.n_splits, DEC_SUM_GROUPS}));
    const dim3 cg((unsigned)std::min<size_t>(rows_all, 65535)), cb(q4, sg);
    e = launch_programmatic(dq_splits_sum_kernel, cg, cb, stream, (const float*)pws, dQ, a.n_splits,
                            (int)rows_all, p.D, (int)(p.out_dtype == FA_BF16));
  }
  const cudaError_t e2 = host::scratch_free(pws, stream);
  return (e == cudaSuccess && e2 == cudaSuccess) ? FA_OK : FA_ERR_CUDA;
}

template <int DK, bool F32IN>
fa_status run_decode_bwd_rows(const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                              const fa_params& p, cudaStream_t stream) {
  if (p.H / p.HKV * p.Sq <= 4)
    return run_decode_bwd<DK, 4, F32IN>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream);
  return run_decode_bwd<DK, DEC_ROWS, F32IN>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream);
}

}  // namespace

fa_status launch_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* LSE, void* dQ, void* dK, void* dV, const fa_params& p,
                     cudaStream_t stream, bool dsmat) {
  if (dsmat && p.in_dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
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
  // decode shapes (a few query rows per kv head): the CUDA-core backward, for both input
  // types (the materialised-dS route keeps its own kernels)
  if (!dsmat && decode_shaped(p)) {
    const bool f32 = p.in_dtype != FA_BF16;
    if (p.D <= 64)
      return f32 ? run_decode_bwd_rows<64, true>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream)
                 : run_decode_bwd_rows<64, false>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream);
    return f32 ? run_decode_bwd_rows<128, true>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream)
               : run_decode_bwd_rows<128, false>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream);
  }
  // head dims below a kernel's D run in it with the missing columns read as zeros
  if (p.in_dtype == FA_BF16) {
    // (the D = 32 kernels write fp32 outputs and recompute dS for dQ)
    if (p.D <= 32 && p.out_dtype == FA_F32 && !dsmat)
      return run_bwd<32, IN_BF16>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream, false);
    if (p.D <= 64) return run_bwd<64, IN_BF16>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream, dsmat);
    if (p.D <= 128) return run_bwd<128, IN_BF16>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream, dsmat);
  } else if (p.f32_mma == FA_F32_MMA_TF32X3) {
    if (p.D <= 64) return run_bwd<64, IN_F32_TF32>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream, false);
  } else {
    if (p.D <= 64) return run_bwd<64, IN_F32_X16>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream, false);
    if (p.D <= 128) return run_bwd<128, IN_F32_X16>(Q, K, V, O, dO, LSE, dQ, dK, dV, p, stream, false);
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
