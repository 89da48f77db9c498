// fa_fwd.cu -- forward attention on sm_103a: TMA-fed, warp-specialised, tcgen05/TMEM.
//
// A work item is NQ query tiles of 128 rows of one (batch, head); it walks the key
// tiles they may see (forge "flash_attention.metal", flash_attn_fwd: threadgroup of
// consecutive query rows, K/V staged once per group, blocks outside the causal /
// window band skipped, online softmax with m starting at -FLT_MAX; rustytorch
// "flash_attention_forward.metal": O = softmax(Q K^T * scale) V and the LSE row
// output). One persistent CTA per SM runs a sequence of items. Roles:
//   warps [0, 4*NQ)   softmax: thread = one query row = one TMEM lane. Reads the
//                     S row from TMEM, masks boundary tiles, keeps the running max
//                     m (log2 units) and sum l, writes P back into TMEM (fp16 for
//                     bf16 inputs; fp16 or tf32 hi + lo for fp32 inputs), rescales its O
//                     row in TMEM when m grows by more than RESCALE_THRESHOLD, and
//                     in the epilogue writes LSE = (m + log2 l) ln 2 and O = acc / l
//                     (staged in a V ring stage, written by TMA stores).
//   warp 4*NQ         MMA issuer (one thread): S_q = Q_q K_j^T, O_q += P_q V_j,
//                     bursts in a fixed tile order so the tiles alternate.
//   warp 4*NQ + 1     TMA producer (one thread): Q per item, K_j ring.
//   warp 4*NQ + 2     TMA producer (one thread): V_j ring and the epilogue stages.
//   warp 4*NQ + 3     load relay: mbarrier waits passed on to the issuer.
// Every barrier wait is bounded; on expiry the kernel raises the device status
// word, drains its in-flight copies and MMAs, frees TMEM and returns.
#include <algorithm>
#include <cmath>
#include <cfloat>
#include <climits>
#include <cstdio>
#include <mutex>
#include "fa_common.cuh"
#include "ptx.cuh"
#include "fa_prepass.cuh"
#include "fa_epilogue.cuh"
#include "fa_decode.cuh"

namespace fa {
using namespace ptx;

static __device__ unsigned int g_fwd_status = 0;

struct FwdArgs {
  void* O;
  float* LSE;
  int H, HKV, Sq, Sk;
  float scale_log2;  // softmax scale * log2(e)
  int causal, window;
  int out_bf16;
  int n_qgroups;  // row groups per head: 128 rows (head pairs) or 256 rows
  int n_splits;  // key ranges per (query group, head (pair)): > 1 writes partial O / LSE per range
  int tps;       // key tiles per range
  int n_items;  // BHi * n_qgroups * n_splits
  int Dv;       // head dim of the tensors (<= the kernel's D; missing columns read as 0)
  int lpt;  // 1: the heaviest query groups first (causal)
  int BH;
  int BHi;  // work units per query group: heads (BH), or head pairs (BH / 2)
  unsigned long long limit_ns;
  const OperandScales* sc;  // bf16 inputs: o_mul = 2^-eV undoes the scaled fp16 copy of V
};

template <int D_, int PREC, int NQ_ = 0>
struct FwdCfg {
  static constexpr int D = D_;
  static constexpr bool F32 = PREC != IN_BF16;
  // fp32 inputs: two scaled fp16 terms per operand (X16: x 2^e = hi + lo, three
  // kind::f16 products per GEMM), or 3xTF32 (hi / lo tf32 splits) up to D = 64, above
  // which the tf32 tiles would not fit shared memory
  static constexpr bool X16 = PREC == IN_F32_X16;
  static constexpr bool TF32 = PREC == IN_F32_TF32;
  static_assert(!TF32 || D <= 64, "3xTF32 tiles up to D = 64");
  // query tiles per item: two (their softmaxes alternate with each other's MMAs) where
  // the operand tiles leave room for them, unless NQ_ asks for one
  static constexpr int NQ = (TF32 || (X16 && D > 64) || NQ_ == 1) ? 1 : 2;
  static_assert(F32 || NQ == 2, "bf16 items hold two query tiles");
  static constexpr int ESZ = TF32 ? 4 : 2;                 // operand bytes in smem
  // smem rows of RB bytes with the swizzle of that width: 128, or 64 for bf16 at D = 32
  static constexpr int RB = F32 ? 128 : tile_row_bytes(D);
  static constexpr uint32_t SWZ = RB == 128 ? SWZ_128B : SWZ_64B;
  static constexpr uint32_t ATOM = 8u * RB;                // 8-row swizzle atom
  static constexpr int ROW_ELEMS = RB / ESZ;               // elements per row
  static constexpr int NCB = D / ROW_ELEMS;                // column blocks per row-tile
  static constexpr uint32_t CB_BYTES = 128u * RB;          // one column block of a 128-row tile
  static constexpr uint32_t TILE_BYTES = NCB * CB_BYTES;   // a 128 x D operand tile
  static constexpr uint32_t VT_CB_BYTES = D * 128u;        // fp32 V^T: 32 keys x D rows
  static constexpr int NSPLIT = F32 ? 2 : 1;               // hi / lo copies
  static constexpr int KST = NQ == 1 ? 1 : ((D == 128 || X16) ? 2 : 3);  // K ring depth
  static constexpr int VST = NQ == 1 ? 1 : 3;                             // V ring depth
  // a V ring stage also stages an item's epilogue, the NQ tiles side by side: at least
  // one 32 x 128-byte box per warp of each tile
  static constexpr uint32_t V_STAGE = NSPLIT * TILE_BYTES > 4 * NQ * EPI_BOX_BYTES
                                          ? NSPLIT * TILE_BYTES
                                          : 4 * NQ * EPI_BOX_BYTES;
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + NQ * NSPLIT * TILE_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + KST * NSPLIT * TILE_BYTES;
  static constexpr uint32_t SMEM_BYTES = V_OFF + VST * V_STAGE;
  static constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;
  static constexpr int SOFTMAX_WARPS = 4 * NQ;
  // The last warpgroup holds the control warps: the MMA issuer (which also owns
  // TMEM), the Q / K producer, the V producer and the load relay.
  static constexpr int MMA_WARP = SOFTMAX_WARPS;
  static constexpr int KQ_WARP = SOFTMAX_WARPS + 1;
  static constexpr int V_WARP = SOFTMAX_WARPS + 2;
  static constexpr int RELAY_WARP = SOFTMAX_WARPS + 3;  // relays load completions to the issuer
  // named barriers: 1 + q = P_q written (softmax -> issuer), RELAY_BAR = operands
  // loaded (relay -> issuer), EPI_BAR0 + q = the four warps of tile q (epilogue),
  // EPI_JOIN = every tile's epilogue stores have read their part of the stage
  static constexpr uint32_t RELAY_BAR = 3;
  static constexpr uint32_t EPI_BAR0 = 4;
  static constexpr uint32_t EPI_JOIN = 6;
  static constexpr int THREADS = 32 * (SOFTMAX_WARPS + 4);
  // Register split for NQ = 2 (launched at 168 per thread for 384 threads): the
  // softmax warpgroups hold a whole 128-column S row in registers.
  static constexpr uint32_t REGS_SOFTMAX = 216, REGS_CONTROL = 64;
  static_assert(NQ == 1 || (2 * 128 * REGS_SOFTMAX + 128 * REGS_CONTROL) <= 384 * 168,
                "register split exceeds the launch allocation");
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t PLO_COL = 128;                  // fp32 path: P_lo columns
  __host__ __device__ static constexpr uint32_t s_col(int q) { return 128u * q; }
  __host__ __device__ static constexpr uint32_t o_col(int q) { return 256u + (uint32_t)D * q; }
  static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory budget");
  static_assert(F32 ? (256 + D <= 512) : (256 + 2 * D <= 512), "TMEM budget");
  // Epilogue: each softmax warp stages its 32 O rows in its share of the tile's part
  // (1 / NQ) of a V ring stage.
  static constexpr uint32_t STAGE_PER_WARP = V_STAGE / (4 * NQ);
  static constexpr int STAGE_BOXES = (int)(STAGE_PER_WARP / EPI_BOX_BYTES);
  static_assert(STAGE_BOXES >= 1 && STAGE_PER_WARP % 1024 == 0, "O staging layout");
};

template <class C>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t sq, uint32_t sq_lo, uint32_t sk,
                                         uint32_t sk_lo) {
  if constexpr (!C::F32) {
    constexpr uint32_t id = make_idesc(128, 128, FMT_BF16, FMT_BF16, false, false);
#pragma unroll
    for (int kk = 0; kk < C::D / 16; ++kk) {
      const uint32_t off = (kk * 16 / C::ROW_ELEMS) * C::CB_BYTES + (kk * 16 % C::ROW_ELEMS) * 2;
      mma_f16_ss(d_tmem, make_sdesc(sq + off, 16, C::ATOM, C::SWZ),
                 make_sdesc(sk + off, 16, C::ATOM, C::SWZ), id, kk > 0);
    }
  } else if constexpr (C::X16) {
    // (Qh + Ql)(Kh + Kl)^T without the lo * lo term, fp16 terms
    constexpr uint32_t id = make_idesc(128, 128, FMT_F16, FMT_F16, false, false);
#pragma unroll
    for (int kk = 0; kk < C::D / 16; ++kk) {
      const uint32_t off = (kk * 16 / 64) * C::CB_BYTES + (kk * 16 % 64) * 2;
      const uint64_t qh = make_sdesc(sq + off, 16, SW128_ATOM);
      const uint64_t ql = make_sdesc(sq_lo + off, 16, SW128_ATOM);
      const uint64_t kh = make_sdesc(sk + off, 16, SW128_ATOM);
      const uint64_t kl = make_sdesc(sk_lo + off, 16, SW128_ATOM);
      mma_f16_ss(d_tmem, qh, kh, id, kk > 0);
      mma_f16_ss(d_tmem, qh, kl, id, 1);
      mma_f16_ss(d_tmem, ql, kh, id, 1);
    }
  } else {
    constexpr uint32_t id = make_idesc(128, 128, FMT_TF32, FMT_TF32, false, false);
#pragma unroll
    for (int kk = 0; kk < C::D / 8; ++kk) {
      const uint32_t off = (kk * 8 / 32) * C::CB_BYTES + (kk * 8 % 32) * 4;
      const uint64_t qh = make_sdesc(sq + off, 16, SW128_ATOM);
      const uint64_t ql = make_sdesc(sq_lo + off, 16, SW128_ATOM);
      const uint64_t kh = make_sdesc(sk + off, 16, SW128_ATOM);
      const uint64_t kl = make_sdesc(sk_lo + off, 16, SW128_ATOM);
      mma_tf32_ss(d_tmem, qh, kh, id, kk > 0);
      mma_tf32_ss(d_tmem, qh, kl, id, 1);
      mma_tf32_ss(d_tmem, ql, kh, id, 1);
    }
  }
}

template <class C, bool PSPLIT = false>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t plo_tmem,
                                         uint32_t sv, uint32_t sv_lo, bool accumulate) {
  if constexpr (!C::F32) {
    // A = P (fp16, TMEM, 8 columns per 16 keys); B = V (fp16, MN-major in smem).
    // PSPLIT: then A = P_lo, 64 columns further on.
    constexpr uint32_t id = make_idesc(128, C::D, FMT_F16, FMT_F16, false, true);
#pragma unroll
    for (int kk = 0; kk < BLOCK_N / 16; ++kk)
      mma_f16_ts(o_tmem, p_tmem + kk * 8, make_sdesc(sv + kk * 16 * C::RB, C::CB_BYTES, C::ATOM, C::SWZ),
                 id, (accumulate || kk > 0) ? 1u : 0u);
    if constexpr (PSPLIT) {
#pragma unroll
      for (int kk = 0; kk < BLOCK_N / 16; ++kk)
        mma_f16_ts(o_tmem, p_tmem + 64 + kk * 8,
                   make_sdesc(sv + kk * 16 * C::RB, C::CB_BYTES, C::ATOM, C::SWZ), id, 1u);
    }
  } else if constexpr (C::X16) {
    // (Ph + Pl)(Vh + Vl) without the lo * lo term: P hi / lo in the S slot's two column
    // halves, V hi / lo MN-major in smem
    constexpr uint32_t id = make_idesc(128, C::D, FMT_F16, FMT_F16, false, true);
#pragma unroll
    for (int kk = 0; kk < BLOCK_N / 16; ++kk) {
      const uint64_t vh = make_sdesc(sv + kk * 16 * 128, C::CB_BYTES, SW128_ATOM);
      const uint64_t vl = make_sdesc(sv_lo + kk * 16 * 128, C::CB_BYTES, SW128_ATOM);
      mma_f16_ts(o_tmem, p_tmem + kk * 8, vh, id, (accumulate || kk > 0) ? 1u : 0u);
      mma_f16_ts(o_tmem, p_tmem + kk * 8, vl, id, 1u);
      mma_f16_ts(o_tmem, p_tmem + 64 + kk * 8, vh, id, 1u);
    }
  } else {
    // A = P_hi / P_lo (fp32, TMEM, one column per key); B = V^T (K-major: rows = d).
    constexpr uint32_t id = make_idesc(128, C::D, FMT_TF32, FMT_TF32, false, false);
#pragma unroll
    for (int kk = 0; kk < BLOCK_N / 8; ++kk) {
      const uint32_t off = (kk / 4) * C::VT_CB_BYTES + (kk % 4) * 32;
      const uint64_t vh = make_sdesc(sv + off, 16, SW128_ATOM);
      const uint64_t vl = make_sdesc(sv_lo + off, 16, SW128_ATOM);
      mma_tf32_ts(o_tmem, p_tmem + kk * 8, vh, id, (accumulate || kk > 0) ? 1u : 0u);
      mma_tf32_ts(o_tmem, p_tmem + kk * 8, vl, id, 1);
      mma_tf32_ts(o_tmem, plo_tmem + kk * 8, vh, id, 1);
    }
  }
}

// TMA loads of key tile t into ring slot it % KST (K) / it % VST (V).
template <class C>
__device__ __forceinline__ void issue_k_load(uint8_t* smem, int it, int t, int bg,
                                             const CUtensorMap* tmK, const CUtensorMap* tmKlo,
                                             uint64_t* bar_kfull) {
  const int ks = it % C::KST;
  mbar_arrive_expect_tx(&bar_kfull[ks], C::NSPLIT * C::TILE_BYTES);
  for (int sp = 0; sp < C::NSPLIT; ++sp)
    for (int cb = 0; cb < C::NCB; ++cb)
      tma_load_3d(smem + C::K_OFF + (ks * C::NSPLIT + sp) * C::TILE_BYTES + cb * C::CB_BYTES,
                  sp ? tmKlo : tmK, &bar_kfull[ks], cb * C::ROW_ELEMS, t * BLOCK_N, bg);
}
template <class C>
__device__ __forceinline__ void issue_v_load(uint8_t* smem, int it, int t, int bg,
                                             const CUtensorMap* tmV, const CUtensorMap* tmVlo,
                                             uint64_t* bar_vfull) {
  const int vs = it % C::VST;
  mbar_arrive_expect_tx(&bar_vfull[vs], C::NSPLIT * C::TILE_BYTES);
  for (int sp = 0; sp < C::NSPLIT; ++sp) {
    uint8_t* dst = smem + C::V_OFF + vs * C::V_STAGE + sp * C::TILE_BYTES;
    if constexpr (!C::TF32) {
      for (int cb = 0; cb < C::NCB; ++cb)
        tma_load_3d(dst + cb * C::CB_BYTES, sp ? tmVlo : tmV, &bar_vfull[vs], cb * C::ROW_ELEMS,
                    t * BLOCK_N, bg);
    } else {  // V^T: 4 boxes of 32 keys x D rows
      for (int cb = 0; cb < 4; ++cb)
        tma_load_3d(dst + cb * C::VT_CB_BYTES, sp ? tmVlo : tmV, &bar_vfull[vs], t * BLOCK_N + cb * 32,
                    0, bg);
    }
  }
}

// Persistent: min(#work items, #SMs) CTAs; CTA c walks the work items (pairs of query
// tiles of one (batch, head), heaviest causal groups first) in rounds of gridDim.x,
// taking item c of even rounds and item G-1-c of odd ones so that every CTA's total
// stays close to the mean. Every ring and hand-off barrier counts across items: key
// tiles by g (K ring, S barriers), items with keys by j (Q tiles, O completion), and
// the V ring by position, where each item also takes NQ positions for its epilogue's
// staging. So the next item's Q tiles and first K tile load while the current item
// finishes, its first S MMAs are issued right after the current item's last PV, and
// the epilogue (O through the V ring to TMA stores) overlaps the other tile's MMAs.
// A phase of a per-item barrier can only complete after every role has observed the
// previous one (Q_q of item j+1 loads only after the last S MMA of item j completed,
// which needs Q_q of item j), so a parity wait never misses a phase.
//
// HP (head pairs, NQ = 2 only): the two query tiles of an item are the same 128 rows
// of two query heads of one kv head, which read the same K / V tiles, instead of two
// consecutive row tiles of one head. Both tiles then need exactly the item's key
// tiles (two row tiles of a causal or windowed item need different ones, so one of
// them computes a tile that is masked for it), and at Sq <= 128 no tile is padding.
//
// PSPLIT (bf16 inputs, short query sequences): P enters O += P V as two fp16 terms,
// P = hi + lo with hi = fp16(P), lo = fp16(P - hi): hi in the S slot's first 64
// columns as usual, lo in the other 64 (free once the softmax has read S), and a
// second PV MMA per tile. The next S MMA on the slot follows both in the issuer's
// order. Where one key takes almost all of a row's weight, one fp16 term (11
// significant bits) puts an error in O that the backward's D_i = dO_i . O_i then
// passes on to dS at exactly the dominant keys.
template <int D, int F32, bool HP, bool PSPLIT, int NQ_ = 0>
__global__ void __launch_bounds__(FwdCfg<D, F32, NQ_>::THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQlo,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmKlo,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmVlo,
                  const FwdArgs a) {
  using C = FwdCfg<D, F32, NQ_>;
  constexpr int NQ = C::NQ, KST = C::KST, VST = C::VST;
  if constexpr (C::F32) {
    // fp32 inputs: a programmatic dependent of the kernel that wrote the operand copies
    // and their scales (every thread reads one or the other)
    grid_launch_dependents();
    grid_dependency_wait();
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_q[NQ], bar_qfree[NQ], bar_kfull[KST], bar_kempty[KST],
      bar_vfull[VST], bar_vempty[VST], bar_grant[NQ], bar_s[NQ], bar_o[NQ], bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = warp_id();
  const int lane = lane_id();
  volatile int* abort_flag = &abort_sh;

  // ---- work items: query group qg (NQ tiles of 128 rows of head bh, or with HP 128
  // rows of heads bh, bh + 1) and key range sp (tiles [sp * tps, (sp + 1) * tps) when
  // the keys are split), linear index w = (qg_lin * BHi + u) * n_splits + sp, u the
  // head (pair), so the heads of one kv group are adjacent. Tile q's outputs go to
  // slab zo (+ q with HP), zo = sp * BH + bh (partial outputs when split).
  constexpr int ITEM_ROWS = HP ? BLOCK_M : BLOCK_M * NQ;
  static_assert(!HP || NQ == 2, "head pairs need two query tiles per item");
  struct Item { int bh, bg, zo, row0, t_lo, n; };
  auto item = [&](int w) {
    Item it;
    const int sp = w % a.n_splits, wq = w / a.n_splits;
    const int qg_lin = wq / a.BHi;
    const int u = wq % a.BHi;
    it.bh = HP ? 2 * u : u;
    it.zo = sp * a.BH + it.bh;
    const int qg = a.lpt ? (a.n_qgroups - 1 - qg_lin) : qg_lin;
    const int b = it.bh / a.H, h = it.bh % a.H;
    it.bg = b * a.HKV + h / (a.H / a.HKV);
    it.row0 = qg * ITEM_ROWS;
    int r1 = it.row0 + ITEM_ROWS - 1;
    if (r1 > a.Sq - 1) r1 = a.Sq - 1;
    int lo, hi;
    kv_tile_range(it.row0, r1, a.Sk, a.causal, a.window, &lo, &hi);
    if (a.n_splits > 1) {
      lo = max(lo, sp * a.tps);
      hi = min(hi, (sp + 1) * a.tps);
    }
    it.t_lo = lo;
    it.n = hi > lo ? hi - lo : 0;
    return it;
  };
  auto item_w = [&](int k) {
    const int G = gridDim.x, c = blockIdx.x;
    return k * G + ((k & 1) ? G - 1 - c : c);
  };
  const Item first = item(item_w(0));  // gridDim.x <= n_items: every CTA has round 0
  const bool setup_issued = first.n > 0;

  if (threadIdx.x == 0) {
    for (int q = 0; q < NQ; ++q) {
      mbar_init(&bar_q[q], 1);  // one per tile: S_0 need not wait for Q_1
      mbar_init(&bar_qfree[q], 1);
      mbar_init(&bar_s[q], 1);
      mbar_init(&bar_o[q], 1);
      mbar_init(&bar_grant[q], 1);
    }
    // a K / V stage is free once the MMAs of every tile that read it have completed
    // (or, for a V stage lent to an epilogue, once its TMA stores have read it)
    for (int s = 0; s < KST; ++s) { mbar_init(&bar_kfull[s], 1); mbar_init(&bar_kempty[s], 1); }
    for (int s = 0; s < VST; ++s) { mbar_init(&bar_vfull[s], 1); mbar_init(&bar_vempty[s], 1); }
    mbar_init(&bar_drain, 1);
    abort_sh = 0;
    fence_mbar_init();
    if (setup_issued) {
      // The first item's Q tiles and first K / V tiles are issued here, before the
      // TMEM allocation and the CTA-wide sync, so their latency overlaps the setup.
      for (int q = 0; q < NQ; ++q) {
        mbar_arrive_expect_tx(&bar_q[q], C::NSPLIT * C::TILE_BYTES);
        for (int sp = 0; sp < C::NSPLIT; ++sp)
          for (int cb = 0; cb < C::NCB; ++cb)
            tma_load_3d(smem + C::Q_OFF + (q * C::NSPLIT + sp) * C::TILE_BYTES + cb * C::CB_BYTES,
                        sp ? &tmQlo : &tmQ, &bar_q[q], cb * C::ROW_ELEMS,
                        first.row0 + (HP ? 0 : q * BLOCK_M), first.bh + (HP ? q : 0));
      }
      issue_k_load<C>(smem, 0, first.t_lo, first.bg, &tmK, &tmKlo, bar_kfull);
      issue_v_load<C>(smem, 0, first.t_lo, first.bg, &tmV, &tmVlo, bar_vfull);
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
  auto sQ = [&](int q, int sp) { return sbase + C::Q_OFF + (q * C::NSPLIT + sp) * C::TILE_BYTES; };
  auto sK = [&](int st, int sp) { return sbase + C::K_OFF + (st * C::NSPLIT + sp) * C::TILE_BYTES; };
  auto sV = [&](int st, int sp) { return sbase + C::V_OFF + st * C::V_STAGE + sp * C::TILE_BYTES; };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait(bar, parity, abort_flag, &g_fwd_status, DEV_TIMEOUT, a.limit_ns);
  };
  auto drain = [&](uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < a.limit_ns) {}
  };

  if (warp >= C::SOFTMAX_WARPS) {
  if constexpr (NQ == 2) regs_decrease<C::REGS_CONTROL>();
  if (warp == C::KQ_WARP) {
    // ------------------------------------------------------------ Q / K producer
    if (lane == 0) {
      int g = 0, j = 0;  // key tiles, items with keys
      int last_k[KST], last_q = setup_issued ? 0 : -1;
      for (int s = 0; s < KST; ++s) last_k[s] = (setup_issued && s == 0) ? 0 : -1;
      bool ok = true;
      for (int k = 0, w = item_w(0); ok && w < a.n_items; w = item_w(++k)) {
        const Item it = item(w);
        if (it.n == 0) continue;
        for (int t = 0; t < it.n; ++t, ++g) {
          if (k == 0 && t == 0) continue;  // issued with the setup
          const int ks = g % KST;
          if (!(ok = wait(&bar_kempty[ks], ((g / KST) & 1) ^ 1))) break;
          issue_k_load<C>(smem, g, it.t_lo + t, it.bg, &tmK, &tmKlo, bar_kfull);
          last_k[ks] = g / KST;
          if (t == 0) {
            // the item's Q tiles, each once the previous item's last S MMA on it completed
            for (int q = 0; ok && q < NQ; ++q) {
              if (j > 0 && !(ok = wait(&bar_qfree[q], (j - 1) & 1))) break;
              mbar_arrive_expect_tx(&bar_q[q], C::NSPLIT * C::TILE_BYTES);
              for (int sp = 0; sp < C::NSPLIT; ++sp)
                for (int cb = 0; cb < C::NCB; ++cb)
                  tma_load_3d(smem + C::Q_OFF + (q * C::NSPLIT + sp) * C::TILE_BYTES + cb * C::CB_BYTES,
                              sp ? &tmQlo : &tmQ, &bar_q[q], cb * C::ROW_ELEMS,
                              it.row0 + (HP ? 0 : q * BLOCK_M), it.bh + (HP ? q : 0));
            }
            if (!ok) break;
            last_q = j;
          }
        }
        ++j;
      }
      // Drain: every issued copy must land before the CTA may exit.
      for (int s = 0; s < KST; ++s)
        if (last_k[s] >= 0) drain(&bar_kfull[s], last_k[s] & 1);
      if (last_q >= 0)
        for (int q = 0; q < NQ; ++q) drain(&bar_q[q], last_q & 1);
    }
  } else if (warp == C::V_WARP) {
    // ------------------------------------------------------------ V producer
    // Every use of a V stage -- a key tile, or the staging area of an item's
    // epilogue -- has a ring position (per item: its key tiles, then one for the
    // epilogue) and is released once (by the MMAs' commit, or by the last query
    // tile's epilogue once its TMA stores have read the stage). This thread starts
    // every use in position order and is the only waiter on the empty barriers, so
    // it sees every release of a stage in order (seen[] counts them) and no parity
    // wait can skip a phase. Key tiles complete on the full barriers (only loads
    // count there); the epilogue stage goes to every query tile at once on the tiles'
    // grant barriers (one phase per item, only after the previous epilogue stage was
    // released), each tile staging through its own 1 / NQ of it, and the last tile
    // releases it once every tile's stores have read their part (EPI_JOIN).
    if (lane == 0) {
      uint32_t pos = 0;
      int seen[VST], loads[VST];  // releases seen, copies issued, per stage
      for (int s = 0; s < VST; ++s) { seen[s] = 0; loads[s] = (setup_issued && s == 0) ? 1 : 0; }
      int prev_stage = -1;
      bool ok = true;
      // wait until the use at position p has been released
      auto wait_release = [&](uint32_t p) {
        const int s = p % VST, u = p / VST;
        if (seen[s] > u) return true;
        if (!wait(&bar_vempty[s], u & 1)) return false;
        seen[s] = u + 1;
        return true;
      };
      for (int k = 0, w = item_w(0); ok && w < a.n_items; w = item_w(++k)) {
        const Item it = item(w);
        for (int t = 0; t < it.n; ++t, ++pos) {
          if (k == 0 && t == 0) continue;  // issued with the setup
          if (pos >= (uint32_t)VST && !(ok = wait_release(pos - VST))) break;
          issue_v_load<C>(smem, (int)pos, it.t_lo + t, it.bg, &tmV, &tmVlo, bar_vfull);
          ++loads[pos % VST];
        }
        if (!ok) break;
        if (pos >= (uint32_t)VST && !(ok = wait_release(pos - VST))) break;
        if (prev_stage >= 0 && !(ok = wait_release((uint32_t)prev_stage))) break;
        for (int q = 0; q < NQ; ++q) mbar_arrive(&bar_grant[q]);
        prev_stage = (int)pos;
        ++pos;
      }
      // Drain: every issued copy must land before the CTA may exit.
      for (int s = 0; s < VST; ++s)
        if (loads[s] > 0) drain(&bar_vfull[s], (loads[s] - 1) & 1);
    }
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // One warp issues every MMA (lane 0): per item S_0 = Q_0 K_0^T, S_1 = Q_1 K_0^T,
    // then in a fixed order per key tile g:
    //   O_0 += P_0 V_g, S_0 = Q_0 K_{g+1}^T, O_1 += P_1 V_g, S_1 = Q_1 K_{g+1}^T
    // (no S after the item's last tile; the next item's first S tiles follow its last
    // PVs in the pipe). The
    // tensor pipe runs them in that order, so S_0(g+1) completes one burst before
    // S_1(g+1): tile 0's softmax runs while tile 1's MMAs execute and vice versa.
    // (With one issuer per tile the two streams interleave in the pipe, both S tiles
    // complete together and both softmaxes compete for the exponential units.)
    // Inside the loop the issuer waits only on named barriers -- "P_q written"
    // (1 + q, from the softmax) and "operands loaded" (RELAY_BAR, from the relay
    // warp): an mbarrier wait right after a burst of MMAs returns only once the
    // burst has drained, which would idle the pipe between bursts. P_q aliases S_q
    // in TMEM; a thread's MMAs run in issue order, so S_q(g+1) after O_q += P_q V_g
    // is safe, and the next item's first O_q = P_q V (no accumulate) is issued only
    // after its softmax has read the previous O_q out of TMEM.
    const bool leader = lane == 0;
    int g = 0, j = 0;
    uint32_t pos = 0;
    for (int k = 0, w = item_w(0); w < a.n_items; w = item_w(++k)) {
      const int n = item(w).n;
      if (n == 0) { pos += 1; continue; }
      // item start: S_q(0) on the item's Q tiles and first K tile, once the relay has
      // seen them land (after the previous item's last PVs in the pipe)
      const int k0 = g % KST;
      for (int q = 0; q < NQ; ++q) {
        named_bar_sync(C::RELAY_BAR, 64);
        tc_fence_after();
        if (leader) {
          issue_qk<C>(tmem + C::s_col(q), sQ(q, 0), sQ(q, C::NSPLIT - 1), sK(k0, 0), sK(k0, C::NSPLIT - 1));
          tc_commit(&bar_s[q]);
          if (n == 1) tc_commit(&bar_qfree[q]);
        }
        __syncwarp();
      }
      if (leader) tc_commit(&bar_kempty[k0]);
      __syncwarp();
      // Every role takes part in every round of the named barriers, in order, whatever
      // happens: the issuer runs all rounds (it has no wait of its own that could
      // fail; after an abort its MMAs compute garbage that nobody stores), the relay
      // syncs each round, and a softmax warpgroup that gave up syncs (not merely
      // arrives) for its remaining rounds. A named barrier counts arrivals, so a role
      // that arrived for two rounds before its partner synced once would complete a
      // round without that partner and leave it waiting forever; in the normal flow
      // the softmax cannot run a round ahead (P_q(g+1) needs S_q(g+1), issued only
      // after the issuer passed round g).
      for (int t = 0; t < n; ++t, ++g, ++pos) {
        const int vs = pos % VST, ks = (g + 1) % KST;
        const bool more = t + 1 < n;
        named_bar_sync(C::RELAY_BAR, 64);  // V_g (and K_{g+1}) are in smem
        for (int q = 0; q < NQ; ++q) {
          named_bar_sync(1 + q, 128 + 32);  // P_q(g) is in TMEM
          tc_fence_after();
          if (leader) {
            issue_pv<C, PSPLIT>(tmem + C::o_col(q), tmem + C::s_col(q), tmem + C::PLO_COL, sV(vs, 0),
                        sV(vs, C::NSPLIT - 1), t > 0);
            if (more) {
              issue_qk<C>(tmem + C::s_col(q), sQ(q, 0), sQ(q, C::NSPLIT - 1), sK(ks, 0),
                          sK(ks, C::NSPLIT - 1));
              tc_commit(&bar_s[q]);
              if (t + 2 == n) tc_commit(&bar_qfree[q]);  // that was the item's last S_q
            } else {
              tc_commit(&bar_o[q]);  // tile q's last MMA: its epilogue may start
            }
          }
          __syncwarp();
        }
        if (leader) {
          tc_commit(&bar_vempty[vs]);
          if (more) tc_commit(&bar_kempty[ks]);
        }
        __syncwarp();
      }
      pos += 1;  // the epilogue's staging position
      ++j;
    }
    if (j > 0 && leader) {
      // Drain: no MMA may still be running when TMEM is released.
      tc_commit(&bar_drain);
      drain(&bar_drain, 0);
    }
    __syncwarp();
  } else if (warp == C::RELAY_WARP) {
    // ------------------------------------------------------------ load relay
    // Waits (on mbarriers, which this warp can do without stalling any MMA) until the
    // operands of the issuer's next bursts have landed and passes that on through
    // RELAY_BAR, the same number of syncs as the issuer (never a bare arrive: see the
    // issuer), also after an abort. It observes every phase of the full barriers in
    // order: per item Q_q and the first K tile, then K_{g+1} and V_g per key tile (the
    // V barriers count loads only, vc[] per stage); the issuer releases a K stage only
    // after its relay round, so no K phase can pass unobserved.
    bool ok = true;
    int g = 0, j = 0;
    uint32_t pos = 0;
    int vc[VST];
    for (int s = 0; s < VST; ++s) vc[s] = 0;
    for (int k = 0, w = item_w(0); w < a.n_items; w = item_w(++k)) {
      const int n = item(w).n;
      if (n == 0) { pos += 1; continue; }
      for (int q = 0; q < NQ; ++q) {  // item start: Q_q (and the first K tile)
        if (ok)
          ok = __all_sync(0xffffffffu, wait(&bar_q[q], j & 1) &&
                                           (q > 0 || wait(&bar_kfull[g % KST], (g / KST) & 1)));
        named_bar_sync(C::RELAY_BAR, 64);
      }
      for (int t = 0; t < n; ++t, ++g, ++pos) {
        const bool more = t + 1 < n;
        const int vs = pos % VST;
        if (ok)
          ok = __all_sync(0xffffffffu,
                          wait(&bar_vfull[vs], vc[vs] & 1) &&
                              (!more || wait(&bar_kfull[(g + 1) % KST], ((g + 1) / KST) & 1)));
        ++vc[vs];
        named_bar_sync(C::RELAY_BAR, 64);
      }
      pos += 1;
      ++j;
    }
  }  // idle warps of the control warpgroup fall through
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    if constexpr (NQ == 2) regs_increase<C::REGS_SOFTMAX>();
    const int q = warp / 4;
    const int wq = warp % 4;
    const int r_in = wq * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t s_addr = lane_addr + C::s_col(q);
    const uint32_t o_addr = lane_addr + C::o_col(q);
    // X16: the scores come from scaled copies of Q and K (sl2 carries 2^-(eQ + eK))
    const float sl2 = C::X16 ? a.sc->sl2 : a.scale_log2;
    const float o_mul = a.sc ? a.sc->o_mul : 1.f;  // O from the scaled V copy, back to V's units
    bool ok = true;
    int g = 0, j = 0;
    uint32_t pos = 0;
    // The last tile's epilogue gives the stage back to the V ring once every tile's
    // warps have read their parts of it back (EPI_JOIN): done after this warpgroup's
    // next hand-off, so that the join does not delay the next P.
    bool pending = false;
    int pend_slot = 0;
    auto release = [&]() {
      __syncwarp();
      if constexpr (NQ == 1) named_bar_sync(C::EPI_BAR0 + q, 128);
      else named_bar_sync(C::EPI_JOIN, 128 * NQ);
      if (wq == 0 && lane == 0) mbar_arrive(&bar_vempty[pend_slot]);
      pending = false;
    };
    for (int k = 0, w = item_w(0); w < a.n_items; w = item_w(++k)) {
      const Item itm = item(w);
      const int n = itm.n;
      const int r0 = itm.row0 + (HP ? 0 : q * BLOCK_M);
      const int zo = itm.zo + (HP ? q : 0);  // this tile's output slab
      const int i = r0 + r_in;  // this thread's query row
      // visible keys of row i: [lo_i, hi_i]
      const int hi_i = a.causal ? min(i, a.Sk - 1) : a.Sk - 1;
      const int lo_i = a.window > 0 ? i - a.window + 1 : INT_MIN / 2;
      float m = -FLT_MAX;  // running max of scale*log2(e)*S, possibly stale by < threshold
      float l = 0.f;
      for (int t = 0; t < n; ++t, ++g) {
        if (ok) ok = __all_sync(0xffffffffu, wait(&bar_s[q], g & 1));
        if (!ok) {
          // The issuer takes one round of named barrier 1 + q per key tile: join the
          // remaining rounds one by one (sync, not arrive) so that it can run out.
          named_bar_sync(1 + q, 128 + 32);
          if (pending) release();
          continue;
        }
        tc_fence_after();
        float s[128];
        {
          uint32_t v0[32], v1[32], v2[32], v3[32];
          tmem_ld32x4(s_addr, s_addr + 32, s_addr + 64, s_addr + 96, v0, v1, v2, v3);
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) {
            s[kk] = __uint_as_float(v0[kk]);
            s[32 + kk] = __uint_as_float(v1[kk]);
            s[64 + kk] = __uint_as_float(v2[kk]);
            s[96 + kk] = __uint_as_float(v3[kk]);
          }
        }
        const int c0 = (itm.t_lo + t) * BLOCK_N;
        if (tile_needs_mask(r0, r0 + BLOCK_M - 1, c0, c0 + BLOCK_N - 1, a.Sk, a.causal, a.window)) {
          mask_outside<128>(s, lo_i - c0, hi_i - c0);
        }
        // row max: eight chains of three-input maxima
        float mx[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mx[kk] = max3(s[kk], s[8 + kk], s[16 + kk]);
#pragma unroll
        for (int c = 24; c < 120; c += 16)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mx[kk] = max3(mx[kk], s[c + kk], s[c + 8 + kk]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mx[kk] = fmaxf(mx[kk], s[120 + kk]);
        const float mt =
            max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sl2;
        const bool need = mt > m + RESCALE_THRESHOLD;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m, mt);
          const float corr = ex2(m - m_new);
          l *= corr;
          if (t > 0) {
#pragma unroll
            for (int c = 0; c < C::D / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(o_addr + c * 32, r);
#pragma unroll
              for (int kk = 0; kk < 32; ++kk) r[kk] = __float_as_uint(__uint_as_float(r[kk]) * corr);
              tmem_st32(o_addr + c * 32, r);
            }
          }
          m = m_new;
        }
        const float nm = -m;
        float l0 = 0.f, l1 = 0.f;
        if constexpr (!C::TF32) {
          constexpr bool TWO = PSPLIT || C::X16;  // P as fp16 hi + lo
          // exponent arguments and the row sum on packed pairs
          const float2 sl2x2 = make_float2(sl2, sl2), nmx2 = make_float2(nm, nm);
          float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[32], pl[TWO ? 32 : 1];
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) {
              const float2 x = fma2(make_float2(s[c * 64 + 2 * kk], s[c * 64 + 2 * kk + 1]), sl2x2, nmx2);
              const float2 pp = make_float2(ex2(x.x), ex2(x.y));
              ls[kk & 1] = add2(ls[kk & 1], pp);
              if constexpr (TWO) {
                const __half2 h = __floats2half2_rn(pp.x, pp.y);
                const float2 hf = __half22float2(h);
                pk[kk] = *reinterpret_cast<const uint32_t*>(&h);
                pl[kk] = pack_half2(pp.x - hf.x, pp.y - hf.y);
              } else {
                pk[kk] = pack_half2(pp.x, pp.y);
              }
            }
            tmem_st32(s_addr + c * 32, pk);
            if constexpr (TWO) tmem_st32(s_addr + 64 + c * 32, pl);  // (S read in full above)
          }
          l0 = ls[0].x + ls[1].x;
          l1 = ls[0].y + ls[1].y;
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t ph[32], pl[32];
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) {
              const float p = ex2(fmaf(s[c * 32 + kk], sl2, nm));
              if (kk & 1) l1 += p; else l0 += p;
              const uint32_t hb = __float_as_uint(p) & 0xFFFFE000u;
              ph[kk] = hb;
              pl[kk] = __float_as_uint(p - __uint_as_float(hb));
            }
            tmem_st32(s_addr + c * 32, ph);
            tmem_st32(lane_addr + C::PLO_COL + c * 32, pl);
          }
        }
        l += l0 + l1;
        tmem_st_wait();
        tc_fence_before();
        named_bar_arrive(1 + q, 128 + 32);
        if (pending) release();
      }
      pos += n;
      if (n > 0) {
        if (ok) ok = __all_sync(0xffffffffu, wait(&bar_o[q], j & 1));
        tc_fence_after();
        ++j;
      }
      if (pending) release();
      // ---- epilogue: LSE, and O = acc / l staged in this tile's part of the item's V
      // ring stage (granted to every tile by the V producer), TMA stores.
      const int slot = pos % VST;
      if (ok) ok = __all_sync(0xffffffffu, wait(&bar_grant[q], k & 1));
      const float inv = (l > 0.f) ? (o_mul / l) : 0.f;
      if (ok && i < a.Sq)
        a.LSE[(size_t)zo * a.Sq + i] = (l > 0.f) ? (m + log2f(l)) * LN2 : -INFINITY;
      const int r_base = r0 + wq * 32;
      const uint32_t stage = sV(slot, 0) + (uint32_t)q * (C::V_STAGE / NQ) + wq * C::STAGE_PER_WARP;
      // (bf16 outputs: 64-column boxes, so D >= 64 kernels only; the host routes
      // bf16 outputs at smaller head dims to the D = 64 kernels)
      constexpr bool BF_OUT = D >= 64;
      // O rows staged box by box in this warp's share of the stage and written by the
      // warp itself (coalesced 16-byte stores): the share is free again when the call
      // returns, no copy-engine read to wait for
      if (ok) {
        if (BF_OUT && a.out_bf16)
          store_rows_direct<D, BF_OUT>(a.O, o_addr, n > 0, inv, stage, r_base, a.Sq, zo, a.Dv);
        else
          store_rows_direct<D, false>(a.O, o_addr, n > 0, inv, stage, r_base, a.Sq, zo, a.Dv);
      }
      if (q < NQ - 1) {
        // this tile is done with its part: the last tile may release the stage. (After
        // an abort a sync, so that this tile cannot arrive for the next item before the
        // last tile's release has taken this generation.)
        if (ok) named_bar_arrive(C::EPI_JOIN, 128 * NQ);
        else named_bar_sync(C::EPI_JOIN, 128 * NQ);
      } else {
        pending = true;
        pend_slot = slot;
      }
      pos += 1;
    }
    if (pending) release();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Rows that see no key at all (Sk == 0): O = 0, LSE = -inf.
__global__ void fill_empty_kernel(void* O, float* LSE, size_t rows, int D, int out_bf16) {
  for (size_t r = blockIdx.x * (size_t)blockDim.x + threadIdx.x; r < rows;
       r += (size_t)gridDim.x * blockDim.x) {
    LSE[r] = -INFINITY;
    if (out_bf16) {
      for (int d = 0; d < D; ++d) static_cast<__nv_bfloat16*>(O)[r * D + d] = __float2bfloat16(0.f);
    } else {
      for (int d = 0; d < D; ++d) static_cast<float*>(O)[r * D + d] = 0.f;
    }
  }
}

// The exponent of V's fp16 copy (the copy was made with exponent 0 by the conversion
// kernel, whose blocks left their largest |V| in part[]): every block reduces the
// partial maxima; block 0 publishes the multipliers, and if the exponent is not 0 the
// grid rewrites the copy as fp16(V * 2^eV).
__global__ void __launch_bounds__(1024) fwd_scales_kernel(const uint32_t* __restrict__ part,
                                                          int n_part, const __nv_bfloat16* V,
                                                          __half* V16, size_t n8,
                                                          OperandScales* out) {
  // launched as a programmatic dependent of the conversion: wait until that grid has
  // completed and its writes (the copy, part[]) are visible
  grid_dependency_wait();
  uint32_t m[1];
  reduce_partials<1>(part, n_part, m);
  const int ev = copy_exponent(m[0]);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    OperandScales sc = {};
    sc.sl2 = sc.dp_mul = sc.dq_mul = sc.dk_mul = sc.dv_mul = 1.f;
    sc.o_mul = pow2i(-ev);
    sc.e[SC_V] = ev;
    *out = sc;
  }
  if (ev != 0) rescale_copy(V, V16, n8, ev);
}

// fp32 inputs as two fp16 terms (X16): every block reduces the amax kernel's per-block maxima
// of |Q|, |K|, |V|, picks each tensor's exponent (x16_exponent), and the grid writes
// x 2^e = hi + lo as fp16 pairs; block 0 publishes the multipliers (scores:
// scale log2(e) 2^-(eQ + eK); O: 2^-eV).
struct X16FwdArgs {
  const uint32_t* part;
  int n_part;
  const float* src[3];  // Q, K, V
  __half* hi[3];
  __half* lo[3];
  size_t n4[3];
  float scale_log2;
  OperandScales* out;
};
__global__ void __launch_bounds__(256) x16_fwd_split_kernel(const __grid_constant__ X16FwdArgs a) {
  // a programmatic dependent of the amax pass: its partial maxima once it has completed
  grid_launch_dependents();
  grid_dependency_wait();
  uint32_t m[3];
  reduce_partials<3>(a.part, a.n_part, m);
  int e[3];
  for (int k = 0; k < 3; ++k) e[k] = x16_exponent(m[k]);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    OperandScales sc = {};
    sc.sl2 = ldexpf(a.scale_log2, -(e[0] + e[1]));
    sc.dp_mul = sc.dq_mul = sc.dk_mul = sc.dv_mul = 1.f;
    sc.o_mul = pow2i(-e[2]);
    sc.e[SC_Q] = e[0];
    sc.e[SC_K] = e[1];
    sc.e[SC_V] = e[2];
    *a.out = sc;
  }
  for (int k = 0; k < 3; ++k) split_x16(a.src[k], a.hi[k], a.lo[k], a.n4[k], e[k]);
}

// Key ranges of one query row computed separately: partial outputs O_s
// (each normalised by its own row sum) and natural-log LSE_s per range, slab
// s * rows + r. The row's result is the softmax over all its keys:
//   LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s
// (ranges with no visible key have LSE_s = -inf and weigh 0; a row with none at all
// gets O = 0, LSE = -inf). One pass over the ranges in order (deterministic), with a
// running maximum m: the sums are rescaled by exp(m_old - m_new) when a larger LSE_s
// arrives, so the LSE and partial-O loads of KEY_RANGE_GROUP ranges go out together
// (a separate pass for the maximum would cost another round trip to memory). Thread
// (x, y) of a block takes columns 4x.. of row blockIdx.x * blockDim.y + y of head
// blockIdx.y (+ multiples of gridDim.y).
__global__ void combine_splits_kernel(const float* __restrict__ Op, const float* __restrict__ Lp,
                                      void* __restrict__ O, float* __restrict__ LSE, int n_splits,
                                      int BH, int Sq, int Dv, int out_bf16) {
  constexpr int G = KEY_RANGE_GROUP;
  // a programmatic dependent of the forward kernel: its partial results once it has
  // completed (every thread waits, so this grid cannot complete before that one)
  grid_dependency_wait();
  const int i = blockIdx.x * blockDim.y + threadIdx.y;
  const int c = threadIdx.x * 4;
  if (i >= Sq || c >= Dv) return;
  const size_t rows = (size_t)BH * Sq;
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    const size_t r = (size_t)bh * Sq + i;
    float m = -INFINITY, sum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g0 = 0; g0 < n_splits; g0 += G) {
      float ls[G];
      float4 ov[G];
#pragma unroll
      for (int k = 0; k < G; ++k) {
        if (g0 + k < n_splits) {
          ls[k] = Lp[(g0 + k) * rows + r];
          ov[k] = *reinterpret_cast<const float4*>(Op + ((g0 + k) * rows + r) * Dv + c);
        }
      }
#pragma unroll
      for (int k = 0; k < G; ++k) {
        if (g0 + k < n_splits && ls[k] != -INFINITY) {
          if (ls[k] > m) {  // new maximum: rescale what was summed (exp(-inf) = 0 at first)
            const float sc = expf(m - ls[k]);
            sum *= sc;
            acc.x *= sc;
            acc.y *= sc;
            acc.z *= sc;
            acc.w *= sc;
            m = ls[k];
          }
          const float wgt = expf(ls[k] - m);
          sum += wgt;
          acc.x += wgt * ov[k].x;
          acc.y += wgt * ov[k].y;
          acc.z += wgt * ov[k].z;
          acc.w += wgt * ov[k].w;
        }
      }
    }
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    if (c == 0) LSE[r] = sum > 0.f ? m + logf(sum) : -INFINITY;
    if (out_bf16) {
      __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo2);
      u.y = *reinterpret_cast<uint32_t*>(&hi2);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(O) + r * Dv + c) = u;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(O) + r * Dv + c) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
  }
}

// The same merge for few rows with many ranges (the decode kernel's partial results):
// block (Dv / 4, SG) per row (rows blockIdx.x + multiples of gridDim.x), its SG thread
// groups dealt the ranges -- group g takes ranges g, g + SG, .. in order, with the
// running maximum above -- and the groups' (m, sum, O) merged in group order through
// shared memory: a row's loads go out from SG times as many threads, the order is fixed
// (deterministic). Dv <= 128, SG <= COMBINE_GROUPS.
constexpr int COMBINE_GROUPS = 16;
__global__ void combine_splits_grouped_kernel(const float* __restrict__ Op, const float* __restrict__ Lp,
                                              void* __restrict__ O, float* __restrict__ LSE,
                                              int n_splits, int rows, int Dv, int out_bf16) {
  constexpr int G = KEY_RANGE_GROUP;
  __shared__ float m_s[COMBINE_GROUPS], sum_s[COMBINE_GROUPS];
  __shared__ __align__(16) float acc_s[COMBINE_GROUPS][128];
  // a programmatic dependent of the decode kernel, as combine_splits_kernel
  grid_dependency_wait();
  const int c = threadIdx.x * 4, grp = threadIdx.y, SG = blockDim.y;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    float m = -INFINITY, sum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = grp; s0 < n_splits; s0 += SG * G) {
      float ls[G];
      float4 ov[G];
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int sp = s0 + k * SG;
        if (sp < n_splits) {
          ls[k] = Lp[(size_t)sp * rows + r];
          ov[k] = *reinterpret_cast<const float4*>(Op + ((size_t)sp * rows + r) * Dv + c);
        }
      }
#pragma unroll
      for (int k = 0; k < G; ++k) {
        if (s0 + k * SG < n_splits && ls[k] != -INFINITY) {
          if (ls[k] > m) {  // new maximum: rescale what was summed (exp(-inf) = 0 at first)
            const float sc = expf(m - ls[k]);
            sum *= sc;
            acc.x *= sc;
            acc.y *= sc;
            acc.z *= sc;
            acc.w *= sc;
            m = ls[k];
          }
          const float wgt = expf(ls[k] - m);
          sum += wgt;
          acc.x += wgt * ov[k].x;
          acc.y += wgt * ov[k].y;
          acc.z += wgt * ov[k].z;
          acc.w += wgt * ov[k].w;
        }
      }
    }
    if (threadIdx.x == 0) {
      m_s[grp] = m;
      sum_s[grp] = sum;
    }
    *reinterpret_cast<float4*>(&acc_s[grp][c]) = acc;
    __syncthreads();
    if (grp == 0) {
      float M = -INFINITY;
      for (int h = 0; h < SG; ++h) M = fmaxf(M, m_s[h]);
      float S = 0.f;
      float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
        for (int h = 0; h < SG; ++h) {
          const float w = expf(m_s[h] - M);  // (a group that saw no key: exp(-inf) = 0)
          const float4 a4 = *reinterpret_cast<const float4*>(&acc_s[h][c]);
          S += sum_s[h] * w;
          A.x += a4.x * w;
          A.y += a4.y * w;
          A.z += a4.z * w;
          A.w += a4.w * w;
        }
      }
      const float inv = S > 0.f ? 1.f / S : 0.f;
      if (c == 0) LSE[r] = S > 0.f ? M + logf(S) : -INFINITY;
      if (out_bf16) {
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(A.x * inv, A.y * inv);
        __nv_bfloat162 hi2 = __floats2bfloat162_rn(A.z * inv, A.w * inv);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo2);
        u.y = *reinterpret_cast<uint32_t*>(&hi2);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(O) + (size_t)r * Dv + c) = u;
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(O) + (size_t)r * Dv + c) =
            make_float4(A.x * inv, A.y * inv, A.z * inv, A.w * inv);
      }
    }
    __syncthreads();  // (the next row's groups overwrite the merge area)
  }
}

// ------------------------------------------------------------------ launcher
namespace {

// X16 (fp32 inputs as two fp16 terms): scratch bytes for the fp16 hi / lo copies of Q, K, V, the
// OperandScales and the amax kernel's n_amax x 3 partial maxima.
size_t x16_fwd_bytes(const fa_params& p, int n_amax) {
  const size_t nq = (size_t)p.B * p.H * p.Sq * p.D, nk = (size_t)p.B * p.HKV * p.Sk * p.D;
  return (2 * nq + 4 * nk) * 2 + 256 + (size_t)n_amax * 3 * 4;
}

// X16: the copies and scales in `ws` (x16_fwd_bytes of it) and their tensor maps.
bool prep_x16_fwd(void* ws, const void* Q, const void* K, const void* V, const fa_params& p,
                  int n_amax, cudaStream_t stream, CUtensorMap* mQ, CUtensorMap* mQlo,
                  CUtensorMap* mK, CUtensorMap* mKlo, CUtensorMap* mV, CUtensorMap* mVlo,
                  OperandScales** sc_out) {
  const int Dv = p.D;
  const size_t nq = (size_t)p.B * p.H * p.Sq * Dv, nk = (size_t)p.B * p.HKV * p.Sk * Dv;
  const uint64_t BHq = (uint64_t)p.B * p.H, BHk = (uint64_t)p.B * p.HKV;
  __half* qh = static_cast<__half*>(ws);
  __half* ql = qh + nq;
  __half* kh = ql + nq;
  __half* kl = kh + nk;
  __half* vh = kl + nk;
  __half* vl = vh + nk;
  char* tail = reinterpret_cast<char*>(vl + nk);
  OperandScales* sc = reinterpret_cast<OperandScales*>(tail);
  uint32_t* part = reinterpret_cast<uint32_t*>(tail + 256);
  AmaxJobs aj = {};
  aj.a[0] = static_cast<const float*>(Q);
  aj.a[1] = static_cast<const float*>(K);
  aj.a[2] = static_cast<const float*>(V);
  aj.n4[0] = nq / 4;
  aj.n4[1] = aj.n4[2] = nk / 4;
  aj.n = 3;
  {
    host::KernelTimer kt("amax(Q,K,V)", stream);
    amax_f32_kernel<3><<<n_amax, 256, 0, stream>>>(aj, part);
  }
  X16FwdArgs xa;
  xa.part = part;
  xa.n_part = n_amax;
  xa.src[0] = aj.a[0]; xa.src[1] = aj.a[1]; xa.src[2] = aj.a[2];
  xa.hi[0] = qh; xa.hi[1] = kh; xa.hi[2] = vh;
  xa.lo[0] = ql; xa.lo[1] = kl; xa.lo[2] = vl;
  xa.n4[0] = nq / 4; xa.n4[1] = xa.n4[2] = nk / 4;
  xa.scale_log2 = p.scale * LOG2E;
  xa.out = sc;
  {
    host::KernelTimer kt("x16_split(Q,K,V)", stream);
    // a programmatic dependent of the amax pass (it waits for it before reading)
    if (launch_programmatic(x16_fwd_split_kernel, dim3(n_amax), dim3(256), stream, xa) != cudaSuccess)
      return false;
  }
  const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  bool enc = host::encode_tiled_3d(mQ, F16, 2, qh, Dv, p.Sq, BHq, Dv, 64, 128);
  enc &= host::encode_tiled_3d(mQlo, F16, 2, ql, Dv, p.Sq, BHq, Dv, 64, 128);
  enc &= host::encode_tiled_3d(mK, F16, 2, kh, Dv, p.Sk, BHk, Dv, 64, 128);
  enc &= host::encode_tiled_3d(mKlo, F16, 2, kl, Dv, p.Sk, BHk, Dv, 64, 128);
  enc &= host::encode_tiled_3d(mV, F16, 2, vh, Dv, p.Sk, BHk, Dv, 64, 128);
  enc &= host::encode_tiled_3d(mVlo, F16, 2, vl, Dv, p.Sk, BHk, Dv, 64, 128);
  *sc_out = sc;
  return enc && cudaGetLastError() == cudaSuccess;
}

// The forward kernel instantiation: head-pair items (two-tile kernels only) or not;
// two-term P (bf16 inputs; fp32 inputs always carry P as two terms) or not.
template <int D, int F32, int NQ_ = 0>
auto fwd_kernel_for(bool hp, bool psplit) {
  auto kern = fa_fwd_kernel<D, F32, false, false, NQ_>;
  if constexpr (FwdCfg<D, F32, NQ_>::NQ == 2) {
    if (hp) kern = fa_fwd_kernel<D, F32, true, false, NQ_>;
    if constexpr (F32 == IN_BF16) {
      if (psplit) kern = hp ? fa_fwd_kernel<D, F32, true, true, NQ_> : fa_fwd_kernel<D, F32, false, true, NQ_>;
    }
  }
  return kern;
}

template <int D, int F32, int NQ_ = 0>
fa_status run_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                  const fa_params& p, cudaStream_t stream) {
  using C = FwdCfg<D, F32, NQ_>;
  const int Dv = p.D;
  const size_t nq = (size_t)p.B * p.H * p.Sq * Dv;
  const size_t nk = (size_t)p.B * p.HKV * p.Sk * Dv;
  const int grid_pp = 4 * host::sm_count();
  void* ws = nullptr;
  CUtensorMap mQ, mQlo, mK, mKlo, mV, mVlo;
  const uint64_t BHq = (uint64_t)p.B * p.H, BHk = (uint64_t)p.B * p.HKV;
  bool enc = true;
  OperandScales* sc = nullptr;
  if constexpr (!F32) {
    // fp16 copy of V | the call's OperandScales | the conversion blocks' partial maxima
    const int n_cvt = 2 * grid_pp;
    const size_t sc_off = (nk * 2 + 255) / 256 * 256;
    if (host::scratch_alloc(&ws, sc_off + 256 + (size_t)n_cvt * 4, stream) != cudaSuccess)
      return FA_ERR_CUDA;
    sc = reinterpret_cast<OperandScales*>(static_cast<char*>(ws) + sc_off);
    uint32_t* part = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + sc_off + 256);
    {
      host::KernelTimer kt("cvt_bf16_to_f16(V)", stream);
      cvt_bf16_to_f16_kernel<<<n_cvt, 256, 0, stream>>>(static_cast<const uint4*>(V),
                                                        static_cast<uint4*>(ws), nk / 8, part);
    }
    {
      host::KernelTimer kt("fwd_scales", stream);
      if (launch_programmatic(fwd_scales_kernel, dim3(host::sm_count()), dim3(1024), stream,
                              (const uint32_t*)part, n_cvt, static_cast<const __nv_bfloat16*>(V),
                              static_cast<__half*>(ws), nk / 8, sc) != cudaSuccess) {
        host::scratch_free(ws, stream);
        return FA_ERR_CUDA;
      }
    }
    enc &= host::encode_tiled_3d(&mQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Q, Dv, p.Sq, BHq, Dv,
                                 C::ROW_ELEMS, 128, C::RB);
    enc &= host::encode_tiled_3d(&mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, Dv, p.Sk, BHk, Dv,
                                 C::ROW_ELEMS, 128, C::RB);
    enc &= host::encode_tiled_3d(&mV, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ws, Dv, p.Sk, BHk, Dv,
                                 C::ROW_ELEMS, 128, C::RB);
    mQlo = mQ; mKlo = mK; mVlo = mV;
  } else if constexpr (C::X16) {
    const int n_amax = 8 * host::sm_count();
    if (host::scratch_alloc(&ws, x16_fwd_bytes(p, n_amax), stream) != cudaSuccess) return FA_ERR_CUDA;
    enc &= prep_x16_fwd(ws, Q, K, V, p, n_amax, stream, &mQ, &mQlo, &mK, &mKlo, &mV, &mVlo, &sc);
  } else {
    const int ldt = (p.Sk + 3) / 4 * 4;  // transposed V rows padded to 16 bytes
    const size_t nvt = (size_t)p.B * p.HKV * Dv * ldt;
    const size_t bytes = (2 * nq + 2 * nk + 2 * nvt) * 4;
    if (host::scratch_alloc(&ws, bytes, stream) != cudaSuccess) return FA_ERR_CUDA;
    float* qh = static_cast<float*>(ws);
    float* ql = qh + nq;
    float* kh = ql + nq;
    float* kl = kh + nk;
    float* vth = kl + nk;
    float* vtl = vth + nvt;
    host::KernelTimer kt("split_tf32(Q,K,V)", stream);
    launch_split_tf32({{static_cast<const float*>(Q), qh, ql, nullptr, nullptr, p.Sq, 0, (int)BHq},
                       {static_cast<const float*>(K), kh, kl, nullptr, nullptr, p.Sk, 0, (int)BHk},
                       {static_cast<const float*>(V), nullptr, nullptr, vth, vtl, p.Sk, ldt, (int)BHk}},
                      Dv, grid_pp, stream);
    enc &= host::encode_tiled_3d(&mQ, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, qh, Dv, p.Sq, BHq, Dv, 32, 128);
    enc &= host::encode_tiled_3d(&mQlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ql, Dv, p.Sq, BHq, Dv, 32, 128);
    enc &= host::encode_tiled_3d(&mK, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kh, Dv, p.Sk, BHk, Dv, 32, 128);
    enc &= host::encode_tiled_3d(&mKlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kl, Dv, p.Sk, BHk, Dv, 32, 128);
    // V^T: [BHk][D][ldt], inner extent Sk (row stride ldt), box 32 keys x D rows
    enc &= host::encode_tiled_3d(&mV, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, vth, p.Sk, Dv, BHk, ldt, 32, D);
    enc &= host::encode_tiled_3d(&mVlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, vtl, p.Sk, Dv, BHk, ldt, 32, D);
  }
  if (!enc) {
    host::scratch_free(ws, stream);
    return FA_ERR_CUDA;
  }
  FwdArgs a;
  a.O = O;
  a.LSE = LSE;
  a.H = p.H;
  a.HKV = p.HKV;
  a.Sq = p.Sq;
  a.Sk = p.Sk;
  a.scale_log2 = p.scale * LOG2E;
  a.causal = p.causal;
  a.window = p.window;
  a.out_bf16 = p.out_dtype == FA_BF16;
  // Two query tiles per item: two heads of one kv head when the group size is even,
  // else two row tiles of one head.
  const bool hp = C::NQ == 2 && (p.H / p.HKV) % 2 == 0;
  const int item_rows = hp ? BLOCK_M : BLOCK_M * C::NQ;
  a.n_qgroups = (p.Sq + item_rows - 1) / item_rows;
  a.BHi = hp ? (int)BHq / 2 : (int)BHq;
  // Fewer (query group, head (pair)) items than SMs -- short query sequences: split each
  // item's keys into ranges of tps tiles, each range a work item writing a partial O
  // and LSE, combined afterwards (key_range_tiles picks tps).
  const int sms = host::sm_count();
  const int n_kt = (p.Sk + BLOCK_N - 1) / BLOCK_N;
  const int base_items = a.BHi * a.n_qgroups;
  a.tps = key_range_tiles(base_items, n_kt, sms);
  a.n_splits = (n_kt + a.tps - 1) / a.tps;
  a.n_items = base_items * a.n_splits;
  a.Dv = Dv;
  a.lpt = p.causal ? 1 : 0;
  a.BH = (int)BHq;
  a.limit_ns = WAIT_LIMIT_NS;
  a.sc = sc;
  void* pws = nullptr;  // partial O [splits][BH][Sq][Dv] and LSE [splits][BH][Sq], fp32
  const size_t rows = (size_t)BHq * p.Sq;
  if (a.n_splits > 1) {
    const size_t o_floats = (size_t)a.n_splits * rows * Dv;
    if (host::scratch_alloc(&pws, (o_floats + (size_t)a.n_splits * rows) * 4, stream) != cudaSuccess) {
      host::scratch_free(ws, stream);
      return FA_ERR_CUDA;
    }
    a.O = pws;
    a.LSE = static_cast<float*>(pws) + o_floats;
    a.out_bf16 = 0;
  }
  const unsigned grid = (unsigned)std::min(a.n_items, sms);
  // two-term P for the shapes whose backward takes two-term P / dS (see split_operands)
  const bool psplit = !F32 && split_operands(p.H / p.HKV, (p.Sq + BLOCK_M - 1) / BLOCK_M);
  auto kern = fwd_kernel_for<D, F32, NQ_>(hp, psplit);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::SMEM_ALLOC);
  if (e == cudaSuccess) {
    host::KernelTimer kt(C::TF32 ? "fa_fwd_kernel<64,tf32>"
                         : F32 ? (D == 128 ? "fa_fwd_kernel<128,f32>" : "fa_fwd_kernel<64,f32>")
                             : (D == 128 ? "fa_fwd_kernel<128,bf16>"
                                         : (D == 64 ? "fa_fwd_kernel<64,bf16>" : "fa_fwd_kernel<32,bf16>")),
                         stream);
    if constexpr (F32 != IN_BF16) {
      // fp32: a programmatic dependent of the kernel that split the operands
      e = launch_programmatic_smem(kern, dim3(grid), dim3(C::THREADS), C::SMEM_ALLOC, stream, mQ,
                                   mQlo, mK, mKlo, mV, mVlo, a);
    } else {
      kern<<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(mQ, mQlo, mK, mKlo, mV, mVlo, a);
      e = cudaGetLastError();
    }
  }
  if (e == cudaSuccess && a.n_splits > 1) {
    host::KernelTimer kt("combine_splits", stream);
    const float* op = static_cast<const float*>(pws);
    dim3 cg, cb;
    combine_launch_shape((int)BHq, p.Sq, Dv, &cg, &cb);
    // a programmatic dependent of the forward kernel (it waits for it before reading)
    e = launch_programmatic(combine_splits_kernel, cg, cb, stream, op,
                            op + (size_t)a.n_splits * rows * Dv, O, LSE, a.n_splits, (int)BHq,
                            p.Sq, Dv, (int)(p.out_dtype == FA_BF16));
  }
  cudaError_t e2 = host::scratch_free(ws, stream);
  const cudaError_t e3 = host::scratch_free(pws, stream);
  return (e == cudaSuccess && e2 == cudaSuccess && e3 == cudaSuccess) ? FA_OK : FA_ERR_CUDA;
}

// The decode forward (fa_decode.cuh): the keys of each (batch, kv head) split into ranges
// so that one wave of CTAs (as many per SM as fit) streams K and V, each range at least
// one chunk per warp; with more than one range, partial O / LSE in scratch and the
// range-order combine.
// (fixed_ws: the no-allocation entry point's array, FA_NOALLOC_SCRATCH_BYTES, for the
// partial results instead of the memory pool)
template <int DK, int ROWS, bool F32IN>
fa_status run_decode(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     const fa_params& p, cudaStream_t stream, void* fixed_ws = nullptr) {
  DecodeArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
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
  a.scale_log2 = p.scale * LOG2E;
  a.out_bf16 = p.out_dtype == FA_BF16;
  a.k_wide = reinterpret_cast<uintptr_t>(K) % 32 == 0;
  constexpr size_t smem = decode_smem_bytes<DK, ROWS, F32IN>();
  auto kern = fa_decode_kernel<DK, ROWS, F32IN>;
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
    const size_t need = ((size_t)a.n_splits * rows_all * p.D + (size_t)a.n_splits * rows_all) * 4;
    if (fixed_ws) {
      if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;  // (nothing enqueued yet)
      pws = fixed_ws;
    } else if (host::scratch_alloc(&pws, need, stream) != cudaSuccess) {
      return FA_ERR_CUDA;
    }
    a.O = pws;
    a.LSE = static_cast<float*>(pws) + (size_t)a.n_splits * rows_all * p.D;
  } else {
    a.O = O;
    a.LSE = LSE;
  }
  {
    host::KernelTimer kt("fa_decode_kernel", stream);
    kern<<<dim3((unsigned)groups, (unsigned)a.n_splits), DEC_WARPS * 32, smem, stream>>>(a);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess && a.n_splits > 1) {
    host::KernelTimer kt("combine_splits", stream);
    const int q4 = p.D / 4;
    const int sg = std::max(1, std::min({256 / q4, a.n_splits, COMBINE_GROUPS}));
    const dim3 cg((unsigned)std::min<size_t>(rows_all, 65535)), cb(q4, sg);
    const float* op = static_cast<const float*>(pws);
    e = launch_programmatic(combine_splits_grouped_kernel, cg, cb, stream, op,
                            op + (size_t)a.n_splits * rows_all * p.D, O, LSE, a.n_splits, (int)rows_all,
                            p.D, (int)(p.out_dtype == FA_BF16));
  }
  const cudaError_t e2 = fixed_ws ? cudaSuccess : host::scratch_free(pws, stream);
  return (e == cudaSuccess && e2 == cudaSuccess) ? FA_OK : FA_ERR_CUDA;
}

template <int DK, bool F32IN>
fa_status run_decode_rows(const void* Q, const void* K, const void* V, void* O, float* LSE,
                          const fa_params& p, cudaStream_t stream, void* fixed_ws = nullptr) {
  const int rows = p.H / p.HKV * p.Sq;
  if (rows <= 4) return run_decode<DK, 4, F32IN>(Q, K, V, O, LSE, p, stream, fixed_ws);
  return run_decode<DK, DEC_ROWS, F32IN>(Q, K, V, O, LSE, p, stream, fixed_ws);
}

}  // namespace

fa_status launch_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     const fa_params& p, cudaStream_t stream) {
  if (p.Sk == 0) {
    const size_t rows = (size_t)p.B * p.H * p.Sq;
    fill_empty_kernel<<<4 * host::sm_count(), 256, 0, stream>>>(O, LSE, rows, p.D,
                                                                p.out_dtype == FA_BF16);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }
  if (decode_shaped(p)) {
    const bool f32 = p.in_dtype != FA_BF16;
    if (p.D <= 64) return f32 ? run_decode_rows<64, true>(Q, K, V, O, LSE, p, stream)
                              : run_decode_rows<64, false>(Q, K, V, O, LSE, p, stream);
    return f32 ? run_decode_rows<128, true>(Q, K, V, O, LSE, p, stream)
               : run_decode_rows<128, false>(Q, K, V, O, LSE, p, stream);
  }
  // head dims below a kernel's D run in it with the missing columns read as zeros
  if (p.in_dtype == FA_BF16) {
    // (the D = 32 kernel writes fp32 outputs only)
    if (p.D <= 32 && p.out_dtype == FA_F32) return run_fwd<32, IN_BF16>(Q, K, V, O, LSE, p, stream);
    if (p.D <= 64) return run_fwd<64, IN_BF16>(Q, K, V, O, LSE, p, stream);
    if (p.D <= 128) return run_fwd<128, IN_BF16>(Q, K, V, O, LSE, p, stream);
  } else if (p.f32_mma == FA_F32_MMA_TF32X3) {
    if (p.D <= 64) return run_fwd<64, IN_F32_TF32>(Q, K, V, O, LSE, p, stream);
  } else {
    if (p.D <= 64) {
      // two query tiles per item, unless that leaves SMs idle which one tile per item
      // would fill: key ranges split items only where the keys are long
      const int sms = host::sm_count(), n_qt = (p.Sq + BLOCK_M - 1) / BLOCK_M;
      const int n_kt = (p.Sk + BLOCK_N - 1) / BLOCK_N;
      const long long bh = (long long)p.B * p.H, items1 = bh * n_qt, items2 = bh * ((n_qt + 1) / 2);
      const bool one = items2 < sms && (items1 >= sms || key_range_tiles((int)items2, n_kt, sms) == n_kt);
      return one ? run_fwd<64, IN_F32_X16, 1>(Q, K, V, O, LSE, p, stream)
                 : run_fwd<64, IN_F32_X16>(Q, K, V, O, LSE, p, stream);
    }
    if (p.D <= 128) return run_fwd<128, IN_F32_X16>(Q, K, V, O, LSE, p, stream);
  }
  return FA_ERR_UNSUPPORTED;
}

// ------------------------------------------------------- barrier-timeout self test
// A one-CTA kernel with the same control skeleton as the attention kernels
// (TMEM allocation, a producer, a consumer waiting on a full barrier, bounded
// waits, abort propagation, TMEM release), in which the producer deliberately
// never issues its copy: the consumer's wait must expire after `limit_ns`, record
// DEV_TIMEOUT in the device status word, make every other role leave, free TMEM
// and let the kernel return normally.
__global__ void __launch_bounds__(128, 1) selftest_timeout_kernel(unsigned long long limit_ns,
                                                                  int* roles_done) {
  __shared__ __align__(8) uint64_t bar_full, bar_empty;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = warp_id(), lane = lane_id();
  volatile int* abort_flag = &abort_sh;
  if (threadIdx.x == 0) {
    mbar_init(&bar_full, 1);
    mbar_init(&bar_empty, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(&tmem_base_sh, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (warp == 1) {
    // producer: the first slot is free at once; it "forgets" the copy, then waits
    // for the consumer to release the slot, which never happens
    if (lane == 0) {
      mbar_wait(&bar_empty, 1, abort_flag, &g_fwd_status, DEV_TIMEOUT, limit_ns);
      mbar_wait(&bar_empty, 0, abort_flag, &g_fwd_status, DEV_TIMEOUT, limit_ns);
      atomicAdd(roles_done, 1);
    }
  } else if (warp == 2) {
    // consumer: waits for data that never arrives
    if (lane == 0) {
      if (mbar_wait(&bar_full, 0, abort_flag, &g_fwd_status, DEV_TIMEOUT, limit_ns))
        mbar_arrive(&bar_empty);
      atomicAdd(roles_done, 1);
    }
  } else if (warp == 3) {
    // a whole warp blocked behind the consumer; it must leave once the abort is raised
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_empty, 0, abort_flag, &g_fwd_status,
                                                      DEV_TIMEOUT, limit_ns));
    if (lane == 0 && !ok) atomicAdd(roles_done, 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

fa_status launch_selftest_timeout(unsigned long long limit_ns, int* roles_done, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 128, 0, s>>>(limit_ns, roles_done);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ------------------------------------------------- forward without allocation
// fa_fwd_noalloc runs the same kernels as fa_fwd, but the temporary operand
// copies live in this file-scope device array instead of the library's memory
// pool, so the call itself never allocates device memory. Every GPU that loads
// the library holds these bytes until the process exits.
static __device__ __align__(256) uint8_t g_fwd_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[NOALLOC_MAX_DEVICES] = {};

// Device address of the array on the current device. The symbol's host-side name
// is only a stand-in; the address is looked up once per device, with that device
// current, and cached.
fa_status noalloc_scratch_addr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES)
    return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fwd_noalloc_scratch) != cudaSuccess || !ptr)
      return FA_ERR_CUDA;
    g_noalloc_addr[dev] = ptr;
  }
  *out = g_noalloc_addr[dev];
  return FA_OK;
}

// Scratch bytes the problem needs, in double so that no product can wrap around
// (exact while it is anywhere near the array's size). bf16: the fp16 copy of V, padded
// to 256 bytes, then the OperandScales and one partial maximum per conversion block.
template <bool F32, bool X16>
double noalloc_bytes(const fa_params& p, int n_cvt) {
  const double nq = (double)p.B * p.H * p.Sq * p.D;
  const double nk = (double)p.B * p.HKV * p.Sk * p.D;
  if constexpr (!F32) {
    return std::ceil(nk * 2 / 256) * 256 + 256 + 4.0 * n_cvt;
  } else if constexpr (X16) {  // fp16 hi / lo of Q, K, V, the scales, the amax partials
    return (2 * nq + 4 * nk) * 2 + 256 + 12.0 * n_cvt;
  } else {
    const double ldt = (double)(((long long)p.Sk + 3) / 4 * 4);
    const double nvt = (double)p.B * p.HKV * p.D * ldt;
    return (2 * nq + 2 * nk + 2 * nvt) * 4;
  }
}

template <int D, int F32>
fa_status run_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE,
                          const fa_params& p, cudaStream_t stream) {
  using C = FwdCfg<D, F32>;
  const int n_cvt = 8 * host::sm_count();  // conversion blocks (bf16 inputs)
  if (noalloc_bytes<C::F32, C::X16>(p, n_cvt) > (double)FA_NOALLOC_SCRATCH_BYTES)
    return FA_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  const fa_status st = noalloc_scratch_addr(&ws);
  if (st != FA_OK) return st;
  const int Dv = p.D;
  const size_t nq = (size_t)p.B * p.H * p.Sq * Dv;
  const size_t nk = (size_t)p.B * p.HKV * p.Sk * Dv;
  const int grid_pp = 4 * host::sm_count();
  CUtensorMap mQ, mQlo, mK, mKlo, mV, mVlo;
  const uint64_t BHq = (uint64_t)p.B * p.H, BHk = (uint64_t)p.B * p.HKV;
  bool enc = true;
  // The whole scratch region used below is rewritten by the pre-pass kernels on
  // every call (the V copy, every conversion block's partial maximum, the scales),
  // so nothing left over from an earlier call is ever read.
  OperandScales* sc = nullptr;
  if constexpr (!F32) {
    const size_t sc_off = (nk * 2 + 255) / 256 * 256;
    sc = reinterpret_cast<OperandScales*>(static_cast<char*>(ws) + sc_off);
    uint32_t* part = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + sc_off + 256);
    cvt_bf16_to_f16_kernel<<<n_cvt, 256, 0, stream>>>(static_cast<const uint4*>(V),
                                                      static_cast<uint4*>(ws), nk / 8, part);
    if (launch_programmatic(fwd_scales_kernel, dim3(host::sm_count()), dim3(1024), stream,
                            (const uint32_t*)part, n_cvt, static_cast<const __nv_bfloat16*>(V),
                            static_cast<__half*>(ws), nk / 8, sc) != cudaSuccess)
      return FA_ERR_CUDA;
    enc &= host::encode_tiled_3d(&mQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Q, Dv, p.Sq, BHq, Dv,
                                 C::ROW_ELEMS, 128, C::RB);
    enc &= host::encode_tiled_3d(&mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, Dv, p.Sk, BHk, Dv,
                                 C::ROW_ELEMS, 128, C::RB);
    enc &= host::encode_tiled_3d(&mV, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ws, Dv, p.Sk, BHk, Dv,
                                 C::ROW_ELEMS, 128, C::RB);
    mQlo = mQ; mKlo = mK; mVlo = mV;
  } else if constexpr (C::X16) {
    enc &= prep_x16_fwd(ws, Q, K, V, p, n_cvt, stream, &mQ, &mQlo, &mK, &mKlo, &mV, &mVlo, &sc);
  } else {
    const int ldt = (p.Sk + 3) / 4 * 4;
    const size_t nvt = (size_t)p.B * p.HKV * Dv * ldt;
    float* qh = static_cast<float*>(ws);
    float* ql = qh + nq;
    float* kh = ql + nq;
    float* kl = kh + nk;
    float* vth = kl + nk;
    float* vtl = vth + nvt;
    launch_split_tf32({{static_cast<const float*>(Q), qh, ql, nullptr, nullptr, p.Sq, 0, (int)BHq},
                       {static_cast<const float*>(K), kh, kl, nullptr, nullptr, p.Sk, 0, (int)BHk},
                       {static_cast<const float*>(V), nullptr, nullptr, vth, vtl, p.Sk, ldt, (int)BHk}},
                      Dv, grid_pp, stream);
    enc &= host::encode_tiled_3d(&mQ, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, qh, Dv, p.Sq, BHq, Dv, 32, 128);
    enc &= host::encode_tiled_3d(&mQlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ql, Dv, p.Sq, BHq, Dv, 32, 128);
    enc &= host::encode_tiled_3d(&mK, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kh, Dv, p.Sk, BHk, Dv, 32, 128);
    enc &= host::encode_tiled_3d(&mKlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kl, Dv, p.Sk, BHk, Dv, 32, 128);
    enc &= host::encode_tiled_3d(&mV, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, vth, p.Sk, Dv, BHk, ldt, 32, D);
    enc &= host::encode_tiled_3d(&mVlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, vtl, p.Sk, Dv, BHk, ldt, 32, D);
  }
  if (!enc || cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  FwdArgs a;
  a.O = O;
  a.LSE = LSE;
  a.H = p.H;
  a.HKV = p.HKV;
  a.Sq = p.Sq;
  a.Sk = p.Sk;
  a.scale_log2 = p.scale * LOG2E;
  a.causal = p.causal;
  a.window = p.window;
  a.out_bf16 = p.out_dtype == FA_BF16;
  const bool hp = C::NQ == 2 && (p.H / p.HKV) % 2 == 0;  // head pairs (see run_fwd)
  const int item_rows = hp ? BLOCK_M : BLOCK_M * C::NQ;
  a.n_qgroups = (p.Sq + item_rows - 1) / item_rows;
  a.BHi = hp ? (int)BHq / 2 : (int)BHq;
  a.n_splits = 1;  // (split keys need scratch for the partial outputs)
  a.tps = (p.Sk + BLOCK_N - 1) / BLOCK_N;
  a.n_items = a.BHi * a.n_qgroups;
  a.Dv = Dv;
  a.lpt = p.causal ? 1 : 0;
  a.BH = (int)BHq;
  a.limit_ns = WAIT_LIMIT_NS;
  a.sc = sc;
  const unsigned grid = (unsigned)std::min(a.n_items, host::sm_count());
  // two-term P for the shapes whose backward takes two-term P / dS (see split_operands)
  const bool psplit = !F32 && split_operands(p.H / p.HKV, (p.Sq + BLOCK_M - 1) / BLOCK_M);
  auto kern = fwd_kernel_for<D, F32>(hp, psplit);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::SMEM_ALLOC);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if constexpr (F32 != IN_BF16) {
    // fp32: a programmatic dependent of the kernel that split the operands
    e = launch_programmatic_smem(kern, dim3(grid), dim3(C::THREADS), C::SMEM_ALLOC, stream, mQ, mQlo,
                                 mK, mKlo, mV, mVlo, a);
  } else {
    kern<<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(mQ, mQlo, mK, mKlo, mV, mVlo, a);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE,
                             const fa_params& p, cudaStream_t stream) {
  if (p.Sk == 0) {  // no key at all: no scratch needed
    const size_t rows = (size_t)p.B * p.H * p.Sq;
    fill_empty_kernel<<<4 * host::sm_count(), 256, 0, stream>>>(O, LSE, rows, p.D,
                                                                p.out_dtype == FA_BF16);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }
  if (decode_shaped(p)) {  // fa_fwd's decode kernel, its partial results in the array
    void* ws = nullptr;
    const fa_status st = noalloc_scratch_addr(&ws);
    if (st != FA_OK) return st;
    const bool f32 = p.in_dtype != FA_BF16;
    if (p.D <= 64) return f32 ? run_decode_rows<64, true>(Q, K, V, O, LSE, p, stream, ws)
                              : run_decode_rows<64, false>(Q, K, V, O, LSE, p, stream, ws);
    return f32 ? run_decode_rows<128, true>(Q, K, V, O, LSE, p, stream, ws)
               : run_decode_rows<128, false>(Q, K, V, O, LSE, p, stream, ws);
  }
  if (p.in_dtype == FA_BF16) {
    if (p.D <= 64) return run_fwd_noalloc<64, IN_BF16>(Q, K, V, O, LSE, p, stream);
    if (p.D <= 128) return run_fwd_noalloc<128, IN_BF16>(Q, K, V, O, LSE, p, stream);
  } else if (p.f32_mma == FA_F32_MMA_TF32X3) {
    if (p.D <= 64) return run_fwd_noalloc<64, IN_F32_TF32>(Q, K, V, O, LSE, p, stream);
  } else {
    if (p.D <= 64) return run_fwd_noalloc<64, IN_F32_X16>(Q, K, V, O, LSE, p, stream);
    if (p.D <= 128) return run_fwd_noalloc<128, IN_F32_X16>(Q, K, V, O, LSE, p, stream);
  }
  return FA_ERR_UNSUPPORTED;
}

unsigned int read_and_clear_fwd_status(cudaError_t* err) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_fwd_status, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(zero));
  if (err) *err = e;
  return v;
}

}  // namespace fa
