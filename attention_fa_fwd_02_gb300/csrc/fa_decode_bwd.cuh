// Backward pass for decode-shaped problems: the shapes the decode forward takes (at most
// DEC_ROWS query rows per kv head: the grouped heads' Sq rows), against many keys.
//
// The tensor-core backward pads those few rows to 128-row MMA tiles in both of its
// kernels. Here the gradients of each key depend on a handful of rows, so one pass over
// K and V on the CUDA cores, in fp32 (exact products of the bf16 or fp32 inputs), does
// all of it:
//
//   grid (B * HKV, key ranges), 8 warps per CTA; a CTA takes one kv head's rows over one
//   key range (the decode forward's split), each warp 16-key chunks of it. Lanes kl and
//   kl + 16 own key j = j0 + kl and hold half of its K and V rows (loaded straight from
//   global memory, the next chunk's while this one's gradients are formed):
//     S_rj  = q_r . k_j and dP_rj = dO_r . v_j, each lane over its half of the dims, one
//             shuffle adding the halves;
//     P_rj  = exp(scale S_rj - LSE_r) (visible keys, else 0), dS_rj = P_rj (dP_rj - D_r)
//             with D_r = dO_r . O_r formed by the CTA for its rows; P and dS of the
//             chunk go to per-warp [key][row] buffers.
//   Then, key by key, lane = DK / 32 columns (q_r and dO_r of those columns held in
//   registers, k_j from a per-warp shared copy of the chunk's K rows, cp.async):
//     dV_j  = sum_r P_rj dO_r and dK_j = scale sum_r dS_rj q_r, stored as whole rows
//             (coalesced): every key belongs to one warp of one CTA, so no sum crosses
//             CTAs and nothing is atomic;
//     dQ_r += dS_rj k_j, rows in pairs.
//   The 8 warps' dQ sum in warp order in shared memory; the CTA writes its range's
//   scale * dQ, which dq_splits_sum_kernel adds up in a fixed order -- or, with one
//   range, dQ itself.
#pragma once

#include "fa_decode.cuh"

namespace fa {

struct DecodeBwdArgs {
  const void* Q;
  const void* K;
  const void* V;
  const void* O;    // the forward's output, its type out_bf16
  const void* dO;   // the input type
  const float* LSE;
  void* dK;         // [B, HKV, Sk, Dv], the output type
  void* dV;
  void* dQ;         // final dQ (n_splits == 1) or partial dQ [n_splits][B*H*Sq][Dv] fp32
  int B, H, HKV, Sq, Sk, Dv, rep, rows;
  int causal, window;
  int keys_per_split, n_splits;
  int out_bf16;     // O, dQ, dK, dV in bf16
  int k_wide, v_wide;  // K / V 32-byte aligned: their rows read 32 bytes per load
  float scale, scale_log2;
};

// shared-memory layout: the K buffers [warps][DEC_KEYS][DK] of the input type (after the
// key loop the dQ merge area [warps][ROWS][DK] fp32 over them), q and dO [ROWS][DK] fp32,
// dS and P [warps][DEC_KEYS][ROWS] fp32, then LSE (log2 domain) and D [ROWS]
template <int DK, int ROWS, bool F32IN>
constexpr size_t decode_bwd_smem_bytes() {
  return decode_v_bytes<DK, F32IN>() + 4ull * (2 * ROWS * DK + 2 * DEC_WARPS * DEC_KEYS * ROWS + 2 * ROWS);
}

// CTAs per SM the kernel is built for: two at D <= 64 with 4 rows; else one (the K and V
// halves of the next chunk, q and dO at the lane's columns, and the dQ sums do not fit
// 128 registers per thread without spilling)
template <int DK, int ROWS, bool F32IN>
__host__ __device__ constexpr int decode_bwd_min_ctas() {
  return ROWS == 4 && DK == 64 ? 2 : 1;
}

template <int DK, int ROWS, bool F32IN>
__global__ void __launch_bounds__(DEC_WARPS * 32, (decode_bwd_min_ctas<DK, ROWS, F32IN>()))
fa_decode_bwd_kernel(const DecodeBwdArgs a) {
  static_assert(DK == 64 || DK == 128, "head dims up to 64 or 128: 2 or 4 columns per lane");
  static_assert(ROWS % 4 == 0 && ROWS <= DEC_ROWS, "rows per kv head: 4 or 8");
  static_assert(ROWS <= DEC_WARPS, "warp r forms row r's D_r");
  static_assert((size_t)DEC_WARPS * ROWS * DK * 4 <= decode_v_bytes<DK, F32IN>(),
                "the dQ merge area fits over the K buffers");
  constexpr int CPL = DK / 32;
  using T = typename std::conditional<F32IN, float, __nv_bfloat16>::type;
  constexpr int EPV = 16 / (int)sizeof(T);  // elements per 16-byte vector
  constexpr int CPR = DK / EPV;             // 16-byte vectors per DK row: 8 to 32
  constexpr int NH = DK / EPV / 2;          // vectors per half row: 4 to 16
  extern __shared__ __align__(16) unsigned char dsm_raw[];
  T* k_st = reinterpret_cast<T*>(dsm_raw);
  float* dq_s = reinterpret_cast<float*>(dsm_raw);
  float* q_s = reinterpret_cast<float*>(dsm_raw + decode_v_bytes<DK, F32IN>());
  float* do_s = q_s + ROWS * DK;
  float* ds_s = do_s + ROWS * DK;
  float* p_s = ds_s + DEC_WARPS * DEC_KEYS * ROWS;
  float* lse_s = p_s + DEC_WARPS * DEC_KEYS * ROWS;
  float* dd_s = lse_s + ROWS;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bg = blockIdx.x, split = blockIdx.y;  // bg = b * HKV + g
  const int b = bg / a.HKV, g = bg % a.HKV;
  const int k0 = split * a.keys_per_split;
  const int k1 = min(a.Sk, k0 + a.keys_per_split);
  const size_t kv_base = (size_t)bg * a.Sk * a.Dv;
  const T* Kg = static_cast<const T*>(a.K) + kv_base;
  const T* Vg = static_cast<const T*>(a.V) + kv_base;
  // row r of the group -> its index in [B, H, Sq]
  auto row_index = [&](int r) -> size_t {
    return ((size_t)b * a.H + g * a.rep + r / a.Sq) * a.Sq + r % a.Sq;
  };

  float* dsw = ds_s + warp * DEC_KEYS * ROWS;
  float* psw = p_s + warp * DEC_KEYS * ROWS;
  T* kw = k_st + warp * DEC_KEYS * DK;
  const uint32_t kw_s = (uint32_t)__cvta_generic_to_shared(kw);
  const int piece = lane % CPR;
  const bool copies = piece * EPV < a.Dv;  // (Dv a multiple of 16: whole vectors in or out)
  // the chunk's K rows into the warp's buffer (rows past the range repeat its last row:
  // their dS are 0)
  auto copy_k = [&](int j0) {
    if (copies) {
#pragma unroll
      for (int t = lane / CPR; t < DEC_KEYS; t += 32 / CPR) {
        const int jr = min(j0 + t, k1 - 1);
        dec_cp16(kw_s + (uint32_t)((t * DK + piece * EPV) * (int)sizeof(T)),
                 Kg + (size_t)jr * a.Dv + piece * EPV);
      }
    }
    dec_cp_commit();
  };
  const int kl = lane % DEC_KEYS, half = lane / DEC_KEYS, v0 = half * NH;
  // the lane's half of row j of `src` (K or V): vectors [v0, v0 + NH), zeros past Dv or
  // past the range
  auto load_half = [&](const T* src, int j, bool wide, uint4 (&raw)[NH]) {
    const T* row = src + (size_t)j * a.Dv;
    if (j < k1 && wide) {
#pragma unroll
      for (int t = 0; t < NH; t += 2) {
        const int d = (v0 + t) * EPV;
        if (d < a.Dv) {
          dec_ld32(row + d, raw[t], raw[t + 1]);
        } else {
          raw[t] = make_uint4(0u, 0u, 0u, 0u);
          raw[t + 1] = raw[t];
        }
      }
    } else {
#pragma unroll
      for (int t = 0; t < NH; ++t) {
        const int d = (v0 + t) * EPV;
        raw[t] = j < k1 && d < a.Dv ? *reinterpret_cast<const uint4*>(row + d)
                                    : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };

  // the first chunk's K copies and K, V halves are in flight while the rows are set up
  int j0 = k0 + warp * DEC_KEYS;
  uint4 kpre[NH], vpre[NH];
  if (j0 < k1) copy_k(j0);
  load_half(Kg, j0 + kl, a.k_wide != 0, kpre);
  load_half(Vg, j0 + kl, a.v_wide != 0, vpre);

  // the group's rows: q and dO (fp32), LSE in the log2 domain, D_r = dO_r . O_r
  for (int e = threadIdx.x; e < ROWS * DK; e += blockDim.x) {
    const int r = e / DK, d = e % DK;
    float q = 0.f, dov = 0.f;
    if (r < a.rows && d < a.Dv) {
      const size_t qi = row_index(r) * a.Dv + d;
      if constexpr (F32IN) {
        q = static_cast<const float*>(a.Q)[qi];
        dov = static_cast<const float*>(a.dO)[qi];
      } else {
        q = __bfloat162float(static_cast<const __nv_bfloat16*>(a.Q)[qi]);
        dov = __bfloat162float(static_cast<const __nv_bfloat16*>(a.dO)[qi]);
      }
    }
    q_s[e] = q;
    do_s[e] = dov;
  }
  if (warp < ROWS) {  // warp r forms row r's D (ROWS <= DEC_WARPS)
    const int r = warp;
    float acc = 0.f;
    if (r < a.rows) {
      const size_t base = row_index(r) * a.Dv;
      for (int d = lane; d < a.Dv; d += 32) {
        const float dov = F32IN ? static_cast<const float*>(a.dO)[base + d]
                                : __bfloat162float(static_cast<const __nv_bfloat16*>(a.dO)[base + d]);
        const float o = a.out_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.O)[base + d])
                                   : static_cast<const float*>(a.O)[base + d];
        acc = fmaf(dov, o, acc);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      dd_s[r] = acc;
      lse_s[r] = r < a.rows ? a.LSE[row_index(r)] * LOG2E : 0.f;
    }
  }
  __syncthreads();

  // s2[r] += x_r . y over the lane's half row, the even and odd dims apart
  auto dot = [&](const uint4 (&raw)[NH], const float* xs, float2 (&s2)[ROWS]) {
#pragma unroll
    for (int t = 0; t < NH; ++t) {
      float2 kp[EPV / 2];
      if constexpr (F32IN) {
        kp[0] = make_float2(__uint_as_float(raw[t].x), __uint_as_float(raw[t].y));
        kp[1] = make_float2(__uint_as_float(raw[t].z), __uint_as_float(raw[t].w));
      } else {
        const uint32_t w4[4] = {raw[t].x, raw[t].y, raw[t].z, raw[t].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          kp[e] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
      }
      const int d = (v0 + t) * EPV;
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
#pragma unroll
        for (int e4 = 0; e4 < EPV; e4 += 4) {
          const float4 x4 = *reinterpret_cast<const float4*>(xs + r * DK + d + e4);
          s2[r] = __ffma2_rn(make_float2(x4.x, x4.y), kp[e4 / 2], s2[r]);
          s2[r] = __ffma2_rn(make_float2(x4.z, x4.w), kp[e4 / 2 + 1], s2[r]);
        }
      }
    }
  };

  // q_r and dO_r at this lane's columns lane * CPL .., in column pairs
  float2 q_reg[ROWS][CPL / 2], do_reg[ROWS][CPL / 2];
#pragma unroll
  for (int r = 0; r < ROWS; ++r)
#pragma unroll
    for (int c2 = 0; c2 < CPL / 2; ++c2) {
      q_reg[r][c2] = *reinterpret_cast<const float2*>(q_s + r * DK + lane * CPL + 2 * c2);
      do_reg[r][c2] = *reinterpret_cast<const float2*>(do_s + r * DK + lane * CPL + 2 * c2);
    }
  float2 dq2[ROWS / 2][CPL];  // (dQ[2 rp][c], dQ[2 rp + 1][c]) at this lane's columns
#pragma unroll
  for (int rp = 0; rp < ROWS / 2; ++rp)
#pragma unroll
    for (int c = 0; c < CPL; ++c) dq2[rp][c] = make_float2(0.f, 0.f);

  for (; j0 < k1; j0 += DEC_WARPS * DEC_KEYS) {
    const int j = j0 + kl;
    float2 s2[ROWS], p2[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      s2[r] = make_float2(0.f, 0.f);
      p2[r] = make_float2(0.f, 0.f);
    }
    dot(kpre, q_s, s2);
    dot(vpre, do_s, p2);
    // the next chunk's K and V halves are in flight through the rest of this one
    const int jn = j0 + DEC_WARPS * DEC_KEYS;
    load_half(Kg, jn + kl, a.k_wide != 0, kpre);
    load_half(Vg, jn + kl, a.v_wide != 0, vpre);
    // P and dS of key j for every row (both lanes of the key hold the same values)
    float P[ROWS], dS[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      float s = s2[r].x + s2[r].y, dp = p2[r].x + p2[r].y;
      s += __shfl_xor_sync(0xffffffffu, s, DEC_KEYS);
      dp += __shfl_xor_sync(0xffffffffu, dp, DEC_KEYS);
      const bool vis = r < a.rows && dec_visible(j, r % a.Sq, k1, a.causal, a.window);
      P[r] = vis ? exp2f(fmaf(s, a.scale_log2, -lse_s[r])) : 0.f;
      dS[r] = P[r] * (dp - dd_s[r]);
    }
    // P and dS of the chunk's keys into the warp's [key][row] buffers
    if (half == 0) {
#pragma unroll
      for (int r4 = 0; r4 < ROWS; r4 += 4) {
        *reinterpret_cast<float4*>(psw + kl * ROWS + r4) =
            make_float4(P[r4], P[r4 + 1], P[r4 + 2], P[r4 + 3]);
        *reinterpret_cast<float4*>(dsw + kl * ROWS + r4) =
            make_float4(dS[r4], dS[r4 + 1], dS[r4 + 2], dS[r4 + 3]);
      }
    }
    dec_cp_wait_all();
    __syncwarp();
    // ---- per key of the chunk, lane = columns lane * CPL ..:
    //   dV_j = sum_r P_rj dO_r and dK_j = scale sum_r dS_rj q_r (q, dO of the lane's
    //   columns in registers), stored as whole rows; dQ_r += dS_rj k_j (k_j from the
    //   chunk's shared copy, rows in pairs)
    if (lane * CPL < a.Dv) {  // (Dv a multiple of 16: a lane's columns are all in or all out)
#pragma unroll 1
      for (int jj = 0; jj < DEC_KEYS; ++jj) {
        float kv[CPL];
        const T* kp = kw + jj * DK + lane * CPL;
        if constexpr (F32IN) {
          if constexpr (CPL == 4) {
            const float4 x = *reinterpret_cast<const float4*>(kp);
            kv[0] = x.x; kv[1] = x.y; kv[2] = x.z; kv[3] = x.w;
          } else {
            const float2 x = *reinterpret_cast<const float2*>(kp);
            kv[0] = x.x; kv[1] = x.y;
          }
        } else {
          if constexpr (CPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(kp);
            const float2 x0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
            const float2 x1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
            kv[0] = x0.x; kv[1] = x0.y; kv[2] = x1.x; kv[3] = x1.y;
          } else {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(kp));
            kv[0] = x.x; kv[1] = x.y;
          }
        }
        const float* pj = psw + jj * ROWS;
        const float* dj = dsw + jj * ROWS;
        float2 av[CPL / 2], ak[CPL / 2];  // dV_j, dK_j at the lane's columns, in pairs
#pragma unroll
        for (int c2 = 0; c2 < CPL / 2; ++c2) av[c2] = ak[c2] = make_float2(0.f, 0.f);
#pragma unroll
        for (int r4 = 0; r4 < ROWS; r4 += 4) {
          const float4 p4 = *reinterpret_cast<const float4*>(pj + r4);
          const float4 d4v = *reinterpret_cast<const float4*>(dj + r4);
          const float pr[4] = {p4.x, p4.y, p4.z, p4.w}, dr[4] = {d4v.x, d4v.y, d4v.z, d4v.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 pp = make_float2(pr[u], pr[u]), dd = make_float2(dr[u], dr[u]);
#pragma unroll
            for (int c2 = 0; c2 < CPL / 2; ++c2) {
              av[c2] = __ffma2_rn(pp, do_reg[r4 + u][c2], av[c2]);
              ak[c2] = __ffma2_rn(dd, q_reg[r4 + u][c2], ak[c2]);
            }
          }
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const float2 kk = make_float2(kv[c], kv[c]);
            dq2[r4 / 2][c] = __ffma2_rn(make_float2(d4v.x, d4v.y), kk, dq2[r4 / 2][c]);
            dq2[r4 / 2 + 1][c] = __ffma2_rn(make_float2(d4v.z, d4v.w), kk, dq2[r4 / 2 + 1][c]);
          }
        }
        if (j0 + jj < k1) {
          const size_t o = kv_base + (size_t)(j0 + jj) * a.Dv + lane * CPL;
          const float2 sc = make_float2(a.scale, a.scale);
#pragma unroll
          for (int c2 = 0; c2 < CPL / 2; ++c2) ak[c2] = __fmul2_rn(ak[c2], sc);
          if (a.out_bf16) {
            uint32_t uv[CPL / 2], uk[CPL / 2];
#pragma unroll
            for (int c2 = 0; c2 < CPL / 2; ++c2) {
              __nv_bfloat162 h = __floats2bfloat162_rn(av[c2].x, av[c2].y);
              uv[c2] = *reinterpret_cast<uint32_t*>(&h);
              h = __floats2bfloat162_rn(ak[c2].x, ak[c2].y);
              uk[c2] = *reinterpret_cast<uint32_t*>(&h);
            }
            __nv_bfloat16* dVo = static_cast<__nv_bfloat16*>(a.dV) + o;
            __nv_bfloat16* dKo = static_cast<__nv_bfloat16*>(a.dK) + o;
            if constexpr (CPL == 4) {
              *reinterpret_cast<uint2*>(dVo) = make_uint2(uv[0], uv[1]);
              *reinterpret_cast<uint2*>(dKo) = make_uint2(uk[0], uk[1]);
            } else {
              *reinterpret_cast<uint32_t*>(dVo) = uv[0];
              *reinterpret_cast<uint32_t*>(dKo) = uk[0];
            }
          } else {
            float* dVo = static_cast<float*>(a.dV) + o;
            float* dKo = static_cast<float*>(a.dK) + o;
            if constexpr (CPL == 4) {
              *reinterpret_cast<float4*>(dVo) = make_float4(av[0].x, av[0].y, av[1].x, av[1].y);
              *reinterpret_cast<float4*>(dKo) = make_float4(ak[0].x, ak[0].y, ak[1].x, ak[1].y);
            } else {
              *reinterpret_cast<float2*>(dVo) = av[0];
              *reinterpret_cast<float2*>(dKo) = ak[0];
            }
          }
        }
      }
    }
    __syncwarp();  // (the next chunk's copies and dS overwrite both buffers)
    if (jn < k1) copy_k(jn);
  }

  // every warp is past its last read of the K buffers before the merge area covers them
  __syncthreads();
#pragma unroll
  for (int r = 0; r < ROWS; ++r)
#pragma unroll
    for (int c = 0; c < CPL; ++c)
      dq_s[(warp * ROWS + r) * DK + lane * CPL + c] = (r & 1) ? dq2[r / 2][c].y : dq2[r / 2][c].x;
  __syncthreads();
  for (int e = threadIdx.x; e < a.rows * DK; e += blockDim.x) {
    const int r = e / DK, d = e % DK;
    if (d >= a.Dv) continue;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) acc += dq_s[(w * ROWS + r) * DK + d];
    const float val = acc * a.scale;
    const size_t row = row_index(r);
    if (a.n_splits == 1) {
      if (a.out_bf16) static_cast<__nv_bfloat16*>(a.dQ)[row * a.Dv + d] = __float2bfloat16(val);
      else static_cast<float*>(a.dQ)[row * a.Dv + d] = val;
    } else {
      const size_t rows_all = (size_t)a.B * a.H * a.Sq;
      static_cast<float*>(a.dQ)[((size_t)split * rows_all + row) * a.Dv + d] = val;
    }
  }
  // the range sum launched after this grid waits for it before reading
  ptx::grid_launch_dependents();
}

// dQ = the sum of the key ranges' partial dQ [n_splits][rows][Dv] (fp32): block
// (Dv / 4, SG) per row (rows blockIdx.x + multiples of gridDim.x), group h adding ranges
// h, h + SG, .. in order, the groups' sums then added in group order (deterministic).
// Dv <= 128, SG <= DEC_SUM_GROUPS.
constexpr int DEC_SUM_GROUPS = 16;
__global__ void dq_splits_sum_kernel(const float* __restrict__ part, void* __restrict__ dQ,
                                     int n_splits, int rows, int Dv, int out_bf16) {
  constexpr int G = 8;  // ranges' loads in flight per thread
  __shared__ __align__(16) float acc_s[DEC_SUM_GROUPS][128];
  // a programmatic dependent of the decode backward kernel
  ptx::grid_dependency_wait();
  const int c = threadIdx.x * 4, grp = threadIdx.y, SG = blockDim.y;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = grp; s0 < n_splits; s0 += SG * G) {
      float4 v[G];
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int sp = s0 + k * SG;
        if (sp < n_splits) v[k] = *reinterpret_cast<const float4*>(part + ((size_t)sp * rows + r) * Dv + c);
      }
#pragma unroll
      for (int k = 0; k < G; ++k) {
        if (s0 + k * SG < n_splits) {
          acc.x += v[k].x;
          acc.y += v[k].y;
          acc.z += v[k].z;
          acc.w += v[k].w;
        }
      }
    }
    *reinterpret_cast<float4*>(&acc_s[grp][c]) = acc;
    __syncthreads();
    if (grp == 0) {
      float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int h = 0; h < SG; ++h) {
        const float4 a4 = *reinterpret_cast<const float4*>(&acc_s[h][c]);
        A.x += a4.x;
        A.y += a4.y;
        A.z += a4.z;
        A.w += a4.w;
      }
      if (out_bf16) {
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(A.x, A.y), hi2 = __floats2bfloat162_rn(A.z, A.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo2);
        u.y = *reinterpret_cast<uint32_t*>(&hi2);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(dQ) + (size_t)r * Dv + c) = u;
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(dQ) + (size_t)r * Dv + c) = A;
      }
    }
    __syncthreads();  // (the next row's groups overwrite the sums)
  }
}

}  // namespace fa
