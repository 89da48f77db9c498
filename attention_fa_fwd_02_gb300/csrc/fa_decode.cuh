// Forward pass for decode-shaped problems: a handful of query rows per kv head (the
// grouped heads' Sq rows, at most DEC_ROWS of them) against many keys.
//
// There the tensor-core forward spends a 128-row MMA tile on each few rows and is bound
// by that padding, while the work itself -- every K and V row read once, a few dot
// products per key -- is bound by HBM bandwidth. This kernel streams K and V once with
// plain loads and does the arithmetic on the CUDA cores in fp32 (the products of bf16 or
// fp32 inputs are exact in fp32, so it is at least as accurate as the tensor paths), two
// lanes of it per instruction (the packed fp32 FMA):
//
//   grid (B * HKV, key ranges), 8 warps per CTA; a CTA takes one kv head's rows (head
//   r / Sq of the group, query r % Sq) over one key range, each warp 16-key chunks of it:
//     scores   lanes kl and kl + 16 = key j: each forms q_r . k_j over half the dims (q,
//              pre-scaled by scale * log2 e, from shared memory; its half of k_j straight
//              from global memory, 32 bytes per load; even and odd dims summed apart),
//              one shuffle adds the halves; masked per row -- while the chunk's V rows
//              copy into the warp's shared buffer (cp.async), and the next chunk's K row
//              is loaded as soon as this one's scores are formed;
//     softmax  per row online in the exp2 domain: m the running maximum (warp-uniform,
//              -inf until a key is visible), l the running sum (kept per lane, summed at
//              the end), O rescaled by 2^(m_old - m_new) when m grows;
//     PV       lane = DK / 32 columns: O_r += sum_j p_rj v_j, v_j from that buffer, the
//              weights of all rows through a second per-warp buffer [key][row], rows
//              taken in pairs.
//   The 8 warps' (m, l, O) merge in shared memory (over the V buffers, free by then); the
//   CTA writes its key range's partial O (normalised by its own l) and LSE, which
//   combine_splits_kernel merges in range order -- or, with one range, the final O and
//   LSE.
#pragma once

#include <type_traits>

namespace fa {

constexpr int DEC_ROWS = 8;      // query rows per kv head the decode kernel takes at most
constexpr int DEC_WARPS = 8;
constexpr int DEC_KEYS = 16;     // keys per warp chunk (two lanes per key)

struct DecodeArgs {
  const void* Q;
  const void* K;
  const void* V;
  void* O;        // final O (n_splits == 1) or partial O [n_splits][B*H][Sq][Dv] fp32
  float* LSE;     // final LSE or partial LSE [n_splits][B*H][Sq]
  int B, H, HKV, Sq, Sk, Dv, rep, rows;
  int causal, window;
  int keys_per_split, n_splits;
  int out_bf16;   // final outputs only
  int k_wide;     // K 32-byte aligned: its rows read 32 bytes per lane and load
  float scale_log2;
};

// Row r of a kv group: its query index i = r % Sq sees key j iff j < Sk, j <= i when
// causal, j >= i - window + 1 when windowed.
__device__ __forceinline__ bool dec_visible(int j, int i, int Sk, int causal, int window) {
  return j < Sk && (!causal || j <= i) && (window <= 0 || j >= i - window + 1);
}

// 16-byte global -> shared copies (cp.async, L2 only) and their completion
__device__ __forceinline__ void dec_cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void dec_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void dec_cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// one 32-byte global load (address 32-byte aligned) into two 16-byte halves: a whole
// sector per lane, so that no sector is asked of L2 twice
__device__ __forceinline__ void dec_ld32(const void* src, uint4& lo, uint4& hi) {
  asm("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
      : "l"(src));
}

// shared-memory layout: the V buffers [warps][DEC_KEYS][DK] of the input type (after the
// key loop the merge area [warps][ROWS][DK] fp32 over them), q [ROWS][DK] fp32, the
// weights [warps][DEC_KEYS][ROWS] fp32, then m and l [warps][ROWS]
template <int DK, bool F32IN>
__host__ __device__ constexpr size_t decode_v_bytes() { return (size_t)DEC_WARPS * DEC_KEYS * DK * (F32IN ? 4 : 2); }

// CTAs per SM the kernel is built for (registers per thread capped to fit them): the
// grid has about one wave of CTAs, each warp a chunk or two, so more warps in flight
// hide more of the loads' latency -- two for 4 rows; 8 rows need more registers than
// that leaves without spilling (and three CTAs of 4 rows spill and ran slower)
template <int ROWS>
__host__ __device__ constexpr int decode_min_ctas() { return ROWS == 4 ? 2 : 1; }

template <int DK, int ROWS, bool F32IN>
__global__ void __launch_bounds__(DEC_WARPS * 32, decode_min_ctas<ROWS>())
fa_decode_kernel(const DecodeArgs a) {
  static_assert(DK == 64 || DK == 128, "head dims up to 64 or 128: 2 or 4 columns per lane");
  static_assert(ROWS % 4 == 0 && ROWS <= DEC_ROWS, "rows per kv head: 4 or 8");
  static_assert((size_t)DEC_WARPS * ROWS * DK * 4 <= decode_v_bytes<DK, F32IN>(),
                "the merge area fits over the V buffers");
  constexpr int CPL = DK / 32;  // O columns per lane
  using T = typename std::conditional<F32IN, float, __nv_bfloat16>::type;
  constexpr int EPV = 16 / (int)sizeof(T);  // elements per 16-byte vector: 8 bf16 or 4 fp32
  constexpr int CPR = DK / EPV;             // 16-byte vectors per DK row: 8 to 32
  extern __shared__ __align__(16) unsigned char dsm_raw[];
  T* v_st = reinterpret_cast<T*>(dsm_raw);
  float* o_s = reinterpret_cast<float*>(dsm_raw);
  float* q_s = reinterpret_cast<float*>(dsm_raw + decode_v_bytes<DK, F32IN>());
  float* p_s = q_s + ROWS * DK;
  float* m_s = p_s + DEC_WARPS * DEC_KEYS * ROWS;
  float* l_s = m_s + DEC_WARPS * ROWS;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bg = blockIdx.x, split = blockIdx.y;  // bg = b * HKV + g (grid x: any count)
  const int b = bg / a.HKV, g = bg % a.HKV;
  const int k0 = split * a.keys_per_split;
  const int k1 = min(a.Sk, k0 + a.keys_per_split);
  const size_t kv_base = (size_t)bg * a.Sk * a.Dv;
  const T* Kg = static_cast<const T*>(a.K) + kv_base;
  const T* Vg = static_cast<const T*>(a.V) + kv_base;

  float* pw = p_s + warp * DEC_KEYS * ROWS;
  T* vw = v_st + warp * DEC_KEYS * DK;
  const uint32_t vw_s = (uint32_t)__cvta_generic_to_shared(vw);
  // this lane's V copies: vector lane % CPR of the rows lane / CPR + n * (32 / CPR)
  const int piece = lane % CPR;
  const bool copies = piece * EPV < a.Dv;  // (Dv a multiple of 16: whole vectors in or out)
  // the chunk's V rows into the warp's buffer (rows past the range repeat its last row:
  // their weights are 0)
  auto copy_v = [&](int j0) {
    if (copies) {
#pragma unroll
      for (int t = lane / CPR; t < DEC_KEYS; t += 32 / CPR) {
        const int jr = min(j0 + t, k1 - 1);
        dec_cp16(vw_s + (uint32_t)((t * DK + piece * EPV) * (int)sizeof(T)),
                 Vg + (size_t)jr * a.Dv + piece * EPV);
      }
    }
    dec_cp_commit();
  };
  // the lane's half of key j's K row: the 16-byte vectors [v0, v0 + NH) (zeros past Dv
  // or past the range)
  constexpr int NH = DK / EPV / 2;  // vectors per half row: 4 to 16
  const int kl = lane % DEC_KEYS, half = lane / DEC_KEYS, v0 = half * NH;
  auto load_k = [&](int j, uint4 (&raw)[NH]) {
    const T* krow = Kg + (size_t)j * a.Dv;
    if (j < k1 && a.k_wide) {
      // (Dv a multiple of 16 elements, d one of 2 EPV: a 32-byte load is all in or out)
#pragma unroll
      for (int t = 0; t < NH; t += 2) {
        const int d = (v0 + t) * EPV;
        if (d < a.Dv) {
          dec_ld32(krow + d, raw[t], raw[t + 1]);
        } else {
          raw[t] = make_uint4(0u, 0u, 0u, 0u);
          raw[t + 1] = raw[t];
        }
      }
    } else {
#pragma unroll
      for (int t = 0; t < NH; ++t) {
        const int d = (v0 + t) * EPV;
        raw[t] = j < k1 && d < a.Dv ? *reinterpret_cast<const uint4*>(krow + d)
                                    : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };

  // the first chunk's V copies and K row are in flight while the query rows are set up
  int j0 = k0 + warp * DEC_KEYS;
  uint4 kpre[NH];
  if (j0 < k1) copy_v(j0);
  load_k(j0 + kl, kpre);

  // the group's query rows, scaled: row r -> head g * rep + r / Sq, query r % Sq
  for (int e = threadIdx.x; e < ROWS * DK; e += blockDim.x) {
    const int r = e / DK, d = e % DK;
    float x = 0.f;
    if (r < a.rows && d < a.Dv) {
      const size_t qi = (((size_t)b * a.H + g * a.rep + r / a.Sq) * a.Sq + r % a.Sq) * a.Dv + d;
      x = F32IN ? static_cast<const float*>(a.Q)[qi]
                : __bfloat162float(static_cast<const __nv_bfloat16*>(a.Q)[qi]);
    }
    q_s[e] = x * a.scale_log2;
  }
  __syncthreads();

  // o2[rp][c] = (O[2 rp][c], O[2 rp + 1][c]) at this lane's columns c
  float m[ROWS], l[ROWS];
  float2 o2[ROWS / 2][CPL];
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
  }
#pragma unroll
  for (int rp = 0; rp < ROWS / 2; ++rp)
#pragma unroll
    for (int c = 0; c < CPL; ++c) o2[rp][c] = make_float2(0.f, 0.f);

  // s2[r] += q_r . k over the lane's half row, the even and odd dims in the two halves
  // of s2
  auto dot = [&](const uint4 (&raw)[NH], float2 (&s2)[ROWS]) {
#pragma unroll
    for (int t = 0; t < NH; ++t) {
      float2 kp[EPV / 2];  // (k_d, k_d+1) pairs
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
          const float4 q4 = *reinterpret_cast<const float4*>(q_s + r * DK + d + e4);
          s2[r] = __ffma2_rn(make_float2(q4.x, q4.y), kp[e4 / 2], s2[r]);
          s2[r] = __ffma2_rn(make_float2(q4.z, q4.w), kp[e4 / 2 + 1], s2[r]);
        }
      }
    }
  };

  for (; j0 < k1; j0 += DEC_WARPS * DEC_KEYS) {
    // ---- scores: lanes kl and kl + 16 = key j, each over half the row, then summed
    // (the same sum, in the same order, on both)
    const int j = j0 + kl;
    float2 s2[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) s2[r] = make_float2(0.f, 0.f);
    dot(kpre, s2);
    float s[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      s[r] = s2[r].x + s2[r].y;
      s[r] += __shfl_xor_sync(0xffffffffu, s[r], DEC_KEYS);
    }
    // the next chunk's K row is in flight through the softmax and PV
    const int jn = j0 + DEC_WARPS * DEC_KEYS;
    load_k(jn + kl, kpre);
    // ---- online softmax per row (m warp-uniform, l per lane: each key counted by both
    // of its lanes); four rows' weights at a time into the warp's [key][row] buffer
#pragma unroll
    for (int r4 = 0; r4 < ROWS; r4 += 4) {
      float p4[4], corr[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = r4 + u;
        const bool vis = r < a.rows && dec_visible(j, r % a.Sq, k1, a.causal, a.window);
        const float x = vis ? s[r] : -INFINITY;
        float mx = x;  // (both halves of the warp hold the same 16 keys)
#pragma unroll
        for (int off = DEC_KEYS / 2; off > 0; off >>= 1)
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m[r], mx);
        // (no visible key yet: m_new = -inf, every p = 0 and nothing is rescaled)
        corr[u] = m_new == -INFINITY ? 1.f : exp2f(m[r] - m_new);
        p4[u] = vis ? exp2f(x - m_new) : 0.f;
        l[r] = l[r] * corr[u] + p4[u];
        m[r] = m_new;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float2 cc = make_float2(corr[2 * h], corr[2 * h + 1]);
#pragma unroll
        for (int c = 0; c < CPL; ++c) o2[r4 / 2 + h][c] = __fmul2_rn(o2[r4 / 2 + h][c], cc);
      }
      if (half == 0)
        *reinterpret_cast<float4*>(pw + kl * ROWS + r4) = make_float4(p4[0], p4[1], p4[2], p4[3]);
    }
    dec_cp_wait_all();
    __syncwarp();
    // ---- O_r += sum_j p_rj v_j, lane = columns lane * CPL .., rows in pairs
    if (lane * CPL < a.Dv) {  // (Dv a multiple of 16: a lane's columns are all in or all out)
#pragma unroll 4
      for (int jj = 0; jj < DEC_KEYS; ++jj) {
        float v[CPL];
        const T* vp = vw + jj * DK + lane * CPL;
        if constexpr (F32IN) {
          if constexpr (CPL == 4) {
            const float4 x = *reinterpret_cast<const float4*>(vp);
            v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
          } else {
            const float2 x = *reinterpret_cast<const float2*>(vp);
            v[0] = x.x; v[1] = x.y;
          }
        } else {
          if constexpr (CPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(vp);
            const float2 x0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
            const float2 x1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
            v[0] = x0.x; v[1] = x0.y; v[2] = x1.x; v[3] = x1.y;
          } else {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vp));
            v[0] = x.x; v[1] = x.y;
          }
        }
        const float* pj = pw + jj * ROWS;
#pragma unroll
        for (int r4 = 0; r4 < ROWS; r4 += 4) {
          const float4 p4 = *reinterpret_cast<const float4*>(pj + r4);
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const float2 vv = make_float2(v[c], v[c]);
            o2[r4 / 2][c] = __ffma2_rn(make_float2(p4.x, p4.y), vv, o2[r4 / 2][c]);
            o2[r4 / 2 + 1][c] = __ffma2_rn(make_float2(p4.z, p4.w), vv, o2[r4 / 2 + 1][c]);
          }
        }
      }
    }
    __syncwarp();  // (the next chunk's copies and weights overwrite both buffers)
    if (jn < k1) copy_v(jn);
  }

  // every warp is past its last read of the V buffers before the merge area covers them
  __syncthreads();
  // ---- merge the warps: per row M = max_w m_w, L = sum_w l_w 2^(m_w - M), O likewise
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    float lr = l[r];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lr += __shfl_xor_sync(0xffffffffu, lr, off);
    lr *= 0.5f;  // (every key counted twice, by identical values: the halving is exact)
    if (lane == 0) {
      m_s[warp * ROWS + r] = m[r];
      l_s[warp * ROWS + r] = lr;
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c)
      o_s[(warp * ROWS + r) * DK + lane * CPL + c] = (r & 1) ? o2[r / 2][c].y : o2[r / 2][c].x;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < a.rows * DK; e += blockDim.x) {
    const int r = e / DK, d = e % DK;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) M = fmaxf(M, m_s[w * ROWS + r]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < DEC_WARPS; ++w) {
        const float f = exp2f(m_s[w * ROWS + r] - M);  // (a warp that saw no key: 2^-inf = 0)
        L += l_s[w * ROWS + r] * f;
        acc += o_s[(w * ROWS + r) * DK + d] * f;
      }
    }
    if (d >= a.Dv) continue;
    const size_t row = ((size_t)b * a.H + g * a.rep + r / a.Sq) * a.Sq + r % a.Sq;
    const float val = L > 0.f ? acc / L : 0.f;
    const float lse = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    if (a.n_splits == 1) {
      if (a.out_bf16) static_cast<__nv_bfloat16*>(a.O)[row * a.Dv + d] = __float2bfloat16(val);
      else static_cast<float*>(a.O)[row * a.Dv + d] = val;
      if (d == 0) a.LSE[row] = lse;
    } else {
      const size_t rows_all = (size_t)a.B * a.H * a.Sq;
      static_cast<float*>(a.O)[((size_t)split * rows_all + row) * a.Dv + d] = val;
      if (d == 0) a.LSE[(size_t)split * rows_all + row] = lse;
    }
  }
  // the combine kernel launched after this grid waits for it before reading
  ptx::grid_launch_dependents();
}

// Whether fa_fwd and fa_bwd take the decode kernels: every kv head's query rows (the
// grouped heads' Sq rows each) fit one CTA's DEC_ROWS.
inline bool decode_shaped(const fa_params& p) {
  return p.Sk > 0 && (long long)(p.H / p.HKV) * p.Sq <= DEC_ROWS;
}

template <int DK, int ROWS, bool F32IN>
constexpr size_t decode_smem_bytes() {
  return decode_v_bytes<DK, F32IN>() +
         4ull * (ROWS * DK + DEC_WARPS * DEC_KEYS * ROWS + 2 * DEC_WARPS * ROWS);
}

}  // namespace fa
