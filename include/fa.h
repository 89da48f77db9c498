/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library, libfa.so.
 *
 * The operation is exact softmax attention with the online-softmax forward and
 * the recompute-from-LSE backward described on the source pages:
 *
 *   O = softmax(scale * Q K^T + mask) V,   LSE_i = m_i + log(sum_j exp(S_ij - m_i))
 *
 *   - rustytorch "flash_attention_forward.metal": kernel header comment (the
 *     formula), parameter block (batch, heads, seq_q, seq_kv, head_dim,
 *     softmax_scale, causal) and the LSE output, one float per query row;
 *   - forge "flash_attention.metal": FlashParams {B, T, H, HKV, scale, causal,
 *     window}, GQA head mapping hkv = h / (H / HKV), the sliding window that
 *     keeps keys j >= i - window + 1 (self included, 0 = full), and the backward
 *     kernels flash_attn_bwd_dq / _dv / _dk that rebuild P from L and use
 *     D_i = dO_i . O_i;
 *   - boostr "flash.wgsl": FlashParams with separate seq_len_q / seq_len_k and
 *     num_kv_heads, tensors laid out [B, heads, S, head_dim].
 *
 * Mask (top-left aligned when Sq != Sk): key j is visible to query i iff
 *   (!causal || j <= i) && (window == 0 || j >= i - window + 1) && j < Sk.
 * A query row that sees no key gets O_i = 0 and LSE_i = -inf, and contributes
 * nothing to the gradients.
 *
 * Precision. in_dtype FA_BF16: QK^T and dO V^T run on bf16/fp16 tensor cores
 * with fp32 accumulation; the probabilities P and dS enter the second GEMMs as
 * fp16. Their partner operands (V in the forward; Q, K, V, dO in the backward) are
 * copied to fp16 as x * 2^e, with one power of two e per tensor and call chosen from
 * the tensor's largest magnitude, and dS likewise from a bound on |dS|; the scaling is
 * undone in fp32. e = 0 when the largest magnitude is already in [0.25, 32768), else
 * e moves it into [2^14, 2^15). A copied value is exact where x * 2^e is an fp16
 * normal number; below that it rounds to fp16's subnormal spacing, an absolute error
 * of at most 2^-23 (e = 0) or 2^-39 (e != 0) of the tensor's largest magnitude. So
 * bf16 inputs of any magnitude whose scores and outputs fit in fp32 are supported
 * (e.g. gradients dO of 1e-7, V of 1e5).
 * in_dtype FA_F32: every GEMM uses three tensor-core products of a hi/lo split of its
 * operands, a = a_hi + a_lo, a_hi b_hi + a_hi b_lo + a_lo b_hi, giving close to fp32
 * accuracy (about 22 significant bits per operand). fa_params.f32_mma picks the terms:
 * FA_F32_MMA_F16X2 (0, the default) uses fp16 terms of x * 2^e (one power of two per
 * tensor and call, chosen from its largest magnitude as for the bf16 path) on the
 * fp16 tensor-core rate, at every supported head dim; FA_F32_MMA_TF32X3 uses tf32
 * terms (fp32's exponent range, no scaling) at half that rate, for D <= 64 only.
 * P and dS enter the second GEMMs as the same kind of pair. Outputs are written in
 * out_dtype (FA_F32 recommended; FA_BF16 rounds O / dQ / dK / dV to bf16 on store).
 * LSE is always fp32, natural log.
 *
 * Supported in this build: head dims D that are multiples of 16, 16 <= D <= 128, for
 * both input types (the pages' set 16, 32, 48, 64, 80, 96, 128 among them); other head
 * dims return FA_ERR_UNSUPPORTED. Each D runs in the kernels built for the next of 32
 * (bf16 inputs with fp32 outputs), 64 and 128, whose tensor-core work then includes
 * the zero columns up to that width.
 */
#ifndef FA_H_
#define FA_H_

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

/* ABI-compatible with cudaStream_t (a CUDA runtime / driver stream handle);
 * NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* fa_stream_t;

typedef enum { FA_F32 = 0, FA_BF16 = 1 } fa_dtype;

/* Tensor-core terms of the fp32-input path (see Precision above). */
typedef enum { FA_F32_MMA_F16X2 = 0, FA_F32_MMA_TF32X3 = 1 } fa_f32_mma;

typedef struct {
  int B;            /* batch size, >= 1 */
  int H;            /* query heads, >= 1 */
  int HKV;          /* key/value heads, >= 1, H % HKV == 0 (query head h reads kv head h / (H/HKV)) */
  int Sq;           /* query rows per head, >= 0 */
  int Sk;           /* key rows per head, >= 0 */
  int D;            /* head dim */
  float scale;      /* softmax scale applied to Q K^T (commonly 1/sqrt(D)); finite and > 0 */
  int causal;       /* 0 or 1: key j visible only if j <= i (top-left aligned) */
  int window;       /* >= 0; 0 = no window, else key j visible only if j >= i - window + 1 */
  fa_dtype in_dtype;  /* dtype of Q, K, V, dO */
  fa_dtype out_dtype; /* dtype of O, dQ, dK, dV */
  fa_f32_mma f32_mma; /* in_dtype FA_F32 only (a valid value is still required for bf16):
                         FA_F32_MMA_F16X2 (0) or FA_F32_MMA_TF32X3 (D <= 64, else
                         FA_ERR_UNSUPPORTED); a zero-initialised struct gets the first */
} fa_params;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* NULL pointer, bad shape, H % HKV != 0, bad enum */
  FA_ERR_UNSUPPORTED = 2, /* valid request this build does not implement (head dim, dtype pair) */
  FA_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned */
  FA_ERR_CUDA = 4,        /* a CUDA runtime / driver call or a kernel launch failed */
  FA_ERR_TIMEOUT = 5,     /* a kernel gave up waiting on an internal barrier (device status) */
  FA_ERR_SCRATCH_LIMIT = 6, /* fa_fwd_noalloc: the problem needs more than FA_NOALLOC_SCRATCH_BYTES */
  FA_ERR_LAYOUT = 7         /* a kernel found less shared memory than its layout needs (device
                               status; the kernel skipped its work, outputs undefined) */
} fa_status;

/*
 * Forward pass.
 *   Q   [B, H,   Sq, D]  in_dtype, contiguous, device memory
 *   K   [B, HKV, Sk, D]  in_dtype
 *   V   [B, HKV, Sk, D]  in_dtype
 *   O   [B, H,   Sq, D]  out_dtype, written (overwritten, never accumulated)
 *   LSE [B, H,   Sq]     fp32, written: natural-log log-sum-exp of each row's
 *                        scaled scores, -inf for rows with no visible key.
 * All pointers are caller-owned device memory, 16-byte aligned; outputs must not
 * alias inputs. The library keeps per-device state for the life of the process (its
 * memory pool, the fa_fwd_noalloc scratch address, the status word): do not call it
 * again on a device after cudaDeviceReset() on that device, which invalidates that
 * state. The call validates its arguments synchronously, then enqueues
 * work on `stream` and returns without waiting. Decode shapes -- at most 8 query rows
 * per kv head, (H / HKV) * Sq <= 8 -- run in a CUDA-core kernel that reads K and V once
 * and computes in fp32 for either input type (f32_mma does not apply there); every
 * other shape runs on the tensor cores. Temporary buffers (the scaled fp16 copy of V
 * and its scale factors for bf16 inputs; the hi/lo splits of Q, K, V for fp32 inputs;
 * for short query sequences, whose work items are fewer than the SMs, fp32 partial O
 * and LSE of up to 32 key ranges, combined in range order; for decode shapes, partial
 * O and LSE of as many key ranges as fill the GPU once, combined in a fixed order: so
 * results stay deterministic) are taken stream-ordered from a library-owned CUDA
 * memory pool and released on the same stream. Errors: FA_ERR_INVALID_ARG / _UNSUPPORTED / _ALIGNMENT before any work
 * is enqueued; FA_ERR_CUDA if a CUDA call or launch fails. Device-side barrier
 * timeouts are reported later by fa_device_status().
 */
FA_API fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                 const fa_params* p, fa_stream_t stream);

/*
 * Forward pass that never allocates device memory (no counterpart on the source
 * pages; an addition for callers that cannot allocate).
 *
 * fa_fwd takes its temporary buffers from a memory pool that the library grows
 * on demand. Some callers cannot let a library do that: runtimes that allocate
 * everything up front and must keep a fixed device-memory footprint afterwards
 * (real-time or safety-certified inference), hosts whose own allocator owns the
 * whole device and would be starved or fragmented by a second pool, and code
 * that runs where a cudaMalloc is not allowed or would block on a lock. For them
 * this entry point computes exactly what fa_fwd computes, with the same arguments,
 * rules and errors, but its scratch (the fp16 copy of V for bf16 inputs; the hi/lo
 * splits of Q, K, V for fp32 inputs; at decode shapes the decode kernel's partial
 * results) lives in a file-scope device array of FA_NOALLOC_SCRATCH_BYTES inside
 * libfa.so. Every GPU on which the library is loaded holds that array until the
 * process exits.
 *   - A problem whose scratch would not fit returns FA_ERR_SCRATCH_LIMIT before
 *     anything is enqueued. Decode shapes ((H / HKV) * Sq <= 8) need 4*(D+1)*B*H*Sq*n
 *     bytes for n key ranges (n = 1, no scratch, once B*HKV reaches twice the SM
 *     count; at most about 3 MB). Other shapes: bf16 inputs need
 *     round_up(B*HKV*Sk*D*2, 256) + 256 +
 *     32 * (the device's SM count) bytes (the fp16 copy of V, its scale factors and
 *     the conversion's partial maxima); fp32 inputs need
 *     2*(2*B*H*Sq*D + 4*B*HKV*Sk*D) + 256 + 96 * (SM count) bytes with
 *     FA_F32_MMA_F16X2 and 4*(2*B*H*Sq*D + 2*B*HKV*Sk*D + 2*B*HKV*D*round_up(Sk,4))
 *     bytes with FA_F32_MMA_TF32X3.
 *   - The first call on each device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture begins.
 *   - All calls on a device share the one array. Each call rewrites the part it
 *     uses before reading it, but two calls whose work overlaps on the GPU (on
 *     different streams, without ordering between them) race on it and give
 *     undefined results: order such calls on one stream or with events.
 *   - It makes no cudaMalloc, cudaFree or other allocating call.
 */
#define FA_NOALLOC_SCRATCH_BYTES ((unsigned long long)32 << 20)
FA_API fa_status fa_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                const fa_params* p, fa_stream_t stream);

/* FA_NOALLOC_SCRATCH_BYTES as compiled into this libfa.so (so that a caller built
 * against another copy of this header can check the size it relies on). Makes no
 * CUDA call. */
FA_API unsigned long long fa_noalloc_scratch_bytes(void);

/*
 * Backward pass for the loss L with upstream gradient dO = dL/dO.
 *   Q, K, V  as in fa_fwd;  O [B,H,Sq,D] out_dtype and LSE [B,H,Sq] fp32 as
 *   written by fa_fwd for the same inputs and params;  dO [B,H,Sq,D] in_dtype.
 *   dQ [B,H,Sq,D], dK [B,HKV,Sk,D], dV [B,HKV,Sk,D]  out_dtype, overwritten.
 * P is rebuilt tile by tile from LSE (never stored); D_i = rowsum(dO_i * O_i) is
 * computed first by a preprocess kernel; dK/dV are accumulated per key tile over
 * the grouped query heads without atomics (deterministic: two calls on the same
 * inputs give bit-identical results). Decode shapes ((H / HKV) * Sq <= 8, as for
 * fa_fwd) run in one CUDA-core kernel in fp32 for either input type: one pass over K
 * and V, D_i formed by that kernel, each key's dK / dV formed once, dQ summed over
 * key ranges in a fixed order. Workspace (D_i, the scaled fp16 or hi/lo-split operand
 * copies and their scale factors; for short query sequences with bf16 inputs, fp32
 * partial dQ of up to 32 key ranges, summed in range order; for short key
 * sequences, fp32 partial dK and dV of up to 32 query ranges, summed in range order;
 * for decode shapes, fp32 partial dQ of as many key ranges as fill the GPU
 * once) is stream-ordered from the library pool. O must be the output of fa_fwd for the same inputs (the dS
 * scaling bounds D_i by the largest |dO| and |V|). Same ownership, alignment and
 * error rules as fa_fwd. Outside decode shapes, for both input types the dQ kernel is
 * launched on `stream` as a programmatic dependent of the dK/dV kernel: it starts on
 * the SMs that dK/dV leaves idle and completes only after dK/dV has, so work enqueued
 * on `stream` afterwards sees all three gradients. (Inside both calls, most kernels after the
 * first are launched as programmatic dependents of the kernel before them; each such
 * kernel waits for that one before it reads its results and before it exits, and the
 * first kernel of a call is an ordinary launch, so stream order as the caller sees it
 * is unchanged.)
 */
FA_API fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, const fa_params* p,
                 fa_stream_t stream);

/*
 * Backward pass with dS materialised in device memory: the same contract, results and
 * errors as fa_bwd (for in_dtype FA_BF16; FA_F32 returns FA_ERR_UNSUPPORTED), by the
 * 5-product route of the metal-flash-attention README's backward-pass discussion
 * instead of fa_bwd's 7: the dK / dV kernel forms S^T, dP^T, P^T, dS^T per key tile,
 * accumulates dV and dK on chip and also writes dS^T (scaled fp16; two fp16 terms for
 * short query sequences) to a workspace of B*H*Sk*round_up(Sq,128)*2 bytes per term;
 * dQ = scale dS K is then a tensor-core GEMM over that buffer, with no second
 * recomputation of S and dP. The buffer costs its write and read in memory traffic
 * (about 2 GB at B=2, H=32, S=4096), which is more than the GEMM work it saves on
 * this GPU at long sequences; fa_bwd never takes this route by itself. Deterministic,
 * like fa_bwd. Workspace from the library pool, as for fa_bwd.
 */
FA_API fa_status fa_bwd_dsmat(const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                              const fa_params* p, fa_stream_t stream);

/*
 * Synchronizes `stream`, then reads and clears the library's device status word
 * on the current device: FA_ERR_LAYOUT if a kernel since the last call found less
 * shared memory than its layout needs, FA_ERR_TIMEOUT if one gave up on a barrier
 * wait (outputs are then undefined in both cases), FA_ERR_CUDA if the
 * synchronization itself failed, else FA_OK.
 * The status word is one per device, not per stream: kernels on every stream of
 * the device set bits in it, and the first fa_device_status() call after a fault
 * (on any stream) reports and clears it. A caller that runs the library on several
 * streams at once and needs to know which call failed must serialize status checks
 * with its own launches (or treat a reported fault as affecting all of them).
 */
FA_API fa_status fa_device_status(fa_stream_t stream);

/* Static, NUL-terminated description of a status code (never NULL). */
FA_API const char* fa_status_string(fa_status s);

/* Library version string, e.g. "fa-sm103a 0.1". */
FA_API const char* fa_version(void);

/*
 * Failure-detection self test (a diagnostic; no counterpart on the source pages).
 * Enqueues one small kernel built like the attention kernels -- TMEM allocation,
 * a producer, a consumer and a third role synchronised by mbarriers -- in which
 * the producer never issues its copy. Every wait in it gives up after `limit_ns`
 * nanoseconds (0 < limit_ns <= 1e10); the expiry must be reported as
 * FA_ERR_TIMEOUT by the next fa_device_status(), each of the three roles must
 * leave (adding 1 to *roles_done, a caller-owned, 16-byte aligned device int
 * that starts at 0), TMEM must be released, and the context stays usable.
 * Returns FA_OK once enqueued.
 */
FA_API fa_status fa_selftest_timeout(unsigned long long limit_ns, int* roles_done,
                                     fa_stream_t stream);

/*
 * Kernel timing (a measurement aid; no counterpart on the source pages).
 * fa_timing_enable(1) makes every later fa_fwd / fa_bwd call record a CUDA event
 * pair around each kernel it launches, on the caller's stream; fa_timing_enable(0)
 * stops recording and discards what was recorded. fa_timing_read() waits for the
 * recorded events, aggregates them per kernel name into out[0..max_entries) and
 * forgets them; it returns the number of distinct kernels (which may exceed
 * max_entries), or -1 on a CUDA error. Names are static strings owned by the
 * library. Not thread-safe with respect to concurrent fa_* calls on other threads.
 */
typedef struct {
  const char* name;  /* kernel name, e.g. "fa_fwd_kernel<128,bf16>" */
  int launches;      /* launches recorded since the last read */
  double total_ms;   /* sum of their event-measured durations */
} fa_kernel_time;

FA_API fa_status fa_timing_enable(int on);
FA_API int fa_timing_read(fa_kernel_time* out, int max_entries);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
