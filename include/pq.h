/*
 * pq.h -- C ABI of the weight-only-quantized linear layer for GB300 (sm_103a).
 *
 * The layer computes y[M][N] = x[M][K] . W[K][N] where W is held as packed
 * low-bit codes with per-group scales:
 *
 *   4-bit GPTQ frame (W4A16) -- "mate: Marlin-class W4A16 GEMM for mp_31
 *   (SQMMA int4 x fp16) - #6", PR description: qweight words of eight 4-bit
 *   codes along K, fp16 scales per 128-row group, optional zero points and
 *   act-order g_idx.  w(k,n) = (code(k,n) - z(g,n)) * s(g,n), g the group of
 *   row k (g_idx[k] under act order).  Activations fp16/bf16, fp32
 *   accumulation, fp16/bf16 output.
 *
 *   ternary PQ2 (W2A8) -- "Kernel experiments: recorded evidence", Test 1 and
 *   Diagram 1 (34-byte blocks: fp16 scale + 32 code bytes per 128 weights,
 *   value = code - 1), Test 6 (int8 activation groups: scale = max|a|/127,
 *   nearest-even rounding, exact integer block dots), Test 21 (plane order,
 *   minus-one correction).  y[m][n] = sum_b S[m][n][b] * xs[m][b] * ws[n][b]
 *   with S the exact int32 block sum of (code-1)*q.
 *
 *   MLX affine 4-bit -- "qwen CUDA: --prompt-precision int8 ... - #1176":
 *   codes 0..15 with a scale and a bias per 64 inputs, w = s * q + b;
 *   fp16/bf16 activations.  y = sum_h s[h] (q . x over 64-group h) +
 *   b[h] (sum of x over h): the group dots on the tensor cores, scale and
 *   bias in fp32.
 *
 * Two calls make up the path: pq_prepare_* once at load time repacks the
 * caller's codes and scales into kernel-native planes; pq_linear runs the
 * layer on a stream.  Everything runs in this library's CUDA kernels; there is
 * no CPU fallback.
 *
 * Ownership: the caller allocates every device buffer (prepared planes,
 * workspace, x, y) and keeps it alive while the handle is used.  The library
 * allocates no device memory.  A pq_prepared handle is a small host object
 * pointing into the caller's memory; pq_destroy frees only that object.
 *
 * Streams are passed as `void*` holding a cudaStream_t (NULL = legacy default
 * stream).  Device pointers are plain CUDA device addresses.
 *
 * Errors: every entry point returns a pq_status.  Argument, shape and
 * alignment errors are detected on the host before any launch; the message
 * naming the violated invariant is available from pq_last_error() (thread
 * local).  Launch failures map to PQ_ERR_CUDA.  Bounded device-side waits
 * that expire record PQ_ERR_DEVICE_TIMEOUT in a status word inside the
 * workspace, read by pq_device_status.
 */
#ifndef PQ_H
#define PQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PQ_API __attribute__((visibility("default")))
#else
#define PQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define PQ_OK                    0
#define PQ_ERR_INVALID_ARG      -1  /* null pointer, bad enum, bad size      */
#define PQ_ERR_SHAPE            -2  /* K % 128 != 0, N < 1, M out of range   */
#define PQ_ERR_ALIGN            -3  /* device pointer not 16-byte aligned    */
#define PQ_ERR_GIDX             -4  /* act-order g_idx malformed             */
#define PQ_ERR_ZP_CONVENTION    -5  /* zero points given/missing vs the named convention */
#define PQ_ERR_UNSUPPORTED      -6  /* valid request this build does not run */
#define PQ_ERR_CUDA             -7  /* CUDA runtime/launch error             */
#define PQ_ERR_DEVICE_TIMEOUT   -8  /* a bounded device wait expired         */
#define PQ_ERR_BUFFER_TOO_SMALL -9  /* prepared / workspace buffer too small */

/* ---- enums ------------------------------------------------------------- */
#define PQ_FMT_W4_GPTQ   1  /* 4-bit codes, group 128 (MATE PR #6 frame)   */
#define PQ_FMT_W2_PQ2    2  /* ternary 2-bit PQ2 blocks (PRISM Test 1)     */
#define PQ_FMT_W4_AFFINE 3  /* MLX affine 4-bit: codes 0..15 with a scale
                               and a bias per 64 inputs, w = s*q + b
                               ("qwen CUDA: --prompt-precision int8 ...
                               #1176")                                  */

/* Zero-point convention, named by the caller and never guessed ("mate ...
 * #6", "Two defects": two packed conventions share shape and value multiset,
 * so the frame must be named).  Zero points are always passed UNPACKED. */
#define PQ_ZP_SYMMETRIC_8  0  /* no zero-point buffer; z = 8              */
#define PQ_ZP_EXPLICIT_U8  1  /* uint8 z[K/128][N] in 0..15, used as given */

#define PQ_F16   1
#define PQ_BF16  2

/* ---- layer descriptor -------------------------------------------------- */
typedef struct pq_desc {
    int32_t fmt;        /* PQ_FMT_*                                          */
    int32_t N;          /* output features, >= 1                             */
    int32_t K;          /* input features, multiple of 128 (W2: <= 65536)    */
    int32_t group;      /* weights per scale group along K: 128 (64 for
                           PQ_FMT_W4_AFFINE)                                 */
    int32_t zp;         /* PQ_ZP_* (W4 only; W2 must pass PQ_ZP_SYMMETRIC_8) */
    int32_t has_gidx;   /* W4 only: 1 if an act-order g_idx is supplied      */
    int32_t act_dtype;  /* PQ_F16 / PQ_BF16: dtype of x                      */
    int32_t out_dtype;  /* PQ_F16 / PQ_BF16: dtype of y                      */
    int32_t act_group;  /* W2 only: activation quantisation group, 128 or K  */
    int32_t max_m;      /* largest M passed to pq_linear (sizes workspace)   */
} pq_desc;

typedef struct pq_prepared pq_prepared;   /* opaque host handle */

/* Device bytes the caller must allocate for the prepared planes of `d`
 * (each plane starts on a 256-byte boundary).  Returns 0 if `d` is invalid
 * (pq_last_error says why).  Host-only; needs no GPU. */
PQ_API size_t pq_prepared_bytes(const pq_desc* d);

/* Device scratch bytes pq_linear needs for M <= d->max_m (act-order gather,
 * activation quantisation, split-K partials, the device status word, and for
 * max_m > 16 the prefill GEMM's flags and fp32 partial tiles: about 42 MB
 * once max_m >= 256).  Handles that never run concurrently may share one
 * workspace.  Never 0 for a valid descriptor.  Host-only; needs no GPU. */
PQ_API size_t pq_workspace_bytes(const pq_desc* d);

/* Repack a 4-bit GPTQ frame ("mate ... #6": prepare_w4a16_from_gptq_frame,
 * resolve_act_order).
 *   d_qweight  uint32 [K/8][N], code of row k in bits 4*(k%8) of word (k/8, n)
 *   d_scales   fp16   [K/128][N]
 *   d_zeros    uint8  [K/128][N] (values 0..15) iff d->zp == PQ_ZP_EXPLICIT_U8,
 *              else NULL (PQ_ERR_ZP_CONVENTION otherwise)
 *   h_g_idx    HOST int32 [K] iff d->has_gidx, else NULL.  Must assign exactly
 *              128 rows to every group 0..K/128-1 (PQ_ERR_GIDX names the first
 *              group that does not).  Rows are stored sorted by group
 *              (stable), and pq_linear gathers x with the same permutation,
 *              so x[:,perm] @ W[perm] == x @ W ("Act order").
 *   d_prepared  caller buffer of >= pq_prepared_bytes(d) bytes, 256-B aligned
 *   d_workspace caller buffer of >= pq_workspace_bytes(d) bytes, 256-B aligned;
 *              bound to the handle and used by every pq_linear call on it
 * Synchronises `stream` before returning (load-time call).  On success
 * *out receives a new handle (free with pq_destroy). */
PQ_API int32_t pq_prepare_w4(const pq_desc* d, const uint32_t* d_qweight,
                      const uint16_t* d_scales, const uint8_t* d_zeros,
                      const int32_t* h_g_idx, void* d_prepared,
                      size_t prepared_bytes, void* d_workspace,
                      size_t workspace_bytes, void* stream, pq_prepared** out);

/* Repack ternary PQ2 rows ("Kernel experiments: recorded evidence", Test 1
 * prepare_pq2 and Test 4: a code plane and a scale plane in one allocation,
 * same 34 bytes per 128 weights).
 *   d_raw   uint8 [N] rows of K/128 blocks of 34 bytes: little-endian fp16
 *           scale, then 32 code bytes; byte i holds weights 4i..4i+3 of the
 *           block, weight 4i+j in bits 2j..2j+1; value = code - 1.
 *   row_stride_bytes  distance between rows, >= K/128*34
 * Other arguments as pq_prepare_w4. */
PQ_API int32_t pq_prepare_w2(const pq_desc* d, const uint8_t* d_raw,
                      size_t row_stride_bytes, void* d_prepared,
                      size_t prepared_bytes, void* d_workspace,
                      size_t workspace_bytes, void* stream, pq_prepared** out);

/* Repack an MLX affine 4-bit weight (fmt = PQ_FMT_W4_AFFINE, group = 64,
 * zp = PQ_ZP_SYMMETRIC_8 meaning "no zero-point plane", has_gidx = 0).
 *   d_wq      uint32 [N][K/8]: code of input k of output row n in bits
 *             4*(k%8) of word (n, k/8), least significant first
 *   d_scales  [N][K/64] act_dtype (fp16 / bf16), the per-group scale s
 *   d_biases  [N][K/64] act_dtype, the per-group bias b; w = s * q + b
 * The codes are stored K-permuted inside every 128 inputs so that each
 * tensor-core k-step of the decode kernels stays inside one 64-group (the
 * GEMM reads each 64-group's codes back out of a block's tile).  K must be a
 * multiple of 128.  Other arguments as pq_prepare_w4.  pq_linear runs the
 * decode GEMV for M <= 16 and the tensor-core GEMM above; the GEMM's sums of
 * x live in the workspace, so it runs only for max_m > 16. */
PQ_API int32_t pq_prepare_affine4(const pq_desc* d, const uint32_t* d_wq, const uint16_t* d_scales,
                                  const uint16_t* d_biases, void* d_prepared, size_t prepared_bytes,
                                  void* d_workspace, size_t workspace_bytes, void* stream,
                                  pq_prepared** out);

/* y = x . W on `stream`; asynchronous, no host synchronisation, no
 * allocation.  The variant (decode GEMV or tensor-core GEMM) is chosen from
 * M by the dispatcher (see pq_plan).  A prefill GEMM whose CTAs share tiles
 * is launched cooperatively (all its CTAs resident at once).
 *   d_x  [M][K] act_dtype, rows contiguous, 16-B aligned
 *   d_y  [M][N] out_dtype, rows contiguous, 16-B aligned
 *   1 <= M <= desc.max_m
 * Calls on the same handle share its workspace: calls that overlap on the
 * GPU (different streams without ordering) race. */
PQ_API int32_t pq_linear(const void* d_x, const pq_prepared* p, void* d_y, int32_t M,
                  void* stream);

/* The ternary decode of pq_linear (activation quantiser, then the GEMV) for
 * callers that cannot allocate device memory at all -- for example code
 * hosted inside a framework that owns every device buffer and forbids new
 * allocations once it is serving, or that cannot accept the device-wide
 * synchronisation an allocation may cause.  The pages have no counterpart;
 * this is an addition of this library.
 *   Scratch: the quantised activations, their per-block sums and scales live
 *   in a fixed 128 KiB array inside the library's device image (every GPU that
 *   loads the library holds it until the process exits), not in the handle's
 *   workspace.  Calls need M*K up to about 120000 (checked: larger sizes
 *   return PQ_ERR_BUFFER_TOO_SMALL naming the need); M = 1..16; ternary
 *   handles only.  Nothing is allocated; nothing needs clearing (each call
 *   rewrites every scratch byte it reads).
 *   Every call on a device shares the one array and it keeps the last call's
 *   contents: calls that overlap on the GPU (unordered streams) race.
 *   The first call on each device looks up the array's device address (with
 *   that device current) and keeps it for the life of the process's primary
 *   context there; make that first call before any stream capture.
 * Arguments as pq_linear (1 <= M <= desc.max_m as well). */
PQ_API int32_t pq_linear_w2a8_static(const void* d_x, const pq_prepared* p, void* d_y,
                                     int32_t M, void* stream);

/* ---- quantised activations and the fused activation producer ------------
 *
 * Ternary layers run on int8 activations.  pq_linear quantises x itself on
 * every call; these entry points let the caller quantise once and run several
 * layers that read the same input (for example the q, k and v projections
 * after one norm), and fuse the quantiser into the producer of the layer
 * input: "Kernel experiments: recorded evidence", section E, Test 18 and
 * Diagram 5 (RMSNorm + Hadamard + Q8 in one pass).
 *
 * The quantised activations live in a caller buffer of pq_act_bytes(d, M)
 * bytes, 256-byte aligned.  Its contents depend on the descriptor's K,
 * act_group and act_dtype and on M only, so one buffer serves every ternary
 * handle that shares those values.  The buffer is opaque; its layout
 * differs between M <= 16 (decode) and M > 16 (prefill). */

/* Bytes of the quantised-activation buffer for M tokens of a ternary
 * descriptor (1 <= M <= max_m); 0 for any other descriptor (pq_last_error
 * says why).  Host-only. */
PQ_API size_t pq_act_bytes(const pq_desc* d, int32_t M);

/* Quantise x [M][K] (act_dtype, 16-B aligned) into d_act with the Test 6
 * group quantiser, exactly as pq_linear does.  Asynchronous on `stream`. */
PQ_API int32_t pq_quantize_act(const void* d_x, const pq_prepared* p, void* d_act,
                               size_t act_bytes, int32_t M, void* stream);

/* Parameters of the fused producer. */
typedef struct pq_norm {
    const void* gamma;      /* [K] act_dtype norm weight, 16-B aligned          */
    const int8_t* signs;    /* [K] transform signs: entries < 0 negate the
                               value before the transform; NULL = all +1       */
    float eps;              /* > 0, added to the mean square                    */
    int32_t unit_offset;    /* 1: weight is stored as an offset from one
                               (w = 1 + gamma, as Test 18); 0: w = gamma        */
    int32_t had_block;      /* 0: no transform; else a power of two 2..1024
                               dividing K: orthonormal Walsh-Hadamard transform
                               of every block of had_block values              */
} pq_norm;

/* Fused activation producer (Test 18), one pass per token row, all in fp32:
 *   u     = h + r                       (r NULL: u = h)
 *   r_out = u rounded to act_dtype      (if d_r_out is non-NULL)
 *   inv   = 1 / sqrt(sum(u*u) / K + eps)
 *   n     = (u * inv) * w rounded to act_dtype    (written to d_norm_out if
 *                                                  non-NULL)
 *   v     = H(signs * n) / sqrt(had_block) rounded to act_dtype (or v = n)
 *   d_act = the group quantiser applied to v, as pq_quantize_act(v).
 * The sum of squares runs in a fixed order: 2048 lanes, lane i adding
 * u[i]^2, u[i+2048]^2, ... in turn, then the lanes added pairwise by halving
 * (lane i += lane i+h for h = 1024, 512, ..., 1); every multiply and add is
 * a separately rounded fp32 operation and the square root and reciprocal
 * are correctly rounded, so the codes are reproducible bit for bit.
 *   d_h, d_r, d_r_out, d_norm_out: [M][K] act_dtype, 16-B aligned.  d_r_out
 *   may be d_h or d_r itself (an in-place residual update); otherwise no
 *   output may overlap an input.
 * Arguments are checked on the host (PQ_ERR_INVALID_ARG / _ALIGN / _SHAPE /
 * _BUFFER_TOO_SMALL); asynchronous on `stream`; no allocation. */
PQ_API int32_t pq_norm_quantize(const void* d_h, const void* d_r, const pq_norm* norm,
                                const pq_prepared* p, void* d_r_out, void* d_norm_out,
                                void* d_act, size_t act_bytes, int32_t M, void* stream);

/* y = x . W for a ternary handle with x given as quantised activations
 * (d_act written by pq_quantize_act or pq_norm_quantize for the same M, with
 * a handle of the same K, act_group and act_dtype).  The kernels are those
 * pq_linear picks, without their quantiser, so the result is the same bit
 * for bit: M = 1..2 the CUDA-core GEMV (the buffer then holds int8 codes),
 * 3..16 the cluster split-K decode (the bf16 split-K decode for rows longer
 * than the cluster holds), above 16 the tensor-core GEMM (for M > 2 the
 * buffer holds bf16 codes).
 *   act_bytes  size of the d_act buffer; PQ_ERR_BUFFER_TOO_SMALL if it is
 *              below pq_act_bytes(desc, M), before any launch
 * PQ_ERR_UNSUPPORTED if no kernel runs (d, M).  Asynchronous, no allocation. */
PQ_API int32_t pq_linear_act(const void* d_act, size_t act_bytes, const pq_prepared* p, void* d_y,
                             int32_t M, void* stream);

/* ---- dispatcher --------------------------------------------------------- */
#define PQ_VARIANT_AUTO          0
#define PQ_VARIANT_W4_GEMV       1  /* mma.sync fragment GEMV, M <= 16: whole
                                       rows in shared memory for M <= 4, else
                                       split-K across CTAs (needs max_m > 1) */
#define PQ_VARIANT_W4_GEMM       2  /* TMA + tcgen05/TMEM GEMM, any M
                                       (affine 4-bit: a pre-pass of the sums
                                       of x first; needs max_m > 16)        */
#define PQ_VARIANT_W2_GEMV_FUSED 3  /* dp4a GEMV, quantisation in-kernel     */
#define PQ_VARIANT_W2_GEMV       4  /* quantise pre-pass + dp4a GEMV         */
#define PQ_VARIANT_W2_GEMM       5  /* quantise pre-pass + tcgen05 GEMM      */
#define PQ_VARIANT_W2_GEMV_TC    6  /* quantise pre-pass + int8 mma.sync split-K
                                       decode, M <= 16 (needs max_m > 1)   */
#define PQ_VARIANT_W2_GEMV_BF    7  /* quantise pre-pass (bf16 codes) + bf16
                                       mma.sync split-K decode on exact
                                       integer operands, M <= 16 (needs
                                       max_m > 1)                          */
#define PQ_VARIANT_W2_GEMV_CL    8  /* one launch, M <= 16: a thread-block
                                       cluster of up to 8 CTAs splits K, each
                                       CTA quantises its slice (row maxima
                                       exchanged in the cluster), fp16
                                       mma.sync on exact integer operands,
                                       the slices added across the cluster;
                                       K <= 24576 (needs no max_m > 1)     */

typedef struct pq_plan_info {
    int32_t variant;      /* PQ_VARIANT_*                                   */
    int32_t grid;         /* CTAs of the main kernel                        */
    int32_t block;        /* threads per CTA of the main kernel             */
    int32_t smem_bytes;   /* dynamic shared memory of the main kernel       */
    int32_t launches;     /* kernels launched per pq_linear call            */
    int32_t m_tile;       /* tokens per tile (GEMV column tile / GEMM BM)   */
    int32_t k_split;      /* warps (GEMV) or CTAs (GEMM) sharing one output */
} pq_plan_info;

/* The dispatcher's decision for (d, M) on a device with `num_sms` SMs, as a
 * pure host function (cached per shape inside pq_linear).  Needs no GPU. */
PQ_API int32_t pq_plan(const pq_desc* d, int32_t M, int32_t num_sms, pq_plan_info* out);

/* pq_linear with the variant forced (PQ_VARIANT_AUTO = dispatcher).  A
 * variant that cannot run (M, format) returns PQ_ERR_UNSUPPORTED. */
PQ_API int32_t pq_linear_variant(const void* d_x, const pq_prepared* p, void* d_y,
                          int32_t M, int32_t variant, void* stream);

/* Synchronise `stream`, read and clear the handle's device status word.
 * Returns PQ_OK or the first device-side error recorded since the last
 * call (PQ_ERR_DEVICE_TIMEOUT).  When it reports an error it also clears the
 * prefill GEMM's shared-tile flags in the workspace (a launch that gave up a
 * bounded wait can leave them raised), so the next call on the workspace
 * starts clean. */
PQ_API int32_t pq_device_status(const pq_prepared* p, void* stream);

/* Free the host handle (not the caller's device buffers). */
PQ_API void pq_destroy(pq_prepared* p);

/* Thread-local message describing the last error of this thread. */
PQ_API const char* pq_last_error(void);

/* ---- measurement --------------------------------------------------------- */

/* Copy-only read probe ("Kernel experiments: recorded evidence", Test 24):
 * reads every byte of d_src[0..bytes) once with 16-byte loads and no other
 * work, and XORs checksums of the words into d_sink, so that the rate a
 * plain streaming read reaches on this device can be set beside the decode
 * GEMVs, which must read every weight byte once as well.
 *   d_src       16-byte aligned device buffer; bytes a multiple of 16, > 0
 *   d_sink      4-byte aligned device words [64] (read-modify-write): the
 *               XOR of all 64 words changes by the XOR of every 32-bit word
 *               of the buffer
 *   ctas_per_sm CTAs of 256 threads per SM (0: 8), at most 8
 *   dependent   1: the launch waits for its predecessor on the stream to
 *               finish before its first load (as a layer reading the
 *               previous layer's output under programmatic dependent
 *               launch); 0: it may overlap the predecessor's tail
 * Asynchronous on `stream`; errors are returned before any launch. */
PQ_API int32_t pq_probe_read(const void* d_src, size_t bytes, uint32_t* d_sink, int32_t ctas_per_sm,
                             int32_t dependent, void* stream);

/* ---- test exports (bit-exact checks against the CPU oracle) ------------- */

/* Dequantised weights from the prepared planes, fp32 [K][N] in the ORIGINAL
 * row order (act order undone): w = (code - z) * s for W4, (code - 1) * ws
 * for W2.  Exact in fp32. */
PQ_API int32_t pq_debug_unpack(const pq_prepared* p, float* d_w, void* stream);

/* W2 only: the activation quantiser of pq_linear.  d_q int8 [M][K] in
 * natural k order; d_xs fp32 [M][K/act_group]. */
PQ_API int32_t pq_debug_w2a8_quantize(const void* d_x, const pq_prepared* p,
                               int8_t* d_q, float* d_xs, int32_t M,
                               void* stream);

/* W2 only: exact int32 block sums S[M][N][K/128] = sum_k (code-1)*q, computed
 * with the GEMV's decode and dot-product device code. */
PQ_API int32_t pq_debug_w2a8_group_sums(const void* d_x, const pq_prepared* p,
                                 int32_t* d_S, int32_t M, void* stream);

/* W2 only: the contents of a quantised-activation buffer (pq_quantize_act /
 * pq_norm_quantize for the same M; act_bytes its size, checked as by
 * pq_linear_act): d_q int8 [M][K] in natural k order, d_xs fp32
 * [M][K/act_group], d_sq int32 [M][K/128] block sums of q. */
PQ_API int32_t pq_debug_act_unpack(const void* d_act, size_t act_bytes, const pq_prepared* p,
                                   int32_t M, int8_t* d_q, float* d_xs, int32_t* d_sq, void* stream);

/* Expire a bounded device wait on purpose: launches one CTA whose wait on an
 * mbarrier that nothing arrives at gives up after `spin_limit` polls, records
 * PQ_ERR_DEVICE_TIMEOUT in the handle's status word and returns.  Lets the
 * failure path be tested without hanging or faulting the GPU. */
PQ_API int32_t pq_debug_expire_wait(const pq_prepared* p, int32_t spin_limit,
                             void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PQ_H */
