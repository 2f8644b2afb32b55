/*
 * qmm.h -- fused-dequantisation GGUF quantized matmul on one NVIDIA GB300
 * (sm_103a).  C ABI: plain pointers and sizes, no C++ or framework types.
 *
 * The operation (all entry points): multiply by a weight matrix held in its
 * GGUF block encoding, decoding each block in registers at the moment its
 * weights enter the dot product, never expanding the matrix into a
 * full-precision buffer.  "Building a Rust Inference Engine That Matches
 * Llama.cpp", section "What Ferrox actually is" (weights never fully
 * decompressed; dequantisation fused into the dot product) and section
 * "Where the wins came from" (the dequant math happens inline, paid once, in
 * cache, instead of a separate memory-bound pass).  Activations are kept in
 * f32 and are never quantized ("Frink Inference: the Rust alternative to
 * llama.cpp", section "Where llama.cpp is still ahead").
 *
 * Weight layouts (GGUF; little-endian; the pages name these formats but do
 * not print them):
 *   QMM_Q4_K  super-block of 256 weights in 144 bytes:
 *             [fp16 d][fp16 dmin][12 bytes: eight 6-bit scales + eight 6-bit
 *             mins, llama.cpp get_scale_min_k4 packing][128 bytes of 4-bit
 *             quants: weight 64c+l is the low nibble of qs[32c+l] (l<32, sub-
 *             block 2c) or the high nibble of qs[32c+l-32] (sub-block 2c+1)].
 *             w = d*sc_j*q - dmin*m_j.
 *   QMM_Q8_0  block of 32 weights in 34 bytes: [fp16 d][32 x int8 q];
 *             w = d*q.
 *   Further formats ("Frink Inference: the Rust alternative to llama.cpp",
 *   "Where Frink is already better than llama.cpp": Q8_0 and the K-quants
 *   written byte-identically to llama-quantize; "Where llama.cpp is still
 *   ahead": IQ4_NL logits that match), for qmm_create, qmm_gemv, qmm_gemv_group, qmm_gemv_batched,
 *   qmm_ffn_decode and qmm_dequantize[_bf16]; the expert and prefill calls
 *   refuse them (QMM_ERR_UNSUPPORTED):
 *   QMM_Q5_K  176 bytes / 256 weights: [fp16 d][fp16 dmin][the 12 scale/min
 *             bytes of Q4_K][32 bytes of fifth bits: bit j of byte l belongs
 *             to weight l of sub-block j][128 bytes of low nibbles, the Q4_K
 *             order]; w = d*sc_j*q - dmin*m_j, q in 0..31.
 *   QMM_Q6_K  210 bytes / 256 weights: [128 bytes of low nibbles][64 bytes of
 *             2-bit high parts][16 int8 scales, one per 16 weights][fp16 d];
 *             weight i: half n = i/128, t = (i%128)/32, l = i%32; low bits =
 *             nibble (t >= 2) of byte 64n + 32*(t&1) + l, high bits = bits
 *             2t..2t+1 of high-part byte 32n + l; w = d*scale[i/16]*(q - 32).
 *   QMM_IQ4_NL 18 bytes / 32 weights: [fp16 d][16 bytes: weight l < 16 is the
 *             low nibble of byte l, weight 16+l its high nibble]; w = d*T[q]
 *             with GGUF's 16-entry IQ4_NL code book T.
 *   K-quants need K % 256 == 0; Q8_0 and IQ4_NL take any K % 32 == 0 (rows
 *   that are not whole 256-weight groups are only 2-byte aligned and go
 *   through the per-group kernels: decode GEMV, batched GEMV, groups, block
 *   decode, and for Q8_0 the no-allocation GEMV; the other calls refuse them).
 *   A matrix of N rows and K columns is N rows back to back, each row K/256
 *   (K-quants) or K/32 (Q8_0, IQ4_NL) blocks.  An expert-stacked tensor is n_experts such
 *   matrices back to back: row r of expert e is row e*N_e + r.
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device addresses on the current device; the
 *     caller owns them and keeps them alive until the work that uses them has
 *     finished.  Host pointers are named *_host.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous and stream-ordered; outputs are overwritten, never
 *     accumulated into.
 *   - One handle owns a small workspace (split-K partials and tickets) and a
 *     device status word: calls that use the same handle must be ordered on
 *     one stream.  Use one handle per concurrent stream.
 *   - Arguments are checked on the host before anything is launched.  A call
 *     that cannot do exactly what was asked does nothing and returns a
 *     non-zero qmm_status; qmm_last_error() then holds a sentence naming what
 *     is wrong.  The library never computes something other than what was
 *     asked, never traps the GPU, and has no CPU fallback.
 *   - Faults found on the device (an expert id out of range, a pipeline wait
 *     that ran out of time) set the handle's status word; read it with
 *     qmm_get_status() after synchronising.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QMM_API __attribute__((visibility("default")))
#else
#define QMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* GGUF tensor-type ids of the supported encodings. */
typedef enum { QMM_Q8_0 = 8, QMM_Q4_K = 12, QMM_Q5_K = 13, QMM_Q6_K = 14, QMM_IQ4_NL = 20 } qmm_format;

typedef enum {
    QMM_OK = 0,
    QMM_ERR_NULL = -1,        /* a required pointer is NULL */
    QMM_ERR_FORMAT = -2,      /* not one of Q4_K, Q8_0, Q5_K, Q6_K, IQ4_NL */
    QMM_ERR_SHAPE = -3,       /* a size is out of range or does not fill whole blocks */
    QMM_ERR_ALIGN = -4,       /* a pointer or leading dimension is not aligned as required */
    QMM_ERR_CUDA = -5,        /* the CUDA runtime reported an error (named in qmm_last_error) */
    QMM_ERR_TIMEOUT = -6,     /* a device-side pipeline wait gave up (status word) */
    QMM_ERR_UNSUPPORTED = -7, /* a valid request this version does not implement */
    QMM_ERR_NOMEM = -8,       /* a workspace allocation failed */
    QMM_ERR_EXPERT = -9       /* an expert id outside [0, n_experts) (status word) */
} qmm_status;

typedef struct qmm_matrix *qmm_t;
typedef void *qmm_stream; /* cudaStream_t */

/* Describe a quantized matrix of N rows x K columns at w_dev (borrowed, not
 * copied).  Requires: fmt one of Q4_K, Q8_0, Q5_K, Q6_K, IQ4_NL; N >= 1;
 * K % 256 == 0 for the K-quants, K % 32 == 0 for Q8_0 and IQ4_NL;
 * K <= 2^20; w_dev 16-byte aligned.  Allocates the handle's workspace and
 * status word on the current device.  On success *out is a new handle.
 * The bytes at w_dev must be fully written before the first call on the
 * handle is enqueued and stay unchanged while calls on it may run: the
 * kernels start fetching weights while earlier work in the stream is still
 * finishing (programmatic dependent launch), so a kernel that writes them
 * must have completed first (synchronise after loading the weights). */
QMM_API qmm_status qmm_create(qmm_format fmt, int64_t N, int64_t K, const void *w_dev,
                      qmm_t *out);

/* Free the handle and its workspace (synchronises the device first). */
QMM_API qmm_status qmm_destroy(qmm_t h);

/* Decode GEMV (one activation vector):  y[n] = sum_k w[n][k] * x[k].
 * x: K fp32 (device, 16-byte aligned), y: N fp32 (device, 4-byte aligned).
 * Any split of K over CTAs is reduced in a fixed order: results are bitwise
 * repeatable.  Never allocates (the handle's scratch covers it). */
QMM_API qmm_status qmm_gemv(qmm_t h, const float *x, float *y, qmm_stream stream);

/* Several matrices that share one input vector in one launch (the q/k/v or
 * gate/up projections of a layer).  All n handles have the same format and
 * K; ys[i] receives matrix i's N_i outputs.  n <= 8.  hs and ys are host
 * arrays of n entries; x and every ys[i] are device pointers as in qmm_gemv.
 * The work and workspace of hs[0] are used. */
QMM_API qmm_status qmm_gemv_group(const qmm_t *hs, int32_t n, const float *x,
                          float *const *ys, qmm_stream stream);

/* Batched decode: M activation rows share one read of the weights -- the
 * decode step of a server that batches requests continuously ("Frink
 * Inference: the Rust alternative to llama.cpp", "The goal, stated once":
 * the server bullet, continuous batching over paged KV).  Y[m*ldy + n] = sum_k w[n][k] * X[m*ldx + k], 1 <= M <= 16,
 * ldx >= K, ldy >= N, both multiples of 4.  Q4_K from two rows on: all rows
 * in one pass; the first call with a larger M may grow the handle's scratch
 * (a synchronising allocation: make it before capturing a CUDA graph). */
QMM_API qmm_status qmm_gemv_batched(qmm_t h, const float *X, int64_t M, int64_t ldx,
                            float *Y, int64_t ldy, qmm_stream stream);

/* Grouped mixture-of-experts GEMV driven by router expert ids, the expert
 * layers of the mixture-of-experts models the pages run ("Frink Inference:
 * the Rust alternative to llama.cpp", "Where Frink is already better than
 * llama.cpp": OLMoE decode on Metal; "Architecture coverage: 100 models with
 * evidence": dense and mixture-of-experts alike).  The handle
 * holds n_experts stacked matrices of N_e = N / n_experts rows each.
 * expert_ids: [T, top_k] int32 (device); the input of slot (t, s) is X[t]
 * when x_per_slot == 0 (X is [T, K]) or X[t*top_k + s] when x_per_slot == 1
 * (X is [T*top_k, K]).  route_w == NULL: Y is [T*top_k, N_e], Y[t*top_k+s] =
 * W_{ids[t,s]} x.  route_w != NULL ([T, top_k] fp32) and route_on_input == 0:
 * Y is [T, N_e], Y[t] = sum_s route_w[t,s] * W_{ids[t,s]} x (summed in slot
 * order).  route_on_input == 1 (route_w required; the Llama 4 form, where
 * the routing weight multiplies the expert's input -- "Architecture
 * coverage: 100 models with evidence"): Y is [T*top_k, N_e],
 * Y[t*top_k+s] = W_{ids[t,s]} (route_w[t,s] * x), no sum over slots (Q4_K:
 * the product r*x rounded to fp32 as the activations are loaded; Q8_0: r
 * times the slot's fp32 dot product, the same value up to rounding).  Each
 * expert's rows are read once per call for all of its slots.  An id outside
 * [0, n_experts) leaves that slot's contribution 0 and sets QMM_ERR_EXPERT in
 * the status word.  1 <= T*top_k <= 4096, top_k <= 16.  Formats: Q4_K, and
 * Q8_0 with K a multiple of 256 (Q8_0: "Frink Inference: the Rust
 * alternative to llama.cpp", "Where llama.cpp is still ahead"); anything
 * else is refused with QMM_ERR_UNSUPPORTED. */
QMM_API qmm_status qmm_moe_gemv(qmm_t h, int32_t n_experts, const int32_t *expert_ids,
                        int32_t T, int32_t top_k, const float *X,
                        int32_t x_per_slot, const float *route_w, int32_t route_on_input,
                        float *Y, qmm_stream stream);

/* h = silu(g) * u elementwise, silu(z) = z / (1 + exp(-z)); n fp32 values.
 * The SwiGLU between an expert's gate/up and down projections. */
QMM_API qmm_status qmm_swiglu(const float *g, const float *u, float *h, int64_t n,
                      qmm_stream stream);

/* A whole expert FFN: gate and up (both n_experts x d_ff x d_model), SwiGLU,
 * down (n_experts x d_model x d_ff) and the routing-weighted sum over each
 * token's top_k experts.  X [T, d_model] fp32, route_w [T, top_k] fp32,
 * Y [T, d_model] fp32.  route_on_input == 0: y_t = sum_s r * Wd h with
 * h = silu(Wg x) * (Wu x) (OLMoE, Mixtral, Qwen-MoE).  route_on_input == 1:
 * the Llama 4 form ("Frink Inference: the Rust alternative to llama.cpp",
 * "Architecture coverage: 100 models with evidence": the expert weight
 * applied to the input of the expert), h = silu(Wg (r x)) * (Wu (r x)),
 * y_t = sum_s Wd h; SwiGLU makes the two differ.  Uses hg's workspace for
 * the [T*top_k, d_ff] intermediate.  Same limits, formats and id checking as
 * qmm_moe_gemv; gate and up must share a format (they run in one launch;
 * QMM_ERR_FORMAT otherwise), down may be the other one. */
QMM_API qmm_status qmm_moe_ffn(qmm_t hg, qmm_t hu, qmm_t hd, int32_t n_experts,
                       const int32_t *expert_ids, int32_t T, int32_t top_k,
                       const float *X, const float *route_w, int32_t route_on_input,
                       float *Y, qmm_stream stream);

/* A dense SwiGLU FFN for one token (decode):  h = silu(Wg x) * (Wu x),
 * y = Wd h.  hg, hu: d_ff x d_model (same format), hd: d_model x d_ff.
 * x: d_model fp32, h: d_ff fp32 (the intermediate, also returned), y: d_model
 * fp32 (device; x and h 16-byte aligned, y 4-byte aligned).  Where the decode
 * kernel takes the shape (every format with K a multiple of 256; Q6_K 2048),
 * gate and up run in one launch with SwiGLU applied in its output phase (the
 * gate and up products never reach memory); otherwise (Q4_K) the earlier
 * tensor-core kernel's pair mode does the same, or gate and up run as one
 * grouped GEMV, the up product going to scratch held by the up handle
 * (allocated on the first such call; make that call before capturing a CUDA
 * graph), and SwiGLU runs as its own kernel.
 * Errors: QMM_ERR_SHAPE for mismatched shapes or formats, QMM_ERR_NULL,
 * QMM_ERR_ALIGN, QMM_ERR_NOMEM (scratch), QMM_ERR_CUDA; nothing is launched
 * on an argument error.
 * Sources: "Building a Rust Inference Engine That Matches Llama.cpp", "Where
 * the wins came from" (fused projections); the SwiGLU FFN of the Llama and
 * OLMoE architectures. */
QMM_API qmm_status qmm_ffn_decode(qmm_t hg, qmm_t hu, qmm_t hd, const float *x, float *h, float *y,
                                  qmm_stream stream);

/* Prefill GEMM on the tensor cores -- prompt processing, the one phase
 * where the pages' CUDA engine trails most ("Frink Inference: the Rust
 * alternative to llama.cpp", "Where llama.cpp is still ahead": prefill 25x
 * to 43x slower on CUDA; a tensor-core GEMM as the newer work).  Q4_K, and
 * Q8_0 with K % 256 == 0 (other formats: QMM_ERR_UNSUPPORTED):
 * Y[m*N + n] = sum_k bf16(w[n][k]) * X[m*K + k], fp32 accumulation, where
 * bf16(w) rounds the exact weight to fp32 and then to bf16 (nearest even).
 * X: [M, K] bfloat16 bit patterns, 16-byte aligned; Y: [M, N] fp32.
 * 1 <= M <= 2^24.  Results are bitwise repeatable (a split of K is added in
 * slice order). */
QMM_API qmm_status qmm_gemm(qmm_t h, const uint16_t *X_bf16, int64_t M, float *Y,
                    qmm_stream stream);

/* qmm_gemm for n matrices that share X (the q/k/v or gate/up projections of
 * a layer's prefill) in one launch: Ys[i] is [M, N_i].  All n handles have
 * the same format (Q4_K, or Q8_0 as above) and K, n <= 4; hs and Ys are host arrays of n entries.  The
 * split-K scratch of hs[0] is used. */
QMM_API qmm_status qmm_gemm_group(const qmm_t *hs, int32_t n, const uint16_t *X_bf16, int64_t M,
                                  float *const *Ys, qmm_stream stream);

/* Decode rows row0 .. row0+nrows-1 to fp32: out[i*K + k] = RN_fp32(w), which
 * is the exact weight (Q8_0) or the exact weight rounded once (Q4_K; d*sc
 * and dmin*m are exact in fp32).  For tests and inspection, not the hot
 * path. */
QMM_API qmm_status qmm_dequantize(qmm_t h, int64_t row0, int64_t nrows, float *out,
                          qmm_stream stream);

/* As qmm_dequantize, then rounded to bfloat16 (nearest even); out holds bit
 * patterns.  These are exactly the weights qmm_gemm multiplies with. */
QMM_API qmm_status qmm_dequantize_bf16(qmm_t h, int64_t row0, int64_t nrows,
                               uint16_t *out, qmm_stream stream);

/* Decode GEMV that allocates nothing, for callers that cannot call
 * cudaMalloc (code running inside a fixed memory pool, a driver-managed
 * allocator or a plug-in that must not grow the process's device footprint).
 * The pages have no counterpart: it is this library's addition.
 *
 * Computes y[n] = sum_k w[n][k] * x[k] like qmm_gemv, but takes the matrix
 * description directly (fmt, N, K, w_dev as in qmm_create) instead of a
 * handle, and keeps its split-K scratch -- partial sums and tickets -- in one
 * 1 MiB device array inside the library image (held by every GPU that loads
 * the library until the process exits).  No cudaMalloc, cudaFree or other
 * allocating call is made.  Every call looks up that array's device address
 * in the current context (cudaGetSymbolAddress; the first lookup in a context
 * may load the library's module, so make the first call before any stream
 * capture); a context reset therefore needs nothing from the caller.  Each
 * call clears the tickets on `stream` before launching.  All calls share the
 * one array: calls whose work can overlap on the GPU (different streams, or
 * concurrent host threads) race and must be serialised by the caller.  Shapes
 * whose split-K scratch exceeds the array are refused (QMM_ERR_SHAPE) with
 * the sizes named.  Unlike qmm_gemv, a device-side timeout is not reported:
 * the kernel records it in a word of the same array that no call reads back,
 * so a wedged pipeline shows only as a wrong y. */
QMM_API qmm_status qmm_gemv_noalloc(qmm_format fmt, int64_t N, int64_t K, const void *w_dev,
                                    const float *x, float *y, qmm_stream stream);

/* ---- The integer-dot variant (opt-in): Q8_K activations ----------------
 * "Frink Inference: the Rust alternative to llama.cpp", section "Where
 * llama.cpp is still ahead": llama.cpp quantizes the activations to Q8_K
 * before a K-quant dot product, and its K-quant logits drift slightly from
 * an engine that keeps f32 activations.  These calls are that path; the f32
 * calls above stay the reference behaviour.
 *
 * Q8_K (GGUF; the pages name it only): 256 activations per 292-byte block,
 * [binary32 d][256 x int8 q][16 x int16 bsums], bsums[g] = q[16g] + ... +
 * q[16g+15].  max = the signed value of the first element of largest
 * magnitude in the block; iscale = -127 / max; q = min(127,
 * round-half-even(iscale * x)); d = 1 / iscale; all three steps in binary32
 * (an all-zero block gives d = 0 and q = 0).  The block stands for d * q.
 *
 * Drift against the f32 path: every activation moves by at most |d|/2 (half
 * a code step of its block), so |y_q8k - y_f32| <= sum over blocks b of
 * (sum of |w| over block b) * |d_b| / 2, plus fp32 rounding. */

/* Quantize K fp32 activations (K a positive multiple of 256) to K/256 Q8_K
 * blocks at xq (K/256 * 292 bytes, device).  x 16-byte aligned, xq 4-byte
 * aligned; both device pointers owned by the caller.  One launch; bitwise
 * equal to the definition above.  Errors: QMM_ERR_NULL, QMM_ERR_SHAPE,
 * QMM_ERR_ALIGN, QMM_ERR_CUDA; nothing is launched on an argument error. */
QMM_API qmm_status qmm_quantize_q8_k(const float *x, int64_t K, void *xq, qmm_stream stream);

/* y[n] = sum over super-blocks of d_w d_x * (integer dot of the 4-bit codes
 * and the Q8_K codes, per sub-block times its 6-bit scale) - dmin d_x * (sum
 * over sub-blocks of the 6-bit min times the sub-block's Q8_K code sum):
 * exactly (up to fp32 rounding of the per-super-block scaling and the sum)
 * sum_k w[n][k] * d q_k.  h: a Q4_K matrix (other formats:
 * QMM_ERR_UNSUPPORTED); xq: K/256 Q8_K blocks as written by
 * qmm_quantize_q8_k (device, 4-byte aligned); y: N fp32 (device, 4-byte
 * aligned).  Each row is reduced inside one warp in a fixed order: bitwise
 * repeatable.  No scratch, no allocation. */
QMM_API qmm_status qmm_gemv_q8k(qmm_t h, const void *xq, float *y, qmm_stream stream);

/* qmm_gemv_q8k for n <= 8 Q4_K matrices of one K sharing xq (the q/k/v or
 * gate/up projections of a layer) in one launch; hs and ys are host arrays
 * of n entries, ys[i] receives matrix i's outputs. */
QMM_API qmm_status qmm_gemv_q8k_group(const qmm_t *hs, int32_t n, const void *xq,
                                      float *const *ys, qmm_stream stream);

/* qmm_gemv_q8k and qmm_gemv_q8k_group on f32 activations x (K values,
 * device, 16-byte aligned): the launch quantizes x to Q8_K itself (every CTA
 * the blocks it reads, in shared memory; the same bytes as
 * qmm_quantize_q8_k) and runs the same integer-dot GEMV, so the results are
 * bitwise those of qmm_quantize_q8_k followed by qmm_gemv_q8k[_group], in one
 * launch instead of two and without the xq buffer.  Errors as for those
 * calls; x NULL: QMM_ERR_NULL. */
QMM_API qmm_status qmm_gemv_q8k_fused(qmm_t h, const float *x, float *y, qmm_stream stream);
QMM_API qmm_status qmm_gemv_q8k_fused_group(const qmm_t *hs, int32_t n, const float *x,
                                            float *const *ys, qmm_stream stream);

/* Read and clear the handle's device status word (synchronises the handle's
 * last stream first).  QMM_OK when no device-side fault was recorded. */
QMM_API qmm_status qmm_get_status(qmm_t h);

/* The calling thread's last refusal or error sentence ("" if none). */
QMM_API const char *qmm_last_error(void);

/* Library version as an integer (major*10000 + minor*100 + patch). */
QMM_API int32_t qmm_version(void);

/* Kernel launches this library has issued in this process so far (all entry
 * points, all devices), for instrumentation: the difference across a region
 * counts the library's kernels in it.  Never fails. */
QMM_API int64_t qmm_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* QMM_H */
