/*
 * mha.h -- C ABI of the GB300 (sm_103a) multi-head scaled dot-product
 * attention library (libmha.so): forward, backward, decode step and the
 * surrounding encoder-layer pieces.
 *
 * The operation (cited by page title and section):
 *
 *   Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k) + mask) V
 *     "Attention Is All You Need" (azimuth.plus), "The idea: every word
 *     queries every word"; "The Transformer: Attention Is All You Need"
 *     (cuijiawei.cn), "The core idea: scaled dot-product attention" and its
 *     scaled_dot_product_attention(q, k, v, mask) with masked_fill(-inf).
 *
 *   MultiHead = Concat(head_1, ..., head_h) W^O,
 *   head_i = Attention(X_q W_i^Q, X_kv W_i^K, X_kv W_i^V)
 *     "Attention Is All You Need: The Research Paper That Changed AI"
 *     (muhitai.com), "Multi-Head Attention Formula"; notebook chapter
 *     "Attention is All You Need", "Multi-Head Self-Attention" and "The
 *     Decoder's Cross-Attention" (queries from the decoder, keys and values
 *     from the encoder output).
 *
 *   Masks: causal -- query i sees key j only if j <= i (notebook chapter,
 *   "Masked Attention in the Decoder"; muhitai.com "What Is Masked
 *   Attention?"); key padding -- keys j >= key_lens[b] get weight zero.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers to caller-owned memory,
 *     row-major and contiguous (sdpa_forward_host alone takes host tensors).
 *     The library never allocates device memory, frees or synchronises
 *     (sdpa_forward_host keeps two copy streams and a few events per device);
 *     every launch is enqueued on `stream` (0 = legacy default stream) and the
 *     call returns immediately.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and returned synchronously (nothing is launched).  A failed launch
 *     returns MHA_ERR_CUDA.
 *   - `status_dev` (optional, may be NULL) is a device int the caller zeroes
 *     before the call.  Every wait inside the kernels is bounded; a wait that
 *     runs out stores MHA_ERR_TIMEOUT there and the kernel returns early
 *     (its outputs are then undefined).  Read it after synchronising.
 *   - `key_lens` is a DEVICE int32 array of B entries, used only with a
 *     key-padding mask (NULL otherwise).  Values are clamped to [0, T_k].  A
 *     query row that sees no key at all (key_lens[b] == 0) outputs zeros.
 *   - Causal visibility is top-left aligned: key j is visible to query i iff
 *     j <= i, also when T_q != T_k.
 *   - The bf16 paths accumulate in fp32 (tensor memory), keep the softmax in
 *     fp32, round the probabilities to bf16 for the P.V product and round
 *     every stored tensor to bf16 (round to nearest even).
 */
#ifndef MHA_H
#define MHA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MHA_OK = 0,
    MHA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum, missing key_lens */
    MHA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. bf16 with d_k != 64) */
    MHA_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than mha_workspace_bytes() */
    MHA_ERR_MISALIGNED = 4,  /* a bf16 pointer is not 16-byte aligned (TMA rule) */
    MHA_ERR_CUDA = 5,        /* a CUDA runtime/driver call or a launch failed */
    MHA_ERR_TIMEOUT = 6,     /* written to *status_dev by a kernel whose wait ran out */
    MHA_ERR_BOUNDS = 7       /* written to *status_dev by a device-side bounds check; only a
                                library built with MHA_BOUNDS_CHECK has the checks */
} mha_status;

typedef enum {
    MHA_MASK_NONE = 0,
    MHA_MASK_CAUSAL = 1,
    MHA_MASK_KEY_PADDING = 2,
    MHA_MASK_CAUSAL_KEY_PADDING = 3
} mha_mask;

typedef enum { MHA_F32 = 0, MHA_BF16 = 1 } mha_dtype;

/*
 * Scaled dot-product attention, o = softmax(scale * q k^T + mask) v.
 *
 *   q (B, h, T_q, d_k), k (B, h, T_k, d_k), v (B, h, T_k, d_v),
 *   o (B, h, T_q, d_v): element type `dt` (fp32 or bf16).
 *   scale: usually 1/sqrt(d_k) (aiany.app, Step 5: "divide by 8" for 64).
 *
 * MHA_F32: fp32 SIMT kernel (FFMA + expf), d_k, d_v <= 128, 4-byte aligned
 *   arrays (with T_k <= 32, d_k == d_v == 64 and 16-byte aligned q, k a
 *   register kernel holding a row's whole key set runs instead, with the same
 *   result bit for bit).
 * MHA_BF16: fused tcgen05 kernel (TMA tiles, QK^T and PV on the tensor cores
 *   with fp32 accumulators in tensor memory, online softmax in registers; the
 *   T_q x T_k score matrix never reaches global memory).  Requires
 *   d_k == d_v == 64 and 16-byte aligned q, k, v, o.
 * B, h, T_q, T_k >= 0 (a zero extent is a no-op; T_k == 0 with T_q > 0
 * outputs zeros); B * h < 2^31.
 */
mha_status sdpa_forward(mha_dtype dt, const void *q, const void *k, const void *v, void *o,
                        int B, int h, int T_q, int T_k, int d_k, int d_v, float scale,
                        mha_mask mask, const int32_t *key_lens, int *status_dev,
                        cudaStream_t stream);

/*
 * Which of its two key splits the MHA_BF16 attention kernel takes for a
 * problem of this shape (host-only; no device call): 1 when the two softmax
 * warp groups take alternate 128-key tiles (a 128-row query tile sees, on
 * average, 8 or more key tiles, key padding not counted), 0 when they take
 * the two 64-key halves of every tile; -1 for negative extents or an invalid
 * mask.  Both splits compute the same function (they round differently); the
 * choice is a speed heuristic, exposed so that tests can cover both.
 */
int sdpa_bf16_key_split(int T_q, int T_k, mha_mask mask);

/*
 * Failure-detection drill (testing only; no product path uses it).  Runs the
 * MHA_BF16 attention of sdpa_forward on (B, h, T, 64) tensors, but every CTA's
 * loader issues no copy for its skip_tile-th key tile (counted over the
 * CTA's work in order, from 0), so the waits on that tile never complete,
 * and every wait of the kernel gives up after wait_limit_ns (1e5 .. 1e9 ns)
 * instead of the usual 1 s.  The kernel then records MHA_ERR_TIMEOUT in
 * *status_dev (required, a DEVICE int the caller zeroes first), drains the
 * copies and tensor-core products it has in flight, frees its tensor memory
 * and returns; the output is unspecified.  The context stays usable: a
 * following call on the same stream computes normally.  A CTA with fewer
 * than skip_tile + 1 key tiles completes normally.  Returns MHA_OK when the
 * launch succeeded (the timeout is reported on the device), argument errors
 * as sdpa_forward (here every extent must be positive).
 */
mha_status sdpa_forward_timeout_drill(const void *q, const void *k, const void *v, void *o,
                                      int B, int h, int T_q, int T_k, float scale,
                                      mha_mask mask, const int32_t *key_lens,
                                      unsigned long long wait_limit_ns, int skip_tile,
                                      int *status_dev, cudaStream_t stream);

/*
 * sdpa_forward (bf16 only) that also writes, per query row, the log-sum-exp of
 * its visible scores,
 *   lse[b, h, i] = log sum_{j visible} exp(scale * q_i . k_j)   (natural log),
 * the softmax normaliser (the weights are exp(scale q_i.k_j - lse)), which a
 * backward pass needs to recompute the weights.  lse: DEVICE fp32 array of
 * B*h*T_q entries (required when the problem is not empty); -inf for a row
 * with no visible key.  MHA_F32 returns MHA_ERR_UNSUPPORTED.
 * The value is the log of the normaliser the output was divided by: the sum
 * of the bf16-rounded weights the P.V product used, so it lies within the
 * relative bf16 rounding (2^-8) of the exact sum, |lse - exact| <= 2^-8 plus
 * fp32 rounding, and is consistent with o (exp(lse) o is the weighted value
 * sum the kernel formed, as a merge of partial results over key ranges needs).
 */
mha_status sdpa_forward_lse(mha_dtype dt, const void *q, const void *k, const void *v, void *o,
                            float *lse, int B, int h, int T_q, int T_k, int d_k, int d_v,
                            float scale, mha_mask mask, const int32_t *key_lens, int *status_dev,
                            cudaStream_t stream);

/*
 * sdpa_forward with HOST buffers: q, k, v (and key_lens) are read from, and o
 * written to, caller-owned HOST memory with the layouts, types and limits of
 * sdpa_forward.  Page-locked memory (cudaHostAlloc / cudaHostRegister) lets
 * the copies run asynchronously; pageable memory works but every copy then
 * completes before the call goes on.  workspace: DEVICE memory of at least
 * sdpa_forward_host_workspace_bytes() bytes, 256-byte aligned, owned by the
 * caller (the device copies of q, k, v, o and key_lens).  key_lens: HOST
 * int32 array of B entries (key-padding masks only).
 *
 * The heads are taken in up to 6 chunks (groups of heads of one batch item,
 * or whole batch items): chunk i's host-to-device copies, its attention launch
 * on `stream` and its device-to-host copy of o are chained by events, the
 * copies run on two internal copy streams (created on first use, one pair per
 * device, kept for the life of the process), so the copies of one chunk
 * overlap the attention of another.  The whole sequence is ordered after the
 * work enqueued on `stream` before the call and before the work enqueued on
 * it afterwards: synchronise `stream` before reading o, and keep the host
 * buffers valid and unchanged until then.  Calls are serialised per device by
 * a mutex while they enqueue.  Errors as sdpa_forward; a workspace that is
 * missing or too small is MHA_ERR_INVALID_ARG, a misaligned one
 * MHA_ERR_MISALIGNED (both detected before anything is enqueued).
 */
size_t sdpa_forward_host_workspace_bytes(mha_dtype dt, int B, int h, int T_q, int T_k, int d_k,
                                         int d_v);
mha_status sdpa_forward_host(mha_dtype dt, const void *q_host, const void *k_host,
                             const void *v_host, void *o_host, void *workspace,
                             size_t workspace_bytes, int B, int h, int T_q, int T_k, int d_k,
                             int d_v, float scale, mha_mask mask, const int32_t *key_lens_host,
                             int *status_dev, cudaStream_t stream);

/*
 * Gradients of sdpa_forward (bf16): given q, k, v, the forward's output o
 * and log-sum-exp lse (from sdpa_forward_lse) and the output gradient dout,
 * writes
 *   dv = P^T dout,  dq = scale dS k,  dk = scale dS^T q,
 *   dS = P (.) (dout v^T - rowsum(dout (.) o)),  P = exp(scale q k^T - lse)
 * (the chain rule of the forward definition; masked entries of P are 0).
 *   q, o, dout, dq (B, h, T_q, 64); k, v, dk, dv (B, h, T_k, 64); bf16,
 *   16-byte aligned; lse (B, h, T_q) fp32.  mask / key_lens / scale as the
 *   forward.  workspace: >= sdpa_backward_workspace_bytes() bytes, 256-byte
 *   aligned (an fp32 dq accumulator and two per-row vectors).
 * Three launches (row terms, the tcgen05 kernel -- one CTA per (b, h, block
 * of 128 keys) that keeps dk and dv in tensor memory and adds its dq
 * contributions to the fp32 accumulator -- and the dq conversion).  d_k ==
 * d_v == 64 only; MHA_F32 returns MHA_ERR_UNSUPPORTED.
 */
size_t sdpa_backward_workspace_bytes(int B, int h, int T_q, int T_k, int d_k, int d_v);
mha_status sdpa_backward(mha_dtype dt, const void *q, const void *k, const void *v, const void *o,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv,
                         void *workspace, size_t workspace_bytes, int B, int h, int T_q, int T_k,
                         int d_k, int d_v, float scale, mha_mask mask, const int32_t *key_lens,
                         int *status_dev, cudaStream_t stream);

/*
 * Adds the sinusoidal positional encoding to embedding rows (bf16):
 *   out[b, t, 2i]   = x[b, t, 2i]   + sin(pos / 10000^(2i/d_model)),
 *   out[b, t, 2i+1] = x[b, t, 2i+1] + cos(pos / 10000^(2i/d_model)),
 * pos = pos0 + t ("Attention is All You Need" notebook chapter, Positional
 * Encoding; aiany.app Step 8).  x, out (B, T, d_model), 16-byte aligned, may
 * be the same buffer; d_model % 8 == 0; pos0 + T < 2^24.
 */
mha_status positional_encoding_add(const void *x, void *out, int B, int T, int d_model, int pos0,
                                   cudaStream_t stream);

/*
 * One encoder layer with post-normalisation (bf16), the Transformer's
 * "self-attention -> add & normalise -> feed-forward -> add & normalise"
 * block (aiany.app Steps 9-10; notebook chapter "Feed-Forward Network"):
 *   y   = LayerNorm1(x + MultiHead(x, x)),
 *   out = LayerNorm2(y + FFN(y)),  FFN(y) = max(0, y W1 + b1) W2 + b2.
 *   x, out (B, T, d_model); W^Q, W^K, W^V, W^O (d_model, d_model) with h heads
 *   of 64 (d_model == 64 h); W1 (d_model, d_ff), b1 (d_ff), W2 (d_ff,
 *   d_model), b2, gamma1/beta1, gamma2/beta2 (d_model); all bf16 device
 *   arrays, 16-byte aligned.  d_ff % 64 == 0; d_model as
 *   mha_forward_add_layernorm.  mask, key_lens, scale, eps, status_dev as there.
 *   workspace: >= encoder_layer_workspace_bytes() bytes, 256-byte aligned.
 * Five launches: the three of the attention sublayer (its output projection
 * normalises), the first FFN GEMM with a bias + ReLU epilogue, the second FFN
 * GEMM with the bias, residual and normalisation in its epilogue.
 */
size_t encoder_layer_workspace_bytes(int B, int T, int d_model, int h, int d_ff);
mha_status encoder_layer_forward(const void *x, const void *w_q, const void *w_k, const void *w_v,
                                 const void *w_o, const void *gamma1, const void *beta1,
                                 const void *w1, const void *b1, const void *w2, const void *b2,
                                 const void *gamma2, const void *beta2, float eps, void *out,
                                 void *workspace, size_t workspace_bytes, int B, int T, int d_model,
                                 int h, int d_ff, float scale, mha_mask mask,
                                 const int32_t *key_lens, int *status_dev, cudaStream_t stream);

/*
 * Attention for decoding steps (bf16): each of the T_q new query rows of a
 * (b, h) attends to the first cache_lens[b] rows of that sequence's key/value
 * cache,
 *   o = softmax(scale * q k[0:len_b]^T) v[0:len_b].
 * Generation emits one token at a time and feeds it back in (aiany.app,
 * Step 10 "The decoder"); the newest row's causal mask ("Masked Attention in
 * the Decoder") reduces to this length limit, and cross-attention over the
 * encoder output ("The Decoder's Cross-Attention") is the same call with the
 * source length.  The result equals sdpa_forward with a key-padding mask.
 *
 *   q (B, h, T_q, 64), k_cache and v_cache (B, h, T_k, 64) with T_k the
 *   cache capacity, o (B, h, T_q, 64); bf16, contiguous, 16-byte aligned.
 *   cache_lens: DEVICE int32 array of B entries (clamped to [0, T_k]), or
 *   NULL for T_k keys everywhere.  1 <= T_q <= 8; d_k == d_v == 64 (other
 *   head sizes: MHA_ERR_UNSUPPORTED).  A row with no cached key outputs 0.
 *
 * One launch: the keys of each (b, h) are split over an 8-CTA thread-block
 * cluster, each CTA streams its range once from HBM (SIMT; the work per key
 * is too small for the tensor cores), and the partial softmax states are
 * merged exactly through distributed shared memory.  No workspace, no wait
 * that can time out (status words are not needed).
 */
mha_status sdpa_decode_forward(const void *q, const void *k_cache, const void *v_cache, void *o,
                               int B, int h, int T_q, int T_k, int d_k, int d_v, float scale,
                               const int32_t *cache_lens, cudaStream_t stream);

/*
 * Bytes of device workspace mha_forward needs: the projected Q, K, V in
 * head-split layout (B, h, T, d) and the merged attention output
 * (B, T_q, h * d_v), all bf16, each region 256-byte aligned.
 * Returns 0 for negative sizes.
 */
size_t mha_workspace_bytes(int B, int h, int T_q, int T_k, int d_k, int d_v);

/*
 * Multi-head attention forward, bf16 only:
 *   out = Concat_i(softmax(scale * (x_q W_i^Q)(x_kv W_i^K)^T + mask)
 *                  (x_kv W_i^V)) W^O
 *
 *   x_q (B, T_q, d_model); x_kv (B, T_k, d_model), may equal x_q for
 *   self-attention; W^Q, W^K (d_model, h*d_k); W^V (d_model, h*d_v);
 *   W^O (h*d_v, d_model); out (B, T_q, d_model).  Row-vector convention
 *   y = x W (notebook chapter: W^Q in R^{d_model x d_k}); head i owns
 *   columns [i*d_k, (i+1)*d_k) of W^Q/W^K/W^V; no bias.
 *   workspace: device buffer of at least mha_workspace_bytes() bytes,
 *   256-byte aligned, owned by the caller, not read before it is written.
 *
 * Three launches on `stream`: one grouped projection GEMM (Q, K, V with a
 * head-split epilogue), the fused attention kernel (writing the merged
 * (B, T_q, h*d_v) layout directly), and the W^O GEMM.
 * Requires d_k == d_v == 64, d_model % 64 == 0 and 16-byte aligned pointers.
 */
mha_status mha_forward(mha_dtype dt, const void *x_q, const void *x_kv, const void *w_q,
                       const void *w_k, const void *w_v, const void *w_o, void *out,
                       void *workspace, size_t workspace_bytes, int B, int h, int T_q, int T_k,
                       int d_model, int d_k, int d_v, float scale, mha_mask mask,
                       const int32_t *key_lens, int *status_dev, cudaStream_t stream);

/*
 * The attention sublayer with its residual connection and post-layer
 * normalisation, bf16:
 *   out = LayerNorm(x_q + MultiHead(x_q, x_kv)),
 *   LayerNorm(v) = (v - mean(v)) / sqrt(var(v) + eps) * gamma + beta per row
 * ("Attention Is All You Need" (aiany.app) Step 9, LayerNorm(x + Sublayer(x));
 * notebook chapter "Layer Normalization and Residual Connections").  mean and
 * var over the d_model features, var the population variance; eps >= 0 is the
 * caller's (the pages print none; 1e-5 is usual).  gamma, beta: d_model bf16
 * each, device, 16-byte aligned.  Other arguments, workspace and layouts as
 * mha_forward; additionally d_model must be a multiple of 128 and at most 2048
 * (else MHA_ERR_UNSUPPORTED).
 *
 * Three launches: the projection GEMM and attention as in mha_forward, then
 * the output projection with the residual add and the normalisation in its
 * epilogue -- a 128-row block is computed by a cluster of d_model/256 (or
 * /128) CTAs that exchange per-row partial sums through distributed shared
 * memory, so the normalised row never makes an extra trip through memory.
 */
mha_status mha_forward_add_layernorm(mha_dtype dt, const void *x_q, const void *x_kv,
                                     const void *w_q, const void *w_k, const void *w_v,
                                     const void *w_o, const void *gamma, const void *beta,
                                     float eps, void *out, void *workspace,
                                     size_t workspace_bytes, int B, int h, int T_q, int T_k,
                                     int d_model, int d_k, int d_v, float scale, mha_mask mask,
                                     const int32_t *key_lens, int *status_dev,
                                     cudaStream_t stream);

/*
 * Multi-head attention forward exactly as mha_forward, but with no workspace
 * argument: the scratch lives in a device array inside the library, so the
 * call allocates nothing.  (The pages have no counterpart: this is a
 * deployment convenience, not part of the method.)
 *
 * For callers that cannot call cudaMalloc or reach any device allocator --
 * for example a plugin hosted by a framework that owns all device memory and
 * exposes no allocation hook, or a serving loop whose memory plan forbids
 * allocation after start-up.
 *
 * Limit: the problem's mha_workspace_bytes(B, h, T_q, T_k, d_k, d_v) must not
 * exceed MHA_STATIC_WORKSPACE_BYTES (32 MiB); larger problems return
 * MHA_ERR_WORKSPACE and launch nothing.  Every GPU that loads the library
 * holds those 32 MiB until the process exits.
 *
 * Arguments are checked first, exactly as mha_forward checks them (errors
 * and the empty-problem MHA_OK come back before any device work).  Then every
 * call looks up the array's device address (cudaGetSymbolAddress, on the
 * caller's current device and context); nothing is cached, so the call stays
 * valid after cudaDeviceReset or under another context.  The first call in a
 * context is the one that loads the library's device code there (the
 * runtime's set-up), so make that first call before any stream capture.  A
 * failed lookup returns MHA_ERR_CUDA with the detail in mha_last_error().
 * All calls on a device share the one array and it keeps the previous call's
 * contents (every byte read is written earlier in the same call, so nothing
 * needs clearing): calls that overlap on the GPU -- on different streams, or
 * from different host threads -- race on it and must be serialised by the
 * caller.  Other arguments and errors as mha_forward.
 */
#define MHA_STATIC_WORKSPACE_BYTES (32u << 20)
mha_status mha_forward_static_workspace(mha_dtype dt, const void *x_q, const void *x_kv,
                                        const void *w_q, const void *w_k, const void *w_v,
                                        const void *w_o, void *out, int B, int h, int T_q,
                                        int T_k, int d_model, int d_k, int d_v, float scale,
                                        mha_mask mask, const int32_t *key_lens,
                                        int *status_dev, cudaStream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char *mha_status_string(mha_status status);

/* Detail of the most recent MHA_ERR_CUDA returned on the calling thread
 * (which step failed and the CUDA error name), or "" if none.  The string is
 * owned by the library and stays valid until the thread's next call. */
const char *mha_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MHA_H */
