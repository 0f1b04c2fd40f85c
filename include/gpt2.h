/*
 * gpt2.h -- C ABI of the GB300 (sm_103a) GPT-2 pre-norm forward library.
 *
 * The library computes the GPT-2 pre-norm decoder block, the full uncached
 * forward (embedding, L blocks, final LayerNorm, tied head) and cached decode,
 * with hand-written CUDA kernels.  Every function takes plain pointers and
 * sizes; device pointers are CUDA device addresses owned by the caller.
 *
 * Sources (web pages, by title and section):
 *   "GPT-2 Decoder Block" (AI Engineer Exhaustive), "How it works": the block
 *       a = Attn(LN1(x)); x += a; m = MLP(LN2(x)); x += m, LN eps 1e-5,
 *       n_head heads of width d/n_head, a 4d GELU MLP, present returned.
 *   "GPT-2 Full Forward Pass" (AI Engineer Exhaustive), "How it works":
 *       H0 = gather(W_e, X) + gather(W_p, pos(X, l_past)); L blocks; ln_f;
 *       logits = LN_f(H) W_e^T; fused c_attn to 3d; past [B, 2, h, T_past,
 *       d_h] per layer concatenated on the sequence axis; present stacked as
 *       [B, L, 2, h, T, d_h]; positions stay below n_ctx.
 *   "GPT-2 Transformer block" (open-model-atlas), openai/gpt-2 ``norm``
 *       excerpt: u = mean(x), s = mean((x-u)^2), (x-u) rsqrt(s+eps) g + b.
 *   "GPT-2 Block - TorchCode", "Reference Solution": scores q k^T/sqrt(d_k),
 *       upper-triangular -inf mask, softmax over keys, weights @ v.
 *   "Decoder-only" (CodeBlanks): pre-LN loop and the tied head.
 *
 * Conventions common to every entry point:
 *   - Return value: a gpt2_status.  On any validation error nothing is
 *     launched and no memory is touched.  Errors raised inside a kernel
 *     (a bounded wait that ran out, a token id out of range, a value past
 *     the fp16 operand range) surface at gpt2_sync_status.
 *   - Asynchrony: work is enqueued on `stream` (a cudaStream_t value; NULL is
 *     the legacy default stream) and the call returns before it completes.
 *   - Dtypes: in GPT2_BF16 mode parameters, the block input/output and the KV
 *     cache are bf16 (16-bit words).  Inside, the operands of the Linear
 *     products are fp16 -- the normalised, attention and GELU activations, and
 *     fp16 copies of the bf16 weights (exact for 2^-14 <= |w| <= 65504) -- and
 *     Q, K, V and the attention probabilities are bf16; every product
 *     accumulates in fp32 and the residual stream is fp32.  (fp16 operands
 *     carry 3 more mantissa bits than bf16; with bf16 operands the tied-head
 *     argmax of random-weight models agrees with exact arithmetic at only
 *     ~99.1% of positions, with fp16 operands at ~99.7%.)  A weight or an
 *     activation past the fp16 range is reported as GPT2_ERR_RANGE by
 *     gpt2_sync_status, never rounded to infinity silently.  In GPT2_FP32 mode
 *     everything is fp32.  Logits are always fp32.  Token ids are int32.
 *   - Layouts are dense row-major C order.  Linear weights are [out, in]
 *     (the nn.Linear convention); c_attn rows are Q | K | V, head j taking
 *     rows [j*d_h, (j+1)*d_h) of each block.
 *   - Alignment: every device pointer must be 16-byte aligned.
 *   - Shapes: BF16 mode needs d_h = d / n_head = 64; FP32 mode needs only
 *     d % n_head == 0 and d_h <= 256.  T_past + T <= n_ctx.
 *   - Ownership: the caller owns every buffer, including the workspace it
 *     hands to gpt2_ctx_create; the library frees nothing it did not create.
 */
#ifndef GPT2_H
#define GPT2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GPT2_OK = 0,
  GPT2_ERR_INVALID_ARG = 1,    /* null pointer, non-positive size, bad enum */
  GPT2_ERR_UNSUPPORTED = 2,    /* shape the chosen mode does not implement */
  GPT2_ERR_CTX_OVERFLOW = 3,   /* T_past + T > n_ctx, or a cache too small */
  GPT2_ERR_ALIGNMENT = 4,      /* a device pointer not 16-byte aligned */
  GPT2_ERR_CUDA = 5,           /* a CUDA runtime call failed */
  GPT2_ERR_DEVICE_TIMEOUT = 6, /* a kernel's bounded wait ran out */
  GPT2_ERR_WORKSPACE = 7,      /* workspace too small for the request */
  GPT2_ERR_NO_DEVICE = 8,      /* no sm_100-family GPU is current */
  GPT2_ERR_RANGE = 9           /* (device) a value outside the fp16 operand range
                                  of the bf16 mode (|v| > 65504), or not finite */
} gpt2_status;

typedef enum { GPT2_BF16 = 0, GPT2_FP32 = 1 } gpt2_dtype;

/* Model hyper-parameters (default_hparams of the official code, as the Full
 * Forward Pass page names them).  dtype is a gpt2_dtype. */
typedef struct {
  int n_vocab, n_ctx, n_embd, n_head, n_layer;
  int dtype;
} gpt2_hparams;

/* One block's parameters, device pointers in the mode's dtype:
 *   ln1_g, ln1_b, ln2_g, ln2_b   [d]
 *   attn_w [3d, d], attn_b [3d]   c_attn (Q | K | V)
 *   proj_w [d, d],  proj_b [d]    attention c_proj
 *   fc_w   [4d, d], fc_b   [4d]   mlp c_fc
 *   mlp_proj_w [d, 4d], mlp_proj_b [d]   mlp c_proj                       */
typedef struct {
  const void *ln1_g, *ln1_b, *attn_w, *attn_b, *proj_w, *proj_b;
  const void *ln2_g, *ln2_b, *fc_w, *fc_b, *mlp_proj_w, *mlp_proj_b;
} gpt2_block_params;

/* Whole-model parameters: wte [n_vocab, d], wpe [n_ctx, d], lnf_g/lnf_b [d]
 * (device, mode dtype); blocks is a HOST array of n_layer block records.   */
typedef struct {
  const void *wte, *wpe, *lnf_g, *lnf_b;
  const gpt2_block_params *blocks;
} gpt2_params;

/* A KV cache.  data is device memory of shape
 *   [B, L, 2, h, T_cap, d_h]  for gpt2_forward (L = n_layer), or
 *   [B, 2, h, T_cap, d_h]     for gpt2_block_forward,
 * index 0 of the "2" axis holding keys and 1 values.  Positions
 * [0, T_len) are valid.  This is the pages' past/present layout with the
 * sequence axis allocated to a capacity T_cap >= T_len.                   */
typedef struct {
  void *data;
  int T_cap;
  int T_len;
} gpt2_kv;

typedef struct gpt2_ctx gpt2_ctx;

/* ------------------------------------------------------------ context ---- */

/* Bytes of device workspace a context needs for batches of up to max_B
 * sequences of up to max_T new tokens with hyper-parameters *hp.          */
int gpt2_workspace_bytes(const gpt2_hparams *hp, int max_B, int max_T, size_t *bytes);

/* Creates a context on the current CUDA device.  workspace: caller-owned
 * device memory of at least gpt2_workspace_bytes bytes, 256-byte aligned,
 * which the context uses for intermediates and its device error word until
 * it is destroyed.  *out receives the context (host memory the library owns).
 * Errors: INVALID_ARG, UNSUPPORTED (shape the dtype cannot run),
 * WORKSPACE (too small), NO_DEVICE, CUDA.                                   */
int gpt2_ctx_create(const gpt2_hparams *hp, int max_B, int max_T, void *workspace,
                    size_t workspace_bytes, gpt2_ctx **out);

/* Releases the context's host state and CUDA events.  The workspace stays
 * the caller's.  NULL is accepted.                                         */
void gpt2_ctx_destroy(gpt2_ctx *ctx);

/* Waits for `stream`, then reads and clears the context's device error
 * word: GPT2_OK, GPT2_ERR_DEVICE_TIMEOUT (a bounded wait ran out),
 * GPT2_ERR_INVALID_ARG (a token id outside [0, n_vocab)), GPT2_ERR_RANGE (in
 * bf16 mode, a value past the fp16 range of the products' operands: a weight
 * with |w| > 65504, or a LayerNorm, attention or GELU output beyond 65504 or
 * not finite; the outputs of that call are not to be trusted), or
 * GPT2_ERR_CUDA for a failed launch or an asynchronous CUDA error.  When
 * several bits are set the first of that list is returned.                 */
int gpt2_sync_status(gpt2_ctx *ctx, void *stream);

/* bf16 mode converts each weight matrix to an fp16 working copy (in the
 * workspace) before its product.  enable != 0: keep those copies across
 * calls, keyed by the weight's device address, and convert a matrix only the
 * first time its address is seen -- the caller promises not to change weight
 * contents in place while caching is on (call again to forget all copies).
 * enable == 0 (the default): convert on every call.                       */
int gpt2_ctx_cache_weights(gpt2_ctx *ctx, int enable);

/* Static description of a status code. */
const char *gpt2_status_string(int status);

/* ------------------------------------------------------------ forward ---- */

/* One pre-norm decoder block ("GPT-2 Decoder Block", "How it works"):
 *   a = c_proj(causal_MHA(c_attn(LN1(x)))); x += a;
 *   m = mlp_proj(GELU_tanh(c_fc(LN2(x)))); out = x + m.
 * x, out: device [B, T, d] in the mode dtype (out may equal x).
 * params: host pointer to device parameter pointers.  d, n_head must equal
 * the context's n_embd, n_head.
 * past: NULL (no cache) or a [B, 2, h, T_cap, d_h] cache holding T_past =
 * past->T_len positions; the queries sit at positions T_past .. T_past+T-1
 * and see every cached and new key at or before their own position.
 * present: NULL (keys/values are not returned) or a cache that receives all
 * T_past + T positions; present->T_len is set to T_past + T when the call is
 * enqueued.  present->data == past->data appends in place; otherwise the
 * past positions are copied into present first.
 * Errors: INVALID_ARG, UNSUPPORTED, CTX_OVERFLOW (T_past + T > n_ctx or
 * > present->T_cap), ALIGNMENT, WORKSPACE (B*T beyond the context's sizing),
 * CUDA.                                                                    */
int gpt2_block_forward(gpt2_ctx *ctx, const void *x, const gpt2_block_params *params, int B, int T,
                       int d, int n_head, const gpt2_kv *past, gpt2_kv *present, void *out,
                       void *stream);

/* The post-norm arrangement of the same block, which the pages contrast
 * with GPT-2's pre-norm ("GPT-2 Decoder Block", "Overview": the original
 * Transformer normalises after each residual add):
 *   x1 = LN1(x + c_proj(causal_MHA(c_attn(x))));
 *   out = LN2(x1 + mlp_proj(GELU_tanh(c_fc(x1)))).
 * Same parameters, arguments, layouts and errors as gpt2_block_forward, with
 * no cache.  In bf16 mode the products take the bf16 weights as they are and
 * the normalised stream x1 is kept in bf16 (no fp16 working copies).       */
int gpt2_block_forward_postnorm(gpt2_ctx *ctx, const void *x, const gpt2_block_params *params,
                                int B, int T, int d, int n_head, void *out, void *stream);

/* The full forward ("GPT-2 Full Forward Pass", "How it works"):
 * H = wte[ids] + wpe[T_past + t]; L blocks; logits = LN_f(H) wte^T.
 * ids: device int32 [B, T], each in [0, n_vocab).
 * params: host pointer; L must equal the context's n_layer.
 * past / present: NULL or [B, L, 2, h, T_cap, d_h] caches as above.
 * logits: device fp32 [B, T, n_vocab] (exactly n_vocab columns, no bias).
 * Out-of-range token ids are clamped into range on the device and reported
 * as GPT2_ERR_INVALID_ARG by gpt2_sync_status.
 * Errors: as gpt2_block_forward.                                            */
int gpt2_forward(gpt2_ctx *ctx, const int32_t *ids, int B, int T, const gpt2_params *params, int L,
                 const gpt2_kv *past, gpt2_kv *present, float *logits, void *stream);

/* The next-token loss of the full forward without the logits ("GPT-2 Full
 * Forward Pass", "Overview": next-token language modelling of p(s_i | s_<i);
 * "How it works": callers take the logits and a next-token cross-entropy).
 * Runs as gpt2_forward up to LN_f, then reduces the tied head on the fly, per
 * position t of [B, T]:
 *   loss[t]     = logsumexp_v z[t, v] - z[t, targets[t]]  (0 where targets[t] < 0)
 *   next_ids[t] = argmax_v z[t, v]  (the lowest index among equal maxima)
 * without writing the [B, T, V] logits.  targets: device int32 [B, T] with
 * entries in [0, n_vocab) or negative (required when loss is given); loss:
 * device fp32 [B, T] or NULL; next_ids: device int32 [B, T] or NULL (not both
 * NULL).  bf16 mode only (UNSUPPORTED in fp32 mode).  A target >= n_vocab
 * gives a NaN loss and INVALID_ARG from gpt2_sync_status.  Other errors: as
 * gpt2_forward.                                                             */
int gpt2_forward_loss(gpt2_ctx *ctx, const int32_t *ids, const int32_t *targets, int B, int T,
                      const gpt2_params *params, int L, const gpt2_kv *past, gpt2_kv *present,
                      float *loss, int32_t *next_ids, void *stream);

/* The k most likely next tokens of every position, without the logits: the
 * candidates a top-k sampler draws from ("GPT-2 Full Forward Pass", "How it
 * works": the logits give the next token's distribution; greedy decoding takes
 * its argmax, k = 1).  Runs as gpt2_forward up to LN_f, then reduces the tied
 * head on the fly, per position t of [B, T]:
 *   top_logits[t, i], top_ids[t, i] for i < k: the k largest z[t, v] in
 *     descending order with their ids (among equal values the lower id
 *     first; NaN and -inf logits are never chosen: id -1 and value -inf fill
 *     slots beyond the other entries);
 *   lse[t] = logsumexp_v z[t, v], so that top_logits[t, i] - lse[t] are the
 *     log-probabilities of the candidates (NaN when a logit is NaN).
 * 1 <= k <= 8 and k <= n_vocab (INVALID_ARG otherwise).  top_logits: device
 * fp32 [B, T, k]; top_ids: device int32 [B, T, k]; lse: device fp32 [B, T] or
 * NULL; each 16-byte aligned.  bf16 mode only (UNSUPPORTED in fp32 mode).
 * Other errors: as gpt2_forward.                                             */
int gpt2_forward_topk(gpt2_ctx *ctx, const int32_t *ids, int B, int T, const gpt2_params *params,
                      int L, const gpt2_kv *past, gpt2_kv *present, int k, float *top_logits,
                      int32_t *top_ids, float *lse, void *stream);

/* Greedy generation: the model's consumer ("GPT-2 Full Forward Pass": the
 * logits of the last position give the next token; greedy takes their
 * argmax, the lowest index among equal maxima).  Runs the prompt ids [B,
 * T_prompt] through gpt2_forward after the cache's T_len positions (with the
 * cache as past when T_len > 0, and as present), then n_new times: the argmax
 * of the last position's logits becomes out_ids[b, i] (device int32 [B,
 * n_new]) and, except after the last one, one cached gpt2_forward step of
 * that token.  All work is enqueued on `stream` with no host synchronisation
 * (the chosen ids stay on the device), so the whole loop can be captured in
 * a CUDA graph.  logits: device fp32 scratch of at least B * T_prompt *
 * n_vocab values (holds the last step's logits on return).  cache->T_len
 * becomes T_len + T_prompt + n_new - 1.
 * Errors: as gpt2_forward; CTX_OVERFLOW when T_len + T_prompt + n_new - 1
 * exceeds n_ctx or cache->T_cap.                                             */
int gpt2_generate_greedy(gpt2_ctx *ctx, const int32_t *ids, int B, int T_prompt,
                         const gpt2_params *params, int L, gpt2_kv *cache, int n_new,
                         float *logits, int32_t *out_ids, void *stream);

/* ------------------------------------------------- single operations ---- */
/* The steps of the forward, exposed one by one so each kernel can be checked
 * and timed alone.  All pointers are device pointers.                      */

/* LayerNorm over the last axis (openai/gpt-2 ``norm`` excerpt, eps 1e-5,
 * biased variance): y = (x - u) rsqrt(s + eps) g + b for `rows` rows of d.
 * x_dtype: dtype of x (GPT2_FP32 or GPT2_BF16); g, b, y: mode dtype.      */
int gpt2_layer_norm(int mode, const void *x, int x_dtype, const void *g, const void *b, int rows,
                    int d, void *y, void *stream);

typedef enum {
  GPT2_EPI_BIAS = 0,       /* out = A W^T + bias                     (mode dtype) */
  GPT2_EPI_BIAS_GELU = 1,  /* out = gelu_tanh(A W^T + bias)          (mode dtype) */
  GPT2_EPI_BIAS_RESID = 2, /* out = resid + A W^T + bias             (fp32 resid/out) */
  GPT2_EPI_LOGITS = 3      /* out = A W^T, no bias                   (fp32 out) */
} gpt2_epilogue;

/* Linear layer C[M, N] = A[M, K] W[N, K]^T with a fused epilogue (the c_attn
 * / c_proj / c_fc / mlp c_proj / tied-head products of the Full Forward Pass
 * page).  A, W: mode dtype.  bias [N] (ignored for LOGITS).  resid and out
 * are [M, N]; resid may equal out.  K must be a multiple of 8.            */
int gpt2_linear(gpt2_ctx *ctx, int epilogue, const void *A, const void *W, const void *bias,
                const float *resid, void *out, int M, int N, int K, void *stream);

/* Causal multi-head attention ("GPT-2 Block - TorchCode", "Reference
 * Solution", with the cache offset of the Full Forward Pass page).
 * q: [B, h, T, d_h]; kv: [B, 2, h, T_cap, d_h] holding T_past + T valid
 * positions (the new keys/values already appended); out: [B, T, h*d_h]
 * (heads merged).  Mode dtype throughout.  T == 1 with T_past > 0 takes the
 * split-KV decode kernel.                                                 */
int gpt2_attention(gpt2_ctx *ctx, const void *q, const void *kv, int B, int n_head, int T,
                   int T_past, int T_cap, int d_h, void *out, void *stream);

/* Single-token decode attention that allocates nothing.  The pages have no
 * counterpart: this exists for callers that cannot allocate device memory
 * and so cannot hand gpt2_ctx_create a workspace -- a plugin that its host
 * application gives only pointers and a stream, a process whose device
 * memory another allocator has already reserved in full, or a
 * latency-critical path that must not take cudaMalloc's implicit
 * synchronisation.  It computes what gpt2_attention computes for T = 1 and
 * T_past > 0 (bf16, d_h = 64), keeping the split-KV partial results in a
 * 1 MiB array compiled into the library, which every GPU that loads the
 * library holds until the process exits.
 *   q: [B, h, 1, 64]; kv: [B, 2, h, T_cap, 64] with T_past + 1 valid
 *   positions (the new key/value already at position T_past);
 *   out: [B, 1, h * 64].  The caller still provides all three.
 *   splits: key chunks per (sequence, head); 0 chooses as gpt2_attention.
 * The first call on a device looks up the array's device address, once per
 * device and with that device current; make that first call before any
 * stream capture.  All calls share the one array, which keeps the previous
 * call's contents; nothing in it has to start at zero, since each call writes
 * every partial result before reading it.  Calls that overlap on the GPU
 * (other streams, other host threads) race on the array.
 * If one of the kernel's bounded waits runs out (2 s by default), that
 * (sequence, head)'s output row is written as NaN instead of being left as
 * it was, and the timeout bit of the entry point's own device error word is
 * set: gpt2_attention_decode_noalloc_status reports it.
 * Errors: INVALID_ARG, UNSUPPORTED (d_h != 64, or B * h > 65535),
 * CTX_OVERFLOW (T_past + 1 > T_cap), ALIGNMENT, WORKSPACE (B * h * splits
 * partial results of 66 floats exceed the 1 MiB array), NO_DEVICE, CUDA.    */
int gpt2_attention_decode_noalloc(const void *q, const void *kv, int B, int n_head, int T_past,
                                  int T_cap, int d_h, int splits, void *out, void *stream);

/* The device error word of gpt2_attention_decode_noalloc on the current
 * device: synchronises `stream`, reads the word and clears it.  Returns
 * DEVICE_TIMEOUT if a call since the last read had a bounded wait run out
 * (its NaN rows are the ones affected), else OK; NO_DEVICE or CUDA when
 * the device or the runtime fails.  Like the entry point it uses no context
 * and allocates nothing (the word is compiled into the library, one per
 * device).                                                                  */
int gpt2_attention_decode_noalloc_status(void *stream);

/* Test support: the limit of gpt2_attention_decode_noalloc's bounded waits,
 * for all devices of the process, in nanoseconds; limit_ns <= 0 restores the
 * 2 s default.  A limit of a few nanoseconds makes the first wait that is
 * not already satisfied run out on ordinary work, so the timeout path can be
 * tested without a fault.  Returns OK.                                      */
int gpt2_attention_decode_noalloc_set_wait_limit(long long limit_ns);

/* Embedding: H[b, t] = wte[ids[b, t]] + wpe[T_past + t] (fp32 out [B, T, d]).
 * wte [n_vocab, d], wpe [n_ctx, d] in the mode dtype.                      */
int gpt2_embed(gpt2_ctx *ctx, const int32_t *ids, const void *wte, const void *wpe, int B, int T,
               int T_past, float *H, void *stream);

/* ----------------------------------------------------------- self-test ---- */

/* Exercises the device-side failure path that every kernel of the library
 * uses: one thread waits, with the kernels' own bounded wait but a limit of
 * limit_us microseconds, on an mbarrier that nothing completes.  The wait
 * runs out, sets the context's error word and the kernel returns; the next
 * gpt2_sync_status reports GPT2_ERR_DEVICE_TIMEOUT (and clears the word) and
 * the context stays usable.  Nothing faults, traps or hangs.  The pages have
 * no counterpart: this is test support for the library.
 * Errors: INVALID_ARG (null ctx, limit_us outside 1 .. 1000000), CUDA.      */
int gpt2_selftest_wait_timeout(gpt2_ctx *ctx, int limit_us, void *stream);

/* Sets the limit of the bounded waits inside the tensor-core GEMM and the
 * prefill attention launched through `ctx` (limit_ns > 0), or restores the
 * default of 2 s (limit_ns <= 0).  Test support, no counterpart on the pages:
 * a limit of a few nanoseconds makes the first wait that is not already
 * satisfied run out, so the kernels' failure path (raise the error word,
 * drain the copies already issued, retire the issued MMAs, free TMEM,
 * return) runs on real work; the next gpt2_sync_status then reports
 * GPT2_ERR_DEVICE_TIMEOUT, and with the default restored the context computes
 * normally again.  The waits that drain copies keep the 2 s limit.
 * Errors: INVALID_ARG (null ctx).                                          */
int gpt2_ctx_set_wait_limit(gpt2_ctx *ctx, long long limit_ns);

/* ---------------------------------------------------------- profiling ---- */

/* When enabled, every kernel launch the context makes is bracketed by CUDA
 * events on its stream; the per-kernel totals accumulate until read.      */
int gpt2_profile_enable(gpt2_ctx *ctx, int enable);

/* Number of kernel kinds the profiler distinguishes. */
int gpt2_profile_kinds(void);

/* Waits for the recorded events and returns, for kernel kind `kind`, its
 * name, the number of launches, their summed duration in ms and the summed
 * algorithmic flops and bytes of those launches.                          */
int gpt2_profile_read(gpt2_ctx *ctx, int kind, const char **name, long long *launches,
                      double *total_ms, double *flops, double *bytes);

/* Clears the accumulated profile. */
int gpt2_profile_reset(gpt2_ctx *ctx);

#ifdef __cplusplus
}
#endif

#endif /* GPT2_H */
