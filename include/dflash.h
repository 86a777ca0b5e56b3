/*
 * dflash.h — C ABI of the GB300 (sm_103a) DFlash draft-cycle library.
 *
 * One draft cycle of the DFlash block-diffusion drafter ("DFlash: Block
 * Diffusion for Flash Speculative Decoding", §4.1 Inference, §7.3 KV Injection
 * Mechanism; explainer page of the same name, "Putting It Together") is:
 *
 *   dflash_inject_context  stages 1+2: fuse the m target-layer hidden states of
 *                          newly committed tokens into H_t and append
 *                          W^K_i H_t (RoPE'd) and W^V_i H_t to every draft
 *                          layer's persistent context cache;
 *   dflash_draft_block     stages 3+4: one non-causal drafter pass over
 *                          [anchor, mask x (block_size-1)] and the shared LM
 *                          head with argmax -> block_size-1 draft tokens;
 *   dflash_verify_greedy   stage 5: greedy lossless verification against the
 *                          target's argmax -> accepted length tau, emitted
 *                          tokens and the next anchor.
 *
 * Conventions (all entry points):
 *  - Every pointer named *_dev, every weight and the cache/workspace memory is
 *    DEVICE memory owned by the caller; pointers named *_host are host memory.
 *    Nothing is copied: weight pointers are borrowed for the model's lifetime.
 *  - Matrices are row-major [out_features, in_features] (the Linear layout).
 *    Weights and target features are stored in the model's dtype
 *    (DFLASH_DTYPE_F32 or DFLASH_DTYPE_BF16).  Everything computed from them —
 *    the context K/V cache and every activation — is kept at fp32 precision and
 *    accumulated in fp32 (bf16 models feed the tensor cores each activation as
 *    a hi + lo bf16 pair against the exact bf16 weights).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Arguments are validated on the host before any launch;
 *    a non-zero return means nothing was launched, and dflash_last_error()
 *    gives a message.  Errors only the device can see (a cache that would
 *    overflow, a bounded wait that ran out) set the model's device status word,
 *    read with dflash_get_status().
 *  - No entry point allocates device memory except dflash_model_create (a few
 *    hundred bytes of model state).  Scratch memory is the caller's workspace.
 *  - Integer token ids are int32 in [0, vocab).
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque stream handle, ABI-compatible with cudaStream_t. */
typedef struct CUstream_st* dflash_stream_t;

/* Return codes. */
#define DFLASH_OK 0
#define DFLASH_ERR_INVALID_ARG (-1) /* null pointer, bad enum, negative size      */
#define DFLASH_ERR_SHAPE (-2)       /* shape the kernels do not support            */
#define DFLASH_ERR_CAPACITY (-3)    /* cache would overflow its capacity           */
#define DFLASH_ERR_CUDA (-4)        /* a CUDA runtime call failed                  */
#define DFLASH_ERR_TIMEOUT (-5)     /* (device status) a bounded wait ran out      */
#define DFLASH_ERR_UNSUPPORTED (-6) /* feature not built for this device           */
#define DFLASH_ERR_WORKSPACE (-7)   /* workspace smaller than dflash_workspace_bytes */

#define DFLASH_DTYPE_F32 0
#define DFLASH_DTYPE_BF16 1

/* Drafter shape.  Paper §5 Implementation: 5 draft layers, block size 16,
 * m = 5 target feature layers; §7.3: W_c in R^{D x mD}.  Qwen3-style layer:
 * RMSNorm, GQA attention with RoPE (rotate-half pairing), SwiGLU FFN.
 * Supported: hidden % 128 == 0, head_dim in {64, 128}, n_q_heads % n_kv_heads
 * == 0, ffn % 64 == 0, vocab % 128 == 0, n_target_feats in [1, 8],
 * 1 <= max_block <= 32. */
typedef struct {
  int32_t hidden;         /* D */
  int32_t layers;         /* draft layers */
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t ffn;            /* SwiGLU width F */
  int32_t vocab;          /* V (shared embedding and LM head rows) */
  int32_t n_target_feats; /* m */
  int32_t max_block;      /* largest block_size accepted by dflash_draft_block */
  float rope_theta;
  float rms_eps;
  int32_t mask_token_id;  /* embedding row used at every masked block position */
  int32_t dtype;          /* DFLASH_DTYPE_* */
  int32_t qk_norm;        /* 0, or 1: every query and key head (block and injected context keys) is
                             RMS-normalised over head_dim and scaled by the layer's g_q / g_k
                             before RoPE (Qwen3's q_norm / k_norm; not on the pages, off in their
                             configuration).  Models with it run the multi-kernel path. */
  int32_t input_fusion;   /* 0, or 1: the ablation of paper §5.5.5 — the fused context enters once, as
                             the context positions' input hidden states, and every draft layer
                             processes those positions (causal among the context) to produce its own
                             context K/V, instead of projecting H_t straight into every layer's K/V.
                             Changes dflash_inject_context only (multi-kernel path); drafting is the
                             same.  Not combined with qk_norm. */
  int32_t kv_bf16;        /* bf16 models: 0 keeps every cached context K/V value as a hi and a lo bf16
                             plane (fp32-level precision, 4 bytes a value); 1 keeps it rounded to one
                             bf16 (2 bytes a value: for the 8B shape 20,480 bytes a token over the 5
                             layers, the storage paper §7.3 counts).  Halves the cache and the bytes
                             the attention reads; the logits then follow the exact definition within
                             the bf16 rounding of the cache.  fp32 models: must be 0.  Not combined
                             with qk_norm. */
  int32_t head_bf16;      /* bf16 models: 1 hands the final normed hidden state to the LM head as one
                             bf16 (rounded to nearest) instead of a hi/lo pair, so the 151,936-wide
                             head projection runs at twice the tensor rate at batch scale; every other
                             tensor keeps fp32-level precision.  Models with it run the multi-kernel
                             path.  fp32 models: must be 0. */
} dflash_config;

/* Device pointers of one draft layer (borrowed).  Shapes with
 * Hq = n_q_heads*head_dim, Hk = n_kv_heads*head_dim:
 *   g_in [D], w_q [Hq,D], w_k [Hk,D], w_v [Hk,D], w_o [D,Hq],
 *   g_post [D], w_g [F,D], w_u [F,D], w_d [D,F],
 *   g_q [head_dim], g_k [head_dim] (QK-norm gains; read only when qk_norm, else may be NULL). */
typedef struct {
  const void* g_in;
  const void* w_q;
  const void* w_k;
  const void* w_v;
  const void* w_o;
  const void* g_post;
  const void* w_g;
  const void* w_u;
  const void* w_d;
  const void* g_q;
  const void* g_k;
} dflash_layer_weights;

/* Device pointers of the whole drafter (borrowed): embed [V,D] and
 * lm_head [V,D] (shared with the target, paper §4.2), w_c [D, m*D], g_c [D]
 * (fusion RMSNorm gain), g_final [D] (norm before the LM head).  `layers` is a
 * HOST array of `layers` entries, copied by dflash_model_create. */
typedef struct {
  const void* embed;
  const void* lm_head;
  const void* w_c;
  const void* g_c;
  const void* g_final;
  const dflash_layer_weights* layers;
} dflash_weights;

typedef struct dflash_model dflash_model;
typedef struct dflash_cache dflash_cache;

/* Library version (major*10000 + minor*100 + patch). */
int32_t dflash_version(void);

/* Thread-local message of the last failed call on this thread ("" if none). */
const char* dflash_last_error(void);

/* Validate `cfg`, copy it and the weight pointers, allocate the model's small
 * device state (status word, RoPE frequency table) on the current device and
 * prepare the tensor-core operand descriptors of every weight matrix.
 * On success *out owns that state until dflash_model_destroy. */
int32_t dflash_model_create(const dflash_config* cfg, const dflash_weights* w, dflash_model** out);
int32_t dflash_model_destroy(dflash_model* model);

/* Device status word: DFLASH_OK, or the first device-detected error since the
 * last clear (DFLASH_ERR_CAPACITY, DFLASH_ERR_TIMEOUT).  Synchronises `stream`. */
int32_t dflash_get_status(const dflash_model* model, dflash_stream_t stream, int32_t* status_host);
int32_t dflash_clear_status(const dflash_model* model, dflash_stream_t stream);

/* Self-test of device-side failure detection (the paper has no counterpart).
 * Launches one CTA on `stream` that waits, with the same bounded wait the
 * kernels' pipelines use, on an mbarrier in its own shared memory that
 * nothing ever arrives on.  After `budget_cycles` SM clock cycles (0 <
 * budget_cycles <= 4e9; 2e6 is about a millisecond) the wait gives up, the
 * kernel sets DFLASH_ERR_TIMEOUT in the model's status word and returns: no
 * fault, and the context stays usable.  Read the result with
 * dflash_get_status and clear it with dflash_clear_status.  Returns
 * DFLASH_ERR_INVALID_ARG for a NULL model or a budget outside the range. */
int32_t dflash_selftest_wait_timeout(const dflash_model* model, int64_t budget_cycles, dflash_stream_t stream);

/* --- persistent draft KV cache (paper §4.1: context K/V stored in the draft
 * model's KV cache and reused across drafting iterations) ----------------------
 * Layout inside the caller's block of device memory (each region 256-B aligned):
 *   fp32 models:  K [batch][layers][n_kv_heads][capacity][head_dim] fp32 (RoPE applied)
 *   bf16 models:  K [batch][layers][n_kv_heads][2][capacity][head_dim] bf16: planes
 *                 hi and lo with k = hi + lo (lo = the rounding residual of hi),
 *                 i.e. fp32-level precision in the same bytes
 *   V likewise
 *   ctx_len int32 [batch]                                (tokens held per request)
 * Only context entries live in the cache; a block's own K/V never does. */
size_t dflash_cache_bytes(const dflash_config* cfg, int32_t batch, int32_t capacity);

/* Carve a cache for `batch` requests of up to `capacity` tokens out of
 * `dev_mem` (>= dflash_cache_bytes) and zero every ctx_len on `stream`. */
int32_t dflash_cache_init(const dflash_model* model, void* dev_mem, size_t bytes, int32_t batch,
                          int32_t capacity, dflash_stream_t stream, dflash_cache** out);
int32_t dflash_cache_destroy(dflash_cache* cache);

/* Byte offsets of the K, V and ctx_len regions from dev_mem. */
int32_t dflash_cache_layout(const dflash_cache* cache, size_t* k_off, size_t* v_off, size_t* len_off);

/* Overwrite every request's ctx_len from host memory (e.g. to drop a request
 * or rewind).  Entries must lie in [0, capacity]. */
int32_t dflash_cache_set_lengths(dflash_cache* cache, const int32_t* ctx_len_host, dflash_stream_t stream);

/* --- workspace ----------------------------------------------------------------
 * Bytes of caller-owned device scratch that dflash_inject_context (with up to
 * `max_inject_rows` rows) and dflash_draft_block (with any block size up to
 * `block_size`) need for a cache of `batch` requests and `capacity` tokens.  One workspace may serve
 * every call on one stream; calls that overlap on the GPU need separate ones. */
size_t dflash_workspace_bytes(const dflash_model* model, int32_t batch, int32_t capacity, int32_t block_size,
                              int32_t max_inject_rows);

/* --- stage 1+2: context fusion and K/V injection ------------------------------
 * Paper §7.3: H_t = RMSNorm(W_c [H^(l1); ...; H^(lm)]);  per layer i the context
 * keys/values W^K_i H_t and W^V_i H_t; §4.1: persistent in the cache.
 *   feats       [max_rows][m][D] (dtype): the new tokens' target hidden states,
 *               request 0's rows first, then request 1's, ... (packed).
 *   n_new_dev   int32 [batch] device: rows per request this call.
 *   n_new_host  int32 [batch] host copy of n_new_dev, or NULL.  When given, the
 *               host checks sum <= max_rows and capacity exactly and returns
 *               DFLASH_ERR_CAPACITY without launching; when NULL (e.g. the
 *               counts come from dflash_verify_greedy on the device) the device
 *               drops rows that do not fit and sets DFLASH_ERR_CAPACITY in the
 *               status word.
 *   max_rows    rows the launch covers (>= sum of n_new); rows past the sum are
 *               ignored.
 * Token j of request b is placed at position ctx_len[b] + j (RoPE position of
 * its key) and ctx_len[b] grows by n_new[b]. */
int32_t dflash_inject_context(const dflash_model* model, dflash_cache* cache, const void* feats,
                              const int32_t* n_new_dev, const int32_t* n_new_host, int32_t max_rows,
                              void* workspace, size_t workspace_bytes, dflash_stream_t stream);

/* --- allocation-free injection --------------------------------------------------
 * The paper has no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory, so cannot provide the workspace that
 * dflash_inject_context needs: code that runs under a fixed, already committed
 * memory budget, runtimes that hand the library only the buffers of the
 * request being served, or hosts without access to a device allocator.
 *
 * Same arguments, results and checks as dflash_inject_context, minus the
 * workspace: the scratch lives in one file-scope device array of
 * dflash_noalloc_scratch_bytes() bytes (8 MiB) that every GPU loading this
 * library holds until the process exits.  No call allocates or frees memory.
 *   - A launch whose scratch plan exceeds that size (an 8B-shaped drafter
 *     fits the 16 to 32 rows of a cycle's injection) returns
 *     DFLASH_ERR_CAPACITY without launching; inject fewer rows per call.
 *   - The first call on a device looks the array's device address up with
 *     cudaGetSymbolAddress (with that device current) and caches it; make that
 *     first call before any stream capture.  The cache is keyed on the
 *     device's current context, so a call after cudaDeviceReset (which
 *     unloads the module holding the array) looks the address up again —
 *     that call, too, belongs before any capture.
 *   - Every call on a device shares the one array and leaves the last call's
 *     contents in it (what must start at zero is cleared by each call), so
 *     calls that overlap on the GPU — two streams, or two threads — race. */
size_t dflash_noalloc_scratch_bytes(void);
int32_t dflash_inject_context_noalloc(const dflash_model* model, dflash_cache* cache, const void* feats,
                                      const int32_t* n_new_dev, const int32_t* n_new_host, int32_t max_rows,
                                      dflash_stream_t stream);

/* --- stage 3+4: drafter forward pass, shared LM head, argmax -------------------
 * Paper §4.2 / explainer step 3: block = [anchor, mask x (block_size-1)] at
 * positions ctx_len[b] .. ctx_len[b]+block_size-1; every block row attends to
 * all of the request's context K/V and to every block row (no causal mask);
 * per layer RMSNorm -> Q,K,V (+RoPE) -> GQA attention -> W_O + residual ->
 * RMSNorm -> SwiGLU -> W_D + residual; then RMSNorm and the LM head on the
 * block_size-1 mask rows; draft = argmax (lowest token id on ties).
 *   anchor_dev  int32 [batch]: the clean anchor token of each request.
 *   draft_dev   int32 [batch][block_size-1]: written.
 *   logits_dev  fp32 [batch][block_size-1][vocab] or NULL: written if given.
 * The cache is read, never written. */
int32_t dflash_draft_block(const dflash_model* model, const dflash_cache* cache, const int32_t* anchor_dev,
                           int32_t block_size, int32_t* draft_dev, float* logits_dev, void* workspace,
                           size_t workspace_bytes, dflash_stream_t stream);

/* --- stages 1-4 in one call ---------------------------------------------------
 * dflash_inject_context(feats, n_new, max_rows) followed by
 * dflash_draft_block(anchor, block_size): the cycle of the explainer's
 * "Putting It Together" from the committed tokens' features to the drafts,
 * with the same arguments, checks and results (up to the order of fp32
 * additions).  When both fit one persistent launch (bf16 model without
 * qk_norm or input_fusion, max_rows <= 16, batch * block_size <= 16) they run
 * as ONE launch: the fusion projection first, then every layer's Q/K/V
 * projection computes the block's queries, keys and values and the injected
 * rows' context keys and values from one read of W_K and W_V.  Otherwise the
 * two calls run one after the other.  The workspace must hold
 * dflash_workspace_bytes(model, batch, capacity, block_size, max_rows). */
int32_t dflash_draft_cycle(const dflash_model* model, dflash_cache* cache, const void* feats,
                           const int32_t* n_new_dev, const int32_t* n_new_host, int32_t max_rows,
                           const int32_t* anchor_dev, int32_t block_size, int32_t* draft_dev, float* logits_dev,
                           void* workspace, size_t workspace_bytes, dflash_stream_t stream);

/* --- stage 5: greedy lossless verification -----------------------------------
 * Explainer, "The Target Verifier Remains the Correctness Anchor": accept drafts
 * left to right while they equal the target's greedy token, stop at the first
 * rejection; paper §3.1: tau in [1, gamma+1] counts the target's own token.
 *   draft_dev          int32 [batch][block_size-1]   d_1..d_{g-1}
 *   target_argmax_dev  int32 [batch][block_size]     y_0..y_{g-1}, y_k = target's
 *                      greedy token after block position k (y_0 judges d_1)
 *   accept_len_dev     int32 [batch] written: tau = n + 1, n = leading matches
 *   out_tokens_dev     int32 [batch][block_size] written: d_1..d_n, y_n, then -1
 *   next_anchor_dev    int32 [batch] written: y_n (correction or bonus)
 * Needs no model; batch may be 0 (no launch). */
int32_t dflash_verify_greedy(const int32_t* draft_dev, const int32_t* target_argmax_dev, int32_t batch,
                             int32_t block_size, int32_t* accept_len_dev, int32_t* out_tokens_dev,
                             int32_t* next_anchor_dev, dflash_stream_t stream);

/* --- stage 5, sampled: stochastic lossless verification -----------------------
 * Explainer, "The Target Verifier Remains the Correctness Anchor" (acceptance
 * probability min(1, p_t/p_d), stop at the first rejection, correction from
 * the residual distribution, bonus token when the whole block survives);
 * paper §5.1 (temperature-1 results).  p_d and p_t are softmax(logits / T) of
 * the drafter's and the target's fp32 logits rows.  Left to right, draft d_k
 * (proposed from p_d row k-1) is kept iff u_accept[b][k-1] < min(1,
 * p_t(d_k) / p_d(d_k)); a draft with p_d = 0 counts as kept, an id outside
 * [0, vocab) as rejected.  At the first rejection, position k, the target
 * draws the correction from max(0, p_t - p_d) of row k, normalised (the
 * residual that makes the rule lossless), and the rest of the block is
 * dropped; when every draft is kept it draws the bonus from target row
 * block-1.  Each draw is an inverse-CDF draw with one uniform u: the smallest
 * id (increasing order) whose cumulative mass exceeds u times the total mass
 * (the last id with mass if rounding leaves none).
 *   draft_logits_dev   fp32 [batch][block-1][vocab] (dflash_draft_block's logits)
 *   target_logits_dev  fp32 [batch][block][vocab]; row k: the target's logits
 *                      for the token after block position k (row 0 judges d_1)
 *   draft_dev          int32 [batch][block-1]: the proposed tokens
 *   u_accept_dev       fp32 [batch][block-1] and u_sample_dev fp32 [batch]:
 *                      uniforms in [0, 1) from the caller (the library draws none)
 *   accept_len_dev, out_tokens_dev, next_anchor_dev: as dflash_verify_greedy
 *   workspace          >= dflash_sampling_workspace_bytes(batch*(2*block-1), batch, vocab)
 * Requires vocab % 4 == 0, vocab <= 2^24, 16-byte aligned logits, batch *
 * (2*block-1) <= 65535, 0 < temperature < inf; batch may be 0 (no launch).
 * The logits are read once for the rows' normalisers and once more for the
 * one or two rows each request draws from. */
size_t dflash_sampling_workspace_bytes(int32_t rows, int32_t draws, int32_t vocab);
int32_t dflash_verify_sampled(const float* draft_logits_dev, const float* target_logits_dev, const int32_t* draft_dev,
                              const float* u_accept_dev, const float* u_sample_dev, int32_t batch, int32_t block_size,
                              int32_t vocab, float temperature, int32_t* accept_len_dev, int32_t* out_tokens_dev,
                              int32_t* next_anchor_dev, void* workspace, size_t workspace_bytes,
                              dflash_stream_t stream);

/* Inverse-CDF draw of one token per logits row: tokens[r] = the smallest id
 * whose cumulative mass under softmax(logits[r] / T) exceeds u[r] — how a
 * sampling drafter proposes its block from dflash_draft_block's logits before
 * dflash_verify_sampled (explainer, same section: x_k drawn from p_d).
 *   logits_dev fp32 [rows][vocab], u_dev fp32 [rows] in [0, 1), tokens_dev int32 [rows]
 *   workspace >= dflash_sampling_workspace_bytes(rows, rows, vocab)
 * Same requirements as dflash_verify_sampled (rows <= 65535). */
int32_t dflash_sample_tokens(const float* logits_dev, int32_t rows, int32_t vocab, float temperature,
                             const float* u_dev, int32_t* tokens_dev, void* workspace, size_t workspace_bytes,
                             dflash_stream_t stream);

/* --- training-time packed block attention (forward) ---------------------------
 * Paper §4.2: training samples anchors from a sequence, opens a block of
 * block_size positions at each, concatenates all blocks and runs them in one
 * pass under a sparse mask; explainer "Training Rehearses the Same Masked
 * Blocks Used at Runtime" (Figure 4): clean target context features are
 * visible to each block, positions attend bidirectionally inside their own
 * block, and nothing crosses between blocks.  Reading (matches inference,
 * where the block starts right after the injected context): block n, anchored
 * at position a_n, sees context keys 0 .. a_n - 1 and its own block_size rows.
 * softmax(q k^T / sqrt(head_dim)) v with grouped-query heads (q head h reads
 * kv head h / (n_q_heads / n_kv_heads)); no mask is materialised.
 *   q_dev       [n_blocks][block][n_q_heads][head_dim]   block queries (RoPE applied)
 *   k_ctx_dev, v_ctx_dev  [seq_len][n_kv_heads][head_dim]  the sequence's context keys / values
 *   k_blk_dev, v_blk_dev  [n_blocks][block][n_kv_heads][head_dim]  the blocks' own keys / values
 *               (all five in `dtype`: DFLASH_DTYPE_F32 or DFLASH_DTYPE_BF16)
 *   anchors_dev int32 [n_blocks] device; anchors_host: the same on the host, or
 *               NULL.  Given, every anchor is checked to lie in [0, seq_len] and
 *               DFLASH_ERR_INVALID_ARG is returned without a launch; otherwise
 *               the device clamps an anchor outside and sets the status word.
 *   out_dev     fp32 [n_blocks][block][n_q_heads][head_dim]
 *   workspace   >= dflash_packed_attention_workspace_bytes(...) bytes, 256-byte
 *               aligned; its first int32 is the call's status word (0, or
 *               DFLASH_ERR_INVALID_ARG / DFLASH_ERR_TIMEOUT), read with
 *               dflash_packed_attention_status.
 * Operands run through the tensor cores at fp32 precision (hi/lo bf16 pairs).
 * head_dim 64 or 128; 1 <= block <= 32; n_blocks * n_kv_heads <= 65535.
 * The workspace size depends on the current device's SM count. */
size_t dflash_packed_attention_workspace_bytes(int32_t n_blocks, int32_t block, int32_t seq_len, int32_t n_q_heads,
                                               int32_t n_kv_heads, int32_t head_dim);
int32_t dflash_packed_block_attention(const void* q_dev, const void* k_ctx_dev, const void* v_ctx_dev,
                                      const void* k_blk_dev, const void* v_blk_dev, const int32_t* anchors_dev,
                                      const int32_t* anchors_host, int32_t n_blocks, int32_t block, int32_t seq_len,
                                      int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t dtype,
                                      float* out_dev, void* workspace, size_t workspace_bytes,
                                      dflash_stream_t stream);
/* Synchronises `stream` and copies the call's status word to *status_host. */
int32_t dflash_packed_attention_status(const void* workspace, dflash_stream_t stream, int32_t* status_host);

/* --- block-size scheduling (host policy) ---------------------------------------
 * Paper §5.5.4: a drafter trained at a large block size serves smaller
 * inference-time block sizes nearly as well, and large blocks raise the
 * verification cost when the target is compute-bound (large batches), so the
 * block size can be chosen per cycle.  This policy runs on the host, between
 * cycles, over the existing kernels:
 *   - dflash_block_policy_observe records a cycle's accepted lengths tau
 *     (one per request, read back from dflash_verify_greedy/_sampled): draft
 *     position j was attempted when every earlier draft of its block was kept
 *     and j < block_size, and kept when j <= tau - 1; the counts of earlier
 *     cycles are first multiplied by `decay`.
 *   - alpha_j = (kept_j + prior_accept * prior_weight) / (attempted_j + prior_weight)
 *     estimates P(draft j kept | earlier drafts kept).
 *   - dflash_block_policy_choose returns the candidate g maximising
 *     batch * E[tau | g] / cost(g), E[tau | g] = 1 + sum_{i<g} prod_{j<=i}
 *     alpha_j (blog "Inside DFlash ...", section 1), cost(g) = cost_fixed_ms +
 *     cost_per_row_ms * batch * g + cost_per_request_ms * batch (a linear
 *     model of drafting and verifying batch * g token rows, measured by the
 *     caller); ties go to the smaller block.  Arithmetic in double precision.
 * Candidates are strictly ascending in [1, DFLASH_POLICY_MAX_BLOCK];
 * 0 < decay <= 1, prior_accept in [0, 1], prior_weight > 0, costs >= 0 with a
 * positive sum.  A policy is plain host memory and is not thread-safe. */
#define DFLASH_POLICY_MAX_CANDIDATES 16
#define DFLASH_POLICY_MAX_BLOCK 32
typedef struct {
  int32_t n_candidates;
  int32_t candidates[DFLASH_POLICY_MAX_CANDIDATES];
  float cost_fixed_ms;
  float cost_per_row_ms;
  float cost_per_request_ms;
  float decay;
  float prior_accept;
  float prior_weight;
} dflash_block_policy_config;
typedef struct dflash_block_policy dflash_block_policy;

int32_t dflash_block_policy_create(const dflash_block_policy_config* cfg, dflash_block_policy** out);
int32_t dflash_block_policy_destroy(dflash_block_policy* policy);
/* accept_len_host: int32 [batch] HOST array of one cycle's tau, 1 <= tau <= block_size. */
int32_t dflash_block_policy_observe(dflash_block_policy* policy, int32_t block_size, const int32_t* accept_len_host,
                                    int32_t batch);
/* *block_size_out = the chosen candidate; *expected_tau_out (may be NULL) = its E[tau]. */
int32_t dflash_block_policy_choose(const dflash_block_policy* policy, int32_t batch, int32_t* block_size_out,
                                   double* expected_tau_out);
/* alpha_out[j] = the estimate for draft position j+1 (0 beyond the largest candidate - 1). */
int32_t dflash_block_policy_acceptance(const dflash_block_policy* policy, double* alpha_out, int32_t n);

/* --- benchmark utility (not part of the method) --------------------------------
 * The synthetic target the benchmark and tests put between dflash_draft_block
 * and dflash_verify_greedy in place of a real target model, as one kernel.
 * With p = *pattern_idx_dev (int64, device), for every request b:
 *   target[b][k] = draft[b][k]                        if match[p][b][k] != 0
 *                = (draft[b][k] + 1 + off[p][b][k]) % vocab   otherwise  (k < block-1)
 *   target[b][block-1] = bonus[p][b]
 * then *pattern_idx_dev = (p + 1) % n_patterns, and, when tau_dev and
 * tau_sum_dev are given, *tau_sum_dev += sum_b tau_dev[b] (the accepted
 * lengths of the previous verification).  match: uint8 [n_patterns][batch][block-1],
 * off: int32 [n_patterns][batch][block-1], bonus: int32 [n_patterns][batch],
 * target: int32 [batch][block]. */
int32_t dflash_synthetic_target(const int32_t* draft_dev, const uint8_t* match_dev, const int32_t* off_dev,
                                const int32_t* bonus_dev, int32_t n_patterns, int64_t* pattern_idx_dev,
                                const int32_t* tau_dev, int64_t* tau_sum_dev, int32_t batch, int32_t block_size,
                                int32_t vocab, int32_t* target_dev, dflash_stream_t stream);

/* --- tracing -------------------------------------------------------------------
 * Kernel launches made by this library in this process (every entry point,
 * every device), for launch accounting. */
uint64_t dflash_launch_count(void);

/* Per-CTA timestamps, for performance work.  When the environment variable
 * DFLASH_TRACE_GEMM=<k> is set at model creation, the model's k-th GEMM launch
 * of the multi-kernel path (counting from 0) records, for every CTA c, 8
 * values at host[8c .. 8c+7]: globaltimer ns at start, after set-up, when the
 * first and the last K stage landed, when the accumulator was ready and at
 * the end; the SM id; 1 if the CTA ran the split-K reduction.  With
 * DFLASH_TRACE_PERSIST=1 instead, every persistent drafter launch records 18
 * values per (CTA, phase) at host[(c*56 + phase)*18 ..]: phase start and end,
 * first/last weight load issued, activation loads released, first/last MMA
 * issued, the SM id, the cycles the MMA issuer and the producers waited, and
 * the steps of the phase's last output tile (persist.cu lists them).
 * Copies min(n, 8*65536) values; DFLASH_ERR_UNSUPPORTED when tracing is off. */
int32_t dflash_trace_read(const dflash_model* model, uint64_t* host, size_t n);

/* Stage ids reported by the profiler. */
#define DFLASH_STAGE_FUSE 0     /* fusion GEMM (W_c)                          */
#define DFLASH_STAGE_INJECT 1   /* K/V injection GEMM (all layers)            */
#define DFLASH_STAGE_QKV 2      /* drafter Q/K/V GEMMs                        */
#define DFLASH_STAGE_ATTN 3     /* block attention (split + merge)            */
#define DFLASH_STAGE_O 4        /* W_O GEMMs                                  */
#define DFLASH_STAGE_GATEUP 5   /* W_G/W_U GEMMs with SwiGLU                  */
#define DFLASH_STAGE_DOWN 6     /* W_D GEMMs                                  */
#define DFLASH_STAGE_LMHEAD 7   /* LM head GEMM with argmax                   */
#define DFLASH_STAGE_OTHER 8    /* embedding, norms, row maps, argmax read-out */
#define DFLASH_STAGE_INJECT_PERSIST 9  /* one-launch injection (fusion + K/V), <= 16 rows */
#define DFLASH_STAGE_DRAFT_PERSIST 10  /* one-launch drafter pass (layers + LM head), <= 16 rows */
#define DFLASH_STAGE_CYCLE_PERSIST 11  /* one-launch injection + drafter pass (dflash_draft_cycle) */
#define DFLASH_NUM_STAGES 12

/* Start recording a CUDA event pair around each launch the model's entry
 * points make (up to max_launches launches), on the stream each call is given.
 * Meant for measurement runs, not for stream capture. */
int32_t dflash_profile_start(dflash_model* model, int32_t max_launches);

/* Synchronise `stream`, stop recording and return per stage the summed launch
 * time in milliseconds and the launch count (arrays of n_stages entries,
 * n_stages <= DFLASH_NUM_STAGES). */
int32_t dflash_profile_stop(dflash_model* model, dflash_stream_t stream, float* ms_by_stage,
                            int32_t* launches_by_stage, int32_t n_stages);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H_ */
