/*
 * llm.h — C ABI of the GB300 (sm_103a) Llama decoder forward pass.
 *
 * One model (weights in library-owned device memory), one or more contexts
 * (KV cache + workspaces + captured decode graphs), and a batch call that
 * runs prefill or decode over it.  The calls follow the pages' statement of
 * the problem:
 *   - "Inside the inference engine: model architectures and forward pass",
 *     section "Detailed explanation: Llama's forward pass in Go" — the math of
 *     Model.Forward and layer.Forward; section "KV Cache: memory for causal
 *     attention" — the per-layer, per-sequence cache; section "Token sampling
 *     pipeline" — temperature 0 is argmax.
 *   - "LLama.cpp — how it works", "Step 10" (llama_batch and the defaults of
 *     llama_batch_allocr::init), "Steps 11–12" (llama_decode, the ubatch split
 *     of init_batch, the return codes), "Steps 14–15" (llama_get_logits_ith),
 *     "KV-cache and the Prefill / Decode stages" (seq_pos_max).
 *
 * Conventions for every call:
 *   - Device pointers are CUDA global-memory addresses on the device that is
 *     current when the model is created; host pointers are ordinary host
 *     memory.  Each argument says which it is.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All device work of a context is ordered on its stream; a
 *     context given NULL creates its own blocking stream, which the legacy
 *     default stream orders against, because the legacy stream cannot be
 *     captured into a CUDA graph.
 *   - Return codes: LLM_OK (0) success; LLM_NO_KV_ROOM (1) the batch does not
 *     fit the KV cache, nothing was written (the non-error "1" of
 *     llama_decode); LLM_ERR_INVALID (-1) invalid argument or batch;
 *     LLM_ERR_ALLOC (-2) device or host allocation failed; LLM_ERR_COMPUTE (-3)
 *     a CUDA launch or copy failed, or a kernel raised its error flag.
 *     A failed call leaves the context's cache metadata unchanged.
 *   - llm_last_error(ctx) gives a one-line description of the last failure of
 *     that context (or of the last failed create call when ctx is NULL).
 *   - No call is thread-safe against other calls on the same context.
 */
#ifndef LLM_H
#define LLM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LLM_OK 0
#define LLM_NO_KV_ROOM 1
#define LLM_ERR_INVALID (-1)
#define LLM_ERR_ALLOC (-2)
#define LLM_ERR_COMPUTE (-3)

typedef struct llm_model llm_model;
typedef struct llm_ctx llm_ctx;

/* Model hyper-parameters (llama.cpp "hparams": n_vocab, n_embd, n_layer,
 * n_head, n_head_kv, head dimension, n_ff, RMSNorm eps, RoPE base).
 * tied_output != 0 means the output projection is token_embd
 * (GGUF tag "output,alt:token_embd").  Requirements: n_head % n_head_kv == 0;
 * head_dim in {32, 64, 128}; n_embd, n_head*head_dim and n_vocab multiples of
 * 128; n_head_kv*head_dim a multiple of 64; n_ff >= 1 (padded internally). */
typedef struct {
    int32_t n_vocab, n_embd, n_layer, n_head, n_head_kv, head_dim, n_ff;
    float rms_eps, rope_theta;
    int32_t tied_output;
} llm_hparams;

/* Weight pointers (all DEVICE, bf16, row-major [out][in]; read only during
 * llm_model_create, which copies and repacks them, so the caller may free
 * them afterwards).  Per-layer entries are HOST arrays of n_layer DEVICE
 * pointers.  Shapes: token_embd/output [n_vocab][n_embd]; norms [n_embd];
 * wq [n_head*hd][n_embd]; wk, wv [n_head_kv*hd][n_embd]; wo [n_embd][n_head*hd];
 * w_gate, w_up [n_ff][n_embd]; w_down [n_embd][n_ff].  `output` must be NULL
 * iff hparams.tied_output != 0. */
typedef struct {
    const void *token_embd, *output_norm, *output;
    const void *const *attn_norm, *const *wq, *const *wk, *const *wv, *const *wo;
    const void *const *ffn_norm, *const *w_gate, *const *w_up, *const *w_down;
} llm_weights;

/* Copy the weights into library-owned device memory in the kernels' layout:
 * Wq, Wk, Wv concatenated per layer; gate and up interleaved in groups of 8
 * rows; the FFN dimension zero-padded to a multiple of 128; norm gains
 * widened to fp32.  Matrices are stored as fp16, the operand type of every
 * tensor-core contraction and of the KV cache: bf16 -> fp16 is exact for
 * 2^-14 <= |w| <= 65504 and rounds smaller magnitudes to the fp16 subnormal
 * grid (absolute error <= 2^-25); a weight above 65504 makes the call fail
 * with LLM_ERR_INVALID.  Runs on `stream` and synchronizes it before
 * returning.  On failure *out = NULL and a negative code is returned. */
int32_t llm_model_create(const llm_hparams *hp, const llm_weights *w, void *stream,
                         llm_model **out);
/* Free a model.  All its contexts must have been freed first. */
void llm_model_free(llm_model *m);

/* Weight types of llm_model_quantize. */
#define LLM_WTYPE_Q8_0 1

/* Re-encode the model's matrices as Q8_0 blocks.  "LLama.cpp — how it
 * works", section "The GGUF format (reference)", names Q8_0 among the
 * quantised tensor element types without giving its layout; the one taken:
 * each row of Wq, Wk, Wv, Wo, gate, up, down and the output projection is cut
 * into blocks of 32 consecutive elements; a block keeps d = max|w| / 127
 * (float32 division, stored rounded to fp16) and codes q = the nearest
 * integer to w / d (float32 division, ties to even; |q| <= 127), and stands
 * for the weights q * d (stored d); a block of zeros has d = 0, q = 0.
 * Afterwards the model computes with those weights everywhere: its fp16
 * copies become f16(q * d) (one rounding; read by prefill and by steps of 2-8
 * rows), and when n_embd, n_head*head_dim and the padded n_ff are multiples of
 * 256 the Q8_0 rows are kept beside them (N rows of K + K/16 bytes: the codes,
 * then the fp16 scales) for the one-row streamed decode GEMVs, which then
 * read 17/32 of the fp16 bytes.  The token embedding is a lookup and stays as
 * created, unless it is the output projection (tied).  Call it before any
 * context of the model exists.  Returns LLM_ERR_INVALID (nothing changed) for
 * an unknown wtype, a model that has live contexts or is already quantised;
 * LLM_ERR_ALLOC if the Q8_0 rows cannot be allocated (nothing changed);
 * LLM_ERR_COMPUTE if a launch fails, after which the model's weights are
 * undefined and it should be freed.  Runs on `stream` and synchronizes it. */
int32_t llm_model_quantize(llm_model *m, int32_t wtype, void *stream);

/* Create a context ("llama_new_context"): an fp16 KV cache of n_ctx positions
 * for each of n_seq_max sequences and every layer, laid out
 * [seq][layer][kv_head][pos][head_dim] for K and for V; activation
 * workspaces for ubatches of up to n_ubatch tokens (1..4096); fp32 RoPE
 * cos/sin tables for positions [0, n_ctx) computed in double precision on the
 * host.  Decode steps (ubatches of 1..8 tokens that are all output rows) are
 * captured into a CUDA graph on first use and replayed afterwards.  The
 * context keeps a reference to `m`, which must outlive it. */
int32_t llm_kv_alloc(llm_model *m, int32_t n_ctx, int32_t n_seq_max, int32_t n_ubatch,
                     void *stream, llm_ctx **out);
void llm_kv_free(llm_ctx *c);

/* The batch of one llm_decode call ("llama_batch", one sequence id per
 * token).  All arrays have n_tokens entries and are HOST memory, except
 * `token`, which is DEVICE memory when (flags & LLM_BATCH_TOKENS_ON_DEVICE).
 *   pos    NULL: each sequence continues at seq_pos_max(seq)+1, in batch order.
 *          Given: must equal exactly those values (no gaps, no rewrites).
 *   seq_id NULL: every token belongs to sequence 0.  Values in [0, n_seq_max).
 *   output NULL: logits for the last row only.  Nonzero: logits for that row.
 * Host token ids are checked to lie in [0, n_vocab); device token ids are
 * checked by the embedding kernel, which raises the context's error flag
 * (reported by llm_synchronize) and embeds a zero row instead. */
#define LLM_BATCH_TOKENS_ON_DEVICE 1
typedef struct {
    int32_t n_tokens;
    const int32_t *token;
    const int32_t *pos;
    const int32_t *seq_id;
    const int8_t *output;
    int32_t flags;
} llm_batch;

/* Run a batch through the model ("llama_decode"): validate it and fill its
 * defaults, return LLM_NO_KV_ROOM if any position would reach n_ctx, cut it
 * into consecutive ubatches of at most n_ubatch tokens, and for each ubatch
 * enqueue on the context's stream: embedding, every layer (K and V of all
 * rows appended to the cache before attention; only the output rows kept
 * before the last layer's MLP), final RMSNorm and output projection of the
 * output rows.  Ubatches of 1..8 rows run the decode kernels (GEMV + split
 * attention), larger ones the prefill kernels (tensor-core GEMM + tiled
 * attention).  Logits of all output rows are kept in batch order.
 * Asynchronous: returns once the work is enqueued; the logits are valid after
 * the stream reaches that point (llm_synchronize, or any later call that
 * reads them to the host). */
int32_t llm_decode(llm_ctx *c, const llm_batch *b);

/* DEVICE pointer to the logits of the last llm_decode / llm_generate:
 * fp32 [n_outputs][n_vocab], rows in batch order.  Owned by the context and
 * valid until the next decode call.  *n_outputs (if not NULL) receives the
 * row count.  NULL if there are none. */
const float *llm_get_logits(llm_ctx *c, int32_t *n_outputs);

/* DEVICE pointer to the logits row of batch index i of the last llm_decode
 * ("llama_get_logits_ith"); i < 0 counts from the end of the output rows
 * (-1 = last output).  NULL if row i was not an output or is out of range. */
const float *llm_get_logits_ith(llm_ctx *c, int32_t i);

/* Greedy choice ("temperature 0 -> argmax"; ties go to the lowest token id)
 * for every output row of the last decode.  Writes n_outputs token ids to the
 * HOST array `out` (capacity entries) and synchronizes the stream.  Returns
 * n_outputs, or a negative code. */
int32_t llm_get_argmax(llm_ctx *c, int32_t *out, int32_t capacity);

/* The token sampling chain ("Inside the inference engine: model architectures
 * and forward pass", section "Token sampling pipeline"; "LLama.cpp — how it
 * works", "Steps 14–15", the sampler chain), applied to each output row of
 * the last decode in this order:
 *   temperature <= 0: greedy argmax (ties to the lowest id); otherwise
 *   repeat penalty: each distinct token among the last penalty_last_n entries
 *     of `history` has its logit divided by repeat_penalty if positive, else
 *     multiplied by it (1 = off; must be > 0);
 *   top-K: the top_k largest logits (1..1024, ties to the lowest id), ordered
 *     by logit descending then id ascending;
 *   temperature: logits / temperature; softmax;
 *   top-P: the shortest prefix whose cumulative probability reaches top_p
 *     (>= 1 = off; must be > 0);
 *   min-P: the tokens with probability >= min_p * the top probability
 *     (<= 0 = off; must be < 1);
 *   draw: the first kept token whose running probability sum exceeds
 *     u * (kept total).
 * The float32 sums are taken in that order by one thread, so equal inputs give
 * equal tokens.  u: HOST array of n_outputs uniforms in [0, 1), one per row
 * (not read when greedy): the caller owns the random stream, which makes the
 * output reproducible.  history: HOST array of n_history earlier tokens (may
 * be NULL when n_history is 0), shared by every row.  Writes n_outputs tokens
 * to the HOST array `out` and synchronizes the stream.  Returns n_outputs, or
 * a negative code (LLM_ERR_INVALID for parameters outside these ranges or a
 * vocabulary above 262144). */
typedef struct {
    float temperature;
    int32_t top_k;
    float top_p;
    float min_p;
    float repeat_penalty;
    int32_t penalty_last_n;
} llm_sampling;
int32_t llm_sample(llm_ctx *c, const llm_sampling *s, const float *u, const int32_t *history,
                   int32_t n_history, int32_t *out, int32_t capacity);

/* Greedy generation on the device for one sequence, with no host round trip
 * per token: take the argmax of the last output row of the previous decode,
 * decode that token at the sequence's next position, take the argmax of its
 * logits, and so on, n_steps times.  tokens_out is a DEVICE int32 array of
 * n_steps entries that receives the chosen tokens in order.  Each step replays
 * the captured 1-token decode graph.  Asynchronous like llm_decode.  Returns
 * LLM_NO_KV_ROOM (nothing run) if the sequence would pass n_ctx. */
int32_t llm_generate(llm_ctx *c, int32_t seq_id, int32_t n_steps, int32_t *tokens_out);

/* Highest cached position of sequence s, or -1 if empty ("seq_pos_max"). */
int32_t llm_seq_pos_max(llm_ctx *c, int32_t seq_id);
/* Forget every cached position of sequence s. */
int32_t llm_seq_clear(llm_ctx *c, int32_t seq_id);
/* Context shift ("Inside the inference engine: model architectures and
 * forward pass", "KV Cache": when the cache is full the model's Shift
 * function adjusts the RoPE position encoding so the window slides forward):
 * drop positions [p0, p0 + n_discard) of sequence s; every later cached
 * position p moves to p - n_discard, its key re-rotated by the RoPE rotation
 * of -n_discard, its value unchanged.  The sequence then continues at
 * seq_pos_max + 1 - n_discard.  Asynchronous on the context stream.  Returns
 * LLM_ERR_INVALID (nothing changed) unless 0 <= p0, n_discard >= 1 and
 * p0 + n_discard <= seq_pos_max + 1. */
int32_t llm_seq_shift(llm_ctx *c, int32_t seq_id, int32_t p0, int32_t n_discard);

/* Host-only check of a batch (no GPU needed): applies exactly the rules of
 * llm_decode to a cache whose sequences end at seq_pos_max[0..n_seq_max)
 * (HOST array, -1 = empty).  On LLM_OK fills, when not NULL, the HOST arrays
 * pos_out[n_tokens] (positions), out_index[n_tokens] (logits row of each
 * batch row, -1 if none) and ubatch_starts[*n_ubatches] (first row of each
 * ubatch of at most n_ubatch rows).  Returns the code llm_decode would. */
int32_t llm_batch_check(int32_t n_vocab, int32_t n_ctx, int32_t n_seq_max, int32_t n_ubatch,
                        const int32_t *seq_pos_max, const llm_batch *b, int32_t *pos_out,
                        int32_t *out_index, int32_t *ubatch_starts, int32_t *n_ubatches);

/* Wait for the context's stream; return LLM_ERR_COMPUTE if a CUDA error
 * occurred or a kernel raised the error flag (the flag is then cleared),
 * LLM_OK otherwise.  llm_last_error names what the flag records: a token id
 * outside the vocabulary, a sequence / position / row index out of range, a
 * bounded wait that timed out, or an activation that had to be narrowed to
 * fp16 (tensor-core operands, the KV cache, the SwiGLU output) while not
 * finite or beyond +-65504 (the fp16 range the library's precision relies
 * on). */
int32_t llm_synchronize(llm_ctx *c);

/* One-line description of the last failure (static storage; never NULL). */
const char *llm_last_error(const llm_ctx *c);

/* Diagnostics: when dst is not NULL, every following llm_decode copies the
 * hidden state after each layer into DEVICE fp32 memory dst laid out
 * [ubatch][layer][row][n_embd] with max_rows rows per (ubatch, layer) slot
 * (the last layer holds only the output rows).  max_ubatches bounds the
 * ubatch index.  Pass dst = NULL to stop. */
int32_t llm_debug_hidden(llm_ctx *c, float *dst, int32_t max_rows, int32_t max_ubatches);

/* Tests of the failure paths.  llm_debug_fail_alloc(n): in the next
 * llm_kv_alloc call (only), its device allocation number n (0-based, in the
 * order the call makes them) fails as if the device were out of memory, so
 * the call returns LLM_ERR_ALLOC after releasing what it had allocated; -1
 * disarms.  Process-wide; returns LLM_ERR_INVALID for n < -1. */
int32_t llm_debug_fail_alloc(int32_t n);

/* Tuning/diagnostic switches (key, value); returns LLM_ERR_INVALID for an
 * unknown key or value.  Keys:
 *   "graphs"       1 = capture decode steps in CUDA graphs (default 1);
 *   "pdl"          programmatic dependent launch for the decode GEMVs and the
 *                  small kernels (default 0: a one-wave GEMV grid that starts
 *                  beside the previous kernel's CTAs spreads unevenly over the SMs);
 *   "pdl_attn"     the same for decode attention, which then streams its cached
 *                  K/V rows while the QKV kernel still runs (default 1);
 *   "pdl_prefill"  the same for the prefill kernels (default 1);
 *   "gemm"         prefill GEMM schedule, all tcgen05/TMEM on CTA pairs
 *                  (cta_group::2, 256-row tiles fed by TMA): 2 = one tile a
 *                  pair, persistent with double-buffered accumulators when the
 *                  tiles exceed one wave (default); 3 = persistent for every
 *                  GEMM; 4 = stream-K: every resident pair takes an equal run
 *                  of K stages across the 256-wide tiles, split tiles finished
 *                  by the pair holding their first stages (GEMMs whose N is
 *                  not a multiple of 256 use schedule 2);
 *   "attn_prefill" 1 = prefill attention on tcgen05, one CTA per query head
 *                  (default; fp16 cache, head_dim 64 or 128); 2 = tcgen05
 *                  with the two query heads of a GQA group on a CTA pair
 *                  (head_dim 128 and an even H / Hkv, else as 1); 0 = the
 *                  mma.sync kernel (always used for head_dim 32 and the FP8
 *                  cache);
 *   "gemv_stream"  1 = one-row steps run their GEMVs streamed through shared
 *                  memory, one CTA per SM, each launch overlapping the previous
 *                  kernel's tail (default, when every GEMV shape allows it:
 *                  K a multiple of 256 up to 16384); 0 = the register-fragment
 *                  GEMV for every row count;
 *   "gemv_stage_kb"  largest ring stage (KB) of the streamed GEMVs, 16..128: each
 *                  warp then takes several rows of a stage (0 = default: one
 *                  row a warp for fp16 rows, up to 96 KB stages for Q8_0 rows);
 *   "gemv_q8"      1 = the streamed one-row GEMVs of a Q8_0 model read its Q8_0
 *                  rows (default); 0 = its fp16 copies (the same weights up to
 *                  one fp16 rounding, twice the bytes);
 *   "gemv_prefetch_kb"  streamed GEMVs: KB per CTA of the next GEMV's weights
 *                  prefetched into L2 while the current one drains (default
 *                  128; the output projection's weights are prefetched whole
 *                  during attention); 0 = off;
 *   "gemm_resid_tma"  1 = the prefill residual GEMMs (O, down) read their tile
 *                  of h into shared memory by TMA while their last MMAs run and
 *                  write h and the next norm's input back by TMA stores
 *                  (default); 0 = each thread reads and writes its row;
 *   "gemm_split_k"  1 = a prefill residual GEMM with K >= 8192 (down) runs on
 *                  256-wide tiles with K split in two, the halves exchanging
 *                  their partial accumulators (default); 0 = 128-wide tiles;
 *   "gemv_prefetch2_kb"  KB per CTA of the gate/up weights the QKV GEMV also
 *                  prefetches into L2, read while decode attention leaves HBM
 *                  idle (default 256); 0 = off;
 *   "kv_fp8"       1 = the KV cache holds FP8 E4M3 elements (nearest, saturating
 *                  at +-448, no scale; half the bytes of the fp16 cache), 0 =
 *                  fp16 (default); allowed only while every sequence is empty
 *                  (the cache is reallocated);
 *   "swa_window"   sliding-window attention ("KV Cache" of the pages): a query at
 *                  position p sees only keys at p - W < position <= p of its
 *                  sequence (0 = every earlier position, the default);
 *   "gemv_path_max_rows"  largest ubatch sent to the decode kernels, 0..8;
 *   "ksplit_qkv", "ksplit_o", "ksplit_gateup", "ksplit_down", "ksplit_lm"
 *                  K splits of the decode GEMVs, 0 = the library's choice (the
 *                  largest split whose grid fits one wave of resident CTAs);
 *   "attn_split"   sequence splits of one-row decode attention, 0 = auto;
 *   "attn_split_rows"  the same for 2-8-row decode steps. */
int32_t llm_set_option(llm_ctx *c, const char *key, int32_t value);

/* Number of kernel launches the context has enqueued so far (graph replays
 * count each captured kernel).  Used to report launch counts. */
int64_t llm_kernel_launches(const llm_ctx *c);

/* Diagnostics: per-kernel timing.  With enable != 0 every following launch is
 * bracketed by CUDA events on the context stream (decode graphs and
 * programmatic dependent launch are bypassed meanwhile, so each kernel runs
 * alone); the totals restart at zero on every call.  llm_kernel_time
 * synchronizes the stream and reports, for kernel class `kernel` (0 ..
 * LLM_KERNEL_CLASSES-1), the summed duration in milliseconds, the launch count
 * and a static name ("gemv_gateup_swiglu", "attn_decode", ...); it returns
 * LLM_ERR_INVALID past the last class. */
#define LLM_KERNEL_CLASSES 16
int32_t llm_kernel_timing(llm_ctx *c, int32_t enable);
int32_t llm_kernel_time(llm_ctx *c, int32_t kernel, double *total_ms, int64_t *count, const char **name);

/* --------------------------------------------------------------------------
 * Single-kernel entry points, for parity tests of each kernel in isolation.
 * Each is one step of layer.Forward ("Inside the inference engine: model
 * architectures and forward pass", section "Detailed explanation: Llama's
 * forward pass in Go"): the GEMV and GEMM are its linear layers (Q, K, V,
 * output, gate, up, down, the output projection) over a decode step or a
 * prefill ubatch; the attention calls are its ScaledDotProduct over the
 * layer's cache (section "KV Cache: memory for causal attention").
 * All pointers are DEVICE pointers unless stated; all run on `stream`.
 * ------------------------------------------------------------------------*/

/* y[t][n] = sum_k W[n][k] * x[t][k] for t < T <= 8 (the decode GEMV, fp16 x
 * and W, fp32 accumulate).  W fp16 [N][K] (N % 64 == 0, K % 128 == 0); x fp16
 * [T][K]; y fp32 [T][N].  ksplit: number of K slices (K % (128*ksplit) == 0),
 * 0 = library choice.  scratch: fp32 [ksplit][N][8] plus uint32 counters
 * [N/64] (zeroed once before the first use; the kernel leaves them zero). */
int32_t llm_op_gemv(const void *W, const void *x, float *y, int32_t N, int32_t K, int32_t T,
                    int32_t ksplit, void *scratch, int64_t scratch_bytes, void *stream);

/* The bounded wait of the pipelined kernels on its own, to check its time-out
 * path: one thread initialises a shared-memory mbarrier for one arrival,
 * arrives on it when `arrive` is nonzero, and polls its phase at most `polls`
 * times (polls >= 1).  A wait that never completes ORs 4 (the time-out bit of
 * the kernels' error word) into the DEVICE word *err and returns; the device
 * stays usable.  No step of the forward pass runs it. */
int32_t llm_op_wait_check(int32_t arrive, int32_t polls, uint32_t *err, void *stream);

/* Q8_0 encoding (the blocks of llm_model_quantize) of the fp16 matrix W
 * [N][K], K a multiple of 256, into out: N rows of K + K/16 bytes, each the
 * K int8 codes in element order followed by the K/32 fp16 block scales.  W is
 * only read.  LLM_ERR_INVALID for a null pointer, N < 1 or a K that is not a
 * positive multiple of 256. */
int32_t llm_op_quantize_q8_0(const void *W, int32_t N, int32_t K, void *out, void *stream);

/* y[n] = sum over blocks b of d[n][b] * sum over k in b of q[n][k] * x[k]:
 * the one-row decode GEMV streamed from Q8_0 rows (as written by
 * llm_op_quantize_q8_0), fp32 products and sums; x fp16 [K] (16-byte
 * aligned), y fp32 [N].  LLM_ERR_INVALID when the streamed GEMV has no plan
 * for (N, K) on this GPU: K must be a multiple of 256, and every multiple of
 * 2048 up to 16384 has one. */
int32_t llm_op_gemv_q8_0(const void *Wq, const void *x, float *y, int32_t N, int32_t K, void *stream);

/* C[m][n] = sum_k A[m][k] * W[n][k] (the prefill GEMM), A fp16 [M][K], W fp16
 * [N][K], C fp32 [M][N]; M >= 1, N % 128 == 0, K % 64 == 0.  kernel: 0 = the
 * schedule the forward pass uses (tcgen05 on CTA pairs, 256-row tiles:
 * stream-K when N % 256 == 0, else width and persistence chosen by the
 * library); 1 / 2 / 3 = CTA pairs with tiles 128 / 192 / 256 wide, one tile
 * a pair; 4 / 5 / 6 = the same widths on persistent CTA pairs; 7 = stream-K
 * (N % 256 == 0; its partial slots are allocated and freed on `stream`).  A
 * width that does not divide N gives LLM_ERR_INVALID. */
int32_t llm_op_gemm(const void *A, const void *W, float *C, int32_t M, int32_t N, int32_t K,
                    int32_t kernel, void *stream);

/* Decode attention (flash-decoding): for each row t < T <= 8 and query head h,
 * o[t][h] = softmax_c(q[t][h] . K[c] / sqrt(hd)) V[c] over cache positions
 * c <= pos[t] of sequence seq[t].  q fp32 [T][H*hd]; caches fp16
 * [n_seq][Hkv][n_ctx][hd] (one layer); pos, seq int32 [T]; o fp16 [T][H*hd].
 * head_dim 32, 64 or 128; H/Hkv 1, 2, 4 or 8; n_split: sequence splits per
 * (row, kv head), 1..128; each split covers whole 64-key tiles, so short
 * sequences use fewer.  Shapes outside these return LLM_ERR_INVALID (reason
 * in llm_last_error(NULL)) before anything is enqueued.
 * scratch: llm_op_attn_decode_scratch_bytes bytes (split partials, counters,
 * an error word; caller-owned, contents need not be initialised).  The call
 * waits for the kernel: a row whose pos lies outside [0, n_ctx) or whose seq
 * lies outside [0, n_seq) is skipped (its output is zero) and the call
 * returns LLM_ERR_COMPUTE, saying so in llm_last_error(NULL). */
int64_t llm_op_attn_decode_scratch_bytes(int32_t T, int32_t H, int32_t hd, int32_t n_split);
int32_t llm_op_attn_decode(const float *q, const void *k_cache, const void *v_cache,
                           const int32_t *pos, const int32_t *seq, void *o, int32_t T,
                           int32_t H, int32_t Hkv, int32_t hd, int32_t n_ctx, int32_t n_seq,
                           int32_t n_split, void *scratch, int64_t scratch_bytes, void *stream);

/* Prefill attention: rows r < T of q fp16 [T][H*hd] belong to sequence seq[r]
 * at position pos[r]; each row attends to its sequence's cache positions
 * c <= pos[r].  Rows of one sequence must be consecutive with consecutive
 * positions.  Caches as above (one layer, n_seq sequences).  o fp16
 * [T][H*hd].  pos, seq are HOST arrays (the tile list is built on the host):
 * a position outside [0, n_ctx), a sequence outside [0, n_seq) or a gap in
 * a sequence's positions returns LLM_ERR_INVALID before anything is
 * enqueued.  The kernel is the tcgen05 one on CTA pairs where it applies
 * (head_dim 128, an even H / Hkv), else the forward pass's default for the
 * shape.  The call waits for the kernel. */
int32_t llm_op_attn_prefill(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *pos, const int32_t *seq, void *o, int32_t T,
                            int32_t H, int32_t Hkv, int32_t hd, int32_t n_ctx, int32_t n_seq,
                            void *stream);

/* The sampling chain of llm_sample on arbitrary rows: logits fp32
 * [n_rows][n_vocab], u fp32 [n_rows], history int32 [n_history] and out int32
 * [n_rows] are DEVICE pointers; n_vocab is a multiple of 4, at most 262144,
 * and logits is 16-byte aligned (rows are read as float4), else
 * LLM_ERR_INVALID. */
int32_t llm_op_sample(const float *logits, int32_t n_rows, int32_t n_vocab, const llm_sampling *s,
                      const float *u, const int32_t *history, int32_t n_history, int32_t *out,
                      void *stream);

/* Decode attention exactly as llm_op_attn_decode (same arguments but the
 * scratch, same kernel, same result), for callers that cannot allocate
 * device memory: a host framework whose caching allocator owns all device
 * memory, a fixed-footprint serving process, or a latency-critical loop that
 * must never enter the driver's allocator (cudaMalloc can synchronize the
 * device).  It calls no allocation routine.  Its split scratch is one
 * file-scope device array of 1048576 floats of partials plus 512 counters and
 * an error word (4 MiB + 2 KiB), which every GPU that loads this library
 * holds until the process exits.  Limits: T*H*n_split*(hd+2) <= 1048576 and
 * T*Hkv <= 512; larger requests return LLM_ERR_INVALID and
 * llm_last_error(NULL) says why.  The first call on each device looks up the
 * array's device address (with that device current), so make that first call
 * before any stream capture.  All calls share the one array: calls that
 * overlap on the GPU (other streams, other threads) race and corrupt each
 * other's results, so serialize them.  Each call clears the counters and the
 * error word on `stream` before launching, and waits for the kernel as
 * llm_op_attn_decode does.  No step of the forward pass needs it: this entry
 * point exists only for such callers, and the pages have no counterpart. */
int32_t llm_op_attn_decode_noalloc(const float *q, const void *k_cache, const void *v_cache,
                                   const int32_t *pos, const int32_t *seq, void *o, int32_t T,
                                   int32_t H, int32_t Hkv, int32_t hd, int32_t n_ctx, int32_t n_seq,
                                   int32_t n_split, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* LLM_H */
