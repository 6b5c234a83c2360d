/*
 * laneformer.h — C ABI of the GB300 (sm_103a) batch-1 decode engine for the
 * lane-structured decoder with Delayed Tensor Parallelism.
 *
 * The problem these calls serve is the one the pages describe: a single
 * request decoded one token at a time at batch 1, greedy, in FP16, within a
 * 4096-token context ("Kog Laneformer 2B generates 3000 tokens per second
 * thanks to delayed tensor parallelism", section "Performance and
 * infrastructure"; "Kog Laneformer 2B: the latency-first model behind Kog
 * Inference Engine", sections "TL;DR" and "Designing the architecture").
 *
 * Conventions for every call:
 *  - Plain C types only; pointers are HOST pointers unless a name says
 *    "device".  The engine owns all device memory it allocates; the caller
 *    keeps ownership of every buffer it passes.
 *  - Every call returns an lf_status.  After LF_ERR_CUDA, LF_ERR_TIMEOUT or
 *    LF_ERR_BOUNDS (or a bad token found on the device by a chained step,
 *    reported as LF_ERR_INVALID_ARG) the engine is poisoned: every call but lf_reset and
 *    lf_destroy returns that status again until lf_reset succeeds.
 *  - Calls run on the engine stream (default: the legacy stream, or the one
 *    given to lf_set_stream) and are synchronous unless stated otherwise.
 *  - One engine per thread; there is no internal locking.
 */
#ifndef LANEFORMER_H
#define LANEFORMER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LF_MAX_LAYERS 64

typedef enum {
    LF_OK = 0,
    LF_ERR_INVALID_ARG = 1,   /* bad pointer, size, token id or config value */
    LF_ERR_OOM = 2,           /* device or host allocation failed */
    LF_ERR_CUDA = 3,          /* a CUDA call failed (no device, launch error, ...) */
    LF_ERR_NOT_LOADED = 4,    /* decode or prefill before lf_load_weights */
    LF_ERR_CTX_OVERFLOW = 5,  /* the position would reach ctx_cap */
    LF_ERR_TIMEOUT = 6,       /* a bounded device-side wait ran out */
    LF_ERR_UNSUPPORTED = 7,   /* a valid config this build has no kernel for */
    LF_ERR_BOUNDS = 8         /* debug build only: a device-side bounds check or a
                                 canary around an engine buffer failed */
} lf_status;

/*
 * Model shape and run options.  The lane structure follows "Kog Laneformer
 * 2B: the latency-first model behind Kog Inference Engine", section
 * "Designing the architecture": n_lanes lanes, each owning an equal, contiguous
 * block of query heads (and the KV heads those read, q head h reading KV head
 * h / (n_q_heads / n_kv_heads)) and an equal block of FFN units.
 *
 * Delayed lane sum: sub-block s (2l = attention, 2l+1 = FFN of layer l) reads
 * the residual e + sum_{u <= s-1-2*dtp_delay} sum_lanes P[u], where P[u] is the
 * row-parallel o_proj / down_proj output of sub-block u; every pending partial
 * is added before the final norm.  dtp_delay = 0 is ordinary per-layer
 * tensor-parallel synchronisation.  (Sections "Hiding overhead" of the blog
 * and "Architectural decisions" of the news page fix only that the
 * synchronisation is delayed by 2 layers; this exact form is the reading this
 * library implements by default.)  own_lane_immediate = 1 selects the other
 * reading: lane i's residual also holds its own partials P_i[u] of sub-blocks
 * s-2d <= u <= s-1 at once (the lane's own output is local to it), the other
 * lanes' share arriving 2*dtp_delay sub-blocks later; with dtp_delay = 0 the
 * two readings are the same function.  The own-lane reading runs each lane's
 * sub-blocks in dependency order with a lane-local sum after every one.
 */
typedef struct {
    int n_layers, d_model, n_q_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    int n_lanes;             /* lanes = SM groups of one GPU; divides n_q_heads and ffn_dim */
    int dtp_delay;           /* >= 0, in layers */
    int ctx_cap;             /* maximum context (positions 0 .. ctx_cap-1) */
    float rms_eps, rope_theta;
    int swa_window[LF_MAX_LAYERS]; /* per layer: keys j > p - W; 0 = full causal */
    int own_lane_immediate;  /* 0: delayed sum as above; 1: each lane adds its own partial at once */
} lf_config;

typedef struct lf_engine lf_engine;

/* Host-only check of a config (no GPU needed).  LF_ERR_INVALID_ARG for values
 * that define no model, LF_ERR_UNSUPPORTED for shapes without a kernel
 * (built: d_model 4096 with head_dim 128, d_model 256 with head_dim 32). */
lf_status lf_validate_config(const lf_config *cfg);

/* Creates an engine on the current CUDA device: validates the config, plans
 * the lane -> SM mapping for the device's SM count and allocates the KV cache,
 * the delayed-sum buffers, the logits and the weight stream.  *out is NULL on
 * failure. */
lf_status lf_create(const lf_config *cfg, lf_engine **out);

/* Copies an FP16 weight blob (nbytes = 2 * number of parameters; tensor order
 * E, per layer [g_attn, Wq, Wk, Wv, Wo, g_ffn, Wg, Wu, Wd], g_f, W_lm; each
 * matrix row-major [out][in]) to the device and repacks it into the per-SM
 * streaming layout.  The caller keeps the blob.  Resets the position to 0. */
lf_status lf_load_weights(lf_engine *e, const void *host_blob, size_t nbytes);

/* Fills KV-cache slots [0, n_pos) of every layer from a host FP16 array in
 * layout [layer][K|V][pos][kv_head][head_dim] (nbytes must match) and sets the
 * position to n_pos.  Used to start decoding from a given cache. */
lf_status lf_load_kv(lf_engine *e, const void *host_kv, size_t nbytes, int n_pos);

/* Decodes n tokens one after another from the current position (prefill by
 * sequential decode steps, which equals a causal prefill exactly).  logits
 * (vocab floats, nullable) and argmax (nullable) receive the result of the
 * last token.  LF_ERR_CTX_OVERFLOW if position + n > ctx_cap (nothing run). */
lf_status lf_prefill(lf_engine *e, const int32_t *tokens, int n, float *logits, int32_t *argmax);

/* One decode step of `token` at the current position; advances the position.
 * logits: host array of vocab floats or NULL; argmax: host int32 or NULL
 * (lowest index among equal maxima).  When both are NULL the step is only
 * enqueued on the engine stream and the call returns without waiting; its
 * results stay on the device (lf_get_logits_device, lf_get_argmax_device) and
 * a device-side error surfaces at the next synchronising call. */
lf_status lf_decode_step(lf_engine *e, int32_t token, float *logits, int32_t *argmax);

/* Greedy generation with no host round trip between steps: the per-request
 * token rate at batch 1 that News (asector), "Performance and
 * infrastructure", quotes, decoded greedily as in its "Training and data
 * specialisation" section.  Runs n >= 1 decode steps from the current
 * position: step 0 reads `first_token`, step i > 0 reads the argmax of step
 * i - 1 straight from device memory.  All n steps run in one launch of the
 * persistent kernel: each SM's weight copies run on into step i + 1 while
 * step i drains its last lane sums and its LM head, and step i + 1 embeds
 * step i's argmax as soon as it is published.  The results are those of n
 * lf_decode_step calls.  tokens_out (host, n int32, required) receives the n
 * argmax tokens; logits (host, vocab floats, nullable) those of the last
 * step.  Advances the position by n.  Synchronous.
 * LF_ERR_INVALID_ARG for n < 1, a NULL tokens_out or first_token outside
 * [0, vocab); LF_ERR_CTX_OVERFLOW if position + n > ctx_cap (nothing run). */
lf_status lf_generate(lf_engine *e, int32_t first_token, int n, int32_t *tokens_out, float *logits);

/* Completion time of each of the first n steps of the last lf_generate call
 * (the device's global timer, ns, taken when the step's argmax is
 * published) into ns (host, n uint64).  Differences give per-token latency.
 * LF_ERR_INVALID_ARG if n exceeds that call's step count. */
lf_status lf_generate_stamps(lf_engine *e, uint64_t *ns, int n);

/* Stochastic decoding for pass@N (News (asector), "Performance and
 * infrastructure": several sampled solutions per prompt are affordable
 * because one pass is fast; the pages name no method, this is temperature +
 * nucleus sampling): like lf_generate, but each step's token is drawn from
 * its logits instead of taken as the argmax.  p_i = exp((z_i - max z) / T);
 * the kept set is every token whose p_i is at least tau, the largest p value
 * for which the tokens at or above it hold at least top_p of the total mass;
 * u = (x0 >> 8) / 2^24 with x0 the first word of Philox4x32-10 (Salmon et
 * al., SC 2011) for key (seed low 32 bits, seed high 32 bits) and counter
 * (position of the step, sample, 0, 0); the token is the first kept index
 * whose running kept mass exceeds u times the kept mass.  Different `sample`
 * values give independent streams, so N samples from the same prompt state
 * are N calls that each start at the prompt's end (lf_set_position).
 * temperature == 0 is greedy.  tokens_out (host, n int32) receives the n
 * sampled tokens, logits (host, nullable) the last step's logits.
 * LF_ERR_INVALID_ARG for n < 1, NULL tokens_out, first_token outside
 * [0, vocab), temperature < 0 or top_p outside (0, 1]; LF_ERR_CTX_OVERFLOW if
 * position + n > ctx_cap; LF_ERR_UNSUPPORTED for a vocabulary above 51200. */
lf_status lf_generate_sampled(lf_engine *e, int32_t first_token, int n, float temperature, float top_p,
                              uint64_t seed, uint32_t sample, int32_t *tokens_out, float *logits);

/* The draw of lf_generate_sampled on its own: *token_device = sample of the
 * vocab fp32 logits at logits_device (both DEVICE pointers), enqueued on
 * cuda_stream (NULL = legacy stream) without waiting.  Same definition and
 * error statuses as lf_generate_sampled. */
lf_status lf_sample(const float *logits_device, int vocab, float temperature, float top_p, uint64_t seed,
                    uint32_t position, uint32_t sample, int32_t *token_device, void *cuda_stream);

/* One chained decode step, the building block of lf_generate: enqueued on the
 * engine stream without waiting; its input token is read on the device from
 * *token_device when the step starts (e.g. the previous step's argmax) and
 * its argmax is written to *argmax_device.  Both must be 4-byte aligned words
 * the GPU can access (device memory of the engine's device, managed or
 * registered host memory), else LF_ERR_INVALID_ARG; they may be the same word.
 * A token outside [0, vocab) found on the device is read as 0 and the next
 * synchronising call returns LF_ERR_INVALID_ARG (engine poisoned until
 * lf_reset).  LF_ERR_CTX_OVERFLOW at position == ctx_cap. */
lf_status lf_decode_step_chained(lf_engine *e, const int32_t *token_device, int32_t *argmax_device);

/* Waits for the engine stream and reports a device-side error, if any. */
lf_status lf_synchronize(lf_engine *e);

/* Position control.  lf_set_position accepts 0 <= pos <= ctx_cap; cache slots
 * below pos keep whatever they hold. */
lf_status lf_set_position(lf_engine *e, int pos);
lf_status lf_get_position(const lf_engine *e, int *pos);

/* Sets the position to 0 and clears the device synchronisation state; also
 * the way out of a poisoned engine. */
lf_status lf_reset(lf_engine *e);

void lf_destroy(lf_engine *e);
const char *lf_status_string(lf_status s);

/* Uses `cuda_stream` (a cudaStream_t owned by the caller, e.g. PyTorch's) for
 * every later call; NULL selects the legacy default stream. */
lf_status lf_set_stream(lf_engine *e, void *cuda_stream);

/* Device pointers to the logits (vocab fp32) and argmax (int32) of the last
 * step run through the engine's own buffers (lf_decode_step, lf_prefill,
 * lf_prefill_batched, the generation calls); valid until lf_destroy.  A
 * lf_decode_step_static_scratch step writes only the caller's buffers and
 * leaves these as they were. */
lf_status lf_get_logits_device(lf_engine *e, const float **dptr);
lf_status lf_get_argmax_device(lf_engine *e, const int32_t **dptr);

/* Reads the cached K and V (head_dim values each, as fp32) of `layer`,
 * global KV head `kv_head` and position `pos` (copy held by the first lane
 * that reads that head). */
lf_status lf_read_kv(lf_engine *e, int layer, int kv_head, int pos, float *k, float *v);

/* Limit of every device-side wait, in nanoseconds (default 2e9).  A wait that
 * runs out makes the step fail with LF_ERR_TIMEOUT instead of hanging. */
lf_status lf_set_timeout_ns(lf_engine *e, uint64_t ns);

/* Tuning: how far (bytes per SM, multiples of 16) each SM's weight stream is
 * prefetched into L2 beyond its shared-memory stages, so that HBM keeps
 * streaming while the SM does latency-bound work.  bytes_per_sm applies to the
 * layers (default 128 KiB), lm_bytes_per_sm to the LM-head rows, which are
 * reached while the step drains its last lane sums (default 128 KiB).  0 turns
 * a prefetch off. */
lf_status lf_set_l2_prefetch(lf_engine *e, uint32_t bytes_per_sm, uint32_t lm_bytes_per_sm);

/* Tuning: when an SM's weight copies have waited after_ns for a free stage
 * (its consumers are held up, e.g. by the last lane sums before the LM head),
 * the SM prefetches further rows of its stream into L2, 32 KiB at a time,
 * until it is bytes_per_sm (a multiple of 16) ahead of its copies; HBM then
 * works during the wait (default 768 KiB after 4000 ns).  0 bytes turns it
 * off. */
lf_status lf_set_idle_prefetch(lf_engine *e, uint32_t bytes_per_sm, uint32_t after_ns);

/* Test hook: in the next decode step, CTA `cta` skips its first lane-barrier
 * arrival (-1 = off), so that the lane's other CTAs time out.  Proves that the
 * step ends with LF_ERR_TIMEOUT rather than a hang. */
lf_status lf_debug_skip_arrival(lf_engine *e, int cta);

/* Tracing: with enable != 0 every later step records, per CTA and per op of
 * the step's op list, LF_TRACE_WORDS words (global timer ns; the buffer is
 * allocated on first use):
 *   [0] start, [1] end, [2] ns blocked on cross-CTA counters, [3] ns blocked
 *   on tile arrival (streaming warps; attention warps for ATTN ops),
 *   [4] ns the weight-copy warp waited for a free stage while issuing this
 *   op's rows, [5] time of its first copy for this op (0 = op has no rows);
 *   for an ATTN op [4] and [5] are the ns the attention warps spent in the
 *   score and in the P.V phases.
 * The slot of a lane-sum op (REDUCE) holds, on the CTAs that sum a chunk
 * (cta < d_model / 32), [wait start, publish time, ns waiting for the
 * partials, ns copying them, 0, 0]; it stays zero on the other CTAs.
 * A launch of several steps (lf_generate) leaves its
 * last step's record: every step rewrites the same slots as its ops end.
 * lf_debug_read_trace copies the last step's record: n_words must equal
 * n_sm * n_ops * LF_TRACE_WORDS (lf_engine_info [0] and [6]); `ops`
 * (nullable, n_ops entries) receives the op list, each entry
 * type | (argument << 8). */
#define LF_TRACE_WORDS 6
lf_status lf_debug_trace(lf_engine *e, int enable);
lf_status lf_debug_read_trace(lf_engine *e, uint64_t *out, size_t n_words, int32_t *ops);

/*
 * Decode step that allocates nothing.  The pages have no counterpart to this
 * call: it exists for callers that may not call the CUDA allocator while they
 * decode, e.g. a host that gives the library a fixed device-memory budget up
 * front and accounts for every byte itself, or a latency-bound serving loop
 * for which a cudaMalloc (which may synchronise the whole device and stall
 * its other streams) is not acceptable.  Such a caller creates and loads the
 * engine beforehand and passes its own output buffers here.
 *
 * Same step as lf_decode_step (same kernel, same results, advances the
 * position, appends to the engine's KV cache), but the step's working memory
 * (lane-sum partials and sums, q/k/v and attention partials, counters, argmax
 * candidates, error word) comes from one fixed device array inside the
 * library, LF_STATIC_SCRATCH_BYTES long, that every GPU which loads this part
 * of the library keeps until the process exits.  The call makes no
 * cudaMalloc, cudaFree or other allocating call.
 *   logits_device: DEVICE array of vocab floats, written by the step.
 *   argmax_device: DEVICE int32, written by the step.
 * Both must be 4-byte aligned and reachable from the engine's device: device
 * memory of that device (for logits, an allocation with room for vocab
 * floats from the pointer on) or managed / mapped host memory; anything else
 * (a plain host pointer, memory of another device) is LF_ERR_INVALID_ARG.
 * The results go only to these buffers: lf_get_logits_device and
 * lf_get_argmax_device keep pointing at the last lf_decode_step's results.
 * The engine's device must be the current device.  The first call on a
 * device looks up the array's device address (once per device); make that
 * first call before any stream capture.  Every call uses the same array and
 * finds in it what the previous call left; the call clears the parts that
 * must start at zero itself.  Calls whose work overlaps on the GPU (on other
 * streams, or from other engines on the same device) race on the array: issue
 * them one after another.  Synchronous: waits for the step and reports a
 * device-side timeout.  Returns LF_ERR_UNSUPPORTED when the engine's working
 * set does not fit the array (the full 2.3B lane model needs about 26 MB on
 * 152 SMs) or the config asks for the own-lane-immediate reading,
 * LF_ERR_INVALID_ARG for outputs that fail the checks above or another
 * current device,
 * and the same statuses as lf_decode_step otherwise.
 */
#define LF_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)
lf_status lf_decode_step_static_scratch(lf_engine *e, int32_t token, float *logits_device,
                                        int32_t *argmax_device);

/* Prefill of n tokens from the current position in one batched pass: the
 * same function as lf_prefill (each position's logits depend only on the
 * positions before it, Blog, "Designing the architecture": causal GQA with
 * sliding windows; the lane sums delayed as in "Hiding overhead"), computed
 * sub-block by sub-block over all n positions at once, with the projections
 * as tensor-core GEMMs (lf_matmul_f16) against the FP16 weights in file
 * layout, which the engine keeps on the device from lf_load_weights on.
 * Because every lane's residual copy is the same vector under the delayed
 * sum, sub-block s of every position reads e + the projection outputs of
 * sub-blocks u <= s - 1 - 2d.  Appends all n positions to the KV cache,
 * advances the position by n; logits (host, vocab floats, nullable) and
 * argmax (host, nullable) receive the last position's result, which also
 * stays on the device (lf_get_logits_device / lf_get_argmax_device).
 * Scratch is allocated on first use and kept (about 0.18 MB per position
 * at full shape, delay 2, plus a transposed copy of the V caches, the size
 * of the V cache, for the tensor-core attention), and so are a second
 * stream and events: consecutive sub-blocks, which the delayed sum leaves
 * independent, run on the engine's stream and that one, which the engine's
 * stream waits for before the call returns.  Synchronous.  LF_ERR_INVALID_ARG for n < 1, a
 * NULL tokens array or a token outside [0, vocab); LF_ERR_CTX_OVERFLOW if
 * position + n > ctx_cap; LF_ERR_OOM when the resident weights or the
 * scratch could not be allocated; LF_ERR_TIMEOUT if a GEMM's device-side
 * wait ran out (engine poisoned). */
lf_status lf_prefill_batched(lf_engine *e, const int32_t *tokens, int n, float *logits, int32_t *argmax);

/* Which attention lf_prefill_batched uses: tensor_cores = 1 (default) runs
 * S = Q K^T and O = P V as tcgen05 MMAs (head_dim 128; other head sizes use
 * the CUDA-core kernel anyway), 0 the CUDA-core kernel.  Same function up to
 * rounding (P and q are FP16 operands on the tensor-core path).
 * LF_ERR_INVALID_ARG for other values. */
lf_status lf_set_prefill_attention(lf_engine *e, int tensor_cores);

/* Tensor-core matrix product of the batched prefill (lf_prefill_batched),
 * exported for tests and for callers that build their own batched passes:
 * c[m][n] = sum_k a[m][k] * b[n][k], with a (m x k) and b (n x k) row-major
 * FP16 DEVICE arrays (16-byte aligned) and c an m x n row-major fp32 DEVICE
 * array, i.e. activations times a weight matrix in its [out][in] layout, the
 * projection shape of every layer (Blog, "Designing the architecture": a
 * standard decoder).  k must be a multiple of 64; m, n >= 1.  Runs on
 * `cuda_stream` (NULL = legacy stream) and waits for it.  LF_ERR_INVALID_ARG
 * for bad sizes, NULL or misaligned pointers; LF_ERR_TIMEOUT if a
 * device-side wait ran out; LF_ERR_CUDA on a CUDA error. */
lf_status lf_matmul_f16(const void *a_device, const void *b_device, float *c_device, int m, int n, int k,
                        void *cuda_stream);

/* c[m][n] = c_in[m][n] + sum_k a[m][k] * b[n][k]: the product of
 * lf_matmul_f16 added to c_in (fp32 DEVICE array of c's shape, row-major)
 * as it leaves the accumulator, the residual update that follows every
 * attention and FFN block (Blog, "Designing the architecture": a standard
 * decoder; the batched prefill adds each block's output to the residual that
 * way).  Each element is c_in + the fp32 product in one rounding; c_in may
 * be c itself (added in place); c_in and c otherwise must not overlap.
 * Sizes and alignment as lf_matmul_f16, and c_in and c have the same
 * address modulo 16 bytes.  Synchronous on `cuda_stream`; errors as
 * lf_matmul_f16. */
lf_status lf_matmul_add_f16(const void *a_device, const void *b_device, const float *c_in_device, float *c_device,
                            int m, int n, int k, void *cuda_stream);

/* The same product, only enqueued on `cuda_stream` (no wait, no status read
 * back): for callers that chain several products, and for timing the kernel
 * alone.  *err_device (device word, 4-byte aligned, cleared by the caller)
 * becomes non-zero if a device-side wait ran out.  LF_ERR_INVALID_ARG for bad
 * sizes or pointers, LF_ERR_CUDA if the launch failed. */
lf_status lf_matmul_f16_async(const void *a_device, const void *b_device, float *c_device, int m, int n, int k,
                              uint32_t *err_device, void *cuda_stream);

/* Batched decode for pass@N (News, "Performance and infrastructure":
 * several sampled solutions per prompt): n_batch samples (1..16) continue
 * the engine's current sequence together, one position per step, each with
 * its own KV cache, so every weight byte streamed from HBM serves all of
 * them.  Each sample computes the forward of lf_decode_step under the
 * delayed lane sum (own_lane_immediate = 0; with 1 it is LF_ERR_UNSUPPORTED)
 * with FP16 activations into tensor-core GEMVs, fp32 accumulation.
 *
 * lf_batch_begin copies positions [0, position) of the engine's KV cache
 * into every sample's cache and sets the batch position to the engine's
 * position; the engine's own sequence is untouched by the batch calls.  The
 * batch state (about B * 4 * L * n_kv * ctx_cap * head_dim bytes of caches)
 * is owned by the engine until lf_batch_end, lf_batch_begin or lf_destroy.
 * LF_ERR_INVALID_ARG for n_batch outside 1..16; LF_ERR_NOT_LOADED before
 * lf_load_weights; LF_ERR_CTX_OVERFLOW at position == ctx_cap;
 * LF_ERR_UNSUPPORTED for shapes the batched kernels do not take (d_model,
 * n_q_heads * head_dim or ffn_dim not a multiple of 64, 128 not a multiple
 * of head_dim, more than 8 query heads per KV head); LF_ERR_OOM. */
lf_status lf_batch_begin(lf_engine *e, int n_batch);
lf_status lf_batch_end(lf_engine *e);
/* *n_batch and *position of the current batch (0 and 0 when there is none). */
lf_status lf_batch_info(const lf_engine *e, int *n_batch, int *position);

/* One step of every sample: tokens (host, n_batch int32, required) at the
 * batch position; logits (host, n_batch x vocab fp32, nullable) and argmax
 * (host, n_batch int32, lowest index among equal maxima, nullable) per
 * sample.  Synchronous; advances the batch position by one.
 * LF_ERR_NOT_LOADED without lf_batch_begin; LF_ERR_INVALID_ARG for a token
 * outside [0, vocab); LF_ERR_CTX_OVERFLOW at position == ctx_cap;
 * LF_ERR_TIMEOUT / LF_ERR_CUDA poison the engine (and end the batch). */
lf_status lf_batch_step(lf_engine *e, const int32_t *tokens, float *logits, int32_t *argmax);

/* n_steps sampled steps of every sample, the draw of lf_generate_sampled:
 * sample b draws with counter (position of the step, b), so sample b of a
 * batch makes the same draws as lf_generate_sampled(..., sample = b) on the
 * same logits.  first_tokens (host, n_batch int32) are the inputs of the
 * first step; tokens_out (host, n_batch x n_steps int32, row b = sample b)
 * receives the drawn tokens.  temperature 0 is greedy.  Synchronous;
 * advances the batch position by n_steps.  Errors as lf_batch_step, plus
 * LF_ERR_INVALID_ARG for temperature < 0 or top_p outside (0, 1] and
 * LF_ERR_UNSUPPORTED for a vocabulary above 51200. */
lf_status lf_batch_generate(lf_engine *e, const int32_t *first_tokens, int n_steps, float temperature, float top_p,
                            uint64_t seed, int32_t *tokens_out);

/* The tensor-core GEMV of the batched decode, exported for tests:
 * y[b][r] = sum_k w[r][k] * x[b][k] for b < batch (1..16), r < n, with w
 * (n x k) and x (batch x k) row-major FP16 DEVICE arrays (16-byte aligned)
 * and y a batch x n row-major fp32 DEVICE array; k a multiple of 64.  The
 * weights are streamed once; the reduction is split over the SMs and summed
 * in a fixed order (deterministic).  Allocates its scratch per call; runs on
 * `cuda_stream` (NULL = legacy stream) and waits for it.  LF_ERR_INVALID_ARG
 * for bad sizes or pointers; LF_ERR_TIMEOUT if a device-side wait ran out. */
lf_status lf_gemv_f16(const void *w_device, const void *x_device, float *y_device, int n, int k, int batch,
                      void *cuda_stream);

/*
 * Debug build.  liblaneformer_debug.so is the same library compiled with
 * LF_DEBUG: before every weight-tile, KV, q/k/v, partial, lane-sum,
 * attention-partial and logit access the decode kernel checks the index
 * against its buffer; a failed check skips the access, records the site
 * and the index in the step's error word and the step returns
 * LF_ERR_BOUNDS (no trap, the context stays usable).  Every buffer the
 * engine allocates at create and load time sits between two 256-byte canary
 * regions, which the host checks after every step that reports a status
 * (lf_decode_step with outputs, lf_synchronize, lf_prefill, the generation
 * calls): an overwritten canary poisons the engine with LF_ERR_BOUNDS.
 *
 * lf_debug_canaries checks every canary now (synchronously) and writes the
 * number of guarded buffers to *n_guarded (nullable): LF_OK, or
 * LF_ERR_BOUNDS for an overwritten canary.  lf_debug_corrupt_canary writes
 * one word into the front (back = 0) or back canary of guarded buffer i,
 * from the host, so that a test can see the check fire.  Both return
 * LF_ERR_UNSUPPORTED in the release library.
 */
lf_status lf_debug_canaries(lf_engine *e, int *n_guarded);
lf_status lf_debug_corrupt_canary(lf_engine *e, int i, int back);

/* Measurement call, not a step of the decode: one read of `bytes` of device
 * memory at `src_device` in the decode kernel's weight-copy pattern (one CTA
 * per SM, each reading one contiguous range with 32 KB bulk copies into a
 * ring of four shared-memory stages, evict-first), with no arithmetic on the
 * data.  Its duration is the read-only ceiling of the decode step's weight
 * stream (the step is bound by reading its weights once: Blog, "Designing
 * the architecture").  `bytes` a multiple of 32768, src_device 16-byte
 * aligned; sink_device receives one checksum float per SM (sink_len >= the
 * SM count); *status_device (4-byte aligned device word, left as it is on
 * success) is set to 1 if a device-side wait ran out.  Asynchronous on
 * `cuda_stream` (NULL = legacy stream); returns LF_ERR_INVALID_ARG for bad
 * arguments, LF_ERR_CUDA if the launch failed. */
lf_status lf_stream_read(const void *src_device, size_t bytes, float *sink_device, int sink_len,
                         uint32_t *status_device, void *cuda_stream);

/* Host-only plan statistics for `n_sm` SMs (no GPU needed): stats[0] = weight
 * rows in the stream, [1] = min rows per SM, [2] = max rows per SM, [3] = ops
 * per step, [4] = 1 if every weight row of every lane appears exactly once,
 * [5] = SMs per lane (smallest), [6] = SMs per lane (largest). */
lf_status lf_plan_stats(const lf_config *cfg, int n_sm, int64_t stats[8]);

/* Engine facts: [0] SMs used, [1] weight-stream bytes, [2] device bytes
 * allocated, [3] smem bytes per CTA, [4] threads per CTA, [5] kernel launches
 * made since creation, [6] ops per step. */
lf_status lf_engine_info(const lf_engine *e, int64_t info[8]);

#ifdef __cplusplus
}
#endif
#endif /* LANEFORMER_H */
