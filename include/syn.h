/*
 * syn.h -- C ABI of libsyn: the per-token forward of a GGUF decoder described by an .archdef text,
 * on one GB300 GPU (sm_103a).
 *
 * The model is a text file plus weights ("Local inference and architectures", synsema.dev,
 * section "Why an architecture is a file here"): the operations are compiled into this library,
 * the order and parameters come from the .archdef text handed to syn_create, and the weights are
 * loaded by their GGUF tensor names. The lifecycle follows "Execution contract" (cyber.page):
 * load -> forward (token by token, or in bulk) -> reset_kv_cache -> drop, with structured errors.
 *
 * Conventions shared by every call:
 *   - Every call returns a syn_status and never aborts; SYN_OK is 0. After an error,
 *     syn_last_error(model) gives a one-line message that names the file and line, tensor, op or
 *     byte count involved ("Execution contract", section "Error semantics").
 *   - Pointers marked "host" are read or written synchronously within the call. Pointers marked
 *     "device" must be CUDA device (or managed) memory of the model's GPU. Sizes are in elements
 *     unless a name ends in "bytes".
 *   - A model is not thread-safe: one thread at a time, and one forward at a time per model (the
 *     KV cache is per model; concurrent forwards on one cache race, "Execution contract",
 *     section "Concurrency"). The kernel launchers also keep process-wide caches (function
 *     attributes, occupancy per shared-memory size), so calls on different models must not
 *     overlap in time either: serialise them when several host threads drive models.
 *   - All device work is issued on the stream given to syn_create (or one the library creates).
 *     Calls that return host data synchronise that stream.
 */
#ifndef SYN_H
#define SYN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct syn_model syn_model; /* opaque; created by syn_create, freed by syn_destroy */
typedef struct syn_kv syn_kv;       /* opaque; one conversation's KV cache on a model (syn_kv_create) */

/* Status codes. The first eight mirror the ExecutionError kinds of "Execution contract", section
 * "Error semantics"; the rest cover archdef parsing ("Local inference and architectures", section
 * "Errors"), the KV cache bound, CUDA failures and calls made in the wrong state. */
typedef enum {
    SYN_OK = 0,
    SYN_E_UNSUPPORTED_OP = 1,  /* an op or operand form this library does not implement */
    SYN_E_SHAPE_MISMATCH = 2,  /* a tensor or register has the wrong shape for its op */
    SYN_E_MISSING_TENSOR = 3,  /* a tensor named by the archdef was never loaded */
    SYN_E_WEIGHT_FORMAT = 4,   /* dtype / byte count of a loaded tensor does not match its shape */
    SYN_E_OOM = 5,             /* device allocation failed (message gives the requested bytes) */
    SYN_E_BACKEND_INIT = 6,    /* no usable CUDA device, or not an sm_103 device */
    SYN_E_INVALID_CONFIG = 7,  /* missing or invalid GGUF metadata */
    SYN_E_ARCHDEF = 8,         /* the archdef text does not parse or validate */
    SYN_E_CONTEXT_FULL = 9,    /* pos + n would exceed the KV cache's max_ctx */
    SYN_E_CUDA = 10,           /* a CUDA runtime call failed */
    SYN_E_STATE = 11,          /* call not allowed now (before finalize, pos != KV length, ...) */
    SYN_E_INVALID_ARG = 12     /* NULL pointer, negative size, unknown option ... */
} syn_status;

/* GGUF tensor type ids (ggml_type) accepted by syn_load_weights. */
typedef enum { SYN_F32 = 0, SYN_F16 = 1, SYN_Q4_0 = 2, SYN_Q8_0 = 8 } syn_dtype;

/* Flags of syn_forward. */
#define SYN_TOKENS_ON_DEVICE 1u /* `tokens` points to device memory */
#define SYN_LOGITS_ON_DEVICE 2u /* `logits` points to device memory */
#define SYN_ARGMAX_ON_DEVICE 4u /* `argmax_out` points to device memory */

/* Per-forward timing breakdown ("Execution contract", section "Observability"), milliseconds,
 * measured with CUDA events on the model's stream. */
typedef struct {
    double load_ms;        /* syn_create .. end of syn_finalize (host wall clock) */
    double last_prefill_ms;/* device time of the last forward with n > 1 */
    double last_step_ms;   /* device time of the last forward with n == 1 (0 when timing is off) */
    int64_t n_forward;     /* forwards since create */
    int64_t n_launches;    /* kernels launched by the last forward (graph nodes when replayed) */
    int64_t pool_bytes;    /* bytes held by the activation frame pool */
    int64_t kv_bytes;      /* bytes of the KV cache */
    int64_t weight_bytes;  /* bytes of weights resident on the device */
} syn_timings;

/*
 * Check an .archdef text without creating a model (host only, no GPU needed).
 *   file_arch : the file's base name (<arch>.archdef); must equal the text's `arch` line, or NULL.
 *   text/len  : the definition (host).
 *   steps_per_layer (host, nullable): receives the number of op lines in the `block` section.
 *   err/errlen (host, nullable): receives "file: line N: message" on failure.
 * Returns SYN_OK or SYN_E_ARCHDEF. Unknown ops (including every control-flow or I/O word) are
 * rejected ("Local inference and architectures", sections "No control flow, and that is the
 * security property" and "Errors"); a misspelt operation, section header, param key or value, or
 * register gets the nearest known word as a suggestion when it is within two edits.
 */
syn_status syn_archdef_check(const char *file_arch, const char *text, size_t len, int *steps_per_layer,
                             char *err, size_t errlen);

/*
 * sha256 of a definition text (host; text may be NULL when len is 0): 64 lower-case hex digits and
 * a NUL into hex65. The identity the pages print for every definition in effect ("Local inference
 * and architectures", section "What is in effect right now": two runs with the same sha ran the
 * same architecture). Needs no GPU.
 */
syn_status syn_archdef_sha256(const char *text, size_t len, char *hex65);

/*
 * One status line of a model (host out, NUL-terminated, space-separated key=value pairs; the same
 * section of the pages): arch, file, steps_per_layer, prologue_steps, epilogue_steps, sha256 (of
 * the definition text handed to syn_create), layers, hidden, heads, kv_heads, head_dim, max_ctx,
 * kv (cache element type); after syn_finalize also vocab, weights (tensor count per storage type),
 * tied (1 when the logits use token_embd.weight), fused (1 if the fusion pass rewrote anything) and
 * kernels_per_step; always the bulk-prefill configuration: bulk_matmul (tc or cuda_core),
 * bulk_attention (tc or ring) and tc_planes (off, auto, on, or the bytes of resident planes once
 * built). SYN_E_INVALID_ARG if len is too small (the message gives the size needed).
 */
syn_status syn_describe(syn_model *m, char *buf, size_t len);

/*
 * Create a model: parse and validate the archdef, read the metadata and bind the CUDA device that
 * is current on the calling thread.
 *   file_arch : archdef file base name, or NULL (then the text's `arch` line is taken as is).
 *   text/len  : the archdef text (host).
 *   metadata  : GGUF metadata as "key=value\n" lines (host, NUL-terminated), e.g.
 *               "llama.embedding_length=4096\n". Keys read: <arch>.block_count, embedding_length,
 *               attention.head_count, attention.head_count_kv, attention.key_length (optional,
 *               default embedding_length/head_count), attention.layer_norm_rms_epsilon,
 *               rope.freq_base, attention.sliding_window (optional).
 *   max_ctx   : KV cache capacity in positions (> 0); the cache is allocated by syn_finalize.
 *   cuda_stream : cudaStream_t to issue work on; it must not be the legacy default stream (decode
 *               steps are captured into a CUDA graph). NULL: the library creates a non-blocking
 *               stream of its own.
 *   out (host): receives the model. On failure *out is still set (so syn_last_error can explain)
 *               unless the failure was an allocation of the model object itself; free it with
 *               syn_destroy either way.
 * Errors, in the order they are checked (the definition and the metadata before any device call):
 * SYN_E_INVALID_ARG (NULL out, text or metadata); SYN_E_ARCHDEF (the definition, with its line,
 * including a `scale` factor that is neither a finite number nor a metadata key);
 * SYN_E_INVALID_CONFIG (a required key missing; a value that is empty, not a 32-bit integer or not
 * a finite number; non-positive block_count, embedding_length or max_ctx; head_count not a
 * multiple of head_count_kv; a negative epsilon or window; a non-positive rope base);
 * SYN_E_UNSUPPORTED_OP (head_dim other than 64, 128, 256, or more than 8 query heads per KV head,
 * 4 with head_dim 256); SYN_E_BACKEND_INIT (no CUDA device, or not sm_103); SYN_E_CUDA.
 */
syn_status syn_create(const char *file_arch, const char *text, size_t len, const char *metadata,
                      int max_ctx, void *cuda_stream, syn_model **out);

/*
 * Load one tensor by its GGUF name ("Local inference and architectures", section "The format":
 * definitions name tensors exactly as the GGUF does).
 *   dtype      : SYN_F32, SYN_F16, SYN_Q8_0 or SYN_Q4_0 for matrices; SYN_F32 or SYN_F16 for
 *                vectors (norm weights, biases), which are kept as f32.
 *   ne/n_dims  : GGUF shape (host), ne[0] the contiguous in-feature axis; 1 <= n_dims <= 2; each
 *                dimension at most 2^31 - 1 (the kernels index with 32-bit integers).
 *   host_bytes : the tensor in GGUF storage format (host); nbytes must match the shape exactly.
 * The bytes are copied (and re-laid out for the kernels) before the call returns; the caller keeps
 * ownership of its buffer. Loading a name twice replaces the tensor. Only allowed before
 * syn_finalize.
 * Errors: SYN_E_INVALID_ARG (NULL name, shape or bytes), SYN_E_WEIGHT_FORMAT (byte count, dtype,
 * dimension count or size, block alignment), SYN_E_OOM, SYN_E_CUDA (upload), SYN_E_STATE.
 */
syn_status syn_load_weights(syn_model *m, const char *gguf_name, syn_dtype dtype, const int64_t *ne,
                            int n_dims, const void *host_bytes, size_t nbytes);

/*
 * Finish loading ("Execution contract", section "Load phase"): check that every tensor the archdef
 * names is present (resolving `a | b` alternatives, "Local inference and architectures", section
 * "Rules"), infer register shapes, allocate the KV cache sized to max_ctx, build the RoPE cos/sin
 * cache (max_ctx x head_dim/2) and run the load-time fusion pass ("Execution contract", section
 * "Fused op policy").
 * Errors: SYN_E_MISSING_TENSOR, SYN_E_SHAPE_MISMATCH, SYN_E_OOM, SYN_E_UNSUPPORTED_OP, SYN_E_CUDA,
 * SYN_E_STATE (called twice).
 */
syn_status syn_finalize(syn_model *m);

/* Empty the KV cache ("Execution contract", section "Memory lifecycle / KV cache"): the next
 * forward starts at position 0. SYN_E_STATE before syn_finalize. */
syn_status syn_reset_kv(syn_model *m);

/*
 * One forward over n tokens at absolute positions pos .. pos+n-1 ("Execution contract", section
 * "Forward phase"): n == 1 is a decode (or token-by-token prefill) step; n > 1 is bulk prefill,
 * whose result must equal n single steps within tolerance. The K and V of the n positions are
 * appended to the cache.
 *   tokens     : n token ids (host, or device with SYN_TOKENS_ON_DEVICE).
 *   pos        : must equal the number of positions in the cache (SYN_E_STATE otherwise);
 *                pos + n must not exceed max_ctx (SYN_E_CONTEXT_FULL).
 *   logits     : nullable; receives the vocab-size logits of the last position (host, or device
 *                with SYN_LOGITS_ON_DEVICE; caller-owned).
 *   argmax_out : nullable; receives the index of the largest logit, lowest index on ties (host,
 *                or device with SYN_ARGMAX_ON_DEVICE).
 * With device outputs the call returns without waiting for the GPU.
 * Errors: SYN_E_STATE (before syn_finalize, or pos != KV length), SYN_E_CONTEXT_FULL,
 * SYN_E_INVALID_ARG (n < 1, NULL tokens, a host token id outside [0, vocab)), SYN_E_CUDA. Faults the
 * kernels detect themselves (a device-resident token id outside the vocabulary: SYN_E_INVALID_ARG; a
 * bounded wait that gave up: SYN_E_CUDA) stay recorded on the device and are reported by the first
 * forward, this one or a later one, that returns host logits or a host argmax; the results of the
 * forwards since then are invalid.
 */
syn_status syn_forward(syn_model *m, const int32_t *tokens, int n, int pos, float *logits,
                       int32_t *argmax_out, unsigned flags);

/* Device pointer to the model's own logits buffer (valid until the next forward). */
syn_status syn_logits_device(syn_model *m, const float **ptr, int *n_vocab);

/* Timing and memory counters (host out). */
syn_status syn_get_timings(syn_model *m, syn_timings *out);

/*
 * Options (before or after finalize):
 *   "fusion"  1 (default) / 0: load-time fusion pass on or off (takes effect at finalize for
 *             decode, at the next bulk forward for prefill; bulk plans take the patterns that hold
 *             for many rows: shared-input matmuls with their biases, matmul + residual, act * mul
 *             in one pass, the per-head transforms in one kernel).
 *   "graph"   1 (default) / 0: replay decode steps from a captured CUDA graph.
 *   "timing"  0 (default) / 1: time every forward with CUDA events (syncs the stream).
 *   "splits"  >0: split count of the decode attention kernel; 0 (default): the largest power of two
 *             (at most 64) with KV heads x rows x splits <= the SM count.
 *   "profile" 0 (default) / 1: accumulate per-kind device time (see syn_get_profile); forwards
 *             then run without graph replay.
 *   "tc"      1 (default) / 0: run the matmuls of bulk prefill (n > 1 rows) on the tensor cores
 *             (three f16 products of scaled hi/lo splits, f32 sums); 0 = CUDA-core f32 GEMM.
 *             Takes effect at the next bulk forward. Shapes the tensor-core path does not take
 *             (in-features not a multiple of 8) use the CUDA-core GEMM either way.
 *   "tc_planes" -1 (default) / 1 / 0: keep the f16 hi/lo operand planes of every matmul weight of
 *             the block resident in device memory (4 bytes per weight, converted once; info key
 *             "tc_plane_bytes"), so that bulk forwards skip that conversion. -1: built at the first
 *             bulk forward when they take at most half of the free device memory then (decode-only
 *             use never holds them); 1: always, built at once if the model is finalized (SYN_E_OOM
 *             if they do not fit); 0: convert per bulk forward (frees them). Same results bit for bit.
 *   "attn_tc" 1 (default) / 0: run the attention of bulk prefill on the tensor cores (S = Q K^T
 *             and O = P V as three f16 products of scaled hi/lo splits each, softmax in f32);
 *             0 = the CUDA-core kernel, one CTA per query row. Takes effect at the next bulk
 *             forward; head sizes other than 64 and 128 use the CUDA-core kernel either way.
 */
syn_status syn_set_option(syn_model *m, const char *key, int64_t value);

/*
 * Per-kind device-time breakdown of the forwards run while option "profile" was 1 (those forwards
 * run eagerly, with a CUDA event pair around every kernel group; "Execution contract", section
 * "Observability"). Writes NUL-terminated lines "kind launches total_ms algorithmic_bytes flops\n" into
 * buf (host, len bytes; SYN_E_INVALID_ARG if too small). reset != 0 clears the counters afterwards.
 * Each line ends with a fifth field, the arithmetic (flops, f32-equivalent) of the bulk matmuls
 * and of the tensor-core prefill attention of that kind.
 * Kinds: gemv, gemm, gemm_tc, attention, attention_tc, heads, embed, rmsnorm, eltwise, copy, argmax.
 */
syn_status syn_get_profile(syn_model *m, char *buf, size_t len, int reset);

/* Model facts: "n_vocab", "n_embd", "n_layer", "n_head", "n_head_kv", "head_dim", "max_ctx",
 * "kv_len", "steps_per_layer", "n_plan_nodes" (kernels per decode step), "fused" (1 if the fusion
 * pass rewrote anything), "tc_plane_bytes" (device bytes
 * of the resident tensor-core operand planes, 0 if none), "kv_f16" (1 if the cache holds f16).
 * Unknown keys: SYN_E_INVALID_ARG. */
syn_status syn_get_info(syn_model *m, const char *key, int64_t *value);

/*
 * Test support: write positions [pos0, pos0+n) of one layer's cache (host k, v laid out
 * [n_head_kv][n][head_dim] f32). pos0 must not exceed the current KV length; the KV length becomes
 * max(current, pos0 + n). Used to stand in for a long prompt.
 */
syn_status syn_debug_write_kv(syn_model *m, int layer, int pos0, int n, const float *k, const float *v);

/* Test support: read positions [pos0, pos0+n) of one layer's cache into host k, v. */
syn_status syn_debug_read_kv(syn_model *m, int layer, int pos0, int n, float *k, float *v);

/*
 * Test support: read a register after the last forward (host out, the first `count` floats of the
 * register: its last row after `last`, the only row in decode; count <= register width). Names as
 * in the archdef ("x", "logits", ...). Registers that the fusion pass folded away are not
 * materialised (SYN_E_STATE). When the fusion pass folded an in-place `x = rms_norm(x, w)` into the
 * matmuls that read x next (the decode epilogue: norm, last, logits), x keeps the values it had
 * before that norm, i.e. the residual after the last block.
 */
syn_status syn_debug_read_register(syn_model *m, const char *name, float *out, int count);

/*
 * Test support: dequantise rows [row0, row0+nrows) of a loaded matrix on the device with the same
 * device code the kernels use, into host out (nrows x ne[0] f32).
 */
syn_status syn_debug_dequant(syn_model *m, const char *gguf_name, int row0, int nrows, float *out);

/*
 * Decode attention for callers that cannot allocate device memory (the pages have no counterpart:
 * this is an addition of this library). One query row at absolute position n_ctx - 1 attends over
 * the keys [lo, n_ctx) of a cache, lo = 0, or n_ctx - window when window > 0, exactly as the
 * attention inside syn_forward does, split over `splits` key slices.
 *   q       : device, n_head * head_dim floats (post-rope query of one position).
 *   k_cache, v_cache : device, [n_head_kv][max_ctx][head_dim] floats, 16-byte aligned (else
 *             SYN_E_INVALID_ARG: rows are streamed with bulk copies); rows < n_ctx are read.
 *   out     : device, n_head * head_dim floats (caller-owned).
 *   cuda_stream : stream to run on (NULL = legacy default stream).
 * The call allocates nothing: its scratch lives in a fixed 4 MiB device array inside the library,
 * present on every GPU that loads it until the process exits. Limits: head_dim 64, 128 or 256;
 * n_head a multiple of n_head_kv with at most 8 query heads per KV head (4 with head_dim 256);
 * n_head_kv <= 1024; 1 <= splits <= 64; splits * n_head * (head_dim + 4) * 4 bytes <= 4 MiB - 4352.
 * Larger sizes return SYN_E_INVALID_ARG (SYN_E_UNSUPPORTED_OP for a head layout the kernel lacks).
 * The first call on each device looks up the array's address; make that first call before any
 * stream capture. All calls share the array, which keeps the previous call's contents (the call
 * clears what must start at zero): calls that overlap on the GPU, from any stream or thread, race
 * and must be serialised by the caller. Returns after enqueueing; the result is ready when the
 * stream reaches it. The kernel's waits on its own bulk copies are bounded: a wait that gives up
 * leaves `out` invalid and sets an error word in the array, which SYN_OK from this call cannot
 * report (it returns before the GPU runs). syn_attention_static_status reports it.
 */
syn_status syn_attention_static(const float *q, const float *k_cache, const float *v_cache, int n_head,
                                int n_head_kv, int head_dim, int max_ctx, int n_ctx, int window, int splits,
                                float *out, void *cuda_stream);

/*
 * Outcome of the syn_attention_static calls on the current device since the last status call:
 * waits for cuda_stream (NULL = legacy default stream) to finish, then reads the array's sticky
 * error word and clears it. SYN_OK: no bounded wait gave up, and every `out` those calls wrote is
 * valid. SYN_E_CUDA: a wait gave up (or a CUDA call failed here), and the outputs of those calls
 * are invalid. Allocates nothing. Like the calls themselves, it must not overlap another call on
 * the same device.
 */
syn_status syn_attention_static_status(void *cuda_stream);

/*
 * Test support: the number of polls after which the bounded waits of syn_attention_static give up
 * (process-wide). polls < 0 restores the default bound (2^24 polls); 0 makes every such wait give
 * up at once, so that the error path (the kernel records the error, waits with the full bound for
 * its bulk copies still in flight, and returns) is exercised without a fault or a hang.
 */
void syn_debug_set_spin_limit(int polls);

/*
 * Several conversations on one loaded model ("Execution contract", section "Concurrency / Multiple
 * conversations": each conversation has its own KV cache, the weights are shared). syn_kv_create (after syn_finalize)
 * allocates a second cache of the same size and element type as the model's, with its own
 * position record and, once used, its own captured decode plan. syn_kv_select makes a handle the
 * model's current conversation (NULL: the model's own cache); from then on syn_forward,
 * syn_reset_kv, syn_debug_write_kv / syn_debug_read_kv and syn_get_info("kv_len") act on it, and
 * the positions of each conversation are independent. Forwards of different conversations run
 * one after another on the model's stream (the activation pool is shared); running two at once
 * is a caller error, as for one model. syn_kv_destroy frees a handle (selecting the model's own
 * cache first if it was current); handles left at syn_destroy lose their device memory there and
 * still need syn_kv_destroy to free the host object.
 */
syn_status syn_kv_create(syn_model *m, syn_kv **out);
syn_status syn_kv_select(syn_model *m, syn_kv *kv);
void syn_kv_destroy(syn_kv *kv);

/* The message of the last failed call on this model (never NULL). */
const char *syn_last_error(const syn_model *m);

/* Free everything the model holds. NULL-safe; a model must be destroyed exactly once
 * ("Execution contract", section "Shutdown"). */
void syn_destroy(syn_model *m);

#ifdef __cplusplus
}
#endif
#endif /* SYN_H */
