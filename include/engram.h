/*
 * engram.h -- C ABI of the Engram conditional-memory layer forward on one
 * GB300 GPU (sm_103a).
 *
 * The layer is the one printed in the code excerpts of atlas.klimoza.dev
 * "deepseek-v4.1 / engram-second" (classes `Engram` and
 * `ParallelEngramEmbedding`).  For each token it
 *   1. reads n_cols ids, each a global row of the table (ids outside [0, R)
 *      give a zero row, as the single-rank case of the sharded embedding does);
 *   2. dequantises each row: fp8-e4m3 code widened to fp32, times the fp32 scale
 *      of its scale_block-channel block (one fp32 rounding), cast to bf16;
 *   3. flattens the rows to K = n_cols*head_dim values (element c*head_dim + f);
 *   4. projects through wkv to N = dim*(hc_mult+1) values, fp32 accumulation,
 *      bf16 result: hc_mult per-stream keys, then one shared value;
 *   5. per (token, stream): rstd = rsqrt(mean h^2 + eps) * rsqrt(mean key^2 + eps),
 *      dot = sum(h * q_weight*k_weight * key) * rstd * dim^-0.5,
 *      gate = sigmoid(copysign(sqrt(max(|dot|, clamp)), dot)), 0 where the
 *      token mask is False;
 *   6. out = bf16(h + gate * value) for every stream; a masked token's streams
 *      are returned bit-for-bit (the excerpt's docstring leaves them as they are).
 * The split into lookup+projection and gating follows zhuai.tech "Engram in
 * DeepSeek V4.1 Flash" (section "Run projection early: overlap CPU work with
 * the GPU"): the lookup and projection depend only on the ids and may run
 * ahead; only the gating needs the hidden state.
 *
 * Conventions for every call
 *  - Pointers named as device pointers must be device (or managed) memory of
 *    the current device; the caller owns them and keeps them alive until the
 *    work queued on `stream` has finished.  The context never frees them.
 *  - bf16 and fp8 values are passed as their bit patterns (uint16_t, uint8_t).
 *  - Row-major layouts, no padding: hash_ids [M, n_cols] int64; x and out
 *    [M, hc_mult, dim]; kv [M, dim*(hc_mult+1)]; rows [M, n_cols*head_dim];
 *    token_mask [M] uint8 (non-zero = the layer applies) or NULL (all apply);
 *    M = B*T tokens.
 *  - Work is queued on `stream` (NULL = the legacy default stream) and runs
 *    asynchronously.  Argument errors are returned at once and queue nothing.
 *    Errors the device detects (ids out of range when check_ids is set, a
 *    pipeline wait that ran out of time) are recorded in the context and
 *    returned by engram_sync_status().
 *  - 16-byte alignment is required for x, out, kv, rows and the table; 8 bytes
 *    for hash_ids and the scales.
 *  - A context is not thread-safe: calls on one context must be serialised by
 *    the caller, and calls on one context must not overlap on the GPU (they
 *    share the context's scratch); use one stream per context.
 */
#ifndef ENGRAM_H
#define ENGRAM_H

#include <stdint.h>

/* Symbols of the shared library (it is built with hidden default visibility). */
#if defined(__GNUC__)
#define ENGRAM_API __attribute__((visibility("default")))
#else
#define ENGRAM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* engram_stream_t;

typedef enum {
  ENGRAM_OK = 0,
  ENGRAM_EINVAL = -1,        /* bad argument: null pointer, size, alignment */
  ENGRAM_ENOMEM = -2,        /* device or host allocation failed (create only) */
  ENGRAM_ECUDA = -3,         /* a CUDA runtime call or kernel launch failed */
  ENGRAM_ERANGE = -4,        /* check_ids: some id was outside [0, num_rows) */
  ENGRAM_ETIMEOUT = -5,      /* a kernel's bounded wait ran out; its output is invalid */
  ENGRAM_EUNSUPPORTED = -6   /* shape or format this build does not implement */
} engram_status;

typedef enum {
  ENGRAM_SCALE_F32 = 0,      /* one fp32 scale per scale_block channels */
  ENGRAM_SCALE_E8M0 = 1      /* one E8M0 byte (2^(e-127)) per scale_block channels */
} engram_scale_fmt;

/* Format of the projection weight wkv.  The V4.1 tables and projections are
 * FP8 (monishver11.github.io "DeepSeek's Other Modules", section "V4.1's two
 * tables, reconciled"); the tables' format is MXFP8, E4M3 codes with one E8M0
 * scale per 32 values (zhuai.tech "Engram in DeepSeek V4.1 Flash", section
 * "Step 2").  ENGRAM_WKV_MXFP8 reads the weight in the same format along its
 * input dimension:  W[j, k] = e4m3(wkv[j, k]) * 2^(wkv_scale[j, k/32] - 127).
 * It requires an MXFP8 table (scale_fmt = ENGRAM_SCALE_E8M0, scale_block = 32):
 * the projection then multiplies the table's codes and the weight's codes on
 * the block-scaled FP8 tensor-core path, each with its own scales, with fp32
 * accumulation; kv is rounded to bf16 as in the bf16 path. */
typedef enum {
  ENGRAM_WKV_BF16 = 0,       /* wkv: bf16 [N, K] */
  ENGRAM_WKV_MXFP8 = 1       /* wkv: e4m3 codes [N, K]; wkv_scale: E8M0 [N, K/32] */
} engram_wkv_fmt;

typedef struct {
  int32_t dim;          /* per-stream hidden size (5120 in V4.1); multiple of 256, <= 5120 */
  int32_t hc_mult;      /* residual streams (4 in V4.1); 1..4 */
  int32_t n_cols;       /* ids per token: (max_ngram_size-1)*n_heads (24 in V4.1) */
  int32_t head_dim;     /* channels per table row (256 in V4.1); multiple of 16 */
  int32_t scale_block;  /* channels per scale; divides head_dim, multiple of 16 */
  int32_t scale_fmt;    /* engram_scale_fmt */
  int64_t num_rows;     /* R: rows of the table */
  float eps;            /* added to both mean squares (the V4.1 config's norm_eps is 1e-20) */
  float clamp;          /* lower clamp of |dot| before the square root (1e-6 in V4.1) */
  int32_t max_tokens;   /* largest B*T of any later call; sizes the scratch */
  int32_t check_ids;    /* non-zero: count ids outside [0, R) and report ENGRAM_ERANGE */
  int32_t fuse_gate;    /* where engram_forward forms the gate and the residual add when the
                           projection runs without split-K: 1 = in the projection's epilogue
                           (kv never reaches HBM), -1 = in a separate kernel that reads kv,
                           0 = the library chooses by batch size (the way that measured
                           faster on GB300: the epilogue of the CTA-pair projection from
                           1,024 tokens on, when all SMs are the projection's; the separate
                           kernel otherwise).  Same bits either way, and the same as
                           engram_lookup_project + engram_gate_apply: a batch that takes the
                           fused epilogue keeps whole tiles in its plan (no remainder split,
                           see engram_plan), so that both ways sum kv alike.  The fused
                           projection takes its tiles from a work counter, in an order where
                           an M tile's key tiles come well before its value tiles, whose
                           epilogues wait (bounded) for the gates the key tiles form: only
                           running CTAs take tiles, so the wait never depends on a CTA that
                           has not started, whatever else shares the GPU.  On CTA pairs the
                           epilogue warps stage x in shared memory by tensor copies and write
                           the output by tensor stores. */
  int32_t wkv_fmt;      /* engram_wkv_fmt; ENGRAM_WKV_MXFP8 needs K a multiple of 128 and
                           takes no fused epilogue (fuse_gate is ignored) */
  int64_t row_offset;   /* global id of the table's first row, >= 0: the table holds rows
                           [row_offset, row_offset + num_rows) of the whole table, one shard of
                           a table split by rows over several GPUs, as `ParallelEngramEmbedding`
                           splits it (atlas.klimoza.dev "deepseek-v4.1 / engram-second": rank r
                           owns rows [r*P, r*P + P), P = ceil(R / world_size)); 0 for a whole
                           table.  An id outside the shard gives a zero row (and is counted by
                           check_ids), so the shards' gathered rows, summed over the ranks, are
                           the whole table's rows: see engram_forward_rows() */
} engram_config;

/* table and scale may live in device memory or in host memory that the device
 * reads in place: pinned host memory (cudaHostAlloc, or cudaHostRegister with
 * cudaHostRegisterMapped) whose device address equals its host address, as it
 * does under unified addressing.  A host-resident table is gathered by the
 * same kernel, its rows crossing the host link on every call (NVLink-C2C on a
 * Grace-Blackwell node): the pages keep the tables in host memory.  engram_create
 * returns ENGRAM_EINVAL for a table or scale pointer the device cannot read at
 * that address (unregistered host memory, another device's memory), and so it
 * does for wkv, wkv_scale, q_weight and k_weight; engram_forward_noalloc()
 * makes the same checks on every call. */
typedef struct {
  const uint8_t* table;     /* device or mapped pinned host, [R, head_dim] fp8-e4m3 codes */
  const void* scale;        /* device or mapped pinned host, [R, head_dim/scale_block]
                               fp32 or uint8 E8M0 */
  const void* wkv;          /* device, [dim*(hc_mult+1), n_cols*head_dim], the Linear's
                               [out, in] weight: keys of stream s at rows s*dim ..
                               s*dim+dim-1, the value at rows hc_mult*dim ..; bf16 bits
                               (uint16_t), or e4m3 codes (uint8_t) for ENGRAM_WKV_MXFP8 */
  const uint16_t* q_weight; /* device, [hc_mult, dim] bf16 */
  const uint16_t* k_weight; /* device, [hc_mult, dim] bf16 */
  const uint8_t* wkv_scale; /* device, [dim*(hc_mult+1), n_cols*head_dim/32] E8M0 for
                               ENGRAM_WKV_MXFP8; ignored (may be NULL) for bf16 */
} engram_weights;

typedef struct engram_ctx engram_ctx;

/* Validates the configuration, allocates the context's scratch on the current
 * device (sized by max_tokens), forms the fp32 product q_weight*k_weight
 * (used only as a product, per the `Engram` excerpt) and copies wkv into a
 * buffer of its own (N*K*2 bytes for bf16, N*K + N*K/32 for MXFP8) in 32 KB
 * tiles of 256 rows x 128 bytes, each stored as the projection's shared-memory
 * stage holds it, so that every weight read of a forward call is one
 * contiguous 32 KB stream.  The table and scales are referenced, not copied,
 * and must outlive the context; wkv, wkv_scale, q_weight and k_weight are read
 * only here (a changed weight needs a new context).  Synchronous.
 * Returns ENGRAM_EINVAL / ENGRAM_EUNSUPPORTED for bad or unsupported shapes,
 * ENGRAM_ENOMEM if the scratch cannot be allocated, ENGRAM_ECUDA otherwise. */
ENGRAM_API engram_status engram_create(engram_ctx** out, const engram_config* cfg, const engram_weights* w);

/* Frees the context's scratch (synchronises the device first).  NULL is a no-op. */
ENGRAM_API void engram_destroy(engram_ctx* ctx);

/* The whole layer (`Engram.forward` with token_mask): out = layer(x).  out may
 * equal x (in place); otherwise the two must not overlap.  hash_ids, x,
 * token_mask and out are device pointers.  B*T must not exceed max_tokens;
 * B*T == 0 queues nothing. */
ENGRAM_API engram_status engram_forward(engram_ctx* ctx, const int64_t* hash_ids, const uint16_t* x,
                             const uint8_t* token_mask, uint16_t* out, int64_t B, int64_t T,
                             engram_stream_t stream);

/* Steps 1-4 only (independent of the hidden state, so they can run ahead on a
 * side stream): writes kv [B*T, dim*(hc_mult+1)] bf16 to the device buffer kv.
 * engram_gate_apply() on this kv gives bit-for-bit the result of
 * engram_forward(). */
ENGRAM_API engram_status engram_lookup_project(engram_ctx* ctx, const int64_t* hash_ids, uint16_t* kv,
                                    int64_t B, int64_t T, engram_stream_t stream);

/* Steps 5-6 on a kv produced by engram_lookup_project (or by the caller):
 * out = layer(x) given kv.  gates (device, [B*T, hc_mult] fp32, 0 on masked
 * tokens) is written when non-NULL.  out may equal x. */
ENGRAM_API engram_status engram_gate_apply(engram_ctx* ctx, const uint16_t* kv, const uint16_t* x,
                                const uint8_t* token_mask, uint16_t* out, float* gates,
                                int64_t B, int64_t T, engram_stream_t stream);

/* Steps 1-3 only: the gathered, dequantised rows, [B*T, n_cols*head_dim] bf16,
 * written to the device buffer rows (the `ParallelEngramEmbedding` output,
 * flattened; on a shard context, before its all-reduce: zero rows for ids
 * outside the shard). */
ENGRAM_API engram_status engram_lookup(engram_ctx* ctx, const int64_t* hash_ids, uint16_t* rows,
                            int64_t B, int64_t T, engram_stream_t stream);

/* Steps 4-6 on gathered rows the caller provides: rows [B*T, n_cols*head_dim]
 * bf16 (device), as engram_lookup() writes them, -> out = layer(x).  This is
 * the second half of the row-sharded layer: each GPU gathers the rows of its
 * shard with engram_lookup() (zero rows for ids outside it), the GPUs sum the
 * rows over the ranks -- the one exchange of the sharded layer, the
 * `dist.all_reduce` of `ParallelEngramEmbedding.forward` (atlas.klimoza.dev
 * "deepseek-v4.1 / engram-second"); exactly one rank holds each row, so a sum
 * of the bit patterns as integers reproduces the rows bit for bit -- and each
 * GPU then calls engram_forward_rows() on the summed rows.  On rows from
 * engram_lookup() of the whole table the result equals engram_forward() bit
 * for bit.  out may equal x.  Takes the bf16 weight only (ENGRAM_EUNSUPPORTED
 * for ENGRAM_WKV_MXFP8, whose projection reads the table's codes).  rows must
 * not be written until the call's work on `stream` has finished. */
ENGRAM_API engram_status engram_forward_rows(engram_ctx* ctx, const uint16_t* rows, const uint16_t* x,
                                             const uint8_t* token_mask, uint16_t* out, int64_t B, int64_t T,
                                             engram_stream_t stream);

/* Waits for `stream`, then returns and clears the device-detected error
 * recorded by earlier calls on this context: ENGRAM_ERANGE (with check_ids),
 * ENGRAM_ETIMEOUT, or ENGRAM_OK.  *bad_ids (may be NULL) receives the number of
 * out-of-range ids counted since the last call. */
ENGRAM_API engram_status engram_sync_status(engram_ctx* ctx, engram_stream_t stream, int64_t* bad_ids);

/* Split-K factor and CTA count the projection would use for B*T = m_tokens on
 * this context's device (for tests and benchmarks; queues nothing). */
ENGRAM_API engram_status engram_plan(const engram_ctx* ctx, int64_t m_tokens, int32_t* splits, int32_t* ctas);
/* (Without split-K, when a small number of tiles would fill only part of a
 * last wave of the grid, the plan also cuts those last tiles into 2-4 K ranges
 * whose fp32 sums a small kernel after the projection adds up in range order;
 * this changes kv's summation order for those tiles, not its tolerance.
 * Contexts with max_tokens <= 128, and batches that take the fused gate
 * epilogue, keep whole tiles.) */

/* The projection's whole plan for B*T = m_tokens on this context (queues
 * nothing).  ENGRAM_EINVAL for a NULL context or pointer or a negative count. */
typedef struct {
  int32_t splits;       /* split-K factor (1: every tile over the whole K) */
  int32_t ctas;         /* CTAs of the projection's persistent grid */
  int32_t cta_pairs;    /* 1: tiles of 256 x 256 on pairs of CTAs (tcgen05 cta_group::2, clusters of two),
                           0: tiles of 128 x 256 on single CTAs */
  int32_t rem_tiles;    /* tiles of a partial last wave cut into K ranges (0: none) */
  int32_t rem_splits;   /* the K ranges each of them is cut into */
  int32_t fused_gate;   /* 1: engram_forward forms the gate in the projection's epilogue */
} engram_plan_info;
ENGRAM_API engram_status engram_describe_plan(const engram_ctx* ctx, int64_t m_tokens, engram_plan_info* info);

/* Number of kernels one engram_forward over m_tokens tokens launches on this
 * context (gather, projection, the remainder sums when the plan has them, gate;
 * 2 with the fused gate epilogue; 0 for no tokens).  Queues nothing.
 * ENGRAM_EINVAL for a NULL context or pointer or a negative count. */
ENGRAM_API engram_status engram_forward_kernels(const engram_ctx* ctx, int64_t m_tokens, int32_t* kernels);

/* Caps the number of SMs the projection's persistent grid occupies (and that
 * its split-K plan is made for) at `sms`; 0 or more than the device has
 * restores all of them.  For running lookup_project ahead on a side stream
 * while other kernels use the rest of the GPU.  The plan, and with it the
 * summation order of kv, may change with the budget.  Host-only; affects
 * later calls.  ENGRAM_EINVAL for a NULL context or a negative count. */
ENGRAM_API engram_status engram_set_sm_budget(engram_ctx* ctx, int32_t sms);

/* Failure-detection test hook.  ENGRAM_TEST_HOLD_GATE_FLAGS makes the fused
 * gate epilogue (fuse_gate with a single-pass plan) never raise its
 * gates-ready flags, so that the value tiles' bounded wait runs out: the
 * call's output is then invalid, engram_sync_status() returns
 * ENGRAM_ETIMEOUT, and the context stays usable once the hook is cleared.
 * Nothing faults, traps or hangs; the wait ends after two seconds.  0 clears
 * the hooks.  ENGRAM_EINVAL for a NULL context or unknown bits. */
#define ENGRAM_TEST_HOLD_GATE_FLAGS 1
ENGRAM_API engram_status engram_test_hook(engram_ctx* ctx, int32_t hooks);

/* Stage timing, for benchmarks.  With enable = n > 0 the context creates CUDA
 * events for its last n calls (n <= 4096) and every later engram_forward /
 * engram_lookup_project records one before the gather and one after each of
 * its kernels on the call's stream, cycling through the n sets; enable == 0
 * destroys them (and a new enable starts the count afresh).  Events between
 * the kernels keep them from overlapping, so these are each kernel's own
 * durations.  engram_stage_times() waits for the last recorded event and
 * writes the durations of the last call's stages in milliseconds: ms[0]
 * gather + dequantise, ms[1] projection, ms[2] gate and residual add (the
 * split-K reduction, for lookup_project; ~0 when the gate ran in the
 * projection's epilogue).  engram_stage_times_n() does the same for the last
 * n calls, oldest first, into ms[3 * n]: queued back to back, they time the
 * kernels in the steady state of a run of calls.  ENGRAM_EINVAL for a NULL
 * context or pointer, timing not enabled, or n outside [1, calls timed]
 * (at most the n given to enable). */
ENGRAM_API engram_status engram_enable_stage_timing(engram_ctx* ctx, int32_t enable);
ENGRAM_API engram_status engram_stage_times(engram_ctx* ctx, float* ms);
ENGRAM_API engram_status engram_stage_times_n(engram_ctx* ctx, int32_t n, float* ms);

/* ---- n-gram hash: the step before the layer ----------------------------------
 * The hash `forward` excerpt of atlas.klimoza.dev "deepseek-v4.1 / engram-second"
 * (and monishver11.github.io "DeepSeek's Other Modules", section "The lookup
 * pipeline"): token ids -> the global table rows of every Engram layer.
 *   1. c = token_map[id]; ids outside [0, vocab_size) and positions whose
 *      token_mask is 0 become dead_id (they take part in no n-gram);
 *   2. cache[b, start_pos + l] = c (the session's history of compressed ids);
 *   3. look-back s = 0 .. max_ngram_size-1: the id s positions back; once a
 *      look-back reaches before position 0 or a dead_id, it and every longer
 *      one are pad_id;
 *   4. with 64-bit wrapping products p_s = id_s * multipliers[g, s], the XOR of
 *      p_0 .. p_i hashes the (i+1)-gram;
 *   5. row = hash mod primes[g, i-1, h] (remainder with the divisor's sign) +
 *      offsets[g, (i-1)*n_heads + h].
 * Calls for one session must come in position order; a call may cover any
 * chunk [start_pos, start_pos + L) of it (earlier positions are read from the
 * cache). */
typedef struct {
  int32_t n_layers;        /* Engram layers that share the hash (2 in V4.1) */
  int32_t max_ngram_size;  /* n-grams of 2 .. max_ngram_size tokens (4 in V4.1); 2..8 */
  int32_t n_heads;         /* hash heads per n-gram order (8 in V4.1); 1..32 */
  int32_t max_batch;       /* rows of the session cache */
  int64_t max_len;         /* positions per cache row */
  int64_t vocab_size;      /* entries of token_map */
  int32_t pad_id;          /* id of a blocked look-back (engram_pad_id, 2 in V4.1) */
  int32_t dead_id;         /* id of a position in no n-gram (e.g. -1) */
} engram_hash_config;

/* All pointers are device pointers, caller-owned.  token_map: [vocab_size]
 * int32; multipliers: [n_layers, max_ngram_size] int64; primes: [n_layers,
 * max_ngram_size-1, n_heads] int64 (positive); offsets: [n_layers,
 * (max_ngram_size-1)*n_heads] int64; cache: [max_batch, max_len] int32, the
 * session state (read below start_pos, written at [start_pos, start_pos+L));
 * input_ids: [B, L] int64; token_mask: [B, L] uint8 or NULL; hash_ids:
 * [n_layers, B, L, (max_ngram_size-1)*n_heads] int64 -- hash_ids[g] is the id
 * array of Engram layer g for engram_forward.  B <= max_batch and start_pos + L
 * <= max_len, else ENGRAM_EINVAL; more than 6144 primes (n_layers *
 * (max_ngram_size-1) * n_heads) give ENGRAM_EUNSUPPORTED.  Asynchronous on
 * `stream`. */
ENGRAM_API engram_status engram_hash(const engram_hash_config* cfg, const int32_t* token_map,
                                     const int64_t* multipliers, const int64_t* primes, const int64_t* offsets,
                                     int32_t* cache, const int64_t* input_ids, const uint8_t* token_mask,
                                     int64_t start_pos, int64_t* hash_ids, int64_t B, int64_t L,
                                     engram_stream_t stream);

/* ---- allocation-free variant ------------------------------------------------
 * The pages have no counterpart to this entry point; it exists for callers of
 * this library that cannot allocate device memory.  A serving engine that
 * reserves nearly all of HBM at start-up for its weights and KV cache and hands
 * out every other byte through its own allocator, or a plugin running inside a
 * host process that owns the GPU's memory budget, cannot let a library call
 * cudaMalloc: the allocation may fail or synchronise at a point the caller does
 * not control, and it escapes the caller's accounting.  engram_create() needs
 * such allocations for its scratch; this call does not.
 *
 * engram_forward_noalloc() computes the same layer as engram_forward(), with
 * the same kernels, for at most ENGRAM_NOALLOC_MAX_TOKENS tokens, without a
 * context and without allocating: it calls no cudaMalloc, cudaFree or other
 * allocating routine.  Its scratch (gathered rows, split-K partial sums,
 * q_weight*k_weight, an error word) is one file-scope static __device__ array
 * of ENGRAM_NOALLOC_SCRATCH_BYTES bytes; the CUDA driver places it in device
 * memory when it loads this part of the library on a device, and every device
 * that loads it keeps those bytes until the process exits.
 *  - cfg and w are as for engram_create() (max_tokens, check_ids and
 *    fuse_gate are ignored); the weights are read on every call.  Shapes with
 *    n_cols*head_dim > 6144 or dim*(hc_mult+1) > 25600 give ENGRAM_EUNSUPPORTED.
 *  - B*T > ENGRAM_NOALLOC_MAX_TOKENS gives ENGRAM_EINVAL and queues nothing;
 *    so does a table, scale, wkv, q_weight or k_weight pointer that the
 *    current device cannot read where it is (pageable host memory, another
 *    device's memory).
 *  - The first call on each device looks up the device address of the scratch
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture on the device.  The address is looked up again
 *    when the device's context has changed since (after cudaDeviceReset the
 *    module, and the array with it, is loaded anew); the first call after such
 *    a reset should therefore also come before any stream capture.
 *  - Every call on a device shares the one scratch array, which keeps the last
 *    call's contents; the call clears the part that must start at zero (the
 *    error word) on `stream` before its kernels run.  Calls that overlap on the
 *    GPU (other streams, other threads) race on the scratch: serialise them.
 *  - Errors the device detects are not reported (there is no context to hold
 *    them); every device wait stays bounded. */
#define ENGRAM_NOALLOC_MAX_TOKENS 64
#define ENGRAM_NOALLOC_SCRATCH_BYTES 20529408
ENGRAM_API engram_status engram_forward_noalloc(const engram_config* cfg, const engram_weights* w,
                                                const int64_t* hash_ids, const uint16_t* x,
                                                const uint8_t* token_mask, uint16_t* out, int64_t B, int64_t T,
                                                engram_stream_t stream);

/* Static description of a status code. */
ENGRAM_API const char* engram_status_string(engram_status s);

/* ABI version of this library: 100 * major + minor. */
ENGRAM_API int32_t engram_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_H */
