/*
 * verkv.h -- C ABI of libverkv.so: KVFetch verified attention over a
 * PoissonComp-compressed KV cache, on one NVIDIA GB300 (sm_103a).
 *
 * The operations follow "Verify Before You Fetch: Reliable KV Cache
 * Compression for LLM Inference":
 *   verkv_compress  -- PoissonComp, Algorithm 1 (Sec. 4.1, eq. (3)), plus the
 *                      token-level key sketch of Appendix A.1.
 *   verkv_decode    -- KVFetch, Algorithm 2 (Sec. 4.2: Definition 2 / eq. (5),
 *                      Lemma 1 / eq. (7), eqs. (9)-(10), Theorem 2), followed by
 *                      the weighted attention named in the comment closing
 *                      Algorithm 2.
 *
 * Conventions
 *   - Every entry point returns a verkv_status; nothing is thrown across the
 *     ABI.  On any status other than VERKV_OK, verkv_last_error(ctx) holds a
 *     one-line message.  Asynchronous CUDA faults surface as VERKV_ECUDA at
 *     the next call that synchronises.
 *   - "device" pointers are CUDA device (or managed) memory of the GPU that was
 *     current when the context was created; "host" pointers are CPU memory.
 *     "pinned" means page-locked (cudaHostAlloc / cudaHostRegister) memory the
 *     GPU can read over the host link.
 *   - A verkv_stream is a cudaStream_t (NULL = the legacy default stream).
 *     Work is enqueued on that stream; one context is driven from one host
 *     thread at a time and has no internal threads.
 *   - The context owns all device memory it allocates.  Caller buffers are
 *     borrowed for the duration of a call, except `kv_host` of
 *     verkv_compress, which is borrowed until verkv_release of that slot.
 *   - Layouts are row-major.  K/V rows of one token and one KV head are stored
 *     K then V: [n_kv_heads][n][2][head_dim] in the element type `kv_dtype`.
 */
#ifndef VERKV_H
#define VERKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct verkv_ctx verkv_ctx;
typedef void* verkv_stream;

typedef enum {
    VERKV_OK = 0,
    VERKV_EINVAL = 1,        /* bad argument or shape */
    VERKV_ENOMEM = 2,        /* device or pinned allocation failed */
    VERKV_ECUDA = 3,         /* a CUDA call or kernel failed */
    VERKV_ETIMEOUT = 4,      /* a bounded device-side wait gave up */
    VERKV_EUNSUPPORTED = 5,  /* configuration not built (e.g. head_dim != 128) */
    VERKV_ESTATE = 6         /* call out of order (e.g. decode before compress) */
} verkv_status;

typedef enum {
    VERKV_SKETCH_EXACT = 0,  /* the "perfect sketch": sketch weights = exact weights */
    VERKV_SKETCH_INT8 = 1,   /* per-token symmetric int8 keys with an fp32 scale */
    VERKV_SKETCH_2BIT = 2    /* Appendix A.1: d/8 rotate-half channel pairs, 2-bit, fp16 zero/scale per group */
} verkv_sketch;

/* The coefficients lambda_i of the shrinkage estimator. */
typedef enum {
    VERKV_SHRINK_CLIPPED = 0,  /* Definition 2: lambda_i = clip_[r_i,1](beta r_i / (w^_i (1 - r_i))) at the fixed
                                  point beta = sum_L w^_i (1 - lambda_i), the unique MSE minimiser (Theorem 1) */
    VERKV_SHRINK_BINARY = 1    /* Appendix A.2: lambda_i in {1, r_i}; L visited by decreasing
                                  w^_i (1 - r_i) / r_i (ties: lower L index first), each token set to r_i while
                                  that value exceeds twice the bias beta accumulated so far */
} verkv_shrinkage;

typedef enum {
    VERKV_DTYPE_BF16 = 0,
    VERKV_DTYPE_F32 = 1
} verkv_dtype;

typedef struct {
    int32_t n_layers;      /* number of layer slots                                   */
    int32_t n_seqs;        /* number of sequence slots per layer                      */
    int32_t max_batch;     /* largest B passed to verkv_decode                         */
    int32_t n_kv_heads;    /* KV heads                                                */
    int32_t n_q_heads;     /* query heads, a multiple of n_kv_heads (GQA group <= 8)  */
    int32_t head_dim;      /* 128 (the only head dimension built)                     */
    int32_t max_tokens;    /* upper bound on n per slot                               */
    int32_t n_sink;        /* first tokens always kept (forced into H)                */
    int32_t n_local;       /* last tokens always kept (forced into H)                 */
    int32_t sketch_group;  /* 2-bit sketch: tokens per min/max group (128)            */
    int32_t shrinkage;     /* verkv_shrinkage (0 = clipped, Definition 2)            */
    double eta;            /* kept fraction: expected |H u S| = eta * n (Alg. 1)      */
    uint64_t seed;         /* Philox4x32-10 key of the Poisson sample                 */
    verkv_sketch sketch;
    verkv_dtype kv_dtype;  /* element type of K and V                                 */
} verkv_config;

/* Per KV head, filled by verkv_compress (host memory, valid on return). */
typedef struct {
    double c;              /* water-filling constant of eq. (3); +inf if every token is kept */
    int32_t n_capped;      /* tokens outside the sink/local windows with r = 1                */
    int32_t n_h;           /* |H| (r = 1, sink and local included)                           */
    int32_t n_l;           /* |L| (0 < r < 1)                                                 */
    int32_t n_s;           /* |S|, the sampled part of L                                      */
    int32_t n_resident;    /* |H| + |S| rows kept on the GPU                                  */
    int32_t pad;
} verkv_head_stats;

/* Per query row (sequence b, query head h) of the last verkv_decode. */
typedef struct {
    double m;              /* logit shift used for the weights                                */
    double D;              /* certificate denominator: sum_H w_i + sum_L w^_i                  */
    double beta;           /* fixed point of Definition 2 (in units of exp(-m))               */
    double sum_a;          /* beta(L) of eq. (7) = sum_L w^_i (1 - lambda_i)                  */
    double V;              /* V(L) of eq. (7)                                                 */
    double b;              /* b(L) of eq. (7)                                                 */
    double eps_hat;        /* eq. (7) on the whole of L                                       */
    int32_t n_l;           /* |L|                                                             */
    int32_t kstar;         /* eq. (10); 0 when no fetch is needed                              */
    int32_t no_fetch;      /* eps_hat < eps (Algorithm 2, the no-fetch test)                   */
    int32_t fallback;      /* k* was beyond the on-chip candidate width: full-row path used   */
    int32_t n_fetch;       /* |L_g[:k*] \ S|, tokens of this row read from the host            */
    int32_t beta_iters;    /* passes the beta solve took                                       */
    int32_t sel_passes;    /* radix-select passes of the on-chip ranking                       */
    uint32_t phase_ns[6];  /* on-chip decision: ns in weights, beta, eq. (7), gain keys, k* search, exact set */
    int32_t n_shrunk;      /* VERKV_SHRINK_BINARY: tokens of L given lambda = r_i; 0 with clipped coefficients */
} verkv_row_trace;

/* Create a context for one GPU (the current device).  All slots empty.
 * EINVAL: bad sizes, n_q_heads not a multiple of n_kv_heads, eta outside
 * (0, 1], unknown shrinkage; EUNSUPPORTED: head_dim != 128 or GQA group > 8. */
verkv_status verkv_create(const verkv_config* cfg, verkv_ctx** out);

/* Free all device memory of the context.  Pending work on the streams the
 * context was used with must be finished by the caller. */
verkv_status verkv_destroy(verkv_ctx* ctx);

/*
 * PoissonComp (Algorithm 1) for one (layer, sequence) slot.
 *   n_tokens  context length n, n_sink + n_local <= n <= max_tokens.
 *   kv_host   pinned host [n_kv_heads][n][2][head_dim] kv_dtype: the offloaded
 *             full cache.  Borrowed until verkv_release(layer, seq); decode
 *             reads fetched rows from it.
 *   kv_dev    optional device copy with the same layout (what prefill leaves
 *             on the GPU).  NULL: compression reads kv_host over the host link.
 *   obs_q     device [n_q_heads][W][head_dim] fp32 observation queries for the
 *             synthetic importance score (Algorithm 1, scoring step: per token, the
 *             largest softmax weight any observation query of the KV head's
 *             group gives it, divided by its maximum over tokens); or NULL.
 *   tau       device [n_kv_heads][n] fp32 importance scores supplied by the
 *             caller (any scorer C), used when obs_q is NULL.  Scores are
 *             clamped to [2^-38, 1]; sink and local tokens get 1.
 *   stats     optional host [n_kv_heads] output.
 * Computes tau, the water-filling constant c with sum_i min(1, c tau_i) =
 * eta n (eq. (3)), r_i = min(1, c tau_i) (stored as fp32; H = {r = 1}), the
 * Poisson sample Z_i = [u_i < r_i] with u_i the top 24 bits of word 0 of
 * Philox4x32-10 at key `seed` and counter (token, kv_head, layer, seq),
 * compacts K/V rows of H u S into device memory (ascending token order) and
 * builds the key sketch.  Synchronises `stream` before returning (the
 * resident sizes decide allocations).  Replaces any previous state of the slot.
 * EINVAL: eta n <= n_sink + n_local, sizes out of range, both obs_q and tau NULL.
 */
verkv_status verkv_compress(verkv_ctx* ctx, int32_t layer, int32_t seq, int32_t n_tokens, const void* kv_host,
                            const void* kv_dev, const float* obs_q, int32_t W, const float* tau,
                            verkv_stream stream, verkv_head_stats* stats);

/*
 * KVFetch (Algorithm 2) and the final attention for B query rows sets.
 *   layer     layer slot.
 *   seq_ids   host [B] sequence slots (each compressed in this layer).
 *   q         device [B][n_q_heads][head_dim] fp32 queries.
 *   eps       tolerance eps >= 0 on the relative error of the denominator.
 *   delta     failure probability, 0 < delta < 1.
 *   out       device [B][n_q_heads][head_dim] fp32 attention outputs.
 * Per query row: sketch weights w^_i = exp(<q, k^_i>/sqrt(d) - m) on L and
 * exact weights on H; the fixed point beta of Definition 2; the certificate
 * eps^(L) of eq. (7) with D = sum_H w_i + sum_L w^_i; if eps^(L) >= eps, the
 * gains g_i = eps^(L) - eps^(L \ {i}) (eq. (9)), the order L_g (descending,
 * ties by token index) and k* of eq. (10); the rows of L_g[:k*] \ S of every
 * query head of a KV head are fetched once (their union) from kv_host; the
 * output is o = N^/D^ with weight 1 on H and on L_g[:k*] and lambda_i / r_i
 * on the rest of S.  With cfg.shrinkage = VERKV_SHRINK_BINARY the fixed point is
 * replaced by the binary coefficients of Appendix A.2 (beta is then their bias).
 * Asynchronous on `stream`: no host synchronisation.
 * EINVAL: bad eps/delta/B; ESTATE: a slot was not compressed; EUNSUPPORTED:
 * binary shrinkage on a row whose |L| exceeds the on-chip decision (16 x 8192
 * entries, or 8 x 8192 on a GPU without 16-block clusters).
 */
verkv_status verkv_decode(verkv_ctx* ctx, int32_t layer, const int32_t* seq_ids, int32_t B, const float* q,
                          double eps, double delta, float* out, verkv_stream stream);

/* Drop the compressed state of a slot and end the borrow of its kv_host. */
verkv_status verkv_release(verkv_ctx* ctx, int32_t layer, int32_t seq);

/*
 * Inspection (copies to caller host buffers; synchronises `stream`).
 * verkv_get_compress_state: for KV head `kv_head` of slot (layer, seq):
 *   c (may be NULL), tau [n] fp32 (NULL to skip), r [n] fp32, flags [n]
 *   (2 = H, 1 = S, 0 = L \ S).  Any array pointer may be NULL.
 */
verkv_status verkv_get_compress_state(verkv_ctx* ctx, int32_t layer, int32_t seq, int32_t kv_head, double* c,
                                      float* tau, float* r, uint8_t* flags, verkv_stream stream);

/* Sketch of one KV head, in the layout the decode reads:
 *   INT8:  codes [n][head_dim] int8, scale [n] fp32.
 *   2BIT:  pairs [head_dim/8] int32, codes [n][head_dim/4] (one 2-bit code per
 *          byte, unpacked for inspection), zero and scale
 *          [ceil(n/group)][head_dim/4] fp16 bit patterns.
 *   EXACT: nothing (returns EINVAL). */
verkv_status verkv_get_sketch(verkv_ctx* ctx, int32_t layer, int32_t seq, int32_t kv_head, int8_t* codes_i8,
                              float* scale_f32, int32_t* pairs, uint8_t* codes_2bit, uint16_t* zero_f16,
                              uint16_t* scale_f16, verkv_stream stream);

/* Traces of the last verkv_decode: rows [B * n_q_heads] (row = b * n_q_heads + h). */
verkv_status verkv_get_decode_trace(verkv_ctx* ctx, verkv_row_trace* rows, int32_t n_rows, verkv_stream stream);

/* Tokens made exact for query row (b, h) in the last decode, L_g[:k*] (as a
 * set, ascending), and the union of fetched rows of KV head (b, kv_head).
 * `count` receives the size; at most `cap` tokens are written. */
verkv_status verkv_get_exact_set(verkv_ctx* ctx, int32_t b, int32_t h, int32_t* tokens, int32_t cap,
                                 int32_t* count, verkv_stream stream);
verkv_status verkv_get_fetch_set(verkv_ctx* ctx, int32_t b, int32_t kv_head, int32_t* tokens, int32_t cap,
                                 int32_t* count, verkv_stream stream);

/* Rows of the last verkv_decode for KV head (b, kv_head): n_union = |the union of its query heads'
 * L_g[:k*] \ S| (the rows the step needs beyond the resident ones), n_host = how many of them the
 * attention read over the host link (the others came from the staging cache or the prefetch buffer).
 * Either pointer may be NULL. */
verkv_status verkv_get_fetch_stats(verkv_ctx* ctx, int32_t b, int32_t kv_head, int32_t* n_union, int32_t* n_host,
                                   verkv_stream stream);

/*
 * Staging cache (the re-use of rows staged in earlier steps, Appendix A.3.2 "Fetching"): a row of
 * L \ S that a decode reads over the host link is also written to device memory, and later decodes
 * of the same slot read it from there.  The cache belongs to the (layer, sequence) slot and is emptied
 * by verkv_compress and freed by verkv_release; the host cache it mirrors is unchanged while borrowed,
 * so staged rows are exact copies.  rows_per_kv_head:
 *   VERKV_STAGE_ETA_N (-2, the default): ceil(eta n) rows per KV head, the size of the resident sample
 *                    again, so that resident and staged rows together hold at most about 2 eta of the
 *                    cache (12.5 % at eta = 1/16; 512 B per row in bf16);
 *   VERKV_STAGE_ALL (-1): room for every row of L \ S of a head (the whole offloaded cache);
 *   0: off (every fetched row crosses the host link at every step);
 *   k > 0: at most k rows per head.
 * A full cache keeps what it holds: rows are staged in the order they are first fetched and never
 * evicted before the next verkv_compress of the slot (an eviction could overwrite a row that another
 * block of the same decode is still reading).  Takes effect at the next verkv_compress of a slot.
 * EINVAL: rows_per_kv_head < -2.  No counterpart in the algorithms themselves: results are identical
 * with any setting.
 */
#define VERKV_STAGE_ETA_N (-2)
#define VERKV_STAGE_ALL (-1)
verkv_status verkv_set_stage_capacity(verkv_ctx* ctx, int64_t rows_per_kv_head);

/*
 * Speculative prefetch (no counterpart in the algorithms: results are identical with it on or off).
 * The host link idles while the decision runs, and the rows a decode fetches are mostly the tokens of
 * L \ S with the largest alpha = w^ (1 - r).  Beside the decision, up to rows_per_kv_head such tokens
 * of each (sequence, KV head) -- neither sampled nor staged, ranked by their largest alpha over the
 * head's query rows relative to each row's largest sketch weight (within 255/16 in log) -- have their
 * K/V rows copied from the pinned host cache into a per-context device buffer; the copying stops once
 * every query row of the call is decided.  It runs on calls whose decision leaves at least eight
 * multiprocessors free.  The attention reads each row it needs from that buffer when the buffer holds
 * it, and over the host link otherwise.  Default 4096 (a buffer of max_batch x n_kv_heads x 4096
 * rows, 512 B each in bf16, allocated at the next verkv_decode); 0 = off.  Takes effect at the next
 * verkv_decode.  EINVAL: rows_per_kv_head outside [0, 65536].
 * verkv_get_prefetch_stats: for KV head (b, kv_head) of the last verkv_decode, n_copied = rows the
 * prefetch copied, n_used = of the rows the step needed beyond the resident and staged ones, how
 * many came from the prefetch buffer (the others crossed the host link during the attention).
 */
verkv_status verkv_set_prefetch(verkv_ctx* ctx, int32_t rows_per_kv_head);
verkv_status verkv_get_prefetch_stats(verkv_ctx* ctx, int32_t b, int32_t kv_head, int32_t* n_copied, int32_t* n_used,
                                      verkv_stream stream);

/*
 * Call timeline (tracing; no counterpart in the paper).  verkv_set_timeline(ctx, 1) makes every
 * following verkv_decode record device times (the GPU's global timer, read by the first CTA to reach
 * a point and by the last to leave it) at two extra small copies per call; 0 turns it off (default).
 * verkv_get_timeline synchronises `stream` and writes VERKV_TIMELINE_N values for the last
 * verkv_decode, in microseconds after the scoring kernel's first CTA started:
 *   [0] decision started (its dependency on the scoring kernel resolved, so the scoring complete),
 *   [1] decision complete (last query row decided), [2] prefetch started, [3] prefetch binning done,
 *   [4] prefetch complete, [5] attention started (after its dependency wait), [6] attention complete
 *   (last KV head merged).
 * NaN where that kernel did not run in the call (the prefetch off or skipped; the multi-kernel
 * decision of rows beyond 262144 L entries records neither [0] nor [1]).  EINVAL when the last
 * verkv_decode recorded no timeline.
 */
#define VERKV_TIMELINE_N 7
verkv_status verkv_set_timeline(verkv_ctx* ctx, int32_t on);
verkv_status verkv_get_timeline(verkv_ctx* ctx, double* out_us, verkv_stream stream);

/*
 * Shortlist (Appendix A.1): at every decode, among the tokens of L outside the sample, the k of each KV
 * head with the largest sketch logit over the head's query rows (ties: lower token index) have their
 * keys read from the pinned host cache and scored exactly, and the decision (beta, eq. (7), gains,
 * k*) uses exact weights for them and for the sampled (resident) tokens, sketch weights for the rest
 * of L.  k = 0 (default) keeps sketch weights on all of L.  Takes effect at the next verkv_decode.
 * EINVAL: k outside [0, 1024].
 */
verkv_status verkv_set_shortlist(verkv_ctx* ctx, int32_t k);

/*
 * Decode-time growth (Appendix A.3.1: the per-(layer, head) list of resident positions is extended
 * as tokens are generated).  verkv_set_append_capacity reserves, at every later verkv_compress, room
 * for rows_per_kv_head appended tokens per KV head of a slot (512 B per row in bf16, capped at
 * max_tokens - n).  Default 0.  EINVAL: rows_per_kv_head < 0.
 *
 * verkv_append adds n_new generated tokens to the (layer, seq) slot: token ids n + n_appended ...,
 * the same tokens for every KV head.  They join H (r = 1): resident, scored with exact keys, in the
 * certificate's denominator and attended with weight 1 by every later verkv_decode; the prefix's
 * L, S, r and sketch stay as verkv_compress left them.  kv_new: [Hkv][n_new][2][d] rows (K then V)
 * in the storage dtype, 16-byte aligned, in device or pinned host memory, read by one kernel on
 * `stream` (caller-owned; free to reuse once the stream has passed the call).  The appended rows live
 * in the slot's device memory until its next verkv_compress or verkv_release.  n_new = 0 is a no-op.
 * EINVAL: n_new < 0, kv_new NULL with n_new > 0, misaligned or in pageable host memory, or more rows
 * than the reserved room;
 * ESTATE: the slot holds no compressed context.
 */
verkv_status verkv_set_append_capacity(verkv_ctx* ctx, int32_t rows_per_kv_head);
verkv_status verkv_append(verkv_ctx* ctx, int32_t layer, int32_t seq, int32_t n_new, const void* kv_new,
                          verkv_stream stream);
/* Tokens appended to the slot since its last verkv_compress. */
verkv_status verkv_get_appended(verkv_ctx* ctx, int32_t layer, int32_t seq, int32_t* n_appended);

/* The shortlist of KV head (b, kv_head) in the last verkv_decode (ascending tokens; count 0 when the
 * shortlist is off).  At most `cap` tokens are written. */
verkv_status verkv_get_shortlist(verkv_ctx* ctx, int32_t b, int32_t kv_head, int32_t* tokens, int32_t cap,
                                 int32_t* count, verkv_stream stream);

/* Sketch weights w^_i (fp32, in units of exp(-m)) of row (b, h) over L in
 * ascending token order, and those tokens. */
verkv_status verkv_get_row_weights(verkv_ctx* ctx, int32_t b, int32_t h, float* w_hat, int32_t* tokens,
                                   int32_t cap, int32_t* count, verkv_stream stream);

/* Failure-path self test (no counterpart in the paper).  Every device-side wait of the decode and
 * compress kernels (mbarrier waits for asynchronous copies) is bounded: when it gives up, the kernel
 * raises the context's mapped error word, leaves its in-flight copies to land and returns, and the
 * next call reports VERKV_ETIMEOUT.  This call takes that path on purpose: it launches one block whose
 * bounded wait is given a barrier that nothing completes, synchronises `stream`, and returns
 * VERKV_ETIMEOUT (VERKV_OK would mean the wait did not give up).  The context stays usable. */
verkv_status verkv_selftest_wait_timeout(verkv_ctx* ctx, verkv_stream stream);

/* Number of kernels the last verkv_decode / verkv_compress enqueued. */
int32_t verkv_last_launch_count(const verkv_ctx* ctx);

/* Per-kernel timing (the per-phase breakdown of a decode step).  When enabled, every later
 * verkv_decode / verkv_compress records a CUDA event on its stream before its first kernel and
 * after each kernel it launches; no host synchronisation is added.  Records accumulate across calls
 * (up to 4096 kernels) until verkv_get_kernel_times, which synchronises on the last event, returns
 * the kernel names (static strings) and the device milliseconds of each launch (for compress these
 * include host-side gaps between launches), and clears the record.  `count` receives the number of
 * records; at most `cap` are written.  Enabling clears the record. */
verkv_status verkv_set_kernel_timing(verkv_ctx* ctx, int32_t enable);
verkv_status verkv_get_kernel_times(verkv_ctx* ctx, const char** names, float* ms, int32_t cap, int32_t* count,
                                    verkv_stream stream);

/*
 * Allocation-free decision for one query row.  This entry point has no counterpart in the paper.  It
 * runs the same per-row decision as verkv_decode -- the shrinkage fixed point beta, the error
 * certificate eps_hat, the per-token gains, their full ranking and the number k* of tokens to make
 * exact -- without a context and without allocating any device memory.  It is for callers that
 * cannot call cudaMalloc: code whose memory is fixed up front (an engine with its own arena, a
 * real-time loop that must not allocate), or code running while a CUDA stream is being captured
 * into a graph, where an allocation would either fail or become part of the graph.
 *   w_hat   device [n_l] fp32 sketch weights of the row's L tokens (any common scale), >= 0 and finite,
 *   r       device [n_l] fp32 inclusion probabilities of those tokens, 0 < r < 1,
 *   D       the certificate denominator in the same scale (sum_H w + sum_L w_hat), > 0,
 *   scalars device [4] output: beta, eps_hat, sum_L w_hat (1 - lambda), the variance term V,
 *   kstar   device [1] output: k* (0 when eps_hat < eps or n_l = 0),
 *   exact   device [n_l] output: the first k* entries are the indices (into w_hat) of the tokens to
 *           make exact, best gain first; nothing is written when k* = 0 (exact may be NULL when n_l = 0).
 * An entry of r outside (0, 1), or of w_hat negative or not finite, is reported on the device:
 * kstar = -1 and NaN scalars (the host cannot see the values without a copy).
 * Scratch is a library-wide static device array of VERKV_STATIC_MAX_L 64-bit keys (512 KiB, held by
 * every GPU that loads the library until the process exits): n_l > VERKV_STATIC_MAX_L returns
 * VERKV_EINVAL.  All calls share that array and it keeps the last call's contents (every call
 * rewrites the part it reads), so calls whose kernels overlap on a GPU (different streams, or several
 * host threads) race and must be serialised by the caller.  The first call on each device looks up
 * the array's device address (with that device current) and keeps it for the life of the process:
 * make that first call before any stream capture, and do not use this entry point on a device after
 * cudaDeviceReset (the kept address would be stale).  Asynchronous on `stream`. */
#define VERKV_STATIC_MAX_L 65536
verkv_status verkv_certify_row_static(const float* w_hat, const float* r, int32_t n_l, double D, double eps,
                                      double delta, double* scalars, int32_t* kstar, int32_t* exact,
                                      verkv_stream stream);

const char* verkv_status_str(verkv_status s);
const char* verkv_last_error(const verkv_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* VERKV_H */
