/*
 * gdn.h - C ABI of the Gated DeltaNet speculative verify/commit library (libgdn.so).
 *
 * The operation.  Gated DeltaNet (GDN) layers keep a fixed-size recurrent state
 * per request and head, read and rewritten for every token; ReplaySSM keeps a
 * checkpoint of that state, computes the draft tokens' outputs from the
 * checkpoint and the buffered inputs, and on rejection keeps only the accepted
 * prefix (OCRia write-up "OCRia 推理栈：单卡 B200 提速近 10 倍", section "Make
 * speculative verification cheaper"; the same in "Wie OCRia einen 10-fachen
 * Inference-Speedup auf B200-GPUs erreichte", section "Wie es funktioniert").  The state
 * update is the gated delta rule, with S the dv x dk state of one unit
 * (request r, head h):
 *
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t q_t
 *
 * Layout (all row-major, all device memory, all caller-owned):
 *   state tile  float32 [dk][dv], tile[i][j] = S[j][i] (key index i is the row,
 *               value index j contiguous); 64 KiB at dk = dv = 128.
 *   pool        float32 [pool_slots][heads][dk][dv]; request r's checkpoint is
 *               pool[slot_ids[r]][h].
 *   q, k        [N_tok][heads][dk], v [N_tok][heads][dv], bfloat16 or float32
 *               (qkv_dtype); token rows of request r are [cu[r], cu[r+1]) with
 *               cu = cu_seqlens, or [r*max_T, (r+1)*max_T) when cu_seqlens is NULL.
 *   alpha, beta float32 [N_tok][heads] (alpha is the decay gate, beta the write
 *               strength; both given directly, no activation applied; with
 *               GDN_FLAG_LOG_GATE alpha holds g and the decay is expf(g)).
 *   o           float32 [N_tok][heads][dv] (bfloat16 with GDN_FLAG_O_BF16).
 *   accepted    int32 [batch], a_r in [0, T_r].
 *
 * Calls.  All compute calls are asynchronous on `stream`; they validate their
 * arguments on the host first and return an error without launching anything
 * if a check fails.  They allocate no memory and keep no state between calls.
 *   gdn_verify               o_t for every draft token; never writes the pool.
 *   gdn_commit               pool[slot_r][h] <- state after a_r tokens, for
 *                            every r with a_r > 0; slots with a_r = 0 and slots
 *                            no request names are left bit-identical.
 *   gdn_verify_commit_fused  both in one pass: reads each checkpoint once,
 *                            writes o for every token and the state once.
 *   gdn_commit_verify        the previous step's commit, then this step's
 *                            verify, in one pass (the order an engine can run
 *                            them in: a step's accepted lengths are known only
 *                            after all its layers verified).
 *   gdn_*_layers             the same calls for the layers of one step, in as
 *                            few launches as possible.
 *   gdn_replay_verify/commit a multi-step ReplaySSM buffer: outputs from the
 *                            checkpoint plus buffered rows, periodic flush.
 *   gdn_accept_prefix        greedy accepted lengths from token ids, on the
 *                            device.
 *   gdn_selftest_wait_timeout  runs the bounded wait to its expiry (diagnostic).
 *
 * Device-side argument errors (a slot id outside [0, pool_slots), a_r outside
 * [0, T_r], a ragged length outside [0, max_T]) cannot be seen on the host
 * without a synchronisation; the kernel ORs a GDN_DEVERR_* bit into *dev_err
 * (when dev_err is not NULL) and skips that unit, writing nothing for it.  It
 * never traps.  The chunked kernel's internal waits give up after about two
 * seconds and report GDN_DEVERR_TIMEOUT instead of hanging.  Duplicate slot
 * ids among the requests of one call are a precondition violation: commit
 * results are then undefined.
 */
#ifndef GDN_H
#define GDN_H

#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_NULL_PTR = 1,     /* a required pointer is NULL */
    GDN_ERR_BAD_DIM = 2,      /* batch/heads/max_T/pool_slots/n_tok out of range (token rows,
                                 batch*max_T or n_tok, above 2^31 - 1), or unknown flags */
    GDN_ERR_BAD_DTYPE = 3,    /* qkv_dtype is not a gdn_dtype */
    GDN_ERR_UNSUPPORTED = 4,  /* dk/dv (or a forced algo) not supported */
    GDN_ERR_DEVICE_ARG = 5,   /* reported by gdn_read_device_error only */
    GDN_ERR_CUDA = 6,         /* a CUDA call failed; see gdn_last_error_string */
    GDN_ERR_ALIGN = 7,        /* a pointer is not aligned (16 bytes for q/k/v/pool/o) */
    GDN_ERR_ALIAS = 8,        /* o overlaps an input, or the pool overlaps q/k/v/o */
    GDN_ERR_LAYER_MISMATCH = 9 /* the problems of a layer batch disagree on a shared field */
} gdn_status;

typedef enum gdn_dtype {
    GDN_FP32 = 0,
    GDN_BF16 = 1
} gdn_dtype;

/* Which kernel runs.  AUTO: the chunked tensor-core kernel where it applies
 * (bf16 q/k/v, dk = dv = 128, any max_T: blocks of 16 tokens chained through
 * the state), else the recurrent kernel. */
typedef enum gdn_algo {
    GDN_ALGO_AUTO = 0,
    GDN_ALGO_RECURRENT = 1,   /* per-token update on CUDA cores, any supported shape */
    GDN_ALGO_CHUNK = 2,       /* WY/chunk form, bf16 mma.sync for the state products; 16-token
                                 chunks, the state carried from one chunk to the next */
    GDN_ALGO_CHUNK_TC = 3     /* the same chunk form with the two state-sized products on
                                 tcgen05.mma (A = H^T staged in tensor memory, accumulators in
                                 tensor memory) and the small solves on CUDA cores; same shapes
                                 as GDN_ALGO_CHUNK, results within the same tolerance; opt-in
                                 (slower than GDN_ALGO_CHUNK on 16-token chunks); no replay
                                 buffer calls; layer batches run one launch per layer */
} gdn_algo;

/* Bits ORed into *dev_err by the kernels. */
#define GDN_DEVERR_SLOT     1   /* slot_ids[r] outside [0, pool_slots) */
#define GDN_DEVERR_ACCEPTED 2   /* accepted[r] outside [0, T_r]        */
#define GDN_DEVERR_SEQLEN   4   /* cu[r+1] - cu[r] outside [0, max_T], or rows outside [0, n_tok) */
#define GDN_DEVERR_TIMEOUT  8   /* an internal pipeline wait gave up (about 2 s); results incomplete.
                                   The block that gave up also bounds its wait for its own
                                   copies in flight; if that wait gives up too, copies (or, on
                                   the tcgen05 kernel, products) may still land after the kernel
                                   ends.  Treat every later result on the stream as suspect until
                                   the CUDA context has been rebuilt. */
#define GDN_DEVERR_REPLAY  16   /* replay buffer: len_in[slot] < 0, or buffered plus new rows > capacity */

/* Variant bits of gdn_problem.flags (the same in every problem of a layer batch). */
#define GDN_FLAG_O_BF16    1    /* o is bfloat16 [N_tok][heads][dv], round to nearest even of the
                                   float32 result; otherwise o is float32 */
#define GDN_FLAG_LOG_GATE  2    /* alpha holds the log-space gate g; the kernels use alpha =
                                   expf(g) (CUDA's expf) */

/* Limits checked on the host. */
#define GDN_MAX_T 1024          /* draft tokens per request */

typedef struct gdn_problem {
    int32_t batch;               /* B >= 0 requests (B = 0: calls return GDN_OK, no launch) */
    int32_t heads;               /* H >= 1 */
    int32_t dk;                  /* key dim: 32, 64, 128 or 256 */
    int32_t dv;                  /* value dim: a multiple of 32, <= 128 or 256 */
    int32_t max_T;               /* uniform draft length (cu_seqlens NULL) or the ragged maximum, 0..GDN_MAX_T */
    int32_t qkv_dtype;           /* gdn_dtype of q, k, v */
    int32_t algo;                /* gdn_algo */
    int32_t flags;               /* GDN_FLAG_* bits; all other bits must be 0 */
    const int32_t *cu_seqlens;   /* device [batch+1] token-row offsets, or NULL (uniform) */
    const void *q;               /* device [N_tok][heads][dk], 16-byte aligned; may be NULL for
                                    the commit calls (gdn_commit, gdn_commit_layers,
                                    gdn_replay_commit), which read no q */
    const void *k;               /* device [N_tok][heads][dk], 16-byte aligned */
    const void *v;               /* device [N_tok][heads][dv], 16-byte aligned */
    const float *alpha;          /* device [N_tok][heads]: alpha, or g = log(alpha) with GDN_FLAG_LOG_GATE */
    const float *beta;           /* device [N_tok][heads] */
    float *pool;                 /* device [pool_slots][heads][dk][dv], 16-byte aligned */
    int64_t pool_slots;          /* >= batch */
    const int32_t *slot_ids;     /* device [batch], distinct, in [0, pool_slots) */
    int32_t *dev_err;            /* device int32 error word (GDN_DEVERR_* bits), or NULL */
    int64_t n_tok;               /* rows of q/k/v/alpha/beta/o.  Ignored for uniform input
                                    (batch*max_T); REQUIRED for ragged input: the kernels
                                    flag GDN_DEVERR_SEQLEN for a request whose rows
                                    [cu[r], cu[r+1]) do not lie in [0, n_tok) */
} gdn_problem;

/* o_t for every draft token of every unit.  o: device float32 (or, with
 * GDN_FLAG_O_BF16, bfloat16) [N_tok][heads][dv],
 * 16-byte aligned, must not overlap any input.  Reads the pool, never writes it. */
GDN_API gdn_status gdn_verify(const gdn_problem *p, void *o, cudaStream_t stream);

/* For every request r with accepted[r] > 0: pool[slot_ids[r]][h] <- state after
 * accepted[r] tokens, replayed from the checkpoint in that same slot (in place).
 * Requests with accepted[r] = 0 write nothing.  accepted: device int32 [batch]. */
GDN_API gdn_status gdn_commit(const gdn_problem *p, const int32_t *accepted, cudaStream_t stream);

/* gdn_verify and then gdn_commit with the same inputs, in one pass: each
 * checkpoint is read once, o is written for every token, the state once. */
GDN_API gdn_status gdn_verify_commit_fused(const gdn_problem *p, const int32_t *accepted,
                                           void *o, cudaStream_t stream);

/* Layer batches: the same calls for the n_layers problems of one step (one per
 * model layer), in as few launches as possible (the chunked kernel takes up to
 * 32 layers per launch, so the fill and drain of a launch are paid once for
 * all of them instead of once per layer).
 *
 * problems: host array of n_layers gdn_problem.  They must agree on the
 * request-level fields (batch, heads, dk, dv, max_T, qkv_dtype, algo,
 * cu_seqlens, slot_ids, pool_slots, and n_tok when ragged), else
 * GDN_ERR_LAYER_MISMATCH; each names its own q, k, v, alpha, beta, pool (that
 * layer's pool) and dev_err.  o: host array of n_layers device pointers, o[l]
 * for problem l as in gdn_verify.  accepted: one device array, shared by all
 * layers.  Each problem is validated as by the single-problem call; besides,
 * no layer's o, nor (commit, fused) its pool, may overlap another layer's
 * arrays (GDN_ERR_ALIAS).  The results equal those of the single-problem call
 * made once per layer.  n_layers = 0 launches nothing. */
GDN_API gdn_status gdn_verify_layers(const gdn_problem *problems, int32_t n_layers,
                                     void *const *o, cudaStream_t stream);
GDN_API gdn_status gdn_commit_layers(const gdn_problem *problems, int32_t n_layers,
                                     const int32_t *accepted, cudaStream_t stream);
GDN_API gdn_status gdn_verify_commit_fused_layers(const gdn_problem *problems, int32_t n_layers,
                                                  const int32_t *accepted, void *const *o,
                                                  cudaStream_t stream);

/* Greedy accepted lengths on the device, so that the commit needs no host round
 * trip: accepted[r] = the largest a in [0, T_r] such that
 *     draft_ids[c_r + t] == target_ids[c_r + t]   for every t < a,
 * with c_r, T_r the token rows of request r as for gdn_problem (cu_seqlens, or
 * r * max_T and max_T when cu_seqlens is NULL).  Speculative decoding keeps the
 * draft tokens that agree with the target model and rolls back to that prefix
 * (OCRia write-up, sections "Generate more tokens per target pass: speculative
 * decoding" and "Make speculative verification cheaper"); this is the greedy
 * form of that check.  The caller lines up both arrays so that row c_r + t
 * holds the draft id of the token fed at that row and the target's own choice
 * for it (a row that is always kept is passed with equal ids).
 *
 * draft_ids, target_ids: device int32 [n_tok] (uniform: batch * max_T rows);
 * accepted: device int32 [batch], written; it must not overlap the other
 * arrays.  A ragged request whose rows leave [0, n_tok) or whose length
 * leaves [0, max_T] sets GDN_DEVERR_SEQLEN in *dev_err and its accepted[r] is
 * not written.  batch = 0 launches nothing.  All pointers 4-byte aligned. */
GDN_API gdn_status gdn_accept_prefix(int32_t batch, int32_t max_T, const int32_t *cu_seqlens,
                                     int64_t n_tok, const int32_t *draft_ids,
                                     const int32_t *target_ids, int32_t *accepted,
                                     int32_t *dev_err, cudaStream_t stream);

/* ReplaySSM buffer (multi-step speculation).  ReplaySSM keeps a checkpoint of
 * the state next to a small buffer of recent inputs, computes outputs from
 * both, writes the full checkpoint only at periodic flushes, and rolls a
 * rejection back by moving the buffer pointer (OCRia write-up, section "Make
 * speculative verification cheaper").  Here pool[slot] is the checkpoint as
 * of the slot's last flush, and the slot's buffer holds the rows accepted
 * since then: rows slot * capacity + [0, len_in[slot]) of k, v, alpha, beta
 * (the layout of the token arrays, with pool_slots * capacity rows).
 *
 * A step, for request r in slot s with n = len_in[s]:
 *   1. the caller writes the step's draft rows of k, v, alpha, beta at buffer
 *      rows s * capacity + n + [0, T_r) (n + T_r <= capacity), and q as usual
 *      at rows cu[r] + [0, T_r) of p->q;
 *   2. gdn_replay_verify: o for the draft rows (rows cu[r] + t of o), from
 *      pool[s] and buffer rows [0, n + T_r); writes neither pool nor buffer;
 *   3. gdn_replay_commit with accepted[r] = a_r: keep = n + a_r.  If
 *      keep + max_T > capacity (a full next draft would not fit) the slot is
 *      flushed: pool[s][h] <- the state after buffer rows [0, keep) and
 *      len_out[s] = 0; otherwise the pool is not touched and len_out[s] = keep
 *      (rejected rows are overwritten by the next step's drafts);
 *   4. the caller swaps len_in and len_out for the next step.
 * Only the chunked kernel runs these calls (bf16 q/k/v, dk = dv = 128);
 * other shapes return GDN_ERR_UNSUPPORTED.  p->k, p->v, p->alpha and p->beta
 * are not used (the buffer holds those rows); every other field of p means
 * what it means for gdn_verify and gdn_commit.  A unit whose buffer does not
 * hold its rows (n < 0, n + T_r > capacity in verify, keep > capacity in
 * commit) sets GDN_DEVERR_REPLAY and is skipped; len_out[s] is then not
 * written.  len_out[s] is written for every named slot, by one thread;
 * entries of other slots are left as they are. */
typedef struct gdn_replay {
    int32_t capacity;            /* buffer rows per slot, >= max_T */
    int32_t reserved;            /* must be 0 */
    const void *k;               /* device [pool_slots * capacity][heads][dk], qkv_dtype, 16-byte aligned */
    const void *v;               /* device [pool_slots * capacity][heads][dv], 16-byte aligned */
    const float *alpha;          /* device [pool_slots * capacity][heads] */
    const float *beta;           /* device [pool_slots * capacity][heads] */
    const int32_t *len_in;       /* device [pool_slots]: rows buffered in each slot */
    int32_t *len_out;            /* device [pool_slots]: written by gdn_replay_commit; must not
                                    overlap len_in or any other array */
} gdn_replay;

GDN_API gdn_status gdn_replay_verify(const gdn_problem *p, const gdn_replay *rb, void *o,
                                     cudaStream_t stream);
GDN_API gdn_status gdn_replay_commit(const gdn_problem *p, const gdn_replay *rb,
                                     const int32_t *accepted, cudaStream_t stream);

/* Commit the previous step, then verify the next one, in one pass over each
 * checkpoint (OCRia write-up, section "Make speculative verification
 * cheaper": rollback keeps the accepted prefix; in an engine the accepted
 * lengths of a step are known only after all its layers have verified, so a
 * layer's commit of step n - 1 can run at its verify of step n).
 *
 * For every request r and head h, with S the state in pool[slot_ids[r]][h]:
 *   1. if prev->accepted[r] = a > 0: S <- the state after the first a rows of
 *      the previous step replayed from S, written back to the slot (as
 *      gdn_commit with that step's problem would);
 *   2. o <- the outputs of this step's drafts from S (as gdn_verify would).
 * The previous step's own W (a by-product of its call, written to its `w`) is
 * what makes step 1 a single rank-a update: no products of the checkpoint.
 *
 *   p     this step: everything gdn_verify takes.  bf16 q/k/v, dk = dv = 128,
 *         1 <= max_T <= 16 (GDN_ERR_UNSUPPORTED otherwise); AUTO or GDN_ALGO_CHUNK.
 *   prev  the previous step of the same requests (same batch, heads, slot ids),
 *         or NULL for the first step (nothing is committed).
 *   o     as gdn_verify.
 *   w     device float32 [N_tok][heads][dv], 16-byte aligned, written: this
 *         step's W, for the next call's prev->w (the caller alternates two
 *         buffers).  Must not overlap any other array of the call.
 * Device errors: prev->accepted[r] outside [0, T_prev,r] sets
 * GDN_DEVERR_ACCEPTED, bad previous row offsets GDN_DEVERR_SEQLEN; the unit is
 * skipped (no write, no outputs). */
typedef struct gdn_prev_step {
    const int32_t *cu_seqlens;   /* device [batch+1] row offsets of the previous step, or NULL (uniform max_T) */
    int32_t max_T;               /* its uniform length, or its ragged maximum; 0..16 */
    int32_t reserved;            /* must be 0 */
    int64_t n_tok;               /* rows of its arrays (ragged; ignored when cu_seqlens is NULL) */
    const void *k;               /* device, its k [n_tok][heads][dk], 16-byte aligned */
    const float *alpha;          /* device, its alpha (or g with GDN_FLAG_LOG_GATE) [n_tok][heads] */
    const float *w;              /* device, the w its call wrote [n_tok][heads][dv], 16-byte aligned */
    const int32_t *accepted;     /* device [batch]: its accepted lengths */
} gdn_prev_step;

GDN_API gdn_status gdn_commit_verify(const gdn_problem *p, const gdn_prev_step *prev, void *o,
                                     float *w, cudaStream_t stream);

/* Waits for `stream`, copies *p->dev_err to *host_code (0 when dev_err is NULL).
 * Returns GDN_ERR_DEVICE_ARG when the word is non-zero, GDN_OK when it is zero. */
GDN_API gdn_status gdn_read_device_error(const gdn_problem *p, cudaStream_t stream,
                                         int32_t *host_code);

/* Self-check of the bounded waits (diagnostic; not part of a decode step).
 * The chunked kernel waits on shared-memory barriers for its copies and
 * products, and gives up after about two seconds with GDN_DEVERR_TIMEOUT
 * rather than hang.  This call runs that same wait in one block, on a barrier
 * that nothing completes: after about two seconds the block ORs
 * GDN_DEVERR_TIMEOUT into *dev_err and exits, and the CUDA context stays
 * usable.  Asynchronous on `stream` (one SM is busy meanwhile).
 * dev_err: device int32, caller-owned, 4-byte aligned, not NULL (else
 * GDN_ERR_NULL_PTR / GDN_ERR_ALIGN before any CUDA call). */
GDN_API gdn_status gdn_selftest_wait_timeout(int32_t *dev_err, cudaStream_t stream);

/* The algo that AUTO resolves to for this problem (host only, no CUDA call),
 * or -1 when the shape fails validation. */
GDN_API int32_t gdn_select_algo(const gdn_problem *p);

/* Static, never NULL. */
GDN_API const char *gdn_status_string(gdn_status s);

/* Text of the last CUDA error seen by this thread ("" if none). */
GDN_API const char *gdn_last_error_string(void);

/* Library version, e.g. "0.1.0". */
GDN_API const char *gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
