// C ABI of libgdn.so: host-side validation, kernel selection and launch.
// Every check runs before any CUDA call, so a rejected call launches nothing
// (and the checks work on a machine without a GPU).
#include <cstdint>
#include <cstdio>

#include "gdn.h"
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace {

thread_local char g_last_error[256] = "";

void set_cuda_error(cudaError_t e, const char *where) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where,
                  cudaGetErrorString(e), (int)e);
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }
bool aligned4(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

// An absent array (NULL) covers no bytes.
Range range(const void *ptr, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
    return Range{lo, ptr ? lo + (uintptr_t)(bytes > 0 ? bytes : 0) : lo};
}

bool overlap(Range a, Range b) {
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

// Rows of the token arrays.
int64_t token_rows(const gdn_problem *p) {
    return p->cu_seqlens ? p->n_tok : (int64_t)p->batch * p->max_T;
}

// The byte ranges of one problem's per-layer arrays.
struct LayerRanges {
    Range q, k, v, alpha, beta, pool;
};

// kv_rows: rows of k, v, alpha and beta (-1: the token rows).
LayerRanges layer_ranges(const gdn_problem *p, int64_t kv_rows = -1) {
    const int64_t H = p->heads;
    const int64_t n_tok = token_rows(p);
    const int64_t nkv = kv_rows < 0 ? n_tok : kv_rows;
    const int64_t esz = p->qkv_dtype == GDN_BF16 ? 2 : 4;
    LayerRanges r;
    r.q = range(p->q, n_tok * H * p->dk * esz);
    r.k = range(p->k, nkv * H * p->dk * esz);
    r.v = range(p->v, nkv * H * p->dv * esz);
    r.alpha = range(p->alpha, nkv * H * 4);
    r.beta = range(p->beta, nkv * H * 4);
    r.pool = range(p->pool, p->pool_slots * H * p->dk * p->dv * 4);
    return r;
}

Range o_range(const gdn_problem *p, const void *o) {
    const int64_t esz = (p->flags & GDN_FLAG_O_BF16) ? 2 : 4;
    return range(o, token_rows(p) * p->heads * p->dv * esz);
}

constexpr int32_t kKnownFlags = GDN_FLAG_O_BF16 | GDN_FLAG_LOG_GATE;

bool dims_supported(int dk, int dv) {
    const bool dk_ok = dk == 32 || dk == 64 || dk == 128 || dk == 256;
    const bool dv_ok = dv >= 32 && dv <= 256 && dv % 32 == 0 && (dv <= 128 || dv % 128 == 0);
    return dk_ok && dv_ok;
}

bool shape_ok(const gdn_problem *p) {
    return p->batch >= 0 && p->heads >= 1 && p->max_T >= 0 && p->max_T <= GDN_MAX_T &&
           (int64_t)p->batch * p->heads <= 0x7fffffffLL;
}

// Which kernel AUTO picks.  The chunked tensor-core kernel covers bf16 q/k/v at
// dk = dv = 128 and any draft length (16-token chunks chained through the state);
// the recurrent kernel the rest.
int resolve_algo(const gdn_problem *p) {
    // The chunked kernel also needs at least one token row (ragged input may have none).
    const bool chunk_ok = gdn::chunk_supported(p->qkv_dtype == GDN_BF16, p->dk, p->dv, p->max_T) &&
                          (!p->cu_seqlens || p->n_tok >= 1);
    if (p->algo == GDN_ALGO_RECURRENT) return GDN_ALGO_RECURRENT;
    if (p->algo == GDN_ALGO_CHUNK) return chunk_ok ? GDN_ALGO_CHUNK : -1;
    if (p->algo == GDN_ALGO_CHUNK_TC) return chunk_ok ? GDN_ALGO_CHUNK_TC : -1;
    return (chunk_ok && gdn::chunk_preferred(p->max_T)) ? GDN_ALGO_CHUNK : GDN_ALGO_RECURRENT;
}

// Host validation shared by all entry points.  On success *algo is the kernel
// to run and *empty tells whether there is nothing to launch.
gdn_status validate(const gdn_problem *p, bool with_o, const void *o, bool with_acc,
                    const int32_t *accepted, int *algo, bool *empty, int64_t kv_rows = -1) {
    if (!p) return GDN_ERR_NULL_PTR;
    if ((p->flags & ~kKnownFlags) != 0 || !shape_ok(p)) return GDN_ERR_BAD_DIM;
    if (p->qkv_dtype != GDN_FP32 && p->qkv_dtype != GDN_BF16) return GDN_ERR_BAD_DTYPE;
    if (!dims_supported(p->dk, p->dv)) return GDN_ERR_UNSUPPORTED;
    if (p->algo < GDN_ALGO_AUTO || p->algo > GDN_ALGO_CHUNK_TC) return GDN_ERR_UNSUPPORTED;
    *algo = resolve_algo(p);
    if (*algo < 0) return GDN_ERR_UNSUPPORTED;
    *empty = p->batch == 0;
    if (*empty) return GDN_OK;
    if (p->pool_slots < p->batch) return GDN_ERR_BAD_DIM;
    if (p->cu_seqlens && p->n_tok < 0) return GDN_ERR_BAD_DIM;
    // Token rows are indexed with 32-bit ints on the device.
    if (token_rows(p) > 0x7fffffffLL || kv_rows > 0x7fffffffLL) return GDN_ERR_BAD_DIM;
    if (!p->pool || !p->slot_ids) return GDN_ERR_NULL_PTR;
    // q is read only by calls that produce outputs (a commit may pass NULL).
    if (p->max_T > 0 && ((with_o && !p->q) || !p->k || !p->v || !p->alpha || !p->beta))
        return GDN_ERR_NULL_PTR;
    if (with_o && !o) return GDN_ERR_NULL_PTR;
    if (with_acc && !accepted) return GDN_ERR_NULL_PTR;
    if (!aligned16(p->q) || !aligned16(p->k) || !aligned16(p->v) || !aligned16(p->pool) ||
        !aligned16(o) || !aligned4(p->alpha) || !aligned4(p->beta) || !aligned4(p->slot_ids) ||
        !aligned4(p->cu_seqlens) || !aligned4(accepted) || !aligned4(p->dev_err))
        return GDN_ERR_ALIGN;

    // Aliasing: o must not overlap any input; the pool must not overlap q/k/v/gates/metadata.
    const LayerRanges lr = layer_ranges(p, kv_rows);
    const Range rq = lr.q, rk = lr.k, rv = lr.v, ra = lr.alpha, rb = lr.beta, rp = lr.pool;
    const Range rs = range(p->slot_ids, (int64_t)p->batch * 4);
    const Range rc = range(p->cu_seqlens, p->cu_seqlens ? ((int64_t)p->batch + 1) * 4 : 0);
    const Range racc = range(accepted, with_acc ? (int64_t)p->batch * 4 : 0);
    const Range re = range(p->dev_err, p->dev_err ? 4 : 0);
    const Range others[] = {rq, rk, rv, ra, rb, rs, rc, racc, re};
    for (const Range &x : others)
        if (overlap(rp, x)) return GDN_ERR_ALIAS;
    if (with_o) {
        const Range ro = o_range(p, o);
        const Range all[] = {rq, rk, rv, ra, rb, rp, rs, rc, racc, re};
        for (const Range &x : all)
            if (overlap(ro, x)) return GDN_ERR_ALIAS;
    }
    return GDN_OK;
}

gdn::Args make_args(const gdn_problem *p, const int32_t *accepted, void *o) {
    gdn::Args a;
    a.B = p->batch;
    a.H = p->heads;
    a.dk = p->dk;
    a.dv = p->dv;
    a.max_T = p->max_T;
    a.n_tok = p->cu_seqlens ? p->n_tok : (long long)p->batch * p->max_T;
    a.cu_seqlens = p->cu_seqlens;
    a.q = p->q;
    a.k = p->k;
    a.v = p->v;
    a.alpha = p->alpha;
    a.beta = p->beta;
    a.pool = p->pool;
    a.pool_slots = p->pool_slots;
    a.slot_ids = p->slot_ids;
    a.accepted = accepted;
    a.o = o;
    a.dev_err = p->dev_err;
    a.kv_rows = a.n_tok;
    a.flags = p->flags;
    a.tc = p->algo == GDN_ALGO_CHUNK_TC;
    return a;
}

gdn_status run(const gdn_problem *p, int mode, const int32_t *accepted, void *o,
               cudaStream_t stream) {
    int algo = 0;
    bool empty = false;
    const bool with_o = mode != gdn::kCommit;
    const bool with_acc = mode != gdn::kVerify;
    const gdn_status st = validate(p, with_o, o, with_acc, accepted, &algo, &empty);
    if (st != GDN_OK || empty) return st;
    const gdn::Args a = make_args(p, with_acc ? accepted : nullptr, with_o ? o : nullptr);
    const bool bf16 = p->qkv_dtype == GDN_BF16;
    const bool chunk = algo == GDN_ALGO_CHUNK || algo == GDN_ALGO_CHUNK_TC;
    const cudaError_t e = chunk ? gdn::launch_chunk(&a, 1, mode, stream)
                                : gdn::launch_recurrent(a, mode, bf16, stream);
    if (e != cudaSuccess) {
        set_cuda_error(e, "kernel launch");
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

// The request-level fields that all problems of a layer batch share.
bool same_requests(const gdn_problem *a, const gdn_problem *b) {
    return a->batch == b->batch && a->heads == b->heads && a->dk == b->dk && a->dv == b->dv &&
           a->max_T == b->max_T && a->qkv_dtype == b->qkv_dtype && a->algo == b->algo &&
           a->flags == b->flags &&
           a->cu_seqlens == b->cu_seqlens && a->slot_ids == b->slot_ids &&
           a->pool_slots == b->pool_slots && (!a->cu_seqlens || a->n_tok == b->n_tok);
}

// Layer batch: every problem passes the single-problem checks, all share the
// request-level fields, and no layer's output (o, or the pool it commits
// into) overlaps another layer's arrays.  Then up to gdn::kChunkMaxLayers
// layers go into each launch of the chunked kernel; the recurrent kernel runs
// once per layer.
gdn_status run_layers(const gdn_problem *ps, int32_t n, int mode, const int32_t *accepted,
                      void *const *o, cudaStream_t stream) {
    if (n < 0) return GDN_ERR_BAD_DIM;
    if (n == 0) return GDN_OK;
    if (!ps) return GDN_ERR_NULL_PTR;
    const bool with_o = mode != gdn::kCommit;
    const bool with_acc = mode != gdn::kVerify;
    if (with_o && !o) return GDN_ERR_NULL_PTR;
    int algo = 0;
    bool empty = false;
    for (int32_t l = 0; l < n; ++l) {
        const gdn_status st =
            validate(&ps[l], with_o, with_o ? o[l] : nullptr, with_acc, accepted, &algo, &empty);
        if (st != GDN_OK) return st;
        if (l > 0 && !same_requests(&ps[0], &ps[l])) return GDN_ERR_LAYER_MISMATCH;
    }
    if (empty) return GDN_OK;
    for (int32_t i = 0; i < n; ++i) {
        const Range ro = with_o ? o_range(&ps[i], o[i]) : Range{0, 0};
        const Range rpool = layer_ranges(&ps[i]).pool;
        for (int32_t j = 0; j < n; ++j) {
            if (i == j) continue;
            const LayerRanges r = layer_ranges(&ps[j]);
            const Range ins[] = {r.q, r.k, r.v, r.alpha, r.beta, r.pool};
            for (const Range &x : ins) {
                if (with_o && overlap(ro, x)) return GDN_ERR_ALIAS;
                if (with_acc && overlap(rpool, x)) return GDN_ERR_ALIAS;
            }
            if (with_o && overlap(ro, o_range(&ps[j], o[j]))) return GDN_ERR_ALIAS;
        }
    }
    const bool bf16 = ps[0].qkv_dtype == GDN_BF16;
    for (int32_t l0 = 0; l0 < n; l0 += gdn::kChunkMaxLayers) {
        const int m = n - l0 < gdn::kChunkMaxLayers ? n - l0 : gdn::kChunkMaxLayers;
        gdn::Args a[gdn::kChunkMaxLayers];
        for (int l = 0; l < m; ++l)
            a[l] = make_args(&ps[l0 + l], with_acc ? accepted : nullptr,
                             with_o ? o[l0 + l] : nullptr);
        cudaError_t e = cudaSuccess;
        if (algo == GDN_ALGO_CHUNK || algo == GDN_ALGO_CHUNK_TC) {
            e = gdn::launch_chunk(a, m, mode, stream);
        } else {
            for (int l = 0; l < m && e == cudaSuccess; ++l)
                e = gdn::launch_recurrent(a[l], mode, bf16, stream);
        }
        if (e != cudaSuccess) {
            set_cuda_error(e, "kernel launch");
            return GDN_ERR_CUDA;
        }
    }
    return GDN_OK;
}

gdn_status run_replay(const gdn_problem *p, const gdn_replay *rb, int mode,
                      const int32_t *accepted, void *o, cudaStream_t stream) {
    if (!p || !rb) return GDN_ERR_NULL_PTR;
    if (rb->reserved != 0 || rb->capacity < 1) return GDN_ERR_BAD_DIM;
    // The problem as the kernel sees it: k, v and the gates come from the buffer.
    gdn_problem pp = *p;
    pp.k = rb->k;
    pp.v = rb->v;
    pp.alpha = rb->alpha;
    pp.beta = rb->beta;
    const int64_t kv_rows = p->pool_slots * (int64_t)rb->capacity;
    const bool with_o = mode == gdn::kVerify;
    const bool with_acc = mode == gdn::kCommit;
    int algo = 0;
    bool empty = false;
    gdn_status st = validate(&pp, with_o, o, with_acc, accepted, &algo, &empty, kv_rows);
    if (st != GDN_OK) return st;
    if (algo != GDN_ALGO_CHUNK) return GDN_ERR_UNSUPPORTED;
    if (empty) return GDN_OK;
    if (rb->capacity < p->max_T || kv_rows > (1ll << 31)) return GDN_ERR_BAD_DIM;
    if (!rb->len_in || (with_acc && !rb->len_out)) return GDN_ERR_NULL_PTR;
    if (!aligned4(rb->len_in) || !aligned4(rb->len_out)) return GDN_ERR_ALIGN;
    if (with_acc) {
        const Range rl = range(rb->len_out, p->pool_slots * 4);
        const LayerRanges lr = layer_ranges(&pp, kv_rows);
        const Range others[] = {lr.q, lr.k, lr.v, lr.alpha, lr.beta, lr.pool,
                                range(rb->len_in, p->pool_slots * 4),
                                range(p->slot_ids, (int64_t)p->batch * 4),
                                range(p->cu_seqlens, p->cu_seqlens ? ((int64_t)p->batch + 1) * 4 : 0),
                                range(accepted, (int64_t)p->batch * 4),
                                range(p->dev_err, p->dev_err ? 4 : 0)};
        for (const Range &x : others)
            if (overlap(rl, x)) return GDN_ERR_ALIAS;
    }
    gdn::Args a = make_args(&pp, with_acc ? accepted : nullptr, with_o ? o : nullptr);
    a.cap = rb->capacity;
    a.kv_rows = kv_rows;
    a.len_in = rb->len_in;
    a.len_out = rb->len_out;
    const cudaError_t e = gdn::launch_chunk(&a, 1, mode, stream);
    if (e != cudaSuccess) {
        set_cuda_error(e, "kernel launch");
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}


// Commit-then-verify: `p` is this step (verify part), `prev` the previous step
// of the same requests (NULL: nothing to commit), `w` this call's W output.
gdn_status run_commit_verify(const gdn_problem *p, const gdn_prev_step *prev, void *o, float *w,
                             cudaStream_t stream) {
    int algo = 0;
    bool empty = false;
    gdn_status st = validate(p, true, o, false, nullptr, &algo, &empty);
    if (st != GDN_OK) return st;
    if (prev && prev->reserved != 0) return GDN_ERR_BAD_DIM;
    if (prev && (prev->max_T < 0 || (prev->cu_seqlens && prev->n_tok < 0))) return GDN_ERR_BAD_DIM;
    if (empty) return GDN_OK;
    // Single 16-token chunks on the mma.sync chunk kernel only.
    if (algo != GDN_ALGO_CHUNK || p->max_T > 16 || (prev && prev->max_T > 16))
        return GDN_ERR_UNSUPPORTED;
    if (!w) return GDN_ERR_NULL_PTR;
    if (!aligned16(w)) return GDN_ERR_ALIGN;
    const int64_t H = p->heads, n_tok = token_rows(p);
    const int64_t prows = prev ? (prev->cu_seqlens ? prev->n_tok : (int64_t)p->batch * prev->max_T) : 0;
    if (prev && prows > 0) {
        if (!prev->k || !prev->alpha || !prev->w || !prev->accepted) return GDN_ERR_NULL_PTR;
        if (!aligned16(prev->k) || !aligned16(prev->w) || !aligned4(prev->alpha) ||
            !aligned4(prev->accepted) || !aligned4(prev->cu_seqlens))
            return GDN_ERR_ALIGN;
    }
    // Aliasing: w is written, so it must not overlap anything else of the call;
    // the pool (written by the commit) must not overlap the previous step's arrays.
    const LayerRanges lr = layer_ranges(p);
    const Range rw = range(w, n_tok * H * p->dv * 4);
    const Range rp = lr.pool, ro = o_range(p, o);
    const Range pk = range(prev ? prev->k : nullptr, prows * H * p->dk * (p->qkv_dtype == GDN_BF16 ? 2 : 4));
    const Range pa = range(prev ? prev->alpha : nullptr, prows * H * 4);
    const Range pw = range(prev ? prev->w : nullptr, prows * H * p->dv * 4);
    const Range pacc = range(prev ? prev->accepted : nullptr, prev && prows > 0 ? (int64_t)p->batch * 4 : 0);
    const Range pcu = range(prev ? prev->cu_seqlens : nullptr,
                            prev && prev->cu_seqlens ? ((int64_t)p->batch + 1) * 4 : 0);
    const Range rs = range(p->slot_ids, (int64_t)p->batch * 4);
    const Range rc = range(p->cu_seqlens, p->cu_seqlens ? ((int64_t)p->batch + 1) * 4 : 0);
    const Range re = range(p->dev_err, p->dev_err ? 4 : 0);
    const Range all_w[] = {lr.q, lr.k, lr.v, lr.alpha, lr.beta, rp, ro, pk, pa, pw, pacc, pcu, rs, rc, re};
    for (const Range &x : all_w)
        if (overlap(rw, x)) return GDN_ERR_ALIAS;
    const Range prev_in[] = {pk, pa, pw, pacc, pcu};
    for (const Range &x : prev_in)
        if (overlap(rp, x) || overlap(ro, x)) return GDN_ERR_ALIAS;

    gdn::Args a = make_args(p, nullptr, o);
    a.w_out = w;
    if (prev && prows > 0) {
        a.p_cu = prev->cu_seqlens;
        a.p_maxT = prev->max_T;
        a.p_ntok = prows;
        a.p_k = prev->k;
        a.p_alpha = prev->alpha;
        a.p_w = prev->w;
        a.p_acc = prev->accepted;
    }
    const cudaError_t e = gdn::launch_chunk(&a, 1, gdn::kLagged, stream);
    if (e != cudaSuccess) {
        set_cuda_error(e, "kernel launch");
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_commit_verify(const gdn_problem *p, const gdn_prev_step *prev, void *o, float *w,
                             cudaStream_t stream) {
    return run_commit_verify(p, prev, o, w, stream);
}

gdn_status gdn_verify(const gdn_problem *p, void *o, cudaStream_t stream) {
    return run(p, gdn::kVerify, nullptr, o, stream);
}

gdn_status gdn_commit(const gdn_problem *p, const int32_t *accepted, cudaStream_t stream) {
    return run(p, gdn::kCommit, accepted, nullptr, stream);
}

gdn_status gdn_verify_commit_fused(const gdn_problem *p, const int32_t *accepted, void *o,
                                   cudaStream_t stream) {
    return run(p, gdn::kFused, accepted, o, stream);
}

gdn_status gdn_verify_layers(const gdn_problem *problems, int32_t n_layers, void *const *o,
                             cudaStream_t stream) {
    return run_layers(problems, n_layers, gdn::kVerify, nullptr, o, stream);
}

gdn_status gdn_commit_layers(const gdn_problem *problems, int32_t n_layers,
                             const int32_t *accepted, cudaStream_t stream) {
    return run_layers(problems, n_layers, gdn::kCommit, accepted, nullptr, stream);
}

gdn_status gdn_verify_commit_fused_layers(const gdn_problem *problems, int32_t n_layers,
                                          const int32_t *accepted, void *const *o,
                                          cudaStream_t stream) {
    return run_layers(problems, n_layers, gdn::kFused, accepted, o, stream);
}

gdn_status gdn_replay_verify(const gdn_problem *p, const gdn_replay *rb, void *o,
                             cudaStream_t stream) {
    return run_replay(p, rb, gdn::kVerify, nullptr, o, stream);
}

gdn_status gdn_replay_commit(const gdn_problem *p, const gdn_replay *rb, const int32_t *accepted,
                             cudaStream_t stream) {
    return run_replay(p, rb, gdn::kCommit, accepted, nullptr, stream);
}

gdn_status gdn_accept_prefix(int32_t batch, int32_t max_T, const int32_t *cu_seqlens,
                             int64_t n_tok, const int32_t *draft_ids, const int32_t *target_ids,
                             int32_t *accepted, int32_t *dev_err, cudaStream_t stream) {
    if (batch < 0 || max_T < 0 || max_T > GDN_MAX_T) return GDN_ERR_BAD_DIM;
    if (batch == 0) return GDN_OK;
    if (cu_seqlens && n_tok < 0) return GDN_ERR_BAD_DIM;
    if (!accepted) return GDN_ERR_NULL_PTR;
    const int64_t rows = cu_seqlens ? n_tok : (int64_t)batch * max_T;
    if (rows > 0 && (!draft_ids || !target_ids)) return GDN_ERR_NULL_PTR;
    if (!aligned4(cu_seqlens) || !aligned4(draft_ids) || !aligned4(target_ids) ||
        !aligned4(accepted) || !aligned4(dev_err))
        return GDN_ERR_ALIGN;
    const Range ra = range(accepted, (int64_t)batch * 4);
    const Range ins[] = {range(draft_ids, rows * 4), range(target_ids, rows * 4),
                         range(cu_seqlens, cu_seqlens ? ((int64_t)batch + 1) * 4 : 0),
                         range(dev_err, dev_err ? 4 : 0)};
    for (const Range &x : ins)
        if (overlap(ra, x)) return GDN_ERR_ALIAS;
    const cudaError_t e = gdn::launch_accept(batch, max_T, cu_seqlens, n_tok, draft_ids,
                                             target_ids, accepted, dev_err, stream);
    if (e != cudaSuccess) {
        set_cuda_error(e, "kernel launch");
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

gdn_status gdn_selftest_wait_timeout(int32_t *dev_err, cudaStream_t stream) {
    if (!dev_err) return GDN_ERR_NULL_PTR;
    if (!aligned4(dev_err)) return GDN_ERR_ALIGN;
    const cudaError_t e = gdn::launch_wait_selftest(dev_err, stream);
    if (e != cudaSuccess) {
        set_cuda_error(e, "kernel launch");
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

gdn_status gdn_read_device_error(const gdn_problem *p, cudaStream_t stream, int32_t *host_code) {
    if (!p || !host_code) return GDN_ERR_NULL_PTR;
    *host_code = 0;
    if (!p->dev_err) return GDN_OK;
    int32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, p->dev_err, sizeof(word), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        set_cuda_error(e, "gdn_read_device_error");
        return GDN_ERR_CUDA;
    }
    *host_code = word;
    return word ? GDN_ERR_DEVICE_ARG : GDN_OK;
}

int32_t gdn_select_algo(const gdn_problem *p) {
    // Shape-level checks only: pointers are not needed to pick a kernel.
    if (!p || !shape_ok(p)) return -1;
    if (p->qkv_dtype != GDN_FP32 && p->qkv_dtype != GDN_BF16) return -1;
    if (!dims_supported(p->dk, p->dv)) return -1;
    if (p->algo < GDN_ALGO_AUTO || p->algo > GDN_ALGO_CHUNK_TC) return -1;
    return resolve_algo(p);
}

const char *gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_NULL_PTR: return "a required pointer is NULL";
        case GDN_ERR_BAD_DIM: return "a size is out of range";
        case GDN_ERR_BAD_DTYPE: return "unknown q/k/v dtype";
        case GDN_ERR_UNSUPPORTED: return "shape or algo not supported";
        case GDN_ERR_DEVICE_ARG:
            return "a kernel reported a bad slot id, accepted length or sequence length";
        case GDN_ERR_CUDA: return "a CUDA call failed";
        case GDN_ERR_ALIGN: return "a pointer is not aligned (16 bytes for q/k/v/pool/o)";
        case GDN_ERR_ALIAS: return "an output overlaps an input";
        case GDN_ERR_LAYER_MISMATCH:
            return "the problems of a layer batch disagree on a request-level field";
    }
    return "unknown status";
}

const char *gdn_last_error_string(void) { return g_last_error; }

const char *gdn_version(void) { return "0.1.0"; }

}  // extern "C"
