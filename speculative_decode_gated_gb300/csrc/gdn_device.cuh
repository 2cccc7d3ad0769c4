// Shared device-side pieces of the Gated DeltaNet verify/commit kernels:
// the kernel argument block, per-unit metadata resolution with the
// device-side argument checks, and small load/convert helpers.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn.h"

namespace gdn {

// kLagged: commit the previous step's accepted prefix (from the W its call
// cached), then verify this step's drafts from the committed state.
enum Mode : int { kVerify = 0, kCommit = 1, kFused = 2, kLagged = 3 };

// Everything a kernel needs; a plain copy of gdn_problem plus the call's outputs.
struct Args {
    int B, H, dk, dv, max_T;
    long long n_tok;  // rows of the token arrays
    const int32_t *cu_seqlens;
    const void *q, *k, *v;
    const float *alpha, *beta;
    float *pool;
    long long pool_slots;
    const int32_t *slot_ids;
    const int32_t *accepted;  // NULL for verify
    void *o;                  // NULL for commit; float, or bf16 with GDN_FLAG_O_BF16
    int32_t *dev_err;
    int flags = 0;            // GDN_FLAG_* bits
    int tc = 0;               // chunk kernel: tcgen05 products (GDN_ALGO_CHUNK_TC)
    // ReplaySSM buffer (replay calls only; k, v, alpha, beta then point into
    // the buffer, whose rows are slot * cap + row).
    int cap = 0;              // rows per slot, 0 when there is no buffer
    long long kv_rows = 0;    // rows of k, v, alpha, beta: n_tok, or pool_slots * cap
    const int32_t *len_in = nullptr;
    int32_t *len_out = nullptr;
    // Commit-then-verify calls (kLagged): the previous step of the same requests.
    const int32_t *p_cu = nullptr;   // its row offsets [B+1], or NULL (uniform p_maxT rows)
    int p_maxT = 0;
    long long p_ntok = 0;            // rows of its arrays
    const void *p_k = nullptr;       // its k [p_ntok][H][dk]
    const float *p_alpha = nullptr;  // its alpha (or g) [p_ntok][H]
    const float *p_w = nullptr;      // the W its call wrote [p_ntok][H][dv]
    const int32_t *p_acc = nullptr;  // its accepted lengths [B]
    float *w_out = nullptr;          // this call's W [n_tok][H][dv]
};

// Token range, accepted length and state tile of one (request r, head h).
struct Unit {
    int row0;     // first token row
    int T;        // draft tokens T_r
    int a;        // accepted length (-1 in verify)
    float *tile;  // pool[slot_r][h], dk x dv
};

// A unit's metadata as loaded, before any check (so the loads can be issued
// well ahead of their first use).
struct RawMeta {
    int cu0, cu1;  // token rows [cu0, cu1)
    int slot;
    int acc;       // accepted length, -1 in verify
    // Commit-then-verify calls: the previous step's rows [pcu0, pcu1) and accepted length.
    int pcu0 = 0, pcu1 = 0, pacc = 0;
};

// Read-only loads that stay where they are written: issued early on purpose,
// their first use is an iteration later (the optimiser would otherwise sink
// them next to the use and expose their latency).
__device__ __forceinline__ int ld_early(const int32_t *ptr) {
    int v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(ptr));
    return v;
}
__device__ __forceinline__ float ld_early(const float *ptr) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
    return v;
}

__device__ __forceinline__ RawMeta load_meta(const Args &p, int r, int mode) {
    RawMeta m;
    if (p.cu_seqlens) {
        m.cu0 = ld_early(p.cu_seqlens + r);
        m.cu1 = ld_early(p.cu_seqlens + r + 1);
    } else {
        m.cu0 = r * p.max_T;
        m.cu1 = m.cu0 + p.max_T;
    }
    m.slot = ld_early(p.slot_ids + r);
    m.acc = mode != kVerify ? ld_early(p.accepted + r) : -1;
    return m;
}

// Applies the device-side checks to loaded metadata.  Only thread 0 of the
// block reports an error bit, so callers on other threads stay silent.
// Returns false when the unit must be skipped (nothing is written for it).
__device__ __forceinline__ bool check_meta(const Args &p, const RawMeta &m, int h, int mode,
                                           Unit &u) {
    int err = 0;
    u.row0 = m.cu0;
    u.T = m.cu1 - m.cu0;
    if (p.cu_seqlens && (u.T < 0 || u.T > p.max_T || u.row0 < 0 || (long long)m.cu1 > p.n_tok))
        err |= GDN_DEVERR_SEQLEN;
    if (m.slot < 0 || (long long)m.slot >= p.pool_slots) err |= GDN_DEVERR_SLOT;
    u.a = m.acc;
    if (mode != kVerify && !err && (u.a < 0 || u.a > u.T)) err |= GDN_DEVERR_ACCEPTED;
    if (err) {
        if (threadIdx.x == 0 && p.dev_err) atomicOr(p.dev_err, err);
        return false;
    }
    u.tile = p.pool + ((size_t)m.slot * p.H + h) * (size_t)p.dk * p.dv;
    return true;
}

// Reads the unit's metadata and applies the device-side checks.  Every thread
// of the block evaluates the same condition; thread 0 reports the error bit.
// Returns false when the unit must be skipped (nothing is written for it).
__device__ __forceinline__ bool resolve_unit(const Args &p, int r, int h, int mode, Unit &u) {
    return check_meta(p, load_meta(p, r, mode), h, mode, u);
}

// Hides a pointer's value from the optimiser, so addresses derived from it are
// recomputed where they are used instead of being kept live in registers.
template <typename T>
__device__ __forceinline__ T *opaque(T *ptr) {
    asm volatile("" : "+l"(ptr));
    return ptr;
}

// 8 bf16 (one 16-byte vector) -> 8 floats.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 &w, float *out) {
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        out[2 * e] = __uint_as_float(x[e] << 16);
        out[2 * e + 1] = __uint_as_float(x[e] & 0xFFFF0000u);
    }
}

}  // namespace gdn
