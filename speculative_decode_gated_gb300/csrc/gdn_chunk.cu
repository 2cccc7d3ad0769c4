// Chunked (WY) form of the gated delta rule for one block of up to 16 draft
// tokens, with the two state-sized products on tensor cores, as a persistent
// kernel with two resident blocks per SM, each of which loads its next unit's
// checkpoint tile and token block with TMA while it computes the current unit.
//
// With the tile H_0 (dk x dv, H = S^T), tokens t = 0..T-1 and
//   D[t][s] = prod_{s<r<=t} alpha_r        (D[t][t] = 1),   gamma_t = D[t][0] * alpha_0,
// the recurrence H_t = alpha_t H_{t-1} + k_t w_t^T, w_t = beta_t (v_t - alpha_t H_{t-1}^T k_t)
// unrolls to
//   P = H_0^T Q^T,  Z = H_0^T K^T                        (dv x T, tensor cores)
//   w_t = beta_t (v_t - gamma_t Z_t) - sum_{s<t} A[t][s] w_s,  A[t][s] = beta_t D[t][s] k_t.k_s
//   o_t = gamma_t P_t + sum_{s<=t} M[t][s] w_s,              M[t][s] = D[t][s] q_t.k_s
//   H_a = gamma_{a-1} H_0 + sum_{s<a} D[a-1][s] k_s w_s^T    (tensor cores)
// In matrix form, with Tinv = (I + A)^-1 (lower triangular, rows t >= T_r zeroed)
// and R = diag(beta) (V - diag(gamma) Z), both small solves are products:
//   W^T = R^T Tinv^T,   O^T = P^T diag(gamma) + W^T M^T          (tensor cores)
// Each value column j is independent given the token block, so warp w of a
// 4-warp block owns the 32 columns [32w, 32w + 32) of the unit (request r,
// head h); every product keeps the value columns as fragment rows, so the
// accumulator of one product is the A operand of the next without any
// shuffle or shared-memory transpose.
//
// Pipeline of one block (the block walks units blockIdx.x, + gridDim.x, ...):
//   * the 64 KiB tile stage is eight half-boxes (32 value columns x 64 key
//     rows), one mbarrier each: warp w reads only its own 32 columns, so it
//     waits only for its two half-boxes, and as soon as it has read the upper
//     (lower) half of its columns in the first product (and the products have
//     consumed the loaded values), its lane 0 issues the same half-box of the
//     next unit that has work into the freed space, behind a proxy fence; one
//     thread of warp 3 issues the 16-token boxes of its k, q and v rows into
//     the other of two token buffers when the current unit starts; all with
//     the 128-byte swizzle;
//   * before the wait on the previous kernel, thread 0 asks TMA to pull the
//     block's first unit into L2 (the only L2 prefetch: prefetches of later
//     units share the copy engine's queue with the loads that are needed
//     first, and measured slower);
//   * metadata is loaded three units ahead (mid-unit, not behind the stores)
//     and the gates one unit ahead, so no thread waits on a load it has just
//     issued.
// Waits on the TMA mbarriers are bounded (about 2 s by %globaltimer); on expiry
// the block reports GDN_DEVERR_TIMEOUT and stops after its copies have landed.
//
// Precision: q, k are bf16 (exact operands).  The fp32 operands (H_0 in the
// first product, the scaled w in the second) are split into bf16 hi + lo and
// both halves multiplied, with fp32 accumulation: about 16 mantissa bits per
// operand.  The triangular solve and the outputs run in fp32 on CUDA cores.
// Token rows past T_r (the next request's rows, or zero fill past the end) are
// loaded with the box but never reach a result: w_t for t >= T_r is set to 0 by
// selection, and every other use of those rows is multiplied by such a w_t.
//
// Fragment layout of H_0: lane (g = lane/4, c = lane%4) of warp w reads rows
// 16 kb + 2c + {0, 1, 8, 9} (kb = 0..7) and columns 32w + 4g + {0..3}.  This is
// at once the A-fragment layout of H_0^T for mma.m16n8k16 (value columns as
// rows: fragment row g <-> column 4g + 2m, row g + 8 <-> 4g + 2m + 1 in m-tile
// m) and the accumulator layout of H_a^T; with the 128-byte swizzle (16-byte
// chunk index XOR row % 8) the 16-byte shared loads are conflict-free, and the
// committed tile leaves as 16-byte stores with full 32-byte sectors.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_device.cuh"
#include "gdn_launch.h"
#include "gdn_wait.cuh"

namespace gdn {
namespace {

constexpr int CT = 16;   // token block
constexpr int D = 128;   // dk = dv
constexpr int kBlocksPerSM = 2;
constexpr uint32_t kBoxBytes = 32 * D * 4;        // one warp's columns: 32 value columns x 128 key rows
constexpr uint32_t kHalfBytes = kBoxBytes / 2;    // one TMA box: 32 value columns x 64 key rows
constexpr uint32_t kTileBytes = 4 * kBoxBytes;    // 64 KiB
constexpr uint32_t kTokHalfBytes = CT * 64 * 2;   // token box: 64 of 128 bf16 x 16 tokens
constexpr uint32_t kTokBytes = 2 * kTokHalfBytes; // one [16][128] bf16 tile

// Token tiles of one step, 1024-byte aligned, each a swizzled [16][128] bf16
// tile in two halves of 64 columns (one TMA box each).  The q and k halves of
// the same columns sit next to each other, so [q; k] is one 32-row operand of
// uniform row-group stride for the tensor cores.
constexpr uint32_t kQKStride = 2 * kTokHalfBytes;  // q/k: bytes from one column half to the next
struct TokBuf {
    unsigned char qk[2][2][kTokHalfBytes];  // [column half][0: q, 1: k]
    unsigned char v[kTokBytes];             // halves kTokHalfBytes apart
    unsigned char kp[kTokBytes];            // commit-then-verify: the previous step's k rows
    __device__ const unsigned char *q() const { return qk[0][0]; }
    __device__ const unsigned char *k() const { return qk[0][1]; }
};

struct Aux {
    float gram[2][CT][CT];  // [0][t][s] = k_t.k_s, [1][t][s] = q_t.k_s
    float A[CT][CT];        // beta_t D[t][s] k_t.k_s for s < t < T, else 0
    float M[CT][CT];        // D[t][s] q_t.k_s for s <= t, else 0
    float Tinv[CT][CT];     // (I + A)^-1, rows t >= T zeroed
    float alpha[CT], beta[CT], gamma[CT];
    float dcol[CT];         // D[a'-1][s] for s < a' (a' = the commit point within the chunk), else 0
    float dlast[CT];        // D[15][s]: the whole chunk's decay to its end
    // Commit-then-verify: the previous step's gates and its commit weights.
    float palpha[CT];       // alpha of its rows t < a_prev (1 beyond)
    float pdcol[CT];        // prod_{s<r<a_prev} alpha_r for s < a_prev, else 0
    float pgam;             // prod_{r<a_prev} alpha_r
    unsigned long long tile_full[4][2];  // [warp][key-row half]: that warp's columns of those rows
    unsigned long long tok_full[2];
    unsigned long long mma_full;  // tcgen05 products completed
    uint32_t tmem_base;           // TMEM address of this block's columns
    int abort_flag;
};

constexpr uint32_t kWpBoxBytes = 32 * CT * 4;  // W box: 32 value columns x 16 token rows
struct Smem {
    unsigned char tile[kTileBytes];
    TokBuf tok[2];
    unsigned char wprev[4 * kWpBoxBytes];  // commit-then-verify: the previous step's W rows
    Aux aux;
};
constexpr size_t kSmemBytes = 1024 + sizeof(Smem);
static_assert(sizeof(TokBuf) % 1024 == 0, "token buffers stay 1024-byte aligned");
static_assert(kBlocksPerSM * (kSmemBytes + 1024) <= 233472, "two blocks per SM");

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// fp32 pair -> bf16x2 hi and lo with x = hi + lo + O(2^-17 |x|).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ void mma(float &d0, float &d1, float &d2, float &d3, uint32_t a0,
                                    uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                              uint32_t &r3, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Byte offset of bf16 element (t, i) in a swizzled [16][128] token tile
// (two boxes of 64 columns, 128 bytes per token row).
// `half` = bytes from one column half to the next: kQKStride for q and k,
// kTokHalfBytes for v.
__device__ __forceinline__ uint32_t tok_off(int t, int i, uint32_t half) {
    return (uint32_t)((i >> 6) * half + t * 128 + ((((i & 63) >> 3) ^ (t & 7)) << 4) + (i & 7) * 2);
}

// Two adjacent bf16 of q or k (half stride kQKStride).
__device__ __forceinline__ uint32_t ld_tok32(const unsigned char *tile, int t, int i) {
    return *reinterpret_cast<const uint32_t *>(tile + tok_off(t, i, kQKStride));
}

// ------------------------------------------------------------ tcgen05 helpers
//
// Tensor memory (TMEM) of one block: 256 of the SM's 512 columns (two blocks
// per SM), 128 lanes of 32 bits each.  A TMEM address is (lane << 16) | column;
// warp w of the block reaches lanes [32w, 32w + 32) only, lane 32w + t from
// its thread t.
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmP = 0;      // P^T = H^T Q^T accumulator: 16 columns (one per token)
constexpr uint32_t kTmZ = 16;     // Z^T = H^T K^T accumulator: 16 columns
constexpr uint32_t kTmAhi = 32;   // A = H^T as bf16 hi, 64 columns (two key rows per column)
constexpr uint32_t kTmAlo = 96;   // A = H^T as bf16 lo, 64 columns
constexpr uint32_t kTmS = 32;     // state-update accumulator (128 columns, over A once it is used)
constexpr uint32_t kTmWhi = 160;  // (diag(d) W)^T as bf16 hi, 8 columns (two tokens per column)
constexpr uint32_t kTmWlo = 168;  // and lo

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(kTmemCols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// Thread t of warp w: 16 (or 8) consecutive 32-bit columns of lane 32w + t.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16};\n" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&f)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (16-byte units), version 1, 128-byte swizzle.  The
// matrices it describes are the TMA-written token tiles: rows of 128 bytes in
// 1024-byte groups of eight, 16-byte chunks XOR-swizzled by row % 8.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version
    d |= (uint64_t)2 << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 accumulator, A
// K-major (it comes from TMEM), B K-major or MN-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t umma_idesc(uint32_t n, bool b_mn_major) {
    return (1u << 4)                       // accumulator: f32
           | (1u << 7) | (1u << 10)        // A, B: bf16
           | ((b_mn_major ? 1u : 0u) << 16)
           | ((n >> 3) << 17)              // N / 8
           | ((128u >> 4) << 24);          // M / 16
}

// D (TMEM) = A (TMEM) B (shared memory) [+ D]: one 128 x N x 16 product, issued
// by one thread, completing asynchronously (see umma_commit).
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The mbarrier receives one arrival once every product issued before by this
// thread has completed (and its TMEM results are visible).
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                     bar)
                 : "memory");
}


// ------------------------------------------------------------ per-unit plan

struct UnitPlan {
    Unit u = {0, 0, -1, nullptr};  // u.row0: first row of k, v and the gates
    int h = 0;
    int layer = 0;  // which problem of the launch
    int tile = 0;   // slot * H + h: the tile's index in its layer's pool
    int teff = 0;   // rows that matter: T_r, or a_r for commit (replay: buffered rows too)
    int qrow0 = 0;  // row of q and o that goes with row u.row0
    int nskip = 0;  // rows before this one have no output (replay: the buffered rows)
    int slot = 0;
    int n = 0;      // replay: rows buffered in the slot (loaded with the plan)
    int prow0 = 0;  // commit-then-verify: the previous step's first row of the request
    int pa = 0;     // and its accepted length (0: nothing to commit)
    bool skip = true;
};

struct Maps {
    CUtensorMap pool, q, k, v;
    CUtensorMap kp;  // commit-then-verify: the previous step's k
    CUtensorMap wp;  // and the W its call cached
};

// One launch: NL problems that share every request-level field (batch, heads,
// lengths, slot ids, accepted lengths) and differ in their tokens, gates,
// outputs and pool.  Unit w of the launch is unit w % U of layer w / U.
template <int NL>
struct Launch {
    Maps maps[NL];
    Args a[NL];
    int n;  // layers in use, 1..NL
};

// Metadata of launch unit `w`, loaded unconditionally (the index is clamped to
// a valid one) so that no select or branch ever waits on these loads: they are
// consumed an iteration later, when the plan decides whether the unit exists.
template <int MODE, bool RAGGED, int NL>
__device__ __forceinline__ RawMeta load_unit_meta(const Args &p, int w, int W, int U) {
    const int wc = w < W ? w : W - 1;
    const int r = (NL == 1 ? wc : wc % U) / p.H;
    RawMeta m;
    if (RAGGED) {
        m.cu0 = ld_early(p.cu_seqlens + r);
        m.cu1 = ld_early(p.cu_seqlens + r + 1);
    } else {
        m.cu0 = r * p.max_T;
        m.cu1 = m.cu0 + p.max_T;
    }
    m.slot = ld_early(p.slot_ids + r);
    m.acc = (MODE == kCommit || MODE == kFused) ? ld_early(p.accepted + r) : -1;
    if (MODE == kLagged) {
        if (p.p_cu) {
            m.pcu0 = ld_early(p.p_cu + r);
            m.pcu1 = ld_early(p.p_cu + r + 1);
        } else {
            m.pcu0 = r * p.p_maxT;
            m.pcu1 = m.pcu0 + p.p_maxT;
        }
        m.pacc = p.p_acc ? ld_early(p.p_acc + r) : 0;
    }
    return m;
}

template <int MODE, int NL, bool REPLAY>
__device__ __forceinline__ UnitPlan plan_unit(const Launch<NL> &L, int w, int U, const RawMeta &m) {
    UnitPlan pl;
    pl.layer = NL == 1 ? 0 : w / U;
    const int unit = w - pl.layer * U;
    const Args &p = L.a[pl.layer];
    pl.h = unit - (unit / p.H) * p.H;
    bool ok = check_meta(p, m, pl.h, MODE == kLagged ? kVerify : MODE, pl.u);
    if (MODE == kLagged && ok && p.p_acc) {
        // The previous step: its rows must lie in its arrays, a_prev in [0, T_prev].
        const int pT = m.pcu1 - m.pcu0;
        int err = 0;
        if (p.p_cu && (pT < 0 || pT > p.p_maxT || m.pcu0 < 0 || (long long)m.pcu1 > p.p_ntok))
            err |= GDN_DEVERR_SEQLEN;
        else if (m.pacc < 0 || m.pacc > pT)
            err |= GDN_DEVERR_ACCEPTED;
        if (err) {
            if (threadIdx.x == 0 && p.dev_err) atomicOr(p.dev_err, err);
            ok = false;
        }
        pl.prow0 = m.pcu0;
        pl.pa = ok ? m.pacc : 0;
    }
    pl.tile = ok ? m.slot * p.H + pl.h : 0;
    pl.slot = ok ? m.slot : 0;
    pl.qrow0 = pl.u.row0;
    if (REPLAY) {
        // The buffered length is only loaded here; finalize_replay uses it one
        // iteration later, when this plan becomes the next unit.
        pl.n = ok ? ld_early(p.len_in + m.slot) : 0;
        pl.u.row0 = pl.slot * p.cap;
        pl.skip = !ok;
        return pl;
    }
    pl.teff = ok ? ((MODE == kCommit) ? pl.u.a : pl.u.T) : 0;
    // Commit-then-verify: a request with no new rows may still have a prefix to commit.
    pl.skip = !ok || (pl.teff == 0 && (MODE != kLagged || pl.pa == 0));
    return pl;
}

// Replay calls: the rows of a unit are its slot's buffer rows [0, n + T_r)
// (verify: outputs for rows n.., at q/o rows cu[r] + row - n) or [0, keep)
// with keep = n + a_r (commit: only when the slot is flushed, keep + max_T >
// cap).  The commit also records the slot's new buffered length (once, by the
// unit of head 0).  A unit whose rows leave the buffer reports
// GDN_DEVERR_REPLAY and is skipped.
template <int MODE>
__device__ __forceinline__ void finalize_replay(const Args &p, UnitPlan &pl, int tid) {
    if (pl.skip) return;  // its metadata was rejected (and reported) already
    const int n = pl.n;
    bool bad;
    if (MODE == kVerify) {
        bad = n < 0 || n + pl.u.T > p.cap;
        pl.teff = n + pl.u.T;
        pl.nskip = n;
        pl.qrow0 -= n;  // q and o rows of the drafts start at cu[r]
        pl.skip = bad || pl.u.T == 0;
    } else {
        const int keep = n + pl.u.a;
        bad = n < 0 || keep > p.cap;
        const bool flush = keep + p.max_T > p.cap;
        if (!bad && pl.h == 0 && tid == 0) p.len_out[pl.slot] = flush ? 0 : keep;
        pl.u.a = keep;
        pl.teff = flush ? keep : 0;
        pl.skip = bad || !flush || keep == 0;
    }
    if (bad && tid == 0 && p.dev_err) atomicOr(p.dev_err, GDN_DEVERR_REPLAY);
}

// One thread: the token boxes (k, v and, unless committing, q) of chunk `ch` of
// one unit: token rows row0 + 16 ch + [0, 16).
template <int MODE>
__device__ __forceinline__ void issue_tokens(const Maps &maps, const UnitPlan &pl, int ch,
                                             TokBuf &tb, uint32_t tok_bar) {
    const int row = pl.u.row0 + CT * ch;
    const int qrow = pl.qrow0 + CT * ch;  // may be negative (replay): those rows read as zero
    const bool prev = MODE == kLagged && pl.pa > 0;  // the previous step's k rows too
    mbar_arrive_expect_tx(tok_bar, (MODE == kCommit ? 2u : 3u) * kTokBytes + (prev ? kTokBytes : 0u));
    if (prev)
#pragma unroll
        for (int hb = 0; hb < 2; ++hb)
            tma_load_3d(smem_u32(tb.kp) + hb * kTokHalfBytes, &maps.kp, 64 * hb, pl.h, pl.prow0, tok_bar);
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
        tma_load_3d(smem_u32(tb.qk[hb][1]), &maps.k, 64 * hb, pl.h, row, tok_bar);
        tma_load_3d(smem_u32(tb.v) + hb * kTokHalfBytes, &maps.v, 64 * hb, pl.h, row, tok_bar);
        if (MODE != kCommit)
            tma_load_3d(smem_u32(tb.qk[hb][0]), &maps.q, 64 * hb, pl.h, qrow, tok_bar);
    }
}

// One thread: half-box `hf` (key rows 64 hf .. 64 hf + 63) of warp w's columns
// 32 w .. 32 w + 31 of one unit's tile, on barrier tile_full[w][hf].
// Commit-then-verify units with a prefix to commit also bring, with the upper
// half, warp w's columns of the previous step's W rows of the request (one box
// of 32 columns x 16 rows).
template <int MODE>
__device__ __forceinline__ void issue_tile_half(const Maps &maps, const UnitPlan &pl, int w, int hf,
                                                unsigned char *tile, uint32_t bar,
                                                unsigned char *wprev) {
    const bool wp = MODE == kLagged && pl.pa > 0 && hf == 0;
    mbar_arrive_expect_tx(bar, kHalfBytes + (wp ? kWpBoxBytes : 0u));
    tma_load_3d(smem_u32(tile) + w * kBoxBytes + hf * kHalfBytes, &maps.pool, 32 * w, 64 * hf,
                pl.tile, bar);
    if (wp) tma_load_3d(smem_u32(wprev) + w * kWpBoxBytes, &maps.wp, 32 * w, pl.h, pl.prow0, bar);
}

// One thread: all eight half-boxes of one unit (no part of the stage is in use).
template <int MODE>
__device__ __forceinline__ void issue_tile(const Maps &maps, const UnitPlan &pl, unsigned char *tile,
                                           Aux &ax, unsigned char *wprev);

// Lane 0 of warp w: both half-boxes of warp w's columns of one unit (that
// warp's part of the stage is not in use).
template <int MODE>
__device__ __forceinline__ void issue_warp_tile(const Maps &maps, const UnitPlan &pl, int w,
                                                unsigned char *tile, Aux &ax, unsigned char *wprev) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
        issue_tile_half<MODE>(maps, pl, w, hf, tile, smem_u32(&ax.tile_full[w][hf]), wprev);
}

template <int MODE>
__device__ __forceinline__ void issue_tile(const Maps &maps, const UnitPlan &pl, unsigned char *tile,
                                           Aux &ax, unsigned char *wprev) {
#pragma unroll
    for (int w = 0; w < 4; ++w) issue_warp_tile<MODE>(maps, pl, w, tile, ax, wprev);
}

// Read through L2 only (no L1 line is left behind), for the hints below.
__device__ __forceinline__ int ld_l2(const int32_t *ptr) {
    int v;
    asm volatile("ld.global.cg.b32 %0, [%1];" : "=r"(v) : "l"(ptr));
    return v;
}

// Thread 0, before the wait on the previous kernel of the stream: ask for the
// tile and token rows of this block's first unit in L2.  Prefetches change no
// memory, so issuing them early is safe even when the previous kernel is still
// writing what they touch (the real loads come after the wait and read the
// current data from L2).  The metadata read here may be stale for the same
// reason; it only picks addresses, clamped into the arrays, and is read again
// after the wait.
template <int MODE, bool RAGGED, int NL, bool REPLAY>
__device__ __forceinline__ void early_prefetch(const Launch<NL> &L, int w, int W, int U) {
    if (w >= W) return;
    const Args &p = L.a[0];
    const int layer = NL == 1 ? 0 : w / U;
    const int unit = w - layer * U;
    const int r = unit / p.H;
    const int h = unit - r * p.H;
    const int row0 = RAGGED ? ld_l2(p.cu_seqlens + r) : r * p.max_T;
    const int slot = ld_l2(p.slot_ids + r);
    const Maps &maps = L.maps[layer];
    const long long row = row0 < 0 ? 0 : (row0 >= p.n_tok ? p.n_tok - 1 : row0);
    const long long sl = slot < 0 ? 0 : (slot >= p.pool_slots ? p.pool_slots - 1 : slot);
    if (!REPLAY) {  // replay: the buffered length is not known yet, so the tile only
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            tma_prefetch_3d(&maps.k, 64 * hb, h, (int)row);
            tma_prefetch_3d(&maps.v, 64 * hb, h, (int)row);
            if (MODE != kCommit) tma_prefetch_3d(&maps.q, 64 * hb, h, (int)row);
        }
    }
#pragma unroll
    for (int b = 0; b < 8; ++b)
        tma_prefetch_3d(&maps.pool, 32 * (b & 3), 64 * (b >> 2), (int)(sl * p.H + h));
}

// Gate of token 16 ch + min(tid, left - 1) of a unit, left = the unit's tokens
// from chunk ch on (any clamped row when the unit is skipped or the token is
// past the end): always a valid address (the chunk kernel runs only with
// n_tok >= 1), so the load never sits behind a branch.
__device__ __forceinline__ float gate_load(const float *gate, const Args &p, const UnitPlan &pl,
                                           int ch, int tid) {
    const int left = pl.teff - CT * ch;
    long long row = (long long)pl.u.row0 + CT * ch + (tid < left ? tid : left - 1);
    row = row < 0 ? 0 : (row >= p.kv_rows ? p.kv_rows - 1 : row);
    const int h = pl.h < 0 ? 0 : (pl.h >= p.H ? p.H - 1 : pl.h);
    return ld_early(gate + (size_t)row * p.H + h);
}

// Commit-then-verify: the previous step's gate of its row min(tid, a_prev - 1)
// (1 when there is nothing to commit).
template <int MODE>
__device__ __forceinline__ float prev_gate_load(const Args &p, const UnitPlan &pl, int tid) {
    if (MODE != kLagged || pl.pa <= 0 || pl.skip) return 1.0f;
    long long row = (long long)pl.prow0 + (tid < pl.pa ? tid : pl.pa - 1);
    row = row < 0 ? 0 : (row >= p.p_ntok ? p.p_ntok - 1 : row);
    return ld_early(p.p_alpha + (size_t)row * p.H + pl.h);
}

// ------------------------------------------------------------ the kernel

// Four warps share one unit: warp w owns the 32 value columns [32w, 32w + 32),
// two m-tiles of 16 columns; lane (g, c) holds the 4 adjacent columns
// 32w + 4g + {0..3} (m-tile m: fragment row g is column 4g + 2m, row g + 8 is
// 4g + 2m + 1).
constexpr int NW = 4;
constexpr int kThreads = 32 * NW;
constexpr int CW = D / NW;       // 32 columns per warp
constexpr int MT = CW / 16;      // 2 m-tiles
constexpr int CPT = 2 * MT;      // 4 columns per lane
constexpr int kTinvLanes = CT / NW;  // Tinv columns per warp
// The thread that issues the token boxes (a copy issue may stall its warp for a
// while when the copy engine is busy; warp 0 issues the tcgen05 products).  The
// tile half-boxes are issued by lane 0 of the warp that reads them.
constexpr int kTokIssuer = 96;

// Columns CPT g + [0, CPT) of warp w's slice, key row `row`, from the swizzled tile.
__device__ __forceinline__ float4 ld_tile_row(const unsigned char *tile, int warp, int g, int row) {
    const int col = warp * CW + CPT * g;  // first column, 0..127
    const unsigned char *box = tile + (col >> 5) * kBoxBytes;
    const int chunk = (col & 31) >> 2;
    return *reinterpret_cast<const float4 *>(box + row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Key rows of this lane in iteration kb, element rr of a fragment: 16 kb + 2c + {0, 1, 8, 9}.
__device__ __forceinline__ int key_row(int kb, int c, int rr) {
    return 16 * kb + 2 * c + (rr & 1) + 8 * (rr >> 1);
}

// The weights of a rank-16 state update, (dvec . W)^T split into bf16 hi + lo
// A fragments: W in the accumulator layout of the W product (token
// 8 ntt + 2c + (e & 1), column col0 + 2m + (e >> 1)), dvec[s] = 0 for tokens
// not taken.
__device__ __forceinline__ void update_weights(const float (&wq)[MT][2][4], const float *dvec, int c,
                                               uint32_t (&ah)[MT][4], uint32_t (&al)[MT][4]) {
#pragma unroll
    for (int ntt = 0; ntt < 2; ++ntt) {
        const float d0 = dvec[8 * ntt + 2 * c], d1 = dvec[8 * ntt + 2 * c + 1];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            split2(d0 * wq[m][ntt][0], d1 * wq[m][ntt][1], ah[m][2 * ntt], al[m][2 * ntt]);
            split2(d0 * wq[m][ntt][2], d1 * wq[m][ntt][3], ah[m][2 * ntt + 1], al[m][2 * ntt + 1]);
        }
    }
}

// Key rows 16 kb .. 16 kb + 15 of the update H^T <- gam H^T + (dvec . W)^T K:
// `hv` holds those rows of H^T on entry (the A-fragment layout of H^T is also
// the accumulator layout of this product) and of the result on exit.
// `khalf`: bytes from one column half of the k tile to the next.
__device__ __forceinline__ void update_rows(float (&hv)[4][CPT], int kb, const uint32_t (&ah)[MT][4],
                                            const uint32_t (&al)[MT][4], float gam, uint32_t k_smem,
                                            uint32_t khalf, int lane) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
        for (int e = 0; e < CPT; ++e) hv[rr][e] *= gam;
    // ldmatrix.trans row address of this lane: matrix lane/8 -> (token half, dk half).
    const int mi = lane >> 3;
    const int krow = (lane & 7) + 8 * (mi & 1);
    uint32_t b00, b01, b10, b11;  // (n-tile 2kb: b0, b1), (n-tile 2kb+1: b0, b1)
    ldsm_x4_trans(b00, b01, b10, b11, k_smem + tok_off(krow, 16 * kb + 8 * (mi >> 1), khalf));
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        mma(hv[0][2 * m], hv[1][2 * m], hv[0][2 * m + 1], hv[1][2 * m + 1], ah[m][0], ah[m][1],
            ah[m][2], ah[m][3], b00, b01);
        mma(hv[2][2 * m], hv[3][2 * m], hv[2][2 * m + 1], hv[3][2 * m + 1], ah[m][0], ah[m][1],
            ah[m][2], ah[m][3], b10, b11);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        mma(hv[0][2 * m], hv[1][2 * m], hv[0][2 * m + 1], hv[1][2 * m + 1], al[m][0], al[m][1],
            al[m][2], al[m][3], b00, b01);
        mma(hv[2][2 * m], hv[3][2 * m], hv[2][2 * m + 1], hv[3][2 * m + 1], al[m][0], al[m][1],
            al[m][2], al[m][3], b10, b11);
    }
}

// This thread's four columns of key rows 16 kb .. 16 kb + 15 of a pool tile (16-byte stores).
__device__ __forceinline__ void store_rows(float *dst, int kb, int c, const float (&hv)[4][CPT]) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr)
        *reinterpret_cast<float4 *>(dst + key_row(kb, c, rr) * D) =
            make_float4(hv[rr][0], hv[rr][1], hv[rr][2], hv[rr][3]);
}

// The state after `dvec`-weighted tokens of the chunk, from the state in `hr`:
//   H^T <- gam H^T + (dvec . W)^T K       (dvec[s] = 0 for tokens not taken)
// STORE: the result goes to `dst` (this thread's columns of the pool tile);
// KEEP: it replaces `hr`.
template <bool STORE, bool KEEP>
__device__ __forceinline__ void state_update(float (&hr)[8][4][CPT], const float (&wq)[MT][2][4],
                                             const float *dvec, float gam, uint32_t k_smem,
                                             uint32_t khalf, int lane, int c, float *dst) {
    uint32_t ah[MT][4], al[MT][4];
    update_weights(wq, dvec, c, ah, al);
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
        float hv[4][CPT];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int e = 0; e < CPT; ++e) hv[rr][e] = hr[kb][rr][e];
        update_rows(hv, kb, ah, al, gam, k_smem, khalf, lane);
        if (STORE) store_rows(dst, kb, c, hv);
        if (KEEP)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                for (int e = 0; e < CPT; ++e) hr[kb][rr][e] = hv[rr][e];
    }
}

// MULTI: units may have more than 16 tokens (several chunks, the state carried
// in registers from one to the next); otherwise every unit is one chunk and
// the verify kernel keeps no state in registers.  VAR: the call's flags (bf16
// o, log-space gates) are read at run time; otherwise they are 0 at compile
// time, so the default calls carry no code for the variants.
//
// TC: the two state-sized products on tcgen05 (A = H^T in TMEM, accumulators in
// TMEM, one issuing thread) instead of mma.sync; the small solves and the
// outputs then run on CUDA cores with one value column per thread.
template <int MODE, bool RAGGED, int NL, bool MULTI, bool REPLAY, bool VAR, bool TC>
__global__ void __launch_bounds__(kThreads, kBlocksPerSM)
    chunk_kernel(const __grid_constant__ Launch<NL> L) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u));
    Aux &ax = sm.aux;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const Args &p = L.a[0];  // the request-level fields every layer shares
    const int flags = VAR ? p.flags : 0;
    const int U = p.B * p.H;  // units per layer
    const int W = NL == 1 ? U : U * L.n;  // units of the launch
    const int G = gridDim.x;
    const size_t row_stride = (size_t)p.H * D;
    const int col0 = warp * CW + CPT * g;  // this thread's first value column

    // Programmatic dependent launch: the next kernel on the stream may be
    // launched right away (its blocks become resident as ours exit and wait in
    // their own prologue), and this kernel issues only L2 prefetches until the
    // previous kernel on the stream has completed.  Stream order is kept.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            mbar_init(smem_u32(&ax.tile_full[w][0]), 1);
            mbar_init(smem_u32(&ax.tile_full[w][1]), 1);
        }
        mbar_init(smem_u32(&ax.tok_full[0]), 1);
        mbar_init(smem_u32(&ax.tok_full[1]), 1);
        mbar_init(smem_u32(&ax.mma_full), 1);
        ax.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
#pragma unroll
        for (int m = 0; m < 4; ++m)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&L.maps[0].pool + m))
                         : "memory");
    }
    if (TC && warp == 0) tmem_alloc(smem_u32(&ax.tmem_base));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = TC ? ax.tmem_base : 0u;           // lane 0, first column
    const uint32_t tl = tm + ((uint32_t)(32 * warp) << 16);  // this warp's first lane
    const uint32_t mma_bar = smem_u32(&ax.mma_full);
    int mma_phase = 0;
    const int j = 32 * warp + lane;  // tcgen05 path: this thread's value column
    if (tid == 0) early_prefetch<MODE, RAGGED, NL, REPLAY>(L, blockIdx.x, W, U);
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Plans: `cur` is the unit being computed, `nxt` the next one (its loads are
    // issued during `cur`), `raw` the metadata of the one after.
    // The metadata of the first three units is loaded at once (the loads are
    // independent), then the first unit's copies go out before anything else.
    int unit = blockIdx.x;  // launch unit
    UnitPlan cur, nxt;
    cur.skip = true;
    nxt.skip = true;
    // (Kernels for units of several chunks plan the units one after the other:
    // their state registers leave no room for three units' metadata at once.)
    RawMeta m1, raw;
    if (MULTI) {
        if (unit < W) {
            cur = plan_unit<MODE, NL, REPLAY>(L, unit, U, load_unit_meta<MODE, RAGGED, NL>(p, unit, W, U));
            if (REPLAY) finalize_replay<MODE>(L.a[cur.layer], cur, tid);
        }
        if (unit + G < W)
            nxt = plan_unit<MODE, NL, REPLAY>(L, unit + G, U,
                                              load_unit_meta<MODE, RAGGED, NL>(p, unit + G, W, U));
        raw = load_unit_meta<MODE, RAGGED, NL>(p, unit + 2 * G, W, U);
    } else {
        const RawMeta m0 = load_unit_meta<MODE, RAGGED, NL>(p, unit, W, U);
        m1 = load_unit_meta<MODE, RAGGED, NL>(p, unit + G, W, U);
        raw = load_unit_meta<MODE, RAGGED, NL>(p, unit + 2 * G, W, U);
        if (unit < W) {
            cur = plan_unit<MODE, NL, REPLAY>(L, unit, U, m0);
            if (REPLAY) finalize_replay<MODE>(L.a[cur.layer], cur, tid);
        }
    }

    // A step is one 16-token chunk of one unit.  Step k (in the order this block
    // computes them) uses token buffer k & 1; its token boxes go out when step
    // k-1 starts (that buffer was last used by step k-2).  A unit's tile goes
    // out half-box by half-box as the previous unit's first product consumes
    // its own (units of several chunks: after that product); later chunks
    // start from the state held in registers.
    int issued = 0;      // units whose tile load was issued
    int processed = 0;   // units whose tile was consumed
    int tok_issued = 0;  // steps whose token load was issued
    int steps = 0;       // steps computed
    if (!cur.skip) {
        // the first unit's token boxes (warp 3) and each warp's own half-boxes
        // (kernels for units of several chunks keep it on one thread: their state
        // registers leave no room for the spread issue)
        if (tid == kTokIssuer)
            issue_tokens<MODE>(L.maps[cur.layer], cur, 0, sm.tok[0], smem_u32(&ax.tok_full[0]));
        if (MULTI ? tid == 0 : lane == 0) {
            if (MULTI)
                issue_tile<MODE>(L.maps[cur.layer], cur, sm.tile, ax, sm.wprev);
            else
                issue_warp_tile<MODE>(L.maps[cur.layer], cur, warp, sm.tile, ax, sm.wprev);
        }
    }
    if (!MULTI && unit + G < W) nxt = plan_unit<MODE, NL, REPLAY>(L, unit + G, U, m1);
    if (!cur.skip) {
        ++issued;
        ++tok_issued;
    }
    // Gates of the next step: thread t < 16 holds alpha_t, beta_t, loaded
    // unconditionally from a clamped (always valid) row; rows t >= T are
    // replaced by alpha = 1, beta = 0 where the values are used.
    float ga = gate_load(L.a[cur.layer].alpha, p, cur, 0, tid);
    float gb = gate_load(L.a[cur.layer].beta, p, cur, 0, tid);
    // Commit-then-verify: the previous step's gate of the next unit (its row tid).
    float gpa = prev_gate_load<MODE>(L.a[cur.layer], cur, tid);

    // The unit's state as H^T in the A-fragment layout: the checkpoint tile,
    // then the state after each chunk (single-chunk verify needs none).
    // (commit-then-verify keeps none: its update is folded into the first product)
    constexpr bool kKeep = MULTI || MODE == kCommit || MODE == kFused;
    float hr[kKeep ? 8 : 1][4][CPT];  // mma.sync path (unused, and removed, on the tcgen05 path)
    // tcgen05 path: this thread's column of the state (key rows 0..127).
    float hcol[(kKeep && TC) ? D : 1];

    bool aborted = false;
    for (; unit < W; unit += G) {
        // Advance the metadata pipeline.
        const UnitPlan me = cur;
        cur = nxt;
        if (REPLAY) finalize_replay<MODE>(L.a[cur.layer], cur, tid);
        nxt.skip = true;
        if (unit + 2 * G < W) nxt = plan_unit<MODE, NL, REPLAY>(L, unit + 2 * G, U, raw);
        if (me.skip) {
            raw = load_unit_meta<MODE, RAGGED, NL>(p, unit + 3 * G, W, U);
            // Gates of the next unit (consumed one iteration later).
            ga = gate_load(L.a[cur.layer].alpha, p, cur, 0, tid);
            gb = gate_load(L.a[cur.layer].beta, p, cur, 0, tid);
            gpa = prev_gate_load<MODE>(L.a[cur.layer], cur, tid);
            if (!cur.skip && issued == processed) {
                // Nothing is in flight: the next unit's loads can all go now.
                if (tid == kTokIssuer)
                    issue_tokens<MODE>(L.maps[cur.layer], cur, 0, sm.tok[tok_issued & 1],
                                       smem_u32(&ax.tok_full[tok_issued & 1]));
                if (MULTI ? tid == 0 : lane == 0) {
                    if (MULTI)
                        issue_tile<MODE>(L.maps[cur.layer], cur, sm.tile, ax, sm.wprev);
                    else
                        issue_warp_tile<MODE>(L.maps[cur.layer], cur, warp, sm.tile, ax, sm.wprev);
                }
                ++issued;
                ++tok_issued;
            }
            continue;
        }
        // Commit-then-verify: the previous step's gate (thread t < 16: row t) and the
        // W its call cached for this thread's columns and rows t < a_prev (0 beyond),
        // in the accumulator layout of the W product (token 8 ntt + 2c + (e & 1),
        // column col0 + 2m + (e >> 1)); consumed after the tile wait.
        const int Tu = me.teff;  // tokens of the unit that matter: T_r, or a_r for commit
        const int nch = MULTI ? (Tu + CT - 1) / CT : 1;
        // The commit point: chunk `ca` holds token a_r - 1.
        const int ca = (MODE != kVerify && me.u.a > 0) ? (me.u.a - 1) / CT : -1;

        for (int ch = 0; ch < nch; ++ch) {
            const int T = Tu - CT * ch < CT ? Tu - CT * ch : CT;  // tokens of this chunk
            const bool more = MULTI && ch + 1 < nch;  // another chunk of this unit follows
            const TokBuf &tb = sm.tok[steps & 1];

            // 1. Gates into shared memory; token block arrival.
            fence_proxy_async_smem();  // reads of the token buffer refilled below come first
            __syncthreads();  // the previous step is done with the small matrices
            // The next step's token block goes into the other buffer now.
            if (tok_issued == steps + 1 && (more || !cur.skip)) {
                if (tid == kTokIssuer) {
                    TokBuf &nb = sm.tok[tok_issued & 1];
                    const uint32_t nbar = smem_u32(&ax.tok_full[tok_issued & 1]);
                    if (more)
                        issue_tokens<MODE>(L.maps[me.layer], me, ch + 1, nb, nbar);
                    else
                        issue_tokens<MODE>(L.maps[cur.layer], cur, 0, nb, nbar);
                }
                ++tok_issued;
            }
            if (tid < CT) {
                // A log-space gate becomes alpha = expf(g) here, once per token.
                const float at = (flags & GDN_FLAG_LOG_GATE) ? expf(ga) : ga;
                ax.alpha[tid] = tid < T ? at : 1.0f;
                ax.beta[tid] = tid < T ? gb : 0.0f;
                if (MODE == kLagged)
                    ax.palpha[tid] = tid < me.pa ? ((flags & GDN_FLAG_LOG_GATE) ? expf(gpa) : gpa) : 1.0f;
            }
            // Gates of the next step, loaded straight into the registers just
            // freed (consumed one step later, so this load is never waited on here).
            // A single-chunk unit loads the next unit's gates after its tile wait
            // instead, away from the stores the previous unit just issued.
            if (more) {
                ga = gate_load(L.a[me.layer].alpha, p, me, ch + 1, tid);
                gb = gate_load(L.a[me.layer].beta, p, me, ch + 1, tid);
            } else if (MULTI && ch > 0) {
                ga = gate_load(L.a[cur.layer].alpha, p, cur, 0, tid);
                gb = gate_load(L.a[cur.layer].beta, p, cur, 0, tid);
                gpa = prev_gate_load<MODE>(L.a[cur.layer], cur, tid);
            }
            if (!wait_parity(smem_u32(&ax.tok_full[steps & 1]), (steps >> 1) & 1))
                ax.abort_flag = 1;
            __syncthreads();
            if (ax.abort_flag) {
                aborted = true;
                break;
            }

            // 2. Gram blocks k_t.k_s and q_t.k_s: warp w computes matrix w / 2,
            //    columns 8 (w % 2) + [0, 8), over all 128 key dims.
            {
                const unsigned char *At = (warp >> 1) ? tb.q() : tb.k();
                const int nt = warp & 1;
                float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kb = 0; kb < 8; ++kb) {
                    const int col = 16 * kb + 2 * c;
                    float *acc = (kb & 1) ? a1 : a0;
                    mma(acc[0], acc[1], acc[2], acc[3], ld_tok32(At, g, col),
                        ld_tok32(At, g + 8, col), ld_tok32(At, g, col + 8),
                        ld_tok32(At, g + 8, col + 8), ld_tok32(tb.k(), 8 * nt + g, col),
                        ld_tok32(tb.k(), 8 * nt + g, col + 8));
                }
                float(*Gm)[CT] = ax.gram[warp >> 1];
                Gm[g][8 * nt + 2 * c] = a0[0] + a1[0];
                Gm[g][8 * nt + 2 * c + 1] = a0[1] + a1[1];
                Gm[g + 8][8 * nt + 2 * c] = a0[2] + a1[2];
                Gm[g + 8][8 * nt + 2 * c + 1] = a0[3] + a1[3];
            }
            __syncthreads();

            // 3. Decay products and the triangular matrices, 256 / kThreads (t, s) pairs per thread.
            {
                float al[CT];
#pragma unroll
                for (int r4 = 0; r4 < CT; r4 += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(&ax.alpha[r4]);
                    al[r4] = a4.x;
                    al[r4 + 1] = a4.y;
                    al[r4 + 2] = a4.z;
                    al[r4 + 3] = a4.w;
                }
                const int tc = ch == ca ? me.u.a - CT * ch - 1 : -1;  // commit row of this chunk
#pragma unroll
                for (int e2 = 0; e2 < CT * CT / kThreads; ++e2) {
                    const int e = tid + kThreads * e2;
                    const int t = e >> 4, s = e & 15;
                    float d = 1.0f;  // D[t][s] = prod_{s<r<=t} alpha_r
#pragma unroll
                    for (int r = 1; r < CT; ++r) d *= (r > s && r <= t) ? al[r] : 1.0f;
                    const float kk = ax.gram[0][t][s], qk = ax.gram[1][t][s];
                    ax.A[t][s] = (s < t && t < T) ? ax.beta[t] * d * kk : 0.0f;
                    ax.M[t][s] = (s <= t) ? d * qk : 0.0f;
                    if (s == 0) ax.gamma[t] = d * al[0];
                    if (MODE != kVerify && t == tc) ax.dcol[s] = (s <= t) ? d : 0.0f;
                    if (MULTI && t == CT - 1) ax.dlast[s] = d;
                }
                if (MODE == kLagged && tid <= CT) {
                    // The previous step's commit weights: pdcol[s] = prod_{s<r<a_prev} alpha_r
                    // (thread s < 16), pgam = prod_{r<a_prev} alpha_r (thread 16).
                    const int lo = tid < CT ? tid + 1 : 0;  // first factor's row
                    float d = 1.0f;
#pragma unroll
                    for (int r = 0; r < CT; ++r) d *= (r >= lo && r < me.pa) ? ax.palpha[r] : 1.0f;
                    if (tid < CT)
                        ax.pdcol[tid] = tid < me.pa ? d : 0.0f;
                    else
                        ax.pgam = d;
                }
            }
            __syncthreads();

            // 4. The checkpoint tile of this unit (first chunk only): the tcgen05
            //    path and units of several chunks wait here for the warp's two
            //    half-boxes; single-chunk units wait for each half where the first
            //    product reads it.  The metadata of the unit three ahead is loaded
            //    here, mid-unit: at the top of the loop these loads would queue
            //    behind the previous unit's stores.
            bool tile_ok = true;
            const uint32_t hbar0 = smem_u32(&ax.tile_full[warp][0]);
            const uint32_t hbar1 = smem_u32(&ax.tile_full[warp][1]);
            if (!MULTI || ch == 0) {
                if constexpr (TC || MULTI) {
                    // (units of several chunks read the whole tile into registers)
                    if (!wait_parity2(hbar0, hbar1, processed & 1)) ax.abort_flag = 1;
                    __syncthreads();
                    if (ax.abort_flag) {
                        aborted = true;
                        break;
                    }
                } else if (MODE == kLagged) {
                    // the previous step's W rows come with the upper half-box
                    tile_ok = mbar_try_wait(hbar0, processed & 1) || wait_parity(hbar0, processed & 1);
                }
                raw = load_unit_meta<MODE, RAGGED, NL>(p, unit + 3 * G, W, U);
                if (!more) {  // a single-chunk unit: the next unit's gates
                    ga = gate_load(L.a[cur.layer].alpha, p, cur, 0, tid);
                    gb = gate_load(L.a[cur.layer].beta, p, cur, 0, tid);
                    gpa = prev_gate_load<MODE>(L.a[cur.layer], cur, tid);
                }
            }

            // 4b. Commit-then-verify: the weights of the previous step's accepted
            //     prefix (its W, cached by its call and staged with the tile: box
            //     `warp`, row t, 128-byte swizzle), split for the tensor cores.  The
            //     update itself runs 16 key rows at a time inside the first product
            //     below, which then works on the committed state; each block of rows
            //     is written to the slot as it is made.
            uint32_t lah[MODE == kLagged ? MT : 1][4], lal[MODE == kLagged ? MT : 1][4];
            if constexpr (MODE == kLagged) {
                if (me.pa > 0) {
                    float wp[MT][2][4];  // token 8 ntt + 2c + (e & 1), column col0 + 2m + (e >> 1)
                    const unsigned char *wb = sm.wprev + warp * kWpBoxBytes;
#pragma unroll
                    for (int m = 0; m < MT; ++m)
#pragma unroll
                        for (int ntt = 0; ntt < 2; ++ntt)
#pragma unroll
                            for (int eo = 0; eo < 2; ++eo) {
                                const int t = 8 * ntt + 2 * c + eo;
                                const float2 x = *reinterpret_cast<const float2 *>(
                                    wb + t * 128 + ((g ^ (t & 7)) << 4) + 8 * m);
                                // rows past a_prev meet a zero weight; keep them finite
                                const bool live = t < me.pa;
                                wp[m][ntt][eo] = live ? x.x : 0.0f;
                                wp[m][ntt][2 + eo] = live ? x.y : 0.0f;
                            }
                    update_weights(wp, ax.pdcol, c, lah, lal);
                }
            }
            if constexpr (TC) {
                // 5. The state at the chunk's start as A = H^T in TMEM, bf16 hi and
                //    lo (thread t of warp w holds value column j = 32w + t: TMEM lane j,
                //    two key rows per 32-bit column), then, issued by thread 0 on the
                //    tensor cores: P^T = H^T Q^T and Z^T = H^T K^T (M = 128 value
                //    columns, N = 16 tokens, K = 128 key rows, hi and lo products).
                //    From the staged tile (first chunk) or from the state in registers.
                const bool outs = MODE != kCommit && (!REPLAY || CT * ch + T > me.nskip);
                {
                    const unsigned char *box = sm.tile + warp * kBoxBytes + (lane & 3) * 4;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t wh[16], wl[16];
#pragma unroll
                        for (int pp = 0; pp < 16; ++pp) {
                            const int i0 = 32 * q4 + 2 * pp;
                            float x0, x1;
                            if (!MULTI || ch == 0) {
                                x0 = *reinterpret_cast<const float *>(
                                    box + i0 * 128 + (((lane >> 2) ^ (i0 & 7)) << 4));
                                x1 = *reinterpret_cast<const float *>(
                                    box + (i0 + 1) * 128 + (((lane >> 2) ^ ((i0 + 1) & 7)) << 4));
                                if (kKeep) {
                                    hcol[kKeep ? i0 : 0] = x0;
                                    hcol[kKeep ? i0 + 1 : 0] = x1;
                                }
                            } else {
                                x0 = hcol[kKeep ? i0 : 0];
                                x1 = hcol[kKeep ? i0 + 1 : 0];
                            }
                            split2(x0, x1, wh[pp], wl[pp]);
                        }
                        tmem_st16(tl + kTmAhi + 16 * q4, wh);
                        tmem_st16(tl + kTmAlo + 16 * q4, wl);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                fence_proxy_async_smem();  // the reads of the stage come before its refill
                __syncthreads();
                // The tile is in TMEM (and registers): the stage is free for the next unit.
                if (!MULTI || ch == 0) {
                    ++processed;
                    if (!cur.skip) {
                        if (tid == 0) issue_tile<MODE>(L.maps[cur.layer], cur, sm.tile, ax, sm.wprev);
                        ++issued;
                    }
                }
                if (tid == 0) {
                    // [Q; K] (32 token rows: P and Z in one product) or K alone (16 rows).
                    tc_fence_after();
                    const uint32_t id = outs ? umma_idesc(32, false) : umma_idesc(16, false);
                    const uint32_t d = outs ? tm + kTmP : tm + kTmZ;
                    const uint32_t b0 = smem_u32(outs ? tb.qk[0][0] : tb.qk[0][1]);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t b = sw128_desc(b0 + (kk >> 2) * kQKStride + (kk & 3) * 32, 16, 1024);
                        umma_ts(d, tm + kTmAhi + 8 * kk, b, id, kk > 0 ? 1u : 0u);
                        umma_ts(d, tm + kTmAlo + 8 * kk, b, id, 1u);
                    }
                    umma_commit(mma_bar);
                }

                // While the products run: Tinv = (I + A)^-1 by forward substitution.
                // Lane groups compute column tj = w + 4 (lane % 4); the first 4 lanes
                // store it.  x_t = [t == tj, t < T] - sum_{s<t} A[t][s] x_s gives zeros
                // above the diagonal and in rows t >= T (A is zero there).
                {
                    const int tj = warp + NW * (lane % kTinvLanes);
                    float xt[CT];
#pragma unroll
                    for (int t = 0; t < CT; ++t) {
                        float acc = (t == tj && t < T) ? 1.0f : 0.0f;
#pragma unroll
                        for (int s4 = 0; s4 < t; s4 += 4) {
                            const float4 a4 = *reinterpret_cast<const float4 *>(&ax.A[t][s4]);
                            acc = fmaf(-a4.x, xt[s4], acc);
                            if (s4 + 1 < t) acc = fmaf(-a4.y, xt[s4 + 1], acc);
                            if (s4 + 2 < t) acc = fmaf(-a4.z, xt[s4 + 2], acc);
                            if (s4 + 3 < t) acc = fmaf(-a4.w, xt[s4 + 3], acc);
                        }
                        xt[t] = acc;
                        if (lane < kTinvLanes) ax.Tinv[t][tj] = acc;
                    }
                }
                const bool mma_ok = wait_parity(mma_bar, mma_phase & 1);
                ++mma_phase;
                if (__syncthreads_or(!mma_ok)) {  // also: Tinv is complete
                    aborted = true;
                    break;
                }
                tc_fence_after();
                float pz[CT], zz[CT];
                if (outs) tmem_ld16(tl + kTmP, pz);
                tmem_ld16(tl + kTmZ, zz);
                tmem_wait_ld();

                // 6. r_t = beta_t (v_t - gamma_t Z_t) for this thread's column (0 for t >= T);
                // 7. w = Tinv r (Tinv is zero above its diagonal and in rows t >= T).
                float w[CT];
                {
                    float r[CT];
#pragma unroll
                    for (int t = 0; t < CT; ++t) {
                        const uint32_t vb =
                            *reinterpret_cast<const unsigned short *>(tb.v + tok_off(t, j, kTokHalfBytes));
                        const float vt = __uint_as_float(vb << 16);
                        r[t] = t < T ? ax.beta[t] * (vt - ax.gamma[t] * zz[t]) : 0.0f;
                    }
#pragma unroll
                    for (int t = 0; t < CT; ++t) {
                        float acc = 0.0f;
#pragma unroll
                        for (int s4 = 0; s4 <= t; s4 += 4) {
                            const float4 a4 = *reinterpret_cast<const float4 *>(&ax.Tinv[t][s4]);
                            acc = fmaf(a4.x, r[s4], acc);
                            acc = fmaf(a4.y, r[s4 + 1], acc);
                            acc = fmaf(a4.z, r[s4 + 2], acc);
                            acc = fmaf(a4.w, r[s4 + 3], acc);
                        }
                        w[t] = acc;
                    }
                }

                // 8. o_t = gamma_t P_t + sum_{s<=t} M[t][s] w_s (M is zero above its
                //    diagonal); a warp stores 32 adjacent columns of one token row.
                if (MODE != kCommit && outs) {
                    const long long orow = (long long)me.qrow0 + CT * ch;
                    const bool o_bf16 = flags & GDN_FLAG_O_BF16;
                    float *go = static_cast<float *>(L.a[me.layer].o) + me.h * D + j;
                    __nv_bfloat16 *gob = static_cast<__nv_bfloat16 *>(L.a[me.layer].o) + me.h * D + j;
                    float ov[CT];  // all outputs first: no store sits between the M loads
#pragma unroll
                    for (int t = 0; t < CT; ++t) {
                        float acc = ax.gamma[t] * pz[t];
#pragma unroll
                        for (int s4 = 0; s4 <= t; s4 += 4) {
                            const float4 m4 = *reinterpret_cast<const float4 *>(&ax.M[t][s4]);
                            acc = fmaf(m4.x, w[s4], acc);
                            acc = fmaf(m4.y, w[s4 + 1], acc);
                            acc = fmaf(m4.z, w[s4 + 2], acc);
                            acc = fmaf(m4.w, w[s4 + 3], acc);
                        }
                        ov[t] = acc;
                    }
#pragma unroll
                    for (int t = 0; t < CT; ++t) {
                        if (t < T && CT * ch + t >= me.nskip) {
                            const size_t i = (size_t)(orow + t) * row_stride;
                            if (o_bf16)
                                gob[i] = __float2bfloat16_rn(ov[t]);
                            else
                                go[i] = ov[t];
                        }
                    }
                }

                // 9. The committed state (its chunk only), then the state after the
                //    whole chunk when another chunk follows:
                //      H^T <- gam H^T + (diag(dvec) W)^T K  (tensor cores: M = 128 value
                //      columns, N = 128 key rows, K = 16 tokens, K from its MN-major tile)
                const bool commit_here = MODE == kCommit ? !more : (MODE == kFused && ch == ca);
                if constexpr (kKeep) {
                    bool mma_failed = false;
#pragma unroll 1
                    for (int pass = 0; pass < 2; ++pass) {
                        const bool store = pass == 0;
                        if (store ? !commit_here : !more) continue;
                        const float *dvec = store ? ax.dcol : ax.dlast;
                        const float gam = store ? ax.gamma[me.u.a - CT * ch - 1] : ax.gamma[CT - 1];
                        {
                            uint32_t wh[8], wl[8];
#pragma unroll
                            for (int pp = 0; pp < 8; ++pp)
                                split2(dvec[2 * pp] * w[2 * pp], dvec[2 * pp + 1] * w[2 * pp + 1], wh[pp],
                                       wl[pp]);
                            tmem_st8(tl + kTmWhi, wh);
                            tmem_st8(tl + kTmWlo, wl);
                            tmem_wait_st();
                        }
                        tc_fence_before();
                        __syncthreads();
                        if (tid == 0) {
                            tc_fence_after();
                            constexpr uint32_t id128 = umma_idesc(128, true);
                            const uint64_t bk = sw128_desc(smem_u32(tb.qk[0][1]), kQKStride, 1024);
                            umma_ts(tm + kTmS, tm + kTmWhi, bk, id128, 0u);
                            umma_ts(tm + kTmS, tm + kTmWlo, bk, id128, 1u);
                            umma_commit(mma_bar);
                        }
                        const bool ok2 = wait_parity(mma_bar, mma_phase & 1);
                        ++mma_phase;
                        if (__syncthreads_or(!ok2)) {
                            mma_failed = true;
                            break;
                        }
                        tc_fence_after();
                        float *dst = opaque(me.u.tile) + j;
#pragma unroll
                        for (int q8 = 0; q8 < 8; ++q8) {
                            float sv[16];
                            tmem_ld16(tl + kTmS + 16 * q8, sv);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int i = 16 * q8 + e;
                                const float hv = fmaf(gam, hcol[kKeep ? i : 0], sv[e]);
                                if (store)
                                    dst[i * D] = hv;
                                else
                                    hcol[kKeep ? i : 0] = hv;
                            }
                        }
                    }
                    if (mma_failed) {
                        aborted = true;
                        break;
                    }
                }
                ++steps;
                continue;
            }

            // 5. P = H^T Q^T and Z = H^T K^T for this warp's columns, H the state at
            //    the chunk's start (N-tiles: Q 0-7, Q 8-15, K 0-7, K 8-15; commit
            //    needs only Z).  Interleaved with the products (it only needs A,
            //    finished above): Tinv = (I + A)^-1 by forward substitution, rows
            //    2kb and 2kb+1 in iteration kb.  Lane groups compute column
            //    j = w + 4 (lane % 4); the first 4 lanes store it.
            //    x_t = [t == j, t < T] - sum_{s<t} A[t][s] x_s gives zeros above
            //    the diagonal and in rows t >= T (A is zero there).
            constexpr int NT0 = (MODE == kCommit) ? 2 : 0;
            // Replay: a chunk of buffered rows only has no outputs (no P, no O).
            const bool outs = MODE != kCommit && (!REPLAY || CT * ch + T > me.nskip);
            const int tj = warp + NW * (lane % kTinvLanes);
            float xt[CT];
            float y[MT][4][4];
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) y[m][nt][e] = 0.0f;
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
                for (int t = 2 * kb; t < 2 * kb + 2; ++t) {
                    float acc = (t == tj && t < T) ? 1.0f : 0.0f;
#pragma unroll
                    for (int s4 = 0; s4 < t; s4 += 4) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(&ax.A[t][s4]);
                        acc = fmaf(-a4.x, xt[s4], acc);
                        if (s4 + 1 < t) acc = fmaf(-a4.y, xt[s4 + 1], acc);
                        if (s4 + 2 < t) acc = fmaf(-a4.z, xt[s4 + 2], acc);
                        if (s4 + 3 < t) acc = fmaf(-a4.w, xt[s4 + 3], acc);
                    }
                    xt[t] = acc;
                    if (lane < kTinvLanes) ax.Tinv[t][tj] = acc;
                }
                float hv[4][CPT];
                if (!MULTI || ch == 0) {
                    // This warp's half-box of these rows: wait for it at the first
                    // rows of each half (it goes to the next unit after the products
                    // of the half's last rows, below).
                    if (!MULTI && (kb & 3) == 0 && (MODE != kLagged || kb == 4)) {
                        const uint32_t hb = kb == 0 ? hbar0 : hbar1;
                        tile_ok = (mbar_try_wait(hb, processed & 1) || wait_parity(hb, processed & 1)) &&
                                  tile_ok;
                    }
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr) {
                        const float4 x = ld_tile_row(sm.tile, warp, g, key_row(kb, c, rr));
                        hv[rr][0] = x.x;
                        hv[rr][1] = x.y;
                        hv[rr][2] = x.z;
                        hv[rr][3] = x.w;
                        if (kKeep)
#pragma unroll
                            for (int e = 0; e < CPT; ++e) hr[kKeep ? kb : 0][rr][e] = hv[rr][e];
                    }
                } else {
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                        for (int e = 0; e < CPT; ++e) hv[rr][e] = hr[kKeep ? kb : 0][rr][e];
                }
                if constexpr (MODE == kLagged) {
                    // These rows of the committed state, written to the slot, then used.
                    if (me.pa > 0) {
                        update_rows(hv, kb, lah, lal, ax.pgam, smem_u32(tb.kp), kTokHalfBytes, lane);
                        if (tile_ok) store_rows(opaque(me.u.tile) + col0, kb, c, hv);
                    }
                }
                uint32_t b[4][2];
#pragma unroll
                for (int nt = NT0; nt < 4; ++nt) {
                    const unsigned char *Bt = nt < 2 ? tb.q() : tb.k();
                    const int tok = 8 * (nt & 1) + g;
                    b[nt][0] = ld_tok32(Bt, tok, 16 * kb + 2 * c);
                    b[nt][1] = ld_tok32(Bt, tok, 16 * kb + 2 * c + 8);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint32_t ah[4], al[4];
                    split2(hv[0][2 * m], hv[1][2 * m], ah[0], al[0]);
                    split2(hv[0][2 * m + 1], hv[1][2 * m + 1], ah[1], al[1]);
                    split2(hv[2][2 * m], hv[3][2 * m], ah[2], al[2]);
                    split2(hv[2][2 * m + 1], hv[3][2 * m + 1], ah[3], al[3]);
#pragma unroll
                    for (int nt = NT0; nt < 4; ++nt) {
                        if (nt < 2 && !outs) continue;
                        mma(y[m][nt][0], y[m][nt][1], y[m][nt][2], y[m][nt][3], ah[0], ah[1], ah[2],
                            ah[3], b[nt][0], b[nt][1]);
                    }
#pragma unroll
                    for (int nt = NT0; nt < 4; ++nt) {
                        if (nt < 2 && !outs) continue;
                        mma(y[m][nt][0], y[m][nt][1], y[m][nt][2], y[m][nt][3], al[0], al[1], al[2],
                            al[3], b[nt][0], b[nt][1]);
                    }
                }
                // The last rows of a half-box are consumed (the products above used
                // them): hand this warp's half-box to the next unit.  The proxy fence
                // orders each lane's shared-memory reads of it before the copy that
                // overwrites it.  (Units of several chunks keep their state in
                // registers through the loop; they send the next tile after it.)
                if (!MULTI && (kb & 3) == 3 && !cur.skip) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && tile_ok)
                        issue_tile_half<MODE>(L.maps[cur.layer], cur, warp, kb >> 2, sm.tile,
                                              kb == 3 ? hbar0 : hbar1, sm.wprev);
                }
            }

            // Tinv is complete.  After the first chunk the tile is in registers,
            // and every warp has sent (or, for units of several chunks, now sends)
            // its half-boxes of the next unit's tile.
            if (MULTI) {
                if (ch == 0) fence_proxy_async_smem();
                __syncthreads();
            } else if (__syncthreads_or(!tile_ok)) {
                aborted = true;
                break;
            }
            if (!MULTI || ch == 0) {
                ++processed;
                if (MULTI && !cur.skip && tid == 0)
                    issue_tile<MODE>(L.maps[cur.layer], cur, sm.tile, ax, sm.wprev);
                if (!cur.skip) ++issued;
            }

            // Token indices of this thread in the fragments: n-tile half ntt, element e:
            //   t = 8 ntt + 2c + (e & 1);   column = col0 + 2m + (e >> 1).
            // 6. R^T = beta_t (v_t - gamma_t Z_t), zero for t >= T.
            float rr_[MT][2][4];
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int ntt = 0; ntt < 2; ++ntt)
#pragma unroll
                    for (int eo = 0; eo < 2; ++eo) {
                        const int t = 8 * ntt + 2 * c + eo;
                        const uint32_t vv =
                            *reinterpret_cast<const uint32_t *>(tb.v + tok_off(t, col0 + 2 * m, kTokHalfBytes));
                        const float v0 = __uint_as_float(vv << 16);
                        const float v1 = __uint_as_float(vv & 0xFFFF0000u);
                        const float bt = ax.beta[t], gt = ax.gamma[t];
                        const bool live = t < T;
                        rr_[m][ntt][eo] = live ? bt * (v0 - gt * y[m][2 + ntt][eo]) : 0.0f;
                        rr_[m][ntt][2 + eo] = live ? bt * (v1 - gt * y[m][2 + ntt][2 + eo]) : 0.0f;
                    }

            // 7. W^T = R^T Tinv^T: A = R^T (accumulator layout, split), B = Tinv^T (split).
            float wq[MT][2][4];
            {
                uint32_t bh[2][2], bl[2][2];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float *tr = ax.Tinv[8 * nt + g];
                    split2(tr[2 * c], tr[2 * c + 1], bh[nt][0], bl[nt][0]);
                    split2(tr[2 * c + 8], tr[2 * c + 9], bh[nt][1], bl[nt][1]);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint32_t ah[4], al[4];
                    split2(rr_[m][0][0], rr_[m][0][1], ah[0], al[0]);
                    split2(rr_[m][0][2], rr_[m][0][3], ah[1], al[1]);
                    split2(rr_[m][1][0], rr_[m][1][1], ah[2], al[2]);
                    split2(rr_[m][1][2], rr_[m][1][3], ah[3], al[3]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        float *d = wq[m][nt];
                        d[0] = d[1] = d[2] = d[3] = 0.0f;
                        mma(d[0], d[1], d[2], d[3], ah[0], ah[1], ah[2], ah[3], bh[nt][0], bh[nt][1]);
                        mma(d[0], d[1], d[2], d[3], ah[0], ah[1], ah[2], ah[3], bl[nt][0], bl[nt][1]);
                        mma(d[0], d[1], d[2], d[3], al[0], al[1], al[2], al[3], bh[nt][0], bh[nt][1]);
                    }
                }
            }

            // 7b. Commit-then-verify: W of this step's drafts, cached for the next call's
            //     commit (same layout as o: [row][head][column], rows t < T only).
            if constexpr (MODE == kLagged) {
                float *gw = L.a[me.layer].w_out + me.h * D + col0;
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int ntt = 0; ntt < 2; ++ntt)
#pragma unroll
                        for (int eo = 0; eo < 2; ++eo) {
                            const int t = 8 * ntt + 2 * c + eo;
                            if (t < T)
                                *reinterpret_cast<float2 *>(gw + (size_t)(me.u.row0 + t) * row_stride + 2 * m) =
                                    make_float2(wq[m][ntt][eo], wq[m][ntt][2 + eo]);
                        }
            }

            // 8. O^T = P^T diag(gamma) + W^T M^T, stored as float2 pairs of adjacent columns.
            if (MODE != kCommit && outs) {
                uint32_t bh[2][2], bl[2][2];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float *mr = ax.M[8 * nt + g];
                    split2(mr[2 * c], mr[2 * c + 1], bh[nt][0], bl[nt][0]);
                    split2(mr[2 * c + 8], mr[2 * c + 9], bh[nt][1], bl[nt][1]);
                }
                // Row t of this chunk is output row qrow0 + 16 ch + t; rows before
                // nskip (replay: buffered rows) have none.
                const long long orow = (long long)me.qrow0 + CT * ch;
                const bool o_bf16 = flags & GDN_FLAG_O_BF16;
                float *go = static_cast<float *>(L.a[me.layer].o) + me.h * D + col0;
                __nv_bfloat16 *gob = static_cast<__nv_bfloat16 *>(L.a[me.layer].o) + me.h * D + col0;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint32_t ah[4], al[4];
                    split2(wq[m][0][0], wq[m][0][1], ah[0], al[0]);
                    split2(wq[m][0][2], wq[m][0][3], ah[1], al[1]);
                    split2(wq[m][1][0], wq[m][1][1], ah[2], al[2]);
                    split2(wq[m][1][2], wq[m][1][3], ah[3], al[3]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int t0 = 8 * nt + 2 * c;
                        const float g0 = ax.gamma[t0], g1 = ax.gamma[t0 + 1];
                        float d[4] = {g0 * y[m][nt][0], g1 * y[m][nt][1], g0 * y[m][nt][2],
                                      g1 * y[m][nt][3]};
                        mma(d[0], d[1], d[2], d[3], ah[0], ah[1], ah[2], ah[3], bh[nt][0], bh[nt][1]);
                        mma(d[0], d[1], d[2], d[3], ah[0], ah[1], ah[2], ah[3], bl[nt][0], bl[nt][1]);
                        mma(d[0], d[1], d[2], d[3], al[0], al[1], al[2], al[3], bh[nt][0], bh[nt][1]);
                        if (t0 < T && CT * ch + t0 >= me.nskip) {
                            const size_t i = (orow + t0) * row_stride + 2 * m;
                            if (o_bf16)
                                *reinterpret_cast<__nv_bfloat162 *>(gob + i) =
                                    __floats2bfloat162_rn(d[0], d[2]);
                            else
                                *reinterpret_cast<float2 *>(go + i) = make_float2(d[0], d[2]);
                        }
                        if (t0 + 1 < T && CT * ch + t0 + 1 >= me.nskip) {
                            const size_t i = (orow + t0 + 1) * row_stride + 2 * m;
                            if (o_bf16)
                                *reinterpret_cast<__nv_bfloat162 *>(gob + i) =
                                    __floats2bfloat162_rn(d[1], d[3]);
                            else
                                *reinterpret_cast<float2 *>(go + i) = make_float2(d[1], d[3]);
                        }
                    }
                }
            }

            // 9. The committed state (its chunk only), then the state after the
            //    whole chunk when another chunk follows.  A commit covers exactly
            //    the chunks up to the commit point, so there the two never meet.
            const bool commit_here = MODE == kCommit ? !more : (MODE == kFused && ch == ca);
            if constexpr (kKeep) {
                if (commit_here)
                    state_update<true, false>(hr, wq, ax.dcol, ax.gamma[me.u.a - CT * ch - 1],
                                              smem_u32(tb.k()), kQKStride, lane, c,
                                              opaque(me.u.tile) + col0);
                if (more)
                    state_update<false, true>(hr, wq, ax.dlast, ax.gamma[CT - 1], smem_u32(tb.k()),
                                              kQKStride, lane, c, nullptr);
            }
            ++steps;
        }
        if (aborted) break;
    }

    // Copies still in flight must land before the block exits.
    if (tid == 0) {
        bool ok = true;
        if (issued > processed)
            for (int b = 0; b < 8; ++b)
                ok = wait_parity(smem_u32(&ax.tile_full[b & 3][b >> 2]), processed & 1) && ok;
        for (int k = steps; k < tok_issued; ++k)
            ok = wait_parity(smem_u32(&ax.tok_full[k & 1]), (k >> 1) & 1) && ok;
        if (!ok) aborted = true;
    }
    if (tid == 0 && aborted)
        for (int l = 0; l < (NL == 1 ? 1 : L.n); ++l)
            if (L.a[l].dev_err) atomicOr(L.a[l].dev_err, GDN_DEVERR_TIMEOUT);
    if (TC) {
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tm);
    }
}

// ------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// A [rows][H][128] bf16 token array as a 3-D tensor (dk, head, row); boxes of
// 64 dk x 1 head x 16 rows, 128-byte swizzle.  Rows past `rows` read as zero.
bool encode_tokens(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *map, const void *base,
                   int H, long long rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)CT};
    const cuuint32_t elem[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int sms = 0;
    bool smem_set[4][2][2][2][2][2][2] = {};  // [mode][ragged][batched][multi][replay][var][tc]
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

static_assert(sizeof(Launch<kChunkMaxLayers>) <= 32764, "kernel parameter space");

template <int MODE, bool RAGGED, int NL, bool MULTI, bool REPLAY = false, bool VAR = false,
          bool TC = false>
cudaError_t launch_mode(const Launch<NL> &L, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        DeviceInfo &info = g_dev[dev];
        if (info.sms == 0) {
            e = cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
        }
        if (!info.smem_set[MODE][RAGGED][NL != 1][MULTI][REPLAY][VAR][TC]) {
            e = cudaFuncSetAttribute(chunk_kernel<MODE, RAGGED, NL, MULTI, REPLAY, VAR, TC>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
            if (e != cudaSuccess) return e;
            info.smem_set[MODE][RAGGED][NL != 1][MULTI][REPLAY][VAR][TC] = true;
        }
        sms = info.sms;
    }
    const long long units = (long long)L.a[0].B * L.a[0].H * L.n;
    const int slots = kBlocksPerSM * sms;
    const int grid = units < slots ? (int)units : slots;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chunk_kernel<MODE, RAGGED, NL, MULTI, REPLAY, VAR, TC>, L);
}

// The pool and token tensor maps of one layer.
cudaError_t encode_layer(const Args &p, Maps *maps) {
    const unsigned long long tiles = (unsigned long long)p.pool_slots * (unsigned long long)p.H;
    if (tiles == 0 || tiles > (1ull << 31) || p.n_tok < 1 || p.n_tok > (1ll << 31) ||
        p.kv_rows < 1 || p.kv_rows > (1ll << 31))
        return cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    // The pool as a 3-D tensor: value column (contiguous), key row, slot * H + head.
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)D, (cuuint64_t)tiles};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)D * D * 4};
    const cuuint32_t box[3] = {32, (cuuint32_t)D / 2, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    if (encode(&maps->pool, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.pool, dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (!encode_tokens(encode, &maps->k, p.k, p.H, p.kv_rows) ||
        !encode_tokens(encode, &maps->v, p.v, p.H, p.kv_rows) ||
        // A commit reads no q and may pass none: k stands in for the unused map.
        !encode_tokens(encode, &maps->q, p.q ? p.q : p.k, p.H, p.q ? p.n_tok : p.kv_rows))
        return cudaErrorInvalidValue;
    if (p.p_k && !encode_tokens(encode, &maps->kp, p.p_k, p.H, p.p_ntok))  // the previous step's k
        return cudaErrorInvalidValue;
    if (p.p_w) {  // the previous step's W: [rows][H][dv] fp32, boxes of 32 columns x 16 rows
        const cuuint64_t wdims[3] = {(cuuint64_t)D, (cuuint64_t)p.H, (cuuint64_t)p.p_ntok};
        const cuuint64_t wstrides[2] = {(cuuint64_t)D * 4, (cuuint64_t)p.H * D * 4};
        const cuuint32_t wbox[3] = {32, 1, (cuuint32_t)CT};
        if (encode(&maps->wp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(p.p_w), wdims,
                   wstrides, wbox, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <int NL, bool MULTI>
cudaError_t dispatch(const Launch<NL> &L, int mode, bool ragged, cudaStream_t stream) {
    switch (mode) {
        case kVerify:
            return ragged ? launch_mode<kVerify, true, NL, MULTI>(L, stream)
                          : launch_mode<kVerify, false, NL, MULTI>(L, stream);
        case kCommit:
            return ragged ? launch_mode<kCommit, true, NL, MULTI>(L, stream)
                          : launch_mode<kCommit, false, NL, MULTI>(L, stream);
        default:
            return ragged ? launch_mode<kFused, true, NL, MULTI>(L, stream)
                          : launch_mode<kFused, false, NL, MULTI>(L, stream);
    }
}

template <int NL>
cudaError_t launch_layers(const Args *layers, int n, int mode, cudaStream_t stream) {
    Launch<NL> L = {};
    L.n = n;
    for (int l = 0; l < n; ++l) {
        L.a[l] = layers[l];
        const cudaError_t e = encode_layer(layers[l], &L.maps[l]);
        if (e != cudaSuccess) return e;
    }
    const bool ragged = layers[0].cu_seqlens != nullptr;
    if constexpr (NL == 1) {
        if (mode == kLagged) {  // commit-then-verify: single chunks, mma.sync products
            if (layers[0].max_T > CT || layers[0].p_maxT > CT || layers[0].tc || layers[0].cap > 0)
                return cudaErrorNotSupported;
            if (layers[0].flags != 0)
                return ragged ? launch_mode<kLagged, true, NL, false, false, true>(L, stream)
                              : launch_mode<kLagged, false, NL, false, false, true>(L, stream);
            return ragged ? launch_mode<kLagged, true, NL, false>(L, stream)
                          : launch_mode<kLagged, false, NL, false>(L, stream);
        }
        if (layers[0].cap > 0) {  // replay buffer (single problems): verify or commit
            if (mode == kVerify)
                return ragged ? launch_mode<kVerify, true, NL, true, true, true>(L, stream)
                              : launch_mode<kVerify, false, NL, true, true, true>(L, stream);
            return ragged ? launch_mode<kCommit, true, NL, true, true, true>(L, stream)
                          : launch_mode<kCommit, false, NL, true, true, true>(L, stream);
        }
        if (layers[0].tc) {  // tcgen05 products (opt-in): one multi-chunk instantiation per mode
            switch (mode) {
                case kVerify:
                    return ragged ? launch_mode<kVerify, true, NL, true, false, true, true>(L, stream)
                                  : launch_mode<kVerify, false, NL, true, false, true, true>(L, stream);
                case kCommit:
                    return ragged ? launch_mode<kCommit, true, NL, true, false, true, true>(L, stream)
                                  : launch_mode<kCommit, false, NL, true, false, true, true>(L, stream);
                default:
                    return ragged ? launch_mode<kFused, true, NL, true, false, true, true>(L, stream)
                                  : launch_mode<kFused, false, NL, true, false, true, true>(L, stream);
            }
        }
        if (layers[0].flags != 0) {  // variants: single-chunk and multi-chunk instantiations
            if (layers[0].max_T <= CT) {
                switch (mode) {
                    case kVerify:
                        return ragged ? launch_mode<kVerify, true, NL, false, false, true>(L, stream)
                                      : launch_mode<kVerify, false, NL, false, false, true>(L, stream);
                    case kCommit:
                        return ragged ? launch_mode<kCommit, true, NL, false, false, true>(L, stream)
                                      : launch_mode<kCommit, false, NL, false, false, true>(L, stream);
                    default:
                        return ragged ? launch_mode<kFused, true, NL, false, false, true>(L, stream)
                                      : launch_mode<kFused, false, NL, false, false, true>(L, stream);
                }
            }
            switch (mode) {
                case kVerify:
                    return ragged ? launch_mode<kVerify, true, NL, true, false, true>(L, stream)
                                  : launch_mode<kVerify, false, NL, true, false, true>(L, stream);
                case kCommit:
                    return ragged ? launch_mode<kCommit, true, NL, true, false, true>(L, stream)
                                  : launch_mode<kCommit, false, NL, true, false, true>(L, stream);
                default:
                    return ragged ? launch_mode<kFused, true, NL, true, false, true>(L, stream)
                                  : launch_mode<kFused, false, NL, true, false, true>(L, stream);
            }
        }
    } else {
        if (layers[0].cap > 0 || layers[0].flags != 0 || layers[0].tc || mode == kLagged)
            return cudaErrorNotSupported;
    }
    if (layers[0].max_T > CT) return dispatch<NL, true>(L, mode, ragged, stream);
    return dispatch<NL, false>(L, mode, ragged, stream);
}

}  // namespace

bool chunk_supported(bool bf16, int dk, int dv, int max_T) {
    return bf16 && dk == D && dv == D && max_T >= 1;
}

bool chunk_preferred(int max_T) { return max_T >= 1; }

cudaError_t launch_chunk(const Args *layers, int n, int mode, cudaStream_t stream) {
    if (n > 0 && (layers[0].flags != 0 || layers[0].cap > 0 || layers[0].tc || mode == kLagged)) {
        // Variants, replay buffers, commit-then-verify and the tcgen05 kernel run one
        // problem per launch.
        for (int l = 0; l < n; ++l) {
            const cudaError_t e = launch_layers<1>(layers + l, 1, mode, stream);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    for (int l0 = 0; l0 < n; l0 += kChunkMaxLayers) {
        const int m = n - l0 < kChunkMaxLayers ? n - l0 : kChunkMaxLayers;
        const cudaError_t e = m == 1 ? launch_layers<1>(layers + l0, 1, mode, stream)
                                     : launch_layers<kChunkMaxLayers>(layers + l0, m, mode, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gdn
