// Chunked (WY) form of the gated delta rule for one block of up to 16 draft
// tokens, with the two state-sized products on tensor cores, as a persistent
// pipelined kernel: one block per SM walks its share of the units while a
// producer warp streams their checkpoint tiles into a 3-stage shared-memory
// ring with TMA.
//
// With the tile H_0 (dk x dv, H = S^T), tokens t = 0..T-1 and
//   D[t][s] = prod_{s<r<=t} alpha_r        (D[t][t] = 1),   gamma_t = D[t][0] * alpha_0,
// the recurrence H_t = alpha_t H_{t-1} + k_t w_t^T, w_t = beta_t (v_t - alpha_t H_{t-1}^T k_t)
// unrolls to
//   P = H_0^T Q^T,  Z = H_0^T K^T                        (dv x T, tensor cores)
//   w_t = beta_t (v_t - gamma_t Z_t) - sum_{s<t} A[t][s] w_s,  A[t][s] = beta_t D[t][s] k_t.k_s
//   o_t = gamma_t P_t + sum_{s<=t} M[t][s] w_s,              M[t][s] = D[t][s] q_t.k_s
//   H_a = gamma_{a-1} H_0 + sum_{s<a} D[a-1][s] k_s w_s^T    (tensor cores)
// Each value column j is independent given the token block, so consumer warp
// w owns the 32 columns [32w, 32w + 32) of the unit (request r, head h).
//
// Roles (block of 5 warps, one block per SM):
//   warp 4 (producer, one lane): for each of the block's units, waits for a
//     free stage, then loads the 64 KiB tile with four 3-D TMA copies (boxes of
//     32 value columns x 128 key rows, 128-byte swizzle) onto the stage's
//     "full" mbarrier.
//   warps 0-3 (consumers): prefetch the next unit's q/k/v/gates into
//     registers, stage the current unit's tokens in shared memory, build the
//     small triangular matrices, wait for the tile, run the products, write
//     the outputs and the committed tile, and release the stage on its
//     "empty" mbarrier.
// Every wait is bounded (about 2 s by %globaltimer); on expiry the block
// reports GDN_DEVERR_TIMEOUT and stops, after waiting for its copies in flight.
//
// Precision: q, k are bf16 (exact operands).  The fp32 operands (H_0 in the
// first product, the scaled w in the second) are split into bf16 hi + lo and
// both halves multiplied, with fp32 accumulation: about 16 mantissa bits per
// operand.  The triangular solve and the outputs run in fp32 on CUDA cores.
//
// Fragment layout of H_0: lane (g = lane/4, c = lane%4) of consumer warp w
// reads rows 16 kb + 2c + {0, 1, 8, 9} (kb = 0..7) and columns 32w + 4g + {0..3}.
// This is at once the A-fragment layout of H_0^T for mma.m16n8k16 (value
// columns as rows: fragment row g <-> column 4g + 2m, row g + 8 <-> 4g + 2m + 1
// in m-tile m) and the accumulator layout of H_a^T; with the 128-byte swizzle
// (16-byte chunk index XOR row % 8) the 16-byte shared loads are conflict-free,
// and the committed tile leaves as 16-byte stores with full 32-byte sectors.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int CT = 16;   // token block
constexpr int D = 128;   // dk = dv
constexpr int KS = 136;  // bf16 row stride of the token tiles (padding: conflict-free fragments)
constexpr int YS = 36;   // float row stride of the per-warp [column][P | Z] buffer
constexpr int WS = 18;   // float row stride of the per-warp [column][scaled w] buffer
constexpr int kStages = 3;
constexpr int kConsumers = 4;  // consumer warps
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr uint32_t kBoxBytes = 32 * D * 4;       // 32 value columns x 128 key rows
constexpr uint32_t kTileBytes = 4 * kBoxBytes;   // 64 KiB
constexpr unsigned long long kWaitNs = 2000000000ull;

struct Aux {
    __nv_bfloat16 k[CT][KS];
    __nv_bfloat16 q[CT][KS];
    float gram[2][CT][CT];  // [0][t][s] = k_t.k_s, [1][t][s] = q_t.k_s
    float A[CT][CT];        // beta_t D[t][s] k_t.k_s for s < t, else 0
    float M[CT][CT];        // D[t][s] q_t.k_s for s <= t, else 0
    float alpha[CT], beta[CT], gamma[CT];
    float dcol[CT];         // D[a-1][s] for s < a, else 0
    float y[kConsumers][32][YS];  // per warp; reused for the scaled w
    unsigned long long full[kStages], empty[kStages];
    int abort_flag;  // a consumer's wait expired: all consumers stop together
};
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kTileBytes + sizeof(Aux);
static_assert(kSmemBytes <= 232448, "shared memory budget");

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with parity `parity` to complete; false after ~2 s.
__device__ __noinline__ bool wait_parity(uint32_t bar, uint32_t parity) {
    unsigned long long t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            const unsigned long long now = globaltimer();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitNs) {
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                             int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kConsumers) : "memory");
}

__device__ __forceinline__ uint32_t lds32(const __nv_bfloat16 *p) {
    return *reinterpret_cast<const uint32_t *>(p);
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
                                              uint32_t &r3, const void *row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(row)));
}

// Row `row`, 16-byte chunk `chunk` of a 128-byte-swizzled box (32 floats per row).
__device__ __forceinline__ float4 ld_box(const char *box, int row, int chunk) {
    return *reinterpret_cast<const float4 *>(box + row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ------------------------------------------------------------ per-unit data

// What both roles know about a unit; `skip` when nothing is to be done.
struct UnitPlan {
    Unit u;
    int h;
    int teff;  // tokens that matter: T_r, or a_r for commit
    bool skip;
};

template <int MODE>
__device__ __forceinline__ RawMeta load_unit_meta(const Args &p, int unit) {
    return load_meta(p, unit / p.H, MODE);
}

template <int MODE>
__device__ __forceinline__ UnitPlan plan_unit(const Args &p, int unit, const RawMeta &m) {
    UnitPlan pl;
    pl.h = unit - (unit / p.H) * p.H;
    const bool ok = check_meta(p, m, pl.h, MODE, pl.u);
    pl.teff = ok ? ((MODE == kCommit) ? pl.u.a : pl.u.T) : 0;
    pl.skip = !ok || pl.teff == 0;
    return pl;
}

// Token block of one unit held in registers by a consumer thread (tid < 128):
// four 16-byte chunks of the k / q tiles, this lane's v column (raw bf16 bits,
// converted only where used so the loads stay in flight), and alpha/beta of
// token tid (tid < 16).
struct TokRegs {
    uint4 qk[4];
    unsigned short v[CT];
    float a, b;
};

template <int MODE>
__device__ __forceinline__ void load_tokens(const Args &p, const UnitPlan &pl, int tid, TokRegs &tr) {
    const size_t row_stride = (size_t)p.H * D;
    const size_t tok0 = ((size_t)pl.u.row0 * p.H + pl.h) * D;
    const __nv_bfloat16 *gq = reinterpret_cast<const __nv_bfloat16 *>(p.q) + tok0;
    const __nv_bfloat16 *gk = reinterpret_cast<const __nv_bfloat16 *>(p.k) + tok0;
    const int T = pl.skip ? 0 : pl.teff;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = tid + 128 * i;
        const int which = e >> 8;  // 0: k, 1: q
        const int t = (e >> 4) & (CT - 1);
        const int ch = e & 15;
        tr.qk[i] = make_uint4(0u, 0u, 0u, 0u);
        if (t < T && (which == 0 || MODE != kCommit))
            tr.qk[i] = *reinterpret_cast<const uint4 *>((which ? gq : gk) + t * row_stride + 8 * ch);
    }
    const unsigned short *gv = reinterpret_cast<const unsigned short *>(p.v) + tok0 + tid;
#pragma unroll
    for (int t = 0; t < CT; ++t) {
        tr.v[t] = 0;
        if (t < T) tr.v[t] = gv[t * row_stride];
    }
    tr.a = 1.0f;
    tr.b = 0.0f;
    if (tid < T) {
        const size_t x = (size_t)(pl.u.row0 + tid) * p.H + pl.h;
        tr.a = p.alpha[x];
        tr.b = p.beta[x];
    }
}

__device__ __forceinline__ float bf16_bits_to_float(unsigned short b) {
    return __uint_as_float((uint32_t)b << 16);
}

// ------------------------------------------------------------ the kernel

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_kernel(const Args p, const __grid_constant__ CUtensorMap tmap) {
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment of the stage ring (required by the 128-byte swizzle).
    const uint32_t raw_addr = smem_u32(smem_raw);
    unsigned char *stages = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    Aux &sm = *reinterpret_cast<Aux *>(stages + (size_t)kStages * kTileBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int U = p.B * p.H;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), kConsumers);
        }
        sm.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    // ---------------------------------------------------------- producer
    if (warp == kConsumers) {
        if (lane != 0) return;
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        uint32_t last_parity[kStages] = {0, 0, 0};
        bool timed_out = false;
        // Metadata is loaded one unit ahead of its use.
        RawMeta raw = load_unit_meta<MODE>(p, blockIdx.x < U ? blockIdx.x : 0);
        for (int unit = blockIdx.x; unit < U; unit += gridDim.x) {
            const UnitPlan pl = plan_unit<MODE>(p, unit, raw);
            if (unit + (int)gridDim.x < U) raw = load_unit_meta<MODE>(p, unit + gridDim.x);
            if (pl.skip) continue;
            if (!wait_parity(smem_u32(&sm.empty[stage]), phase ^ 1u)) {
                timed_out = true;
                break;
            }
            const uint32_t full = smem_u32(&sm.full[stage]);
            mbar_arrive_expect_tx(full, kTileBytes);
            const int slot_unit = (int)((pl.u.tile - p.pool) / (D * D));  // slot * H + h
            const uint32_t dst = smem_u32(stages + (size_t)stage * kTileBytes);
#pragma unroll
            for (int b = 0; b < 4; ++b) tma_load_box(dst + b * kBoxBytes, &tmap, 32 * b, 0, slot_unit, full);
            last_parity[stage] = phase;
            ++issued;
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // Copies still in flight must land before the block exits.
        for (int s = 0; s < kStages && s < issued; ++s)
            if (!wait_parity(smem_u32(&sm.full[s]), last_parity[s])) timed_out = true;
        if (timed_out && p.dev_err) atomicOr(p.dev_err, GDN_DEVERR_TIMEOUT);
        return;
    }

    // ---------------------------------------------------------- consumers
    const int g = lane >> 2, c = lane & 3;
    const size_t row_stride = (size_t)p.H * D;
    int stage = 0;
    uint32_t phase = 0;

    // Pipeline of the consumers' own loads: metadata two units ahead, the token
    // block one unit ahead, so no load is waited on in the iteration that issues it.
    const int G = gridDim.x;
    UnitPlan nxt;
    TokRegs tn;
    RawMeta raw2;
    int unit = blockIdx.x;
    if (unit < U) {
        nxt = plan_unit<MODE>(p, unit, load_unit_meta<MODE>(p, unit));
        load_tokens<MODE>(p, nxt, tid, tn);
        if (unit + G < U) raw2 = load_unit_meta<MODE>(p, unit + G);
    }
    for (; unit < U; unit += G) {
        const UnitPlan cur = nxt;
        const TokRegs tc = tn;
        if (unit + G < U) {
            nxt = plan_unit<MODE>(p, unit + G, raw2);
            if (unit + 2 * G < U) raw2 = load_unit_meta<MODE>(p, unit + 2 * G);
            load_tokens<MODE>(p, nxt, tid, tn);
        }
        if (cur.skip) continue;
        const int T = cur.teff;
        const bool write_state = MODE != kVerify && cur.u.a > 0;

        // 1. Stage the token block (the previous unit is done with it).
        consumer_sync();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = tid + 128 * i;
            const int t = (e >> 4) & (CT - 1);
            const int ch = e & 15;
            *reinterpret_cast<uint4 *>((e >> 8) ? &sm.q[t][8 * ch] : &sm.k[t][8 * ch]) = tc.qk[i];
        }
        if (tid < CT) {
            sm.alpha[tid] = tc.a;
            sm.beta[tid] = tc.b;
        }
        consumer_sync();

        // 2. Gram blocks k_t.k_s and q_t.k_s: warp w computes matrix w/2, columns 8 (w%2) + [0, 8).
        {
            const __nv_bfloat16(*At)[KS] = (warp >> 1) ? sm.q : sm.k;
            const int nt = warp & 1;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
                const int col = 16 * kb + 2 * c;
                mma(acc[0], acc[1], acc[2], acc[3], lds32(&At[g][col]), lds32(&At[g + 8][col]),
                    lds32(&At[g][col + 8]), lds32(&At[g + 8][col + 8]),
                    lds32(&sm.k[8 * nt + g][col]), lds32(&sm.k[8 * nt + g][col + 8]));
            }
            float(*G)[CT] = sm.gram[warp >> 1];
            G[g][8 * nt + 2 * c] = acc[0];
            G[g][8 * nt + 2 * c + 1] = acc[1];
            G[g + 8][8 * nt + 2 * c] = acc[2];
            G[g + 8][8 * nt + 2 * c + 1] = acc[3];
        }
        consumer_sync();

        // 3. Decay products and the two triangular matrices (lane t of warp 0 owns row t).
        if (warp == 0 && lane < CT) {
            const int t = lane;
            const int a_last = (MODE == kVerify) ? -1 : cur.u.a - 1;
            float d = 1.0f;  // D[t][s], walking s = t, t-1, ..., 0
#pragma unroll
            for (int s = CT - 1; s >= 0; --s) {
                if (s <= t) {
                    sm.A[t][s] = s < t ? sm.beta[t] * d * sm.gram[0][t][s] : 0.0f;
                    sm.M[t][s] = d * sm.gram[1][t][s];
                    if (t == a_last) sm.dcol[s] = d;
                    d *= sm.alpha[s];  // D[t][s-1] = D[t][s] alpha_s; after s = 0: gamma_t
                } else {
                    sm.A[t][s] = 0.0f;
                    sm.M[t][s] = 0.0f;
                    if (t == a_last) sm.dcol[s] = 0.0f;
                }
            }
            sm.gamma[t] = d;
        }
        consumer_sync();

        // 4. The checkpoint tile of this unit.  Every consumer thread's wait is
        //    bounded; they then agree, so none is left at a barrier alone.
        if (!wait_parity(smem_u32(&sm.full[stage]), phase)) sm.abort_flag = 1;
        consumer_sync();
        if (sm.abort_flag) {
            if (tid == 0 && p.dev_err) atomicOr(p.dev_err, GDN_DEVERR_TIMEOUT);
            break;
        }
        const char *box = reinterpret_cast<const char *>(stages + (size_t)stage * kTileBytes) +
                          warp * kBoxBytes;

        // 5. P = H_0^T Q^T and Z = H_0^T K^T for this warp's 32 columns (N-tiles: Q 0-7,
        //    Q 8-15, K 0-7, K 8-15; commit needs only Z).
        constexpr int NT0 = (MODE == kCommit) ? 2 : 0;
        float y[2][4][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) y[m][nt][e] = 0.0f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
            float hv[4][4];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const float4 x = ld_box(box, 16 * kb + 2 * c + (rr & 1) + 8 * (rr >> 1), g);
                hv[rr][0] = x.x;
                hv[rr][1] = x.y;
                hv[rr][2] = x.z;
                hv[rr][3] = x.w;
            }
            uint32_t b[4][2];
#pragma unroll
            for (int nt = NT0; nt < 4; ++nt) {
                const __nv_bfloat16(*Bt)[KS] = nt < 2 ? sm.q : sm.k;
                const int tok = 8 * (nt & 1) + g;
                b[nt][0] = lds32(&Bt[tok][16 * kb + 2 * c]);
                b[nt][1] = lds32(&Bt[tok][16 * kb + 2 * c + 8]);
            }
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                uint32_t ah[4], al[4];
                split2(hv[0][2 * m], hv[1][2 * m], ah[0], al[0]);
                split2(hv[0][2 * m + 1], hv[1][2 * m + 1], ah[1], al[1]);
                split2(hv[2][2 * m], hv[3][2 * m], ah[2], al[2]);
                split2(hv[2][2 * m + 1], hv[3][2 * m + 1], ah[3], al[3]);
#pragma unroll
                for (int nt = NT0; nt < 4; ++nt) {
                    float *d = y[m][nt];
                    mma(d[0], d[1], d[2], d[3], ah[0], ah[1], ah[2], ah[3], b[nt][0], b[nt][1]);
                    mma(d[0], d[1], d[2], d[3], al[0], al[1], al[2], al[3], b[nt][0], b[nt][1]);
                }
            }
        }
        const uint32_t empty = smem_u32(&sm.empty[stage]);
        if (!write_state) {  // the tile is not read again: hand the stage back now
            __syncwarp();
            if (lane == 0) mbar_arrive(empty);
        }

        // 6. Fragments -> per-warp [column][P | Z] buffer -> lane j holds column 32w + j.
        float(*yb)[YS] = sm.y[warp];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int nt = NT0; nt < 4; ++nt) {
                const int tk = 16 * (nt >> 1) + 8 * (nt & 1) + 2 * c;
                *reinterpret_cast<float2 *>(&yb[4 * g + 2 * m][tk]) =
                    make_float2(y[m][nt][0], y[m][nt][1]);
                *reinterpret_cast<float2 *>(&yb[4 * g + 2 * m + 1][tk]) =
                    make_float2(y[m][nt][2], y[m][nt][3]);
            }
        __syncwarp();
        float pq[CT], z[CT];
#pragma unroll
        for (int t4 = 0; t4 < CT; t4 += 4) {
            const float4 zz = *reinterpret_cast<const float4 *>(&yb[lane][16 + t4]);
            z[t4] = zz.x;
            z[t4 + 1] = zz.y;
            z[t4 + 2] = zz.z;
            z[t4 + 3] = zz.w;
            if (MODE != kCommit) {
                const float4 pp = *reinterpret_cast<const float4 *>(&yb[lane][t4]);
                pq[t4] = pp.x;
                pq[t4 + 1] = pp.y;
                pq[t4 + 2] = pp.z;
                pq[t4 + 3] = pp.w;
            }
        }

        // 7. Forward substitution for w (fp32), one column per lane.
        float w[CT];
#pragma unroll
        for (int t = 0; t < CT; ++t) {
            float acc = sm.beta[t] * (bf16_bits_to_float(tc.v[t]) - sm.gamma[t] * z[t]);
#pragma unroll
            for (int s = 0; s < t; ++s) acc = fmaf(-sm.A[t][s], w[s], acc);
            w[t] = acc;
        }

        // 8. Outputs o_t for t < T_r.
        if (MODE != kCommit) {
            float *go = p.o + ((size_t)cur.u.row0 * p.H + cur.h) * D + 32 * warp + lane;
#pragma unroll
            for (int t = 0; t < CT; ++t) {
                if (t < T) {
                    float acc = sm.gamma[t] * pq[t];
#pragma unroll
                    for (int s = 0; s <= t; ++s) acc = fmaf(sm.M[t][s], w[s], acc);
                    go[t * row_stride] = acc;
                }
            }
        }

        // 9. Commit: H_a^T = gamma_{a-1} H_0^T + (D[a-1][.] w)^T K, tile by tile of 16 rows.
        if (write_state) {
            __syncwarp();  // yb is reused
            float(*wb)[WS] = reinterpret_cast<float(*)[WS]>(&sm.y[warp][0][0]);
#pragma unroll
            for (int s = 0; s < CT; s += 2)
                *reinterpret_cast<float2 *>(&wb[lane][s]) =
                    make_float2(sm.dcol[s] * w[s], sm.dcol[s + 1] * w[s + 1]);
            __syncwarp();
            uint32_t ah[2][4], al[2][4];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const float *r0 = wb[4 * g + 2 * m];
                const float *r1 = wb[4 * g + 2 * m + 1];
                split2(r0[2 * c], r0[2 * c + 1], ah[m][0], al[m][0]);
                split2(r1[2 * c], r1[2 * c + 1], ah[m][1], al[m][1]);
                split2(r0[2 * c + 8], r0[2 * c + 9], ah[m][2], al[m][2]);
                split2(r1[2 * c + 8], r1[2 * c + 9], ah[m][3], al[m][3]);
            }
            const float gam = sm.gamma[cur.u.a - 1];
            // ldmatrix.trans row address of this lane: matrix lane/8 -> (token half, dk half).
            const int mi = lane >> 3;
            const __nv_bfloat16 *krow = &sm.k[(lane & 7) + 8 * (mi & 1)][8 * (mi >> 1)];
            float *dst = opaque(cur.u.tile) + 32 * warp + 4 * g;
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
                float hv[4][4];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const float4 x = ld_box(box, 16 * kb + 2 * c + (rr & 1) + 8 * (rr >> 1), g);
                    hv[rr][0] = gam * x.x;
                    hv[rr][1] = gam * x.y;
                    hv[rr][2] = gam * x.z;
                    hv[rr][3] = gam * x.w;
                }
                uint32_t b00, b01, b10, b11;  // (n-tile 2kb: b0, b1), (n-tile 2kb+1: b0, b1)
                ldsm_x4_trans(b00, b01, b10, b11, krow + 16 * kb);
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    mma(hv[0][2 * m], hv[1][2 * m], hv[0][2 * m + 1], hv[1][2 * m + 1], ah[m][0],
                        ah[m][1], ah[m][2], ah[m][3], b00, b01);
                    mma(hv[0][2 * m], hv[1][2 * m], hv[0][2 * m + 1], hv[1][2 * m + 1], al[m][0],
                        al[m][1], al[m][2], al[m][3], b00, b01);
                    mma(hv[2][2 * m], hv[3][2 * m], hv[2][2 * m + 1], hv[3][2 * m + 1], ah[m][0],
                        ah[m][1], ah[m][2], ah[m][3], b10, b11);
                    mma(hv[2][2 * m], hv[3][2 * m], hv[2][2 * m + 1], hv[3][2 * m + 1], al[m][0],
                        al[m][1], al[m][2], al[m][3], b10, b11);
                }
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int row = 16 * kb + 2 * c + (rr & 1) + 8 * (rr >> 1);
                    *reinterpret_cast<float4 *>(dst + row * D) =
                        make_float4(hv[rr][0], hv[rr][1], hv[rr][2], hv[rr][3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty);
        }
        if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
        }
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

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int sms = 0;
    bool smem_set[3] = {false, false, false};
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

template <int MODE>
cudaError_t launch_mode(const Args &p, const CUtensorMap &map, cudaStream_t stream) {
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
        if (!info.smem_set[MODE]) {
            e = cudaFuncSetAttribute(chunk_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
            if (e != cudaSuccess) return e;
            info.smem_set[MODE] = true;
        }
        sms = info.sms;
    }
    const int units = p.B * p.H;
    const int grid = units < sms ? units : sms;
    chunk_kernel<MODE><<<grid, kThreads, kSmemBytes, stream>>>(p, map);
    return cudaGetLastError();
}

}  // namespace

bool chunk_supported(bool bf16, int dk, int dv, int max_T) {
    return bf16 && dk == D && dv == D && max_T >= 1 && max_T <= CT;
}

bool chunk_preferred(int max_T) { return max_T >= 1; }

cudaError_t launch_chunk(const Args &p, int mode, cudaStream_t stream) {
    // The pool as a 3-D tensor: value column (contiguous), key row, slot * H + head.
    const unsigned long long tiles = (unsigned long long)p.pool_slots * (unsigned long long)p.H;
    if (tiles == 0 || tiles > (1ull << 31)) return cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)D, (cuuint64_t)tiles};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)D * D * 4};
    const cuuint32_t box[3] = {32, (cuuint32_t)D, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.pool, dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    switch (mode) {
        case kVerify: return launch_mode<kVerify>(p, map, stream);
        case kCommit: return launch_mode<kCommit>(p, map, stream);
        default: return launch_mode<kFused>(p, map, stream);
    }
}

}  // namespace gdn
