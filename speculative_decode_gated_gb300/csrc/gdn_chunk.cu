// Chunked (WY) form of the gated delta rule for one block of up to 16 draft
// tokens, with the two state-sized products on tensor cores.
//
// With the tile H_0 (dk x dv, H = S^T), tokens t = 0..T-1 and
//   D[t][s] = prod_{s<r<=t} alpha_r        (D[t][t] = 1),   gamma_t = D[t][0] * alpha_0,
// the recurrence H_t = alpha_t H_{t-1} + k_t w_t^T, w_t = beta_t (v_t - alpha_t H_{t-1}^T k_t)
// unrolls to
//   P = H_0^T Q^T,  Z = H_0^T K^T                        (dv x T, tensor cores)
//   w_t = beta_t (v_t - gamma_t Z_t) - sum_{s<t} A[t][s] w_s,  A[t][s] = beta_t D[t][s] k_t.k_s
//   o_t = gamma_t P_t + sum_{s<=t} M[t][s] w_s,              M[t][s] = D[t][s] q_t.k_s
//   H_a = gamma_{a-1} H_0 + sum_{s<a} D[a-1][s] k_s w_s^T    (tensor cores)
// Each value column j is independent given the token block, so warp w owns the
// 32 columns [32w, 32w + 32) of one unit (request r, head h); a block of 4
// warps owns one unit of dk = dv = 128.
//
// Precision: q, k are bf16 (exact operands).  The fp32 operands (H_0 in the
// first product, the scaled w in the second) are split into bf16 hi + lo and
// both halves multiplied, with fp32 accumulation: about 16 mantissa bits per
// operand.  The triangular solve and the outputs run in fp32 on CUDA cores.
//
// Register layout of H_0 (and of the committed state, which accumulates in
// the same registers): lane (g = lane/4, c = lane%4) of warp w holds rows
// 16 kb + 2c + {0, 1, 8, 9} (kb = 0..7) and columns 32w + 4g + {0..3}.  This is
// at once the A-fragment layout of H_0^T for mma.m16n8k16 (value columns as
// rows: fragment row g <-> column 4g + 2m, row g + 8 <-> 4g + 2m + 1 in m-tile
// m) and the accumulator layout of H_a^T, and every load and store of the
// tile is a 16-byte vector with full 32-byte sectors.
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int CT = 16;   // token block
constexpr int D = 128;   // dk = dv
constexpr int KS = 136;  // bf16 row stride of the token tiles (padding: conflict-free fragments)
constexpr int YS = 36;   // float row stride of the per-warp [column][P | Z] buffer
constexpr int WS = 18;   // float row stride of the per-warp [column][scaled w] buffer

struct __align__(16) ChunkSmem {
    __nv_bfloat16 k[CT][KS];
    __nv_bfloat16 q[CT][KS];
    float gram[2][CT][CT];  // [0][t][s] = k_t.k_s, [1][t][s] = q_t.k_s
    float A[CT][CT];        // beta_t D[t][s] k_t.k_s for s < t, else 0
    float M[CT][CT];        // D[t][s] q_t.k_s for s <= t, else 0
    float alpha[CT], beta[CT], gamma[CT];
    float dcol[CT];         // D[a-1][s] for s < a, else 0
    float y[4][32][YS];     // per warp; reused for the scaled w
};

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
    const uint32_t addr = (uint32_t)__cvta_generic_to_shared(row);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <int MODE>
__global__ void __launch_bounds__(128, 2) chunk_kernel(const Args p) {
    __shared__ ChunkSmem sm;
    const int unit = blockIdx.x;
    const int r = unit / p.H;
    const int h = unit - r * p.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;

    Unit u;
    if (!resolve_unit(p, r, h, MODE, u)) return;
    // Tokens that matter: all of them for outputs, the accepted prefix for commit.
    const int T = (MODE == kCommit) ? u.a : u.T;
    if (T == 0) return;
    const bool write_state = MODE != kVerify && u.a > 0;

    // 1. Checkpoint tile -> registers (slot gather), 32 x 16-byte loads per thread.
    float hr[8][4][4];
    {
        const float *src = u.tile + 32 * warp + 4 * g;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int row = 16 * kb + 2 * c + (rr & 1) + 8 * (rr >> 1);
                const float4 x = *reinterpret_cast<const float4 *>(src + row * D);
                hr[kb][rr][0] = x.x;
                hr[kb][rr][1] = x.y;
                hr[kb][rr][2] = x.z;
                hr[kb][rr][3] = x.w;
            }
    }

    // 2. Token block: q, k (bf16, zero rows past T), gates, this lane's v column.
    const size_t row_stride = (size_t)p.H * D;
    const size_t tok0 = ((size_t)u.row0 * p.H + h) * D;
    {
        const __nv_bfloat16 *gq = reinterpret_cast<const __nv_bfloat16 *>(p.q) + tok0;
        const __nv_bfloat16 *gk = reinterpret_cast<const __nv_bfloat16 *>(p.k) + tok0;
#pragma unroll
        for (int e = tid; e < 2 * CT * 16; e += 128) {
            const int which = e / (CT * 16);  // 0: k, 1: q
            const int t = (e >> 4) & (CT - 1);
            const int ch = e & 15;
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (t < T && (which == 0 || MODE != kCommit))
                val = *reinterpret_cast<const uint4 *>((which ? gq : gk) + t * row_stride + 8 * ch);
            *reinterpret_cast<uint4 *>(which ? &sm.q[t][8 * ch] : &sm.k[t][8 * ch]) = val;
        }
        if (tid < CT) {
            const size_t x = (size_t)(u.row0 + tid) * p.H + h;
            sm.alpha[tid] = tid < T ? p.alpha[x] : 1.0f;
            sm.beta[tid] = tid < T ? p.beta[x] : 0.0f;
        }
    }
    float vv[CT];
    {
        const __nv_bfloat16 *gv =
            reinterpret_cast<const __nv_bfloat16 *>(p.v) + tok0 + 32 * warp + lane;
#pragma unroll
        for (int t = 0; t < CT; ++t)
            vv[t] = t < T ? __bfloat162float(gv[t * row_stride]) : 0.0f;
    }
    __syncthreads();

    // 3. Gram blocks k_t.k_s and q_t.k_s: warp w computes matrix w/2, columns 8 (w%2) + [0, 8).
    {
        const __nv_bfloat16(*At)[KS] = (warp >> 1) ? sm.q : sm.k;
        const int nt = warp & 1;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
            const int col = 16 * kb + 2 * c;
            mma(acc[0], acc[1], acc[2], acc[3], lds32(&At[g][col]), lds32(&At[g + 8][col]),
                lds32(&At[g][col + 8]), lds32(&At[g + 8][col + 8]), lds32(&sm.k[8 * nt + g][col]),
                lds32(&sm.k[8 * nt + g][col + 8]));
        }
        float(*G)[CT] = sm.gram[warp >> 1];
        G[g][8 * nt + 2 * c] = acc[0];
        G[g][8 * nt + 2 * c + 1] = acc[1];
        G[g + 8][8 * nt + 2 * c] = acc[2];
        G[g + 8][8 * nt + 2 * c + 1] = acc[3];
    }
    __syncthreads();

    // 4. Decay products and the two triangular matrices (lane t of warp 0 owns row t).
    if (warp == 0 && lane < CT) {
        const int t = lane;
        const int a_last = (MODE == kVerify) ? -1 : u.a - 1;
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
    __syncthreads();

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
            split2(hr[kb][0][2 * m], hr[kb][1][2 * m], ah[0], al[0]);
            split2(hr[kb][0][2 * m + 1], hr[kb][1][2 * m + 1], ah[1], al[1]);
            split2(hr[kb][2][2 * m], hr[kb][3][2 * m], ah[2], al[2]);
            split2(hr[kb][2][2 * m + 1], hr[kb][3][2 * m + 1], ah[3], al[3]);
#pragma unroll
            for (int nt = NT0; nt < 4; ++nt) {
                float *d = y[m][nt];
                mma(d[0], d[1], d[2], d[3], ah[0], ah[1], ah[2], ah[3], b[nt][0], b[nt][1]);
                mma(d[0], d[1], d[2], d[3], al[0], al[1], al[2], al[3], b[nt][0], b[nt][1]);
            }
        }
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
        float acc = sm.beta[t] * (vv[t] - sm.gamma[t] * z[t]);
#pragma unroll
        for (int s = 0; s < t; ++s) acc = fmaf(-sm.A[t][s], w[s], acc);
        w[t] = acc;
    }

    // 8. Outputs o_t for t < T_r.
    if (MODE != kCommit) {
        float *go = p.o + ((size_t)u.row0 * p.H + h) * D + 32 * warp + lane;
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

    // 9. Commit: H_a^T = gamma_{a-1} H_0^T + (D[a-1][.] w)^T K, accumulated in hr.
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
        const float gam = sm.gamma[u.a - 1];
#pragma unroll
        for (int kb = 0; kb < 8; ++kb)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                for (int e = 0; e < 4; ++e) hr[kb][rr][e] *= gam;
        // ldmatrix.trans row address of this lane: matrix lane/8 -> (token half, dk half).
        const int mi = lane >> 3;
        const __nv_bfloat16 *krow = &sm.k[(lane & 7) + 8 * (mi & 1)][8 * (mi >> 1)];
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
            uint32_t b00, b01, b10, b11;  // (n-tile 2kb: b0, b1), (n-tile 2kb+1: b0, b1)
            ldsm_x4_trans(b00, b01, b10, b11, krow + 16 * kb);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                mma(hr[kb][0][2 * m], hr[kb][1][2 * m], hr[kb][0][2 * m + 1], hr[kb][1][2 * m + 1],
                    ah[m][0], ah[m][1], ah[m][2], ah[m][3], b00, b01);
                mma(hr[kb][0][2 * m], hr[kb][1][2 * m], hr[kb][0][2 * m + 1], hr[kb][1][2 * m + 1],
                    al[m][0], al[m][1], al[m][2], al[m][3], b00, b01);
                mma(hr[kb][2][2 * m], hr[kb][3][2 * m], hr[kb][2][2 * m + 1], hr[kb][3][2 * m + 1],
                    ah[m][0], ah[m][1], ah[m][2], ah[m][3], b10, b11);
                mma(hr[kb][2][2 * m], hr[kb][3][2 * m], hr[kb][2][2 * m + 1], hr[kb][3][2 * m + 1],
                    al[m][0], al[m][1], al[m][2], al[m][3], b10, b11);
            }
        }
        float *dst = opaque(u.tile) + 32 * warp + 4 * g;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int row = 16 * kb + 2 * c + (rr & 1) + 8 * (rr >> 1);
                *reinterpret_cast<float4 *>(dst + row * D) =
                    make_float4(hr[kb][rr][0], hr[kb][rr][1], hr[kb][rr][2], hr[kb][rr][3]);
            }
    }
}

}  // namespace

bool chunk_supported(bool bf16, int dk, int dv, int max_T) {
    return bf16 && dk == D && dv == D && max_T >= 1 && max_T <= CT;
}

bool chunk_preferred(int max_T) { return max_T >= 1; }

cudaError_t launch_chunk(const Args &p, int mode, cudaStream_t stream) {
    const dim3 grid((unsigned)(p.B * p.H)), block(128);
    switch (mode) {
        case kVerify: chunk_kernel<kVerify><<<grid, block, 0, stream>>>(p); break;
        case kCommit: chunk_kernel<kCommit><<<grid, block, 0, stream>>>(p); break;
        default: chunk_kernel<kFused><<<grid, block, 0, stream>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace gdn
