// Recurrent (per-token) form of the gated delta rule on CUDA cores.
//
// RS threads own one value column j of one unit's state tile, each dk/RS of its
// rows, in registers.  With the tile H (dk x dv, H = S^T) and h_j its column j:
//     u_j = h_j . k_t            p_j = h_j . q_t
//     w_j = beta_t (v_tj - alpha_t u_j)
//     h_j <- alpha_t h_j + w_j k_t
//     o_tj = h_j . q_t = alpha_t p_j + w_j (k_t . q_t)
// which is S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
// o_t = S_t q_t with the column j of H being row j of S.  The only reduction
// that crosses threads is the RS-way sum of the partial dot products (warp
// shuffles between the threads of one column).  The decay is kept as a scalar
// factor, h_j = s * g_j, so the update is one FMA per element
// (g_j += k_t * (w_j / s)); g is rescaled when s leaves [2^-60, 2^60] (and so
// when alpha_t = 0).
//
// Block: up to 128 threads = (value columns) x RS; lane = column + (32/RS) * part,
// so one warp covers 32/RS columns.  Grid: x = unit (r * H + h), y = column block.
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int kChunk = 16;     // tokens staged in shared memory at a time
constexpr int kThreads = 128;  // threads per block at most

template <int DK>
struct RecShape {
    static constexpr int RS = DK >= 256 ? 4 : (DK >= 128 ? 2 : 1);  // threads per column
    static constexpr int R = DK / RS;             // rows per thread
    static constexpr int CPW = 32 / RS;           // columns per warp
};

template <int DK, bool BF16, int MODE>
__global__ void __launch_bounds__(kThreads) rec_kernel(const Args p) {
    using Shape = RecShape<DK>;
    constexpr int R = Shape::R, CPW = Shape::CPW;
    __shared__ __align__(16) float sk[kChunk][DK];
    __shared__ __align__(16) float sq[kChunk][DK];
    __shared__ __align__(16) float sv[kChunk][kThreads];
    __shared__ float sa[kChunk], sb[kChunk], skq[kChunk];

    const int unit = blockIdx.x;
    const int r = unit / p.H;
    const int h = unit - r * p.H;
    const int ncols = blockDim.x / Shape::RS;
    const int c0 = blockIdx.y * ncols;
    const int lane_ = threadIdx.x & 31;
    const int cl = (threadIdx.x >> 5) * CPW + (lane_ % CPW);  // column within the block
    const int part = lane_ / CPW;                             // which rows of the column
    const int i0 = part * R;
    const int j = c0 + cl;

    Unit u;
    if (!resolve_unit(p, r, h, MODE, u)) return;
    const int T_run = (MODE == kCommit) ? u.a : u.T;
    if (T_run == 0) return;  // commit of a = 0 writes nothing; no tokens, no outputs

    float *col = u.tile + (size_t)i0 * p.dv + j;  // element (i0 + i, j) at col[i * dv]
    float g[R];
#pragma unroll
    for (int i = 0; i < R; ++i) g[i] = col[(size_t)i * p.dv];
    float s = 1.0f;

    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;

#pragma unroll 1
    for (int t0 = 0; t0 < T_run; t0 += kChunk) {
        const int n = min(kChunk, T_run - t0);
        __syncthreads();  // previous chunk fully consumed
        // Stage q (not for commit: it has no outputs), k (n x DK), v (n x ncols),
        // alpha, beta as float.
        constexpr int VEC = BF16 ? 8 : 4;
        for (int e = tid * VEC; e < n * DK; e += nthr * VEC) {
            const int tt = e / DK, c = e - tt * DK;
            const size_t off = ((size_t)(u.row0 + t0 + tt) * p.H + h) * DK + c;
            if (BF16) {
                if (MODE != kCommit) {
                    const uint4 wq = *reinterpret_cast<const uint4 *>(
                        reinterpret_cast<const __nv_bfloat16 *>(p.q) + off);
                    bf16x8_to_f32(wq, &sq[tt][c]);
                }
                const uint4 wk = *reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const __nv_bfloat16 *>(p.k) + off);
                bf16x8_to_f32(wk, &sk[tt][c]);
            } else {
                if (MODE != kCommit)
                    *reinterpret_cast<float4 *>(&sq[tt][c]) =
                        *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.q) + off);
                *reinterpret_cast<float4 *>(&sk[tt][c]) =
                    *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.k) + off);
            }
        }
        for (int e = tid * VEC; e < n * ncols; e += nthr * VEC) {
            const int tt = e / ncols, c = e - tt * ncols;
            const size_t off = ((size_t)(u.row0 + t0 + tt) * p.H + h) * p.dv + c0 + c;
            if (BF16) {
                const uint4 wv = *reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const __nv_bfloat16 *>(p.v) + off);
                bf16x8_to_f32(wv, &sv[tt][c]);
            } else {
                *reinterpret_cast<float4 *>(&sv[tt][c]) =
                    *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.v) + off);
            }
        }
        if (tid < n) {
            const size_t x = (size_t)(u.row0 + t0 + tid) * p.H + h;
            const float a = p.alpha[x];
            sa[tid] = (p.flags & GDN_FLAG_LOG_GATE) ? expf(a) : a;  // log-space gate: expf(g)
            sb[tid] = p.beta[x];
        }
        __syncthreads();
        // k_t . q_t, one warp per token (outputs only).
        for (int tt = warp; MODE != kCommit && tt < n; tt += nwarps) {
            float acc = 0.0f;
#pragma unroll
            for (int i = lane; i < DK; i += 32) acc = fmaf(sk[tt][i], sq[tt][i], acc);
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
            if (lane == 0) skq[tt] = acc;
        }
        __syncthreads();

#pragma unroll 1
        for (int tt = 0; tt < n; ++tt) {
            const int t = t0 + tt;
            const float a_t = sa[tt], b_t = sb[tt];
            float uu[4] = {0.f, 0.f, 0.f, 0.f}, pp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < R; i += 4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(&sk[tt][i0 + i]);
                uu[0] = fmaf(k4.x, g[i + 0], uu[0]);
                uu[1] = fmaf(k4.y, g[i + 1], uu[1]);
                uu[2] = fmaf(k4.z, g[i + 2], uu[2]);
                uu[3] = fmaf(k4.w, g[i + 3], uu[3]);
                if (MODE != kCommit) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(&sq[tt][i0 + i]);
                    pp[0] = fmaf(q4.x, g[i + 0], pp[0]);
                    pp[1] = fmaf(q4.y, g[i + 1], pp[1]);
                    pp[2] = fmaf(q4.z, g[i + 2], pp[2]);
                    pp[3] = fmaf(q4.w, g[i + 3], pp[3]);
                }
            }
            // u_j and p_j use h_{t-1} = s * g; sum the RS parts of the column.
            float us = (uu[0] + uu[1]) + (uu[2] + uu[3]);
            float ps = (pp[0] + pp[1]) + (pp[2] + pp[3]);
#pragma unroll
            for (int m = CPW; m < 32; m <<= 1) {
                us += __shfl_xor_sync(0xffffffffu, us, m);
                if (MODE != kCommit) ps += __shfl_xor_sync(0xffffffffu, ps, m);
            }
            const float u_j = s * us;
            const float p_j = s * ps;
            const float w_j = b_t * (sv[tt][cl] - a_t * u_j);
            float s_new = a_t * s;
            if (!(s_new >= 0x1p-60f && s_new <= 0x1p60f)) {  // block-uniform branch
#pragma unroll
                for (int i = 0; i < R; ++i) g[i] *= s_new;
                s_new = 1.0f;
            }
            const float c = w_j / s_new;
#pragma unroll
            for (int i = 0; i < R; i += 4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(&sk[tt][i0 + i]);
                g[i + 0] = fmaf(k4.x, c, g[i + 0]);
                g[i + 1] = fmaf(k4.y, c, g[i + 1]);
                g[i + 2] = fmaf(k4.z, c, g[i + 2]);
                g[i + 3] = fmaf(k4.w, c, g[i + 3]);
            }
            s = s_new;
            if (MODE != kCommit && part == 0) {
                const size_t oi = ((size_t)(u.row0 + t) * p.H + h) * p.dv + j;
                const float ov = fmaf(a_t, p_j, w_j * skq[tt]);
                if (p.flags & GDN_FLAG_O_BF16)
                    static_cast<__nv_bfloat16 *>(p.o)[oi] = __float2bfloat16_rn(ov);
                else
                    static_cast<float *>(p.o)[oi] = ov;
            }
            if (MODE == kFused && t + 1 == u.a) {
                float *dst = opaque(col);
#pragma unroll
                for (int i = 0; i < R; ++i) dst[(size_t)i * p.dv] = s * g[i];
            }
        }
    }
    if (MODE == kCommit) {
        float *dst = opaque(col);
#pragma unroll
        for (int i = 0; i < R; ++i) dst[(size_t)i * p.dv] = s * g[i];
    }
}

template <int DK, bool BF16>
cudaError_t launch_dk(const Args &p, int mode, cudaStream_t stream) {
    constexpr int RS = RecShape<DK>::RS;
    int ncols = kThreads / RS;  // columns per block: a multiple of 32 that divides dv
    while (p.dv % ncols) ncols -= 32;
    const dim3 grid((unsigned)(p.B * p.H), (unsigned)(p.dv / ncols));
    const dim3 block((unsigned)(ncols * RS));
    switch (mode) {
        case kVerify: rec_kernel<DK, BF16, kVerify><<<grid, block, 0, stream>>>(p); break;
        case kCommit: rec_kernel<DK, BF16, kCommit><<<grid, block, 0, stream>>>(p); break;
        default: rec_kernel<DK, BF16, kFused><<<grid, block, 0, stream>>>(p); break;
    }
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_bf(const Args &p, int mode, cudaStream_t stream) {
    switch (p.dk) {
        case 32: return launch_dk<32, BF16>(p, mode, stream);
        case 64: return launch_dk<64, BF16>(p, mode, stream);
        case 128: return launch_dk<128, BF16>(p, mode, stream);
        default: return launch_dk<256, BF16>(p, mode, stream);
    }
}

}  // namespace

// Host launcher.  The caller has validated: dk in {32, 64, 128, 256}, dv a multiple
// of 32 (and of 128 when above 128), B * H >= 1.
cudaError_t launch_recurrent(const Args &p, int mode, bool bf16, cudaStream_t stream) {
    return bf16 ? launch_bf<true>(p, mode, stream) : launch_bf<false>(p, mode, stream);
}

}  // namespace gdn
