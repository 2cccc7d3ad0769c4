// Greedy accepted length of each request: the number of leading positions of
// its draft block at which the draft token id equals the target model's id
// (speculative decoding keeps the draft tokens that agree with the target
// model and rolls the state back to that prefix: OCRia write-up, sections
// "Generate more tokens per target pass: speculative decoding" and "Make
// speculative verification cheaper").  One warp per request: each lane
// compares one position of a 32-token window, a ballot finds the first
// disagreement, and the warp stops at the first window that has one.
#include <cstdint>

#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int kWarps = 8;  // requests per block (one warp each)

__global__ void __launch_bounds__(32 * kWarps)
    accept_kernel(int B, int max_T, const int32_t *cu_seqlens, long long n_tok,
                  const int32_t *draft, const int32_t *target, int32_t *accepted,
                  int32_t *dev_err) {
    // Programmatic dependent launch: the next kernel may start its prologue
    // now; the ids are read only after the previous kernel has completed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    for (long long r = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); r < B;
         r += (long long)gridDim.x * kWarps) {
        long long c0 = r * (long long)max_T;
        int T = max_T;
        if (cu_seqlens) {
            const long long c1 = cu_seqlens[r + 1];
            c0 = cu_seqlens[r];
            const long long len = c1 - c0;
            if (len < 0 || len > max_T || c0 < 0 || c1 > n_tok) {
                if (lane == 0 && dev_err) atomicOr(dev_err, GDN_DEVERR_SEQLEN);
                continue;  // nothing is written for this request
            }
            T = (int)len;
        }
        int a = T;
        for (int t0 = 0; t0 < T; t0 += 32) {
            const int t = t0 + lane;
            const bool differ = t < T && draft[c0 + t] != target[c0 + t];
            const unsigned m = __ballot_sync(0xffffffffu, differ);
            if (m) {
                a = t0 + __ffs(m) - 1;
                break;
            }
        }
        if (lane == 0) accepted[r] = a;
    }
}

}  // namespace

cudaError_t launch_accept(int B, int max_T, const int32_t *cu_seqlens, long long n_tok,
                          const int32_t *draft, const int32_t *target, int32_t *accepted,
                          int32_t *dev_err, cudaStream_t stream) {
    const long long blocks = ((long long)B + kWarps - 1) / kWarps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(blocks < 65535 ? blocks : 65535));
    cfg.blockDim = dim3(32 * kWarps);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accept_kernel, B, max_T, cu_seqlens, n_tok, draft, target,
                              accepted, dev_err);
}

}  // namespace gdn
