// Host-side launchers of the kernels (internal to libgdn.so).
#pragma once

#include <cuda_runtime.h>

#include "gdn_device.cuh"

namespace gdn {

// Recurrent kernel: dk in {32, 64, 128, 256}; dv a multiple of 32, <= 128 or a
// multiple of 128 up to 256; q/k/v bf16 or fp32; any max_T.
cudaError_t launch_recurrent(const Args &p, int mode, bool bf16, cudaStream_t stream);

// Chunked tensor-core kernel and its applicability.  One call covers n
// problems (layers) that share every request-level field; up to
// kChunkMaxLayers of them run in one launch, more are split into several.
constexpr int kChunkMaxLayers = 32;
bool chunk_supported(bool bf16, int dk, int dv, int max_T);
bool chunk_preferred(int max_T);
cudaError_t launch_chunk(const Args *layers, int n, int mode, cudaStream_t stream);

// Greedy accepted lengths (arguments already validated on the host).
cudaError_t launch_accept(int B, int max_T, const int32_t *cu_seqlens, long long n_tok,
                          const int32_t *draft, const int32_t *target, int32_t *accepted,
                          int32_t *dev_err, cudaStream_t stream);

// One block that waits on a barrier nothing completes, until the bounded wait
// gives up; ORs GDN_DEVERR_TIMEOUT into *dev_err (not NULL).
cudaError_t launch_wait_selftest(int32_t *dev_err, cudaStream_t stream);

}  // namespace gdn
