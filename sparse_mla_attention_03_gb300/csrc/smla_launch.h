// Host-side launchers shared between the translation units of libsparse_mla.
#pragma once
#include "smla_common.cuh"

namespace smla {
int mma_heads_per_cta(int H);
cudaError_t launch_mma(const KParams& p, cudaStream_t stream);
cudaError_t launch_combine(const KParams& p, cudaStream_t stream);
cudaError_t launch_resolve(const KParams& p, int32_t* rows, int64_t rows_stride, cudaStream_t stream);
}  // namespace smla
