// Host-side launchers shared between the translation units of libsparse_mla.
#pragma once
#include "smla_common.cuh"

namespace smla {
int mma_heads_per_cta(int H);
cudaError_t launch_mma(const KParams& p, cudaStream_t stream);
bool tc_supported(int H);
cudaError_t launch_tc(const KParams& p, cudaStream_t stream);
// The attention kernel for these parameters: tcgen05 for H % 64 == 0, warp-MMA otherwise.
inline int heads_per_cta(int H) { return tc_supported(H) ? 64 : mma_heads_per_cta(H); }
inline cudaError_t launch_attention(const KParams& p, cudaStream_t stream) {
  return tc_supported(p.H) ? launch_tc(p, stream) : launch_mma(p, stream);
}
cudaError_t launch_combine(const KParams& p, cudaStream_t stream);
cudaError_t launch_resolve(const KParams& p, int32_t* rows, int64_t rows_stride, cudaStream_t stream);
}  // namespace smla
