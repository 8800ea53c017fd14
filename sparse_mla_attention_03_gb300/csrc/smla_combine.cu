// Split-K decode combine and the index-resolution kernel.
//
// Combine (AppMana forks-flash-mla-ampere-dsv4 releases, "decode H6: warp-wide
// combine -- one split per lane, branchless"): one warp per (token, head);
// lane s holds split s's LSE, a warp reduction gives lse = log sum_s
// exp(lse_s), and the output is sum_s exp(lse_s - lse) o_s, scaled by
// exp(lse) / (exp(lse) + exp(sink)) for the per-head sink.  Splits with
// lse_s = -inf weigh 0; if every split is empty, out = 0 and lse = -inf.
#include "smla_launch.h"

namespace smla {

__global__ void __launch_bounds__(128) combine_kernel(const KParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * 4 + warp;
  if (gw >= (int64_t)p.T * p.H) return;
  const int t = (int)(gw / p.H), h = (int)(gw % p.H);
  const int S = p.num_splits;
  const float* ls = p.ws_lse + gw * S;
  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, ls[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __nv_bfloat16* orow = p.out + (int64_t)t * p.out_stride_t + (int64_t)h * kDV;
  if (mx == -INFINITY) {
#pragma unroll
    for (int i = 0; i < 4; ++i) *reinterpret_cast<uint2*>(orow + 128 * i + 4 * lane) = make_uint2(0u, 0u);
    if (lane == 0) p.lse[(int64_t)t * p.lse_stride_t + h] = -INFINITY;
    return;
  }
  float sum = 0.f;
  for (int s = lane; s < S; s += 32) sum += expf(ls[s] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float L = mx + logf(sum);
  const float sinkf = p.attn_sink ? 1.f / (1.f + expf(__ldg(p.attn_sink + h) - L)) : 1.f;
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* ob = p.ws_o + gw * S * kDV;
  for (int s = 0; s < S; ++s) {
    const float w = expf(ls[s] - L) * sinkf;
    if (w == 0.f) continue;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = *reinterpret_cast<const float4*>(ob + (int64_t)s * kDV + 128 * i + 4 * lane);
      acc[i].x = fmaf(w, v.x, acc[i].x);
      acc[i].y = fmaf(w, v.y, acc[i].y);
      acc[i].z = fmaf(w, v.z, acc[i].z);
      acc[i].w = fmaf(w, v.w, acc[i].w);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 a = __floats2bfloat162_rn(acc[i].x, acc[i].y);
    __nv_bfloat162 b = __floats2bfloat162_rn(acc[i].z, acc[i].w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&a);
    pk.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(orow + 128 * i + 4 * lane) = pk;
  }
  if (lane == 0) p.lse[(int64_t)t * p.lse_stride_t + h] = L;
}

cudaError_t launch_combine(const KParams& p, cudaStream_t stream) {
  const int64_t warps = (int64_t)p.T * p.H;
  const int64_t blocks = (warps + 3) / 4;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  combine_kernel<<<(unsigned)blocks, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

// rows[t * rows_stride + s] = cache row of combined slot s of token t, or -1
// (second-list rows of the dual-cache form are encoded as rows1 + row).  The
// same slot routines as the attention kernels, with the dual-capable
// instantiation, which also serves one list (x_base INT32_MAX, topk2 0).
__global__ void resolve_kernel(const KParams p, int width, int32_t* rows, int64_t rows_stride) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)p.T * width) return;
  const int t = (int)(i / width), s = (int)(i % width);
  const TokSlots ts = token_slots<true>(p, t);
  int r = -1;
  if (s < ts.end && slot_readable<true>(p, s, ts.len1))
    r = resolve_slot<true>(p, bt_row_of(p, t), bt2_row_of(p, t), s, slot_index<true>(p, t, s));
  rows[(int64_t)t * rows_stride + s] = r;
}

cudaError_t launch_resolve(const KParams& p, int32_t* rows, int64_t rows_stride, cudaStream_t stream) {
  const int width = p.dual ? p.x_base + p.topk2 : p.topk;
  const int64_t n = (int64_t)p.T * width;
  const int64_t blocks = (n + 255) / 256;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  resolve_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, width, rows, rows_stride);
  return cudaGetLastError();
}

}  // namespace smla
