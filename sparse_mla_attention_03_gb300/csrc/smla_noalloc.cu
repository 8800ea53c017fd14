// Decode entry point that allocates nothing: the split-K partials live in a
// fixed-size array compiled into the library instead of a caller workspace.
//
// Some callers cannot allocate device memory: a host engine that owns all
// device memory through its own pool allocator and hands a kernel library
// only tensors and a stream (a cudaMalloc there either fails because the pool
// reserved the memory, or escapes the engine's accounting), and callers on a
// latency-critical path where a device allocation and its implicit
// synchronisation are not acceptable.  For them, sparse_mla_decode_noalloc
// runs the same split and combine kernels as sparse_mla_decode on this array.
#include <stdio.h>

#include <mutex>

#include "../../include/sparse_mla.h"
#include "smla_launch.h"

namespace smla {
namespace host {
int validate_args(const smla_args* a);
int setup_device(int* dev);
KParams params_for(const smla_args* a, int dev);
int num_sms(int dev);
int64_t l2_bytes(int dev);
int decode_splits(int T, int H, int topk, int num_splits, int sms, int64_t l2_bytes);
size_t decode_ws_bytes(int64_t T, int64_t H, int64_t S);
int set_error(int code, const char* msg);
void clear_error();
}  // namespace host
}  // namespace smla

namespace {

// Scratch for the split partials: fp32 outputs [T, H, S, 512] then LSEs
// [T, H, S].  Every GPU that loads this module keeps it until the process
// exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SMLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  In host code
// g_noalloc_scratch names a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.
int scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(no-alloc scratch) failed: %s", cudaGetErrorString(e));
      return smla::host::set_error(SMLA_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SMLA_OK;
}

}  // namespace

extern "C" size_t sparse_mla_noalloc_scratch_bytes(void) { return sizeof(g_noalloc_scratch); }

extern "C" int sparse_mla_decode_noalloc(const smla_args* a, int32_t num_splits, smla_stream_t stream) {
  smla::host::clear_error();
  int rc = smla::host::validate_args(a);
  if (rc != SMLA_OK) return rc;
  if (num_splits < 0 || num_splits > SMLA_MAX_SPLITS)
    return smla::host::set_error(SMLA_ERR_INVALID, "num_splits must be in [0, 64]");
  if (a->T == 0) return SMLA_OK;
  int dev = 0;
  if ((rc = smla::host::setup_device(&dev)) != SMLA_OK) return rc;
  if (dev >= kMaxDev) return smla::host::set_error(SMLA_ERR_UNSUPPORTED, "device ordinal above 63");
  int S = smla::host::decode_splits(a->T, a->H, a->topk, num_splits, smla::host::num_sms(dev),
                                    smla::host::l2_bytes(dev));
  if (num_splits == 0) {
    // automatic choice: the largest split count up to the model's pick whose
    // partials fit the array (one split needs none, so some count always fits)
    while (S > 1 && smla::host::decode_ws_bytes(a->T, a->H, S) > sizeof(g_noalloc_scratch))
      S = smla::host::decode_splits(a->T, a->H, a->topk, S - 1, 0, 0);
  }
  smla::KParams p = smla::host::params_for(a, dev);
  const int chunks = (a->topk + 63) / 64;
  p.num_splits = S;
  p.split_len = ((chunks + S - 1) / S) * 64;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (S == 1) {  // one split: final outputs straight from the attention kernel, no scratch
    cudaError_t e = smla::launch_attention(p, st);
    if (e != cudaSuccess) return smla::host::set_error(SMLA_ERR_CUDA, cudaGetErrorString(e));
    return SMLA_OK;
  }
  const size_t need = smla::host::decode_ws_bytes(a->T, a->H, S);
  if (need > (size_t)SMLA_NOALLOC_SCRATCH_BYTES) {
    char msg[320];
    snprintf(msg, sizeof(msg),
             "sparse_mla_decode_noalloc: T=%d, H=%d, %d splits need %zu bytes of scratch but the built-in "
             "array holds %zu; use fewer tokens or splits per call, or sparse_mla_decode with a workspace",
             a->T, a->H, S, need, (size_t)SMLA_NOALLOC_SCRATCH_BYTES);
    return smla::host::set_error(SMLA_ERR_INVALID, msg);
  }
  void* scratch = nullptr;
  if ((rc = scratch_address(dev, &scratch)) != SMLA_OK) return rc;
  // Every partial slot [t, h, s] is written by the split kernel before the
  // combine reads it (empty splits write lse = -inf), so nothing left in the
  // array by an earlier call needs clearing.
  const size_t o_bytes = (size_t)a->T * a->H * S * SMLA_D_V * sizeof(float);
  p.ws_o = static_cast<float*>(scratch);
  p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(scratch) + ((o_bytes + 255) / 256) * 256);
  cudaError_t e = smla::launch_attention(p, st);
  if (e != cudaSuccess) return smla::host::set_error(SMLA_ERR_CUDA, cudaGetErrorString(e));
  e = smla::launch_combine(p, st);
  if (e != cudaSuccess) return smla::host::set_error(SMLA_ERR_CUDA, cudaGetErrorString(e));
  return SMLA_OK;
}
