// C ABI of libsparse_mla.so: argument validation, kernel choice and launches.
// The operations themselves are defined in include/sparse_mla.h.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <mutex>

#include "../../include/sparse_mla.h"
#include "smla_launch.h"

namespace {

thread_local char g_last_error[512] = "";

// Limit of every bounded in-kernel wait, for the calls that follow.
constexpr uint64_t kDefaultWaitNs = 1000000000ull;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int32_t> g_test_stall{0};

// One NVTX range per entry point (named after it), for profiler timelines.
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
};

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

// One error word per device; its address is looked up once per device.
__device__ int g_error_word;
constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];
int64_t g_l2_bytes[kMaxDevices];
std::mutex g_dev_mu;

int device_setup(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(SMLA_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(cudaGetLastError()));
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_err_ptr[dev] == nullptr) {
    int* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_error_word);
    if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    int l2 = 0;
    e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    g_num_sms[dev] = sms;
    g_l2_bytes[dev] = l2;
    g_err_ptr[dev] = ptr;
  }
  *dev_out = dev;
  return SMLA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
// The tcgen05 kernel's load policy for a cache of `bytes`: 0 while it fits in
// a quarter of L2 (rows come from L2: one burst of loads per tile), 1 beyond
// that (rows mostly from HBM: early per-group loads and an L2 prefetch one
// tile ahead), 2 beyond L2 itself (also 256 bytes per row and load
// instruction, the 128-dim groups released in pairs).  Policy 2 measured 3%
// faster on a 1.37 GB decode cache and 6% on a 1.7 GB dual-cache decode, but
// slower on an 86 MB cache, whose rows L2 partly keeps.
int32_t load_policy(int64_t bytes, int64_t l2) { return bytes > l2 ? 2 : (bytes > l2 / 4 ? 1 : 0); }

int validate(const smla_args* a) {
  if (a == nullptr) return fail(SMLA_ERR_INVALID, "args is NULL");
  if (a->T < 0) return fail(SMLA_ERR_INVALID, "T = %d < 0", a->T);
  if (a->H < 1 || a->H > SMLA_MAX_HEADS) return fail(SMLA_ERR_INVALID, "H = %d not in [1, 128]", a->H);
  if (a->topk < 1) return fail(SMLA_ERR_INVALID, "topk = %d < 1", a->topk);
  if (a->kv_format != SMLA_KV_E4M3 && a->kv_format != SMLA_KV_INT8)
    return fail(SMLA_ERR_INVALID, "kv_format = %d is neither SMLA_KV_E4M3 nor SMLA_KV_INT8", a->kv_format);
  if (a->layout != SMLA_LAYOUT_ROPE64 && a->layout != SMLA_LAYOUT_NOPE)
    return fail(SMLA_ERR_INVALID, "layout = %d is neither SMLA_LAYOUT_ROPE64 nor SMLA_LAYOUT_NOPE", a->layout);
  if (a->reserved1 != 0) return fail(SMLA_ERR_INVALID, "reserved1 must be 0");
  if (!(a->sm_scale == a->sm_scale) || a->sm_scale > 3.0e38f || a->sm_scale < -3.0e38f)
    return fail(SMLA_ERR_INVALID, "sm_scale is not finite");
  if (a->T == 0) return SMLA_OK;
  if (!a->q || !a->indices || !a->out || !a->lse)
    return fail(SMLA_ERR_INVALID, "q, indices, out and lse must be non-NULL");
  if (a->num_pages < 0 || a->num_pages * SMLA_PAGE > 0x7FFFFFFFLL)
    return fail(SMLA_ERR_INVALID, "num_pages = %lld out of range", (long long)a->num_pages);
  if (a->num_pages > 0 && !a->kv) return fail(SMLA_ERR_INVALID, "kv is NULL");
  if (a->kv && !aligned(a->kv, 16)) return fail(SMLA_ERR_INVALID, "kv must be 16-byte aligned");
  if (a->q_stride_t < (int64_t)a->H * (a->layout == SMLA_LAYOUT_NOPE ? 512 : SMLA_D_QK))
    return fail(SMLA_ERR_INVALID, "q_stride_t = %lld < H*d_qk", (long long)a->q_stride_t);
  if (a->out_stride_t < (int64_t)a->H * SMLA_D_V || a->out_stride_t % 4 != 0)
    return fail(SMLA_ERR_INVALID, "out_stride_t = %lld must be >= H*512 and a multiple of 4",
                (long long)a->out_stride_t);
  if (a->lse_stride_t < a->H) return fail(SMLA_ERR_INVALID, "lse_stride_t < H");
  if (a->idx_stride_t < a->topk) return fail(SMLA_ERR_INVALID, "idx_stride_t < topk");
  if (!aligned(a->q, 2) || !aligned(a->out, 8) || !aligned(a->lse, 4) || !aligned(a->indices, 4))
    return fail(SMLA_ERR_INVALID, "misaligned q/out/lse/indices (need 2/8/4/4 bytes)");
  if (a->topk_length && !aligned(a->topk_length, 4)) return fail(SMLA_ERR_INVALID, "misaligned topk_length");
  if (a->attn_sink && !aligned(a->attn_sink, 4)) return fail(SMLA_ERR_INVALID, "misaligned attn_sink");
  if (a->block_table) {
    if (a->tokens_per_req < 1) return fail(SMLA_ERR_INVALID, "tokens_per_req < 1");
    if (a->bt_cols < 1 || a->bt_stride < a->bt_cols || a->bt_rows < 1)
      return fail(SMLA_ERR_INVALID, "bad block table shape (rows %d, cols %d, stride %lld)", a->bt_rows,
                  a->bt_cols, (long long)a->bt_stride);
    if ((int64_t)a->bt_rows * a->tokens_per_req < a->T)
      return fail(SMLA_ERR_INVALID, "block table has %d rows for %d tokens at %d tokens/request", a->bt_rows,
                  a->T, a->tokens_per_req);
    if (!aligned(a->block_table, 4)) return fail(SMLA_ERR_INVALID, "misaligned block_table");
  }
  return SMLA_OK;
}

smla::KParams make_params(const smla_args* a, int dev) {
  smla::KParams p;
  memset(&p, 0, sizeof(p));
  p.q = static_cast<const __nv_bfloat16*>(a->q);
  p.q_stride_t = a->q_stride_t;
  p.kv = a->kv;
  p.num_pages = a->num_pages;
  p.block_table = a->block_table;
  p.bt_stride = a->bt_stride;
  p.bt_rows = a->bt_rows;
  p.bt_cols = a->bt_cols;
  p.tokens_per_req = a->block_table ? a->tokens_per_req : 1;
  p.indices = a->indices;
  p.idx_stride_t = a->idx_stride_t;
  p.topk = a->topk;
  p.topk_length = a->topk_length;
  p.attn_sink = a->attn_sink;
  p.sm_scale = a->sm_scale;
  p.T = a->T;
  p.H = a->H;
  p.out = static_cast<__nv_bfloat16*>(a->out);
  p.out_stride_t = a->out_stride_t;
  p.lse = a->lse;
  p.lse_stride_t = a->lse_stride_t;
  p.num_splits = 1;
  p.split_len = ((a->topk + 63) / 64) * 64;
  // The gathered rows of a cache within a quarter of L2 are re-read from L2
  // after their first touch; a larger cache (long-context decode, 100k-token
  // prefill) is read mostly from HBM, which the tcgen05 kernel's producers
  // meet with L2 prefetch and earlier register loads.
  p.big_cache = load_policy((int64_t)a->num_pages * SMLA_PAGE * SMLA_ROW_BYTES, g_l2_bytes[dev]);
  p.err = g_err_ptr[dev];
  p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  p.test_stall = g_test_stall.load(std::memory_order_relaxed);
  p.kv_format = a->kv_format;
  p.nope = a->layout == SMLA_LAYOUT_NOPE ? 1 : 0;
  // one list: the second-list fields stay inert
  p.dual = 0;
  p.x_base = 0x7FFFFFFF;
  p.rows1 = (int32_t)(a->num_pages * SMLA_PAGE);
  p.topk2 = 0;
  return p;
}

// Combined slot width of the dual-cache form: the first list padded to whole
// 64-slot chunks, then the second list.
int64_t dual_width(int64_t topk, int64_t topk2) { return ((topk + 63) / 64) * 64 + topk2; }

int validate_extra(const smla_args* a, const smla_extra_args* x) {
  if (x == nullptr) return fail(SMLA_ERR_INVALID, "extra is NULL");
  if (x->reserved0 != 0) return fail(SMLA_ERR_INVALID, "extra->reserved0 must be 0");
  if (x->topk < 1) return fail(SMLA_ERR_INVALID, "extra->topk = %d < 1", x->topk);
  if (dual_width(a->topk, x->topk) > (1 << 24))
    return fail(SMLA_ERR_INVALID, "combined slot width %lld too large", (long long)dual_width(a->topk, x->topk));
  if (a->T == 0) return SMLA_OK;
  if (!x->indices) return fail(SMLA_ERR_INVALID, "extra->indices is NULL");
  if (x->idx_stride_t < x->topk) return fail(SMLA_ERR_INVALID, "extra->idx_stride_t < extra->topk");
  if (x->num_pages < 0 || x->num_pages * SMLA_PAGE > 0x7FFFFFFFLL)
    return fail(SMLA_ERR_INVALID, "extra->num_pages = %lld out of range", (long long)x->num_pages);
  if ((a->num_pages + x->num_pages) * SMLA_PAGE > 0x7FFFFFFFLL)
    return fail(SMLA_ERR_INVALID, "the two caches hold more than 2^31 - 1 rows together");
  if (x->num_pages > 0 && !x->kv) return fail(SMLA_ERR_INVALID, "extra->kv is NULL");
  if (x->kv && !aligned(x->kv, 16)) return fail(SMLA_ERR_INVALID, "extra->kv must be 16-byte aligned");
  if (!aligned(x->indices, 4)) return fail(SMLA_ERR_INVALID, "misaligned extra->indices");
  if (x->topk_length && !aligned(x->topk_length, 4)) return fail(SMLA_ERR_INVALID, "misaligned extra->topk_length");
  if (x->block_table) {
    if (a->tokens_per_req < 1) return fail(SMLA_ERR_INVALID, "tokens_per_req < 1");
    if (x->bt_cols < 1 || x->bt_stride < x->bt_cols || x->bt_rows < 1)
      return fail(SMLA_ERR_INVALID, "bad extra block table shape (rows %d, cols %d, stride %lld)", x->bt_rows,
                  x->bt_cols, (long long)x->bt_stride);
    if ((int64_t)x->bt_rows * a->tokens_per_req < a->T)
      return fail(SMLA_ERR_INVALID, "extra block table has %d rows for %d tokens at %d tokens/request",
                  x->bt_rows, a->T, a->tokens_per_req);
    if (!aligned(x->block_table, 4)) return fail(SMLA_ERR_INVALID, "misaligned extra->block_table");
  }
  return SMLA_OK;
}

smla::KParams make_params_dual(const smla_args* a, const smla_extra_args* x, int dev) {
  smla::KParams p = make_params(a, dev);
  p.dual = 1;
  p.x_base = (int32_t)(((a->topk + 63) / 64) * 64);
  p.topk2 = x->topk;
  p.kv2 = x->kv;
  p.num_pages2 = x->num_pages;
  p.block_table2 = x->block_table;
  p.bt2_stride = x->bt_stride;
  p.bt2_cols = x->bt_cols;
  p.indices2 = x->indices;
  p.idx2_stride_t = x->idx_stride_t;
  p.topk_length2 = x->topk_length;
  if (x->block_table) p.tokens_per_req = a->tokens_per_req;
  p.split_len = (int32_t)(((dual_width(a->topk, x->topk) + 63) / 64) * 64);
  p.big_cache = load_policy((a->num_pages + x->num_pages) * SMLA_PAGE * SMLA_ROW_BYTES, g_l2_bytes[dev]);
  return p;
}

// Decode split choice.  An explicit request is honoured up to the number of
// 64-slot chunks; the automatic choice minimises waves x CTA length for the
// kernel that will run (measured against split sweeps on GB300), subject to
// an L2-footprint guard.
//
// The guard (FlashInfer PR #4802, commit note on the analytical cpb model:
// the "L2-footprint guard rail" over min(G, S) * cpb * W): when the rows of a
// token are gathered by more than one CTA (one per head group, R > 1), the
// later readers find them in L2 only while the rows streamed between the
// first and the last read -- min(G, resident CTA slots) x 64-slot chunks per
// CTA x 64 rows x 656 bytes -- fit in L2.  Split counts beyond it are
// excluded; if none fits, the unconstrained pick stands.  G is the span of
// CTAs, in dispatch order, from a row's first reader to its last: this grid
// numbers the head-group CTAs of one (token, split) S apart, so G = (R-1) S
// + 1 and all readers of a row normally run at the same time.  (Taking G as
// the whole grid, as for a kernel whose readers are a grid apart, moved H=128
// decode on GB300 from one split to two, measured 19-24% slower.)  With one
// CTA per token and split (R == 1) no row is read twice and the guard does
// not apply.
constexpr double kChunkBytes = 64.0 * SMLA_ROW_BYTES;

struct SplitModel {
  int64_t base;     // CTAs per split: tokens x head-group CTAs per token
  int64_t slots;    // resident CTA slots: SMs x CTAs per SM
  int rereads;      // CTAs that gather the same rows (head groups per token)
  double fixed;     // per-CTA fixed cost, in chunk units
  double per_chunk; // cost of one 64-slot chunk
  bool tile128;     // cost in 128-slot tiles (tcgen05 kernel): (chunks + 1) / 2
  double merge;     // cost per split of the combine's merge
};

SplitModel split_model(int H, int num_sms) {
  const int sms = num_sms > 0 ? num_sms : 148;
  SplitModel m;
  if (smla::tc_supported(H)) {
    // tcgen05 kernel: one CTA per SM, each paying a fixed cost (q load, first
    // gather latency, epilogue: about 2.5 tiles' worth) plus one unit per
    // 128-row tile
    m = SplitModel{H / 64, sms, H / 64, 2.5, 1.0, true, 0.0};
  } else {
    // warp-MMA kernel: a wave of SMs x resident CTAs (4 per SM for 8-head
    // CTAs, 2 for 16-head CTAs), a fixed cost of about 1.5 64-slot chunks, one
    // unit per chunk, and 0.05 units per split for the combine's merge
    const int hpc = smla::heads_per_cta(H);
    const int groups = (H + hpc - 1) / hpc;
    m = SplitModel{groups, (int64_t)sms * (hpc == 8 ? 4 : 2), groups, 1.5, 1.0, false, 0.05};
  }
  return m;
}

int splits_for(int T, int H, int topk, int num_splits, int num_sms, int64_t l2_bytes) {
  const int chunks = (topk + 63) / 64;
  int S = 1;
  if (num_splits > 0) {
    S = num_splits < chunks ? num_splits : chunks;
  } else {
    const SplitModel m = split_model(H, num_sms);
    const int64_t base = (int64_t)T * m.base;
    double best_any = 0.0, best_fit = 0.0;
    int s_any = 1, s_fit = 0;
    for (int s = 1; s <= SMLA_MAX_SPLITS && s <= chunks; ++s) {
      const int per = (chunks + s - 1) / s;                 // 64-slot chunks per split
      if (s > 1 && (chunks + per - 1) / per < s) continue;  // same partition as a smaller s
      const int64_t ctas = base * s;
      const double waves = (double)((ctas + m.slots - 1) / m.slots);
      const double len = m.tile128 ? (double)((per + 1) / 2) : (double)per * m.per_chunk;
      const double cost = waves * (m.fixed + len) + m.merge * s;
      if (s == 1 || cost < best_any * 0.97) {
        best_any = cost;
        s_any = s;
      }
      const int64_t span = (int64_t)(m.rereads - 1) * s + 1;  // CTAs from a row's first reader to its last
      const double footprint = (double)(span < m.slots ? span : m.slots) * per * kChunkBytes;
      const bool fits = m.rereads <= 1 || l2_bytes <= 0 || footprint <= (double)l2_bytes;
      if (fits && (s_fit == 0 || cost < best_fit * 0.97)) {
        best_fit = cost;
        s_fit = s;
      }
    }
    S = s_fit > 0 ? s_fit : s_any;
  }
  if (S < 1) S = 1;
  // effective count: chunks per split rounded up, then splits that hold slots
  const int per = (chunks + S - 1) / S;
  return (chunks + per - 1) / per;
}

size_t ws_bytes(int64_t T, int64_t H, int64_t S) {
  const size_t o = (size_t)(T * H * S * SMLA_D_V) * sizeof(float);
  const size_t l = (size_t)(T * H * S) * sizeof(float);
  return ((o + 255) / 256) * 256 + ((l + 255) / 256) * 256;
}

// Split launch plus combine over a slot width of `width` (topk, or the
// combined width of the dual-cache form).
int decode_launch(smla::KParams p, int width, int num_splits, void* workspace, size_t workspace_bytes,
                  smla_stream_t stream, int dev) {
  const int S = splits_for(p.T, p.H, width, num_splits, g_num_sms[dev], g_l2_bytes[dev]);
  const size_t need = ws_bytes(p.T, p.H, S);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(SMLA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
  if (!aligned(workspace, 256)) return fail(SMLA_ERR_INVALID, "workspace must be 256-byte aligned");
  const int chunks = (width + 63) / 64;
  p.num_splits = S;
  p.split_len = ((chunks + S - 1) / S) * 64;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (S == 1) {
    // one split: the attention kernel writes out and lse itself (the prefill
    // epilogue), with no partials and no combine
    cudaError_t e = smla::launch_attention(p, st);
    if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    return SMLA_OK;
  }
  const size_t o_bytes = (size_t)p.T * p.H * S * SMLA_D_V * sizeof(float);
  p.ws_o = static_cast<float*>(workspace);
  p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((o_bytes + 255) / 256) * 256);
  cudaError_t e = smla::launch_attention(p, st);
  if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "decode split launch: %s", cudaGetErrorString(e));
  e = smla::launch_combine(p, st);
  if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "decode combine launch: %s", cudaGetErrorString(e));
  return SMLA_OK;
}

}  // namespace

extern "C" {

int32_t sparse_mla_abi_version(void) { return 5; }

uint64_t sparse_mla_set_wait_limit_ns(uint64_t ns) { return g_wait_ns.exchange(ns); }

int32_t sparse_mla_set_test_stall(int32_t on) { return g_test_stall.exchange(on != 0 ? 1 : 0); }

const char* sparse_mla_last_error(void) { return g_last_error; }

int sparse_mla_prefill(const smla_args* a, smla_stream_t stream) {
  g_last_error[0] = 0;
  Range range("sparse_mla_prefill");
  int rc = validate(a);
  if (rc != SMLA_OK) return rc;
  if (a->T == 0) return SMLA_OK;
  int dev;
  if ((rc = device_setup(&dev)) != SMLA_OK) return rc;
  smla::KParams p = make_params(a, dev);
  cudaError_t e = smla::launch_attention(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  return SMLA_OK;
}

int32_t sparse_mla_plan_num_splits(int32_t T, int32_t H, int32_t topk, int32_t num_splits, int32_t num_sms,
                                   int64_t l2_bytes) {
  if (T < 0 || H < 1 || H > SMLA_MAX_HEADS || topk < 1 || num_splits < 0 || num_splits > SMLA_MAX_SPLITS ||
      num_sms < 1 || l2_bytes < 0)
    return 0;
  return splits_for(T, H, topk, num_splits, num_sms, l2_bytes);
}

int32_t sparse_mla_decode_num_splits(int32_t T, int32_t H, int32_t topk, int32_t num_splits) {
  if (T < 0 || H < 1 || H > SMLA_MAX_HEADS || topk < 1 || num_splits < 0 || num_splits > SMLA_MAX_SPLITS) return 0;
  int sms = 0;
  int64_t l2 = 0;
  if (num_splits == 0) {
    int dev;
    if (device_setup(&dev) != SMLA_OK) return 0;
    sms = g_num_sms[dev];
    l2 = g_l2_bytes[dev];
  }
  return splits_for(T, H, topk, num_splits, sms, l2);
}

size_t sparse_mla_decode_workspace_size(int32_t T, int32_t H, int32_t topk, int32_t num_splits) {
  if (T <= 0) return 0;
  const int S = sparse_mla_decode_num_splits(T, H, topk, num_splits);
  if (S <= 0) return 0;
  return ws_bytes(T, H, S);
}

int sparse_mla_decode(const smla_args* a, int32_t num_splits, void* workspace, size_t workspace_bytes,
                      smla_stream_t stream) {
  g_last_error[0] = 0;
  Range range("sparse_mla_decode");
  int rc = validate(a);
  if (rc != SMLA_OK) return rc;
  if (num_splits < 0 || num_splits > SMLA_MAX_SPLITS)
    return fail(SMLA_ERR_INVALID, "num_splits = %d not in [0, 64]", num_splits);
  if (a->T == 0) return SMLA_OK;  // zero tokens: nothing to launch
  int dev;
  if ((rc = device_setup(&dev)) != SMLA_OK) return rc;
  return decode_launch(make_params(a, dev), a->topk, num_splits, workspace, workspace_bytes, stream, dev);
}

int32_t sparse_mla_dual_width(int32_t topk, int32_t extra_topk) {
  if (topk < 1 || extra_topk < 1 || dual_width(topk, extra_topk) > (1 << 24)) return 0;
  return (int32_t)dual_width(topk, extra_topk);
}

int sparse_mla_prefill_dual(const smla_args* a, const smla_extra_args* x, smla_stream_t stream) {
  g_last_error[0] = 0;
  Range range("sparse_mla_prefill_dual");
  int rc = validate(a);
  if (rc != SMLA_OK) return rc;
  if ((rc = validate_extra(a, x)) != SMLA_OK) return rc;
  if (a->T == 0) return SMLA_OK;
  int dev;
  if ((rc = device_setup(&dev)) != SMLA_OK) return rc;
  smla::KParams p = make_params_dual(a, x, dev);
  cudaError_t e = smla::launch_attention(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "dual prefill launch: %s", cudaGetErrorString(e));
  return SMLA_OK;
}

int sparse_mla_decode_dual(const smla_args* a, const smla_extra_args* x, int32_t num_splits, void* workspace,
                           size_t workspace_bytes, smla_stream_t stream) {
  g_last_error[0] = 0;
  Range range("sparse_mla_decode_dual");
  int rc = validate(a);
  if (rc != SMLA_OK) return rc;
  if ((rc = validate_extra(a, x)) != SMLA_OK) return rc;
  if (num_splits < 0 || num_splits > SMLA_MAX_SPLITS)
    return fail(SMLA_ERR_INVALID, "num_splits = %d not in [0, 64]", num_splits);
  if (a->T == 0) return SMLA_OK;
  int dev;
  if ((rc = device_setup(&dev)) != SMLA_OK) return rc;
  return decode_launch(make_params_dual(a, x, dev), (int)dual_width(a->topk, x->topk), num_splits, workspace,
                       workspace_bytes, stream, dev);
}

int sparse_mla_resolve_rows(const smla_args* a, int32_t* rows_out, int64_t rows_stride_t, smla_stream_t stream) {
  g_last_error[0] = 0;
  Range range("sparse_mla_resolve_rows");
  int rc = validate(a);
  if (rc != SMLA_OK) return rc;
  if (a->T == 0) return SMLA_OK;
  if (rows_out == nullptr || rows_stride_t < a->topk)
    return fail(SMLA_ERR_INVALID, "rows_out is NULL or rows_stride_t < topk");
  int dev;
  if ((rc = device_setup(&dev)) != SMLA_OK) return rc;
  smla::KParams p = make_params(a, dev);
  cudaError_t e = smla::launch_resolve(p, rows_out, rows_stride_t, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "resolve launch: %s", cudaGetErrorString(e));
  return SMLA_OK;
}

int sparse_mla_resolve_rows_dual(const smla_args* a, const smla_extra_args* x, int32_t* rows_out,
                                 int64_t rows_stride_t, smla_stream_t stream) {
  g_last_error[0] = 0;
  Range range("sparse_mla_resolve_rows_dual");
  int rc = validate(a);
  if (rc != SMLA_OK) return rc;
  if ((rc = validate_extra(a, x)) != SMLA_OK) return rc;
  if (a->T == 0) return SMLA_OK;
  const int64_t width = dual_width(a->topk, x->topk);
  if (rows_out == nullptr || rows_stride_t < width)
    return fail(SMLA_ERR_INVALID, "rows_out is NULL or rows_stride_t < the combined width %lld", (long long)width);
  int dev;
  if ((rc = device_setup(&dev)) != SMLA_OK) return rc;
  smla::KParams p = make_params_dual(a, x, dev);
  cudaError_t e = smla::launch_resolve(p, rows_out, rows_stride_t, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "resolve launch: %s", cudaGetErrorString(e));
  return SMLA_OK;
}

int sparse_mla_get_error_word(smla_stream_t stream, int32_t* out_flags) {
  g_last_error[0] = 0;
  if (out_flags == nullptr) return fail(SMLA_ERR_INVALID, "out_flags is NULL");
  int dev;
  int rc = device_setup(&dev);
  if (rc != SMLA_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int));
  if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "read error word: %s", cudaGetErrorString(e));
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
  if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "clear error word: %s", cudaGetErrorString(e));
  *out_flags = v;
  return SMLA_OK;
}

}  // extern "C"

// Accessors for other translation units of the library (same behaviour as the
// helpers above; nothing here changes the entry points defined in this file).
namespace smla {
namespace host {
int validate_args(const smla_args* a) { return validate(a); }
int setup_device(int* dev) { return device_setup(dev); }
KParams params_for(const smla_args* a, int dev) { return make_params(a, dev); }
int num_sms(int dev) { return g_num_sms[dev]; }
int64_t l2_bytes(int dev) { return g_l2_bytes[dev]; }
int decode_splits(int T, int H, int topk, int num_splits, int sms, int64_t l2_bytes) {
  return splits_for(T, H, topk, num_splits, sms, l2_bytes);
}
size_t decode_ws_bytes(int64_t T, int64_t H, int64_t S) { return ws_bytes(T, H, S); }
int set_error(int code, const char* msg) { return fail(code, "%s", msg); }
void clear_error() { g_last_error[0] = 0; }
}  // namespace host
}  // namespace smla
