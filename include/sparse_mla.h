/*
 * sparse_mla.h -- C ABI of libsparse_mla.so: sparse MLA attention forward
 * (prefill and decode) for NVIDIA GB300 (sm_103a).
 *
 * What is computed.  For each query token t and head h, over the valid slots j
 * of the token's index row (see "Slots" below):
 *
 *   s_j      = sm_scale * < q[t,h,0:576], K[row_j] >
 *   m        = max_j s_j,   l = sum_j exp(s_j - m)
 *   out[t,h] = sum_j exp(s_j - m) V[row_j] / (l + exp(attn_sink[h] - m))   (bf16)
 *   lse[t,h] = m + log(l)                                                  (fp32)
 *
 * with K[r] the 576-vector of cache row r dequantised (512 e4m3 codes times
 * their per-128 fp32 scale, then 64 bf16 rope values) and V[r] = K[r][0:512].
 * Sources: FlashInfer PR #4802 "Refactor Sparse MLA SM120" (review note on the
 * DSv3.2 per-token KV layout: [0:512) e4m3, [512:528) 4 x fp32 scale, one per
 * 128-element tile, [528:656) 64 x bf16 rope; d_v == d_nope per its Summary;
 * page block 64; index row stride taken from the tensor; zero-token decode),
 * vLLM PR #57673 "[Perf][DSv4.1] Native-head Triton sparse MLA for SM90
 * few-head prefill" (Test Plan / Test Result: attn_sink, topk_length,
 * non-contiguous q/out views written in place), and the AppMana
 * forks-flash-mla-ampere-dsv4 releases page ("decode H6: warp-wide combine",
 * split-K decode merged by LSE).
 *
 * Readings where the pages are silent: attn_sink[h] is a logit in the units
 * of s_j that adds exp(attn_sink[h]) to the denominator only (NULL = no sink);
 * lse excludes the sink and uses the natural log; a token with no valid slot
 * gets out = 0 and lse = -inf.
 *
 * Slots.  Slot j of token t (j < topk) is valid iff
 *   j < clamp(topk_length[t], 0, topk)   (topk_length NULL: topk), and
 *   its index i = indices[t*idx_stride_t + j] resolves to a cache row:
 *     flat  (block_table NULL): row = i, 0 <= i < num_pages*64;
 *     paged: r = t / tokens_per_req (< bt_rows), page = i / 64 (< bt_cols),
 *            p = block_table[r*bt_stride + page] (0 <= p < num_pages),
 *            row = p*64 + i % 64.
 * -1 is padding.  Any other index that does not resolve is masked like -1 and
 * sets bit SMLA_ERRF_INDEX_RANGE in the device error word.  Index entries at
 * or past topk_length are not read.
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     keeps none of them after the call returns and never frees them.
 *   - Calls are asynchronous on the given stream (0 = legacy default stream).
 *     They do not synchronise and do not allocate device memory.
 *   - T == 0 returns SMLA_OK without launching anything.
 *   - Return codes: SMLA_OK, SMLA_ERR_INVALID (bad argument: the call did
 *     nothing), SMLA_ERR_UNSUPPORTED, SMLA_ERR_CUDA (a launch failed).
 *     sparse_mla_last_error() gives a message for the calling thread.
 *   - Range of the cache values: the kernels hold dequantised values in fp16,
 *     so every |code * scale| must be at most 65504 (scales at most 128,
 *     in either cache format).
 */
#ifndef SPARSE_MLA_H_
#define SPARSE_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* smla_stream_t;

enum {
  SMLA_OK = 0,
  SMLA_ERR_INVALID = 1,
  SMLA_ERR_UNSUPPORTED = 2,
  SMLA_ERR_CUDA = 3,
  SMLA_ERR_DEVICE = 4
};

/* Bits of the device error word (sparse_mla_get_error_word). */
enum {
  SMLA_ERRF_INDEX_RANGE = 1, /* an index other than -1 did not resolve (masked) */
  SMLA_ERRF_TIMEOUT = 2,     /* a bounded in-kernel wait gave up; outputs invalid */
  SMLA_ERRF_SCALE_RANGE = 4  /* a cache row scale above 128 was seen */
};

#define SMLA_D_QK 576
#define SMLA_D_V 512
#define SMLA_ROW_BYTES 656
#define SMLA_PAGE 64
#define SMLA_MAX_HEADS 128
#define SMLA_MAX_SPLITS 64

/*
 * Cache formats (the code bytes [0:512) of a 656-byte row; the per-128 fp32
 * scales and the bf16 rope are the same in both):
 *  SMLA_KV_E4M3  OCP FP8 E4M3FN codes, the DSv3.2 layout (FlashInfer PR
 *                #4802, KV layout note; power-of-two scales).
 *  SMLA_KV_INT8  signed int8 codes (two's complement), value = code * scale.
 *                The AppMana releases page names the INT8 latent-cache kernels
 *                (fwd_sparse_int8_decode_mla, fwd_sparse_int8_prefill_mla;
 *                "int8 width 1024" at the 16k footprint) but prints no byte
 *                layout; this keeps the DSv3.2 row layout with int8 codes in
 *                place of e4m3, the plainest reading.  Scales need not be
 *                powers of two; the kernels round them to fp16.
 */
#define SMLA_KV_E4M3 0
#define SMLA_KV_INT8 1

/*
 * Row layouts (FlashInfer PR #4802, review note on the KV layout comment of
 * the DSv3.2 decode kernel):
 *  SMLA_LAYOUT_ROPE64  [528, 656) holds 64 bf16 rope values; d_qk = 576 and
 *                      q is [T, H, 576] (head stride 576).
 *  SMLA_LAYOUT_NOPE    GLM53_NOPE: the same 656-byte row with d_rope = 0;
 *                      [528, 656) is reserved padding and is never read;
 *                      d_qk = 512 and q is [T, H, 512] (head stride 512).
 * GLM_NSA's arbitrary (not power-of-two) fp32 scales need no flag: every
 * scale is taken as stored (rounded to fp16 by the kernels).
 */
#define SMLA_LAYOUT_ROPE64 0
#define SMLA_LAYOUT_NOPE 1

/*
 * Arguments shared by prefill and decode.  Strides are in ELEMENTS of the
 * pointed-to type.
 *
 *  q            bf16 [T, H, 576]: head stride 576, token stride q_stride_t
 *               (>= H*576; a view into a wider buffer is fine).  With
 *               SMLA_LAYOUT_NOPE: [T, H, 512], head stride 512, q_stride_t
 *               >= H*512.
 *  kv           uint8 [num_pages, 64, 656], contiguous rows, 16-byte aligned.
 *  block_table  int32 [bt_rows, >= bt_cols] with row stride bt_stride, or
 *               NULL for flat row ids.  tokens_per_req query tokens share a
 *               block-table row (decode: request r owns tokens
 *               r*tokens_per_req ... ; needs bt_rows*tokens_per_req >= T).
 *  indices      int32 [T, >= topk]: row stride idx_stride_t (>= topk), last
 *               dimension contiguous.
 *  topk_length  int32 [T] or NULL.
 *  attn_sink    fp32 [H] or NULL.
 *  out          bf16 [T, H, 512]: head stride 512, token stride out_stride_t
 *               (>= H*512, multiple of 4), 8-byte aligned; written in place.
 *  lse          fp32 [T, H]: token stride lse_stride_t (>= H).
 *  kv_format    SMLA_KV_E4M3 or SMLA_KV_INT8 (see above).
 *  layout       SMLA_LAYOUT_ROPE64 or SMLA_LAYOUT_NOPE (see above); both
 *               caches of a dual call share it.  reserved1 must be 0.
 *  H in [1, 128]; T >= 0; topk >= 1.
 */
typedef struct smla_args {
  const void* q;
  int64_t q_stride_t;
  const uint8_t* kv;
  int64_t num_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  int32_t bt_rows;
  int32_t bt_cols;
  int32_t tokens_per_req;
  int32_t topk;
  const int32_t* indices;
  int64_t idx_stride_t;
  const int32_t* topk_length;
  const float* attn_sink;
  float sm_scale;
  int32_t T;
  int32_t H;
  int32_t kv_format; /* SMLA_KV_E4M3 (0) or SMLA_KV_INT8 (1), for every cache of the call */
  void* out;
  int64_t out_stride_t;
  float* lse;
  int64_t lse_stride_t;
  int32_t layout;
  int32_t reserved1;
} smla_args;

/*
 * Prefill: one pass over every token's selected rows, with gather, dequant,
 * QK^T, sink softmax, PV and the epilogue fused per token (the fused path of
 * the AppMana releases page, "Remove the legacy staged sparse-MLA prefill
 * kernel": no materialised gather).  H % 64 == 0 runs on the tcgen05/TMEM
 * kernel; other head counts run at their native width on the warp-MMA kernel
 * (vLLM PR #57673: no zero-padding of few heads to 64).
 */
int sparse_mla_prefill(const smla_args* args, smla_stream_t stream);

/*
 * Decode: the topk slots of each token are cut into num_splits contiguous
 * chunks (multiples of 64 slots); each chunk is attended by its own CTA,
 * which writes an fp32 partial (output normalised over its slots, sink-free,
 * and its LSE) to the caller's workspace; a combine kernel then merges the
 * partials with weights exp(lse_s - lse) and applies the sink (FlashInfer PR
 * #4802, "Runner and CUDA graphs": split-K scratch owned by the caller; AppMana
 * releases, "decode H6: warp-wide combine").  With one split (automatic for
 * few tokens x long lists) the attention kernel writes out and lse directly
 * and no combine runs; the workspace is then not touched.
 *
 *  num_splits   0 = automatic, else 1..64 (reduced so that no split is empty
 *               of slots: effective splits = ceil(topk / chunk)).
 *  workspace    device memory, 256-byte aligned, at least
 *               sparse_mla_decode_workspace_size(T, H, topk, num_splits)
 *               bytes; its contents on entry do not matter.  Calls that share a
 *               workspace must be ordered on one stream.
 */
int sparse_mla_decode(const smla_args* args, int32_t num_splits, void* workspace,
                      size_t workspace_bytes, smla_stream_t stream);

/*
 * Workspace bytes that sparse_mla_decode needs for these sizes on the
 * current device.  num_splits == 0 sizes for the automatic choice.  Returns 0
 * for invalid sizes.  T == 0 needs no workspace (returns 0).
 */
size_t sparse_mla_decode_workspace_size(int32_t T, int32_t H, int32_t topk,
                                        int32_t num_splits);

/*
 * The split count sparse_mla_decode uses for num_splits (0 = automatic).
 * The automatic choice minimises (CTA waves) x (per-CTA fixed cost + its
 * share of the 64-slot chunks) for the kernel that will run, and applies the
 * L2-footprint guard of FlashInfer PR #4802 (commit note on the analytical
 * cpb model: min(G, S) * cpb * W must fit in L2): when a token's rows are
 * gathered by more than one CTA (head groups of 64, or of the warp-MMA
 * kernel's width), split counts are not chosen whose rows streamed between a
 * row's first and last reader -- min(G, resident CTAs) x chunks per CTA x 64
 * rows x 656 bytes, G being the span of CTAs from the first reader to the
 * last, (head groups - 1) x splits + 1 in this grid's order -- exceed the
 * device's L2, unless none fits.  Returns 0 for invalid sizes.
 */
int32_t sparse_mla_decode_num_splits(int32_t T, int32_t H, int32_t topk, int32_t num_splits);

/*
 * The same choice for a device described by its SM count and L2 size in
 * bytes instead of the current one (host only: no CUDA call).  Returns 0 for
 * invalid sizes.
 */
int32_t sparse_mla_plan_num_splits(int32_t T, int32_t H, int32_t topk, int32_t num_splits, int32_t num_sms,
                                   int64_t l2_bytes);

/*
 * Index handling only: rows_out[t*rows_stride_t + j] (int32, device) receives
 * the physical cache row of slot j of token t, or -1 if the slot is invalid,
 * for j < topk.  Runs the same device resolution routine as the attention
 * kernels; used to check index handling bit for bit.
 */
int sparse_mla_resolve_rows(const smla_args* args, int32_t* rows_out, int64_t rows_stride_t,
                            smla_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word (SMLA_ERRF_* bits) into *out_flags.
 */
int sparse_mla_get_error_word(smla_stream_t stream, int32_t* out_flags);

/*
 * Limit, in nanoseconds of GPU global time, of every bounded in-kernel wait
 * of the calls made after it, on any thread (default 1000000000, one
 * second).  Returns the previous limit.  Every wait of the tcgen05 kernel on
 * an mbarrier is bounded, so that a pipeline stage that never completes ends
 * the CTA with an error status instead of a hang (FlashInfer PR #4802 page,
 * follow-up fix note on the DGX Spark hang: IO warps that no barrier counted
 * spun forever on mbarrier_wait_parity).  When a limit runs out, the CTA sets
 * SMLA_ERRF_TIMEOUT, stops every role, waits for its issued MMAs, frees its
 * tensor memory and returns without writing its outputs; the context stays
 * usable.  A waiting thread retries with a suspend-time hint of 20 us, so a
 * wait notices an exhausted limit (or another role's abort) within about
 * 20 us of it.  The limit in force is read when a call is made; calls
 * already queued keep theirs.
 */
uint64_t sparse_mla_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook for the path above: while on (non-zero), the producers of the
 * tcgen05 kernel (H % 64 == 0) gather nothing in the calls made after it, on
 * any thread, so the MMA issue's first wait is never completed and runs out
 * after the wait limit; the call ends with SMLA_ERRF_TIMEOUT and unwritten
 * outputs.  Off by default; returns the previous setting.  Not for use
 * outside tests.
 */
int32_t sparse_mla_set_test_stall(int32_t on);

/*
 * Decode without any device allocation -- no counterpart on the pages; added
 * for callers that cannot allocate device memory: a host engine that owns all
 * device memory through its own pool and gives a library only tensors and a
 * stream (cudaMalloc there fails or escapes the pool's accounting), or a
 * latency-critical path where an allocation and its implicit synchronisation
 * are not acceptable.  Same operation, kernels and results as
 * sparse_mla_decode, but the split partials live in a fixed array compiled
 * into the library (SMLA_NOALLOC_SCRATCH_BYTES per GPU, kept by every GPU
 * that loads it until the process exits).  The caller still passes every
 * input and output through args.
 *  - With num_splits == 0 the split count is the automatic choice lowered,
 *    if needed, to the largest count whose partials fit the array; such a
 *    call is never rejected for its size.  An explicit num_splits whose
 *    partials need more than SMLA_NOALLOC_SCRATCH_BYTES (see
 *    sparse_mla_decode_workspace_size) is rejected with SMLA_ERR_INVALID.
 *    A call that runs with one split has no partials and is never rejected.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, once per device); make that first call before any
 *    stream capture begins.
 *  - All calls on a device share the array, which keeps the last call's
 *    contents: calls that overlap on the GPU (different streams, no ordering
 *    between them) race.  Order them on one stream.
 *  - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define SMLA_NOALLOC_SCRATCH_BYTES (64u << 20)
int sparse_mla_decode_noalloc(const smla_args* args, int32_t num_splits, smla_stream_t stream);

/* Size in bytes of the no-alloc decode's built-in array, as compiled. */
size_t sparse_mla_noalloc_scratch_bytes(void);

/*
 * Dual-cache form: one softmax over the candidates of two index lists, each
 * into its own cache (FlashInfer PR #4802: the "DSv4 secondary cache" whose
 * index row stride comes from the tensor, the dual-cache decode-form calls
 * that must not ignore the secondary cache, and the "topk=1024+2176 dual"
 * decode shape).  args describes the first list and cache exactly as for
 * sparse_mla_prefill / sparse_mla_decode; extra describes the second:
 *
 *  kv, num_pages   the second cache, same row format and page size.
 *  block_table     int32 [bt_rows, >= bt_cols], row stride bt_stride, or
 *                  NULL for flat row ids; shares args->tokens_per_req.
 *  topk, indices, idx_stride_t, topk_length
 *                  the second list, with the same slot rules as the first.
 *
 * For each token the result is the sink softmax of the Introduction over the
 * union of both lists' valid slots (a row of each cache counts as many times
 * as it is selected).  The lists are laid end to end as "combined slots": the
 * first list padded with invalid slots to a multiple of 64, then the second,
 * i.e. sparse_mla_dual_width(topk, extra->topk) slots per token.  Decode
 * splits cut the combined slots into chunks of 64, so size its workspace as
 *   sparse_mla_decode_workspace_size(T, H, sparse_mla_dual_width(topk,
 *                                    extra->topk), num_splits).
 * Readings where the pages are silent: the sink enters once per token (not
 * once per list), and the second list's row ids are resolved in the second
 * cache only.  Extra constraint: both caches together hold fewer than 2^31
 * rows.  Error behaviour as for the single-list calls (SMLA_ERR_INVALID for
 * a bad extra; out-of-range indices of either list set SMLA_ERRF_INDEX_RANGE).
 */
typedef struct smla_extra_args {
  const uint8_t* kv;
  int64_t num_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  int32_t bt_rows;
  int32_t bt_cols;
  int32_t topk;
  int32_t reserved0; /* must be 0 */
  const int32_t* indices;
  int64_t idx_stride_t;
  const int32_t* topk_length;
} smla_extra_args;

/* Combined slots per token of the dual-cache form (0 for invalid sizes). */
int32_t sparse_mla_dual_width(int32_t topk, int32_t extra_topk);

int sparse_mla_prefill_dual(const smla_args* args, const smla_extra_args* extra, smla_stream_t stream);

int sparse_mla_decode_dual(const smla_args* args, const smla_extra_args* extra, int32_t num_splits,
                           void* workspace, size_t workspace_bytes, smla_stream_t stream);

/*
 * Index handling of the dual-cache form: rows_out[t*rows_stride_t + s] for
 * every combined slot s (rows_stride_t >= the combined width) receives the
 * first cache's row for a first-list slot, args->num_pages*64 + the second
 * cache's row for a second-list slot, or -1 for an invalid or padding slot.
 */
int sparse_mla_resolve_rows_dual(const smla_args* args, const smla_extra_args* extra, int32_t* rows_out,
                                 int64_t rows_stride_t, smla_stream_t stream);

/* Message for the last failing call on this thread ("" if none). */
const char* sparse_mla_last_error(void);

/* ABI version (bumped on any change of this header). */
int32_t sparse_mla_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SPARSE_MLA_H_ */
