// Shared device-side definitions for the sparse MLA kernels (sm_103a).
//
// Row format (FlashInfer PR #4802 "Refactor Sparse MLA SM120", review note on
// the DSv3.2 per-token KV layout): 656 bytes per cached token,
//   [0, 512)   512 x e4m3 "nope" codes
//   [512, 528) 4 x fp32 scale, one per 128 codes (powers of two)
//   [528, 656) 64 x bf16 rope values
// cached in pages of 64 rows.  K of a row is the 576-vector (nope*scale, rope);
// V is its first 512 entries (d_v == d_nope, same PR, Summary).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace smla {

constexpr int kRowBytes = 656;
constexpr int kDNope = 512;
constexpr int kDRope = 64;
constexpr int kDQK = 576;
constexpr int kDV = 512;
constexpr int kPage = 64;
constexpr int kScaleOff = 512;
constexpr int kRopeOff = 528;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device error word bits (read back with sparse_mla_get_error_word).
enum : int {
  kErrIndexRange = 1,  // an index other than -1 was out of range (masked like -1)
  kErrTimeout = 2,     // a bounded wait gave up
  kErrScaleRange = 4,  // a row scale outside the supported range was seen
};

// Kernel parameters (by value).  Pointers are device pointers.
struct KParams {
  const __nv_bfloat16* q;
  int64_t q_stride_t;  // elements between tokens; heads are 576 apart
  const uint8_t* kv;
  int64_t num_pages;
  const int32_t* block_table;  // nullptr: flat row ids
  int64_t bt_stride;
  int32_t bt_rows;
  int32_t bt_cols;
  int32_t tokens_per_req;
  const int32_t* indices;
  int64_t idx_stride_t;
  int32_t topk;
  const int32_t* topk_length;  // nullptr: topk
  const float* attn_sink;      // nullptr: no sink
  float sm_scale;
  int32_t T;
  int32_t H;
  __nv_bfloat16* out;
  int64_t out_stride_t;
  float* lse;
  int64_t lse_stride_t;
  // split-K decode (num_splits == 1 and ws_o == nullptr: write final outputs)
  int32_t num_splits;
  int32_t split_len;  // slots per split, multiple of the tile width
  float* ws_o;        // [T, H, S, 512] fp32 partial outputs (normalised, sink-free)
  float* ws_lse;      // [T, H, S] fp32 partial LSE (natural log)
  int32_t big_cache;   // load policy: 0 cache within a quarter of L2, 1 larger (rows mostly
                       // from HBM), 2 larger than L2 itself
  // Dual-cache form: a second list of slots into a second cache follows the
  // first list, whose width is padded to a multiple of 64 slots.  Unused
  // (dual 0, x_base INT32_MAX, topk2 0) for one list.
  int32_t dual;
  int32_t x_base;              // first combined slot of the second list
  int32_t rows1;               // num_pages * 64: second-cache rows are encoded as rows1 + row
  int32_t topk2;
  const uint8_t* kv2;
  int64_t num_pages2;
  const int32_t* block_table2;  // nullptr: flat row ids
  int64_t bt2_stride;
  int32_t bt2_cols;
  int32_t kv_format;  // 0: e4m3 codes, 1: int8 codes (both caches)
  int32_t nope;       // 1: no rope (q is [T, H, 512]; row bytes [528, 656) are never read)
  int32_t pad_;
  const int32_t* indices2;
  int64_t idx2_stride_t;
  const int32_t* topk_length2;  // nullptr: topk2
  int* err;           // device error word
  uint64_t wait_ns;   // limit of each bounded in-kernel wait (GPU global time)
  int32_t test_stall; // test hook: the tcgen05 kernel's producers gather nothing
  int32_t pad2_;
};

// ---------------------------------------------------------------------------
// Slot validity and address translation.
// Slot j of token t is valid iff j < clamp(topk_length[t], 0, topk) and its
// index is in range; -1 is silent padding, any other out-of-range value is
// masked the same way and flagged.  Flat: row = idx.  Paged: row =
// block_table[t / tokens_per_req][idx / 64] * 64 + idx % 64.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int token_len(const KParams& p, int t) {
  if (p.topk_length == nullptr) return p.topk;
  int l = __ldg(p.topk_length + t);
  return l < 0 ? 0 : (l > p.topk ? p.topk : l);
}

// Row of index idx in a cache of num_pages pages (flat when bt_row is null).
__device__ __forceinline__ int resolve_in(int64_t num_pages, const int32_t* bt_row, int bt_cols, int idx, int* err) {
  if (idx < 0) {
    if (idx != -1) atomicOr(err, kErrIndexRange);
    return -1;
  }
  if (bt_row == nullptr) {
    if ((int64_t)idx >= num_pages * kPage) {
      atomicOr(err, kErrIndexRange);
      return -1;
    }
    return idx;
  }
  const int lp = idx >> 6;
  if (lp >= bt_cols) {
    atomicOr(err, kErrIndexRange);
    return -1;
  }
  const int pp = __ldg(bt_row + lp);
  if (pp < 0 || (int64_t)pp >= num_pages) {
    atomicOr(err, kErrIndexRange);
    return -1;
  }
  return pp * kPage + (idx & (kPage - 1));
}

__device__ __forceinline__ int resolve_row(const KParams& p, const int32_t* bt_row, int idx) {
  return resolve_in(p.num_pages, bt_row, p.bt_cols, idx, p.err);
}

__device__ __forceinline__ const int32_t* bt_row_of(const KParams& p, int t) {
  return p.block_table == nullptr
             ? nullptr
             : p.block_table + (int64_t)(t / p.tokens_per_req) * p.bt_stride;
}

// ---------------------------------------------------------------------------
// Combined slots.  With one list, slot s of token t is slot s of its index
// row.  In the dual-cache form (kDual, p.dual) slots [0, x_base) are the first
// list (valid only below its topk_length) and slots [x_base, x_base + topk2)
// the second list, resolved in the second cache and encoded as rows1 + row.
// All candidates of a token enter one softmax.  kDual == false compiles the
// single-list path with no trace of the second list.
// ---------------------------------------------------------------------------
struct TokSlots {
  int len1;  // first-list entries at or past len1 are not read
  int end;   // slots [0, end) may hold valid candidates
};

template <bool kDual>
__device__ __forceinline__ TokSlots token_slots(const KParams& p, int t) {
  const int l1 = token_len(p, t);
  if (!kDual) return {l1, l1};
  int l2 = p.topk2;
  if (p.topk_length2 != nullptr) {
    const int l = __ldg(p.topk_length2 + t);
    l2 = l < 0 ? 0 : (l > p.topk2 ? p.topk2 : l);
  }
  return {l1, l2 > 0 ? p.x_base + l2 : l1};
}

template <bool kDual>
__device__ __forceinline__ bool in_list2(const KParams& p, int s) {
  return kDual && s >= p.x_base;
}

// Whether slot s's index entry may be read (the caller checks s < end).
template <bool kDual>
__device__ __forceinline__ bool slot_readable(const KParams& p, int s, int len1) {
  return s < len1 || in_list2<kDual>(p, s);
}

template <bool kDual>
__device__ __forceinline__ int slot_index(const KParams& p, int t, int s) {
  if (in_list2<kDual>(p, s)) return __ldg(p.indices2 + (int64_t)t * p.idx2_stride_t + (s - p.x_base));
  return __ldg(p.indices + (int64_t)t * p.idx_stride_t + s);
}

__device__ __forceinline__ const int32_t* bt2_row_of(const KParams& p, int t) {
  return p.block_table2 == nullptr
             ? nullptr
             : p.block_table2 + (int64_t)(t / p.tokens_per_req) * p.bt2_stride;
}

// Row of slot s with index idx (-1: invalid), given the token's block-table
// rows of both lists.
template <bool kDual>
__device__ __forceinline__ int resolve_slot(const KParams& p, const int32_t* btr, const int32_t* btr2, int s,
                                            int idx) {
  if (!in_list2<kDual>(p, s)) return resolve_row(p, btr, idx);
  const int r = resolve_in(p.num_pages2, btr2, p.bt2_cols, idx, p.err);
  return r < 0 ? -1 : p.rows1 + r;
}

template <bool kDual>
__device__ __forceinline__ const uint8_t* row_ptr(const KParams& p, int r) {
  if (kDual && r >= p.rows1) return p.kv2 + (int64_t)(r - p.rows1) * kRowBytes;
  return p.kv + (int64_t)r * kRowBytes;
}

// ---------------------------------------------------------------------------
// Small PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes == 0 zero-fills.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Two e4m3 codes (low byte first) -> f16x2 (exact: every e4m3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(v));
  return r;
}
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = e4m3x2_to_f16x2((uint16_t)(w & 0xFFFFu));
  hi = e4m3x2_to_f16x2((uint16_t)(w >> 16));
}

// Four signed int8 codes (byte 0 first) -> two f16x2, exactly: each code c is
// biased to c + 128 in [0, 255] and placed as the low mantissa byte of the
// f16 0x6400 (= 1024, whose unit in the last place is 1), which reads
// 1152 + c; subtracting 1152 is exact for every integer below 2048.
__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  const uint32_t b = 0x64646464u, off = 0x64806480u;  // f16x2 (1152, 1152)
  uint32_t l, h;
  asm("prmt.b32 %0, %1, %2, 0x4140;\n" : "=r"(l) : "r"(x), "r"(b));
  asm("prmt.b32 %0, %1, %2, 0x4342;\n" : "=r"(h) : "r"(x), "r"(b));
  asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(lo) : "r"(l), "r"(off));
  asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(hi) : "r"(h), "r"(off));
}

// Cache codes of either format -> f16 (unscaled).
template <bool kInt8>
__device__ __forceinline__ void codes4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if (kInt8)
    s8x4_to_f16x2x2(w, lo, hi);
  else
    e4m3x4_to_f16x2x2(w, lo, hi);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Per-head power-of-two pre-scale for q.  q is bf16; the contraction runs on
// f16 operands, so each head is multiplied by 2^-e with e chosen so that its
// largest |q| lands in [2^14, 2^15): every bf16 value within 2^28 of the head's
// maximum is then an exact f16, and 2^e is folded back into the score scale.
__device__ __forceinline__ int q_prescale_exp(float amax) {
  if (!(amax > 0.f) || !isfinite(amax)) return 0;
  int e;
  frexpf(amax, &e);  // amax = m * 2^e, m in [0.5, 1)
  e -= 15;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}
// 2^e as a float, exact for |e| <= 126.
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

}  // namespace smla
