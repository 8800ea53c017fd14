// tcgen05 / TMEM sparse MLA kernel for head groups of 64 (H % 64 == 0).
//
// One CTA = (token, 64-head group, split of the token's slots).  The per-token
// contractions are real dense GEMMs, so they run on the 5th-generation tensor
// cores with fp32 accumulators in tensor memory.  Operand roles are swapped
// (the "swapAB" idea of FlashInfer PR #4802): the 128 candidate rows of a tile
// fill the MMA M dimension and the 64 heads fill N, so every MMA is a full
// 128-row instruction at the native head count.
//
//   S^T[128 cand x 64 h]   = K_tile[128 x 576] . Q^T        (TMEM cols 0..63)
//   O^T[512 dv  x 64 h]   += V_tile^T[512 x 128] . P^T     (TMEM cols 64..319,
//                                                            four M=128 chunks)
//
// Shared memory (SW128 canonical layouts, 1024-byte aligned atoms):
//   tile   128 KB: the dequantised nope part of 128 rows, f16, eight 64-dim
//          blocks of [128 rows x 128 B].  Read K-major as the A operand of
//          S^T and MN-major (dv contiguous) as the A operand of O^T -- one
//          copy serves both.
//   rope    16 KB: the rows' bf16 rope (A operand of the rope part of S^T);
//          reused for P^T [128 cand x 64 h] f16 once S^T is done.
//   q       72 KB: q of the token, nope f16 / rope bf16, B operand of S^T,
//          with one power-of-two prescale for the whole token.
//
// Warp roles (512 threads; setmaxnreg gives 136 / 160 / 80 registers):
//   warps 0-7   producers: warp w gathers rows 16w..16w+15 of each tile with
//               coalesced 16-byte loads, converts the codes (e4m3 or int8) to
//               f16 times the row's scale and stores them swizzled; the bf16
//               rope is copied as is.  The next tile's rows are loaded in one
//               burst after a tile is stored (kLoad 0: L2-resident cache) or
//               group by group as soon as each group is stored, with an L2
//               prefetch one tile further ahead (kLoad 1: cache larger than
//               a quarter of L2; kLoad 2: larger than L2, where the rows are
//               also read 256 bytes per row and load instruction and the
//               128-dim groups go out in pairs).
//   warps 8-11  softmax/epilogue: thread = TMEM lane.  Per tile it reads its
//               candidate's 64 scores once, keeps a per-head reference max that
//               is only raised when a score exceeds it by 2^8 (then O^T columns
//               and the sums are rescaled), writes P (f16) for the PV MMA and
//               adds P into per-head sums with warp transpose-reductions.  The
//               token's score factor and the 64 reference maxima stay in
//               registers, and the four warps meet at one barrier per tile.
//   warp 12     MMA issue: S^T of a tile group by group as the producers
//               release them, PV after the softmax; one converged warp issuing
//               through elect.sync.
//   warps 12-15 with warps 8-11: the load and conversion of q before the first
//               tile, and half of the epilogue's stores after the last.
//
// Every mbarrier wait is bounded (KParams::wait_ns of global time, one second
// unless the caller set another limit; retries carry a 20 us suspend hint);
// when a limit runs out the CTA sets the error word, stops, drains its issued
// MMAs, frees TMEM and returns without writing outputs.
#include "smla_common.cuh"
#include "smla_launch.h"

namespace smla {
namespace tc_path {

constexpr int BM = 128;  // candidate rows per tile (MMA M)
constexpr int HG = 64;   // heads per CTA (MMA N)
constexpr int NT = 512;   // 8 producer warps, 4 softmax warps, 1 MMA warp, 3 helpers (q, epilogue)
constexpr int W_SOFT = 8;
constexpr int W_MMA = 12;
// Limit of the final wait for already-issued MMAs (they always complete; the
// call's own wait limit, which may be set as low as zero, does not apply).
constexpr uint64_t kDrainLimitNs = 1000000000ull;

// shared memory map (offsets from a 1024-aligned base)
constexpr int OFF_TILE = 0;                       // 8 x 16384
constexpr int OFF_ROPE = 131072;                  // 16384 (rope, then P^T)
constexpr int OFF_Q = 147456;                     // 9 x 8192
constexpr int OFF_QMUL = 221184;                  // float [64]
constexpr int OFF_TMAX = OFF_QMUL + 256;          // float [4][64]
constexpr int OFF_MREF = OFF_TMAX + 1024;         // float [64]
constexpr int OFF_ALPHA = OFF_MREF + 256;         // float [64]
constexpr int OFF_LSUM = OFF_ALPHA + 256;         // float [4][64]
constexpr int OFF_MNEG = OFF_LSUM + 1024;         // float [64]: -reference max (0 while unset)
constexpr int OFF_SCALE = OFF_MNEG + 256;         // float [8 warps][16 rows][4]
constexpr int OFF_MISC = OFF_SCALE + 2048;        // barriers, flags, tmem base
constexpr int SMEM_USED = OFF_MISC + 256;
constexpr int SMEM_BYTES = SMEM_USED + 1024;      // + alignment slack

// barrier slots in OFF_MISC (8 bytes each)
enum { B_KV0 = 0, B_SFULL = 5, B_PFULL = 6, B_PV0 = 7, B_DRAIN = 11, B_QCONV = 12, N_BARS = 13 };
constexpr int OFF_FLAGS = OFF_MISC + N_BARS * 8;  // int abort, int rescale, uint32 tmem base

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same test, with a hint that the thread may be suspended for up to ns
// nanoseconds while the phase is incomplete (it resumes when the phase
// completes).
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
constexpr uint32_t kSuspendNs = 20000;  // per retry of a wait that did not succeed at once
// Bounded wait (limit: KParams::wait_ns).  Returns false if the CTA is
// aborting (the limit ran out here or in another role).  Retries carry the
// suspend hint: long waits (rows from HBM) then poll far less, which measured
// 1.4% faster on the decode workload and 1.7% on the 131k prefill, and the
// limit and the abort flag are checked after every retry.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, const KParams& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait_hint(bar, parity, kSuspendNs)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > p.wait_ns) {
      atomicOr(p.err, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Warp-uniform bounded wait: every lane polls (a lane-0-only poll leaves the
// warp diverged, and MMAs issued by a diverged warp run several times
// slower), and the warp agrees on the outcome.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               const KParams& p) {
  const bool ok = mbar_wait(bar, parity, abort_flag, p);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool bar_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, %2, %3, pi;\n selp.u32 %0, 1, 0, po;\n}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// SW128 shared-memory matrix descriptor (tcgen05 format).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}
// kind::f16 instruction descriptor: fp32 accumulate, M=128, N=64.
// fmt 0 = f16, 1 = bf16; major 0 = K-major, 1 = MN-major.
__host__ __device__ constexpr uint32_t idesc(uint32_t fmt, uint32_t a_major, uint32_t b_major) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_major << 15) | (b_major << 16) | ((uint32_t)(HG >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}
// The same descriptor split in its two 32-bit words: the low word holds the
// start address >> 4 and the leading byte offset >> 4; the high word (stride
// 1024 B between 8-row groups, version bit 46, 128-byte swizzle) is the same
// for every operand here.  Advancing an operand is then one 32-bit add.
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ void mma_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, e;\n .reg .b64 da, db;\n setp.ne.b32 p, %4, 0;\n mov.b64 da, {%1, %5};\n"
      " mov.b64 db, {%2, %5};\n elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(id), "r"(acc), "r"(kDescHi)
      : "memory");
}
// One MMA issued by one elected lane of a converged warp.
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  tmem_ld16(taddr, v);
  tmem_ld16(taddr + 16, v + 16);
  tmem_ld16(taddr + 32, v + 32);
  tmem_ld16(taddr + 48, v + 48);
  tmem_ld_wait();
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Byte offset of 16-byte chunk `ch` of row `r` inside a [rows x 128 B] SW128 block.
__device__ __forceinline__ uint32_t sw128(int r, int ch) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4));
}

// Offset in the q buffer of the 16-byte chunk j (dims 8j .. 8j+7) of head row hh.
__device__ __forceinline__ uint32_t q_chunk_off(int hh, int j) {
  return j < 64 ? (uint32_t)(OFF_Q + (j >> 3) * 8192) + sw128(hh, j & 7)
                : (uint32_t)(OFF_Q + 8 * 8192) + sw128(hh, j - 64);
}

// Warp transpose-reduction of 64 per-lane values: lane l receives the
// reduction over all 32 lanes of entries 2l and 2l+1.

// Warp transpose-reduction of 32 per-lane values x[B .. B+32): lane l receives
// the reduction over all 32 lanes of entry B + l.
template <bool kMax, int B, int N>
__device__ __forceinline__ float xreduce32_at(const float (&xa)[N]) {
  const float* x = xa + B;
  const int lane = threadIdx.x & 31;
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float b[16];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float send = hi ? x[j] : x[16 + j];
      const float keep = hi ? x[16 + j] : x[j];
      b[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
  }
  float c[8];
  {
    const bool hi = lane & 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float send = hi ? b[j] : b[8 + j];
      const float keep = hi ? b[8 + j] : b[j];
      c[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
  }
  float d[4];
  {
    const bool hi = lane & 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float send = hi ? c[j] : c[4 + j];
      const float keep = hi ? c[4 + j] : c[j];
      d[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
  }
  float e[2];
  {
    const bool hi = lane & 2;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float send = hi ? d[j] : d[2 + j];
      const float keep = hi ? d[2 + j] : d[j];
      e[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
  }
  const bool hi = lane & 1;
  const float send = hi ? e[0] : e[1];
  const float keep = hi ? e[1] : e[0];
  return op(keep, __shfl_xor_sync(0xffffffffu, send, 1));
}

// Warp transpose-reduction of 32 per-lane values: lane l receives the
// reduction over all 32 lanes of entry l.
template <bool kMax>
__device__ __forceinline__ float xreduce32(const float (&x)[32]) {
  const int lane = threadIdx.x & 31;
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float b[16];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float send = hi ? x[j] : x[16 + j];
      const float keep = hi ? x[16 + j] : x[j];
      b[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
  }
  float c[8];
  {
    const bool hi = lane & 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float send = hi ? b[j] : b[8 + j];
      const float keep = hi ? b[8 + j] : b[j];
      c[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
  }
  float d[4];
  {
    const bool hi = lane & 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float send = hi ? c[j] : c[4 + j];
      const float keep = hi ? c[4 + j] : c[j];
      d[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
  }
  float e[2];
  {
    const bool hi = lane & 2;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float send = hi ? d[j] : d[2 + j];
      const float keep = hi ? d[2 + j] : d[j];
      e[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
  }
  const bool hi = lane & 1;
  const float send = hi ? e[0] : e[1];
  const float keep = hi ? e[1] : e[0];
  return op(keep, __shfl_xor_sync(0xffffffffu, send, 1));
}

template <bool kMax>
__device__ __forceinline__ void xreduce64(const float (&x)[64], float& r0, float& r1) {
  const int lane = threadIdx.x & 31;
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float a[32];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float send = hi ? x[j] : x[32 + j];
      const float keep = hi ? x[32 + j] : x[j];
      a[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
  }
  float b[16];
  {
    const bool hi = lane & 8;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float send = hi ? a[j] : a[16 + j];
      const float keep = hi ? a[16 + j] : a[j];
      b[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
  }
  float c[8];
  {
    const bool hi = lane & 4;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float send = hi ? b[j] : b[8 + j];
      const float keep = hi ? b[8 + j] : b[j];
      c[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
  }
  float d[4];
  {
    const bool hi = lane & 2;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float send = hi ? c[j] : c[4 + j];
      const float keep = hi ? c[4 + j] : c[j];
      d[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
  }
  {
    const bool hi = lane & 1;
    const float s0 = hi ? d[0] : d[2], k0 = hi ? d[2] : d[0];
    const float s1 = hi ? d[1] : d[3], k1 = hi ? d[3] : d[1];
    r0 = op(k0, __shfl_xor_sync(0xffffffffu, s0, 1));
    r1 = op(k1, __shfl_xor_sync(0xffffffffu, s1, 1));
  }
}

// Producer warp pw (0..7) owns tile rows 16pw .. 16pw+15.  Its loads are
// coalesced (4 lanes read 64 contiguous bytes of one row), and the 16 rows'
// scale and rope chunks (9 per row) are read as 144 consecutive (row, chunk)
// pairs.
template <int kLoad, bool kDual, bool kInt8>
__device__ __forceinline__ void producer(const KParams& p, uint8_t* smem, uint32_t sbase, uint32_t bars, int t,
                                         int len1, int lo, int hi, int ntiles, int pw, int lane,
                                         volatile int* s_abort) {
  constexpr bool kEarly = kLoad >= 1;  // rows mostly from HBM: early per-group loads, L2 prefetch
  constexpr bool kPairs = kLoad == 2;  // cache beyond L2: 256-byte row reads, groups in pairs
  // test hook (sparse_mla_set_test_stall): no row is gathered, so the MMA
  // issue's first wait runs out and the CTA takes its abort path
  if (p.test_stall) return;
  const int32_t* btr = bt_row_of(p, t);
  const int32_t* btr2 = kDual ? bt2_row_of(p, t) : nullptr;
  float* s_sc = reinterpret_cast<float*>(smem + OFF_SCALE) + pw * 64;  // [16 rows][4]
  // nope[g][j]: lane l holds row 8(j/2) + 2(l/8) + (l/4)%2, chunk 8g + 4(j%2) + l%4.
  // Each 8-lane store phase then covers two adjacent rows, whose different
  // swizzles put its 8 chunks in 8 distinct bank groups.
  uint4 nope[4][4];
  uint4 tail[5];     // flat (row, chunk) f = 32k + lane: row f/9, chunk 32 + f%9
  // index reads (lanes 0..15: one row each)
  auto load_idx = [&](int it) -> int {
    const int slot = lo + it * BM + 16 * pw + lane;
    return (lane < 16 && it < ntiles && slot < hi && slot_readable<kDual>(p, slot, len1))
               ? slot_index<kDual>(p, t, slot)
               : -1;
  };
  // Slot indices are read two tiles ahead of the conversion.  With rows that
  // stay in L2 (!kEarly), the next tile is loaded into registers in one burst
  // after the current tile is stored, while the S^T tail, softmax and PV keep
  // the producers idle.  With a cache larger than L2 can hold (kEarly), whose
  // rows come from HBM, the next tile's row ids are resolved as the current
  // tile starts and each 128-dim group (and the tail) is loaded as soon as
  // the same group of the current tile is stored, so that it stays in flight
  // for a whole tile period; the rows of the tile after that are prefetched
  // into L2, so the register loads see L2 latency and only the prefetch waits
  // on HBM.  (For L2-resident rows early loads only compete with the
  // conversion for the L1/shared-memory path.)
  int idx_a = load_idx(0), idx_b = load_idx(1);
  auto resolve = [&](int it) -> int {
    int rowid = -1;
    const int idx = idx_a, idx1 = idx_b;
    idx_a = idx_b;
    idx_b = load_idx(it + 2);
    if (lane < 16) {
      const int slot = lo + it * BM + 16 * pw + lane;
      if (slot < hi) rowid = resolve_slot<kDual>(p, btr, btr2, slot, idx);
      if (kEarly && it + 1 < ntiles && slot + BM < hi) {
        const int r1 = resolve_slot<kDual>(p, btr, btr2, slot + BM, idx1);
        if (r1 >= 0)
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row_ptr<kDual>(p, r1)),
                       "r"(kRowBytes)
                       : "memory");
      }
    }
    return rowid;
  };
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  auto load_group = [&](int g, int rowid) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = __shfl_sync(0xffffffffu, rowid, 8 * (j >> 1) + 2 * (lane >> 3) + ((lane >> 2) & 1));
      const uint4* src = reinterpret_cast<const uint4*>(row_ptr<kDual>(p, r < 0 ? 0 : r));
      nope[g][j] = r >= 0 ? __ldg(src + 8 * g + 4 * (j & 1) + (lane & 3)) : z;
    }
  };
  // kPairs: pair h (0, 1) = groups 2h and 2h+1.  nope[2h + j/4][j%4] holds
  // rows 2j (lanes 0-15) and 2j+1 (lanes 16-31), chunk 16h + l%16: each
  // 8-lane phase of a load reads 128 contiguous bytes of one row (about 1.9
  // cache lines, against 2.75 for two rows' 64 bytes).  Lanes 4-7 of each
  // eight convert their upper 8 codes first, so that each 8-lane store phase
  // covers the odd and the even 16-byte chunks of its row's two 64-dim blocks.
  auto load_pair = [&](int h, int rowid) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = __shfl_sync(0xffffffffu, rowid, 2 * j + (lane >> 4));
      const uint4* src = reinterpret_cast<const uint4*>(row_ptr<kDual>(p, r < 0 ? 0 : r));
      nope[2 * h + (j >> 2)][j & 3] = r >= 0 ? __ldg(src + 16 * h + (lane & 15)) : z;
    }
  };
  auto load_tail = [&](int rowid) {
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      const int f = 32 * k + lane;
      const int rr = f < 144 ? f / 9 : 0;
      const int r = __shfl_sync(0xffffffffu, rowid, rr);
      const uint4* src = reinterpret_cast<const uint4*>(row_ptr<kDual>(p, r < 0 ? 0 : r));
      tail[k] = (f < 144 && r >= 0) ? __ldg(src + 32 + (f - 9 * rr)) : z;
    }
  };
  if (ntiles > 0) {
    const int rowid = resolve(0);
    if constexpr (kPairs) {
      load_pair(0, rowid);
      load_pair(1, rowid);
    } else {
#pragma unroll
      for (int g = 0; g < 4; ++g) load_group(g, rowid);
    }
    load_tail(rowid);
  }
  for (int it = 0; it < ntiles; ++it) {
    const bool more = it + 1 < ntiles;
    const int rowid_next = (kEarly && more) ? resolve(it + 1) : -1;
    // scales of the 16 rows (invalid rows have zero data and zero scale)
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      const int f = 32 * k + lane;
      if (f < 144 && f % 9 == 0) {
        const int rr = f / 9;
        s_sc[rr * 4 + 0] = __uint_as_float(tail[k].x);
        s_sc[rr * 4 + 1] = __uint_as_float(tail[k].y);
        s_sc[rr * 4 + 2] = __uint_as_float(tail[k].z);
        s_sc[rr * 4 + 3] = __uint_as_float(tail[k].w);
        if (!(__uint_as_float(tail[k].x) <= 128.f && __uint_as_float(tail[k].y) <= 128.f &&
              __uint_as_float(tail[k].z) <= 128.f && __uint_as_float(tail[k].w) <= 128.f))
          atomicOr(p.err, kErrScaleRange);
      }
    }
    __syncwarp();
    if constexpr (kPairs) {
#pragma unroll
      for (int gp = 0; gp < 3; ++gp) {  // groups 0-1, groups 2-3, then the tail (rope)
        // PV chunks complete in order: the pair's later chunk frees both
        if (it > 0 && !mbar_wait(bars + 8u * (B_PV0 + (gp < 2 ? 2 * gp + 1 : 3)), (it - 1) & 1, s_abort, p))
          return;
        if (gp < 2) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int rl = 2 * j + (lane >> 4);
            const int row = 16 * pw + rl;
            const int c = 16 * gp + (lane & 15);  // nope chunk: dims 16c .. 16c+15
            const int odd = (lane >> 2) & 1;      // convert the upper 8 codes first
            const uint4 nv = nope[2 * gp + (j >> 2)][j & 3];
            const __half2 sc2 = __float2half2_rn(s_sc[rl * 4 + (c >> 3)]);
            const uint32_t sc2u = *reinterpret_cast<const uint32_t*>(&sc2);
            const uint32_t w[4] = {odd ? nv.z : nv.x, odd ? nv.w : nv.y, odd ? nv.x : nv.z, odd ? nv.y : nv.w};
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if constexpr (kInt8) {
                s8x4_to_f16x2x2(w[i], h[2 * i], h[2 * i + 1]);
              } else {
                asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n"
                    " cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
                    : "=r"(h[2 * i]), "=r"(h[2 * i + 1])
                    : "r"(w[i]));
              }
              h[2 * i] = hmul2_u32(h[2 * i], sc2u);
              h[2 * i + 1] = hmul2_u32(h[2 * i + 1], sc2u);
            }
            const uint32_t base = sbase + OFF_TILE + (c >> 2) * 16384;
            const int oc = 2 * (c & 3);
            sts128(base + sw128(row, oc + odd), make_uint4(h[0], h[1], h[2], h[3]));
            sts128(base + sw128(row, oc + 1 - odd), make_uint4(h[4], h[5], h[6], h[7]));
          }
        } else {
#pragma unroll
          for (int k = 0; k < 5; ++k) {
            const int f = 32 * k + lane;
            if (f < 144 && f % 9 != 0) {
              const int rr = f / 9;
              sts128(sbase + OFF_ROPE + sw128(16 * pw + rr, f - 9 * rr - 1), tail[k]);
            }
          }
        }
        fence_proxy_async();
        if (gp < 2) {
          mbar_arrive(bars + 8u * (B_KV0 + 2 * gp));
          mbar_arrive(bars + 8u * (B_KV0 + 2 * gp + 1));
        } else {
          mbar_arrive(bars + 8u * (B_KV0 + 4));
        }
        if (more) {  // kPairs implies kEarly
          if (gp < 2)
            load_pair(gp, rowid_next);
          else
            load_tail(rowid_next);
        }
      }
    } else {
#pragma unroll
      for (int g = 0; g < 5; ++g) {
        // this region of the tile is free once the previous tile's PV used it
        // (a per-lane wait: the lanes of the converged warp poll the barrier in
        // the same instructions and see the same phase; a warp-wide agreement on
        // every wait cost 1% of the 16k prefill)
        if (it > 0 && !mbar_wait(bars + 8u * (B_PV0 + (g < 4 ? g : 3)), (it - 1) & 1, s_abort, p)) return;
        if (g < 4) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int rl = 8 * (j >> 1) + 2 * (lane >> 3) + ((lane >> 2) & 1);
            const int row = 16 * pw + rl;
            const int c = 8 * g + 4 * (j & 1) + (lane & 3);  // nope chunk: dims 16c .. 16c+15
            const __half2 sc2 = __float2half2_rn(s_sc[rl * 4 + g]);
            const uint32_t sc2u = *reinterpret_cast<const uint32_t*>(&sc2);
            const uint32_t w[4] = {nope[g][j].x, nope[g][j].y, nope[g][j].z, nope[g][j].w};
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if constexpr (kInt8) {
                s8x4_to_f16x2x2(w[i], h[2 * i], h[2 * i + 1]);
              } else {
                asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n"
                    " cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
                    : "=r"(h[2 * i]), "=r"(h[2 * i + 1])
                    : "r"(w[i]));
              }
              h[2 * i] = hmul2_u32(h[2 * i], sc2u);
              h[2 * i + 1] = hmul2_u32(h[2 * i + 1], sc2u);
            }
            const uint32_t base = sbase + OFF_TILE + (c >> 2) * 16384;
            const int oc = 2 * (c & 3);
            sts128(base + sw128(row, oc), make_uint4(h[0], h[1], h[2], h[3]));
            sts128(base + sw128(row, oc + 1), make_uint4(h[4], h[5], h[6], h[7]));
          }
        } else {
#pragma unroll
          for (int k = 0; k < 5; ++k) {
            const int f = 32 * k + lane;
            if (f < 144 && f % 9 != 0) {
              const int rr = f / 9;
              sts128(sbase + OFF_ROPE + sw128(16 * pw + rr, f - 9 * rr - 1), tail[k]);
            }
          }
        }
        fence_proxy_async();
        mbar_arrive(bars + 8u * (B_KV0 + g));
        // the registers of this group are free: start the next tile's loads
        if (kEarly && more) {
          if (g < 4)
            load_group(g, rowid_next);
          else
            load_tail(rowid_next);
        }
      }
    }
    if (!kEarly && more) {
      const int rowid = resolve(it + 1);
#pragma unroll
      for (int g = 0; g < 4; ++g) load_group(g, rowid);
      load_tail(rowid);
    }
  }
}

// Epilogue: parts [part_lo, part_hi) of the 8 (d_v chunk, 32-head half)
// parts of O^T, by a warp whose TMEM lane quarter is q4.  s_alpha holds
// the per-head normaliser.  kStream: final out is written with the
// evict-first (streaming) cache operator, so that it does not push gathered
// rows of a cache larger than L2 out of L2 (the HBM-resident load policy).
template <bool kStream>
__device__ __forceinline__ void store_parts(const KParams& p, const float* s_alpha, uint32_t T_O,
                                            uint32_t lane_off, int t, int h0, int split, int ntiles, int q4,
                                            int lane, int part_lo, int part_hi) {
  const bool final_out = p.ws_o == nullptr;
  // O^T -> registers, 32 head columns at a time -> two transpose stages
  // through lane pairs and quads: lane l ends up with 4 consecutive d_v
  // values (4*(l/4) .. +3 of this warp's 32) for 8 heads
  // (hq = 32*half + 16*(l&1) + 8*((l>>1)&1) + j), stored as one 8-byte
  // (bf16 out) or 16-byte (fp32 partial) word per head.
  const bool odd = lane & 1, hi2 = lane & 2;
  const bool out_al8 = ((reinterpret_cast<uintptr_t>(p.out) | (uintptr_t)(p.out_stride_t * 2)) & 7) == 0;
#pragma unroll 1
  for (int part = part_lo; part < part_hi; ++part) {
    const int ch = part >> 1, half = part & 1;
    const int dv0 = 128 * ch + 32 * q4 + 4 * (lane >> 2);
    const int hq = 32 * half + 16 * (lane & 1) + 8 * ((lane >> 1) & 1);
    float o[32];
    if (ntiles > 0) {
      tmem_ld16(T_O + 64 * ch + 32 * half + lane_off, o);
      tmem_ld16(T_O + 64 * ch + 32 * half + 16 + lane_off, o + 16);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int h = 0; h < 32; ++h) o[h] = 0.f;
    }
#pragma unroll
    for (int h4 = 0; h4 < 8; ++h4) {
      const float4 a4 = *reinterpret_cast<const float4*>(s_alpha + 32 * half + 4 * h4);
      o[4 * h4 + 0] *= a4.x;
      o[4 * h4 + 1] *= a4.y;
      o[4 * h4 + 2] *= a4.z;
      o[4 * h4 + 3] *= a4.w;
    }
    if (final_out) {
      uint32_t wv[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float send = odd ? o[j] : o[16 + j];
        const float keep = odd ? o[16 + j] : o[j];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
        const __nv_bfloat162 bv = odd ? __floats2bfloat162_rn(recv, keep) : __floats2bfloat162_rn(keep, recv);
        wv[j] = *reinterpret_cast<const uint32_t*>(&bv);
      }
      __nv_bfloat16* ob = p.out + (int64_t)t * p.out_stride_t + (int64_t)(h0 + hq) * kDV + dv0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t send = hi2 ? wv[j] : wv[8 + j];
        const uint32_t keep = hi2 ? wv[8 + j] : wv[j];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 2);
        const uint2 st = hi2 ? make_uint2(recv, keep) : make_uint2(keep, recv);
        if (out_al8) {
          if (kStream)
            __stcs(reinterpret_cast<uint2*>(ob + (int64_t)j * kDV), st);
          else
            *reinterpret_cast<uint2*>(ob + (int64_t)j * kDV) = st;
        } else {
          unsigned short* os = reinterpret_cast<unsigned short*>(ob + (int64_t)j * kDV);
          os[0] = (unsigned short)(st.x & 0xFFFFu);
          os[1] = (unsigned short)(st.x >> 16);
          os[2] = (unsigned short)(st.y & 0xFFFFu);
          os[3] = (unsigned short)(st.y >> 16);
        }
      }
    } else {
      float2 f2[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float send = odd ? o[j] : o[16 + j];
        const float keep = odd ? o[16 + j] : o[j];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
        f2[j] = odd ? make_float2(recv, keep) : make_float2(keep, recv);
      }
      const int64_t hstride = (int64_t)p.num_splits * kDV;
      float* wb = p.ws_o + (((int64_t)t * p.H + h0 + hq) * p.num_splits + split) * kDV + dv0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 send = hi2 ? f2[j] : f2[8 + j];
        const float2 keep = hi2 ? f2[8 + j] : f2[j];
        float2 recv;
        recv.x = __shfl_xor_sync(0xffffffffu, send.x, 2);
        recv.y = __shfl_xor_sync(0xffffffffu, send.y, 2);
        const float4 st = hi2 ? make_float4(recv.x, recv.y, keep.x, keep.y)
                              : make_float4(keep.x, keep.y, recv.x, recv.y);
        *reinterpret_cast<float4*>(wb + (int64_t)j * hstride) = st;
      }
    }
  }
}

// q of one token, loaded and converted while the producers gather the first
// tile, by the 256 threads of the softmax warps and the last warpgroup (whose
// MMA-issue warp waits for q anyway; the other three have no other work).  The
// 64 head rows (one contiguous 72 KB block, or 64 KB without rope) are copied
// into their swizzled places in the q buffer, then converted in place: thread
// qc handles head qc/4, chunks [18 (qc%4), 18 (qc%4) + 18) of its 72.  The
// token gets one power-of-two prescale, putting the largest |q| of its 64
// heads in [2^14, 2^15).  Each head's maximum exponent is the largest
// exponent field of its bf16 values (an integer max over 16-bit halves),
// except when that field is 0 or 255 (all zero or subnormal; Inf/NaN), where
// the float maximum decides; the token takes the largest over its heads.
// kStream: q is read with the evict-first (streaming) cache operator (it is
// read once), for the HBM-resident load policy, whose cached rows should keep
// their L2 lines; otherwise it is copied with cp.async.
template <bool kStream>
__device__ __forceinline__ void load_q(const KParams& p, uint8_t* smem, uint32_t sbase, int t, int h0, int qc,
                                       float* s_qmul, float* s_mref, float* s_mneg, uint32_t bars) {
  const __nv_bfloat16* qsrc = p.q + (int64_t)t * p.q_stride_t + (int64_t)h0 * (p.nope ? kDNope : kDQK);
  if (p.nope) {
    // 512-dim heads (512 apart); the q buffer's rope chunks are zeroed (the
    // rope MMAs are skipped without rope)
    const unsigned short* qs = reinterpret_cast<const unsigned short*>(qsrc);
#pragma unroll 2
    for (int f = qc; f < HG * 72; f += 256) {
      const int hh = f / 72, ch = f % 72;
      const uint32_t dst = sbase + q_chunk_off(hh, ch);
      if (ch < 64) {
        const unsigned short* e = qs + (int64_t)hh * kDNope + 8 * ch;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = (uint32_t)__ldg(e + 2 * i) | ((uint32_t)__ldg(e + 2 * i + 1) << 16);
        sts128(dst, make_uint4(w[0], w[1], w[2], w[3]));
      } else {
        sts128(dst, make_uint4(0u, 0u, 0u, 0u));
      }
    }
  } else if ((reinterpret_cast<uintptr_t>(qsrc) & 15) == 0) {
    if (kStream) {
      const uint4* qv = reinterpret_cast<const uint4*>(qsrc);
#pragma unroll 6
      for (int f = qc; f < HG * 72; f += 256) sts128(sbase + q_chunk_off(f / 72, f % 72), __ldcs(qv + f));
    } else {
#pragma unroll 2
      for (int f = qc; f < HG * 72; f += 256) cp_async16(sbase + q_chunk_off(f / 72, f % 72), qsrc + 8 * f, 16);
      cp_async_commit();
      cp_async_wait<0>();
    }
  } else {
    const unsigned short* qs = reinterpret_cast<const unsigned short*>(qsrc);
#pragma unroll 2
    for (int f = qc; f < HG * 72; f += 256) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = (uint32_t)__ldg(qs + 8 * f + 2 * i) | ((uint32_t)__ldg(qs + 8 * f + 2 * i + 1) << 16);
      sts128(sbase + q_chunk_off(f / 72, f % 72), make_uint4(w[0], w[1], w[2], w[3]));
    }
  }
  named_bar(2, 256);
  const int hh = qc >> 2, quarter = qc & 3;
  uint32_t m = 0;
#pragma unroll 3
  for (int k = 0; k < 18; ++k) {
    const uint4 v = *reinterpret_cast<const uint4*>(smem + q_chunk_off(hh, 18 * quarter + k));
    m = __vmaxu2(m, v.x & 0x7F807F80u);
    m = __vmaxu2(m, v.y & 0x7F807F80u);
    m = __vmaxu2(m, v.z & 0x7F807F80u);
    m = __vmaxu2(m, v.w & 0x7F807F80u);
  }
  m = max(m & 0xFFFFu, m >> 16);
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
  const int ef = (int)(m >> 7);  // largest exponent field of the head
  int e = ef - 141;              // the exponent of max|q| is ef - 126; prescale to [2^14, 2^15)
  e = e < -100 ? -100 : (e > 100 ? 100 : e);
  bool e_valid = ef > 0 && ef < 255;  // the head has a finite, nonzero, normal maximum
  if (__any_sync(0xffffffffu, ef == 0 || ef == 255)) {
    float amax = 0.f;
#pragma unroll 2
    for (int k = 0; k < 18; ++k) {
      const uint4 v = *reinterpret_cast<const uint4*>(smem + q_chunk_off(hh, 18 * quarter + k));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(wv[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(wv[i] & 0xFFFF0000u)));
      }
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if (ef == 0 || ef == 255) {
      e = q_prescale_exp(amax);
      e_valid = amax > 0.f && isfinite(amax);
    }
  }
  // One prescale for the whole token: that of its largest head (heads with
  // no finite nonzero value do not count).  Every head then shares one score
  // factor, which the softmax keeps in a register instead of reading 64 of
  // them from shared memory per tile.  A head's bf16 values stay exact in f16
  // down to 2^-28 of the token's largest |q|; smaller ones only carry scores
  // below that relative size.
  int ev = e_valid ? e : -1000;
  ev = max(ev, __shfl_xor_sync(0xffffffffu, ev, 4));
  ev = max(ev, __shfl_xor_sync(0xffffffffu, ev, 8));
  ev = max(ev, __shfl_xor_sync(0xffffffffu, ev, 16));
  int* s_emax = reinterpret_cast<int*>(smem + OFF_TMAX);  // free until the softmax's first slow path
  if ((qc & 31) == 0) s_emax[qc >> 5] = ev;
  named_bar(2, 256);
  ev = s_emax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) ev = max(ev, s_emax[w]);
  e = ev == -1000 ? 0 : ev;
  const float down = pow2f(-e);
#pragma unroll 3
  for (int k = 0; k < 18; ++k) {
    const int ch = 18 * quarter + k;  // 8 dims: 8ch .. 8ch+7
    const uint32_t off = q_chunk_off(hh, ch);
    const uint4 v = *reinterpret_cast<const uint4*>(smem + off);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = __uint_as_float(wv[i] << 16) * down;
      const float b = __uint_as_float(wv[i] & 0xFFFF0000u) * down;
      if (ch < 64) {
        const __half2 hv = __floats2half2_rn(a, b);
        o[i] = *reinterpret_cast<const uint32_t*>(&hv);
      } else {
        const __nv_bfloat162 bv = __floats2bfloat162_rn(a, b);
        o[i] = *reinterpret_cast<const uint32_t*>(&bv);
      }
    }
    sts128(sbase + off, make_uint4(o[0], o[1], o[2], o[3]));
  }
  if (quarter == 0) {
    s_qmul[hh] = p.sm_scale * kLog2e * pow2f(e);
    s_mref[hh] = -INFINITY;
    s_mneg[hh] = 0.f;
  }
  fence_proxy_async();
  mbar_arrive(bars + 8u * B_QCONV);  // q is ready for the S^T MMAs
  named_bar(2, 256);                 // q, s_qmul and s_mref visible to the softmax warps and the issuer
}

template <int kLoad, bool kDual, bool kInt8>
__global__ void __launch_bounds__(NT, 1) tc_kernel(const KParams p) {
  constexpr bool kEarly = kLoad >= 1;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, by pointer arithmetic on the __shared__ array so
  // that accesses through it stay shared-memory (not generic) accesses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int n_hg = p.H / HG;
  int bid = blockIdx.x;
  const int split = bid % p.num_splits;
  bid /= p.num_splits;
  const int hg = bid % n_hg;
  const int t = bid / n_hg;
  const int h0 = hg * HG;
  const TokSlots ts = token_slots<kDual>(p, t);
  const int lo = split * p.split_len;
  const int hi = min(ts.end, lo + p.split_len);
  const int ntiles = hi > lo ? (hi - lo + BM - 1) / BM : 0;

  float* s_qmul = reinterpret_cast<float*>(smem + OFF_QMUL);
  float* s_tmax = reinterpret_cast<float*>(smem + OFF_TMAX);
  float* s_mref = reinterpret_cast<float*>(smem + OFF_MREF);
  float* s_alpha = reinterpret_cast<float*>(smem + OFF_ALPHA);
  float* s_lsum = reinterpret_cast<float*>(smem + OFF_LSUM);
  float* s_mneg = reinterpret_cast<float*>(smem + OFF_MNEG);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_FLAGS);
  volatile int* s_flag = reinterpret_cast<volatile int*>(smem + OFF_FLAGS + 4);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_FLAGS + 8);
  volatile int* s_epi = reinterpret_cast<volatile int*>(smem + OFF_FLAGS + 12);  // epilogue runs
  const uint32_t bars = sbase + OFF_MISC;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };

  // ---------------------------------------------------------------- setup
  if (warp == W_SOFT) {
    if (lane == 0) {
      for (int g = 0; g < 5; ++g) mbar_init(bar(B_KV0 + g), 256);
      mbar_init(bar(B_SFULL), 1);
      mbar_init(bar(B_PFULL), 128);
      for (int c = 0; c < 4; ++c) mbar_init(bar(B_PV0 + c), 1);
      mbar_init(bar(B_DRAIN), 1);
      mbar_init(bar(B_QCONV), 256);
      *s_abort = 0;
      *s_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(s_tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t T_S = tmem;        // S^T: cols [0, 64)
  const uint32_t T_O = tmem + 64;   // O^T chunk c: cols [64 + 64c, 128 + 64c)

  if (warp < W_SOFT) {
    // ============================================================ producers
    asm volatile("setmaxnreg.inc.sync.aligned.u32 136;" ::: "memory");
    producer<kLoad, kDual, kInt8>(p, smem, sbase, bars, t, ts.len1, lo, hi, ntiles, warp, lane, s_abort);
  } else if (warp >= W_MMA) {
    // ============================================ q conversion, MMA issue (warp 12), epilogue
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
    load_q<kEarly>(p, smem, sbase, t, h0, tid - 256, reinterpret_cast<float*>(smem + OFF_QMUL),
           reinterpret_cast<float*>(smem + OFF_MREF), reinterpret_cast<float*>(smem + OFF_MNEG), bars);
    if (warp == W_MMA) {
      const uint32_t id_f16 = idesc(0, 0, 0);
      const uint32_t id_bf16 = idesc(1, 0, 0);
      const uint32_t id_pv = idesc(0, 1, 1);
      const uint32_t ad_tile = sdesc_lo(sbase + OFF_TILE, 16);      // K-major view (S^T)
      const uint32_t ad_tile_mn = sdesc_lo(sbase + OFF_TILE, 16384);  // MN-major view (PV)
      const uint32_t ad_rope = sdesc_lo(sbase + OFF_ROPE, 16);
      const uint32_t bd_p = sdesc_lo(sbase + OFF_ROPE, 8192);
      const uint32_t bd_q = sdesc_lo(sbase + OFF_Q, 16);
      // S^T(it) = K_tile . Q^T, 128-dim group by group as the producers finish them
      auto issue_st = [&](int it) -> bool {
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          if (!mbar_wait_warp(bar(B_KV0 + g), it & 1, s_abort, p)) return false;
          tc_fence_after();
          uint32_t ag = ad_tile + (uint32_t)g * (2 * 16384 >> 4), bg = bd_q + (uint32_t)g * (2 * 8192 >> 4);
          asm volatile("" : "+r"(ag), "+r"(bg));  // keep the group's bases in registers, not its 16 operands
#pragma unroll
          for (int kb2 = 0; kb2 < 2; ++kb2)
#pragma unroll
            for (int st = 0; st < 4; ++st)
              mma_lo(T_S, ag + (uint32_t)((kb2 * 16384 + st * 32) >> 4), bg + (uint32_t)((kb2 * 8192 + st * 32) >> 4),
                     id_f16, (g | kb2 | st) != 0);
        }
        // the rope group is waited for even without rope (p.nope: its bytes are
        // padding and its MMAs are skipped), so that the tile region where P^T
        // will be written is no longer being stored to
        if (!mbar_wait_warp(bar(B_KV0 + 4), it & 1, s_abort, p)) return false;
        tc_fence_after();
        if (!p.nope) {
#pragma unroll
          for (int st = 0; st < 4; ++st)
            mma_lo(T_S, ad_rope + (uint32_t)((st * 32) >> 4), bd_q + (uint32_t)((8 * 8192 + st * 32) >> 4), id_bf16,
                   1);
        }
        mma_commit(bar(B_SFULL));
        return true;
      };
      // O^T += V_tile^T . P^T, one commit per 128-row d_v chunk
      auto issue_pv = [&](int it) -> bool {
        if (!mbar_wait_warp(bar(B_PFULL), it & 1, s_abort, p)) return false;
        tc_fence_after();
        const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          const uint32_t ac = ad_tile_mn + (uint32_t)ch * (2 * 16384 >> 4);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_lo(T_O + 64 * ch, ac + (uint32_t)((ks * 2048) >> 4), bd_p + (uint32_t)((ks * 2048) >> 4), id_pv,
                   ks > 0 ? 1u : acc0);
          mma_commit(bar(B_PV0 + ch));
        }
        return true;
      };
      const bool q_ok = ntiles == 0 || mbar_wait_warp(bar(B_QCONV), 0, s_abort, p);
      for (int it = 0; it < ntiles && q_ok; ++it) {
        if (!issue_st(it)) break;
        if (!issue_pv(it)) break;
      }
      // every issued MMA completes before TMEM is released
      mma_commit(bar(B_DRAIN));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(B_DRAIN), 0)) {
        if (globaltimer() - t0 > kDrainLimitNs) {
          if (lane == 0) atomicOr(p.err, kErrTimeout);
          break;
        }
      }
      __syncwarp();
    }
    // second half of the epilogue (every issued MMA has completed: the issuer
    // drained them, and the softmax warps waited for the last PV)
    named_bar(2, 256);
    if (*s_epi) {
      tc_fence_after();
      store_parts<kEarly>(p, s_alpha, T_O, (uint32_t)((warp & 3) * 32) << 16, t, h0, split, ntiles, warp & 3, lane, 4, 8);
    }
  } else {
    // ============================================================ softmax + epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 160;" ::: "memory");
    const int q4 = warp & 3;
    const int c = q4 * 32 + lane;  // TMEM lane: candidate (S^T) / dv row (O^T)
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    // the sinks of this warp's two heads (warp 8 computes the normalisers),
    // read now so that the load is long done by the epilogue
    const float sink_lo = (q4 == 0 && p.attn_sink) ? __ldg(p.attn_sink + h0 + lane) : 0.f;
    const float sink_hi = (q4 == 0 && p.attn_sink) ? __ldg(p.attn_sink + h0 + lane + 32) : 0.f;
    load_q<kEarly>(p, smem, sbase, t, h0, c, s_qmul, s_mref, s_mneg, bars);
    const float qmul = s_qmul[0];  // the token's score factor (one q prescale for all heads)
    // the negated reference max of every head, kept in registers: it changes
    // only in the slow path, and reading it from shared memory on every tile
    // put 16 broadcast loads per warp on the softmax's critical path
    float mn[64];
#pragma unroll
    for (int h = 0; h < 64; ++h) mn[h] = s_mneg[h];

    // running sums of P per head: lane l keeps heads l and l+32 of this warp's
    // 32 candidates (summed over the warp by a transpose-reduction per tile)
    float lsum0 = 0.f, lsum1 = 0.f;
    bool alive = true;
    bool refs_set = false;  // uniform: every head has a finite reference max
    const int32_t* btr = bt_row_of(p, t);
    const int32_t* btr2 = kDual ? bt2_row_of(p, t) : nullptr;
    auto index_at = [&](int sl) -> int {  // -1 past the token's slots
      return (sl < hi && slot_readable<kDual>(p, sl, ts.len1)) ? slot_index<kDual>(p, t, sl) : -1;
    };
    // the slot index of tile it+1 is read during tile it and resolved at its
    // end, off the softmax's critical path
    bool valid_next = false;
    if (ntiles > 0) valid_next = resolve_slot<kDual>(p, btr, btr2, lo + c, index_at(lo + c)) >= 0;
    int idx_ahead = ntiles > 1 ? index_at(lo + BM + c) : -1;
    for (int it = 0; it < ntiles; ++it) {
      const int slot = lo + it * BM + c;
      const bool valid = valid_next;
      const int idx1 = idx_ahead;
      const int slot2 = slot + 2 * BM;
      idx_ahead = it + 2 < ntiles ? index_at(slot2) : -1;
      // A failed wait (the CTA is aborting) is agreed on together with the
      // slow-path vote below, so that a normal tile pays one barrier of the
      // four softmax warps: the scores loaded meanwhile are then discarded.
      const bool failed = !mbar_wait(bar(B_SFULL), it & 1, s_abort, p);
      tc_fence_after();
      float x[64];
      tmem_ld64(T_S + lane_off, x);  // one TMEM round trip per tile
      // x = score (log2 units) minus the head's reference max
      float dmax = -INFINITY;
#pragma unroll
      for (int h4 = 0; h4 < 16; ++h4) {
        x[4 * h4 + 0] = fmaf(x[4 * h4 + 0], qmul, mn[4 * h4 + 0]);
        x[4 * h4 + 1] = fmaf(x[4 * h4 + 1], qmul, mn[4 * h4 + 1]);
        x[4 * h4 + 2] = fmaf(x[4 * h4 + 2], qmul, mn[4 * h4 + 2]);
        x[4 * h4 + 3] = fmaf(x[4 * h4 + 3], qmul, mn[4 * h4 + 3]);
        dmax = fmaxf(dmax, fmaxf(fmaxf(x[4 * h4], x[4 * h4 + 1]), fmaxf(x[4 * h4 + 2], x[4 * h4 + 3])));
      }
      if (!valid) dmax = -INFINITY;
      // Slow path (first tile with data, or a score 2^8 above its reference):
      // exact per-head tile maxima, raise the references, rescale sums and O^T.
      if (bar_or(1, 128, failed || (!refs_set && valid) || dmax > 8.f)) {
        if (bar_or(1, 128, failed)) {
          alive = false;
          break;
        }
#pragma unroll
        for (int h = 0; h < 64; ++h) x[h] = valid ? x[h] - s_mneg[h] : -INFINITY;  // raw scores
        s_tmax[q4 * 64 + lane] = xreduce32_at<true, 0>(x);
        s_tmax[q4 * 64 + 32 + lane] = xreduce32_at<true, 32>(x);
        named_bar(1, 128);
        if (q4 == 0) {
          bool any_set = true;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int h = lane + 32 * j;
            const float tm = fmaxf(fmaxf(s_tmax[h], s_tmax[64 + h]), fmaxf(s_tmax[128 + h], s_tmax[192 + h]));
            const float mo = s_mref[h];
            float al = 1.f;
            if (tm > mo + 8.f || (mo == -INFINITY && tm > -INFINITY)) {
              al = mo == -INFINITY ? 0.f : exp2f(mo - tm);
              s_mref[h] = tm;
              s_mneg[h] = -tm;
            }
            any_set = any_set && (s_mref[h] > -INFINITY);
            s_alpha[h] = al;
          }
          any_set = __all_sync(0xffffffffu, any_set);
          if (lane == 0) *s_flag = any_set ? 1 : 0;
        }
        named_bar(1, 128);
        refs_set = *s_flag != 0;
        lsum0 *= s_alpha[lane];
        lsum1 *= s_alpha[lane + 32];
        if (it > 0) {
          // O^T columns of rescaled heads (the previous PV has completed: S^T of
          // this tile was issued after it and has been waited for)
#pragma unroll 1
          for (int part = 0; part < 16; ++part) {
            const int col = 16 * part, hb = col & 63;
            float o[16];
            tmem_ld16(T_O + col + lane_off, o);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 16; ++h) o[h] *= s_alpha[hb + h];
            tmem_st16(T_O + col + lane_off, o);
          }
          tmem_st_wait();
        }
        // scores again from TMEM, against the new references
        tmem_ld64(T_S + lane_off, x);
#pragma unroll
        for (int h = 0; h < 64; ++h) mn[h] = s_mneg[h];  // the references just raised
#pragma unroll
        for (int h4 = 0; h4 < 16; ++h4) {
          x[4 * h4 + 0] = fmaf(x[4 * h4 + 0], qmul, mn[4 * h4 + 0]);
          x[4 * h4 + 1] = fmaf(x[4 * h4 + 1], qmul, mn[4 * h4 + 1]);
          x[4 * h4 + 2] = fmaf(x[4 * h4 + 2], qmul, mn[4 * h4 + 2]);
          x[4 * h4 + 3] = fmaf(x[4 * h4 + 3], qmul, mn[4 * h4 + 3]);
        }
      }
      // P = exp2(x) rounded to f16 -> row c of P^T (MN-major: heads contiguous)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t pk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int h = 8 * j + 2 * k;
          const float e0 = valid ? ex2(x[h]) : 0.f;
          const float e1 = valid ? ex2(x[h + 1]) : 0.f;
          x[h] = e0;
          x[h + 1] = e1;
          const __half2 hv = __floats2half2_rn(e0, e1);
          pk[k] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        sts128(sbase + OFF_ROPE + sw128(c, j), make_uint4(pk[0], pk[1], pk[2], pk[3]));
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
      lsum0 += xreduce32_at<false, 0>(x);
      lsum1 += xreduce32_at<false, 32>(x);
      valid_next = (it + 1 < ntiles && slot + BM < hi) && resolve_slot<kDual>(p, btr, btr2, slot + BM, idx1) >= 0;
    }
    // ---------------------------------------------------------- epilogue
    bool failed = !alive;
    if (alive && ntiles > 0 && !mbar_wait(bar(B_PV0 + 3), (ntiles - 1) & 1, s_abort, p)) failed = true;
    s_lsum[q4 * 64 + lane] = lsum0;
    s_lsum[q4 * 64 + 32 + lane] = lsum1;
    alive = !bar_or(1, 128, failed);
    if (alive) {
      tc_fence_after();
      const bool final_out = p.ws_o == nullptr;
      // per-head normaliser and lse (warp 8: lane handles heads l and l+32)
      if (q4 == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int hh = lane + 32 * j;
          const int h = h0 + hh;
          const float lt = s_lsum[hh] + s_lsum[64 + hh] + s_lsum[128 + hh] + s_lsum[192 + hh];
          const float m = s_mref[hh];
          const float mu = m == -INFINITY ? 0.f : m;
          const float lse_v = lt > 0.f ? (mu + log2f(lt)) * kLn2 : -INFINITY;
          float inv;
          if (final_out) {
            const float sk = p.attn_sink ? exp2f((j == 0 ? sink_lo : sink_hi) * kLog2e - mu) : 0.f;
            const float den = lt + sk;
            inv = den > 0.f ? 1.f / den : 0.f;
            p.lse[(int64_t)t * p.lse_stride_t + h] = lse_v;
          } else {
            inv = lt > 0.f ? 1.f / lt : 0.f;
            p.ws_lse[((int64_t)t * p.H + h) * p.num_splits + split] = lse_v;
          }
          s_alpha[hh] = inv;  // reuse as the normaliser
        }
      }
      named_bar(1, 128);
    }
    // the last warpgroup stores half of the parts: s_alpha and the outcome
    // are published to it by the barrier below
    if (warp == W_SOFT && lane == 0) *s_epi = alive ? 1 : 0;
    named_bar(2, 256);
    if (alive) store_parts<kEarly>(p, s_alpha, T_O, lane_off, t, h0, split, ntiles, q4, lane, 0, 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == W_SOFT) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

}  // namespace tc_path

bool tc_supported(int H) { return H % tc_path::HG == 0; }

cudaError_t launch_tc(const KParams& p, cudaStream_t stream) {
  const int64_t grid = (int64_t)p.T * (p.H / tc_path::HG) * p.num_splits;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  // load policy by cache size (p.big_cache: 0 within a quarter of L2, 1
  // larger, 2 larger than L2); the dual-cache form and the int8 cache format
  // have their own instantiations
  using K = void (*)(const KParams);
  static const K kerns[12] = {
      tc_path::tc_kernel<0, false, false>, tc_path::tc_kernel<1, false, false>, tc_path::tc_kernel<2, false, false>,
      tc_path::tc_kernel<0, true, false>,  tc_path::tc_kernel<1, true, false>,  tc_path::tc_kernel<2, true, false>,
      tc_path::tc_kernel<0, false, true>,  tc_path::tc_kernel<1, false, true>,  tc_path::tc_kernel<2, false, true>,
      tc_path::tc_kernel<0, true, true>,   tc_path::tc_kernel<1, true, true>,   tc_path::tc_kernel<2, true, true>};
  const int load = p.big_cache < 0 ? 0 : (p.big_cache > 2 ? 2 : p.big_cache);
  const K kern = kerns[load + (p.dual ? 3 : 0) + (p.kv_format == 1 ? 6 : 0)];
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc_path::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, tc_path::NT, tc_path::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
