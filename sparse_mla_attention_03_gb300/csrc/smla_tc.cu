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
//   q       72 KB: q of the token, nope f16 / rope bf16, B operand of S^T.
//
// Warp roles (288 threads):
//   warps 0-3  producers: thread p gathers row p of the tile straight from
//              global memory, converts e4m3 -> f16 times its scale (exact while
//              |value| <= 65504) and stores it swizzled; the bf16 rope is copied.
//   warps 4-7  softmax/epilogue: thread = TMEM lane.  Per tile it reads its
//              candidate's 64 scores, forms per-head tile maxima and sums with a
//              warp transpose-reduction, keeps a per-head reference max that is
//              only raised when a score exceeds it by 2^8 (then O^T columns and
//              the sums are rescaled), and writes P (f16) for the PV MMA.
//   warp 8     allocates TMEM; lane 0 issues every MMA and commit.
//
// Every mbarrier wait is bounded (about one second of global time); on timeout
// the CTA sets the error word, stops, drains its issued MMAs, frees TMEM and
// returns without writing outputs.
#include "smla_common.cuh"
#include "smla_launch.h"

namespace smla {
namespace tc_path {

constexpr int BM = 128;  // candidate rows per tile (MMA M)
constexpr int HG = 64;   // heads per CTA (MMA N)
constexpr int NT = 288;
constexpr uint64_t kTimeoutNs = 1000000000ull;

// shared memory map (offsets from a 1024-aligned base)
constexpr int OFF_TILE = 0;                       // 8 x 16384
constexpr int OFF_ROPE = 131072;                  // 16384 (rope, then P^T)
constexpr int OFF_Q = 147456;                     // 9 x 8192
constexpr int OFF_QMUL = 221184;                  // float [64]
constexpr int OFF_TMAX = OFF_QMUL + 256;          // float [4][64]
constexpr int OFF_MREF = OFF_TMAX + 1024;         // float [64]
constexpr int OFF_ALPHA = OFF_MREF + 256;         // float [64]
constexpr int OFF_LSUM = OFF_ALPHA + 256;         // float [4][64]
constexpr int OFF_MISC = OFF_LSUM + 1024;         // barriers, flags, tmem base
constexpr int SMEM_USED = OFF_MISC + 256;
constexpr int SMEM_BYTES = SMEM_USED + 1024;      // + alignment slack

// barrier slots in OFF_MISC (8 bytes each)
enum { B_KV0 = 0, B_SFULL = 5, B_PFULL = 6, B_PV0 = 7, B_DRAIN = 11, B_QFULL = 12, N_BARS = 13 };
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
// Bounded wait.  Returns false if the CTA is aborting (timeout here or elsewhere).
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kTimeoutNs) {
        atomicOr(err, kErrTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
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
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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

// Warp transpose-reduction of 64 per-lane values: lane l receives the
// reduction over all 32 lanes of entries 2l and 2l+1.
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

__global__ void __launch_bounds__(NT, 1) tc_kernel(const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int n_hg = p.H / HG;
  int bid = blockIdx.x;
  const int split = bid % p.num_splits;
  bid /= p.num_splits;
  const int hg = bid % n_hg;
  const int t = bid / n_hg;
  const int h0 = hg * HG;
  const int len = token_len(p, t);
  const int lo = split * p.split_len;
  const int hi = min(len, lo + p.split_len);
  const int ntiles = hi > lo ? (hi - lo + BM - 1) / BM : 0;

  float* s_qmul = reinterpret_cast<float*>(smem + OFF_QMUL);
  float* s_tmax = reinterpret_cast<float*>(smem + OFF_TMAX);
  float* s_mref = reinterpret_cast<float*>(smem + OFF_MREF);
  float* s_alpha = reinterpret_cast<float*>(smem + OFF_ALPHA);
  float* s_lsum = reinterpret_cast<float*>(smem + OFF_LSUM);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_FLAGS);
  volatile int* s_rescale = reinterpret_cast<volatile int*>(smem + OFF_FLAGS + 4);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_FLAGS + 8);
  const uint32_t bars = sbase + OFF_MISC;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };

  // ---------------------------------------------------------------- setup
  if (warp == 8) {
    if (lane == 0) {
      for (int g = 0; g < 5; ++g) mbar_init(bar(B_KV0 + g), 128);
      mbar_init(bar(B_SFULL), 1);
      mbar_init(bar(B_PFULL), 128);
      for (int c = 0; c < 4; ++c) mbar_init(bar(B_PV0 + c), 1);
      mbar_init(bar(B_DRAIN), 1);
      mbar_init(bar(B_QFULL), 128);
      *s_abort = 0;
      *s_rescale = 0;
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

  if (warp < 4) {
    // ============================================================ producers
    const int pr = tid;  // row of the tile
    const int32_t* idx_row = p.indices + (int64_t)t * p.idx_stride_t;
    const int32_t* btr = bt_row_of(p, t);
    for (int it = 0; it < ntiles; ++it) {
      const int slot = lo + it * BM + pr;
      const int row = slot < hi ? resolve_row(p, btr, __ldg(idx_row + slot)) : -1;
      const uint4* src = reinterpret_cast<const uint4*>(p.kv + (int64_t)(row < 0 ? 0 : row) * kRowBytes);
      const bool ok = row >= 0;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      const uint4 scv = ok ? __ldg(src + 32) : z;
      uint4 cur[8], nxt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) cur[j] = ok ? __ldg(src + j) : z;
      bool alive = true;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        if (g < 3) {
#pragma unroll
          for (int j = 0; j < 8; ++j) nxt[j] = ok ? __ldg(src + 8 * (g + 1) + j) : z;
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) nxt[j] = ok ? __ldg(src + 33 + j) : z;  // rope
        }
        const float sc = __uint_as_float(g == 0 ? scv.x : (g == 1 ? scv.y : (g == 2 ? scv.z : scv.w)));
        if (ok && !(sc <= 128.f)) atomicOr(p.err, kErrScaleRange);
        const __half2 sc2 = __float2half2_rn(sc);
        const uint32_t sc2u = *reinterpret_cast<const uint32_t*>(&sc2);
        // the block pair 2g, 2g+1 of this tile is free once PV of the previous tile used chunk g
        if (it > 0 && !mbar_wait(bar(B_PV0 + g), (it - 1) & 1, s_abort, p.err)) {
          alive = false;
          break;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          // 16 codes = dims 128g + 16j .. +15 -> two 16-byte f16 chunks
          const uint32_t w[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
          uint32_t h[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            e4m3x4_to_f16x2x2(w[k], h[2 * k], h[2 * k + 1]);
            h[2 * k] = hmul2_u32(h[2 * k], sc2u);
            h[2 * k + 1] = hmul2_u32(h[2 * k + 1], sc2u);
          }
          const int kb = 2 * g + (j >> 2);
          const int oc = 2 * (j & 3);
          const uint32_t base = sbase + OFF_TILE + kb * 16384;
          sts128(base + sw128(pr, oc), make_uint4(h[0], h[1], h[2], h[3]));
          sts128(base + sw128(pr, oc + 1), make_uint4(h[4], h[5], h[6], h[7]));
        }
        fence_proxy_async();
        mbar_arrive(bar(B_KV0 + g));
#pragma unroll
        for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
      }
      if (!alive) break;
      // rope: the region also holds P^T of the previous tile -> wait for its PV to finish
      if (it > 0 && !mbar_wait(bar(B_PV0 + 3), (it - 1) & 1, s_abort, p.err)) break;
#pragma unroll
      for (int j = 0; j < 8; ++j) sts128(sbase + OFF_ROPE + sw128(pr, j), cur[j]);
      fence_proxy_async();
      mbar_arrive(bar(B_KV0 + 4));
    }
  } else if (warp < 8) {
    // ============================================================ softmax
    const int q4 = warp & 3;
    const int c = q4 * 32 + lane;  // TMEM lane: candidate (S^T) / dv row (O^T)
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    // q of this token (while the producers gather the first tile): warp w
    // converts heads 16(w-4) .. +15 in two rounds of 8; lane l owns head
    // (l / 4) of the round and 16-byte chunks (l % 4) + 4k, k < 18.
#pragma unroll 1
    for (int round = 0; round < 2; ++round) {
      const int hh = 16 * q4 + 8 * round + (lane >> 2);
      const int sub = lane & 3;
      const __nv_bfloat16* qrow = p.q + (int64_t)t * p.q_stride_t + (int64_t)(h0 + hh) * kDQK;
      const bool vec = (reinterpret_cast<uintptr_t>(qrow) & 15) == 0;
      uint4 v[18];
#pragma unroll
      for (int k = 0; k < 18; ++k) {
        const int ch = sub + 4 * k;
        if (vec) {
          v[k] = __ldg(reinterpret_cast<const uint4*>(qrow) + ch);
        } else {
          uint16_t e[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) e[i] = __ldg(reinterpret_cast<const unsigned short*>(qrow) + ch * 8 + i);
          v[k] = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16),
                            e[4] | ((uint32_t)e[5] << 16), e[6] | ((uint32_t)e[7] << 16));
        }
      }
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < 18; ++k) {
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
          amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int e = q_prescale_exp(amax);
#pragma unroll
      for (int k = 0; k < 18; ++k) {
        const int ch = sub + 4 * k;  // 8 dims: 8ch .. 8ch+7
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = ldexpf(__uint_as_float(w[i] << 16), -e);
          const float b = ldexpf(__uint_as_float(w[i] & 0xFFFF0000u), -e);
          if (ch < 64) {
            const __half2 hv = __floats2half2_rn(a, b);
            o[i] = *reinterpret_cast<const uint32_t*>(&hv);
          } else {
            const __nv_bfloat162 bv = __floats2bfloat162_rn(a, b);
            o[i] = *reinterpret_cast<const uint32_t*>(&bv);
          }
        }
        const uint32_t off = ch < 64 ? OFF_Q + (ch >> 3) * 8192 + sw128(hh, ch & 7)
                                     : OFF_Q + 8 * 8192 + sw128(hh, ch - 64);
        sts128(sbase + off, make_uint4(o[0], o[1], o[2], o[3]));
      }
      if (sub == 0) {
        s_qmul[hh] = p.sm_scale * kLog2e * ldexpf(1.f, e);
        s_mref[hh] = -INFINITY;
      }
    }
    fence_proxy_async();
    mbar_arrive(bar(B_QFULL));
    named_bar(1, 128);  // s_qmul / s_mref visible to the other softmax warps

    float lsum0 = 0.f, lsum1 = 0.f;
    bool alive = true;
    const int32_t* idx_row = p.indices + (int64_t)t * p.idx_stride_t;
    const int32_t* btr = bt_row_of(p, t);
    for (int it = 0; it < ntiles; ++it) {
      const int slot = lo + it * BM + c;
      const bool valid = slot < hi && resolve_row(p, btr, __ldg(idx_row + slot)) >= 0;
      const bool failed = !mbar_wait(bar(B_SFULL), it & 1, s_abort, p.err);
      if (bar_or(1, 128, failed)) {
        alive = false;
        break;
      }
      tc_fence_after();
      float x[64];
      tmem_ld64(T_S + lane_off, x);
#pragma unroll
      for (int h = 0; h < 64; ++h) x[h] = valid ? x[h] * s_qmul[h] : -INFINITY;
      float m0, m1;
      xreduce64<true>(x, m0, m1);
      s_tmax[q4 * 64 + 2 * lane] = m0;
      s_tmax[q4 * 64 + 2 * lane + 1] = m1;
      named_bar(1, 128);
      if (q4 == 0) {
        bool need = false;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int h = 2 * lane + j;
          const float tm = fmaxf(fmaxf(s_tmax[h], s_tmax[64 + h]), fmaxf(s_tmax[128 + h], s_tmax[192 + h]));
          const float mo = s_mref[h];
          float al = 1.f;
          if (tm > mo + 8.f) {  // also when mo == -inf and tm is finite
            al = exp2f(mo - tm);
            s_mref[h] = tm;
            need = true;
          }
          s_alpha[h] = al;
        }
        need = __any_sync(0xffffffffu, need);
        if (lane == 0) *s_rescale = need ? 1 : 0;
      }
      named_bar(1, 128);
      const bool rescale = *s_rescale != 0;
      // P = exp2(x - mref) rounded to f16, row c of P^T (MN-major: heads contiguous)
      float pf[64];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t pk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int h = 8 * j + 2 * k;
          const float r0 = s_mref[h], r1 = s_mref[h + 1];
          const float e0 = exp2f(x[h] - (r0 == -INFINITY ? 0.f : r0));
          const float e1 = exp2f(x[h + 1] - (r1 == -INFINITY ? 0.f : r1));
          const __half2 hv = __floats2half2_rn(e0, e1);
          pk[k] = *reinterpret_cast<const uint32_t*>(&hv);
          const float2 back = __half22float2(hv);
          pf[h] = back.x;
          pf[h + 1] = back.y;
        }
        sts128(sbase + OFF_ROPE + sw128(c, j), make_uint4(pk[0], pk[1], pk[2], pk[3]));
      }
      float t0, t1;
      xreduce64<false>(pf, t0, t1);
      lsum0 = fmaf(lsum0, s_alpha[2 * lane], t0);
      lsum1 = fmaf(lsum1, s_alpha[2 * lane + 1], t1);
      if (rescale && it > 0) {
        // O^T columns of rescaled heads (the previous PV has completed: S^T of
        // this tile was issued after it and has been waited for)
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          float o[64];
          tmem_ld64(T_O + 64 * ch + lane_off, o);
#pragma unroll
          for (int h = 0; h < 64; ++h) o[h] *= s_alpha[h];
          tmem_st16(T_O + 64 * ch + lane_off, o);
          tmem_st16(T_O + 64 * ch + 16 + lane_off, o + 16);
          tmem_st16(T_O + 64 * ch + 32 + lane_off, o + 32);
          tmem_st16(T_O + 64 * ch + 48 + lane_off, o + 48);
        }
        tmem_st_wait();
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    // ---------------------------------------------------------- epilogue
    bool failed = !alive;
    if (alive && ntiles > 0 && !mbar_wait(bar(B_PV0 + 3), (ntiles - 1) & 1, s_abort, p.err)) failed = true;
    s_lsum[q4 * 64 + 2 * lane] = lsum0;
    s_lsum[q4 * 64 + 2 * lane + 1] = lsum1;
    alive = !bar_or(1, 128, failed);
    if (alive) {
      tc_fence_after();
      const bool final_out = p.ws_o == nullptr;
      // per-head normaliser and lse (lane handles heads 2l, 2l+1 in warp 4)
      if (q4 == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int hh = 2 * lane + j;
          const int h = h0 + hh;
          const float lt = s_lsum[hh] + s_lsum[64 + hh] + s_lsum[128 + hh] + s_lsum[192 + hh];
          const float m = s_mref[hh];
          const float mu = m == -INFINITY ? 0.f : m;
          const float lse_v = lt > 0.f ? (mu + log2f(lt)) * kLn2 : -INFINITY;
          float inv;
          if (final_out) {
            const float sk = p.attn_sink ? exp2f(__ldg(p.attn_sink + h) * kLog2e - mu) : 0.f;
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
      // stage [64 heads x 512 dv] in the (now idle) tile buffer, then store rows
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        float o[64];
        if (ntiles > 0) {
          tmem_ld64(T_O + 64 * ch + lane_off, o);
        } else {
#pragma unroll
          for (int h = 0; h < 64; ++h) o[h] = 0.f;
        }
        const int dv = 128 * ch + c;
        if (final_out) {
          __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(smem + OFF_TILE);
#pragma unroll
          for (int h = 0; h < 64; ++h) st[h * kDV + dv] = __float2bfloat16_rn(o[h] * s_alpha[h]);
        } else {
          float* st = reinterpret_cast<float*>(smem + OFF_TILE);
#pragma unroll
          for (int h = 0; h < 64; ++h) st[h * kDV + dv] = o[h] * s_alpha[h];
        }
      }
      named_bar(1, 128);
      const int tl = tid - 128;
      if (final_out) {
        for (int i = tl; i < 64 * 128; i += 128) {  // 64 rows x 128 x 8 B
          const int hh = i >> 7, part = i & 127;
          const uint2 v = *reinterpret_cast<const uint2*>(smem + OFF_TILE + hh * 1024 + part * 8);
          __nv_bfloat16* orow = p.out + (int64_t)t * p.out_stride_t + (int64_t)(h0 + hh) * kDV;
          *reinterpret_cast<uint2*>(orow + part * 4) = v;
        }
      } else {
        for (int i = tl; i < 64 * 128; i += 128) {  // 64 rows x 128 x 16 B
          const int hh = i >> 7, part = i & 127;
          const uint4 v = *reinterpret_cast<const uint4*>(smem + OFF_TILE + hh * 2048 + part * 16);
          float* wrow = p.ws_o + (((int64_t)t * p.H + h0 + hh) * p.num_splits + split) * kDV;
          *reinterpret_cast<uint4*>(wrow + part * 4) = v;
        }
      }
    }
  } else if (lane == 0) {
    // ============================================================ MMA issuer
    const uint32_t id_f16 = idesc(0, 0, 0);
    const uint32_t id_bf16 = idesc(1, 0, 0);
    const uint32_t id_pv = idesc(0, 1, 1);
    const uint32_t a_tile = sbase + OFF_TILE, a_rope = sbase + OFF_ROPE, b_q = sbase + OFF_Q;
    const bool q_ok = mbar_wait(bar(B_QFULL), 0, s_abort, p.err);
    for (int it = 0; it < (q_ok ? ntiles : 0); ++it) {
      bool alive = true;
      for (int g = 0; g < 4 && alive; ++g) {
        if (!mbar_wait(bar(B_KV0 + g), it & 1, s_abort, p.err)) {
          alive = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kb2 = 0; kb2 < 2; ++kb2) {
          const int kb = 2 * g + kb2;
#pragma unroll
          for (int s = 0; s < 4; ++s)
            mma(T_S, sdesc(a_tile + kb * 16384 + s * 32, 16, 1024), sdesc(b_q + kb * 8192 + s * 32, 16, 1024),
                id_f16, (kb | s) != 0);
        }
      }
      if (!alive) break;
      if (!mbar_wait(bar(B_KV0 + 4), it & 1, s_abort, p.err)) break;
      tc_fence_after();
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(T_S, sdesc(a_rope + s * 32, 16, 1024), sdesc(b_q + 8 * 8192 + s * 32, 16, 1024), id_bf16, 1);
      mma_commit(bar(B_SFULL));
      if (!mbar_wait(bar(B_PFULL), it & 1, s_abort, p.err)) break;
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma(T_O + 64 * ch, sdesc(a_tile + 2 * ch * 16384 + ks * 2048, 16384, 1024),
              sdesc(a_rope + ks * 2048, 8192, 1024), id_pv, (it > 0 || ks > 0) ? 1u : 0u);
        mma_commit(bar(B_PV0 + ch));
      }
    }
    // all issued MMAs complete before TMEM is released
    mma_commit(bar(B_DRAIN));
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar(B_DRAIN), 0)) {
      if (globaltimer() - t0 > kTimeoutNs) {
        atomicOr(p.err, kErrTimeout);
        break;
      }
    }
  }
  if (warp == 8) __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
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
  cudaError_t e =
      cudaFuncSetAttribute(tc_path::tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc_path::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  tc_path::tc_kernel<<<(unsigned)grid, tc_path::NT, tc_path::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
