// Warp-MMA sparse MLA kernel (mma.sync m16n8k16), any head count at its
// native width: heads are processed in groups of 8 or 16 with no padding to 64
// (vLLM PR #57673, Purpose: the few-head case should not run dummy heads).
//
// Operand roles are swapped as in the "swapAB" prefill of FlashInfer PR #4802
// (candidate rows fill the MMA M dimension, heads fill N), but the rest is this
// file's own design:
//
//  * One CTA = (token, head group, split).  4 warps; a tile is 64 candidate
//    rows; warp w gathers rows 16w..16w+15 of each tile with 16-byte cp.async,
//    row by row (one contiguous 512-byte copy of the codes per row and warp,
//    then the scales and rope).  8-head groups stage one tile per CTA and run
//    4 CTAs per SM; 16-head groups stage two tiles.
//  * S^T = K Q^T: warp w computes its 16 rows x all heads of the group.  The
//    e4m3 (or int8) codes are converted to f16 in registers (one cvt per two codes, no
//    scale); the per-128 scale multiplies the fp32 partial sum of each
//    128-dim group.  The rope part runs as a bf16 MMA.  The contraction index
//    is permuted inside each 64-dim block so that a thread's fragment is 16
//    contiguous bytes of a row (the same permutation is applied to q).
//  * Softmax: running max per head over the whole tile (exact, no lazy
//    threshold), P rounded to f16 and shared through shared memory.
//  * O^T = V^T P^T: warp w owns d_v columns [128w, 128w+128) -- exactly scale
//    group w -- for all 64 rows of the tile.  V fragments are built from 4x4
//    byte blocks transposed with prmt, converted to f16 and multiplied by the
//    row scale (f16, exact while |v| <= 65504).
//  * Prefill writes bf16 out / fp32 lse; split mode writes fp32 partials.
#include "smla_common.cuh"
#include "smla_launch.h"

namespace smla {
namespace mma_path {

constexpr int BC = 64;    // candidate rows per tile
constexpr int TS = 704;   // shared row stride in bytes (44 x 16)
constexpr int QS = 1168;  // shared q row stride in bytes (73 x 16)
constexpr int PS = 160;   // shared P row stride in bytes (64 f16 + pad)
constexpr int NT = 128;   // threads per CTA
constexpr float kPScale = 256.f;  // power-of-two factor on the PV B operand (see the PV loop)

// Bank-conflict swizzle of 16-byte chunks inside a staged row.  Chunks 0..39
// are XOR-permuted by (row / 4) % 4 so that the transposing V reads of four
// rows 4 apart hit distinct banks; chunk 40 stays in place.
__device__ __forceinline__ int swz(int row, int ch) {
  return ch < 40 ? (ch ^ (((row >> 2) & 3) << 1)) : ch;
}

// NST staged tiles: 2 overlap a CTA's own gather with its compute; 1 halves
// the CTA's shared memory so that 4 CTAs (16 warps) share an SM and hide the
// gather latency across CTAs instead.
template <int NH8, int NST>
struct Layout {
  static constexpr int HG = NH8 * 8;
  static constexpr int kv = 0;
  static constexpr int q = NST * BC * TS;
  static constexpr int p = q + HG * QS;
  static constexpr int red = p + HG * PS;
  static constexpr int lsum = red + 4 * HG * 4;
  static constexpr int qmul = lsum + 4 * HG * 4;
  static constexpr int total = qmul + HG * 4;
};

// 16 zero bytes to shared memory (the slot of an invalid row; no global
// address is formed for it, so an empty cache may have a null pointer).
__device__ __forceinline__ void sts_zero16(uint32_t dst) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(dst), "r"(0) : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ uint32_t wsel(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

template <int NH8, int NST, bool kDual, bool kInt8>
__global__ void __launch_bounds__(NT, NST == 1 ? 4 : 2) mma_kernel(const KParams p) {
  constexpr int HG = NH8 * 8;
  using L = Layout<NH8, NST>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;

  const int n_hg = (p.H + HG - 1) / HG;
  int bid = blockIdx.x;
  const int split = bid % p.num_splits;
  bid /= p.num_splits;
  const int hg = bid % n_hg;
  const int t = bid / n_hg;
  const int h0 = hg * HG;

  const TokSlots ts = token_slots<kDual>(p, t);
  const int lo = split * p.split_len;
  const int hi = min(ts.end, lo + p.split_len);
  const int ntiles = hi > lo ? (hi - lo + BC - 1) / BC : 0;
  const int32_t* btr = bt_row_of(p, t);
  const int32_t* btr2 = kDual ? bt2_row_of(p, t) : nullptr;

  float* s_red = reinterpret_cast<float*>(smem + L::red);
  float* s_lsum = reinterpret_cast<float*>(smem + L::lsum);
  float* s_qmul = reinterpret_cast<float*>(smem + L::qmul);

  // ---- q: load, per-head power-of-two pre-scale, f16 nope / bf16 rope ----
  for (int hh = warp; hh < HG; hh += 4) {
    const int h = h0 + hh;
    uint8_t* qrow = smem + L::q + hh * QS;
    if (h < p.H) {
      const __nv_bfloat16* qg = p.q + (int64_t)t * p.q_stride_t + (int64_t)h * (p.nope ? kDNope : kDQK);
      float v[18];
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 18; ++i) {
        v[i] = (i < 16 || !p.nope) ? __bfloat162float(qg[i * 32 + lane]) : 0.f;  // no rope: zero q rope
        amax = fmaxf(amax, fabsf(v[i]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const int e = q_prescale_exp(amax);
#pragma unroll
      for (int i = 0; i < 18; ++i) {
        const int d = i * 32 + lane;
        const float x = ldexpf(v[i], -e);
        if (d < kDNope) {
          reinterpret_cast<__half*>(qrow)[d] = __float2half_rn(x);
        } else {
          const int r = d - kDNope, c = r >> 3;
          const int unit = 64 + 2 * (c & 3) + (c >> 2);
          reinterpret_cast<__nv_bfloat16*>(qrow + unit * 16)[r & 7] = __float2bfloat16_rn(x);
        }
      }
      if (lane == 0) s_qmul[hh] = p.sm_scale * kLog2e * ldexpf(1.f, e);
    } else {
      for (int u = lane; u < QS / 16; u += 32) *reinterpret_cast<uint4*>(qrow + u * 16) = make_uint4(0, 0, 0, 0);
      if (lane == 0) s_qmul[hh] = 0.f;
    }
  }

  // ---- gather: warp w stages tile rows 16w..16w+15 (whole rows per warp) ----
  // Row by row: lane l copies chunk l (the 512 code bytes: one contiguous
  // 512-byte read per warp) and lanes 0..8 copy chunk 32+l (scales and rope).
  // A row's swizzle term ((16w + r) / 4) % 4 = (r / 4) % 4 is fixed for each
  // unrolled r, and its row id is uniform across the warp, so an empty row
  // costs no divergence.  swz() moves chunks 0..39 by an XOR of the term,
  // which on byte offsets is an XOR of term * 32 (chunk 40, lane 8's second
  // chunk, stays).
  const uint32_t lo16 = (uint32_t)lane << 4;
  const uint32_t hi16 = (uint32_t)(32 + lane) << 4;           // lanes 0..8: chunks 32..40
  const uint32_t hi_xmask = lane < 8 ? 0xFFFFFFFFu : 0u;      // chunk 40 is not permuted
  auto issue = [&](int tile, int stage) -> uint32_t {
    const int slot = lo + tile * BC + warp * 16 + (lane & 15);
    int row = -1;
    if (lane < 16 && slot < hi && slot_readable<kDual>(p, slot, ts.len1))
      row = resolve_slot<kDual>(p, btr, btr2, slot, slot_index<kDual>(p, t, slot));
    const uint32_t base = smem_u32(smem + L::kv + stage * BC * TS + warp * 16 * TS);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int rr = __shfl_sync(0xffffffffu, row, r);
      const uint32_t drow = base + r * TS;
      const uint32_t xo = (uint32_t)((r >> 2) & 3) << 5;  // swizzle term of row 16w + r, in bytes
      const uint32_t dlo = drow + (lo16 ^ xo), dhi = drow + (hi16 ^ (xo & hi_xmask));
      if (rr >= 0) {
        const uint8_t* srow = row_ptr<kDual>(p, rr);
        cp_async16(dlo, srow + lo16, 16);
        if (lane < 9) cp_async16(dhi, srow + hi16, 16);
      } else {
        sts_zero16(dlo);
        if (lane < 9) sts_zero16(dhi);
      }
    }
    return __ballot_sync(0xffffffffu, lane < 16 && row >= 0) & 0xFFFFu;
  };

  float m_run[NH8][2], l_part[NH8][2];
  float o[8][NH8][4];
#pragma unroll
  for (int n = 0; n < NH8; ++n) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      m_run[n][j] = -INFINITY;
      l_part[n][j] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[mt][n][k] = 0.f;
  }

  uint32_t vmask[2] = {0u, 0u};
  __syncthreads();  // q visible
  if (ntiles > 0) vmask[0] = issue(0, 0);
  cp_async_commit();
  if (NST == 2) {
    if (ntiles > 1) vmask[1] = issue(1, 1);
    cp_async_commit();
  }

  const int rg = warp * 16 + g, rg8 = rg + 8;
  uint8_t* s_p = smem + L::p;

  for (int it = 0; it < ntiles; ++it) {
    const int st = NST == 2 ? (it & 1) : 0;
    if (NST == 2)
      cp_async_wait<1>();
    else
      cp_async_wait<0>();
    __syncthreads();
    const uint8_t* tile = smem + L::kv + st * BC * TS;
    const uint8_t* pg = tile + rg * TS;
    const uint8_t* pg8 = tile + rg8 * TS;

    // ---------------- S^T = K Q^T (rows rg, rg8; all heads of the group) --------------
    float acc[NH8][4];
#pragma unroll
    for (int n = 0; n < NH8; ++n)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[n][k] = 0.f;
#pragma unroll 1
    for (int grp = 0; grp < 4; ++grp) {
      float tmp[NH8][4];
#pragma unroll
      for (int n = 0; n < NH8; ++n)
#pragma unroll
        for (int k = 0; k < 4; ++k) tmp[n][k] = 0.f;
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const int b = grp * 2 + bb;
        const uint4 ka = lds128(pg + swz(rg, 4 * b + tq) * 16);
        const uint4 kb = lds128(pg8 + swz(rg8, 4 * b + tq) * 16);
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          uint4 qv[NH8];
#pragma unroll
          for (int n = 0; n < NH8; ++n)
            qv[n] = lds128(smem + L::q + (n * 8 + g) * QS + (8 * b + 2 * tq + s2) * 16);
#pragma unroll
          for (int ss = 0; ss < 2; ++ss) {
            const int s = 2 * s2 + ss;
            uint32_t a0, a1, a2, a3;
            codes4_to_f16x2x2<kInt8>(wsel(ka, s), a0, a2);
            codes4_to_f16x2x2<kInt8>(wsel(kb, s), a1, a3);
#pragma unroll
            for (int n = 0; n < NH8; ++n)
              mma_f16_16816(tmp[n], a0, a1, a2, a3, ss ? qv[n].z : qv[n].x, ss ? qv[n].w : qv[n].y);
          }
        }
      }
      const float scg = *reinterpret_cast<const float*>(pg + swz(rg, 32) * 16 + grp * 4);
      const float scg8 = *reinterpret_cast<const float*>(pg8 + swz(rg8, 32) * 16 + grp * 4);
#pragma unroll
      for (int n = 0; n < NH8; ++n) {
        acc[n][0] = fmaf(scg, tmp[n][0], acc[n][0]);
        acc[n][1] = fmaf(scg, tmp[n][1], acc[n][1]);
        acc[n][2] = fmaf(scg8, tmp[n][2], acc[n][2]);
        acc[n][3] = fmaf(scg8, tmp[n][3], acc[n][3]);
      }
    }
    if (!p.nope) {  // rope dims: bf16 x bf16 (without rope the row bytes there are padding)
      const uint4 ra0 = lds128(pg + swz(rg, 33 + tq) * 16);
      const uint4 ra1 = lds128(pg + swz(rg, 37 + tq) * 16);
      const uint4 rb0 = lds128(pg8 + swz(rg8, 33 + tq) * 16);
      const uint4 rb1 = lds128(pg8 + swz(rg8, 37 + tq) * 16);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint4 qr[NH8];
#pragma unroll
        for (int n = 0; n < NH8; ++n)
          qr[n] = lds128(smem + L::q + (n * 8 + g) * QS + (64 + 2 * tq + half) * 16);
        const uint4& xa = half ? ra1 : ra0;
        const uint4& xb = half ? rb1 : rb0;
#pragma unroll
        for (int ss = 0; ss < 2; ++ss) {
          const int w0 = 2 * ss;
#pragma unroll
          for (int n = 0; n < NH8; ++n)
            mma_bf16_16816(acc[n], wsel(xa, w0), wsel(xb, w0), wsel(xa, w0 + 1), wsel(xb, w0 + 1),
                           wsel(qr[n], w0), wsel(qr[n], w0 + 1));
        }
      }
    }

    // ---------------- online softmax over the tile ----------------
    const uint32_t vm = vmask[st];
    const bool vg = (vm >> g) & 1u, vg8 = (vm >> (g + 8)) & 1u;
    float sc[NH8][4];
#pragma unroll
    for (int n = 0; n < NH8; ++n) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float qm = s_qmul[n * 8 + 2 * tq + j];
        sc[n][j] = vg ? acc[n][j] * qm : -INFINITY;
        sc[n][2 + j] = vg8 ? acc[n][2 + j] * qm : -INFINITY;
        float mx = fmaxf(sc[n][j], sc[n][2 + j]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (g == 0) s_red[warp * HG + n * 8 + 2 * tq + j] = mx;
      }
    }
    __syncthreads();
#pragma unroll
    for (int n = 0; n < NH8; ++n) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int hh = n * 8 + 2 * tq + j;
        const float tm = fmaxf(fmaxf(s_red[hh], s_red[HG + hh]), fmaxf(s_red[2 * HG + hh], s_red[3 * HG + hh]));
        const float mnew = fmaxf(m_run[n][j], tm);
        const float muse = mnew == -INFINITY ? 0.f : mnew;
        const float alpha = exp2f(m_run[n][j] - muse);
        m_run[n][j] = mnew;
        const __half p0 = __float2half_rn(exp2f(sc[n][j] - muse));
        const __half p1 = __float2half_rn(exp2f(sc[n][2 + j] - muse));
        l_part[n][j] = fmaf(l_part[n][j], alpha, __half2float(p0) + __half2float(p1));
        __half* prow = reinterpret_cast<__half*>(s_p + hh * PS);
        prow[warp * 16 + g] = p0;
        prow[warp * 16 + g + 8] = p1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][n][j] *= alpha;
          o[mt][n][2 + j] *= alpha;
        }
      }
    }
    __syncthreads();

    // ---------------- O^T += V^T P^T for d_v [128w, 128w+128) ----------------
#pragma unroll 1
    for (int kk = 0; kk < 4; ++kk) {
      const int cb = 16 * kk + 4 * tq;
      const uint8_t* r0 = tile + (cb + 0) * TS;
      const uint8_t* r1 = tile + (cb + 1) * TS;
      const uint8_t* r2 = tile + (cb + 2) * TS;
      const uint8_t* r3 = tile + (cb + 3) * TS;
      const float v0 = *reinterpret_cast<const float*>(r0 + swz(cb + 0, 32) * 16 + warp * 4);
      const float v1 = *reinterpret_cast<const float*>(r1 + swz(cb + 1, 32) * 16 + warp * 4);
      const float v2 = *reinterpret_cast<const float*>(r2 + swz(cb + 2, 32) * 16 + warp * 4);
      const float v3 = *reinterpret_cast<const float*>(r3 + swz(cb + 3, 32) * 16 + warp * 4);
      const uint32_t sclo = pack_f16x2(v0 * kPScale, v1 * kPScale), schi = pack_f16x2(v2 * kPScale, v3 * kPScale);
      // The row scales multiply P, not V: warp w's d_v columns are exactly
      // scale block w, so candidate c's scale is one number for all of them,
      // and P'[c][h] = P[c][h] * scale[c][w] * kPScale costs 2 multiplies per
      // head group here instead of one per converted V pair.  kPScale (a
      // power of two, removed in the epilogue) keeps P' in f16's normal range
      // for small P (scale 2^-7, P down to about 2^-15) while the largest
      // allowed scale (128) keeps it below 2^15.
      uint32_t bfr[NH8][2];
#pragma unroll
      for (int n = 0; n < NH8; ++n) {
        const uint2 bv = *reinterpret_cast<const uint2*>(s_p + (n * 8 + g) * PS + (16 * kk + 4 * tq) * 2);
        bfr[n][0] = hmul2_u32(bv.x, sclo);
        bfr[n][1] = hmul2_u32(bv.y, schi);
      }
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const int dvb = 128 * warp + 32 * pp + 4 * g;
        const int ch = dvb >> 4, wo = dvb & 15;
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(r0 + swz(cb + 0, ch) * 16 + wo);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(r1 + swz(cb + 1, ch) * 16 + wo);
        const uint32_t w2 = *reinterpret_cast<const uint32_t*>(r2 + swz(cb + 2, ch) * 16 + wo);
        const uint32_t w3 = *reinterpret_cast<const uint32_t*>(r3 + swz(cb + 3, ch) * 16 + wo);
        const uint32_t t01l = prmt(w0, w1, 0x5140), t23l = prmt(w2, w3, 0x5140);
        const uint32_t t01h = prmt(w0, w1, 0x7362), t23h = prmt(w2, w3, 0x7362);
        const uint32_t x0 = prmt(t01l, t23l, 0x5410), x1 = prmt(t01l, t23l, 0x7632);
        const uint32_t x2 = prmt(t01h, t23h, 0x5410), x3 = prmt(t01h, t23h, 0x7632);
        uint32_t l0, h0_, l1, h1_, l2, h2_, l3, h3_;
        codes4_to_f16x2x2<kInt8>(x0, l0, h0_);
        codes4_to_f16x2x2<kInt8>(x1, l1, h1_);
        codes4_to_f16x2x2<kInt8>(x2, l2, h2_);
        codes4_to_f16x2x2<kInt8>(x3, l3, h3_);
#pragma unroll
        for (int n = 0; n < NH8; ++n) {
          mma_f16_16816(o[2 * pp][n], l0, l1, h0_, h1_, bfr[n][0], bfr[n][1]);
          mma_f16_16816(o[2 * pp + 1][n], l2, l3, h2_, h3_, bfr[n][0], bfr[n][1]);
        }
      }
    }
    __syncthreads();  // stage st and P are free
    if (it + NST < ntiles) vmask[st] = issue(it + NST, st);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // ---------------- epilogue ----------------
#pragma unroll
  for (int n = 0; n < NH8; ++n) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = l_part[n][j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (g == 0) s_lsum[warp * HG + n * 8 + 2 * tq + j] = l;
    }
  }
  __syncthreads();
  const bool final_out = p.ws_o == nullptr;
#pragma unroll
  for (int n = 0; n < NH8; ++n) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int hh = n * 8 + 2 * tq + j;
      const int h = h0 + hh;
      if (h >= p.H) continue;
      const float lt = s_lsum[hh] + s_lsum[HG + hh] + s_lsum[2 * HG + hh] + s_lsum[3 * HG + hh];
      const float m = m_run[n][j];
      const float muse = m == -INFINITY ? 0.f : m;
      const float lse_v = lt > 0.f ? (muse + log2f(lt)) * kLn2 : -INFINITY;
      if (final_out) {
        const float sk = p.attn_sink ? exp2f(__ldg(p.attn_sink + h) * kLog2e - muse) : 0.f;
        const float den = lt + sk;
        const float inv = den > 0.f ? 1.f / (den * kPScale) : 0.f;
        __nv_bfloat16* orow = p.out + (int64_t)t * p.out_stride_t + (int64_t)h * kDV;
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const int dvb = 128 * warp + 32 * pp + 4 * g;
          __nv_bfloat162 a = __floats2bfloat162_rn(o[2 * pp][n][j] * inv, o[2 * pp][n][2 + j] * inv);
          __nv_bfloat162 b = __floats2bfloat162_rn(o[2 * pp + 1][n][j] * inv, o[2 * pp + 1][n][2 + j] * inv);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t*>(&a);
          pk.y = *reinterpret_cast<uint32_t*>(&b);
          *reinterpret_cast<uint2*>(orow + dvb) = pk;
        }
        if (warp == 0 && g == 0) p.lse[(int64_t)t * p.lse_stride_t + h] = lse_v;
      } else {
        const float inv = lt > 0.f ? 1.f / (lt * kPScale) : 0.f;
        const int64_t th = ((int64_t)t * p.H + h) * p.num_splits + split;
        float* wrow = p.ws_o + th * kDV;
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const int dvb = 128 * warp + 32 * pp + 4 * g;
          *reinterpret_cast<float4*>(wrow + dvb) =
              make_float4(o[2 * pp][n][j] * inv, o[2 * pp][n][2 + j] * inv, o[2 * pp + 1][n][j] * inv,
                          o[2 * pp + 1][n][2 + j] * inv);
        }
        if (warp == 0 && g == 0) p.ws_lse[th] = lse_v;
      }
    }
  }
}

template <int NH8, int NST, bool kDual, bool kInt8>
static cudaError_t launch(const KParams& p, cudaStream_t stream) {
  using L = Layout<NH8, NST>;
  const int n_hg = (p.H + NH8 * 8 - 1) / (NH8 * 8);
  const int64_t grid = (int64_t)p.T * n_hg * p.num_splits;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  cudaError_t e =
      cudaFuncSetAttribute(mma_kernel<NH8, NST, kDual, kInt8>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total);
  if (e != cudaSuccess) return e;
  mma_kernel<NH8, NST, kDual, kInt8><<<(unsigned)grid, NT, L::total, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mma_path

int mma_heads_per_cta(int H) { return H <= 8 ? 8 : 16; }

cudaError_t launch_mma(const KParams& p, cudaStream_t stream) {
  using L = cudaError_t (*)(const KParams&, cudaStream_t);
  static const L launchers[8] = {
      mma_path::launch<1, 1, false, false>, mma_path::launch<2, 2, false, false>,
      mma_path::launch<1, 1, true, false>,  mma_path::launch<2, 2, true, false>,
      mma_path::launch<1, 1, false, true>,  mma_path::launch<2, 2, false, true>,
      mma_path::launch<1, 1, true, true>,   mma_path::launch<2, 2, true, true>};
  return launchers[(mma_heads_per_cta(p.H) == 8 ? 0 : 1) + (p.dual ? 2 : 0) + (p.kv_format == 1 ? 4 : 0)](p, stream);
}

}  // namespace smla
