// pa_mma.cuh -- tensor-core consumer for the paged decode kernel, for groups
// of query heads that share one kv head (GQA).  Per staged block the group's
// scores and weighted values are two small dense contractions:
//
//   S[tokens x heads]  = K[tokens x D] . Q^T[D x heads]       (mma m16n8k16, M = 16 tokens)
//   O^T[D x heads]    += V^T[D x tokens] . P^T[tokens x heads] (mma m16n8k16, M = 16 dims)
//
// with 8 query heads as the N = 8 side of the instruction.  Both cache layouts
// of the page "paged_attention_v2_triton.py -- Triton PagedAttention V2 for
// BI-V100" already are the operands ldmatrix wants: a K block [D/8][BS][8]
// stores 16 bytes (8 dims) of one token contiguously, i.e. one ldmatrix row of
// K[tokens x dims]; a V block [D][BS] stores 8 tokens of one dim contiguously,
// i.e. one row of V^T[dims x tokens].  The score fragment is turned into the
// P^T operand with movmatrix (an in-register 8x8 transpose).
//
// Softmax arithmetic is that of the phase-1 kernel `_paged_attn_v2_partition_kernel`
// (scores in fp32, running max, exp, running sum, rescaled accumulation); the
// weights enter the second product rounded to the element type.
#pragma once

#include <cuda_fp8.h>

#include <type_traits>

#include "pa_common.cuh"

namespace pa {

// FP8_: the caches hold E4M3 codes (one byte per element, key layout
// [D/16][BS][16]); operand fragments are then read code pair by code pair and
// widened to T (every E4M3 value is exact in fp16 and bf16).
template <typename T_, int D_, int BS_, bool FP8_ = false>
struct MmaConsumer {
  using T = T_;
  static constexpr int D = D_, BS = BS_, GT = 8;
  static constexpr bool kMma = true;
  static constexpr bool kFp8 = FP8_;
  static constexpr int KV_ESZ = FP8_ ? 1 : 2;  // bytes per cached element
  static constexpr int NK = D / 16;    // k-steps of the score product
  static constexpr int NMT = D / 16;   // 16-dim tiles of the value product
  static constexpr int NTT = BS / 16;  // 16-token tiles per block
  static constexpr int SCRATCH_FLOATS = 0;
  static constexpr bool kSplitWeights = std::is_same<T_, __nv_bfloat16>::value;

  uint32_t qb[NK][2];  // Q^T fragments (B operand), packed element pairs
  float m[2], l[2];    // heads 2*(lane%4) and 2*(lane%4)+1
  float acc[NMT][4];
  float scale_log2;
  int lim[2];  // positions [0, lim) the lane's two heads see (causal rows of multi-query decode)

  // The two E4M3 codes at shared address addr as a packed pair of T (the
  // lower code in the lower half, as the fragments want it).
  __device__ __forceinline__ static uint32_t fp8_pair(uint32_t addr) {
    uint16_t raw;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(raw) : "r"(addr));
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(raw, __NV_E4M3);
    if constexpr (std::is_same<T, __half>::value) {
      return (uint32_t)h.x | ((uint32_t)h.y << 16);
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
      return F16Traits<T>::pack(f.x, f.y);
    }
  }

  // Positions each of this lane's two heads (hq, hq + 1) may see; a
  // single-query unit sees every position of the sequence.
  __device__ __forceinline__ void set_limits(int lim_hq, int lim_hq1) {
    lim[0] = lim_hq;
    lim[1] = lim_hq1;
  }

  __device__ __forceinline__ void begin_unit(const T* qs, int nh, float sl2, int lane) {
    const int n = lane >> 2, kq = (lane & 3) * 2;
    const uint16_t* q16 = reinterpret_cast<const uint16_t*>(qs);
#pragma unroll
    for (int ks = 0; ks < NK; ++ks) {
      uint32_t lo = 0, hi = 0;
      if (n < nh) {
        lo = *reinterpret_cast<const uint32_t*>(q16 + n * D + ks * 16 + kq);
        hi = *reinterpret_cast<const uint32_t*>(q16 + n * D + ks * 16 + kq + 8);
      }
      qb[ks][0] = lo;
      qb[ks][1] = hi;
    }
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][i] = 0.f;
    scale_log2 = sl2;
  }

  __device__ __forceinline__ void block(const uint8_t* ks, uint8_t* vs, int ntok, int lane, float*,
                                        int tok0) {
    const uint32_t kbase = smem_addr(ks), vbase = smem_addr(vs);
    const int r = lane >> 2;
    float sc[NTT][4];
#pragma unroll
    for (int tt = 0; tt < NTT; ++tt) {
      // Two accumulators (even / odd k-steps) halve the dependent mma chain.
      float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < NK; ++kk) {
        uint32_t a[4];
        if constexpr (kFp8) {
          // A = K[16 tokens x 16 dims]: rows tt*16 + r (+8), columns (lane%4)*2 (+8);
          // chunk kk of the key block holds dims 16kk.. of every token in 16 bytes.
          const uint32_t lo = kbase + (kk * BS + tt * 16 + r) * 16 + (lane & 3) * 2, hi = lo + 8 * 16;
          a[0] = fp8_pair(lo);
          a[1] = fp8_pair(hi);
          a[2] = fp8_pair(lo + 8);
          a[3] = fp8_pair(hi + 8);
        } else {
          const int tok = tt * 16 + (lane & 15), chunk = 2 * kk + (lane >> 4);
          ldmatrix_x4(kbase + (chunk * BS + tok) * 16, a);
        }
        if (kk & 1) Mma<T>::run(c2, a, qb[kk][0], qb[kk][1]);
        else Mma<T>::run(c, a, qb[kk][0], qb[kk][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] += c2[i];
      const int t_lo = tt * 16 + r, t_hi = t_lo + 8;
      sc[tt][0] = (t_lo < ntok && tok0 + t_lo < lim[0]) ? c[0] * scale_log2 : -INFINITY;
      sc[tt][1] = (t_lo < ntok && tok0 + t_lo < lim[1]) ? c[1] * scale_log2 : -INFINITY;
      sc[tt][2] = (t_hi < ntok && tok0 + t_hi < lim[0]) ? c[2] * scale_log2 : -INFINITY;
      sc[tt][3] = (t_hi < ntok && tok0 + t_hi < lim[1]) ? c[3] * scale_log2 : -INFINITY;
    }
    float alpha[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float bm = fmaxf(sc[0][j], sc[0][j + 2]);
#pragma unroll
      for (int tt = 1; tt < NTT; ++tt) bm = fmaxf(bm, fmaxf(sc[tt][j], sc[tt][j + 2]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
      const float mn = fmaxf(m[j], bm);
      // A causal row that has seen no position yet keeps m = -inf: subtract
      // 0 instead, so its weights and rescale come out 0, not NaN.
      const float ms = (mn == -INFINITY) ? 0.f : mn;
      alpha[j] = exp2f(m[j] - ms);
      m[j] = mn;
      float ps = 0.f;
#pragma unroll
      for (int tt = 0; tt < NTT; ++tt) {
        sc[tt][j] = exp2f(sc[tt][j] - ms);
        sc[tt][j + 2] = exp2f(sc[tt][j + 2] - ms);
        ps += sc[tt][j] + sc[tt][j + 2];
      }
      l[j] = fmaf(l[j], alpha[j], ps);
    }
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) {
      acc[mt][0] *= alpha[0];
      acc[mt][1] *= alpha[1];
      acc[mt][2] *= alpha[0];
      acc[mt][3] *= alpha[1];
    }
    if (ntok < BS) {
      // Slots past the sequence end hold arbitrary cache contents; zero them
      // so that 0 * (NaN or Inf) cannot reach the accumulator.
      for (int i = lane; i < D * (BS - ntok); i += 32) {
        const int d = i / (BS - ntok), t = ntok + i % (BS - ntok);
        if constexpr (kFp8) reinterpret_cast<uint8_t*>(vs)[d * BS + t] = 0;
        else reinterpret_cast<uint16_t*>(vs)[d * BS + t] = 0;
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
#pragma unroll
    for (int tt = 0; tt < NTT; ++tt) {
      // P fragment rows = tokens, cols = heads; transpose to the B operand.
      const uint32_t p0 = F16Traits<T>::pack(sc[tt][0], sc[tt][1]);
      const uint32_t p1 = F16Traits<T>::pack(sc[tt][2], sc[tt][3]);
      const uint32_t b0 = movmatrix_trans(p0), b1 = movmatrix_trans(p1);
      // bf16 keeps 8 significant bits, so a weight rounded once can be off by
      // 2^-9 of itself: enough, over a handful of tokens, to miss the parity
      // tolerance.  The rounding remainder goes through a second product
      // (P = P_hi + P_lo, both bf16), leaving an error near 2^-17.  fp16's
      // 11 bits need no second product.
      uint32_t r0 = 0, r1 = 0;
      if constexpr (kSplitWeights) {
        const float2 h0 = F16Traits<T>::to_float2(p0), h1 = F16Traits<T>::to_float2(p1);
        r0 = movmatrix_trans(F16Traits<T>::pack(sc[tt][0] - h0.x, sc[tt][1] - h0.y));
        r1 = movmatrix_trans(F16Traits<T>::pack(sc[tt][2] - h1.x, sc[tt][3] - h1.y));
      }
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
        uint32_t a[4];
        if constexpr (kFp8) {
          // A = V[16 dims x 16 tokens]: rows mt*16 + r (+8), columns tt*16 + (lane%4)*2 (+8).
          const uint32_t lo = vbase + (mt * 16 + r) * BS + tt * 16 + (lane & 3) * 2, hi = lo + 8 * BS;
          a[0] = fp8_pair(lo);
          a[1] = fp8_pair(hi);
          a[2] = fp8_pair(lo + 8);
          a[3] = fp8_pair(hi + 8);
        } else {
          const int row = mt * 16 + (lane & 15), chunk = tt * 2 + (lane >> 4);
          ldmatrix_x4(vbase + row * (BS * 2) + chunk * 16, a);
        }
        Mma<T>::run(acc[mt], a, b0, b1);
        if constexpr (kSplitWeights) Mma<T>::run(acc[mt], a, r0, r1);
      }
    }
  }

  __device__ __forceinline__ void finish(float* acc_out, float* ml, int lane) {
    const int r = lane >> 2, hq = (lane & 3) * 2;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float ls = l[j];
      ls += __shfl_xor_sync(0xffffffffu, ls, 4);
      ls += __shfl_xor_sync(0xffffffffu, ls, 8);
      ls += __shfl_xor_sync(0xffffffffu, ls, 16);
      if (r == 0) {
        ml[(hq + j) * 2] = m[j];
        ml[(hq + j) * 2 + 1] = ls;
      }
    }
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) {
      acc_out[hq * D + mt * 16 + r] = acc[mt][0];
      acc_out[(hq + 1) * D + mt * 16 + r] = acc[mt][1];
      acc_out[hq * D + mt * 16 + r + 8] = acc[mt][2];
      acc_out[(hq + 1) * D + mt * 16 + r + 8] = acc[mt][3];
    }
  }
};

}  // namespace pa
