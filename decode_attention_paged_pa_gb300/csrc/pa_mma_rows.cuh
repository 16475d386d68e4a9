// pa_mma_rows.cuh -- tensor-core consumer for units of 16 query rows of one
// kv head (more than 8 query rows per kv head: large GQA groups, or several
// query tokens per sequence in multi-query decode), 16-bit caches, head sizes
// 64 and 128, blocks of 16 or 32 tokens.
//
// The 16 rows fill the M = 16 side of mma.sync m16n8k16, and the tokens and
// dims are its N = 8 column tiles:
//
//   S[rows x tokens]  = Q[rows x D] . K^T[D x tokens]      (two 8-token tiles per 16 tokens)
//   O[rows x D]      += P[rows x tokens] . V[tokens x D]   (D / 8 dim tiles)
//
// With the rows in M the score fragment of the first product already is the
// weight fragment (A operand) of the second, so the weights need no
// transpose, and a row's maximum and sum over the tokens reduce over the four
// lanes of a quad.  Both cache layouts of the page "paged_attention_v2_triton.py
// -- Triton PagedAttention V2 for BI-V100" give the B operands by plain
// ldmatrix: a K block [D/8][BS][8] holds 8 dims of one token in 16 bytes (a
// column of K^T), a V block [D][BS] holds 8 tokens of one dim in 16 bytes (a
// column of V).  The query rows' A fragments are loaded once per unit.
//
// Softmax arithmetic is that of the phase-1 kernel `_paged_attn_v2_partition_kernel`
// (scores in fp32, running max, exp, running sum, rescaled accumulation); the
// weights enter the second product rounded to the element type (bf16: as the
// sum of two bf16 terms, as in MmaConsumer).  Staging is MmaConsumer's: the
// key block by a bulk copy, the value block by a swizzled tensor copy.
#pragma once

#include <type_traits>

#include "pa_mma.cuh"

namespace pa {

template <typename T_, int D_, int BS_>
struct MmaRowConsumer {
  using T = T_;
  static constexpr int D = D_, BS = BS_, GT = 16;
  static_assert((D_ == 64 || D_ == 128) && (BS_ == 16 || BS_ == 32), "head sizes 64/128, blocks of 16/32");
  static constexpr bool kTma = true;
  static constexpr bool kMma = true;
  static constexpr bool kCausal = false;  // (every unit is masked by its limits)
  static constexpr bool kFp8 = false;
  static constexpr int KVU = 1;
  static constexpr int KV_ESZ = 2;
  static constexpr uint32_t KTILE = (uint32_t)D_ * BS_ * 2;
  static constexpr uint32_t KBLK = KTILE;
  static constexpr uint32_t KREGION = al1024(KBLK);
  static constexpr uint32_t STAGE_BYTES = al1024(KREGION + KBLK);
  static constexpr uint32_t STAGE_TX = 2 * KBLK;
  static constexpr int kIssueBatch = (KBLK <= 2048) ? 32 : 16;  // as MmaConsumer
  static constexpr int kItemBlocks = 1;
  static constexpr int NK = D / 16;   // k-steps (16 dims) of the score product
  static constexpr int NN = D / 8;    // 8-dim column tiles of the value product
  static constexpr int NTT = BS / 16; // 16-token tiles per block
  static constexpr int SCRATCH_FLOATS = 0;
  // Row strides (elements) of a staged query row and of a handed-over state
  // row: the 8 rows one ldmatrix or one 8-byte store touches fall in distinct
  // shared-memory banks.
  static constexpr int QROW = D_ + 16 / (int)sizeof(T_);
  static constexpr int AROW = D_ + 8;
  static constexpr bool kSplitWeights = std::is_same<T_, __nv_bfloat16>::value;

  // Swizzled value rows of VROW = 2 BS bytes (see MmaConsumer::vchunk).
  static constexpr uint32_t VROW = (uint32_t)BS_ * 2;
  __device__ __forceinline__ static uint32_t vchunk(int d, int c) {
    return (uint32_t)d * VROW + ((uint32_t)(c ^ (((uint32_t)d * VROW >> 7) & (VROW / 16u - 1u))) << 4);
  }

  uint32_t qa[NK][4];  // A fragments of the unit's 16 query rows
  float m[2], l[2];    // rows lane / 4 and lane / 4 + 8
  float acc[NN][4];    // O fragments: dims 8n + 2 (lane % 4) (+1) of those rows
  float scale_log2;
  int lim[2];          // positions [0, lim) each of the two rows sees

  template <class F>
  __device__ __forceinline__ void set_limits(F limit_of, int lane) {
    lim[0] = limit_of(lane >> 2);
    lim[1] = limit_of((lane >> 2) + 8);
  }

  // qs: the unit's query rows [16][QROW]; rows >= nh are taken as zero.
  __device__ __forceinline__ void begin_unit(const T* qs, int nh, float sl2, int lane, int /*G*/) {
    const int r = lane >> 2;
    // ldmatrix x4 of k-step kk: matrices (rows 0-7 | 8-15) x (dims +0 | +8).
    const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), ldim = 8 * (lane >> 4);
    const uint32_t base = smem_addr(qs) + (uint32_t)(lrow * QROW + ldim) * 2u;
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      ldmatrix_x4(base + kk * 32, qa[kk]);
      if (r >= nh) qa[kk][0] = qa[kk][2] = 0u;
      if (r + 8 >= nh) qa[kk][1] = qa[kk][3] = 0u;
    }
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int n = 0; n < NN; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;
    scale_log2 = sl2;
  }

  // One staged block (its NTT 16-token tiles, one softmax update): ks = key
  // block, vs = value block; ntok of its tokens lie before the sequence end;
  // tok0 = position of its first token.
  __device__ __forceinline__ void block(const uint8_t* ks, uint8_t* vs, int ntok, int lane, float*, int tok0) {
    const int r = lane >> 2, cq = 2 * (lane & 3);
    // Scores: sc[tt][j][i], token tile j (tokens 16 tt + 8 j ..), C fragment i.
    float sc[NTT][2][4];
    // ldmatrix x4 of the keys: lane supplies token row (lane & 7) + 8 (lane >> 4)
    // of chunk 2 kk + ((lane >> 3) & 1): matrices b0, b1 of token tile 0, then of tile 1.
    const int ktok = (lane & 7) + 8 * (lane >> 4), kch = (lane >> 3) & 1;
#pragma unroll
    for (int tt = 0; tt < NTT; ++tt) {
      float c[2][4], c2[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[j][i] = c2[j][i] = 0.f;
      const uint32_t kb = smem_addr(ks) + (uint32_t)(kch * BS + tt * 16 + ktok) * 16u;
#pragma unroll
      for (int kk = 0; kk < NK; ++kk) {
        uint32_t b[4];
        ldmatrix_x4(kb + kk * 2 * BS * 16, b);
        // Two accumulators (even / odd k-steps) per token tile halve the dependent chain.
        if (kk & 1) {
          Mma<T>::run(c2[0], qa[kk], b[0], b[1]);
          Mma<T>::run(c2[1], qa[kk], b[2], b[3]);
        } else {
          Mma<T>::run(c[0], qa[kk], b[0], b[1]);
          Mma<T>::run(c[1], qa[kk], b[2], b[3]);
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int t = tt * 16 + j * 8 + cq;
        sc[tt][j][0] = (t < ntok && tok0 + t < lim[0]) ? (c[j][0] + c2[j][0]) * scale_log2 : -INFINITY;
        sc[tt][j][1] = (t + 1 < ntok && tok0 + t + 1 < lim[0]) ? (c[j][1] + c2[j][1]) * scale_log2 : -INFINITY;
        sc[tt][j][2] = (t < ntok && tok0 + t < lim[1]) ? (c[j][2] + c2[j][2]) * scale_log2 : -INFINITY;
        sc[tt][j][3] = (t + 1 < ntok && tok0 + t + 1 < lim[1]) ? (c[j][3] + c2[j][3]) * scale_log2 : -INFINITY;
      }
    }
    // Online softmax per row (row r: fragment entries 0, 1; row r + 8: 2, 3).
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float bm = -INFINITY;
#pragma unroll
      for (int tt = 0; tt < NTT; ++tt)
#pragma unroll
        for (int j = 0; j < 2; ++j) bm = fmaxf(bm, fmaxf(sc[tt][j][2 * h], sc[tt][j][2 * h + 1]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      const float mn = fmaxf(m[h], bm);
      // A causal row that has seen no position yet keeps m = -inf: subtract
      // 0 instead, so its weights and rescale come out 0, not NaN.
      const float ms = (mn == -INFINITY) ? 0.f : mn;
      alpha[h] = exp2f(m[h] - ms);
      m[h] = mn;
      float ps = 0.f;
#pragma unroll
      for (int tt = 0; tt < NTT; ++tt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          sc[tt][j][2 * h] = exp2f(sc[tt][j][2 * h] - ms);
          sc[tt][j][2 * h + 1] = exp2f(sc[tt][j][2 * h + 1] - ms);
          ps += sc[tt][j][2 * h] + sc[tt][j][2 * h + 1];
        }
      l[h] = fmaf(l[h], alpha[h], ps);
    }
#pragma unroll
    for (int n = 0; n < NN; ++n) {
      acc[n][0] *= alpha[0];
      acc[n][1] *= alpha[0];
      acc[n][2] *= alpha[1];
      acc[n][3] *= alpha[1];
    }
    // Values: ldmatrix x4 gives b0, b1 (tokens +0..7, +8..15) of dim tiles
    // 2 nn and 2 nn + 1: lane supplies dim 16 nn + (lane & 7) + 8 (lane >> 4),
    // 16-byte chunk 2 tt + ((lane >> 3) & 1) of its row.
    const int vd = (lane & 7) + 8 * (lane >> 4), vch = (lane >> 3) & 1;
    const bool ragged = ntok < BS;
#pragma unroll
    for (int tt = 0; tt < NTT; ++tt) {
      // The score fragment is the weight fragment: a0 (row r, tokens cq, cq+1),
      // a1 (row r+8, same tokens), a2, a3 (tokens 8+cq, 9+cq).
      uint32_t pa[4], pr[4] = {0u, 0u, 0u, 0u};
      pa[0] = F16Traits<T>::pack(sc[tt][0][0], sc[tt][0][1]);
      pa[1] = F16Traits<T>::pack(sc[tt][0][2], sc[tt][0][3]);
      pa[2] = F16Traits<T>::pack(sc[tt][1][0], sc[tt][1][1]);
      pa[3] = F16Traits<T>::pack(sc[tt][1][2], sc[tt][1][3]);
      if constexpr (kSplitWeights) {
        // bf16 keeps 8 significant bits: the rounding remainder of each weight
        // goes through a second product (see MmaConsumer).
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = i >> 1, e = 2 * (i & 1);
          const float2 hv = F16Traits<T>::to_float2(pa[i]);
          pr[i] = F16Traits<T>::pack(sc[tt][j][e] - hv.x, sc[tt][j][e + 1] - hv.y);
        }
      }
      // Value slots past the sequence end hold arbitrary contents: cleared in
      // the fragments so that 0 * (NaN or Inf) cannot reach the accumulator.
      uint32_t k0 = 0xffffffffu, k1 = 0xffffffffu;
      if (ragged) {
        const int t = tt * 16 + cq;
        k0 = (t < ntok ? 0xffffu : 0u) | (t + 1 < ntok ? 0xffff0000u : 0u);
        k1 = (t + 8 < ntok ? 0xffffu : 0u) | (t + 9 < ntok ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int nn = 0; nn < NN / 2; ++nn) {
        uint32_t b[4];
        ldmatrix_x4(smem_addr(vs) + vchunk(nn * 16 + vd, 2 * tt + vch), b);
        if (ragged) {
          b[0] &= k0; b[1] &= k1; b[2] &= k0; b[3] &= k1;
        }
        Mma<T>::run(acc[2 * nn], pa, b[0], b[1]);
        Mma<T>::run(acc[2 * nn + 1], pa, b[2], b[3]);
        if constexpr (kSplitWeights) {
          Mma<T>::run(acc[2 * nn], pr, b[0], b[1]);
          Mma<T>::run(acc[2 * nn + 1], pr, b[2], b[3]);
        }
      }
    }
  }

  // Write this warp's state: acc_out [16][AROW] (unnormalised), ml [16][2] = (m, l).
  __device__ __forceinline__ void finish(float* acc_out, float* ml, int lane) {
    const int r = lane >> 2, cq = 2 * (lane & 3);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float ls = l[h];
      ls += __shfl_xor_sync(0xffffffffu, ls, 1);
      ls += __shfl_xor_sync(0xffffffffu, ls, 2);
      if ((lane & 3) == 0) {
        ml[(r + 8 * h) * 2] = m[h];
        ml[(r + 8 * h) * 2 + 1] = ls;
      }
    }
#pragma unroll
    for (int n = 0; n < NN; ++n) {
      *reinterpret_cast<float2*>(acc_out + r * AROW + 8 * n + cq) = make_float2(acc[n][0], acc[n][1]);
      *reinterpret_cast<float2*>(acc_out + (r + 8) * AROW + 8 * n + cq) = make_float2(acc[n][2], acc[n][3]);
    }
  }
};

}  // namespace pa
