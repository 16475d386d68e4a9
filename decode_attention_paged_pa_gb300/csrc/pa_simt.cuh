// pa_simt.cuh -- CUDA-core consumer for the paged decode kernel: one warp
// turns one staged physical block (K block [D/x][BS][x] with x = 16 bytes of
// elements -- 8 for fp16/bf16, 4 for fp32 -- and V block [D][BS]) into an
// online-softmax update of its private (m, l, acc) state for GT query heads.
//
// Follows the phase-1 kernel `_paged_attn_v2_partition_kernel` of the page
// "paged_attention_v2_triton.py -- Triton PagedAttention V2 for BI-V100":
// scores = scale * q . k (fp32), masked tokens -> -inf, block max, exp, running
// sum and rescaled V accumulation.  Unlike the page, each K/V block is read
// once for all GT query heads of its kv head, and the accumulator is kept
// unnormalised per warp (normalised once, when the warps' states are combined).
#pragma once

#include "pa_common.cuh"

namespace pa {

// CAUSAL_: the instance for the causal rows of multi-query decode (each
// head masked to the positions it may see; used for fp32 elements, whose
// multi-query rows run on this family).
template <typename T_, int D_, int BS_, int GT_, bool CAUSAL_ = false>
struct SimtConsumer {
  using T = T_;
  static constexpr int D = D_, BS = BS_, GT = GT_;
  static constexpr bool kMma = false;
  static constexpr bool kCausal = CAUSAL_;
  // Blocks the producer warp issues together (MHA batch: 8 / 24 / 32 blocks
  // 363.5 / 355.3 / 359.4 us).
  static constexpr int kIssueBatch = 24;
  static constexpr bool kFp8 = false;
  static constexpr int KV_ESZ = (int)sizeof(T_);  // bytes per cached element
  // A ring stage holds one whole block, key then value, each one bulk copy.
  static constexpr bool kTma = false;
  static constexpr uint32_t KTILE = (uint32_t)D_ * BS_ * sizeof(T_);
  static constexpr uint32_t KREGION = KTILE, STAGE_BYTES = 2 * KTILE, STAGE_TX = 2 * KTILE;
  static constexpr int KVU = 1;  // kv heads per unit
  static constexpr int kItemBlocks = 1;  // blocks per work item
  static constexpr uint32_t KBLK = KTILE;
  static constexpr int EPC = elems_per_chunk<T_>();  // elements per 16-byte chunk
  // q.k: each lane takes QKD dims of one token; LPT lanes share a token
  // (32 dims for fp32, whose registers hold half as many per byte; half the
  // head for head sizes 80, 96, 112).
  static constexpr bool kPow2D = (D & (D - 1)) == 0;
  // 8-token fp32 blocks: a quarter of the head a lane (8 tokens a pass: the
  // block is one pass), 32 dims at head size 256 (two passes).
  static constexpr bool kB8 = BS_ == 8 && KV_ESZ == 4;
  static constexpr int QKD = kB8 ? (D == 256 ? 32 : D / 4)
                                 : !kPow2D ? D / 2 : (D >= 128 && KV_ESZ == 2) ? 64 : 32;
  static constexpr int LPT = D / QKD;
  static constexpr int TPP = 32 / LPT;        // tokens per pass over the warp
  static constexpr int NPASS = BS / TPP;
  static constexpr int QCH = QKD / EPC;       // 16-byte K chunks per lane and token
  // p.V: lane (row r, chunk c) reads the 16-byte chunk c (EPC tokens) of V
  // rows r, r + RPP, ...; consecutive lanes read consecutive 16-byte words.
  static constexpr int CPR = BS / EPC;        // chunks per V row
  static constexpr int RPP = 32 / CPR;        // rows per warp pass
  static constexpr int NROW = D / RPP;        // rows per lane
  static constexpr int SCRATCH_FLOATS = GT * BS;  // per warp: p of the current block

  static_assert(NPASS >= 1 && BS % TPP == 0, "block size must cover whole passes");
  static_assert(QKD % EPC == 0 && 32 % LPT == 0 && D % RPP == 0, "head size must split over the lanes");

  float qf[GT][QKD];
  float m[GT], l[GT];
  float acc[GT][NROW];
  int lim[GT];  // causal instances: positions [0, lim) each head sees

  // q rows [GT][D] in shared memory; rows >= nh are treated as zero.
  // Row strides, in elements, of a staged query row and of a handed-over
  // state row (no padding: a warp's loads and stores here stay in one row).
  static constexpr int QROW = D;
  static constexpr int AROW = D;

  __device__ __forceinline__ void begin_unit(const T* qs, int nh, float scale_log2, int lane, int /*G*/) {
    const int slice = lane / TPP;
#pragma unroll
    for (int g = 0; g < GT; ++g) {
#pragma unroll
      for (int i = 0; i < QCH; ++i) {
        float f[EPC];
        if (g < nh) {
          const uint4 raw = *reinterpret_cast<const uint4*>(qs + g * QROW + slice * QKD + i * EPC);
          unpack_chunk<T>(raw, f);
        } else {
#pragma unroll
          for (int e = 0; e < EPC; ++e) f[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < EPC; ++e) qf[g][i * EPC + e] = f[e] * scale_log2;
      }
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int r = 0; r < NROW; ++r) acc[g][r] = 0.f;
    }
  }

  // Positions each head of the unit may see (causal instances only).
  template <class F>
  __device__ __forceinline__ void set_limits(F limit_of, int) {
    if constexpr (kCausal) {
#pragma unroll
      for (int g = 0; g < GT; ++g) lim[g] = limit_of(g);
    }
  }

  // One staged block: ks = K block, vs = V block (shared memory), ntok valid
  // tokens (1..BS) starting at position tok0.  pw = this warp's scratch
  // (SCRATCH_FLOATS floats).
  __device__ __forceinline__ void block(const uint8_t* ks, uint8_t* vs, int ntok, int lane,
                                        float* pw, int tok0) {
    const int tl = lane % TPP, slice = lane / TPP;
    float sc[NPASS][GT];
#pragma unroll
    for (int ps = 0; ps < NPASS; ++ps) {
      const int t = ps * TPP + tl;
      // One partial sum per 16-byte chunk keeps the FMA chains short.
      float part[QCH][GT];
#pragma unroll
      for (int i = 0; i < QCH; ++i) {
        const int c = slice * QCH + i;
        const uint4 raw = *reinterpret_cast<const uint4*>(ks + (c * BS + t) * 16);
        float f[EPC];
        unpack_chunk<T>(raw, f);
#pragma unroll
        for (int g = 0; g < GT; ++g) {
          float a = qf[g][i * EPC] * f[0];
#pragma unroll
          for (int e = 1; e < EPC; ++e) a = fmaf(qf[g][i * EPC + e], f[e], a);
          part[i][g] = a;
        }
      }
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        if constexpr ((QCH & (QCH - 1)) == 0) {
#pragma unroll
          for (int w = QCH / 2; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) part[i][g] += part[i + w][g];
        } else {
#pragma unroll
          for (int i = 1; i < QCH; ++i) part[0][g] += part[i][g];
        }
        sc[ps][g] = part[0][g];
#pragma unroll
        for (int off = TPP; off < 32; off <<= 1) sc[ps][g] += __shfl_xor_sync(0xffffffffu, sc[ps][g], off);
        if (t >= ntok) sc[ps][g] = -INFINITY;
        if constexpr (kCausal) {
          if (tok0 + t >= lim[g]) sc[ps][g] = -INFINITY;
        }
      }
    }
    // Online softmax update (log2 domain: q carries scale * log2(e)).
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      float bm = sc[0][g];
#pragma unroll
      for (int ps = 1; ps < NPASS; ++ps) bm = fmaxf(bm, sc[ps][g]);
#pragma unroll
      for (int off = 1; off < TPP; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
      const float mn = fmaxf(m[g], bm);
      // A causal row that has seen no position yet keeps m = -inf: subtract
      // 0 instead, so its weights and rescale come out 0, not NaN.
      const float ms = (kCausal && mn == -INFINITY) ? 0.f : mn;
      const float alpha = exp2f(m[g] - ms);
      m[g] = mn;
      float psum = 0.f;
#pragma unroll
      for (int ps = 0; ps < NPASS; ++ps) {
        const float p = exp2f(sc[ps][g] - ms);
        sc[ps][g] = p;
        psum += p;
      }
      l[g] = fmaf(l[g], alpha, psum);
#pragma unroll
      for (int r = 0; r < NROW; ++r) acc[g][r] *= alpha;
      if (slice == 0) {
#pragma unroll
        for (int ps = 0; ps < NPASS; ++ps) pw[g * BS + ps * TPP + tl] = sc[ps][g];
      }
    }
    if (ntok < BS) {
      // Slots past the sequence end hold arbitrary cache contents; zero them
      // so that 0 * (NaN or Inf) cannot reach the accumulator.  Rows of up to
      // 32 tokens: a lane clears its dims' tails (no index division; the
      // head-size-256 batch +0.7%); longer rows: consecutive slots over the
      // lanes (a lane a row would put every lane's stores in one bank).
      if constexpr (BS <= 32) {
        for (int d = lane; d < D; d += 32)
          for (int t = ntok; t < BS; ++t) {
            if constexpr (sizeof(T) == 4) reinterpret_cast<uint32_t*>(vs)[d * BS + t] = 0u;
            else reinterpret_cast<uint16_t*>(vs)[d * BS + t] = 0;
          }
      } else {
        for (int i = lane; i < D * (BS - ntok); i += 32) {
          const int d = i / (BS - ntok), t = ntok + i % (BS - ntok);
          if constexpr (sizeof(T) == 4) reinterpret_cast<uint32_t*>(vs)[d * BS + t] = 0u;
          else reinterpret_cast<uint16_t*>(vs)[d * BS + t] = 0;
        }
      }
      fence_proxy_async_smem();
    }
    __syncwarp();
    const int r0 = lane / CPR, c = lane % CPR;
    float pv[GT][EPC];
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
      for (int e4 = 0; e4 < EPC; e4 += 4) {
        const float4 a = *reinterpret_cast<const float4*>(pw + g * BS + c * EPC + e4);
        pv[g][e4] = a.x; pv[g][e4 + 1] = a.y; pv[g][e4 + 2] = a.z; pv[g][e4 + 3] = a.w;
      }
#pragma unroll
    for (int r = 0; r < NROW; ++r) {
      const int d = r0 + r * RPP;
      const uint4 raw = *reinterpret_cast<const uint4*>(vs + (d * BS + c * EPC) * KV_ESZ);
      float f[EPC];
      unpack_chunk<T>(raw, f);
#pragma unroll
      for (int g = 0; g < GT; ++g)
#pragma unroll
        for (int e = 0; e < EPC; ++e) acc[g][r] = fmaf(pv[g][e], f[e], acc[g][r]);
    }
    __syncwarp();
  }

  // Write this warp's state: acc_out [GT][D] (unnormalised), ml [GT][2] = (m, l).
  __device__ __forceinline__ void finish(float* acc_out, float* ml, int lane) {
    const int r0 = lane / CPR, c = lane % CPR;
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      float ls = l[g];
#pragma unroll
      for (int off = 1; off < TPP; off <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
#pragma unroll
      for (int r = 0; r < NROW; ++r) {
        float v = acc[g][r];
#pragma unroll
        for (int off = 1; off < CPR; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (c == 0) acc_out[g * AROW + r0 + r * RPP] = v;
      }
      if (lane == 0) {
        ml[g * 2] = m[g];
        ml[g * 2 + 1] = ls;
      }
    }
  }
};

}  // namespace pa
