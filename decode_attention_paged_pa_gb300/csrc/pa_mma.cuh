// pa_mma.cuh -- tensor-core consumer for the paged decode kernel, for groups
// of query heads that share one kv head (GQA).  Per staged block the group's
// scores and weighted values are two small dense contractions:
//
//   S[tokens x heads]  = K[tokens x D] . Q^T[D x heads]       (mma m16n8k16, M = 16 tokens)
//   O^T[D x heads]    += V^T[D x tokens] . P^T[tokens x heads] (mma m16n8k16, M = 16 dims)
//
// with 8 query heads as the N = 8 side of the instruction (units of 16 query
// rows of one kv head take MmaRowConsumer, pa_mma_rows.cuh).  Both cache layouts
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
//
// Staging.  A ring stage holds one physical block of one kv head: the key
// block [D/8][BS][8] by a 1-D bulk copy (it is contiguous), and, with 16-bit
// caches in blocks of 16 tokens or more (kTma), the value block [D][BS] by a
// 3-D tensor copy (the value cache viewed as [blocks * kv heads][D][BS]) that
// stores its rows of R = 2 BS bytes in the R-byte swizzle: the 16-byte chunk
// index of a row (address bits 4..) is XORed with address bits 7.. .  Without
// it, the rows an ldmatrix reads (8 consecutive dims, one 16-byte chunk each)
// are R bytes apart and fall in 8 R / 128 distinct bank groups only (a 2-, 4-
// or 8-way conflict for R = 32, 64, 128); with it they fall in 8 (checked on
// the CPU for every head size).  fp8 caches and 8-token blocks are staged by
// 1-D bulk copies of the contiguous value block.
#pragma once

#include <cuda_fp8.h>

#include <type_traits>

#include "pa_common.cuh"

namespace pa {

constexpr uint32_t al1024(uint32_t x) { return (x + 1023u) & ~1023u; }

// FP8_: the caches hold E4M3 codes (one byte per element, key layout
// [D/16][BS][16]).  Every E4M3 value is exact in fp16, so both products then
// run as fp16 MMAs whatever T is: K and V codes widen to fp16 in registers
// (one conversion per code pair), the query is scaled by a power of two into
// fp16's range (exact for bf16 queries too: bf16 keeps 8 significant bits,
// fp16 11) with the inverse factor folded into the score scale, and the
// weights enter the value product rounded once to fp16, as in the fp16 path.
//
// The fp8 fragments are read with 4-byte shared loads.  Within a 16-dim
// k-step, lane quad c holds dims 4c..4c+3 of its token rows (slots k = 2c,
// 2c+1 and 2c+8, 2c+9; the query fragments use the same assignment), and MMA
// row i of a 16-token tile holds token kTok(i) below: a lane's value word
// then covers four consecutive tokens of one dim, and the eight token rows a
// lane quad reads fall in distinct shared-memory banks.  Two 8-token blocks
// fill one tile (its tokens 0..7 from the first), and a 64-token block runs
// as two softmax updates of two tiles each.
// KVU_: kv heads per unit.  With fewer than 8 query heads per kv head (G),
// the 8 columns of a tile hold the query heads of KVU = 8 / G consecutive kv
// heads: a stage then holds one block of each of them (the cache keeps the kv
// heads of a block contiguous, so still one copy for the keys and one for the
// values), and each product runs once per kv head with the query (scores) or
// weight (values) columns of the other kv heads zeroed, into the same
// accumulators.  The softmax, the weights and the stage's waits then serve
// KVU kv heads at once, and the copies are KVU times larger.
template <typename T_, int D_, int BS_, bool FP8_ = false, int KVU_ = 1>
struct MmaConsumer {
  using T = T_;
  using MT = typename std::conditional<FP8_, __half, T_>::type;  // operand type of the products
  static constexpr int NT = 1;  // 8-head column tiles per unit
  // kTma: the value block is staged by a swizzled tensor copy.
  static constexpr bool kTma = !FP8_ && BS_ >= 16;
  static constexpr int D = D_, BS = BS_, GT = 8 * NT;
  static constexpr int KVU = KVU_;
  static_assert(KVU_ == 1 || 8 % KVU_ == 0, "kv-head groups share one 8-column tile");
  static constexpr bool kMma = true;
  static constexpr bool kCausal = false;  // (every unit is masked by its limits)
  static constexpr bool kFp8 = FP8_;
  static constexpr int KV_ESZ = FP8_ ? 1 : 2;  // bytes per cached element
  // A stage: the key blocks of the unit's KVU kv heads (KTILE bytes each,
  // contiguous), then (at KREGION, 1024-byte aligned for the swizzled tensor
  // copy) their value blocks; STAGE_TX bytes land per stage.  A kv head's
  // value block starts KTILE bytes after the previous one's: a multiple of the
  // swizzle's repeat (8 rows), as every head size is a multiple of 8.
  static constexpr uint32_t KTILE = (uint32_t)D_ * BS * KV_ESZ;
  static constexpr uint32_t KBLK = (uint32_t)KVU_ * KTILE;
  static constexpr uint32_t KREGION = kTma ? al1024(KBLK) : KBLK;
  static constexpr uint32_t STAGE_BYTES = kTma ? al1024(KREGION + KBLK) : KREGION + KBLK;
  static constexpr uint32_t STAGE_TX = 2 * KBLK;
  // Blocks the producer warp issues together (one per lane, as their stages
  // free up): 16, or 32 for copies of 2 KB or less.  (Batches of 4 / 8 / 16
  // blocks: the multi-query GQA batch 558 / 464 / 459 us, the fp8 one
  // 298 / 259 / 257 us; the producer re-polls a batch's stages with a
  // growing back-off, which small batches hit more often.)
  static constexpr int kIssueBatch = (KBLK <= 2048) ? 32 : 16;
  static constexpr int NK = D / 16;    // k-steps of the score product
  static constexpr int NMT = D / 16;   // 16-dim tiles of the value product
  // 16-token tiles per block.  An 8-token block fills half of one tile: the
  // score rows of tokens 8..15 are masked and their value columns are zero.
  static constexpr int NTT = BS >= 16 ? BS / 16 : 1;
  // Blocks per work item: a pair for 8-token blocks (one 16-token tile) and
  // for 16-token fp8 blocks of one kv head (one softmax update over two
  // tiles); one otherwise.
  static constexpr int kItemBlocks = (BS == 8) ? 2 : (BS == 16 && FP8_ && KVU_ == 1) ? 2 : 1;
  static_assert(D % 16 == 0 && (BS == 8 || BS % 16 == 0), "head size a multiple of 16; block 8 or 16k");
  static constexpr int SCRATCH_FLOATS = 0;
  // Row strides, in elements, of a staged query row and of a handed-over
  // state row: 16 bytes past the row, so that the 8 rows a fragment load or
  // a state store touches (rows a multiple of 128 bytes long otherwise) fall
  // in distinct shared-memory banks.
  static constexpr int QROW = D_ + 16 / (int)sizeof(T_);
  static constexpr int AROW = D_ + 4;
  static constexpr bool kSplitWeights = std::is_same<MT, __nv_bfloat16>::value;

  // Byte offset, in a staged value block, of the 16-byte chunk c (tokens
  // 8c .. 8c + 7) of dim d's row.  Tensor-copied blocks have rows of
  // VROW = 2 BS bytes in the VROW-byte swizzle: the chunk index is XORed
  // with the row's address bits 7 and up (VROW / 16 - 1 of them matter).
  static constexpr uint32_t VROW = (uint32_t)BS_ * KV_ESZ;
  __device__ __forceinline__ static uint32_t vchunk(int d, int c) {
    if constexpr (kTma) {
      return (uint32_t)d * VROW + ((uint32_t)(c ^ (((uint32_t)d * VROW >> 7) & (VROW / 16u - 1u))) << 4);
    } else {
      return (uint32_t)d * VROW + (uint32_t)c * 16u;
    }
  }

  // Q^T fragments (B operand) per column tile and kv head of the unit, packed
  // element pairs (with KVU > 1, the columns of the other kv heads zero).
  uint32_t qb[NK][NT * KVU_][2];
  int ub;  // KVU > 1: the kv head (0 .. KVU - 1) of this lane's weight column
  float m[NT][2], l[NT][2];  // heads 8t + 2*(lane%4) and 8t + 2*(lane%4) + 1 of tile t
  float acc[NMT][NT][4];
  float scale_log2;
  int lim[NT][2];  // positions [0, lim) the lane's heads see (causal rows of multi-query decode)

  // fp8 caches: the token (within its 16-token tile) that MMA row i holds.
  // Rows 2c, 2c+1 and 2c+8, 2c+9 -- the score rows that become the weight
  // slots of lane quad c -- hold tokens 4c..4c+3, the lower pair on rows
  // 2c, 2c+1 for c < 2 and on rows 2c+8, 2c+9 for c >= 2.
  __device__ __forceinline__ static int kTok(int i) {
    const int c = (i & 7) >> 1;
    return 4 * c + 2 * ((c >> 1) ^ (i >> 3)) + (i & 1);
  }

  __device__ __forceinline__ static uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
  }

  // Two E4M3 codes (the low code in bits 0-7) as a packed fp16 pair.
  __device__ __forceinline__ static uint32_t e4m3x2(uint32_t codes) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(codes & 0xffffu), __NV_E4M3);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
  }

  // Positions each of this lane's heads may see: limit_of(h) for head h of
  // the unit (a single-query unit sees every position of the sequence).
  template <class F>
  __device__ __forceinline__ void set_limits(F limit_of, int lane) {
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int j = 0; j < 2; ++j) lim[t][j] = limit_of(8 * t + (lane & 3) * 2 + j);
  }

  // G: query heads per kv head (columns n of a KVU > 1 unit belong to kv
  // head n / G of the unit).
  __device__ __forceinline__ void begin_unit(const T* qs, int nh, float sl2, int lane, int G) {
    const int n = lane >> 2, kq = (lane & 3) * 2;
    ub = KVU_ > 1 ? n / G : 0;
    const uint16_t* q16 = reinterpret_cast<const uint16_t*>(qs);
    if constexpr (kFp8) {
      // Dims 16ks + 4c .. +3 of head n, scaled by 2^s so that the unit's
      // largest |q| lies below 2^15 (fp16 tops out near 2^16).
      float amax = 0.f;
#pragma unroll
      for (int ks = 0; ks < NK; ++ks) {
        if (n < nh) {
          const uint2 w = *reinterpret_cast<const uint2*>(q16 + n * QROW + ks * 16 + 2 * kq);
          const float2 a = F16Traits<T>::to_float2(w.x), b = F16Traits<T>::to_float2(w.y);
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y))));
        }
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // amax < 2^(E - 126) for a normal binary32 with biased exponent E;
      // zero, subnormal, Inf or NaN leave the query unscaled.
      const int E = (__float_as_int(amax) >> 23) & 0xff;
      const int s = (E == 0 || E == 255) ? 0 : max(-110, min(110, 141 - E));
      const float up = __int_as_float((127 + s) << 23), down = __int_as_float((127 - s) << 23);
#pragma unroll
      for (int ks = 0; ks < NK; ++ks) {
        uint32_t lo = 0, hi = 0;
        if (n < nh) {
          const uint2 w = *reinterpret_cast<const uint2*>(q16 + n * QROW + ks * 16 + 2 * kq);
          const float2 a = F16Traits<T>::to_float2(w.x), b = F16Traits<T>::to_float2(w.y);
          lo = F16Traits<__half>::pack(a.x * up, a.y * up);
          hi = F16Traits<__half>::pack(b.x * up, b.y * up);
        }
#pragma unroll
        for (int u = 0; u < KVU_; ++u) {
          const bool mine = KVU_ == 1 || ub == u;
          qb[ks][u][0] = mine ? lo : 0u;
          qb[ks][u][1] = mine ? hi : 0u;
        }
      }
      sl2 *= down;
    } else {
#pragma unroll
      for (int ks = 0; ks < NK; ++ks)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int h = 8 * t + n;
          uint32_t lo = 0, hi = 0;
          if (h < nh) {
            lo = *reinterpret_cast<const uint32_t*>(q16 + h * QROW + ks * 16 + kq);
            hi = *reinterpret_cast<const uint32_t*>(q16 + h * QROW + ks * 16 + kq + 8);
          }
#pragma unroll
          for (int u = 0; u < KVU_; ++u) {
            const bool mine = KVU_ == 1 || ub == u;
            qb[ks][t * KVU_ + u][0] = mine ? lo : 0u;
            qb[ks][t * KVU_ + u][1] = mine ? hi : 0u;
          }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      m[t][0] = m[t][1] = -INFINITY;
      l[t][0] = l[t][1] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][t][i] = 0.f;
    scale_log2 = sl2;
  }

  __device__ __forceinline__ void block(const uint8_t* ks, uint8_t* vs, int ntok, int lane, float*,
                                        int tok0) {
    if constexpr (kFp8) {
      if constexpr (BS == 8) {
        // Half a tile: the rows of tokens 8..15 read block A again (masked).
        fp8_pair8(ks, vs, ks, vs, ntok, lane, tok0);
      } else {
        // At most two tiles per softmax update (a 64-token block takes two
        // updates): the value words of a whole update stay in registers.
        constexpr int NTU = NTT < 2 ? NTT : 2;
#pragma unroll
        for (int h = 0; h < NTT / NTU; ++h) {
          if (h > 0 && ntok <= h * 16 * NTU) break;
          uint32_t klo[NTU], khi[NTU], vv[NTU];
#pragma unroll
          for (int tt = 0; tt < NTU; ++tt) {
            const int tile = h * NTU + tt;
            fp8_rows(smem_addr(ks) + tile * 16 * 16, smem_addr(vs) + tile * 16, lane, klo[tt], khi[tt], vv[tt]);
          }
          fp8_tiles<NTU>(klo, khi, vv, ntok - h * 16 * NTU, lane, tok0 + h * 16 * NTU);
        }
      }
      return;
    }
    if constexpr (!kFp8) {
      // The NTT tiles of one block (an 8-token block: half a tile).
      uint32_t kt[NTT], vt[NTT];
      int vc[NTT];
#pragma unroll
      for (int tt = 0; tt < NTT; ++tt) {
        kt[tt] = smem_addr(ks) + tt * 16 * 16;
        vt[tt] = smem_addr(vs);
        vc[tt] = 2 * tt;
      }
      tiles<NTT>(kt, vt, vc, false, ntok, lane, tok0);
    }
  }

  // Two consecutive 8-token blocks of a unit as one 16-token tile: block A
  // (tokens 0..7, full) and block B (tokens 8..15, ntok - 8 of them valid).
  // Over an fp8 cache in 16-token blocks: two consecutive blocks A and B
  // (ntok tokens of 17..32 valid) as the two tiles of one work item.
  __device__ __forceinline__ void block_pair(const uint8_t* ksA, uint8_t* vsA, const uint8_t* ksB,
                                             uint8_t* vsB, int ntok, int lane, int tok0) {
    if constexpr (kFp8 && BS == 8) {
      fp8_pair8(ksA, vsA, ksB, vsB, ntok, lane, tok0);
    } else if constexpr (kFp8) {
      static_assert(BS == 16, "fp8 pairs are 8- or 16-token blocks");
      uint32_t klo[2], khi[2], vv[2];
      fp8_rows(smem_addr(ksA), smem_addr(vsA), lane, klo[0], khi[0], vv[0]);
      fp8_rows(smem_addr(ksB), smem_addr(vsB), lane, klo[1], khi[1], vv[1]);
      fp8_tiles<2>(klo, khi, vv, ntok, lane, tok0);
    } else if constexpr (BS == 8) {
      // One tile: K fragment rows 8..15 (lanes 8..15, 24..31) and V fragment
      // token columns 8..15 (lanes 16..31) come from block B.
      const uint32_t kt[1] = {smem_addr((lane & 8) ? ksB : ksA)};
      const uint32_t vt[1] = {smem_addr((lane >> 4) ? vsB : vsA)};
      const int vc[1] = {0};
      tiles<1>(kt, vt, vc, true, ntok, lane, tok0);
    } else {
      static_assert(BS == 16, "16-bit pairs are 8- or 16-token blocks");
      const uint32_t kt[2] = {smem_addr(ksA), smem_addr(ksB)};
      const uint32_t vt[2] = {smem_addr(vsA), smem_addr(vsB)};
      const int vc[2] = {0, 0};
      tiles<2>(kt, vt, vc, false, ntok, lane, tok0);
    }
  }

  // The 16-bit products over the NTI 16-token tiles of one work item (tokens
  // 16 tt .. 16 tt + 15 of the item in tile tt): this lane's ldmatrix rows of
  // tile tt's keys at kt[tt] + (chunk * BS + row) * 16, its value columns in
  // the 16-byte chunk vc[tt] + (lane >> 4) of the dim rows at vt[tt].  8-token
  // blocks (NTI = 1) fill one tile from two blocks through the lanes'
  // addresses; without block B (has_b false) rows 8..15 repeat A's and are
  // masked, their value columns are zero.  ntok: the item's tokens that lie
  // before the sequence end.
  template <int NTI>
  __device__ __forceinline__ void tiles(const uint32_t (&kt)[NTI], const uint32_t (&vt)[NTI], const int (&vc)[NTI],
                                        bool has_b, int ntok, int lane, int tok0) {
    const int r = lane >> 2;
    float sc[NTI][NT][4];
#pragma unroll
    for (int tt = 0; tt < NTI; ++tt) {
      // Two accumulators (even / odd k-steps) per column tile halve the
      // dependent mma chain.
      float c[NT][4], c2[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[t][i] = c2[t][i] = 0.f;
#pragma unroll
      for (int kk = 0; kk < NK; ++kk) {
        // (An 8-token block: rows 8..15 are block B's, or repeat rows 0..7 and are masked below.)
        const int tok = lane & (BS >= 16 ? 15 : 7), chunk = 2 * kk + (lane >> 4);
#pragma unroll
        for (int u = 0; u < KVU; ++u) {
          uint32_t a[4];
          ldmatrix_x4(kt[tt] + u * KTILE + (chunk * BS + tok) * 16, a);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if ((kk * KVU + u) & 1) Mma<T>::run(c2[t], a, qb[kk][t * KVU + u][0], qb[kk][t * KVU + u][1]);
            else Mma<T>::run(c[t], a, qb[kk][t * KVU + u][0], qb[kk][t * KVU + u][1]);
          }
        }
      }
      const int t_lo = tt * 16 + r, t_hi = t_lo + 8;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int i = 0; i < 4; ++i) c[t][i] += c2[t][i];
        sc[tt][t][0] = (t_lo < ntok && tok0 + t_lo < lim[t][0]) ? c[t][0] * scale_log2 : -INFINITY;
        sc[tt][t][1] = (t_lo < ntok && tok0 + t_lo < lim[t][1]) ? c[t][1] * scale_log2 : -INFINITY;
        sc[tt][t][2] = (t_hi < ntok && tok0 + t_hi < lim[t][0]) ? c[t][2] * scale_log2 : -INFINITY;
        sc[tt][t][3] = (t_hi < ntok && tok0 + t_hi < lim[t][1]) ? c[t][3] * scale_log2 : -INFINITY;
      }
    }
    float alpha[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float bm = fmaxf(sc[0][t][j], sc[0][t][j + 2]);
#pragma unroll
        for (int tt = 1; tt < NTI; ++tt) bm = fmaxf(bm, fmaxf(sc[tt][t][j], sc[tt][t][j + 2]));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        const float mn = fmaxf(m[t][j], bm);
        // A causal row that has seen no position yet keeps m = -inf: subtract
        // 0 instead, so its weights and rescale come out 0, not NaN.
        const float ms = (mn == -INFINITY) ? 0.f : mn;
        alpha[t][j] = exp2f(m[t][j] - ms);
        m[t][j] = mn;
        float ps = 0.f;
#pragma unroll
        for (int tt = 0; tt < NTI; ++tt) {
          sc[tt][t][j] = exp2f(sc[tt][t][j] - ms);
          sc[tt][t][j + 2] = exp2f(sc[tt][t][j + 2] - ms);
          ps += sc[tt][t][j] + sc[tt][t][j + 2];
        }
        l[t][j] = fmaf(l[t][j], alpha[t][j], ps);
      }
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        acc[mt][t][0] *= alpha[t][0];
        acc[mt][t][1] *= alpha[t][1];
        acc[mt][t][2] *= alpha[t][0];
        acc[mt][t][3] *= alpha[t][1];
      }
    // Slots past the sequence end hold arbitrary cache contents: the value
    // fragments' elements of those tokens are zeroed in registers, so that
    // 0 * (NaN or Inf) cannot reach the accumulator.  A lane's value fragment
    // covers tokens 2c, 2c + 1 (registers 0, 1) and 2c + 8, 2c + 9
    // (registers 2, 3) of each tile, c = lane % 4; low halves first.
    const bool ragged = ntok < 16 * NTI;
    const int tq = 2 * (lane & 3);
#pragma unroll
    for (int tt = 0; tt < NTI; ++tt) {
      // P fragment rows = tokens, cols = heads; transpose to the B operand.
      // bf16 keeps 8 significant bits, so a weight rounded once can be off by
      // 2^-9 of itself: enough, over a handful of tokens, to miss the parity
      // tolerance.  The rounding remainder goes through a second product
      // (P = P_hi + P_lo, both bf16), leaving an error near 2^-17.  fp16's
      // 11 bits need no second product.
      uint32_t b0[NT], b1[NT], r0[NT], r1[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint32_t p0 = F16Traits<T>::pack(sc[tt][t][0], sc[tt][t][1]);
        const uint32_t p1 = F16Traits<T>::pack(sc[tt][t][2], sc[tt][t][3]);
        b0[t] = movmatrix_trans(p0);
        b1[t] = movmatrix_trans(p1);
        r0[t] = r1[t] = 0u;
        if constexpr (kSplitWeights) {
          const float2 h0 = F16Traits<T>::to_float2(p0), h1 = F16Traits<T>::to_float2(p1);
          r0[t] = movmatrix_trans(F16Traits<T>::pack(sc[tt][t][0] - h0.x, sc[tt][t][1] - h0.y));
          r1[t] = movmatrix_trans(F16Traits<T>::pack(sc[tt][t][2] - h1.x, sc[tt][t][3] - h1.y));
        }
      }
#pragma unroll
      for (int u = 0; u < KVU; ++u) {
        // kv head u's value product takes the weight columns of its own query heads.
        const bool mine = KVU == 1 || ub == u;
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
          uint32_t a[4];
          const int chunk = vc[tt] + (BS >= 16 ? (lane >> 4) : 0);
          ldmatrix_x4(vt[tt] + u * KTILE + vchunk(mt * 16 + (lane & 15), chunk), a);
          if (BS < 16 && !has_b) a[2] = a[3] = 0u;  // tokens 8..15 of the tile do not exist
          if (ragged) {
            const int t = tt * 16 + tq;
            const uint32_t k0 = (t < ntok ? 0xffffu : 0u) | (t + 1 < ntok ? 0xffff0000u : 0u);
            const uint32_t k1 = (t + 8 < ntok ? 0xffffu : 0u) | (t + 9 < ntok ? 0xffff0000u : 0u);
            a[0] &= k0; a[1] &= k0; a[2] &= k1; a[3] &= k1;
          }
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            Mma<T>::run(acc[mt][t], a, mine ? b0[t] : 0u, mine ? b1[t] : 0u);
            if constexpr (kSplitWeights) Mma<T>::run(acc[mt][t], a, mine ? r0[t] : 0u, mine ? r1[t] : 0u);
          }
        }
      }
    }
  }

  // This lane's fragment addresses in a 16-token fp8 tile whose key rows start
  // at kb (token row t of chunk kk at kb + (kk * BS + t) * 16) and whose value
  // rows start at vb (dim d at vb + d * BS): its two key rows (MMA rows
  // lane / 4 and lane / 4 + 8) in chunk 0, and its four tokens in dim row 0.
  __device__ __forceinline__ static void fp8_rows(uint32_t kb, uint32_t vb, int lane, uint32_t& klo,
                                                  uint32_t& khi, uint32_t& vv) {
    const int r = lane >> 2, c = lane & 3;
    klo = kb + kTok(r) * 16 + c * 4;
    khi = kb + kTok(r + 8) * 16 + c * 4;
    vv = vb + c * 4;
  }

  // One 16-token tile of two 8-token fp8 blocks: tokens 0..7 from block A,
  // 8..15 from block B (ntok of the 16 before the sequence end).
  __device__ __forceinline__ void fp8_pair8(const uint8_t* ksA, const uint8_t* vsA, const uint8_t* ksB,
                                            const uint8_t* vsB, int ntok, int lane, int tok0) {
    const int r = lane >> 2, c = lane & 3;
    const int tl = kTok(r), th = kTok(r + 8);
    const uint32_t klo[1] = {smem_addr(tl < 8 ? ksA : ksB) + (tl & 7) * 16 + c * 4};
    const uint32_t khi[1] = {smem_addr(th < 8 ? ksA : ksB) + (th & 7) * 16 + c * 4};
    const uint32_t vv[1] = {smem_addr(c < 2 ? vsA : vsB) + (c & 1) * 4};
    fp8_tiles<1>(klo, khi, vv, ntok, lane, tok0);
  }

  // NT2 16-token tiles of E4M3 codes (see the note above the struct), by this
  // lane's fragment addresses (fp8_rows): its key words of chunk kk at
  // klo[tt] / khi[tt] + kk * BS * 16, its value word of dim d at vv[tt] + d * BS.
  template <int NT2>
  __device__ __forceinline__ void fp8_tiles(const uint32_t (&klo)[NT2], const uint32_t (&khi)[NT2],
                                            const uint32_t (&vv)[NT2], int ntok, int lane, int tok0) {
    const int r = lane >> 2, c = lane & 3;
    const int trow_lo = kTok(r), trow_hi = kTok(r + 8);
    float sc[NT2][4];
#pragma unroll
    for (int tt = 0; tt < NT2; ++tt) {
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int u = 0; u < KVU; ++u) {
        // Chunk kk of a key block holds dims 16kk..16kk+15 of every token in 16 bytes.
        uint32_t wk[NK][2];
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
          wk[kk][0] = lds32(klo[tt] + u * KTILE + kk * BS * 16);
          wk[kk][1] = lds32(khi[tt] + u * KTILE + kk * BS * 16);
        }
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
          const uint32_t a[4] = {e4m3x2(wk[kk][0]), e4m3x2(wk[kk][1]), e4m3x2(wk[kk][0] >> 16),
                                 e4m3x2(wk[kk][1] >> 16)};
          if ((kk * KVU + u) & 1) Mma<__half>::run(c1, a, qb[kk][u][0], qb[kk][u][1]);
          else Mma<__half>::run(c0, a, qb[kk][u][0], qb[kk][u][1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) c0[i] += c1[i];
      const int t_lo = tt * 16 + trow_lo, t_hi = tt * 16 + trow_hi;
      sc[tt][0] = (t_lo < ntok && tok0 + t_lo < lim[0][0]) ? c0[0] * scale_log2 : -INFINITY;
      sc[tt][1] = (t_lo < ntok && tok0 + t_lo < lim[0][1]) ? c0[1] * scale_log2 : -INFINITY;
      sc[tt][2] = (t_hi < ntok && tok0 + t_hi < lim[0][0]) ? c0[2] * scale_log2 : -INFINITY;
      sc[tt][3] = (t_hi < ntok && tok0 + t_hi < lim[0][1]) ? c0[3] * scale_log2 : -INFINITY;
    }
    // Value words (dims mt*16 + r and + 8, tokens tt*16 + 4c .. +3) do not
    // depend on the weights: read them before the softmax.
    // (Those of the unit's first kv head; the others' are read in their turn.)
    uint32_t wv[NT2][NMT][2];
#pragma unroll
    for (int tt = 0; tt < NT2; ++tt)
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
        wv[tt][mt][0] = lds32(vv[tt] + (mt * 16 + r) * BS);
        wv[tt][mt][1] = lds32(vv[tt] + (mt * 16 + r + 8) * BS);
      }
    float alpha[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float bm = fmaxf(sc[0][j], sc[0][j + 2]);
#pragma unroll
      for (int tt = 1; tt < NT2; ++tt) bm = fmaxf(bm, fmaxf(sc[tt][j], sc[tt][j + 2]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
      const float mn = fmaxf(m[0][j], bm);
      const float ms = (mn == -INFINITY) ? 0.f : mn;  // a causal row that has seen nothing yet
      alpha[j] = exp2f(m[0][j] - ms);
      m[0][j] = mn;
      float ps = 0.f;
#pragma unroll
      for (int tt = 0; tt < NT2; ++tt) {
        sc[tt][j] = exp2f(sc[tt][j] - ms);
        sc[tt][j + 2] = exp2f(sc[tt][j + 2] - ms);
        ps += sc[tt][j] + sc[tt][j + 2];
      }
      l[0][j] = fmaf(l[0][j], alpha[j], ps);
    }
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) {
      acc[mt][0][0] *= alpha[0];
      acc[mt][0][1] *= alpha[1];
      acc[mt][0][2] *= alpha[0];
      acc[mt][0][3] *= alpha[1];
    }
    // The weights' B fragments per tile (quads c >= 2 find their tokens 4c,
    // 4c+1 in score rows 2c+8, 2c+9), and the value bytes each tile keeps:
    // slots past the sequence end hold arbitrary codes (E4M3 has NaNs), which
    // are cleared so that 0 * NaN cannot reach the accumulator.
    uint32_t bw[NT2][2], vmask[NT2];
#pragma unroll
    for (int tt = 0; tt < NT2; ++tt) {
      const int keep = ntok - (tt * 16 + c * 4);
      vmask[tt] = keep >= 4 ? 0xffffffffu : (keep <= 0 ? 0u : (1u << (8 * keep)) - 1u);
      const uint32_t p0 = F16Traits<__half>::pack(sc[tt][0], sc[tt][1]);
      const uint32_t p1 = F16Traits<__half>::pack(sc[tt][2], sc[tt][3]);
      const uint32_t b0 = movmatrix_trans(p0), b1 = movmatrix_trans(p1);
      bw[tt][0] = c >= 2 ? b1 : b0;
      bw[tt][1] = c >= 2 ? b0 : b1;
    }
#pragma unroll
    for (int u = 0; u < KVU; ++u) {
      if (u > 0) {
#pragma unroll
        for (int tt = 0; tt < NT2; ++tt)
#pragma unroll
          for (int mt = 0; mt < NMT; ++mt) {
            wv[tt][mt][0] = lds32(vv[tt] + u * KTILE + (mt * 16 + r) * BS);
            wv[tt][mt][1] = lds32(vv[tt] + u * KTILE + (mt * 16 + r + 8) * BS);
          }
      }
      // kv head u's value product takes the weight columns of its own query heads.
      const bool mine = KVU == 1 || ub == u;
#pragma unroll
      for (int tt = 0; tt < NT2; ++tt) {
        const uint32_t b0 = mine ? bw[tt][0] : 0u, b1 = mine ? bw[tt][1] : 0u;
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
          const uint32_t v0 = wv[tt][mt][0] & vmask[tt], v1 = wv[tt][mt][1] & vmask[tt];
          const uint32_t a[4] = {e4m3x2(v0), e4m3x2(v1), e4m3x2(v0 >> 16), e4m3x2(v1 >> 16)};
          Mma<__half>::run(acc[mt][0], a, b0, b1);
        }
      }
    }
  }

  __device__ __forceinline__ void finish(float* acc_out, float* ml, int lane) {
    const int r = lane >> 2, hq = (lane & 3) * 2;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float ls = l[t][j];
        ls += __shfl_xor_sync(0xffffffffu, ls, 4);
        ls += __shfl_xor_sync(0xffffffffu, ls, 8);
        ls += __shfl_xor_sync(0xffffffffu, ls, 16);
        if (r == 0) {
          ml[(8 * t + hq + j) * 2] = m[t][j];
          ml[(8 * t + hq + j) * 2 + 1] = ls;
        }
      }
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        // Accumulator rows r and r + 8 of value tile mt hold dims mt * 16 + r and + 8.
        float* o = acc_out + (8 * t + hq) * AROW;
        const int d_lo = mt * 16 + r, d_hi = d_lo + 8;
        o[d_lo] = acc[mt][t][0];
        o[AROW + d_lo] = acc[mt][t][1];
        o[d_hi] = acc[mt][t][2];
        o[AROW + d_hi] = acc[mt][t][3];
      }
  }
};

}  // namespace pa
