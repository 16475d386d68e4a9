// pa_combine.cuh -- phase 2 of paged decode attention: the cross-partition
// log-sum-exp combine of the page "paged_attention_v2_triton.py -- Triton
// PagedAttention V2 for BI-V100" (`_paged_attn_v2_reduce_kernel` and the
// module docstring's Phase 2 formula):
//
//   M = max_p m_p,   total = sum_p e^(m_p - M) l_p,
//   out = sum_p (e^(m_p - M) l_p / total) o_p,   lse = M + log(total),
//
// over the partition states (m_p, l_p, o_p) phase 1 stored for every row
// (sequence, head) of a sequence with two or more partitions; sequences with
// one partition were finished by phase 1 (single pass).  No cap on the number
// of partitions (the page drops those past its MAX_NUM_PARTS).
//
// Launch: grid (S, ceil(H / RPC)), 8 warps a CTA.  WPR warps share a row
// (WPR = 8 / RPC, chosen by the host from the largest partition count the
// table allows): warp sub of a row takes a contiguous range of its
// partitions, each lane a float4 column of the head (two at head size 256),
// loads in batches of 16 partitions (8 at head size 256); the WPR warp states of a row are then merged in shared memory
// in warp order, so the result is deterministic.  The kernel is launched as a
// programmatic dependent of phase 1: it reads the lengths first and waits for
// phase 1 to complete (griddepcontrol.wait) before it reads any state.  The
// maxima and sums of a batch come in one coalesced load each (lane j holds
// partition j's) and reach the other lanes by shuffles.
#pragma once

#include "pa_common.cuh"

namespace pa {

struct CParams {
  void* out;       // [S, H, D] (multi-query: [S, q_len, Hu, D]) of T
  float* lse;      // rows' log-sum-exp, or null
  const float* ws_m;  // [S, H, Pmax] partition maxima (natural-log units)
  const float* ws_l;  // [S, H, Pmax] partition sums
  const float* ws_o;  // [S, H, Pmax, D] normalised partition outputs
  const int32_t* lens;
  int S, H, Pmax, P, max_len;
  int wpr;             // warps per row: 1, 2, 4 or 8
  int q_len, Hu, Gu, G;  // multi-query rows (q_len > 1): row head -> output row
};

// 8 warps: with 16, CTAs of 512 threads fit one to an SM by registers and a
// long-context batch's 448 CTAs ran in three waves (phase 2: 7 -> 11 us).
constexpr int kCombineWarps = 8;

// Output row of row head h of sequence s (as in phase 1).
__device__ __forceinline__ size_t combine_out_row(const CParams& prm, int s, int h) {
  if (prm.q_len <= 1) return (size_t)s * prm.H + h;
  const int kv = h / prm.G, l = h - kv * prm.G, i = l / prm.Gu;
  return ((size_t)s * prm.q_len + i) * prm.Hu + kv * prm.Gu + (l - i * prm.Gu);
}

template <typename T, int D>
__global__ void __launch_bounds__(kCombineWarps * 32) pa_combine_kernel(const __grid_constant__ CParams prm) {
  constexpr int D4 = D / 4;                 // float4 columns of a head
  constexpr int CPL = (D4 + 31) / 32;       // columns per lane
  // Partitions whose states are loaded together (all in flight at once):
  // 16, or 8 where a lane takes two columns (registers).
  constexpr int kCombineBatch = 16 / CPL;
  __shared__ float4 s_acc[kCombineWarps][D4];
  __shared__ float s_m[kCombineWarps], s_t[kCombineWarps];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x;
  const int rpc = kCombineWarps / prm.wpr;
  const int row_local = warp / prm.wpr, sub = warp - row_local * prm.wpr;
  const int h = blockIdx.y * rpc + row_local;
  const int L = min(max(prm.lens[s], 0), prm.max_len);
  const int np = (L + prm.P - 1) / prm.P;
  if (np <= 1) return;  // finished by phase 1 (or empty: zeros written there)
  // Partition states are phase 1's output.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  float M = -INFINITY, tot = 0.f;
  float4 acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  const bool row_ok = h < prm.H;
  // Phase 1 kept the states in L2 (evict-last); they are read once here.
  const uint64_t pol_once = l2_policy_evict_first();
  if (row_ok) {
    const int per = (np + prm.wpr - 1) / prm.wpr;
    const int p_beg = min(sub * per, np), p_end = min(p_beg + per, np);
    const size_t base = ((size_t)s * prm.H + h) * prm.Pmax;
    const float4* o4 = reinterpret_cast<const float4*>(prm.ws_o) + base * D4;
    for (int p0 = p_beg; p0 < p_end; p0 += kCombineBatch) {
      // Lane j < batch holds m and l of partition p0 + j (one coalesced load
      // each); every lane holds its columns of the batch's outputs.
      const bool inj = lane < kCombineBatch && p0 + lane < p_end;
      const float mj = inj ? ld_f32_policy(prm.ws_m + base + p0 + lane, pol_once) : -INFINITY;
      const float lj = inj ? ld_f32_policy(prm.ws_l + base + p0 + lane, pol_once) : 0.f;
      float4 ov[kCombineBatch][CPL];
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) {
        const bool in = p0 + j < p_end;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int col = lane + 32 * c;
          ov[j][c] = (in && col < D4) ? ld_f4_policy(o4 + (size_t)(p0 + j) * D4 + col, pol_once)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float gm = mj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
      const float Mn = fmaxf(M, gm);
      // States a causal row never reached are (-inf, 0): while every state so
      // far is one, subtract 0 so that they weigh 0 instead of NaN.
      const float Ms = (Mn == -INFINITY) ? 0.f : Mn;
      const float sc = exp2f((M - Ms) * kLog2e);
      tot *= sc;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        acc[c].x *= sc; acc[c].y *= sc; acc[c].z *= sc; acc[c].w *= sc;
      }
      // Each lane's partition weight, then taken in partition order.
      const float wj = exp2f((mj - Ms) * kLog2e) * lj;
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) {
        const float w = __shfl_sync(0xffffffffu, wj, j);
        tot += w;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          acc[c].x = fmaf(w, ov[j][c].x, acc[c].x); acc[c].y = fmaf(w, ov[j][c].y, acc[c].y);
          acc[c].z = fmaf(w, ov[j][c].z, acc[c].z); acc[c].w = fmaf(w, ov[j][c].w, acc[c].w);
        }
      }
      M = Mn;
    }
  }
  // Merge the row's warp states in warp order.
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const int col = lane + 32 * c;
    if (col < D4) s_acc[warp][col] = acc[c];
  }
  if (lane == 0) {
    s_m[warp] = M;
    s_t[warp] = tot;
  }
  __syncthreads();
  if (!row_ok || sub != 0) return;
  const int w0 = row_local * prm.wpr;
  float Mr = -INFINITY;
  for (int w = 0; w < prm.wpr; ++w) Mr = fmaxf(Mr, s_m[w0 + w]);
  const float Ms = (Mr == -INFINITY) ? 0.f : Mr;
  float total = 0.f;
  float wt[kCombineWarps];
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) {
    wt[w] = w < prm.wpr ? exp2f((s_m[w0 + w] - Ms) * kLog2e) : 0.f;
    if (w < prm.wpr) total = fmaf(wt[w], s_t[w0 + w], total);
  }
  const float inv = total > 0.f ? 1.f / total : 0.f;
  const size_t orow = combine_out_row(prm, s, h);
  T* out = static_cast<T*>(prm.out) + orow * D;
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const int col = lane + 32 * c;
    if (col >= D4) continue;
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      if (w >= prm.wpr) break;
      const float4 a = s_acc[w0 + w][col];
      r.x = fmaf(wt[w], a.x, r.x); r.y = fmaf(wt[w], a.y, r.y);
      r.z = fmaf(wt[w], a.z, r.z); r.w = fmaf(wt[w], a.w, r.w);
    }
    store4<T>(out + col * 4, make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv));
  }
  // log-sum-exp of all the row's scores: M + log(total) (natural-log units).
  if (lane == 0 && prm.lse) prm.lse[orow] = Mr + logf(total);
}

}  // namespace pa
