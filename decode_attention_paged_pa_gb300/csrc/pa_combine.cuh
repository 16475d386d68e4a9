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
// Work is cut into row groups: RPC rows of one sequence, WPR = NW / RPC warps
// a row.  Warp sub of a row takes a contiguous range of its partitions, each
// lane a float4 column of the head (two at head size 256), loads in batches
// of 16 partitions (8 at head size 256; the batch's maxima and sums in one
// coalesced load each, lane j holding partition j's, shuffled to the other
// lanes); the WPR warp states of a row are then merged in shared memory in
// warp order, so the result is deterministic.
//
// Two launch shapes, both programmatic dependents of phase 1 that read the
// lengths first and wait for phase 1 to complete (griddepcontrol.wait) before
// they read any state:
//  - pa_combine_rows_kernel (up to kRowsMaxSeqs sequences, when the table
//    allows more than 16 partitions): one CTA of 16
//    warps per SM, persistent over the batch's row groups, each sequence's WPR
//    chosen from its own partition count (the smallest power of two that
//    leaves a warp at most 16 partitions, up to 16).  A long row then spreads
//    over 16 warps (one batch of loads each) while short rows pack 16 to a CTA,
//    and the grid is one wave however skewed the lengths.
//  - pa_combine_kernel (otherwise): grid (S, ceil(H / RPC)), 8 warps a CTA,
//    one WPR for the launch from the table's largest partition count.
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
  int wpr;             // pa_combine_kernel: warps per row, 1, 2, 4 or 8
  int q_len, Hu, Gu, G;  // multi-query rows (q_len > 1): row head -> output row
};

// pa_combine_kernel: 8 warps where a row takes 8 of them, 4 otherwise (with
// 16, CTAs of 512 threads fit one to an SM by registers and a long-context
// batch's 448 CTAs ran in three waves).
constexpr int kCombineWarps = 8;
// pa_combine_rows_kernel: 16 warps, one CTA per SM; batches of up to this many
// sequences (their row-group prefix is kept in shared memory).
constexpr int kRowsWarps = 16;
constexpr int kRowsMaxSeqs = 2048;

// Output row of row head h of sequence s (as in phase 1).
__device__ __forceinline__ size_t combine_out_row(const CParams& prm, int s, int h) {
  if (prm.q_len <= 1) return (size_t)s * prm.H + h;
  const int kv = h / prm.G, l = h - kv * prm.G, i = l / prm.Gu;
  return ((size_t)s * prm.q_len + i) * prm.Hu + kv * prm.Gu + (l - i * prm.Gu);
}

__device__ __forceinline__ int seq_partitions(const CParams& prm, int s) {
  const int L = min(max(prm.lens[s], 0), prm.max_len);
  return (L + prm.P - 1) / prm.P;
}

// Combine the row group of rows h0 .. h0 + NW / wpr - 1 (those below H) of
// sequence s, which has np >= 2 partitions: wpr warps a row.  Every thread of
// the CTA calls it; it ends with the shared-memory merge done (the caller
// separates two calls by a barrier).
template <typename T, int D, int NW>
__device__ __forceinline__ void combine_rows(const CParams& prm, int s, int np, int wpr, int h0, int warp,
                                             int lane, float4 (*s_acc)[D / 4], float* s_m, float* s_t) {
  constexpr int D4 = D / 4;                 // float4 columns of a head
  constexpr int CPL = (D4 + 31) / 32;       // columns per lane
  // Partitions whose states are loaded together (all in flight at once):
  // 16, or 8 where a lane takes two columns (registers).
  constexpr int kCombineBatch = 16 / CPL;
  const int row_local = warp / wpr, sub = warp - row_local * wpr;
  const int h = h0 + row_local;

  float M = -INFINITY, tot = 0.f;
  float4 acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  const bool row_ok = h < prm.H;
  // Phase 1 kept the states in L2 (evict-last); they are read once here.
  const uint64_t pol_once = l2_policy_evict_first();
  if (row_ok) {
    const int per = (np + wpr - 1) / wpr;
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
  const int w0 = row_local * wpr;
  float Mr = -INFINITY;
  for (int w = 0; w < wpr; ++w) Mr = fmaxf(Mr, s_m[w0 + w]);
  const float Ms = (Mr == -INFINITY) ? 0.f : Mr;
  float total = 0.f;
  float wt[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    wt[w] = w < wpr ? exp2f((s_m[w0 + w] - Ms) * kLog2e) : 0.f;
    if (w < wpr) total = fmaf(wt[w], s_t[w0 + w], total);
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
    for (int w = 0; w < NW; ++w) {
      if (w >= wpr) break;
      const float4 a = s_acc[w0 + w][col];
      r.x = fmaf(wt[w], a.x, r.x); r.y = fmaf(wt[w], a.y, r.y);
      r.z = fmaf(wt[w], a.z, r.z); r.w = fmaf(wt[w], a.w, r.w);
    }
    store4<T>(out + col * 4, make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv));
  }
  // log-sum-exp of all the row's scores: M + log(total) (natural-log units).
  if (lane == 0 && prm.lse) prm.lse[orow] = Mr + logf(total);
}

template <typename T, int D, int NW>
__global__ void __launch_bounds__(NW * 32) pa_combine_kernel(const __grid_constant__ CParams prm) {
  __shared__ float4 s_acc[NW][D / 4];
  __shared__ float s_m[NW], s_t[NW];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x;
  const int np = seq_partitions(prm, s);
  if (np <= 1) return;  // finished by phase 1 (or empty: zeros written there)
  // Partition states are phase 1's output.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int rpc = NW / prm.wpr;
  combine_rows<T, D, NW>(prm, s, np, prm.wpr, blockIdx.y * rpc, warp, lane, s_acc, s_m, s_t);
}

// Warps per row of a sequence with np partitions (pa_combine_rows_kernel).
__device__ __forceinline__ int rows_wpr(int np) {
  int w = 1;
  while (w < kRowsWarps && w * 16 < np) w <<= 1;
  return w;
}

template <typename T, int D>
__global__ void __launch_bounds__(kRowsWarps * 32, 1) pa_combine_rows_kernel(const __grid_constant__ CParams prm) {
  __shared__ float4 s_acc[kRowsWarps][D / 4];
  __shared__ float s_m[kRowsWarps], s_t[kRowsWarps];
  __shared__ int s_pref[kRowsMaxSeqs + 1];  // row groups before each sequence
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = prm.S;
  // Row groups per sequence (none below two partitions) and their prefix:
  // one warp, 32 sequences a step, an inclusive shuffle scan.
  if (warp == 0) {
    int carry = 0;
    for (int b = 0; b < S; b += 32) {
      const int s = b + lane;
      int ng = 0;
      if (s < S) {
        const int np = seq_partitions(prm, s);
        if (np > 1) {
          const int rpc = kRowsWarps / rows_wpr(np);
          ng = (prm.H + rpc - 1) / rpc;
        }
      }
      int x = ng;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (s < S) s_pref[s + 1] = carry + x;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) s_pref[0] = 0;
  }
  __syncthreads();
  const int total = s_pref[S];
  if ((int)blockIdx.x >= total) return;
  // Partition states are phase 1's output.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int v = blockIdx.x; v < total; v += gridDim.x) {
    int lo = 0, hi = S;  // s_pref[lo] <= v < s_pref[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pref[mid] <= v) lo = mid; else hi = mid;
    }
    const int s = lo, np = seq_partitions(prm, s), wpr = rows_wpr(np), rpc = kRowsWarps / wpr;
    combine_rows<T, D, kRowsWarps>(prm, s, np, wpr, (v - s_pref[s]) * rpc, warp, lane, s_acc, s_m, s_t);
    __syncthreads();  // the next row group reuses s_acc, s_m, s_t
  }
}

}  // namespace pa
