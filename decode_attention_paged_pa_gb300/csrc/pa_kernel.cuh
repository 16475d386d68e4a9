// pa_kernel.cuh -- persistent, warp-specialised paged decode attention kernel.
//
// Work unit = (sequence s, partition p, head group hg): the tokens
// [p*P, min((p+1)*P, L)) of s against GT query heads that share one kv head.
// This is the phase-1 program of the page "paged_attention_v2_triton.py --
// Triton PagedAttention V2 for BI-V100" (`_paged_attn_v2_partition_kernel`,
// grid (seq, head, partition)), except that only used partitions become units
// and the GT heads of a group share every K/V load.
//
// One CTA per SM runs until the units run out:
//   * warp NC (producer): takes units from a global counter (dynamic
//     scheduling balances skewed sequence lengths), publishes each unit's
//     description and query rows through a 2-slot unit queue, and streams the
//     unit's physical K and V blocks -- each a contiguous D*BS*2-byte run in
//     the page's layouts -- into an NSTAGE-deep shared-memory ring with 1-D
//     bulk async copies completing on mbarriers;
//   * warps 0..NC-1 (consumers): block j of a unit goes to warp j % NC, which
//     folds it into its private online-softmax state (SimtConsumer or
//     MmaConsumer).  At the end of a unit the warps' states are combined in
//     shared memory into the partition's (m_p, l_p, o_p).
// Sequences with one partition write the output directly (single pass).  For
// longer sequences each unit stores its partition state in the workspace and
// takes a ticket; the CTA that completes a (sequence, head group) performs the
// phase-2 combine of `_paged_attn_v2_reduce_kernel` (M = max m_p,
// w_p = e^(m_p - M) l_p / sum, out = sum w_p o_p) for all its partitions.
// Unused partitions get the sentinels (m = -inf, l = 0) of the page.
#pragma once

#include "pa_common.cuh"

namespace pa {

struct KParams {
  void* out;
  const void* q;
  const void* kc;
  const void* vc;
  const int32_t* bt;
  const int32_t* lens;
  float* ws_m;   // [S, H, Pmax]
  float* ws_l;   // [S, H, Pmax]
  float* ws_o;   // [S, H, Pmax, D]
  int* hdr;      // kHdrInts ints
  int* tickets;  // [S, n_hg]
  float scale_log2;
  int S, H, KH, G, MB, num_blocks, P, Pmax;
  int hg_per_kv;  // ceil(G / GT)
  int n_hg;       // KH * hg_per_kv
  long long timeout_ns;
};

struct UnitInfo {
  int s, p, hg, t0, t1, nb, np, nh, h0;
  int pad[3];
};

constexpr uint32_t al16(uint32_t x) { return (x + 15u) & ~15u; }

template <class C, int NC_, int NSTAGE_>
struct Layout {
  static constexpr int NC = NC_, NSTAGE = NSTAGE_, UQ = 2;
  static constexpr int NCT = NC * 32;          // consumer threads
  static constexpr int THREADS = NCT + 32;     // + producer warp
  static constexpr int RCH = 64;               // partitions per combine chunk
  static constexpr uint32_t KBYTES = C::D * C::BS * 2;
  static constexpr uint32_t STAGE = 2 * KBYTES;
  static constexpr uint32_t RING = NSTAGE * STAGE;
  static constexpr uint32_t QSLOT = C::GT * C::D * 2;
  static constexpr uint32_t OFF_Q = RING;
  static constexpr uint32_t OFF_EPI_ACC = al16(OFF_Q + UQ * QSLOT);
  static constexpr uint32_t OFF_EPI_ML = al16(OFF_EPI_ACC + NC * C::GT * C::D * 4);
  static constexpr uint32_t OFF_SCR = al16(OFF_EPI_ML + NC * C::GT * 2 * 4);
  static constexpr uint32_t OFF_RED = al16(OFF_SCR + NC * C::SCRATCH_FLOATS * 4);
  static constexpr uint32_t OFF_RSTAT = al16(OFF_RED + C::GT * RCH * 4);
  static constexpr uint32_t OFF_SCAN = al16(OFF_RSTAT + C::GT * 2 * 4);
  static constexpr uint32_t OFF_INFO = al16(OFF_SCAN + THREADS * 4);
  static constexpr uint32_t OFF_BAR = al16(OFF_INFO + UQ * sizeof(UnitInfo));
  static constexpr uint32_t OFF_FLAGS = al16(OFF_BAR + (2 * NSTAGE + 2 * UQ) * 8);
  static constexpr uint32_t OFF_PREF = al16(OFF_FLAGS + 16);
  static constexpr uint32_t FIXED = OFF_PREF;
  static constexpr uint32_t bytes(int S) { return al16(OFF_PREF + (uint32_t)(S + 1) * 4); }
  static constexpr int OUTS = (C::GT * C::D + NCT - 1) / NCT;  // combine outputs per thread
};

template <class C, class LY>
__device__ __forceinline__ void producer_loop(const KParams& prm, uint8_t* smem, const int* pref,
                                              UnitInfo* info, volatile int* abort_flag, int lane) {
  using T = typename C::T;
  constexpr int D = C::D, BS = C::BS, GT = C::GT, NS = LY::NSTAGE, UQ = LY::UQ;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_full = sbase + LY::OFF_BAR, bar_empty = bar_full + NS * 8;
  const uint32_t bar_ufull = bar_empty + NS * 8, bar_uempty = bar_ufull + UQ * 8;
  int* err = prm.hdr + kHdrError;
  const uint64_t pol_stream = l2_policy_evict_first();
  const uint64_t pol_keep = l2_policy_evict_last();
  const int S = prm.S;
  const int total = pref[S] * prm.n_hg;
  const int max_len = prm.MB * BS;

  uint32_t g = 0;   // K/V blocks issued by this CTA
  uint32_t kq = 0;  // units published
  int u = 0;
  if (lane == 0) u = atomicAdd(prm.hdr + kHdrWork, 1);
  u = __shfl_sync(0xffffffffu, u, 0);
  bool ok = true;
  while (true) {
    const int slot = kq % UQ;
    const uint32_t par = (kq / UQ) & 1u;
    if (lane == 0) ok = wait_bounded(bar_uempty + 8 * slot, par ^ 1u, abort_flag, err, prm.timeout_ns);
    ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
    if (!ok) break;
    if (u >= total) {
      if (lane == 0) {
        info[slot].s = -1;
        mbar_arrive(bar_ufull + 8 * slot);
      }
      break;
    }
    const int pair = u / prm.n_hg, hg = u - pair * prm.n_hg;
    int lo = 0, hi = S;  // pref[lo] <= pair < pref[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pref[mid] <= pair) lo = mid; else hi = mid;
    }
    const int s = lo, p = pair - pref[s], np = pref[s + 1] - pref[s];
    const int L = min(max(prm.lens[s], 0), max_len);
    const int t0 = p * prm.P, t1 = min(t0 + prm.P, L);
    const int nb = (t1 - t0 + BS - 1) / BS;
    const int kv = hg / prm.hg_per_kv, hgk = hg - kv * prm.hg_per_kv;
    const int h0 = kv * prm.G + hgk * GT;
    const int nh = min(GT, prm.G - hgk * GT);
    int u_next = 0;
    if (lane == 0) {
      u_next = atomicAdd(prm.hdr + kHdrWork, 1);
      UnitInfo& I = info[slot];
      I.s = s; I.p = p; I.hg = hg; I.t0 = t0; I.t1 = t1; I.nb = nb; I.np = np; I.nh = nh; I.h0 = h0;
      const uint32_t qbytes = (uint32_t)(nh * D * 2);
      mbar_arrive_expect_tx(bar_ufull + 8 * slot, qbytes);
      bulk_copy_g2s(sbase + LY::OFF_Q + slot * LY::QSLOT,
                    static_cast<const T*>(prm.q) + ((size_t)s * prm.H + h0) * D, qbytes,
                    bar_ufull + 8 * slot, pol_keep);
    }
    ++kq;
    const int32_t* btrow = prm.bt + (size_t)s * prm.MB + t0 / BS;
    for (int jb = 0; jb < nb && ok; jb += 32) {
      const int cnt = min(32, nb - jb);
      int b = 0;
      if (lane < cnt) {
        b = __ldg(btrow + jb + lane);
        if ((unsigned)b >= (unsigned)prm.num_blocks) {
          atomicCAS(err, 0, kErrDeviceBounds);
          b = 0;  // keep the pipeline going on a valid block; the result is flagged
        }
      }
      for (int i = 0; i < cnt; ++i) {
        const int bi = __shfl_sync(0xffffffffu, b, i);
        if (lane == 0) {
          const uint32_t st = g % NS, ph = (g / NS) & 1u;
          ok = wait_bounded(bar_empty + 8 * st, ph ^ 1u, abort_flag, err, prm.timeout_ns);
          if (ok) {
            const uint32_t dst = sbase + st * LY::STAGE;
            const size_t off = ((size_t)bi * prm.KH + kv) * (size_t)(D * BS);
            mbar_arrive_expect_tx(bar_full + 8 * st, LY::STAGE);
            bulk_copy_g2s(dst, static_cast<const T*>(prm.kc) + off, LY::KBYTES, bar_full + 8 * st, pol_stream);
            bulk_copy_g2s(dst + LY::KBYTES, static_cast<const T*>(prm.vc) + off, LY::KBYTES,
                          bar_full + 8 * st, pol_stream);
          }
        }
        ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
        if (!ok) break;
        ++g;
      }
    }
    if (!ok) break;
    u = __shfl_sync(0xffffffffu, u_next, 0);
  }
  if (!ok && lane == 0) {
    // Aborted: let copies that may still be in flight land before the CTA
    // exits (bounded; the abort flag is ignored here).
    const long long drain_ns = prm.timeout_ns;
    for (uint32_t i = (g > (uint32_t)NS ? g - NS : 0u); i < g; ++i) {
      const uint32_t bar = bar_full + 8 * (i % NS), ph = (i / NS) & 1u;
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar, ph) && (long long)(global_timer_ns() - t0) < drain_ns) {}
    }
    for (uint32_t i = (kq > (uint32_t)UQ ? kq - UQ : 0u); i < kq; ++i) {
      const uint32_t bar = bar_ufull + 8 * (i % UQ), ph = (i / UQ) & 1u;
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar, ph) && (long long)(global_timer_ns() - t0) < drain_ns) {}
    }
  }
}

template <class C, class LY>
__device__ __forceinline__ void consumer_loop(const KParams& prm, uint8_t* smem, const int* pref,
                                              const UnitInfo* info, volatile int* abort_flag,
                                              int* last_flag, int warp, int lane) {
  using T = typename C::T;
  constexpr int D = C::D, BS = C::BS, GT = C::GT, NC = LY::NC, NCT = LY::NCT, NS = LY::NSTAGE,
                UQ = LY::UQ, RCH = LY::RCH, OUTS = LY::OUTS;
  const int ctid = warp * 32 + lane;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_full = sbase + LY::OFF_BAR, bar_empty = bar_full + NS * 8;
  const uint32_t bar_ufull = bar_empty + NS * 8, bar_uempty = bar_ufull + UQ * 8;
  float* epi_acc = reinterpret_cast<float*>(smem + LY::OFF_EPI_ACC);
  float* epi_ml = reinterpret_cast<float*>(smem + LY::OFF_EPI_ML);
  float* scr = reinterpret_cast<float*>(smem + LY::OFF_SCR) + warp * C::SCRATCH_FLOATS;
  float* rw = reinterpret_cast<float*>(smem + LY::OFF_RED);
  float* rstat = reinterpret_cast<float*>(smem + LY::OFF_RSTAT);
  int* err = prm.hdr + kHdrError;
  const int S = prm.S, H = prm.H, Pmax = prm.Pmax;
  T* out = static_cast<T*>(prm.out);

  // Unused partitions: sentinels (m = -inf, l = 0).  Empty sequences: zeros.
  {
    const long long n1 = (long long)S * H * Pmax;
    for (long long i = (long long)blockIdx.x * NCT + ctid; i < n1; i += (long long)gridDim.x * NCT) {
      const int s = (int)(i / ((long long)H * Pmax));
      const int p = (int)(i % Pmax);
      if (p >= pref[s + 1] - pref[s]) {
        prm.ws_m[i] = -INFINITY;
        prm.ws_l[i] = 0.f;
      }
    }
    const long long n2 = (long long)S * H * (D / 8);
    for (long long i = (long long)blockIdx.x * NCT + ctid; i < n2; i += (long long)gridDim.x * NCT) {
      const int s = (int)(i / ((long long)H * (D / 8)));
      if (pref[s + 1] == pref[s]) reinterpret_cast<uint4*>(out)[i] = make_uint4(0, 0, 0, 0);
    }
  }

  C cons;
  uint32_t g = 0, k = 0;
  while (true) {
    const int slot = k % UQ;
    const uint32_t par = (k / UQ) & 1u;
    const bool okw = wait_bounded(bar_ufull + 8 * slot, par, abort_flag, err, prm.timeout_ns);
    const UnitInfo I = info[slot];
    const bool stop = named_barrier_or(1, NCT, !okw || I.s < 0 || *abort_flag != 0);
    if (stop) break;
    cons.begin_unit(reinterpret_cast<const T*>(smem + LY::OFF_Q + slot * LY::QSLOT), I.nh,
                    prm.scale_log2, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_uempty + 8 * slot);
    ++k;

    for (int j = warp; j < I.nb; j += NC) {
      const uint32_t gj = g + j, st = gj % NS, ph = (gj / NS) & 1u;
      bool okb = wait_bounded(bar_full + 8 * st, ph, abort_flag, err, prm.timeout_ns);
      okb = __all_sync(0xffffffffu, okb);
      const int ntok = min(BS, I.t1 - I.t0 - j * BS);
      if (okb) cons.block(smem + st * LY::STAGE, smem + st * LY::STAGE + LY::KBYTES, ntok, lane, scr);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }
    g += I.nb;

    // Combine the NC warp states into the partition's (m_p, l_p, o_p).
    cons.finish(epi_acc + warp * GT * D, epi_ml + warp * GT * 2, lane);
    named_barrier_sync(1, NCT);
    const bool single = (I.np == 1);
#pragma unroll
    for (int o = 0; o < OUTS; ++o) {
      const int idx = ctid + o * NCT;
      if (idx >= GT * D) break;
      const int gh = idx / D, d = idx - gh * D;
      if (gh >= I.nh) continue;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w) M = fmaxf(M, epi_ml[(w * GT + gh) * 2]);
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float f = exp2f(epi_ml[(w * GT + gh) * 2] - M);
        num = fmaf(f, epi_acc[(w * GT + gh) * D + d], num);
        den = fmaf(f, epi_ml[(w * GT + gh) * 2 + 1], den);
      }
      const float val = num / den;
      const int h = I.h0 + gh;
      const size_t sh = (size_t)I.s * H + h;
      if (single) {
        out[sh * D + d] = F16Traits<T>::from_float(val);
      } else {
        prm.ws_o[(sh * Pmax + I.p) * D + d] = val;
      }
      if (d == 0) {
        prm.ws_m[sh * Pmax + I.p] = M * kLn2;
        prm.ws_l[sh * Pmax + I.p] = den;
      }
    }
    if (!single) {
      __threadfence();
      named_barrier_sync(1, NCT);
      if (ctid == 0) {
        int* ticket = prm.tickets + (size_t)I.s * prm.n_hg + I.hg;
        const int t = atomicAdd(ticket, 1);
        const int last = (t == I.np - 1);
        if (last) *ticket = 0;
        *last_flag = last;
      }
      named_barrier_sync(1, NCT);
      if (*last_flag) {
        __threadfence();
        // Phase 2 for this (sequence, head group): per head M and 1/total
        // (warp per head), then the weighted sum of the o_p in chunks.
        for (int gh = warp; gh < I.nh; gh += NC) {
          const size_t base = ((size_t)I.s * H + I.h0 + gh) * Pmax;
          float M = -INFINITY;
          for (int p = lane; p < I.np; p += 32) M = fmaxf(M, __ldcg(prm.ws_m + base + p));
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
          float tot = 0.f;
          for (int p = lane; p < I.np; p += 32)
            tot = fmaf(exp2f((__ldcg(prm.ws_m + base + p) - M) * kLog2e), __ldcg(prm.ws_l + base + p), tot);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
          if (lane == 0) {
            rstat[gh * 2] = M;
            rstat[gh * 2 + 1] = 1.f / tot;
          }
        }
        float racc[OUTS];
#pragma unroll
        for (int o = 0; o < OUTS; ++o) racc[o] = 0.f;
        for (int c0 = 0; c0 < I.np; c0 += RCH) {
          const int cn = min(RCH, I.np - c0);
          named_barrier_sync(1, NCT);
          for (int i = ctid; i < I.nh * RCH; i += NCT) {
            const int gh = i / RCH, pp = i - gh * RCH;
            if (pp < cn) {
              const size_t e = ((size_t)I.s * H + I.h0 + gh) * Pmax + c0 + pp;
              rw[i] = exp2f((__ldcg(prm.ws_m + e) - rstat[gh * 2]) * kLog2e) * __ldcg(prm.ws_l + e) *
                      rstat[gh * 2 + 1];
            }
          }
          named_barrier_sync(1, NCT);
#pragma unroll
          for (int o = 0; o < OUTS; ++o) {
            const int idx = ctid + o * NCT;
            if (idx >= GT * D) break;
            const int gh = idx / D, d = idx - gh * D;
            if (gh >= I.nh) continue;
            const float* src = prm.ws_o + (((size_t)I.s * H + I.h0 + gh) * Pmax + c0) * D + d;
            float a = racc[o];
#pragma unroll 4
            for (int pp = 0; pp < cn; ++pp) a = fmaf(rw[gh * RCH + pp], __ldcg(src + (size_t)pp * D), a);
            racc[o] = a;
          }
        }
#pragma unroll
        for (int o = 0; o < OUTS; ++o) {
          const int idx = ctid + o * NCT;
          if (idx >= GT * D) break;
          const int gh = idx / D, d = idx - gh * D;
          if (gh >= I.nh) continue;
          out[((size_t)I.s * H + I.h0 + gh) * D + d] = F16Traits<T>::from_float(racc[o]);
        }
      }
    }
    named_barrier_sync(1, NCT);
  }
}

template <class C, int NC, int NSTAGE>
__global__ void __launch_bounds__(Layout<C, NC, NSTAGE>::THREADS, 1)
    pa_decode_kernel(const __grid_constant__ KParams prm) {
  using LY = Layout<C, NC, NSTAGE>;
  constexpr int NS = NSTAGE, UQ = LY::UQ;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::OFF_FLAGS);
  int* last_flag = reinterpret_cast<int*>(smem + LY::OFF_FLAGS + 4);
  int* pref = reinterpret_cast<int*>(smem + LY::OFF_PREF);
  int* scan = reinterpret_cast<int*>(smem + LY::OFF_SCAN);
  UnitInfo* info = reinterpret_cast<UnitInfo*>(smem + LY::OFF_INFO);

  if (tid == 0) {
    const uint32_t bar = sbase + LY::OFF_BAR;
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar + 8 * i, 1);            // full: producer arrive + bytes
      mbar_init(bar + 8 * (NS + i), 1);     // empty: one consumer warp
    }
    for (int i = 0; i < UQ; ++i) {
      mbar_init(bar + 8 * (2 * NS + i), 1);        // unit full
      mbar_init(bar + 8 * (2 * NS + UQ + i), NC);  // unit empty: every consumer warp
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  // pref[s] = number of used partitions before sequence s (lengths clamped to
  // [0, MB*BS]; an out-of-range length is recorded as a device error).
  {
    const int S = prm.S, nthr = LY::THREADS, max_len = prm.MB * C::BS;
    const int per = (S + nthr - 1) / nthr;
    const int beg = min(tid * per, S), end = min(beg + per, S);
    int sum = 0;
    for (int s = beg; s < end; ++s) {
      int L = prm.lens[s];
      if (L < 0 || L > max_len) {
        atomicCAS(prm.hdr + kHdrError, 0, kErrDeviceBounds);
        L = min(max(L, 0), max_len);
      }
      sum += (L + prm.P - 1) / prm.P;
    }
    scan[tid] = sum;
    __syncthreads();
    if (tid == 0) {
      int run = 0;
      for (int i = 0; i < nthr; ++i) {
        const int v = scan[i];
        scan[i] = run;
        run += v;
      }
      pref[S] = run;
    }
    __syncthreads();
    int run = scan[tid];
    for (int s = beg; s < end; ++s) {
      pref[s] = run;
      run += (min(max(prm.lens[s], 0), max_len) + prm.P - 1) / prm.P;
    }
  }
  __syncthreads();
  if (warp == NC) {
    producer_loop<C, LY>(prm, smem, pref, info, abort_flag, lane);
  } else {
    consumer_loop<C, LY>(prm, smem, pref, info, abort_flag, last_flag, warp, lane);
  }
}

}  // namespace pa
