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
//     the page's layouts -- into shared memory with 1-D bulk async copies
//     completing on mbarriers;
//   * warps 0..NC-1 (consumers): block j of a unit goes to warp j % NC (a
//     fixed grouping, so results do not depend on scheduling), which folds it
//     into its private online-softmax state (SimtConsumer or MmaConsumer).
//     The CTA's g-th block (counted over all its units) lives in ring stage
//     g % NSTAGE.  Warps run at different speeds, so a fast warp
//     could reach stage g % NSTAGE while the stage's previous copy (block
//     g - NSTAGE) is still in flight, and an mbarrier parity wait cannot tell
//     those two phases apart.  A consumer therefore first waits until the
//     producer has issued block g (a shared-memory counter): the producer
//     issues block g only after block g - NSTAGE was consumed, so by then the
//     stage's previous phase is complete and the parity wait is exact.
//     At the end of a unit the warps' states are combined in shared memory
//     into the partition's (m_p, l_p, o_p).
// Sequences with one partition write the output directly (single pass).  For
// longer sequences each unit stores its partition state in the workspace and
// takes a ticket (checked one unit later, off the critical path); the last
// writer runs the phase-2 combine of `_paged_attn_v2_reduce_kernel`
// (M = max m_p, w_p = e^(m_p - M) l_p / sum, out = sum w_p o_p).  Up to
// kChunk = 16 partitions are combined in one step; longer sequences are
// combined per chunk of 16 partitions by each chunk's last writer, and the
// chunk states by the last chunk (the combine is associative), so no CTA
// walks hundreds of partitions alone.
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
  float* ws_cm;  // [S, H, Cmax]     combined state of each chunk of kChunk partitions
  float* ws_cl;  // [S, H, Cmax]
  float* ws_co;  // [S, H, Cmax, D]
  int* hdr;      // kHdrInts ints
  int* tickets;  // [S, n_hg]        partitions (or chunks) of a sequence completed
  int* ctickets; // [S, n_hg, Cmax]  partitions of a chunk completed
  float scale_log2;
  int S, H, KH, G, MB, num_blocks, P, Pmax, Cmax;
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
  static constexpr int THREADS = NCT + 64;     // + producer warp + epilogue warp
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
  static constexpr uint32_t OFF_EF = al16(OFF_RSTAT + C::GT * 2 * 4);   // NC*GT warp weights + GT sums
  static constexpr uint32_t OFF_SCAN = al16(OFF_EF + (NC + 1) * C::GT * 4);
  static constexpr uint32_t OFF_INFO = al16(OFF_SCAN + THREADS * 4);
  static constexpr uint32_t OFF_EPI_INFO = al16(OFF_INFO + UQ * sizeof(UnitInfo));
  static constexpr uint32_t OFF_BAR = al16(OFF_EPI_INFO + sizeof(UnitInfo));
  static constexpr uint32_t NBAR = 2 * NSTAGE + 2 * UQ + 2;
  static constexpr uint32_t OFF_FLAGS = al16(OFF_BAR + NBAR * 8);
  static constexpr uint32_t OFF_PREF = al16(OFF_FLAGS + 64);
  static constexpr uint32_t FIXED = OFF_PREF;
  static constexpr uint32_t bytes(int S) { return al16(OFF_PREF + (uint32_t)(S + 1) * 4); }
  static constexpr int OUTS = (C::GT * C::D + NCT - 1) / NCT;  // combine outputs per thread
};

template <class LY>
__device__ __forceinline__ uint32_t stage_of(uint32_t g) {
  return g % LY::NSTAGE;
}
template <class LY>
__device__ __forceinline__ uint32_t phase_of(uint32_t g) {
  return (g / LY::NSTAGE) & 1u;
}

// Wait (bounded) until the producer has issued at least `target` blocks.
__device__ __forceinline__ bool wait_issued(const volatile uint32_t* issued, uint32_t target,
                                            volatile int* abort_flag, int* err_word,
                                            long long timeout_ns) {
  if (*issued >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (*issued >= target) return true;
    if (*abort_flag) return false;
    if ((long long)(global_timer_ns() - t0) > timeout_ns) {
      *abort_flag = 1;
      atomicCAS(err_word, 0, kErrTimeout);
      return false;
    }
  }
}

// A work unit as the producer sees it.
struct UnitPlan {
  int s, p, hg, t0, t1, nb, np, nh, h0, kv;
};

template <class C>
__device__ __forceinline__ UnitPlan plan_unit(const KParams& prm, const int* pref, int u) {
  constexpr int BS = C::BS, GT = C::GT;
  UnitPlan U;
  const int pair = u / prm.n_hg;
  U.hg = u - pair * prm.n_hg;
  int lo = 0, hi = prm.S;  // pref[lo] <= pair < pref[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= pair) lo = mid; else hi = mid;
  }
  U.s = lo;
  U.p = pair - pref[lo];
  U.np = pref[lo + 1] - pref[lo];
  const int L = min(max(prm.lens[lo], 0), prm.MB * BS);
  U.t0 = U.p * prm.P;
  U.t1 = min(U.t0 + prm.P, L);
  U.nb = (U.t1 - U.t0 + BS - 1) / BS;
  U.kv = U.hg / prm.hg_per_kv;
  const int hgk = U.hg - U.kv * prm.hg_per_kv;
  U.h0 = U.kv * prm.G + hgk * GT;
  U.nh = min(GT, prm.G - hgk * GT);
  return U;
}

// This lane's block-table entry among blocks [c0, c0 + 32) of unit U (0 past
// the unit's end).  An id outside the pool is recorded and replaced by 0, so
// nothing is read out of bounds.
template <class C>
__device__ __forceinline__ int load_block_id(const KParams& prm, const UnitPlan& U, int c0, int lane) {
  int b = 0;
  if (c0 + lane < U.nb) {
    b = __ldg(prm.bt + (size_t)U.s * prm.MB + U.t0 / C::BS + c0 + lane);
    if ((unsigned)b >= (unsigned)prm.num_blocks) {
      atomicCAS(prm.hdr + kHdrError, 0, kErrDeviceBounds);
      b = 0;
    }
  }
  return b;
}

template <class C, class LY>
__device__ __forceinline__ void producer_loop(const KParams& prm, uint8_t* smem, const int* pref,
                                              UnitInfo* info, volatile int* abort_flag,
                                              volatile uint32_t* issued, int lane) {
  using T = typename C::T;
  constexpr int D = C::D, NS = LY::NSTAGE, UQ = LY::UQ;
  // Blocks issued together, one per lane, as their stages free up.
  constexpr int BATCH = NS < 8 ? NS : 8;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_full = sbase + LY::OFF_BAR, bar_empty = bar_full + NS * 8;
  const uint32_t bar_ufull = bar_empty + NS * 8, bar_uempty = bar_ufull + UQ * 8;
  int* err = prm.hdr + kHdrError;
  const uint64_t pol_stream = l2_policy_evict_first();
  const uint64_t pol_keep = l2_policy_evict_last();
  const int total = pref[prm.S] * prm.n_hg;

  uint32_t g = 0;   // blocks whose copies are issued, in order
  uint32_t kq = 0;  // units published (the end marker included)
  bool ok = true;

  // Publish unit U (or, if !have, the end marker) into the next queue slot:
  // its description, and a bulk copy of its query rows.
  auto publish = [&](const UnitPlan& Up, bool have) -> bool {
    const int slot = kq % UQ;
    const uint32_t par = (kq / UQ) & 1u;
    bool okp = true;
    if (lane == 0) {
      okp = wait_bounded(bar_uempty + 8 * slot, par ^ 1u, abort_flag, err, prm.timeout_ns);
      if (okp && !have) {
        info[slot].s = -1;
        mbar_arrive(bar_ufull + 8 * slot);
      } else if (okp) {
        UnitInfo& I = info[slot];
        I.s = Up.s; I.p = Up.p; I.hg = Up.hg; I.t0 = Up.t0; I.t1 = Up.t1; I.nb = Up.nb;
        I.np = Up.np; I.nh = Up.nh; I.h0 = Up.h0;
        const uint32_t qbytes = (uint32_t)(Up.nh * D * 2);
        mbar_arrive_expect_tx(bar_ufull + 8 * slot, qbytes);
        bulk_copy_g2s(sbase + LY::OFF_Q + slot * LY::QSLOT,
                      static_cast<const T*>(prm.q) + ((size_t)Up.s * prm.H + Up.h0) * D, qbytes,
                      bar_ufull + 8 * slot, pol_keep);
      }
    }
    okp = __shfl_sync(0xffffffffu, (int)okp, 0) != 0;
    if (okp) ++kq;
    return okp;
  };

  // The work counter is read two units ahead: while unit k streams, unit k+1
  // is already planned and published and the index of unit k+2 is in flight,
  // so neither the atomic nor the block-table loads stall the stream.
  int u_cur = 0, u_req = 0;
  if (lane == 0) {
    u_cur = atomicAdd(prm.hdr + kHdrWork, 1);
    u_req = atomicAdd(prm.hdr + kHdrWork, 1);
  }
  u_cur = __shfl_sync(0xffffffffu, u_cur, 0);
  bool have = u_cur < total;
  UnitPlan U{};
  int bids = 0;  // this lane's block id among the unit's first 32 blocks
  if (have) {
    U = plan_unit<C>(prm, pref, u_cur);
    bids = load_block_id<C>(prm, U, 0, lane);
  }
  ok = publish(U, have);
  while (have && ok) {
    const int u_nx = __shfl_sync(0xffffffffu, u_req, 0);
    const bool have_next = u_nx < total;
    UnitPlan Un{};
    int bids_next = 0;
    if (have_next) {
      Un = plan_unit<C>(prm, pref, u_nx);
      bids_next = load_block_id<C>(prm, Un, 0, lane);
      if (lane == 0) u_req = atomicAdd(prm.hdr + kHdrWork, 1);
    }
    ok = publish(Un, have_next);
    if (!ok) break;
    for (int c0 = 0; c0 < U.nb && ok; c0 += 32) {
      const int b32 = (c0 == 0) ? bids : load_block_id<C>(prm, U, c0, lane);
      const int cend = min(c0 + 32, U.nb);
      for (int jb = c0; jb < cend && ok; jb += BATCH) {
        const int cnt = min(BATCH, cend - jb);
        const int bi = __shfl_sync(0xffffffffu, b32, (jb - c0) + (lane < cnt ? lane : 0));
        // Lanes < cnt issue block g + lane once its stage is free; the
        // shared `issued` counter follows the prefix of issued blocks.
        const uint32_t gi = g + lane, st = stage_of<LY>(gi), ph = phase_of<LY>(gi);
        bool done = lane >= cnt;
        bool timing = false;
        uint64_t t_start = 0;
        while (true) {
          if (!done && mbar_test_wait(bar_empty + 8 * st, ph ^ 1u)) {
            const uint32_t dst = sbase + st * LY::STAGE;
            const size_t off = ((size_t)bi * prm.KH + U.kv) * (size_t)(D * C::BS);
            mbar_arrive_expect_tx(bar_full + 8 * st, LY::STAGE);
            bulk_copy_g2s(dst, static_cast<const T*>(prm.kc) + off, LY::KBYTES, bar_full + 8 * st, pol_stream);
            bulk_copy_g2s(dst + LY::KBYTES, static_cast<const T*>(prm.vc) + off, LY::KBYTES,
                          bar_full + 8 * st, pol_stream);
            done = true;
          }
          const unsigned m = __ballot_sync(0xffffffffu, done);
          const int prefix = (m == 0xffffffffu) ? 32 : (__ffs(~m) - 1);
          if (lane == 0) *issued = g + (uint32_t)min(prefix, cnt);
          if (m == 0xffffffffu) break;
          int stop = 0;
          if (lane == 0) {
            if (*abort_flag) {
              stop = 1;
            } else {
              const uint64_t now = global_timer_ns();
              if (!timing) {
                timing = true;
                t_start = now;
              } else if ((long long)(now - t_start) > prm.timeout_ns) {
                *abort_flag = 1;
                atomicCAS(err, 0, kErrTimeout);
                stop = 1;
              } else {
                __nanosleep(32);
              }
            }
          }
          if (__shfl_sync(0xffffffffu, stop, 0)) {
            // Aborted: let this batch's issued copies land before leaving.
            ok = false;
            if (done && lane < cnt) {
              const uint64_t t0 = global_timer_ns();
              while (!mbar_try_wait(bar_full + 8 * st, ph) && (long long)(global_timer_ns() - t0) < 100000000LL) {
              }
            }
            __syncwarp();
            break;
          }
        }
        if (!ok) break;
        g += cnt;
      }
    }
    U = Un;
    bids = bids_next;
    have = have_next;
  }
  if (!ok && lane == 0) {
    // Aborted: let copies that may still be in flight (the last NSTAGE
    // blocks and the last UQ query rows issued) land before the CTA exits.
    // Each wait is bounded (100 ms, independent of the caller's timeout,
    // which may be tiny) and ignores the abort flag.
    const uint32_t hi = g;
    const long long drain_ns = 100000000LL;
    for (uint32_t i = (hi > (uint32_t)NS ? hi - NS : 0u); i < hi; ++i) {
      const uint32_t bar = bar_full + 8 * stage_of<LY>(i), ph = phase_of<LY>(i);
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

// Partitions per combine chunk (kept equal to kChunkParts of the launcher).
constexpr int kChunk = 16;

// A combine job: the partitions of one (sequence, head group) -- all of them
// (kind 0, at most kChunk), or chunk c of them (kind 1), whose combined state
// is then folded with the other chunks' by the last chunk to finish.
struct RedInfo {
  int s, hg, h0, nh, np, kind, c, cnt;
};

// Lane 0's job, for every lane of the warp.
__device__ __forceinline__ RedInfo broadcast_job(const RedInfo& J) {
  RedInfo R;
  R.s = __shfl_sync(0xffffffffu, J.s, 0);
  R.hg = __shfl_sync(0xffffffffu, J.hg, 0);
  R.h0 = __shfl_sync(0xffffffffu, J.h0, 0);
  R.nh = __shfl_sync(0xffffffffu, J.nh, 0);
  R.np = __shfl_sync(0xffffffffu, J.np, 0);
  R.kind = __shfl_sync(0xffffffffu, J.kind, 0);
  R.c = __shfl_sync(0xffffffffu, J.c, 0);
  R.cnt = __shfl_sync(0xffffffffu, J.cnt, 0);
  return R;
}

__device__ __forceinline__ int* ticket_of(const KParams& prm, const RedInfo& R) {
  const size_t sg = (size_t)R.s * prm.n_hg + R.hg;
  return R.kind == 0 ? prm.tickets + sg : prm.ctickets + sg * prm.Cmax + R.c;
}

// Log-sum-exp combine of `count` states (m, l, o) of the heads of R, by one
// warp: per head M = max m_i and total = sum e^(m_i - M) l_i, then
// o = sum_i (e^(m_i - M) l_i / total) o_i with the weights staged in shared
// memory in chunks of RCH (the page's Phase 2 formula).  State i of head h is
// m[(s*H + h)*stride + first + i] and o[((s*H + h)*stride + first + i)*D + ..].
// TO_OUT writes o, rounded, to the output; otherwise (M, total, o) becomes
// chunk state `dst_c`.
template <class C, class LY, bool TO_OUT>
__device__ __forceinline__ void combine_states(const KParams& prm, const RedInfo& R, const float* sm,
                                               const float* sl, const float* so, int stride, int first,
                                               int count, int dst_c, float* rw, float* rstat, int lane) {
  using T = typename C::T;
  constexpr int D = C::D, GT = C::GT, RCH = LY::RCH;
  constexpr int D4 = D / 4, OUT4 = (GT * D4 + 31) / 32;
  const int H = prm.H;
  for (int gh = 0; gh < R.nh; ++gh) {
    const size_t base = ((size_t)R.s * H + R.h0 + gh) * stride + first;
    float M = -INFINITY;
    for (int i = lane; i < count; i += 32) M = fmaxf(M, __ldcg(sm + base + i));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float tot = 0.f;
    for (int i = lane; i < count; i += 32)
      tot = fmaf(exp2f((__ldcg(sm + base + i) - M) * kLog2e), __ldcg(sl + base + i), tot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    if (lane == 0) {
      rstat[gh * 2] = M;
      rstat[gh * 2 + 1] = tot;
    }
  }
  float4 acc[OUT4];
#pragma unroll
  for (int o = 0; o < OUT4; ++o) acc[o] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < count; c0 += RCH) {
    const int cn = min(RCH, count - c0);
    __syncwarp();
    for (int i = lane; i < R.nh * RCH; i += 32) {
      const int gh = i / RCH, pp = i - gh * RCH;
      if (pp < cn) {
        const size_t e = ((size_t)R.s * H + R.h0 + gh) * stride + first + c0 + pp;
        rw[i] = exp2f((__ldcg(sm + e) - rstat[gh * 2]) * kLog2e) * __ldcg(sl + e) / rstat[gh * 2 + 1];
      }
    }
    __syncwarp();
#pragma unroll
    for (int o = 0; o < OUT4; ++o) {
      const int idx = lane + o * 32;
      if (idx >= GT * D4) break;
      const int gh = idx / D4, d4 = idx - gh * D4;
      if (gh >= R.nh) continue;
      const float4* src = reinterpret_cast<const float4*>(
                              so + (((size_t)R.s * H + R.h0 + gh) * stride + first + c0) * D) + d4;
      float4 a = acc[o], b = make_float4(0.f, 0.f, 0.f, 0.f);
      int pp = 0;
#pragma unroll 4
      for (; pp + 1 < cn; pp += 2) {
        const float w0 = rw[gh * RCH + pp], w1 = rw[gh * RCH + pp + 1];
        const float4 v0 = __ldcg(src + (size_t)pp * D4), v1 = __ldcg(src + (size_t)(pp + 1) * D4);
        a.x = fmaf(w0, v0.x, a.x); a.y = fmaf(w0, v0.y, a.y); a.z = fmaf(w0, v0.z, a.z); a.w = fmaf(w0, v0.w, a.w);
        b.x = fmaf(w1, v1.x, b.x); b.y = fmaf(w1, v1.y, b.y); b.z = fmaf(w1, v1.z, b.z); b.w = fmaf(w1, v1.w, b.w);
      }
      if (pp < cn) {
        const float w0 = rw[gh * RCH + pp];
        const float4 v0 = __ldcg(src + (size_t)pp * D4);
        a.x = fmaf(w0, v0.x, a.x); a.y = fmaf(w0, v0.y, a.y); a.z = fmaf(w0, v0.z, a.z); a.w = fmaf(w0, v0.w, a.w);
      }
      acc[o] = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
    }
  }
#pragma unroll
  for (int o = 0; o < OUT4; ++o) {
    const int idx = lane + o * 32;
    if (idx >= GT * D4) break;
    const int gh = idx / D4, d4 = idx - gh * D4;
    if (gh >= R.nh) continue;
    const size_t sh = (size_t)R.s * H + R.h0 + gh;
    if constexpr (TO_OUT) {
      uint2 v;
      v.x = F16Traits<T>::pack(acc[o].x, acc[o].y);
      v.y = F16Traits<T>::pack(acc[o].z, acc[o].w);
      *reinterpret_cast<uint2*>(static_cast<T*>(prm.out) + sh * D + d4 * 4) = v;
    } else {
      reinterpret_cast<float4*>(prm.ws_co + (sh * prm.Cmax + dst_c) * D)[d4] = acc[o];
      if (d4 == 0) {
        prm.ws_cm[sh * prm.Cmax + dst_c] = rstat[gh * 2];
        prm.ws_cl[sh * prm.Cmax + dst_c] = rstat[gh * 2 + 1];
      }
    }
  }
  __syncwarp();
}

// Run the combine job R (one warp).  A chunk job writes the chunk's state,
// then takes the sequence-level ticket; the last chunk folds all chunk states
// into the output.
template <class C, class LY>
__device__ __forceinline__ void run_combine(const KParams& prm, const RedInfo& R, float* rw, float* rstat,
                                            int lane) {
  if (R.kind == 0) {
    combine_states<C, LY, true>(prm, R, prm.ws_m, prm.ws_l, prm.ws_o, prm.Pmax, 0, R.np, 0, rw, rstat, lane);
    return;
  }
  combine_states<C, LY, false>(prm, R, prm.ws_m, prm.ws_l, prm.ws_o, prm.Pmax, R.c * kChunk, R.cnt, R.c,
                               rw, rstat, lane);
  const int nchunks = (R.np + kChunk - 1) / kChunk;
  int last = 0;
  if (lane == 0) {
    // The warp's chunk-state stores (ordered before lane 0 by the __syncwarp
    // that ends combine_states) are released with the ticket.
    int* tk = prm.tickets + (size_t)R.s * prm.n_hg + R.hg;
    const int t = atomic_add_release_gpu(tk, 1);
    last = (t == nchunks - 1);
    if (last) {
      *tk = 0;
      fence_acq_rel_gpu();
    }
  }
  if (__shfl_sync(0xffffffffu, last, 0))
    combine_states<C, LY, true>(prm, R, prm.ws_cm, prm.ws_cl, prm.ws_co, prm.Cmax, 0, nchunks, 0, rw,
                                rstat, lane);
}

// Consumer warp: stream the blocks of every unit assigned to it and hand its
// online-softmax state for each unit to the epilogue warp through shared
// memory.  Consumer warps never wait for each other.
template <class C, class LY>
__device__ __forceinline__ void consumer_loop(const KParams& prm, uint8_t* smem, const int* pref,
                                              const UnitInfo* info, volatile int* abort_flag,
                                              const volatile uint32_t* issued, int warp, int lane) {
  using T = typename C::T;
  constexpr int D = C::D, BS = C::BS, GT = C::GT, NC = LY::NC, NCT = LY::NCT, NS = LY::NSTAGE,
                UQ = LY::UQ;
  const int ctid = warp * 32 + lane;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_full = sbase + LY::OFF_BAR, bar_empty = bar_full + NS * 8;
  const uint32_t bar_ufull = bar_empty + NS * 8, bar_uempty = bar_ufull + UQ * 8;
  const uint32_t bar_efull = bar_uempty + UQ * 8, bar_eempty = bar_efull + 8;
  float* epi_acc = reinterpret_cast<float*>(smem + LY::OFF_EPI_ACC);
  float* epi_ml = reinterpret_cast<float*>(smem + LY::OFF_EPI_ML);
  UnitInfo* epi_info = reinterpret_cast<UnitInfo*>(smem + LY::OFF_EPI_INFO);
  float* scr = reinterpret_cast<float*>(smem + LY::OFF_SCR) + warp * C::SCRATCH_FLOATS;
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
    const bool okw = __all_sync(0xffffffffu, wait_bounded(bar_ufull + 8 * slot, par, abort_flag, err,
                                                          prm.timeout_ns));
    const UnitInfo I = info[slot];
    if (!okw) break;
    if (I.s < 0) {
      // End of work: pass the end marker on to the epilogue warp, once it has
      // taken the previous hand-over (the k-th hand-over waits for the
      // (k-1)-th to be consumed).
      if (!__all_sync(0xffffffffu, wait_bounded(bar_eempty, (k & 1u) ^ 1u, abort_flag, err,
                                                prm.timeout_ns)))
        break;
      if (warp == 0 && lane == 0) epi_info->s = -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_efull);
      break;
    }
    cons.begin_unit(reinterpret_cast<const T*>(smem + LY::OFF_Q + slot * LY::QSLOT), I.nh,
                    prm.scale_log2, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_uempty + 8 * slot);

    for (int j = warp; j < I.nb; j += NC) {
      const uint32_t gj = g + j, st = stage_of<LY>(gj), ph = phase_of<LY>(gj);
      bool okb = wait_issued(issued, gj + 1, abort_flag, err, prm.timeout_ns) &&
                 wait_bounded(bar_full + 8 * st, ph, abort_flag, err, prm.timeout_ns);
      okb = __all_sync(0xffffffffu, okb);
      const int ntok = min(BS, I.t1 - I.t0 - j * BS);
      if (okb) cons.block(smem + st * LY::STAGE, smem + st * LY::STAGE + LY::KBYTES, ntok, lane, scr);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }
    g += I.nb;

    // Hand this warp's state for unit k to the epilogue warp, once it has
    // taken unit k-1's.
    if (!__all_sync(0xffffffffu, wait_bounded(bar_eempty, (k & 1u) ^ 1u, abort_flag, err,
                                              prm.timeout_ns)))
      break;
    ++k;
    cons.finish(epi_acc + warp * GT * D, epi_ml + warp * GT * 2, lane);
    if (warp == 0 && lane == 0) *epi_info = I;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_efull);
  }
}

// Epilogue warp: for every unit, merge the consumer warps' states into the
// partition's (m_p, l_p, o_p) (or the output, for a single-partition
// sequence), take the completion ticket (checked one unit later, off the
// critical path) and run the combine jobs that fall to this CTA.
template <class C, class LY>
__device__ __forceinline__ void epilogue_loop(const KParams& prm, uint8_t* smem, volatile int* abort_flag,
                                              int lane) {
  using T = typename C::T;
  constexpr int D = C::D, GT = C::GT, NC = LY::NC, NS = LY::NSTAGE, UQ = LY::UQ;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_efull = sbase + LY::OFF_BAR + (2 * NS + 2 * UQ) * 8, bar_eempty = bar_efull + 8;
  const float* epi_acc = reinterpret_cast<const float*>(smem + LY::OFF_EPI_ACC);
  const float* epi_ml = reinterpret_cast<const float*>(smem + LY::OFF_EPI_ML);
  const UnitInfo* epi_info = reinterpret_cast<const UnitInfo*>(smem + LY::OFF_EPI_INFO);
  float* rw = reinterpret_cast<float*>(smem + LY::OFF_RED);
  float* rstat = reinterpret_cast<float*>(smem + LY::OFF_RSTAT);
  float* ef = reinterpret_cast<float*>(smem + LY::OFF_EF);  // [NC][GT] weights, then [GT] sums
  int* err = prm.hdr + kHdrError;
  const int H = prm.H, Pmax = prm.Pmax;
  T* out = static_cast<T*>(prm.out);

  // Lane 0 only: a ticket taken and not yet checked, and its job.
  bool pend = false;
  int pend_t = 0;
  RedInfo pinfo{};
  for (uint32_t k = 0;; ++k) {
    const bool ok = __all_sync(0xffffffffu, wait_bounded(bar_efull, k & 1u, abort_flag, err,
                                                         prm.timeout_ns));
    if (!ok) return;  // aborted: the results are abandoned
    const UnitInfo I = *epi_info;
    if (I.s < 0) {
      // End of work: settle the last ticket.
      int last = 0;
      if (lane == 0 && pend && pend_t == pinfo.cnt - 1) {
        last = 1;
        *ticket_of(prm, pinfo) = 0;
        fence_acq_rel_gpu();
      }
      const RedInfo R = broadcast_job(pinfo);  // pinfo is kept by lane 0 only
      if (__shfl_sync(0xffffffffu, last, 0)) run_combine<C, LY>(prm, R, rw, rstat, lane);
      return;
    }
    // Per head: M = max over warps, each warp's weight 2^(m_w - M), and the sum l.
    for (int i = lane; i < GT; i += 32) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w) M = fmaxf(M, epi_ml[(w * GT + i) * 2]);
      float den = 0.f;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float f = exp2f(epi_ml[(w * GT + i) * 2] - M);
        ef[w * GT + i] = f;
        den = fmaf(f, epi_ml[(w * GT + i) * 2 + 1], den);
      }
      ef[NC * GT + i] = den;
      rstat[i * 2] = M;
    }
    __syncwarp();
    const bool single = (I.np == 1);
    for (int idx = lane; idx < I.nh * D; idx += 32) {
      const int gh = idx / D, d = idx - gh * D;
      float num = 0.f;
#pragma unroll
      for (int w = 0; w < NC; ++w) num = fmaf(ef[w * GT + gh], epi_acc[(w * GT + gh) * D + d], num);
      const float val = num / ef[NC * GT + gh];
      const size_t sh = (size_t)I.s * H + I.h0 + gh;
      if (single) out[sh * D + d] = F16Traits<T>::from_float(val);
      else prm.ws_o[(sh * Pmax + I.p) * D + d] = val;
      if (d == 0) {
        prm.ws_m[sh * Pmax + I.p] = rstat[gh * 2] * kLn2;
        prm.ws_l[sh * Pmax + I.p] = ef[NC * GT + gh];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_eempty);  // the hand-over slot may be refilled

    // Settle the previous ticket; take this unit's (release: the warp's
    // partition stores above, ordered by __syncwarp, become visible first).
    int go = 0;
    RedInfo job = pinfo;
    if (lane == 0) {
      if (pend && pend_t == pinfo.cnt - 1) {
        go = 1;
        *ticket_of(prm, pinfo) = 0;
        fence_acq_rel_gpu();
      }
      pend = !single;
      if (pend) {
        pinfo.s = I.s; pinfo.hg = I.hg; pinfo.h0 = I.h0; pinfo.nh = I.nh; pinfo.np = I.np;
        if (I.np <= kChunk) {
          pinfo.kind = 0; pinfo.c = 0; pinfo.cnt = I.np;
        } else {
          pinfo.kind = 1; pinfo.c = I.p / kChunk; pinfo.cnt = min(kChunk, I.np - pinfo.c * kChunk);
        }
        pend_t = atomic_add_release_gpu(ticket_of(prm, pinfo), 1);
      }
    }
    const RedInfo R = broadcast_job(job);  // pinfo is kept by lane 0 only
    if (__shfl_sync(0xffffffffu, go, 0)) run_combine<C, LY>(prm, R, rw, rstat, lane);
  }
}

template <class C, int NC, int NSTAGE, int CTAS_PER_SM>
__global__ void __launch_bounds__(Layout<C, NC, NSTAGE>::THREADS, CTAS_PER_SM)
    pa_decode_kernel(const __grid_constant__ KParams prm) {
  using LY = Layout<C, NC, NSTAGE>;
  constexpr int NS = LY::NSTAGE, UQ = LY::UQ;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::OFF_FLAGS);
  volatile uint32_t* issued = reinterpret_cast<volatile uint32_t*>(smem + LY::OFF_FLAGS + 8);
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
    mbar_init(bar + 8 * (2 * NS + 2 * UQ), NC);     // hand-over full: every consumer warp
    mbar_init(bar + 8 * (2 * NS + 2 * UQ + 1), 1);  // hand-over empty: the epilogue warp
    *abort_flag = 0;
    *issued = 0;
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
    producer_loop<C, LY>(prm, smem, pref, info, abort_flag, issued, lane);
  } else if (warp == NC + 1) {
    epilogue_loop<C, LY>(prm, smem, abort_flag, lane);
  } else {
    consumer_loop<C, LY>(prm, smem, pref, info, abort_flag, issued, warp, lane);
  }
}

}  // namespace pa
