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
//     unit's physical K and V blocks -- each a contiguous D*BS*(element
//     size)-byte run in the page's layouts -- into shared memory with 1-D
//     bulk async copies completing on mbarriers;
//   * warps 0..NC-1 (consumers): block j of unit u goes to warp (j + u) % NC
//     (a fixed grouping, so results do not depend on scheduling), which folds it
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
  float* lse;    // [S, H] log-sum-exp of the scaled scores, or null
  int q_len;     // query tokens per sequence (multi-query kernels; 1 otherwise)
  int Hu, Gu;    // the caller's heads and heads per kv head; H and G below count row
                 // heads, q_len of them per caller head (H = q_len * Hu, G = q_len * Gu)
  float scale_log2;   // softmax scale (times k_scale for an fp8 cache) times log2 e
  float v_scale;      // multiplies every output: 1, or an fp8 cache's v_scale
  int S, H, KH, G, MB, num_blocks, P, Pmax, Cmax;
  int hg_per_kv;  // ceil(G / GT)
  int n_hg;       // KH * hg_per_kv
  long long timeout_ns;
};

// Cached tokens of sequence s, clamped to [0, max_len].  A length outside
// [MQ ? q_len : 0, max_len] is flagged (*bad): a multi-query sequence holds
// its q_len new tokens.
template <bool MQ>
__device__ __forceinline__ int seq_tokens(const KParams& prm, int s, int max_len, bool* bad) {
  const int L = prm.lens[s];
  if (L < (MQ ? prm.q_len : 0) || L > max_len) *bad = true;
  return min(max(L, 0), max_len);
}

// Multi-query decode keeps the single-query work decomposition and gives the
// rows of a unit to (query token, head) pairs: within kv head kv, row head
// h = kv * G + l (l < G = q_len * Gu) is query token i = l / Gu and caller
// head kv * Gu + l % Gu.  Every row head streams the same K/V blocks (one
// load serves q_len * Gu rows); token i sits at position L - q_len + i and
// sees positions 0 .. L - q_len + i.  (Multi-query kernels are separate
// instances: carrying q_len through the single-query kernel cost it 5%.)
template <bool MQ>
__device__ __forceinline__ size_t out_row(const KParams& prm, int s, int h) {
  if constexpr (!MQ) {
    return (size_t)s * prm.H + h;
  } else {
    const int kv = h / prm.G, l = h - kv * prm.G, i = l / prm.Gu;
    return ((size_t)s * prm.q_len + i) * prm.Hu + kv * prm.Gu + (l - i * prm.Gu);
  }
}
// out_row for code shared by both kernel kinds (final writes only).
__device__ __forceinline__ size_t out_row_rt(const KParams& prm, int s, int h) {
  return prm.q_len > 1 ? out_row<true>(prm, s, h) : out_row<false>(prm, s, h);
}
// Positions [0, limit) that row head h of a sequence of L tokens sees.
template <bool MQ>
__device__ __forceinline__ int row_limit(const KParams& prm, int L, int h) {
  if constexpr (!MQ) {
    return L;
  } else {
    return L - prm.q_len + (h % prm.G) / prm.Gu + 1;
  }
}

struct UnitInfo {
  int s, p, hg, t0, t1, nb, np, nh, h0;
  int L;  // the sequence's tokens
  int pad[2];
};

constexpr uint32_t al16(uint32_t x) { return (x + 15u) & ~15u; }

template <class C, int NC_, int NSTAGE_>
struct Layout {
  static constexpr int NC = NC_, NSTAGE = NSTAGE_, UQ = 2;
  static constexpr int NCT = NC * 32;          // consumer threads
  static constexpr int THREADS = NCT + 64;     // + producer warp + epilogue warp
  static constexpr uint32_t KBYTES = C::D * C::BS * C::KV_ESZ;  // one block of one kv head
  // A stage holds the K block, then the V block in C::kVPieces pieces (with
  // C::kVPad bytes of padding between them); its copies deliver STAGE_TX bytes.
  static constexpr uint32_t STAGE = 2 * KBYTES + C::kVPad;
  static constexpr uint32_t STAGE_TX = 2 * KBYTES;
  static_assert(C::kVPieces * C::kVPieceBytes == KBYTES, "value pieces cover the block");
  static constexpr uint32_t RING = NSTAGE * STAGE;
  static constexpr uint32_t QSLOT = C::GT * C::D * (uint32_t)sizeof(typename C::T);
  static constexpr uint32_t OFF_Q = RING;
  static constexpr uint32_t OFF_EPI_ACC = al16(OFF_Q + UQ * QSLOT);
  static constexpr uint32_t OFF_EPI_ML = al16(OFF_EPI_ACC + NC * C::GT * C::D * 4);
  static constexpr uint32_t OFF_SCR = al16(OFF_EPI_ML + NC * C::GT * 2 * 4);
  static constexpr uint32_t OFF_RSTAT = al16(OFF_SCR + NC * C::SCRATCH_FLOATS * 4);
  static constexpr uint32_t OFF_EF = al16(OFF_RSTAT + C::GT * 2 * 4);   // NC*GT warp weights + GT sums
  static constexpr uint32_t OFF_SCAN = al16(OFF_EF + (NC + 1) * C::GT * 4);
  static constexpr uint32_t OFF_INFO = al16(OFF_SCAN + THREADS * 4);
  static constexpr uint32_t OFF_EPI_INFO = al16(OFF_INFO + UQ * sizeof(UnitInfo));
  static constexpr uint32_t OFF_JOBQ = al16(OFF_EPI_INFO + sizeof(UnitInfo));   // 16 queued jobs
  static constexpr uint32_t OFF_JOBREC = al16(OFF_JOBQ + 16 * 32);               // posted-job slots
  static constexpr uint32_t OFF_BAR = al16(OFF_JOBREC + 8 * 32);
  static constexpr uint32_t NBAR = 2 * NSTAGE + 2 * UQ + 2 + 8;
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

// Wait sites recorded by a timeout (workspace header words 2..5).
enum WaitSite {
  kSitePublish = 1,     // producer: a unit-queue slot to free up
  kSiteStage = 2,       // producer: a ring stage to free up
  kSiteUnit = 3,        // consumer: the next unit's description
  kSiteIssued = 4,      // consumer: a block to be issued
  kSiteFull = 5,        // consumer: a block to land
  kSiteHandover = 6,    // consumer: the hand-over slot to free up
  kSiteHandEnd = 7,     // consumer: the hand-over slot, for the end marker
  kSiteServe = 8,       // consumer: the epilogue warp to finish its jobs
  kSiteEpiFull = 9,     // epilogue: the consumers' states of a unit
  kSiteJobDone = 10     // epilogue: the helpers of a shared combine job
};

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
      record_timeout(abort_flag, err_word, kSiteIssued, (int)target);
      return false;
    }
  }
}

// A work unit as the producer sees it.
struct UnitPlan {
  int s, p, hg, t0, t1, nb, np, nh, h0, kv, L;
};

template <class C, bool MQ>
__device__ __forceinline__ UnitPlan plan_unit(const KParams& prm, const int* pref, int u) {
  constexpr int BS = C::BS, GT = C::GT;
  UnitPlan U;
  const int pair = u / prm.n_hg;
  U.hg = u - pair * prm.n_hg;
  int lo = 0, hi = prm.S;  // pref[lo] <= pair < pref[lo + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= pair) lo = mid; else hi = mid;
  }
  bool bad = false;  // flagged by the prefix scan already
  U.s = lo;
  U.p = pair - pref[lo];
  U.np = pref[lo + 1] - pref[lo];
  const int L = seq_tokens<MQ>(prm, lo, prm.MB * BS, &bad);
  U.L = L;
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
template <class C, bool MQ>
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

template <class C, class LY, bool MQ>
__device__ __forceinline__ void producer_loop(const KParams& prm, uint8_t* smem, const int* pref,
                                              UnitInfo* info, volatile int* abort_flag,
                                              volatile uint32_t* issued, int lane) {
  using T = typename C::T;
  constexpr int D = C::D, NS = LY::NSTAGE, UQ = LY::UQ;
  // Blocks issued together, one per lane, as their stages free up.
  static_assert(C::kIssueBatch >= 1 && C::kIssueBatch <= 32, "one block per lane");
  constexpr int BATCH = NS < C::kIssueBatch ? NS : C::kIssueBatch;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_full = sbase + LY::OFF_BAR, bar_empty = bar_full + NS * 8;
  const uint32_t bar_ufull = bar_empty + NS * 8, bar_uempty = bar_ufull + UQ * 8;
  int* err = prm.hdr + kHdrError;
  const uint64_t pol_stream = l2_policy_evict_first();
  const uint64_t pol_keep = l2_policy_evict_last();
  const int total = pref[prm.S] * prm.n_hg;
  auto plan_next = [&](int u, UnitPlan& Up) -> bool {
    if (u >= total) return false;
    Up = plan_unit<C, MQ>(prm, pref, u);
    return true;
  };

  uint32_t g = 0;   // blocks whose copies are issued, in order
  uint32_t kq = 0;  // units published (the end marker included)
  uint32_t reissued = 0;  // after an abort inside a batch: lanes whose block g + lane was issued
  bool ok = true;

  // Publish unit U (or, if !have, the end marker) into the next queue slot:
  // its description, and a bulk copy of its query rows.
  auto publish = [&](const UnitPlan& Up, bool have) -> bool {
    const int slot = kq % UQ;
    const uint32_t par = (kq / UQ) & 1u;
    bool okp = true;
    if (lane == 0) {
      okp = wait_bounded(bar_uempty + 8 * slot, par ^ 1u, abort_flag, err, prm.timeout_ns, kSitePublish,
                         (int)kq);
      if (okp && !have) {
        info[slot].s = -1;
        mbar_arrive(bar_ufull + 8 * slot);
      } else if (okp) {
        UnitInfo& I = info[slot];
        I.s = Up.s; I.p = Up.p; I.hg = Up.hg; I.t0 = Up.t0; I.t1 = Up.t1; I.nb = Up.nb;
        I.np = Up.np; I.nh = Up.nh; I.h0 = Up.h0; I.L = Up.L;
        const uint32_t qbytes = (uint32_t)(Up.nh * D * sizeof(T));
        mbar_arrive_expect_tx(bar_ufull + 8 * slot, qbytes);
        if constexpr (!MQ)
          bulk_copy_g2s(sbase + LY::OFF_Q + slot * LY::QSLOT,
                        static_cast<const T*>(prm.q) + ((size_t)Up.s * prm.H + Up.h0) * D, qbytes,
                        bar_ufull + 8 * slot, pol_keep);
      }
    }
    okp = __shfl_sync(0xffffffffu, (int)okp, 0) != 0;
    if constexpr (MQ) {
      // The row heads of a multi-query unit are scattered over the caller's
      // [S, q_len, H] rows: one row copy per lane.
      if (okp && have && lane < Up.nh)
        bulk_copy_g2s(sbase + LY::OFF_Q + slot * LY::QSLOT + lane * D * (uint32_t)sizeof(T),
                      static_cast<const T*>(prm.q) + out_row<true>(prm, Up.s, Up.h0 + lane) * D,
                      (uint32_t)(D * sizeof(T)), bar_ufull + 8 * slot, pol_keep);
    }
    if (okp) ++kq;
    return okp;
  };

  // The work counter is read one unit ahead: the next unit is claimed when
  // unit k starts streaming, and planned and published once k's first batch
  // of copies is issued (the atomic has returned by then).  A CTA thus holds
  // at most the unit it streams and the next one, which keeps the end of the
  // work even across CTAs.
  int u_cur = 0;
  if (lane == 0) u_cur = atomicAdd(prm.hdr + kHdrWork, 1);
  u_cur = __shfl_sync(0xffffffffu, u_cur, 0);
  UnitPlan U{};
  bool have = plan_next(u_cur, U);
  int bids = 0;  // this lane's block id among the unit's first 32 blocks
  if (have) bids = load_block_id<C, MQ>(prm, U, 0, lane);
  ok = publish(U, have);
  while (have && ok) {
    int u_req = 0;
    if (lane == 0) u_req = atomicAdd(prm.hdr + kHdrWork, 1);
    bool have_next = false, published_next = false;
    UnitPlan Un{};
    int bids_next = 0;
    auto publish_next = [&]() {
      const int u_nx = __shfl_sync(0xffffffffu, u_req, 0);
      have_next = plan_next(u_nx, Un);
      if (have_next) bids_next = load_block_id<C, MQ>(prm, Un, 0, lane);
      ok = publish(Un, have_next);
      published_next = true;
    };
    for (int c0 = 0; c0 < U.nb && ok; c0 += 32) {
      const int b32 = (c0 == 0) ? bids : load_block_id<C, MQ>(prm, U, c0, lane);
      const int cend = min(c0 + 32, U.nb);
      for (int jb = c0; jb < cend && ok; jb += BATCH) {
        if (jb > 0 && !published_next) {
          publish_next();
          if (!ok) break;
        }
        if (__shfl_sync(0xffffffffu, lane == 0 ? *abort_flag : 0, 0)) {
          ok = false;
          break;
        }
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
            mbar_arrive_expect_tx(bar_full + 8 * st, LY::STAGE_TX);
            bulk_copy_g2s(dst, static_cast<const uint8_t*>(prm.kc) + off * C::KV_ESZ, LY::KBYTES,
                          bar_full + 8 * st, pol_stream);
            const uint8_t* vsrc = static_cast<const uint8_t*>(prm.vc) + off * C::KV_ESZ;
#pragma unroll
            for (int pc = 0; pc < C::kVPieces; ++pc)
              bulk_copy_g2s(dst + LY::KBYTES + pc * (C::kVPieceBytes + 16u), vsrc + pc * C::kVPieceBytes,
                            C::kVPieceBytes, bar_full + 8 * st, pol_stream);
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
                record_timeout(abort_flag, err, kSiteStage, (int)g);
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
            reissued = __ballot_sync(0xffffffffu, done && lane < cnt);
            break;
          }
        }
        if (!ok) break;
        g += cnt;
      }
    }
    if (ok && !published_next) publish_next();
    U = Un;
    bids = bids_next;
    have = have_next;
  }
  if (lane == 0) {
    // Let copies that may still be in flight (the last NSTAGE blocks and the
    // last UQ query rows issued) land before this warp exits, so that the CTA
    // never ends with a copy outstanding, whatever the consumer warps did.
    // (Without an abort they have landed already.)  Each wait is bounded
    // (100 ms, independent of the caller's timeout, which may be tiny) and
    // ignores the abort flag.
    const uint32_t hi = g;
    const long long drain_ns = 100000000LL;
    for (uint32_t i = (hi > (uint32_t)NS ? hi - NS : 0u); i < hi; ++i) {
      // A stage taken over by block i + NS of an aborted batch was waited for there.
      const uint32_t lane_of_i = i + NS - hi;
      if (lane_of_i < 32u && ((reissued >> lane_of_i) & 1u)) continue;
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

// A combine job for one (sequence, head group):
//   kind 0: all np (<= kChunk) partition states -> output;
//   kind 1: the cnt partition states of chunk c -> chunk state c;
//   kind 2: the ceil(np / kChunk) chunk states -> output.
struct Job {
  int s, hg, h0, nh, np, kind, c, cnt;
};
static_assert(sizeof(Job) <= 48, "combine job must fit in the shared flag area");

// Jobs that read more float4 values than this (or have more output columns
// than the epilogue warp has lanes) are shared with the consumer warps;
// smaller ones are done by the epilogue warp alone.
#ifndef PA_SHARE_JOB_LOADS
#define PA_SHARE_JOB_LOADS 512
#endif
constexpr int kShareJobLoads = PA_SHARE_JOB_LOADS;

// Lane 0's job, for every lane of the warp.
__device__ __forceinline__ Job broadcast_job(const Job& J) {
  Job R;
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

__device__ __forceinline__ int* ticket_of(const KParams& prm, const Job& J) {
  const size_t sg = (size_t)J.s * prm.n_hg + J.hg;
  return J.kind == 0 ? prm.tickets + sg : prm.ctickets + sg * prm.Cmax + J.c;
}

__device__ __forceinline__ int job_count(const Job& J) {
  return J.kind == 0 ? J.np : (J.kind == 1 ? J.cnt : (J.np + kChunk - 1) / kChunk);
}

// One participant's share of a combine job: the float4 output columns
// idx = part*32 + lane (+ nparts*32 ...).  Each lane combines its column over
// all `count` states on its own (the page's Phase 2 formula): M = max m_i,
// total = sum e^(m_i - M) l_i, o = sum_i (e^(m_i - M) l_i / total) o_i.
template <class C>
__device__ __forceinline__ void combine_share(const KParams& prm, const Job& J, int part, int nparts,
                                              int lane) {
  using T = typename C::T;
  // States per round of loads (fewer where registers are tight).
  constexpr int D = C::D, D4 = D / 4, G8 = (C::kMma && D >= 256) ? 8 : 16;
  const float *sm, *sl, *so;
  int stride, first;
  if (J.kind == 2) {
    sm = prm.ws_cm; sl = prm.ws_cl; so = prm.ws_co; stride = prm.Cmax; first = 0;
  } else {
    sm = prm.ws_m; sl = prm.ws_l; so = prm.ws_o; stride = prm.Pmax; first = J.kind == 1 ? J.c * kChunk : 0;
  }
  const int count = job_count(J);
  for (int idx = part * 32 + lane; idx < J.nh * D4; idx += nparts * 32) {
    const int gh = idx / D4, d4 = idx - gh * D4;
    const size_t row = (size_t)J.s * prm.H + J.h0 + gh;
    const size_t base = row * stride + first;
    const float4* src = reinterpret_cast<const float4*>(so + base * D) + d4;
    // One pass in groups of 8 states, all loads of a group in flight at once,
    // with the running maximum rescaling the running sums.
    float M = -INFINITY, tot = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < count; i0 += G8) {
      float mv[G8], lv[G8];
      float4 ov[G8];
#pragma unroll
      for (int j = 0; j < G8; ++j) {
        if (i0 + j < count) {
          mv[j] = __ldcg(sm + base + i0 + j);
          lv[j] = __ldcg(sl + base + i0 + j);
          ov[j] = __ldcg(src + (size_t)(i0 + j) * D4);
        } else {
          mv[j] = -INFINITY;
          lv[j] = 0.f;
          ov[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float gm = mv[0];
#pragma unroll
      for (int j = 1; j < G8; ++j) gm = fmaxf(gm, mv[j]);
      const float Mn = fmaxf(M, gm);
      // States a causal row never reached are (-inf, 0): while every state so
      // far is one, subtract 0 so that they weigh 0 instead of NaN.
      const float Ms = (Mn == -INFINITY) ? 0.f : Mn;
      const float sc = exp2f((M - Ms) * kLog2e);
      tot *= sc;
      acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
#pragma unroll
      for (int j = 0; j < G8; ++j) {
        const float w = exp2f((mv[j] - Ms) * kLog2e) * lv[j];
        tot += w;
        acc.x = fmaf(w, ov[j].x, acc.x); acc.y = fmaf(w, ov[j].y, acc.y);
        acc.z = fmaf(w, ov[j].z, acc.z); acc.w = fmaf(w, ov[j].w, acc.w);
      }
      M = Mn;
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    const float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (J.kind == 1) {
      reinterpret_cast<float4*>(prm.ws_co + (row * prm.Cmax + J.c) * D)[d4] = r;
      if (d4 == 0) {
        prm.ws_cm[row * prm.Cmax + J.c] = M;
        prm.ws_cl[row * prm.Cmax + J.c] = tot;
      }
    } else {
      const size_t orow = out_row_rt(prm, J.s, J.h0 + gh);
      store4<T>(static_cast<T*>(prm.out) + orow * D + d4 * 4, r);
      // Final combine: the log-sum-exp of all the sequence's scores is
      // M + log(total) (natural-log units: the partition and chunk maxima are).
      if (d4 == 0 && prm.lse) prm.lse[orow] = M + logf(tot);
    }
  }
}

// Shared state of the job protocol between the epilogue warp (which posts
// jobs) and the consumer warps (which help with heavy ones).  Up to kJobSlots
// posted jobs can be in flight; job i uses slot i % kJobSlots: its record and
// an mbarrier that completes when all NC + 1 warps have taken their share.
constexpr int kJobSlots = 4;
struct JobChannel {
  volatile int* posted;    // number of jobs posted for help
  volatile int* finished;  // set once the epilogue warp posts no more jobs
  Job* rec;                // kJobSlots records
  uint32_t bar_done;       // kJobSlots mbarriers (8 bytes apart)
};

#ifndef PA_SETTLE_WHEN_IDLE
#define PA_SETTLE_WHEN_IDLE 1
#endif
constexpr bool kSettleWhenIdle = PA_SETTLE_WHEN_IDLE != 0;
// Consumer warps of the tensor-core kernel (several heads per unit, so
// combine jobs are shared) also look for posted jobs before every block.
#ifndef PA_MMA_HELP_PER_BLOCK
#define PA_MMA_HELP_PER_BLOCK 1
#endif
constexpr bool kMmaHelpPerBlock = PA_MMA_HELP_PER_BLOCK != 0;

// A consumer warp's help with every posted job it has not taken yet.
template <class C, class LY>
__device__ __forceinline__ void help_with_job(const KParams& prm, const JobChannel& ch, int& seen, int warp,
                                              int lane) {
  // Lane 0's reading decides for the whole warp.
  const int posted = __shfl_sync(0xffffffffu, *ch.posted, 0);
  while (seen < posted) {
    __threadfence_block();
    const int slot = seen % kJobSlots;
    const Job J = ch.rec[slot];
    combine_share<C>(prm, J, warp, LY::NC + 1, lane);
    // A chunk state is read by another CTA once the epilogue warp has retired
    // this job and released the sequence ticket: every lane's stores must be
    // visible GPU-wide before this warp counts its share done.
    if (J.kind == 1) fence_acq_rel_gpu();
    __syncwarp();
    if (lane == 0) mbar_arrive(ch.bar_done + 8 * slot);
    ++seen;
  }
}

template <class C, class LY>
__device__ __noinline__ void help_with_job_out_of_line(const KParams& prm, const JobChannel& ch, int& seen,
                                                       int warp, int lane) {
  help_with_job<C, LY>(prm, ch, seen, warp, lane);
}

// Consumer warp: wait (bounded) for the hand-over slot to be free for
// hand-over k, helping with any combine job posted meanwhile.  (The epilogue
// warp may be waiting for this warp's help before it can free the slot.)
template <class C, class LY>
__device__ __forceinline__ bool wait_handover(const KParams& prm, const JobChannel& ch, int& seen,
                                              uint32_t bar_eempty, uint32_t k, volatile int* abort_flag,
                                              int* err, int site, int warp, int lane) {
  const uint32_t parity = (k & 1u) ^ 1u;
  if (__all_sync(0xffffffffu, mbar_test_wait(bar_eempty, parity))) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    help_with_job<C, LY>(prm, ch, seen, warp, lane);
    if (__all_sync(0xffffffffu, mbar_test_wait(bar_eempty, parity))) return true;
    if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
    if ((long long)(global_timer_ns() - t0) > prm.timeout_ns) {
      if (lane == 0) record_timeout(abort_flag, err, site, (int)k);
      return false;
    }
    __nanosleep(32);
  }
}

// Epilogue warp's combine-job engine.  Jobs are queued; a heavy job is posted
// for the consumer warps (up to kJobSlots in flight), who take their shares at
// their next unit boundary, while the epilogue warp takes its own share and
// goes back to merging hand-overs.  Completion is polled in posting order; a
// completed chunk job (kind 1) then takes the sequence ticket, and the last
// chunk's final job (kind 2) is queued.  All members are warp-uniform; queued
// jobs live in a shared-memory ring.
template <class C, class LY>
struct JobEngine {
  static constexpr int JQ = 16;
  const KParams& prm;
  const JobChannel& ch;
  Job* q;               // JQ slots
  volatile int* abort_flag;
  int* err;
  int lane;
  int head = 0, tail = 0;       // queued jobs
  int nposted = 0, ndone = 0;   // posted jobs, and those completed (in order)

  __device__ __forceinline__ JobEngine(const KParams& p, const JobChannel& c, Job* qq, volatile int* ab,
                                       int* e, int l)
      : prm(p), ch(c), q(qq), abort_flag(ab), err(e), lane(l) {}

  // Shared if it is large, or if the epilogue warp alone would need more than
  // one output column per lane (columns are combined one after another, each
  // a round trip to L2).
  __device__ __forceinline__ bool heavy(const Job& J) const {
    const int columns = J.nh * (C::D / 4);
    return columns > 32 || (long long)columns * job_count(J) > kShareJobLoads;
  }

  // Sequence-level ticket after a chunk job; true if it completed the sequence.
  __device__ __forceinline__ bool chunk_done(const Job& J) {
    int last = 0;
    if (lane == 0) {
      int* tk = prm.tickets + (size_t)J.s * prm.n_hg + J.hg;
      const int t = atomic_add_release_gpu(tk, 1);
      last = (t == (J.np + kChunk - 1) / kChunk - 1);
      if (last) {
        *tk = 0;
        fence_acq_rel_gpu();
      }
    }
    return __shfl_sync(0xffffffffu, last, 0) != 0;
  }

  // Run J alone, now (and its follow-up).
  __device__ __forceinline__ void run_alone(Job J) {
    while (true) {
      combine_share<C>(prm, J, 0, 1, lane);
      if (J.kind == 1) fence_acq_rel_gpu();  // every lane's chunk state, before the ticket
      __syncwarp();
      if (J.kind != 1 || !chunk_done(J)) return;
      J.kind = 2;
    }
  }

  __device__ __forceinline__ void push(const Job& J) {
    if (tail - head >= JQ) {  // queue full (not expected): no waiting, just do it
      run_alone(J);
      return;
    }
    if (lane == 0) q[tail % JQ] = J;
    __syncwarp();
    ++tail;
  }

  // Start J: post it (heavy; the caller guarantees a free slot) or run it alone.
  __device__ __forceinline__ void launch(const Job& J) {
    {
      if (heavy(J)) {
        const int slot = nposted % kJobSlots;
        if (lane == 0) {
          ch.rec[slot] = J;
          __threadfence_block();
          *ch.posted = nposted + 1;
        }
        ++nposted;
        combine_share<C>(prm, J, LY::NC, LY::NC + 1, lane);
        if (J.kind == 1) fence_acq_rel_gpu();  // every lane's chunk state, before the ticket
        __syncwarp();
        if (lane == 0) mbar_arrive(ch.bar_done + 8 * slot);
        return;
      }
      run_alone(J);
      return;
    }
  }

  // Make progress without blocking (block = false) or until idle (block = true,
  // each wait bounded).  Returns false once the CTA is aborting.
  __device__ __forceinline__ bool poll(bool block) {
    while (true) {
      while (ndone < nposted) {
        const int slot = ndone % kJobSlots;
        const uint32_t par = (uint32_t)(ndone / kJobSlots) & 1u;
        const uint32_t bar = ch.bar_done + 8 * slot;
        bool done = __all_sync(0xffffffffu, mbar_test_wait(bar, par));
        if (!done && block)
          done = __all_sync(0xffffffffu, wait_bounded(bar, par, abort_flag, err, prm.timeout_ns,
                                                      kSiteJobDone, ndone));
        if (!done) break;
        // Every helper's arrival was observed: their stores are ordered
        // before the release in chunk_done.
        Job J = broadcast_job(ch.rec[slot]);
        ++ndone;
        if (J.kind == 1 && chunk_done(J)) {
          J.kind = 2;
          push(J);
        }
      }
      if (block && ndone < nposted) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
        continue;  // the bounded wait above gave up: loop re-checks the flag
      }
      while (head != tail && nposted - ndone < kJobSlots) {
        const Job J = broadcast_job(q[head % JQ]);
        ++head;
        launch(J);
      }
      if (!block || (ndone == nposted && head == tail)) return __all_sync(0xffffffffu, *abort_flag == 0);
    }
  }

  __device__ __forceinline__ bool drain() {
    while (ndone < nposted || head != tail)
      if (!poll(true)) return false;
    return true;
  }
};

// Consumer warp: stream the blocks of every unit assigned to it and hand its
// online-softmax state for each unit to the epilogue warp through shared
// memory.  Consumer warps never wait for each other.
template <class C, class LY, bool MQ>
__device__ __forceinline__ void consumer_loop(const KParams& prm, uint8_t* smem, const int* pref,
                                              const UnitInfo* info, volatile int* abort_flag,
                                              const volatile uint32_t* issued, const JobChannel& ch,
                                              int warp, int lane) {
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

  // Unused partitions: sentinels (m = -inf, l = 0).  Empty sequences: zeros
  // (a multi-query sequence is never empty: it holds its new tokens).
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
    if constexpr (!MQ) {
      constexpr int D16 = D * (int)sizeof(T) / 16;  // 16-byte words per output row
      const long long n2 = (long long)S * H * D16;
      for (long long i = (long long)blockIdx.x * NCT + ctid; i < n2; i += (long long)gridDim.x * NCT) {
        const int s = (int)(i / ((long long)H * D16));
        if (pref[s + 1] == pref[s]) reinterpret_cast<uint4*>(out)[i] = make_uint4(0, 0, 0, 0);
      }
      if (prm.lse) {  // no scores: the log-sum-exp is log 0
        for (int i = blockIdx.x * NCT + ctid; i < S * H; i += gridDim.x * NCT)
          if (pref[i / H + 1] == pref[i / H]) prm.lse[i] = -INFINITY;
      }
    }
  }

  C cons;
  uint32_t g = 0, k = 0;
  int seen = 0;  // combine jobs helped with
  while (true) {
    const int slot = k % UQ;
    const uint32_t par = (k / UQ) & 1u;
    const bool okw = __all_sync(0xffffffffu, wait_bounded(bar_ufull + 8 * slot, par, abort_flag, err,
                                                          prm.timeout_ns, kSiteUnit, (int)k));
    const UnitInfo I = info[slot];
    if (!okw) break;
    if (I.s < 0) {
      // End of work: pass the end marker on to the epilogue warp, once it has
      // taken the previous hand-over (the k-th hand-over waits for the
      // (k-1)-th to be consumed), then help with combine jobs until the
      // epilogue warp has run its last one.
      if (!wait_handover<C, LY>(prm, ch, seen, bar_eempty, k, abort_flag, err, kSiteHandEnd, warp, lane))
        break;
      if (warp == 0 && lane == 0) epi_info->s = -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_efull);
      const uint64_t t0 = global_timer_ns();
      while (true) {
        help_with_job<C, LY>(prm, ch, seen, warp, lane);
        if (__any_sync(0xffffffffu, *ch.finished != 0 || *abort_flag != 0)) break;
        if ((long long)(global_timer_ns() - t0) > prm.timeout_ns) {
          if (lane == 0) record_timeout(abort_flag, err, kSiteServe, seen);
          break;
        }
        __nanosleep(64);
      }
      break;
    }
    cons.begin_unit(reinterpret_cast<const T*>(smem + LY::OFF_Q + slot * LY::QSLOT), I.nh,
                    prm.scale_log2, lane);
    if constexpr (C::kMma)
      cons.set_limits([&](int h) { return row_limit<MQ>(prm, I.L, I.h0 + h); }, lane);
    fence_proxy_async_smem();  // the query slot is refilled by a bulk copy: same ordering as a stage
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_uempty + 8 * slot);

    // Work item i of unit u goes to warp (i + u) % NC: when a unit's item
    // count is not a multiple of NC, the extra items fall on different warps
    // from unit to unit instead of on warps 0, 1, ... every time.  The
    // grouping depends only on the unit, never on which CTA runs it.  An item
    // is one block, or for the tensor-core consumer over 8-token blocks two
    // consecutive blocks (one 16-token tile of the products).
    constexpr int PB = (C::kMma && BS == 8 && !C::kFp8) ? 2 : 1;
    const int u_id = (pref[I.s] + I.p) * prm.n_hg + I.hg;
    const int nitem = (I.nb + PB - 1) / PB;
    for (int it = (warp + NC - u_id % NC) % NC; it < nitem; it += NC) {
      if constexpr (C::kMma && kMmaHelpPerBlock) {
        if (__shfl_sync(0xffffffffu, *ch.posted, 0) > seen) help_with_job<C, LY>(prm, ch, seen, warp, lane);
      }
      const int j = it * PB, nbi = min(PB, I.nb - j);
      const uint32_t gj = g + j, st = stage_of<LY>(gj);
      bool okb = wait_issued(issued, gj + nbi, abort_flag, err, prm.timeout_ns);
      for (int b = 0; b < nbi && okb; ++b)
        okb = wait_bounded(bar_full + 8 * stage_of<LY>(gj + b), phase_of<LY>(gj + b), abort_flag, err,
                           prm.timeout_ns, kSiteFull, (int)(gj + b));
      // A stage whose copy this warp has not seen land is never released:
      // on a failed wait the warp stops (the producer sees the abort and
      // waits for its copies before the CTA exits).
      if (!__all_sync(0xffffffffu, okb)) break;
      const int ntok = min(nbi * BS, I.t1 - I.t0 - j * BS);
      uint8_t* sa = smem + st * LY::STAGE;
      if constexpr (PB == 2) {
        if (nbi == 2) {
          uint8_t* sb = smem + stage_of<LY>(gj + 1) * LY::STAGE;
          cons.block_pair(sa, sa + LY::KBYTES, sb, sb + LY::KBYTES, ntok, lane, I.t0 + j * BS);
        } else {
          cons.block(sa, sa + LY::KBYTES, ntok, lane, scr, I.t0 + j * BS);
        }
      } else {
        cons.block(sa, sa + LY::KBYTES, ntok, lane, scr, I.t0 + j * BS);
      }
      // The stage is refilled by a bulk copy (async proxy) once released:
      // every lane's reads of it (generic proxy) are ordered before that
      // write by a proxy fence, or the copy can land under reads still
      // queued (the last V tile read stale data without it).
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        for (int b = 0; b < nbi; ++b) mbar_arrive(bar_empty + 8 * stage_of<LY>(gj + b));
    }
    if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
    g += I.nb;

    // Hand this warp's state for unit k to the epilogue warp, once it has
    // taken unit k-1's (helping with combine jobs meanwhile).
    if (!wait_handover<C, LY>(prm, ch, seen, bar_eempty, k, abort_flag, err, kSiteHandover, warp, lane))
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
                                              const JobChannel& ch, int lane) {
  using T = typename C::T;
  constexpr int D = C::D, GT = C::GT, NC = LY::NC, NS = LY::NSTAGE, UQ = LY::UQ;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_efull = sbase + LY::OFF_BAR + (2 * NS + 2 * UQ) * 8, bar_eempty = bar_efull + 8;
  const float* epi_acc = reinterpret_cast<const float*>(smem + LY::OFF_EPI_ACC);
  const float* epi_ml = reinterpret_cast<const float*>(smem + LY::OFF_EPI_ML);
  const UnitInfo* epi_info = reinterpret_cast<const UnitInfo*>(smem + LY::OFF_EPI_INFO);
  float* rstat = reinterpret_cast<float*>(smem + LY::OFF_RSTAT);
  float* ef = reinterpret_cast<float*>(smem + LY::OFF_EF);  // [NC][GT] weights, then [GT] sums
  int* err = prm.hdr + kHdrError;
  const int H = prm.H, Pmax = prm.Pmax;
  T* out = static_cast<T*>(prm.out);
  JobEngine<C, LY> jobs(prm, ch, reinterpret_cast<Job*>(smem + LY::OFF_JOBQ), abort_flag, err, lane);

  // Lane 0 only: a ticket taken and not yet checked, and its job.
  bool pend = false;
  int pend_t = 0;
  Job pinfo{};
  // Lane 0: if the pending ticket was the last of its group, its job (the
  // acquire fence orders the other CTAs' partition states before it).
  auto settle = [&]() -> int {
    int go = 0;
    if (lane == 0 && pend && pend_t == pinfo.cnt - 1) {
      go = 1;
      *ticket_of(prm, pinfo) = 0;
      fence_acq_rel_gpu();
    }
    pend = false;
    return __shfl_sync(0xffffffffu, go, 0);
  };

  for (uint32_t k = 0;; ++k) {
    // Wait for hand-over k, advancing combine jobs meanwhile.
    bool ok = __all_sync(0xffffffffu, mbar_test_wait(bar_efull, k & 1u));
    if (!ok) {
      // Idle: settle the pending ticket now rather than at the next merge
      // (its atomic has long returned), so a job it completes starts early.
      if (kSettleWhenIdle) {
        const Job R = broadcast_job(pinfo);
        if (settle()) jobs.push(R);
      }
      const uint64_t t0 = global_timer_ns();
      while (!ok) {
        if (!jobs.poll(false)) return;
        ok = __all_sync(0xffffffffu, mbar_test_wait(bar_efull, k & 1u));
        if (ok) break;
        if (__any_sync(0xffffffffu, *abort_flag != 0)) return;
        if ((long long)(global_timer_ns() - t0) > prm.timeout_ns) {
          if (lane == 0) record_timeout(abort_flag, err, kSiteEpiFull, (int)k);
          return;
        }
        __nanosleep(32);
      }
    }
    const UnitInfo I = *epi_info;
    if (I.s < 0) {
      // End of work: settle the last ticket, finish every job (the consumer
      // warps are waiting to help), then release them.
      const Job R = broadcast_job(pinfo);  // pinfo is kept by lane 0 only
      if (settle()) jobs.push(R);
      jobs.drain();
      if (lane == 0) *ch.finished = 1;
      return;
    }
    // Per head: M = max over warps, each warp's weight 2^(m_w - M), and the sum l.
    for (int i = lane; i < GT; i += 32) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w) M = fmaxf(M, epi_ml[(w * GT + i) * 2]);
      float den = 0.f;
      // A causal row with no position in this partition has M = -inf: its
      // weights come out 0 (subtracting 0), its state (-inf, 0, 0).
      const float Ms = (M == -INFINITY) ? 0.f : M;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float f = exp2f(epi_ml[(w * GT + i) * 2] - Ms);
        ef[w * GT + i] = f;
        den = fmaf(f, epi_ml[(w * GT + i) * 2 + 1], den);
      }
      ef[NC * GT + i] = den;
      rstat[i * 2] = M;
    }
    __syncwarp();
    const bool single = (I.np == 1);
    constexpr int D4 = D / 4;
    for (int idx = lane; idx < I.nh * D4; idx += 32) {
      const int gh = idx / D4, d4 = idx - gh * D4;
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float f = ef[w * GT + gh];
        const float4 v = reinterpret_cast<const float4*>(epi_acc + (w * GT + gh) * D)[d4];
        num.x = fmaf(f, v.x, num.x); num.y = fmaf(f, v.y, num.y);
        num.z = fmaf(f, v.z, num.z); num.w = fmaf(f, v.w, num.w);
      }
      const float den = ef[NC * GT + gh];
      const float inv = (den > 0.f ? 1.f / den : 0.f) * prm.v_scale;
      const float4 val = make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
      const size_t sh = (size_t)I.s * H + I.h0 + gh;
      if (single) {
        store4<T>(out + out_row_rt(prm, I.s, I.h0 + gh) * D + d4 * 4, val);
      } else {
        reinterpret_cast<float4*>(prm.ws_o + (sh * Pmax + I.p) * D)[d4] = val;
      }
      if (d4 == 0) {
        prm.ws_m[sh * Pmax + I.p] = rstat[gh * 2] * kLn2;
        prm.ws_l[sh * Pmax + I.p] = ef[NC * GT + gh];
        // A single-partition sequence ends here: its log-sum-exp is the
        // merged maximum (log2 units -> natural) plus the log of the merged sum.
        if (single && prm.lse) prm.lse[out_row_rt(prm, I.s, I.h0 + gh)] = rstat[gh * 2] * kLn2 + logf(ef[NC * GT + gh]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_eempty);  // the hand-over slot may be refilled

    // Settle the previous ticket; take this unit's (release: the warp's
    // partition stores above, ordered by __syncwarp, become visible first).
    const Job R = broadcast_job(pinfo);
    const int go = settle();
    if (lane == 0) {
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
    if (go) jobs.push(R);
    if (!jobs.poll(false)) return;
  }
}

template <class C, int NC, int NSTAGE, int CTAS_PER_SM, bool MQ>
__global__ void __launch_bounds__(Layout<C, NC, NSTAGE>::THREADS, CTAS_PER_SM)
    pa_decode_kernel(const __grid_constant__ KParams prm) {
  using LY = Layout<C, NC, NSTAGE>;
  constexpr int NS = LY::NSTAGE, UQ = LY::UQ;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::OFF_FLAGS);
  volatile uint32_t* issued = reinterpret_cast<volatile uint32_t*>(smem + LY::OFF_FLAGS + 8);
  JobChannel ch;
  ch.posted = reinterpret_cast<volatile int*>(smem + LY::OFF_FLAGS + 4);
  ch.finished = reinterpret_cast<volatile int*>(smem + LY::OFF_FLAGS + 12);
  ch.rec = reinterpret_cast<Job*>(smem + LY::OFF_JOBREC);
  ch.bar_done = sbase + LY::OFF_BAR + 8 * (2 * NS + 2 * UQ + 2);
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
    for (int i = 0; i < kJobSlots; ++i)
      mbar_init(bar + 8 * (2 * NS + 2 * UQ + 2 + i), NC + 1);  // shared combine job done: all helpers
    *abort_flag = 0;
    *issued = 0;
    *ch.posted = 0;
    *ch.finished = 0;
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
      bool bad = false;
      const int L = seq_tokens<MQ>(prm, s, max_len, &bad);
      if (bad) atomicCAS(prm.hdr + kHdrError, 0, kErrDeviceBounds);
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
      bool bad = false;
      run += (seq_tokens<MQ>(prm, s, max_len, &bad) + prm.P - 1) / prm.P;
    }
  }
  __syncthreads();
  if (warp == NC) {
    producer_loop<C, LY, MQ>(prm, smem, pref, info, abort_flag, issued, lane);
  } else if (warp == NC + 1) {
    epilogue_loop<C, LY>(prm, smem, abort_flag, ch, lane);
  } else {
    consumer_loop<C, LY, MQ>(prm, smem, pref, info, abort_flag, issued, ch, warp, lane);
  }
}

}  // namespace pa
