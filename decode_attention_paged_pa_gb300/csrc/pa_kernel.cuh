// pa_kernel.cuh -- persistent, warp-specialised paged decode attention kernel
// (phase 1).
//
// Work unit = (sequence s, partition p, head group hg): the tokens
// [p*P, min((p+1)*P, L)) of s against GT query heads that share one kv head
// (or, for consumers with KVU > 1, the query heads of KVU consecutive kv
// heads: one block of each of them per ring stage).
// This is the phase-1 program of the page "paged_attention_v2_triton.py --
// Triton PagedAttention V2 for BI-V100" (`_paged_attn_v2_partition_kernel`,
// grid (seq, head, partition)), except that only used partitions become units
// and the GT heads of a group share every K/V load.
//
// One CTA per SM runs until the units run out:
//   * warp NC (producer): takes units from a global counter (dynamic
//     scheduling balances skewed sequence lengths; the next unit is claimed
//     and planned during the current unit's last batches), publishes each unit's
//     description and query rows through a 2-slot unit queue, and streams the
//     unit's physical K and V blocks -- each a contiguous D*BS*(element
//     size)-byte run in the page's layouts -- into shared memory, completing
//     on mbarriers: the key block by a 1-D bulk async copy, the value block by
//     a 1-D bulk copy or (tensor-core consumer over 16-bit caches, C::kTma) a
//     3-D tensor copy that lays its rows out in the swizzle of their width;
//   * warps 0..NC-1 (consumers): work item j of unit (p, hg) (a block, or two
//     consecutive blocks: C::kItemBlocks) goes to warp (j + p * n_hg + hg) % NC
//     (a fixed grouping, so results do not depend on scheduling), which folds
//     it into its private online-softmax state
//     (SimtConsumer, MmaConsumer or MmaRowConsumer).  The CTA's g-th block (counted over all
//     its units) lives in ring stage g % NSTAGE.  Warps run at different
//     speeds, so a fast warp could reach stage g % NSTAGE while the stage's
//     previous copy (block g - NSTAGE) is still in flight, and an mbarrier
//     parity wait cannot tell those two phases apart.  A consumer therefore
//     first waits until the producer has issued block g (a shared-memory
//     counter): the producer issues block g only after block g - NSTAGE was
//     consumed, so by then the stage's previous phase is complete and the
//     parity wait is exact.  At the end of a unit each warp hands its state
//     to the epilogue warp;
//   * warp NC + 1 (epilogue): merges the consumer warps' states of each unit
//     into the partition's (m_p, l_p, o_p) in the workspace, or, for a
//     sequence with one partition, into the output (single pass).
// Unused partitions get the sentinels (m = -inf, l = 0) of the page.  The
// cross-partition combine of `_paged_attn_v2_reduce_kernel` is phase 2
// (pa_combine.cuh), launched as a programmatic dependent of this kernel: each
// CTA signals it once its producer has run out of units.
#pragma once

#include "pa_common.cuh"

namespace pa {

// Sequences per launch: the kernel keeps the longest-first order and a prefix
// sum of partitions per sequence in shared memory (6 bytes a sequence, taken
// from the ring); longer batches are split into several launches.
#ifndef PA_MAX_SEQS_PER_LAUNCH
#define PA_MAX_SEQS_PER_LAUNCH 512
#endif
constexpr int kMaxSeqsPerLaunch = PA_MAX_SEQS_PER_LAUNCH;
static_assert(kMaxSeqsPerLaunch <= 65536, "ranks are kept as 16-bit sequence indices");

struct KParams {
  // Tensor map of the value cache (C::kTma consumers only): [NB * KH][D][BS]
  // elements, box [C::KVU][D][BS] (the unit's kv heads of one block),
  // shared-memory rows in the swizzle of their width (BS * 2 bytes: 32, 64
  // or 128).
  CUtensorMap tmv;
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
  float* lse;    // [S, H] log-sum-exp of the scaled scores, or null
  int q_len;     // query tokens per sequence (multi-query kernels; 1 otherwise)
  int Hu, Gu;    // the caller's heads and heads per kv head; H and G below count row
                 // heads, q_len of them per caller head (H = q_len * Hu, G = q_len * Gu)
  float scale_log2;   // softmax scale (times k_scale for an fp8 cache) times log2 e
  float v_scale;      // multiplies every output: 1, or an fp8 cache's v_scale
  int S, H, KH, G, MB, num_blocks, P, Pmax;
  int hg_per_kv;  // ceil(G / GT)
  int n_hg;       // head groups per partition: KH * hg_per_kv, or KH / KVU
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
  // A stage holds one block of one kv head: the K block, then at VOFF the V
  // block; its copies deliver STAGE_TX bytes.
  static constexpr uint32_t KBYTES = C::KBLK;
  static constexpr uint32_t VOFF = C::KREGION;
  static constexpr uint32_t STAGE = C::STAGE_BYTES;
  static constexpr uint32_t STAGE_TX = C::STAGE_TX;
  static_assert(!C::kTma || (STAGE % 1024 == 0 && VOFF % 1024 == 0), "swizzled value blocks 1024-byte aligned");
  static constexpr uint32_t RING = NSTAGE * STAGE;
  static constexpr uint32_t QROW_BYTES = (uint32_t)C::QROW * sizeof(typename C::T);
  static_assert(QROW_BYTES % 16 == 0, "query rows start on 16-byte boundaries (bulk copies)");
  static constexpr uint32_t QSLOT = C::GT * QROW_BYTES;
  static constexpr uint32_t OFF_Q = RING;
  static constexpr uint32_t OFF_EPI_ACC = al16(OFF_Q + UQ * QSLOT);
  static constexpr uint32_t OFF_EPI_ML = al16(OFF_EPI_ACC + NC * C::GT * C::AROW * 4);
  static constexpr uint32_t OFF_SCR = al16(OFF_EPI_ML + NC * C::GT * 2 * 4);
  static constexpr uint32_t OFF_RSTAT = al16(OFF_SCR + NC * C::SCRATCH_FLOATS * 4);
  static constexpr uint32_t OFF_EF = al16(OFF_RSTAT + C::GT * 2 * 4);   // NC*GT warp weights + GT sums
  static constexpr uint32_t OFF_INFO = al16(OFF_EF + (NC + 1) * C::GT * 4);
  static constexpr uint32_t OFF_EPI_INFO = al16(OFF_INFO + UQ * sizeof(UnitInfo));
  static constexpr uint32_t OFF_BAR = al16(OFF_EPI_INFO + sizeof(UnitInfo));
  static constexpr uint32_t NBAR = 2 * NSTAGE + 2 * UQ + 2;
  static constexpr uint32_t OFF_FLAGS = al16(OFF_BAR + NBAR * 8);
  static constexpr uint32_t OFF_PREF = al16(OFF_FLAGS + 64);
  static constexpr uint32_t FIXED = OFF_PREF;
  // pref: [S + 1] int32 partitions before each rank; then perm: [S] uint16
  // sequence of each rank (longest first).
  static constexpr uint32_t perm_off(int S) { return al16(OFF_PREF + (uint32_t)(S + 1) * 4); }
  static constexpr uint32_t bytes(int S) { return al16(perm_off(S) + (uint32_t)S * 2); }
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
  kSiteEpiFull = 9      // epilogue: the consumers' states of a unit
};

// Longest sleep of the producer warp between polls of the ring.
constexpr unsigned kMaxBackoffNs = 512;

// Wait (bounded) until the producer has issued at least `target` blocks.
__device__ __forceinline__ bool wait_issued(const volatile uint32_t* issued, uint32_t target,
                                            volatile int* abort_flag, int* err_word,
                                            long long timeout_ns) {
  if (*issued >= target) return true;
  // Not issued yet: its copy is at least a memory latency away, so poll
  // sparingly.
  const uint64_t t0 = global_timer_ns();
  while (true) {
    __nanosleep(64);
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

// Unit u = (partition pair, head group): pairs are numbered over the
// sequences in longest-first order (rank r holds sequence perm[r] and
// partitions pref[r] .. pref[r + 1] - 1), so the sequences with the most
// partitions, whose combines are the longest chains, start first, and the
// last units handed out belong to the shortest sequences.
template <class C, bool MQ>
__device__ __forceinline__ UnitPlan plan_unit(const KParams& prm, const int* pref, const uint16_t* perm, int u) {
  constexpr int BS = C::BS, GT = C::GT;
  UnitPlan U;
  const int pair = u / prm.n_hg;
  U.hg = u - pair * prm.n_hg;
  int lo = 0, hi = prm.S;  // pref[lo] <= pair < pref[lo + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= pair) lo = mid; else hi = mid;
  }
  bool bad = false;  // flagged by the prologue already
  U.s = perm[lo];
  U.p = pair - pref[lo];
  U.np = pref[lo + 1] - pref[lo];
  const int L = seq_tokens<MQ>(prm, U.s, prm.MB * C::BS, &bad);
  U.L = L;
  U.t0 = U.p * prm.P;
  U.t1 = min(U.t0 + prm.P, L);
  U.nb = (U.t1 - U.t0 + BS - 1) / BS;
  if constexpr (C::KVU > 1) {
    // Head group hg: kv heads KVU hg .. KVU hg + KVU - 1, their G * KVU query heads.
    U.kv = U.hg * C::KVU;
    U.h0 = U.kv * prm.G;
    U.nh = min(GT, prm.G * C::KVU);
  } else {
    U.kv = U.hg / prm.hg_per_kv;
    const int hgk = U.hg - U.kv * prm.hg_per_kv;
    U.h0 = U.kv * prm.G + hgk * GT;
    U.nh = min(GT, prm.G - hgk * GT);
  }
  return U;
}

// This lane's block-table entry among blocks [c0, c0 + 32) of unit U, as
// loaded (0 past the unit's end): issuing the load and checking the entry
// (check_block_id) are split so that the load's latency can overlap other
// work.
template <class C>
__device__ __forceinline__ int fetch_block_id(const KParams& prm, const UnitPlan& U, int c0, int lane) {
  return (c0 + lane < U.nb) ? __ldg(prm.bt + (size_t)U.s * prm.MB + U.t0 / C::BS + c0 + lane) : 0;
}
// An id outside the pool is recorded and replaced by 0, so nothing is read
// out of bounds.
__device__ __forceinline__ int check_block_id(const KParams& prm, int b) {
  if ((unsigned)b >= (unsigned)prm.num_blocks) {
    atomicCAS(prm.hdr + kHdrError, 0, kErrDeviceBounds);
    b = 0;
  }
  return b;
}
template <class C>
__device__ __forceinline__ int load_block_id(const KParams& prm, const UnitPlan& U, int c0, int lane) {
  return check_block_id(prm, fetch_block_id<C>(prm, U, c0, lane));
}

template <class C, class LY, bool MQ>
__device__ __forceinline__ void producer_loop(const KParams& prm, uint8_t* smem, const int* pref,
                                              const uint16_t* perm, UnitInfo* info, volatile int* abort_flag,
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
    Up = plan_unit<C, MQ>(prm, pref, perm, u);
    return true;
  };

  // The prologue kept temporaries in the ring: order those generic-proxy
  // writes before the copies (async proxy) that will overwrite them.
  fence_proxy_async_smem();
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
        if constexpr (!MQ && C::QROW == D)
          bulk_copy_g2s(sbase + LY::OFF_Q + slot * LY::QSLOT,
                        static_cast<const T*>(prm.q) + ((size_t)Up.s * prm.H + Up.h0) * D, qbytes,
                        bar_ufull + 8 * slot, pol_keep);
      }
    }
    okp = __shfl_sync(0xffffffffu, (int)okp, 0) != 0;
    if constexpr (MQ || C::QROW != D) {
      // One row copy per lane: the row heads of a multi-query unit are
      // scattered over the caller's [S, q_len, H] rows, and padded rows
      // (QROW > D) are not contiguous in the slot.
      if (okp && have && lane < Up.nh)
        bulk_copy_g2s(sbase + LY::OFF_Q + slot * LY::QSLOT + lane * LY::QROW_BYTES,
                      static_cast<const T*>(prm.q) + out_row<MQ>(prm, Up.s, Up.h0 + lane) * D,
                      (uint32_t)(D * sizeof(T)), bar_ufull + 8 * slot, pol_keep);
    }
    if (okp) ++kq;
    return okp;
  };

  // The work counter is read late: the next unit is claimed when unit k's
  // second-to-last batch of copies starts (its last, for a unit of one
  // batch), planned when the last batch starts, with the load of its first
  // block ids in flight while that batch issues, and published once the
  // batch is issued.  A CTA thus commits to a unit only shortly before it
  // streams it, which keeps the end of the work even across CTAs (claiming
  // at the start of unit k left up to two units to a CTA when the counter
  // ran out), and the two round trips (the atomic, the block-table load)
  // stay off the gap between the units' copies.  CTA i's first unit is unit
  // i, without an atomic (all CTAs start at once, and their first claims
  // would queue on one word); the counter hands out units gridDim.x,
  // gridDim.x + 1, ...
  int u_cur = blockIdx.x;
  UnitPlan U{};
  bool have = plan_next(u_cur, U);
  int bids = 0;  // this lane's block id among the unit's first 32 blocks
  if (have) bids = load_block_id<C>(prm, U, 0, lane);
  ok = publish(U, have);
  while (have && ok) {
    int u_req = 0;
    bool claimed = false;
    auto claim_next = [&]() {
      if (lane == 0) u_req = atomicAdd(prm.hdr + kHdrWork, 1) + (int)gridDim.x;
      claimed = true;
    };
    bool have_next = false, planned_next = false;
    UnitPlan Un{};
    int bids_next = 0;  // as fetched: checked when the unit is published
    auto plan_fetch_next = [&]() {
      const int u_nx = __shfl_sync(0xffffffffu, u_req, 0);
      have_next = plan_next(u_nx, Un);
      if (have_next) bids_next = fetch_block_id<C>(prm, Un, 0, lane);
      planned_next = true;
    };
    // Batches of the unit: those of its 32-block chunks (a batch never crosses one).
    const int nbatch = (U.nb / 32) * ((32 + BATCH - 1) / BATCH) + (U.nb % 32 + BATCH - 1) / BATCH;
    int ib = 0;
    for (int c0 = 0; c0 < U.nb && ok; c0 += 32) {
      const int b32 = (c0 == 0) ? bids : load_block_id<C>(prm, U, c0, lane);
      const int cend = min(c0 + 32, U.nb);
      for (int jb = c0; jb < cend && ok; jb += BATCH, ++ib) {
        if (!claimed && ib + 2 >= nbatch) {
          claim_next();  // the unit's second-to-last batch (its only one)
        } else if (claimed && !planned_next && ib + 1 == nbatch) {
          plan_fetch_next();  // the last batch: the claim issued a batch ago has returned
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
        // Back off while no stage frees up: the polls take issue slots from
        // the consumer warps of this sub-partition, and the ring holds
        // microseconds of copies, so a late reissue costs nothing.
        unsigned backoff = 32, seen = 0;
        while (true) {
          if (!done && mbar_test_wait(bar_empty + 8 * st, ph ^ 1u)) {
            const uint32_t dst = sbase + st * LY::STAGE;
            const size_t off = ((size_t)bi * prm.KH + U.kv) * (size_t)(D * C::BS) * C::KV_ESZ;
            mbar_arrive_expect_tx(bar_full + 8 * st, LY::STAGE_TX);
            bulk_copy_g2s(dst, static_cast<const uint8_t*>(prm.kc) + off, LY::KBYTES, bar_full + 8 * st,
                          pol_stream);
            if constexpr (C::kTma) {
              // The whole value block (x = 0: the 16-byte alignment rule holds).
              tma_load_3d(dst + LY::VOFF, &prm.tmv, 0, 0, bi * prm.KH + U.kv, bar_full + 8 * st, pol_stream);
            } else {
              bulk_copy_g2s(dst + LY::VOFF, static_cast<const uint8_t*>(prm.vc) + off, LY::KBYTES,
                            bar_full + 8 * st, pol_stream);
            }
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
                const unsigned n_done = __popc(m);
                backoff = n_done > seen ? 32u : min(backoff * 2u, kMaxBackoffNs);
                seen = n_done;
                __nanosleep(backoff);
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
    if (ok && !claimed) claim_next();
    if (ok && !planned_next) plan_fetch_next();
    if (ok) {
      if (have_next) bids_next = check_block_id(prm, bids_next);
      ok = publish(Un, have_next);
    }
    U = Un;
    bids = bids_next;
    have = have_next;
  }
  // No more units for this CTA: phase 2 may be launched once every CTA has
  // said so (it waits for this grid to complete before it reads anything).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// Consumer warp: wait (bounded) for the hand-over slot to be free for
// hand-over k (the epilogue warp has merged hand-over k - 1).
__device__ __forceinline__ bool wait_handover(const KParams& prm, uint32_t bar_eempty, uint32_t k,
                                              volatile int* abort_flag, int* err, int site, int lane) {
  const uint32_t parity = (k & 1u) ^ 1u;
  // try_wait suspends the warp in hardware (for a bounded time) instead of
  // spinning on issue slots the other warps of its sub-partition need.
  if (__all_sync(0xffffffffu, mbar_try_wait(bar_eempty, parity))) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar_eempty, parity))) return true;
    if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
    if ((long long)(global_timer_ns() - t0) > prm.timeout_ns) {
      if (lane == 0) record_timeout(abort_flag, err, site, (int)k);
      return false;
    }
  }
}

// Consumer warp: stream the blocks of every unit assigned to it and hand its
// online-softmax state for each unit to the epilogue warp through shared
// memory.  Consumer warps never wait for each other.
template <class C, class LY, bool MQ>
__device__ __forceinline__ void consumer_loop(const KParams& prm, uint8_t* smem, const UnitInfo* info,
                                              volatile int* abort_flag, const volatile uint32_t* issued, int warp,
                                              int lane) {
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
    auto parts_of = [&](int s) {
      bool bad = false;  // flagged by the prologue already
      return (seq_tokens<MQ>(prm, s, prm.MB * C::BS, &bad) + prm.P - 1) / prm.P;
    };
    const long long n1 = (long long)S * H * Pmax;
    for (long long i = (long long)blockIdx.x * NCT + ctid; i < n1; i += (long long)gridDim.x * NCT) {
      const int s = (int)(i / ((long long)H * Pmax));
      const int p = (int)(i % Pmax);
      if (p >= parts_of(s)) {
        prm.ws_m[i] = -INFINITY;
        prm.ws_l[i] = 0.f;
      }
    }
    if constexpr (!MQ) {
      constexpr int D16 = D * (int)sizeof(T) / 16;  // 16-byte words per output row
      const long long n2 = (long long)S * H * D16;
      for (long long i = (long long)blockIdx.x * NCT + ctid; i < n2; i += (long long)gridDim.x * NCT) {
        const int s = (int)(i / ((long long)H * D16));
        if (parts_of(s) == 0) reinterpret_cast<uint4*>(out)[i] = make_uint4(0, 0, 0, 0);
      }
      if (prm.lse) {  // no scores: the log-sum-exp is log 0
        for (int i = blockIdx.x * NCT + ctid; i < S * H; i += gridDim.x * NCT)
          if (parts_of(i / H) == 0) prm.lse[i] = -INFINITY;
      }
    }
  }

  C cons;
  uint32_t g = 0, k = 0;
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
      // (k-1)-th to be consumed).
      if (!wait_handover(prm, bar_eempty, k, abort_flag, err, kSiteHandEnd, lane)) break;
      if (warp == 0 && lane == 0) epi_info->s = -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_efull);
      break;
    }
    cons.begin_unit(reinterpret_cast<const T*>(smem + LY::OFF_Q + slot * LY::QSLOT), I.nh,
                    prm.scale_log2, lane, prm.G);
    if constexpr (C::kMma || MQ)
      cons.set_limits([&](int h) { return row_limit<MQ>(prm, I.L, I.h0 + h); }, lane);
    fence_proxy_async_smem();  // the query slot is refilled by a bulk copy: same ordering as a stage
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_uempty + 8 * slot);

    // Work item i of unit (p, hg) goes to warp (i + p * n_hg + hg) % NC: when
    // a unit's item count is not a multiple of NC, the extra items fall on
    // different warps from unit to unit instead of on warps 0, 1, ... every
    // time.  The grouping depends only on the partition and head group, never
    // on which CTA runs the unit or on the other sequences of the batch, so a
    // sequence's output is bitwise the same in any batch.  An item is one
    // block, or two consecutive blocks where the consumer says so
    // (kItemBlocks: one 16-token tile of 8-token blocks, or one softmax update
    // over two 16-token tiles).
    constexpr int PB = C::kItemBlocks;
    const int u_id = I.p * prm.n_hg + I.hg;
    const int nitem = (I.nb + PB - 1) / PB;
    for (int it = (warp + NC - u_id % NC) % NC; it < nitem; it += NC) {
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
          cons.block_pair(sa, sa + LY::VOFF, sb, sb + LY::VOFF, ntok, lane, I.t0 + j * BS);
        } else {
          cons.block(sa, sa + LY::VOFF, ntok, lane, scr, I.t0 + j * BS);
        }
      } else {
        cons.block(sa, sa + LY::VOFF, ntok, lane, scr, I.t0 + j * BS);
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
    // taken unit k-1's.
    if (!wait_handover(prm, bar_eempty, k, abort_flag, err, kSiteHandover, lane)) break;
    ++k;
    cons.finish(epi_acc + warp * GT * C::AROW, epi_ml + warp * GT * 2, lane);
    if (warp == 0 && lane == 0) *epi_info = I;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_efull);
  }
}

// Epilogue warp: for every unit, merge the consumer warps' states into the
// partition's (m_p, l_p, o_p) in the workspace, or, for a sequence with one
// partition, into the output and its log-sum-exp (single pass).
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
  float* rstat = reinterpret_cast<float*>(smem + LY::OFF_RSTAT);
  float* ef = reinterpret_cast<float*>(smem + LY::OFF_EF);  // [NC][GT] weights, then [GT] sums
  int* err = prm.hdr + kHdrError;
  const int H = prm.H, Pmax = prm.Pmax;
  T* out = static_cast<T*>(prm.out);
  // Partition states are read back by phase 2 right after this kernel: keep
  // them in L2 ahead of the streamed K/V (which is marked evict-first).
  const uint64_t pol_keep = l2_policy_evict_last();

  for (uint32_t k = 0;; ++k) {
    // Wait (bounded) for hand-over k, suspended in hardware between tries.
    bool ok = __all_sync(0xffffffffu, mbar_try_wait(bar_efull, k & 1u));
    if (!ok) {
      const uint64_t t0 = global_timer_ns();
      while (!ok) {
        ok = __all_sync(0xffffffffu, mbar_try_wait(bar_efull, k & 1u));
        if (ok) break;
        if (__any_sync(0xffffffffu, *abort_flag != 0)) return;
        if ((long long)(global_timer_ns() - t0) > prm.timeout_ns) {
          if (lane == 0) record_timeout(abort_flag, err, kSiteEpiFull, (int)k);
          return;
        }
      }
    }
    const UnitInfo I = *epi_info;
    if (I.s < 0) return;  // end of work
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
        const float4 v = reinterpret_cast<const float4*>(epi_acc + (w * GT + gh) * C::AROW)[d4];
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
        st_f4_policy(reinterpret_cast<float4*>(prm.ws_o + (sh * Pmax + I.p) * D) + d4, val, pol_keep);
      }
      if (d4 == 0) {
        st_f32_policy(prm.ws_m + sh * Pmax + I.p, rstat[gh * 2] * kLn2, pol_keep);
        st_f32_policy(prm.ws_l + sh * Pmax + I.p, ef[NC * GT + gh], pol_keep);
        // A single-partition sequence ends here: its log-sum-exp is the
        // merged maximum (log2 units -> natural) plus the log of the merged sum.
        if (single && prm.lse) prm.lse[out_row_rt(prm, I.s, I.h0 + gh)] = rstat[gh * 2] * kLn2 + logf(ef[NC * GT + gh]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_eempty);  // the hand-over slot may be refilled
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
  int* bad_len = reinterpret_cast<int*>(smem + LY::OFF_FLAGS + 16);  // a length out of range
  int* pref = reinterpret_cast<int*>(smem + LY::OFF_PREF);
  uint16_t* perm = reinterpret_cast<uint16_t*>(smem + LY::perm_off(prm.S));
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
    *bad_len = 0;
    fence_mbarrier_init();
  }
  // Longest-first order.  Every CTA computes the same order from the lengths:
  // perm[r] = the sequence of rank r, sequences sorted by partition count,
  // most first (counts of 127 or more as equals), ties in batch order (a
  // stable counting sort); pref[r] = partitions of ranks before r.  Lengths
  // are clamped to [0, MB*BS]; an out-of-range length is recorded as a device
  // error.  Temporaries live in the ring, unused until the producer starts.
  {
    constexpr int NW = LY::THREADS / 32;
    constexpr int NBK = 128;  // sort buckets
    static_assert(LY::THREADS % 32 == 0 && NW <= 32, "whole warps, at most 32");
    static_assert(LY::RING >= (NBK + kMaxSeqsPerLaunch + 2 * NW) * 4, "prologue temporaries fit in the ring");
    const int S = prm.S, nthr = LY::THREADS, max_len = prm.MB * C::BS;
    int* bucket = reinterpret_cast<int*>(smem);       // [NBK] counts, then next free rank
    int* parts = bucket + NBK;                          // [S] partitions per sequence
    int* scan = parts + kMaxSeqsPerLaunch;              // [2 * NW] warp totals, then warp starts
    for (int i = tid; i < NBK; i += nthr) bucket[i] = 0;
    __syncthreads();
    for (int s = tid; s < S; s += nthr) {
      bool bad = false;
      const int L = seq_tokens<MQ>(prm, s, max_len, &bad);
      if (bad) *bad_len = 1;
      const int np = (L + prm.P - 1) / prm.P;
      parts[s] = np;
      atomicAdd(&bucket[NBK - 1 - min(np, NBK - 1)], 1);
    }
    __syncthreads();
    if (warp == 0) {
      constexpr int PER = NBK / 32;  // buckets per lane: exclusive scan of the counts
      int v[PER], tot = 0;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        v[j] = bucket[lane * PER + j];
        tot += v[j];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      int start = incl - tot;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        bucket[lane * PER + j] = start;
        start += v[j];
      }
      __syncwarp();
      // 32 sequences at a time, in batch order: lanes with the same bucket
      // take consecutive ranks in lane order.
      for (int c0 = 0; c0 < S; c0 += 32) {
        const int s = c0 + lane;
        const int key = s < S ? NBK - 1 - min(parts[s], NBK - 1) : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int before = __popc(peers & ((1u << lane) - 1u));
        const int base = s < S ? bucket[key] : 0;
        __syncwarp();
        if (s < S) {
          perm[base + before] = (uint16_t)s;
          if (before == 0) bucket[key] = base + __popc(peers);
        }
        __syncwarp();
      }
    }
    __syncthreads();
    // pref over ranks: thread t sums a contiguous range of ranks; an exclusive
    // scan of those sums (within each warp, then over the warp totals).
    const int per = (S + nthr - 1) / nthr;
    const int beg = min(tid * per, S), end = min(beg + per, S);
    int sum = 0;
    for (int r = beg; r < end; ++r) sum += parts[perm[r]];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int t = lane < NW ? scan[lane] : 0;
      int ti = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, ti, o);
        if (lane >= o) ti += n;
      }
      if (lane < NW) scan[NW + lane] = ti - t;  // warp starts
      if (lane == NW - 1) pref[S] = ti;
    }
    __syncthreads();
    int run = scan[NW + warp] + incl - sum;
    for (int r = beg; r < end; ++r) {
      pref[r] = run;
      run += parts[perm[r]];
    }
  }
  __syncthreads();
  // This launch is a programmatic dependent of the kernel that clears the
  // workspace header: everything above overlaps it, nothing below may touch
  // the header before it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0 && *bad_len) atomicCAS(prm.hdr + kHdrError, 0, kErrDeviceBounds);
  if (warp == NC) {
    producer_loop<C, LY, MQ>(prm, smem, pref, perm, info, abort_flag, issued, lane);
  } else if (warp == NC + 1) {
    epilogue_loop<C, LY>(prm, smem, abort_flag, lane);
  } else {
    consumer_loop<C, LY, MQ>(prm, smem, info, abort_flag, issued, warp, lane);
  }
}

}  // namespace pa
