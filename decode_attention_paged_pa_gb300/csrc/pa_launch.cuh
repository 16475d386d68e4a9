// pa_launch.cuh -- shared-memory sizing and launch of one kernel instance.
#pragma once

#include <atomic>

#include "pa_launch.h"

namespace pa {

// Consumer warps per CTA and CTAs per SM.
#ifndef PA_CONSUMER_WARPS
#define PA_CONSUMER_WARPS 8
#endif
#ifndef PA_CTAS_PER_SM
#define PA_CTAS_PER_SM 1
#endif
constexpr int kConsumerWarps = PA_CONSUMER_WARPS;
// The tensor-core kernel's consumer warps: six (eight warps in all) leave
// each thread up to 255 registers (ten warps cap it at 168 by the SM
// sub-partitions' register files) and shrink the hand-over buffer, which
// lengthens the ring.
#ifndef PA_MMA_CONSUMER_WARPS
#define PA_MMA_CONSUMER_WARPS 6
#endif
constexpr int kMmaConsumerWarps = PA_MMA_CONSUMER_WARPS;
// Over an fp8 KV cache a block carries half the bytes for the same
// arithmetic, and the consumer warps' latency sets the pace: eight of them
// where their registers fit under the ten-warp cap (D <= 128), six otherwise.
template <int D>
constexpr int mma8_consumer_warps() {
  return D <= 128 ? 8 : 6;
}
constexpr int kCtasPerSm = PA_CTAS_PER_SM;

// Shared memory per CTA: the SM's 228 KB less 1 KB reserved per CTA.
constexpr uint32_t kSmemBudget = (kCtasPerSm == 1) ? 227u * 1024u : (228u * 1024u / kCtasPerSm - 1024u);

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }

// Ring depth: as many K+V stages as fit next to the fixed regions and the
// largest per-launch order and prefix arrays.  Each stage beyond the first
// adds its bytes and two 8-byte mbarriers (both multiples of 16, so no
// alignment in the layout moves).
template <class C, int NC>
struct Sizing {
  using L1 = Layout<C, NC, 1>;
  static_assert(L1::STAGE % 16 == 0, "stages are whole 16-byte units");
  static constexpr uint32_t base = L1::bytes(kMaxSeqsPerLaunch);
  static_assert(base <= kSmemBudget, "shared memory over budget");
  static constexpr int NS = cmin(64, 1 + (int)((kSmemBudget - base) / (L1::STAGE + 16)));
  static_assert(NS >= 2, "shared memory holds fewer than two ring stages");
  using LY = Layout<C, NC, NS>;
  static_assert(LY::bytes(kMaxSeqsPerLaunch) <= kSmemBudget, "shared memory over budget");
  static_assert(NS == 64 || Layout<C, NC, NS + 1>::bytes(kMaxSeqsPerLaunch) > kSmemBudget, "ring as deep as fits");
};

template <class C, int NC>
cudaError_t launch_one(const KParams& prm, int max_ctas, cudaStream_t stream) {
  using SZ = Sizing<C, NC>;
  using LY = typename SZ::LY;
  // Multi-query rows run on the tensor-core consumer, and on the CUDA-core
  // consumer's causal instances (fp32); those have no single-query kernel.
  void (*kern)(KParams) = nullptr;
  if constexpr (C::kMma) {
    kern = prm.q_len > 1 ? pa_decode_kernel<C, NC, SZ::NS, kCtasPerSm, true>
                         : pa_decode_kernel<C, NC, SZ::NS, kCtasPerSm, false>;
  } else if constexpr (C::kCausal) {
    if (prm.q_len <= 1) return cudaErrorInvalidValue;
    kern = pa_decode_kernel<C, NC, SZ::NS, kCtasPerSm, true>;
  } else {
    if (prm.q_len > 1) return cudaErrorInvalidValue;
    kern = pa_decode_kernel<C, NC, SZ::NS, kCtasPerSm, false>;
  }
  // The shared-memory opt-in is set once per kernel instance and device.
  static std::atomic<uint64_t> opted_in[2] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int mq = prm.q_len > 1 ? 1 : 0;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (!bit || !(opted_in[mq].load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::bytes(kMaxSeqsPerLaunch));
    if (e != cudaSuccess) return e;
    opted_in[mq].fetch_or(bit, std::memory_order_acq_rel);
  }
  int grid = device_sm_count() * kCtasPerSm;
  if (max_ctas > 0 && max_ctas < grid) grid = max_ctas;
  if (grid < 1) grid = 1;
  // A programmatic dependent of the header-clearing kernel just before it.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(LY::THREADS, 1, 1);
  cfg.dynamicSmemBytes = LY::bytes(prm.S);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace pa
