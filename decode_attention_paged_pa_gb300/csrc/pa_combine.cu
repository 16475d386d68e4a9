// pa_combine.cu -- launches of the phase-2 combine kernel (pa_combine.cuh), one
// instance per output element type and head size.
#include "pa_combine.cuh"
#include "pa_launch.h"

namespace pa {

namespace {

template <typename T, int D>
cudaError_t go(const CParams& prm, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  // A programmatic dependent of the phase-1 launch just before it on the
  // stream: it may start as soon as every phase-1 CTA has run out of work,
  // and waits (griddepcontrol.wait) for phase 1 to complete before it reads.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (prm.S <= kRowsMaxSeqs && prm.Pmax > 16) {
    // Rows that a single warp would take in two batches or more: one
    // persistent CTA per SM (no more than the batch's rows could need).  With
    // short rows only, the per-sequence grid is as good (its CTAs, 8 rows of
    // one warp each, are short) and the persistent one lost 0.2-0.9%.
    const long long rows = (long long)prm.S * prm.H;
    const int sms = device_sm_count();
    cfg.gridDim = dim3((unsigned)(rows < sms ? rows : sms), 1, 1);
    cfg.blockDim = dim3(kRowsWarps * 32, 1, 1);
    return cudaLaunchKernelEx(&cfg, pa_combine_rows_kernel<T, D>, prm);
  }
  // CTAs of 4 warps where a row takes at most 4 (five CTAs of a 98-register
  // kernel fit an SM where two of 8 warps did: 20 warps in flight, not 16).
  const int nw = prm.wpr <= 4 ? 4 : kCombineWarps;
  const int rpc = nw / prm.wpr;
  cfg.gridDim = dim3((unsigned)prm.S, (unsigned)((prm.H + rpc - 1) / rpc), 1);
  cfg.blockDim = dim3(nw * 32, 1, 1);
  if (nw == 4) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<T, D, 4>, prm);
  return cudaLaunchKernelEx(&cfg, pa_combine_kernel<T, D, kCombineWarps>, prm);
}

template <typename T>
cudaError_t by_head_size(const CParams& prm, int D, cudaStream_t st) {
  switch (D) {
    case 64: return go<T, 64>(prm, st);
    case 80: return go<T, 80>(prm, st);
    case 96: return go<T, 96>(prm, st);
    case 112: return go<T, 112>(prm, st);
    case 128: return go<T, 128>(prm, st);
    case 256: return go<T, 256>(prm, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_combine(const CParams& prm, int elem_bytes, bool bf16, int D, cudaStream_t st) {
  if (elem_bytes == 4) return by_head_size<float>(prm, D, st);
  return bf16 ? by_head_size<__nv_bfloat16>(prm, D, st) : by_head_size<__half>(prm, D, st);
}

}  // namespace pa
