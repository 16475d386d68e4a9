// pa_simt_bf16.cu -- instances of the paged decode kernel with the CUDA-core
// consumer, element type __nv_bfloat16.
#include "pa_launch.cuh"
#include "pa_simt.cuh"

namespace pa {

template <int D, int BS, int GT>
static cudaError_t go(const KParams& prm, int max_ctas, cudaStream_t st) {
  return launch_one<SimtConsumer<__nv_bfloat16, D, BS, GT>, 4>(prm, max_ctas, st);
}

template <int D, int BS>
static cudaError_t by_gt(const KParams& prm, int gt, int max_ctas, cudaStream_t st) {
  return gt == 1 ? go<D, BS, 1>(prm, max_ctas, st) : go<D, BS, 2>(prm, max_ctas, st);
}

cudaError_t launch_simt_bf16(const KParams& prm, int D, int BS, int gt, int max_ctas, cudaStream_t st) {
  if (D == 64) return BS == 16 ? by_gt<64, 16>(prm, gt, max_ctas, st) : by_gt<64, 32>(prm, gt, max_ctas, st);
  if (D == 128) return BS == 16 ? by_gt<128, 16>(prm, gt, max_ctas, st) : by_gt<128, 32>(prm, gt, max_ctas, st);
  return BS == 16 ? by_gt<256, 16>(prm, gt, max_ctas, st) : by_gt<256, 32>(prm, gt, max_ctas, st);
}

}  // namespace pa
