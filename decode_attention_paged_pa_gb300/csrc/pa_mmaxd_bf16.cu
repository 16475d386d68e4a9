// pa_mmaxd_bf16.cu -- instances of the paged decode kernel with the tensor-core
// (mma.sync) consumer for head sizes 80, 96 and 112 (block sizes 16 and 32),
// element type __nv_bfloat16.
#include "pa_launch.cuh"
#include "pa_mma.cuh"

namespace pa {

template <int D, int BS>
static cudaError_t go(const KParams& prm, int max_ctas, cudaStream_t st) {
  return launch_one<MmaConsumer<__nv_bfloat16, D, BS>, kMmaConsumerWarps>(prm, max_ctas, st);
}

template <int BS>
static cudaError_t by_d(const KParams& prm, int D, int max_ctas, cudaStream_t st) {
  if (D == 80) return go<80, BS>(prm, max_ctas, st);
  if (D == 96) return go<96, BS>(prm, max_ctas, st);
  return go<112, BS>(prm, max_ctas, st);
}

cudaError_t launch_mma_xd_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st) {
  return BS == 16 ? by_d<16>(prm, D, max_ctas, st) : by_d<32>(prm, D, max_ctas, st);
}

}  // namespace pa
