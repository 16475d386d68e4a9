// pa_simtmqx_f32.cu -- multi-query instances of the paged decode kernel with
// the CUDA-core consumer's causal instances, element type float, at the
// shapes beyond 64/128/256 x 16/32 (as pa_simtx_f32.cu).
#include "pa_launch.cuh"
#include "pa_simt.cuh"

namespace pa {

template <int D, int BS>
static cudaError_t go(const KParams& prm, int max_ctas, cudaStream_t st) {
  return launch_one<SimtConsumer<float, D, BS, 1, true>, kConsumerWarps>(prm, max_ctas, st);
}

template <int D>
static cudaError_t by_bs(const KParams& prm, int BS, int max_ctas, cudaStream_t st) {
  if (BS == 16) return go<D, 16>(prm, max_ctas, st);
  if (BS == 32) return go<D, 32>(prm, max_ctas, st);
  return go<D, 64>(prm, max_ctas, st);
}

cudaError_t launch_simtx_mq_f32(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st) {
  switch (D) {
    case 80: return by_bs<80>(prm, BS, max_ctas, st);
    case 96: return by_bs<96>(prm, BS, max_ctas, st);
    case 112: return by_bs<112>(prm, BS, max_ctas, st);
    case 64: return go<64, 64>(prm, max_ctas, st);
    default: return go<128, 64>(prm, max_ctas, st);
  }
}

}  // namespace pa
