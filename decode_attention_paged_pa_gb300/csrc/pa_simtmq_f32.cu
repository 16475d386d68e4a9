// pa_simtmq_f32.cu -- multi-query instances of the paged decode kernel with
// the CUDA-core consumer's causal instances (one row head per pass, masked to
// its causal limit), element type float, head sizes 64/128/256 with blocks of
// 16 or 32 tokens.
#include "pa_launch.cuh"
#include "pa_simt.cuh"

namespace pa {

template <int D, int BS>
static cudaError_t go(const KParams& prm, int max_ctas, cudaStream_t st) {
  return launch_one<SimtConsumer<float, D, BS, 1, true>, kConsumerWarps>(prm, max_ctas, st);
}

cudaError_t launch_simt_mq_f32(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st) {
  if (D == 64) return BS == 16 ? go<64, 16>(prm, max_ctas, st) : go<64, 32>(prm, max_ctas, st);
  if (D == 128) return BS == 16 ? go<128, 16>(prm, max_ctas, st) : go<128, 32>(prm, max_ctas, st);
  return BS == 16 ? go<256, 16>(prm, max_ctas, st) : go<256, 32>(prm, max_ctas, st);
}

}  // namespace pa
