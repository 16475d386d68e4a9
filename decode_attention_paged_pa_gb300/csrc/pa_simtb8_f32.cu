// pa_simtb8_f32.cu -- instances of the paged decode kernel with the CUDA-core
// consumer over fp32 caches in 8-token blocks (every supported head size),
// single-query and the causal instances of multi-query decode.
#include "pa_launch.cuh"
#include "pa_simt.cuh"

namespace pa {

template <int D, bool CAUSAL>
static cudaError_t go(const KParams& prm, int max_ctas, cudaStream_t st) {
  return launch_one<SimtConsumer<float, D, 8, 1, CAUSAL>, kConsumerWarps>(prm, max_ctas, st);
}

template <bool CAUSAL>
static cudaError_t by_d(const KParams& prm, int D, int max_ctas, cudaStream_t st) {
  switch (D) {
    case 64: return go<64, CAUSAL>(prm, max_ctas, st);
    case 80: return go<80, CAUSAL>(prm, max_ctas, st);
    case 96: return go<96, CAUSAL>(prm, max_ctas, st);
    case 112: return go<112, CAUSAL>(prm, max_ctas, st);
    case 128: return go<128, CAUSAL>(prm, max_ctas, st);
    default: return go<256, CAUSAL>(prm, max_ctas, st);
  }
}

cudaError_t launch_simt_b8_f32(const KParams& prm, int D, int max_ctas, cudaStream_t st) {
  return prm.q_len > 1 ? by_d<true>(prm, D, max_ctas, st) : by_d<false>(prm, D, max_ctas, st);
}

}  // namespace pa
