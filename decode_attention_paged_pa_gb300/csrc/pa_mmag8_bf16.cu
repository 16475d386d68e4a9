// pa_mmag8_bf16.cu -- instances of the paged decode kernel with the tensor-core
// (mma.sync) consumer over pairs of kv heads (4 query heads per kv head: one
// unit's 8 columns hold two kv heads' query heads), 8-token blocks, element
// type __nv_bfloat16, head sizes up to 128.
#include "pa_launch.cuh"
#include "pa_mma.cuh"

namespace pa {

template <int D>
static cudaError_t go(const KParams& prm, int max_ctas, cudaStream_t st) {
  return launch_one<MmaConsumer<__nv_bfloat16, D, 8, false, 2>, kMmaConsumerWarps>(prm, max_ctas, st);
}

cudaError_t launch_mma_g8_bf16(const KParams& prm, int D, int max_ctas, cudaStream_t st) {
  switch (D) {
    case 64: return go<64>(prm, max_ctas, st);
    case 80: return go<80>(prm, max_ctas, st);
    case 96: return go<96>(prm, max_ctas, st);
    case 112: return go<112>(prm, max_ctas, st);
    default: return go<128>(prm, max_ctas, st);
  }
}

}  // namespace pa
