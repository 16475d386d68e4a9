// pa_mma8b64_f16.cu -- instances of the paged decode kernel with the tensor-core
// (mma.sync) consumer over an fp8 (E4M3) KV cache in 64-token blocks (every
// supported head size), queries and output __half.
#include "pa_launch.cuh"
#include "pa_mma.cuh"

namespace pa {

template <int D>
static cudaError_t go(const KParams& prm, int max_ctas, cudaStream_t st) {
  return launch_one<MmaConsumer<__half, D, 64, true>, mma8_consumer_warps<D>()>(prm, max_ctas, st);
}

cudaError_t launch_mma8_b64_f16(const KParams& prm, int D, int max_ctas, cudaStream_t st) {
  switch (D) {
    case 64: return go<64>(prm, max_ctas, st);
    case 80: return go<80>(prm, max_ctas, st);
    case 96: return go<96>(prm, max_ctas, st);
    case 112: return go<112>(prm, max_ctas, st);
    case 128: return go<128>(prm, max_ctas, st);
    default: return go<256>(prm, max_ctas, st);
  }
}

}  // namespace pa
