// pa_mma16_f16.cu -- instances of the paged decode kernel with the tensor-core
// (mma.sync) consumer for units of 16 query rows of one kv head (the rows in
// the M = 16 side of the products), for groups of more than 8 query rows per
// kv head (head sizes 64 and 128: at 256 the accumulators no longer fit the
// registers), element type __half.
#include "pa_launch.cuh"
#include "pa_mma_rows.cuh"

namespace pa {

template <int D, int BS>
static cudaError_t go(const KParams& prm, int max_ctas, cudaStream_t st) {
  return launch_one<MmaRowConsumer<__half, D, BS>, kMmaConsumerWarps>(prm, max_ctas, st);
}

cudaError_t launch_mma16_f16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st) {
  if (D == 64) return BS == 16 ? go<64, 16>(prm, max_ctas, st) : go<64, 32>(prm, max_ctas, st);
  return BS == 16 ? go<128, 16>(prm, max_ctas, st) : go<128, 32>(prm, max_ctas, st);
}

}  // namespace pa
