// pa_mma8g_bf16.cu -- instances of the paged decode kernel with the tensor-core
// (mma.sync) consumer over an fp8 (E4M3) KV cache and pairs of kv heads (4
// query heads per kv head: one unit's 8 columns hold two kv heads' query
// heads), queries and output __nv_bfloat16, head sizes 64 and 128.
#include "pa_launch.cuh"
#include "pa_mma.cuh"

namespace pa {

template <int D, int BS>
static cudaError_t go(const KParams& prm, int max_ctas, cudaStream_t st) {
  return launch_one<MmaConsumer<__nv_bfloat16, D, BS, true, 2>, mma8_consumer_warps<D>()>(prm, max_ctas, st);
}

cudaError_t launch_mma8_g_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st) {
  if (D == 64) return BS == 16 ? go<64, 16>(prm, max_ctas, st) : go<64, 32>(prm, max_ctas, st);
  return BS == 16 ? go<128, 16>(prm, max_ctas, st) : go<128, 32>(prm, max_ctas, st);
}

}  // namespace pa
