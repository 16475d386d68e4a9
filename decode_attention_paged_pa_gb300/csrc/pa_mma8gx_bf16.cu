// pa_mma8gx_bf16.cu -- instances of the paged decode kernel with the tensor-core
// (mma.sync) consumer over an fp8 (E4M3) KV cache and pairs of kv heads (4
// query heads per kv head) at head sizes 80, 96 and 112 with blocks of 16 or
// 32 tokens, queries and output __nv_bfloat16.
#include "pa_launch.cuh"
#include "pa_mma.cuh"

namespace pa {

template <int D, int BS>
static cudaError_t go(const KParams& prm, int max_ctas, cudaStream_t st) {
  return launch_one<MmaConsumer<__nv_bfloat16, D, BS, true, 2>, mma8_consumer_warps<D>()>(prm, max_ctas, st);
}

template <int BS>
static cudaError_t by_d(const KParams& prm, int D, int max_ctas, cudaStream_t st) {
  if (D == 80) return go<80, BS>(prm, max_ctas, st);
  if (D == 96) return go<96, BS>(prm, max_ctas, st);
  return go<112, BS>(prm, max_ctas, st);
}

cudaError_t launch_mma8_gx_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st) {
  return BS == 16 ? by_d<16>(prm, D, max_ctas, st) : by_d<32>(prm, D, max_ctas, st);
}

}  // namespace pa
