// pa_launch.h -- internal interface between the C ABI (pa_api.cu) and the
// kernel instantiation units.
#pragma once

#include <cuda_runtime.h>

#include "pa_combine.cuh"
#include "pa_kernel.cuh"

namespace pa {

// Query heads per work unit of each kernel family (the tensor-core family
// takes 16 where a kv head has more than 8 query rows).
constexpr int kSimtGroup = 1;
constexpr int kMmaGroup = 8;
constexpr int kMmaGroupWide = 16;

// Launch the persistent kernel for one chunk of sequences.  Returns a cudaError_t.
cudaError_t launch_simt_f16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_simt_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_simt_f32(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
// CUDA-core instances of head sizes 80, 96, 112 (blocks of 16, 32, 64) and of
// 64-token blocks at head sizes 64, 128 (fp16 / bf16).
cudaError_t launch_simtx_f16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_simtx_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_simtx_f32(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
// Multi-query rows with fp32 elements: the causal instances, base and further shapes.
cudaError_t launch_simt_mq_f32(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_simtx_mq_f32(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
// fp32 caches in 8-token blocks, single- and multi-query.
cudaError_t launch_simt_b8_f32(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_f16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma16_f16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma16_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
// Tensor-core instances of the other shapes: head sizes 80, 96, 112 (block
// sizes 16, 32), and 8- or 64-token blocks (head sizes 64, 80, 96, 112, 128, 256).
cudaError_t launch_mma_xd_f16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_xd_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_b8_f16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_b8_bf16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_b64_f16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_b64_bf16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
// Tensor-core instances over pairs of kv heads (4 query heads per kv head,
// head sizes up to 128), in 8-, 16- and 32-token blocks.
cudaError_t launch_mma_g8_f16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_g8_bf16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_g16_f16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_g16_bf16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_g32_f16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma_g32_bf16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
// The same over an fp8 (E4M3) KV cache, queries and output fp16 / bf16.
cudaError_t launch_mma8_f16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
// (head sizes 64, 128, 256 with 16- or 32-token blocks), at head sizes 80, 96,
// 112 with 16- or 32-token blocks (_x), and in 8- or 64-token blocks (_b8, _b64).
cudaError_t launch_mma8_x_f16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_x_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_b8_f16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_b8_bf16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_b64_f16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_b64_bf16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
// ... and over pairs of kv heads (4 query heads per kv head): head sizes 64
// and 128 with 16- or 32-token blocks, 80, 96, 112 with 16- or 32-token
// blocks (_gx), and every head size up to 128 in 8-token blocks (_gb8).
cudaError_t launch_mma8_g_f16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_g_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_gx_f16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_gx_bf16(const KParams& prm, int D, int BS, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_gb8_f16(const KParams& prm, int D, int max_ctas, cudaStream_t st);
cudaError_t launch_mma8_gb8_bf16(const KParams& prm, int D, int max_ctas, cudaStream_t st);

// Phase 2: the cross-partition combine of every multi-partition row, launched
// as a programmatic dependent of the phase-1 launch before it on `st`.
cudaError_t launch_combine(const CParams& prm, int elem_bytes, bool bf16, int D, cudaStream_t st);

// SM count of the current device (cached per device).
int device_sm_count();

}  // namespace pa
