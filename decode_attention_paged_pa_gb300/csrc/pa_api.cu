// pa_api.cu -- C ABI of the paged decode attention library (include/pa_decode.h):
// argument validation, workspace layout, kernel-family choice and launches.
#include <climits>
#include <cstdint>
#include <cstring>

#include "pa_decode.h"
#include "pa_launch.h"

namespace pa {

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) {
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
  }
  if (cache[dev] == 0) {
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n;
  }
  return cache[dev];
}

// Clears header words [first, first + count) of the workspace before a phase-1
// launch.  It is itself launched as a programmatic dependent of whatever
// precedes it on the stream, so its launch overlaps that work's end: it first
// waits for that work to complete (its writes -- the caller's inputs among
// them -- visible), and only then lets phase 1, its own programmatic
// dependent, be scheduled; phase 1 waits for this kernel before it touches
// the header.
__global__ void __launch_bounds__(64) pa_clear_header_kernel(int* hdr, int first, int count) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = threadIdx.x; i < count; i += blockDim.x) hdr[first + i] = 0;
}

// The header clear, launched as described above.
static cudaError_t launch_clear_header(int* hdr, int first, int count, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(64, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pa_clear_header_kernel, hdr, first, count);
}

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct WsLayout {
  size_t hdr, m, l, o, total;
  int pmax;
};

bool valid_sizes(int S, int H, int KH, int D, int MB, int BS, int P) {
  if (S < 0 || H <= 0 || KH <= 0 || H % KH != 0 || MB <= 0 || BS <= 0 || P <= 0 || D <= 0) return false;
  if ((long long)MB * BS > INT_MAX / 2) return false;
  return true;
}

size_t elem_bytes(int dtype) { return dtype == PA_DTYPE_FP32 ? 4 : 2; }

// Shapes every kernel family handles; the tensor-core family also takes head
// sizes 80, 96, 112 and 8- or 64-token blocks.
bool base_shape(int D, int BS) {
  return (D == 64 || D == 128 || D == 256) && (BS == 16 || BS == 32);
}

// The CUDA-core family's further shapes: head sizes 80, 96, 112 with
// blocks of 16, 32 or 64 tokens, and 64-token blocks at head sizes 64, 128.
bool simt_extra_shape(int D, int BS) {
  return ((D == 80 || D == 96 || D == 112) && (BS == 16 || BS == 32 || BS == 64)) ||
         ((D == 64 || D == 128) && BS == 64);
}

bool supported(int D, int BS, int P) {
  const bool d_ok = D == 64 || D == 80 || D == 96 || D == 112 || D == 128 || D == 256;
  const bool bs_ok = BS == 8 || BS == 16 || BS == 32 || BS == 64;
  return d_ok && bs_ok && P % BS == 0;
}

bool ws_layout(int S, int H, int KH, int D, int MB, int BS, int P, WsLayout* w) {
  if (!valid_sizes(S, H, KH, D, MB, BS, P)) return false;
  const long long pmax = ((long long)MB * BS + P - 1) / P;
  if (pmax > INT_MAX) return false;
  w->pmax = (int)pmax;
  const size_t shp = (size_t)S * H * (size_t)pmax;
  w->hdr = 0;
  w->m = align_up(kHdrInts * sizeof(int));
  w->l = align_up(w->m + shp * sizeof(float));
  w->o = align_up(w->l + shp * sizeof(float));
  w->total = align_up(w->o + shp * (size_t)D * sizeof(float));
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link the driver library itself).
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// Tensor map of a 16-bit paged value cache for the tensor-core kernels:
// value_cache [NB, KH, D, BS] as a 3-D tensor [NB*KH][D][BS] with a box of one
// whole block ([1][D][BS]), stored in shared memory in the swizzle of the
// rows' width (BS * 2 bytes: 32, 64 or 128).
// kvu: kv heads per box (the unit's consecutive kv heads of one block).
bool encode_value_map(KParams* prm, const void* value_cache, int num_blocks, int KH, int D, int BS, int kvu) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const CUtensorMapSwizzle sw = BS == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                                : BS == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : CU_TENSOR_MAP_SWIZZLE_128B;
  const cuuint32_t unit[3] = {1, 1, 1};
  const cuuint64_t vdim[3] = {(cuuint64_t)BS, (cuuint64_t)D, (cuuint64_t)num_blocks * (cuuint64_t)KH};
  const cuuint64_t vstride[2] = {(cuuint64_t)BS * 2, (cuuint64_t)D * BS * 2};
  const cuuint32_t vbox[3] = {(cuuint32_t)BS, (cuuint32_t)D, (cuuint32_t)kvu};
  return enc(&prm->tmv, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(value_cache), vdim, vstride, vbox,
             unit, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_v2_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                               int head_size, int max_blocks_per_seq, int block_size,
                                               int partition_size) {
  WsLayout w;
  if (!ws_layout(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq, block_size,
                 partition_size, &w))
    return 0;
  return w.total;
}

extern "C" int pa_decode_v2_workspace_layout(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                             int max_blocks_per_seq, int block_size, int partition_size,
                                             size_t offsets[5], int* max_partitions) {
  WsLayout w;
  if (!offsets || !ws_layout(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq,
                             block_size, partition_size, &w))
    return PA_ERR_INVALID_ARG;
  offsets[0] = w.m;
  offsets[1] = w.l;
  offsets[2] = w.o;
  offsets[3] = w.hdr;
  offsets[4] = w.total;
  if (max_partitions) *max_partitions = w.pmax;
  return PA_OK;
}

namespace {

int decode_impl(void* out, float* lse, const void* query, const void* key_cache,
                const void* value_cache, const int32_t* block_tables, const int32_t* seq_lens,
                float scale, int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_size,
                int block_size, int partition_size, int dtype, void* stream, int max_blocks_per_seq,
                int num_blocks, void* workspace, size_t workspace_bytes, int variant, int max_ctas,
                long long timeout_ns, bool kv_fp8 = false, float k_scale = 1.f, float v_scale = 1.f) {
  // Multi-query: the kernel sees q_len "row heads" per caller head (H below
  // counts them), q_len * G per kv head, all sharing the kv head's blocks.
  if (q_len < 1 || q_len > kMaxSeqsPerLaunch || num_heads <= 0 ||
      (long long)num_heads * q_len > 65535)
    return PA_ERR_INVALID_ARG;
  const int S = num_seqs, H = num_heads * q_len, KH = num_kv_heads, D = head_size, BS = block_size,
            P = partition_size, MB = max_blocks_per_seq;
  if (!valid_sizes(S, H, KH, D, MB, BS, P) || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (dtype != PA_DTYPE_FP16 && dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_FP32) return PA_ERR_INVALID_ARG;
  if (variant < PA_VARIANT_AUTO || variant > PA_VARIANT_MMA || max_ctas < 0 || timeout_ns < 0)
    return PA_ERR_INVALID_ARG;
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return PA_ERR_INVALID_ARG;
  if (!(k_scale == k_scale) || k_scale == INFINITY || k_scale == -INFINITY || !(v_scale == v_scale) ||
      v_scale == INFINITY || v_scale == -INFINITY)
    return PA_ERR_INVALID_ARG;
  if (!supported(D, BS, P)) return PA_ERR_UNSUPPORTED;
  if (kv_fp8 && variant == PA_VARIANT_SIMT) return PA_ERR_UNSUPPORTED;  // fp8 runs on tensor cores
  // (8-token blocks on the CUDA cores: fp32 only; the 16-bit types take the tensor cores there.)
  const bool simt_ok = base_shape(D, BS) || simt_extra_shape(D, BS) || (dtype == PA_DTYPE_FP32 && BS == 8);
  if (variant == PA_VARIANT_SIMT && !simt_ok) return PA_ERR_UNSUPPORTED;
  // fp32 runs on the CUDA-core family only (its shapes; multi-query rows on
  // its causal instances).
  if (dtype == PA_DTYPE_FP32 && (kv_fp8 || variant == PA_VARIANT_MMA || !simt_ok))
    return PA_ERR_UNSUPPORTED;
  if (S == 0) return PA_OK;
  if (!out || !query || !key_cache || !value_cache || !block_tables || !seq_lens)
    return PA_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(query, 16) || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || !aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
      (workspace && !aligned(workspace, 16)) || (lse && !aligned(lse, 4)))
    return PA_ERR_INVALID_ARG;
  WsLayout w;
  if (!ws_layout(S, H, KH, D, MB, BS, P, &w)) return PA_ERR_INVALID_ARG;
  if (workspace && workspace_bytes < w.total) return PA_ERR_WORKSPACE;

  const int G = H / KH;
  if (variant == PA_VARIANT_AUTO)
    variant = ((G == 1 || dtype == PA_DTYPE_FP32) && !kv_fp8 && simt_ok) ? PA_VARIANT_SIMT : PA_VARIANT_MMA;
  // More than 8 query rows per kv head: the tensor-core instances for units
  // of 16 rows (the rows on the M side of the products) read each K/V block
  // once for 16 rows (head sizes 64 and 128, blocks of 16 or 32 tokens,
  // 16-bit caches).
  const bool wide = variant == PA_VARIANT_MMA && G > kMmaGroup && !kv_fp8 && D <= 128 &&
                    base_shape(D, BS);
  const int gt = (variant == PA_VARIANT_MMA) ? (wide ? kMmaGroupWide : kMmaGroup) : kSimtGroup;
  // Four query rows per kv head (query heads, or multi-query row heads): a
  // unit's 8 columns take two kv heads (one block copy each for keys and
  // values covers both), head sizes up to 128 and blocks of 8, 16 or 32 tokens.
  const bool pairs = variant == PA_VARIANT_MMA && !wide && G * 2 == kMmaGroup && KH % 2 == 0 &&
                     D <= 128 && (BS == 8 || BS == 16 || BS == 32);
  const int kvu = pairs ? 2 : 1;
  const int hg_per_kv = (G + gt - 1) / gt;
  const int n_hg = KH * hg_per_kv / kvu;
  const int rows_per_launch = kMaxSeqsPerLaunch;  // sequences per launch
  const int chunk = S < rows_per_launch ? S : rows_per_launch;
  if ((long long)chunk * w.pmax * n_hg > INT_MAX / 2) return PA_ERR_UNSUPPORTED;
  // The tensor-core kernels over 16-bit caches in blocks of 16 tokens or more
  // stage value blocks by swizzled tensor copies (z coordinates are int32).
  const bool tma_values = variant == PA_VARIANT_MMA && !kv_fp8 && BS >= 16;
  KParams maps;
  std::memset(&maps, 0, sizeof maps);
  if (tma_values) {
    if ((long long)num_blocks * KH > INT_MAX) return PA_ERR_UNSUPPORTED;
    if (!encode_value_map(&maps, value_cache, num_blocks, KH, D, BS, kvu)) return PA_ERR_CUDA;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  bool own = false;
  if (!ws) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&ws), w.total, st) != cudaSuccess) return PA_ERR_CUDA;
    own = true;
  }
  int status = PA_OK;
  const size_t esz = elem_bytes(dtype);
  for (int s0 = 0; s0 < S && status == PA_OK; s0 += rows_per_launch) {
    const int n = (S - s0) < rows_per_launch ? (S - s0) : rows_per_launch;
    // The header (error word, work counter, timeout record) starts at zero;
    // a later launch of the same call restarts the work counter only.
    if (launch_clear_header(reinterpret_cast<int*>(ws + w.hdr), s0 == 0 ? 0 : kHdrWork,
                            s0 == 0 ? kHdrInts : 1, st) != cudaSuccess) {
      status = PA_ERR_CUDA;
      break;
    }
    KParams prm;
    std::memset(&prm, 0, sizeof prm);
    prm.tmv = maps.tmv;
    prm.out = static_cast<uint8_t*>(out) + (size_t)s0 * H * D * esz;
    prm.q = static_cast<const uint8_t*>(query) + (size_t)s0 * H * D * esz;
    prm.kc = key_cache;
    prm.vc = value_cache;
    prm.bt = block_tables + (size_t)s0 * MB;
    prm.lens = seq_lens + s0;
    prm.q_len = q_len;
    prm.Hu = num_heads;
    prm.Gu = num_heads / KH;
    prm.ws_m = reinterpret_cast<float*>(ws + w.m) + (size_t)s0 * H * w.pmax;
    prm.ws_l = reinterpret_cast<float*>(ws + w.l) + (size_t)s0 * H * w.pmax;
    prm.ws_o = reinterpret_cast<float*>(ws + w.o) + (size_t)s0 * H * w.pmax * D;
    prm.hdr = reinterpret_cast<int*>(ws + w.hdr);
    prm.lse = lse ? lse + (size_t)s0 * H : nullptr;
    prm.scale_log2 = scale * k_scale * kLog2e;
    prm.v_scale = v_scale;
    prm.S = n;
    prm.H = H;
    prm.KH = KH;
    prm.G = G;
    prm.MB = MB;
    prm.num_blocks = num_blocks;
    prm.P = P;
    prm.Pmax = w.pmax;
    prm.hg_per_kv = hg_per_kv;
    prm.n_hg = n_hg;
    prm.timeout_ns = timeout_ns > 0 ? timeout_ns : (1LL << 31);
    cudaError_t e;
    if (kv_fp8 && pairs && BS == 8)
      e = dtype == PA_DTYPE_FP16 ? launch_mma8_gb8_f16(prm, D, max_ctas, st)
                                 : launch_mma8_gb8_bf16(prm, D, max_ctas, st);
    else if (kv_fp8 && pairs && (D == 64 || D == 128))
      e = dtype == PA_DTYPE_FP16 ? launch_mma8_g_f16(prm, D, BS, max_ctas, st)
                                 : launch_mma8_g_bf16(prm, D, BS, max_ctas, st);
    else if (kv_fp8 && pairs)
      e = dtype == PA_DTYPE_FP16 ? launch_mma8_gx_f16(prm, D, BS, max_ctas, st)
                                 : launch_mma8_gx_bf16(prm, D, BS, max_ctas, st);
    else if (kv_fp8 && BS == 8)
      e = dtype == PA_DTYPE_FP16 ? launch_mma8_b8_f16(prm, D, max_ctas, st)
                                 : launch_mma8_b8_bf16(prm, D, max_ctas, st);
    else if (kv_fp8 && BS == 64)
      e = dtype == PA_DTYPE_FP16 ? launch_mma8_b64_f16(prm, D, max_ctas, st)
                                 : launch_mma8_b64_bf16(prm, D, max_ctas, st);
    else if (kv_fp8 && base_shape(D, BS))
      e = dtype == PA_DTYPE_FP16 ? launch_mma8_f16(prm, D, BS, max_ctas, st)
                                 : launch_mma8_bf16(prm, D, BS, max_ctas, st);
    else if (kv_fp8)
      e = dtype == PA_DTYPE_FP16 ? launch_mma8_x_f16(prm, D, BS, max_ctas, st)
                                 : launch_mma8_x_bf16(prm, D, BS, max_ctas, st);
    else if (wide)
      e = dtype == PA_DTYPE_FP16 ? launch_mma16_f16(prm, D, BS, max_ctas, st)
                                 : launch_mma16_bf16(prm, D, BS, max_ctas, st);
    else if (pairs && BS == 8)
      e = dtype == PA_DTYPE_FP16 ? launch_mma_g8_f16(prm, D, max_ctas, st) : launch_mma_g8_bf16(prm, D, max_ctas, st);
    else if (pairs && BS == 16)
      e = dtype == PA_DTYPE_FP16 ? launch_mma_g16_f16(prm, D, max_ctas, st) : launch_mma_g16_bf16(prm, D, max_ctas, st);
    else if (pairs)
      e = dtype == PA_DTYPE_FP16 ? launch_mma_g32_f16(prm, D, max_ctas, st) : launch_mma_g32_bf16(prm, D, max_ctas, st);
    else if (variant == PA_VARIANT_MMA && BS == 8)
      e = dtype == PA_DTYPE_FP16 ? launch_mma_b8_f16(prm, D, max_ctas, st)
                                 : launch_mma_b8_bf16(prm, D, max_ctas, st);
    else if (variant == PA_VARIANT_MMA && BS == 64)
      e = dtype == PA_DTYPE_FP16 ? launch_mma_b64_f16(prm, D, max_ctas, st)
                                 : launch_mma_b64_bf16(prm, D, max_ctas, st);
    else if (variant == PA_VARIANT_MMA && !base_shape(D, BS))
      e = dtype == PA_DTYPE_FP16 ? launch_mma_xd_f16(prm, D, BS, max_ctas, st)
                                 : launch_mma_xd_bf16(prm, D, BS, max_ctas, st);
    else if (variant == PA_VARIANT_MMA)
      e = dtype == PA_DTYPE_FP16 ? launch_mma_f16(prm, D, BS, max_ctas, st)
                                 : launch_mma_bf16(prm, D, BS, max_ctas, st);
    else if (dtype == PA_DTYPE_FP32 && BS == 8)
      e = launch_simt_b8_f32(prm, D, max_ctas, st);
    else if (dtype == PA_DTYPE_FP32 && q_len > 1)
      e = base_shape(D, BS) ? launch_simt_mq_f32(prm, D, BS, max_ctas, st)
                            : launch_simtx_mq_f32(prm, D, BS, max_ctas, st);
    else if (dtype == PA_DTYPE_FP32)
      e = base_shape(D, BS) ? launch_simt_f32(prm, D, BS, max_ctas, st)
                            : launch_simtx_f32(prm, D, BS, max_ctas, st);
    else if (!base_shape(D, BS))
      e = dtype == PA_DTYPE_FP16 ? launch_simtx_f16(prm, D, BS, max_ctas, st)
                                 : launch_simtx_bf16(prm, D, BS, max_ctas, st);
    else
      e = dtype == PA_DTYPE_FP16 ? launch_simt_f16(prm, D, BS, max_ctas, st)
                                 : launch_simt_bf16(prm, D, BS, max_ctas, st);
    if (e != cudaSuccess) status = PA_ERR_CUDA;
  }
  // Phase 2 over the whole batch (no sequence has more than one partition if
  // the table holds at most P tokens).  Warps per row: enough that a warp
  // takes at most 16 partitions (one batch of loads), up to 8.
  if (status == PA_OK && w.pmax > 1) {
    CParams cp;
    std::memset(&cp, 0, sizeof cp);
    cp.out = out;
    cp.lse = lse;
    cp.ws_m = reinterpret_cast<const float*>(ws + w.m);
    cp.ws_l = reinterpret_cast<const float*>(ws + w.l);
    cp.ws_o = reinterpret_cast<const float*>(ws + w.o);
    cp.lens = seq_lens;
    cp.S = S;
    cp.H = H;
    cp.Pmax = w.pmax;
    cp.P = P;
    cp.max_len = MB * BS;
    cp.wpr = w.pmax > 64 ? 8 : w.pmax > 32 ? 4 : w.pmax > 16 ? 2 : 1;
    cp.q_len = q_len;
    cp.Hu = num_heads;
    cp.Gu = num_heads / KH;
    cp.G = G;
    if (launch_combine(cp, (int)esz, dtype == PA_DTYPE_BF16, D, st) != cudaSuccess) status = PA_ERR_CUDA;
  }
  if (own && cudaFreeAsync(ws, st) != cudaSuccess && status == PA_OK) status = PA_ERR_CUDA;
  return status;
}

}  // namespace

extern "C" int pa_decode_v2_ex(void* out, const void* query, const void* key_cache,
                               const void* value_cache, const int32_t* block_tables,
                               const int32_t* seq_lens, float scale, int num_seqs, int num_heads,
                               int num_kv_heads, int head_size, int block_size, int partition_size,
                               int dtype, void* stream, int max_blocks_per_seq, int num_blocks,
                               void* workspace, size_t workspace_bytes, int variant, int max_ctas,
                               long long timeout_ns) {
  return decode_impl(out, nullptr, query, key_cache, value_cache, block_tables, seq_lens, scale,
                     num_seqs, 1, num_heads, num_kv_heads, head_size, block_size, partition_size,
                     dtype, stream, max_blocks_per_seq, num_blocks, workspace, workspace_bytes,
                     variant, max_ctas, timeout_ns);
}

extern "C" int pa_decode_v2_lse(void* out, float* lse, const void* query, const void* key_cache,
                                const void* value_cache, const int32_t* block_tables,
                                const int32_t* seq_lens, float scale, int num_seqs, int num_heads,
                                int num_kv_heads, int head_size, int block_size, int partition_size,
                                int dtype, void* stream, int max_blocks_per_seq, int num_blocks,
                                void* workspace, size_t workspace_bytes) {
  return decode_impl(out, lse, query, key_cache, value_cache, block_tables, seq_lens, scale,
                     num_seqs, 1, num_heads, num_kv_heads, head_size, block_size, partition_size,
                     dtype, stream, max_blocks_per_seq, num_blocks, workspace, workspace_bytes,
                     PA_VARIANT_AUTO, 0, 0);
}

extern "C" int pa_decode_v2_fp8(void* out, float* lse, const void* query, const void* key_cache,
                                const void* value_cache, const int32_t* block_tables,
                                const int32_t* seq_lens, float scale, float k_scale, float v_scale,
                                int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                int block_size, int partition_size, int dtype, void* stream,
                                int max_blocks_per_seq, int num_blocks, void* workspace,
                                size_t workspace_bytes) {
  return decode_impl(out, lse, query, key_cache, value_cache, block_tables, seq_lens, scale,
                     num_seqs, 1, num_heads, num_kv_heads, head_size, block_size, partition_size,
                     dtype, stream, max_blocks_per_seq, num_blocks, workspace, workspace_bytes,
                     PA_VARIANT_AUTO, 0, 0, true, k_scale, v_scale);
}

extern "C" int pa_decode_v2_mq(void* out, float* lse, const void* query, const void* key_cache,
                               const void* value_cache, const int32_t* block_tables,
                               const int32_t* seq_lens, float scale, int num_seqs, int q_len,
                               int num_heads, int num_kv_heads, int head_size, int block_size,
                               int partition_size, int dtype, void* stream, int max_blocks_per_seq,
                               int num_blocks, void* workspace, size_t workspace_bytes) {
  return decode_impl(out, lse, query, key_cache, value_cache, block_tables, seq_lens, scale,
                     num_seqs, q_len, num_heads, num_kv_heads, head_size, block_size,
                     partition_size, dtype, stream, max_blocks_per_seq, num_blocks, workspace,
                     workspace_bytes, PA_VARIANT_AUTO, 0, 0);
}

extern "C" int pa_decode_v2_mq_fp8(void* out, float* lse, const void* query, const void* key_cache,
                                   const void* value_cache, const int32_t* block_tables,
                                   const int32_t* seq_lens, float scale, float k_scale, float v_scale,
                                   int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_size,
                                   int block_size, int partition_size, int dtype, void* stream,
                                   int max_blocks_per_seq, int num_blocks, void* workspace,
                                   size_t workspace_bytes) {
  return decode_impl(out, lse, query, key_cache, value_cache, block_tables, seq_lens, scale,
                     num_seqs, q_len, num_heads, num_kv_heads, head_size, block_size,
                     partition_size, dtype, stream, max_blocks_per_seq, num_blocks, workspace,
                     workspace_bytes, PA_VARIANT_AUTO, 0, 0, true, k_scale, v_scale);
}

extern "C" int pa_decode_v2(void* out, const void* query, const void* key_cache, const void* value_cache,
                            const int32_t* block_tables, const int32_t* seq_lens, float scale,
                            int num_seqs, int num_heads, int num_kv_heads, int head_size,
                            int block_size, int partition_size, int dtype, void* stream,
                            int max_blocks_per_seq, int num_blocks, void* workspace,
                            size_t workspace_bytes) {
  return pa_decode_v2_ex(out, query, key_cache, value_cache, block_tables, seq_lens, scale, num_seqs,
                         num_heads, num_kv_heads, head_size, block_size, partition_size, dtype, stream,
                         max_blocks_per_seq, num_blocks, workspace, workspace_bytes, PA_VARIANT_AUTO, 0, 0);
}

namespace {
// Staging for the host-I/O entry point, placed after the regular workspace.
struct HostIoLayout {
  size_t q, out, bt, lens, total;
};
bool host_io_layout(int S, int H, int KH, int D, int MB, int BS, int P, HostIoLayout* h, WsLayout* w) {
  if (!ws_layout(S, H, KH, D, MB, BS, P, w)) return false;
  const size_t qbytes = (size_t)S * H * D * 4;  // room for the widest element type
  h->q = w->total;
  h->out = align_up(h->q + qbytes);
  h->bt = align_up(h->out + qbytes);
  h->lens = align_up(h->bt + (size_t)S * MB * sizeof(int32_t));
  h->total = align_up(h->lens + (size_t)S * sizeof(int32_t));
  return true;
}
}  // namespace

extern "C" size_t pa_decode_v2_host_io_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                                       int head_size, int max_blocks_per_seq,
                                                       int block_size, int partition_size) {
  HostIoLayout h;
  WsLayout w;
  if (!host_io_layout(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq, block_size,
                      partition_size, &h, &w))
    return 0;
  return h.total;
}

extern "C" int pa_decode_v2_host_io(void* out_host, const void* query_host, const void* key_cache,
                                    const void* value_cache, const int32_t* block_tables_host,
                                    const int32_t* seq_lens_host, float scale, int num_seqs,
                                    int num_heads, int num_kv_heads, int head_size, int block_size,
                                    int partition_size, int dtype, void* stream,
                                    int max_blocks_per_seq, int num_blocks, void* workspace,
                                    size_t workspace_bytes) {
  const int S = num_seqs, H = num_heads, D = head_size, MB = max_blocks_per_seq;
  HostIoLayout h;
  WsLayout w;
  if (!host_io_layout(S, H, num_kv_heads, D, MB, block_size, partition_size, &h, &w))
    return PA_ERR_INVALID_ARG;
  if (S == 0) return PA_OK;
  if (!out_host || !query_host || !block_tables_host || !seq_lens_host || !workspace)
    return PA_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < h.total) return PA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype != PA_DTYPE_FP16 && dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_FP32) return PA_ERR_INVALID_ARG;
  const size_t qbytes = (size_t)S * H * D * elem_bytes(dtype);
  if (cudaMemcpyAsync(ws + h.q, query_host, qbytes, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(ws + h.bt, block_tables_host, (size_t)S * MB * sizeof(int32_t),
                      cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(ws + h.lens, seq_lens_host, (size_t)S * sizeof(int32_t), cudaMemcpyHostToDevice,
                      st) != cudaSuccess)
    return PA_ERR_CUDA;
  const int status = pa_decode_v2(ws + h.out, ws + h.q, key_cache, value_cache,
                                  reinterpret_cast<const int32_t*>(ws + h.bt),
                                  reinterpret_cast<const int32_t*>(ws + h.lens), scale, S, H,
                                  num_kv_heads, D, block_size, partition_size, dtype, stream, MB,
                                  num_blocks, ws, w.total);
  if (status != PA_OK) return status;
  if (cudaMemcpyAsync(out_host, ws + h.out, qbytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

extern "C" int pa_decode_v2_device_status(const void* workspace, void* stream, int* status) {
  if (!workspace || !status) return PA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  *status = v;
  return PA_OK;
}

extern "C" const char* pa_decode_v2_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_WORKSPACE: return "workspace too small";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_DEVICE_BOUNDS: return "device-side bounds violation (block id or sequence length)";
    case PA_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}
