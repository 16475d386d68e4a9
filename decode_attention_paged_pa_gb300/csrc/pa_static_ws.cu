// pa_static_ws.cu -- a decode entry point that never allocates device memory.
//
// pa_decode_v2 needs a scratch workspace (partition states, counters).  Most
// callers pass one, or let the library take one with cudaMallocAsync.  Some
// callers cannot do either: a serving process whose device memory is entirely
// reserved up front by another allocator has no room for a fresh allocation;
// a latency-critical loop cannot afford an allocation call that may
// synchronise the device or stall other streams; a deployment that fixes its
// memory footprint when it starts may forbid allocating afterwards.  For them
// this file keeps the scratch in a fixed-size array in the library's own
// device memory, which exists from the moment the library's module is loaded
// on a device until the process exits.
#include <mutex>

#include "pa_decode.h"
#include "pa_launch.h"

namespace {

// The shared scratch, one copy per device that loads the library.
static __device__ __align__(256) unsigned char g_pa_static_scratch[PA_DECODE_V2_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  The host-side
// name of the array is only a stand-in; the real address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
int scratch_address(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_static_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_v2_static_scratch(void* out, const void* query, const void* key_cache,
                                           const void* value_cache, const int32_t* block_tables,
                                           const int32_t* seq_lens, float scale, int num_seqs,
                                           int num_heads, int num_kv_heads, int head_size,
                                           int block_size, int partition_size, int dtype, void* stream,
                                           int max_blocks_per_seq, int num_blocks) {
  const size_t need = pa_decode_v2_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_size,
                                                   max_blocks_per_seq, block_size, partition_size);
  if (need == 0) return PA_ERR_INVALID_ARG;
  if (need > (size_t)PA_DECODE_V2_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != PA_OK) return st;
  // The regular entry point zeroes the counters it needs at the start of every
  // call (stream-ordered memset) and writes every other scratch byte it reads.
  return pa_decode_v2(out, query, key_cache, value_cache, block_tables, seq_lens, scale, num_seqs,
                      num_heads, num_kv_heads, head_size, block_size, partition_size, dtype, stream,
                      max_blocks_per_seq, num_blocks, scratch, (size_t)PA_DECODE_V2_STATIC_SCRATCH_BYTES);
}
