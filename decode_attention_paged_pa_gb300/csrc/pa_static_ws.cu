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
#include <cuda.h>  // CUcontext and CUresult types only: the driver calls are looked up at run time

#include <mutex>

#include "pa_decode.h"
#include "pa_launch.h"

namespace {

// The shared scratch, one copy per device that loads the library.
static __device__ __align__(256) unsigned char g_pa_static_scratch[PA_DECODE_V2_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchSlot {
  void* ptr;                 // device address of the array in the context below
  unsigned long long ctx;    // unique id of the context the address belongs to (0: unknown)
};
ScratchSlot g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context, or 0 if there is none or
// it cannot be read.  A device's module (and with it the scratch array) is
// loaded again when its context is destroyed and recreated (cudaDeviceReset),
// so the cached address is only valid while this id stays the same.  Caller
// holds g_setup_mutex.
unsigned long long current_context_id() {
  static bool looked_up = false;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (!looked_up) {
    looked_up = true;
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", reinterpret_cast<void**>(&get_current), 12000,
                                         cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess)
      get_current = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", reinterpret_cast<void**>(&get_id), 12000,
                                         cudaEnableDefault, &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      get_id = nullptr;
  }
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device.  The host-side
// name of the array is only a stand-in; the real address comes from
// cudaGetSymbolAddress, looked up with the device current: once per device,
// and again whenever the device's context has been recreated since (or on
// every call if the context's id cannot be read).
int scratch_address(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchSlot& slot = g_scratch[dev];
  const unsigned long long ctx = current_context_id();
  if (slot.ptr && ctx != 0 && slot.ctx == ctx) {
    *ptr = slot.ptr;
    return PA_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_pa_static_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
  slot.ptr = p;
  slot.ctx = current_context_id();  // the lookup made the device's context current if it was not
  *ptr = p;
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
