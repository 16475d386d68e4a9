// pa_common.cuh -- device helpers shared by the paged decode attention kernels:
// inline-PTX wrappers for mbarriers, 1-D bulk async copies and 3-D tensor
// copies (the Tensor Memory Accelerator), ldmatrix / movmatrix / mma.sync,
// bounded waits, and element conversions (fp16, bf16, fp32).
#pragma once

#include <cuda.h>  // CUtensorMap (the type only)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace pa {

// Status codes shared with include/pa_decode.h.
constexpr int kOk = 0;
constexpr int kErrDeviceBounds = 5;
constexpr int kErrTimeout = 6;

// Workspace header: int32 words.
constexpr int kHdrError = 0;    // first device-side error code (0 = none)
constexpr int kHdrWork = 1;     // dynamic work counter (units handed out)
constexpr int kHdrWhere = 2;    // first timed-out wait: site, CTA, warp, detail (4 ints)
constexpr int kHdrInts = 64;    // header size in ints (256 bytes)

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of phase `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Record a timed-out wait: kErrTimeout in the error word and, for the first
// one, where it happened (wait site, CTA, warp, a site-specific detail).
__device__ __forceinline__ void record_timeout(volatile int* abort_flag, int* err_word, int site,
                                               int detail) {
  *abort_flag = 1;
  atomicCAS(err_word, 0, kErrTimeout);
  if (atomicCAS(err_word + kHdrWhere, 0, site) == 0) {
    err_word[kHdrWhere + 1] = blockIdx.x;
    err_word[kHdrWhere + 2] = threadIdx.x >> 5;
    err_word[kHdrWhere + 3] = detail;
  }
}

// Wait for phase `parity` of an mbarrier with a time bound.  Returns false if
// the CTA's abort flag is raised or the bound runs out (which raises the flag
// and records the timeout).  Never spins forever.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             int* err_word, long long timeout_ns, int site = 1,
                                             int detail = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((long long)(global_timer_ns() - t0) > timeout_ns) {
      record_timeout(abort_flag, err_word, site, detail);
      return false;
    }
  }
}

// ---------------------------------------------------------------- bulk copy
// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// Both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
// 3-D tensor copy global -> shared of one box of the tensor map `tmap` (a
// __grid_constant__ kernel parameter) at element coordinates (x, y, z),
// completion counted on `bar` in bytes.  `dst` must be 1024-byte aligned (the
// value tiles use the 32-byte swizzle, whose pattern follows the shared-memory
// address bits); x times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tmap, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// Global stores / loads of fp32 data with an L2 eviction-priority policy.
__device__ __forceinline__ void st_f4_policy(float4* dst, const float4& v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void st_f32_policy(float* dst, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(dst), "f"(v), "l"(policy) : "memory");
}
__device__ __forceinline__ float4 ld_f4_policy(const float4* src, uint64_t policy) {
  float4 v;
  asm volatile("ld.global.cg.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(src), "l"(policy));
  return v;
}
__device__ __forceinline__ float ld_f32_policy(const float* src, uint64_t policy) {
  float v;
  asm volatile("ld.global.cg.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(src), "l"(policy));
  return v;
}

// L2 policy for data read once (K/V pages): evict first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- global atomics
// atomicAdd with release semantics at GPU scope: every write that happens
// before it (in this thread, or in threads it synchronised with through a
// barrier) is visible GPU-wide before the add is.
__device__ __forceinline__ int atomic_add_release_gpu(int* addr, int v) {
  int old;
  asm volatile("atom.release.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// ---------------------------------------------------------------- barriers
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also ORs a predicate across the participating threads.
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------- 16-bit floats
template <typename T> struct F16Traits;
template <> struct F16Traits<__half> {
  __device__ __forceinline__ static float2 to_float2(uint32_t v) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static __half from_float(float f) { return __float2half_rn(f); }
};
template <> struct F16Traits<__nv_bfloat16> {
  __device__ __forceinline__ static float2 to_float2(uint32_t v) {
    // bfloat16 is the upper half of a binary32: widening is a shift.
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static __nv_bfloat16 from_float(float f) { return __float2bfloat16_rn(f); }
};

// Elements of T in one 16-byte chunk (the page's key layout packs x of them).
template <typename T>
constexpr int elems_per_chunk() {
  return 16 / (int)sizeof(T);
}

// One 16-byte chunk of T as floats.
template <typename T>
__device__ __forceinline__ void unpack_chunk(const uint4& raw, float (&f)[elems_per_chunk<T>()]) {
  if constexpr (sizeof(T) == 4) {
    f[0] = __uint_as_float(raw.x); f[1] = __uint_as_float(raw.y);
    f[2] = __uint_as_float(raw.z); f[3] = __uint_as_float(raw.w);
  } else {
    float2 a = F16Traits<T>::to_float2(raw.x), b = F16Traits<T>::to_float2(raw.y);
    float2 c = F16Traits<T>::to_float2(raw.z), d = F16Traits<T>::to_float2(raw.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
}

// Four consecutive output elements, rounded to T (round to nearest even).
template <typename T>
__device__ __forceinline__ void store4(T* dst, const float4& v) {
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(dst) = v;
  } else {
    uint2 w;
    w.x = F16Traits<T>::pack(v.x, v.y);
    w.y = F16Traits<T>::pack(v.z, v.w);
    *reinterpret_cast<uint2*>(dst) = w;
  }
}

// ---------------------------------------------------------------- tensor-core helpers
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
template <typename T> struct Mma;
template <> struct Mma<__half> {
  __device__ __forceinline__ static void run(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};
template <> struct Mma<__nv_bfloat16> {
  __device__ __forceinline__ static void run(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

}  // namespace pa
