// Asynchronous-copy helpers (sm_100+ PTX): shared-memory mbarriers with bounded waits,
// the untiled bulk copy global -> shared, proxy fences and gpu-scope counters.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dory {

// try_wait rounds before a wait gives up (each round suspends for a bounded time in the
// hardware, so the limit is well above any legitimate wait)
constexpr uint32_t MBAR_WAIT_LIMIT = 1u << 20;

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// The same shared-memory address as a pointer the compiler can see is in shared memory. A
// pointer handed across a call that is not inlined arrives generic, and loads and stores
// through it take the generic path; rebuilt from the shared window's base it is shared again.
template <typename T>
__device__ __forceinline__ T *in_shared(T *p) {
  extern __shared__ uint8_t dyn_smem_base[];
  return reinterpret_cast<T *>(dyn_smem_base + ((int)smem_addr(p) - (int)smem_addr(dyn_smem_base)));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of parity `parity` to complete; false when the limit ran out or
// `*stop` became nonzero (stop may be null).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int *stop = nullptr) {
  for (uint32_t i = 0; i < MBAR_WAIT_LIMIT; i++) {
    if (mbar_test(bar, parity)) return true;
    if (stop && *stop) return false;
  }
  return false;
}

__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(n) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// `bytes` (a multiple of 16, both addresses 16-byte aligned) from global to shared memory,
// completion counted on `bar`
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// An L2 policy that evicts first what it tags (for data read once, such as a weight stream,
// so that it does not displace what is read again soon).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy for the source reads
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Order this thread's generic-proxy global writes before later async-proxy (bulk copy)
// reads of the same memory, and the reverse on the reading side.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Order earlier generic-proxy accesses of shared memory (after a barrier, the whole team's)
// before a bulk copy that overwrites it.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Start moving `bytes` (a multiple of 16, 16-byte aligned) from global memory into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(int *p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_release_gpu(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Tagged words: a float and the tag of the stage that wrote it in one 64-bit word (value in
// the low half), stored and loaded as single 64-bit accesses, so a reader sees either the old
// word or the new one whole. A reader polls until the tag is the one it expects: the word is
// its own completion flag, with no fence and no separate counter.
__device__ __forceinline__ unsigned long long tag_word(float v, uint32_t tag) {
  return ((unsigned long long)tag << 32) | __float_as_uint(v);
}

__device__ __forceinline__ void st_tagged(unsigned long long *p, float v, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(tag_word(v, tag)) : "memory");
}

// 4 consecutive values (16-byte aligned words p[0..3])
__device__ __forceinline__ void st_tagged4(unsigned long long *p, const float4 &v, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(tag_word(v.x, tag)),
               "l"(tag_word(v.y, tag))
               : "memory");
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p + 2), "l"(tag_word(v.z, tag)),
               "l"(tag_word(v.w, tag))
               : "memory");
}

// true when the word carries `tag` (v is then its value)
__device__ __forceinline__ bool ld_tagged(const unsigned long long *p, uint32_t tag, float &v) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p));
  v = __uint_as_float((uint32_t)w);
  return (uint32_t)(w >> 32) == tag;
}

// 2 consecutive values (16-byte aligned words p[0..1])
__device__ __forceinline__ void st_tagged2(unsigned long long *p, float a, float b, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(tag_word(a, tag)), "l"(tag_word(b, tag))
               : "memory");
}

// true when both words p[0..1] (16-byte aligned) carry `tag`
__device__ __forceinline__ bool ld_tagged2(const unsigned long long *p, uint32_t tag, float2 &v) {
  unsigned long long a, b;
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
  v = make_float2(__uint_as_float((uint32_t)a), __uint_as_float((uint32_t)b));
  return (uint32_t)(a >> 32) == tag && (uint32_t)(b >> 32) == tag;
}

// true when all 4 words p[0..3] (16-byte aligned) carry `tag`
__device__ __forceinline__ bool ld_tagged4(const unsigned long long *p, uint32_t tag, float4 &v) {
  unsigned long long a, b, c, d;
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(c), "=l"(d) : "l"(p + 2));
  v = make_float4(__uint_as_float((uint32_t)a), __uint_as_float((uint32_t)b), __uint_as_float((uint32_t)c),
                  __uint_as_float((uint32_t)d));
  return (uint32_t)(a >> 32) == tag && (uint32_t)(b >> 32) == tag && (uint32_t)(c >> 32) == tag &&
         (uint32_t)(d >> 32) == tag;
}


}  // namespace dory
