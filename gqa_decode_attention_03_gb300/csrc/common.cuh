// common.cuh -- device helpers shared by the decode-attention kernels (sm_103a).
//
// mbarrier / TMA / cp.async wrappers in inline PTX, bounded waits, and the small numeric helpers
// (exp2 with log2(e) folded into the score scale, NaN-safe masking).  Every wait here has an
// iteration limit: a wait that runs out returns false, the caller records GQA_ERR_TIMEOUT in the
// error word and leaves, so no kernel can spin forever.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gqa_decode.h"

namespace gqa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kSpinLimit = 1u << 20;  // try_wait polls before a wait gives up (>= ~20 ms)

// ------------------------------------------------------------------------------------ mbarrier

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes the barrier initialisation visible to the async proxy (TMA) and the other threads.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; false after kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// ------------------------------------------------------------------------------------ TMA

// 3-D tiled bulk tensor load global -> shared, completing as transaction bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Untiled bulk copy global -> shared of `bytes` (a multiple of 16; both addresses 16-byte
// aligned), completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------------------------ cp.async

// 16-byte (or 8-byte) asynchronous copy global -> shared, bypassing L1.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

// The barrier's pending count drops by one when all cp.async issued so far by this thread
// have landed (the arrival is not pre-counted: the barrier's count includes this thread).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// ------------------------------------------------------------------------------------ misc

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

// ---------------------------------------------------------------- thread-block clusters

// Every thread of every CTA of the cluster: arrive (release), then wait (acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}

// The address of this CTA's shared word `a` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

// The inverse rotation of a TurboQuant row (flash_attention_tq.metal's epilogue), on a row held
// D/32 consecutive dims per lane: scale by 1/sqrt(D), the Walsh-Hadamard butterflies (within
// the lane for strides below D/32, across lanes by shuffle above), then the sign flip.
template <int D>
__device__ __forceinline__ void rotate_back(float (&a)[D / 32], const float* signs, int lane) {
  constexpr int DPL = D / 32;
  const float s = rsqrtf(static_cast<float>(D));
#pragma unroll
  for (int k = 0; k < DPL; ++k) a[k] *= s;
#pragma unroll
  for (int stride = 1; stride < DPL; stride <<= 1)
#pragma unroll
    for (int k = 0; k < DPL; ++k)
      if ((k & stride) == 0) {
        const float x = a[k], y = a[k + stride];
        a[k] = x + y;
        a[k + stride] = x - y;
      }
#pragma unroll
  for (int stride = DPL; stride < D; stride <<= 1) {
    const int lmask = stride / DPL;
    const bool high = (lane & lmask) != 0;
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
      const float other = __shfl_xor_sync(0xffffffffu, a[k], lmask);
      a[k] = high ? other - a[k] : a[k] + other;
    }
  }
#pragma unroll
  for (int k = 0; k < DPL; ++k) a[k] *= __ldg(signs + lane * DPL + k);
}

__device__ __forceinline__ void flag_error(int32_t* err_word, int bits) {
  if (err_word) atomicOr(err_word, bits);
}

// Byte offset of 16-byte chunk `c` of tile row `r` in a staged tile laid out as boxes of
// 128-byte rows with the 128-byte TMA swizzle: box b = c / 8 holds rows of 8 chunks, and the
// chunk slot within a row is (c % 8) xor (r % 8).  Box b starts at b * rows * 128.
__device__ __forceinline__ uint32_t swz_off(int r, int c, int rows) {
  return static_cast<uint32_t>((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

}  // namespace gqa
