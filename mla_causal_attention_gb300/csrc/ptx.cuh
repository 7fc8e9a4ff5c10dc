// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers, bulk and tensor copies,
// bounded waits and the device status word.  No CUDA math library internals are used.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "mla_attn.h"

namespace mla {

// Upper bound on any single wait inside a kernel (nanoseconds of %globaltimer).  A wait
// that runs past it records MLA_ERR_TIMEOUT in the status word and the kernel unwinds.
// MLA_WAIT_LIMIT_NS overrides it only in the test build that checks this unwinding; the
// library itself is always built with the default.
#ifndef MLA_WAIT_LIMIT_NS
#define MLA_WAIT_LIMIT_NS 1000000000ull
#endif
constexpr uint64_t kWaitLimitNs = MLA_WAIT_LIMIT_NS;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// First error wins; later ones are dropped.
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---- mbarrier ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async proxy (bulk copies, tensor cores).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
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

// try_wait that may park the thread until the phase completes (at most the hint, 1 ms).  A
// parked waiter issues nothing, so it does not take issue slots from the warps that share
// its scheduler (a spinning waiter measurably slowed the softmax warps next to it).
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed.  Bounded: after
// kWaitLimitNs it records MLA_ERR_TIMEOUT, sets *abort and returns false.  Once *abort is
// set (by this or another thread of the CTA, via shared memory) every later wait returns
// false at once, so a CTA unwinds instead of waiting on work that will never arrive.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_hint(a, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      set_status(status, MLA_ERR_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

// ---- programmatic dependent launch ----------------------------------------------------
// The next kernel on the stream, launched with programmatic stream serialization, may start
// once every block of this one has called grid_dep_launch (or exited); it must call
// grid_dep_wait before reading anything this kernel writes.  Both are no-ops in a kernel
// launched without the attribute.
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- bulk copies (async proxy) ----------------------------------------------------------
// 1-D bulk copy global -> shared, completion counted in bytes on an mbarrier.  Both
// addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

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

// 3-D tiled tensor copy global -> shared through a tensor map (TMA).  The innermost
// coordinate c0 times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// The same without an L2 cache hint.
__device__ __forceinline__ void tma_load_3d_nohint(void* smem_dst, const void* tmap,
                                                   uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// 2-D and 4-D tiled tensor copies global -> shared (no cache hint); the innermost coordinate
// times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---- small math helpers -----------------------------------------------------------------
// 2^x with the hardware approximation (MUFU); ftz.  exp2(-inf) = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) {
  return __uint_as_float(w & 0xffff0000u);
}

// Packed fp32 pairs (sm_100 family): two lanes of fp32 arithmetic per instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Round-to-nearest-even pack of two floats into a bf16x2 word (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- rotary embedding (rotate-half form on the 64 rotary columns) ----------------------
// y[d] = x[d] cos_d - x[d+32] sin_d,  y[d+32] = x[d+32] cos_d + x[d] sin_d  (d < 32), in
// fp32, rounded once to bf16.  Eight columns at a time: `own` holds columns [c, c+8) of one
// row and `other` the columns 32 away; `upper` says whether `own` is the half at 32..63.
// cos_d / sin_d for the eight d of this slice.
__device__ __forceinline__ uint4 rope_rotate8(const uint4 own, const uint4 other,
                                              const float* cs_cos, const float* cs_sin,
                                              bool upper) {
  const uint32_t ow[4] = {own.x, own.y, own.z, own.w};
  const uint32_t ot[4] = {other.x, other.y, other.z, other.w};
  uint32_t r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float y[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float xo = h ? bf16hi_to_f32(ow[k]) : bf16lo_to_f32(ow[k]);
      const float xt = h ? bf16hi_to_f32(ot[k]) : bf16lo_to_f32(ot[k]);
      const float c = cs_cos[2 * k + h], sn = cs_sin[2 * k + h];
      // x1 = x[d], x2 = x[d+32]: lower half y = x1 c - x2 s, upper half y = x2 c + x1 s
      y[h] = upper ? fmaf(xo, c, xt * sn) : fmaf(xo, c, -xt * sn);
    }
    r[k] = pack_bf16x2(y[0], y[1]);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

}  // namespace mla
