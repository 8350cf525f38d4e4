// pa_device.cuh — device-side helpers shared by the libpa kernels (sm_103a).
//
// Error reporting: kernels never trap. A range error or a wait that gives up
// sets a bit in a per-device error word (owned by pa_host.cu, passed to every
// kernel as a pointer) and the offending work is skipped or clamped.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

enum : unsigned {
  kErrBounds = 1u,   // an index pointed outside its buffer
  kErrTimeout = 2u,  // a bounded wait gave up
};

// Upper bound of any device-side wait, in nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ void raise_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// One arrival that counts as `count` of the barrier's expected arrivals.
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, unsigned count) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(count)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Returns false (and
// raises kErrTimeout) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      raise_error(err, kErrTimeout);
      return false;
    }
  }
}

// ------------------------------------------- programmatic dependent launch
// A kernel that produces split partials lets the merge kernel that follows
// it on the stream be scheduled early (launch_dependents, called by every
// CTA at its start); the merge waits (grid_dependency_wait) until the
// producing grid has completed and its writes are visible. Both are no-ops
// for kernels launched without the programmatic-serialization attribute.
__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// --------------------------------------------------------- bulk async copies

// One contiguous global -> shared copy completed on `bar` (transaction bytes).
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, unsigned bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 16 bytes global -> shared through L2 only (cp.async.cg), tracked by the
// executing thread's async-copy groups.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until every async-copy group of this thread has landed.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Named barrier over `count` threads (a multiple of 32). The caller's warp
// is reconverged first, and the non-aligned form is used, so a warp whose
// lanes arrive from different branches cannot leave the barrier incomplete.
__device__ __forceinline__ void named_bar_sync(unsigned id, unsigned count) {
  __syncwarp();
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier over `count` threads that also ORs a predicate over them:
// every participant gets the same answer (for decisions that must agree).
__device__ __forceinline__ bool named_bar_or(unsigned id, unsigned count, bool pred) {
  __syncwarp();
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ numbers

// Two fp32 lanes in one 64-bit register pair, for the sm_100-family packed
// fp32 instructions (one instruction does two multiply-adds).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// 2^x on the special-function unit, results below 2^-126 flushed to zero
// (softmax weights: exp2(-inf) = 0, exp2(0) = 1 exactly).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (sm_100 family)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Eight bf16 in a uint4 -> eight floats (exact).
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Two E4M3 codes (low byte first) -> two floats, exact (E4M3 values are
// representable in f16, and f16 in f32).
__device__ __forceinline__ void e4m3x2_to_f32(uint16_t codes, float& lo, float& hi) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tmov.b16 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(h2)
      : "h"(codes));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  float2 f = __half22float2(h);
  lo = f.x;
  hi = f.y;
}

// Sixteen E4M3 codes in a uint4 -> sixteen floats.
__device__ __forceinline__ void e4m3x16_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    e4m3x2_to_f32(static_cast<uint16_t>(w[i] & 0xFFFF), f[4 * i + 0], f[4 * i + 1]);
    e4m3x2_to_f32(static_cast<uint16_t>(w[i] >> 16), f[4 * i + 2], f[4 * i + 3]);
  }
}

// Eight E4M3 codes in a uint2 -> eight floats.
__device__ __forceinline__ void e4m3x8_to_f32(const uint2& v, float* f) {
  e4m3x2_to_f32(static_cast<uint16_t>(v.x & 0xFFFF), f[0], f[1]);
  e4m3x2_to_f32(static_cast<uint16_t>(v.x >> 16), f[2], f[3]);
  e4m3x2_to_f32(static_cast<uint16_t>(v.y & 0xFFFF), f[4], f[5]);
  e4m3x2_to_f32(static_cast<uint16_t>(v.y >> 16), f[6], f[7]);
}

}  // namespace pa
