// Internal helpers shared by the libpkv translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

// ---------------------------------------------------------------------------
// Sticky device error word.  Each translation unit has its own copy (no
// relocatable device code); host code reads them through the per-unit
// read_device_error_* functions declared in internal.h.  Encoding: bits
// 63..56 = pkv_status, bits 55..0 = the offending index (truncated).
// The first error wins.
// ---------------------------------------------------------------------------
static __device__ unsigned long long g_dev_error = 0ull;

__device__ __forceinline__ void record_error(pkv_status code, int64_t detail) {
  unsigned long long v = (static_cast<unsigned long long>(code) << 56) |
                         (static_cast<unsigned long long>(detail) & ((1ull << 56) - 1));
  atomicCAS(&g_dev_error, 0ull, v);
}

// Host side: read and clear this unit's word (synchronises the device).
static inline cudaError_t read_and_clear_unit_error(unsigned long long *out) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_dev_error, sizeof(*out));
  if (e != cudaSuccess) return e;
  const unsigned long long zero = 0ull;
  return cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(zero));
}

// ---------------------------------------------------------------------------
// Element types.  Storage is raw 16-bit; conversion to fp32 is exact.
// ---------------------------------------------------------------------------
struct BF16 {
  using storage = __nv_bfloat16;
  using pair = __nv_bfloat162;
  // exact widening of a packed pair (low half = first element)
  static __device__ __forceinline__ float2 to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  static __device__ __forceinline__ uint32_t from_f2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
  static __device__ __forceinline__ float to_f(uint16_t s) {
    return __uint_as_float(static_cast<uint32_t>(s) << 16);
  }
};

struct FP16 {
  using storage = __half;
  using pair = __half2;
  static __device__ __forceinline__ float2 to_f2(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    return __half22float2(h);
  }
  static __device__ __forceinline__ uint32_t from_f2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
  static __device__ __forceinline__ float to_f(uint16_t s) {
    return __half2float(__ushort_as_half(s));
  }
};

// ---------------------------------------------------------------------------
// Bounded waits.  Every spin in this library gives up after kWaitLimitNs of
// %globaltimer time, records PKV_ERR_TIMEOUT and reports failure so the
// caller can drain and return instead of hanging the GPU.
// ---------------------------------------------------------------------------
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s; legit waits are us

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false on timeout
// (PKV_ERR_TIMEOUT recorded with `where` as detail).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int64_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_error(PKV_ERR_TIMEOUT, where);
      return false;
    }
  }
}

// 4-D tiled TMA load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel of its stream finishes;
// past grid_dependency_wait() that kernel has completed and its writes are
// visible (a no-op for an ordinary launch).  grid_launch_dependents() lets
// the next such kernel be scheduled before this one completes.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// Four E4M3 codes (low byte first) -> two fp16 pairs (low half first),
// exactly: every E4M3 value is an fp16 value.
__device__ __forceinline__ uint2 e4m3x4_to_h4(uint32_t u) {
  uint2 r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(r.x), "=r"(r.y)
      : "r"(u));
  return r;
}

// Four floats (first in the low byte) as E4M3 codes, nearest even,
// saturating: hi; and the codes of what hi leaves over: lo.
__device__ __forceinline__ void split_e4m3x4(float v0, float v1, float v2, float v3, uint32_t &hi,
                                             uint32_t &lo) {
  auto pack = [](float a, float b, float c, float d) -> uint32_t {
    uint16_t p01, p23;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(p01) : "f"(a), "f"(b));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(p23) : "f"(c), "f"(d));
    return static_cast<uint32_t>(p01) | (static_cast<uint32_t>(p23) << 16);
  };
  hi = pack(v0, v1, v2, v3);
  const uint2 h = e4m3x4_to_h4(hi);  // exact: every E4M3 value is an fp16 value
  const float2 f01 = FP16::to_f2(h.x), f23 = FP16::to_f2(h.y);
  lo = pack(v0 - f01.x, v1 - f01.y, v2 - f23.x, v3 - f23.y);
}

// Packed fp32 pairs (Blackwell f32x2 FMA/ADD/MUL) and the 3-input max: the
// attention inner loops are instruction-bound, and the packed forms halve
// their per-element arithmetic.
__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long fmul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

}  // namespace pkv
