// Device helpers for the sm_103a selective-scan kernels: shared-memory addresses, mbarriers,
// TMA tiled loads, packed f32x2 arithmetic, hardware transcendental approximations and
// bf16 <-> f32 conversion.  Everything here is written with documented PTX instructions.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace ssm {

// ------------------------------------------------------------------ status word
// kStatusTimeout (internal.h): a pipeline wait gave up.  The word lives in scan_fwd.cu and is read and
// cleared by ssm_device_status().

// ------------------------------------------------------------------ checked builds
// Built with -DSSM_CHECK=1 (libssm_b300_check.so), every global-memory access whose index a kernel
// computes goes through checked(): an index outside its buffer sets kStatusBounds in this
// translation unit's check word and the access is redirected to a small sink inside this library's
// device image, so that the kernel carries on without touching memory it does not own.  The result
// of that call is then wrong, and ssm_device_status() reports SSM_ERR_CHECK.  Without SSM_CHECK the
// helper is the plain pointer arithmetic.
#if SSM_CHECK
static __device__ unsigned int g_tu_check_status = 0;
static __device__ __align__(16) unsigned char g_tu_check_sink[256];
#endif

// &base[idx], valid for `width` elements, in a buffer of n elements.
template <typename T>
__device__ __forceinline__ T* checked(T* base, int64_t idx, int64_t n, int width = 1) {
#if SSM_CHECK
  if (base == nullptr || idx < 0 || idx + width > n || width * static_cast<int64_t>(sizeof(T)) > 256) {
    atomicOr(&g_tu_check_status, kStatusBounds);
    return reinterpret_cast<T*>(g_tu_check_sink);
  }
#endif
  return base + idx;
}

// Reads and clears this translation unit's check word (0 in unchecked builds).
static inline cudaError_t tu_check_read_and_clear(unsigned int* out) {
#if SSM_CHECK
  cudaError_t e = cudaMemcpyFromSymbol(out, g_tu_check_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_tu_check_status, &zero, sizeof(unsigned int));
#else
  *out = 0;
  return cudaSuccess;
#endif
}

// ------------------------------------------------------------------ shared memory / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// One arrival (release semantics at CTA scope for the arriving thread's prior writes).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase with the given parity to complete.  Gives up after `limit_ns` of wall time,
// records kStatusTimeout in *status and returns false.  try_wait itself suspends for a bounded
// time per call.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned int* status,
                                                  uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// 2D tiled TMA load of a box at (x = inner coordinate in elements, y = row) into shared memory,
// completing on `bar` with a byte count.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 3D tiled TMA load of a box at (x = inner coordinate in elements, y = row, z = block).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ packed f32x2
// A pair of floats in one 64-bit register: low word = .x, high word = .y.
struct f2 {
  unsigned long long v;
};

__device__ __forceinline__ f2 f2_make(float lo, float hi) {
  f2 r;
  r.v = (static_cast<unsigned long long>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
  return r;
}
__device__ __forceinline__ f2 f2_splat(float a) { return f2_make(a, a); }
__device__ __forceinline__ float f2_lo(f2 a) { return __uint_as_float(static_cast<unsigned>(a.v)); }
__device__ __forceinline__ float f2_hi(f2 a) { return __uint_as_float(static_cast<unsigned>(a.v >> 32)); }

__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return d;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
  return d;
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
  return d;
}

// ------------------------------------------------------------------ hardware approximations (MUFU)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// softplus(v) = log(1 + e^v) with MUFU ex2/lg2.  With e = e^v: for v < -3 the Taylor series of
// log(1 + e) to e^4 is used (truncation below e^4/5, i.e. 7e-8 relative there); for v > 15,
// softplus(v) = v to float32 precision; in between, ln2 * log2(1 + e), whose relative error is
// below 6e-6 (the absolute error of lg2.approx over log2(1 + e) >= 0.07).
__device__ __forceinline__ float softplus_fast(float v) {
  const float e = ex2_approx(v * kLog2e);
  const float series = e * fmaf(e, fmaf(e, fmaf(e, -0.25f, 0.33333334f), -0.5f), 1.0f);
  const float logpath = kLn2 * lg2_approx(1.0f + e);
  float r = v < -3.0f ? series : logpath;
  return v > 15.0f ? v : r;
}

// Accurate softplus with the CUDA math library (float32 io path).
__device__ __forceinline__ float softplus_accurate(float v) {
  return v > 0.0f ? v + log1pf(expf(-v)) : log1pf(expf(v));
}

// SiLU(z) = z / (1 + e^{-z}) with MUFU ex2/rcp.
__device__ __forceinline__ float silu_fast(float z) {
  return z * rcp_approx(1.0f + ex2_approx(-z * kLog2e));
}
__device__ __forceinline__ float silu_accurate(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------------------ bf16 <-> f32
// A 32-bit word holding two bf16 values: element 0 in the low half, element 1 in the high half.
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round two floats to bf16 (round to nearest even) and pack: a in the low half, b in the high half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

template <typename T>
struct IoTraits;

template <>
struct IoTraits<float> {
  static constexpr int kBytes = 4;
  static constexpr int kVec = 4;  // elements per 16-byte chunk
  __device__ static float to_f32(float x) { return x; }
  __device__ static float from_f32(float x) { return x; }
};

template <>
struct IoTraits<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr int kVec = 8;
  __device__ static float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

// Unpack one 16-byte chunk into kVec floats.
__device__ __forceinline__ void unpack_chunk(const uint4& c, float (&out)[4], float) {
  out[0] = __uint_as_float(c.x);
  out[1] = __uint_as_float(c.y);
  out[2] = __uint_as_float(c.z);
  out[3] = __uint_as_float(c.w);
}
__device__ __forceinline__ void unpack_chunk(const uint4& c, float (&out)[8], __nv_bfloat16) {
  out[0] = bf16lo_to_f32(c.x);
  out[1] = bf16hi_to_f32(c.x);
  out[2] = bf16lo_to_f32(c.y);
  out[3] = bf16hi_to_f32(c.y);
  out[4] = bf16lo_to_f32(c.z);
  out[5] = bf16hi_to_f32(c.z);
  out[6] = bf16lo_to_f32(c.w);
  out[7] = bf16hi_to_f32(c.w);
}

__device__ __forceinline__ uint4 pack_chunk(const float (&v)[4]) {
  return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
}
__device__ __forceinline__ uint4 pack_chunk(const float (&v)[8]) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

}  // namespace ssm
