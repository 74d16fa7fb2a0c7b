// Device-side helpers: vector memory access, lane masks, number conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace ep {

constexpr unsigned kFullMask = 0xFFFFFFFFu;

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// 16-byte load of data that no kernel writes while this one runs; it is read
// once, so it is not kept in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// 16-byte read-only load that may be served from L1 (rows a token reads twice).
__device__ __forceinline__ uint4 ld_ro16(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ void st16(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// L2-coherent 32-bit load (bypasses L1): data another CTA wrote in this kernel.
__device__ __forceinline__ int ld_cg(const int32_t* p) { return __ldcg(p); }

// two bf16 (packed in a 32-bit word, low half first) -> two floats; exact
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w) {
  float2 r;
  r.x = __uint_as_float(w << 16);
  r.y = __uint_as_float(w & 0xFFFF0000u);
  return r;
}

// fp32 -> bf16, round to nearest even; a and b packed with a in the low half
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// fp32 -> OCP E4M3, round to nearest even, saturating to +-448; a in the low byte
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

}  // namespace ep
