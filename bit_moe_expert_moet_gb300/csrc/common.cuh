// Shared device helpers of the moet library (sm_103a).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moet.h"

namespace moet {

// First device-side problem recorded by a kernel of this translation unit
// (0 = none).  Lives in the module image: one word per device per unit, never
// allocated at run time.  Each unit exposes it to the host through
// MOET_ERROR_ACCESSOR, which moet_last_device_error calls for every unit.
static __device__ int g_device_error = 0;

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_device_error, 0, code); }

// ---------------------------------------------------------------- programmatic dependent launch
// The decode regime's kernels are launched with programmatic stream serialization (pdl_launch):
// a kernel may be scheduled while the kernel before it in the stream is still running, and runs its
// set-up (shared-memory barriers, TMEM allocation) meanwhile.  pdl_wait() returns once that
// kernel has completed and its memory operations are visible; every kernel calls it before its
// first access to global memory.  pdl_trigger(), called after the wait, lets the next kernel be
// scheduled early in turn (so at most one kernel waits ahead).  Both are no-ops for a kernel
// launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// pdl = false launches plainly.  The decode regime's chain of short kernels uses the attribute
// (T = 64: 0.833 -> 0.826 ms per step); the prefill regime does not (its step was 1.5 % slower
// with it).
template <typename... P, typename... A>
inline cudaError_t pdl_launch(bool pdl, void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              A&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...);
}

// ---------------------------------------------------------------- e4m3fn
// Exact fp32 value of a non-negative e4m3fn byte (sign ignored, 0x7F never
// produced by this library).  Normal codes: the 7 low bits placed at fp32 bits
// 20..26 give 2^(e-127) (1 + m/8); multiplying by 2^120 rebases the exponent
// (bias 7).  Subnormal codes land on fp32 subnormals m 2^-129 and the same
// multiply gives m 2^-9.  Exact in both cases (no FTZ in this library).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  return __uint_as_float((b & 0x7Fu) << 20) * 0x1p120f;
}

// RNE to e4m3fn (satfinite) of a value given as a fp32 number; one cvt.
// Both halves of the packed result hold the same value, so the byte order of
// the x2 conversion does not matter.
__device__ __forceinline__ uint32_t f32_to_e4m3_rn(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x), "f"(x));
  return r & 0xFFu;
}

// e4m3 satfinite RNE of the exact ratio a / d (a >= 0, d in {3, 6}).  The
// first guess comes from a rounded fp32 quotient; it is then corrected by
// comparing 2a with d (lo + hi), the doubled midpoint with each neighbour,
// which is exact in fp32 because a, d and the midpoints have few
// significant bits.  Ties go to the even code.
__device__ __forceinline__ uint32_t e4m3_rne_ratio_small(float a, float d) {
  uint32_t c = f32_to_e4m3_rn(a / d);
  float v = e4m3_to_f32(c);
  if (c < 126u) {
    float up = e4m3_to_f32(c + 1);
    float m2 = d * (v + up);
    if (2.0f * a > m2 || (2.0f * a == m2 && (c & 1u))) c += 1;
  }
  if (c > 0u) {
    float v2 = e4m3_to_f32(c);
    float dn = e4m3_to_f32(c - 1);
    float m2 = d * (dn + v2);
    if (2.0f * a < m2 || (2.0f * a == m2 && (c & 1u))) c -= 1;
  }
  return c;
}

// e2m1 magnitude code of RNE(a / s) for a >= 0, s > 0, saturating at 6,
// ties to the even code, by comparison with the seven midpoints scaled by s
// (each product is exact in fp32).
__device__ __forceinline__ uint32_t e2m1_rne_mag(float a, float s) {
  uint32_t c = 0;
  c += (a > 0.25f * s);
  c += (a >= 0.75f * s);
  c += (a > 1.25f * s);
  c += (a >= 1.75f * s);
  c += (a > 2.5f * s);
  c += (a >= 3.5f * s);
  c += (a > 5.0f * s);
  return c;
}

__device__ __forceinline__ float e2m1_mag_value(uint32_t m) {
  // {0, .5, 1, 1.5, 2, 3, 4, 6}
  const float lo = (float)(m & 1u) * 0.5f;
  switch (m >> 1) {
    case 0: return lo;            // 0, 0.5
    case 1: return 1.0f + lo;     // 1, 1.5
    case 2: return 2.0f * (1.0f + lo);  // 2, 3
    default: return 4.0f * (1.0f + lo); // 4, 6
  }
}

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + 0, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// e2m1x2 byte (low nibble -> low half) to f16x2.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "r"(byte));
  return r;
}

// Opt-in launch timing (moet_profile_enable): host-side event pairs around
// each launch of kind `kind` on `st`.  No-ops while profiling is off.
void prof_begin(int kind, cudaStream_t st);
void prof_end(int kind, cudaStream_t st);

struct ProfScope {
  int kind;
  cudaStream_t st;
  ProfScope(int k, cudaStream_t s) : kind(k), st(s) { prof_begin(k, s); }
  ~ProfScope() { prof_end(kind, st); }
};

}  // namespace moet

// Defines `int name(void)`: reads and clears this unit's device error flag
// (blocking copy; the caller has synchronised the stream).  Returns -1 if the
// copy fails.
#define MOET_ERROR_ACCESSOR(name)                                                   \
  extern "C" __attribute__((visibility("hidden"))) int name(void) {                                                       \
    int v = 0;                                                                      \
    if (cudaMemcpyFromSymbol(&v, moet::g_device_error, sizeof(int)) != cudaSuccess) \
      return -1;                                                                    \
    if (v != 0) {                                                                   \
      const int zero = 0;                                                           \
      if (cudaMemcpyToSymbol(moet::g_device_error, &zero, sizeof(int)) != cudaSuccess) \
        return -1;                                                                  \
    }                                                                               \
    return v;                                                                       \
  }

#define MOET_CUDA_TRY(expr)                          \
  do {                                               \
    if ((expr) != cudaSuccess) return MOET_ERR_CUDA; \
  } while (0)
