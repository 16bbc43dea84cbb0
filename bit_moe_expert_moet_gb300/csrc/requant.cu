// Load-time kernels: fp32 -> NVFP4 quantiser and NVFP4 -> 2-bit planes (+ delta).
//
// README "Frontier MoE on consumer Blackwell (SM120)", "GLM-5.2 (753B)" par. 1
// (modelopt NVFP4 = e2m1 x e4m3 block-16 x fp32 scale_2, requantised at load)
// and "How it fits -- 2-bit experts at FP4 quality" bullets 1-2.
//
// Both kernels are HBM-bound streams: one thread owns 32-weight groups of
// one row (16 bytes of NVFP4 codes + 2 scale bytes in, one sign word + one
// magnitude word + 2 scale bytes (+16 + 2 delta bytes) out), so consecutive
// threads touch consecutive 16-byte chunks and every access is a coalesced
// 128-bit (or narrower, contiguous) transaction.
#include "common.cuh"

namespace moet {

// ---------------------------------------------------------------- requant
__global__ void __launch_bounds__(256) requant_2bit_kernel(
    long long n_groups, const uint4* __restrict__ codes, const uint16_t* __restrict__ s4,
    uint32_t* __restrict__ sign_out, uint32_t* __restrict__ mag_out,
    uint16_t* __restrict__ s16_out, uint4* __restrict__ dcodes_out,
    uint16_t* __restrict__ ds4_out) {
  long long gi = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (; gi < n_groups; gi += stride) {
    const uint4 cw = __ldg(codes + gi);
    const uint32_t sc = __ldg(s4 + gi);
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
    uint32_t sign = 0, mag = 0, s16pair = 0, ds4pair = 0;
    uint32_t dwords[4] = {0, 0, 0, 0};
#pragma unroll
    for (int b = 0; b < 2; ++b) {  // two blocks of 16 per 32-weight group
      const float s4f = e4m3_to_f32((sc >> (8 * b)) & 0xFFu);
      float v[16];
      float bmax = 0.0f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t c = (words[2 * b + (j >> 3)] >> (4 * (j & 7))) & 0xFu;
        const float a = e2m1_mag_value(c & 7u) * s4f;  // exact
        v[j] = (c & 8u) ? -a : a;
        bmax = fmaxf(bmax, a);
        sign |= (c >> 3) << (16 * b + j);
      }
      const uint32_t s16 = e4m3_rne_ratio_small(bmax, 3.0f);
      const float s16f = e4m3_to_f32(s16);
      s16pair |= s16 << (8 * b);
      float d[16];
      float dmax = 0.0f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t m = fabsf(v[j]) >= 2.0f * s16f;
        mag |= m << (16 * b + j);
        const float q = (m ? 3.0f : 1.0f) * s16f;
        const float w2 = ((sign >> (16 * b + j)) & 1u) ? -q : q;
        d[j] = v[j] - w2;  // exact in fp32 (short dyadics of nearby magnitude)
        dmax = fmaxf(dmax, fabsf(d[j]));
      }
      if (dcodes_out != nullptr) {
        const uint32_t ds4 = e4m3_rne_ratio_small(dmax, 6.0f);
        const float dsf = e4m3_to_f32(ds4);
        ds4pair |= ds4 << (8 * b);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t dm = dsf > 0.0f ? e2m1_rne_mag(fabsf(d[j]), dsf) : 0u;
          const uint32_t code = dm | ((d[j] < 0.0f && dm != 0u) ? 8u : 0u);
          dwords[2 * b + (j >> 3)] |= code << (4 * (j & 7));
        }
      }
    }
    sign_out[gi] = sign;
    mag_out[gi] = mag;
    s16_out[gi] = (uint16_t)s16pair;
    if (dcodes_out != nullptr) {
      dcodes_out[gi] = make_uint4(dwords[0], dwords[1], dwords[2], dwords[3]);
      ds4_out[gi] = (uint16_t)ds4pair;
    }
  }
}

// ---------------------------------------------------------------- requant, planes only
// Fast path without the delta.  All 16 weights of a block share s4, so
// v = e2m1(code) * s4 is monotone in the magnitude code: max|v| is the value of
// the largest magnitude code, and |v| >= 2 s16 holds exactly for the codes at
// or above a threshold code.  Both s16 and that threshold depend only on
// (largest code, s4); every CTA tabulates them once in shared memory with the
// exact rounding above, and the per-weight work is integer arithmetic on
// eight nibbles at a time.
__device__ __forceinline__ uint32_t gather_nibble_bit3(uint32_t x) {
  // bit 3 of nibble i -> bit i (i = 0..7)
  uint32_t t = (x >> 3) & 0x11111111u;
  t = (t | (t >> 3)) & 0x03030303u;
  t = (t | (t >> 6)) & 0x000F000Fu;
  return (t | (t >> 12)) & 0xFFu;
}

__device__ __forceinline__ uint32_t max_mag_code(uint32_t w0, uint32_t w1) {
  uint32_t m = __vmaxu4(__vmaxu4(w0 & 0x07070707u, (w0 >> 4) & 0x07070707u),
                        __vmaxu4(w1 & 0x07070707u, (w1 >> 4) & 0x07070707u));
  m = __vmaxu4(m, m >> 16);
  m = __vmaxu4(m, m >> 8);
  return m & 0xFFu;
}

// mag bits (|q| = 3) of the 8 nibbles of w, given the block's threshold code
__device__ __forceinline__ uint32_t mag_bits(uint32_t w, uint32_t add) {
  return gather_nibble_bit3(((w & 0x77777777u) + add) & 0x88888888u);
}

constexpr int kGroupsPerIter = 2;

__global__ void __launch_bounds__(256) requant_planes_kernel(
    long long n_groups, const uint4* __restrict__ codes, const uint16_t* __restrict__ s4,
    uint32_t* __restrict__ sign_out, uint32_t* __restrict__ mag_out, uint16_t* __restrict__ s16_out) {
  // lut[s4 * 8 + maxcode] = s16 | (threshold code << 8)
  __shared__ uint16_t lut[128 * 8];
  for (int i = threadIdx.x; i < 127 * 8; i += blockDim.x) {
    const uint32_t sc = i >> 3, mc = i & 7;
    const float s4f = e4m3_to_f32(sc);
    const uint32_t s16 = e4m3_rne_ratio_small(e2m1_mag_value(mc) * s4f, 3.0f);
    const float two_s16 = 2.0f * e4m3_to_f32(s16);
    uint32_t thr = 0;
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c) thr += (e2m1_mag_value(c) * s4f < two_s16);
    lut[i] = (uint16_t)(s16 | (thr << 8));
  }
  __syncthreads();
  const long long stride = (long long)gridDim.x * blockDim.x * kGroupsPerIter;
  for (long long g0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * kGroupsPerIter; g0 < n_groups;
       g0 += stride) {
    uint4 cw[kGroupsPerIter];
    uint32_t sc[kGroupsPerIter];
#pragma unroll
    for (int u = 0; u < kGroupsPerIter; ++u) {
      if (g0 + u < n_groups) {
        cw[u] = __ldg(codes + g0 + u);
        sc[u] = __ldg(s4 + g0 + u);
      }
    }
#pragma unroll
    for (int u = 0; u < kGroupsPerIter; ++u) {
      if (g0 + u >= n_groups) break;
      const uint32_t w[4] = {cw[u].x, cw[u].y, cw[u].z, cw[u].w};
      uint32_t sign = 0, mag = 0, s16pair = 0;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t e = lut[((sc[u] >> (8 * b)) & 0x7Fu) * 8 + max_mag_code(w[2 * b], w[2 * b + 1])];
        s16pair |= (e & 0xFFu) << (8 * b);
        const uint32_t add = (8u - (e >> 8)) * 0x11111111u;
        sign |= (gather_nibble_bit3(w[2 * b]) | (gather_nibble_bit3(w[2 * b + 1]) << 8)) << (16 * b);
        mag |= (mag_bits(w[2 * b], add) | (mag_bits(w[2 * b + 1], add) << 8)) << (16 * b);
      }
      sign_out[g0 + u] = sign;
      mag_out[g0 + u] = mag;
      s16_out[g0 + u] = (uint16_t)s16pair;
    }
  }
}

// ---------------------------------------------------------------- quantiser
__global__ void __launch_bounds__(256) amax_kernel(long long per_matrix4, const float4* __restrict__ w,
                                                   unsigned int* __restrict__ amax_bits) {
  const int m = blockIdx.y;
  const float4* wm = w + (long long)m * per_matrix4;
  float mx = 0.0f;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < per_matrix4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 f = __ldg(wm + i);
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits + m, __float_as_uint(mx));
}

__global__ void scale2_kernel(int M, float* scale_2) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m < M) scale_2[m] = __fdiv_rn(scale_2[m], 2688.0f);  // scale_2 held amax bits
}

// e4m3 RNE of a / d with d = 6 scale_2 (a 26-bit number): exact comparisons
// in fp64, where d (lo + hi) is exact.
__device__ __forceinline__ uint32_t e4m3_rne_ratio_f64(float a, double d) {
  uint32_t c = f32_to_e4m3_rn((float)((double)a / d));
  const double a2 = 2.0 * (double)a;
  if (c < 126u) {
    const double m2 = d * ((double)e4m3_to_f32(c) + (double)e4m3_to_f32(c + 1));
    if (a2 > m2 || (a2 == m2 && (c & 1u))) c += 1;
  }
  if (c > 0u) {
    const double m2 = d * ((double)e4m3_to_f32(c - 1) + (double)e4m3_to_f32(c));
    if (a2 < m2 || (a2 == m2 && (c & 1u))) c -= 1;
  }
  return c;
}

__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(
    long long n_groups, long long groups_per_matrix, const float4* __restrict__ w,
    const float* __restrict__ scale_2, uint4* __restrict__ codes_out,
    uint16_t* __restrict__ s4_out) {
  long long gi = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (; gi < n_groups; gi += stride) {
    const float sc2 = __ldg(scale_2 + gi / groups_per_matrix);
    uint32_t out[4] = {0, 0, 0, 0};
    uint32_t s4pair = 0;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      float x[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 f = __ldg(w + gi * 8 + b * 4 + q);
        x[4 * q + 0] = f.x; x[4 * q + 1] = f.y; x[4 * q + 2] = f.z; x[4 * q + 3] = f.w;
      }
      float bmax = 0.0f;
#pragma unroll
      for (int j = 0; j < 16; ++j) bmax = fmaxf(bmax, fabsf(x[j]));
      uint32_t s4 = 0;
      if (sc2 > 0.0f) s4 = e4m3_rne_ratio_f64(bmax, 6.0 * (double)sc2);
      s4pair |= s4 << (8 * b);
      const double step = (double)e4m3_to_f32(s4) * (double)sc2;  // exact
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        uint32_t c = 0;
        if (step > 0.0) {
          const double a = fabs((double)x[j]);
          c += (a > 0.25 * step);
          c += (a >= 0.75 * step);
          c += (a > 1.25 * step);
          c += (a >= 1.75 * step);
          c += (a > 2.5 * step);
          c += (a >= 3.5 * step);
          c += (a > 5.0 * step);
        }
        c |= (__float_as_uint(x[j]) >> 31) << 3;
        out[2 * b + (j >> 3)] |= c << (4 * (j & 7));
      }
    }
    codes_out[gi] = make_uint4(out[0], out[1], out[2], out[3]);
    s4_out[gi] = (uint16_t)s4pair;
  }
}

static int grid_for(long long n, int block) {
  long long g = (n + block - 1) / block;
  const long long cap = 152LL * 16;  // grid-stride beyond 16 CTAs per SM
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace moet

using namespace moet;

MOET_ERROR_ACCESSOR(moet_internal_error_requant)

extern "C" moet_status moet_requant_2bit(int M, int N, int K, const uint8_t* codes,
                                         const uint8_t* s4, uint32_t* sign, uint32_t* mag,
                                         uint8_t* s16, uint8_t* dcodes, uint8_t* ds4,
                                         moet_stream stream) {
  if (M < 1 || N < 1 || K < 32) return MOET_ERR_SHAPE;
  if (K % 32 != 0) return MOET_ERR_SHAPE;
  if (!codes || !s4 || !sign || !mag || !s16) return MOET_ERR_INVALID_ARG;
  if ((dcodes == nullptr) != (ds4 == nullptr)) return MOET_ERR_INVALID_ARG;
  if (((uintptr_t)codes & 15) || ((uintptr_t)s4 & 1) || ((uintptr_t)sign & 3) ||
      ((uintptr_t)mag & 3) || ((uintptr_t)s16 & 1))
    return MOET_ERR_ALIGN;
  if (dcodes && (((uintptr_t)dcodes & 15) || ((uintptr_t)ds4 & 1))) return MOET_ERR_ALIGN;
  const long long n_groups = (long long)M * N * (K / 32);
  {
    ProfScope ps(MOET_K_REQUANT, (cudaStream_t)stream);
    if (dcodes == nullptr) {
      long long g = (n_groups + 256LL * kGroupsPerIter - 1) / (256LL * kGroupsPerIter);
      if (g > 152LL * 8) g = 152LL * 8;
      requant_planes_kernel<<<(int)g, 256, 0, (cudaStream_t)stream>>>(
          n_groups, (const uint4*)codes, (const uint16_t*)s4, sign, mag, (uint16_t*)s16);
    } else {
      requant_2bit_kernel<<<grid_for(n_groups, 256), 256, 0, (cudaStream_t)stream>>>(
          n_groups, (const uint4*)codes, (const uint16_t*)s4, sign, mag, (uint16_t*)s16,
          (uint4*)dcodes, (uint16_t*)ds4);
    }
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}

extern "C" moet_status moet_quantize_nvfp4(int M, int N, int K, const float* w, float* scale_2,
                                           uint8_t* codes, uint8_t* s4, moet_stream stream) {
  if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return MOET_ERR_SHAPE;
  if (!w || !scale_2 || !codes || !s4) return MOET_ERR_INVALID_ARG;
  if (((uintptr_t)w & 15) || ((uintptr_t)codes & 15) || ((uintptr_t)s4 & 1) ||
      ((uintptr_t)scale_2 & 3))
    return MOET_ERR_ALIGN;
  if (M > 65535) return MOET_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  const long long per4 = (long long)N * K / 4;
  MOET_CUDA_TRY(cudaMemsetAsync(scale_2, 0, sizeof(float) * M, st));
  int gx = (int)((per4 + 255) / 256);
  if (gx > 512) gx = 512;
  {
    ProfScope ps(MOET_K_QUANTIZE, st);
    amax_kernel<<<dim3(gx, M), 256, 0, st>>>(per4, (const float4*)w, (unsigned int*)scale_2);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  {
    ProfScope ps(MOET_K_QUANTIZE, st);
    scale2_kernel<<<(M + 255) / 256, 256, 0, st>>>(M, scale_2);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  const long long gpm = (long long)N * (K / 32);
  const long long n_groups = gpm * M;
  {
    ProfScope ps(MOET_K_QUANTIZE, st);
    quantize_nvfp4_kernel<<<grid_for(n_groups, 256), 256, 0, st>>>(
        n_groups, gpm, (const float4*)w, scale_2, (uint4*)codes, (uint16_t*)s4);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}
