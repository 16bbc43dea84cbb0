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

// ---------------------------------------------------------------- requant, planes only
// Fast path without the delta.  All 16 weights of a block share s4, so
// v = e2m1(code) * s4 is monotone in the magnitude code: max|v| is the value of
// the largest magnitude code, and |v| >= 2 s16 holds exactly for the codes at
// or above a threshold code.  Both s16 and that threshold depend only on
// (largest code, s4); every CTA tabulates them once in shared memory with the
// exact rounding above, and the per-weight work is integer arithmetic on
// eight nibbles at a time.  The kernel is bound by integer issue, so the bit
// gathers run as multiplies (the FMA pipe) and byte permutes.

// Bit 3 of each nibble of t (t = x & 0x88888888) gathered by one multiply: the
// partial products of t * 0x249 (shifts 0, 3, 6, 9) put nibbles 0-3's bits at
// bits 12-15 and nibbles 4-7's at bits 28-31, and every other partial product
// lands on a bit of its own, so no carry reaches those eight.
__device__ __forceinline__ uint32_t gather_bit3(uint32_t t) { return t * 0x249u; }

// The 32 gathered bits of four words (gather_bit3 results r0..r3) in word order.
__device__ __forceinline__ uint32_t assemble_bits(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  const uint32_t p01 = __byte_perm(r0, r1, 0x7351), p23 = __byte_perm(r2, r3, 0x7351);
  const uint32_t a = __byte_perm(p01, p23, 0x5410);   // bytes 1 of r0..r3: nibbles 0-3
  const uint32_t b = __byte_perm(p01, p23, 0x7632);   // bytes 3 of r0..r3: nibbles 4-7
  return ((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
}

// Largest magnitude code (nibble & 7) among the 16 nibbles of (w0, w1), given
// o = w | 0x88888888: its bit 2 is an OR of bit 2, then bits 1 and 0 test
// "some nibble >= t" with a per-nibble subtraction (8 + m - t keeps bit 3 iff
// m >= t, and never borrows across a nibble).
__device__ __forceinline__ uint32_t max_mag_code(uint32_t w0, uint32_t w1, uint32_t o0, uint32_t o1) {
  uint32_t t = ((w0 | w1) & 0x44444444u) ? 4u : 0u;
  uint32_t T = (t + 2u) * 0x11111111u;
  if (((o0 - T) | (o1 - T)) & 0x88888888u) t += 2u;
  T = (t + 1u) * 0x11111111u;
  if (((o0 - T) | (o1 - T)) & 0x88888888u) t += 1u;
  return t;
}

constexpr int kGroupsPerIter = 4;

// Thread t of a CTA handles groups base + u * blockDim + t (u < kGroupsPerIter), so every load
// and store instruction of a warp covers consecutive groups; all loads of an iteration are issued
// before its first use.
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
  const long long span = (long long)blockDim.x * kGroupsPerIter;
  for (long long base = (long long)blockIdx.x * span; base < n_groups; base += (long long)gridDim.x * span) {
    uint4 cw[kGroupsPerIter];
    uint32_t sc[kGroupsPerIter];
#pragma unroll
    for (int u = 0; u < kGroupsPerIter; ++u) {
      const long long gi = base + (long long)u * blockDim.x + threadIdx.x;
      if (gi < n_groups) {
        cw[u] = __ldg(codes + gi);
        sc[u] = __ldg(s4 + gi);
      }
    }
#pragma unroll
    for (int u = 0; u < kGroupsPerIter; ++u) {
      const long long gi = base + (long long)u * blockDim.x + threadIdx.x;
      if (gi >= n_groups) break;
      const uint32_t w[4] = {cw[u].x, cw[u].y, cw[u].z, cw[u].w};
      uint32_t o[4], mr[4], s16pair = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = w[q] | 0x88888888u;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t mc = max_mag_code(w[2 * b], w[2 * b + 1], o[2 * b], o[2 * b + 1]);
        const uint32_t e = lut[((sc[u] >> (8 * b)) & 0x7Fu) * 8 + mc];
        s16pair |= (e & 0xFFu) << (8 * b);
        const uint32_t T = (e >> 8) * 0x11111111u;   // |q| = 3 iff magnitude code >= threshold
        mr[2 * b] = gather_bit3((o[2 * b] - T) & 0x88888888u);
        mr[2 * b + 1] = gather_bit3((o[2 * b + 1] - T) & 0x88888888u);
      }
      sign_out[gi] = assemble_bits(gather_bit3(w[0] & 0x88888888u), gather_bit3(w[1] & 0x88888888u),
                                   gather_bit3(w[2] & 0x88888888u), gather_bit3(w[3] & 0x88888888u));
      mag_out[gi] = assemble_bits(mr[0], mr[1], mr[2], mr[3]);
      s16_out[gi] = (uint16_t)s16pair;
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

// Grid of a grid-stride streaming kernel: at most as many CTAs as can be resident at once (the
// occupancy calculator's CTAs per SM x the SM count), so the work splits evenly over one wave
// instead of leaving a partial wave as a tail.
template <typename Kern>
static int resident_grid(Kern kernel, int block, long long n_threads) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    sms = 152;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  long long g = (n_threads + block - 1) / block;
  const long long cap = (long long)sms * per_sm;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace moet

using namespace moet;

MOET_ERROR_ACCESSOR(moet_internal_error_requant)

// ---------------------------------------------------------------- exact integer arithmetic
// The FP8 and MXFP4 inputs are requantised with integer operations only.  Every number the rule
// touches -- an e4m3 or e2m1 value, an fp32 block scale or power-of-two exponent, scale_2, the
// products of these and the residuals -- is a short integer times a power of two.  Each is held
// as an integer and an exponent, and every rounding decision of the rule is an exact integer
// comparison; no quotient is rounded and reused.

// e4m3 value of code c (0..126) times 2^10, an integer below 2^19: (8 + m) 2^e for exponent
// field e >= 1, m 2^1 for the subnormals (e = 0).
__device__ __forceinline__ uint32_t e4m3_units(uint32_t c) {
  const uint32_t e = c >> 3;
  return ((c & 7u) | (e ? 8u : 0u)) << max(e, 1u);
}

// A finite fp32 |x| as m 2^e with the integer m < 2^24.
__device__ __forceinline__ void f32_parts(float x, uint32_t& m, int& e) {
  const uint32_t b = __float_as_uint(x) & 0x7FFFFFFFu, ef = b >> 23;
  m = (b & 0x7FFFFFu) | (ef ? 0x800000u : 0u);
  e = (int)(ef ? ef : 1u) - 150;
}

// Sign of A 2^a - B 2^b for integers A, B < 2^63.  Unequal positions of the top set bits decide
// it; equal positions leave the larger-exponent integer shiftable onto the other's exponent
// without overflow.
__device__ __forceinline__ int xcmp(uint64_t A, int a, uint64_t B, int b) {
  if (A == 0u || B == 0u) return (int)(A != 0u) - (int)(B != 0u);
  const int ta = a - __clzll((long long)A), tb = b - __clzll((long long)B);
  if (ta != tb) return ta > tb ? 1 : -1;
  if (a > b) A <<= (a - b);
  else B <<= (b - a);
  return (int)(A > B) - (int)(A < B);
}

// x 2^k in fp32, saturating to 0 or infinity (for a first guess only).
__device__ __forceinline__ float pow2_scale(float x, int k) {
  k = max(-250, min(250, k));
  const int k1 = k / 2, k2 = k - k1;
  return x * __int_as_float((k1 + 127) << 23) * __int_as_float((k2 + 127) << 23);
}

// e4m3 satfinite RNE code of (A 2^a) / (D 2^d) for integers A, D < 2^48 (A > 0 with D = 0
// saturates): a guess from the fp32 quotient, within one code of the result, then exact
// comparisons of 2 A 2^a with D (e4m3(c) + e4m3(c + 1)) 2^d, the doubled midpoint with each
// neighbour (D times a sum of two code units stays below 2^48); ties go to the even code.
__device__ __forceinline__ uint32_t e4m3_rne_ratio_x(uint64_t A, int a, uint64_t D, int d) {
  if (A == 0u) return 0u;
  if (D == 0u) return 126u;
  uint32_t c = f32_to_e4m3_rn(pow2_scale(__ull2float_rn(A) / __ull2float_rn(D), a - d));
  if (c < 126u) {
    const int s = xcmp(2u * A, a, D * (e4m3_units(c) + e4m3_units(c + 1u)), d - 10);
    if (s > 0 || (s == 0 && (c & 1u))) c += 1u;
  }
  if (c > 0u) {
    const int s = xcmp(2u * A, a, D * (e4m3_units(c - 1u) + e4m3_units(c)), d - 10);
    if (s < 0 || (s == 0 && (c & 1u))) c -= 1u;
  }
  return c;
}

// Magnitude code of e2m1 satfinite RNE(|d| / step) from a = 4 |d| and the step's multiples
// t = (1, 3, 5, 7, 10, 14, 20) x step, all in one integer unit: the code counts the midpoints
// (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) x step that |d| passes, strictly for the even codes'
// upper midpoints and inclusively for the odd ones' (ties to the even code), by bisection.
struct StepMultiples {
  uint64_t t[7];
};

__device__ __forceinline__ StepMultiples step_multiples(uint64_t S) {
  return {{S, 3u * S, 5u * S, 7u * S, 10u * S, 14u * S, 20u * S}};
}

__device__ __forceinline__ uint32_t e2m1_mag_x(uint64_t a, const StepMultiples& m) {
  uint32_t c = a >= m.t[3] ? 4u : 0u;
  c += (c ? a >= m.t[5] : a >= m.t[1]) ? 2u : 0u;
  const uint64_t u = c == 0u ? m.t[0] : c == 2u ? m.t[2] : c == 4u ? m.t[4] : m.t[6];
  return c + (a > u ? 1u : 0u);
}

// The largest key of a CTA's threads (keys >= 0), valid in thread 0.
__device__ __forceinline__ uint64_t cta_max_u64(uint64_t v) {
  __shared__ uint64_t red[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  }
  return v;
}

// scale_2 = fp32(fp64(amax) / 1344) from amax's fp64 bit pattern (for a non-negative double the
// pattern orders like the value, so the largest pattern is the amax).
__device__ __forceinline__ float scale2_from_key(uint64_t key) {
  return __double2float_rn(__ddiv_rn(__longlong_as_double((long long)key), 1344.0));
}

// The amax pass runs P CTAs per matrix.  With P = 1 the CTA writes scale_2 itself; otherwise each
// writes its largest key into the first 2P words of the matrix's sign plane (written over later
// by the requant kernel) and amax_finalize_kernel reduces them.
__device__ __forceinline__ void amax_store(int m, uint64_t key, uint32_t* sign_scratch, long long words,
                                           float* scale_2) {
  if (threadIdx.x != 0) return;
  if (gridDim.x == 1) {
    scale_2[m] = scale2_from_key(key);
  } else {
    uint32_t* s = sign_scratch + (size_t)m * words + 2 * blockIdx.x;
    s[0] = (uint32_t)key;
    s[1] = (uint32_t)(key >> 32);
  }
}

// One warp per matrix: the largest of the P partial keys, then scale_2.
__global__ void amax_finalize_kernel(int M, int P, long long words, const uint32_t* __restrict__ sign_scratch,
                                     float* __restrict__ scale_2) {
  const int m = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (m >= M) return;
  const uint32_t* s = sign_scratch + (size_t)m * words;
  uint64_t v = 0;
  for (int p = lane; p < P; p += 32) v = max(v, (uint64_t)s[2 * p] | ((uint64_t)s[2 * p + 1] << 32));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) scale_2[m] = scale2_from_key(v);
}

// Grid-stride walk over the 32-weight groups of M matrices of [N, K/32] groups with the matrix,
// row and group-in-row indices carried along instead of divided out per step.
struct GroupWalk {
  long long gi;
  int m, n, j;
  int dm, dn, dj;
  __device__ __forceinline__ void init(long long start, long long stride, int N, int Kg) {
    const long long gpm = (long long)N * Kg;
    gi = start;
    m = (int)(start / gpm);
    const long long r = start - (long long)m * gpm;
    n = (int)(r / Kg);
    j = (int)(r - (long long)n * Kg);
    dm = (int)(stride / gpm);
    const long long dr = stride - (long long)dm * gpm;
    dn = (int)(dr / Kg);
    dj = (int)(dr - (long long)dn * Kg);
  }
  __device__ __forceinline__ void next(long long stride, int N, int Kg) {
    gi += stride;
    j += dj;
    n += dn;
    if (j >= Kg) { j -= Kg; ++n; }
    m += dm;
    if (n >= N) { n -= N; ++m; }
  }
};

// ---------------------------------------------------------------- FP8 block-quant input
// README "How it fits -- 2-bit experts at FP4 quality", last paragraph: FP8 block-quant
// checkpoints (an e4m3 code per weight, one fp32 scale per 128 x 128 block) are requantised to
// the same planes.  W = e4m3(code) * bscale is V(code) Mb 2^(Eb - 10) with V < 2^19 the code's
// units and bscale = Mb 2^Eb, so the rule is the NVFP4 one applied to these exact weights with
// scale_2 = fp32(fp64(amax) / 1344).
constexpr int kFp8Block = 128;

// amax key of 16 e4m3 codes under one block scale: the fp64 bit pattern of e4m3(top) * bscale
// (the e4m3 magnitude order is the code order), built from the 43-bit integer product.
__device__ __forceinline__ uint64_t fp8_chunk_key(uint4 c, uint32_t bm, int be) {
  uint32_t x = __vmaxu4(__vmaxu4(c.x & 0x7F7F7F7Fu, c.y & 0x7F7F7F7Fu), __vmaxu4(c.z & 0x7F7F7F7Fu, c.w & 0x7F7F7F7Fu));
  x = __vmaxu4(x, x >> 16);
  x = __vmaxu4(x, x >> 8);
  const uint64_t p = (uint64_t)e4m3_units(x & 0xFFu) * bm;
  if (p == 0u) return 0u;
  const int lz = __clzll((long long)p);
  const uint64_t frac = ((p << lz) << 1) >> 12;                       // the 52 bits below the top
  return ((uint64_t)(63 - lz + be - 10 + 1023) << 52) | frac;
}

// grid (P, M): CTA p of matrix m takes 16-code chunks [p C / P, (p + 1) C / P) of its C chunks.
__global__ void __launch_bounds__(256) fp8_amax_kernel(int N, int K, const uint8_t* __restrict__ codes,
                                                       const float* __restrict__ bscale, float* __restrict__ scale_2,
                                                       uint32_t* __restrict__ sign_scratch) {
  const int m = blockIdx.y, P = gridDim.x, p = blockIdx.x;
  const int Kc = K / 16;
  const long long C = (long long)N * Kc;
  const int nbn = (N + kFp8Block - 1) / kFp8Block, nbk = (K + kFp8Block - 1) / kFp8Block;
  const long long c0 = C * p / P, c1 = C * (p + 1) / P;
  const uint4* cm = reinterpret_cast<const uint4*>(codes) + (size_t)m * C;
  const float* bm_ = bscale + (size_t)m * nbn * nbk;
  const int stride = blockDim.x, sn = stride / Kc, sj = stride - sn * Kc;
  long long i = c0 + threadIdx.x;
  int n = (int)(i / Kc), j = (int)(i - (long long)n * Kc);
  uint64_t key = 0;
  for (; i < c1; i += stride) {
    uint32_t bmant;
    int bexp;
    f32_parts(__ldg(bm_ + (size_t)(n >> 7) * nbk + (j >> 3)), bmant, bexp);
    key = max(key, fp8_chunk_key(__ldg(cm + i), bmant, bexp));
    j += sj;
    n += sn;
    if (j >= Kc) { j -= Kc; ++n; }
  }
  key = cta_max_u64(key);
  amax_store(m, key, sign_scratch, (long long)N * (K / 32), scale_2);
}

struct Block16 {
  uint32_t mag, s16, dlo, dhi, ds4;
};

// The rule on one block of 16 e4m3 codes (four words, byte j = weight j) under one block scale
// bm 2^be, with the codes' sign bits (bit j) and scale_2 = sm 2^se: s16, the magnitude bits and,
// when `delta` is set, the 16 delta codes (two words, low nibble first) and the delta scale.
// Weights and levels share the unit 2^eu, eu = min(be, se) - 10, in which |W_j| = V(c_j) mbs and
// the level is lu; both stay below 2^46 because scale_2 comes from the matrix's amax (so
// bmax <= 1344 scale_2) and a nonzero s16 is at most 2/3 of bmax / scale_2.
__device__ __forceinline__ Block16 fp8_rule_16(const uint32_t (&w)[4], uint32_t sbits, uint32_t bm, int be,
                                               uint32_t sm, int se, bool delta) {
  Block16 r = {0u, 0u, 0u, 0u, 0u};
  uint32_t wm[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) wm[q] = w[q] & 0x7F7F7F7Fu;
  uint32_t x = __vmaxu4(__vmaxu4(wm[0], wm[1]), __vmaxu4(wm[2], wm[3]));
  x = __vmaxu4(x, x >> 16);
  x = __vmaxu4(x, x >> 8);
  const uint32_t cmax = x & 0xFFu;
  r.s16 = e4m3_rne_ratio_x((uint64_t)e4m3_units(cmax) * bm, be - 10, 3ull * sm, se);
  const int eu = min(be, se) - 10;
  const int sw = min(be - 10 - eu, 63), sl = min(se - 10 - eu, 63);
  const uint64_t mbs = (uint64_t)bm << sw;
  const uint64_t lu = r.s16 ? ((uint64_t)e4m3_units(r.s16) * sm) << sl : 0ull;
  // |q| = 3 iff the code is at least thr, the first code with V(c) mbs >= 2 lu: a guess from the
  // fp32 ratio (the nearest code, at most one below), corrected exactly
  uint32_t thr = 0u;
  if (lu != 0u) {
    thr = f32_to_e4m3_rn(__ull2float_rn(2u * lu) / __ull2float_rn(mbs) * 0x1p-10f);
    if ((uint64_t)e4m3_units(thr) * mbs < 2u * lu) thr += 1u;          // 127: no code reaches it
    if (thr > 0u && (uint64_t)e4m3_units(thr - 1u) * mbs >= 2u * lu) thr -= 1u;
  }
  const uint32_t T4 = thr * 0x01010101u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t t = __vcmpgeu4(wm[q], T4) & 0x80808080u;
    r.mag |= ((t * 0x204081u) >> 28) << (4 * q);                      // byte bits 7 -> bits 28..31
  }
  if (!delta) return r;
  const uint64_t l3 = 3u * lu;
  int64_t d[16];
  uint64_t dmax = 0u;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t c = (wm[j >> 2] >> (8 * (j & 3))) & 0xFFu;
    d[j] = (int64_t)((uint64_t)e4m3_units(c) * mbs - (((r.mag >> j) & 1u) ? l3 : lu));
    dmax = max(dmax, (uint64_t)(d[j] < 0 ? -d[j] : d[j]));
  }
  r.ds4 = e4m3_rne_ratio_x(dmax, eu, 6ull * sm, se);
  if (r.ds4 == 0u) return r;                                           // all delta codes +0
  const StepMultiples st = step_multiples(((uint64_t)e4m3_units(r.ds4) * sm) << sl);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const bool neg = d[j] < 0;
    const uint32_t dm = e2m1_mag_x(4u * (uint64_t)(neg ? -d[j] : d[j]), st);
    const uint32_t code = dm | ((dm != 0u && (neg != (bool)((sbits >> j) & 1u))) ? 8u : 0u);
    if (j < 8) r.dlo |= code << (4 * j);
    else r.dhi |= code << (4 * (j - 8));
  }
  return r;
}

// One thread per 32-weight group of a row: 32 codes in, one sign and one magnitude word, two s16
// bytes (and 16 delta code bytes + two delta scale bytes) out.
__global__ void __launch_bounds__(256) requant_fp8_kernel(
    int M, int N, int K, const uint8_t* __restrict__ codes, const float* __restrict__ bscale,
    const float* __restrict__ scale_2, uint32_t* __restrict__ sign_out, uint32_t* __restrict__ mag_out,
    uint16_t* __restrict__ s16_out, uint4* __restrict__ dcodes_out, uint16_t* __restrict__ ds4_out) {
  const int Kg = K / 32;
  const long long n_groups = (long long)M * N * Kg;
  const int nbn = (N + kFp8Block - 1) / kFp8Block, nbk = (K + kFp8Block - 1) / kFp8Block;
  const bool delta = dcodes_out != nullptr;
  const long long stride = (long long)gridDim.x * blockDim.x;
  GroupWalk g;
  g.init((long long)blockIdx.x * blockDim.x + threadIdx.x, stride, N, Kg);
  int m_sc = -1;
  uint32_t sm = 0u;
  int se = 0;
  for (; g.gi < n_groups; g.next(stride, N, Kg)) {
    if (g.m != m_sc) {
      f32_parts(__ldg(scale_2 + g.m), sm, se);
      m_sc = g.m;
    }
    uint32_t bm;
    int be;
    f32_parts(__ldg(bscale + ((size_t)g.m * nbn + (g.n >> 7)) * nbk + (g.j >> 2)), bm, be);
    const uint4* src = reinterpret_cast<const uint4*>(codes) + g.gi * 2;
    const uint4 c0 = __ldg(src), c1 = __ldg(src + 1);
    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    // sign bits: bit 7 of every byte, gathered four bytes at a time
    uint32_t sign = 0u;
#pragma unroll
    for (int q = 0; q < 8; ++q) sign |= (((words[q] & 0x80808080u) * 0x204081u) >> 28) << (4 * q);
    uint32_t mag = 0u, s16pair = 0u, ds4pair = 0u, dw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t wb[4] = {words[4 * b], words[4 * b + 1], words[4 * b + 2], words[4 * b + 3]};
      const Block16 o = fp8_rule_16(wb, sign >> (16 * b), bm, be, sm, se, delta);
      mag |= o.mag << (16 * b);
      s16pair |= o.s16 << (8 * b);
      ds4pair |= o.ds4 << (8 * b);
      dw[2 * b] = o.dlo;
      dw[2 * b + 1] = o.dhi;
    }
    sign_out[g.gi] = sign;
    mag_out[g.gi] = mag;
    s16_out[g.gi] = (uint16_t)s16pair;
    if (delta) {
      dcodes_out[g.gi] = make_uint4(dw[0], dw[1], dw[2], dw[3]);
      ds4_out[g.gi] = (uint16_t)ds4pair;
    }
  }
}

// ---------------------------------------------------------------- MXFP4 (FP4 experts) input
// README "How it fits -- 2-bit experts at FP4 quality", last paragraph: checkpoints with FP4
// experts load by a code remap.  Read as OCP MXFP4 -- an e2m1 code per weight (two per byte, low
// nibble = even k) and one E8M0 scale 2^(e - 127) per 32 weights along K -- remapped by the same
// rule as the FP8 input: W = e2m1(code) 2^(e - 127) = u2(code) 2^(e - 128) with the integer
// u2 = 2 e2m1 in {0, 1, 2, 3, 4, 6, 8, 12}, and scale_2 = fp32(fp64(amax) / 1344).

// u2 of magnitude code c (0..7).
__device__ __forceinline__ uint32_t e2m1_units2(uint32_t c) {
  return c < 4u ? c : (2u + (c & 1u)) << ((c >> 1) - 1u);
}

// Bit v of the result: some nibble of the 16 in (a, b) has magnitude code v.  A byte permute with
// the table {1, 2, 4, .., 128} turns four 3-bit codes (the selector's four low nibbles) into four
// one-hot bytes; the OR of the 16 one-hot bytes is the set.
__device__ __forceinline__ uint32_t codes_present(uint32_t a, uint32_t b) {
  constexpr uint32_t kOneHotLo = 0x08040201u, kOneHotHi = 0x80402010u;
  const uint32_t ma = a & 0x77777777u, mb = b & 0x77777777u;
  const uint32_t r = prmt(kOneHotLo, kOneHotHi, ma) | prmt(kOneHotLo, kOneHotHi, ma >> 16) |
                     prmt(kOneHotLo, kOneHotHi, mb) | prmt(kOneHotLo, kOneHotHi, mb >> 16);
  const uint32_t x = r | (r >> 16);
  return (x | (x >> 8)) & 0xFFu;
}

// amax key of one 32-weight group: the fp64 bit pattern of e2m1(top code) 2^(e - 127), built
// from the code's binade and half-step bit.
__device__ __forceinline__ uint64_t mxfp4_group_key(uint4 c, uint32_t e) {
  const uint32_t pres = codes_present(c.x, c.y) | codes_present(c.z, c.w);
  const uint32_t top = 31u - (uint32_t)__clz(pres | 1u);
  if (top == 0u) return 0u;
  const int binade = (int)(top >> 1) - 1;                              // 0.5: -1, 1 and 1.5: 0, ...
  const uint64_t half = (top >= 2u && (top & 1u)) ? (1ull << 51) : 0ull;
  return ((uint64_t)((int)e - 127 + binade + 1023) << 52) | half;
}

// grid (P, M): CTA p of matrix m takes groups [p G / P, (p + 1) G / P) of its G groups.
__global__ void __launch_bounds__(256) mxfp4_amax_kernel(long long G, const uint4* __restrict__ codes,
                                                         const uint8_t* __restrict__ e8m0,
                                                         float* __restrict__ scale_2,
                                                         uint32_t* __restrict__ sign_scratch) {
  const int m = blockIdx.y, P = gridDim.x, p = blockIdx.x;
  const long long c0 = G * p / P, c1 = G * (p + 1) / P;
  const uint4* cm = codes + (size_t)m * G;
  const uint8_t* em = e8m0 + (size_t)m * G;
  uint64_t key = 0;
  for (long long i = c0 + threadIdx.x; i < c1; i += blockDim.x)
    key = max(key, mxfp4_group_key(__ldg(cm + i), __ldg(em + i)));
  key = cta_max_u64(key);
  amax_store(m, key, sign_scratch, G, scale_2);
}

// Delta codes of the 8 nibbles of w from per-code tables: byte c of (tlo, thi) is the delta code
// of a positive weight with magnitude code c, byte c of (flo, fhi) is 8 when that code is nonzero
// (a negative weight flips it).  Even and odd nibbles go through one byte permute each.
__device__ __forceinline__ uint32_t delta_from_tables(uint32_t w, uint32_t tlo, uint32_t thi, uint32_t flo,
                                                      uint32_t fhi) {
  const uint32_t ce = w & 0x07070707u, co = (w >> 4) & 0x07070707u;   // codes of nibbles 0,2,4,6 / 1,3,5,7
  const uint32_t se = (ce | (ce >> 4)) & 0x00FF00FFu, so = (co | (co >> 4)) & 0x00FF00FFu;
  const uint32_t sel_e = (se | (se >> 8)) & 0xFFFFu, sel_o = (so | (so >> 8)) & 0xFFFFu;
  const uint32_t de = prmt(tlo, thi, sel_e) ^ (prmt(flo, fhi, sel_e) & (w & 0x08080808u));
  const uint32_t dd = prmt(tlo, thi, sel_o) ^ (prmt(flo, fhi, sel_o) & ((w >> 4) & 0x08080808u));
  return de | (dd << 4);
}

// One thread per 32-weight group (16 code bytes and one exponent byte in, like the FP8 kernel
// out).  All 32 weights share 2^(e - 128), so within a 16-block every decision of the rule is a
// function of the 3-bit magnitude code: the rule runs once per block over the 8 codes (s16 from
// the largest code present, the |q| = 3 threshold code, the delta scale from the codes present,
// the 8 delta codes) in the unit 2^eu, eu = min(e - 128, se - 10), where the weights u2(c) << sw
// and the level stay below 2^46 (as in the FP8 rule); the 16 weights take byte permutes only.
// Codes above the block's largest never occur in it, so their table entries are not used.
__global__ void __launch_bounds__(256) requant_mxfp4_kernel(
    int M, long long gpm, const uint4* __restrict__ codes, const uint8_t* __restrict__ e8m0,
    const float* __restrict__ scale_2, uint32_t* __restrict__ sign_out, uint32_t* __restrict__ mag_out,
    uint16_t* __restrict__ s16_out, uint4* __restrict__ dcodes_out, uint16_t* __restrict__ ds4_out) {
  const long long n_groups = (long long)M * gpm;
  const bool delta = dcodes_out != nullptr;
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long gi = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  int m = (int)(gi / gpm);
  long long r = gi - (long long)m * gpm;
  const int dm = (int)(stride / gpm);
  const long long dr = stride - (long long)dm * gpm;
  int m_sc = -1;
  uint32_t sm = 0u;
  int se = 0;
  for (; gi < n_groups; gi += stride) {
    if (m != m_sc) {
      f32_parts(__ldg(scale_2 + m), sm, se);
      m_sc = m;
    }
    const int ew = (int)__ldg(e8m0 + gi) - 128;                        // weights: u2(c) 2^ew
    const uint4 cw = __ldg(codes + gi);
    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
    const int eu = min(ew, se - 10);
    const int sw = min(ew - eu, 63), sl = min(se - 10 - eu, 63);
    uint32_t mr[4], s16pair = 0, ds4pair = 0, dw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t wa = w[2 * b], wb = w[2 * b + 1];
      const uint32_t pres = codes_present(wa, wb);
      const uint32_t cmax = 31u - (uint32_t)__clz(pres);               // pres != 0: 16 codes
      const uint32_t s16 = e4m3_rne_ratio_x(e2m1_units2(cmax), ew, 3ull * sm, se);
      const uint64_t lu = s16 ? ((uint64_t)e4m3_units(s16) * sm) << sl : 0ull;
      uint64_t wu[8];
      uint32_t thr = 0;                                                  // |q| = 3 iff code >= thr
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        wu[c] = (uint64_t)e2m1_units2((uint32_t)c) << sw;
        thr += ((uint32_t)c <= cmax && wu[c] < 2u * lu) ? 1u : 0u;
      }
      s16pair |= s16 << (8 * b);
      const uint32_t T = thr * 0x11111111u;
      mr[2 * b] = gather_bit3(((wa | 0x88888888u) - T) & 0x88888888u);
      mr[2 * b + 1] = gather_bit3(((wb | 0x88888888u) - T) & 0x88888888u);
      if (delta) {
        int64_t d[8];
        uint64_t dmax = 0u;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          d[c] = (int64_t)(wu[c] - ((uint32_t)c >= thr ? 3u * lu : lu));
          if ((pres >> c) & 1u) dmax = max(dmax, (uint64_t)(d[c] < 0 ? -d[c] : d[c]));
        }
        const uint32_t ds4 = e4m3_rne_ratio_x(dmax, eu, 6ull * sm, se);
        uint32_t tlo = 0, thi = 0, flo = 0, fhi = 0;
        if (ds4 != 0u) {
          const StepMultiples st = step_multiples(((uint64_t)e4m3_units(ds4) * sm) << sl);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const bool neg = d[c] < 0;
            const uint32_t dmg = e2m1_mag_x(4u * (uint64_t)(neg ? -d[c] : d[c]), st);
            const uint32_t e = dmg | ((neg && dmg != 0u) ? 8u : 0u);     // for a positive weight
            const uint32_t f = dmg != 0u ? 8u : 0u;
            if (c < 4) { tlo |= e << (8 * c); flo |= f << (8 * c); }
            else { thi |= e << (8 * (c - 4)); fhi |= f << (8 * (c - 4)); }
          }
        }
        ds4pair |= ds4 << (8 * b);
        dw[2 * b] = delta_from_tables(wa, tlo, thi, flo, fhi);
        dw[2 * b + 1] = delta_from_tables(wb, tlo, thi, flo, fhi);
      }
    }
    sign_out[gi] = assemble_bits(gather_bit3(w[0] & 0x88888888u), gather_bit3(w[1] & 0x88888888u),
                                 gather_bit3(w[2] & 0x88888888u), gather_bit3(w[3] & 0x88888888u));
    mag_out[gi] = assemble_bits(mr[0], mr[1], mr[2], mr[3]);
    s16_out[gi] = (uint16_t)s16pair;
    if (delta) {
      dcodes_out[gi] = make_uint4(dw[0], dw[1], dw[2], dw[3]);
      ds4_out[gi] = (uint16_t)ds4pair;
    }
    m += dm;
    r += dr;
    if (r >= gpm) { r -= gpm; ++m; }
  }
}

// ---------------------------------------------------------------- NVFP4 -> planes + delta by tables
// All 16 weights of an NVFP4 block share s4, so every decision of the rule inside a block --
// s16 (from the largest magnitude code), the |q| = 3 threshold code, the delta scale (from the
// largest |d| over the magnitude codes present) and the delta code of each magnitude code -- is a
// function of (s4, the set of magnitude codes present).  requant_delta_lut_kernel evaluates the
// rule once per such pair into g_requant_lut, in fp32, exactly: v = e2m1 x s4 and q s16 are short
// dyadics a few binades apart, so d = v - q s16 is exact, and both e4m3 roundings and the e2m1
// rounding compare doubled midpoints exactly; requant_delta_kernel then gives each weight its planes and delta code with
// integer operations (presence by borrow tests, bit gathers by multiplies, codes by byte
// permutes).  The table is rebuilt by every call (32 K entries, a few microseconds), so nothing
// depends on state left by an earlier call.
//   entry (s4 & 0x7F) * 256 + present:  x, y = delta code bytes of magnitude codes 0-3 / 4-7
//   for a positive weight;  z = s16 | ds4 << 8 | threshold code << 16
constexpr int kLutEntries = 128 * 256;
static __device__ uint4 g_requant_lut[kLutEntries];

__global__ void __launch_bounds__(256) requant_delta_lut_kernel() {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= kLutEntries) return;
  const uint32_t sc = (uint32_t)i >> 8, pres = (uint32_t)i & 0xFFu;
  if (pres == 0u) {                       // never looked up: a block always holds some code
    g_requant_lut[i] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const float s4f = e4m3_to_f32(sc);
  const uint32_t mc = 31u - (uint32_t)__clz(pres);
  const uint32_t s16 = e4m3_rne_ratio_small(e2m1_mag_value(mc) * s4f, 3.0f);
  const float s16f = e4m3_to_f32(s16);
  uint32_t thr = 0;
#pragma unroll
  for (uint32_t c = 0; c < 8; ++c) thr += (e2m1_mag_value(c) * s4f < 2.0f * s16f) ? 1u : 0u;
  float d[8];
  float dmax = 0.0f;
#pragma unroll
  for (uint32_t c = 0; c < 8; ++c) {
    const float q = (c >= thr ? 3.0f : 1.0f) * s16f;
    d[c] = e2m1_mag_value(c) * s4f - q;                      // exact (short dyadics)
    if ((pres >> c) & 1u) dmax = fmaxf(dmax, fabsf(d[c]));
  }
  const uint32_t ds4 = e4m3_rne_ratio_small(dmax, 6.0f);
  const float dsf = e4m3_to_f32(ds4);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (uint32_t c = 0; c < 8; ++c) {
    const uint32_t dm = dsf > 0.0f ? e2m1_rne_mag(fabsf(d[c]), dsf) : 0u;
    const uint32_t code = dm | ((d[c] < 0.0f && dm != 0u) ? 8u : 0u);
    if (c < 4) lo |= code << (8 * c);
    else hi |= code << (8 * (c - 4));
  }
  g_requant_lut[i] = make_uint4(lo, hi, s16 | (ds4 << 8) | (thr << 16), 0u);
}

// Thread t of a CTA handles groups base + u * blockDim + t (u < kGroupsPerIter), as the planes-only
// kernel; per 16-block one table entry.
__global__ void __launch_bounds__(256) requant_delta_kernel(
    long long n_groups, const uint4* __restrict__ codes, const uint16_t* __restrict__ s4,
    uint32_t* __restrict__ sign_out, uint32_t* __restrict__ mag_out, uint16_t* __restrict__ s16_out,
    uint4* __restrict__ dcodes_out, uint16_t* __restrict__ ds4_out) {
  const long long span = (long long)blockDim.x * kGroupsPerIter;
  for (long long base = (long long)blockIdx.x * span; base < n_groups; base += (long long)gridDim.x * span) {
    uint4 cw[kGroupsPerIter];
    uint32_t sc[kGroupsPerIter];
#pragma unroll
    for (int u = 0; u < kGroupsPerIter; ++u) {
      const long long gi = base + (long long)u * blockDim.x + threadIdx.x;
      if (gi < n_groups) {
        cw[u] = __ldg(codes + gi);
        sc[u] = __ldg(s4 + gi);
      }
    }
#pragma unroll
    for (int u = 0; u < kGroupsPerIter; ++u) {
      const long long gi = base + (long long)u * blockDim.x + threadIdx.x;
      if (gi >= n_groups) break;
      const uint32_t w[4] = {cw[u].x, cw[u].y, cw[u].z, cw[u].w};
      uint32_t mr[4], dw[4], s16pair = 0, ds4pair = 0;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t wa = w[2 * b], wb = w[2 * b + 1];
        const uint32_t pres = codes_present(wa, wb);
        const uint4 e = g_requant_lut[(((sc[u] >> (8 * b)) & 0x7Fu) << 8) | pres];
        s16pair |= (e.z & 0xFFu) << (8 * b);
        ds4pair |= ((e.z >> 8) & 0xFFu) << (8 * b);
        const uint32_t T = (e.z >> 16) * 0x11111111u;             // |q| = 3 iff magnitude code >= threshold
        mr[2 * b] = gather_bit3(((wa | 0x88888888u) - T) & 0x88888888u);
        mr[2 * b + 1] = gather_bit3(((wb | 0x88888888u) - T) & 0x88888888u);
        // byte c of (flo, fhi) = 8 when magnitude code c has a nonzero delta magnitude
        const uint32_t flo = ((e.x & 0x07070707u) + 0x07070707u) & 0x08080808u;
        const uint32_t fhi = ((e.y & 0x07070707u) + 0x07070707u) & 0x08080808u;
        dw[2 * b] = delta_from_tables(wa, e.x, e.y, flo, fhi);
        dw[2 * b + 1] = delta_from_tables(wb, e.x, e.y, flo, fhi);
      }
      sign_out[gi] = assemble_bits(gather_bit3(w[0] & 0x88888888u), gather_bit3(w[1] & 0x88888888u),
                                   gather_bit3(w[2] & 0x88888888u), gather_bit3(w[3] & 0x88888888u));
      mag_out[gi] = assemble_bits(mr[0], mr[1], mr[2], mr[3]);
      s16_out[gi] = (uint16_t)s16pair;
      dcodes_out[gi] = make_uint4(dw[0], dw[1], dw[2], dw[3]);
      ds4_out[gi] = (uint16_t)ds4pair;
    }
  }
}

// CTAs per matrix of the amax pass: up to 128, each leaving its partial key in two words of the
// matrix's sign plane, so at most half the plane's words; one CTA (writing scale_2 itself) for
// planes of fewer than four words.
static int amax_parts(long long sign_words) {
  const long long p = sign_words / 2;
  return (int)(p < 2 ? 1 : (p > 128 ? 128 : p));
}

extern "C" moet_status moet_requant_mxfp4_2bit(int M, int N, int K, const uint8_t* codes, const uint8_t* e8m0,
                                               float* scale_2, uint32_t* sign, uint32_t* mag, uint8_t* s16,
                                               uint8_t* dcodes, uint8_t* ds4, moet_stream stream) {
  if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return MOET_ERR_SHAPE;
  if (!codes || !e8m0 || !scale_2 || !sign || !mag || !s16) return MOET_ERR_INVALID_ARG;
  if ((dcodes == nullptr) != (ds4 == nullptr)) return MOET_ERR_INVALID_ARG;
  if (((uintptr_t)codes & 15) || ((uintptr_t)scale_2 & 3) || ((uintptr_t)sign & 3) ||
      ((uintptr_t)mag & 3) || ((uintptr_t)s16 & 1))
    return MOET_ERR_ALIGN;
  if (dcodes && (((uintptr_t)dcodes & 15) || ((uintptr_t)ds4 & 1))) return MOET_ERR_ALIGN;
  if (M > 65535) return MOET_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  const long long gpm = (long long)N * (K / 32);
  const int P = amax_parts(gpm);
  {
    ProfScope ps(MOET_K_REQUANT, st);
    mxfp4_amax_kernel<<<dim3(P, M), 256, 0, st>>>(gpm, (const uint4*)codes, e8m0, scale_2, sign);
    if (P > 1) amax_finalize_kernel<<<(M + 7) / 8, 256, 0, st>>>(M, P, gpm, sign, scale_2);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  {
    ProfScope ps(MOET_K_REQUANT, st);
    const int g = resident_grid(requant_mxfp4_kernel, 256, gpm * M);
    requant_mxfp4_kernel<<<g, 256, 0, st>>>(M, gpm, (const uint4*)codes, e8m0, scale_2, sign, mag, (uint16_t*)s16,
                                            (uint4*)dcodes, (uint16_t*)ds4);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}

extern "C" moet_status moet_requant_fp8_2bit(int M, int N, int K, const uint8_t* codes, const float* bscale,
                                             float* scale_2, uint32_t* sign, uint32_t* mag, uint8_t* s16,
                                             uint8_t* dcodes, uint8_t* ds4, moet_stream stream) {
  if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return MOET_ERR_SHAPE;
  if (!codes || !bscale || !scale_2 || !sign || !mag || !s16) return MOET_ERR_INVALID_ARG;
  if ((dcodes == nullptr) != (ds4 == nullptr)) return MOET_ERR_INVALID_ARG;
  if (((uintptr_t)codes & 15) || ((uintptr_t)bscale & 3) || ((uintptr_t)scale_2 & 3) ||
      ((uintptr_t)sign & 3) || ((uintptr_t)mag & 3) || ((uintptr_t)s16 & 1))
    return MOET_ERR_ALIGN;
  if (dcodes && (((uintptr_t)dcodes & 15) || ((uintptr_t)ds4 & 1))) return MOET_ERR_ALIGN;
  if (M > 65535) return MOET_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  const long long gpm = (long long)N * (K / 32);
  const long long n_groups = (long long)M * gpm;
  const int P = amax_parts(gpm);
  {
    ProfScope ps(MOET_K_REQUANT, st);
    fp8_amax_kernel<<<dim3(P, M), 256, 0, st>>>(N, K, codes, bscale, scale_2, sign);
    if (P > 1) amax_finalize_kernel<<<(M + 7) / 8, 256, 0, st>>>(M, P, gpm, sign, scale_2);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  {
    ProfScope ps(MOET_K_REQUANT, st);
    const int g = resident_grid(requant_fp8_kernel, 256, n_groups);
    requant_fp8_kernel<<<g, 256, 0, st>>>(M, N, K, codes, bscale, scale_2, sign, mag, (uint16_t*)s16,
                                          (uint4*)dcodes, (uint16_t*)ds4);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}

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
      const int g = resident_grid(requant_planes_kernel, 256, (n_groups + kGroupsPerIter - 1) / kGroupsPerIter);
      requant_planes_kernel<<<g, 256, 0, (cudaStream_t)stream>>>(
          n_groups, (const uint4*)codes, (const uint16_t*)s4, sign, mag, (uint16_t*)s16);
    } else {
      requant_delta_lut_kernel<<<kLutEntries / 256, 256, 0, (cudaStream_t)stream>>>();
      const int g = resident_grid(requant_delta_kernel, 256, (n_groups + kGroupsPerIter - 1) / kGroupsPerIter);
      requant_delta_kernel<<<g, 256, 0, (cudaStream_t)stream>>>(
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
    const int g = resident_grid(quantize_nvfp4_kernel, 256, n_groups);
    quantize_nvfp4_kernel<<<g, 256, 0, st>>>(
        n_groups, gpm, (const float4*)w, scale_2, (uint4*)codes, (uint16_t*)s4);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}
