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

// ---------------------------------------------------------------- FP8 block-quant input
// README "How it fits -- 2-bit experts at FP4 quality", last paragraph: FP8 block-quant
// checkpoints (an e4m3 code per weight, one fp32 scale per 128 x 128 block) are requantised to
// the same planes.  W = e4m3(code) * block scale is exact in fp64 (4 + 24 significant bits), so
// the rule is the NVFP4 one applied to W with scale_2 = fp32(fp64(amax) / 1344): every ratio is
// rounded once by exact fp64 comparisons (all products of the short significands involved fit in
// fp64's 53 bits), no quotient is rounded and reused.
constexpr int kFp8Block = 128;

// e4m3 satfinite RNE of a / d for a >= 0, d > 0, both exact in fp64 with d * (two neighbouring
// e4m3 values) exact: a guess from a * inv_d (inv_d ~ 1 / d; the guess is within one code, the
// quotient itself is never used), corrected against the doubled midpoints.
__device__ __forceinline__ uint32_t e4m3_rne_ratio_dd(double a, double d, double inv_d) {
  if (!(a > 0.0)) return 0u;                          // zero (also for an all-zero matrix, d = 0)
  uint32_t c = f32_to_e4m3_rn((float)(a * inv_d));
  const double a2 = 2.0 * a;
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

// e2m1 magnitude code of RNE(a / s), saturating, ties to even, by exact comparison with the seven
// midpoints of the e2m1 grid scaled by s, t[i] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5}[i] * s
// (exact in fp64): the code is the number of thresholds a passes, > for even i and >= for odd i
// (ties to the even code), found by bisection.
__device__ __forceinline__ uint32_t e2m1_rne_mag_bisect(double a, const double (&t)[7]) {
  uint32_t c = a >= t[3] ? 4u : 0u;
  c += (c ? a >= t[5] : a >= t[1]) ? 2u : 0u;
  const double u = c == 0u ? t[0] : c == 2u ? t[2] : c == 4u ? t[4] : t[6];
  return c + (a > u ? 1u : 0u);
}

__device__ __forceinline__ void e2m1_thresholds(double step, double (&t)[7]) {
  t[0] = 0.25 * step; t[1] = 0.75 * step; t[2] = 1.25 * step; t[3] = 1.75 * step;
  t[4] = 2.5 * step; t[5] = 3.5 * step; t[6] = 5.0 * step;
}

__device__ __forceinline__ double fp8_bscale(const float* bscale, int n, int k, int nbk) {
  return (double)__ldg(bscale + (size_t)(n / kFp8Block) * nbk + k / kFp8Block);
}

// One CTA per matrix: amax over |W| in fp64 (the e4m3 magnitude order is the code order, so
// each 16-code chunk contributes its largest code once), then scale_2 = fp32(fp64(amax) / 1344).
__global__ void __launch_bounds__(1024) fp8_scale2_kernel(int N, int K, const uint8_t* __restrict__ codes,
                                                          const float* __restrict__ bscale,
                                                          float* __restrict__ scale_2) {
  const int m = blockIdx.x;
  const int nbn = (N + kFp8Block - 1) / kFp8Block, nbk = (K + kFp8Block - 1) / kFp8Block;
  const uint8_t* cm = codes + (size_t)m * N * K;
  const float* bm = bscale + (size_t)m * nbn * nbk;
  const long long chunks = (long long)N * K / 16;
  double mx = 0.0;
  for (long long i = threadIdx.x; i < chunks; i += blockDim.x) {
    const uint4 c = __ldg(reinterpret_cast<const uint4*>(cm) + i);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t top = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int b = 0; b < 4; ++b) top = max(top, (w[q] >> (8 * b)) & 0x7Fu);
    const long long e0 = i * 16;
    const int n = (int)(e0 / K), k = (int)(e0 - (long long)n * K);
    mx = fmax(mx, (double)e4m3_to_f32(top) * fp8_bscale(bm, n, k, nbk));
  }
  __shared__ double red[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    mx = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (threadIdx.x == 0) scale_2[m] = __double2float_rn(__ddiv_rn(mx, 1344.0));
  }
}

// A matrix's scale_2 with the two divisors of the rule and guesses of their inverses.
struct Scale2 {
  double s2, d3, d6, i3, i6;
};

__device__ __forceinline__ Scale2 make_scale2(float sc2) {
  Scale2 c;
  c.s2 = (double)sc2;
  c.d3 = 3.0 * c.s2;                                  // exact: 26 significant bits
  c.d6 = 6.0 * c.s2;
  c.i3 = 1.0 / c.d3;                                  // inf for a zero matrix, never used there
  c.i6 = 1.0 / c.d6;
  return c;
}

// The NVFP4 rule on one block of 16 exact weights (fp64) with their sign bits (bit j = weight j)
// and the matrix's scale_2: the block's s16 and magnitude bits and, when `delta` is set, its 16
// delta codes (two words, low nibble first) and delta scale.
struct Block16 {
  uint32_t mag, s16, dlo, dhi, ds4;
};

__device__ __forceinline__ Block16 exact_rule_16(const double (&wv)[16], uint32_t sbits, const Scale2& sc,
                                                 bool delta) {
  const double s2 = sc.s2;
  Block16 r = {0u, 0u, 0u, 0u, 0u};
  double bmax = 0.0;
#pragma unroll
  for (int j = 0; j < 16; ++j) bmax = fmax(bmax, fabs(wv[j]));
  r.s16 = e4m3_rne_ratio_dd(bmax, sc.d3, sc.i3);
  const double lvl = (double)e4m3_to_f32(r.s16) * s2;                   // s16 scale_2, exact
  double d[16];
  double dmax = 0.0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t mg = fabs(wv[j]) >= 2.0 * lvl;
    r.mag |= mg << j;
    const double q = (mg ? 3.0 : 1.0) * lvl;
    d[j] = wv[j] - (((sbits >> j) & 1u) ? -q : q);                      // exact
    dmax = fmax(dmax, fabs(d[j]));
  }
  if (delta) {
    r.ds4 = e4m3_rne_ratio_dd(dmax, sc.d6, sc.i6);
    const double step = (double)e4m3_to_f32(r.ds4) * s2;
    double t[7];
    e2m1_thresholds(step, t);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t dm = step > 0.0 ? e2m1_rne_mag_bisect(fabs(d[j]), t) : 0u;
      const uint32_t code = dm | ((d[j] < 0.0 && dm != 0u) ? 8u : 0u);
      if (j < 8) r.dlo |= code << (4 * j);
      else r.dhi |= code << (4 * (j - 8));
    }
  }
  return r;
}

// One thread per 32-weight group of a row: 32 codes in, one sign and one magnitude word, two s16
// bytes (and 16 delta code bytes + two delta scale bytes) out.
__global__ void __launch_bounds__(256) requant_fp8_kernel(
    int M, int N, int K, const uint8_t* __restrict__ codes, const float* __restrict__ bscale,
    const float* __restrict__ scale_2, uint32_t* __restrict__ sign_out, uint32_t* __restrict__ mag_out,
    uint16_t* __restrict__ s16_out, uint4* __restrict__ dcodes_out, uint16_t* __restrict__ ds4_out) {
  const long long gpm = (long long)N * (K / 32);
  const long long n_groups = (long long)M * gpm;
  const int nbn = (N + kFp8Block - 1) / kFp8Block, nbk = (K + kFp8Block - 1) / kFp8Block;
  const bool delta = dcodes_out != nullptr;
  int m_sc = -1;
  Scale2 sc;
  for (long long gi = (long long)blockIdx.x * blockDim.x + threadIdx.x; gi < n_groups;
       gi += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(gi / gpm);
    const long long r = gi - (long long)m * gpm;
    const int n = (int)(r / (K / 32)), k0 = (int)(r - (long long)n * (K / 32)) * 32;
    if (m != m_sc) {
      sc = make_scale2(__ldg(scale_2 + m));
      m_sc = m;
    }
    const double bs = fp8_bscale(bscale + (size_t)m * nbn * nbk, n, k0, nbk);
    const uint4* src = reinterpret_cast<const uint4*>(codes + ((size_t)m * N + n) * K + k0);
    const uint4 c0 = __ldg(src), c1 = __ldg(src + 1);
    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint32_t sign = 0, mag = 0, s16pair = 0, ds4pair = 0;
    uint32_t dwords[4] = {0, 0, 0, 0};
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      double wv[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t c = (words[4 * b + (j >> 2)] >> (8 * (j & 3))) & 0xFFu;
        const double a = (double)e4m3_to_f32(c & 0x7Fu) * bs;          // exact
        wv[j] = (c & 0x80u) ? -a : a;
        sign |= (c >> 7) << (16 * b + j);
      }
      const Block16 o = exact_rule_16(wv, sign >> (16 * b), sc, delta);
      mag |= o.mag << (16 * b);
      s16pair |= o.s16 << (8 * b);
      ds4pair |= o.ds4 << (8 * b);
      dwords[2 * b] = o.dlo;
      dwords[2 * b + 1] = o.dhi;
    }
    sign_out[gi] = sign;
    mag_out[gi] = mag;
    s16_out[gi] = (uint16_t)s16pair;
    if (delta) {
      dcodes_out[gi] = make_uint4(dwords[0], dwords[1], dwords[2], dwords[3]);
      ds4_out[gi] = (uint16_t)ds4pair;
    }
  }
}

// ---------------------------------------------------------------- MXFP4 (FP4 experts) input
// README "How it fits -- 2-bit experts at FP4 quality", last paragraph: checkpoints with FP4
// experts load by a code remap.  Read as OCP MXFP4 -- an e2m1 code per weight (two per byte, low
// nibble = even k) and one E8M0 scale 2^(e - 127) per 32 weights along K -- remapped by the same
// rule as the FP8 input: W = e2m1(code) 2^(e - 127) is exact in fp64 and scale_2 =
// fp32(fp64(amax) / 1344).

// 2^(e - 127) as an fp64, built from its exponent field (e in 0..254 gives a normal fp64).
__device__ __forceinline__ double e8m0_value(uint32_t e) {
  return __longlong_as_double((long long)(e + (1023 - 127)) << 52);
}

// One CTA per matrix: amax over |W| in fp64 (each 32-weight group contributes its largest
// magnitude code once, e2m1 magnitudes being ordered like their codes).
__global__ void __launch_bounds__(1024) mxfp4_scale2_kernel(int N, int K, const uint8_t* __restrict__ codes,
                                                            const uint8_t* __restrict__ e8m0,
                                                            float* __restrict__ scale_2) {
  const int m = blockIdx.x;
  const long long groups = (long long)N * (K / 32);
  const uint4* cm = reinterpret_cast<const uint4*>(codes) + (size_t)m * groups;
  const uint8_t* em = e8m0 + (size_t)m * groups;
  double mx = 0.0;
  for (long long i = threadIdx.x; i < groups; i += blockDim.x) {
    const uint4 c = __ldg(cm + i);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t top = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int b = 0; b < 8; ++b) top = max(top, (w[q] >> (4 * b)) & 7u);
    mx = fmax(mx, (double)e2m1_mag_value(top) * e8m0_value(__ldg(em + i)));
  }
  __shared__ double red[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    mx = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (threadIdx.x == 0) scale_2[m] = __double2float_rn(__ddiv_rn(mx, 1344.0));
  }
}

// Bit v of the result: some nibble of the 16 in (a, b) has magnitude code v.  A nibble of
// x = (w & 7 per nibble) ^ v is zero exactly where the code is v; the borrow test
// (x - 0x1..1) & ~x & 0x8..8 is nonzero iff some nibble of x is zero.
__device__ __forceinline__ uint32_t codes_present(uint32_t a, uint32_t b) {
  const uint32_t ma = a & 0x77777777u, mb = b & 0x77777777u;
  uint32_t pres = 0;
#pragma unroll
  for (uint32_t v = 0; v < 8; ++v) {
    const uint32_t xa = ma ^ (v * 0x11111111u), xb = mb ^ (v * 0x11111111u);
    const uint32_t z = ((xa - 0x11111111u) & ~xa) | ((xb - 0x11111111u) & ~xb);
    pres |= ((z & 0x88888888u) != 0u ? 1u : 0u) << v;
  }
  return pres;
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
// out).  All 32 weights share p2 = 2^(e - 127), so within a 16-block every decision of the rule is
// a function of the 3-bit magnitude code: the fp64 work runs once per block over the 8 codes (s16
// from the largest code present, the |q| = 3 threshold code, the delta scale from the codes
// present, the 8 delta codes), and the 16 weights take integer operations only.
__global__ void __launch_bounds__(256) requant_mxfp4_kernel(
    int M, long long gpm, const uint4* __restrict__ codes, const uint8_t* __restrict__ e8m0,
    const float* __restrict__ scale_2, uint32_t* __restrict__ sign_out, uint32_t* __restrict__ mag_out,
    uint16_t* __restrict__ s16_out, uint4* __restrict__ dcodes_out, uint16_t* __restrict__ ds4_out) {
  const long long n_groups = (long long)M * gpm;
  const bool delta = dcodes_out != nullptr;
  int m_sc = -1;
  Scale2 sc;
  for (long long gi = (long long)blockIdx.x * blockDim.x + threadIdx.x; gi < n_groups;
       gi += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(gi / gpm);
    if (m != m_sc) {
      sc = make_scale2(__ldg(scale_2 + m));
      m_sc = m;
    }
    const double p2 = e8m0_value(__ldg(e8m0 + gi));
    const uint4 cw = __ldg(codes + gi);
    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
    double wv[8];                                                        // e2m1 value of code c times p2
#pragma unroll
    for (int c = 0; c < 8; ++c) wv[c] = (double)e2m1_mag_value((uint32_t)c) * p2;   // exact
    uint32_t mr[4], s16pair = 0, ds4pair = 0, dw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t wa = w[2 * b], wb = w[2 * b + 1];
      const uint32_t pres = codes_present(wa, wb);
      const uint32_t cmax = 31u - (uint32_t)__clz(pres);                 // pres != 0: 16 codes
      double bmax = 0.0;
#pragma unroll
      for (int c = 0; c < 8; ++c) bmax = (uint32_t)c == cmax ? wv[c] : bmax;
      const uint32_t s16 = e4m3_rne_ratio_dd(bmax, sc.d3, sc.i3);
      const double lvl = (double)e4m3_to_f32(s16) * sc.s2;              // exact
      uint32_t thr = 0;                                                  // |q| = 3 iff code >= thr
#pragma unroll
      for (int c = 0; c < 8; ++c) thr += wv[c] < 2.0 * lvl ? 1u : 0u;
      s16pair |= s16 << (8 * b);
      const uint32_t T = thr * 0x11111111u;
      mr[2 * b] = gather_bit3(((wa | 0x88888888u) - T) & 0x88888888u);
      mr[2 * b + 1] = gather_bit3(((wb | 0x88888888u) - T) & 0x88888888u);
      if (delta) {
        double d[8], dmax = 0.0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          d[c] = wv[c] - ((uint32_t)c >= thr ? 3.0 : 1.0) * lvl;         // exact
          if ((pres >> c) & 1u) dmax = fmax(dmax, fabs(d[c]));
        }
        const uint32_t ds4 = e4m3_rne_ratio_dd(dmax, sc.d6, sc.i6);
        const double step = (double)e4m3_to_f32(ds4) * sc.s2;
        double t[7];
        e2m1_thresholds(step, t);
        uint32_t tlo = 0, thi = 0, flo = 0, fhi = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t dm = step > 0.0 ? e2m1_rne_mag_bisect(fabs(d[c]), t) : 0u;
          const uint32_t e = dm | ((d[c] < 0.0 && dm != 0u) ? 8u : 0u);  // for a positive weight
          const uint32_t f = dm != 0u ? 8u : 0u;
          if (c < 4) { tlo |= e << (8 * c); flo |= f << (8 * c); }
          else { thi |= e << (8 * (c - 4)); fhi |= f << (8 * (c - 4)); }
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
  {
    ProfScope ps(MOET_K_REQUANT, st);
    mxfp4_scale2_kernel<<<M, 1024, 0, st>>>(N, K, codes, e8m0, scale_2);
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
  const long long n_groups = (long long)M * N * (K / 32);
  {
    ProfScope ps(MOET_K_REQUANT, st);
    fp8_scale2_kernel<<<M, 1024, 0, st>>>(N, K, codes, bscale, scale_2);
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
