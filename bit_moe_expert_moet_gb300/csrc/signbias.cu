// Sign-bias probe: per-block L2-optimal quantisation of fp32 weights to a 4-level integer
// codebook, with per-row and per-matrix sums of W, W^2, Q - W and (Q - W)^2.
//
// README "Frontier MoE on consumer Blackwell (SM120)", "How it fits -- 2-bit experts at FP4
// quality", bullet 1 (the sign-bias finding): the L2-optimal fit of a naive 2-bit codebook drops
// one sign's tail and biases every expert, a sign-symmetric codebook at the same L2 error does
// not.  Each block of 16 weights along K gets the scale s > 0 minimising
// sum (w - s L[nearest(w / s)])^2.  For s > 0 the nearest-level assignment is monotone in w, so
// the optimum is among the 969 monotone assignments of the sorted block (counts c1 <= c2 <= c3
// of weights below each level boundary); one assignment's best scale is Nc / Dc (Nc = sum a w,
// Dc = sum a^2) and leaves the error sum w^2 - Nc^2 / Dc, so the search maximises Nc^2 / Dc over
// the candidates with Nc > 0.  The argmax decides integers, so it runs in fp32 with one fixed,
// uncontracted operation order; the chosen block's sums are evaluated in fp64.
//
// One warp per row; lane l takes the row's blocks l, l + 32, ...  Per block: four 16-byte loads,
// a 63-comparator sorting network, fp32 prefix sums, the fully unrolled search (every index
// static, so the prefix sums stay in registers), then the fp64 block sums.  Rows reduce their
// lanes by a fixed butterfly; a second kernel sums the rows of each matrix in row order.
#include "common.cuh"

namespace moet {

constexpr int kProbeBlock = 16;

__device__ __forceinline__ void cas(float& a, float& b) {
  const float lo = fminf(a, b), hi = fmaxf(a, b);
  a = lo;
  b = hi;
}

// Batcher's odd-even merge sort on 16 values (63 compare-exchanges, all indices static).
__device__ __forceinline__ void sort16(float (&v)[kProbeBlock]) {
#pragma unroll
  for (int p = 1; p < kProbeBlock; p <<= 1)
#pragma unroll
    for (int k = p; k >= 1; k >>= 1)
#pragma unroll
      for (int j = k % p; j + k < kProbeBlock; j += 2 * k)
#pragma unroll
        for (int i = 0; i < k; ++i)
          if (i + j + k < kProbeBlock && (i + j) / (2 * p) == (i + j + k) / (2 * p)) cas(v[i + j], v[i + j + k]);
}

struct ProbeLevels {
  float L0, L1, L2, L3;
};

// (sum w, sum w^2, sum (Q - w), sum (Q - w)^2) of one block in fp64.
__device__ __forceinline__ void probe_block(const float4* src, const ProbeLevels lv, double (&acc)[4]) {
  float v[kProbeBlock];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 f = __ldg(src + q);
    v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
  }
  sort16(v);
  float P[kProbeBlock + 1];
  P[0] = 0.0f;
#pragma unroll
  for (int j = 0; j < kProbeBlock; ++j) P[j + 1] = __fadd_rn(P[j], v[j]);
  const float A = lv.L0 - lv.L1, B = lv.L1 - lv.L2, C = lv.L2 - lv.L3;   // small integers, exact
  const float dA = lv.L0 * lv.L0 - lv.L1 * lv.L1, dB = lv.L1 * lv.L1 - lv.L2 * lv.L2;
  const float dC = lv.L2 * lv.L2 - lv.L3 * lv.L3, dT = kProbeBlock * lv.L3 * lv.L3;
  float u[kProbeBlock + 1], x[kProbeBlock + 1], z[kProbeBlock + 1];
#pragma unroll
  for (int j = 0; j <= kProbeBlock; ++j) {
    u[j] = __fmul_rn(A, P[j]);
    x[j] = __fmul_rn(B, P[j]);
    z[j] = __fmul_rn(C, P[j]);
  }
  const float tail = __fmul_rn(lv.L3, P[kProbeBlock]);
  float nn_best = 0.0f, d_best = 1.0f;
  int best = -1;
#pragma unroll
  for (int c1 = 0; c1 <= kProbeBlock; ++c1)
#pragma unroll
    for (int c2 = c1; c2 <= kProbeBlock; ++c2)
#pragma unroll
      for (int c3 = c2; c3 <= kProbeBlock; ++c3) {
        const float n = __fadd_rn(__fadd_rn(__fadd_rn(u[c1], x[c2]), z[c3]), tail);
        const float d = dA * (float)c1 + dB * (float)c2 + dC * (float)c3 + dT;   // exact integers
        const float nn = __fmul_rn(n, n);
        if (n > 0.0f && __fmul_rn(nn, d_best) > __fmul_rn(nn_best, d)) {
          nn_best = nn;
          d_best = d;
          best = (c1 << 10) | (c2 << 5) | c3;
        }
      }
  double sw = 0.0, sw2 = 0.0, nc = 0.0, sa = 0.0, dc = 0.0;
  const int c1 = best >> 10, c2 = (best >> 5) & 31, c3 = best & 31;
#pragma unroll
  for (int i = 0; i < kProbeBlock; ++i) {
    const double wd = (double)v[i];
    sw += wd;
    sw2 += wd * wd;
    const float l = i < c1 ? lv.L0 : i < c2 ? lv.L1 : i < c3 ? lv.L2 : lv.L3;
    nc += (double)l * wd;
    sa += (double)l;
    dc += (double)(l * l);
  }
  acc[0] += sw;
  acc[1] += sw2;
  if (best >= 0) {
    acc[2] += nc / dc * sa - sw;
    acc[3] += sw2 - nc * nc / dc;
  } else {                                   // no fit with s > 0: the block quantises to zero
    acc[2] -= sw;
    acc[3] += sw2;
  }
}

// Two CTAs per SM (126 registers, no spills): 1.7x the throughput of one.
__global__ void __launch_bounds__(256, 2) signbias_rows_kernel(long long rows, int K, const float* __restrict__ w,
                                                               ProbeLevels lv, double* __restrict__ row_sums) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float4* src = reinterpret_cast<const float4*>(w + row * K);
  double acc[4] = {0.0, 0.0, 0.0, 0.0};
  for (int b = lane; b < K / kProbeBlock; b += 32) probe_block(src + 4 * b, lv, acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
  if (lane < 4) row_sums[row * 4 + lane] = acc[lane];
}

// One thread per (matrix, statistic): the rows in order.
__global__ void signbias_matrix_kernel(int M, int N, const double* __restrict__ row_sums, double* __restrict__ sums) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= M * 4) return;
  const int m = t >> 2, q = t & 3;
  const double* r = row_sums + (size_t)m * N * 4 + q;
  double s = 0.0;
  for (int n = 0; n < N; ++n) s += r[(size_t)n * 4];
  sums[t] = s;
}

}  // namespace moet

using namespace moet;

extern "C" moet_status moet_sign_bias_probe(int M, int N, int K, const float* w, const int32_t* levels,
                                            double* row_sums, double* sums, moet_stream stream) {
  if (M < 1 || N < 1 || K < kProbeBlock || K % kProbeBlock != 0) return MOET_ERR_SHAPE;
  if (!w || !levels || !row_sums || !sums) return MOET_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i)
    if (levels[i] < -64 || levels[i] > 64 || (i > 0 && levels[i] <= levels[i - 1])) return MOET_ERR_INVALID_ARG;
  if (((uintptr_t)w & 15) || ((uintptr_t)row_sums & 7) || ((uintptr_t)sums & 7)) return MOET_ERR_ALIGN;
  const ProbeLevels lv = {(float)levels[0], (float)levels[1], (float)levels[2], (float)levels[3]};
  cudaStream_t st = (cudaStream_t)stream;
  const long long rows = (long long)M * N;
  const long long ctas = (rows * 32 + 255) / 256;
  if (ctas > 0x7FFFFFFFLL) return MOET_ERR_UNSUPPORTED;
  {
    ProfScope ps(MOET_K_PROBE, st);
    signbias_rows_kernel<<<(unsigned)ctas, 256, 0, st>>>(rows, K, w, lv, row_sums);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  {
    ProfScope ps(MOET_K_PROBE, st);
    signbias_matrix_kernel<<<(M * 4 + 127) / 128, 128, 0, st>>>(M, N, row_sums, sums);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}
