// tcgen05 bf16 FC engine for large token counts (prefill, sm_103a).
//
// README "Frontier MoE on consumer Blackwell (SM120)", "How it fits -- 2-bit
// experts at FP4 quality", "The kernels": with many tokens per expert the FC
// layers are a dense contraction (tensor-bound), not a weight stream.
//
// Weights.  A 2-bit weight times its block scale, q * s16 with q in {+-1, +-3}
// and s16 an e4m3 value (2^-9 .. 1344 in magnitude), has at most 6 significant
// bits, so it is exact in bf16 and in fp16: the planes expand to an exact A
// operand of tcgen05.mma kind::f16 (fp32 accumulation in TMEM); scale_2 is
// applied in the epilogue.  The NVFP4 delta (e2m1 code times an e4m3 scale,
// 2^-10 .. 2688, also exact in both) is expanded the same way and accumulates
// into the same TMEM accumulator against a copy of the inputs whose ungated
// rows are zero, so it only reaches gated pairs.
//
// Precision.  FC1 runs on bf16 (x is bf16, so FC1 is exact up to fp32
// accumulation).  FC2 runs on fp16: rounding h to bf16 (8 significant bits) on
// top of the bf16 output would exceed the layer's max-error budget, fp16 keeps
// 11.  pf_h16_kernel scales each fp32 h row by a power of two that puts its
// maximum in [2^14, 2^15) (no overflow, and everything above 2^-28 of the
// maximum stays normal) and rounds it to fp16; FC2's epilogue undoes the scale.
//
// Layout.  A 32-bit TMEM column holds two 16-bit values of one row; column c
// of a 32-weight group holds weights c and c + 16 (one shift-and-mask extracts
// the sign and magnitude bits of both, a byte permute with sign replication
// turns the magnitude bits into half-word masks).  The bucketing gather (x)
// and pf_h16_kernel (h) write the activations in the same K order.
//
// Pipeline: one persistent CTA per SM (24 warps) over (work item of <= 256
// pairs x 128-row weight tile) units: warp 0 streams 256-weight chunks of the
// planes (or delta) and warps 3, 16, 18, 19 take turns streaming the steps of the
// item's activation rows, with TMA (one lane per box); warps 8-15 expand each step's weights into a TMEM A
// stage (two warps per 32-row quarter); warp 1 issues 4 MMAs
// per step and commits; warp 2 prepares the unit records; warps 4-7 and 20-23 (two per
// lane quarter, alternate 16-column chunks) drain the accumulator (FC1: SiLU(gate) * up ->
// fp32 h; FC2: times the routing weight, scale_2 and the row's h scale -> fp32 o).  Every wait
// is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "common.cuh"
#include "moe_pf.cuh"
#include "tc_common.cuh"

namespace moet {
namespace {

constexpr int kPfThreads = 768;           // 24 warps, roles above
constexpr int kPfEpiWarps = 8;            // epilogue warps: two per TMEM lane quarter (4-7, 20-23)
constexpr int kBProd = 4;                 // activation producer warps (3, 16, 18, 19), steps in turn
constexpr int kPfConvWarps = 8;
constexpr int kPC = 256;                  // weights per weight chunk
// weights per step: 4 MMAs of K = 16, i.e. 32 TMEM columns of A and 128-byte activation rows
constexpr int kStepWeights = 64;
constexpr int kPRing = 3;                 // weight chunks in flight
constexpr int kBRing = 5;                 // activation steps in flight
constexpr int kPAst = 8;                  // TMEM A stages
constexpr int kGrp = 4;                   // steps per converter hand-off (one weight chunk)
constexpr int kNGrp = kPAst / kGrp;       // hand-off groups of A stages in flight
constexpr int kPMeta = 2;                 // unit records in flight
constexpr int kPTmemCols = 512;
constexpr int kPColA = 256;               // D: columns 0..255; A stage s: kPColA + 32 s
static_assert(kPColA + 32 * kPAst <= kPTmemCols, "TMEM columns");
static_assert(kPAst % kGrp == 0 && (kPC / 64) % kGrp == 0, "hand-off groups tile the A ring and the chunks");
// weight chunk stage: planes: sign [128 rows][32 B] (SW32) at 0, magnitude at 4096, row scales
// [128][16 B] at 8192; delta: codes [128][128 B] (SW128) at 0, scales [128][16 B] at 16384
constexpr int kPChunkBytes = 18432;
constexpr int kBStepBytes = 32768;        // activation step: [<= 256 rows][128 B] (SW128)
constexpr int kPBase = 0, kBBase = kPRing * kPChunkBytes;
constexpr int kPMisc = kBBase + kBRing * kBStepBytes;      // barriers and unit records

struct PfMaps {
  CUtensorMap sign, mag, q;      // planes u32 [E N, K/32] box {8, 64} SW32; s16 u8 [E N, K/16] box {16, 64}
  CUtensorMap dcodes, ds4;       // delta u8 [S N, K/2] box {128, 64} SW128; scales box {16, 64}
  CUtensorMap act, actg;         // activations bf16 (FC1) / fp16 (FC2) [pairs, K] box {64, 64} SW128 (all / gated rows)
};

struct PfArgs {
  int T, H, I, k, K, N, tiles;
  const int32_t* offsets;
  const int32_t* perm;
  const float* topk_w;
  const float* scale_2;
  const int32_t* delta_slot;
  int n_slots;
  const uint8_t* gate;
  const int* hdr;
  int* work;                     // units handed out so far (one counter per launch, zeroed beforehand)
  const int4* chunks;
  float* h;                      // FC1 output [pairs, I]
  const float* hscale;           // FC2: per bucketed row, the power of two that undoes the fp16 scaling of h
  float* o;                      // FC2 output
};

struct PfMeta {
  int e, pos0, ntok, ncols;      // e: the planes' expert (pool slot) index
  int dslot;                     // delta slot when the unit runs the delta pass, else -1
  int nck;                       // weight chunks (K / 256, doubled with the delta pass)
  int r0, r1;
  float sc2;
  int ncols_d;                   // delta pass: columns up to the last gated one (multiple of 16)
  int pad[6];
  int pair[kPfTok];              // per column (token of the item): pair id t k + j, -1 = none
  float wts[kPfTok];             // FC2: routing weight x scale_2 x h scale of the pair
  uint8_t gated[kPfTok];         // 1 = the pair's token is gated
};
static_assert(sizeof(PfMeta) == 64 + 9 * kPfTok, "PfMeta layout");

struct PfSmem {
  uint64_t pfull[kPRing], pempty[kPRing];
  uint64_t bfull[kBRing], bdone[kBRing];
  uint64_t staged[kNGrp];         // the A stages of a group of steps expanded
  uint64_t adone[kNGrp];          // MMAs of a group of steps done: their A stages are free
  uint64_t acc_full, acc_empty;
  uint64_t meta_full[kPMeta], meta_empty[kPMeta];
  PfMeta meta[kPMeta];
  uint32_t tmem_base;
  int stuck;
};

constexpr size_t kPfSmemBytes = 1024 + (size_t)kPMisc + sizeof(PfSmem);
static_assert(kPfSmemBytes <= 232448, "shared memory over the per-CTA limit");

__device__ __forceinline__ bool pf_stuck(const PfSmem& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.stuck) != 0;
}

// kind::f16 instruction descriptor: fp32 D, A and B both bf16 (BF = true) or both fp16, both
// K-major, M = 128.  The two operands always share the type.
template <bool BF>
__device__ __forceinline__ uint32_t f16_idesc(int n) {
  const uint32_t t = BF ? 1u : 0u;
  return (1u << 4) | (t << 7) | (t << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// Row of the weight chunk (gate rows 0-63, up rows 64-127 for FC1; output rows for FC2) held by
// TMEM lane t.  FC1 interleaves them per lane quarter: lanes 0-15 of quarter q hold gate rows
// 16 q .. 16 q + 15 and lanes 16-31 the matching up rows, so that every gate value meets its up
// value in the same warp (one shuffle, no shared memory) in the epilogue.
template <bool FC1>
__device__ __forceinline__ int tile_row(int t) {
  return FC1 ? ((t & 16) ? 64 : 0) + 16 * (t >> 5) + (t & 15) : t;
}

// kind::f16 MMA with A in TMEM, issued by one elected lane of a converged warp (warp-uniform
// operands stay in uniform registers).
__device__ __forceinline__ void mma_ta_elect(uint32_t d, uint32_t a_tmem, uint64_t bd, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p, e; setp.ne.b32 p, %4, 0; elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d),
      "r"(a_tmem), "l"(bd), "r"(idesc), "r"(acc));
}

// 16-bit float bits (bf16 if BF, else fp16) of a value that is exact in that format.
template <bool BF>
__device__ __forceinline__ uint32_t h16_bits(float f) {
  return BF ? (__float_as_uint(f) >> 16) : (uint32_t)__half_as_ushort(__float2half_rn(f));
}

// 32 weights (sign word S, magnitude word M) with block scales s0 (weights 0-15)
// and s1 (16-31) -> 16 words: word j = bits (weight j) | bits (weight j + 16) << 16,
// bf16 (BF) or fp16 (both have the sign in bit 15 of a half).  One shift of a plane word by
// 7 - j puts bits j, j + 8, j + 16, j + 24 at the most significant bits of its four bytes, which
// serves words j (bytes 0, 2) and j + 8 (bytes 1, 3): a sign-replicating byte permute turns the
// magnitude bits into half-word masks, and the sign bits sit at bits 15 and 31 already for word
// j + 8 (for word j after one more byte shift, taken once from S << 8).
template <bool BF>
__device__ __forceinline__ void planes_to_16(uint32_t S, uint32_t M, uint32_t s0, uint32_t s1, uint32_t out[16]) {
  const float f0 = e4m3_to_f32(s0), f1 = e4m3_to_f32(s1);
  const uint32_t a0 = h16_bits<BF>(f0), b0 = h16_bits<BF>(3.0f * f0);
  const uint32_t a1 = h16_bits<BF>(f1), b1 = h16_bits<BF>(3.0f * f1);
  const uint32_t one = a0 | (a1 << 16);                    // q = 1 in both halves
  const uint32_t dif = (a0 ^ b0) | ((a1 ^ b1) << 16);      // q = 1 -> q = 3
  const uint32_t S8 = S << 8;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t mj = M << (7 - j), sj = S << (7 - j), s8j = S8 << (7 - j);
    const uint32_t mlo = prmt(mj, 0u, 0xAA88u);            // bits j, j + 16 -> half-word masks
    const uint32_t mhi = prmt(mj, 0u, 0xBB99u);            // bits j + 8, j + 24
    out[j] = (one ^ (mlo & dif)) | (s8j & 0x80008000u);
    out[j + 8] = (one ^ (mhi & dif)) | (sj & 0x80008000u);
  }
}

// e2m1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} as bf16 and as fp16, split into byte tables for prmt
// (first word: codes 0-3, second: codes 4-7); the fp16 values have zero low bytes
constexpr uint32_t kE2m1LoA = 0xC0800000u, kE2m1LoB = 0xC0804000u;   // bf16 low bytes
constexpr uint32_t kE2m1HiA = 0x3F3F3F00u, kE2m1HiB = 0x40404040u;   // bf16 high bytes
constexpr uint32_t kE2m1F16A = 0x3E3C3800u, kE2m1F16B = 0x46444240u; // fp16 high bytes

template <bool BF>
__device__ __forceinline__ uint32_t mul_16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  if (BF)
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two e2m1 codes (bits 0-3 and 8-11 of c) times the 16x2 scales sc -> 16x2 (exact: a code
// value has 2 significant bits, an e4m3 scale 4, and the products stay in the normal range).
template <bool BF>
__device__ __forceinline__ uint32_t e2m1x2_16(uint32_t c, uint32_t sc) {
  const uint32_t sel = c & 0x0707u;
  const uint32_t mag = BF ? (prmt(kE2m1LoA, kE2m1LoB, sel) | (prmt(kE2m1HiA, kE2m1HiB, sel) << 8))
                          : (prmt(kE2m1F16A, kE2m1F16B, sel) << 8);
  return mul_16x2<BF>(mag, sc) ^ (((c & 0x0008u) << 12) | ((c & 0x0800u) << 20));
}

// 32 delta codes (16 bytes: byte t = codes of weights 2t, 2t+1, low nibble first) with block
// scales s0 (weights 0-15), s1 (16-31) -> word j = bits (weight j) | bits (weight j + 16) << 16.
template <bool BF>
__device__ __forceinline__ void delta_to_16(uint4 c, uint32_t s0, uint32_t s1, uint32_t out[16]) {
  const uint32_t sc = h16_bits<BF>(e4m3_to_f32(s0)) | (h16_bits<BF>(e4m3_to_f32(s1)) << 16);
  const uint32_t lo[2] = {c.x, c.y}, hi[2] = {c.z, c.w};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int sh = 4 * (j & 7);
    out[j] = e2m1x2_16<BF>(((lo[j >> 3] >> sh) & 15u) | (((hi[j >> 3] >> sh) & 15u) << 8), sc);
  }
}

// ---------------------------------------------------------------- gather
// Whether the delta pass can read the gated-copy row of pair p: its expert holds a delta slot.
// Rows of the other pairs are never read, so the gated copies skip them.
__device__ __forceinline__ bool pair_in_delta_pass(int p, const int32_t* __restrict__ topk_idx, int n_experts,
                                                   const int32_t* __restrict__ delta_slot, int n_slots) {
  const int e = __ldg(topk_idx + p);
  if (e < 0 || e >= n_experts) return false;
  const int ds = __ldg(delta_slot + e);
  return ds >= 0 && ds < n_slots;
}

// xb[pos] = x[token of perm[pos]] in the permuted K order; xbg the same for
// gated pairs, zero for the others (written for the delta pass's pairs only:
// xbg == null or delta_slot == null writes none).  One CTA per row; a thread takes two
// neighbouring 8-element outputs at a time (16-byte loads of both halves of their 32-group).
constexpr int kGatherThreads = 224;
__global__ void __launch_bounds__(kGatherThreads) pf_gather_kernel(int pairs, int k, int H, const uint16_t* __restrict__ x,
                                                        const int32_t* __restrict__ perm,
                                                        const uint8_t* __restrict__ gate,
                                                        const int32_t* __restrict__ topk_idx, int n_experts,
                                                        const int32_t* __restrict__ delta_slot, int n_slots,
                                                        uint16_t* __restrict__ xb, uint16_t* __restrict__ xbg) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  const int pos = blockIdx.x;
  const int p = __ldg(perm + pos);
  bool gated = false, in_delta = false, ok = p >= 0 && p < pairs;
  if (ok) {
    gated = gate != nullptr && __ldg(gate + p / k) != 0;
    in_delta = xbg != nullptr && delta_slot != nullptr &&
               pair_in_delta_pass(p, topk_idx, n_experts, delta_slot, n_slots);
  } else if (threadIdx.x == 0) {
    record_error(MOET_ERR_DEVICE_INDEX);
  }
  const uint16_t* xr = x + (size_t)(ok ? p / k : 0) * H;
  uint4* out = reinterpret_cast<uint4*>(xb + (size_t)pos * H);
  uint4* outg = reinterpret_cast<uint4*>(xbg + (size_t)pos * H);
  // outputs t and t + 1 (t even): k' = 32 g + 2 c + b holds weight 32 g + c + 16 b, and the pair
  // covers c = 8 r .. 8 r + 7 (t = 4 g + 2 r)
  for (int tt = threadIdx.x; tt < H / 16; tt += kGatherThreads) {
    const int g = tt >> 1, r = tt & 1;
    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
    if (ok) {
      lo = __ldg(reinterpret_cast<const uint4*>(xr + 32 * g + 8 * r));
      hi = __ldg(reinterpret_cast<const uint4*>(xr + 32 * g + 16 + 8 * r));
    }
    const uint4 v0 = make_uint4((lo.x & 0xFFFFu) | (hi.x << 16), (lo.x >> 16) | (hi.x & 0xFFFF0000u),
                                (lo.y & 0xFFFFu) | (hi.y << 16), (lo.y >> 16) | (hi.y & 0xFFFF0000u));
    const uint4 v1 = make_uint4((lo.z & 0xFFFFu) | (hi.z << 16), (lo.z >> 16) | (hi.z & 0xFFFF0000u),
                                (lo.w & 0xFFFFu) | (hi.w << 16), (lo.w >> 16) | (hi.w & 0xFFFF0000u));
    out[2 * tt] = v0;
    out[2 * tt + 1] = v1;
    if (in_delta) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      outg[2 * tt] = gated ? v0 : z;
      outg[2 * tt + 1] = gated ? v1 : z;
    }
  }
}

// FC1's fp32 h (bucketed rows, natural K order) -> FC2's fp16 operand in the permuted K order
// (as xb), each row times the power of two 2^-e that puts its max |h| in [2^14, 2^15), and
// hscale[pos] = 2^e; hg16 the same for gated pairs, zero for the others (for the delta pass's
// pairs only, as xbg).  One CTA per row; a thread holds J pairs of neighbouring 8-element outputs
// (both halves of their 32-group, 64 bytes of h each) in registers, so h is read once: the row's
// max |h| comes from those registers, then the same registers are scaled and stored.
constexpr int kH16MaxThreads = 256;
template <int J>
__global__ void __launch_bounds__(kH16MaxThreads) pf_h16_kernel(int pairs, int k, int I, const float* __restrict__ h,
                                                     const int32_t* __restrict__ perm,
                                                     const uint8_t* __restrict__ gate,
                                                     const int32_t* __restrict__ topk_idx, int n_experts,
                                                     const int32_t* __restrict__ delta_slot, int n_slots,
                                                     uint16_t* __restrict__ h16, uint16_t* __restrict__ hg16,
                                                     float* __restrict__ hscale) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  const int pos = blockIdx.x;
  const float* row = h + (size_t)pos * I;
  const int ntt = I / 16;
  __shared__ float red[kH16MaxThreads / 32];
  // output pair tt covers k' = 16 tt .. 16 tt + 15 of the permuted order, where k' = 32 g + 2 c + b
  // holds element 32 g + c + 16 b: c = 8 r .. 8 r + 7 of group g (tt = 2 g + r)
  float4 v[J][4];
  float mx = 0.0f;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int tt = threadIdx.x + j * blockDim.x;
    if (tt < ntt) {
      const float4* src = reinterpret_cast<const float4*>(row + 32 * (tt >> 1) + 8 * (tt & 1));
      v[j][0] = __ldg(src);
      v[j][1] = __ldg(src + 1);
      v[j][2] = __ldg(src + 4);
      v[j][3] = __ldg(src + 5);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[j][q].x), fabsf(v[j][q].y)), fmaxf(fabsf(v[j][q].z), fabsf(v[j][q].w))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) mx = fmaxf(mx, red[w]);
  // 2^-e with max * 2^-e in [2^14, 2^15): e = (exponent of max) - 15; a zero or non-finite
  // maximum keeps the row as it is
  int e = 0;
  if (mx > 0.0f && mx <= 3.0e38f) {
    frexpf(mx, &e);                                        // mx = f 2^e, f in [0.5, 1)
    e = e - 15 < -112 ? -112 : e - 15;                     // 2^-e stays finite in fp32
  }
  const float down = ldexpf(1.0f, -e);
  const int p = __ldg(perm + pos);
  bool gated = false, in_delta = false;
  if (p >= 0 && p < pairs) {
    gated = gate != nullptr && __ldg(gate + p / k) != 0;
    in_delta = hg16 != nullptr && delta_slot != nullptr &&
               pair_in_delta_pass(p, topk_idx, n_experts, delta_slot, n_slots);
  } else if (threadIdx.x == 0) {
    record_error(MOET_ERR_DEVICE_INDEX);
  }
  if (threadIdx.x == 0) hscale[pos] = ldexpf(1.0f, e);
  uint4* out = reinterpret_cast<uint4*>(h16 + (size_t)pos * I);
  uint4* outg = reinterpret_cast<uint4*>(hg16 + (size_t)pos * I);
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int tt = threadIdx.x + j * blockDim.x;
    if (tt >= ntt) continue;
    const float a[8] = {v[j][0].x, v[j][0].y, v[j][0].z, v[j][0].w, v[j][1].x, v[j][1].y, v[j][1].z, v[j][1].w};
    const float b[8] = {v[j][2].x, v[j][2].y, v[j][2].z, v[j][2].w, v[j][3].x, v[j][3].y, v[j][3].z, v[j][3].w};
    uint32_t wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      wv[i] = (uint32_t)__half_as_ushort(__float2half_rn(a[i] * down)) |
              ((uint32_t)__half_as_ushort(__float2half_rn(b[i] * down)) << 16);
    const uint4 v0 = make_uint4(wv[0], wv[1], wv[2], wv[3]), v1 = make_uint4(wv[4], wv[5], wv[6], wv[7]);
    out[2 * tt] = v0;
    out[2 * tt + 1] = v1;
    if (in_delta) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      outg[2 * tt] = gated ? v0 : z;
      outg[2 * tt + 1] = gated ? v1 : z;
    }
  }
}

// ---------------------------------------------------------------- FC kernel
template <bool FC1>
__global__ void __launch_bounds__(kPfThreads, 1) pf_fc_kernel(const PfArgs a, const __grid_constant__ PfMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem_dyn[];
  unsigned char* base = smem_dyn + ((1024 - (smem_addr(smem_dyn) & 1023)) & 1023);
  PfSmem& sm = *reinterpret_cast<PfSmem*>(base + kPMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wl = wait_limit();
  // Units are handed out one at a time from a global counter (the scheduler warp takes the next
  // one when a record slot is free), so the uneven units (partial items, delta passes) spread over
  // the CTAs; the record after a CTA's last unit has nck = -1 and ends every role's loop.
  const int nkc = a.K / kPC;                   // weight chunks of the main pass

  if (tid == 0) {
    sm.stuck = 0;
    for (int s = 0; s < kPRing; ++s) { mbar_init(&sm.pfull[s], 1); mbar_init(&sm.pempty[s], kPfConvWarps); }
    for (int s = 0; s < kBRing; ++s) { mbar_init(&sm.bfull[s], 1); mbar_init(&sm.bdone[s], 1); }
    for (int s = 0; s < kNGrp; ++s) mbar_init(&sm.staged[s], kPfConvWarps);
    for (int s = 0; s < kNGrp; ++s) mbar_init(&sm.adone[s], 1);
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, kPfEpiWarps);
    for (int s = 0; s < kPMeta; ++s) { mbar_init(&sm.meta_full[s], 1); mbar_init(&sm.meta_empty[s], kPfEpiWarps); }
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&sm.tmem_base)),
                 "r"(kPTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = sm.tmem_base;
  // set-up above overlaps the previous kernel; its outputs are read from here on
  pdl_wait();
  pdl_trigger();
  const int total_units = a.hdr[0] * a.tiles;

  // activation producers 3, 16, 18, 19: none on the MMA thread's sub-partition (warp % 4 == 1)
  const int bprod = warp == 3 ? 0 : warp == 16 ? 1 : warp == 18 ? 2 : warp == 19 ? 3 : -1;
  if (warp == 0 || bprod >= 0) {
    // ---------------- producers, one lane per TMA box: warp 0 streams the weight chunks,
    // the activation producers take the 64-row activation steps in turn
    int gc = 0, gs = 0;
    bool bad = false;
    for (int j = 0; !bad; ++j) {
      const int m = j % kPMeta;
      if (!mbar_wait_warp(&sm.meta_full[m], (j / kPMeta) & 1, wl)) { bad = true; break; }
      const PfMeta& um = sm.meta[m];
      if (um.nck < 0) break;                                 // no more units
      const int pos0 = um.pos0, nck = um.nck, dslot = um.dslot;
      const int nb = (um.ncols + 63) / 64;                 // 64-row activation boxes per step
      const int nbd = (um.ncols_d + 63) / 64;              // ... of a delta step
      const int w0 = um.e * a.N + um.r0, w1 = um.e * a.N + um.r1;
      const int d0 = dslot * a.N + um.r0, d1 = dslot * a.N + um.r1;
      for (int c = 0; c < nck && !bad; ++c, ++gc) {
        const bool dp = c >= nkc;
        const int cc = dp ? c - nkc : c;
        if (warp == 0) {
          const int ps = gc % kPRing;
          if (gc >= kPRing && !mbar_wait_warp(&sm.pempty[ps], ((gc / kPRing) - 1) & 1, wl)) { bad = true; break; }
          unsigned char* pst = base + kPBase + ps * kPChunkBytes;
          if (lane == 0) mbar_expect_tx(&sm.pfull[ps], dp ? 18432u : 10240u);
          __syncwarp();
          if (!dp) {
            if (lane < 6) {
              const int hv = lane & 1;
              const CUtensorMap* map = lane < 2 ? &maps.sign : lane < 4 ? &maps.mag : &maps.q;
              const int off = lane < 2 ? 2048 * hv : lane < 4 ? 4096 + 2048 * hv : 8192 + 1024 * hv;
              tma_load_2d(smem_addr(pst + off), map, lane < 4 ? cc * 8 : cc * 16, hv ? w1 : w0, &sm.pfull[ps]);
            }
          } else {
            if (lane < 4) {
              const int hv = lane & 1;
              const CUtensorMap* map = lane < 2 ? &maps.dcodes : &maps.ds4;
              const int off = lane < 2 ? 8192 * hv : 16384 + 1024 * hv;
              tma_load_2d(smem_addr(pst + off), map, lane < 2 ? cc * 128 : cc * 16, hv ? d1 : d0, &sm.pfull[ps]);
            }
          }
          continue;
        }
        for (int s = 0; s < kPC / kStepWeights; ++s, ++gs) {
          if (gs % kBProd != bprod) continue;
          const int bs = gs % kBRing;
          if (gs >= kBRing && !mbar_wait_warp(&sm.bdone[bs], ((gs / kBRing) - 1) & 1, wl)) { bad = true; break; }
          unsigned char* bst = base + kBBase + bs * kBStepBytes;
          const int nbs = dp ? nbd : nb;
          if (lane == 0) mbar_expect_tx(&sm.bfull[bs], (uint32_t)nbs * 64u * 128u);
          __syncwarp();
          if (lane < nbs)
            tma_load_2d(smem_addr(bst + 8192 * lane), dp ? &maps.actg : &maps.act, cc * kPC + s * kStepWeights,
                        pos0 + 64 * lane, &sm.bfull[bs]);
        }
      }
    }
    if (bad && lane == 0) atomicExch(&sm.stuck, 1);
    if (lane == 0) {
      // every copy this warp issued has landed before the CTA may exit
      if (warp == 0)
        for (int i = gc > kPRing ? gc - kPRing : 0; i < gc; ++i) mbar_wait(&sm.pfull[i % kPRing], (i / kPRing) & 1, wl);
      else
        for (int i = gs > kBRing ? gs - kBRing : 0; i < gs; ++i)
          if (i % kBProd == bprod) mbar_wait(&sm.bfull[i % kBRing], (i / kBRing) & 1, wl);
    }
  } else if (warp == 1) {
    // ---------------- MMA issue.  The whole warp walks the loop, so every operand stays
    // warp-uniform (uniform registers); one elected lane issues each MMA and commit.  An
    // activation stage's descriptor is the ring's base descriptor plus the stage's offset / 16.
    int gs = 0, last = -1;
    bool bad = false;
    const uint64_t b_desc = sw128_desc(smem_addr(base + kBBase));
    for (int j = 0; !bad; ++j) {
      const int m = j % kPMeta;
      if (!mbar_wait_warp(&sm.meta_full[m], (j / kPMeta) & 1, wl)) { bad = true; break; }
      if (sm.meta[m].nck < 0) break;                         // no more units
      if (j >= 1 && !mbar_wait_warp(&sm.acc_empty, (j - 1) & 1, wl)) { bad = true; break; }
      if (__any_sync(0xffffffffu, pf_stuck(sm))) { bad = true; break; }
      asm volatile("tcgen05.fence::after_thread_sync;");
      const int nst = sm.meta[m].nck * (kPC / kStepWeights);
      const uint32_t idesc = f16_idesc<FC1>(sm.meta[m].ncols);   // FC1 bf16, FC2 fp16
      const uint32_t idesc_d = f16_idesc<FC1>(sm.meta[m].ncols_d);   // the delta pass's steps
      // a group of kGrp steps per iteration: its A stages expanded (one wait), then each
      // step's activations (one wait per step: the activation ring is shallower than a group
      // plus the next)
      for (int st = 0; st < nst && !bad; st += kGrp, gs += kGrp) {
        const int grp = gs / kGrp;
        if (!mbar_wait_warp(&sm.staged[grp % kNGrp], (grp / kNGrp) & 1, wl)) {
          bad = true;
          break;
        }
#pragma unroll
        for (int h = 0; h < kGrp; ++h) {
          const int as = (gs + h) % kPAst, bs = (gs + h) % kBRing;
          if (!mbar_wait_warp(&sm.bfull[bs], ((gs + h) / kBRing) & 1, wl)) {
            bad = true;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;");
          const uint64_t bd = b_desc + (uint64_t)((bs * kBStepBytes) >> 4);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mma_ta_elect(tmem, tmem + kPColA + 32 * as + 8 * i, bd + (uint64_t)((32 * i) >> 4),
                         st >= nkc * (kPC / kStepWeights) ? idesc_d : idesc,
                         (st > 0 || h > 0 || i > 0) ? 1u : 0u);
          tc_commit_elect(&sm.bdone[bs]);
          last = gs + h;
        }
        if (bad) break;
        tc_commit_elect(&sm.adone[grp % kNGrp]);
      }
      if (bad) break;
      tc_commit_elect(&sm.acc_full);
    }
    if (bad && lane == 0) atomicExch(&sm.stuck, 1);
    // every MMA this warp issued is complete before TMEM is released
    if (last >= 0 && lane == 0) mbar_wait(&sm.bdone[last % kBRing], (last / kBRing) & 1, wl);
    __syncwarp();
  } else if (warp == 2) {
    // ---------------- scheduler
    for (int j = 0;; ++j) {
      const int m = j % kPMeta;
      if (j >= kPMeta && !mbar_wait_warp(&sm.meta_empty[m], ((j / kPMeta) - 1) & 1, wl)) {
        if (lane == 0) atomicExch(&sm.stuck, 1);
        break;
      }
      if (__any_sync(0xffffffffu, pf_stuck(sm))) break;
      int u = 0;
      if (lane == 0) u = atomicAdd(a.work, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      // (a test can make CTA 0 withhold its first record: every wait on it then runs out)
      const bool withhold = blockIdx.x == 0 && j == 0 && *reinterpret_cast<volatile int*>(&g_dbg_withhold) != 0;
      if (u >= total_units) {
        if (lane == 0) sm.meta[m].nck = -1;                  // the end record
        __syncwarp();
        if (lane == 0 && !withhold) mbar_arrive(&sm.meta_full[m]);
        break;
      }
      const int item = u / a.tiles, tile = u - item * a.tiles;
      const int4 ch = a.chunks[item];
      const int e = ch.x, ntok = ch.z;
      const int pe = ch.w;                 // pool slot of the expert's planes and scale_2
      const int pos0 = __ldg(a.offsets + e) + ch.y;
      int dslot = -1;
      if (a.delta_slot != nullptr && a.gate != nullptr) {
        dslot = __ldg(a.delta_slot + e);
        if (dslot >= a.n_slots) {
          if (lane == 0) record_error(MOET_ERR_DEVICE_INDEX);
          dslot = -1;
        }
      }
      // per-column table of the item: pair id, FC2's output factor (routing weight x scale_2 x the
      // row's h scale), gate flag
      PfMeta& um = sm.meta[m];
      const float sc2 = __ldg(a.scale_2 + pe);
      bool gated = false;
      int last_g = -1;
      for (int t = lane; t < kPfTok; t += 32) {
        int pr = -1;
        float wv = 0.0f;
        uint8_t gf = 0;
        if (t < ntok) {
          const int p = __ldg(a.perm + pos0 + t);
          if (p < 0 || p >= a.T * a.k) {
            record_error(MOET_ERR_DEVICE_INDEX);
          } else {
            pr = p;
            if (!FC1) wv = __ldg(a.topk_w + p) * sc2 * __ldg(a.hscale + pos0 + t);
            if (a.gate != nullptr && __ldg(a.gate + p / a.k)) gf = 1;
          }
        }
        um.pair[t] = pr;
        um.wts[t] = wv;
        um.gated[t] = gf;
        gated = gated || gf != 0;
        if (gf) last_g = t;
      }
      if (!__any_sync(0xffffffffu, gated)) dslot = -1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) last_g = max(last_g, __shfl_xor_sync(0xffffffffu, last_g, o));
      if (lane == 0) {
        um.e = pe; um.pos0 = pos0; um.ntok = ntok;
        um.ncols = ((ntok + 15) / 16) * 16;
        um.ncols_d = ((last_g + 1 + 15) / 16) * 16;   // the delta reaches only gated columns
        um.dslot = dslot;
        um.nck = dslot >= 0 ? 2 * nkc : nkc;
        um.r0 = FC1 ? tile * 64 : tile * 128;
        um.r1 = FC1 ? a.I + tile * 64 : tile * 128 + 64;
        um.sc2 = sc2;
      }
      __syncwarp();
      if (lane == 0 && !withhold) mbar_arrive(&sm.meta_full[m]);
    }
  } else if ((warp >= 4 && warp < 8) || warp >= 20) {
    // ---------------- epilogue: TMEM lane quarter warp & 3; the two warps of a quarter take
    // alternate 16-column chunks
    const int ehalf = warp >= 20 ? 1 : 0;
    const int trow = 32 * (warp & 3) + lane;
    const uint32_t lane_q = (uint32_t)((warp & 3) * 32) << 16;
    const bool lo = lane < 16;                     // FC1: this lane holds a gate row, lane ^ 16 its up row
    for (int j = 0;; ++j) {
      const int m = j % kPMeta;
      bool ok = mbar_wait_warp(&sm.meta_full[m], (j / kPMeta) & 1, wl);
      if (ok && sm.meta[m].nck < 0) break;                   // no more units (same for all eight warps)
      ok = ok && mbar_wait_warp(&sm.acc_full, j & 1, wl);
      asm volatile("tcgen05.fence::after_thread_sync;");
      if (epi_any<32 * kPfEpiWarps>(!ok || pf_stuck(sm))) {
        if (!ok && lane == 0) atomicExch(&sm.stuck, 1);
        break;
      }
      const PfMeta& um = sm.meta[m];
      const int ncols = um.ncols, ntok = um.ntok, pos0 = um.pos0;
      const float sc2 = um.sc2;
      // two of this warp's 16-column chunks (c0 and c0 + 32) per TMEM wait
      for (int c0 = 16 * ehalf; c0 < ncols; c0 += 64) {
        const bool two = c0 + 32 < ncols;                    // the same for the whole warp
        float v2[2][16];
        tmem_ld16_pair(tmem + lane_q + c0, two, v2[0], v2[1]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (hh == 1 && !two) break;
          const int cc = c0 + 32 * hh;
          const float* v = v2[hh];
          if (!FC1) {
            // output row trow; per column the routing weight x scale_2 x the row's h scale
            float* orow = a.o + um.r0 + trow;
            const int4* pp = reinterpret_cast<const int4*>(um.pair + cc);
            const float4* wp = reinterpret_cast<const float4*>(um.wts + cc);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int4 p4 = pp[q];
              const float4 w4 = wp[q];
              const int pq[4] = {p4.x, p4.y, p4.z, p4.w};
              const float wq[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int col = cc + 4 * q + t;
                if (col < ntok && pq[t] >= 0) orow[(size_t)pq[t] * a.H] = v[4 * q + t] * wq[t];
              }
            }
          } else {
            // SiLU(gate) * up: the gate lane finishes columns cc .. cc + 7, the up lane cc + 8 ..
            // cc + 15; each hands the other the half it needs
            float r[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) r[i] = __shfl_xor_sync(0xffffffffu, lo ? v[8 + i] : v[i], 16);
            const int cb = cc + (lo ? 0 : 8);
            const int hcol = um.r0 + 16 * (warp & 3) + (lane & 15);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int col = cb + i;
              if (col < ntok) {
                const float gv = (lo ? v[i] : r[i]) * sc2, uv = (lo ? r[i] : v[8 + i]) * sc2;
                a.h[(size_t)(pos0 + col) * a.I + hcol] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
              }
            }
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.acc_empty);
        mbar_arrive(&sm.meta_empty[m]);
      }
    }
  } else if (warp >= 8 && warp < 16) {
    // ---------------- converters: two warps per 32-row quarter; half h fills TMEM
    // columns 16 h .. 16 h + 15 of each step's A stage for its row
    const int half = (warp - 8) >> 2;
    const int trow = 32 * (warp & 3) + lane;
    const int srow = tile_row<FC1>(trow);              // the weight row this TMEM lane holds
    const uint32_t lane_q = (uint32_t)((warp & 3) * 32) << 16;
    int gc = 0, gs = 0;
    bool bad = false;
    for (int j = 0; !bad; ++j) {
      const int m = j % kPMeta;
      if (!mbar_wait_warp(&sm.meta_full[m], (j / kPMeta) & 1, wl)) { bad = true; break; }
      if (sm.meta[m].nck < 0) break;                         // no more units
      if (__any_sync(0xffffffffu, pf_stuck(sm))) { bad = true; break; }
      const int nck = sm.meta[m].nck;
      for (int c = 0; c < nck && !bad; ++c, ++gc) {
        const int ps = gc % kPRing;
        if (!mbar_wait_warp(&sm.pfull[ps], (gc / kPRing) & 1, wl)) { bad = true; break; }
        const unsigned char* pst = base + kPBase + ps * kPChunkBytes;
        const bool dp = c >= nkc;
        constexpr int kSteps = kPC / kStepWeights;
        // steps in groups of kGrp (the MMA thread consumes them so): one TMEM fence and one arrive
        // per group
        for (int s = 0; s < kSteps; s += kGrp, gs += kGrp) {
          const int grp = gs / kGrp;
          // the group's A stages are free once the MMAs of the group that used them last are done
          if (grp >= kNGrp) {
            const int q = grp - kNGrp;
            if (!mbar_wait_warp(&sm.adone[q % kNGrp], (q / kNGrp) & 1, wl)) { bad = true; break; }
          }
          // half h expands 32-weight group 2 (s + h2) + h of step s + h2 (16-bit pairs of weights
          // c and c + 16 per column)
#pragma unroll
          for (int h2 = 0; h2 < kGrp; ++h2) {
            const int wi = 2 * (s + h2) + half;
            const uint32_t sc = *reinterpret_cast<const uint16_t*>(pst + (dp ? 16384 : 8192) + srow * 16 + 2 * wi);
            const uint32_t s0 = sc & 0xFFu, s1 = sc >> 8;
            uint32_t av[16];
            if (!dp) {
              // 32-byte-swizzled plane rows: 16-byte piece p of row r at p ^ ((r >> 2) & 1)
              const int wo = srow * 32 + ((((wi >> 2) ^ ((srow >> 2) & 1))) << 4) + 4 * (wi & 3);
              planes_to_16<FC1>(*reinterpret_cast<const uint32_t*>(pst + wo),
                                *reinterpret_cast<const uint32_t*>(pst + 4096 + wo), s0, s1, av);
            } else {
              // 128-byte-swizzled code rows: piece p of row r at p ^ (r & 7)
              delta_to_16<FC1>(*reinterpret_cast<const uint4*>(pst + srow * 128 + ((wi ^ (srow & 7)) << 4)), s0, s1,
                               av);
            }
            tmem_st16(tmem + lane_q + kPColA + 32 * ((gs + h2) % kPAst) + 16 * half, av);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;");
          asm volatile("tcgen05.fence::before_thread_sync;");
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.staged[grp % kNGrp]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.pempty[ps]);
      }
    }
    if (bad && lane == 0) atomicExch(&sm.stuck, 1);
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPTmemCols));
  }
  if (tid == 0 && pf_stuck(sm)) record_error(MOET_ERR_TIMEOUT);
}

// ---------------------------------------------------------------- host side
template <bool FC1>
moet_status launch_pf(const PfArgs& a, const moet_planes* pl, const moet_nvfp4* dl, const void* act,
                      const void* actg, int pairs, int E, cudaStream_t st) {
  PfMaps m;
  std::memset(&m, 0, sizeof(m));
  const uint64_t rowsW = (uint64_t)E * a.N, K = (uint64_t)a.K;
  bool ok = make_map(&m.sign, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, pl->sign, rowsW, K / 32, 8, 64, CU_TENSOR_MAP_SWIZZLE_32B) &&
            make_map(&m.mag, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, pl->mag, rowsW, K / 32, 8, 64, CU_TENSOR_MAP_SWIZZLE_32B) &&
            make_map(&m.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pl->s16, rowsW, K / 16, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE) &&
            make_map(&m.act, FC1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, act,
                     (uint64_t)pairs, K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok && a.delta_slot != nullptr) {
    const uint64_t rowsD = (uint64_t)a.n_slots * a.N;
    ok = make_map(&m.dcodes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, dl->codes, rowsD, K / 2, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&m.ds4, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, dl->s4, rowsD, K / 16, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         make_map(&m.actg, FC1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, actg,
                  (uint64_t)pairs, K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return MOET_ERR_CUDA;
  const int grid = sm_count();
  if (grid <= 0) return MOET_ERR_CUDA;
  auto kern = pf_fc_kernel<FC1>;
  MOET_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPfSmemBytes));
  {
    ProfScope ps(FC1 ? MOET_K_FC1 : MOET_K_FC2, st);
    MOET_CUDA_TRY(pdl_launch(false, kern, dim3(grid), dim3(kPfThreads), kPfSmemBytes, st, a, m));
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}

}  // namespace

namespace {
PfArgs pf_common(const PfForwardArgs& f) {
  const bool with_delta = f.delta_slot != nullptr && f.gate != nullptr;
  PfArgs a{};
  a.T = f.T; a.H = f.H; a.I = f.I; a.k = f.k;
  a.offsets = f.offsets; a.perm = f.perm; a.topk_w = f.topk_w;
  a.delta_slot = with_delta ? f.delta_slot : nullptr; a.n_slots = f.n_slots;
  a.gate = with_delta ? f.gate : nullptr;
  a.hdr = f.hdr; a.chunks = f.chunks;
  return a;
}
}  // namespace

moet_status pf_forward_fc1(const PfForwardArgs& f, cudaStream_t st) {
  const int pairs = f.T * f.k;
  const bool with_delta = f.delta_slot != nullptr && f.gate != nullptr;
  {
    ProfScope ps(MOET_K_TERMS, st);
    MOET_CUDA_TRY(pdl_launch(false, pf_gather_kernel, dim3(pairs), dim3(kGatherThreads), 0, st, pairs, f.k, f.H, f.x, f.perm, with_delta ? f.gate : nullptr, f.topk_idx,
                                           f.n_experts, with_delta ? f.delta_slot : nullptr, f.n_slots, f.xb,
                                           with_delta ? f.xbg : nullptr));
  }
  MOET_CUDA_TRY(cudaGetLastError());
  PfArgs a1 = pf_common(f);
  a1.work = f.work;
  a1.K = f.H; a1.N = 2 * f.I; a1.tiles = f.I / 64;
  a1.scale_2 = f.fc1->scale_2;
  a1.h = f.h;
  return launch_pf<true>(a1, f.fc1, f.dfc1, f.xb, f.xbg, pairs, f.E, st);
}

moet_status pf_forward_fc2(const PfForwardArgs& f, cudaStream_t st) {
  const int pairs = f.T * f.k;
  const bool with_delta = f.delta_slot != nullptr && f.gate != nullptr;
  {
    ProfScope ps(MOET_K_TERMS, st);
    // J output pairs per thread, the fewest that fit the row in kH16MaxThreads threads
    // (pf_supported caps I at 4 * 16 * kH16MaxThreads)
    const int ntt = f.I / 16;
    const int J = ntt <= kH16MaxThreads ? 1 : ntt <= 2 * kH16MaxThreads ? 2 : 4;
    const int threads = ((ntt + J - 1) / J + 31) / 32 * 32;
    auto kern = J == 1 ? pf_h16_kernel<1> : J == 2 ? pf_h16_kernel<2> : pf_h16_kernel<4>;
    MOET_CUDA_TRY(pdl_launch(false, kern, dim3(pairs), dim3(threads), 0, st, pairs, f.k, f.I, f.h, f.perm, with_delta ? f.gate : nullptr, f.topk_idx,
                                    f.n_experts, with_delta ? f.delta_slot : nullptr, f.n_slots, f.h16,
                                    with_delta ? f.hg16 : nullptr, f.hscale));
  }
  MOET_CUDA_TRY(cudaGetLastError());
  PfArgs a2 = pf_common(f);
  a2.work = f.work + 1;
  a2.K = f.I; a2.N = f.H; a2.tiles = f.H / 128;
  a2.scale_2 = f.fc2->scale_2;
  a2.hscale = f.hscale;
  a2.o = f.o;
  return launch_pf<false>(a2, f.fc2, f.dfc2, f.h16, f.hg16, pairs, f.E, st);
}

moet_status pf_forward(const PfForwardArgs& f, cudaStream_t st) {
  const moet_status s = pf_forward_fc1(f, st);
  if (s != MOET_OK) return s;
  return pf_forward_fc2(f, st);
}

}  // namespace moet

MOET_ERROR_ACCESSOR(moet_internal_error_moe_pf)
MOET_DEBUG_WAITS_SETTER(moet_internal_debug_waits_moe_pf)
