// tcgen05 block-scaled FC engine for the decode regime (sm_103a).
//
// README "Frontier MoE on consumer Blackwell (SM120)", "How it fits -- 2-bit
// experts at FP4 quality": decode is HBM-bound, so the 2-bit planes must stream
// at memory speed.  The pages' SM120 kernels feed block-scaled MMAs from a
// PRMT-LUT decode; on sm_103a the block-scaled MMA is tcgen05.mma
// kind::mxf4nvf4 (e2m1 operands, ue4m3 scale per 16 elements, fp32 in TMEM).
//
// Weights.  The 2-bit level set {+-1, +-3} is, halved, exactly the e2m1 values
// {+-0.5, +-1.5}, and s16 is exactly a ue4m3 block-16 scale.  So the planes
// become an exact NVFP4 A operand: each thread expands one weight row of the
// 128-row tile (sign and magnitude words -> e2m1 nibbles s|0|m|1) with a
// handful of integer ops per 8 weights and stores it to TMEM (the A operand of
// tcgen05.mma may live there), with the row scales beside it; the tensor core
// applies the block scale.  The factor 2 of the halved levels is applied in the
// epilogue.
//
// Activations.  Each activation row (bf16 token for FC1, fp32 h for FC2) is
// expanded into kTcTerms NVFP4 terms r = sum_t g_t * e2m1 * ue4m3, each term
// quantising the residual of the previous ones (a block's residual shrinks at
// least ~6x per term, so 4 terms leave ~1e-3 of the block maxima, well inside
// the 5e-3 output tolerance).  The MMA's N dimension holds (token, term)
// pairs; the epilogue sums the terms with their fp32 scales g_t.
//
// K order.  Inside each 16-element block the MMA sees the weights in the
// order produced by the expansion (position 4 r + n holds element r + 4 n);
// the activation terms are stored in the same order ("cperm").  The delta (already NVFP4) is used in its natural order
// against a naturally ordered copy of the terms ("cnat") and accumulates in
// a second TMEM region.
//
// Pipeline: a persistent CTA per SM (16 warps, warp-specialised, no CTA-wide
// barrier in the loop) walks (work item, 128-row weight tile) units.  Two
// producer warps stream each unit's K chunks into a ring of raw shared-memory
// stages with TMA, one lane per box (sign and magnitude planes, row scales, the
// item's activation-term rows and their scales); 8 converter warps expand the
// planes into TMEM A stages and write the scale factors to TMEM; the MMA warp
// issues the MMAs (K = 64 each, one elected lane) and commits them to the stage's "done" barrier
// and, at the end of a unit, to one of two TMEM accumulator buffers that the
// epilogue warps drain while the next unit accumulates.  A scheduler warp
// prepares each unit's record (pairs, routing weights, gate flags, term scales)
// ahead of use.  Every wait is bounded; a stuck CTA records an error, waits for
// its copies and MMAs in flight and releases TMEM.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>

#include "common.cuh"
#include "moe_tc.cuh"
#include "tc_common.cuh"

namespace moet {
namespace {

constexpr int kWsThreads = 512;              // 16 warps, roles in fc_tc_kernel
constexpr int kConvGroups = 2;                // converter groups, one per MMA sub-step of a stage
constexpr int kConvWarps = 4;                 // per group: one warp per 32-row quarter
constexpr int kRaw = 5;                       // raw TMA stages in flight
constexpr int kAst = 2;                       // expanded-A stages (in TMEM)
constexpr int kMeta = 4;                      // unit records in flight
constexpr int kKC = 512;                      // weights per plane stage: two MMA sub-steps of 256
constexpr int kKD = 256;                      // weights per delta stage: one sub-step
constexpr int kMaxN = kTcTerms * kTcTok;      // 64 columns of D
constexpr int kTmemCols = 512;
// TMEM columns: accumulator buffer b holds D at 128 b and the delta's D2 at 128 b + 64;
// A stage s (128 rows x 512 e2m1 = 64 columns; sub-step h at +32 h) at kColA + 64 s;
// scale factors of A stage s at kColSFA + 32 s and kColSFB + 32 s (sub-step h at +16 h)
constexpr int kColA = 256, kColSFA = kColA + 64 * kAst, kColSFB = kColSFA + 32 * kAst;
static_assert(kColSFB + 32 * kAst <= kTmemCols, "TMEM columns");
static_assert(kAst <= kRaw, "an A stage is released by the done barrier of its raw stage");
// raw stage (1024-aligned).  Plane stage: sign and magnitude planes [128 rows][64 B] (SW64),
// row scales [128][32 B] (SW32), activation terms [2 sub-steps][<= 64 rows][128 B] (SW128),
// term scales [<= 64 rows][32 B].  Delta stage: codes [128][128 B] (SW128) at 0, scales
// [128][16 B] at kRDS, terms in natural order [<= 64][128 B] at kRB, term scales [<= 64][16 B].
constexpr int kRSign = 0, kRMag = 8192, kRQ = 16384, kRB = 20480, kRSF = 36864, kRawBytes = 38912;
constexpr int kRDS = 16384;


// Instruction descriptor: kind::mxf4nvf4, A and B e2m1, K-major, ue4m3 scales, M = 128.
__device__ __forceinline__ uint32_t mxf4_idesc(int n) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// The block-scaled MMA (A and B from shared memory), issued by one elected lane of a converged
// warp: the operands are warp-uniform, so they stay in uniform registers.
__device__ __forceinline__ void tc_mma_elect(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sfa,
                                             uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p, e; setp.ne.b32 p, %6, 0; elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p; }"
      ::"r"(d), "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc));
}

// Same MMA with the A operand in TMEM (row = lane, K along the columns, 8 e2m1 per column).
__device__ __forceinline__ void tc_mma_ta_elect(uint32_t d, uint32_t a_tmem, uint64_t bd, uint32_t idesc,
                                                uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p, e; setp.ne.b32 p, %6, 0; elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], [%1], %2, %3, [%4], [%5], p; }"
      ::"r"(d), "r"(a_tmem), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc));
}

// Sign word S and magnitude word M of 32 weights (LSB first) -> 4 words of e2m1
// nibbles (s | 0 | m | 1) = +-0.5 / +-1.5.  W_r collects the weights r + 4 n
// (n = 0..7) with the sign moved to nibble bit 3 and the magnitude to bit 1;
// its low half holds block 0 (bits 0..15), its high half block 1.  Two byte
// permutes per block then give 16 MMA positions p = 4 r + n <- weight r + 4 n.
__device__ __forceinline__ uint4 planes_to_e2m1(uint32_t S, uint32_t M) {
  const uint32_t w0 = 0x11111111u | ((S << 3) & 0x88888888u) | ((M << 1) & 0x22222222u);
  const uint32_t w1 = 0x11111111u | ((S << 2) & 0x88888888u) | (M & 0x22222222u);
  const uint32_t w2 = 0x11111111u | ((S << 1) & 0x88888888u) | ((M >> 1) & 0x22222222u);
  const uint32_t w3 = 0x11111111u | (S & 0x88888888u) | ((M >> 2) & 0x22222222u);
  uint4 o;
  o.x = prmt(w0, w1, 0x5410u);   // block 0: weights 0,4,8,12, 1,5,9,13
  o.y = prmt(w2, w3, 0x5410u);   // block 0: weights 2,6,10,14, 3,7,11,15
  o.z = prmt(w0, w1, 0x7632u);   // block 1
  o.w = prmt(w2, w3, 0x7632u);
  return o;
}

// ---------------------------------------------------------------- activation terms
// Grid (source rows, ceil(K / 16 / 128)), 128 threads: one thread expands one
// 16-element block into kTcTerms NVFP4 terms.  Term t has the fp32 scale
// g_t = m / (6 * 448) / 4^t, m = the row maximum (given: per token for FC1,
// per pair from FC1's epilogue for FC2), and a ue4m3 scale per block chosen
// from the block's current residual, so each term quantises what the previous
// ones left (a block's residual shrinks at least ~6x per term while g_t
// shrinks 4x, keeping the block scales in the normal e4m3 range).  Outputs per
// (output row, term): codes in permuted and natural K order (8 bytes each per
// block), one ue4m3 scale per block, and g_t.  FC1 expands each token once and
// writes it to the bucketed rows of its k pairs (inv = pair -> bucketed
// position); FC2 expands each bucketed pair row in place (inv = null, ncopy = 1).
constexpr int kTermThreads = 128;

// Two e2m1 codes (sign | 3-bit magnitude) by one hardware conversion, round to nearest even with
// saturation at +-6: hi in bits 4-7, lo in bits 0-3.
__device__ __forceinline__ uint32_t e2m1x2_rn(float hi, float lo) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The values of the two e2m1 codes in bits 0-3 (lo) and 4-7 (hi) of c.
__device__ __forceinline__ void e2m1x2_values(uint32_t c, float& lo, float& hi) {
  asm("{ .reg .b8 t; .reg .b16 l, h; .reg .b32 d; cvt.u8.u32 t, %2; cvt.rn.f16x2.e2m1x2 d, t;"
      " mov.b32 {l, h}, d; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h; }"
      : "=f"(lo), "=f"(hi) : "r"(c));
}

// Exchange of the nibbles at the positions in m with those d nibbles above them.
__device__ __forceinline__ uint64_t nibble_swap(uint64_t x, int d, uint64_t m) {
  const uint64_t t = ((x >> (4 * d)) ^ x) & m;
  return x ^ t ^ (t << (4 * d));
}

// The kTcTerms NVFP4 terms of one 16-element block r (the residual is updated in place) under the
// row's first term scale g0: per term the codes in natural order (nat) and in the expansion's
// order (per), two words each, and the ue4m3 block scale.  A term's codes are RNE(r_i / sc) in
// e2m1 (one conversion per two elements, ratios rounded to fp32 first; an exact tie may go
// either way, which only changes what the next term quantises) and its residual is
// r_i - value_i * sc in one fused multiply-add.
__device__ __forceinline__ void block_terms(float (&r)[16], float g0, uint32_t (&nat)[kTcTerms][2],
                                            uint32_t (&per)[kTcTerms][2], uint32_t (&sfo)[kTcTerms]) {
#pragma unroll
  for (int t = 0; t < kTcTerms; ++t) {
    const float g = ldexpf(g0, -2 * t);
    float bm = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bm = fmaxf(bm, fabsf(r[i]));
    uint32_t sf = 0;
    float sc = 0.0f;
    if (g > 0.0f) {
      sf = f32_to_e4m3_rn(bm / (6.0f * g));
      sc = e4m3_to_f32(sf) * g;
    }
    const float inv = sc > 0.0f ? 1.0f / sc : 0.0f;     // sc = 0: every code 0, r unchanged
    // natural order: nibble i holds element i
    uint64_t n = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t c = e2m1x2_rn(r[2 * i + 1] * inv, r[2 * i] * inv);
      float v0, v1;
      e2m1x2_values(c, v0, v1);
      r[2 * i] = fmaf(-v0, sc, r[2 * i]);
      r[2 * i + 1] = fmaf(-v1, sc, r[2 * i + 1]);
      n |= (uint64_t)c << (8 * i);
    }
    // expansion order: position p = 4 a + b holds element a + 4 b, the transpose of the 4 x 4
    // nibble matrix (row a = nibbles 4 a .. 4 a + 3) by two exchanges: the off-diagonal 2 x 2
    // blocks (nibbles 2, 3, 6, 7 <-> 8, 9, 12, 13), then inside each 2 x 2 block
    uint64_t q = nibble_swap(n, 6, 0x00000000FF00FF00ull);
    q = nibble_swap(q, 3, 0x0000F0F00000F0F0ull);
    nat[t][0] = (uint32_t)n;
    nat[t][1] = (uint32_t)(n >> 32);
    per[t][0] = (uint32_t)q;
    per[t][1] = (uint32_t)(q >> 32);
    sfo[t] = sf;
  }
}

// The 16 source elements of block b of a row: bf16 (FC1 input x) or fp32 (FC2 input h).
template <bool BF16_IN>
__device__ __forceinline__ void load_block(const void* __restrict__ src, size_t srow, int K, int b, float (&r)[16]) {
  if (BF16_IN) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + srow * K + 16 * b);
    const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      r[2 * i] = __uint_as_float(w[i] << 16);
      r[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + srow * K + 16 * b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = p[i];
      r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
    }
  }
}

__device__ __forceinline__ void store_block_terms(int K, int b, size_t orow, const uint32_t (&nat)[kTcTerms][2],
                                                  const uint32_t (&per)[kTcTerms][2],
                                                  const uint32_t (&sfo)[kTcTerms], uint8_t* __restrict__ cperm,
                                                  uint8_t* __restrict__ cnat, uint8_t* __restrict__ sfb,
                                                  bool want_nat) {
#pragma unroll
  for (int t = 0; t < kTcTerms; ++t) {
    const size_t term_row = orow * kTcTerms + t;
    if (want_nat) *reinterpret_cast<uint2*>(cnat + term_row * (K / 2) + 8 * b) = make_uint2(nat[t][0], nat[t][1]);
    *reinterpret_cast<uint2*>(cperm + term_row * (K / 2) + 8 * b) = make_uint2(per[t][0], per[t][1]);
    sfb[term_row * (K / 16) + b] = (uint8_t)sfo[t];
  }
}

// The natural-order copy of a pair's terms is read only by the delta stages (an expert with a
// delta slot), and only gated pairs' columns count there: other rows are not written.
struct NatRows {
  const int32_t* topk_idx;     // null: no delta table (no row needs the copy)
  const int32_t* delta_slot;
  const uint8_t* gate;
  int k, n_experts, n_slots;
  __device__ __forceinline__ bool want(int p) const {
    if (topk_idx == nullptr) return false;
    const int e = __ldg(topk_idx + p);
    if (e < 0 || e >= n_experts || !__ldg(gate + p / k)) return false;
    const int s = __ldg(delta_slot + e);
    return s >= 0 && s < n_slots;
  }
};

// Grid (source rows, ceil(K / 16 / 128)), 128 threads: one thread expands one 16-element block
// into kTcTerms NVFP4 terms.  Term t has the fp32 scale g_t = m / (6 * 448) / 4^t, m = the row
// maximum (given: per token for FC1, per pair from FC1's epilogue for FC2), and a ue4m3 scale per
// block chosen from the block's current residual, so each term quantises what the previous ones
// left (a block's residual shrinks at least ~6x per term while g_t shrinks 4x, keeping the block
// scales in the normal e4m3 range).  Outputs per (output row, term): codes in permuted and natural
// K order (8 bytes each per block), one ue4m3 scale per block, and g_t.  FC1 expands each token
// once and writes it to the bucketed rows of its k pairs (inv = pair -> bucketed position); FC2
// expands each bucketed pair row in place (inv = null, ncopy = 1; perm gives the row's pair).
// The output rows of source row `row` (ncopy <= 32 of them) and whether each needs the
// natural-order copy, looked up once per warp: lane cp holds copy cp's output row (-1: skipped,
// out of range) and its flag, so the lookups of all copies are in flight together.  The row's
// pair is token row x k + copy (FC1, inv given) or the bucketed row's pair (FC2, inv null).
struct CopyInfo {
  int orow;
  bool want;
};
__device__ __forceinline__ CopyInfo copy_info(int row, int lane, const int32_t* __restrict__ inv, int ncopy,
                                              int out_rows, const int32_t* __restrict__ perm, const NatRows& nr) {
  CopyInfo ci{-1, false};
  if (lane < ncopy) {
    const int r = inv ? __ldg(inv + (size_t)row * ncopy + lane) : row;
    if (r >= 0 && r < out_rows) {
      ci.orow = r;
      const int p = inv ? row * ncopy + lane : __ldg(perm + row);
      ci.want = p >= 0 && p < out_rows && nr.want(p);
    }
  }
  return ci;
}

template <bool BF16_IN>
__global__ void __launch_bounds__(kTermThreads) act_terms_kernel(int K, const void* __restrict__ src,
                                                                const int32_t* __restrict__ inv, int ncopy,
                                                                int out_rows, const float* __restrict__ rowmax,
                                                                uint8_t* __restrict__ cperm, uint8_t* __restrict__ cnat,
                                                                uint8_t* __restrict__ sfb, float* __restrict__ gsc,
                                                                const int32_t* __restrict__ perm, NatRows nr) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const size_t srow = (size_t)row;
  const float m = __ldg(rowmax + srow);
  const float g0 = m / (6.0f * 448.0f);
  const CopyInfo ci = copy_info(row, lane, inv, ncopy, out_rows, perm, nr);
  const int b = blockIdx.y * kTermThreads + tid;            // 16-element block of the row
  const bool active = b < K / 16;
  if (blockIdx.y == 0 && tid < 32) {
    for (int cp = 0; cp < ncopy; ++cp) {
      const int orow = __shfl_sync(0xffffffffu, ci.orow, cp);
      if (orow >= 0 && lane < kTcTerms) gsc[(size_t)orow * kTcTerms + lane] = ldexpf(g0, -2 * lane);
    }
  }
  if (__all_sync(0xffffffffu, !active)) return;            // the whole warp is past the row's end
  // every lane of the warp stays (the copies' rows come from lanes 0 .. ncopy - 1); lanes past
  // the row's end expand zeros and store nothing
  float r[16];
  if (active) {
    load_block<BF16_IN>(src, srow, K, b, r);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = 0.0f;
  }
  uint32_t nat[kTcTerms][2], per[kTcTerms][2], sfo[kTcTerms];
  block_terms(r, g0, nat, per, sfo);
  for (int cp = 0; cp < ncopy; ++cp) {
    const int orow = __shfl_sync(0xffffffffu, ci.orow, cp);
    const bool want = __shfl_sync(0xffffffffu, ci.want ? 1 : 0, cp) != 0;
    if (orow >= 0 && active) store_block_terms(K, b, (size_t)orow, nat, per, sfo, cperm, cnat, sfb, want);
  }
}

// The same expansion for the term rows of a work-item list (the prefill regime's experts with few
// pairs): term row j belongs to slot j % kTcTok of item j / kTcTok, i.e. to the pair at bucketed
// position offsets[e] + first + j % kTcTok (rows past the item's count are not written).  The
// source row is the pair's token (FC1, bf16 x, row maximum per token) or the pair's bucketed
// position (FC2, fp32 h, row maximum per pair).  Grid-stride over (row, 16-element block).
template <bool BF16_IN>
__global__ void __launch_bounds__(256) act_terms_items_kernel(int K, const void* __restrict__ src,
                                                             const int* __restrict__ n_items,
                                                             const int4* __restrict__ chunks,
                                                             const int32_t* __restrict__ offsets,
                                                             const int32_t* __restrict__ perm, int k, int pairs,
                                                             const float* __restrict__ rowmax,
                                                             uint8_t* __restrict__ cperm, uint8_t* __restrict__ cnat,
                                                             uint8_t* __restrict__ sfb, float* __restrict__ gsc,
                                                             NatRows nr) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  const int nb = K / 16;
  const long long total = (long long)__ldg(n_items) * kTcTok * nb;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(idx / nb), b = (int)(idx - (long long)row * nb);
    const int4 ch = __ldg(chunks + row / kTcTok);
    const int slot = row % kTcTok;
    if (slot >= ch.z) continue;
    const int pos = __ldg(offsets + ch.x) + ch.y + slot;
    const int p = pos >= 0 && pos < pairs ? __ldg(perm + pos) : -1;
    if (p < 0 || p >= pairs) {
      record_error(MOET_ERR_DEVICE_INDEX);
      continue;
    }
    const size_t srow = BF16_IN ? (size_t)(p / k) : (size_t)pos;
    const float g0 = __ldg(rowmax + srow) / (6.0f * 448.0f);
    if (b == 0) {
#pragma unroll
      for (int t = 0; t < kTcTerms; ++t) gsc[(size_t)row * kTcTerms + t] = ldexpf(g0, -2 * t);
    }
    float r[16];
    load_block<BF16_IN>(src, srow, K, b, r);
    uint32_t nat[kTcTerms][2], per[kTcTerms][2], sfo[kTcTerms];
    block_terms(r, g0, nat, per, sfo);
    store_block_terms(K, b, (size_t)row, nat, per, sfo, cperm, cnat, sfb, nr.want(p));
  }
}

// ---------------------------------------------------------------- FC kernel
struct TmaMaps {
  CUtensorMap sign, mag, q;        // planes u32 [E N, K/32] box {16, 64} SW64; s16 u8 [E N, K/16] box {32, 64} SW32
  CUtensorMap act, actn;           // terms u8 [pairs 4, K/2] box {128, brows} SW128 (permuted / natural order)
  CUtensorMap sfb2, sfb1;          // term scales u8 [pairs 4, K/16] box {32, brows} / {16, brows}
  CUtensorMap dcodes, ds4;         // delta u8 [S N, K/2] box {128, 64} SW128; scales box {16, 64}
};

struct FcTcArgs {
  int T, H, I, k, K, N;          // N = rows of one expert matrix
  int tiles;                     // 128-row weight tiles per expert matrix
  int brows;                     // rows of one activation-term box: min(16, 4 * term rows)
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
  const float* gsc;
  float* out;
  unsigned* hmax;                // FC1: max |h| per bucketed pair (fp32 bits), for the FC2 terms
  int item_rows;                 // 1: activation-term rows at item * kTcTok (act_terms_items_kernel),
                                 // 0: at the pair's bucketed position
};

// One unit of work = (work item, 128-row weight tile), written by the scheduler warp.
struct UnitMeta {
  int e, pos0, ntok, ncols;      // e: the planes' expert (pool slot) index
  int dslot;                     // delta slot when the unit runs the delta pass, else -1
  int nch;                       // stages: ceil(K/512) plane stages (+ K/256 delta stages)
  int r0, r1;                    // first weight rows of the tile's two 64-row halves
  float sc2;                     // the expert's scale_2
  int crow0;                     // first activation-term source row of the item
  int pad[6];
  int pair[kTcTok];              // pair id t k + j per token column (-1 = none)
  float wts[kTcTok];             // routing weight per token column
  float gate_f[kTcTok];          // 1 = the delta counts for this column
  float gsc[kMaxN];              // term scales g_t, column order
};
static_assert(sizeof(UnitMeta) == 512, "UnitMeta layout");

struct TcSmem {
  uint64_t full[kRaw];           // TMA bytes of the raw stage landed
  uint64_t done[kRaw];           // MMAs of the stage done (raw stage and its A stage free)
  uint64_t staged[kAst];         // converters done (A expanded, scales in TMEM)
  uint64_t acc_full[2];          // unit's accumulation complete
  uint64_t acc_empty[2];         // epilogue has read the accumulators
  uint64_t meta_full[kMeta];
  uint64_t meta_empty[kMeta];
  uint32_t tmem_base;
  int stuck;
};

constexpr size_t kXchgBytes = 64 * kTcTok * sizeof(float);
constexpr size_t kSmemBytes =
    1024 + (size_t)kRaw * kRawBytes + kXchgBytes + kMeta * sizeof(UnitMeta) + sizeof(TcSmem);
static_assert(kSmemBytes <= 232448, "shared memory over the per-CTA limit");

__device__ __forceinline__ bool is_stuck(const TcSmem& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.stuck) != 0;
}

__device__ __forceinline__ void set_stuck(TcSmem& sm) { atomicExch(&sm.stuck, 1); }

// Persistent warp-specialised FC: one CTA per SM walks the units u = blockIdx.x
// + j gridDim.x of the (work item x weight tile) grid.  Warp roles:
//   0, 3   producers, alternate stages: each TMA box of a stage is issued by
//          its own lane (one instruction), into a ring of kRaw raw stages
//   1      TMEM owner; issues the MMAs and their commits (warp-uniform, one elected lane)
//   2      scheduler: per unit, the item's pairs, weights, gate flags and term
//          scales into a ring of kMeta unit records
//   4-7    epilogue (TMEM lane quarters 0-3): term sums, SiLU * up / routing
//          weight, stores; the accumulators are double-buffered in TMEM so the
//          next unit's MMAs run while the epilogue reads this one's
//   8-15   converters in two groups of four warps (one per 32-row quarter);
//          group h takes sub-step h of every stage: planes -> e2m1 A operand
//          and scale factors, both stored straight into TMEM (each thread owns
//          the TMEM lane of its weight row), so the expanded A never touches
//          shared memory
// Main pass per unit: stages of 512 weights from the 2-bit planes (two MMA
// sub-steps of 256; converter group h expands sub-step h).  Delta pass (cached
// expert with a gated pair): the NVFP4 delta in stages of 256 weights, its
// codes used as the A operand straight from shared memory; it accumulates
// into a second TMEM region.
template <bool FC1>
__global__ void __launch_bounds__(kWsThreads, 1) fc_tc_kernel(const FcTcArgs a, const __grid_constant__ TmaMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem_dyn[];
  unsigned char* base = smem_dyn + ((1024 - (smem_addr(smem_dyn) & 1023)) & 1023);
  unsigned char* raw = base;
  float (*xchg)[kTcTok] = reinterpret_cast<float (*)[kTcTok]>(base + kRaw * kRawBytes);
  UnitMeta* meta = reinterpret_cast<UnitMeta*>(base + kRaw * kRawBytes + kXchgBytes);
  TcSmem& sm = *reinterpret_cast<TcSmem*>(meta + kMeta);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wl = wait_limit();
  // Units are handed out one at a time from a global counter (the scheduler warp takes the next
  // one when a record slot is free), so CTAs that draw units with a delta pass (three times the
  // stages) take fewer; items of delta experts come first in the item list.  The record after a
  // CTA's last unit has nch = -1 and ends every role's loop.
  const int nps = (a.K + kKC - 1) / kKC;        // plane stages per unit

  if (tid == 0) {
    sm.stuck = 0;
    for (int s = 0; s < kRaw; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.done[s], 1); }
    for (int s = 0; s < kAst; ++s) mbar_init(&sm.staged[s], kConvGroups * kConvWarps);
    for (int s = 0; s < 2; ++s) { mbar_init(&sm.acc_full[s], 1); mbar_init(&sm.acc_empty[s], 4); }
    for (int s = 0; s < kMeta; ++s) { mbar_init(&sm.meta_full[s], 1); mbar_init(&sm.meta_empty[s], 4); }
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&sm.tmem_base)),
                 "r"(kTmemCols));
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

  if (warp == 0 || warp == 3) {
    // ---------------- producers: warp pw takes the stages g with g % 2 == pw; the
    // stage's boxes are issued by one lane each in the same instruction
    const int pw = warp == 0 ? 0 : 1;
    int g = 0;
    bool bad = false;
    for (int j = 0; !bad; ++j) {
      const int m = j % kMeta;
      if (!mbar_wait_warp(&sm.meta_full[m], (j / kMeta) & 1, wl)) { bad = true; break; }
      const UnitMeta& um = meta[m];
      if (um.nch < 0) break;                                  // no more units
      const int nch = um.nch, dslot = um.dslot;
      const int nbox = um.ncols / 16;
      const int y0 = (dslot >= 0 ? dslot : um.e) * a.N;      // delta rows only used by delta stages
      const int w0 = um.e * a.N + um.r0, w1 = um.e * a.N + um.r1;
      const int trow0 = um.crow0 * kTcTerms;                // first activation-term row of the item
      for (int c = 0; c < nch; ++c, ++g) {
        if ((g & 1) != pw) continue;
        const int rs = g % kRaw, ru = g / kRaw;
        if (ru > 0 && !mbar_wait_warp(&sm.done[rs], (ru - 1) & 1, wl)) { bad = true; break; }
        unsigned char* st = raw + rs * kRawBytes;
        uint64_t* fb = &sm.full[rs];
        const bool dp = c >= nps;
        const int nsub = dp ? 1 : min(2, (a.K - kKC * c) / kKD);
        if (lane == 0) {
          const uint32_t bx_bytes = (uint32_t)a.brows * (dp ? 128u + 16u : 128u * nsub + 32u);
          mbar_expect_tx(fb, (dp ? 16384u + 2048u : 20480u) + (uint32_t)nbox * bx_bytes);
        }
        __syncwarp();
        // lane -> box: weight boxes (two 64-row halves each), then the item's term boxes (16 rows each)
        const CUtensorMap* map = nullptr;
        uint32_t dst = 0;
        int x = 0, y = 0;
        if (!dp) {
          if (lane < 6) {
            const int hv = lane & 1;
            map = lane < 2 ? &maps.sign : lane < 4 ? &maps.mag : &maps.q;
            dst = smem_addr(st + (lane < 2 ? kRSign + 4096 * hv : lane < 4 ? kRMag + 4096 * hv : kRQ + 2048 * hv));
            x = lane < 4 ? c * 16 : c * 32;
            y = hv ? w1 : w0;
          } else if (lane < 6 + nsub * nbox) {
            const int q = lane - 6, sub = q / nbox, bx = q - sub * nbox;
            map = &maps.act;
            dst = smem_addr(st + kRB + 8192 * sub + 2048 * bx);
            x = (2 * c + sub) * 128;
            y = trow0 + 16 * bx;
          } else if (lane < 6 + (nsub + 1) * nbox) {
            const int bx = lane - 6 - nsub * nbox;
            map = &maps.sfb2;
            dst = smem_addr(st + kRSF + 512 * bx);
            x = c * 32;
            y = trow0 + 16 * bx;
          }
        } else {
          const int dc = c - nps;
          if (lane < 4) {
            const int hv = lane & 1;
            map = lane < 2 ? &maps.dcodes : &maps.ds4;
            dst = smem_addr(st + (lane < 2 ? 8192 * hv : kRDS + 1024 * hv));
            x = lane < 2 ? dc * 128 : dc * 16;
            y = y0 + (hv ? um.r1 : um.r0);
          } else if (lane < 4 + nbox) {
            const int bx = lane - 4;
            map = &maps.actn;
            dst = smem_addr(st + kRB + 2048 * bx);
            x = dc * 128;
            y = trow0 + 16 * bx;
          } else if (lane < 4 + 2 * nbox) {
            const int bx = lane - 4 - nbox;
            map = &maps.sfb1;
            dst = smem_addr(st + kRSF + 256 * bx);
            x = dc * 16;
            y = trow0 + 16 * bx;
          }
        }
        if (map != nullptr) tma_load_2d(dst, map, x, y, fb);
      }
    }
    if (bad && lane == 0) set_stuck(sm);
    // every copy this warp issued has landed before the CTA may exit
    if (lane == 0)
      for (int i = g > kRaw ? g - kRaw : 0; i < g; ++i)
        if ((i & 1) == pw) mbar_wait(&sm.full[i % kRaw], (i / kRaw) & 1, wl);
  } else if (warp == 1) {
    // ---------------- MMA issue.  The whole warp walks the loop, so every operand (descriptors,
    // TMEM addresses, loop state) is warp-uniform and stays in the uniform datapath; one elected
    // lane issues each MMA and commit.  A stage's shared-memory descriptors are its base
    // descriptor plus constant offsets (byte offset / 16 in the address field, which cannot
    // carry: shared addresses stay below 256 KB).
    int g = 0, last = -1;
    bool bad = false;
    const uint64_t raw_desc = sw128_desc(smem_addr(raw));
    for (int j = 0; !bad; ++j) {
      const int m = j % kMeta, ab = j & 1;
      if (!mbar_wait_warp(&sm.meta_full[m], (j / kMeta) & 1, wl)) { bad = true; break; }
      if (meta[m].nch < 0) break;                            // no more units
      if (j >= 2 && !mbar_wait_warp(&sm.acc_empty[ab], ((j >> 1) - 1) & 1, wl)) { bad = true; break; }
      if (__any_sync(0xffffffffu, is_stuck(sm))) { bad = true; break; }
      asm volatile("tcgen05.fence::after_thread_sync;");
      const int nch = meta[m].nch;
      const uint32_t idesc = mxf4_idesc(meta[m].ncols);
      const uint32_t dcol = tmem + 128 * ab;
      for (int c = 0; c < nch; ++c, ++g) {
        const int as = g % kAst, au = g / kAst, rs = g % kRaw;
        if (!mbar_wait_warp(&sm.staged[as], au & 1, wl)) { bad = true; break; }
        asm volatile("tcgen05.fence::after_thread_sync;");
        const uint64_t rd = raw_desc + (uint64_t)((rs * kRawBytes) >> 4);
        const uint32_t sfa = tmem + kColSFA + 32 * as, sfb = tmem + kColSFB + 32 * as;
        if (c < nps) {
          const int nsub = min(2, (a.K - kKC * c) / kKD);
          const uint32_t ata = tmem + kColA + 64 * as;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h < nsub) {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                tc_mma_ta_elect(dcol, ata + 32 * h + 8 * i, rd + (uint64_t)((kRB + 8192 * h + 32 * i) >> 4), idesc,
                                sfa + 16 * h + 4 * i, sfb + 16 * h + 4 * i, (c > 0 || h > 0 || i > 0) ? 1u : 0u);
            }
          }
        } else {
          const int dc = c - nps;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            tc_mma_elect(dcol + 64, rd + (uint64_t)((32 * i) >> 4), rd + (uint64_t)((kRB + 32 * i) >> 4), idesc,
                         sfa + 4 * i, sfb + 4 * i, (dc > 0 || i > 0) ? 1u : 0u);
        }
        tc_commit_elect(&sm.done[rs]);
        last = g;
      }
      if (bad) break;
      tc_commit_elect(&sm.acc_full[ab]);
    }
    if (bad && lane == 0) set_stuck(sm);
    // every MMA this warp issued is complete before TMEM is released
    if (last >= 0 && lane == 0) mbar_wait(&sm.done[last % kRaw], (last / kRaw) & 1, wl);
    __syncwarp();
  } else if (warp == 2) {
    // ---------------- scheduler
    for (int j = 0;; ++j) {
      const int m = j % kMeta;
      if (j >= kMeta && !mbar_wait_warp(&sm.meta_empty[m], ((j / kMeta) - 1) & 1, wl)) {
        if (lane == 0) set_stuck(sm);
        break;
      }
      if (__any_sync(0xffffffffu, is_stuck(sm))) break;
      int u = 0;
      if (lane == 0) u = atomicAdd(a.work, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      // (a test can make CTA 0 withhold its first record: every wait on it then runs out)
      const bool withhold = blockIdx.x == 0 && j == 0 && *reinterpret_cast<volatile int*>(&g_dbg_withhold) != 0;
      if (u >= total_units) {
        if (lane == 0) meta[m].nch = -1;                     // the end record
        __syncwarp();
        if (lane == 0 && !withhold) mbar_arrive(&sm.meta_full[m]);
        break;
      }
      const int item = u / a.tiles, tile = u - item * a.tiles;
      const int4 ch = a.chunks[item];
      const int e = ch.x, ntok = ch.z;
      const int pe = ch.w;                 // pool slot of the expert's planes and scale_2
      const int pos0 = __ldg(a.offsets + e) + ch.y;
      const int crow0 = a.item_rows ? item * kTcTok : pos0;
      int dslot = -1;
      if (a.delta_slot != nullptr && a.gate != nullptr) {
        dslot = __ldg(a.delta_slot + e);
        if (dslot >= a.n_slots) {
          if (lane == 0) record_error(MOET_ERR_DEVICE_INDEX);
          dslot = -1;
        }
      }
      int pr = -1;
      float wv = 0.0f, gf = 0.0f;
      if (lane < ntok && lane < kTcTok) {
        const int p = __ldg(a.perm + pos0 + lane);
        if (p < 0 || p >= a.T * a.k) {
          record_error(MOET_ERR_DEVICE_INDEX);
        } else {
          pr = p;
          wv = __ldg(a.topk_w + p);
          if (dslot >= 0 && __ldg(a.gate + p / a.k)) gf = 1.0f;
        }
      }
      if (!__any_sync(0xffffffffu, gf != 0.0f)) dslot = -1;
      UnitMeta& um = meta[m];
      if (lane < kTcTok) { um.pair[lane] = pr; um.wts[lane] = wv; um.gate_f[lane] = gf; }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int col = lane + 32 * h2, tk = col / kTcTerms;
        const int ptk = __shfl_sync(0xffffffffu, pr, tk);
        um.gsc[col] = tk < ntok && ptk >= 0 ? __ldg(a.gsc + (size_t)(crow0 + tk) * kTcTerms + col % kTcTerms) : 0.0f;
      }
      if (lane == 0) {
        um.e = pe; um.pos0 = pos0; um.ntok = ntok; um.crow0 = crow0;
        um.ncols = ((kTcTerms * ntok + 15) / 16) * 16;
        um.dslot = dslot;
        um.nch = dslot >= 0 ? nps + a.K / kKD : nps;
        um.r0 = FC1 ? tile * 64 : tile * 128;
        um.r1 = FC1 ? a.I + tile * 64 : tile * 128 + 64;
        um.sc2 = __ldg(a.scale_2 + pe);
      }
      __syncwarp();
      if (lane == 0 && !withhold) mbar_arrive(&sm.meta_full[m]);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- epilogue: TMEM lane quarter warp & 3
    const int trow = 32 * (warp & 3) + lane;
    const uint32_t lane_q = (uint32_t)((warp & 3) * 32) << 16;
    for (int j = 0;; ++j) {
      const int m = j % kMeta, ab = j & 1;
      bool ok = mbar_wait_warp(&sm.meta_full[m], (j / kMeta) & 1, wl);
      if (ok && meta[m].nch < 0) break;                      // no more units (same for all four warps)
      ok = ok && mbar_wait_warp(&sm.acc_full[ab], (j >> 1) & 1, wl);
      asm volatile("tcgen05.fence::after_thread_sync;");
      if (epi_any(!ok || is_stuck(sm))) {
        if (!ok && lane == 0) set_stuck(sm);
        break;
      }
      const UnitMeta& um = meta[m];
      const int ncols = um.ncols, ntok = um.ntok, pos0 = um.pos0;
      const bool do_delta = um.dslot >= 0;
      const float sc2 = 2.0f * um.sc2;          // 2: the halved e2m1 levels
      const float sc2d = um.sc2;
      const int wrow = trow < 64 ? um.r0 + trow : um.r1 + trow - 64;
      const uint32_t dcol = tmem + lane_q + 128 * ab;
      for (int c0 = 0; c0 < ncols; c0 += 16) {
        float v[16], v2[16];
        tmem_ld16(dcol + c0, v);
        if (do_delta) tmem_ld16(dcol + 64 + c0, v2);
        float acc[16 / kTcTerms];
#pragma unroll
        for (int q = 0; q < 16 / kTcTerms; ++q) {
          const int tk = c0 / kTcTerms + q;
          // delta columns count only for gated pairs (the B box also holds other pairs' rows)
          const bool gated = do_delta && um.gate_f[tk] != 0.0f;
          float sacc = 0.0f;
#pragma unroll
          for (int t = 0; t < kTcTerms; ++t) {
            const int col = q * kTcTerms + t;
            float d = sc2 * v[col];
            if (gated) d = fmaf(sc2d, v2[col], d);
            sacc = fmaf(um.gsc[c0 + col], d, sacc);
          }
          acc[q] = sacc;
        }
        if (!FC1) {
#pragma unroll
          for (int q = 0; q < 16 / kTcTerms; ++q) {
            const int tk = c0 / kTcTerms + q;
            const int pr = um.pair[tk];
            if (tk < ntok && pr >= 0) a.out[(size_t)pr * a.H + wrow] = acc[q] * um.wts[tk];
          }
        } else {
          if (trow >= 64) {
#pragma unroll
            for (int q = 0; q < 16 / kTcTerms; ++q) xchg[trow - 64][c0 / kTcTerms + q] = acc[q];
          }
          asm volatile("bar.sync 1, 128;");
          if (trow < 64) {
#pragma unroll
            for (int q = 0; q < 16 / kTcTerms; ++q) {
              const int tk = c0 / kTcTerms + q;
              const bool valid = tk < ntok && um.pair[tk] >= 0;
              float hv = 0.0f;
              if (valid) {
                const float gv = acc[q], uv = xchg[trow][tk];
                hv = gv / (1.0f + expf(-gv)) * uv;
                a.out[(size_t)(pos0 + tk) * a.I + wrow] = hv;
              }
              float mx = fabsf(hv);
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
              if (lane == 0 && valid) atomicMax(a.hmax + pos0 + tk, __float_as_uint(mx));
            }
          }
          asm volatile("bar.sync 1, 128;");
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.acc_empty[ab]);
        mbar_arrive(&sm.meta_empty[m]);
      }
    }
  } else if (warp >= 8) {
    // ---------------- converters: group grp expands sub-step grp (256 weights) of
    // every plane stage (group 0 handles the delta stages); in a group, one warp per
    // 32-row quarter, each thread one row: its 8 plane words -> 32 TMEM columns, then
    // the sub-step's row scales and activation-term scales
    const int grp = (warp - 8) >> 2;
    const int trow = 32 * (warp & 3) + lane;
    const uint32_t lane_q = (uint32_t)((warp & 3) * 32) << 16;
    // 64-byte-swizzled plane rows: 16-byte piece p of row r sits at piece p ^ ((r >> 1) & 3)
    const int praw0 = trow * 64 + (((2 * grp) ^ ((trow >> 1) & 3)) << 4);
    const int praw1 = trow * 64 + (((2 * grp + 1) ^ ((trow >> 1) & 3)) << 4);
    int g = 0;
    bool bad = false;
    for (int j = 0; !bad; ++j) {
      const int m = j % kMeta;
      if (!mbar_wait_warp(&sm.meta_full[m], (j / kMeta) & 1, wl)) { bad = true; break; }
      if (meta[m].nch < 0) break;                            // no more units
      if (__any_sync(0xffffffffu, is_stuck(sm))) { bad = true; break; }
      const int nch = meta[m].nch, ncols = meta[m].ncols;
      for (int c = 0; c < nch; ++c, ++g) {
        const int rs = g % kRaw, ru = g / kRaw, as = g % kAst;
        if (!mbar_wait_warp(&sm.full[rs], ru & 1, wl)) { bad = true; break; }
        // the A stage is free once the MMAs of stage g - kAst are done
        if (g >= kAst && !mbar_wait_warp(&sm.done[(g - kAst) % kRaw], ((g - kAst) / kRaw) & 1, wl)) { bad = true; break; }
        const bool dp = c >= nps;
        const int nsub = dp ? 1 : min(2, (a.K - kKC * c) / kKD);
        if (grp < nsub) {
          const unsigned char* st = raw + rs * kRawBytes;
          if (!dp) {
            // this thread's 256 weights of the row -> 32 TMEM columns of its lane (K order)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int pr = hh ? praw1 : praw0;
              const uint4 sw = *reinterpret_cast<const uint4*>(st + kRSign + pr);
              const uint4 mw = *reinterpret_cast<const uint4*>(st + kRMag + pr);
              uint32_t av[16];
              const uint4 e0 = planes_to_e2m1(sw.x, mw.x), e1 = planes_to_e2m1(sw.y, mw.y);
              const uint4 e2 = planes_to_e2m1(sw.z, mw.z), e3 = planes_to_e2m1(sw.w, mw.w);
              av[0] = e0.x; av[1] = e0.y; av[2] = e0.z; av[3] = e0.w;
              av[4] = e1.x; av[5] = e1.y; av[6] = e1.z; av[7] = e1.w;
              av[8] = e2.x; av[9] = e2.y; av[10] = e2.z; av[11] = e2.w;
              av[12] = e3.x; av[13] = e3.y; av[14] = e3.z; av[15] = e3.w;
              tmem_st16(tmem + lane_q + kColA + 64 * as + 32 * grp + 16 * hh, av);
            }
          }
          // scale factors to TMEM, replicated layout: rows lane + 32 j -> columns 4 i + j; the row
          // scales (A) and the activation-term scales (B) of this sub-step
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t v[16];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int n = lane + 32 * jj;
              uint4 q = make_uint4(0u, 0u, 0u, 0u);
              if (half == 0) {
                // plane row scales: 32-byte-swizzled rows, piece h of row n at h ^ ((n >> 2) & 1)
                const int off = dp ? kRDS + n * 16 : kRQ + n * 32 + ((grp ^ ((n >> 2) & 1)) << 4);
                q = *reinterpret_cast<const uint4*>(st + off);
              } else if (n < ncols) {
                q = *reinterpret_cast<const uint4*>(st + kRSF + (dp ? n * 16 : n * 32 + 16 * grp));
              }
              v[0 * 4 + jj] = q.x; v[1 * 4 + jj] = q.y; v[2 * 4 + jj] = q.z; v[3 * 4 + jj] = q.w;
            }
            tmem_st16(tmem + lane_q + (half ? kColSFB : kColSFA) + 32 * as + 16 * grp, v);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;");
          asm volatile("tcgen05.fence::before_thread_sync;");
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.staged[as]);
      }
    }
    if (bad && lane == 0) set_stuck(sm);
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
  if (tid == 0 && is_stuck(sm)) record_error(MOET_ERR_TIMEOUT);
}

// ---------------------------------------------------------------- host side
template <bool FC1>
moet_status launch_fc_tc(const FcTcArgs& a, const moet_planes* pl, const moet_nvfp4* dl, const uint8_t* cperm,
                         const uint8_t* cnat, const uint8_t* sfb, int act_rows, int E, int row_tiles,
                         cudaStream_t st) {
  TmaMaps m;
  std::memset(&m, 0, sizeof(m));
  const uint32_t brows = (uint32_t)(act_rows * kTcTerms < 16 ? act_rows * kTcTerms : 16);
  const uint64_t rowsW = (uint64_t)E * a.N, K = (uint64_t)a.K;
  const uint64_t trows = (uint64_t)act_rows * kTcTerms;
  bool ok = make_map(&m.sign, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, pl->sign, rowsW, K / 32, 16, 64, CU_TENSOR_MAP_SWIZZLE_64B) &&
            make_map(&m.mag, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, pl->mag, rowsW, K / 32, 16, 64, CU_TENSOR_MAP_SWIZZLE_64B) &&
            make_map(&m.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pl->s16, rowsW, K / 16, 32, 64, CU_TENSOR_MAP_SWIZZLE_32B) &&
            make_map(&m.act, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, cperm, trows, K / 2, 128, brows, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&m.actn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, cnat, trows, K / 2, 128, brows, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&m.sfb2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, sfb, trows, K / 16, 32, brows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
            make_map(&m.sfb1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, sfb, trows, K / 16, 16, brows, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (ok && a.delta_slot != nullptr) {
    const uint64_t rowsD = (uint64_t)a.n_slots * a.N;
    ok = make_map(&m.dcodes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, dl->codes, rowsD, K / 2, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&m.ds4, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, dl->s4, rowsD, K / 16, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!ok) return MOET_ERR_CUDA;
  FcTcArgs ab = a;
  ab.brows = (int)brows;
  ab.tiles = row_tiles;
  const int grid = sm_count();
  if (grid <= 0) return MOET_ERR_CUDA;
  auto kern = fc_tc_kernel<FC1>;
  MOET_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
  {
    ProfScope ps(FC1 ? MOET_K_FC1 : MOET_K_FC2, st);
    MOET_CUDA_TRY(pdl_launch(a.item_rows == 0, kern, dim3(grid), dim3(kWsThreads), kSmemBytes, st, ab, m));
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}

}  // namespace

namespace {
FcTcArgs common_args(const TcForwardArgs& f) {
  FcTcArgs a{};
  a.T = f.T; a.H = f.H; a.I = f.I; a.k = f.k;
  a.offsets = f.offsets; a.perm = f.perm; a.topk_w = f.topk_w;
  a.delta_slot = f.delta_slot; a.n_slots = f.n_slots; a.gate = f.gate;
  a.hdr = f.hdr; a.chunks = f.chunks;
  a.item_rows = f.item_rows;
  return a;
}

// Grid of the item-mode terms kernel: resident CTAs over all SMs.
int items_grid() {
  const int sms = sm_count();
  return (sms > 0 ? sms : 152) * 8;
}
}  // namespace

// Which rows need the natural-order terms (see NatRows).
NatRows nat_rows(const TcForwardArgs& f) {
  NatRows nr{};
  if (f.delta_slot != nullptr && f.gate != nullptr) {
    nr.topk_idx = f.topk_idx; nr.delta_slot = f.delta_slot; nr.gate = f.gate;
    nr.k = f.k; nr.n_experts = f.n_experts; nr.n_slots = f.n_slots;
  }
  return nr;
}

moet_status tc_forward_fc1(const TcForwardArgs& f, cudaStream_t st) {
  const int pairs = f.T * f.k;
  {
    ProfScope ps(MOET_K_TERMS, st);
    if (f.item_rows) {
      // FC1 input terms of the items' pairs, at item * kTcTok + slot
      MOET_CUDA_TRY(pdl_launch(false, act_terms_items_kernel<true>, dim3(items_grid()), dim3(256), 0, st, f.H, f.x, f.hdr, f.chunks, f.offsets, f.perm, f.k,
                                                                 pairs, f.tokmax, f.buf.x_cperm, f.buf.x_cnat,
                                                                 f.buf.x_sf, f.buf.x_g, nat_rows(f)));
    } else {
      // each token once, written to the bucketed rows of its k pairs so that a work item's term
      // rows are consecutive
      const dim3 grid(f.T, (f.H / 16 + kTermThreads - 1) / kTermThreads);
      MOET_CUDA_TRY(pdl_launch(true, act_terms_kernel<true>, dim3(grid), dim3(kTermThreads), 0, st, f.H, f.x, f.inv, f.k, pairs, f.tokmax, f.buf.x_cperm,
                                                            f.buf.x_cnat, f.buf.x_sf, f.buf.x_g, f.perm, nat_rows(f)));
    }
  }
  MOET_CUDA_TRY(cudaGetLastError());
  FcTcArgs a1 = common_args(f);
  a1.work = f.work;
  a1.K = f.H; a1.N = 2 * f.I;
  a1.scale_2 = f.fc1->scale_2;
  a1.gsc = f.buf.x_g;
  a1.out = f.h;
  a1.hmax = f.hmax;
  return launch_fc_tc<true>(a1, f.fc1, f.dfc1, f.buf.x_cperm, f.buf.x_cnat, f.buf.x_sf, f.act_rows, f.E, f.I / 64,
                            st);
}

moet_status tc_forward_fc2(const TcForwardArgs& f, cudaStream_t st) {
  const int pairs = f.T * f.k;
  {
    ProfScope ps(MOET_K_TERMS, st);
    if (f.item_rows) {
      MOET_CUDA_TRY(pdl_launch(false, act_terms_items_kernel<false>, dim3(items_grid()), dim3(256), 0, st, f.I, f.h, f.hdr, f.chunks, f.offsets, f.perm, f.k,
                                                                  pairs, reinterpret_cast<const float*>(f.hmax),
                                                                  f.buf.h_cperm, f.buf.h_cnat, f.buf.h_sf, f.buf.h_g,
                                                                  nat_rows(f)));
    } else {
      // one row per bucketed pair (h rows are in bucketed order)
      const dim3 grid(pairs, (f.I / 16 + kTermThreads - 1) / kTermThreads);
      MOET_CUDA_TRY(pdl_launch(true, act_terms_kernel<false>, dim3(grid), dim3(kTermThreads), 0, st, f.I, f.h, nullptr, 1, pairs,
                                                             reinterpret_cast<const float*>(f.hmax), f.buf.h_cperm,
                                                             f.buf.h_cnat, f.buf.h_sf, f.buf.h_g, f.perm, nat_rows(f)));
    }
  }
  MOET_CUDA_TRY(cudaGetLastError());
  FcTcArgs a2 = common_args(f);
  a2.work = f.work + 1;
  a2.K = f.I; a2.N = f.H;
  a2.scale_2 = f.fc2->scale_2;
  a2.gsc = f.buf.h_g;
  a2.out = f.o;
  return launch_fc_tc<false>(a2, f.fc2, f.dfc2, f.buf.h_cperm, f.buf.h_cnat, f.buf.h_sf, f.act_rows, f.E, f.H / 128,
                             st);
}

moet_status tc_forward(const TcForwardArgs& f, cudaStream_t st) {
  const moet_status s = tc_forward_fc1(f, st);
  if (s != MOET_OK) return s;
  return tc_forward_fc2(f, st);
}

}  // namespace moet

MOET_ERROR_ACCESSOR(moet_internal_error_moe_tc)
MOET_DEBUG_WAITS_SETTER(moet_internal_debug_waits_moe_tc)
