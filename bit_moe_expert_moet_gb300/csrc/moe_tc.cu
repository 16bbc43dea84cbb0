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
// handful of integer ops per 8 weights, stores it to shared memory in the
// 128-byte-swizzled K-major layout, and writes the row scales to TMEM; the
// tensor core applies the block scale.  The factor 2 of the halved levels is
// applied in the epilogue.
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
// Pipeline per CTA (256 threads; threads t and t + 128 share tile row t):
// raw chunks of 256 weights stream into a kRawRing-deep cp.async ring (planes,
// scales and activation terms, ~19 KB per chunk), refilled as soon as they
// are staged; staging expands a raw chunk into a kOpRing-deep operand ring
// (swizzled A and B tiles in shared memory, scale factors in TMEM).  Each
// iteration has one CTA barrier: thread 0 issues the 4 MMAs (K = 64) of the
// chunk staged in the previous iteration and commits them to that operand
// slot's mbarrier, while everyone stages the next chunk into the other slot
// after a bounded wait for the MMAs that last read it.
#include <cuda_bf16.h>

#include "common.cuh"
#include "moe_tc.cuh"

namespace moet {
namespace {

constexpr int kFcThreads = 256;               // FC kernel: two threads per weight row
constexpr int kRawRing = 3;                   // raw chunks in flight (cp.async)
constexpr int kOpRing = 2;                    // operand slots (A, B, scales) in use by the tensor core
constexpr int kKC = 256;                      // weights per main-pass K chunk (one SW128 atom)
constexpr int kKD = 128;                      // weights per delta-pass K chunk
constexpr int kMaxN = kTcTerms * kTcTok;      // 64 columns of D
constexpr int kTmemCols = 256;
constexpr int kColD = 0, kColD2 = 64, kColSFA = 128, kColSFB = 128 + 16 * kOpRing;
// raw slot: planes [half][row][16 B] (sign, then magnitude; the delta pass puts its
// 32 bytes per half-row in the same two arrays), row scales [row][16 B], B-term
// scales [n][16 B], B-term codes [n][128 B]
constexpr int kRawSign = 0, kRawMag = 4096, kRawQ = 8192, kRawSfb = 10240, kRawB = 11264;
constexpr int kRawBytes = 19456;
// operand slot: A (128 rows x 128 B, swizzled), B (64 rows x 128 B, swizzled)
constexpr int kOpA = 0, kOpB = 16384;
constexpr int kOpBytes = 24576;
constexpr long long kWaitLimit = 1LL << 22;   // polls before a wait is declared stuck

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte asynchronous global->shared copy; src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes = 16) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes));
}
// 8-byte form (8-byte aligned addresses); src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async8(void* dst, const void* src, uint32_t src_bytes = 8) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

// SW128 K-major shared-memory matrix descriptor: 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)2 << 61;                 // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::mxf4nvf4, A and B e2m1, K-major, ue4m3 scales, M = 128.
__device__ __forceinline__ uint32_t mxf4_idesc(int n) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

// Bounded wait for the mbarrier phase with the given parity; false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  for (long long it = 0; it < kWaitLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(a), "r"(parity));
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p; }"
      ::"r"(d), "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc));
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar)));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t v[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
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
// Grid (rows, K / 256): each CTA of 256 threads reads its row once for the
// row maximum m, then 16 threads expand one 16-element block (one element
// each) into kTcTerms NVFP4 terms.  Term t has the fp32 scale
// g_t = m / (6 * 448) / 4^t and a ue4m3 scale per block chosen from the
// block's current residual, so each term quantises what the previous ones
// left (a block's residual shrinks at least ~6x per term while g_t shrinks
// 4x, keeping the block scales in the normal e4m3 range).  Outputs per
// (row, term): codes in permuted and natural K order, one ue4m3 scale per
// 16 elements, and g_t.
constexpr int kTermThreads = 256;

template <bool BF16_IN>
__global__ void __launch_bounds__(kTermThreads) act_terms_kernel(int K, const void* __restrict__ src,
                                                                uint8_t* __restrict__ cperm, uint8_t* __restrict__ cnat,
                                                                uint8_t* __restrict__ sfb, float* __restrict__ gsc) {
  __shared__ float red[kTermThreads / 32];
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const uint16_t* sb = static_cast<const uint16_t*>(src) + (size_t)row * K;
  const float* sf32 = static_cast<const float*>(src) + (size_t)row * K;
  float m = 0.0f;
  if (BF16_IN) {
    const uint4* p = reinterpret_cast<const uint4*>(sb);
    for (int i = tid; i < K / 8; i += kTermThreads) {
      const uint4 v = __ldg(p + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[q] << 16)), fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(sf32);
    for (int i = tid; i < K / 4; i += kTermThreads) {
      const float4 v = p[i];
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[tid >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < kTermThreads / 32; ++w) m = fmaxf(m, red[w]);
  const float g0 = m / (6.0f * 448.0f);
  if (blockIdx.y == 0 && tid < kTcTerms) gsc[(size_t)row * kTcTerms + tid] = ldexpf(g0, -2 * tid);
  const int idx = blockIdx.y * kTermThreads + tid;         // element index in the row
  const int b = idx >> 4, j = idx & 15, lbase = lane & 16;
  const bool live = idx < K;                                // K % 256 == 0: all live
  float r = 0.0f;
  if (live) r = BF16_IN ? __uint_as_float((uint32_t)__ldg(sb + idx) << 16) : sf32[idx];
  // the element whose code lands at permuted position p = 4 r + n is r + 4 n
  const int p0 = 2 * (j & 7), p1 = p0 + 1;
  const int src0 = (p0 >> 2) + 4 * (p0 & 3);
  const int src1 = (p1 >> 2) + 4 * (p1 & 3);
#pragma unroll
  for (int t = 0; t < kTcTerms; ++t) {
    const float g = ldexpf(g0, -2 * t);
    float bm = fabsf(r);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
    uint32_t sf = 0;
    float sc = 0.0f;
    if (g > 0.0f) {
      sf = f32_to_e4m3_rn(bm / (6.0f * g));
      sc = e4m3_to_f32(sf) * g;
    }
    uint32_t code = 0;
    if (sc > 0.0f) {
      const uint32_t mg = e2m1_rne_mag(fabsf(r), sc);
      const bool neg = r < 0.0f && mg != 0u;
      const float q = e2m1_mag_value(mg) * sc;
      r -= neg ? -q : q;
      code = mg | (neg ? 8u : 0u);
    }
    const uint32_t nat_hi = __shfl_down_sync(0xffffffffu, code, 1);
    const uint32_t per_lo = __shfl_sync(0xffffffffu, code, lbase + src0);
    const uint32_t per_hi = __shfl_sync(0xffffffffu, code, lbase + src1);
    if (live) {
      const size_t term_row = (size_t)row * kTcTerms + t;
      if ((j & 1) == 0) cnat[term_row * (K / 2) + 8 * b + (j >> 1)] = (uint8_t)(code | (nat_hi << 4));
      if (j < 8) cperm[term_row * (K / 2) + 8 * b + j] = (uint8_t)(per_lo | (per_hi << 4));
      if (j == 0) sfb[term_row * (K / 16) + b] = (uint8_t)sf;
    }
  }
}

// ---------------------------------------------------------------- FC kernel
struct FcTcArgs {
  int T, H, I, k, K, N;          // N = rows of one expert matrix
  const int32_t* offsets;
  const int32_t* perm;
  const float* topk_w;
  const uint32_t* sign;
  const uint32_t* mag;
  const uint8_t* s16;
  const float* scale_2;
  const int32_t* delta_slot;
  int n_slots;
  const uint8_t* dcodes;
  const uint8_t* ds4;
  const uint8_t* gate;
  const int* hdr;
  const int4* chunks;
  const uint8_t* cperm;          // activation terms (rows: FC1 tokens, FC2 bucketed pairs)
  const uint8_t* cnat;
  const uint8_t* sfb;
  const float* gsc;
  float* out;
};

struct TcSmem {
  uint64_t bar[kOpRing];
  uint32_t tmem_base;
  int stuck;
  int any_gated;
  int slot;
  int src_row[kTcTok];           // activation-term row per token of the work item
  float gate_f[kTcTok];
  float gsc[kMaxN];              // term scales, column order
  float wts[kTcTok];             // FC2: routing weight per pair
  int pair[kTcTok];              // FC2: pair id per column token
};

template <bool FC1>
__global__ void __launch_bounds__(kFcThreads, 2) fc_tc_kernel(const FcTcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_dyn[];
  // 1024-aligned operand stages, then the small shared state
  unsigned char* base = smem_dyn + ((1024 - (smem_addr(smem_dyn) & 1023)) & 1023);
  unsigned char* ops = base;                                   // [kOpRing][kOpBytes]
  unsigned char* raws = base + kOpRing * kOpBytes;             // [kRawRing][kRawBytes]
  TcSmem& sm = *reinterpret_cast<TcSmem*>(raws + kRawRing * kRawBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int trow = tid & 127, half = tid >> 7;   // tile row of this thread, and which 128 weights
  if ((int)blockIdx.y >= a.hdr[0]) return;
  const int4 ch = a.chunks[blockIdx.y];
  const int e = ch.x, ntok = ch.z;
  const int pos0 = __ldg(a.offsets + e) + ch.y;
  const int K = a.K, nkc = K / kKC;
  const int ncols = ((kTcTerms * ntok + 15) / 16) * 16;        // MMA N (multiple of 16, <= 64)

  if (tid == 0) {
    sm.stuck = 0;
    sm.any_gated = 0;
    int slot = -1;
    if (a.delta_slot != nullptr && a.gate != nullptr) {
      slot = __ldg(a.delta_slot + e);
      if (slot >= a.n_slots) { record_error(MOET_ERR_DEVICE_INDEX); slot = -1; }
    }
    sm.slot = slot;
    for (int s = 0; s < kOpRing; ++s) mbar_init(&sm.bar[s], 1);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&sm.tmem_base)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  __syncthreads();
  if (tid < kTcTok) {
    int srow = -1, pr = -1;
    float gf = 0.0f, wv = 0.0f;
    if (tid < ntok) {
      const int p = __ldg(a.perm + pos0 + tid);
      if (p < 0 || p >= a.T * a.k) {
        record_error(MOET_ERR_DEVICE_INDEX);
      } else {
        const int tok = p / a.k;
        srow = FC1 ? tok : pos0 + tid;
        pr = p;
        wv = __ldg(a.topk_w + p);
        if (sm.slot >= 0 && __ldg(a.gate + tok)) { gf = 1.0f; sm.any_gated = 1; }
      }
    }
    sm.src_row[tid] = srow;
    sm.gate_f[tid] = gf;
    sm.pair[tid] = pr;
    sm.wts[tid] = wv;
  }
  __syncthreads();
  if (tid < kMaxN) {
    const int tk = tid / kTcTerms, term = tid % kTcTerms;
    const int srow = tk < kTcTok ? sm.src_row[tk] : -1;
    sm.gsc[tid] = srow >= 0 ? __ldg(a.gsc + (size_t)srow * kTcTerms + term) : 0.0f;
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = sm.tmem_base;
  const bool do_delta = sm.slot >= 0 && sm.any_gated;
  const uint32_t idesc = mxf4_idesc(ncols);

  // the weight row owned by this thread
  int wrow;
  if (FC1) {
    wrow = trow < 64 ? blockIdx.x * 64 + trow : a.I + blockIdx.x * 64 + (trow - 64);
  } else {
    wrow = blockIdx.x * 128 + trow;
  }
  // weight rows whose scales this thread writes to TMEM (replicated layout: rows lane + 32 j)
  int srows[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tr = lane + 32 * j;
    srows[j] = FC1 ? (tr < 64 ? blockIdx.x * 64 + tr : a.I + blockIdx.x * 64 + (tr - 64)) : blockIdx.x * 128 + tr;
  }
  const size_t wpr = (size_t)K / 32, bpr = (size_t)K / 16;
  const uint32_t lane_q = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lane quarter

  // chunk sequence: nkc main-pass chunks of 256 weights, then (with the delta)
  // nkd delta-pass chunks of 128 weights
  const int nkd = do_delta ? K / kKD : 0;
  const int total = nkc + nkd;

  // Per-thread sources, fixed for the whole K loop.  Warps 0-3 (half 0) copy
  // the row scales and write the weight-row scale factors; warps 4-7 (half 1)
  // copy and stage the B-term tiles and write the B-term scale factors.
  const size_t wrow_base = (size_t)e * a.N + wrow;
  const uint4* sign_src = reinterpret_cast<const uint4*>(a.sign + wrow_base * wpr) + half;   // + 2 c
  const uint4* mag_src = reinterpret_cast<const uint4*>(a.mag + wrow_base * wpr) + half;
  const uint4* q_src = reinterpret_cast<const uint4*>(a.s16 + wrow_base * bpr);               // + c
  const int rawp = (half * 128 + trow) * 16;                    // this thread's raw plane offset
  int aoff[4];                                                  // swizzled A offsets of its 4 pieces
#pragma unroll
  for (int w = 0; w < 4; ++w) aoff[w] = kOpA + trow * 128 + (((4 * half + w) ^ (trow & 7)) << 4);
  const int bt = tid - 128;                                     // B-side thread index (half 1)
  // main-pass B items of this thread: it = bt + 128 m, row n = it / 8, piece u = it % 8
  const uint8_t* bsrc[4];
  int bdst[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int it = bt + 128 * m;
    const int n = it >> 3, u = it & 7;
    bsrc[m] = nullptr;
    bdst[m] = -1;
    if (half == 1 && n < ncols) {
      const int tk = n / kTcTerms, term = n % kTcTerms;
      const int srow = tk < ntok ? sm.src_row[tk] : -1;
      bdst[m] = n * 128 + 16 * u;
      if (srow >= 0) bsrc[m] = a.cperm + ((size_t)srow * kTcTerms + term) * (K / 2) + 16 * u;
    }
  }
  const uint8_t* sfb_src = nullptr;                             // B-term scale row (bt < ncols)
  if (half == 1 && bt < ncols) {
    const int tk = bt / kTcTerms, term = bt % kTcTerms;
    const int srow = tk < ntok ? sm.src_row[tk] : -1;
    if (srow >= 0) sfb_src = a.sfb + ((size_t)srow * kTcTerms + term) * bpr;
  }

  // Asynchronous copies of chunk cg into raw slot cg % kRawRing.  One commit
  // group per chunk (possibly empty) keeps the group count uniform.
  auto prefetch = [&](int cg) {
    if (cg < total) {
      const bool dp = cg >= nkc;
      const int c = dp ? cg - nkc : cg;
      unsigned char* raw = raws + (cg % kRawRing) * kRawBytes;
      if (!dp) {
        cp_async16(raw + kRawSign + rawp, sign_src + 2 * c);
        cp_async16(raw + kRawMag + rawp, mag_src + 2 * c);
        if (half == 0) cp_async16(raw + kRawQ + trow * 16, q_src + c);
        else {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            if (bdst[m] >= 0)
              cp_async16(raw + kRawB + bdst[m], bsrc[m] ? bsrc[m] + (size_t)c * 128 : a.cperm, bsrc[m] ? 16u : 0u);
          }
          if (bt < ncols) cp_async16(raw + kRawSfb + bt * 16, sfb_src ? sfb_src + (size_t)c * 16 : a.sfb, sfb_src ? 16u : 0u);
        }
      } else {
        const uint8_t* dsrc = a.dcodes + ((size_t)sm.slot * a.N + wrow) * (K / 2) + (size_t)c * 64 + 32 * half;
        cp_async16(raw + kRawSign + rawp, dsrc);
        cp_async16(raw + kRawMag + rawp, dsrc + 16);
        if (half == 0) {
          cp_async8(raw + kRawQ + trow * 16, a.ds4 + ((size_t)sm.slot * a.N + wrow) * bpr + (size_t)c * 8);
        } else {
          for (int it = bt; it < ncols * 4; it += 128) {              // 64 bytes per B row
            const int n = it >> 2, u = it & 3;
            const int tk = n / kTcTerms, term = n % kTcTerms;
            const int srow = tk < ntok ? sm.src_row[tk] : -1;
            const bool ok = srow >= 0 && sm.gate_f[tk] != 0.0f;
            const uint8_t* src = ok ? a.cnat + ((size_t)srow * kTcTerms + term) * (K / 2) + (size_t)c * 64 + 16 * u : a.cnat;
            cp_async16(raw + kRawB + n * 128 + 16 * u, src, ok ? 16u : 0u);
          }
          if (bt < ncols)
            cp_async8(raw + kRawSfb + bt * 16, sfb_src ? sfb_src + (size_t)c * 8 : a.sfb, sfb_src ? 8u : 0u);
        }
      }
    }
    cp_async_commit();
  };

  // Turn raw chunk cg into the operands of operand slot cg % kOpRing: expand (or
  // copy) A into the swizzled tile, copy B into its swizzled tile, write the
  // scale factors to TMEM.  The caller has made the slot free.
  auto stage = [&](int cg) {
    const bool dp = cg >= nkc;
    const int oi = cg % kOpRing;
    const unsigned char* raw = raws + (cg % kRawRing) * kRawBytes;
    unsigned char* op = ops + oi * kOpBytes;
    const uint4 sw = *reinterpret_cast<const uint4*>(raw + kRawSign + rawp);
    const uint4 mw = *reinterpret_cast<const uint4*>(raw + kRawMag + rawp);
    if (!dp) {
      const uint32_t SW[4] = {sw.x, sw.y, sw.z, sw.w};
      const uint32_t MW[4] = {mw.x, mw.y, mw.z, mw.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) *reinterpret_cast<uint4*>(op + aoff[w]) = planes_to_e2m1(SW[w], MW[w]);
    } else {
      unsigned char* arow = op + kOpA + trow * 128;
      *reinterpret_cast<uint4*>(arow + (((2 * half) ^ (trow & 7)) << 4)) = sw;
      *reinterpret_cast<uint4*>(arow + (((2 * half + 1) ^ (trow & 7)) << 4)) = mw;
    }
    if (half == 1) {
      const int upr = dp ? 4 : 8;                        // 16-byte pieces per B row
      for (int it = bt; it < ncols * upr; it += 128) {
        const int n = it / upr, u = it % upr;
        *reinterpret_cast<uint4*>(op + kOpB + n * 128 + ((u ^ (n & 7)) << 4)) =
            *reinterpret_cast<const uint4*>(raw + kRawB + n * 128 + 16 * u);
      }
    }
    // scale factors, replicated TMEM layout (rows lane + 32 j -> columns 4 i + j);
    // warps 0-3 write the weight-row scales, warps 4-7 the B-term scales
    uint32_t v[16];
    const int src = half ? kRawSfb : kRawQ;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = lane + 32 * j;
      uint4 q = make_uint4(0u, 0u, 0u, 0u);
      if (!half || n < ncols) q = *reinterpret_cast<const uint4*>(raw + src + n * 16);
      if (dp) { q.z = 0u; q.w = 0u; }                  // 128-weight chunk: two MMAs' worth
      v[0 * 4 + j] = q.x; v[1 * 4 + j] = q.y; v[2 * 4 + j] = q.z; v[3 * 4 + j] = q.w;
    }
    tmem_st16(tmem + lane_q + (half ? kColSFB : kColSFA) + 16 * oi, v);
    asm volatile("fence.proxy.async.shared::cta;");
    asm volatile("tcgen05.wait::st.sync.aligned;");
    asm volatile("tcgen05.fence::before_thread_sync;");
  };

#pragma unroll 1
  for (int cg = 0; cg < kRawRing; ++cg) prefetch(cg);
  cp_async_wait<kRawRing - 1>();
  __syncthreads();
  stage(0);

  int cg = 0;
#pragma unroll 1
  for (; cg < total; ++cg) {
    cp_async_wait<kRawRing - 2>();               // this thread's copies of chunk cg + 1 landed
    __syncthreads();                             // operands of cg staged; raw cg + 1 visible
    if (sm.stuck) break;
    const bool dp = cg >= nkc;
    const int oi = cg % kOpRing;
    if (tid == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;");
      const uint32_t a0 = smem_addr(ops + oi * kOpBytes + kOpA), b0 = smem_addr(ops + oi * kOpBytes + kOpB);
      const uint32_t dcol = dp ? kColD2 : kColD;
      const int nmma = dp ? kKD / 64 : kKC / 64;
      const int c = dp ? cg - nkc : cg;
      for (int i = 0; i < nmma; ++i) {
        tc_mma(tmem + dcol, sw128_desc(a0 + 32 * i), sw128_desc(b0 + 32 * i), idesc,
               tmem + kColSFA + 16 * oi + 4 * i, tmem + kColSFB + 16 * oi + 4 * i, (c > 0 || i > 0) ? 1u : 0u);
      }
      tc_commit(&sm.bar[oi]);
    }
    if (cg + 1 < total) {
      // the next operand slot was last read by the MMAs of chunk cg + 1 - kOpRing
      if (cg + 1 >= kOpRing) {
        const int prev = cg + 1 - kOpRing;
        if (!mbar_wait(&sm.bar[prev % kOpRing], (prev / kOpRing) & 1)) atomicExch(&sm.stuck, 1);
      }
      stage(cg + 1);
    }
    prefetch(cg + kRawRing);                     // raw slot of chunk cg is free since the barrier
  }
  cp_async_wait<0>();
  // ---- drain: the last use of every operand slot (bounded), then read the accumulators
  const int issued = cg;
  for (int s2 = 0; s2 < kOpRing && s2 < issued; ++s2) {
    const int last = issued - 1 - ((issued - 1 - s2) % kOpRing);
    if (!mbar_wait(&sm.bar[s2], (last / kOpRing) & 1)) atomicExch(&sm.stuck, 1);
  }
  asm volatile("tcgen05.fence::after_thread_sync;");
  __syncthreads();
  if (sm.stuck) {
    if (tid == 0) record_error(MOET_ERR_TIMEOUT);
  } else if (half == 0) {
    // FC1: up rows hand their values to the gate rows through the (now idle) ring memory
    float (*xchg)[kTcTok] = reinterpret_cast<float (*)[kTcTok]>(base);
    const float sc2 = 2.0f * __ldg(a.scale_2 + e);           // 2: the halved e2m1 levels
    const float sc2d = __ldg(a.scale_2 + e);
    for (int c0 = 0; c0 < ncols; c0 += 16) {
      float v[16], v2[16];
      tmem_ld16(tmem + lane_q + kColD + c0, v);
      if (do_delta) tmem_ld16(tmem + lane_q + kColD2 + c0, v2);
      float acc[16 / kTcTerms];
#pragma unroll
      for (int q = 0; q < 16 / kTcTerms; ++q) {
        float sacc = 0.0f;
#pragma unroll
        for (int t = 0; t < kTcTerms; ++t) {
          const int col = q * kTcTerms + t;
          float d = sc2 * v[col];
          if (do_delta) d = fmaf(sc2d, v2[col], d);
          sacc = fmaf(sm.gsc[c0 + col], d, sacc);
        }
        acc[q] = sacc;
      }
      if (!FC1) {
#pragma unroll
        for (int q = 0; q < 16 / kTcTerms; ++q) {
          const int tk = c0 / kTcTerms + q;
          if (tk < ntok && sm.src_row[tk] >= 0) a.out[(size_t)sm.pair[tk] * a.H + wrow] = acc[q] * sm.wts[tk];
        }
      } else {
        // up rows (threads 64..127) hand their values to the gate rows (threads 0..63)
        if (tid >= 64) {
#pragma unroll
          for (int q = 0; q < 16 / kTcTerms; ++q) xchg[tid - 64][c0 / kTcTerms + q] = acc[q];
        }
        asm volatile("bar.sync 1, 128;");        // warps 0-3 only
        if (tid < 64) {
#pragma unroll
          for (int q = 0; q < 16 / kTcTerms; ++q) {
            const int tk = c0 / kTcTerms + q;
            if (tk < ntok && sm.src_row[tk] >= 0) {
              const float gv = acc[q], uv = xchg[tid][tk];
              a.out[(size_t)(pos0 + tk) * a.I + wrow] = gv / (1.0f + expf(-gv)) * uv;
            }
          }
        }
        asm volatile("bar.sync 1, 128;");
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

template <bool FC1>
moet_status launch_fc_tc(const FcTcArgs& a, int row_tiles, int grid_y, cudaStream_t st) {
  const size_t smem = 1024 + kOpRing * kOpBytes + kRawRing * kRawBytes + sizeof(TcSmem);
  auto kern = fc_tc_kernel<FC1>;
  MOET_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  {
    ProfScope ps(FC1 ? MOET_K_FC1 : MOET_K_FC2, st);
    kern<<<dim3(row_tiles, grid_y), kFcThreads, smem, st>>>(a);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}

}  // namespace

moet_status tc_forward(const TcForwardArgs& f, cudaStream_t st) {
  const int pairs = f.T * f.k;
  // FC1 input terms: one row per token
  {
    ProfScope ps(MOET_K_TERMS, st);
    const dim3 grid(f.T, (f.H + kTermThreads - 1) / kTermThreads);
    act_terms_kernel<true><<<grid, kTermThreads, 0, st>>>(f.H, f.x, f.buf.x_cperm, f.buf.x_cnat, f.buf.x_sf,
                                                      f.buf.x_g);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  FcTcArgs a{};
  a.T = f.T; a.H = f.H; a.I = f.I; a.k = f.k;
  a.offsets = f.offsets; a.perm = f.perm; a.topk_w = f.topk_w;
  a.delta_slot = f.delta_slot; a.n_slots = f.n_slots; a.gate = f.gate;
  a.hdr = f.hdr; a.chunks = f.chunks;
  FcTcArgs a1 = a;
  a1.K = f.H; a1.N = 2 * f.I;
  a1.sign = f.fc1->sign; a1.mag = f.fc1->mag; a1.s16 = f.fc1->s16; a1.scale_2 = f.fc1->scale_2;
  if (f.delta_slot) { a1.dcodes = f.dfc1->codes; a1.ds4 = f.dfc1->s4; }
  a1.cperm = f.buf.x_cperm; a1.cnat = f.buf.x_cnat; a1.sfb = f.buf.x_sf; a1.gsc = f.buf.x_g;
  a1.out = f.h;
  moet_status s = launch_fc_tc<true>(a1, f.I / 64, f.max_items, st);
  if (s != MOET_OK) return s;
  // FC2 input terms: one row per bucketed pair (h rows are in bucketed order)
  {
    ProfScope ps(MOET_K_TERMS, st);
    const dim3 grid(pairs, (f.I + kTermThreads - 1) / kTermThreads);
    act_terms_kernel<false><<<grid, kTermThreads, 0, st>>>(f.I, f.h, f.buf.h_cperm, f.buf.h_cnat, f.buf.h_sf,
                                                       f.buf.h_g);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  FcTcArgs a2 = a;
  a2.K = f.I; a2.N = f.H;
  a2.sign = f.fc2->sign; a2.mag = f.fc2->mag; a2.s16 = f.fc2->s16; a2.scale_2 = f.fc2->scale_2;
  if (f.delta_slot) { a2.dcodes = f.dfc2->codes; a2.ds4 = f.dfc2->s4; }
  a2.cperm = f.buf.h_cperm; a2.cnat = f.buf.h_cnat; a2.sfb = f.buf.h_sf; a2.gsc = f.buf.h_g;
  a2.out = f.o;
  return launch_fc_tc<false>(a2, f.H / 128, f.max_items, st);
}

}  // namespace moet

MOET_ERROR_ACCESSOR(moet_internal_error_moe_tc)
