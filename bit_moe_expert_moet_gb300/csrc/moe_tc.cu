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
// Pipeline per CTA (10 warps, warp-specialised, no CTA-wide barrier in the K
// loop): warp 0 (one thread) streams each 256-weight K chunk into one of
// kSlots shared-memory slots with TMA (sign and magnitude planes, row scales,
// the work item's 64 activation-term rows and their scales); warps 2-9 (two
// threads per weight row; rows = TMEM lanes) expand the planes into the
// swizzled A tile and write the scale factors to TMEM; warp 1 (one thread)
// issues the 4 MMAs (K = 64) per chunk and commits them to the slot's
// "empty" mbarrier.  Hand-offs: full (TMA bytes landed) -> staged (256
// converter arrivals) -> empty (MMA commit); every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>

#include "common.cuh"
#include "moe_tc.cuh"

namespace moet {
namespace {

constexpr int kWsThreads = 320;              // warp 0: TMA producer, warp 1: MMA, warps 2-9: converters
constexpr int kConvThreads = 256;             // two converter threads per weight row
constexpr int kSlots = 3;                     // K chunks in flight
constexpr int kKC = 256;                      // weights per K chunk (one SW128 atom)
constexpr int kMaxN = kTcTerms * kTcTok;      // 64 columns of D
constexpr int kTmemCols = 256;
constexpr int kColD = 0, kColD2 = 64, kColSFA = 128, kColSFB = 128 + 16 * kSlots;
// slot layout (1024-aligned): A operand (128 rows x 128 B, SW128), B operand (64 rows x 128 B,
// SW128), raw sign and magnitude planes [128 rows][32 B], raw row scales [128][16 B], raw B-term
// scales [64 rows][16 B]
constexpr int kSA = 0, kSB = 16384, kSSign = 24576, kSMag = 28672, kSQ = 32768, kSF = 34816;
constexpr int kSlotBytes = 36864;
constexpr long long kWaitLimit = 1LL << 22;   // polls before a wait is declared stuck

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

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
// Grid (rows, K / 256), 256 threads: 16 threads expand one 16-element block
// (one element each) into kTcTerms NVFP4 terms.  Term t has the fp32 scale
// g_t = m / (6 * 448) / 4^t, m = the row maximum (given: per token for FC1,
// per pair from FC1's epilogue for FC2), and a ue4m3 scale per block chosen
// from the block's current residual, so each term quantises what the previous
// ones left (a block's residual shrinks at least ~6x per term while g_t
// shrinks 4x, keeping the block scales in the normal e4m3 range).  Outputs
// per (row, term): codes in permuted and natural K order, one ue4m3 scale per
// 16 elements, and g_t.
constexpr int kTermThreads = 256;

template <bool BF16_IN>
__global__ void __launch_bounds__(kTermThreads) act_terms_kernel(int K, const void* __restrict__ src,
                                                                const int32_t* __restrict__ row_map, int map_div,
                                                                const float* __restrict__ rowmax,
                                                                uint8_t* __restrict__ cperm, uint8_t* __restrict__ cnat,
                                                                uint8_t* __restrict__ sfb, float* __restrict__ gsc) {
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  // output row `row` expands source row row_map[row] / map_div (or `row` itself)
  const size_t srow = row_map ? (size_t)(__ldg(row_map + row) / map_div) : (size_t)row;
  const float m = __ldg(rowmax + srow);
  const float g0 = m / (6.0f * 448.0f);
  if (blockIdx.y == 0 && tid < kTcTerms) gsc[(size_t)row * kTcTerms + tid] = ldexpf(g0, -2 * tid);
  const int idx = blockIdx.y * kTermThreads + tid;          // element of the row (K % 256 == 0)
  const int b = idx >> 4, j = idx & 15, lbase = lane & 16;
  float r = BF16_IN ? __uint_as_float((uint32_t)__ldg(static_cast<const uint16_t*>(src) + srow * K + idx) << 16)
                    : static_cast<const float*>(src)[srow * K + idx];
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
    const size_t term_row = (size_t)row * kTcTerms + t;
    if ((j & 1) == 0) cnat[term_row * (K / 2) + 8 * b + (j >> 1)] = (uint8_t)(code | (nat_hi << 4));
    if (j < 8) cperm[term_row * (K / 2) + 8 * b + j] = (uint8_t)(per_lo | (per_hi << 4));
    if (j == 0) sfb[term_row * (K / 16) + b] = (uint8_t)sf;
  }
}

// ---------------------------------------------------------------- FC kernel
struct TmaMaps {
  CUtensorMap sign, mag, q;        // planes u32 [E N, K/32] box {8, 64} SW32; s16 u8 [E N, K/16] box {16, 64}
  CUtensorMap act, actn, sfb;      // terms u8 [pairs 4, K/2] box {128, 16} SW128 (perm / natural); scales box {16, 16}
  CUtensorMap dcodes, ds4;         // delta u8 [S N, K/2] box {128, 64} SW128; scales box {16, 64}
};

struct FcTcArgs {
  int T, H, I, k, K, N;          // N = rows of one expert matrix
  int brows;                     // rows of one activation-term box: min(16, 4 * term rows)
  const int32_t* offsets;
  const int32_t* perm;
  const float* topk_w;
  const float* scale_2;
  const int32_t* delta_slot;
  int n_slots;
  const uint8_t* gate;
  const int* hdr;
  const int4* chunks;
  const float* gsc;
  float* out;
  unsigned* hmax;                // FC1: max |h| per bucketed pair (fp32 bits), for the FC2 terms
};

struct TcSmem {
  uint64_t full[kSlots];         // TMA bytes landed
  uint64_t staged[kSlots];       // converters done (A expanded, scales in TMEM)
  uint64_t empty[kSlots];        // MMAs of the slot done
  uint32_t tmem_base;
  int stuck;
  int issued;                    // MMA chunks issued
  int any_gated;
  int slot;
  int src_row[kTcTok];           // activation-term row per token of the work item
  float gate_f[kTcTok];
  float gsc[kMaxN];              // term scales, column order
  float wts[kTcTok];             // FC2: routing weight per pair
  int pair[kTcTok];              // FC2: pair id per column token
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool is_stuck(const TcSmem& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.stuck) != 0;
}

// Warp-specialised FC over one 128-row weight tile of one expert and one work
// item of <= kTcTok routed pairs.  Main pass: K chunks of 256 weights from the
// 2-bit planes; delta pass (cached expert with gated pairs): the same chunks
// of the NVFP4 delta into a second accumulator.
template <bool FC1>
__global__ void __launch_bounds__(kWsThreads, 2) fc_tc_kernel(const FcTcArgs a, const __grid_constant__ TmaMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem_dyn[];
  unsigned char* base = smem_dyn + ((1024 - (smem_addr(smem_dyn) & 1023)) & 1023);
  TcSmem& sm = *reinterpret_cast<TcSmem*>(base + kSlots * kSlotBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((int)blockIdx.y >= a.hdr[0]) return;
  const int4 ch = a.chunks[blockIdx.y];
  const int e = ch.x, ntok = ch.z;
  const int pos0 = __ldg(a.offsets + e) + ch.y;
  const int K = a.K, nkc = K / kKC;
  const int ncols = ((kTcTerms * ntok + 15) / 16) * 16;        // MMA N (multiple of 16, <= 64)

  if (tid == 0) {
    sm.stuck = 0;
    sm.issued = 0;
    sm.any_gated = 0;
    int slot = -1;
    if (a.delta_slot != nullptr && a.gate != nullptr) {
      slot = __ldg(a.delta_slot + e);
      if (slot >= a.n_slots) { record_error(MOET_ERR_DEVICE_INDEX); slot = -1; }
    }
    sm.slot = slot;
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.staged[s], kConvThreads);
      mbar_init(&sm.empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  if (warp == 1) {
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
    sm.gsc[tid] = tk < ntok && sm.src_row[tk] >= 0 ? __ldg(a.gsc + (size_t)(pos0 + tk) * kTcTerms + term) : 0.0f;
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = sm.tmem_base;
  const bool do_delta = sm.slot >= 0 && sm.any_gated;
  const int total = do_delta ? 2 * nkc : nkc;
  // the two 64-row halves of the tile in the expert's matrix (FC1: gate rows, then up rows)
  const int r0 = FC1 ? blockIdx.x * 64 : blockIdx.x * 128;
  const int r1 = FC1 ? a.I + blockIdx.x * 64 : blockIdx.x * 128 + 64;

  if (warp == 0) {
    // ---------------- producer: one thread issues every TMA copy
    if (lane == 0) {
      for (int cg = 0; cg < total; ++cg) {
        const int s = cg % kSlots, u = cg / kSlots;
        if (u > 0 && !mbar_wait(&sm.empty[s], (u - 1) & 1)) { atomicExch(&sm.stuck, 1); break; }
        if (is_stuck(sm)) break;
        const bool dp = cg >= nkc;
        const int c = dp ? cg - nkc : cg;
        unsigned char* sl = base + s * kSlotBytes;
        const int nbox = (ncols + 15) / 16;         // 16-row boxes of activation terms
        const uint32_t bytes = (dp ? 16384u + 2048u : 4096u + 4096u + 2048u) + (uint32_t)(nbox * a.brows) * (128u + 16u);
        mbar_expect_tx(&sm.full[s], bytes);
        if (!dp) {
          const int y0 = e * a.N + r0, y1 = e * a.N + r1;
          tma_load_2d(smem_addr(sl + kSSign), &maps.sign, c * 8, y0, &sm.full[s]);
          tma_load_2d(smem_addr(sl + kSSign + 2048), &maps.sign, c * 8, y1, &sm.full[s]);
          tma_load_2d(smem_addr(sl + kSMag), &maps.mag, c * 8, y0, &sm.full[s]);
          tma_load_2d(smem_addr(sl + kSMag + 2048), &maps.mag, c * 8, y1, &sm.full[s]);
          tma_load_2d(smem_addr(sl + kSQ), &maps.q, c * 16, y0, &sm.full[s]);
          tma_load_2d(smem_addr(sl + kSQ + 1024), &maps.q, c * 16, y1, &sm.full[s]);
        } else {
          const int y0 = sm.slot * a.N + r0, y1 = sm.slot * a.N + r1;
          tma_load_2d(smem_addr(sl + kSA), &maps.dcodes, c * 128, y0, &sm.full[s]);
          tma_load_2d(smem_addr(sl + kSA + 8192), &maps.dcodes, c * 128, y1, &sm.full[s]);
          tma_load_2d(smem_addr(sl + kSQ), &maps.ds4, c * 16, y0, &sm.full[s]);
          tma_load_2d(smem_addr(sl + kSQ + 1024), &maps.ds4, c * 16, y1, &sm.full[s]);
        }
        // the work item's pairs are consecutive bucketed rows: ncols / 16 boxes of 16 term rows
        for (int bx = 0; bx < nbox; ++bx) {
          tma_load_2d(smem_addr(sl + kSB + bx * 2048), dp ? &maps.actn : &maps.act, c * 128, pos0 * kTcTerms + 16 * bx,
                      &sm.full[s]);
          tma_load_2d(smem_addr(sl + kSF + bx * 256), &maps.sfb, c * 16, pos0 * kTcTerms + 16 * bx, &sm.full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issue: one thread
    if (lane == 0) {
      const uint32_t idesc = mxf4_idesc(ncols);
      int cg = 0;
      for (; cg < total; ++cg) {
        const int s = cg % kSlots, u = cg / kSlots;
        if (!mbar_wait(&sm.staged[s], u & 1)) { atomicExch(&sm.stuck, 1); break; }
        if (is_stuck(sm)) break;
        asm volatile("tcgen05.fence::after_thread_sync;");
        const bool dp = cg >= nkc;
        const int c = dp ? cg - nkc : cg;
        unsigned char* sl = base + s * kSlotBytes;
        const uint32_t a0 = smem_addr(sl + kSA), b0 = smem_addr(sl + kSB);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tc_mma(tmem + (dp ? kColD2 : kColD), sw128_desc(a0 + 32 * i), sw128_desc(b0 + 32 * i), idesc,
                 tmem + kColSFA + 16 * s + 4 * i, tmem + kColSFB + 16 * s + 4 * i, (c > 0 || i > 0) ? 1u : 0u);
        }
        tc_commit(&sm.empty[s]);
      }
      sm.issued = cg;
    }
  } else {
    // ---------------- converters: two threads per tile row (= TMEM lane); half h
    // expands weight words 4h..4h+3 of the chunk; half 0 writes the row scales to
    // TMEM, half 1 the activation-term scales
    const int half = (warp - 2) >> 2;
    const int trow = 32 * (warp & 3) + lane;
    const uint32_t lane_q = (uint32_t)((warp & 3) * 32) << 16;
    // 32-byte-swizzled raw plane rows: 16-byte piece h of row r sits at piece h ^ ((r >> 2) & 1)
    const int praw = trow * 32 + ((half ^ ((trow >> 2) & 1)) << 4);
    int aoff[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) aoff[w] = kSA + trow * 128 + (((4 * half + w) ^ (trow & 7)) << 4);
    for (int cg = 0; cg < total; ++cg) {
      const int s = cg % kSlots, u = cg / kSlots;
      if (!mbar_wait(&sm.full[s], u & 1)) { atomicExch(&sm.stuck, 1); break; }
      if (is_stuck(sm)) break;
      const bool dp = cg >= nkc;
      unsigned char* sl = base + s * kSlotBytes;
      if (!dp) {
        const uint4 sw = *reinterpret_cast<const uint4*>(sl + kSSign + praw);
        const uint4 mw = *reinterpret_cast<const uint4*>(sl + kSMag + praw);
        *reinterpret_cast<uint4*>(sl + aoff[0]) = planes_to_e2m1(sw.x, mw.x);
        *reinterpret_cast<uint4*>(sl + aoff[1]) = planes_to_e2m1(sw.y, mw.y);
        *reinterpret_cast<uint4*>(sl + aoff[2]) = planes_to_e2m1(sw.z, mw.z);
        *reinterpret_cast<uint4*>(sl + aoff[3]) = planes_to_e2m1(sw.w, mw.w);
      }
      // scale factors to TMEM, replicated layout: rows lane + 32 j -> columns 4 i + j
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = lane + 32 * j;
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        if (half == 0) q = *reinterpret_cast<const uint4*>(sl + kSQ + n * 16);
        else if (n < ncols) q = *reinterpret_cast<const uint4*>(sl + kSF + n * 16);
        v[0 * 4 + j] = q.x; v[1 * 4 + j] = q.y; v[2 * 4 + j] = q.z; v[3 * 4 + j] = q.w;
      }
      tmem_st16(tmem + lane_q + (half ? kColSFB : kColSFA) + 16 * s, v);
      asm volatile("fence.proxy.async.shared::cta;");
      asm volatile("tcgen05.wait::st.sync.aligned;");
      asm volatile("tcgen05.fence::before_thread_sync;");
      mbar_arrive(&sm.staged[s]);
    }
    // ---------------- epilogue (warps 2-5): wait for the last MMA chunk, read the accumulators
    if (half == 0) {
    if (!is_stuck(sm) && total > 0) {
      const int last = total - 1;
      if (!mbar_wait(&sm.empty[last % kSlots], (last / kSlots) & 1)) atomicExch(&sm.stuck, 1);
    }
    asm volatile("tcgen05.fence::after_thread_sync;");
    asm volatile("bar.sync 1, 128;");
    if (!is_stuck(sm)) {
      // FC1: up rows hand their values to the gate rows through slot 0's raw B-scale area
      float (*xchg)[kTcTok] = reinterpret_cast<float (*)[kTcTok]>(base + kSSign);
      const float sc2 = 2.0f * __ldg(a.scale_2 + e);         // 2: the halved e2m1 levels
      const float sc2d = __ldg(a.scale_2 + e);
      const int wrow = trow < 64 ? r0 + trow : r1 + trow - 64;
      for (int c0 = 0; c0 < ncols; c0 += 16) {
        float v[16], v2[16];
        tmem_ld16(tmem + lane_q + kColD + c0, v);
        if (do_delta) tmem_ld16(tmem + lane_q + kColD2 + c0, v2);
        float acc[16 / kTcTerms];
#pragma unroll
        for (int q = 0; q < 16 / kTcTerms; ++q) {
          const int tk = c0 / kTcTerms + q;
          // delta columns count only for gated pairs (the B box also holds other pairs' rows)
          const bool gated = do_delta && tk < kTcTok && sm.gate_f[tk] != 0.0f;
          float sacc = 0.0f;
#pragma unroll
          for (int t = 0; t < kTcTerms; ++t) {
            const int col = q * kTcTerms + t;
            float d = sc2 * v[col];
            if (gated) d = fmaf(sc2d, v2[col], d);
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
          if (trow >= 64) {
#pragma unroll
            for (int q = 0; q < 16 / kTcTerms; ++q) xchg[trow - 64][c0 / kTcTerms + q] = acc[q];
          }
          asm volatile("bar.sync 1, 128;");
          if (trow < 64) {
#pragma unroll
            for (int q = 0; q < 16 / kTcTerms; ++q) {
              const int tk = c0 / kTcTerms + q;
              float hv = 0.0f;
              if (tk < ntok && sm.src_row[tk] >= 0) {
                const float gv = acc[q], uv = xchg[trow][tk];
                hv = gv / (1.0f + expf(-gv)) * uv;
                a.out[(size_t)(pos0 + tk) * a.I + wrow] = hv;
              }
              float mx = fabsf(hv);
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
              if (lane == 0 && tk < ntok && sm.src_row[tk] >= 0) atomicMax(a.hmax + pos0 + tk, __float_as_uint(mx));
            }
          }
          asm volatile("bar.sync 1, 128;");
        }
      }
    }
    }
  }
  __syncthreads();
  if (warp == 1) {
    // every MMA this CTA issued must be complete before TMEM is released
    const int issued = sm.issued;
    if (lane == 0 && is_stuck(sm) && issued > 0) {
      const int last = issued - 1;
      mbar_wait(&sm.empty[last % kSlots], (last / kSlots) & 1);
    }
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
  if (tid == 0 && is_stuck(sm)) record_error(MOET_ERR_TIMEOUT);
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D row-major tensor of `rows` x `cols` elements; box = box_cols x box_rows.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* ptr, uint64_t rows, uint64_t cols,
              uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || ptr == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FC1>
moet_status launch_fc_tc(const FcTcArgs& a, const moet_planes* pl, const moet_nvfp4* dl, const uint8_t* cperm,
                         const uint8_t* cnat, const uint8_t* sfb, int act_rows, int E, int row_tiles, int grid_y,
                         cudaStream_t st) {
  TmaMaps m;
  std::memset(&m, 0, sizeof(m));
  const uint32_t brows = (uint32_t)(act_rows * kTcTerms < 16 ? act_rows * kTcTerms : 16);
  const uint64_t rowsW = (uint64_t)E * a.N, K = (uint64_t)a.K;
  bool ok = make_map(&m.sign, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, pl->sign, rowsW, K / 32, 8, 64, CU_TENSOR_MAP_SWIZZLE_32B) &&
            make_map(&m.mag, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, pl->mag, rowsW, K / 32, 8, 64, CU_TENSOR_MAP_SWIZZLE_32B) &&
            make_map(&m.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pl->s16, rowsW, K / 16, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE) &&
            make_map(&m.act, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, cperm, (uint64_t)act_rows * kTcTerms, K / 2, 128,
                     brows, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&m.actn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, cnat, (uint64_t)act_rows * kTcTerms, K / 2, 128,
                     brows, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&m.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, sfb, (uint64_t)act_rows * kTcTerms, K / 16, 16,
                     brows, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (ok && a.delta_slot != nullptr) {
    const uint64_t rowsD = (uint64_t)a.n_slots * a.N;
    ok = make_map(&m.dcodes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, dl->codes, rowsD, K / 2, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&m.ds4, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, dl->s4, rowsD, K / 16, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!ok) return MOET_ERR_CUDA;
  FcTcArgs ab = a;
  ab.brows = (int)brows;
  const size_t smem = 1024 + kSlots * kSlotBytes + sizeof(TcSmem);
  auto kern = fc_tc_kernel<FC1>;
  MOET_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  {
    ProfScope ps(FC1 ? MOET_K_FC1 : MOET_K_FC2, st);
    kern<<<dim3(row_tiles, grid_y), kWsThreads, smem, st>>>(ab, m);
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
    // one row per bucketed pair (the pair's token), so a work item's rows are consecutive
    const dim3 grid(pairs, f.H / kTermThreads);
    act_terms_kernel<true><<<grid, kTermThreads, 0, st>>>(f.H, f.x, f.perm, f.k, f.tokmax, f.buf.x_cperm,
                                                          f.buf.x_cnat, f.buf.x_sf, f.buf.x_g);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  FcTcArgs a{};
  a.T = f.T; a.H = f.H; a.I = f.I; a.k = f.k;
  a.offsets = f.offsets; a.perm = f.perm; a.topk_w = f.topk_w;
  a.delta_slot = f.delta_slot; a.n_slots = f.n_slots; a.gate = f.gate;
  a.hdr = f.hdr; a.chunks = f.chunks;
  FcTcArgs a1 = a;
  a1.K = f.H; a1.N = 2 * f.I;
  a1.scale_2 = f.fc1->scale_2;
  a1.gsc = f.buf.x_g;
  a1.out = f.h;
  a1.hmax = f.hmax;
  moet_status s = launch_fc_tc<true>(a1, f.fc1, f.dfc1, f.buf.x_cperm, f.buf.x_cnat, f.buf.x_sf, pairs, f.E,
                                     f.I / 64, f.max_items, st);
  if (s != MOET_OK) return s;
  // FC2 input terms: one row per bucketed pair (h rows are in bucketed order)
  {
    ProfScope ps(MOET_K_TERMS, st);
    const dim3 grid(pairs, f.I / kTermThreads);
    act_terms_kernel<false><<<grid, kTermThreads, 0, st>>>(f.I, f.h, nullptr, 1,
                                                           reinterpret_cast<const float*>(f.hmax), f.buf.h_cperm,
                                                           f.buf.h_cnat, f.buf.h_sf, f.buf.h_g);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  FcTcArgs a2 = a;
  a2.K = f.I; a2.N = f.H;
  a2.scale_2 = f.fc2->scale_2;
  a2.gsc = f.buf.h_g;
  a2.out = f.o;
  return launch_fc_tc<false>(a2, f.fc2, f.dfc2, f.buf.h_cperm, f.buf.h_cnat, f.buf.h_sf, pairs, f.E, f.H / 128,
                             f.max_items, st);
}

}  // namespace moet

MOET_ERROR_ACCESSOR(moet_internal_error_moe_tc)
