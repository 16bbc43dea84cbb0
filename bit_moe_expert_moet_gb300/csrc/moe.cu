// MoE expert-layer forward over 2-bit sign/magnitude planes with the NVFP4 delta.
//
// README "Frontier MoE on consumer Blackwell (SM120)", "How it fits -- 2-bit
// experts at FP4 quality", bullet 2: decode streams the 2-bit experts (an FP4
// read is twice the bytes); experts in the delta cache add the FP4 residual
// for tokens the confidence gate flags.
//
// Launch chain on the caller's stream (no host synchronisation):
//   1. prologue   chunk list (expert, first pair, count<=64) from the expert
//                 offsets; per-token power-of-two activation scales; zeroes
//                 the per-pair |h| maxima.
//   2. fc<FC1>    h = SiLU(x Wg^T) * (x Wu^T) per routed pair (+ delta on gated
//                 pairs of cached experts), fp32, bucketed order.
//   3. fc<FC2>    o_p = w_p * h_p W2^T (+ delta), fp32, in pair order t*k+j.
//   4. combine    y_t = sum_j o_{t*k+j} in a fixed order, rounded to bf16.
//
// Inner product engine (fc kernels).  A warp owns a 16-row MMA tile of one
// expert's weight matrix (FC1: 8 gate rows + the 8 matching up rows, so
// SiLU*mul happens in registers; FC2: 16 output rows) and streams its 2-bit
// planes with 128-bit read-only loads, 128 weights per row per step.  The
// codes are expanded in registers to f16 A fragments of mma.sync.m16n8k16:
// f16 +-1 and +-3 have a zero low byte, so one PRMT over a 4-entry byte
// table turns two 2-bit codes into one f16x2 register.  K is permuted inside
// each 16-block so that every lane's codes sit at a fixed stride in the
// plane word; the activations (B operand, staged once per CTA in shared
// memory as f16) carry the same permutation.  One MMA covers exactly one
// 16-weight scale block, and its fp32 result is scaled by that block's s16
// and accumulated in fp32.  Activations reach f16 through a power-of-two
// scale per row (token or pair) so that the conversion from bf16 is exact
// except for values 2^31 below the row maximum.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "moe_pf.cuh"
#include "moe_tc.cuh"

namespace moet {

constexpr int kChunk = 64;          // pairs per work item
constexpr int kThreads = 256;       // 8 warps
constexpr int kSmemBudget = 96 * 1024;
constexpr uint32_t kCodeLut = 0xC242BC3Cu;  // f16 high bytes of +1, -1, +3, -3

struct WsLayout {
  size_t hdr, tok_scale, tok_max, hmax, inv, pvalid, chunks, chunks_s, h, o, xt, ht, pfa, perm2, total;
};

// Largest T routed through the tcgen05 engine (small tokens-per-expert regime).
constexpr int kTcMaxT = 512;

// Prefill regime (T > kTcMaxT): an expert routed at most this many pairs is a weight stream with
// few tokens, where the bf16 engine's 128-row tiles would cost as much as for 256 pairs; its pairs
// go through the block-scaled decode engine in items of kTcTok instead (a second work list).
constexpr int kPfSmallMax = 32;

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline int max_chunks(int T, int E, int k, int chunk) {
  const long long pairs = (long long)T * k;
  return (int)((pairs < E ? pairs : E) + (pairs + chunk - 1) / chunk);
}

// Capacity of the prefill regime's second work list: items of <= kTcTok pairs of experts with at
// most kPfSmallMax pairs.
inline int pf_small_items(int T, int E, int k) {
  const long long a = max_chunks(T, E, k, kTcTok);
  const long long b = (long long)E * ((kPfSmallMax + kTcTok - 1) / kTcTok);
  return (int)(a < b ? a : b);
}

inline bool pf_hybrid(int T, int H, int I) {
  return T > kTcMaxT && pf_supported(H, I) && tc_supported(H, I) && kPfSmallMax > 0;
}

inline WsLayout ws_layout(int T, int H, int I, int E, int k) {
  WsLayout L;
  const size_t pairs = (size_t)T * k;
  size_t off = 0;
  L.hdr = off;       off += align256(32);              // [0..2] item counts, ok; [4..7] unit counters
  L.tok_scale = off; off += align256(sizeof(float) * T);
  L.tok_max = off;   off += align256(sizeof(float) * T);
  L.hmax = off;      off += align256(sizeof(unsigned) * pairs);
  L.inv = off;       off += align256(sizeof(int32_t) * pairs);
  L.pvalid = off;    off += align256(pairs);
  L.chunks = off;    off += align256(sizeof(int4) * (size_t)max_chunks(T, E, k, kTcTok));
  L.h = off;         off += align256(sizeof(float) * pairs * I);
  L.o = off;         off += align256(sizeof(float) * pairs * H);
  L.xt = off; L.ht = off; L.pfa = off; L.chunks_s = off; L.perm2 = off;
  if (T <= kTcMaxT && tc_supported(H, I)) {
    L.xt = off;      off += align256(tc_terms_bytes(pairs, (size_t)H));
    L.ht = off;      off += align256(tc_terms_bytes(pairs, (size_t)I));
  } else if (T > kTcMaxT && pf_supported(H, I)) {
    L.pfa = off;     off += align256(pf_act_bytes(pairs, (size_t)H, (size_t)I) + 5 * 256);
    L.perm2 = off;   off += align256(sizeof(int32_t) * pairs);
    if (pf_hybrid(T, H, I)) {
      const size_t items = (size_t)pf_small_items(T, E, k), rows = items * kTcTok;
      L.chunks_s = off; off += align256(sizeof(int4) * items);
      L.xt = off;       off += align256(tc_terms_bytes(rows, (size_t)H));
      L.ht = off;       off += align256(tc_terms_bytes(rows, (size_t)I));
    }
  }
  L.total = off;
  return L;
}

// Prefill regime with the delta: the engines walk the pairs in a private order, the bucketed
// order with each cached expert's pairs stably split into its gated pairs first, then the rest.
// A work item is a run of consecutive pairs of one expert, so only the items that reach into
// the gated run make the delta pass, and within an item the gated pairs are the leading
// columns.  Every pair's result depends only on its own column, so the layer's output is the
// same as in the bucketed order.  One CTA per expert: the gated count first (all loads in
// flight), then 1024-pair chunks, four consecutive pairs per thread, placed by a block-wide
// exclusive scan.  A pair id out of range counts as ungated (the engines report it).
constexpr int kGfPer = 4;                       // pairs per thread per chunk

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const int t = warp_tot[w];
    base += w < warp ? t : 0;
    all += t;
  }
  __syncthreads();                               // warp_tot is reused by the next call
  *total = all;
  return base + incl - v;
}

__global__ void __launch_bounds__(kThreads) gated_first_kernel(int k, int n_pairs, const int32_t* __restrict__ offsets,
                                                               const int32_t* __restrict__ perm,
                                                               const int32_t* __restrict__ delta_slot,
                                                               const uint8_t* __restrict__ gate,
                                                               int32_t* __restrict__ perm2) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  __shared__ int warp_tot[kThreads / 32];
  const int e = blockIdx.x, tid = threadIdx.x;
  const int off = __ldg(offsets + e), n = __ldg(offsets + e + 1) - off;
  if (n <= 0 || off < 0 || off + n > n_pairs) return;
  if (__ldg(delta_slot + e) < 0) {
    for (int i = tid; i < n; i += kThreads) perm2[off + i] = __ldg(perm + off + i);
    return;
  }
  auto is_gated = [&](int p) { return p >= 0 && p < n_pairs && __ldg(gate + p / k) != 0; };
  int mine = 0;
  for (int i = tid; i < n; i += kThreads) mine += is_gated(__ldg(perm + off + i)) ? 1 : 0;
  int G = 0;
  (void)block_exclusive_scan(mine, warp_tot, &G);
  int gi = 0, ui = G;                            // next gated / ungated destination
  for (int c = 0; c < n; c += kThreads * kGfPer) {
    int p[kGfPer];
    bool g[kGfPer];
    int ng = 0, nu = 0;
#pragma unroll
    for (int q = 0; q < kGfPer; ++q) {
      const int i = c + tid * kGfPer + q;
      p[q] = i < n ? __ldg(perm + off + i) : -1;
      g[q] = i < n && is_gated(p[q]);
      ng += g[q] ? 1 : 0;
      nu += (i < n && !g[q]) ? 1 : 0;
    }
    int tg = 0, tu = 0;
    int pg = block_exclusive_scan(ng, warp_tot, &tg);
    int pu = block_exclusive_scan(nu, warp_tot, &tu);
#pragma unroll
    for (int q = 0; q < kGfPer; ++q) {
      const int i = c + tid * kGfPer + q;
      if (i >= n) break;
      if (g[q]) perm2[off + gi + pg++] = p[q];
      else perm2[off + ui + pu++] = p[q];
    }
    gi += tg;
    ui += tu;
  }
}

// power-of-two multiplier that brings max|row| into [2^14, 2^15)
__device__ __forceinline__ float pow2_scale_for(float amax) {
  if (!(amax > 0.0f) || !isfinite(amax)) return 1.0f;
  int e;
  frexpf(amax, &e);          // amax = f * 2^e, f in [0.5, 1)
  int s = 15 - e;            // amax * 2^s in [2^14, 2^15)
  s = s > 100 ? 100 : (s < -100 ? -100 : s);
  return ldexpf(1.0f, s);
}

// ---------------------------------------------------------------- prologue
// With an expert slot table (pooled forward), experts that are not resident get no work items,
// their routed pairs are counted (miss_count, miss_mask) and marked invalid for the combine, and
// each work item carries the expert's pool slot (.w) for the plane and scale_2 addressing; without
// one, .w is the expert id.
__global__ void __launch_bounds__(kThreads) prologue_kernel(
    int T, int H, int E, int k, int chunk, int chunk_small, int small_max, int4* __restrict__ chunks_small,
    const uint16_t* __restrict__ x, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ perm, int* __restrict__ hdr, float* __restrict__ tok_scale,
    float* __restrict__ tok_max, unsigned* __restrict__ hmax, int32_t* __restrict__ inv, int4* __restrict__ chunks,
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ expert_slot, int n_pool,
    unsigned* __restrict__ miss_count, uint8_t* __restrict__ miss_mask, uint8_t* __restrict__ pvalid,
    const int32_t* __restrict__ delta_slot, int rowmax_mode) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (blockIdx.x == 0) {
    // The work items (lists chunks and chunks_small), built by the block's warps: warp w takes the
    // 32-expert groups w, w + 8, ...  With a delta table the items of experts with a delta slot
    // come first in each list (their units may carry the delta pass, three times the stages of a
    // plain unit, and the engines hand units out in list order), then the others; within each
    // class, expert order.  Per expert four item counts (list x class), scanned inside each group
    // by warp shuffles and across groups in shared memory.
    constexpr int kGroups = 1024 / 32;                  // E <= 1024
    constexpr int kPerWarp = kGroups / (kThreads / 32);
    __shared__ int gpre[kGroups][4];                    // per group: items of (list, class), then their prefix
    __shared__ int tot[4];
    __shared__ int okf;
    if (tid == 0) okf = __ldg(offsets) == 0 && __ldg(offsets + E) == T * k;
    __syncthreads();                                    // okf set before any warp may clear it
    const bool split = delta_slot != nullptr;
    const int ngroups = (E + 31) / 32;
    int nv[kPerWarp], pv[kPerWarp], cnt[kPerWarp][4], excl[kPerWarp][4];
#pragma unroll
    for (int r = 0; r < kPerWarp; ++r) {
      const int g = warp + r * (kThreads / 32), e = 32 * g + lane;
      int n = 0, pslot = e;
      bool heavy = true;
      if (g < ngroups && e < E) {
        n = __ldg(offsets + e + 1) - __ldg(offsets + e);
        if (n < 0) { okf = 0; n = 0; }
        if (expert_slot != nullptr) {
          pslot = __ldg(expert_slot + e);
          if (pslot >= n_pool) { record_error(MOET_ERR_DEVICE_INDEX); pslot = -1; }
          if (pslot < 0 && n > 0) {
            if (miss_count != nullptr) atomicAdd(miss_count, (unsigned)n);
            if (miss_mask != nullptr) miss_mask[e] = 1;
          }
        }
        heavy = !split || __ldg(delta_slot + e) >= 0;
      }
      // an expert with at most small_max pairs goes to the second list (items of chunk_small)
      const bool small = small_max > 0 && n <= small_max;
      const int nch = g < ngroups && e < E && pslot >= 0 && !small ? (n + chunk - 1) / chunk : 0;
      const int nchs = g < ngroups && e < E && pslot >= 0 && small ? (n + chunk_small - 1) / chunk_small : 0;
      nv[r] = n;
      pv[r] = pslot;
      cnt[r][0] = heavy ? nch : 0;   cnt[r][1] = heavy ? 0 : nch;      // list 0 (chunks): heavy, light
      cnt[r][2] = heavy ? nchs : 0;  cnt[r][3] = heavy ? 0 : nchs;     // list 1 (chunks_small)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        int incl = cnt[r][q];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        excl[r][q] = incl - cnt[r][q];
        if (lane == 31 && g < ngroups) gpre[g][q] = incl;
      }
    }
    __syncthreads();
    if (tid < 4) {
      int running = 0;
      for (int g = 0; g < ngroups; ++g) {
        const int v = gpre[g][tid];
        gpre[g][tid] = running;
        running += v;
      }
      tot[tid] = running;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kPerWarp; ++r) {
      const int g = warp + r * (kThreads / 32), e = 32 * g + lane;
      if (g >= ngroups || e >= E) continue;
      const int n = nv[r], pslot = pv[r];
      const int nch = cnt[r][0] + cnt[r][1], nchs = cnt[r][2] + cnt[r][3];
      const int first = cnt[r][0] > 0 ? gpre[g][0] + excl[r][0] : tot[0] + gpre[g][1] + excl[r][1];
      for (int c = 0; c < nch; ++c) chunks[first + c] = make_int4(e, c * chunk, min(chunk, n - c * chunk), pslot);
      const int first_s = cnt[r][2] > 0 ? gpre[g][2] + excl[r][2] : tot[2] + gpre[g][3] + excl[r][3];
      for (int c = 0; c < nchs; ++c)
        chunks_small[first_s + c] = make_int4(e, c * chunk_small, min(chunk_small, n - c * chunk_small), pslot);
    }
    __syncthreads();
    if (tid == 0) {
      const bool ok = okf != 0;
      if (!ok) record_error(MOET_ERR_DEVICE_INDEX);
      hdr[0] = ok ? tot[0] + tot[1] : 0;
      hdr[1] = ok ? 1 : 0;
      hdr[2] = ok ? tot[2] + tot[3] : 0;
      hdr[4] = 0;                                        // the decode engine's unit counters (FC1, FC2)
      hdr[5] = 0;
      hdr[6] = 0;                                        // the bf16 engine's (FC1, FC2)
      hdr[7] = 0;
    }
    return;
  }
  // blocks >= 1: one warp per token, zeroing of hmax and (when asked) the
  // inverse of the bucketing permutation, pair -> bucketed position
  const int gw = (blockIdx.x - 1) * (kThreads / 32) + warp;
  const int nthreads = (gridDim.x - 1) * kThreads;
  for (int i = (blockIdx.x - 1) * kThreads + tid; i < T * k; i += nthreads) {
    hmax[i] = 0u;
    if (pvalid != nullptr) {
      // pair i (= t k + j) counts in the combine only if its expert is resident
      const int e = __ldg(topk_idx + i);
      int sl = -1;
      if (e >= 0 && e < E) sl = __ldg(expert_slot + e);
      pvalid[i] = (sl >= 0 && sl < n_pool) ? 1 : 0;
    }
    if (inv != nullptr) {
      const int p = __ldg(perm + i);
      if (p >= 0 && p < T * k) inv[p] = i;
    }
  }
  if (gw >= T) return;
  // The per-token max |x| (and its power-of-two scale) feeds the decode and mma.sync engines'
  // input quantisation: every token (rowmax_mode 1), none (0: the bf16 engine alone), or in the
  // prefill regime's split only tokens with a pair in the small-expert list (2).
  if (rowmax_mode == 0) return;
  if (rowmax_mode == 2) {
    bool small = false;
    if (lane < k) {
      const int e = __ldg(topk_idx + (size_t)gw * k + lane);
      small = e >= 0 && e < E && __ldg(offsets + e + 1) - __ldg(offsets + e) <= small_max;
    }
    if (!__any_sync(0xffffffffu, small)) return;
  }
  const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)gw * H);
  float m = 0.0f;
  for (int i = lane; i < H / 8; i += 32) {
    const uint4 v = __ldg(row + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      m = fmaxf(m, fabsf(__uint_as_float(w[q] << 16)));
      m = fmaxf(m, fabsf(__uint_as_float(w[q] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) {
    tok_scale[gw] = pow2_scale_for(m);
    tok_max[gw] = m;
  }
}

// ---------------------------------------------------------------- fc kernels
// Staged layout of one 16-element K-block of an activation row: the lane with
// c = lane & 3 reads halves 4c..4c+3 = (x_c, x_{c+8}, x_{c+4}, x_{c+12}),
// which are the B-fragment rows 2c, 2c+1, 2c+8, 2c+9 of mma.m16n8k16; the
// A fragments built from the planes use the same order.

struct FcArgs {
  int T, H, I, E, k, K, N;
  const uint16_t* x;
  const float* h_in;
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
  const float* tok_scale;
  unsigned* hmax;
  float* out;        // FC1: h [pairs, I] bucketed; FC2: o [pairs, H] by pair id
  int ks;            // K slice staged per pass (multiple of 128)
};

template <bool FC1, int NT>
__global__ void __launch_bounds__(kThreads, 2) fc_kernel(const FcArgs a) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  if ((int)blockIdx.y >= a.hdr[0]) return;
  const int4 ch = a.chunks[blockIdx.y];
  const int e = ch.x, count = ch.z;
  const size_t pe = (size_t)ch.w;                        // pool slot of the expert's planes
  const int pos0 = __ldg(a.offsets + e) + ch.y;
  const int K = a.K;
  const int pitch = a.ks + 16;                           // halves per staged row
  __half* xs = reinterpret_cast<__half*>(smem_raw);      // [NT*8 + 1][pitch], last row = zeros
  float* rscale = reinterpret_cast<float*>(smem_raw + sizeof(__half) * (NT * 8 + 1) * pitch);  // [NT*8]
  float* gatef = rscale + NT * 8;                        // [NT*8]
  int* rsrc = reinterpret_cast<int*>(gatef + NT * 8);    // [NT*8] token (FC1) or pair id (FC2)
  __shared__ int any_gated;

  int slot = -1;
  if (a.delta_slot != nullptr && a.gate != nullptr) {
    slot = __ldg(a.delta_slot + e);
    if (slot >= a.n_slots) { record_error(MOET_ERR_DEVICE_INDEX); slot = -1; }
  }
  if (tid == 0) any_gated = 0;
  __syncthreads();
  if (tid < NT * 8) {
    float sc = 0.0f, gf = 0.0f;
    int src = -1;
    if (tid < count) {
      const int p = __ldg(a.perm + pos0 + tid);
      const int tok = p / a.k;
      if (p < 0 || p >= a.T * a.k) {
        record_error(MOET_ERR_DEVICE_INDEX);
      } else {
        src = FC1 ? tok : p;
        if (FC1) {
          sc = __ldg(a.tok_scale + tok);
        } else {
          sc = pow2_scale_for(__uint_as_float(a.hmax[pos0 + tid]));
        }
        if (slot >= 0 && __ldg(a.gate + tok)) { gf = 1.0f; any_gated = 1; }
      }
    }
    rscale[tid] = sc;
    gatef[tid] = gf;
    rsrc[tid] = src;
  }
  __syncthreads();
  const bool do_delta = slot >= 0 && any_gated;
  const int ntiles = (count + 7) >> 3;

  // rows of this warp
  int row_g, row_u;
  if (FC1) {
    const int i0 = blockIdx.x * 64 + warp * 8;
    row_g = i0 + g;
    row_u = a.I + i0 + g;
  } else {
    const int r0 = blockIdx.x * 128 + warp * 16;
    row_g = r0 + g;
    row_u = r0 + g + 8;
  }
  const size_t wpr = (size_t)K / 32, bpr = (size_t)K / 16;
  const uint32_t* Sg = a.sign + (pe * a.N + row_g) * wpr;
  const uint32_t* Mg = a.mag + (pe * a.N + row_g) * wpr;
  const uint32_t* Su = a.sign + (pe * a.N + row_u) * wpr;
  const uint32_t* Mu = a.mag + (pe * a.N + row_u) * wpr;
  const uint8_t* Qg = a.s16 + (pe * a.N + row_g) * bpr;
  const uint8_t* Qu = a.s16 + (pe * a.N + row_u) * bpr;
  const uint8_t* Dg = nullptr; const uint8_t* Du = nullptr;
  const uint8_t* DQg = nullptr; const uint8_t* DQu = nullptr;
  if (do_delta) {
    Dg = a.dcodes + ((size_t)slot * a.N + row_g) * (K / 2);
    Du = a.dcodes + ((size_t)slot * a.N + row_u) * (K / 2);
    DQg = a.ds4 + ((size_t)slot * a.N + row_g) * bpr;
    DQu = a.ds4 + ((size_t)slot * a.N + row_u) * bpr;
  }

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;

  for (int k0 = 0; k0 < K; k0 += a.ks) {
    const int k1 = min(K, k0 + a.ks);
    const int nblk = (k1 - k0) / 16;
    __syncthreads();                                     // previous slice fully consumed
    if (k0 == 0) {                                       // zero row read by padding columns
      for (int i = tid; i < pitch / 8; i += kThreads)
        reinterpret_cast<uint4*>(xs + (size_t)NT * 8 * pitch)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    // ---- stage the chunk's activation rows of this slice: one 16-block per item
    for (int it = tid; it < count * nblk; it += kThreads) {
      const int r = it / nblk, b = it - r * nblk;
      float v[16];
      const int src = rsrc[r];
      if (src >= 0) {
        const float sc = rscale[r];
        if (FC1) {
          const uint4* p = reinterpret_cast<const uint4*>(a.x + (size_t)src * a.H + k0 + 16 * b);
          const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
          const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            v[2 * q] = __uint_as_float(w[q] << 16) * sc;
            v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u) * sc;
          }
        } else {
          const float4* p = reinterpret_cast<const float4*>(a.h_in + (size_t)(pos0 + r) * a.I + k0 + 16 * b);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 f = p[q];
            v[4 * q] = f.x * sc; v[4 * q + 1] = f.y * sc; v[4 * q + 2] = f.z * sc; v[4 * q + 3] = f.w * sc;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.0f;
      }
      // staged order: (x0,x8) (x4,x12) (x1,x9) (x5,x13) (x2,x10) (x6,x14) (x3,x11) (x7,x15)
      uint32_t wv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int j = (q >> 1) + 4 * (q & 1);
        const __half2 hp = __floats2half2_rn(v[j], v[j + 8]);
        wv[q] = *reinterpret_cast<const uint32_t*>(&hp);
      }
      uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)r * pitch + 16 * b);
      dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
    }
    __syncthreads();

    // ---- 2-bit pass over the slice, 128 weights per row per step; the next
    // step's plane loads are issued before the current step is expanded
    const __half* xrow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r = nt * 8 + g;
      xrow[nt] = xs + (size_t)(r < count ? r : NT * 8) * pitch + 4 * c;
    }
    uint4 sg = ldg_nc_v4(Sg + k0 / 32), mg = ldg_nc_v4(Mg + k0 / 32);
    uint4 su = ldg_nc_v4(Su + k0 / 32), mu = ldg_nc_v4(Mu + k0 / 32);
    uint2 qg = ldg_nc_v2(Qg + k0 / 16), qu = ldg_nc_v2(Qu + k0 / 16);
    for (int kk = k0; kk < k1; kk += 128) {
      const int kn = kk + 128 < k1 ? kk + 128 : kk;
      const uint4 nsg = ldg_nc_v4(Sg + kn / 32), nmg = ldg_nc_v4(Mg + kn / 32);
      const uint4 nsu = ldg_nc_v4(Su + kn / 32), nmu = ldg_nc_v4(Mu + kn / 32);
      const uint2 nqg = ldg_nc_v2(Qg + kn / 16), nqu = ldg_nc_v2(Qu + kn / 16);
      const uint32_t SG[4] = {sg.x, sg.y, sg.z, sg.w}, MG[4] = {mg.x, mg.y, mg.z, mg.w};
      const uint32_t SU[4] = {su.x, su.y, su.z, su.w}, MU[4] = {mu.x, mu.y, mu.z, mu.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t cg = ((SG[q] >> c) & 0x11111111u) | (((MG[q] >> c) & 0x11111111u) << 1);
        const uint32_t cu = ((SU[q] >> c) & 0x11111111u) | (((MU[q] >> c) & 0x11111111u) << 1);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t xg = hh ? (cg >> 16) : cg, xu = hh ? (cu >> 16) : cu;
          const uint32_t a0 = prmt(kCodeLut, 0u, (xg << 4) + 0x0404u);
          const uint32_t a2 = prmt(kCodeLut, 0u, xg + 0x0404u);
          const uint32_t a1 = prmt(kCodeLut, 0u, (xu << 4) + 0x0404u);
          const uint32_t a3 = prmt(kCodeLut, 0u, xu + 0x0404u);
          const int bi = 2 * q + hh;                       // block inside the 128-step
          const uint32_t qgw = bi < 4 ? qg.x : qg.y, quw = bi < 4 ? qu.x : qu.y;
          const float sgf = e4m3_to_f32(qgw >> (8 * (bi & 3)));
          const float suf = e4m3_to_f32(quw >> (8 * (bi & 3)));
          const int lb = (kk - k0) / 16 + bi;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (nt < ntiles) {
              const uint2 bv = *reinterpret_cast<const uint2*>(xrow[nt] + 16 * lb);
              float d[4];
              mma_f16_16816(d, a0, a1, a2, a3, bv.x, bv.y);
              acc[nt][0] = fmaf(sgf, d[0], acc[nt][0]);
              acc[nt][1] = fmaf(sgf, d[1], acc[nt][1]);
              acc[nt][2] = fmaf(suf, d[2], acc[nt][2]);
              acc[nt][3] = fmaf(suf, d[3], acc[nt][3]);
            }
          }
        }
      }
      sg = nsg; mg = nmg; su = nsu; mu = nmu; qg = nqg; qu = nqu;
    }

    // ---- delta pass (gated pairs of a cached expert), 32 weights per row per step
    if (do_delta) {
      for (int kk = k0; kk < k1; kk += 32) {
        const uint4 dg = ldg_nc_v4(Dg + kk / 2), du = ldg_nc_v4(Du + kk / 2);
        const uint32_t sq_g = *reinterpret_cast<const uint16_t*>(DQg + kk / 16);
        const uint32_t sq_u = *reinterpret_cast<const uint16_t*>(DQu + kk / 16);
        const uint32_t DG[4] = {dg.x, dg.y, dg.z, dg.w}, DU[4] = {du.x, du.y, du.z, du.w};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // weights c, c+8 -> a0/a1 ; c+4, c+12 -> a2/a3 (same permutation as above)
          const uint32_t lg = DG[2 * hh] >> (4 * c), hg = DG[2 * hh + 1] >> (4 * c);
          const uint32_t lu = DU[2 * hh] >> (4 * c), hu = DU[2 * hh + 1] >> (4 * c);
          const uint32_t tg = (lg & 0x000F000Fu) | ((hg & 0x000F000Fu) << 4);
          const uint32_t tu = (lu & 0x000F000Fu) | ((hu & 0x000F000Fu) << 4);
          const uint32_t a0 = e2m1x2_to_f16x2(tg & 0xFFu), a2 = e2m1x2_to_f16x2((tg >> 16) & 0xFFu);
          const uint32_t a1 = e2m1x2_to_f16x2(tu & 0xFFu), a3 = e2m1x2_to_f16x2((tu >> 16) & 0xFFu);
          const float sgf = e4m3_to_f32(sq_g >> (8 * hh));
          const float suf = e4m3_to_f32(sq_u >> (8 * hh));
          const int lb = (kk - k0) / 16 + hh;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (nt < ntiles) {
              const uint2 bv = *reinterpret_cast<const uint2*>(xrow[nt] + 16 * lb);
              float d[4];
              mma_f16_16816(d, a0, a1, a2, a3, bv.x, bv.y);
              const float g0 = gatef[nt * 8 + 2 * c], g1 = gatef[nt * 8 + 2 * c + 1];
              acc[nt][0] = fmaf(sgf * g0, d[0], acc[nt][0]);
              acc[nt][1] = fmaf(sgf * g1, d[1], acc[nt][1]);
              acc[nt][2] = fmaf(suf * g0, d[2], acc[nt][2]);
              acc[nt][3] = fmaf(suf * g1, d[3], acc[nt][3]);
            }
          }
        }
      }
    }
  }

  // ---- epilogue
  const float sc2 = __ldg(a.scale_2 + pe);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int col = 0; col < 2; ++col) {
      const int n = nt * 8 + 2 * c + col;
      const bool valid = nt < ntiles && n < count && rsrc[min(n, NT * 8 - 1)] >= 0;
      const float inv = valid ? sc2 / rscale[n] : 0.0f;
      if (FC1) {
        const float gv = acc[nt][col] * inv, uv = acc[nt][2 + col] * inv;
        const float hv = valid ? gv / (1.0f + expf(-gv)) * uv : 0.0f;
        if (valid) a.out[(size_t)(pos0 + n) * a.I + row_g] = hv;
        float m = fabsf(hv);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (valid && g == 0) atomicMax(a.hmax + pos0 + n, __float_as_uint(m));
      } else if (valid) {
        const int p = rsrc[n];
        const float wp = __ldg(a.topk_w + p) * inv;
        a.out[(size_t)p * a.H + row_g] = acc[nt][col] * wp;
        a.out[(size_t)p * a.H + row_u] = acc[nt][2 + col] * wp;
      }
    }
  }
}

// ---------------------------------------------------------------- combine
constexpr int kCombineBatch = 8;                // partial rows in flight per thread
constexpr int kCombineCtasPerSm = 4;            // guaranteed by the launch bounds: one full wave
__global__ void __launch_bounds__(kThreads, kCombineCtasPerSm)
    combine_kernel(int T, int H, int k, const int* __restrict__ hdr, const float* __restrict__ o,
                   const uint8_t* __restrict__ pvalid, uint16_t* __restrict__ y) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  const long long n4 = (long long)T * H / 4;
  const bool ok = hdr[1] != 0;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const long long t = (i * 4) / H, r = (i * 4) % H;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ok) {
      // the partial rows are loaded kCombineBatch at a time before their adds (the loads
      // overlap), then summed in pair order; a pair of a non-resident expert (pooled forward) is
      // skipped: its o row is never written
      for (int j0 = 0; j0 < k; j0 += kCombineBatch) {
        float4 v[kCombineBatch];
        bool use[kCombineBatch];
#pragma unroll
        for (int u = 0; u < kCombineBatch; ++u) {
          const int j = j0 + u;
          use[u] = j < k && (pvalid == nullptr || __ldg(pvalid + (size_t)t * k + j) != 0);
          if (use[u]) v[u] = __ldg(reinterpret_cast<const float4*>(o + ((size_t)t * k + j) * H + r));
        }
#pragma unroll
        for (int u = 0; u < kCombineBatch; ++u)
          if (use[u]) { s.x += v[u].x; s.y += v[u].y; s.z += v[u].z; s.w += v[u].w; }
      }
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(s.x, s.y), hi = __floats2bfloat162_rn(s.z, s.w);
    uint2 outv;
    outv.x = *reinterpret_cast<const uint32_t*>(&lo);
    outv.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(y + (size_t)t * H + r) = outv;
  }
}

template <bool FC1, int NT>
static moet_status launch_fc(const FcArgs& a, int row_tiles, int grid_y, cudaStream_t st) {
  const size_t smem = sizeof(__half) * (NT * 8 + 1) * (a.ks + 16) + 3 * sizeof(float) * NT * 8;
  auto kern = fc_kernel<FC1, NT>;
  MOET_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  {
    ProfScope ps(FC1 ? MOET_K_FC1 : MOET_K_FC2, st);
    MOET_CUDA_TRY(pdl_launch(false, kern, dim3(dim3(row_tiles, grid_y)), dim3(kThreads), smem, st, a));
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}

template <bool FC1>
static moet_status dispatch_fc(FcArgs a, int nt, int row_tiles, int grid_y, cudaStream_t st) {
  const int rows = nt * 8;
  int ks = (kSmemBudget / ((rows + 1) * 2) - 16) / 128 * 128;
  if (ks > a.K) ks = a.K;
  a.ks = ks;
  switch (nt) {
    case 1: return launch_fc<FC1, 1>(a, row_tiles, grid_y, st);
    case 2: return launch_fc<FC1, 2>(a, row_tiles, grid_y, st);
    case 4: return launch_fc<FC1, 4>(a, row_tiles, grid_y, st);
    default: return launch_fc<FC1, 8>(a, row_tiles, grid_y, st);
  }
}

}  // namespace moet

using namespace moet;

MOET_ERROR_ACCESSOR(moet_internal_error_moe)

extern "C" size_t moet_forward_workspace_size(int T, int H, int I, int E, int k) {
  if (T < 1 || H < 1 || I < 1 || E < 1 || k < 1) return 0;
  return ws_layout(T, H, I, E, k).total;
}

// The forward behind moet_moe_forward (expert_slot == null: the planes hold all E experts) and
// moet_moe_forward_pooled (the planes hold n_pool slots, expert e in slot expert_slot[e]).
static moet_status forward_impl(int T, int H, int I, int E, int k, const uint16_t* x, const int32_t* topk_idx,
                                const float* topk_w, const int32_t* expert_offsets, const int32_t* perm,
                                const int32_t* expert_slot, int n_pool, const moet_planes* fc1,
                                const moet_planes* fc2, const int32_t* delta_slot, int n_slots,
                                const moet_nvfp4* dfc1, const moet_nvfp4* dfc2, const uint8_t* gate_mask,
                                unsigned* miss_count, uint8_t* miss_mask, uint16_t* y, void* workspace,
                                size_t ws_bytes, moet_stream stream) {
  if (T < 1 || H < 128 || I < 128 || H % 128 || I % 128 || E < 1 || E > 1024 || k < 1 || k > 16 ||
      k > E)
    return MOET_ERR_SHAPE;
  if ((long long)T * k > (1LL << 30) || (long long)T * k * H > (1LL << 40)) return MOET_ERR_UNSUPPORTED;
  if (!x || !topk_idx || !topk_w || !expert_offsets || !perm || !fc1 || !fc2 || !y) return MOET_ERR_INVALID_ARG;
  if (!fc1->sign || !fc1->mag || !fc1->s16 || !fc1->scale_2 || !fc2->sign || !fc2->mag || !fc2->s16 ||
      !fc2->scale_2)
    return MOET_ERR_INVALID_ARG;
  const bool with_delta = delta_slot != nullptr && gate_mask != nullptr;
  if (with_delta) {
    if (n_slots < 1 || !dfc1 || !dfc2 || !dfc1->codes || !dfc1->s4 || !dfc2->codes || !dfc2->s4)
      return MOET_ERR_INVALID_ARG;
    if (((uintptr_t)dfc1->codes & 15) || ((uintptr_t)dfc2->codes & 15) || ((uintptr_t)dfc1->s4 & 1) ||
        ((uintptr_t)dfc2->s4 & 1))
      return MOET_ERR_ALIGN;
  }
  if (((uintptr_t)x & 15) || ((uintptr_t)y & 15) || ((uintptr_t)fc1->sign & 15) ||
      ((uintptr_t)fc1->mag & 15) || ((uintptr_t)fc2->sign & 15) || ((uintptr_t)fc2->mag & 15) ||
      ((uintptr_t)fc1->s16 & 7) || ((uintptr_t)fc2->s16 & 7) || ((uintptr_t)workspace & 255))
    return MOET_ERR_ALIGN;
  const WsLayout L = ws_layout(T, H, I, E, k);
  if (!workspace || ws_bytes < L.total) return MOET_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  char* ws = static_cast<char*>(workspace);
  int* hdr = reinterpret_cast<int*>(ws + L.hdr);
  float* tok_scale = reinterpret_cast<float*>(ws + L.tok_scale);
  float* tok_max = reinterpret_cast<float*>(ws + L.tok_max);
  unsigned* hmax = reinterpret_cast<unsigned*>(ws + L.hmax);
  int32_t* inv = reinterpret_cast<int32_t*>(ws + L.inv);
  int4* chunks = reinterpret_cast<int4*>(ws + L.chunks);
  float* h = reinterpret_cast<float*>(ws + L.h);
  float* o = reinterpret_cast<float*>(ws + L.o);
  uint8_t* pvalid = expert_slot != nullptr ? reinterpret_cast<uint8_t*>(ws + L.pvalid) : nullptr;
  const int n_planes = expert_slot != nullptr ? n_pool : E;     // experts (or slots) the planes hold

  const bool use_tc = T <= kTcMaxT && tc_supported(H, I);
  const bool use_pf = !use_tc && T > kTcMaxT && pf_supported(H, I);
  const bool hybrid = use_pf && pf_hybrid(T, H, I);
  const int chunk = use_tc ? kTcTok : use_pf ? kPfTok : kChunk;
  int4* chunks_s = hybrid ? reinterpret_cast<int4*>(ws + L.chunks_s) : nullptr;
  {
    ProfScope ps(MOET_K_PROLOGUE, st);
    MOET_CUDA_TRY(pdl_launch(use_tc, prologue_kernel, dim3(1 + (T + 7) / 8), dim3(kThreads), 0, st, T, H, E, k, chunk, kTcTok, hybrid ? kPfSmallMax : 0,
                                                           chunks_s, x, expert_offsets, perm, hdr,
                                                           tok_scale, tok_max, hmax, use_tc ? inv : nullptr,
                                                           chunks, topk_idx, expert_slot, n_pool, miss_count,
                                                           miss_mask, pvalid, with_delta ? delta_slot : nullptr,
                                                           hybrid ? 2 : use_pf ? 0 : 1));
  }
  MOET_CUDA_TRY(cudaGetLastError());

  const int mc = max_chunks(T, E, k, chunk);
  // the block-scaled decode engine's part: every item of the decode regime, or the prefill
  // regime's second list (experts with few pairs), with term rows per item slot
  auto carve = [](char* base, size_t rows, size_t K, uint8_t** cperm, uint8_t** cnat, uint8_t** sf, float** g) {
    size_t off = 0;
    *cperm = reinterpret_cast<uint8_t*>(base + off); off += align256(rows * kTcTerms * (K / 2));
    *cnat = reinterpret_cast<uint8_t*>(base + off);  off += align256(rows * kTcTerms * (K / 2));
    *sf = reinterpret_cast<uint8_t*>(base + off);    off += align256(rows * kTcTerms * (K / 16));
    *g = reinterpret_cast<float*>(base + off);
  };
  auto tc_args = [&](bool items) {
    TcForwardArgs f{};
    f.T = T; f.H = H; f.I = I; f.E = n_planes; f.k = k;   // E: experts the planes hold (tensor maps)
    f.x = x; f.offsets = expert_offsets; f.perm = perm; f.topk_w = topk_w;
    f.topk_idx = topk_idx; f.n_experts = E;
    f.fc1 = fc1; f.fc2 = fc2;
    f.delta_slot = with_delta ? delta_slot : nullptr;
    f.n_slots = n_slots; f.dfc1 = dfc1; f.dfc2 = dfc2;
    f.gate = with_delta ? gate_mask : nullptr;
    f.hdr = items ? hdr + 2 : hdr;
    f.work = hdr + 4;
    f.chunks = items ? chunks_s : chunks;
    f.h = h; f.o = o; f.max_items = items ? pf_small_items(T, E, k) : mc;
    f.tokmax = tok_max; f.hmax = hmax; f.inv = inv;
    f.item_rows = items ? 1 : 0;
    const size_t rows = items ? (size_t)pf_small_items(T, E, k) * kTcTok : (size_t)T * k;
    f.act_rows = (int)rows;
    carve(ws + L.xt, rows, (size_t)H, &f.buf.x_cperm, &f.buf.x_cnat, &f.buf.x_sf, &f.buf.x_g);
    carve(ws + L.ht, rows, (size_t)I, &f.buf.h_cperm, &f.buf.h_cnat, &f.buf.h_sf, &f.buf.h_g);
    return f;
  };
  if (use_pf) {
    // with the delta, the engines walk each cached expert's pairs gated first
    const int32_t* eperm = perm;
    if (with_delta) {
      int32_t* perm2 = reinterpret_cast<int32_t*>(ws + L.perm2);
      {
        ProfScope ps(MOET_K_PROLOGUE, st);
        MOET_CUDA_TRY(pdl_launch(false, gated_first_kernel, dim3(E), dim3(kThreads), 0, st, k, T * k, expert_offsets, perm, delta_slot, gate_mask, perm2));
      }
      MOET_CUDA_TRY(cudaGetLastError());
      eperm = perm2;
    }
    PfForwardArgs f{};
    f.T = T; f.H = H; f.I = I; f.E = n_planes; f.k = k;   // E: experts the planes hold (tensor maps)
    f.x = x; f.offsets = expert_offsets; f.perm = eperm; f.topk_w = topk_w;
    f.topk_idx = topk_idx; f.n_experts = E;
    f.fc1 = fc1; f.fc2 = fc2;
    f.delta_slot = with_delta ? delta_slot : nullptr;
    f.n_slots = n_slots; f.dfc1 = dfc1; f.dfc2 = dfc2;
    f.gate = with_delta ? gate_mask : nullptr;
    f.hdr = hdr; f.chunks = chunks; f.o = o;
    f.work = hdr + 6;
    const size_t pairs = (size_t)T * k;
    char* pb = ws + L.pfa;
    f.xb = reinterpret_cast<uint16_t*>(pb);  pb += align256(pairs * H * sizeof(uint16_t));
    f.xbg = reinterpret_cast<uint16_t*>(pb); pb += align256(pairs * H * sizeof(uint16_t));
    f.h = h;
    f.h16 = reinterpret_cast<uint16_t*>(pb);  pb += align256(pairs * I * sizeof(uint16_t));
    f.hg16 = reinterpret_cast<uint16_t*>(pb); pb += align256(pairs * I * sizeof(uint16_t));
    f.hscale = reinterpret_cast<float*>(pb);
    // FC1 of both lists (they write disjoint bucketed rows of h), then FC2 of both (disjoint
    // pairs of o); each engine's FC2 reads only its own rows of h
    if (hybrid) {
      TcForwardArgs g = tc_args(true);
      g.perm = eperm;
      moet_status s = tc_forward_fc1(g, st);
      if (s != MOET_OK) return s;
      s = pf_forward_fc1(f, st);
      if (s != MOET_OK) return s;
      s = tc_forward_fc2(g, st);
      if (s != MOET_OK) return s;
      s = pf_forward_fc2(f, st);
      if (s != MOET_OK) return s;
    } else {
      moet_status s = pf_forward(f, st);
      if (s != MOET_OK) return s;
    }
  } else if (use_tc) {
    moet_status s = tc_forward(tc_args(false), st);
    if (s != MOET_OK) return s;
  } else {
  const int maxn = T < kChunk ? T : kChunk;
  const int nt = maxn <= 8 ? 1 : maxn <= 16 ? 2 : maxn <= 32 ? 4 : 8;
  FcArgs a{};
  a.T = T; a.H = H; a.I = I; a.E = n_planes; a.k = k;
  a.x = x; a.h_in = h; a.offsets = expert_offsets; a.perm = perm; a.topk_w = topk_w;
  a.delta_slot = with_delta ? delta_slot : nullptr;
  a.gate = with_delta ? gate_mask : nullptr;
  a.n_slots = n_slots;
  a.hdr = hdr; a.chunks = chunks; a.tok_scale = tok_scale; a.hmax = hmax;

  FcArgs a1 = a;
  a1.K = H; a1.N = 2 * I;
  a1.sign = fc1->sign; a1.mag = fc1->mag; a1.s16 = fc1->s16; a1.scale_2 = fc1->scale_2;
  if (with_delta) { a1.dcodes = dfc1->codes; a1.ds4 = dfc1->s4; }
  a1.out = h;
  moet_status s = dispatch_fc<true>(a1, nt, I / 64, mc, st);
  if (s != MOET_OK) return s;

  FcArgs a2 = a;
  a2.K = I; a2.N = H;
  a2.sign = fc2->sign; a2.mag = fc2->mag; a2.s16 = fc2->s16; a2.scale_2 = fc2->scale_2;
  if (with_delta) { a2.dcodes = dfc2->codes; a2.ds4 = dfc2->s4; }
  a2.out = o;
  s = dispatch_fc<false>(a2, nt, H / 128, mc, st);
  if (s != MOET_OK) return s;
  }

  long long n4 = (long long)T * H / 4;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    sms = 152;
  long long gcl = (n4 + kThreads - 1) / kThreads;
  if (gcl > (long long)sms * kCombineCtasPerSm) gcl = (long long)sms * kCombineCtasPerSm;
  const int gc = (int)gcl;
  {
    ProfScope ps(MOET_K_COMBINE, st);
    MOET_CUDA_TRY(pdl_launch(use_tc, combine_kernel, dim3(gc), dim3(kThreads), 0, st, T, H, k, hdr, o, pvalid, y));
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}

extern "C" moet_status moet_moe_forward(int T, int H, int I, int E, int k, const uint16_t* x,
                                        const int32_t* topk_idx, const float* topk_w,
                                        const int32_t* expert_offsets, const int32_t* perm,
                                        const moet_planes* fc1, const moet_planes* fc2,
                                        const int32_t* delta_slot, int n_slots, const moet_nvfp4* dfc1,
                                        const moet_nvfp4* dfc2, const uint8_t* gate_mask, uint16_t* y,
                                        void* workspace, size_t ws_bytes, moet_stream stream) {
  return forward_impl(T, H, I, E, k, x, topk_idx, topk_w, expert_offsets, perm, nullptr, E, fc1, fc2, delta_slot,
                      n_slots, dfc1, dfc2, gate_mask, nullptr, nullptr, y, workspace, ws_bytes, stream);
}

extern "C" moet_status moet_moe_forward_pooled(int T, int H, int I, int E, int k, const uint16_t* x,
                                               const int32_t* topk_idx, const float* topk_w,
                                               const int32_t* expert_offsets, const int32_t* perm,
                                               const int32_t* expert_slot, int n_pool,
                                               const moet_planes* fc1, const moet_planes* fc2,
                                               const int32_t* delta_slot, int n_slots, const moet_nvfp4* dfc1,
                                               const moet_nvfp4* dfc2, const uint8_t* gate_mask,
                                               uint32_t* miss_count, uint8_t* miss_mask, uint16_t* y,
                                               void* workspace, size_t ws_bytes, moet_stream stream) {
  if (!expert_slot) return MOET_ERR_INVALID_ARG;
  if (n_pool < 1) return MOET_ERR_SHAPE;
  if ((uintptr_t)expert_slot & 3) return MOET_ERR_ALIGN;
  return forward_impl(T, H, I, E, k, x, topk_idx, topk_w, expert_offsets, perm, expert_slot, n_pool, fc1, fc2,
                      delta_slot, n_slots, dfc1, dfc2, gate_mask, miss_count, miss_mask, y, workspace, ws_bytes,
                      stream);
}
