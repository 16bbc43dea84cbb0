// Router top-k + renormalised softmax + token bucketing by expert.
//
// Routing step of the MoE layer (README "Frontier MoE on consumer Blackwell
// (SM120)", "How it fits"; the airanks page's DeepSeek-V4.1 table, row "MoE at
// decode", counts seven launches from router to FC1 in stock vLLM -- here it is
// one launch for up to 16 tokens, two beyond, three above 4096 pairs).
//
// Top-k: one warp per token; each lane holds ceil(E/32) logits in registers
// and a 64-bit key (order-preserving logit bits, then the complement of the
// expert id) so that one warp-wide max per round picks the largest logit with
// the lower id on ties.  NaN maps below -inf, -0 equals +0.
// Bucketing: one CTA of 1024 threads counts pairs per expert in shared
// memory, scans, and scatters pair ids stably in chunks of 1024 pairs: the
// rank inside a warp comes from __match_any_sync, the rank across warps of
// the chunk from a [32 warps][E] byte table of per-warp counts.  Up to 16
// tokens, the same CTA that ran the top-k buckets by counting over the ids it
// kept in shared memory (bucket_small).
#include "common.cuh"

namespace moet {

__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) return 0u;                         // NaN: below everything
  uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Returns, in lane j < k, the token's j-th expert id (-1 in the other lanes).
template <int VPL>
__device__ __forceinline__ int topk_one_token(int t, int E, int k, const float* __restrict__ logits,
                                              int32_t* __restrict__ topk_idx,
                                              float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  unsigned long long key[VPL];
  float val[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      val[i] = __ldg(logits + (long long)t * E + e);
      key[i] = ((unsigned long long)order_key(val[i]) << 32) | (0xFFFFu - (uint32_t)e);
    } else {
      val[i] = 0.0f;
      key[i] = 0ull;                              // below every real entry
    }
  }
  float my_logit = 0.0f;
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < VPL; ++i) best = key[i] > best ? key[i] : best;
    unsigned long long wbest = best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, wbest, o);
      wbest = other > wbest ? other : wbest;
    }
    const int e = 0xFFFF - (int)(wbest & 0xFFFFull);
    const int owner = e & 31;
    float lv = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      if (key[i] == wbest) {
        lv = val[i];
        key[i] = 0ull;
      }
    }
    lv = __shfl_sync(0xffffffffu, lv, owner);
    if (lane == j) {
      my_logit = lv;
      my_idx = e;
    }
  }
  const float lmax = __shfl_sync(0xffffffffu, my_logit, 0);
  float ex = lane < k ? expf(my_logit - lmax) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    topk_idx[(long long)t * k + lane] = my_idx;
    topk_w[(long long)t * k + lane] = ex / sum;
  }
  return lane < k ? my_idx : -1;
}

template <int VPL>
__global__ void __launch_bounds__(256) topk_kernel(int T, int E, int k, const float* __restrict__ logits,
                                                   int32_t* __restrict__ topk_idx,
                                                   float* __restrict__ topk_w) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (t < T) topk_one_token<VPL>(t, E, k, logits, topk_idx, topk_w);
}

// Bucketing of few pairs (n <= kSmallPairs) by counting, from the pairs' expert ids in shared
// memory (sidx[0 .. n4), n rounded up to a multiple of 4 with -1): offsets[e] = the number of
// valid pairs whose expert is below e (offsets[E] = all valid pairs), and pair p goes to
// offsets[e_p] + the number of pairs q < p with the same expert -- the stable bucketing, as the
// chunked scatter below computes it, without atomics, scans or a per-warp count table.  Every
// thread reads the whole id list (broadcast shared-memory loads, four ids per load), so the work
// grows as n^2: for T <= 16 tokens only (T = 8: step 0.250 -> 0.243 ms; at 512 pairs it took
// 14.8 us against the chunked scatter's 5.6 us).
constexpr int kSmallPairs = 256;
__device__ __forceinline__ void bucket_small(int n, int E, const int* __restrict__ sidx, int32_t* __restrict__ offsets,
                                             int32_t* __restrict__ perm) {
  const int n4 = (n + 3) & ~3;
  const int4* s4 = reinterpret_cast<const int4*>(sidx);
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    int c = 0;
    for (int q = 0; q < n4 / 4; ++q) {
      const int4 f = s4[q];
      c += ((unsigned)f.x < (unsigned)e) + ((unsigned)f.y < (unsigned)e) + ((unsigned)f.z < (unsigned)e) +
           ((unsigned)f.w < (unsigned)e);
    }
    offsets[e] = c;
  }
  for (int p = threadIdx.x; p < n; p += blockDim.x) {
    const int e = sidx[p];
    if ((unsigned)e >= (unsigned)E) {
      record_error(MOET_ERR_DEVICE_INDEX);
      continue;
    }
    int before = 0, same = 0;
    for (int q = 0; q < n4 / 4; ++q) {
      const int4 f = s4[q];
      const int fq[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        before += (unsigned)fq[i] < (unsigned)e;
        same += (4 * q + i < p) & (fq[i] == e);
      }
    }
    perm[before + same] = p;
  }
}

// Routing of up to kFusedMaxT tokens in one CTA of 1024 threads: the top-k of each token (a warp
// per token), its expert ids kept in shared memory, then bucket_small.
template <int VPL>
__global__ void __launch_bounds__(1024) route_small_kernel(int T, int E, int k, const float* __restrict__ logits,
                                                           int32_t* __restrict__ topk_idx,
                                                           float* __restrict__ topk_w,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ perm) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  __shared__ __align__(16) int sidx[kSmallPairs];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = T * k;
  for (int t = warp; t < T; t += 32) {
    const int id = topk_one_token<VPL>(t, E, k, logits, topk_idx, topk_w);
    if (lane < k) sidx[t * k + lane] = id;
  }
  if (tid < 3 && n + tid < kSmallPairs) sidx[n + tid] = -1;   // padding to a multiple of 4
  __syncthreads();
  bucket_small(n, E, sidx, offsets, perm);
}

// Bucketing of up to kBucketMultiPairs pairs in one CTA of 1024 threads (count, scan, chunked
// stable scatter).
__global__ void __launch_bounds__(1024) bucket_kernel(int T, int E, int k, int32_t* __restrict__ topk_idx,
                                                      int32_t* __restrict__ offsets,
                                                      int32_t* __restrict__ perm) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  extern __shared__ int smem[];
  int* counts = smem;                               // [E]
  int* base = smem + E;                             // [E]
  unsigned char* wc = (unsigned char*)(smem + 2 * E);  // [32][E]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int i = tid; i < E; i += 1024) counts[i] = 0;
  for (int i = tid; i < 32 * E; i += 1024) wc[i] = 0;
  __syncthreads();
  const int n = T * k;
  for (int p = tid; p < n; p += 1024) {
    const int e = topk_idx[p];
    if (e < 0 || e >= E) {
      record_error(MOET_ERR_DEVICE_INDEX);
      continue;
    }
    atomicAdd(counts + e, 1);
  }
  __syncthreads();
  // exclusive scan of counts[0..E) by warp 0 (E <= 1024: 32 values per lane)
  if (warp == 0) {
    int running = 0;
    for (int c0 = 0; c0 < E; c0 += 32) {
      const int e = c0 + lane;
      const int v = e < E ? counts[e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < E) {
        base[e] = running + incl - v;
        offsets[e] = running + incl - v;
      }
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) offsets[E] = running;
  }
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < n; c0 += 1024) {
    const int p = c0 + tid;
    int e = -1;
    if (p < n) {
      e = topk_idx[p];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    const int cnt = __popc(peers);
    if (e >= 0 && rank == 0) wc[warp * E + e] = (unsigned char)cnt;
    __syncthreads();
    if (e >= 0) {
      int pre = 0;
      for (int w = 0; w < warp; ++w) pre += wc[w * E + e];
      perm[base[e] + pre + rank] = p;
    }
    __syncthreads();
    if (e >= 0 && rank == 0) {
      atomicAdd(base + e, cnt);
      wc[warp * E + e] = 0;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- bucketing of large batches
// Beyond kBucketMultiPairs pairs the single CTA's chunk loop dominates the routing step (66 us at
// T = 4096, k = 8), so the work is split over one CTA per 1024-pair chunk without any scratch
// buffer: bucket_offsets_kernel (one CTA) counts all pairs per expert and writes the exclusive
// scan to offsets; bucket_scatter_kernel's CTA c counts per expert the pairs before its chunk
// (re-reading those ids from L2), adds them to the offsets, and scatters its own chunk stably
// with the same warp-rank scheme as bucket_kernel.  The permutation is the same as bucket_kernel's.
constexpr int kBucketMultiPairs = 4096;

__global__ void __launch_bounds__(1024) bucket_offsets_kernel(int n, int E, const int32_t* __restrict__ topk_idx,
                                                               int32_t* __restrict__ offsets) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  __shared__ int counts[1024];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < E; i += 1024) counts[i] = 0;
  __syncthreads();
  for (int p = tid; p < n; p += 1024) {
    const int e = __ldg(topk_idx + p);
    if (e < 0 || e >= E) {
      record_error(MOET_ERR_DEVICE_INDEX);
      continue;
    }
    atomicAdd(counts + e, 1);
  }
  __syncthreads();
  if (warp == 0) {
    int running = 0;
    for (int c0 = 0; c0 < E; c0 += 32) {
      const int e = c0 + lane;
      const int v = e < E ? counts[e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < E) offsets[e] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) offsets[E] = running;
  }
}

__global__ void __launch_bounds__(1024) bucket_scatter_kernel(int n, int E, const int32_t* __restrict__ topk_idx,
                                                               const int32_t* __restrict__ offsets,
                                                               int32_t* __restrict__ perm) {
  pdl_wait();                                  // the previous kernel is complete
  pdl_trigger();
  extern __shared__ int smem[];
  int* base = smem;                                   // [E]
  unsigned char* wc = (unsigned char*)(smem + E);     // [32][E]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c0 = blockIdx.x * 1024;
  for (int i = tid; i < E; i += 1024) base[i] = 0;
  for (int i = tid; i < 32 * E; i += 1024) wc[i] = 0;
  __syncthreads();
  // pairs of each expert before this chunk (ids out of range are recorded by bucket_offsets_kernel)
  for (int p = tid; p < c0; p += 1024) {
    const int e = __ldg(topk_idx + p);
    if (e >= 0 && e < E) atomicAdd(base + e, 1);
  }
  __syncthreads();
  for (int i = tid; i < E; i += 1024) base[i] += __ldg(offsets + i);
  const int p = c0 + tid;
  int e = -1;
  if (p < n) {
    e = __ldg(topk_idx + p);
    if (e < 0 || e >= E) e = -1;
  }
  const unsigned lt_mask = (1u << lane) - 1u;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & lt_mask);
  const int cnt = __popc(peers);
  if (e >= 0 && rank == 0) wc[warp * E + e] = (unsigned char)cnt;
  __syncthreads();
  if (e >= 0) {
    int pre = 0;
    for (int w = 0; w < warp; ++w) pre += wc[w * E + e];
    perm[base[e] + pre + rank] = p;
  }
}

// Largest T routed by the single-CTA fused kernel: beyond it the top-k work
// (about k warp-wide arg-max rounds per token) is spread over one warp per
// token on many SMs, and one CTA buckets the result (at T = 64, E = 256, k = 8
// the fused kernel takes 27 us, the two kernels 10 us).
constexpr int kFusedMaxT = 16;

template <int VPL>
static moet_status launch_route(int T, int E, int k, const float* logits, int32_t* idx, float* w,
                                int32_t* offsets, int32_t* perm, cudaStream_t st) {
  const size_t smem = (size_t)E * 8 + (size_t)E * 32;
  const int n = T * k;
  if (T <= kFusedMaxT) {                                // n <= 16 * 16 = kSmallPairs
    ProfScope ps(MOET_K_ROUTE, st);
    MOET_CUDA_TRY(pdl_launch(true, route_small_kernel<VPL>, dim3(1), dim3(1024), 0, st, T, E, k, logits, idx, w,
                             offsets, perm));
  } else if ((long long)n > kBucketMultiPairs) {
    {
      ProfScope ps(MOET_K_ROUTE, st);
      MOET_CUDA_TRY(pdl_launch(false, topk_kernel<VPL>, dim3((T + 7) / 8), dim3(256), 0, st, T, E, k, logits, idx, w));
    }
    MOET_CUDA_TRY(cudaGetLastError());
    {
      ProfScope ps(MOET_K_ROUTE, st);
      MOET_CUDA_TRY(pdl_launch(false, bucket_offsets_kernel, dim3(1), dim3(1024), 0, st, n, E, idx, offsets));
    }
    MOET_CUDA_TRY(cudaGetLastError());
    const size_t ssmem = (size_t)E * 4 + (size_t)E * 32;
    if (ssmem > 48 * 1024)
      MOET_CUDA_TRY(cudaFuncSetAttribute(bucket_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssmem));
    ProfScope ps(MOET_K_ROUTE, st);
    MOET_CUDA_TRY(pdl_launch(false, bucket_scatter_kernel, dim3((n + 1023) / 1024), dim3(1024), ssmem, st, n, E, idx, offsets, perm));
  } else {
    {
      ProfScope ps(MOET_K_ROUTE, st);
      MOET_CUDA_TRY(pdl_launch(true, topk_kernel<VPL>, dim3((T + 7) / 8), dim3(256), 0, st, T, E, k, logits, idx, w));
    }
    MOET_CUDA_TRY(cudaGetLastError());
    if (smem > 48 * 1024)
      MOET_CUDA_TRY(cudaFuncSetAttribute(bucket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    ProfScope ps(MOET_K_ROUTE, st);
    MOET_CUDA_TRY(pdl_launch(true, bucket_kernel, dim3(1), dim3(1024), smem, st, T, E, k, idx, offsets, perm));
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}

// ---------------------------------------------------------------- confidence gate
// One thread per (token, slot j) pair: the gate of its token, and for gated tokens whether its
// expert lacks a delta slot.  Thread j = 0 of a token writes the gate and counts it.
__global__ void __launch_bounds__(256) gate_kernel(int T, int E, int k, const float* __restrict__ conf, float tau,
                                                   const int32_t* __restrict__ topk_idx,
                                                   const int32_t* __restrict__ delta_slot,
                                                   uint8_t* __restrict__ gate_mask, uint8_t* __restrict__ need_mask,
                                                   unsigned* __restrict__ counts) {
  const long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= (long long)T * k) return;
  const int t = (int)(p / k), j = (int)(p - (long long)t * k);
  const bool gated = __ldg(conf + t) < tau;                 // false for NaN
  if (j == 0) {
    gate_mask[t] = gated ? 1 : 0;
    if (gated && counts != nullptr) atomicAdd(counts, 1u);
  }
  if (!gated) return;
  const int e = __ldg(topk_idx + p);
  if (e < 0 || e >= E) {
    record_error(MOET_ERR_DEVICE_INDEX);
    return;
  }
  const bool cached = delta_slot != nullptr && __ldg(delta_slot + e) >= 0;
  if (!cached) {
    if (need_mask != nullptr) need_mask[e] = 1;
    if (counts != nullptr) atomicAdd(counts + 1, 1u);
  }
}

}  // namespace moet

using namespace moet;

MOET_ERROR_ACCESSOR(moet_internal_error_route)

extern "C" moet_status moet_gate_from_confidence(int T, int E, int k, const float* conf, float tau,
                                                 const int32_t* topk_idx, const int32_t* delta_slot,
                                                 uint8_t* gate_mask, uint8_t* need_mask, uint32_t* counts,
                                                 moet_stream stream) {
  if (T < 1 || E < 1 || E > 1024 || k < 1 || k > 16 || k > E) return MOET_ERR_SHAPE;
  if ((long long)T * k > (1LL << 30)) return MOET_ERR_UNSUPPORTED;
  if (!conf || !topk_idx || !gate_mask) return MOET_ERR_INVALID_ARG;
  if (((uintptr_t)conf & 3) || ((uintptr_t)topk_idx & 3) || ((uintptr_t)delta_slot & 3) ||
      ((uintptr_t)counts & 3))
    return MOET_ERR_ALIGN;
  cudaStream_t st = (cudaStream_t)stream;
  const long long n = (long long)T * k;
  {
    ProfScope ps(MOET_K_ROUTE, st);
    gate_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(T, E, k, conf, tau, topk_idx, delta_slot, gate_mask,
                                                             need_mask, counts);
  }
  MOET_CUDA_TRY(cudaGetLastError());
  return MOET_OK;
}

extern "C" moet_status moet_route_topk(int T, int E, int k, const float* logits, int32_t* topk_idx,
                                       float* topk_w, int32_t* expert_offsets, int32_t* perm,
                                       moet_stream stream) {
  if (T < 1 || E < 1 || E > 1024 || k < 1 || k > 16 || k > E) return MOET_ERR_SHAPE;
  if ((long long)T * k > (1LL << 30)) return MOET_ERR_UNSUPPORTED;
  if (!logits || !topk_idx || !topk_w || !expert_offsets || !perm) return MOET_ERR_INVALID_ARG;
  if (((uintptr_t)logits & 3) || ((uintptr_t)topk_idx & 3) || ((uintptr_t)topk_w & 3) ||
      ((uintptr_t)expert_offsets & 3) || ((uintptr_t)perm & 3))
    return MOET_ERR_ALIGN;
  cudaStream_t st = (cudaStream_t)stream;
  const int vpl = (E + 31) / 32;
  if (vpl <= 2) return launch_route<2>(T, E, k, logits, topk_idx, topk_w, expert_offsets, perm, st);
  if (vpl <= 4) return launch_route<4>(T, E, k, logits, topk_idx, topk_w, expert_offsets, perm, st);
  if (vpl <= 8) return launch_route<8>(T, E, k, logits, topk_idx, topk_w, expert_offsets, perm, st);
  if (vpl <= 12) return launch_route<12>(T, E, k, logits, topk_idx, topk_w, expert_offsets, perm, st);
  if (vpl <= 16) return launch_route<16>(T, E, k, logits, topk_idx, topk_w, expert_offsets, perm, st);
  return launch_route<32>(T, E, k, logits, topk_idx, topk_w, expert_offsets, perm, st);
}
