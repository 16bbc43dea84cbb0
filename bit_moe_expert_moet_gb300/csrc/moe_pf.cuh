// Internal interface between the forward's entry point (moe.cu) and the
// tcgen05 bf16 engine for large token counts (moe_pf.cu).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moet.h"

namespace moet {

constexpr int kPfTok = 256;   // routed pairs per work item -> MMA N <= 256

// True when the bf16 engine handles this layer shape.
// I <= 16384: the h -> fp16 kernel holds a row of h in at most 256 threads' registers.
inline bool pf_supported(int H, int I) { return H % 256 == 0 && I % 256 == 0 && I <= 16384; }

// Bytes of the engine's extra activation buffers for `pairs` routed pairs: x in
// bucketed order as bf16 plus its gated copy (rows of ungated pairs zero), h as
// scaled fp16 plus its gated copy, and the per-row scales of h (FC1 writes fp32
// h into the forward's h buffer).
inline size_t pf_act_bytes(size_t pairs, size_t H, size_t I) {
  return pairs * H * 2 * sizeof(uint16_t) + pairs * I * 2 * sizeof(uint16_t) + pairs * sizeof(float);
}

struct PfForwardArgs {
  int T, H, I, E, k;
  const uint16_t* x;
  const int32_t* offsets;
  const int32_t* perm;
  const float* topk_w;
  const int32_t* topk_idx;     // expert of each pair (which pairs the delta pass can read)
  int n_experts;               // experts the ids range over (delta_slot entries)
  const moet_planes* fc1;
  const moet_planes* fc2;
  const int32_t* delta_slot;   // nullable
  int n_slots;
  const moet_nvfp4* dfc1;
  const moet_nvfp4* dfc2;
  const uint8_t* gate;         // nullable
  const int* hdr;              // [0] = number of work items
  int* work;                   // [0] FC1, [1] FC2: units handed out so far (zeroed by the prologue)
  const int4* chunks;          // (expert, first pair, count <= kPfTok, pool slot of the planes)
  uint16_t* xb;                // [T k, H] bf16, bucketed rows, K permuted within 32-groups
  uint16_t* xbg;               // same, rows of ungated pairs zero
  float* h;                    // [T k, I] fp32, FC1 output (bucketed rows, natural order)
  uint16_t* h16;               // [T k, I] fp16, h times 2^-e per row, K permuted within 32-groups
  uint16_t* hg16;              // same, rows of ungated pairs zero
  float* hscale;               // [T k] 2^e per bucketed row
  float* o;                    // [T k, H] pair order
};

// FC1 (the gather of x, then the FC kernel) and FC2 (h to scaled fp16, then the FC kernel);
// pf_forward runs both.
moet_status pf_forward_fc1(const PfForwardArgs& a, cudaStream_t st);
moet_status pf_forward_fc2(const PfForwardArgs& a, cudaStream_t st);
moet_status pf_forward(const PfForwardArgs& a, cudaStream_t st);

}  // namespace moet
