// Internal interface between the forward's entry point (moe.cu) and the
// tcgen05 block-scaled FC engine (moe_tc.cu).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moet.h"

namespace moet {

constexpr int kTcTerms = 4;   // NVFP4 terms per activation row
constexpr int kTcTok = 16;    // tokens (pairs) per tcgen05 work item -> N <= 64

struct TcBuffers {
  // activation terms of the FC1 input (rows = tokens) and FC2 input (rows = bucketed pairs)
  uint8_t* x_cperm; uint8_t* x_cnat; uint8_t* x_sf; float* x_g;
  uint8_t* h_cperm; uint8_t* h_cnat; uint8_t* h_sf; float* h_g;
};

// Bytes of activation-term storage for `rows` rows of length K.
inline size_t tc_terms_bytes(size_t rows, size_t K) {
  return rows * kTcTerms * (K / 2 * 2 + K / 16) + rows * kTcTerms * sizeof(float) + 4 * 256;
}

// True when the tcgen05 engine handles this layer shape.
inline bool tc_supported(int H, int I) { return H % 256 == 0 && I % 256 == 0; }

struct TcForwardArgs {
  int T, H, I, E, k;
  const uint16_t* x;
  const int32_t* offsets;
  const int32_t* perm;
  const float* topk_w;
  const int32_t* topk_idx;     // expert of each pair
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
  const int4* chunks;          // (expert, first pair, count <= kTcTok, pool slot of the planes)
  int item_rows;               // 1: activation-term rows at item * kTcTok + slot (act_rows =
                               //    kTcTok x the item-list capacity); 0: at the pair's bucketed
                               //    position (act_rows = T k)
  int act_rows;                // activation-term source rows the term buffers hold
  float* h;                    // [T k, I] bucketed
  float* o;                    // [T k, H] pair order
  const float* tokmax;         // [T] max |x_t| (written by the prologue)
  unsigned* hmax;              // [T k] max |h| per bucketed pair, zeroed by the prologue
  const int32_t* inv;          // [T k] pair -> bucketed position (written by the prologue)
  TcBuffers buf;
  int max_items;
};

// FC1 (its input terms, then the FC kernel) and FC2 (the same); tc_forward runs both.
moet_status tc_forward_fc1(const TcForwardArgs& a, cudaStream_t st);
moet_status tc_forward_fc2(const TcForwardArgs& a, cudaStream_t st);
moet_status tc_forward(const TcForwardArgs& a, cudaStream_t st);

}  // namespace moet
