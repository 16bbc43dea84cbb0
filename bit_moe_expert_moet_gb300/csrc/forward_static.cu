// moet_moe_forward_static: the MoE forward with its scratch in the library image.
//
// Some callers cannot allocate device memory at the point where they run the
// layer: code that runs inside a memory-budgeted runtime whose allocator is
// owned by someone else, a plug-in handed only the input and output buffers,
// or a C caller without a device allocator of its own.  For them this entry
// point takes the same arguments as moet_moe_forward minus the workspace and
// uses a fixed scratch array that is part of this library's device image
// instead.  It calls no allocating routine at all.
//
// The scratch array (MOET_FORWARD_STATIC_SCRATCH_BYTES, 8 MiB) exists on every GPU that
// loads the library and stays there until the process exits.  Its device
// address is looked up with cudaGetSymbolAddress, with the device current, on
// every call made while `stream` is not being captured into a CUDA graph (a
// cheap host call; it also picks up a new address after a device reset reloads
// the module); a call made during stream capture uses the address found by the
// last call outside capture on that device, so the first call on a device must
// come before any stream capture.  All calls share the one array: calls that overlap on the
// GPU (different streams, or concurrent host threads) race on it and must be
// serialised by the caller.  No part of the scratch has to start at zero: the
// forward's kernels write every scratch word before reading it, so the stale
// contents left by the previous call do not matter.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = MOET_FORWARD_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_forward_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_forward_scratch on the current device: looked up afresh
// outside stream capture, the last address found outside capture during it.
moet_status scratch_on_current_device(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOET_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOET_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return MOET_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_forward_scratch) != cudaSuccess || p == nullptr) return MOET_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  } else if (g_scratch_ptr[dev] == nullptr) {
    return MOET_ERR_UNSUPPORTED;   // no call outside capture has set this device up yet
  }
  *out = g_scratch_ptr[dev];
  return MOET_OK;
}

}  // namespace

extern "C" moet_status moet_moe_forward_static(int T, int H, int I, int E, int k, const uint16_t* x,
                                               const int32_t* topk_idx, const float* topk_w,
                                               const int32_t* expert_offsets, const int32_t* perm,
                                               const moet_planes* fc1, const moet_planes* fc2,
                                               const int32_t* delta_slot, int n_slots,
                                               const moet_nvfp4* dfc1, const moet_nvfp4* dfc2,
                                               const uint8_t* gate_mask, uint16_t* y, moet_stream stream) {
  const size_t need = moet_forward_workspace_size(T, H, I, E, k);
  if (need == 0) return MOET_ERR_SHAPE;
  if (need > kStaticScratchBytes) return MOET_ERR_WORKSPACE;  // layer too large for the fixed scratch
  void* scratch = nullptr;
  const moet_status s = scratch_on_current_device((cudaStream_t)stream, &scratch);
  if (s != MOET_OK) return s;
  return moet_moe_forward(T, H, I, E, k, x, topk_idx, topk_w, expert_offsets, perm, fc1, fc2, delta_slot,
                          n_slots, dfc1, dfc2, gate_mask, y, scratch, kStaticScratchBytes, stream);
}
