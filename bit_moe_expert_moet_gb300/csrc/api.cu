// Status strings and the device error query of the moet C ABI.
#include "common.cuh"

extern "C" int moet_internal_error_requant(void);
extern "C" int moet_internal_error_route(void);
extern "C" int moet_internal_error_moe(void);

extern "C" const char* moet_status_string(moet_status s) {
  switch (s) {
    case MOET_OK: return "MOET_OK";
    case MOET_ERR_INVALID_ARG: return "MOET_ERR_INVALID_ARG";
    case MOET_ERR_SHAPE: return "MOET_ERR_SHAPE";
    case MOET_ERR_ALIGN: return "MOET_ERR_ALIGN";
    case MOET_ERR_UNSUPPORTED: return "MOET_ERR_UNSUPPORTED";
    case MOET_ERR_WORKSPACE: return "MOET_ERR_WORKSPACE";
    case MOET_ERR_CUDA: return "MOET_ERR_CUDA";
    case MOET_ERR_TIMEOUT: return "MOET_ERR_TIMEOUT";
    case MOET_ERR_DEVICE_INDEX: return "MOET_ERR_DEVICE_INDEX";
  }
  return "MOET_ERR_UNKNOWN";
}

extern "C" moet_status moet_last_device_error(moet_stream stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOET_ERR_CUDA;
  int first = 0;
  const int codes[3] = {moet_internal_error_requant(), moet_internal_error_route(),
                        moet_internal_error_moe()};
  for (int c : codes) {
    if (c < 0) return MOET_ERR_CUDA;
    if (first == 0 && c != 0) first = c;
  }
  return (moet_status)first;
}
