"""GB300 (sm_103a) MoE expert layer over sign-symmetric 2-bit experts with an NVFP4 delta.

Thin Python binding of the C ABI in ``include/moet.h`` (libmoet.so).  Every
function here only checks and marshals arguments; all computation runs in the
library's CUDA kernels.  PyTorch is used for device memory and streams only.
There is no CPU fallback: importing this package without the built library,
or calling it on tensors that are not on a CUDA device, raises.

Entry points (same names as the C ABI without the ``moet_`` prefix):
  quantize_nvfp4   fp32 weights -> NVFP4 (codes, s4, scale_2)
  requant_2bit     NVFP4 -> 2-bit sign/magnitude planes + s16 (+ delta)
  requant_fp8_2bit FP8 block-quant -> scale_2, planes + s16 (+ delta)
  requant_mxfp4_2bit  MXFP4 (FP4 experts) -> scale_2, planes + s16 (+ delta)
  sign_bias_probe  bias and L2 error of per-block optimal fits to a 4-level codebook
  route_topk       logits -> top-k ids/weights, expert offsets, permutation
  moe_forward      the MoE layer y = sum_j w_j FFN_e(x) on the 2-bit planes
  moe_forward_pooled  the same over a pool of resident experts (slot table,
                   non-resident experts contribute zero and are counted)
  gate_from_confidence  the confidence gate: gate mask and the experts to promote
  moe_forward_static    moe_forward with its scratch in the library image (no workspace)
  debug_wait_expiry     test control of the engines' bounded waits
"""
from ._lib import (  # noqa: F401
    MoetError,
    Planes,
    DeltaPool,
    lib,
    lib_path,
    status_string,
    last_device_error,
    profile_enable,
    profile_read,
    debug_wait_expiry,
    KERNEL_KINDS,
    quantize_nvfp4,
    requant_2bit,
    requant_fp8_2bit,
    requant_mxfp4_2bit,
    sign_bias_probe,
    route_topk,
    forward_workspace_size,
    moe_forward,
    moe_forward_pooled,
    gate_from_confidence,
    moe_forward_static,
    FORWARD_STATIC_SCRATCH_BYTES,
)
