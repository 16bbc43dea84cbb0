/*
 * moet.h -- C ABI of the GB300 (sm_103a) library for MoE expert layers over
 * sign-symmetric 2-bit expert weights with an NVFP4 delta.
 *
 * Method: vLLM-Moet README ("Frontier MoE on consumer Blackwell (SM120)"),
 * sections "GLM-5.2 (753B) -- the headline model" (modelopt NVFP4 experts,
 * load-time requantisation) and "How it fits -- 2-bit experts at FP4 quality"
 * (sign-symmetric 2-bit codebook, FP4 delta cache, confidence gate).  The
 * pages leave the 2-bit levels open; this library fixes q in {-3,-1,+1,+3}
 * with an e4m3 scale s16 per block of 16 along K.
 *
 * Conventions shared by every entry point
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    never allocates or frees memory (except the one-time 1 KB error flag
 *    that is part of the library image).  Shapes are given in elements.
 *  - Every call is asynchronous on `stream` and returns after enqueueing.
 *    Host-side argument checks run first and nothing is enqueued when one
 *    fails.  No entry point synchronises, except moet_last_device_error.
 *    Stream order holds as usual: some kernels (routing of up to 4096 pairs,
 *    the forward's block-scaled engine for up to 512 tokens) are launched
 *    with programmatic stream serialization,
 *    so they may be scheduled while the previous kernel on `stream` still
 *    runs, but each waits for that kernel's completion before its first
 *    access to global memory.
 *  - Problems that only the device can see (an index out of range, a
 *    bounded wait that expired) never trap: the kernel records the first
 *    such problem in a device flag and skips the offending access; read it
 *    with moet_last_device_error.
 *  - Matrices are row-major.  "Units of scale_2" means a value divided by
 *    the matrix's fp32 per-tensor scale_2.
 *
 * Data formats
 *  NVFP4 matrix [N, K]: codes u8 [N, K/2] (two e2m1 codes per byte, LOW
 *    nibble = even k; code bit 3 = sign, bits 0..2 index {0,.5,1,1.5,2,3,4,6}),
 *    s4 u8 [N, K/16] (e4m3fn scale per 16 along K), scale_2 fp32.
 *  2-bit planes [N, K]: sign u32 [N, K/32], mag u32 [N, K/32] (bit j of word
 *    w holds k = 32 w + j; sign 1 = negative; mag 1 = |q| = 3), s16 u8
 *    [N, K/16] (e4m3fn).  Weight = (sign ? -1 : 1) * (mag ? 3 : 1) * s16 *
 *    scale_2.  The code is never zero.
 *  Delta: an NVFP4 matrix on the SAME scale_2 holding W_nvfp4 - W_2bit.
 */
#ifndef MOET_H
#define MOET_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moet_stream; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  MOET_OK = 0,
  MOET_ERR_INVALID_ARG = 1, /* null pointer where one is required, bad enum/size      */
  MOET_ERR_SHAPE = 2,       /* a dimension violates the stated divisibility or range  */
  MOET_ERR_ALIGN = 3,       /* a pointer is not aligned as the entry point requires   */
  MOET_ERR_UNSUPPORTED = 4, /* shape valid in principle but not handled by the library  */
  MOET_ERR_WORKSPACE = 5,   /* workspace missing or smaller than the size query       */
  MOET_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed            */
  MOET_ERR_TIMEOUT = 7,     /* a bounded device wait expired (device flag)            */
  MOET_ERR_DEVICE_INDEX = 8 /* device saw an index out of range (device flag)         */
} moet_status;

/* Human-readable name of a status.  Never returns NULL. */
const char* moet_status_string(moet_status s);

/* Synchronises `stream`, then returns and clears the first device-side
 * problem recorded by any kernel of this library on the current device
 * (MOET_OK if none).  Returns MOET_ERR_CUDA if the synchronisation fails. */
moet_status moet_last_device_error(moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_quantize_nvfp4 -- fp32 weights -> NVFP4 (the experts' input format).
 * README "Frontier MoE on consumer Blackwell (SM120)", "GLM-5.2 (753B)" par. 1
 * (e2m1 x e4m3 block-16 x fp32 scale_2), read as: scale_2 = fp32(amax/2688);
 * s4 = e4m3 RNE(block amax / (6 scale_2)); code = e2m1 RNE(w / (s4 scale_2)),
 * ties to even, saturating, sign of w kept (-0 stays -0); amax = 0 or s4 = 0
 * give +-0 codes.
 *   M matrices of [N, K] each, K % 32 == 0, M,N >= 1.
 *   w        [M, N, K] fp32, 16-byte aligned
 *   scale_2  [M] fp32 (written)
 *   codes    [M, N, K/2] u8 (written), 16-byte aligned
 *   s4       [M, N, K/16] u8 (written), 2-byte aligned
 * Enqueues a zero-fill of scale_2 and three kernels.  */
moet_status moet_quantize_nvfp4(int M, int N, int K, const float* w, float* scale_2,
                                uint8_t* codes, uint8_t* s4, moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_requant_2bit -- load-time NVFP4 -> 2-bit planes (+ optional delta).
 * README "GLM-5.2 (753B)" par. 1 (exact dequant then sign-symmetric 2-bit
 * requantisation) and "How it fits" bullets 1-2.  In units of scale_2, with
 * v = e2m1(code) * e4m3(s4) exact, per block of 16 along K:
 *   s16 = e4m3 satfinite RNE(max|v| / 3); sign = sign bit of the code;
 *   mag = (|v| >= 2 s16)   (the nearest level of w's sign, ties to |q| = 3).
 * Delta (when dcodes and ds4 are both non-NULL): d = v - q s16 (exact),
 *   ds4 = e4m3 RNE(max|d| / 6), dcode = sign(d) | e2m1 RNE(|d| / ds4),
 *   a zero magnitude written as +0.  The result does not depend on scale_2,
 *   which the delta shares with the planes, so scale_2 is not an argument.
 *   M matrices of [N, K], K % 32 == 0.
 *   codes [M,N,K/2] u8, s4 [M,N,K/16] u8            (read; 16 B / 2 B aligned)
 *   sign, mag [M,N,K/32] u32, s16 [M,N,K/16] u8      (written; 4 B / 2 B aligned)
 *   dcodes [M,N,K/2] u8, ds4 [M,N,K/16] u8            (written if non-NULL)
 * All outputs are bit-exact functions of the inputs.  */
moet_status moet_requant_2bit(int M, int N, int K, const uint8_t* codes, const uint8_t* s4,
                              uint32_t* sign, uint32_t* mag, uint8_t* s16,
                              uint8_t* dcodes, uint8_t* ds4, moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_requant_fp8_2bit -- FP8 block-quant weights -> 2-bit planes (+ delta).
 * README "How it fits -- 2-bit experts at FP4 quality", last paragraph: FP8
 * block-quant checkpoints are requantised to the sign-symmetric codebook at
 * load like the NVFP4 ones.  A matrix holds an e4m3 code per weight and one
 * fp32 scale per 128 x 128 block: W = e4m3(code) * bscale (exact in fp64).
 * The pages give no formula for this input; this library applies the NVFP4
 * rule of moet_requant_2bit to W with a per-matrix
 *   scale_2 = fp32(fp64(amax |W|) / 1344)      (1344 = 3 * 448),
 * so the largest block's s16 lands at 448:
 *   s16 = e4m3 satfinite RNE(max_b |W| / (3 scale_2)); sign = the code's sign
 *   bit; mag = |W| >= 2 s16 scale_2; the delta is the NVFP4 residual of
 *   W - q s16 scale_2 on the same scale_2 (scale e4m3 RNE(max|d| / (6 scale_2)),
 *   codes e2m1 RNE, zero as +0).  Every ratio is rounded once, exactly: the
 *   kernels hold each number as an integer times a power of two and decide by
 *   integer comparisons.
 *   M >= 1 matrices of [N, K], K % 32 == 0.  codes [M, N, K] u8 (16 B aligned;
 *   the NaN codes 0x7F/0xFF are not valid weights); bscale [M, ceil(N/128),
 *   ceil(K/128)] fp32, finite and >= 0 (read; for another value the outputs of
 *   that block and the matrix's scale_2 are unspecified, nothing faults).
 *   scale_2 [M] fp32, sign/mag [M, N, K/32] u32, s16 [M, N, K/16] u8
 *   (written; the first words of each matrix's sign plane also serve as
 *   scratch for the amax pass before the planes are written); dcodes
 *   [M, N, K/2] / ds4 [M, N, K/16] (both NULL = no delta).  Outputs are
 *   bit-exact. */
moet_status moet_requant_fp8_2bit(int M, int N, int K, const uint8_t* codes, const float* bscale,
                                  float* scale_2, uint32_t* sign, uint32_t* mag, uint8_t* s16,
                                  uint8_t* dcodes, uint8_t* ds4, moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_requant_mxfp4_2bit -- FP4-expert (MXFP4) weights -> 2-bit planes (+ delta).
 * README "How it fits -- 2-bit experts at FP4 quality", last paragraph:
 * checkpoints whose experts are FP4 (DeepSeek-V4-Flash) load by a code remap.
 * The pages name no format; this library reads it as OCP MXFP4: an e2m1 code
 * per weight and one E8M0 scale 2^(e - 127) per 32 weights along K, so
 * W = e2m1(code) * 2^(e - 127), exact in fp64.  The remap is the rule of
 * moet_requant_fp8_2bit applied to W: scale_2 = fp32(fp64(amax |W|) / 1344),
 * s16 = e4m3 satfinite RNE(max_b |W| / (3 scale_2)), sign = the code's sign
 * bit, mag = |W| >= 2 s16 scale_2, and the NVFP4 delta of W - q s16 scale_2.
 *   M >= 1 matrices of [N, K], K % 32 == 0.  codes [M, N, K/2] u8, low nibble =
 *   even k (16 B aligned); e8m0 [M, N, K/32] u8 (read; 0xFF = NaN is not a
 *   valid scale: the outputs of its group are unspecified, nothing faults).
 *   scale_2 [M] fp32, sign/mag [M, N, K/32] u32, s16 [M, N, K/16] u8 (written;
 *   the sign plane also serves as scratch for the amax pass, as in
 *   moet_requant_fp8_2bit); dcodes [M, N, K/2] / ds4 [M, N, K/16] (both NULL =
 *   no delta).  Outputs are bit-exact (integer arithmetic, as above). */
moet_status moet_requant_mxfp4_2bit(int M, int N, int K, const uint8_t* codes, const uint8_t* e8m0,
                                    float* scale_2, uint32_t* sign, uint32_t* mag, uint8_t* s16,
                                    uint8_t* dcodes, uint8_t* ds4, moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_sign_bias_probe -- bias and L2 error of per-block optimal 2-bit fits.
 * README "How it fits -- 2-bit experts at FP4 quality", bullet 1 (the
 * sign-bias finding): the L2-optimal fit of a naive 2-bit codebook drops one
 * sign's tail and biases every tensor; a sign-symmetric codebook at the same
 * L2 error does not.  For a codebook of 4 integer levels L, each block of 16
 * weights along K gets the scale s > 0 that minimises
 * sum (w - s L[nearest(w / s)])^2 (exactly: the best of the 969 monotone
 * assignments of the sorted block, chosen in fp32 with a fixed operation
 * order, its sums evaluated in fp64); Q is that fit (0 when no s > 0 fits).
 *   M >= 1 matrices of [N, K] fp32, K % 16 == 0: w (device, 16 B aligned,
 *   read; NaN/inf weights give unspecified sums).  levels: HOST int32[4],
 *   strictly ascending, each in [-64, 64].  row_sums [M, N, 4] and sums [M, 4]
 *   fp64 (device, written): per row and per matrix (rows summed in order)
 *   sum W, sum W^2, sum (Q - W), sum (Q - W)^2. */
moet_status moet_sign_bias_probe(int M, int N, int K, const float* w, const int32_t* levels,
                                 double* row_sums, double* sums, moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_route_topk -- router top-k, renormalised softmax, bucketing by expert.
 * Per token: the k largest logits (ties -> lower expert id; NaN below -inf),
 * ordered by decreasing logit; w_j = exp(l_j - l_max) / sum over the k.
 * counts[e] = pairs routed to e; expert_offsets = exclusive scan [E+1]
 * (offsets[E] = T k); perm lists pair ids p = t k + j grouped by increasing
 * expert and by increasing p inside an expert (a stable sort).
 *   1 <= T, 1 <= E <= 1024, 1 <= k <= min(16, E).
 *   logits [T, E] fp32 (read); topk_idx [T, k] i32, topk_w [T, k] fp32,
 *   expert_offsets [E+1] i32, perm [T k] i32 (written).
 * Indices, offsets and perm are bit-exact; weights are fp32 (|err| < 1e-6).  */
moet_status moet_route_topk(int T, int E, int k, const float* logits, int32_t* topk_idx,
                            float* topk_w, int32_t* expert_offsets, int32_t* perm,
                            moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_gate_from_confidence -- the confidence gate's producer.
 * README "Frontier MoE on consumer Blackwell (SM120)", "How it fits" (the FP4
 * tier): a confidence gate re-runs low-confidence steps at FP4 -- it promotes
 * the step's routed experts into the delta cache, replays the step once and
 * decides again.  The pages do not define the confidence; here it is one
 * float per token supplied by the caller (e.g. the probability of the token
 * the previous step sampled), and the gate of token t is conf[t] < tau
 * (strict; a NaN confidence never gates).
 *   1 <= T, 1 <= E <= 1024, 1 <= k <= min(16, E).
 *   conf [T] fp32 (read); topk_idx [T, k] i32 (read, as from moet_route_topk);
 *   delta_slot [E] i32 (read; NULL = no expert is cached).
 *   gate_mask [T] u8 (written: 1 = gated).
 *   need_mask [E] u8 (nullable; entry e set to 1 when a gated token routes to
 *     e and e has no delta slot -- the experts to promote before the replay;
 *     never cleared here).
 *   counts: nullable u32 [2]; counts[0] += gated tokens, counts[1] += (gated
 *     token, expert) pairs whose expert has no delta slot (atomic; the caller
 *     resets them).
 * An expert id outside [0, E) is a device index error; its pair is skipped. */
moet_status moet_gate_from_confidence(int T, int E, int k, const float* conf, float tau,
                                      const int32_t* topk_idx, const int32_t* delta_slot,
                                      uint8_t* gate_mask, uint8_t* need_mask, uint32_t* counts,
                                      moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_moe_forward -- the MoE expert layer on 2-bit planes with the delta.
 * README "How it fits" bullet 2: y_t = sum_j w_tj FFN_{e_tj}(x_t), with
 * FFN_e(x) = W2_e (SiLU(Wg_e x) * (Wu_e x)) and SiLU(z) = z / (1 + e^-z).
 * FC1 planes hold [2I, H] per expert (gate rows 0..I-1, up rows I..2I-1),
 * FC2 planes hold [H, I].  For a pair whose token has gate_mask[t] != 0 and
 * whose expert has delta_slot[e] >= 0, both matrices become W_2bit + delta
 * (delta pool slot delta_slot[e], same scale_2 as the expert's planes).
 * No SwiGLU clamp.  bf16 activations in and out, fp32 accumulation.
 *   T >= 1, H % 128 == 0, I % 128 == 0, 1 <= E <= 1024, 1 <= k <= min(16,E).
 *   x [T, H] bf16 bits (u16, 16 B aligned); y [T, H] bf16 bits (written).
 *   topk_idx, topk_w, expert_offsets, perm: as written by moet_route_topk.
 *   fc1/fc2: planes of all E experts, scale_2 [E] fp32.
 *   delta_slot [E] i32 (-1 = not cached) and gate_mask [T] u8 may be NULL
 *   (no delta); n_slots bounds the slot values; dfc1/dfc2 hold the pool as
 *   [n_slots, 2I, H/2] / [n_slots, H, I/2] codes with matching s4.
 *   workspace: device buffer of at least moet_forward_workspace_size bytes,
 *   256-byte aligned; its contents on entry do not matter.
 * Output tolerance vs the fp64 definition: relative Frobenius error
 * <= 5e-3 and max abs error <= 2e-2 rms(y).  */
typedef struct {
  const uint32_t* sign; /* [E, N, K/32] */
  const uint32_t* mag;  /* [E, N, K/32] */
  const uint8_t* s16;   /* [E, N, K/16] */
  const float* scale_2; /* [E]          */
} moet_planes;

typedef struct {
  const uint8_t* codes; /* [S, N, K/2]  */
  const uint8_t* s4;    /* [S, N, K/16] */
} moet_nvfp4;

size_t moet_forward_workspace_size(int T, int H, int I, int E, int k);

moet_status moet_moe_forward(int T, int H, int I, int E, int k, const uint16_t* x,
                             const int32_t* topk_idx, const float* topk_w,
                             const int32_t* expert_offsets, const int32_t* perm,
                             const moet_planes* fc1, const moet_planes* fc2,
                             const int32_t* delta_slot, int n_slots, const moet_nvfp4* dfc1,
                             const moet_nvfp4* dfc2, const uint8_t* gate_mask, uint16_t* y,
                             void* workspace, size_t ws_bytes, moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_moe_forward_pooled -- moet_moe_forward over a device-resident pool of
 * experts, for layers whose 2-bit planes do not all fit on the GPU.
 * README "Frontier MoE on consumer Blackwell (SM120)", "When the model doesn't
 * fit at all -- the GPU as an expert cache": the GPU holds a cache of hot
 * experts addressed through a slot table read inside the (graph-captured)
 * forward; a routed expert that is not resident contributes zero to y and is
 * counted, so the caller can fetch every missing expert, update the table
 * and replay the step -- which then equals a fully resident forward bit for
 * bit (an expert's arithmetic does not depend on its pool slot).
 *   expert_slot [E] i32: pool slot of expert e, or -1 (not resident); a slot
 *     >= n_pool is a device index error and the expert counts as missing.
 *   fc1/fc2: planes of the n_pool pool slots ([n_pool, 2I, H/32] ... and
 *     scale_2 [n_pool]); all other arguments as for moet_moe_forward (the
 *     delta table stays indexed by expert id).
 *   miss_count: if non-NULL, one u32 to which the number of routed (token,
 *     expert) pairs whose expert is not resident is added (atomically; the
 *     caller resets it).  miss_mask: if non-NULL, u8 [E]; entry e is set to 1
 *     when expert e was routed and is not resident (never cleared here).
 *   Workspace: moet_forward_workspace_size(T, H, I, E, k), as for
 *     moet_moe_forward.
 * With every routed expert resident the result equals moet_moe_forward's on
 * the same weights bit for bit.  */
moet_status moet_moe_forward_pooled(int T, int H, int I, int E, int k, const uint16_t* x,
                                    const int32_t* topk_idx, const float* topk_w,
                                    const int32_t* expert_offsets, const int32_t* perm,
                                    const int32_t* expert_slot, int n_pool,
                                    const moet_planes* fc1, const moet_planes* fc2,
                                    const int32_t* delta_slot, int n_slots, const moet_nvfp4* dfc1,
                                    const moet_nvfp4* dfc2, const uint8_t* gate_mask,
                                    uint32_t* miss_count, uint8_t* miss_mask, uint16_t* y,
                                    void* workspace, size_t ws_bytes, moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_moe_forward_static -- moet_moe_forward for callers that cannot
 * allocate device memory (a plug-in given only its input and output buffers,
 * code inside a runtime whose device allocator belongs to someone else, a C
 * caller with no allocator).  The pages describe no such entry point; it is
 * an addition of this library.  Same arguments and results as
 * moet_moe_forward, without `workspace`/`ws_bytes`: the scratch is a fixed
 * array of MOET_FORWARD_STATIC_SCRATCH_BYTES in the library's device image,
 * present on every GPU that loads the library until the process exits.
 * Nothing is allocated or freed.
 *  - Returns MOET_ERR_WORKSPACE, enqueueing nothing, when the layer needs
 *    more scratch than that (moet_forward_workspace_size(T,H,I,E,k) >
 *    MOET_FORWARD_STATIC_SCRATCH_BYTES); e.g. H=7168, I=2048, E=256, k=8 fits
 *    up to T=13 tokens.
 *  - A call made while `stream` is not being captured looks the array's
 *    device address up (cudaGetSymbolAddress, on the current device), so a
 *    device reset that reloads the library's module is picked up by the next
 *    such call.  A call made during stream capture reuses the address found by
 *    the last call outside capture on that device and returns
 *    MOET_ERR_UNSUPPORTED if there was none: make the first call on a device
 *    before any stream capture.
 *  - Every call uses the same array and leaves its contents behind; calls
 *    that overlap on the GPU race on it, so the caller must serialise them.
 *    No scratch contents need to start at zero. */
#define MOET_FORWARD_STATIC_SCRATCH_BYTES ((size_t)8 << 20)

moet_status moet_moe_forward_static(int T, int H, int I, int E, int k, const uint16_t* x,
                                    const int32_t* topk_idx, const float* topk_w,
                                    const int32_t* expert_offsets, const int32_t* perm,
                                    const moet_planes* fc1, const moet_planes* fc2,
                                    const int32_t* delta_slot, int n_slots, const moet_nvfp4* dfc1,
                                    const moet_nvfp4* dfc2, const uint8_t* gate_mask, uint16_t* y,
                                    moet_stream stream);

/* ------------------------------------------------------------------------
 * moet_debug_wait_expiry -- test control of the forward engines' bounded waits.
 * The two tcgen05 engines (the block-scaled decode engine and the bf16 prefill
 * engine behind moet_moe_forward) hand work between warps through mbarriers;
 * every wait polls at most 2^20 times (each poll suspended for at most about
 * 2 us).  A wait that runs out marks the CTA stuck: every warp role leaves
 * its loop, the copy and MMA issuers wait (bounded) for what they have in
 * flight, TMEM is released, and MOET_ERR_TIMEOUT is recorded for
 * moet_last_device_error; the outputs of that launch are unspecified, the
 * context stays usable.  This control lets a test drive that path:
 *   polls     > 0 lowers the poll bound of every wait to `polls` (a value at
 *             or above the default leaves it unchanged); 0 restores it.
 *   withhold  1 makes CTA 0 of every engine launch skip publishing its first
 *             unit record, so that every wait on that record runs out;
 *             0 (the default) publishes every record.
 * The setting holds for later launches until changed.  Returns
 * MOET_ERR_INVALID_ARG for polls < 0 or withhold not 0/1, MOET_ERR_CUDA if
 * the setting cannot be copied to the current device.  Blocking; not for use
 * during stream capture.  Not a part of the layer computation: the pages
 * describe no such control. */
moet_status moet_debug_wait_expiry(int polls, int withhold);

/* ------------------------------------------------------------------------
 * Kernel timing (tracing aid, off by default).  While enabled, the library
 * records a CUDA event before and after each of its kernel launches on the
 * launching stream (so timings are on-device and per launch; leave it off
 * during CUDA-graph capture).  moet_profile_read synchronises on the
 * recorded events and returns, per kernel kind, the number of launches and
 * their summed duration in milliseconds since the previous read, then
 * clears the record.  At most 8192 launches are kept between reads; later
 * ones are counted in launches[] but not timed (check `timed`).
 *   launches, timed: int[MOET_KERNEL_KINDS]; total_ms: float[MOET_KERNEL_KINDS]. */
typedef enum {
  MOET_K_REQUANT = 0,
  MOET_K_QUANTIZE = 1,
  MOET_K_ROUTE = 2,
  MOET_K_PROLOGUE = 3,
  MOET_K_FC1 = 4,
  MOET_K_FC2 = 5,
  MOET_K_COMBINE = 6,
  MOET_K_TERMS = 7, /* activation -> NVFP4 term expansion of the tensor-core path */
  MOET_K_PROBE = 8, /* moet_sign_bias_probe */
  MOET_KERNEL_KINDS = 9
} moet_kernel_kind;

moet_status moet_profile_enable(int on);
moet_status moet_profile_read(int* launches, int* timed, float* total_ms);

#ifdef __cplusplus
}
#endif
#endif /* MOET_H */
