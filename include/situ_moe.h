/*
 * situ_moe.h -- C ABI of the GB300 (sm_103a) SiTU routed-MoE expert layer.
 *
 * The layer is the Kimi-K3 routed-expert MoE of the TokenSpeed SiTU page
 * (pypi.org/project/tokenspeed-situ, "Supported contract" and "Activation
 * precision (w4a16 vs w4a8)"): precomputed global top-k routing; a permute
 * of the (token, slot) pairs by local expert that drops experts outside the
 * rank's contiguous shard; FC1 gate/up with the SiTU gated activation; FC2;
 * and a top-k-weighted un-permute sum that is a partial output the caller
 * all-reduces across its MoE TP/EP group (this library performs no
 * collective).
 *
 * Conventions, for every entry point:
 *   - Pointers are DEVICE pointers unless stated otherwise, row-major and
 *     contiguous.  Activation, packed-weight, output and workspace pointers
 *     must be 16-byte aligned, block-scale arrays 2-byte aligned, fp32 and
 *     int32 vectors 4-byte aligned (SITU_ERR_MISALIGNED otherwise).  For
 *     situ_moe_permute and situ_moe_quant_mxfp8 every pointer must be
 *     16-byte aligned.  Packed MXFP4 weights (w1, w2) whose bases are
 *     16- but not 32-byte aligned are accepted, but the block-scaled tcgen05
 *     kernels need 32 (their 4-bit tensor maps), so such calls run on the
 *     slower register / f16 kernels.  The caller owns every buffer,
 *     including the workspace; the library allocates no device memory and
 *     keeps no state between calls.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).
 *   - Arguments are validated on the host before anything is launched.  A
 *     non-SITU_OK return means nothing was enqueued, except SITU_ERR_CUDA,
 *     which reports a launch failure (cudaGetLastError) after enqueueing.
 *   - Element formats: E2M1 (FP4) codes are packed two per byte, element 2i
 *     in the low nibble of byte i; UE8M0 scales are one byte 2^(b-127);
 *     E4M3 is the OCP "fn" variant (max 448, no infinities); bf16 is
 *     IEEE binary32 truncated to its upper 16 bits.
 *   - MXFP4 = E2M1 elements with one UE8M0 scale per 32 consecutive
 *     elements along the contraction dimension; NVFP4 = E2M1 with one E4M3
 *     scale per 16 plus an fp32 per-tensor global scale; MXFP8 = E4M3 with
 *     one UE8M0 scale per 32.
 */
#ifndef SITU_MOE_H
#define SITU_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum situ_status {
  SITU_OK = 0,
  SITU_ERR_NULL_ARG = 1,           /* a required pointer is NULL */
  SITU_ERR_BAD_SHAPE = 2,          /* a size is negative, inconsistent or not a supported multiple */
  SITU_ERR_UNSUPPORTED = 3,        /* unsupported (activation, weight) format pair or limit */
  SITU_ERR_WORKSPACE_TOO_SMALL = 4,
  SITU_ERR_CUDA = 5,               /* a CUDA launch or runtime call failed */
  SITU_ERR_MISALIGNED = 6,         /* a pointer is below the alignment its argument requires */
  SITU_ERR_DEVICE_TIMEOUT = 7      /* a kernel gave up a bounded wait (see situ_moe_device_status) */
} situ_status;

typedef enum situ_act_dtype {
  SITU_ACT_BF16 = 0,   /* w4a16: bf16 activations */
  SITU_ACT_MXFP8 = 1,  /* w4a8: MXFP8 activations + per-token hidden_states_scale */
  SITU_ACT_NVFP4 = 2   /* NVFP4 activations with a per-token fp32 global scale */
} situ_act_dtype;

typedef enum situ_weight_dtype {
  SITU_W_MXFP4 = 0,
  SITU_W_NVFP4 = 1
} situ_weight_dtype;

/* Largest supported top-k and local expert count. */
#define SITU_MAX_TOP_K 16
#define SITU_MAX_LOCAL_EXPERTS 4096

/* Human-readable name of a status code (static storage). */
const char* situ_status_string(situ_status s);

/* ------------------------------------------------------------------------
 * situ_moe_permute -- group the (token, slot) pairs by local expert.
 *
 * Defined by TokenSpeed SiTU, "Supported contract": top-k expert IDs stay
 * global (0..num_experts_total-1); experts outside the contiguous shard
 * [local_expert_offset, local_expert_offset + num_local_experts) are
 * filtered out.  Slot s = t*top_k + j of token t is kept when its ID lies in
 * the shard (IDs outside it, including negative ones, are dropped).
 *
 *   topk_ids        int32 [T, top_k]               (input)
 *   expert_counts   int32 [num_local_experts]      kept slots per local expert
 *   expert_offsets  int32 [num_local_experts + 1]  exclusive prefix sum; the last
 *                                                  entry is R, the kept-slot count
 *   permuted_src    int32 [T*top_k]                row r < R holds the slot it came
 *                                                  from; rows are grouped by local
 *                                                  expert and ascending in slot
 *                                                  index within an expert (a stable
 *                                                  order); rows >= R hold -1
 *   slot_to_row     int32 [T*top_k]                row of each slot, -1 if dropped
 *   workspace       device scratch of at least situ_moe_permute_workspace_size()
 *                   bytes; contents on entry are ignored
 *
 * All outputs are bit-exact and deterministic.  T == 0 launches nothing.
 * Errors: NULL_ARG, BAD_SHAPE (T < 0, top_k not in 1..16, local shard not
 * inside [0, num_experts_total), num_local_experts > 4096), MISALIGNED,
 * WORKSPACE_TOO_SMALL, CUDA.
 * --------------------------------------------------------------------- */
size_t situ_moe_permute_workspace_size(int32_t T, int32_t top_k, int32_t num_local_experts);

situ_status situ_moe_permute(const int32_t* topk_ids, int32_t T, int32_t top_k,
                             int32_t num_experts_total, int32_t num_local_experts,
                             int32_t local_expert_offset, int32_t* expert_counts,
                             int32_t* expert_offsets, int32_t* permuted_src,
                             int32_t* slot_to_row, void* workspace, size_t workspace_bytes,
                             void* stream);

/* ------------------------------------------------------------------------
 * situ_moe_permute_noalloc -- situ_moe_permute without a caller workspace.
 *
 * The paper has no counterpart to this call; it is a convenience of this
 * library for callers that cannot allocate device memory where they route
 * tokens.  Examples: a serving engine that hands all device memory to its own
 * pool at start-up, or code in a region where a cudaMalloc would synchronise
 * the device or is not permitted at all.  Such a caller has nowhere to get
 * the permute's scratch from.
 *
 * Inputs, outputs, ordering and errors are those of situ_moe_permute.  The
 * scratch (the per-chunk expert counts) lives in a fixed array inside the
 * library: SITU_NOALLOC_SCRATCH_INTS int32 (4 MiB), which every GPU that
 * loads the library holds until the process exits.  The call never calls
 * cudaMalloc, cudaFree or any other allocating routine.
 *
 * Limit: ceil(T*top_k / 4096) * num_local_experts must not exceed
 * SITU_NOALLOC_SCRATCH_INTS (for 896 local experts: T*top_k up to 4,792,320
 * slots); a larger request returns SITU_ERR_WORKSPACE_TOO_SMALL and launches
 * nothing.
 *
 * The first call on each device looks up the array's device address with
 * that device current (cudaGetSymbolAddress), so make that first call before
 * any stream capture.  The address is cached per device and context: the
 * first call in a context created anew on a device (after cudaDeviceReset,
 * for instance) looks it up again.  All calls share the one array, which
 * keeps whatever the last call left in it; nothing in it has to start at
 * zero, because
 * each call writes every entry it later reads.  Calls whose kernels can
 * overlap on the GPU (different streams, or unordered host threads) race on
 * the array and must be serialised by the caller.
 * --------------------------------------------------------------------- */
#define SITU_NOALLOC_SCRATCH_INTS (1 << 20)
situ_status situ_moe_permute_noalloc(const int32_t* topk_ids, int32_t T, int32_t top_k,
                                     int32_t num_experts_total, int32_t num_local_experts,
                                     int32_t local_expert_offset, int32_t* expert_counts,
                                     int32_t* expert_offsets, int32_t* permuted_src,
                                     int32_t* slot_to_row, void* stream);

/* ------------------------------------------------------------------------
 * situ_moe_route_topk -- the top-k routing of router logits, upstream of
 * situ_moe_permute.
 *
 * The golden reference MoE of TensorRT-LLM PR #17865 (review comment on
 * test_kimi_k3_situ_moe.py, `_reference_moe`) starts from router logits and
 * `routing_method.apply(router_logits)`; TokenSpeed SiTU ("Supported
 * contract") consumes the resulting top-k IDs and weights.  The pages name
 * no routing method; this call implements top-k selection with a softmax:
 *   topk_ids[t, j]      the K largest logits of token t in descending order,
 *                       two equal logits taken lower expert ID first (+0 and
 *                       -0 are equal);
 *   topk_weights[t, j]  renormalize = 1: exp(l_j - m) / sum over the K
 *                       selected of exp(l_i - m), m the largest logit (a
 *                       softmax over the selected logits, the definition the
 *                       layer's routing weights follow); renormalize = 0:
 *                       the same numerator over the sum across all E logits
 *                       (the selected experts' softmax probabilities).
 *
 *   router_logits  fp32  [T, num_experts_total]  (finite values)
 *   topk_ids       int32 [T, top_k]              global expert IDs
 *   topk_weights   fp32  [T, top_k]
 *
 * The IDs are exact (comparisons of the fp32 logits); the weights are fp32
 * (expf and one division, a few ulps from the exactly rounded value).
 * Pointers 4-byte aligned.  T == 0 launches nothing.  Asynchronous on
 * `stream`.  Errors: NULL_ARG, BAD_SHAPE (T < 0, num_experts_total < 1,
 * top_k not in 1..min(16, num_experts_total)), UNSUPPORTED (renormalize
 * not 0 or 1), MISALIGNED, CUDA.
 * --------------------------------------------------------------------- */
situ_status situ_moe_route_topk(const float* router_logits, int32_t T, int32_t num_experts_total,
                                int32_t top_k, int32_t renormalize, int32_t* topk_ids,
                                float* topk_weights, void* stream);

/* ------------------------------------------------------------------------
 * situ_moe_quant_mxfp8 -- quantise bf16 activations to MXFP8 (w4a8 chain).
 *
 * TokenSpeed SiTU, "Activation precision (w4a16 vs w4a8)" and "Supported
 * contract": MXFP8 activations with a per-token hidden_states_scale
 * block-scale tensor.  The pages do not fix the scale rule; this library
 * uses, per token and per 32 consecutive hidden elements, the smallest
 * power of two 2^e (e in [-127, 127]) with amax * 2^-e <= 448, stored as
 * the UE8M0 byte e + 127 (an all-zero block gets byte 0), and rounds each
 * element x * 2^-e to the nearest E4M3 value, ties to even, saturating.
 *
 *   x_bf16          bf16  [T, H]      (input; finite values)
 *   x_e4m3          uint8 [T, H]      E4M3 codes
 *   x_scale_ue8m0   uint8 [T, H/32]   hidden_states_scale
 *
 * Bit-exact.  H must be a positive multiple of 32; T == 0 launches nothing.
 * Errors: NULL_ARG, BAD_SHAPE, MISALIGNED, CUDA.
 * --------------------------------------------------------------------- */
situ_status situ_moe_quant_mxfp8(const void* x_bf16, int32_t T, int32_t H, uint8_t* x_e4m3,
                                 uint8_t* x_scale_ue8m0, void* stream);

/* ------------------------------------------------------------------------
 * situ_moe_quant_nvfp4 -- quantise bf16 activations to NVFP4 with
 * per-token scaling (the NVFP4 variant's hidden_states / hidden_states_scale
 * / hidden_states_gscale).
 *
 * FlashInfer 0.6.18 SM100a+SM103a MoE-LoRA AOT release notes, Summary: the
 * NVFP4 path scales its activations per token (and TRT-LLM-Gen has no fused
 * SiTU GEMM1 for that case).  The pages do not fix the
 * rule; this library uses, per token row, with every step one fp32
 * operation rounded to nearest even:
 *   gscale = amax_row / 2688 (= 6 * 448; 1 for an all-zero row),
 *   scale  = E4M3(amax_16 / (6 * gscale)) per 16 consecutive elements,
 *   code   = E2M1(x / (value(scale) * gscale)), ties to the even code,
 *            saturating at 6 (0 when that divisor is 0).
 *
 *   x_bf16        bf16  [T, H]      (input; finite values; 16-byte aligned)
 *   x_e2m1        uint8 [T, H/2]    packed codes, element 2i in the low nibble
 *                                   (8-byte aligned)
 *   x_scale_e4m3  uint8 [T, H/16]
 *   x_gscale      fp32  [T]
 *
 * Bit-exact.  H must be a positive multiple of 16; T == 0 launches nothing.
 * Asynchronous on `stream`.  Errors: NULL_ARG, BAD_SHAPE, MISALIGNED, CUDA.
 * --------------------------------------------------------------------- */
situ_status situ_moe_quant_nvfp4(const void* x_bf16, int32_t T, int32_t H, uint8_t* x_e2m1,
                                 uint8_t* x_scale_e4m3, float* x_gscale, void* stream);

/* ------------------------------------------------------------------------
 * situ_moe_forward -- the whole routed-expert layer.
 *
 * For each kept pair (t, j) with local expert e = topk_ids[t,j] - offset:
 *   gate_i = g1_alphas[e]    * gs_gate * xs_t * <x_t, W1[e, i, :]>       i <  I
 *   up_i   = g1_alphas_up[e] * gs_up   * xs_t * <x_t, W1[e, I+i, :]>
 *   h_i    = [b*tanh(gate_i/b)*sigmoid(gate_i)] * [bl*tanh(up_i/bl)]
 *            with b = gemm1_alpha[e], bl = gemm1_beta[e]
 *   y      = g2_alphas[e] * gs_2 * H1 W2[e]^T,  H1 = h rounded to bf16
 *            (w4a16, NVFP4) or MXFP8-quantised per 32 along I and
 *            dequantised (w4a8)
 *   out[t] = sum over kept j, ascending, of topk_weights[t,j] * y
 * Sources: the SiTU formula is the golden `_situ_act` in TensorRT-LLM PR
 * #17865 ("bring up Kimi K3 NVFP4 with CUTLASS and cuteDSL MegaMoE SiTU");
 * the per-expert beta / linear beta from gemm1_alpha / gemm1_beta and the
 * up half rescaled by g1_alphas_up / g1_alphas before the tanh are from the
 * FlashInfer 0.6.18 SM100a+SM103a MoE-LoRA AOT release notes ("Changes since
 * 875b7d7"); the FC1-w4a8 + FC2-w4a16 chain with the FC1 fp8 output
 * dequantised before FC2 is TokenSpeed SiTU, "Activation precision".
 * g1_alphas scales both FC1 halves and the up half is further rescaled by
 * g1_alphas_up / g1_alphas, so the net up scale is g1_alphas_up.  A cap
 * b or bl <= 0 switches that factor to its limit (gate*sigmoid(gate), up).
 * gs_* are the NVFP4 per-tensor global scales (1 for MXFP4) and xs_t the
 * NVFP4 per-token activation scale (1 otherwise).  Tokens with no kept
 * slot get out = 0.  W1 rows 0..I-1 are the gate half, I..2I-1 the up half.
 *
 * Supported (act, weight) pairs: (BF16, MXFP4) w4a16, (MXFP8, MXFP4) w4a8,
 * (NVFP4, NVFP4).  Shapes: H and I positive multiples of 32, top_k 1..16,
 * the local shard inside [0, num_experts_total).  MXFP4 weight scale bytes
 * must lie in [2, 252] so that every dequantised weight is a bf16 normal or
 * zero (the layer's synthetic and real checkpoints are far inside this).
 * Representation: the block-scaled tensor-core paths scale every 32 (MXFP4)
 * or 16 (NVFP4) elements on their own, bf16 rows entering as two MXFP8 rows
 * (exact within 2^14 of their block's maximum, an absolute error below
 * 2^-22 of it further down).  The f16 prefill tiles, which take H or I not
 * multiples of 128 and NVFP4 routings above 512 rows per expert, hold an
 * activation row in f16 under one scale for the row and a weight row
 * relative to its largest block scale: activation elements more than 2^-24
 * below their row's maximum, and weight blocks more than 2^-23 below their
 * row's largest block scale, contribute nothing there.  The NVFP4 FC2 on
 * tiles of up to 64 tokens takes the bf16 H1 as f16 under one power of two
 * for the whole call (its largest magnitude brought into [2^14, 2^15)): exact
 * within 2^31 of that maximum, an absolute error below 2^-32 of it further
 * down.  SiTU's capped factors carry an absolute error of a few fp32 ulps
 * of the cap near 0, so a layer whose pre-activations all lie below about
 * 1e-5 of the caps misses the relative parity bar.
 * --------------------------------------------------------------------- */
/* FC1's gated activation (situ_moe_args.activation). */
typedef enum { SITU_ACT_FN_SITU = 0, SITU_ACT_FN_SWIGLU_BIAS = 1 } situ_act_fn;

typedef struct situ_moe_args {
  int32_t T;                      /* tokens */
  int32_t H;                      /* hidden size (FC1 K, FC2 N) */
  int32_t I;                      /* intermediate size (FC1 has 2*I rows) */
  int32_t num_experts_total;      /* global expert count (896 for Kimi-K3) */
  int32_t num_local_experts;      /* E_loc */
  int32_t local_expert_offset;    /* first global ID of the shard */
  int32_t top_k;
  int32_t act_dtype;              /* situ_act_dtype */
  int32_t weight_dtype;           /* situ_weight_dtype */
  const void* hidden_states;      /* bf16 [T, H] (SITU_ACT_BF16) */
  const uint8_t* hidden_states_q; /* E4M3 [T, H] (MXFP8) or packed E2M1 [T, H/2] (NVFP4) */
  const uint8_t* hidden_states_scale;  /* UE8M0 [T, H/32] (MXFP8) or E4M3 [T, H/16] (NVFP4) */
  const float* hidden_states_gscale;   /* fp32 [T] per-token global scale (NVFP4) */
  const int32_t* topk_ids;        /* int32 [T, top_k] global expert IDs */
  const float* topk_weights;      /* fp32 [T, top_k] */
  const uint8_t* w1;              /* packed E2M1 [E_loc, 2I, H/2] */
  const uint8_t* w1_scale;        /* UE8M0 [E_loc, 2I, H/32] or E4M3 [E_loc, 2I, H/16] */
  const float* w1_gscale;         /* fp32 [E_loc, 2] gate / up global scale (NVFP4) */
  const uint8_t* w2;              /* packed E2M1 [E_loc, H, I/2] */
  const uint8_t* w2_scale;        /* UE8M0 [E_loc, H, I/32] or E4M3 [E_loc, H, I/16] */
  const float* w2_gscale;         /* fp32 [E_loc] (NVFP4) */
  const float* gemm1_alpha;       /* fp32 [E_loc] SiTU beta, required */
  const float* gemm1_beta;        /* fp32 [E_loc] SiTU linear beta, required */
  const float* g1_alphas;         /* fp32 [E_loc] or NULL (1) */
  const float* g1_alphas_up;      /* fp32 [E_loc] or NULL (1) */
  const float* g2_alphas;         /* fp32 [E_loc] or NULL (1) */
  void* out;                      /* bf16 [T, H] partial output of this shard */
  const void* scales_packed;      /* optional: situ_moe_pack_scales output for w1_scale /
                                     w2_scale, or NULL (the forward then packs them into its
                                     workspace on every call) */
  int32_t fuse_combine;           /* 0: FC2 writes each kept slot's row Y and a second kernel
                                     forms the weighted sums in ascending slot order
                                     (deterministic).  1: on the block-scaled prefill tiles,
                                     FC2 adds weight * Y straight into an fp32 accumulator
                                     with vector reductions (red.global.add) and a last
                                     kernel rounds it to bf16; this saves the fp32 Y round
                                     trip through HBM, but the order of the additions varies
                                     from run to run, so outputs are reproducible only to
                                     fp32 rounding.  The other paths ignore it. */
  int32_t activation;             /* FC1's gated activation, situ_act_fn: SITU (default; the
                                     caps gemm1_alpha / gemm1_beta) or SWIGLU_BIAS, CUTLASS's
                                     g * sigmoid(alpha * g) * (u + beta) printed beside SiTU in
                                     PR #17865's golden reference, with alpha = gemm1_alpha and
                                     beta = gemm1_beta per local expert (SwiGLU: SITU with both
                                     caps <= 0, or SWIGLU_BIAS with alpha 1, beta 0) */
  int32_t apply_topk_in_fc1;      /* 1: each slot's routing weight scales its H1 row in FC1's
                                     epilogue, before H1 is rounded for FC2, and the
                                     un-permute sum is unweighted (the MegaMoE option of PR
                                     #17865); 0: the weight is applied in the sum */
  int32_t h1_nvfp4;               /* NVFP4 only.  0 (default): H1 stays bf16 and FC2 multiplies
                                     it with the NVFP4 weights.  1: H1, rounded to bf16, is
                                     requantised per token to NVFP4 with the rule of
                                     situ_moe_quant_nvfp4 (the per-token NVFP4 activation
                                     scaling of the FlashInfer 0.6.18 MoE-LoRA AOT notes, as an
                                     unfused quantisation step), and FC2 runs NVFP4 x NVFP4
                                     (kind::mxf4nvf4 on the NVFP4 tiles).  Needs H a
                                     multiple of 256 and I of 128; other shapes and format
                                     pairs: SITU_ERR_UNSUPPORTED. */
  int32_t tactic[2];              /* kernel configuration of FC1 / FC2, as the TokenSpeed SiTU
                                     runtime API's `tactic` pair: -1 = auto, the first valid
                                     configuration.  This library has one configuration per
                                     shape (its path choice), so -1 and 0 both select it; any
                                     other value returns SITU_ERR_UNSUPPORTED. */
} situ_moe_args;

/* Workspace bytes situ_moe_forward needs for these shapes (0 on bad args).
 * It grows with T*top_k: permute arrays, the permuted activations
 * [T*top_k, H] (f16 or E4M3 rows plus scales), the FC1 output [T*top_k, I]
 * and the FC2 output [T*top_k, H] fp32. */
size_t situ_moe_workspace_size(const situ_moe_args* args);

/* Errors: NULL_ARG (args, required pointers, gemm1_alpha / gemm1_beta --
 * the SiTU caps have no default), BAD_SHAPE, UNSUPPORTED (format pair,
 * activation kind, a tactic other than -1 / 0), MISALIGNED,
 * WORKSPACE_TOO_SMALL, CUDA.  T == 0 launches nothing.
 * Debugging aid: with the environment variable SITU_MOE_DEBUG_SYNC set, the
 * call synchronises its stream after every stage and prints the first stage
 * whose kernels failed to stderr (this serialises the call: not for timing). */
situ_status situ_moe_forward(const situ_moe_args* args, void* workspace, size_t workspace_bytes,
                             void* stream);

/* ------------------------------------------------------------------------
 * situ_moe_forward_profiled -- situ_moe_forward plus stage timing events.
 *
 * Enqueues exactly the launches of situ_moe_forward and records, on the same
 * stream, events[0] before the first launch and events[i] after stage i:
 * 1 permute (3 launches), 2 gather, 3 FC1 + SiTU, 4 FC2, 5 combine.  `events`
 * holds SITU_PROFILE_EVENTS cudaEvent_t handles (passed as void*) created by
 * the caller with timing enabled.  Measurement aid only; the pages define no
 * counterpart.  Errors: those of situ_moe_forward, NULL_ARG for a NULL
 * events array.
 * --------------------------------------------------------------------- */
#define SITU_PROFILE_EVENTS 6
situ_status situ_moe_forward_profiled(const situ_moe_args* args, void* workspace,
                                      size_t workspace_bytes, void* stream, void* const* events);

/* ------------------------------------------------------------------------
 * situ_moe_device_status -- outcome of the device-side waits of the last
 * situ_moe_forward enqueued on `stream` with this workspace.
 *
 * The tensor-core GEMM kernels bound every wait on their asynchronous
 * copies and MMAs (200 ms); a CTA that runs out records a nonzero code in
 * a status word inside the workspace and returns, and the kernels after it
 * stop early, so the CUDA context stays usable.  This call waits for
 * `stream`, reads the word (4 bytes, device to host) and returns SITU_OK
 * when it is 0, SITU_ERR_DEVICE_TIMEOUT otherwise; the raw code (which
 * wait gave up first) goes to *code when `code` is not NULL.  `args` must
 * be the shapes the workspace was used with.  Synchronous; the pages
 * define no counterpart.  Errors: NULL_ARG, BAD_SHAPE, CUDA.
 * --------------------------------------------------------------------- */
situ_status situ_moe_device_status(const situ_moe_args* args, const void* workspace, void* stream,
                                   int32_t* code);

/* ------------------------------------------------------------------------
 * situ_moe_wait_selftest -- the bounded wait of the tensor-core kernels,
 * made to run out.
 *
 * Launches one small kernel that waits, with the same bounded mbarrier wait
 * every GEMM kernel of this library uses (200 ms of the GPU's global timer),
 * for a barrier phase that nothing completes.  The wait gives up, records
 * SITU_SELFTEST_WAIT_CODE in *device_status (one int32 in device memory,
 * which the caller sets to 0 first) and the kernel returns: no trap, no
 * hang, and the CUDA context stays usable.  A test of the failure path;
 * the pages define no counterpart.  Asynchronous on `stream`.
 * Errors: NULL_ARG (device_status), MISALIGNED (not 4-byte aligned), CUDA.
 * --------------------------------------------------------------------- */
#define SITU_SELFTEST_WAIT_CODE 99
situ_status situ_moe_wait_selftest(int32_t* device_status, void* stream);

/* ------------------------------------------------------------------------
 * situ_moe_forward_wait_test -- situ_moe_forward with its failure path
 * taken on purpose.
 *
 * A test of the GEMMs' own unwinding, without a fault: the forward runs as
 * situ_moe_forward does, except that in its FC1 (the block-scaled decode
 * tiles, which these arguments must select, else UNSUPPORTED) every bounded
 * wait gives up after wait_us microseconds instead of 200 ms, and CTA 0's
 * copy producer leaves its K stage number skip_stage (counted across its
 * work items) unissued.  The MMA issuer's wait for that stage then runs out:
 * the kernel records its code in the workspace's status word, waits (bounded)
 * for the copies and MMAs it issued, releases its tensor memory and returns;
 * the other CTAs and the kernels after it see the word and skip their work.
 * The output is then undefined and situ_moe_device_status reports
 * SITU_ERR_DEVICE_TIMEOUT; the next situ_moe_forward with the same
 * workspace clears the word and runs normally.  Asynchronous on `stream`.
 * The pages define no counterpart.  Errors: those of situ_moe_forward,
 * BAD_SHAPE (skip_stage < 0, wait_us outside 1..1000000), UNSUPPORTED.
 * --------------------------------------------------------------------- */
situ_status situ_moe_forward_wait_test(const situ_moe_args* args, void* workspace, size_t workspace_bytes,
                                       void* stream, int32_t skip_stage, int32_t wait_us);

/* ------------------------------------------------------------------------
 * situ_tc_peak -- dense throughput of one tensor-core MMA kind on this GPU.
 *
 * Enqueues one kernel with one CTA per SM.  Each CTA fills a 128-row A tile
 * and a 256-row B tile in shared memory (a fixed byte pattern, scales 1.0),
 * then issues `mmas_per_sm` MMAs of M = 128, N = 256 into one TMEM
 * accumulator back to back, as a GEMM's K loop does but without memory
 * traffic:
 *   SITU_TC_MXF8F6F4  tcgen05.mma.kind::mxf8f6f4.block_scale, E4M3 x E2M1
 *                     with UE8M0 per 32, K = 32 (the MXFP4 GEMMs);
 *   SITU_TC_MXF4NVF4  kind::mxf4nvf4.block_scale.scale_vec::4X, E2M1 x E2M1
 *                     with E4M3 per 16, K = 64 (the NVFP4 FC1);
 *   SITU_TC_BF16      kind::f16 with bf16 operands, K = 16 (the NVFP4 FC2).
 * *flops receives the dense FLOPs of the launch (2*M*N*K per MMA, times
 * mmas_per_sm and the SM count); time the launch with events on `stream`
 * to get the rate.  The final wait is bounded: if it runs out the kernel
 * records 98 in *device_status (one int32 in device memory that the caller
 * sets to 0) and returns.  A measurement aid: the pages define no
 * counterpart; the roofline of each GEMM is taken against its own kind.
 * Errors: NULL_ARG, MISALIGNED (device_status not 4-byte aligned),
 * UNSUPPORTED (kind), BAD_SHAPE (mmas_per_sm not a positive multiple of 4),
 * CUDA.
 * --------------------------------------------------------------------- */
typedef enum { SITU_TC_MXF8F6F4 = 0, SITU_TC_MXF4NVF4 = 1, SITU_TC_BF16 = 2 } situ_tc_kind;
situ_status situ_tc_peak(int32_t kind, int32_t mmas_per_sm, int32_t* device_status, double* flops,
                         void* stream);

/* ------------------------------------------------------------------------
 * situ_moe_forward_launches -- the number of kernels situ_moe_forward
 * enqueues for these arguments (0 for T = 0, -1 when validation fails),
 * e.g. to size a CUDA graph or to count device work.  Host-only; the pages
 * define no counterpart.
 * --------------------------------------------------------------------- */
int32_t situ_moe_forward_launches(const situ_moe_args* args);

/* ------------------------------------------------------------------------
 * situ_moe_packed_scales_size / situ_moe_pack_scales -- the weight scales
 * rearranged for the block-scaled tensor-core GEMMs.
 *
 * The block-scaled GEMMs read each stage's weight scales as contiguous
 * blocks laid out as the tensor memory copy expects.  MXFP4 (the w4a8
 * prefill tiles, and the decode tiles of bf16 and MXFP8 activations): per
 * (local expert, weight tile, 128 elements of K) the UE8M0 bytes of the
 * tile's rows; the buffer holds four such packings (the prefill and the
 * decode tiles of FC1 and of FC2).  NVFP4 (the tiles of NVFP4
 * activations): per (local expert, 128 gate + 128 up rows, 256 elements of
 * K) eight blocks of the E4M3 bytes, one per K = 64 MMA and W1 half; then
 * the same for W2 in tiles of 256 rows of H (two halves of 128) and stages
 * of 256 elements of I (the FC2 of a requantised NVFP4 H1, h1_nvfp4).  Packing depends only on w1_scale, w2_scale, num_local_experts, H
 * and I, so it is done once per weight set; pass the result as
 * args->scales_packed.  Without it the forward packs into its workspace on
 * every call (same result, about 25% more HBM traffic for a decode step).
 * The size is 0 (and pack_scales returns UNSUPPORTED) unless weight_dtype
 * is MXFP4 with H and I multiples of 128, or NVFP4 with H a multiple of 256
 * and I of 128.  `packed` is a device buffer
 * of at least that many bytes, 16-byte aligned, owned by the caller;
 * asynchronous on `stream`.  A layout of this library, not of the pages.
 * Errors: NULL_ARG, BAD_SHAPE, UNSUPPORTED, MISALIGNED, WORKSPACE_TOO_SMALL
 * (packed_bytes too small), CUDA.
 * --------------------------------------------------------------------- */
size_t situ_moe_packed_scales_size(const situ_moe_args* args);
situ_status situ_moe_pack_scales(const situ_moe_args* args, void* packed, size_t packed_bytes,
                                 void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SITU_MOE_H */
