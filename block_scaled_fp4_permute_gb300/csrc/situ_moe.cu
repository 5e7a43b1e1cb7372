// situ_moe.cu -- the C ABI (include/situ_moe.h): host-side validation,
// workspace layout and the launch sequence of the layer.
//
// situ_moe_forward enqueues, on the caller's stream:
//   permute (1 launch up to 4,096 slots, else 3) -> gather -> FC1 (+SiTU)
//   -> FC2 -> combine.
// No host synchronisation: the number of kept rows and the GEMM token tiles
// live on the device (written by the permute) and every later kernel reads
// them there; grids are sized for the worst case and surplus CTAs exit.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "../../include/situ_moe.h"
#include "situ_internal.h"

using namespace situ;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned_to(const void* p, uintptr_t a) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool aligned16(const void* p) { return aligned_to(p, 16); }

struct Layout {
  size_t counts, offsets, tile_offsets, tile_info, meta, psrc, s2r, blk, h1, h1f, y;
  size_t x16, x16s, h16, h16s, xsp, hsp, wsp, wxs, whs, ys, xg, hq, hqs, hg, t2off, t2info, total;
};

// Decode-like routings (about six or fewer rows per expert) take the
// 8-token-tile path when its shared-memory staging fits; everything else a
// tcgen05 prefill path.
bool decode_like(const situ_moe_args* a) {
  return (double)a->T * a->top_k / (double)a->num_experts_total <= 6.0;
}
constexpr size_t kMaxDecodeSmem = 220 * 1024;
bool takes_decode_path(const situ_moe_args* a) {
  const bool nv = a->weight_dtype == SITU_W_NVFP4;
  return decode_like(a) && fcd_smem_bytes(a->H, nv) <= kMaxDecodeSmem && fcd_smem_bytes(a->I, nv) <= kMaxDecodeSmem;
}
// shapes of the block-scaled prefill path (w4a8, K multiples of 128)
bool block_scaled_shapes(const situ_moe_args* a) {
  return a->weight_dtype == SITU_W_MXFP4 && a->H % 128 == 0 && a->I % 128 == 0;
}
// decode-like routings with bf16 or MXFP8 activations on MXFP4 weights of
// those shapes: the block-scaled decode tiles (weights on the MMA M side)
bool fcw_shapes(const situ_moe_args* a) {
  return decode_like(a) && block_scaled_shapes(a) &&
         (a->act_dtype == SITU_ACT_BF16 || a->act_dtype == SITU_ACT_MXFP8);
}
// NVFP4 weights whose FC1 fits the NVFP4 decode tiles (stages of 256
// elements of H, gate / up tiles of 128 rows)
bool nv_tile_shapes(const situ_moe_args* a) {
  return a->weight_dtype == SITU_W_NVFP4 && a->H % 256 == 0 && a->I % 128 == 0;
}
// NVFP4 activations on those weights with up to 512 kept rows per expert on
// average: FC1 on the block-scaled 16-token tiles (kind::mxf4nvf4), FC2 with
// the weights expanded to bf16 (kind::f16) on the same tiles or on 64-token
// ones.  Each tile streams its expert's weights, which beats the 128-token
// f16 prefill tiles (whose dequantisation runs per tile over mostly empty
// rows) until the experts hold a few hundred rows.
constexpr double kNvTileMaxRowsPerExpert = 512.0;
bool fcw_nv_shapes(const situ_moe_args* a) {
  return (double)a->T * a->top_k / (double)a->num_experts_total <= kNvTileMaxRowsPerExpert && nv_tile_shapes(a) &&
         a->act_dtype == SITU_ACT_NVFP4;
}
// Above 16 rows per expert on average the NVFP4 tiles are 64 tokens wide:
// a K stage of these tiles takes about as long with 64 tokens as with 16
// (measured on both GEMMs), so wider tiles cut the stages and the weight
// re-reads per weight byte.
constexpr int kNvWideTile = 64;
bool nv_wide(const situ_moe_args* a) {
  return fcw_nv_shapes(a) && (double)a->T * a->top_k / (double)a->num_experts_total > 16.0;
}
// Above 64 rows per expert FC2 takes 128-token tiles of a second tile table:
// its converter warps expand an expert's weights once per tile, so wider
// tiles expand them fewer times.
constexpr int kNvFc2WideTile = 128;
bool nv_wide_fc2(const situ_moe_args* a) {
  return fcw_nv_shapes(a) && (double)a->T * a->top_k / (double)a->num_experts_total > 64.0;
}
// prefill-sized routings with MXFP8 or bf16 activations on MXFP4 weights of
// those shapes: the block-scaled prefill tiles (bf16 rows as hi + lo)
bool takes_block_scaled_path(const situ_moe_args* a) {
  return (a->act_dtype == SITU_ACT_MXFP8 || a->act_dtype == SITU_ACT_BF16) && block_scaled_shapes(a) &&
         !takes_decode_path(a);
}
// packed weight scales: [FC1 prefill tiles | FC2 prefill tiles | FC1 decode
// tiles | FC2 decode tiles]
size_t packed_fc1_bytes(const situ_moe_args* a) {
  return fcq_packed_scale_bytes(a->num_local_experts, a->H, a->I, true);
}
size_t packed_fc2_bytes(const situ_moe_args* a) {
  return fcq_packed_scale_bytes(a->num_local_experts, a->H, a->I, false);
}
size_t packed_fc1d_bytes(const situ_moe_args* a) {
  return packed_scale_bytes(a->num_local_experts, a->H, a->I, true, fcw_n_rows(true));
}
size_t packed_fc2d_bytes(const situ_moe_args* a) {
  return packed_scale_bytes(a->num_local_experts, a->H, a->I, false, fcw_n_rows(false));
}
// NVFP4: two packings, the FC1 tiles and the FC2 tiles of the requantised
// H1 (h1_nvfp4)
size_t packed_nv1_bytes(const situ_moe_args* a) { return packed_scale_bytes_nv(a->num_local_experts, a->H, a->I); }
size_t packed_total_bytes(const situ_moe_args* a) {
  if (a->weight_dtype == SITU_W_NVFP4)
    return packed_nv1_bytes(a) + packed_scale_bytes_nv2(a->num_local_experts, a->H, a->I);
  return packed_fc1_bytes(a) + packed_fc2_bytes(a) + packed_fc1d_bytes(a) + packed_fc2d_bytes(a);
}
// the packings into one buffer (layout above); fc2_nv: the NVFP4 FC2 one
// too (always for the caller's buffer; inside a call only when H1 is
// requantised)
cudaError_t pack_all_scales(const situ_moe_args* a, uint8_t* dst, cudaStream_t st, bool fc2_nv = true) {
  const int E = a->num_local_experts;
  if (a->weight_dtype == SITU_W_NVFP4) {
    cudaError_t e = launch_pack_scales_nv(a->w1_scale, E, a->H, a->I, dst, st);
    if (e == cudaSuccess && fc2_nv) e = launch_pack_scales_nv2(a->w2_scale, E, a->H, a->I, dst + packed_nv1_bytes(a), st);
    return e;
  }
  cudaError_t e = launch_pack_scales(a->w1_scale, E, a->H, a->I, true, dst, st);
  dst += packed_fc1_bytes(a);
  if (e == cudaSuccess) e = launch_pack_scales(a->w2_scale, E, a->H, a->I, false, dst, st);
  dst += packed_fc2_bytes(a);
  if (e == cudaSuccess) e = launch_pack_scales_nh(a->w1_scale, E, a->H, a->I, true, fcw_n_rows(true), dst, st);
  dst += packed_fc1d_bytes(a);
  if (e == cudaSuccess) e = launch_pack_scales_nh(a->w2_scale, E, a->H, a->I, false, fcw_n_rows(false), dst, st);
  return e;
}
long max_prefill_tiles(const situ_moe_args* a) {
  return (long)a->T * a->top_k / fcp_token_tile() + a->num_local_experts + 1;
}

Layout make_layout(const situ_moe_args* a) {
  Layout L;
  size_t o = 0;
  const size_t S = (size_t)a->T * (size_t)a->top_k;
  const size_t E = (size_t)a->num_local_experts;
  auto take = [&](size_t bytes) { size_t at = o; o += align_up(bytes > 0 ? bytes : 1); return at; };
  L.counts = take(4 * E);
  L.offsets = take(4 * (E + 1));
  L.tile_offsets = take(4 * (E + 1));
  L.tile_info = take(8 * (S / kDecodeTileTokens + E + 2));   // any tile width >= 8
  L.meta = take(16);
  L.psrc = take(4 * S);
  L.s2r = take(4 * S);
  L.blk = take(permute_scratch_bytes(a->T, a->top_k, a->num_local_experts));
  L.h1 = take(2 * S * (size_t)a->I);
  // NVFP4 tiles with bf16 H1: its scaled f16 copy for the FC2's f16 operands
  L.h1f = take(fcw_nv_shapes(a) && a->h1_nvfp4 == 0 ? 2 * S * (size_t)a->I : 0);
  L.y = take(4 * S * (size_t)a->H);
  // decode path: f16 block rows of the input and of H1
  L.x16 = take(2 * S * (size_t)pad128(a->H));
  L.x16s = take(4 * S * (size_t)(pad128(a->H) / 32));
  L.h16 = take(2 * S * (size_t)pad128(a->I));
  L.h16s = take(4 * S * (size_t)(pad128(a->I) / 32));
  // block-scaled path: scale blocks of the token tiles (FC1 input, H1), and
  // the packed weight scales when the caller keeps none
  const bool bs = takes_block_scaled_path(a);
  const long tiles = max_prefill_tiles(a);
  const size_t nblk = a->act_dtype == SITU_ACT_BF16 ? 2 : 1;   // hi and lo blocks for bf16
  L.xsp = take(bs ? nblk * fcq_act_scale_bytes(tiles, a->H) : 0);
  L.hsp = take(bs ? nblk * fcq_act_scale_bytes(tiles, a->I) : 0);
  L.ys = take(bs ? S * (size_t)(a->H / 32) : 0);   // scale bytes of the f16 Y rows
  const bool w = fcw_shapes(a), wnv = fcw_nv_shapes(a);
  L.wsp = take((bs || w || wnv) && !a->scales_packed ? packed_total_bytes(a) : 0);
  // decode tiles: hi / lo scale rows of the input and of H1 (the E4M3 rows
  // reuse the x16 / h16 regions); NVFP4 tiles: the input's E4M3 scales in
  // 16-byte chunks per 64 elements (its packed codes reuse x16) and per-row
  // global scales
  L.wxs = take(w ? 2 * S * (size_t)fcw_scale_stride(a->H) : wnv ? S * (size_t)(a->H / 4) : 0);
  L.whs = take(w ? 2 * S * (size_t)fcw_scale_stride(a->I) : 0);
  L.xg = take(wnv ? 4 * S : 0);
  // H1 requantised to NVFP4: packed codes, scales (chunks of 16 bytes per 64
  // elements, or rows of I/16 bytes), global scales
  const bool h1nv = a->h1_nvfp4 != 0;
  L.hq = take(h1nv ? S * (size_t)(a->I / 2) : 0);
  L.hqs = take(h1nv ? S * (size_t)(a->I / 4) : 0);
  L.hg = take(h1nv ? 4 * S : 0);
  // NVFP4 FC2 on 128-token tiles: its own tile table
  const bool wide2 = nv_wide_fc2(a);
  L.t2off = take(wide2 ? 4 * (E + 1) : 0);
  L.t2info = take(wide2 ? 8 * (S / kNvFc2WideTile + E + 2) : 0);
  L.total = o;
  return L;
}

situ_status check_routing(int32_t T, int32_t top_k, int32_t E_total, int32_t E_loc, int32_t off) {
  if (T < 0 || top_k < 1 || top_k > SITU_MAX_TOP_K) return SITU_ERR_BAD_SHAPE;
  if (E_loc < 1 || E_loc > SITU_MAX_LOCAL_EXPERTS || off < 0 || E_total < 1 ||
      (int64_t)off + E_loc > (int64_t)E_total)
    return SITU_ERR_BAD_SHAPE;
  if ((int64_t)T * top_k > (int64_t)0x7FFFFFFF) return SITU_ERR_BAD_SHAPE;
  return SITU_OK;
}

situ_status validate(const situ_moe_args* a) {
  if (!a) return SITU_ERR_NULL_ARG;
  situ_status s = check_routing(a->T, a->top_k, a->num_experts_total, a->num_local_experts,
                                a->local_expert_offset);
  if (s != SITU_OK) return s;
  if (a->H <= 0 || a->I <= 0 || a->H % 32 || a->I % 32) return SITU_ERR_BAD_SHAPE;
  const bool w4a16 = a->act_dtype == SITU_ACT_BF16 && a->weight_dtype == SITU_W_MXFP4;
  const bool w4a8 = a->act_dtype == SITU_ACT_MXFP8 && a->weight_dtype == SITU_W_MXFP4;
  const bool nv = a->act_dtype == SITU_ACT_NVFP4 && a->weight_dtype == SITU_W_NVFP4;
  if (!(w4a16 || w4a8 || nv)) return SITU_ERR_UNSUPPORTED;
  if (a->activation != SITU_ACT_FN_SITU && a->activation != SITU_ACT_FN_SWIGLU_BIAS) return SITU_ERR_UNSUPPORTED;
  // the requantised NVFP4 H1 is an option of the NVFP4 chain on the shapes of
  // its tiles (H a multiple of 256, I of 128), whichever routing size
  if (a->h1_nvfp4 != 0 && (a->h1_nvfp4 != 1 || !nv || !nv_tile_shapes(a))) return SITU_ERR_UNSUPPORTED;
  // one configuration per shape: -1 (auto) or 0 (the first valid one) select it
  for (int g = 0; g < 2; ++g)
    if (a->tactic[g] != -1 && a->tactic[g] != 0) return SITU_ERR_UNSUPPORTED;
  if (a->T == 0) return SITU_OK;
  if (!a->topk_ids || !a->topk_weights || !a->w1 || !a->w1_scale || !a->w2 || !a->w2_scale ||
      !a->gemm1_alpha || !a->gemm1_beta || !a->out)
    return SITU_ERR_NULL_ARG;
  if (w4a16 && !a->hidden_states) return SITU_ERR_NULL_ARG;
  if ((w4a8 || nv) && (!a->hidden_states_q || !a->hidden_states_scale)) return SITU_ERR_NULL_ARG;
  if (nv && (!a->hidden_states_gscale || !a->w1_gscale || !a->w2_gscale)) return SITU_ERR_NULL_ARG;
  // vector-loaded tensors need 16 bytes, scale rows 2 (NVFP4 reads scale
  // pairs), fp32 / int32 vectors 4
  const void* p16[] = {a->hidden_states, a->hidden_states_q, a->w1, a->w2, a->out};
  const void* p4[] = {a->hidden_states_gscale, a->topk_ids, a->topk_weights, a->w1_gscale,
                      a->w2_gscale, a->gemm1_alpha, a->gemm1_beta, a->g1_alphas,
                      a->g1_alphas_up, a->g2_alphas};
  for (const void* p : p16)
    if (!aligned_to(p, 16)) return SITU_ERR_MISALIGNED;
  for (const void* p : p4)
    if (!aligned_to(p, 4)) return SITU_ERR_MISALIGNED;
  if (!aligned_to(a->w1_scale, 2) || !aligned_to(a->w2_scale, 2)) return SITU_ERR_MISALIGNED;
  if (!aligned_to(a->scales_packed, 16)) return SITU_ERR_MISALIGNED;
  return SITU_OK;
}


situ_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SITU_OK : SITU_ERR_CUDA; }

}  // namespace

extern "C" {

const char* situ_status_string(situ_status s) {
  switch (s) {
    case SITU_OK: return "SITU_OK";
    case SITU_ERR_NULL_ARG: return "SITU_ERR_NULL_ARG: a required pointer is NULL";
    case SITU_ERR_BAD_SHAPE: return "SITU_ERR_BAD_SHAPE: unsupported or inconsistent sizes";
    case SITU_ERR_UNSUPPORTED: return "SITU_ERR_UNSUPPORTED: unsupported format pair";
    case SITU_ERR_WORKSPACE_TOO_SMALL: return "SITU_ERR_WORKSPACE_TOO_SMALL";
    case SITU_ERR_CUDA: return "SITU_ERR_CUDA: a CUDA launch or call failed";
    case SITU_ERR_MISALIGNED: return "SITU_ERR_MISALIGNED: a pointer is below the alignment its argument requires";
    case SITU_ERR_DEVICE_TIMEOUT: return "SITU_ERR_DEVICE_TIMEOUT: a kernel gave up a bounded wait";
  }
  return "unknown situ_status";
}

size_t situ_moe_permute_workspace_size(int32_t T, int32_t top_k, int32_t num_local_experts) {
  if (T < 0 || top_k < 1 || num_local_experts < 1) return 0;
  return permute_scratch_bytes(T, top_k, num_local_experts);
}

situ_status situ_moe_permute(const int32_t* topk_ids, int32_t T, int32_t top_k,
                             int32_t num_experts_total, int32_t num_local_experts,
                             int32_t local_expert_offset, int32_t* expert_counts,
                             int32_t* expert_offsets, int32_t* permuted_src,
                             int32_t* slot_to_row, void* workspace, size_t workspace_bytes,
                             void* stream) {
  situ_status s = check_routing(T, top_k, num_experts_total, num_local_experts, local_expert_offset);
  if (s != SITU_OK) return s;
  if (T == 0) return SITU_OK;
  if (!topk_ids || !expert_counts || !expert_offsets || !permuted_src || !slot_to_row || !workspace)
    return SITU_ERR_NULL_ARG;
  const void* ptrs[] = {topk_ids, expert_counts, expert_offsets, permuted_src, slot_to_row, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return SITU_ERR_MISALIGNED;
  if (workspace_bytes < permute_scratch_bytes(T, top_k, num_local_experts))
    return SITU_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(launch_permute(topk_ids, T, top_k, num_local_experts, local_expert_offset, 1,
                                    expert_counts, expert_offsets, nullptr, nullptr, permuted_src,
                                    slot_to_row, nullptr, (int32_t*)workspace,
                                    (cudaStream_t)stream));
}

situ_status situ_moe_quant_mxfp8(const void* x_bf16, int32_t T, int32_t H, uint8_t* x_e4m3,
                                 uint8_t* x_scale_ue8m0, void* stream) {
  if (T < 0 || H <= 0 || H % 32) return SITU_ERR_BAD_SHAPE;
  if (T == 0) return SITU_OK;
  if (!x_bf16 || !x_e4m3 || !x_scale_ue8m0) return SITU_ERR_NULL_ARG;
  if (!aligned16(x_bf16) || !aligned16(x_e4m3) || !aligned16(x_scale_ue8m0)) return SITU_ERR_MISALIGNED;
  return cuda_status(launch_quant_mxfp8(x_bf16, T, H, x_e4m3, x_scale_ue8m0, (cudaStream_t)stream));
}

situ_status situ_moe_quant_nvfp4(const void* x_bf16, int32_t T, int32_t H, uint8_t* x_e2m1,
                                 uint8_t* x_scale_e4m3, float* x_gscale, void* stream) {
  if (T < 0 || H <= 0 || H % 16) return SITU_ERR_BAD_SHAPE;
  if (T == 0) return SITU_OK;
  if (!x_bf16 || !x_e2m1 || !x_scale_e4m3 || !x_gscale) return SITU_ERR_NULL_ARG;
  if (!aligned16(x_bf16) || !aligned_to(x_e2m1, 8) || !aligned_to(x_gscale, 4)) return SITU_ERR_MISALIGNED;
  return cuda_status(
      launch_quant_nvfp4(x_bf16, T, H, x_e2m1, x_scale_e4m3, x_gscale, (cudaStream_t)stream));
}

size_t situ_moe_workspace_size(const situ_moe_args* args) {
  if (!args) return 0;
  if (check_routing(args->T, args->top_k, args->num_experts_total, args->num_local_experts,
                    args->local_expert_offset) != SITU_OK || args->H <= 0 || args->I <= 0)
    return 0;
  return make_layout(args).total;
}

// The failure-path test's injection into the FC1 of the block-scaled decode
// tiles (situ_moe_forward_wait_test); null for every other call.
struct WaitTest {
  unsigned long long wait_ns;
  int skip_stage;
};

static situ_status forward_impl(const situ_moe_args* a, void* workspace, size_t workspace_bytes,
                                void* stream, void* const* events, const WaitTest* wt = nullptr) {
  situ_status s = validate(a);
  if (s != SITU_OK) return s;
  if (a->T == 0) return SITU_OK;
  if (!workspace) return SITU_ERR_NULL_ARG;
  if (!aligned16(workspace)) return SITU_ERR_MISALIGNED;
  const Layout L = make_layout(a);
  if (workspace_bytes < L.total) return SITU_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  int32_t* counts = (int32_t*)(ws + L.counts);
  int32_t* offsets = (int32_t*)(ws + L.offsets);
  int32_t* tile_offsets = (int32_t*)(ws + L.tile_offsets);
  int2* tile_info = (int2*)(ws + L.tile_info);
  int32_t* meta = (int32_t*)(ws + L.meta);
  int32_t* psrc = (int32_t*)(ws + L.psrc);
  int32_t* s2r = (int32_t*)(ws + L.s2r);
  uint16_t* h1 = (uint16_t*)(ws + L.h1);
  float* y = (float*)(ws + L.y);
  const bool nv = a->weight_dtype == SITU_W_NVFP4;
  const bool fcw = fcw_shapes(a) && fcq_supported(a->H, a->I, a->w1, a->w2);
  const bool fcwnv = fcw_nv_shapes(a);
  const bool decode_path = !fcw && !fcwnv && takes_decode_path(a);
  const int tile_n = fcwnv ? (nv_wide(a) ? kNvWideTile : fcw_token_tile())
                     : fcw ? fcw_token_tile() : decode_path ? kDecodeTileTokens : fcp_token_tile();
  const long S = (long)a->T * a->top_k;
  const long max_tiles = S / tile_n + a->num_local_experts + 1;
  // SITU_MOE_DEBUG_SYNC set: synchronise after every stage and name the
  // first one whose kernels failed (a debugging aid; it serialises the call)
  static const bool debug_sync = std::getenv("SITU_MOE_DEBUG_SYNC") != nullptr;
  auto mark = [&](int i) {
    if (events) cudaEventRecord((cudaEvent_t)events[i], st);
    if (debug_sync && i > 0) {
      static const char* names[] = {"start", "permute", "gather", "FC1", "FC2", "combine"};
      const cudaError_t e = cudaStreamSynchronize(st);
      if (e != cudaSuccess)
        std::fprintf(stderr, "situ_moe_forward: stage %s failed: %s\n", i < 6 ? names[i] : "?",
                     cudaGetErrorString(e));
    }
  };

  bool fused = false;   // FC2 adds into the output accumulator (block-scaled prefill only)
  bool y16 = false;     // FC2 writes Y as f16 rows + scale bytes (block-scaled prefill)
  mark(0);
  cudaError_t err = launch_permute(a->topk_ids, a->T, a->top_k, a->num_local_experts,
                                   a->local_expert_offset, tile_n, counts, offsets, tile_offsets,
                                   tile_info, psrc, s2r, meta, (int32_t*)(ws + L.blk), st);
  const bool h1nv = a->h1_nvfp4 != 0;
  if (err == cudaSuccess && fcwnv && nv_wide_fc2(a) && !h1nv)
    err = launch_tile_table(offsets, a->num_local_experts, kNvFc2WideTile, (int32_t*)(ws + L.t2off),
                            (int2*)(ws + L.t2info), st);
  if (err != cudaSuccess) return SITU_ERR_CUDA;
  mark(1);

  // the packed weight scales of the block-scaled GEMMs: the caller's, or
  // packed into the workspace by this call
  auto packed_scales = [&](const uint8_t*& wsp1, const uint8_t*& wsp2, const uint8_t*& wsp3,
                           const uint8_t*& wsp4) -> cudaError_t {
    wsp1 = (const uint8_t*)a->scales_packed;
    if (!wsp1) {
      cudaError_t e2 = pack_all_scales(a, ws + L.wsp, st, h1nv);
      if (e2 != cudaSuccess) return e2;
      wsp1 = ws + L.wsp;
    }
    wsp2 = wsp1 + packed_fc1_bytes(a);
    wsp3 = wsp2 + packed_fc2_bytes(a);
    wsp4 = wsp3 + packed_fc1d_bytes(a);
    return cudaSuccess;
  };

  if (fcw) {
    // 16-token tiles on the block-scaled tensor cores, weights on the MMA M
    // side: token rows as E4M3 (bf16 as interleaved hi / lo rows), FC1
    // (+SiTU) writing H1 in the same form, FC2
    const uint8_t *wsp1, *wsp2, *wsp3, *wsp4;
    if ((err = packed_scales(wsp1, wsp2, wsp3, wsp4)) != cudaSuccess) return SITU_ERR_CUDA;
    const bool lo = a->act_dtype == SITU_ACT_BF16;
    GatherHLParams g;
    std::memset(&g, 0, sizeof(g));
    g.act = a->act_dtype;
    g.x_bf16 = a->hidden_states;
    g.x_q = a->hidden_states_q;
    g.x_s = a->hidden_states_scale;
    g.permuted_src = psrc;
    g.slot_to_row = s2r;
    g.T = a->T;
    g.meta = meta;
    g.top_k = a->top_k;
    g.K = a->H;
    g.S = S;
    g.x = ws + L.x16;
    g.xs = ws + L.wxs;
    g.s_stride = fcw_scale_stride(a->H);
    if ((err = launch_gather_hl(g, st)) != cudaSuccess) return SITU_ERR_CUDA;
    mark(2);
    FcwParams w;
    std::memset(&w, 0, sizeof(w));
    w.offsets = offsets;
    w.tile_offsets = tile_offsets;
    w.tile_info = tile_info;
    w.E_loc = a->num_local_experts;
    w.I = a->I;
    w.err = meta + 2;
    w.wsp = wsp3;
    w.Mtot = 2 * a->I;
    w.K = a->H;
    w.n_ntiles = (a->I + fcw_n_rows(true) - 1) / fcw_n_rows(true);
    w.beta = a->gemm1_alpha;
    w.beta_lin = a->gemm1_beta;
    w.alpha_g = a->g1_alphas;
    w.alpha_u = a->g1_alphas_up;
    w.act_kind = a->activation;
    w.topk_fc1 = a->apply_topk_in_fc1 != 0;
    w.permuted_src = psrc;
    w.topk_weights = a->topk_weights;
    w.h = ws + L.h16;
    w.hs = ws + L.whs;
    w.hs_stride = fcw_scale_stride(a->I);
    if (wt) {
      w.wait_ns = wt->wait_ns;
      w.skip_stage1 = wt->skip_stage + 1;
    }
    if ((err = launch_fcw(w, a->w1, g.x, g.xs, S, a->num_local_experts, true, lo, max_tiles, st)) != cudaSuccess)
      return SITU_ERR_CUDA;
    w.wait_ns = 0;
    w.skip_stage1 = 0;
    mark(3);
    w.wsp = wsp4;
    w.Mtot = a->H;
    w.K = a->I;
    w.n_ntiles = (a->H + fcw_n_rows(false) - 1) / fcw_n_rows(false);
    w.alpha2 = a->g2_alphas;
    w.y_out = y;
    if ((err = launch_fcw(w, a->w2, w.h, w.hs, S, a->num_local_experts, false, lo, max_tiles, st)) != cudaSuccess)
      return SITU_ERR_CUDA;
    mark(4);
  } else if (fcwnv) {
    // NVFP4 at decode: FC1 (+SiTU) on 16- or 64-token block-scaled tiles
    // with both operands E2M1 (kind::mxf4nvf4), writing H1 as bf16 rows; FC2
    // on the same tiles with the weights expanded to f16 in TMEM, or on
    // 128-token tiles expanded to bf16 in shared memory (kind::f16)
    const uint8_t *wsp1, *wsp2, *wsp3, *wsp4;
    if ((err = packed_scales(wsp1, wsp2, wsp3, wsp4)) != cudaSuccess) return SITU_ERR_CUDA;
    GatherHLParams g;
    std::memset(&g, 0, sizeof(g));
    g.act = SITU_ACT_NVFP4;
    g.x_q = a->hidden_states_q;
    g.x_s = a->hidden_states_scale;
    g.x_gs = a->hidden_states_gscale;
    g.xg = (float*)(ws + L.xg);
    g.permuted_src = psrc;
    g.slot_to_row = s2r;   // by token: each row read once for all its slots
    g.T = a->T;
    g.meta = meta;
    g.top_k = a->top_k;
    g.K = a->H;
    g.S = S;
    g.x = ws + L.x16;
    g.xs = ws + L.wxs;
    if ((err = launch_gather_hl(g, st)) != cudaSuccess) return SITU_ERR_CUDA;
    mark(2);
    FcwParams w;
    std::memset(&w, 0, sizeof(w));
    w.offsets = offsets;
    w.tile_offsets = tile_offsets;
    w.tile_info = tile_info;
    w.E_loc = a->num_local_experts;
    w.I = a->I;
    w.err = meta + 2;
    w.wsp = wsp1;
    w.Mtot = 2 * a->I;
    w.K = a->H;
    w.n_ntiles = (a->I + fcw_n_rows(true) - 1) / fcw_n_rows(true);
    w.beta = a->gemm1_alpha;
    w.beta_lin = a->gemm1_beta;
    w.alpha_g = a->g1_alphas;
    w.alpha_u = a->g1_alphas_up;
    w.act_kind = a->activation;
    w.topk_fc1 = a->apply_topk_in_fc1 != 0;
    w.permuted_src = psrc;
    w.topk_weights = a->topk_weights;
    w.w1_gs = a->w1_gscale;
    w.xg = g.xg;
    w.h_bf16 = h1;
    // H1's largest magnitude, for an FC2 that multiplies on f16 operands
    const int fc2_rows = nv_wide_fc2(a) ? kNvFc2WideTile : tile_n;
    unsigned* h1max = !h1nv && fct_applies(a->I, fc2_rows) ? (unsigned*)(meta + 3) : nullptr;
    w.h1max = h1max;
    if ((err = launch_fcw_nv(w, a->w1, g.x, g.xs, S, a->num_local_experts, tile_n, max_tiles, st)) != cudaSuccess)
      return SITU_ERR_CUDA;
    mark(3);
    if (h1nv) {
      // H1 requantised per row to NVFP4 (scale chunks of the tiles' layout),
      // then FC2 as NVFP4 x NVFP4 on the same token tiles (kind::mxf4nvf4)
      uint8_t* hq = ws + L.hq;
      uint8_t* hqs = ws + L.hqs;
      float* hg = (float*)(ws + L.hg);
      if ((err = launch_requant_h1_nvfp4(h1, a->I, S, meta, hq, hqs, hg, 1, st)) != cudaSuccess) return SITU_ERR_CUDA;
      FcwParams w2;
      std::memset(&w2, 0, sizeof(w2));
      w2.offsets = offsets;
      w2.tile_offsets = tile_offsets;
      w2.tile_info = tile_info;
      w2.E_loc = a->num_local_experts;
      w2.I = a->I;
      w2.err = meta + 2;
      w2.wsp = wsp1 + packed_nv1_bytes(a);
      w2.Mtot = a->H;
      w2.K = a->I;
      w2.n_ntiles = (a->H + fcw_n_rows(false) - 1) / fcw_n_rows(false);
      w2.alpha2 = a->g2_alphas;
      w2.w2_gs = a->w2_gscale;
      w2.xg = hg;
      w2.y_out = y;
      if ((err = launch_fcw_nv2(w2, a->w2, hq, hqs, S, a->num_local_experts, tile_n, max_tiles, st)) != cudaSuccess)
        return SITU_ERR_CUDA;
      mark(4);
    } else {
    FcvParams v;
    std::memset(&v, 0, sizeof(v));
    v.Mtot = a->H;
    v.K = a->I;
    v.w = a->w2;
    v.ws = a->w2_scale;
    v.gs = a->w2_gscale;
    v.alpha2 = a->g2_alphas;
    v.offsets = offsets;
    v.tile_offsets = tile_offsets;
    v.tile_info = tile_info;
    v.E_loc = a->num_local_experts;
    v.n_ntiles = (a->H + fcw_n_rows(false) - 1) / fcw_n_rows(false);
    v.y_out = y;
    v.err = meta + 2;
    v.h1max = h1max;
    int fc2_tile = tile_n;
    long fc2_tiles = max_tiles;
    if (nv_wide_fc2(a)) {
      fc2_tile = kNvFc2WideTile;
      fc2_tiles = S / kNvFc2WideTile + a->num_local_experts + 1;
      v.tile_offsets = (const int32_t*)(ws + L.t2off);
      v.tile_info = (const int2*)(ws + L.t2info);
    }
    uint16_t* h1f = h1max ? (uint16_t*)(ws + L.h1f) : nullptr;
    if (h1f && (err = launch_h1_to_f16(h1, S, a->I, meta, h1max, h1f, st)) != cudaSuccess) return SITU_ERR_CUDA;
    if ((err = launch_fcv(v, h1, h1f, S, a->num_local_experts, fc2_tile, fc2_tiles, st)) != cudaSuccess)
      return SITU_ERR_CUDA;
    mark(4);
    }
  } else if (decode_path) {
    // 8-token tiles: rows are converted once to f16 block rows, then FC1
    // (+SiTU, writing H1 as f16 block rows) and FC2
    Gather16Params g16;
    g16.act = a->act_dtype;
    g16.row_scale = 0;
    g16.x_bf16 = a->hidden_states;
    g16.x_q = a->hidden_states_q;
    g16.x_s = a->hidden_states_scale;
    g16.x_gs = a->hidden_states_gscale;
    g16.permuted_src = psrc;
    g16.meta = meta;
    g16.top_k = a->top_k;
    g16.K = a->H;
    g16.S = S;
    g16.x16 = (uint16_t*)(ws + L.x16);
    g16.xs = (float*)(ws + L.x16s);
    if ((err = launch_gather16(g16, st)) != cudaSuccess) return SITU_ERR_CUDA;
    mark(2);
    FcdParams d;
    std::memset(&d, 0, sizeof(d));
    d.offsets = offsets;
    d.tile_offsets = tile_offsets;
    d.tile_info = tile_info;
    d.E_loc = a->num_local_experts;
    d.I = a->I;
    d.w = a->w1;
    d.ws = a->w1_scale;
    d.Mtot = 2 * a->I;
    d.K = a->H;
    d.x16 = g16.x16;
    d.xs = g16.xs;
    d.ablk = a->act_dtype != SITU_ACT_NVFP4;   // bf16 and MXFP8 rows carry a scale per 32-block
    d.n_mtiles = (a->I + 63) / 64;
    d.mg = 1;
    d.beta = a->gemm1_alpha;
    d.beta_lin = a->gemm1_beta;
    d.alpha_g = a->g1_alphas;
    d.alpha_u = a->g1_alphas_up;
    d.w1_gs = a->w1_gscale;
    d.h_mxfp8 = a->act_dtype == SITU_ACT_MXFP8;
    d.act_kind = a->activation;
    d.topk_fc1 = a->apply_topk_in_fc1 != 0;
    d.permuted_src = psrc;
    d.topk_weights = a->topk_weights;
    d.h16 = (uint16_t*)(ws + L.h16);
    d.hs = (float*)(ws + L.h16s);
    if ((err = launch_fcd(d, true, nv, max_tiles, st)) != cudaSuccess) return SITU_ERR_CUDA;
    mark(3);
    // FC2 reads H1 (f16 block rows, one scale per 32-block) in expert order
    d.w = a->w2;
    d.ws = a->w2_scale;
    d.Mtot = a->H;
    d.K = a->I;
    d.x16 = d.h16;
    d.xs = d.hs;
    d.ablk = 1;
    d.n_mtiles = (a->H + 127) / 128;
    d.mg = 4;
    d.alpha2 = a->g2_alphas;
    d.w2_gs = a->w2_gscale;
    d.y_out = y;
    if ((err = launch_fcd(d, false, nv, max_tiles, st)) != cudaSuccess) return SITU_ERR_CUDA;
    mark(4);
  } else if (takes_block_scaled_path(a) && fcq_supported(a->H, a->I, a->w1, a->w2)) {
    // 128-token tiles on the block-scaled tensor cores: MXFP8 rows (w4a8)
    // or bf16 rows split into hi / lo MXFP8 rows (w4a16) copied into expert
    // order with their tile scale blocks, FC1 (+SiTU) writing H1 in the same
    // form (MXFP8, or bf16 as hi / lo), FC2 reading it as it stands
    const uint8_t *wsp1, *wsp2, *wsp3, *wsp4;
    if ((err = packed_scales(wsp1, wsp2, wsp3, wsp4)) != cudaSuccess) return SITU_ERR_CUDA;
    const bool lo = a->act_dtype == SITU_ACT_BF16;
    fused = a->fuse_combine != 0;
    if (fused && (err = launch_zero_f32(y, (long)a->T * a->H, st)) != cudaSuccess) return SITU_ERR_CUDA;
    Gather8Params g8;
    g8.x_bf16 = lo ? a->hidden_states : nullptr;
    g8.x_q = a->hidden_states_q;
    g8.x_s = a->hidden_states_scale;
    g8.permuted_src = psrc;
    g8.offsets = offsets;
    g8.tile_offsets = tile_offsets;
    g8.tile_info = tile_info;
    g8.E_loc = a->num_local_experts;
    g8.top_k = a->top_k;
    g8.K = a->H;
    g8.s_vec = (reinterpret_cast<uintptr_t>(a->hidden_states_scale) & 3) == 0;
    g8.x8 = ws + L.x16;
    g8.xsp = ws + L.xsp;
    g8.x8_lo = lo ? g8.x8 + (size_t)S * a->H : nullptr;
    g8.xsp_lo = lo ? g8.xsp + fcq_act_scale_bytes(max_tiles, a->H) : nullptr;
    // MXFP8 rows by token (each row read once for its kept slots); bf16 rows
    // are split per row
    g8.slot_to_row = s2r;
    g8.T = a->T;
    if ((err = launch_gather8(g8, max_tiles, st)) != cudaSuccess) return SITU_ERR_CUDA;
    mark(2);
    FcqParams q;
    std::memset(&q, 0, sizeof(q));
    q.offsets = offsets;
    q.tile_offsets = tile_offsets;
    q.tile_info = tile_info;
    q.E_loc = a->num_local_experts;
    q.I = a->I;
    q.err = meta + 2;
    q.wsp = wsp1;
    q.xsp = g8.xsp;
    q.xsp_lo = g8.xsp_lo;
    q.Mtot = 2 * a->I;
    q.K = a->H;
    q.n_ntiles = (a->I + fcq_n_rows(true) - 1) / fcq_n_rows(true);
    q.beta = a->gemm1_alpha;
    q.beta_lin = a->gemm1_beta;
    q.alpha_g = a->g1_alphas;
    q.alpha_u = a->g1_alphas_up;
    q.act_kind = a->activation;
    q.topk_fc1 = a->apply_topk_in_fc1 != 0;
    q.permuted_src = psrc;
    q.topk_weights = a->topk_weights;
    q.hq = ws + L.h16;
    q.hsp = ws + L.hsp;
    q.hq_lo = lo ? q.hq + (size_t)S * a->I : nullptr;
    q.hsp_lo = lo ? q.hsp + fcq_act_scale_bytes(max_tiles, a->I) : nullptr;
    q.hq_stride = a->I;
    if ((err = launch_fcq(q, g8.x8, g8.x8_lo, S, a->w1, a->num_local_experts, true, max_tiles, st)) !=
        cudaSuccess)
      return SITU_ERR_CUDA;
    mark(3);
    q.wsp = wsp2;
    q.xsp = q.hsp;
    q.xsp_lo = q.hsp_lo;
    q.Mtot = a->H;
    q.K = a->I;
    q.n_ntiles = (a->H + fcq_n_rows(false) - 1) / fcq_n_rows(false);
    q.alpha2 = a->g2_alphas;
    q.y_out = y;
    q.fuse = fused ? 1 : 0;
    q.top_k = a->top_k;
    // unfused: Y as f16 rows with a scale per 32 columns (half the bytes of fp32)
    q.y_scale = fused ? nullptr : ws + L.ys;
    q.ys_rows = S;
    y16 = !fused;
    q.out_acc = y;   // fused: the accumulator [T, H] takes the place of Y
    if ((err = launch_fcq(q, q.hq, q.hq_lo, S, a->w2, a->num_local_experts, false, max_tiles, st)) !=
        cudaSuccess)
      return SITU_ERR_CUDA;
    mark(4);
  } else {
    // 128-token tiles on tcgen05: f16 rows with one scale per row, FC1 (+SiTU)
    // writing bf16 H1, H1 to f16 rows, FC2
    int* err_word = meta + 2;
    Gather16Params g16;
    g16.act = a->act_dtype;
    g16.row_scale = 1;
    g16.x_bf16 = a->hidden_states;
    g16.x_q = a->hidden_states_q;
    g16.x_s = a->hidden_states_scale;
    g16.x_gs = a->hidden_states_gscale;
    g16.permuted_src = psrc;
    g16.meta = meta;
    g16.top_k = a->top_k;
    g16.K = a->H;
    g16.S = S;
    g16.x16 = (uint16_t*)(ws + L.x16);
    g16.xs = (float*)(ws + L.x16s);
    if ((err = launch_gather16(g16, st)) != cudaSuccess) return SITU_ERR_CUDA;
    mark(2);
    FcpParams f;
    std::memset(&f, 0, sizeof(f));
    f.offsets = offsets;
    f.tile_offsets = tile_offsets;
    f.tile_info = tile_info;
    f.E_loc = a->num_local_experts;
    f.I = a->I;
    f.err = err_word;
    f.w = a->w1;
    f.ws = a->w1_scale;
    f.Mtot = 2 * a->I;
    f.K = a->H;
    f.n_ntiles = (a->I + 127) / 128;
    f.xs = g16.xs;
    f.xs_stride = pad128(a->H) / 32;
    f.beta = a->gemm1_alpha;
    f.beta_lin = a->gemm1_beta;
    f.alpha_g = a->g1_alphas;
    f.alpha_u = a->g1_alphas_up;
    f.w1_gs = a->w1_gscale;
    f.h_mxfp8 = a->act_dtype == SITU_ACT_MXFP8;
    f.act_kind = a->activation;
    f.topk_fc1 = a->apply_topk_in_fc1 != 0;
    f.permuted_src = psrc;
    f.topk_weights = a->topk_weights;
    f.h_out = h1;
    if ((err = launch_fcp(f, g16.x16, S, pad128(a->H), a->w1, a->num_local_experts, true, nv, max_tiles, st)) !=
        cudaSuccess)
      return SITU_ERR_CUDA;
    // H1 (bf16, expert order) to f16 rows with one scale per row; with the
    // NVFP4 H1 option, requantised to NVFP4 first and converted exactly
    // (code x block scale in f16, the row's global scale as the row scale)
    Gather16Params h16;
    std::memset(&h16, 0, sizeof(h16));
    h16.act = SITU_ACT_BF16;
    h16.row_scale = 1;
    h16.x_bf16 = h1;
    if (h1nv) {
      if ((err = launch_requant_h1_nvfp4(h1, a->I, S, meta, ws + L.hq, ws + L.hqs, (float*)(ws + L.hg), 0, st)) !=
          cudaSuccess)
        return SITU_ERR_CUDA;
      h16.act = SITU_ACT_NVFP4;
      h16.x_q = ws + L.hq;
      h16.x_s = ws + L.hqs;
      h16.x_gs = (const float*)(ws + L.hg);
    }
    h16.permuted_src = nullptr;
    h16.meta = meta;
    h16.K = a->I;
    h16.S = S;
    h16.x16 = (uint16_t*)(ws + L.h16);
    h16.xs = (float*)(ws + L.h16s);
    if ((err = launch_gather16(h16, st)) != cudaSuccess) return SITU_ERR_CUDA;
    mark(3);
    f.w = a->w2;
    f.ws = a->w2_scale;
    f.Mtot = a->H;
    f.K = a->I;
    f.n_ntiles = (a->H + 255) / 256;
    f.xs = h16.xs;
    f.xs_stride = pad128(a->I) / 32;
    f.alpha2 = a->g2_alphas;
    f.w2_gs = a->w2_gscale;
    f.y_out = y;
    if ((err = launch_fcp(f, h16.x16, S, pad128(a->I), a->w2, a->num_local_experts, false, nv, max_tiles, st)) !=
        cudaSuccess)
      return SITU_ERR_CUDA;
    mark(4);
  }

  if (fused)
    err = launch_acc_to_bf16(y, (long)a->T * a->H, a->out, st);
  else if (y16)
    err = launch_combine16(y, ws + L.ys, S, s2r, a->apply_topk_in_fc1 ? nullptr : a->topk_weights, a->T, a->top_k,
                           a->H, a->out, st);
  else
    err = launch_combine(y, s2r, a->apply_topk_in_fc1 ? nullptr : a->topk_weights, a->T, a->top_k, a->H, a->out,
                         st);
  if (err != cudaSuccess) return SITU_ERR_CUDA;
  mark(5);
  return cuda_status(cudaGetLastError());
}

situ_status situ_moe_forward(const situ_moe_args* a, void* workspace, size_t workspace_bytes,
                             void* stream) {
  return forward_impl(a, workspace, workspace_bytes, stream, nullptr);
}

situ_status situ_moe_forward_profiled(const situ_moe_args* a, void* workspace,
                                      size_t workspace_bytes, void* stream, void* const* events) {
  if (!events) return SITU_ERR_NULL_ARG;
  return forward_impl(a, workspace, workspace_bytes, stream, events);
}

situ_status situ_moe_forward_wait_test(const situ_moe_args* a, void* workspace, size_t workspace_bytes, void* stream,
                                       int32_t skip_stage, int32_t wait_us) {
  if (!a) return SITU_ERR_NULL_ARG;
  if (skip_stage < 0 || wait_us < 1 || wait_us > 1000000) return SITU_ERR_BAD_SHAPE;
  if (validate(a) != SITU_OK) return validate(a);
  // only the block-scaled decode tiles carry the injection
  if (!(fcw_shapes(a) && fcq_supported(a->H, a->I, a->w1, a->w2))) return SITU_ERR_UNSUPPORTED;
  const WaitTest wt = {1000ull * (unsigned long long)wait_us, skip_stage};
  return forward_impl(a, workspace, workspace_bytes, stream, nullptr, &wt);
}

size_t situ_moe_packed_scales_size(const situ_moe_args* a) {
  if (!a || a->H <= 0 || a->I <= 0 || a->num_local_experts < 1 || !(block_scaled_shapes(a) || nv_tile_shapes(a)))
    return 0;
  return packed_total_bytes(a);
}

situ_status situ_moe_pack_scales(const situ_moe_args* a, void* packed, size_t packed_bytes, void* stream) {
  if (!a || !packed) return SITU_ERR_NULL_ARG;
  if (a->H <= 0 || a->I <= 0 || a->num_local_experts < 1 || a->num_local_experts > SITU_MAX_LOCAL_EXPERTS)
    return SITU_ERR_BAD_SHAPE;
  if (!(block_scaled_shapes(a) || nv_tile_shapes(a))) return SITU_ERR_UNSUPPORTED;
  if (!a->w1_scale || !a->w2_scale) return SITU_ERR_NULL_ARG;
  if (!aligned16(packed)) return SITU_ERR_MISALIGNED;
  if (packed_bytes < situ_moe_packed_scales_size(a)) return SITU_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(pack_all_scales(a, (uint8_t*)packed, (cudaStream_t)stream));
}

situ_status situ_moe_wait_selftest(int32_t* device_status, void* stream) {
  if (!device_status) return SITU_ERR_NULL_ARG;
  if (!aligned_to(device_status, 4)) return SITU_ERR_MISALIGNED;
  return cuda_status(launch_wait_selftest(device_status, SITU_SELFTEST_WAIT_CODE, (cudaStream_t)stream));
}

int32_t situ_moe_forward_launches(const situ_moe_args* a) {
  if (validate(a) != SITU_OK) return -1;
  if (a->T == 0) return 0;
  const int perm = permute_launches(a->T, a->top_k, a->num_local_experts);
  const int pack = a->scales_packed ? 0 : 4;
  if (fcw_shapes(a) && fcq_supported(a->H, a->I, a->w1, a->w2)) return perm + pack + 4;
  const int h1nv = a->h1_nvfp4 != 0 ? 1 : 0;   // + the requantisation (+ its scale packing)
  if (fcw_nv_shapes(a)) {
    // + H1 to f16 for an FC2 on f16 operands
    const int fc2_rows = nv_wide_fc2(a) ? kNvFc2WideTile : nv_wide(a) ? kNvWideTile : fcw_token_tile();
    const int f16 = !h1nv && fct_applies(a->I, fc2_rows) ? 1 : 0;
    return perm + (nv_wide_fc2(a) && !h1nv ? 1 : 0) + (a->scales_packed ? 0 : 1 + h1nv) + 4 + h1nv + f16;
  }
  if (takes_decode_path(a)) return perm + 4;
  if (takes_block_scaled_path(a) && fcq_supported(a->H, a->I, a->w1, a->w2))
    return perm + pack + 4 + (a->fuse_combine ? 1 : 0);   // + zeroing the accumulator
  return perm + 5 + h1nv;
}

situ_status situ_moe_device_status(const situ_moe_args* a, const void* workspace, void* stream,
                                   int32_t* code) {
  if (code) *code = 0;
  if (!a || !workspace) return SITU_ERR_NULL_ARG;
  if (check_routing(a->T, a->top_k, a->num_experts_total, a->num_local_experts, a->local_expert_offset) !=
          SITU_OK ||
      a->H <= 0 || a->I <= 0)
    return SITU_ERR_BAD_SHAPE;
  if (a->T == 0) return SITU_OK;
  const Layout L = make_layout(a);
  int32_t word = 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&word, (const uint8_t*)workspace + L.meta + 2 * sizeof(int32_t), sizeof(word),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SITU_ERR_CUDA;
  if (code) *code = word;
  return word == 0 ? SITU_OK : SITU_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
