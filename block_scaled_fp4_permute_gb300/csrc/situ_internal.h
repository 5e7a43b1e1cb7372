// situ_internal.h -- launchers shared between the kernel files and the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace situ {

constexpr int kPermChunk = 4096;   // routing slots per permute block

// Serialises the launchers' per-device caches of kernel attributes (each
// raises cudaFuncAttributeMaxDynamicSharedMemorySize once per device and
// kernel).  Unserialised, two host threads could both find a cache unset,
// or one could lower a limit that the other has just raised for its launch.
inline std::mutex& attr_mutex() {
  static std::mutex m;
  return m;
}

// Launches kernel k with the programmatic stream-serialisation attribute
// (see griddep_wait): its prologue may overlap the predecessor's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

// tile_offsets / tile_info / meta may be null (the standalone permute).
// tile_info[t] = (local expert, first expert-ordered row) of GEMM token tile t.
cudaError_t launch_permute(const int32_t* ids, int T, int K, int E_loc, int off, int tile_n,
                           int32_t* counts, int32_t* offsets, int32_t* tile_offsets,
                           int2* tile_info, int32_t* permuted_src, int32_t* slot_to_row,
                           int32_t* meta, int32_t* blk_counts, cudaStream_t st);
size_t permute_scratch_bytes(int T, int K, int E_loc);
// a second tile table (tiles of tile_n rows) over the permute's expert
// offsets [E_loc + 1], for a GEMM with another token tile
cudaError_t launch_tile_table(const int32_t* offsets, int E_loc, int tile_n, int32_t* tile_offsets, int2* tile_info,
                              cudaStream_t st);

int permute_launches(int T, int K, int E_loc);   // kernels launch_permute enqueues

cudaError_t launch_quant_mxfp8(const void* x, int T, int H, uint8_t* q, uint8_t* s,
                               cudaStream_t st);
cudaError_t launch_quant_nvfp4(const void* x, int T, int H, uint8_t* q, uint8_t* s, float* gs, cudaStream_t st);

cudaError_t launch_combine(const void* y, const int32_t* slot_to_row, const float* w, int T, int K,
                           int H, void* out, cudaStream_t st);
// the same over Y as f16 rows [S, H] with scale bytes [S, H/32] (y16_exponent)
cudaError_t launch_combine16(const void* y16, const uint8_t* ys, long ys_rows, const int32_t* slot_to_row, const float* w,
                             int T, int K, int H, void* out, cudaStream_t st);
// fused-combine helpers: zero the fp32 accumulator, round it to bf16 out
cudaError_t launch_zero_f32(float* a, long n, cudaStream_t st);
cudaError_t launch_acc_to_bf16(const float* acc, long n, void* out, cudaStream_t st);

// Decode path.  Activation rows for the decode-tile GEMMs are "f16 block
// rows": f16 mantissas [rows, kpad] (kpad = K rounded up to 128, zero
// padded) and one fp32 scale per (row, 32-block) [rows, kpad/32]; a row's
// value is mantissa * scale.  gather16 builds them from the token-major
// input in expert order; FC1 writes H1 in the same form for FC2.
__host__ __device__ inline int pad128(int k) { return (k + 127) / 128 * 128; }

struct Gather16Params {
  int act;                       // situ_act_dtype of the input
  int row_scale;                 // 1: one scale per row (MXFP8 block scales folded into the mantissas)
  const void* x_bf16;
  const uint8_t* x_q;
  const uint8_t* x_s;
  const float* x_gs;
  const int32_t* permuted_src;   // row r reads source row permuted_src[r] / top_k; null: row r
  const int32_t* meta;           // meta[0] = R
  int top_k, K;
  long S;                        // upper bound on R
  uint16_t* x16;                 // f16 [S, pad128(K)]
  float* xs;                     // fp32 [S, pad128(K)/32]
};
cudaError_t launch_gather16(const Gather16Params& p, cudaStream_t st);

// Decode-tile grouped GEMM (8 tokens per CTA, whole K staged once).
struct FcdParams {
  const uint8_t* w;              // packed E2M1 [E_loc, Mtot, K/2]
  const uint8_t* ws;             // block scales [E_loc, Mtot, K/bs]
  int Mtot, K;
  const uint16_t* x16;           // f16 block rows [S, pad128(K)] in expert order
  const float* xs;               // [S, pad128(K)/32]
  int ablk;                      // scales differ per block (else one per row)
  const int32_t* offsets;
  const int32_t* tile_offsets;
  const int2* tile_info;
  int E_loc, n_mtiles, mg;
  // FC1
  int I;
  const float *beta, *beta_lin, *alpha_g, *alpha_u, *w1_gs;
  int h_mxfp8;                   // H1 is the MXFP8 round trip of h (else bf16 of h)
  int act_kind, topk_fc1;        // FC1's activation (kActSitu / kActSwigluBias); routing weight in H1
  const int32_t* permuted_src;   // topk_fc1: row -> slot, and the slots' weights
  const float* topk_weights;
  uint16_t* h16;                 // f16 block rows [S, pad128(I)]
  float* hs;                     // [S, pad128(I)/32]
  // FC2
  const float *alpha2, *w2_gs;
  float* y_out;                  // fp32 [S, H]
};
constexpr int kDecodeTileTokens = 8;

// Prefill-tile grouped GEMM on tcgen05 (fc_tc.cu): 128 token rows x 256
// weight rows per CTA.  Activations: f16 rows [S, pad128(K)] with one fp32
// scale per row (xs[row * xs_stride]).
struct FcpParams {
  int Mtot, K, I;
  const uint8_t* w;              // packed E2M1 [E_loc, Mtot, K/2]
  const uint8_t* ws;             // block scales [E_loc, Mtot, K/bs]
  const int32_t* offsets;
  const int32_t* tile_offsets;
  const int2* tile_info;
  int E_loc, n_ntiles;
  const float* xs;
  int xs_stride;
  // FC1
  const float *beta, *beta_lin, *alpha_g, *alpha_u, *w1_gs;
  int h_mxfp8;
  int act_kind, topk_fc1;
  const int32_t* permuted_src;
  const float* topk_weights;
  uint16_t* h_out;               // bf16 [S, I]
  // FC2
  const float *alpha2, *w2_gs;
  float* y_out;                  // fp32 [S, H]
  int* err;                      // device status word (0 = ok)
};
int fcp_token_tile();
cudaError_t launch_fcp(const FcpParams& p, const uint16_t* x16, long S, int kpad, const uint8_t* w, int E_loc,
                       bool fc1, bool nvfp4, long max_tiles, cudaStream_t st);

// Block-scaled tcgen05 path for MXFP8 activations x MXFP4 weights (w4a8).
// A operand: E4M3 rows in expert order [S, K] plus, per 128-token tile, the
// scale blocks of its rows (xsp [tiles, K/128, 512 B]); B scales packed per
// (expert, N tile, stage) by launch_pack_scales.  K a multiple of 128.  FC1
// writes H1 as E4M3 rows (hq [S, hq_stride]) and scale blocks (hsp [tiles,
// I/128, 512 B]); FC2 writes fp32 Y [S, Mtot].
struct FcqParams {
  int Mtot, K, I;
  const uint8_t* wsp;            // packed weight scale blocks
  const uint8_t* xsp;            // activation scale blocks per token tile
  const uint8_t* xsp_lo;         // the lo rows' blocks (bf16 activations), else null
  const int32_t* offsets;
  const int32_t* tile_offsets;
  const int2* tile_info;
  int E_loc;
  int n_ntiles;
  const float* beta;
  const float* beta_lin;
  const float* alpha_g;
  const float* alpha_u;
  int act_kind, topk_fc1;        // FC1's activation; routing weight in H1 (uses the fields below)
  uint8_t* hq;
  uint8_t* hsp;
  uint8_t* hq_lo;                // FC1 of bf16 activations: H1's lo rows and blocks
  uint8_t* hsp_lo;
  int hq_stride;
  const float* alpha2;
  float* y_out;
  uint8_t* y_scale;              // non-null: Y as f16 rows [S, Mtot] (at y_out) + these scale bytes,
                                 // block-major: byte of (row r, 32-column block b) at b * ys_rows + r
  long ys_rows;
  // fused combine (FC2): add topk_weights[slot] * Y into out_acc [T, Mtot]
  int fuse;
  const int32_t* permuted_src;
  const float* topk_weights;
  int top_k;
  float* out_acc;
  int* err;                      // device status word
};
bool fcq_supported(int H, int I, const void* w1, const void* w2);
// weight rows per N tile: FC1 gate rows (the tile also holds the matching
// up rows), FC2 rows of H
int fcq_n_rows(bool fc1);
// bytes of the activation scale blocks for max_tiles token tiles, and of
// one weight's packed scale blocks
size_t fcq_act_scale_bytes(long max_tiles, int K);
size_t fcq_packed_scale_bytes(int E_loc, int H, int I, bool fc1);
// packed scale blocks for weight tiles of nh rows (FC1: nh gate rows then
// their nh up rows, nh <= 128; FC2: nh <= 256 rows)
size_t packed_scale_bytes(int E_loc, int H, int I, bool fc1, int nh);
cudaError_t launch_pack_scales(const uint8_t* w_scale, int E_loc, int H, int I, bool fc1, uint8_t* out,
                               cudaStream_t st);
cudaError_t launch_pack_scales_nh(const uint8_t* w_scale, int E_loc, int H, int I, bool fc1, int nh, uint8_t* out,
                                  cudaStream_t st);
// xq_lo non-null: bf16 activations as hi (xq) + lo rows, two MMAs per K block
cudaError_t launch_fcq(const FcqParams& p, const uint8_t* xq, const uint8_t* xq_lo, long S, const uint8_t* w,
                       int E_loc, bool fc1, long max_tiles, cudaStream_t st);

// Per token tile: MXFP8 rows (x_q [T, K], x_s [T, K/32]) copied into
// expert order (x8 [S, K]) and their scales written as the tile's scale
// blocks (xsp); bf16 rows (x_bf16 non-null) split into hi rows (x8, xsp) and
// lo rows (x8_lo, xsp_lo) by split_hl32.  K a multiple of 128, s_vec = 1
// when x_s is 4-byte aligned.
struct Gather8Params {
  const void* x_bf16;            // bf16 rows, split into x8 (hi) and x8_lo (lo); null for MXFP8
  const uint8_t* x_q;
  const uint8_t* x_s;
  const int32_t* permuted_src;
  const int32_t* offsets;
  const int32_t* tile_offsets;
  const int2* tile_info;
  int E_loc, top_k, K, s_vec;
  uint8_t* x8;
  uint8_t* xsp;
  uint8_t* x8_lo;
  uint8_t* xsp_lo;
  // MXFP8 rows by token: each token's row read once for all its kept slots
  // (slot_to_row, required for MXFP8), the scale blocks written per tile
  const int32_t* slot_to_row;
  int T;
};
cudaError_t launch_gather8(const Gather8Params& p, long max_tiles, cudaStream_t st);
// Decode tiles on the block-scaled tensor cores (fc_bsd.cu): weights on
// the MMA's M side, up to 16 expert-ordered token rows on N.  Token-side
// rows are E4M3 [rows, K] with scale rows [rows, fcw_scale_stride(K)] bytes
// (16 bytes per 128-element stage, its four UE8M0 bytes first); a bf16 row
// r is the sum of the hi row 2r and the lo row 2r + 1 (lo = true), an MXFP8
// row r is row r.  FC1 writes H1 in the same form for FC2.  The weight
// scales are packed per weight tile: FC1 tiles of fcw_n_rows(true) gate
// rows plus their up rows, FC2 tiles as the prefill GEMM's.
struct GatherHLParams {
  int act;                       // SITU_ACT_BF16 (hi + lo), SITU_ACT_MXFP8 (hi) or SITU_ACT_NVFP4
  const void* x_bf16;
  const uint8_t* x_q;
  const uint8_t* x_s;
  const float* x_gs;             // NVFP4: per-token global scale, copied to xg [S] in row order
  float* xg;
  const int32_t* permuted_src;
  const int32_t* slot_to_row;    // bf16 rows are gathered per token: slot -> row (-1 dropped)
  int T;
  const int32_t* meta;           // meta[0] = R
  int top_k, K;
  long S;
  uint8_t *x, *xs;
  int s_stride;
};
cudaError_t launch_gather_hl(const GatherHLParams& p, cudaStream_t st);
struct FcwParams {
  int Mtot, K, I;
  const uint8_t* w;              // packed E2M1 [E_loc, Mtot, K/2] (set by launch_fcw)
  const uint8_t* wsp;            // packed weight scale blocks of this GEMM's weight tiles
  const int32_t* offsets;
  const int32_t* tile_offsets;
  const int2* tile_info;
  int E_loc, n_ntiles;
  // FC1
  const float *beta, *beta_lin, *alpha_g, *alpha_u;
  int act_kind, topk_fc1;        // FC1's activation; routing weight in H1
  const int32_t* permuted_src;
  const float* topk_weights;
  uint8_t *h, *hs;               // H1 rows and scale rows, as the token side above
  int hs_stride;
  // NVFP4 FC1 (kind::mxf4nvf4): global scales, and H1 as bf16 rows for
  // the NVFP4 FC2 (launch_fcv)
  const float* w1_gs;            // [E_loc, 2] gate / up global scale
  const float* xg;               // [S] the row's per-token global scale
  uint16_t* h_bf16;              // [S, I]
  unsigned* h1max;               // non-null: raised to the largest |H1| (fp32 bits; cleared before)
  // FC2
  const float* alpha2;
  const float* w2_gs;            // [E_loc] global scale (NVFP4 FC2 on the requantised H1)
  float* y_out;                  // fp32 [S, H]
  int* err;                      // device status word
  // failure-path test (situ_moe_forward_wait_test): every wait's limit in ns
  // (0: the default 200 ms), and 1 + the K stage (the producer's running
  // count) that CTA 0 leaves unissued (0: none), so that a zeroed struct
  // injects nothing
  unsigned long long wait_ns;
  int skip_stage1;
};
// one bounded mbarrier wait that nothing completes: records `code` in
// *status after the wait limit and returns (the failure path's self-test)
cudaError_t launch_wait_selftest(int* status, int code, cudaStream_t st);
int fcw_token_tile();
int fcw_n_rows(bool fc1);
int fcw_scale_stride(int K);
cudaError_t launch_fcw(const FcwParams& p, const uint8_t* w, const uint8_t* x, const uint8_t* xs, long S, int E_loc,
                       bool fc1, bool lo, long max_tiles, cudaStream_t st);
// NVFP4 FC1 on the decode tiles: both operands E2M1 with E4M3 scales per 16
// (tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X).  Token rows: packed
// E2M1 [rows, K/2] with their scale rows [rows, K/16] in expert order (gather
// act = NVFP4); weight scales packed by launch_pack_scales_nv.  K a multiple
// of 256, I of 128.
// tile_rows: token rows per tile, 16 or 64 (the tile table's)
cudaError_t launch_fcw_nv(const FcwParams& p, const uint8_t* w, const uint8_t* x, const uint8_t* xs, long S,
                          int E_loc, int tile_rows, long max_tiles, cudaStream_t st);
size_t packed_scale_bytes_nv(int E_loc, int H, int I);
// NVFP4 FC2 on the same tiles, for an H1 requantised per row to NVFP4
// (requant_h1_nvfp4): weights W2 on the MMA M side in 256-row tiles (two
// M = 128 halves), H1 rows as the token side (packed E2M1 [S, K/2], scale
// chunks [S, K/4], global scales p.xg [S]), K = I a multiple of 128 (a last
// half stage of 128 elements is allowed); Y fp32 = alpha2 * w2_gs * xg * acc.
// Weight scales packed by launch_pack_scales_nv2.
cudaError_t launch_fcw_nv2(const FcwParams& p, const uint8_t* w, const uint8_t* x, const uint8_t* xs, long S,
                           int E_loc, int tile_rows, long max_tiles, cudaStream_t st);
size_t packed_scale_bytes_nv2(int E_loc, int H, int I);
cudaError_t launch_pack_scales_nv2(const uint8_t* w2_scale, int E_loc, int H, int I, uint8_t* out, cudaStream_t st);
// The bf16 H1 rows [S, I] (rows < meta[0]) quantised per row to NVFP4 with
// the per-token rule of quant_nvfp4: packed E2M1 [S, I/2], global scales
// [S], and the E4M3 scales either as rows [S, I/16] (chunked = 0) or as one
// 16-byte chunk per 64 elements, its four bytes first, [S, I/4] (chunked =
// 1, the token-side scale layout of the NVFP4 tiles).  I a multiple of 64.
cudaError_t launch_requant_h1_nvfp4(const uint16_t* h, int I, long S, const int32_t* meta, uint8_t* q, uint8_t* s,
                                    float* gs, int chunked, cudaStream_t st);
// NVFP4 FC2 on the decode tiles: the weights expanded to exact bf16 (code x
// E4M3 block scale) in shared memory by converter warps, times the bf16 H1
// rows [S, K] on tcgen05.mma.kind::f16; 256 rows of H per weight tile, up to
// 16 tokens; Y fp32 [S, Mtot] = alpha2 * gs * acc.  K a multiple of 64.
struct FcvParams {
  int Mtot, K;
  const uint8_t* w;              // packed E2M1 [E_loc, Mtot, K/2]
  const uint8_t* ws;             // E4M3 block scales [E_loc, Mtot, K/16]
  const float* gs;               // [E_loc] global scale
  const float* alpha2;           // [E_loc] or null
  const int32_t* offsets;
  const int32_t* tile_offsets;
  const int2* tile_info;
  int E_loc, n_ntiles;
  float* y_out;
  int* err;
  const unsigned* h1max;         // the largest |H1| (fp32 bits), or null: the 16- and
                                 // 64-row tiles then multiply bf16 operands, not f16 ones
};
// tile_rows: the token tile of p's tile table, 16, 64 or 128; h_f16 (may be
// null): H1 as f16 times 2^-s (launch_h1_to_f16), which the 16- and 64-row
// tiles multiply on f16 operands when p.h1max holds a finite maximum
cudaError_t launch_fcv(const FcvParams& p, const uint16_t* h_bf16, const uint16_t* h_f16, long S, int E_loc,
                       int tile_rows, long max_tiles, cudaStream_t st);
// H1 bf16 [S, I] (meta[0] rows in use) to f16 times 2^-s, s from the largest
// magnitude *h1max that the FC1 recorded; nothing when it is not finite
cudaError_t launch_h1_to_f16(const uint16_t* h_bf16, long S, int I, const int32_t* meta, const unsigned* h1max,
                             uint16_t* h_f16, cudaStream_t st);
// whether launch_fcv takes these tiles on the kernel that can use f16 operands
bool fct_applies(int K, int tile_rows);
cudaError_t launch_pack_scales_nv(const uint8_t* w1_scale, int E_loc, int H, int I, uint8_t* out, cudaStream_t st);
size_t fcd_smem_bytes(int K, bool nvfp4);
cudaError_t launch_fcd(const FcdParams& p, bool fc1, bool nvfp4, long max_tiles, cudaStream_t st);

}  // namespace situ
