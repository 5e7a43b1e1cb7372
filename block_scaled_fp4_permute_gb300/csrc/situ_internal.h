// situ_internal.h -- launchers shared between the kernel files and the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace situ {

constexpr int kPermChunk = 4096;   // routing slots per permute block

// tile_offsets / tile_info / meta may be null (the standalone permute).
// tile_info[t] = (local expert, first expert-ordered row) of GEMM token tile t.
cudaError_t launch_permute(const int32_t* ids, int T, int K, int E_loc, int off, int tile_n,
                           int32_t* counts, int32_t* offsets, int32_t* tile_offsets,
                           int2* tile_info, int32_t* permuted_src, int32_t* slot_to_row,
                           int32_t* meta, int32_t* blk_counts, cudaStream_t st);
size_t permute_scratch_bytes(int T, int K, int E_loc);

cudaError_t launch_quant_mxfp8(const void* x, int T, int H, uint8_t* q, uint8_t* s,
                               cudaStream_t st);

cudaError_t launch_combine(const void* y, const int32_t* slot_to_row, const float* w, int T, int K,
                           int H, void* out, cudaStream_t st);

// Gather the kept rows into expert order as bf16 (exact dequantisation of
// MXFP8 / NVFP4 activations) and, for NVFP4, the per-row activation scale.
struct GatherParams {
  int act;                       // situ_act_dtype
  const void* x_bf16;
  const uint8_t* x_q;
  const uint8_t* x_s;
  const float* x_gs;
  const int32_t* permuted_src;
  const int32_t* meta;           // meta[0] = R
  int top_k, H;
  long S;                        // T * top_k, an upper bound on R
  uint16_t* x_perm;              // bf16 [S, H]
  float* xg_perm;                // fp32 [S] (NVFP4) or nullptr
};
cudaError_t launch_gather(const GatherParams& p, cudaStream_t st);

// One grouped GEMM over the token tiles built by the permute:
// rows of W (block-scaled FP4, one matrix per local expert) times the
// expert's permuted bf16 activation rows, with the FC1 (SiTU) or FC2
// (scale, fp32 output) epilogue.
struct FcParams {
  const uint8_t* w;              // packed E2M1 [E_loc, Mtot, K/2]
  const uint8_t* ws;             // block scales [E_loc, Mtot, K/bs]
  int Mtot, K;
  const uint16_t* x;             // bf16 [S, K], rows in expert order
  const int32_t* offsets;        // [E_loc+1]
  const int32_t* tile_offsets;   // [E_loc+1]
  const int2* tile_info;         // [tiles] (expert, first row)
  int E_loc, n_mtiles;
  // FC1
  int I;
  const float *beta, *beta_lin, *alpha_g, *alpha_u, *w1_gs, *xg;
  int mxfp8_h;
  uint16_t* h_out;               // bf16 [S, I]
  // FC2
  const float *alpha2, *w2_gs;
  float* y_out;                  // fp32 [S, H]
};
cudaError_t launch_fc(const FcParams& p, bool fc1, bool nvfp4, int ns, long max_tiles,
                      cudaStream_t st);

// Decode-tile grouped GEMM (8 tokens per CTA, whole K staged once).  The
// activation rows come from `xa` in one of three formats (act): 0 bf16
// [rows, K]; 1 MXFP8 E4M3 [rows, K] + UE8M0 xs [rows, K/32]; 2 NVFP4 packed
// [rows, K/2] + E4M3 xs [rows, K/16] + fp32 xg [rows].  With row_src set,
// expert-ordered row r reads source row row_src[r] / top_k (FC1 gathers
// from the token-major input); without it, row r itself.
struct FcdParams {
  const uint8_t* w;
  const uint8_t* ws;
  int Mtot, K;
  int act;
  const void* xa;
  const uint8_t* xs;
  const float* xg;
  const int32_t* row_src;
  int top_k;
  const int32_t* offsets;
  const int32_t* tile_offsets;
  const int2* tile_info;
  int E_loc, n_mtiles, mg;
  // FC1
  int I;
  const float *beta, *beta_lin, *alpha_g, *alpha_u, *w1_gs;
  int h_mxfp8;
  uint16_t* h_bf16;              // bf16 [S, I]
  uint8_t* h_q;                  // MXFP8 [S, I] (w4a8)
  uint8_t* h_s;                  // UE8M0 [S, I/32]
  // FC2
  const float *alpha2, *w2_gs;
  float* y_out;                  // fp32 [S, H]
};
constexpr int kDecodeTileTokens = 8;
size_t fcd_smem_bytes(int K, bool nvfp4);
cudaError_t launch_fcd(const FcdParams& p, bool fc1, bool nvfp4, long max_tiles, cudaStream_t st);

}  // namespace situ
