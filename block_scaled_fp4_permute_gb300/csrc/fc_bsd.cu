// fc_bsd.cu -- FC1 (gate/up + SiTU) and FC2 for decode-sized token tiles on
// the block-scaled tensor cores, weights on the MMA's M side.
//
// Kernels here: fcw_kernel (MXFP4 weights, kind::mxf8f6f4; and the NVFP4
// FC1, kind::mxf4nvf4, 16 or 64 tokens per tile), gather_hl_kernel (the
// token rows in expert order), fcv_kernel (the NVFP4 FC2: weights expanded
// to bf16 in shared memory, kind::f16, 16, 64 or 128 tokens per tile; its
// 128-token tile table comes from tile_table_kernel in permute.cu),
// pack_scales_nv_kernel, and wait_selftest_kernel (the bounded wait made to
// run out).
//
// At decode every touched expert's FP4 weights are streamed once for one or
// two tokens, so the layer is bound by HBM bandwidth, and any per-weight
// instruction (a register conversion of the codes, a scale multiply) costs
// issue slots that the stream cannot spare.  Here no instruction touches a
// weight: TMA copies the packed E2M1 codes from HBM into shared memory (the
// tensor-map type that widens each 8-byte group of 16 codes into a 16-byte
// slot, the 4-bit operand layout of the MMA) and
// tcgen05.mma.kind::mxf8f6f4.block_scale reads them there, with their UE8M0
// block scales in TMEM.
//
// Tokens are the MMA's N side: a tile holds up to 16 expert-ordered rows.
// The activations enter as E4M3 rows with one UE8M0 scale per 32 elements.
// An MXFP8 input is that already.  A bf16 input (and the bf16 H1 of w4a16)
// is held as the sum of two such rows, hi + lo: hi is x rounded to E4M3
// under the block's MXFP8 scale 2^e, and lo the remainder rounded to E4M3
// under 2^(e-4).  hi carries the leading four significant bits and lo the
// next four, so every bf16 value whose exponent lies within 2^-14 of the
// block's largest is represented exactly; smaller ones keep an absolute error
// below 2^-22 of the block maximum.  hi and lo rows are stored interleaved
// (rows 2r and 2r + 1), so one box of 32 rows is the MMA's B operand for 16
// tokens and the epilogue adds columns 2t and 2t + 1.
//
// Weight tiles: FC1 takes 128 gate rows and the 128 matching up rows, FC2
// 256 rows of H; both are staged as rows of 128 K-codes and covered by two
// M = 128 MMAs (FC1: gate, up; FC2: rows 0..127 and 128..255).  In FC1 gate
// row i and up row i are then lane i of the two accumulators, so SiTU runs
// on one thread's registers.  Each MMA has its block of packed
// weight scales (pack_scales: per weight tile and stage, 128 rows x four
// K blocks, laid out as tcgen05.cp.32x128b.warpx4 takes them), copied into
// four TMEM columns.
//
// Token-side scales are rows of 16 bytes per stage, the stage's four UE8M0
// bytes first (the other twelve unused), so a 16-byte TMA box of the tile's
// rows lands as the source layout of tcgen05.cp.32x128b.warpx4 with each
// row's scale word in the first TMEM column of the copy.
//
// Warp roles (one CTA per SM, persistent over the (token tile, weight tile)
// items): warps 0..3 epilogue (thread = TMEM lane = weight row), warp 4 one
// lane TMA producer, warp 5 TMEM allocation and one lane scale copies + MMA.
// Two accumulator buffers let an item's epilogue overlap the next item's
// MMAs; the producer runs ahead across item boundaries.  Every mbarrier wait
// is bounded; on expiry the CTA records an error code, drains what it issued,
// releases TMEM and returns.
#include "situ_internal.h"
#include "../../include/situ_moe.h"
#include "tc_common.cuh"
#include <cuda_fp16.h>

namespace situ {

using namespace tc;

namespace {

constexpr int kTok = 16;           // tokens per tile
constexpr int kRowB = 128;         // bytes of one operand row per stage (one 128-byte swizzle row)
constexpr int kBK = 128;           // K elements per stage of 8-bit containers (MXFP4 x E4M3)
constexpr int kBKnv = 256;         // K elements per stage of packed E2M1 (NVFP4 x NVFP4)
constexpr int kNH1 = 128;          // FC1 gate (and up) rows per weight tile
constexpr int kNH2 = 256;          // FC2 rows per weight tile
constexpr int kThreads = 192;
constexpr int kSfBlock = 512;

// NV: NVFP4 FC1 (E2M1 x E2M1, E4M3 scales per 16, kind::mxf4nvf4 with
// scale_vec::4X).  A stage is then 256 elements of K (128 packed bytes per
// row), four K = 64 MMAs per accumulator; each MMA reads four E4M3 bytes
// per row, so every MMA has its own 512-byte scale block (four TMEM
// columns) on both sides: two weight accumulators x four MMAs, and four
// token blocks (the gather writes each row's stage scales as four 16-byte
// chunks, one per MMA, its word first).  TT: token rows per tile, 16, or
// 64 for NVFP4 when experts hold more rows; a 64-row token scale block
// spans two TMEM columns (rows 0..31, then 32..63): the MMA warp first moves
// row i + 32's word into word 1 of row i in shared memory, so one
// tcgen05.cp (its TMEM destination 4-column aligned, as the copy requires)
// lays both columns.
template <bool FC1, bool LO, bool NV = false, int TT = kTok>
struct CfgW {
  static_assert(!NV || !LO, "the NVFP4 tiles take NVFP4 token rows");
  static_assert(TT == kTok || (NV && TT == 64), "64-row tiles are NVFP4 only");
  static constexpr int kStages = NV ? (TT > 32 ? 4 : 5) : 6;
  static constexpr int NB = LO ? 2 * TT : TT;              // MMA N: token rows (hi, lo interleaved)
  static constexpr int kKS = NV ? kBKnv : kBK;             // K elements per stage
  static constexpr int kABytes = 256 * kRowB;              // 32 KB
  static constexpr int kBBytes = NB * kRowB;               // 2 / 4 / 8 KB
  static constexpr int kWSf = NV ? 8 : 2;                  // weight scale blocks per stage
  static constexpr int kTSf = NV ? 4 : 1;                  // token scale blocks per stage
  static constexpr int kTSfBytes = TT * 16 > kSfBlock ? TT * 16 : kSfBlock;
  static constexpr int kSfBytes = kWSf * kSfBlock + kTSf * kTSfBytes;
  static constexpr int kTmemCols = NV ? 512 : 256;
  static constexpr int kAccStride = 2 * NB > 64 ? 2 * NB : 64;   // columns per accumulator buffer
  static constexpr int kSfCol0 = 2 * kAccStride;            // scale columns after the two buffers
  static constexpr int kSfColsPerStage = 4 * (kWSf + kTSf);
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSF = kOffB + kStages * kBBytes;
  static constexpr int kOffBar = kOffSF + kStages * kSfBytes;
  static constexpr int kNumBars = 2 * kStages + 5;         // full, empty; acc_full[2], acc_empty[2]; drain
  static constexpr int kOffTm = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffTm + 16 + 1024;
  // bytes a stage's copies deliver: the 4-bit map of the MXFP4 weights
  // counts the packed bytes (half the widened tile), the NVFP4 map is bytes
  static constexpr uint32_t kTx = NV ? (uint32_t)(2 * kNH1 * kRowB + NB * kRowB + kTSf * TT * 16 + kWSf * kSfBlock)
                                     : (uint32_t)(FC1 ? 2 * kNH1 : kNH2) * (kBK / 2) + (uint32_t)NB * kBK +
                                           (uint32_t)NB * 16 + 2 * kSfBlock;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
  static_assert(2 * NB <= kAccStride, "accumulator buffer");
  static_assert(kOffB % 1024 == 0 && kBBytes % 1024 == 0 && kABytes % 1024 == 0, "swizzle atoms");
  // A = E2M1 (5), B = E4M3 (0), both K-major; N >> 3 at bit 17, UE8M0
  // scales (bit 23), M >> 4 at bit 24; B / A scale byte selectors at bits
  // 4..5 / 29..30.  NVFP4: A = B = E2M1 (1 in the fp4 kinds' encoding),
  // UE4M3 scales (bit 23 clear), selectors 0 (all four bytes are used).
  static constexpr uint32_t kIdesc =
      NV ? ((1u << 7) | (1u << 10) | ((uint32_t)(NB >> 3) << 17) | ((uint32_t)(128 >> 4) << 24))
         : ((5u << 7) | (0u << 10) | ((uint32_t)(NB >> 3) << 17) | (1u << 23) | ((uint32_t)(128 >> 4) << 24));
};

__device__ __forceinline__ void mma_bs(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_nv(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// scale block in shared memory: no swizzle, 8-row groups of 128 bytes
__device__ __forceinline__ uint64_t sf_desc(uint32_t a) {
  uint64_t d = 0;
  d |= (uint64_t)((a >> 4) & 0x3FFFu);
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  return d;
}
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// barrier over the n threads of named barrier id; returns the AND of v
__device__ __forceinline__ bool bar_red_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %3, 0;\n bar.red.and.pred p, %1, %2, q;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(r)
      : "r"(id), "r"(n), "r"((uint32_t)v)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void drain_wait(uint32_t a, uint32_t parity, unsigned long long limit = kWaitNs) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try(a, parity))
    if (globaltimer() - t0 > limit) return;
}

}  // namespace

// The hi/lo MXFP8 pair of one value v (held exactly in fp32) of a block
// with MXFP8 exponent e; the lo scale exponent is e - c, c = min(4, e + 127).
// Returns the hi code and sets the lo code.
__device__ __forceinline__ uint32_t split_hl(float v, int e, int c, uint32_t& lo) {
  const float x = v * exp2i(-e);
  const uint32_t h = f32x2_to_e4m3x2(x, 0.f) & 0xFFu;
  const float r = x - e4m3_code_to_f32(h);
  lo = f32x2_to_e4m3x2(r * exp2i(c), 0.f) & 0xFFu;
  return h;
}

// byte offset of the UE8M0 scale of 32-element block b in a token scale row
__device__ __forceinline__ int tok_scale_byte(int b) { return 16 * (b >> 2) + (b & 3); }

template <bool FC1, bool LO, bool NV, int TT>
__global__ void __launch_bounds__(kThreads, 1)
fcw_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
           const __grid_constant__ CUtensorMap tmS, const FcwParams p) {
  using C = CfgW<FC1, LO, NV, TT>;
  constexpr int kStages = C::kStages;
  constexpr int NB = C::NB;
  constexpr int NH = FC1 ? kNH1 : kNH2;
  constexpr int RM = LO ? 2 : 1;     // token-side rows per token
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // K stages; the NVFP4 FC2 (K = I, a multiple of 128) may end in a half
  // stage, whose missing half TMA fills with zeros and whose MMAs are skipped
  const int nk = (p.K + C::kKS - 1) / C::kKS;
  // every wait's limit (a test may shorten it), and the one stage a test may
  // leave unissued in CTA 0 (-1: none) so that the waits for it run out
  const unsigned long long lim = p.wait_ns ? p.wait_ns : kWaitNs;
  const long skip = (blockIdx.x == 0 && p.skip_stage1 > 0) ? (long)p.skip_stage1 - 1 : -1;

  const uint32_t sbase = saddr(smem);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto full = [&](int s) { return bar0 + 8 * s; };
  auto empty = [&](int s) { return bar0 + 8 * (kStages + s); };
  auto acc_full = [&](int b) { return bar0 + 8 * (2 * kStages + b); };
  auto acc_empty = [&](int b) { return bar0 + 8 * (2 * kStages + 2 + b); };
  const uint32_t drain = bar0 + 8 * (2 * kStages + 4);
  uint32_t* tm_holder = reinterpret_cast<uint32_t*>(smem + C::kOffTm);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 128);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tm_holder)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tm_holder;
  // the set-up above may overlap the predecessor's tail; everything below
  // reads its outputs
  griddep_wait();
  // an earlier CTA that timed out leaves no work (total = 0)
  const long total = *reinterpret_cast<volatile int*>(p.err) != 0
                         ? 0
                         : (long)__ldg(p.tile_offsets + p.E_loc) * p.n_ntiles;

  if ((long)blockIdx.x >= total) {
    // no item for this CTA
  } else if (warp == 4) {
    // ---------------- TMA producer ----------------
    // the whole warp walks the loop; one elected lane issues the copies
    const bool leader = elect_one();
    long it = 0;
    bool ok = true;
    // the tile of the next item is read one item ahead, so that its
    // latency hides behind this item's loads
    int2 ti_next = __ldg(p.tile_info + blockIdx.x / p.n_ntiles);
    for (long item = blockIdx.x; item < total && ok; item += gridDim.x) {
      const int nt = (int)(item % p.n_ntiles);
      const int2 ti = ti_next;
      if (item + gridDim.x < total) ti_next = __ldg(p.tile_info + (item + gridDim.x) / p.n_ntiles);
      const int e = ti.x, row0 = ti.y;
      const int wrow = e * p.Mtot + nt * NH;
      const uint8_t* wsb = p.wsp + ((size_t)e * p.n_ntiles + nt) * nk * (C::kWSf * kSfBlock);
      for (int kk = 0; kk < nk; ++kk, ++it) {
        const int s = (int)(it % kStages);
        const long r = it / kStages;
        if (r > 0 && !mbar_wait_warp(empty(s), (uint32_t)((r - 1) & 1), p.err, 41, lim)) {
          ok = false;
          break;
        }
        if (leader && it != skip) {
          mbar_expect_tx(full(s), C::kTx);
          const uint32_t a_smem = sbase + C::kOffA + s * C::kABytes;
          const uint32_t sf_smem = sbase + C::kOffSF + s * C::kSfBytes;
          // x = kk * 128: codes of the MXFP4 map, bytes of the E4M3 / packed
          // NVFP4 maps; either way one 128-byte row of the stage
          tma_load_2d(a_smem, &tmW, kk * kRowB, wrow, full(s));
          // FC1: the up half; NVFP4 FC2: rows 128..255 (its map's boxes are 128 rows)
          if (FC1 || NV) tma_load_2d(a_smem + kNH1 * kRowB, &tmW, kk * kRowB, wrow + (FC1 ? p.I : kNH1), full(s));
          tma_load_2d(sbase + C::kOffB + s * C::kBBytes, &tmX, kk * kRowB, RM * row0, full(s));
          bulk_load(sf_smem, wsb + (size_t)kk * C::kWSf * kSfBlock, C::kWSf * kSfBlock, full(s));
#pragma unroll
          for (int b = 0; b < C::kTSf; ++b)
            tma_load_2d(sf_smem + C::kWSf * kSfBlock + b * C::kTSfBytes, &tmS, 16 * (C::kTSf * kk + b), RM * row0,
                        full(s));
        }
        __syncwarp();
      }
    }
    if (leader)
      for (long j = it - 1; j >= 0 && j >= it - kStages; --j)
        drain_wait(full((int)(j % kStages)), (uint32_t)((j / kStages) & 1), lim);
    __syncwarp();
  } else if (warp == 5) {
    // ---------------- scale copies + MMA issuer ----------------
    // the whole warp walks the loop; one elected lane issues
    const bool leader = elect_one();
    long it = 0;
    int li = 0;
    bool ok = true;
    for (long item = blockIdx.x; item < total && ok; item += gridDim.x, ++li) {
      const int buf = li & 1, use = li >> 1;
      if (use > 0 && !mbar_wait_warp(acc_empty(buf), (uint32_t)((use - 1) & 1), p.err, 42, lim)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t d1 = tmem + (uint32_t)(buf * C::kAccStride);
      const uint32_t d2 = d1 + NB;
      for (int kk = 0; kk < nk; ++kk, ++it) {
        const int s = (int)(it % kStages);
        if (!mbar_wait_warp(full(s), (uint32_t)((it / kStages) & 1), p.err, 43, lim)) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (TT > 32) {
          // 64-row token scale blocks: lane i puts row i + 32's scale word
          // beside row i's (word 1 of its 16-byte row)
          uint32_t* tb = reinterpret_cast<uint32_t*>(smem + C::kOffSF + s * C::kSfBytes + C::kWSf * kSfBlock);
#pragma unroll
          for (int b = 0; b < C::kTSf; ++b) {
            uint32_t* blk = tb + b * (C::kTSfBytes / 4);
            blk[4 * lane + 1] = blk[4 * (lane + 32)];
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }
        if (leader) {
          const uint32_t sf_smem = sbase + C::kOffSF + s * C::kSfBytes;
          const uint32_t sfw = tmem + (uint32_t)(C::kSfCol0 + s * C::kSfColsPerStage);
          const uint32_t sft = sfw + 4 * C::kWSf;
          const uint32_t sf_tok = sf_smem + C::kWSf * kSfBlock;
#pragma unroll
          for (int b = 0; b < C::kWSf; ++b) tmem_cp_sf(sfw + 4 * b, sf_desc(sf_smem + b * kSfBlock));
#pragma unroll
          for (int b = 0; b < C::kTSf; ++b) tmem_cp_sf(sft + 4 * b, sf_desc(sf_tok + b * C::kTSfBytes));
          const uint32_t a_smem = sbase + C::kOffA + s * C::kABytes;
          const uint64_t ad1 = sdesc(a_smem);
          const uint64_t ad2 = sdesc(a_smem + 128 * kRowB);
          const uint64_t bd = sdesc(sbase + C::kOffB + s * C::kBBytes);
          // four MMAs per accumulator, 32 bytes of each row apart (K = 32
          // 8-bit containers, or K = 64 packed E2M1)
          const int n64 = NV ? min(4, (p.K - kk * C::kKS) / 64) : 4;   // K = 64 steps in this stage
#pragma unroll
          for (uint32_t k4 = 0; k4 < 4; ++k4) {
            const uint32_t acc = (kk | (int)k4) != 0;
            if (NV && (int)k4 >= n64) break;
            if (NV) {
              // scale block k4 of each accumulator and of the tokens
              mma_nv(d1, ad1 + 2 * k4, bd + 2 * k4, C::kIdesc, sfw + 4 * k4, sft + 4 * k4, acc);
              mma_nv(d2, ad2 + 2 * k4, bd + 2 * k4, C::kIdesc, sfw + 16 + 4 * k4, sft + 4 * k4, acc);
            } else {
              // one block per accumulator, byte k4 of each scale word
              const uint32_t idesc = C::kIdesc | (k4 << 4) | (k4 << 29);
              mma_bs(d1, ad1 + 2 * k4, bd + 2 * k4, idesc, sfw, sft, acc);
              mma_bs(d2, ad2 + 2 * k4, bd + 2 * k4, idesc, sfw + 4, sft, acc);
            }
          }
          mma_commit(empty(s));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) mma_commit(acc_full(buf));
      __syncwarp();
    }
    if (leader) {
      mma_commit(drain);
      drain_wait(drain, 0, lim);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: thread = weight row (TMEM lane) ----------------
    const int l = warp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    for (int li = 0;; ++li) {
      const long item = blockIdx.x + (long)li * gridDim.x;
      if (item >= total) break;
      const int buf = li & 1;
      const int tile = (int)(item / p.n_ntiles), nt = (int)(item % p.n_ntiles);
      const int2 ti = __ldg(p.tile_info + tile);
      const int e = ti.x, row0 = ti.y;
      const int nrows = min(TT, __ldg(p.offsets + e + 1) - row0);
      // the item's constants while the MMAs run: the expert's scales (c0, c1:
      // FC1 gate / up, FC2 output; bt, btl: the activation's caps) and, for
      // NVFP4 tokens, lane j's token global scale (tokens j and j + 32)
      float c0s, c1s = 1.f, bt = 0.f, btl = 0.f;
      if (FC1) {
        c0s = p.alpha_g ? __ldg(p.alpha_g + e) : 1.f;
        c1s = p.alpha_u ? __ldg(p.alpha_u + e) : 1.f;
        if (NV) {
          c0s *= __ldg(p.w1_gs + 2 * e);
          c1s *= __ldg(p.w1_gs + 2 * e + 1);
        }
        bt = __ldg(p.beta + e);
        btl = __ldg(p.beta_lin + e);
      } else {
        c0s = (p.alpha2 ? __ldg(p.alpha2 + e) : 1.f) * (NV ? __ldg(p.w2_gs + e) : 1.f);
      }
      float gxl[TT > 32 ? 2 : 1];
#pragma unroll
      for (int h = 0; h < (TT > 32 ? 2 : 1); ++h)
        gxl[h] = (NV && 32 * h + lane < nrows) ? __ldg(p.xg + row0 + 32 * h + lane) : 0.f;
      // every epilogue thread takes the same decision (the waits are
      // bounded, so all 128 reach the reduction)
      if (!bar_red_and(2, 128, mbar_wait(acc_full(buf), (uint32_t)((li >> 1) & 1), p.err, 46, lim))) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t t1 = tmem + lane_off + (uint32_t)(buf * C::kAccStride);
      float a1[kTok], a2[kTok];
      if (NV) {
        // read 16 token columns at a time below
      } else if (LO) {
        // columns 2t (hi) and 2t + 1 (lo) of token t
        float v[16];
#pragma unroll
        for (int acc = 0; acc < 2; ++acc) {
          float* a = acc ? a2 : a1;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tmem_ld16(t1 + (uint32_t)(acc * NB + 16 * h), v);
#pragma unroll
            for (int j = 0; j < 8; ++j) a[8 * h + j] = v[2 * j] + v[2 * j + 1];
          }
        }
      } else {
        tmem_ld16(t1, a1);
        tmem_ld16(t1 + NB, a2);
      }
      if (!NV) {
        // the accumulator is in registers: hand it back to the MMA warp
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        mbar_arrive(acc_empty(buf));
      }

      if constexpr (NV && !FC1) {
        // NVFP4 FC2 on the requantised H1: the accumulators hold sum(code *
        // scale) products of W2 rows n1 = nt * 256 + l and n2 = n1 + 128; the
        // expert's global scale, alpha2 and the row's H1 global scale make them
        // Y.  Y rows leave as 128-byte segments (a warp's 32 consecutive n).
        const float a2s = c0s;
        const int n1 = nt * kNH2 + l, n2 = n1 + 128;
        for (int c0 = 0; c0 < TT; c0 += 16) {
          tmem_ld16(t1 + c0, a1);
          tmem_ld16(t1 + NB + c0, a2);
          if (c0 >= nrows) continue;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = c0 + j;
            const float gx = __shfl_sync(0xffffffffu, (TT > 32 && (t & 32)) ? gxl[TT > 32 ? 1 : 0] : gxl[0], t & 31);
            if (t >= nrows) break;
            const float sc = a2s * gx;
            float* yr = p.y_out + (size_t)(row0 + t) * p.Mtot;
            if (n1 < p.Mtot) yr[n1] = a1[j] * sc;
            if (n2 < p.Mtot) yr[n2] = a2[j] * sc;
          }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        mbar_arrive(acc_empty(buf));
      } else if constexpr (NV) {
        // NVFP4: the accumulators hold sum(code * scale) products; the
        // expert's gate / up global scale and the token's global scale make
        // them dot products.  H1 is bf16 rows [S, I] (the NVFP4 variant keeps
        // H1 in bf16), which the FC2 of NVFP4 weights reads.
        // The tile's token columns 16 at a time.
        const int i0 = nt * kNH1 + warp * 32;
        const float ag = c0s, au = c1s;
        for (int c0 = 0; c0 < TT; c0 += 16) {
          tmem_ld16(t1 + c0, a1);
          tmem_ld16(t1 + NB + c0, a2);
          if (c0 >= nrows || i0 >= p.I) continue;
          uint32_t hmax = 0;   // largest |H1| of the chunk (bf16 bits; ordered as the magnitudes)
          float gx[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)   // zero past nrows (the lanes' loads)
            gx[j] = __shfl_sync(0xffffffffu, (TT > 32 && ((c0 + j) & 32)) ? gxl[TT > 32 ? 1 : 0] : gxl[0], (c0 + j) & 31);
          float hv[16];
          with_act(p.act_kind, bt, btl, [&](auto act) {
#pragma unroll
            for (int j = 0; j < 16; ++j) hv[j] = act(a1[j] * (ag * gx[j]), a2[j] * (au * gx[j]));
          });
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = c0 + j;
            if (t >= nrows) break;
            float h = hv[j];
            if (p.topk_fc1) h *= __ldg(p.topk_weights + __ldg(p.permuted_src + row0 + t));
            const uint32_t hb = f32x2_to_bf16x2(h, 0.f) & 0xFFFFu;
            p.h_bf16[(size_t)(row0 + t) * p.I + i0 + lane] = (uint16_t)hb;
            hmax = max(hmax, hb & 0x7FFFu);
          }
          if (p.h1max) {
            hmax = __reduce_max_sync(0xffffffffu, hmax);
            if (lane == 0 && hmax != 0) atomicMax(p.h1max, hmax << 16);
          }
        }
        // every column is in registers or stored: hand the accumulator back
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        mbar_arrive(acc_empty(buf));
      } else if (FC1) {
        // gate row i = nt * 128 + l and its up row are lane l of the two
        // accumulators; warp w holds the 32-element block i0 .. i0 + 31
        const int i0 = nt * kNH1 + warp * 32;
        if (i0 < p.I) {
          const float ag = c0s, au = c1s;
          const int sbyte = tok_scale_byte(i0 / 32);   // FC2's K block of this warp
          // the activation of all 16 token columns first (independent
          // chains; the columns past nrows hold other rows or zeros and are
          // not stored), then the per-token block scales and stores
          float hv[kTok];
          with_act(p.act_kind, bt, btl, [&](auto act) {
#pragma unroll
            for (int t = 0; t < kTok; ++t) hv[t] = act(a1[t] * ag, a2[t] * au);
          });
#pragma unroll
          for (int t = 0; t < kTok; ++t) {
            if (t >= nrows) break;
            float h = hv[t];
            if (p.topk_fc1) h *= __ldg(p.topk_weights + __ldg(p.permuted_src + row0 + t));
            if (LO) h = bf16_lo(f32x2_to_bf16x2(h, 0.f));   // w4a16: H1 is bf16
            const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h))));
            const int ex = mxfp8_exponent(amax);
            const size_t r = (size_t)RM * (size_t)(row0 + t);
            if (LO) {
              const int c = min(4, ex + 127);
              uint32_t lo;
              const uint32_t hi = split_hl(h, ex, c, lo);
              p.h[r * p.I + i0 + lane] = (uint8_t)hi;
              p.h[(r + 1) * p.I + i0 + lane] = (uint8_t)lo;
              if (lane == 0) {
                p.hs[r * p.hs_stride + sbyte] = (uint8_t)(ex + 127);
                p.hs[(r + 1) * p.hs_stride + sbyte] = (uint8_t)(ex - c + 127);
              }
            } else {
              p.h[r * p.I + i0 + lane] = (uint8_t)(f32x2_to_e4m3x2(h * exp2i(-ex), 0.f) & 0xFFu);
              if (lane == 0) p.hs[r * p.hs_stride + sbyte] = (uint8_t)(ex + 127);
            }
          }
        }
      } else {
        // FC2: row n = nt * 256 + l (first accumulator) and nt * 256 + 128 + l
        // (second); Y rows leave as 128-byte segments
        const float a2s = c0s;
        const int n1 = nt * kNH2 + l, n2 = nt * kNH2 + 128 + l;
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
          if (t >= nrows) break;
          float* yr = p.y_out + (size_t)(row0 + t) * p.Mtot;
          if (n1 < p.Mtot) yr[n1] = a1[t] * a2s;
          if (n2 < p.Mtot) yr[n2] = a2[t] * a2s;
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// gather_hl: the token-side operand of the decode tiles, in expert order.
// Row r takes token permuted_src[r] / top_k.  A bf16 row becomes hi / lo
// E4M3 rows 2r, 2r + 1 with their scale rows (one thread per 32-element
// block); an MXFP8 row is copied to row r with its scales; an NVFP4 row is
// copied to row r with its scale row and global scale.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(128) gather_hl_kernel(const GatherHLParams p) {
  griddep_wait();   // the permute's outputs
  const long r = blockIdx.x;
  if (r >= __ldg(p.meta)) return;
  const int tid = threadIdx.x;
  const int K = p.K, nb = K / 32;
  const long t = __ldg(p.permuted_src + r) / p.top_k;
  if (p.act == 0) {
    const uint4* xrow = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.x_bf16) + (size_t)t * K * 2);
    uint4* hrow = reinterpret_cast<uint4*>(p.x + (size_t)(2 * r) * K);
    uint4* lrow = reinterpret_cast<uint4*>(p.x + (size_t)(2 * r + 1) * K);
    uint8_t* sh = p.xs + (size_t)(2 * r) * p.s_stride;
    uint8_t* sl = sh + p.s_stride;
    for (int b = tid; b < nb; b += 128) {
      float v[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = __ldg(xrow + 4 * b + q);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * q + 2 * j] = bf16_lo(u[j]);
          v[8 * q + 2 * j + 1] = bf16_hi(u[j]);
        }
      }
      uint32_t hi[8], lo[8];
      const uint32_t sb = split_hl32(v, hi, lo);
      hrow[2 * b] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      hrow[2 * b + 1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
      lrow[2 * b] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      lrow[2 * b + 1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
      sh[tok_scale_byte(b)] = (uint8_t)(sb & 0xFFu);
      sl[tok_scale_byte(b)] = (uint8_t)(sb >> 8);
    }
  } else if (p.act == 2) {
    // NVFP4: packed codes (16-byte rows) copied as they are; the E4M3
    // scales of each 64-element K step (one MMA) as a 16-byte chunk, its
    // four bytes first (scale row of K/4 bytes; the caller's scale rows are
    // read bytewise, they need no alignment); the token's global scale
    const uint4* src = reinterpret_cast<const uint4*>(p.x_q + (size_t)t * (K / 2));
    uint4* dst = reinterpret_cast<uint4*>(p.x + (size_t)r * (K / 2));
    for (int i = tid; i < K / 32; i += 128) dst[i] = __ldg(src + i);
    const uint8_t* ss = p.x_s + (size_t)t * (K / 16);
    uint4* sd = reinterpret_cast<uint4*>(p.xs + (size_t)r * (K / 4));
    for (int c = tid; c < K / 64; c += 128) {
      const uint32_t v = (uint32_t)__ldg(ss + 4 * c) | ((uint32_t)__ldg(ss + 4 * c + 1) << 8) |
                         ((uint32_t)__ldg(ss + 4 * c + 2) << 16) | ((uint32_t)__ldg(ss + 4 * c + 3) << 24);
      sd[c] = make_uint4(v, 0u, 0u, 0u);
    }
    if (tid == 0) p.xg[r] = __ldg(p.x_gs + t);
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(p.x_q + (size_t)t * K);
    uint4* dst = reinterpret_cast<uint4*>(p.x + (size_t)r * K);
    for (int i = tid; i < K / 16; i += 128) dst[i] = __ldg(src + i);
    const uint8_t* ss = p.x_s + (size_t)t * nb;
    uint8_t* sh = p.xs + (size_t)r * p.s_stride;
    for (int b = tid; b < nb; b += 128) sh[tok_scale_byte(b)] = __ldg(ss + b);
  }
}

// bf16 token rows by token: each thread splits one 32-element block of
// token t into hi + lo E4M3 blocks once and writes them to the rows of all
// the token's kept slots (up to top_k), so a token's row is read and split
// once instead of once per kept slot.
constexpr int kGatherTokThreads = 32;
__global__ void __launch_bounds__(kGatherTokThreads) gather_hl_tok_kernel(const GatherHLParams p) {
  griddep_wait();   // the permute's outputs
  const long t = blockIdx.x;
  const int lane = threadIdx.x;
  const int K = p.K, nb = K / 32;
  const int b = blockIdx.y * kGatherTokThreads + lane;
  // lane j holds the row of slot j
  const int my_row = lane < p.top_k ? __ldg(p.slot_to_row + t * p.top_k + lane) : -1;
  // every lane stays for the row shuffles below; lanes past the row's last
  // block only take part in them
  const bool valid = b < nb;
  const uint4* xrow = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.x_bf16) + (size_t)t * K * 2);
  float v[32];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = valid ? __ldg(xrow + 4 * b + q) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * q + 2 * j] = bf16_lo(u[j]);
      v[8 * q + 2 * j + 1] = bf16_hi(u[j]);
    }
  }
  uint32_t hi[8], lo[8];
  const uint32_t sb = split_hl32(v, hi, lo);
  const uint4 h0 = make_uint4(hi[0], hi[1], hi[2], hi[3]), h1 = make_uint4(hi[4], hi[5], hi[6], hi[7]);
  const uint4 l0 = make_uint4(lo[0], lo[1], lo[2], lo[3]), l1 = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  for (int j = 0; j < p.top_k; ++j) {
    const int r = __shfl_sync(0xffffffffu, my_row, j);
    if (r < 0 || !valid) continue;
    uint4* hrow = reinterpret_cast<uint4*>(p.x + (size_t)(2 * r) * K);
    uint4* lrow = reinterpret_cast<uint4*>(p.x + (size_t)(2 * r + 1) * K);
    hrow[2 * b] = h0;
    hrow[2 * b + 1] = h1;
    lrow[2 * b] = l0;
    lrow[2 * b + 1] = l1;
    uint8_t* sh = p.xs + (size_t)(2 * r) * p.s_stride;
    sh[tok_scale_byte(b)] = (uint8_t)(sb & 0xFFu);
    sh[p.s_stride + tok_scale_byte(b)] = (uint8_t)(sb >> 8);
  }
}

// NVFP4 token rows by token: token t's packed codes and its scale chunks
// (the E4M3 scales of each 64-element K step as a 16-byte chunk, its four
// bytes first) are read once and written to the rows of all its kept slots,
// with the token's global scale; one CTA per token instead of one per row.
constexpr int kGatherNvThreads = 128;
__global__ void __launch_bounds__(kGatherNvThreads) gather_nv_tok_kernel(const GatherHLParams p) {
  griddep_wait();   // the permute's outputs
  const long t = blockIdx.x;
  const int tid = threadIdx.x;
  const int K = p.K, top_k = p.top_k;
  __shared__ int rows[SITU_MAX_TOP_K];
  if (tid < top_k) rows[tid] = __ldg(p.slot_to_row + t * top_k + tid);
  __syncthreads();
  const uint4* src = reinterpret_cast<const uint4*>(p.x_q + (size_t)t * (K / 2));
  for (int i = tid; i < K / 32; i += kGatherNvThreads) {
    const uint4 v = __ldg(src + i);
    for (int j = 0; j < top_k; ++j) {
      const int r = rows[j];
      if (r >= 0) reinterpret_cast<uint4*>(p.x + (size_t)r * (K / 2))[i] = v;
    }
  }
  const uint8_t* ss = p.x_s + (size_t)t * (K / 16);
  for (int c = tid; c < K / 64; c += kGatherNvThreads) {
    const uint32_t v = (uint32_t)__ldg(ss + 4 * c) | ((uint32_t)__ldg(ss + 4 * c + 1) << 8) |
                       ((uint32_t)__ldg(ss + 4 * c + 2) << 16) | ((uint32_t)__ldg(ss + 4 * c + 3) << 24);
    for (int j = 0; j < top_k; ++j) {
      const int r = rows[j];
      if (r >= 0) reinterpret_cast<uint4*>(p.xs + (size_t)r * (K / 4))[c] = make_uint4(v, 0u, 0u, 0u);
    }
  }
  if (tid < top_k && rows[tid] >= 0) p.xg[rows[tid]] = __ldg(p.x_gs + t);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

int sm_count_w() {
  static std::atomic<int> n[64];   // SM count per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && n[dev] > 0) return n[dev];
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
  if (dev < 64) n[dev] = v;
  return v;
}

template <bool FC1, bool LO, bool NV = false, int TT = kTok>
cudaError_t launch_fcw_t(const FcwParams& p, const CUtensorMap* m, long max_tiles, cudaStream_t st) {
  using C = CfgW<FC1, LO, NV, TT>;
  static int set_for[64];
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (dev >= 64 || set_for[dev] == 0) {
      cudaError_t err =
          cudaFuncSetAttribute(fcw_kernel<FC1, LO, NV, TT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
      if (err != cudaSuccess) return err;
      if (dev < 64) set_for[dev] = 1;
    }
  }
  const long items = max_tiles * p.n_ntiles;   // upper bound; the kernel reads the true count
  const long grid = items < sm_count_w() ? items : sm_count_w();
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(fcw_kernel<FC1, LO, NV, TT>, dim3((unsigned)grid), dim3(kThreads), (size_t)C::kSmem, st, m[0],
                    m[1], m[2], p);
}

}  // namespace

int fcw_token_tile() { return kTok; }
int fcw_n_rows(bool fc1) { return fc1 ? kNH1 : kNH2; }
int fcw_scale_stride(int K) { return K / 8; }   // 16 bytes per 128-element stage

cudaError_t launch_gather_hl(const GatherHLParams& p, cudaStream_t st) {
  if (p.S <= 0) return cudaSuccess;
  if (p.act == 0 && p.slot_to_row) {
    const int nb = p.K / 32;
    const dim3 grid((unsigned)p.T, (unsigned)((nb + kGatherTokThreads - 1) / kGatherTokThreads));
    return launch_pdl(gather_hl_tok_kernel, grid, dim3(kGatherTokThreads), 0, st, p);
  }
  if (p.act == 2 && p.slot_to_row) {
    if (p.T <= 0) return cudaSuccess;
    return launch_pdl(gather_nv_tok_kernel, dim3((unsigned)p.T), dim3(kGatherNvThreads), 0, st, p);
  }
  return launch_pdl(gather_hl_kernel, dim3((unsigned)p.S), dim3(128), 0, st, p);
}

cudaError_t launch_fcw(const FcwParams& p, const uint8_t* w, const uint8_t* x, const uint8_t* xs, long S, int E_loc,
                       bool fc1, bool lo, long max_tiles, cudaStream_t st) {
  if (S <= 0) return cudaSuccess;
  FcwParams q = p;
  q.w = w;
  CUtensorMap m[3];
  const int ss = fcw_scale_stride(p.K);
  const uint64_t rows = (uint64_t)S * (lo ? 2 : 1);   // token-side rows (hi, lo interleaved)
  const uint32_t nb = (uint32_t)(lo ? 2 * kTok : kTok);
  // weights: E2M1 [E_loc * Mtot, K] (K/2 bytes per row), boxes of 128 codes x
  // the tile's rows, each 16 codes in a 16-byte slot, 128-byte swizzle
  if (!make_map(&m[0], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w, (uint64_t)p.K, (uint64_t)E_loc * p.Mtot,
                (uint64_t)(p.K / 2), kBK, (uint32_t)fcw_n_rows(fc1), CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // token rows: E4M3 [rows, K], boxes of 128 bytes x the tile's rows,
  // 128-byte swizzle; scale rows: [rows, ss] bytes, boxes of 16 bytes
  if (!make_map(&m[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, x, (uint64_t)p.K, rows, (uint64_t)p.K, kBK, nb,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, xs, (uint64_t)ss, rows, (uint64_t)ss, 16, nb,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (fc1) return lo ? launch_fcw_t<true, true>(q, m, max_tiles, st) : launch_fcw_t<true, false>(q, m, max_tiles, st);
  return lo ? launch_fcw_t<false, true>(q, m, max_tiles, st) : launch_fcw_t<false, false>(q, m, max_tiles, st);
}

// ---------------------------------------------------------------------------
// NVFP4 FC1 on the decode tiles
// ---------------------------------------------------------------------------

// Packed NVFP4 weight scales of the FC1 decode tiles: per (expert, weight
// tile nt, stage kk of 256 elements, accumulator a (gate, up), MMA k) a
// 512-byte block; in it the four E4M3 bytes of tile row r = i + 32q (K
// blocks 16kk + 4k .. + 3 of source row a * I + nt * 128 + r) sit at byte
// 16i + 4q, the layout tcgen05.cp.32x128b.warpx4 spreads over the four
// TMEM columns the MMA reads.  One thread per 4-byte word.
__global__ void pack_scales_nv_kernel(const uint8_t* __restrict__ ws, int H, int I, int n_nt, int nk, long n_words,
                                      uint32_t* __restrict__ out) {
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_words) return;
  const int w = (int)(idx & 127);
  const int i = w >> 2, q = w & 3;
  long b = idx >> 7;
  const int k = (int)(b & 3);
  b >>= 2;
  const int a = (int)(b & 1);
  b >>= 1;
  const int kk = (int)(b % nk);
  b /= nk;
  const int nt = (int)(b % n_nt);
  const long e = b / n_nt;
  const int ir = nt * kNH1 + i + 32 * q;   // gate / up row within the half
  uint32_t v = 0;
  if (ir < I) {
    const uint8_t* src = ws + ((size_t)e * 2 * I + (size_t)a * I + ir) * (size_t)(H / 16) + 16 * kk + 4 * k;
    v = (uint32_t)src[0] | ((uint32_t)src[1] << 8) | ((uint32_t)src[2] << 16) | ((uint32_t)src[3] << 24);
  }
  out[idx] = v;
}

size_t packed_scale_bytes_nv(int E_loc, int H, int I) {
  const size_t n_nt = (size_t)(I + kNH1 - 1) / kNH1, nk = (size_t)H / kBKnv;
  return (size_t)E_loc * n_nt * nk * 8 * kSfBlock;
}

cudaError_t launch_pack_scales_nv(const uint8_t* w1_scale, int E_loc, int H, int I, uint8_t* out, cudaStream_t st) {
  const int n_nt = (I + kNH1 - 1) / kNH1, nk = H / kBKnv;
  const long n_words = (long)(packed_scale_bytes_nv(E_loc, H, I) / 4);
  if (n_words <= 0) return cudaSuccess;
  pack_scales_nv_kernel<<<(unsigned)((n_words + 255) / 256), 256, 0, st>>>(w1_scale, H, I, n_nt, nk, n_words,
                                                                          reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError();
}

// Packed NVFP4 weight scales of the FC2 tiles: per (expert, 256-row tile
// nt, stage kk of 256 elements of I, half a (rows 0..127, 128..255), MMA k)
// a 512-byte block laid out as pack_scales_nv's, from W2's E4M3 scales
// [E_loc, H, I/16]; the blocks of K steps past I (a last half stage) are 0.
__global__ void pack_scales_nv2_kernel(const uint8_t* __restrict__ ws, int H, int I, int n_nt, int nk, long n_words,
                                       uint32_t* __restrict__ out) {
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_words) return;
  const int w = (int)(idx & 127);
  const int i = w >> 2, q = w & 3;
  long b = idx >> 7;
  const int k = (int)(b & 3);
  b >>= 2;
  const int a = (int)(b & 1);
  b >>= 1;
  const int kk = (int)(b % nk);
  b /= nk;
  const int nt = (int)(b % n_nt);
  const long e = b / n_nt;
  const int row = nt * kNH2 + a * 128 + i + 32 * q;   // row of H
  const int kb = 16 * kk + 4 * k;                     // first 16-element block of the MMA
  uint32_t v = 0;
  if (row < H && kb < I / 16) {
    const uint8_t* src = ws + ((size_t)e * H + row) * (size_t)(I / 16) + kb;
    v = (uint32_t)src[0] | ((uint32_t)src[1] << 8) | ((uint32_t)src[2] << 16) | ((uint32_t)src[3] << 24);
  }
  out[idx] = v;
}

size_t packed_scale_bytes_nv2(int E_loc, int H, int I) {
  const size_t n_nt = (size_t)(H + kNH2 - 1) / kNH2, nk = (size_t)(I + kBKnv - 1) / kBKnv;
  return (size_t)E_loc * n_nt * nk * 8 * kSfBlock;
}

cudaError_t launch_pack_scales_nv2(const uint8_t* w2_scale, int E_loc, int H, int I, uint8_t* out, cudaStream_t st) {
  const int n_nt = (H + kNH2 - 1) / kNH2, nk = (I + kBKnv - 1) / kBKnv;
  const long n_words = (long)(packed_scale_bytes_nv2(E_loc, H, I) / 4);
  if (n_words <= 0) return cudaSuccess;
  pack_scales_nv2_kernel<<<(unsigned)((n_words + 255) / 256), 256, 0, st>>>(w2_scale, H, I, n_nt, nk, n_words,
                                                                           reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError();
}

cudaError_t launch_fcw_nv2(const FcwParams& p, const uint8_t* w, const uint8_t* x, const uint8_t* xs, long S,
                           int E_loc, int tile_rows, long max_tiles, cudaStream_t st) {
  if (S <= 0) return cudaSuccess;
  if (tile_rows != kTok && tile_rows != 64) return cudaErrorInvalidValue;
  if (p.K % 128 != 0) return cudaErrorInvalidValue;
  FcwParams q = p;
  q.w = w;
  CUtensorMap m[3];
  // W2 and the H1 rows: packed E2M1 as bytes [rows, K/2], boxes of 128
  // bytes x 128 weight rows / the tile's token rows, 128-byte swizzle (a box
  // past the row end of a half stage reads zeros); H1 scale rows [S, K/4]
  // bytes, boxes of 16 bytes
  if (!make_map(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, w, (uint64_t)(p.K / 2), (uint64_t)E_loc * p.Mtot,
                (uint64_t)(p.K / 2), kRowB, kNH1, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, x, (uint64_t)(p.K / 2), (uint64_t)S, (uint64_t)(p.K / 2), kRowB,
                (uint32_t)tile_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, xs, (uint64_t)(p.K / 4), (uint64_t)S, (uint64_t)(p.K / 4), 16,
                (uint32_t)tile_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (tile_rows == 64) return launch_fcw_t<false, false, true, 64>(q, m, max_tiles, st);
  return launch_fcw_t<false, false, true, kTok>(q, m, max_tiles, st);
}

cudaError_t launch_fcw_nv(const FcwParams& p, const uint8_t* w, const uint8_t* x, const uint8_t* xs, long S,
                          int E_loc, int tile_rows, long max_tiles, cudaStream_t st) {
  if (S <= 0) return cudaSuccess;
  if (tile_rows != kTok && tile_rows != 64) return cudaErrorInvalidValue;
  FcwParams q = p;
  q.w = w;
  CUtensorMap m[3];
  // weights and token rows: packed E2M1 as bytes [rows, K/2], boxes of 128
  // bytes (256 codes) x the tile's rows, 128-byte swizzle; token scale rows
  // [rows, K/4] bytes (a 16-byte chunk per 64 elements), boxes of 16 bytes
  if (!make_map(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, w, (uint64_t)(p.K / 2), (uint64_t)E_loc * p.Mtot,
                (uint64_t)(p.K / 2), kRowB, kNH1, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, x, (uint64_t)(p.K / 2), (uint64_t)S, (uint64_t)(p.K / 2), kRowB,
                (uint32_t)tile_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, xs, (uint64_t)(p.K / 4), (uint64_t)S, (uint64_t)(p.K / 4), 16,
                (uint32_t)tile_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (tile_rows == 64) return launch_fcw_t<true, false, true, 64>(q, m, max_tiles, st);
  return launch_fcw_t<true, false, true, kTok>(q, m, max_tiles, st);
}

// ---------------------------------------------------------------------------
// fcv_kernel: FC2 of NVFP4 weights on the decode tiles, bf16 H1.
//
// The FC2 input H1 is bf16 (the NVFP4 variant keeps H1 in bf16), which no
// fp4 x fp4 MMA can take, and NVFP4's E4M3 scales per 16 fit no UE8M0
// block-scaled kind.  So the weights are expanded in shared memory: a code
// times its block scale is E2M1 x E4M3, at most six significant bits, held
// exactly by bf16; tcgen05.mma.kind::f16 multiplies it with the bf16 H1 in
// fp32.  The per-expert global scale and alpha2 go to the epilogue.
//
// Tiles as fcw's FC2: 256 rows of H (two M = 128 accumulators) x up to 16
// expert-ordered tokens (N = 16), K = I in stages of 64.  Per stage TMA
// loads the packed codes of the 256 rows (32 bytes each, no swizzle) and the
// tokens' bf16 H1 rows (128 bytes each, 128-byte swizzle); eight converter
// warps (one weight row per thread) write the stage's bf16 A operand in the
// 128-byte-swizzled K-major layout, reading the row's four E4M3 scale bytes
// from global memory one stage ahead.  Warp roles: 0..3 epilogue (thread =
// TMEM lane = weight row), 4 TMA producer, 5 TMEM allocation + MMA issuer,
// 6..13 converters.  Persistent over (token tile, weight tile) items, two
// accumulator buffers; every wait bounded, as in fcw_kernel.
// ---------------------------------------------------------------------------

namespace {

constexpr int kVBK = 64;                        // K elements per stage
constexpr int kVThreads = 448;
constexpr int kVABytes = 256 * 128;             // bf16 A operand: 256 rows x 64 elements
constexpr int kVRBytes = 256 * 32;              // packed codes
// NB: token rows per tile (MMA N), 16, 64 or 128 as experts hold more rows
template <int NB>
struct CfgV {
  static constexpr int kStages = NB > 64 ? 3 : NB > 16 ? 4 : 5;
  static constexpr int kTmemCols = NB > 16 ? 4 * NB : 64;   // two buffers of two NB-column accumulators
  static constexpr int kXBytes = NB * 128;              // bf16 token rows
  static constexpr int kOffA = 0;
  static constexpr int kOffX = kOffA + kStages * kVABytes;
  static constexpr int kOffR = kOffX + kStages * kXBytes;
  static constexpr int kOffBar = kOffR + kStages * kVRBytes;
  static constexpr int kNumBars = 3 * kStages + 5;     // full, conv, empty; acc_full[2], acc_empty[2]; drain
  static constexpr int kOffTm = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffTm + 16 + 1024;
  static constexpr uint32_t kTx = kXBytes + kVRBytes;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(kOffX % 1024 == 0 && kXBytes % 1024 == 0, "swizzle atoms");
  static_assert(4 * NB <= kTmemCols, "TMEM budget");
  // kind::f16: fp32 accumulator (bit 4), A = B = bf16 (1 at bits 7 and 10),
  // both K-major, N >> 3 at bit 17, M >> 4 at bit 24
  static constexpr uint32_t kIdesc =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NB >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
};

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// eight E2M1 codes (one 32-bit word, byte j = elements 2j, 2j + 1) -> f16 pairs
__device__ __forceinline__ void e2m1x8_f16(uint32_t w, uint32_t* d) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(w));
}
__device__ __forceinline__ uint32_t e4m3_pair_f16(uint32_t b) {   // one E4M3 code in both halves
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)(b | (b << 8))));
  return d;
}
// code x scale as an exact f16 pair, then as a bf16 pair (at most six
// significant bits and magnitudes in [2^-10, 2688]: exact in both)
__device__ __forceinline__ uint32_t scaled_bf16x2(uint32_t codes_f16x2, uint32_t scale_f16x2) {
  uint32_t v;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(v) : "r"(codes_f16x2), "r"(scale_f16x2));
  const float lo = __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
  const float hi = __half2float(__ushort_as_half((unsigned short)(v >> 16)));
  return f32x2_to_bf16x2(lo, hi);
}

}  // namespace

template <int NB>
__global__ void __launch_bounds__(kVThreads, 1)
fcv_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const FcvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using C = CfgV<NB>;
  constexpr int kVStages = C::kStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nk = p.K / kVBK;
  const int nsb = p.K / 16;                     // E4M3 scales per weight row

  const uint32_t sbase = saddr(smem);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto full = [&](int s) { return bar0 + 8 * s; };
  auto conv = [&](int s) { return bar0 + 8 * (kVStages + s); };
  auto empty = [&](int s) { return bar0 + 8 * (2 * kVStages + s); };
  auto acc_full = [&](int b) { return bar0 + 8 * (3 * kVStages + b); };
  auto acc_empty = [&](int b) { return bar0 + 8 * (3 * kVStages + 2 + b); };
  const uint32_t drain = bar0 + 8 * (3 * kVStages + 4);
  uint32_t* tm_holder = reinterpret_cast<uint32_t*>(smem + C::kOffTm);

  if (tid == 0) {
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(conv(s), 256);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 128);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tm_holder)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tm_holder;
  griddep_wait();
  const long total = *reinterpret_cast<volatile int*>(p.err) != 0
                         ? 0
                         : (long)__ldg(p.tile_offsets + p.E_loc) * p.n_ntiles;

  if ((long)blockIdx.x >= total) {
    // no item for this CTA
  } else if (warp == 4) {
    // ---------------- TMA producer ----------------
    const bool leader = elect_one();
    long it = 0;
    bool ok = true;
    for (long item = blockIdx.x; item < total && ok; item += gridDim.x) {
      const int nt = (int)(item % p.n_ntiles);
      const int2 ti = __ldg(p.tile_info + item / p.n_ntiles);
      const int wrow = ti.x * p.Mtot + nt * kNH2;
      // the next item's weight rows into L2 now: its packed codes and E4M3
      // scales are two contiguous runs (kNH2 rows of K/2 and K/16 bytes), so
      // two bulk prefetches stand in for a ring deeper than shared memory holds
      const long inext = item + gridDim.x;
      if (leader && inext < total) {
        const int ntn = (int)(inext % p.n_ntiles);
        const int en = __ldg(p.tile_info + inext / p.n_ntiles).x;
        const int r0 = ntn * kNH2;
        const int rows = min(kNH2, p.Mtot - r0);
        const size_t row = (size_t)en * p.Mtot + r0;
        const uint32_t cb = (uint32_t)rows * (uint32_t)(p.K / 2), sb = (uint32_t)rows * (uint32_t)(p.K / 16);
        bulk_prefetch_l2(p.w + row * (size_t)(p.K / 2), cb & ~15u);
        if ((reinterpret_cast<uintptr_t>(p.ws + row * (size_t)(p.K / 16)) & 15u) == 0)
          bulk_prefetch_l2(p.ws + row * (size_t)(p.K / 16), sb & ~15u);
      }
      for (int kk = 0; kk < nk; ++kk, ++it) {
        const int s = (int)(it % kVStages);
        const long r = it / kVStages;
        if (r > 0 && !mbar_wait_warp(empty(s), (uint32_t)((r - 1) & 1), p.err, 51)) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_expect_tx(full(s), C::kTx);
          tma_load_2d(sbase + C::kOffR + s * kVRBytes, &tmW, kk * (kVBK / 2), wrow, full(s));
          tma_load_2d(sbase + C::kOffX + s * C::kXBytes, &tmX, kk * kVBK, ti.y, full(s));
        }
        __syncwarp();
      }
    }
    if (leader)
      for (long j = it - 1; j >= 0 && j >= it - kVStages; --j)
        drain_wait(full((int)(j % kVStages)), (uint32_t)((j / kVStages) & 1));
    __syncwarp();
  } else if (warp >= 6) {
    // ---------------- converters: thread = weight row n of the tile ----------------
    const int n = tid - 192;
    long it = 0;
    for (long item = blockIdx.x; item < total; item += gridDim.x) {
      const int nt = (int)(item % p.n_ntiles);
      const int e = __ldg(p.tile_info + item / p.n_ntiles).x;
      const int grow = nt * kNH2 + n;
      const bool valid = grow < p.Mtot;
      const uint8_t* srow = p.ws + ((size_t)e * p.Mtot + (valid ? grow : 0)) * (size_t)nsb;
      // the row's four scale bytes of a stage (its 16-element blocks)
      auto load_sc = [&](int kk) -> uint32_t {
        if (!valid || kk >= nk) return 0u;
        const uint8_t* q = srow + 4 * kk;
        return (uint32_t)__ldg(q) | ((uint32_t)__ldg(q + 1) << 8) | ((uint32_t)__ldg(q + 2) << 16) |
               ((uint32_t)__ldg(q + 3) << 24);
      };
      uint32_t sc = load_sc(0);
      bool ok = true;
      for (int kk = 0; kk < nk; ++kk, ++it) {
        const uint32_t sc_next = load_sc(kk + 1);
        const int s = (int)(it % kVStages);
        if (!mbar_wait(full(s), (uint32_t)((it / kVStages) & 1), p.err, 54)) {
          ok = false;
          break;
        }
        const uint8_t* raw = smem + C::kOffR + s * kVRBytes + n * 32;
        uint8_t* arow = smem + C::kOffA + s * kVABytes + n * 128;
        const uint4 q0 = *reinterpret_cast<const uint4*>(raw);
        const uint4 q1 = *reinterpret_cast<const uint4*>(raw + 16);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint32_t f[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) f[b] = e4m3_pair_f16((sc >> (8 * b)) & 0xFFu);
#pragma unroll
        for (int j = 0; j < 8; ++j) {   // 16-byte chunk j = elements 8j .. 8j + 7 (block j / 2)
          uint32_t d[4];
          e2m1x8_f16(w[j], d);
#pragma unroll
          for (int i = 0; i < 4; ++i) d[i] = scaled_bf16x2(d[i], f[j >> 1]);
          *reinterpret_cast<uint4*>(arow + ((j ^ (n & 7)) << 4)) = make_uint4(d[0], d[1], d[2], d[3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(conv(s));
        sc = sc_next;
      }
      if (!ok) break;
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    const bool leader = elect_one();
    long it = 0;
    int li = 0;
    bool ok = true;
    for (long item = blockIdx.x; item < total && ok; item += gridDim.x, ++li) {
      const int buf = li & 1, use = li >> 1;
      if (use > 0 && !mbar_wait_warp(acc_empty(buf), (uint32_t)((use - 1) & 1), p.err, 52)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t d1 = tmem + (uint32_t)(buf * 2 * NB);
      const uint32_t d2 = d1 + NB;
      for (int kk = 0; kk < nk; ++kk, ++it) {
        const int s = (int)(it % kVStages);
        const uint32_t par = (uint32_t)((it / kVStages) & 1);
        if (!mbar_wait_warp(full(s), par, p.err, 53) || !mbar_wait_warp(conv(s), par, p.err, 55)) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (leader) {
          const uint64_t ad1 = sdesc(sbase + C::kOffA + s * kVABytes);
          const uint64_t ad2 = sdesc(sbase + C::kOffA + s * kVABytes + 128 * 128);
          const uint64_t bd = sdesc(sbase + C::kOffX + s * C::kXBytes);
#pragma unroll
          for (uint32_t k4 = 0; k4 < kVBK / 16; ++k4) {   // K = 16 per MMA, 32 bytes of each row
            const uint32_t acc = (kk | (int)k4) != 0;
            mma_bf16(d1, ad1 + 2 * k4, bd + 2 * k4, C::kIdesc, acc);
            mma_bf16(d2, ad2 + 2 * k4, bd + 2 * k4, C::kIdesc, acc);
          }
          mma_commit(empty(s));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) mma_commit(acc_full(buf));
      __syncwarp();
    }
    if (leader) {
      mma_commit(drain);
      drain_wait(drain, 0);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: thread = weight row (TMEM lane) ----------------
    const int l = warp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    for (int li = 0;; ++li) {
      const long item = blockIdx.x + (long)li * gridDim.x;
      if (item >= total) break;
      const int buf = li & 1;
      const int nt = (int)(item % p.n_ntiles);
      const int2 ti = __ldg(p.tile_info + item / p.n_ntiles);
      const int e = ti.x, row0 = ti.y;
      const int nrows = min(NB, __ldg(p.offsets + e + 1) - row0);
      const float sc = (p.alpha2 ? __ldg(p.alpha2 + e) : 1.f) * __ldg(p.gs + e);   // while the MMAs run
      if (!bar_red_and(2, 128, mbar_wait(acc_full(buf), (uint32_t)((li >> 1) & 1), p.err, 56))) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t t1 = tmem + lane_off + (uint32_t)(buf * 2 * NB);
      const int n1 = nt * kNH2 + l, n2 = n1 + 128;
      // 16 token columns at a time from each accumulator
      for (int c0 = 0; c0 < NB; c0 += 16) {
        float a1[16], a2[16];
        tmem_ld16(t1 + c0, a1);
        tmem_ld16(t1 + NB + c0, a2);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          if (c0 + t >= nrows) break;
          float* yr = p.y_out + (size_t)(row0 + c0 + t) * p.Mtot;
          if (n1 < p.Mtot) yr[n1] = a1[t] * sc;
          if (n2 < p.Mtot) yr[n2] = a2[t] * sc;
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(acc_empty(buf));
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// fct_kernel: the same FC2 (NVFP4 weights, bf16 H1) with the expanded weights
// in TMEM, for token tiles of 16 and 64 rows.
//
// The converters write each stage's bf16 A operand (256 weight rows x 64
// elements) straight into TMEM with tcgen05.st, and the MMAs read A from
// there (tcgen05.mma.kind::f16 with A in tensor memory: lane = weight row,
// two bf16 of K per column).  Shared memory then holds only the packed codes
// and the token rows, in stages of K = 128: the codes as 64-byte rows (64-byte
// swizzle), since a TMA box moves about one row per three cycles per SM
// whatever its width (32-byte rows held fcv_kernel's weight stream near
// 3 TB/s); each stage feeds two K = 64 A slots.  Each item's E4M3 scales
// (256 rows x K/16 bytes, one contiguous run) arrive in one bulk copy into a
// four-deep buffer instead of per-thread global loads.
//
// Both operands are f16 when the FC1 has recorded H1's largest magnitude m
// (h1max): a code times its E4M3 scale is a normal f16 (2^-10 to 2688 in
// magnitude, at most six significant bits), so one f16 multiply per pair
// makes the A operand; the token rows come from an f16 copy of H1 scaled by
// 2^-s (h1_to_f16_kernel, between the two GEMMs), s chosen so that m lands
// in [2^14, 2^15), and the epilogue multiplies by 2^s.  Every H1 value within 2^31 of
// m is then exact; smaller ones keep an absolute error below 2^-32 m.
// Without h1max (or with a non-finite m) the operands are bf16.  Each item's
// scales come in one bulk copy when the scale array is 16-byte aligned, else
// the converters read their row's bytes from global memory.
// TMEM: the two accumulator buffers (2 x 2 x NB columns), then A slots of
// 64 columns (32 per M = 128 half of the tile).  A converter warp writes the
// TMEM lanes of its quarter (warp % 4), so warp w converts weight rows
// 128 * ((w - 6) / 4) + 32 * (w % 4) + lane.  Warp roles as fcv_kernel.
// ---------------------------------------------------------------------------

namespace {

constexpr int kTScBuf = 4;                      // item scale buffers
constexpr int kTScBytes = 256 * 32;             // one item's scales, K <= 512
constexpr int kTBK = 128;                       // K elements per TMA stage
constexpr int kTRBytes = 256 * 64;              // packed codes of a stage: 256 rows x 64 bytes
template <int NB>
struct CfgT {
  static_assert(NB == 16 || NB == 64, "TMEM tiles: 16 or 64 token rows");
  static constexpr int kStages = NB == 16 ? 8 : 5;     // codes + token rows in shared memory
  static constexpr int kAccCols = 4 * NB;              // two buffers of two NB-column accumulators
  static constexpr int kASlots = (512 - kAccCols) / 64;
  static constexpr int kXBytes = NB * 256;             // bf16 token rows: two boxes of 64 elements
  static constexpr int kOffR = 0;
  static constexpr int kOffX = kOffR + kStages * kTRBytes;
  static constexpr int kOffSc = kOffX + kStages * kXBytes;
  static constexpr int kOffBar = kOffSc + kTScBuf * kTScBytes;
  // full, empty per stage; conv, aempty per A slot; scfull, scfree per scale
  // buffer; acc_full[2], acc_empty[2]; drain
  static constexpr int kNumBars = 2 * kStages + 2 * kASlots + 2 * kTScBuf + 5;
  static constexpr int kOffTm = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffTm + 16 + 1024;
  static constexpr uint32_t kTx = kXBytes + kTRBytes;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(kXBytes % 2048 == 0 && kOffX % 1024 == 0, "swizzle atoms");
  static_assert(kASlots >= 2, "TMEM budget");
  static constexpr uint32_t kIdesc = CfgV<NB>::kIdesc;
};

__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 consecutive TMEM columns of the warp's 32 lanes, one row per thread
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

}  // namespace

template <int NB>
__global__ void __launch_bounds__(kVThreads, 1)
fct_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
           const __grid_constant__ CUtensorMap tmXh, const FcvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using C = CfgT<NB>;
  constexpr int D1 = C::kStages, D2 = C::kASlots;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nk = p.K / kTBK;                    // TMA stages per item, two A slots each
  const int nsb = p.K / 16;                     // E4M3 scales per weight row

  const uint32_t sbase = saddr(smem);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto full = [&](int s) { return bar0 + 8 * s; };
  auto empty = [&](int s) { return bar0 + 8 * (D1 + s); };
  auto conv = [&](int s) { return bar0 + 8 * (2 * D1 + s); };
  auto aempty = [&](int s) { return bar0 + 8 * (2 * D1 + D2 + s); };
  auto scfull = [&](int b) { return bar0 + 8 * (2 * D1 + 2 * D2 + b); };
  auto scfree = [&](int b) { return bar0 + 8 * (2 * D1 + 2 * D2 + kTScBuf + b); };
  auto acc_full = [&](int b) { return bar0 + 8 * (2 * D1 + 2 * D2 + 2 * kTScBuf + b); };
  auto acc_empty = [&](int b) { return bar0 + 8 * (2 * D1 + 2 * D2 + 2 * kTScBuf + 2 + b); };
  const uint32_t drain = bar0 + 8 * (2 * D1 + 2 * D2 + 2 * kTScBuf + 4);
  uint32_t* tm_holder = reinterpret_cast<uint32_t*>(smem + C::kOffTm);

  if (tid == 0) {
    for (int s = 0; s < D1; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int s = 0; s < D2; ++s) {
      mbar_init(conv(s), 256);
      mbar_init(aempty(s), 1);
    }
    for (int b = 0; b < kTScBuf; ++b) {
      mbar_init(scfull(b), 1);
      mbar_init(scfree(b), 256);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 128);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tm_holder)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tm_holder;
  griddep_wait();
  const long total = *reinterpret_cast<volatile int*>(p.err) != 0
                         ? 0
                         : (long)__ldg(p.tile_offsets + p.E_loc) * p.n_ntiles;
  // f16 operands with H1 scaled by 2^-sig (the largest |H1|, recorded by the
  // FC1 before, brought into [2^14, 2^15)); bf16 without the record
  const uint32_t mbits = p.h1max ? *reinterpret_cast<const volatile unsigned*>(p.h1max) : 0x7F800000u;
  const bool f16m = mbits < 0x7F800000u;
  const int sig = mbits >= 0x00800000u ? min(113, max(-126, (int)(mbits >> 23) - 127 - 14)) : 0;
  const bool sc_bulk = (reinterpret_cast<uintptr_t>(p.ws) & 15u) == 0;

  if ((long)blockIdx.x >= total) {
    // no item for this CTA
  } else if (warp == 4) {
    // ---------------- TMA producer ----------------
    const bool leader = elect_one();
    const CUtensorMap* mx = f16m ? &tmXh : &tmX;
    long it = 0;
    int li = 0;
    bool ok = true;
    for (long item = blockIdx.x; item < total && ok; item += gridDim.x, ++li) {
      const int nt = (int)(item % p.n_ntiles);
      const int2 ti = __ldg(p.tile_info + item / p.n_ntiles);
      const int wrow = ti.x * p.Mtot + nt * kNH2;
      // the item's scales: rows wrow .. of K/16 bytes, one contiguous run
      const int b = li % kTScBuf;
      if (li >= kTScBuf && !mbar_wait_warp(scfree(b), (uint32_t)((li / kTScBuf - 1) & 1), p.err, 62)) break;
      if (leader) {
        if (sc_bulk) {
          const uint32_t bytes = (uint32_t)min(kNH2, p.Mtot - nt * kNH2) * (uint32_t)nsb;
          mbar_expect_tx(scfull(b), bytes);
          bulk_load(sbase + C::kOffSc + b * kTScBytes, p.ws + (size_t)wrow * nsb, bytes, scfull(b));
        } else {
          mbar_arrive(scfull(b));   // the converters read the scales themselves
        }
      }
      __syncwarp();
      for (int kk = 0; kk < nk; ++kk, ++it) {
        const int s = (int)(it % D1);
        const long r = it / D1;
        if (r > 0 && !mbar_wait_warp(empty(s), (uint32_t)((r - 1) & 1), p.err, 61)) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_expect_tx(full(s), C::kTx);
          const uint32_t xs = sbase + C::kOffX + s * C::kXBytes;
          tma_load_2d(sbase + C::kOffR + s * kTRBytes, &tmW, kk * (kTBK / 2), wrow, full(s));
          tma_load_2d(xs, mx, kk * kTBK, ti.y, full(s));
          tma_load_2d(xs + NB * 128, mx, kk * kTBK + 64, ti.y, full(s));
        }
        __syncwarp();
      }
    }
    // unwind: the copies of the last stages and scale buffers may still be landing
    if (leader) {
      for (long j = it - 1; j >= 0 && j >= it - D1; --j) drain_wait(full((int)(j % D1)), (uint32_t)((j / D1) & 1));
      for (int j = li - 1; j >= 0 && j >= li - kTScBuf; --j)
        drain_wait(scfull(j % kTScBuf), (uint32_t)((j / kTScBuf) & 1));
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ---------------- converters: thread = weight row n of the tile ----------------
    const int q = warp & 3, mt = (warp - 6) >> 2;
    const int n = mt * 128 + q * 32 + lane;
    const uint32_t tlane = (uint32_t)(q * 32) << 16;
    const int sw = (n >> 1) & 3;   // 64-byte swizzle: 16-byte chunk j of row n sits at chunk j ^ sw
    long it = 0, ia = 0;           // TMA stages, A slots
    int li = 0;
    bool ok = true;
    // The store of a half into TMEM is waited for, and the half handed to the
    // MMA, only after the next half has been converted, so the store's
    // latency overlaps that work (two register sets, one per half of a stage).
    int pend = -1;                 // A slot of the stored, not yet handed over half
    auto hand_over = [&]() {
      if (pend < 0) return;
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(conv(pend));
      pend = -1;
    };
    // the K = 64 half u of stage s1 (row n) as 32 bf16 pairs
    auto convert = [&](int s1, int u, uint32_t sc, uint32_t* a) {
      const uint8_t* raw = smem + C::kOffR + s1 * kTRBytes + n * 64;
      const uint4 q0 = *reinterpret_cast<const uint4*>(raw + (((2 * u) ^ sw) << 4));
      const uint4 q1 = *reinterpret_cast<const uint4*>(raw + (((2 * u + 1) ^ sw) << 4));
      const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      uint32_t f[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) f[j] = e4m3_pair_f16((sc >> (8 * j)) & 0xFFu);
      if (f16m) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {   // word j = elements 8j .. 8j + 7 (block j / 2)
          uint32_t d[4];
          e2m1x8_f16(w[j], d);
#pragma unroll
          for (int i = 0; i < 4; ++i) a[4 * j + i] = mul_f16x2(d[i], f[j >> 1]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t d[4];
          e2m1x8_f16(w[j], d);
#pragma unroll
          for (int i = 0; i < 4; ++i) a[4 * j + i] = scaled_bf16x2(d[i], f[j >> 1]);
        }
      }
    };
    uint32_t a0[32], a1[32];
    for (long item = blockIdx.x; item < total && ok; item += gridDim.x, ++li) {
      const int nt = (int)(item % p.n_ntiles);
      const bool valid = nt * kNH2 + n < p.Mtot;
      const int b = li % kTScBuf;
      if (!mbar_wait(scfull(b), (uint32_t)((li / kTScBuf) & 1), p.err, 65)) break;
      const uint8_t* srow = smem + C::kOffSc + b * kTScBytes + n * nsb;
      // unaligned scale array: the row's bytes straight from global memory
      const uint16_t* grow =
          sc_bulk ? nullptr
                  : reinterpret_cast<const uint16_t*>(
                        p.ws + ((size_t)__ldg(p.tile_info + item / p.n_ntiles).x * p.Mtot + nt * kNH2 + (valid ? n : 0)) *
                                   nsb);
      for (int kk = 0; kk < nk && ok; ++kk, ++it) {
        const int s1 = (int)(it % D1);
        if (!mbar_wait(full(s1), (uint32_t)((it / D1) & 1), p.err, 63)) {
          ok = false;
          break;
        }
        // the row's scale bytes of the stage: four per half (its 16-element blocks)
        uint2 sc = make_uint2(0u, 0u);
        if (valid && sc_bulk) {
          sc = *reinterpret_cast<const uint2*>(srow + 8 * kk);
        } else if (valid) {
          sc.x = (uint32_t)__ldg(grow + 4 * kk) | ((uint32_t)__ldg(grow + 4 * kk + 1) << 16);
          sc.y = (uint32_t)__ldg(grow + 4 * kk + 2) | ((uint32_t)__ldg(grow + 4 * kk + 3) << 16);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u, ++ia) {
          const int s2 = (int)(ia % D2);
          if (ia >= D2 && !mbar_wait(aempty(s2), (uint32_t)((ia / D2 - 1) & 1), p.err, 64)) {
            ok = false;
            break;
          }
          uint32_t* a = u ? a1 : a0;
          convert(s1, u, u ? sc.y : sc.x, a);
          hand_over();   // the previous half, stored while this one converted
          // TMEM column c of the slot holds elements 2c, 2c + 1 of the row
          tmem_st32(tmem + tlane + (uint32_t)(C::kAccCols + s2 * 64 + mt * 32), a);
          pend = s2;
        }
      }
      if (ok) mbar_arrive(scfree(b));
    }
    if (ok) {
      hand_over();
    } else if (pend >= 0) {
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    const bool leader = elect_one();
    // kind::f16 operand types: bf16 (1) or f16 (0) for A (bits 7..9) and B (10..12)
    const uint32_t idesc = f16m ? (C::kIdesc & ~((7u << 7) | (7u << 10))) : C::kIdesc;
    long it = 0, ia = 0;
    int li = 0;
    bool ok = true;
    for (long item = blockIdx.x; item < total && ok; item += gridDim.x, ++li) {
      const int buf = li & 1, use = li >> 1;
      if (use > 0 && !mbar_wait_warp(acc_empty(buf), (uint32_t)((use - 1) & 1), p.err, 66)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t d1 = tmem + (uint32_t)(buf * 2 * NB);
      const uint32_t d2 = d1 + NB;
      for (int kk = 0; kk < nk && ok; ++kk, ++it) {
        const int s1 = (int)(it % D1);
        if (!mbar_wait_warp(full(s1), (uint32_t)((it / D1) & 1), p.err, 67)) {
          ok = false;
          break;
        }
        for (int u = 0; u < 2; ++u, ++ia) {
          const int s2 = (int)(ia % D2);
          if (!mbar_wait_warp(conv(s2), (uint32_t)((ia / D2) & 1), p.err, 68)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          if (leader) {
            const uint32_t a1 = tmem + (uint32_t)(C::kAccCols + s2 * 64);
            // the half's token rows: the stage's u-th box of 64 elements
            const uint64_t bd = sdesc(sbase + C::kOffX + s1 * C::kXBytes + u * NB * 128);
#pragma unroll
            for (uint32_t k4 = 0; k4 < 4; ++k4) {   // K = 16 per MMA: 8 TMEM columns, 32 bytes of each token row
              const uint32_t acc = (kk | u | (int)k4) != 0;
              mma_bf16_ta(d1, a1 + 8 * k4, bd + 2 * k4, idesc, acc);
              mma_bf16_ta(d2, a1 + 32 + 8 * k4, bd + 2 * k4, idesc, acc);
            }
            mma_commit(aempty(s2));
            if (u == 1) mma_commit(empty(s1));
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      if (leader) mma_commit(acc_full(buf));
      __syncwarp();
    }
    if (leader) {
      mma_commit(drain);
      drain_wait(drain, 0);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: thread = weight row (TMEM lane) ----------------
    const int l = warp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    for (int li = 0;; ++li) {
      const long item = blockIdx.x + (long)li * gridDim.x;
      if (item >= total) break;
      const int buf = li & 1;
      const int nt = (int)(item % p.n_ntiles);
      const int2 ti = __ldg(p.tile_info + item / p.n_ntiles);
      const int e = ti.x, row0 = ti.y;
      const int nrows = min(NB, __ldg(p.offsets + e + 1) - row0);
      // while the MMAs run; f16 mode undoes H1's 2^-sig
      const float sc = (p.alpha2 ? __ldg(p.alpha2 + e) : 1.f) * __ldg(p.gs + e) * (f16m ? exp2i(sig) : 1.f);
      if (!bar_red_and(2, 128, mbar_wait(acc_full(buf), (uint32_t)((li >> 1) & 1), p.err, 69))) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t t1 = tmem + lane_off + (uint32_t)(buf * 2 * NB);
      const int n1 = nt * kNH2 + l, n2 = n1 + 128;
      for (int c0 = 0; c0 < NB; c0 += 16) {
        float a1[16], a2[16];
        tmem_ld16(t1 + c0, a1);
        tmem_ld16(t1 + NB + c0, a2);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          if (c0 + t >= nrows) break;
          float* yr = p.y_out + (size_t)(row0 + c0 + t) * p.Mtot;
          if (n1 < p.Mtot) yr[n1] = a1[t] * sc;
          if (n2 < p.Mtot) yr[n2] = a2[t] * sc;
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(acc_empty(buf));
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

template <int NB>
cudaError_t launch_fct_t(const FcvParams& p, const uint16_t* h_bf16, const uint16_t* h_f16, long S, int E_loc,
                         long max_tiles, cudaStream_t st) {
  using C = CfgT<NB>;
  CUtensorMap m[3];
  // packed codes in boxes of 64 bytes (128 codes) x 256 rows, 64-byte
  // swizzle; H1 bf16 in boxes of 64 elements x NB rows, 128-byte swizzle
  if (!make_map(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.w, (uint64_t)(p.K / 2), (uint64_t)E_loc * p.Mtot,
                (uint64_t)(p.K / 2), kTBK / 2, kNH2, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&m[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h_bf16, (uint64_t)p.K, (uint64_t)S, (uint64_t)p.K * 2,
                kVBK, NB, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, h_f16 ? h_f16 : h_bf16, (uint64_t)p.K, (uint64_t)S,
                (uint64_t)p.K * 2, kVBK, NB, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  FcvParams q = p;
  if (!h_f16) q.h1max = nullptr;   // no f16 copy: bf16 operands
  static int set_for[64];
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (dev >= 64 || set_for[dev] == 0) {
      cudaError_t err = cudaFuncSetAttribute(fct_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
      if (err != cudaSuccess) return err;
      if (dev < 64) set_for[dev] = 1;
    }
  }
  const long items = max_tiles * p.n_ntiles;
  const long grid = items < sm_count_w() ? items : sm_count_w();
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(fct_kernel<NB>, dim3((unsigned)grid), dim3(kVThreads), (size_t)C::kSmem, st, m[0], m[1], m[2], q);
}

template <int NB>
cudaError_t launch_fcv_t(const FcvParams& p, const uint16_t* h_bf16, long S, int E_loc, long max_tiles,
                         cudaStream_t st) {
  using C = CfgV<NB>;
  CUtensorMap m[2];
  // packed codes [E_loc * Mtot, K/2] bytes, boxes of 32 bytes (64 codes) x
  // 256 rows, no swizzle; H1 bf16 [S, K], boxes of 64 elements x NB rows,
  // 128-byte swizzle
  if (!make_map(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.w, (uint64_t)(p.K / 2), (uint64_t)E_loc * p.Mtot,
                (uint64_t)(p.K / 2), kVBK / 2, kNH2, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&m[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h_bf16, (uint64_t)p.K, (uint64_t)S, (uint64_t)p.K * 2,
                kVBK, NB, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static int set_for[64];
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (dev >= 64 || set_for[dev] == 0) {
      cudaError_t err = cudaFuncSetAttribute(fcv_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
      if (err != cudaSuccess) return err;
      if (dev < 64) set_for[dev] = 1;
    }
  }
  const long items = max_tiles * p.n_ntiles;
  const long grid = items < sm_count_w() ? items : sm_count_w();
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(fcv_kernel<NB>, dim3((unsigned)grid), dim3(kVThreads), (size_t)C::kSmem, st, m[0], m[1], p);
}

// the TMEM-operand kernel takes the 16- and 64-row tiles (an item's scales,
// 256 rows of K/16 bytes, fit its 8 KB buffers)
bool fct_applies(int K, int tile_rows) { return (tile_rows == kTok || tile_rows == 64) && K <= 512 && K % kTBK == 0; }

// H1 (bf16 [S, I], the first meta[0] rows in use) as f16 times 2^-sig, sig
// from the largest magnitude the FC1 recorded (as fct_kernel derives it);
// 8 elements per thread.
__global__ void __launch_bounds__(256) h1_to_f16_kernel(const uint4* __restrict__ h, const int32_t* meta,
                                                        const unsigned* h1max, int I, uint4* __restrict__ hf) {
  griddep_wait();   // H1 and its maximum are the predecessor's output
  griddep_launch_dependents();
  const uint32_t mbits = *reinterpret_cast<const volatile unsigned*>(h1max);
  if (mbits >= 0x7F800000u) return;   // not finite: the FC2 takes bf16 operands
  const int sig = mbits >= 0x00800000u ? min(113, max(-126, (int)(mbits >> 23) - 127 - 14)) : 0;
  const float sc = exp2i(-sig);
  const long n8 = (long)__ldg(meta) * (I / 8);
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n8; i += (long)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(h + i);
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = pack_f16x2(bf16_lo(in[j]) * sc, bf16_hi(in[j]) * sc);
    hf[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_h1_to_f16(const uint16_t* h_bf16, long S, int I, const int32_t* meta, const unsigned* h1max,
                             uint16_t* h_f16, cudaStream_t st) {
  const long n8 = S * (I / 8);
  const long grid = std::min<long>((n8 + 255) / 256, 4L * sm_count_w());
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(h1_to_f16_kernel, dim3((unsigned)grid), dim3(256), 0, st, (const uint4*)h_bf16, meta, h1max, I,
                    (uint4*)h_f16);
}

cudaError_t launch_fcv(const FcvParams& p, const uint16_t* h_bf16, const uint16_t* h_f16, long S, int E_loc,
                       int tile_rows, long max_tiles, cudaStream_t st) {
  if (S <= 0) return cudaSuccess;
  if (tile_rows == 128) return launch_fcv_t<128>(p, h_bf16, S, E_loc, max_tiles, st);
  const bool ta = fct_applies(p.K, tile_rows);
  if (tile_rows == 64)
    return ta ? launch_fct_t<64>(p, h_bf16, h_f16, S, E_loc, max_tiles, st)
              : launch_fcv_t<64>(p, h_bf16, S, E_loc, max_tiles, st);
  if (tile_rows == kTok)
    return ta ? launch_fct_t<kTok>(p, h_bf16, h_f16, S, E_loc, max_tiles, st)
              : launch_fcv_t<kTok>(p, h_bf16, S, E_loc, max_tiles, st);
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// The failure path's self-test: the bounded wait of the GEMM kernels on a
// barrier phase that no arrival completes.  It gives up after kWaitNs,
// records `code` in *status and returns.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(32) wait_selftest_kernel(int* status, int code) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(saddr(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (mbar_wait(saddr(&bar), 0, status, code)) atomicExch(status, -1);   // cannot complete
  }
}

cudaError_t launch_wait_selftest(int* status, int code, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, code);
  return cudaGetLastError();
}

}  // namespace situ
