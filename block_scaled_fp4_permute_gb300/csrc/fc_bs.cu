// fc_bs.cu -- FC1 (gate/up + SiTU) and FC2 for MXFP8 activations x MXFP4
// weights (w4a8) on the block-scaled tensor cores:
// tcgen05.mma.kind::mxf8f6f4.block_scale, E4M3 x E2M1 with one UE8M0 scale
// per 32 elements of K on both operands, fp32 accumulation in TMEM.
//
// A persistent kernel: one CTA per SM walks the work items (a 128-token
// tile of one local expert x an N tile of weight rows; FC1 N = 96 gate rows
// + the 96 matching up rows, FC2 N = 224 rows of H), K in stages of 128.
//
// Block scales travel in "scale blocks": 512 bytes holding the four UE8M0
// bytes (the four 32-element K blocks of one stage) of 128 rows, as 32
// 16-byte rows in which row i holds the words of rows i, i+32, i+64, i+96 --
// the source layout of tcgen05.cp.32x128b.warpx4, which copies a block
// into four TMEM columns of every 32-lane quarter, where the MMA reads it.
// The activation scales are written in that layout per token tile by the
// gather (FC1) and by FC1's epilogue (FC2); the weight scales are packed
// into it once per weight set (pack_scales), so every stage's scales are two
// contiguous bulk copies.
//
// Warp roles:
//   * warp 0 (one lane), TMA producer: per stage the token tile's E4M3 rows
//     (128 x 128 B, 128-byte swizzle), the weight rows' E2M1 codes and the
//     stage's scale blocks (1 for A, 2 for B).  The weights are read with the
//     tensor-map type that expands each 8-byte group of 16 packed codes into a
//     16-byte slot in shared memory, the operand layout the MMA takes for
//     4-bit types next to 8-bit ones, so the packed weights go from HBM to the
//     tensor core untouched;
//   * warp 1 allocates all 512 TMEM columns (two accumulators plus 12 scale
//     columns per stage); one lane copies each stage's scale blocks into TMEM
//     and issues four MMAs (M = 128, K = 32), the k-th taking byte k of the
//     scale words, committing the stage back to the producer and each
//     finished accumulator to the epilogue;
//   * warps 4..7 and 8..11, epilogue (each thread one token row), one
//     warpgroup per accumulator, so that two items drain while the MMAs run
//     on: FC1 applies the per-expert alphas and SiTU to each gate/up column
//     pair and writes H1 as MXFP8 (E4M3 rows + scale blocks), FC2's A
//     operand as it stands; FC2 writes alpha2 * acc as fp32 through a small
//     shared staging block, so that Y leaves in whole 128-byte row segments.
// K (H for FC1, I for FC2) must be a multiple of 128.  Every mbarrier wait
// is bounded; on expiry the CTA records an error code in the device status
// word, waits (bounded) for its copies and MMAs in flight, releases TMEM
// and returns.
#include "situ_internal.h"
#include "../../include/situ_moe.h"
#include "tc_common.cuh"

namespace situ {

using namespace tc;

namespace {

constexpr int kBM = 128;         // tokens per tile (MMA M, TMEM lanes)
constexpr int kBK = 128;         // K elements per stage
constexpr int kThreads = 384;
constexpr int kTmemCols = 512;
constexpr int kSfBlock = 512;    // one scale block: 128 rows x 4 K blocks
// LO: bf16 token rows as hi + lo MXFP8 rows (split_hl32), two A tiles per
// stage and two MMAs per K block into the same accumulator.
template <bool FC1, bool LO>
struct Cfg {
  static constexpr int BN = FC1 ? 192 : 224;        // MMA N
  static constexpr int NH = FC1 ? BN / 2 : BN;      // rows per weight box
  static constexpr int kNA = LO ? 2 : 1;            // A tiles per stage
  static constexpr int kStages = LO ? 3 : (FC1 ? 5 : 4);
  static constexpr int kATile = kBM * kBK;          // 16 KB of E4M3
  static constexpr int kABytes = kNA * kATile;
  static constexpr int kBBytes = BN * kBK;          // E2M1 in 16-byte slots of 16 codes
  static constexpr int kBTx = BN * kBK / 2;         // bytes the weight loads transfer (packed)
  static constexpr int kSfBytes = (kNA + 2) * kSfBlock;   // A block(s), B rows 0..127, B rows 128..255
  static constexpr int kSfColsPerStage = 4 * (kNA + 2);
  static constexpr int kTx = kABytes + kBTx + kSfBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSF = kOffB + kStages * kBBytes;
  // FC2: per epilogue warp a 32 x 32 fp32 staging block (rows padded to
  // 144 bytes)
  static constexpr int kYRow = 144;
  static constexpr int kOffY = kOffSF + kStages * kSfBytes;
  static constexpr int kYBytes = FC1 ? 0 : 8 * 32 * kYRow;
  static constexpr int kOffBar = kOffY + kYBytes;
  // full, empty per stage; acc_full[2], acc_empty[2]; drain
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kOffTm = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffTm + 16 + 1024;  // + alignment slack
  static constexpr int kSfCol0 = 2 * BN;            // TMEM: accumulators [0, 2 BN), then scales
  static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  // Instruction descriptor, block-scaled kinds: A = E4M3 (0), B = E2M1 (5),
  // both K-major, N >> 3 at bit 17, UE8M0 scales (bit 23), M >> 4 at bit
  // 24; the B and A scale byte selectors sit at bits 4..5 and 29..30.
  static constexpr uint32_t kIdesc = (0u << 7) | (5u << 10) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) |
                                     ((uint32_t)(kBM >> 4) << 24);
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

// Descriptor of a scale block: no swizzle, 8-row groups of 128 contiguous
// bytes.
__device__ __forceinline__ uint64_t sf_desc(uint32_t a) {
  uint64_t d = 0;
  d |= (uint64_t)((a >> 4) & 0x3FFFu);
  d |= (uint64_t)(128u >> 4) << 32;   // stride byte offset
  d |= (uint64_t)1u << 46;            // descriptor version
  return d;
}
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
// contiguous global -> shared copy on the TMA engine, completing on an mbarrier
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Short bounded wait used only while unwinding (no error code recorded).
__device__ __forceinline__ void drain_wait(uint32_t a, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try(a, parity))
    if (globaltimer() - t0 > kWaitNs) return;
}

// out[0..3] += v (fp32 vector reduction in L2)
__device__ __forceinline__ void red_add_v4(float* out, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(out), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// byte offset of (row r, K block kb of the stage) inside a scale block
__device__ __forceinline__ uint32_t sf_offset(int r, int kb) {
  return (uint32_t)((r & 31) * 16 + ((r >> 5) & 3) * 4 + kb);
}

}  // namespace

template <bool FC1, bool LO>
__global__ void __launch_bounds__(kThreads, 1)
fcq_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAl,
           const __grid_constant__ CUtensorMap tmB, const FcqParams p) {
  using C = Cfg<FC1, LO>;
  constexpr int kSfColsPerStage = C::kSfColsPerStage;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int nk = p.K / kBK;

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
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tm_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tm_holder;
  // the set-up above overlaps the predecessor's tail (programmatic launch).
  // The successor is not released early: launched at the start of this
  // persistent kernel, FC2's grid or the combine's 57 k CTAs slowed the w4a8
  // prefill step from 1.11 to 1.24 ms.
  griddep_wait();
  // no items when an earlier kernel's wait ran out
  const long total = *reinterpret_cast<volatile int*>(p.err) != 0
                         ? 0
                         : (long)__ldg(p.tile_offsets + p.E_loc) * p.n_ntiles;

  if ((long)blockIdx.x >= total) {
    // no item for this CTA
  } else if (warp == 0) {
    // ---------------- TMA producer ----------------
    // the whole warp walks the loop; one elected lane issues the copies
    const bool leader = elect_one();
    long it = 0;
    bool ok = true;
    // the tile of the next item is read one item ahead, so that its latency
    // hides behind this item's copies (FC2's items are three stages long)
    int2 ti_next = __ldg(p.tile_info + blockIdx.x / p.n_ntiles);
    for (long item = blockIdx.x; item < total && ok; item += gridDim.x) {
      const int tile = (int)(item / p.n_ntiles), ntile = (int)(item % p.n_ntiles);
      const int2 ti = ti_next;
      if (item + gridDim.x < total) ti_next = __ldg(p.tile_info + (item + gridDim.x) / p.n_ntiles);
      const int e = ti.x, row0 = ti.y;
      const int wrow = e * p.Mtot + ntile * C::NH;
      const uint8_t* xsb = p.xsp + (size_t)tile * nk * kSfBlock;
      const uint8_t* xsb_lo = LO ? p.xsp_lo + (size_t)tile * nk * kSfBlock : nullptr;
      const uint8_t* wsb = p.wsp + ((size_t)e * p.n_ntiles + ntile) * nk * (2 * kSfBlock);
      for (int kk = 0; kk < nk; ++kk, ++it) {
        const int s = (int)(it % kStages);
        const long r = it / kStages;
        if (r > 0 && !mbar_wait_warp(empty(s), (uint32_t)((r - 1) & 1), p.err, 21)) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_expect_tx(full(s), C::kTx);
          const uint32_t b_smem = sbase + C::kOffB + s * C::kBBytes;
          const uint32_t sf_smem = sbase + C::kOffSF + s * C::kSfBytes;
          tma_load_2d(sbase + C::kOffA + s * C::kABytes, &tmA, kk * kBK, row0, full(s));
          if (LO) tma_load_2d(sbase + C::kOffA + s * C::kABytes + C::kATile, &tmAl, kk * kBK, row0, full(s));
          tma_load_2d(b_smem, &tmB, kk * kBK, wrow, full(s));
          if (FC1) tma_load_2d(b_smem + C::NH * kBK, &tmB, kk * kBK, wrow + p.I, full(s));
          bulk_load(sf_smem, xsb + (size_t)kk * kSfBlock, kSfBlock, full(s));
          if (LO) bulk_load(sf_smem + kSfBlock, xsb_lo + (size_t)kk * kSfBlock, kSfBlock, full(s));
          bulk_load(sf_smem + C::kNA * kSfBlock, wsb + (size_t)kk * 2 * kSfBlock, 2 * kSfBlock, full(s));
        }
        __syncwarp();
      }
    }
    // unwind: the loads of the last stages may still be landing
    if (leader)
      for (long j = it - 1; j >= 0 && j >= it - kStages; --j)
        drain_wait(full((int)(j % kStages)), (uint32_t)((j / kStages) & 1));
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- scale copies + MMA issuer ----------------
    // the whole warp walks the loop; one elected lane issues
    const bool leader = elect_one();
    long it = 0;
    int li = 0;
    bool ok = true;
    for (long item = blockIdx.x; item < total && ok; item += gridDim.x, ++li) {
      const int buf = li & 1, use = li >> 1;
      if (use > 0 && !mbar_wait_warp(acc_empty(buf), (uint32_t)((use - 1) & 1), p.err, 22)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t d = tmem + (uint32_t)(buf * C::BN);
      for (int kk = 0; kk < nk; ++kk, ++it) {
        const int s = (int)(it % kStages);
        if (!mbar_wait_warp(full(s), (uint32_t)((it / kStages) & 1), p.err, 23)) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (leader) {
          const uint32_t sf_smem = sbase + C::kOffSF + s * C::kSfBytes;
          const uint32_t sfa = tmem + (uint32_t)(C::kSfCol0 + s * kSfColsPerStage);
          const uint32_t sfb = sfa + 4 * C::kNA;
          tmem_cp_sf(sfa, sf_desc(sf_smem));
          if (LO) tmem_cp_sf(sfa + 4, sf_desc(sf_smem + kSfBlock));
          tmem_cp_sf(sfb, sf_desc(sf_smem + C::kNA * kSfBlock));
          tmem_cp_sf(sfb + 4, sf_desc(sf_smem + (C::kNA + 1) * kSfBlock));
          const uint64_t ad = sdesc(sbase + C::kOffA + s * C::kABytes);
          const uint64_t bd = sdesc(sbase + C::kOffB + s * C::kBBytes);
#pragma unroll
          for (uint32_t k4 = 0; k4 < kBK / 32; ++k4) {   // +32 bytes along K per instruction
            const uint32_t idesc = C::kIdesc | (k4 << 4) | (k4 << 29);
            mma_bs(d, ad + 2 * k4, bd + 2 * k4, idesc, sfa, sfb, (kk | (int)k4) != 0);
            // the lo rows of the same tokens add into the same accumulator
            if (LO) mma_bs(d, ad + (uint64_t)(C::kATile >> 4) + 2 * k4, bd + 2 * k4, idesc, sfa + 4, sfb, 1u);
          }
          mma_commit(empty(s));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) mma_commit(acc_full(buf));
      __syncwarp();
    }
    // unwind: every MMA and scale copy issued so far has completed
    if (leader) {
      mma_commit(drain);
      drain_wait(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- epilogue: thread = token row (TMEM lane) ----------------
    // warpgroup buf drains accumulator buf, i.e. this CTA's items buf, buf + 2, ...
    const int buf = (warp - 4) >> 2;
    const int quarter = warp & 3;        // the TMEM lanes a warp may read: 32 * (warp % 4) ..
    const int m = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    for (int li = buf;; li += 2) {
      const long item = blockIdx.x + (long)li * gridDim.x;
      if (item >= total) break;
      const int tile = (int)(item / p.n_ntiles), ntile = (int)(item % p.n_ntiles);
      const int2 ti = __ldg(p.tile_info + tile);
      const int e = ti.x, row0 = ti.y;
      const int nrows = min(kBM, __ldg(p.offsets + e + 1) - row0);
      const int nbase = ntile * C::NH;
      // FC2's output scale, loaded while the MMAs run
      const float a2 = (!FC1 && p.alpha2) ? __ldg(p.alpha2 + e) : 1.f;
      // warp-uniform outcome: the tcgen05.ld below are .sync.aligned
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full(buf), (uint32_t)((li >> 1) & 1), p.err, 26))) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t trow = tmem + lane_off + (uint32_t)(buf * C::BN);
      const bool vrow = m < nrows;
      const size_t row = (size_t)(row0 + (vrow ? m : 0));
      if (FC1) {
        const float ag = p.alpha_g ? __ldg(p.alpha_g + e) : 1.f;
        const float au = p.alpha_u ? __ldg(p.alpha_u + e) : 1.f;
        const float bt = __ldg(p.beta + e), btl = __ldg(p.beta_lin + e);
        const int nkh = p.I / kBK;   // FC2's stages: H1's scale blocks per tile
        const float rw = (p.topk_fc1 && vrow) ? __ldg(p.topk_weights + __ldg(p.permuted_src + row)) : 1.f;
        for (int c0 = 0; c0 < C::NH; c0 += 32) {
          float gt[32], up[32];
          tmem_ld16(trow + c0, gt);
          tmem_ld16(trow + c0 + 16, gt + 16);
          tmem_ld16(trow + C::NH + c0, up);
          tmem_ld16(trow + C::NH + c0 + 16, up + 16);
          const int i0 = nbase + c0;
          if (!vrow || i0 >= p.I) continue;
          float v[32];
          float amax = 0.f;
          with_act(p.act_kind, bt, btl, [&](auto act) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              v[j] = act(gt[j] * ag, up[j] * au) * rw;
              if (LO) v[j] = bf16_lo(f32x2_to_bf16x2(v[j], 0.f));   // w4a16: H1 is bf16
              amax = fmaxf(amax, fabsf(v[j]));
            }
          });
          const int b = i0 / 32;   // K block of FC2
          const size_t sfo = ((size_t)tile * nkh + b / 4) * kSfBlock + sf_offset(m, b & 3);
          uint32_t qv[8];
          if (LO) {
            // bf16 H1 as FC2's hi / lo rows
            uint32_t ql[8];
            const uint32_t sb = split_hl32(v, qv, ql);
            uint4* dl = reinterpret_cast<uint4*>(p.hq_lo + row * p.hq_stride + i0);
            dl[0] = make_uint4(ql[0], ql[1], ql[2], ql[3]);
            dl[1] = make_uint4(ql[4], ql[5], ql[6], ql[7]);
            p.hsp[sfo] = (uint8_t)(sb & 0xFFu);
            p.hsp_lo[sfo] = (uint8_t)(sb >> 8);
          } else {
            // MXFP8 of the 32-element block: the smallest e with amax * 2^-e <= 448
            const int ex = mxfp8_exponent(amax);
            const float sc = exp2i(-ex);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              qv[j] = f32x2_to_e4m3x2(v[4 * j] * sc, v[4 * j + 1] * sc) |
                      (f32x2_to_e4m3x2(v[4 * j + 2] * sc, v[4 * j + 3] * sc) << 16);
            p.hsp[sfo] = (uint8_t)(ex + 127);
          }
          uint4* dst = reinterpret_cast<uint4*>(p.hq + row * p.hq_stride + i0);
          dst[0] = make_uint4(qv[0], qv[1], qv[2], qv[3]);
          dst[1] = make_uint4(qv[4], qv[5], qv[6], qv[7]);
        }
      } else if (p.y_scale == nullptr) {
        // this warp's staging block; the warp owns tile rows 32 quarter .. + 31
        uint8_t* yst = smem + C::kOffY + (warp - 4) * 32 * C::kYRow;
        const int wrow0 = quarter * 32;
        // fused combine: lane l knows the token and routing weight of row wrow0 + l
        int my_t = 0;
        float my_w = 0.f;
        if (p.fuse && wrow0 + lane < nrows) {
          const int src = __ldg(p.permuted_src + row0 + wrow0 + lane);
          my_t = src / p.top_k;
          my_w = p.topk_fc1 ? 1.f : __ldg(p.topk_weights + src);   // else the weight is in H1
        }
        for (int c0 = 0; c0 < C::BN; c0 += 32) {
          float acc[32];
          tmem_ld16(trow + c0, acc);
          tmem_ld16(trow + c0 + 16, acc + 16);
          // own row into the staging block ...
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(yst + lane * C::kYRow + 16 * q) =
                make_float4(acc[4 * q] * a2, acc[4 * q + 1] * a2, acc[4 * q + 2] * a2, acc[4 * q + 3] * a2);
          __syncwarp();
          // ... and out as 4 rows x 128 bytes per instruction
          const int n = nbase + c0 + 4 * (lane & 7);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = 4 * j + (lane >> 3);
            const float4 v = *reinterpret_cast<const float4*>(yst + r * C::kYRow + 16 * (lane & 7));
            if (p.fuse) {
              const int t = __shfl_sync(0xffffffffu, my_t, r);
              const float w = __shfl_sync(0xffffffffu, my_w, r);
              if (wrow0 + r < nrows && n < p.Mtot)
                red_add_v4(p.out_acc + (size_t)t * p.Mtot + n, v.x * w, v.y * w, v.z * w, v.w * w);
            } else if (wrow0 + r < nrows && n < p.Mtot) {
              *reinterpret_cast<float4*>(p.y_out + (size_t)(row0 + wrow0 + r) * p.Mtot + n) = v;
            }
          }
          __syncwarp();
        }
      } else {
        // Y as f16 rows with a power-of-two scale per 32 columns: half the
        // bytes of the fp32 rows that the combine reads back
        uint8_t* yst = smem + C::kOffY + (warp - 4) * 32 * C::kYRow;
        const int wrow0 = quarter * 32;
        uint16_t* y16 = reinterpret_cast<uint16_t*>(p.y_out);
        for (int c0 = 0; c0 < C::BN; c0 += 32) {
          float acc[32];
          tmem_ld16(trow + c0, acc);
          tmem_ld16(trow + c0 + 16, acc + 16);
          float amax = 0.f;
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            acc[q] *= a2;
            amax = fmaxf(amax, fabsf(acc[q]));
          }
          const int ex = y16_exponent(amax);
          const float inv = exp2i(-ex);
          // own row (64 bytes) into the staging block ...
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(yst + lane * C::kYRow + 16 * q) =
                make_uint4(pack_f16x2(acc[8 * q] * inv, acc[8 * q + 1] * inv),
                           pack_f16x2(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv),
                           pack_f16x2(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv),
                           pack_f16x2(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv));
          const int n0 = nbase + c0;
          // block-major scales: the warp's 32 rows are 32 consecutive bytes
          if (m < nrows && n0 < p.Mtot) p.y_scale[(size_t)(n0 / 32) * p.ys_rows + (row0 + m)] = (uint8_t)(ex + 127);
          __syncwarp();
          // ... and out as 8 rows x 64 bytes per instruction
          const int n = n0 + 8 * (lane & 3);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = 8 * j + (lane >> 2);
            const uint4 v = *reinterpret_cast<const uint4*>(yst + r * C::kYRow + 16 * (lane & 3));
            if (wrow0 + r < nrows && n < p.Mtot)
              *reinterpret_cast<uint4*>(y16 + (size_t)(row0 + wrow0 + r) * p.Mtot + n) = v;
          }
          __syncwarp();
        }
      }
      // this accumulator may be overwritten by the item after next
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(acc_empty(buf));
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// gather8: the token rows of the block-scaled prefill tiles in expert order.
// bf16 rows are split into hi / lo MXFP8 rows per row, their UE8M0 scales
// written into the tile's scale blocks; MXFP8 rows are copied per token
// (gather8_tok_kernel below).
// ---------------------------------------------------------------------------

// One unit of work: 16 rows of a tile, which the CTAs walk grid-stride, so
// that the last wave is not left to a few CTAs (the EP shard's gather 0.048
// -> 0.033 ms against a CTA per 128-row tile).
constexpr int kGatherRowsHL = 16;
__device__ __forceinline__ void gather8_hl_rows(const Gather8Params& p, int tile, int m0) {
  const int2 ti = __ldg(p.tile_info + tile);
  const int row0 = ti.y;
  const int nrows = min(kBM, __ldg(p.offsets + ti.x + 1) - row0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.K, nsb = K / 32, nk = K / kBK;
  uint8_t* blocks = p.xsp + (size_t)tile * nk * kSfBlock;
  // bf16 rows: hi / lo E4M3 rows (split_hl32), one lane per 32-element block
  uint8_t* blocks_lo = p.xsp_lo + (size_t)tile * nk * kSfBlock;
  for (int m = m0 + warp; m < m0 + kGatherRowsHL; m += 8) {
    if (m < nrows) {
      const long r = row0 + m;
      const long t = __ldg(p.permuted_src + r) / p.top_k;
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.x_bf16) + (size_t)t * K * 2);
      uint4* dh = reinterpret_cast<uint4*>(p.x8 + (size_t)r * K);
      uint4* dl = reinterpret_cast<uint4*>(p.x8_lo + (size_t)r * K);
      for (int b = lane; b < nsb; b += 32) {
        float v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w = __ldg(src + 4 * b + q);
          const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v[8 * q + 2 * j] = bf16_lo(u[j]);
            v[8 * q + 2 * j + 1] = bf16_hi(u[j]);
          }
        }
        uint32_t hi[8], lo[8];
        const uint32_t sb = split_hl32(v, hi, lo);
        dh[2 * b] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        dh[2 * b + 1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
        dl[2 * b] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        dl[2 * b + 1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        const size_t o = (size_t)(b / 4) * kSfBlock + sf_offset(m, b & 3);
        blocks[o] = (uint8_t)(sb & 0xFFu);
        blocks_lo[o] = (uint8_t)(sb >> 8);
      }
    } else {
      // rows past the expert's end: finite (2^-127) scales
      for (int kk = lane; kk < nk; kk += 32) {
        *reinterpret_cast<uint32_t*>(blocks + (size_t)kk * kSfBlock + sf_offset(m, 0)) = 0u;
        *reinterpret_cast<uint32_t*>(blocks_lo + (size_t)kk * kSfBlock + sf_offset(m, 0)) = 0u;
      }
    }
  }
}

__global__ void __launch_bounds__(256) gather8_kernel(const Gather8Params p) {
  griddep_wait();   // the tile table and the activations
  constexpr int per = kBM / kGatherRowsHL;
  const int units = __ldg(p.tile_offsets + p.E_loc) * per;
  for (int u = blockIdx.x; u < units; u += gridDim.x) gather8_hl_rows(p, u / per, (u % per) * kGatherRowsHL);
}

// MXFP8 rows by token, a warp per token: token t's E4M3 row is read once
// and written to the rows of all its kept slots (lane j < top_k holds slot
// j's row, which the others take by shuffle).  The scale blocks are then
// written per tile, each as whole 512-byte blocks: lane i of the tile's warp
// holds rows i, i + 32, i + 64 and i + 96, whose words for one stage are the
// 16 bytes at 16 i of the stage's block.  Their words come from the
// token-major scale rows; the padding rows of partly filled tiles get finite
// (2^-127) scales.
constexpr int kGather8TokWarps = 4;
constexpr int kGather8TokUnroll = 8;   // 16-byte pieces per lane per pass
__global__ void __launch_bounds__(32 * kGather8TokWarps) gather8_tok_kernel(const Gather8Params p) {
  griddep_wait();   // the permute's outputs and the activations
  const int lane = threadIdx.x & 31;
  const long gw = (long)blockIdx.x * kGather8TokWarps + (threadIdx.x >> 5);
  const long nw = (long)gridDim.x * kGather8TokWarps;
  const int K = p.K, nk = K / kBK, n16 = K / 16, top_k = p.top_k;
  const int n_tiles = __ldg(p.tile_offsets + p.E_loc);
  for (long tile = gw; tile < n_tiles; tile += nw) {
    const int2 ti = __ldg(p.tile_info + tile);
    const int nrows = min(kBM, __ldg(p.offsets + ti.x + 1) - ti.y);
    const uint8_t* srow[4];
    bool has[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int m = lane + 32 * q;
      has[q] = m < nrows;
      srow[q] = p.x_s + (size_t)(has[q] ? __ldg(p.permuted_src + ti.y + m) / top_k : 0) * (K / 32);
    }
    uint4* blocks = reinterpret_cast<uint4*>(p.xsp + (size_t)tile * nk * kSfBlock) + lane;
    for (int kk = 0; kk < nk; ++kk) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint8_t* ss = srow[q] + 4 * kk;
        w[q] = !has[q] ? 0u
               : p.s_vec ? __ldg(reinterpret_cast<const uint32_t*>(ss))
                         : (uint32_t)__ldg(ss) | ((uint32_t)__ldg(ss + 1) << 8) | ((uint32_t)__ldg(ss + 2) << 16) |
                               ((uint32_t)__ldg(ss + 3) << 24);
      }
      blocks[(size_t)kk * (kSfBlock / 16)] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  for (long t = gw; t < p.T; t += nw) {
    const int my_r = lane < top_k ? __ldg(p.slot_to_row + t * top_k + lane) : -1;
    const uint4* src = reinterpret_cast<const uint4*>(p.x_q + (size_t)t * K);
    for (int i0 = 0; i0 < n16; i0 += 32 * kGather8TokUnroll) {
      uint4 v[kGather8TokUnroll];
#pragma unroll
      for (int u = 0; u < kGather8TokUnroll; ++u) {
        const int i = i0 + 32 * u + lane;
        if (i < n16) v[u] = __ldg(src + i);
      }
      for (int j = 0; j < top_k; ++j) {
        const int r = __shfl_sync(0xffffffffu, my_r, j);
        if (r < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(p.x8 + (size_t)r * K);
#pragma unroll
        for (int u = 0; u < kGather8TokUnroll; ++u) {
          const int i = i0 + 32 * u + lane;
          if (i < n16) dst[i] = v[u];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// pack_scales: a weight's UE8M0 scales [E_loc, Mtot, K/32] rearranged into
// the scale blocks of the GEMM's N tiles: per (expert, N tile, stage) two
// blocks for tile rows 0..127 and 128..255.  FC1 tiles are NH gate rows
// followed by the NH matching up rows.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) pack_scales_kernel(const uint8_t* ws, int Mtot, int K, int I, int fc1,
                                                          int nh, int n_ntiles, int E_loc, int vec, uint8_t* out) {
  const int nk = K / kBK, nsb = K / 32;
  const long nblk = (long)E_loc * n_ntiles * nk;
  for (long blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
    const int kk = (int)(blk % nk);
    const int ntile = (int)((blk / nk) % n_ntiles);
    const int e = (int)(blk / ((long)nk * n_ntiles));
    uint8_t* dst = out + blk * (2 * kSfBlock);
    const int n = threadIdx.x;   // tile row 0..255
    int wr;
    bool v;
    if (fc1) {
      const int i = ntile * nh + (n < nh ? n : n - nh);
      v = n < 2 * nh && i < I;
      wr = (n < nh ? 0 : I) + i;
    } else {
      wr = ntile * nh + n;
      v = n < nh && wr < Mtot;
    }
    uint32_t w = 0u;
    if (v) {
      const uint8_t* s = ws + ((size_t)e * Mtot + wr) * nsb + 4 * kk;
      w = vec ? __ldg(reinterpret_cast<const uint32_t*>(s))
              : (uint32_t)__ldg(s) | ((uint32_t)__ldg(s + 1) << 8) | ((uint32_t)__ldg(s + 2) << 16) |
                    ((uint32_t)__ldg(s + 3) << 24);
    }
    *reinterpret_cast<uint32_t*>(dst + (n >> 7) * kSfBlock + sf_offset(n, 0)) = w;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

int sm_count() {
  static std::atomic<int> n[64];   // SM count per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && n[dev] > 0) return n[dev];
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
  if (dev < 64) n[dev] = v;
  return v;
}

template <bool FC1, bool LO>
cudaError_t launch_fcq_t(const FcqParams& p, const CUtensorMap& a, const CUtensorMap& al, const CUtensorMap& b,
                         long max_tiles, cudaStream_t st) {
  using C = Cfg<FC1, LO>;
  static int set_for[64];
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (dev >= 64 || set_for[dev] == 0) {
      cudaError_t err =
          cudaFuncSetAttribute(fcq_kernel<FC1, LO>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
      if (err != cudaSuccess) return err;
      if (dev < 64) set_for[dev] = 1;
    }
  }
  const long items = max_tiles * p.n_ntiles;   // upper bound; the kernel reads the true count
  const long grid = items < sm_count() ? items : sm_count();
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(fcq_kernel<FC1, LO>, dim3((unsigned)grid), dim3(kThreads), (size_t)C::kSmem, st, a, al, b, p);
}

}  // namespace

int fcq_n_rows(bool fc1) { return fc1 ? Cfg<true, false>::NH : Cfg<false, false>::NH; }

bool fcq_supported(int H, int I, const void* w1, const void* w2) {
  // the 4-bit tensor-map type wants rows of a multiple of 128 codes and a
  // 32-byte aligned base
  auto al = [](const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; };
  return H % kBK == 0 && I % kBK == 0 && al(w1, 32) && al(w2, 32);
}

size_t fcq_act_scale_bytes(long max_tiles, int K) { return (size_t)max_tiles * (K / kBK) * kSfBlock; }

size_t packed_scale_bytes(int E_loc, int H, int I, bool fc1, int nh) {
  const int K = fc1 ? H : I;
  const int n_ntiles = ((fc1 ? I : H) + nh - 1) / nh;
  return (size_t)E_loc * n_ntiles * (K / kBK) * 2 * kSfBlock;
}

size_t fcq_packed_scale_bytes(int E_loc, int H, int I, bool fc1) {
  return packed_scale_bytes(E_loc, H, I, fc1, fcq_n_rows(fc1));
}

cudaError_t launch_pack_scales_nh(const uint8_t* ws, int E_loc, int H, int I, bool fc1, int nh, uint8_t* out,
                                  cudaStream_t st) {
  const int Mtot = fc1 ? 2 * I : H, K = fc1 ? H : I;
  const int n_ntiles = ((fc1 ? I : H) + nh - 1) / nh;
  const long nblk = (long)E_loc * n_ntiles * (K / kBK);
  if (nblk <= 0) return cudaSuccess;
  const int vec = (reinterpret_cast<uintptr_t>(ws) & 3) == 0;   // rows are 4-byte multiples (K % 128 == 0)
  const long grid = nblk < 8L * sm_count() ? nblk : 8L * sm_count();
  pack_scales_kernel<<<(unsigned)grid, 256, 0, st>>>(ws, Mtot, K, I, fc1 ? 1 : 0, nh, n_ntiles, E_loc, vec, out);
  return cudaGetLastError();
}

cudaError_t launch_pack_scales(const uint8_t* ws, int E_loc, int H, int I, bool fc1, uint8_t* out,
                               cudaStream_t st) {
  return launch_pack_scales_nh(ws, E_loc, H, I, fc1, fcq_n_rows(fc1), out, st);
}

cudaError_t launch_gather8(const Gather8Params& p, long max_tiles, cudaStream_t st) {
  if (max_tiles <= 0) return cudaSuccess;
  if (!p.x_bf16) {
    // MXFP8: a warp per tile's scale blocks, then per token's row, at most
    // one wave of 16 CTAs per SM
    if (!p.slot_to_row) return cudaErrorInvalidValue;
    const long units = std::max<long>(p.T, max_tiles);
    const long grid = std::min<long>((units + kGather8TokWarps - 1) / kGather8TokWarps, 16L * sm_count());
    return launch_pdl(gather8_tok_kernel, dim3((unsigned)grid), dim3(32 * kGather8TokWarps), 0, st, p);
  }
  // bf16 rows: one full wave of 8 CTAs per SM (or fewer units)
  const long grid = std::min<long>(max_tiles * (kBM / kGatherRowsHL), 8L * sm_count());
  return launch_pdl(gather8_kernel, dim3((unsigned)grid), dim3(256), 0, st, p);
}

cudaError_t launch_fcq(const FcqParams& p, const uint8_t* xq, const uint8_t* xq_lo, long S, const uint8_t* w,
                       int E_loc, bool fc1, long max_tiles, cudaStream_t st) {
  const bool lo = xq_lo != nullptr;
  CUtensorMap ma, mal, mb;
  // activations: E4M3 [S, K], boxes of 128 bytes x 128 rows, 128-byte swizzle
  // (the lo rows of bf16 activations likewise)
  if (!make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)p.K, (uint64_t)S, (uint64_t)p.K, kBK, kBM,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mal, CU_TENSOR_MAP_DATA_TYPE_UINT8, lo ? xq_lo : xq, (uint64_t)p.K, (uint64_t)S, (uint64_t)p.K, kBK,
                kBM, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // weights: E2M1 [E_loc * Mtot, K] (K/2 bytes per row), boxes of 128 codes x
  // NH rows, each 16 codes landing in a 16-byte slot, 128-byte swizzle
  const uint32_t nh = (uint32_t)fcq_n_rows(fc1);
  if (!make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w, (uint64_t)p.K, (uint64_t)E_loc * p.Mtot,
                (uint64_t)(p.K / 2), kBK, nh, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (fc1)
    return lo ? launch_fcq_t<true, true>(p, ma, mal, mb, max_tiles, st)
              : launch_fcq_t<true, false>(p, ma, mal, mb, max_tiles, st);
  return lo ? launch_fcq_t<false, true>(p, ma, mal, mb, max_tiles, st)
            : launch_fcq_t<false, false>(p, ma, mal, mb, max_tiles, st);
}

}  // namespace situ
