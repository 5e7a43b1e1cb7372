// fc_bs.cu -- FC1 (gate/up + SiTU) and FC2 for MXFP8 activations x MXFP4
// weights (w4a8) on the block-scaled tensor cores:
// tcgen05.mma.kind::mxf8f6f4.block_scale, E4M3 x E2M1 with one UE8M0 scale
// per 32 elements of K on both operands, fp32 accumulation in TMEM.
//
// One CTA computes a [128 tokens x 256 weight rows] tile of one local
// expert, K in stages of 128:
//   * warp 0 (one lane) is the TMA producer: per stage the token tile's
//     E4M3 rows (128 x 128 B, 128-byte swizzle) and the weight rows' E2M1
//     codes (256 x 128 elements).  The weights are read with the tensor-map
//     type that expands each 8-byte group of 16 packed codes into a 16-byte
//     slot in shared memory, the operand layout the MMA takes for 4-bit
//     types next to 8-bit ones, so the packed weights go from HBM to the
//     tensor core untouched;
//   * warps 4..7 stage the block scales: per stage each row's four UE8M0
//     bytes (the four 32-element blocks of the stage) as one 32-bit word,
//     written to shared memory as 32 x 16-byte rows in which row i holds the
//     words of tile rows i, i+32, i+64, i+96 -- the source layout of
//     tcgen05.cp.32x128b.warpx4, which copies it into four TMEM columns of
//     every 32-lane quarter;
//   * warp 1 allocates 512 TMEM columns (256 for the accumulator, 12 per
//     stage for scales); one lane copies each stage's scales into TMEM and
//     issues four MMAs (M = 128, N = 256, K = 32), the k-th taking byte k of
//     the scale words, then commits the stage back to the producer;
//   * warps 4..7 then read the accumulator (each thread one token row):
//     FC1 applies the per-expert alphas and SiTU to each gate/up column pair
//     (the tile's columns are 128 gate rows then the 128 matching up rows)
//     and writes H1 as MXFP8 (E4M3 + one UE8M0 per 32 along I), which is
//     FC2's A operand as it stands; FC2 writes alpha2 * acc as fp32.
// K (H for FC1, I for FC2) must be a multiple of 128.  Every mbarrier wait
// is bounded; on expiry the CTA records an error code in the device status
// word and unwinds, and TMEM is always released.
#include "situ_internal.h"
#include "tc_common.cuh"

namespace situ {

using namespace tc;

namespace {

constexpr int kBM = 128;         // tokens per tile (MMA M, TMEM lanes)
constexpr int kBN = 256;         // weight rows per tile (MMA N)
constexpr int kBK = 128;         // K elements per stage
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr int kTmemCols = 512;
constexpr int kABytes = kBM * kBK;           // 16 KB of E4M3
constexpr int kBBytes = kBN * kBK;           // 32 KB: E2M1 in 16-byte slots of 16 codes
constexpr int kBTxBytes = kBN * kBK / 2;     // what the loads transfer: the packed 16 KB
constexpr int kSfaBytes = kBM * 4;           // four UE8M0 bytes per row
constexpr int kSfbBytes = kBN * 4;
constexpr int kSfStage = kSfaBytes + kSfbBytes;
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffSF = kOffB + kStages * kBBytes;
constexpr int kOffBar = kOffSF + kStages * kSfStage;
constexpr int kNumBars = 3 * kStages + 1;    // full, sf_full, empty per stage; acc_full
constexpr int kOffTm = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffTm + 16 + 1024;   // + alignment slack
// TMEM columns: accumulator [0, 256); stage s's A scales at 256 + 12 s
// (4 columns), its B scales at 256 + 12 s + 4 (4 columns per 128 rows)
constexpr int kSfCol0 = 256;
constexpr int kSfColsPerStage = 12;
static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");

// Instruction descriptor, block-scaled kinds: A = E4M3 (0), B = E2M1 (5),
// both K-major, N >> 3 at bit 17, UE8M0 scales (bit 23), M >> 4 at bit 24;
// the B and A scale byte selectors sit at bits 4..5 and 29..30.
constexpr uint32_t kIdesc = (0u << 7) | (5u << 10) | ((uint32_t)(kBN >> 3) << 17) | (1u << 23) |
                            ((uint32_t)(kBM >> 4) << 24);
__device__ __forceinline__ uint32_t idesc_sf(uint32_t k) { return kIdesc | (k << 4) | (k << 29); }

__device__ __forceinline__ void mma_bs(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Descriptor of a 32 x 16-byte scale block: no swizzle, 8-row groups of
// 128 contiguous bytes.
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

// one 32-bit word of four scale bytes; 4-byte aligned when vec
__device__ __forceinline__ uint32_t ld_sf4(const uint8_t* p, bool vec) {
  if (vec) return __ldg(reinterpret_cast<const uint32_t*>(p));
  return (uint32_t)__ldg(p) | ((uint32_t)__ldg(p + 1) << 8) | ((uint32_t)__ldg(p + 2) << 16) |
         ((uint32_t)__ldg(p + 3) << 24);
}

}  // namespace

template <bool FC1>
__global__ void __launch_bounds__(kThreads, 1)
fcq_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const FcqParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int ntile = blockIdx.x % p.n_ntiles;
  const int tile = blockIdx.x / p.n_ntiles;
  if (tile >= __ldg(p.tile_offsets + p.E_loc)) return;
  if (*reinterpret_cast<volatile int*>(p.err) != 0) return;   // an earlier CTA timed out
  const int2 ti = __ldg(p.tile_info + tile);
  const int e = ti.x, row0 = ti.y;
  const int nrows = min(kBM, __ldg(p.offsets + e + 1) - row0);
  const int nk = p.K / kBK;
  const int nsb = p.K / 32;                       // block scales per row
  const int nbase = FC1 ? ntile * (kBN / 2) : ntile * kBN;

  const uint32_t sbase = saddr(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto full = [&](int s) { return bar0 + 8 * s; };
  auto sf_full = [&](int s) { return bar0 + 8 * (kStages + s); };
  auto empty = [&](int s) { return bar0 + 8 * (2 * kStages + s); };
  const uint32_t acc_full = bar0 + 8 * (3 * kStages);
  uint32_t* tm_holder = reinterpret_cast<uint32_t*>(smem + kOffTm);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(sf_full(s), 128);
      mbar_init(empty(s), 1);
    }
    mbar_init(acc_full, 1);
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

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const int wrow = e * p.Mtot + nbase;
      const int wrow2 = FC1 ? wrow + p.I : wrow + kBN / 2;   // second 128 rows: up rows / next rows
      for (int kk = 0; kk < nk; ++kk) {
        const int s = kk % kStages, r = kk / kStages;
        if (r > 0 && !mbar_wait(empty(s), (r - 1) & 1, p.err, 21)) break;
        mbar_expect_tx(full(s), kABytes + kBTxBytes);
        tma_load_2d(sbase + kOffA + s * kABytes, &tmA, kk * kBK, row0, full(s));
        tma_load_2d(sbase + kOffB + s * kBBytes, &tmB, kk * kBK, wrow, full(s));
        tma_load_2d(sbase + kOffB + s * kBBytes + kBBytes / 2, &tmB, kk * kBK, wrow2, full(s));
      }
    }
  } else if (warp == 1) {
    // ---------------- scale copies + MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      for (int kk = 0; kk < nk && ok; ++kk) {
        const int s = kk % kStages, par = (kk / kStages) & 1;
        ok = mbar_wait(full(s), par, p.err, 22) && mbar_wait(sf_full(s), par, p.err, 23);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t sf_smem = sbase + kOffSF + s * kSfStage;
        const uint32_t sfa = tmem + kSfCol0 + s * kSfColsPerStage;
        const uint32_t sfb = sfa + 4;
        tmem_cp_sf(sfa, sf_desc(sf_smem));
        tmem_cp_sf(sfb, sf_desc(sf_smem + kSfaBytes));
        tmem_cp_sf(sfb + 4, sf_desc(sf_smem + kSfaBytes + 512));
        const uint64_t ad = sdesc(sbase + kOffA + s * kABytes);
        const uint64_t bd = sdesc(sbase + kOffB + s * kBBytes);
#pragma unroll
        for (int k4 = 0; k4 < kBK / 32; ++k4)   // +32 bytes along K per instruction
          mma_bs(tmem, ad + 2 * k4, bd + 2 * k4, idesc_sf((uint32_t)k4), sfa, sfb, (kk | k4) != 0);
        mma_commit(empty(s));
      }
      mma_commit(acc_full);
    }
  } else if (warp >= 4) {
    // ---------------- scale staging, then epilogue ----------------
    const int t = tid - 128;
    const bool a_ok = t < nrows;
    const uint8_t* a_src = p.xs + (size_t)(row0 + (a_ok ? t : 0)) * p.xs_stride;
    const uint8_t* b_src[2];
    bool b_ok[2];
    for (int h = 0; h < 2; ++h) {
      int brow;
      if (FC1) {
        b_ok[h] = nbase + t < p.I;
        brow = (h ? p.I : 0) + nbase + t;
      } else {
        brow = nbase + t + 128 * h;
        b_ok[h] = brow < p.Mtot;
      }
      b_src[h] = p.ws + ((size_t)e * p.Mtot + (b_ok[h] ? brow : 0)) * (size_t)nsb;
    }
    const bool vec = p.ws_vec != 0;
    auto load = [&](int kk, uint32_t* w) {
      const bool in = kk < nk;
      w[0] = (a_ok && in) ? __ldg(reinterpret_cast<const uint32_t*>(a_src + 4 * kk)) : 0u;
      w[1] = (b_ok[0] && in) ? ld_sf4(b_src[0] + 4 * kk, vec) : 0u;
      w[2] = (b_ok[1] && in) ? ld_sf4(b_src[1] + 4 * kk, vec) : 0u;
    };
    // the word of tile row 32 j + i goes to byte (16 i + 4 j) of its 512-byte block
    const int so = (t & 31) * 16 + (t >> 5) * 4;
    uint32_t w0[3], w1[3], w2[3];
    load(0, w0);
    load(1, w1);
    for (int kk = 0; kk < nk; ++kk) {
      load(kk + 2, w2);
      const int s = kk % kStages, r = kk / kStages;
      // the stage's scale block is free once the MMAs of its previous round are done
      if (r > 0 && !mbar_wait(empty(s), (r - 1) & 1, p.err, 24)) break;
      uint8_t* sf = smem + kOffSF + s * kSfStage;
      *reinterpret_cast<uint32_t*>(sf + so) = w0[0];
      *reinterpret_cast<uint32_t*>(sf + kSfaBytes + so) = w0[1];
      *reinterpret_cast<uint32_t*>(sf + kSfaBytes + 512 + so) = w0[2];
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(sf_full(s));
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        w0[i] = w1[i];
        w1[i] = w2[i];
      }
    }
    // ---- epilogue: thread = token row (TMEM lane) ----
    const int m = (warp - 4) * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)((warp - 4) * 32) << 16);
    // warp-uniform outcome: the tcgen05.ld below are .sync.aligned
    const bool acc_ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, p.err, 25));
    if (acc_ok) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const bool vrow = m < nrows;
      const size_t row = (size_t)(row0 + (vrow ? m : 0));
      if (FC1) {
        const float ag = p.alpha_g ? __ldg(p.alpha_g + e) : 1.f;
        const float au = p.alpha_u ? __ldg(p.alpha_u + e) : 1.f;
        const float bt = __ldg(p.beta + e), btl = __ldg(p.beta_lin + e);
        for (int c0 = 0; c0 < kBN / 2; c0 += 32) {
          float gt[32], up[32];
          tmem_ld16(trow + c0, gt);
          tmem_ld16(trow + c0 + 16, gt + 16);
          tmem_ld16(trow + 128 + c0, up);
          tmem_ld16(trow + 128 + c0 + 16, up + 16);
          const int i0 = nbase + c0;
          if (!vrow || i0 >= p.I) continue;
          float v[32];
          float amax = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] = situ_f(gt[j] * ag, up[j] * au, bt, btl);
            amax = fmaxf(amax, fabsf(v[j]));
          }
          // MXFP8 of the 32-element block: the smallest e with amax * 2^-e <= 448
          const int ex = mxfp8_exponent(amax);
          const float sc = exp2i(-ex);
          uint32_t q[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            q[j] = f32x2_to_e4m3x2(v[4 * j] * sc, v[4 * j + 1] * sc) |
                   (f32x2_to_e4m3x2(v[4 * j + 2] * sc, v[4 * j + 3] * sc) << 16);
          uint4* dst = reinterpret_cast<uint4*>(p.hq + row * p.hq_stride + i0);
          dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
          dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
          p.hs[row * (p.hq_stride / 32) + i0 / 32] = (uint8_t)(ex + 127);
        }
      } else {
        const float a2 = p.alpha2 ? __ldg(p.alpha2 + e) : 1.f;
        for (int c0 = 0; c0 < kBN; c0 += 16) {
          float acc[16];
          tmem_ld16(trow + c0, acc);
          const int n0 = nbase + c0;
          if (!vrow || n0 >= p.Mtot) continue;
          float4* dst = reinterpret_cast<float4*>(p.y_out + row * p.Mtot + n0);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_float4(acc[4 * q] * a2, acc[4 * q + 1] * a2, acc[4 * q + 2] * a2, acc[4 * q + 3] * a2);
        }
      }
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
// gather8: MXFP8 activation rows (E4M3 bytes and UE8M0 scale bytes) copied
// into expert order; one warp per row, 16-byte copies.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) gather8_kernel(const Gather8Params p) {
  const long r = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= __ldg(p.meta)) return;
  const long t = __ldg(p.permuted_src + r) / p.top_k;
  const int K = p.K, n16 = K / 16;
  const uint4* src = reinterpret_cast<const uint4*>(p.x_q + (size_t)t * K);
  uint4* dst = reinterpret_cast<uint4*>(p.x8 + (size_t)r * K);
  for (int i = lane; i < n16; i += 32) dst[i] = __ldg(src + i);
  const int nsb = K / 32;
  const uint8_t* ss = p.x_s + (size_t)t * nsb;
  uint8_t* sd = p.x8s + (size_t)r * nsb;
  if (p.s_vec) {
    for (int i = lane; i < nsb / 4; i += 32)
      reinterpret_cast<uint32_t*>(sd)[i] = __ldg(reinterpret_cast<const uint32_t*>(ss) + i);
  } else {
    for (int i = lane; i < nsb; i += 32) sd[i] = __ldg(ss + i);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

template <bool FC1>
cudaError_t launch_fcq_t(const FcqParams& p, const CUtensorMap& a, const CUtensorMap& b, long max_tiles,
                         cudaStream_t st) {
  static int set_for[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || set_for[dev] == 0) {
    cudaError_t err =
        cudaFuncSetAttribute(fcq_kernel<FC1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    if (dev < 64) set_for[dev] = 1;
  }
  const long grid = max_tiles * p.n_ntiles;
  if (grid <= 0) return cudaSuccess;
  fcq_kernel<FC1><<<(unsigned)grid, kThreads, kSmemBytes, st>>>(a, b, p);
  return cudaGetLastError();
}

}  // namespace

bool fcq_supported(int H, int I, const void* w1, const void* w2) {
  // the 4-bit tensor-map type wants rows of a multiple of 128 codes and a
  // 32-byte aligned base
  return H % kBK == 0 && I % kBK == 0 && (reinterpret_cast<uintptr_t>(w1) & 31) == 0 &&
         (reinterpret_cast<uintptr_t>(w2) & 31) == 0;
}

cudaError_t launch_gather8(const Gather8Params& p, cudaStream_t st) {
  if (p.S <= 0) return cudaSuccess;
  gather8_kernel<<<(unsigned)((p.S + 7) / 8), 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fcq(const FcqParams& p, const uint8_t* xq, long S, const uint8_t* w, int E_loc, bool fc1,
                       long max_tiles, cudaStream_t st) {
  CUtensorMap ma, mb;
  // activations: E4M3 [S, K], boxes of 128 bytes x 128 rows, 128-byte swizzle
  if (!make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)p.K, (uint64_t)S, (uint64_t)p.K, kBK, kBM,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // weights: E2M1 [E_loc * Mtot, K] (K/2 bytes per row), boxes of 128 codes x
  // 128 rows, each 16 codes landing in a 16-byte slot, 128-byte swizzle
  if (!make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w, (uint64_t)p.K, (uint64_t)E_loc * p.Mtot,
                (uint64_t)(p.K / 2), kBK, kBN / 2, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  return fc1 ? launch_fcq_t<true>(p, ma, mb, max_tiles, st) : launch_fcq_t<false>(p, ma, mb, max_tiles, st);
}

}  // namespace situ
