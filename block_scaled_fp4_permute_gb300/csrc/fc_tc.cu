// fc_tc.cu -- FC1 (gate/up + SiTU) and FC2 on the 5th-generation tensor
// cores (tcgen05) for prefill-sized token tiles.
//
// One CTA computes a [128 tokens x 256 weight rows] tile of one local
// expert, K in stages of 64:
//   * warp 0 (one lane) is the TMA producer: per stage it loads the token
//     tile's f16 activation rows (128 x 64, 128-byte swizzle, the layout the
//     MMA descriptors expect) and the weight rows' packed E2M1 bytes
//     (256 x 32 B) into a 3-stage shared ring, completion tracked by
//     mbarrier transaction counts;
//   * warps 4..7 (128 threads, two weight rows each) dequantise the packed
//     weights to f16 in shared memory, in the 128-byte-swizzled K-major
//     layout: E2M1 -> f16 with the hardware conversion, times the block scale
//     relative to the row's largest block scale (2^(s_b - s_max), exact for
//     blocks within 2^23 of the row maximum; NVFP4's E4M3 block scales are
//     folded in directly, always exact); the row's 2^(s_max - 127) and any
//     NVFP4 global scale go to the epilogue;
//   * warp 1 allocates 256 TMEM columns and one lane issues
//     tcgen05.mma.kind::f16 (M = 128 tokens, N = 256, K = 16 per
//     instruction, fp32 accumulation in TMEM), committing each stage back to
//     the producer and the final accumulator to the epilogue;
//   * warps 4..7 then read the accumulator (each thread one token row) with
//     tcgen05.ld and apply the per-token and per-row scales and, for FC1,
//     SiTU on the gate/up column pair (the tile's 256 columns are 128 gate
//     rows and the 128 matching up rows), writing H1 as bf16 (or its MXFP8
//     round trip for w4a8); FC2 writes fp32.
// Activations are "f16 rows with one scale per row" (gather16 in row-scale
// mode).  Every mbarrier wait is bounded by a wall-clock limit; on expiry
// the CTA records an error code in the device status word and unwinds, and
// TMEM is always released.
#include "situ_internal.h"
#include "tc_common.cuh"

namespace situ {

using namespace tc;

namespace {

constexpr int kBM = 128;        // tokens per tile (MMA M, TMEM lanes)
constexpr int kBN = 256;        // weight rows per tile (MMA N)
constexpr int kBK = 64;         // K elements per stage
constexpr int kStages = 3;
constexpr int kThreads = 256;
constexpr int kTmemCols = 256;
constexpr int kABytes = kBM * kBK * 2;     // 16 KB
constexpr int kBBytes = kBN * kBK * 2;     // 32 KB
constexpr int kPBytes = kBN * kBK / 2;     // 8 KB packed E2M1
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffP = kOffB + kStages * kBBytes;
constexpr int kOffW = kOffP + kStages * kPBytes;          // float[kBN] epilogue row scales
constexpr int kOffBar = kOffW + kBN * 4;                   // mbarriers
constexpr int kNumBars = 4 * kStages + 1;
constexpr int kOffTm = kOffBar + kNumBars * 8;             // TMEM base address
constexpr int kSmemBytes = kOffTm + 16 + 1024;             // + alignment slack

// kind::f16 instruction descriptor: f16 x f16 -> f32, both K-major,
// N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t* d) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(w));
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)v));
  return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// 2^k as an f16 pair, k in [-24, 15] (0 below)
__device__ __forceinline__ uint32_t f16x2_pow2(int k) {
  uint32_t h;
  if (k >= -14) h = (uint32_t)(k + 15) << 10;
  else if (k >= -24) h = 1u << (k + 24);
  else h = 0u;
  return h | (h << 16);
}

}  // namespace

template <bool FC1, bool WNV>
__global__ void __launch_bounds__(kThreads, 1)
fcp_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const FcpParams p) {
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
  const int K = p.K;
  const int nk = (K + kBK - 1) / kBK;
  const int bsz = WNV ? 16 : 32;
  const int nsb = K / bsz;                        // block scales per weight row
  const int nbase = FC1 ? ntile * (kBN / 2) : ntile * kBN;

  const uint32_t sbase = saddr(smem);
  float* wsc = reinterpret_cast<float*>(smem + kOffW);
  const uint32_t bar0 = sbase + kOffBar;
  auto full_a = [&](int s) { return bar0 + 8 * s; };
  auto full_p = [&](int s) { return bar0 + 8 * (kStages + s); };
  auto full_b = [&](int s) { return bar0 + 8 * (2 * kStages + s); };
  auto empty = [&](int s) { return bar0 + 8 * (3 * kStages + s); };
  const uint32_t acc_full = bar0 + 8 * (4 * kStages);
  uint32_t* tm_holder = reinterpret_cast<uint32_t*>(smem + kOffTm);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_a(s), 1);
      mbar_init(full_p(s), 1);
      mbar_init(full_b(s), 128);
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
    // the whole warp walks the loop; one elected lane issues the copies
    const bool leader = elect_one();
    const int yw = e * p.Mtot + nbase;
    for (int kk = 0; kk < nk; ++kk) {
      const int s = kk % kStages, r = kk / kStages;
      if (r > 0 && !mbar_wait_warp(empty(s), (r - 1) & 1, p.err, 11)) break;
      if (leader) {
        mbar_expect_tx(full_a(s), kABytes);
        tma_load_2d(sbase + kOffA + s * kABytes, &tmA, kk * kBK, row0, full_a(s));
        mbar_expect_tx(full_p(s), kPBytes);
        if (FC1) {
          tma_load_2d(sbase + kOffP + s * kPBytes, &tmB, kk * (kBK / 2), yw, full_p(s));
          tma_load_2d(sbase + kOffP + s * kPBytes + kPBytes / 2, &tmB, kk * (kBK / 2), yw + p.I, full_p(s));
        } else {
          tma_load_2d(sbase + kOffP + s * kPBytes, &tmB, kk * (kBK / 2), yw, full_p(s));
        }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // the whole warp walks the loop; one elected lane issues
    const bool leader = elect_one();
    bool ok = true;
    for (int kk = 0; kk < nk && ok; ++kk) {
      const int s = kk % kStages, par = (kk / kStages) & 1;
      ok = mbar_wait_warp(full_a(s), par, p.err, 12) && mbar_wait_warp(full_b(s), par, p.err, 13);
      if (!ok) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (leader) {
        const uint64_t ad = sdesc(sbase + kOffA + s * kABytes);
        const uint64_t bd = sdesc(sbase + kOffB + s * kBBytes);
#pragma unroll
        for (int k4 = 0; k4 < kBK / 16; ++k4)   // +32 bytes along K per instruction
          mma_f16_ss(tmem, ad + 2 * k4, bd + 2 * k4, (kk | k4) != 0);
        mma_commit(empty(s));
      }
      __syncwarp();
    }
    if (leader) mma_commit(acc_full);
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- converters, then epilogue ----------------
    const int t = tid - 128;
    int grow[2];
    bool gv[2];
    for (int h = 0; h < 2; ++h) {
      const int n = t + 128 * h;
      if (FC1) {
        const int i = nbase + t;
        gv[h] = i < p.I;
        grow[h] = h ? p.I + i : i;
      } else {
        grow[h] = nbase + n;
        gv[h] = grow[h] < p.Mtot;
      }
    }
    const uint8_t* srow[2];
    int smax[2];
    for (int h = 0; h < 2; ++h) {
      srow[h] = p.ws + ((size_t)e * p.Mtot + (gv[h] ? grow[h] : 0)) * (size_t)nsb;
      int m = 0;
      if (!WNV && gv[h]) {
        if ((nsb & 15) == 0 && (reinterpret_cast<uintptr_t>(srow[h]) & 15) == 0) {
          // the row's largest block scale, 16 bytes per load
          uint32_t acc = 0u;
          for (int b = 0; b < nsb; b += 16) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(srow[h] + b));
            acc = __vmaxu4(acc, __vmaxu4(__vmaxu4(v.x, v.y), __vmaxu4(v.z, v.w)));
          }
          m = max(max((int)(acc & 0xFFu), (int)((acc >> 8) & 0xFFu)),
                  max((int)((acc >> 16) & 0xFFu), (int)(acc >> 24)));
        } else {
          for (int b = 0; b < nsb; ++b) m = max(m, (int)__ldg(srow[h] + b));
        }
      }
      smax[h] = m;
      float ws = 0.f;
      if (gv[h]) {
        if (WNV) ws = FC1 ? __ldg(p.w1_gs + 2 * e + h) : __ldg(p.w2_gs + e);
        else ws = exp2i(m - 127);
      }
      wsc[t + 128 * h] = ws;
    }
    // the stage's block-scale bytes of both rows, packed per row (4 x E4M3
    // or 2 x UE8M0), prefetched two stages ahead so their load latency
    // hides behind the conversion
    constexpr int kSB = WNV ? 4 : 2;
    auto load_sc = [&](int kk, int h) -> uint32_t {
      uint32_t v = 0u;
#pragma unroll
      for (int j = 0; j < kSB; ++j) {
        const int b = kk * kSB + j;
        if (gv[h] && kk < nk && b < nsb) v |= (uint32_t)__ldg(srow[h] + b) << (8 * j);
      }
      return v;
    };
    uint32_t sc0[2] = {load_sc(0, 0), load_sc(0, 1)};
    uint32_t sc1[2] = {load_sc(1, 0), load_sc(1, 1)};
    for (int kk = 0; kk < nk; ++kk) {
      const uint32_t sc2[2] = {load_sc(kk + 2, 0), load_sc(kk + 2, 1)};
      const int s = kk % kStages, par = (kk / kStages) & 1;
      if (!mbar_wait(full_p(s), par, p.err, 14)) break;
      const uint8_t* pk = smem + kOffP + s * kPBytes;
      uint8_t* bt = smem + kOffB + s * kBBytes;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int n = t + 128 * h;
        const uint4 q0 = *reinterpret_cast<const uint4*>(pk + n * 32);
        const uint4 q1 = *reinterpret_cast<const uint4*>(pk + n * 32 + 16);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        // dequant factors: word j covers elements 8j..8j+7 of the stage
        uint32_t f[8];
        if (WNV) {
#pragma unroll
          for (int j2 = 0; j2 < 4; ++j2) {   // 16-element blocks of the stage
            const uint32_t sb = (sc0[h] >> (8 * j2)) & 0xFFu;
            f[2 * j2] = f[2 * j2 + 1] = e4m3x2_to_f16x2(sb | (sb << 8));
          }
        } else {
#pragma unroll
          for (int j2 = 0; j2 < 2; ++j2) {   // 32-element blocks
            const int b = kk * 2 + j2;
            const uint32_t fb =
                (gv[h] && b < nsb) ? f16x2_pow2((int)((sc0[h] >> (8 * j2)) & 0xFFu) - smax[h]) : 0u;
            f[4 * j2] = f[4 * j2 + 1] = f[4 * j2 + 2] = f[4 * j2 + 3] = fb;
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {   // 16-byte chunk j = elements 8j..8j+7
          uint32_t d[4];
          e2m1x8_to_f16x8(w[j], d);
#pragma unroll
          for (int i = 0; i < 4; ++i) d[i] = hmul2(d[i], f[j]);
          *reinterpret_cast<uint4*>(bt + n * 128 + ((j ^ (n & 7)) << 4)) = make_uint4(d[0], d[1], d[2], d[3]);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(full_b(s));
      sc0[0] = sc1[0];
      sc0[1] = sc1[1];
      sc1[0] = sc2[0];
      sc1[1] = sc2[1];
    }
    // ---- epilogue: thread = token row (TMEM lane) ----
    const int m = (warp - 4) * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)((warp - 4) * 32) << 16);
    asm volatile("bar.sync 1, 128;" ::: "memory");   // converters' wsc writes visible
    // warp-uniform outcome: the tcgen05.ld below are .sync.aligned
    const bool acc_ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, p.err, 15));
    if (acc_ok) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const bool vrow = m < nrows;
      const size_t row = (size_t)(row0 + (vrow ? m : 0));
      const float xs = vrow ? __ldg(p.xs + row * p.xs_stride) : 0.f;
      if (FC1) {
        const float ag = p.alpha_g ? __ldg(p.alpha_g + e) : 1.f;
        const float au = p.alpha_u ? __ldg(p.alpha_u + e) : 1.f;
        const float bt = __ldg(p.beta + e), btl = __ldg(p.beta_lin + e);
        const float rw = (p.topk_fc1 && vrow) ? __ldg(p.topk_weights + __ldg(p.permuted_src + row)) : 1.f;
        for (int c0 = 0; c0 < kBN / 2; c0 += 32) {
          float gt[32], up[32];
          tmem_ld16(trow + c0, gt);
          tmem_ld16(trow + c0 + 16, gt + 16);
          tmem_ld16(trow + 128 + c0, up);
          tmem_ld16(trow + 128 + c0 + 16, up + 16);
          const int i0 = nbase + c0;
          if (!vrow || i0 >= p.I) continue;
          float v[32];
          with_act(p.act_kind, bt, btl, [&](auto act) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              v[j] = act(gt[j] * (xs * wsc[c0 + j] * ag), up[j] * (xs * wsc[128 + c0 + j] * au)) * rw;
          });
          if (p.h_mxfp8) {   // the MXFP8 round trip FC2 consumes (w4a8)
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
            const int ex = mxfp8_exponent(amax);
            const float sc = exp2i(-ex), back = exp2i(ex);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const uint32_t cc = f32x2_to_e4m3x2(v[j] * sc, v[j + 1] * sc);
              v[j] = e4m3_to_f32(cc & 0xFFu) * back;
              v[j + 1] = e4m3_to_f32(cc >> 8) * back;
            }
          }
          uint4* dst = reinterpret_cast<uint4*>(p.h_out + row * p.I + i0);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(f32x2_to_bf16x2(v[8 * q], v[8 * q + 1]), f32x2_to_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                f32x2_to_bf16x2(v[8 * q + 4], v[8 * q + 5]), f32x2_to_bf16x2(v[8 * q + 6], v[8 * q + 7]));
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
            dst[q] = make_float4(acc[4 * q] * (xs * wsc[c0 + 4 * q] * a2), acc[4 * q + 1] * (xs * wsc[c0 + 4 * q + 1] * a2),
                                 acc[4 * q + 2] * (xs * wsc[c0 + 4 * q + 2] * a2),
                                 acc[4 * q + 3] * (xs * wsc[c0 + 4 * q + 3] * a2));
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
// host side
// ---------------------------------------------------------------------------

namespace {

template <bool FC1, bool WNV>
cudaError_t launch_fcp_t(const FcpParams& p, const CUtensorMap& a, const CUtensorMap& b, long max_tiles,
                         cudaStream_t st) {
  static int set_for[64];
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (dev >= 64 || set_for[dev] == 0) {
      cudaError_t err = cudaFuncSetAttribute(fcp_kernel<FC1, WNV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
      if (err != cudaSuccess) return err;
      if (dev < 64) set_for[dev] = 1;
    }
  }
  const long grid = max_tiles * p.n_ntiles;
  if (grid <= 0) return cudaSuccess;
  fcp_kernel<FC1, WNV><<<(unsigned)grid, kThreads, kSmemBytes, st>>>(a, b, p);
  return cudaGetLastError();
}

}  // namespace

int fcp_token_tile() { return kBM; }

cudaError_t launch_fcp(const FcpParams& p, const uint16_t* x16, long S, int kpad, const uint8_t* w, int E_loc,
                       bool fc1, bool nvfp4, long max_tiles, cudaStream_t st) {
  CUtensorMap ma, mb;
  // activations: f16 [S, kpad], boxes of 64 columns (128 B) x 128 rows, 128-byte swizzle
  if (!make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16, (uint64_t)kpad, (uint64_t)S, (uint64_t)kpad * 2, kBK, kBM,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // packed weights: u8 [E_loc * Mtot, K/2], boxes of 32 bytes x (128 | 256) rows
  if (!make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, (uint64_t)(p.K / 2), (uint64_t)E_loc * p.Mtot,
                (uint64_t)(p.K / 2), kBK / 2, fc1 ? kBN / 2 : kBN, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (fc1) return nvfp4 ? launch_fcp_t<true, true>(p, ma, mb, max_tiles, st) : launch_fcp_t<true, false>(p, ma, mb, max_tiles, st);
  return nvfp4 ? launch_fcp_t<false, true>(p, ma, mb, max_tiles, st) : launch_fcp_t<false, false>(p, ma, mb, max_tiles, st);
}

}  // namespace situ
