// tc_peak.cu -- dense throughput of the tensor-core MMA kinds the layer's
// GEMMs run on, measured on this GPU (a measurement aid: the roofline of a
// block-scaled GEMM is taken against the rate its own MMA kind reaches).
//
// One CTA per SM (the shared-memory request keeps a second CTA off the SM)
// fills a 128-row A tile, a 256-row B tile and their scale blocks in shared
// memory once, copies the scales into TMEM, and then issues `mmas` MMAs of
// M = 128, N = 256 back to back from one elected lane into one TMEM
// accumulator, exactly as a GEMM's K loop does, but with no memory traffic:
//   kind::mxf8f6f4.block_scale  A = E4M3, B = E2M1, UE8M0 per 32, K = 32
//                               (the w4a8 / w4a16 block-scaled GEMMs)
//   kind::mxf4nvf4.block_scale.scale_vec::4X  A = B = E2M1, E4M3 per 16,
//                               K = 64 (the NVFP4 FC1)
//   kind::f16                   A = B = bf16, K = 16 (the NVFP4 FC2)
// The operands are a fixed pseudo-random byte pattern (no E4M3 NaN codes),
// the scales 1.0.  The final commit is waited for with the bounded wait of
// the GEMM kernels; on expiry the CTA records kWaitCode in the status word.
#include "../../include/situ_moe.h"
#include "situ_internal.h"
#include "tc_common.cuh"

namespace situ {

using namespace tc;

namespace {

constexpr int kThreads = 128;
constexpr int kM = 128, kN = 256;
constexpr int kABytes = kM * 128;           // one 128-byte swizzle row per operand row
constexpr int kBBytes = kN * 128;
constexpr int kSfBlock = 512;
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kABytes;
constexpr int kOffSf = kOffB + kBBytes;     // A block, B rows 0..127, B rows 128..255
constexpr int kOffBar = kOffSf + 3 * kSfBlock;
constexpr int kOffTm = kOffBar + 8;
// more than half of an SM's shared memory, so that each SM holds one CTA
constexpr int kSmem = 120 * 1024;
constexpr int kTmemCols = 512;
constexpr int kSfaCol = 256, kSfbCol = 264;  // after the N = 256 accumulator, 4-column aligned
constexpr int kWaitCode = 98;
static_assert(kOffTm + 16 + 1024 <= kSmem, "shared memory layout");

__device__ __forceinline__ uint64_t sf_desc(uint32_t a) {
  uint64_t d = 0;
  d |= (uint64_t)((a >> 4) & 0x3FFFu);
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  return d;
}

template <int KIND>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                    uint32_t acc) {
  if (KIND == SITU_TC_MXF8F6F4) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
  } else if (KIND == SITU_TC_MXF4NVF4) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
  } else {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  }
}

// instruction descriptors, M = 128, N = 256, both operands K-major
template <int KIND>
__host__ __device__ constexpr uint32_t idesc_of() {
  return KIND == SITU_TC_MXF8F6F4
             // A = E4M3 (0), B = E2M1 (5), UE8M0 scales (bit 23)
             ? ((0u << 7) | (5u << 10) | ((uint32_t)(kN >> 3) << 17) | (1u << 23) | ((uint32_t)(kM >> 4) << 24))
         : KIND == SITU_TC_MXF4NVF4
             // A = B = E2M1 (1 in the fp4 kinds' encoding), UE4M3 scales
             ? ((1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24))
             // fp32 accumulator (bit 4), A = B = bf16
             : ((1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24));
}

// K elements per MMA of each kind (32 bytes of every operand row)
__host__ __device__ constexpr int k_per_mma(int kind) {
  return kind == SITU_TC_MXF8F6F4 ? 32 : kind == SITU_TC_MXF4NVF4 ? 64 : 16;
}

__device__ __forceinline__ uint32_t hash32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) tc_peak_kernel(long mmas, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t sbase = saddr(smem);
  const uint32_t bar = sbase + kOffBar;
  uint32_t* tm_holder = reinterpret_cast<uint32_t*>(smem + kOffTm);

  // operands: bytes with the E4M3 NaN pattern (S.1111.111) masked off; for
  // bf16 the exponent field stays below 0x7F (finite values of modest size)
  uint32_t* ops = reinterpret_cast<uint32_t*>(smem + kOffA);
  const uint32_t mask = KIND == SITU_TC_BF16 ? 0x3F7F3F7Fu : 0x77777777u;
  for (int i = tid; i < (kABytes + kBBytes) / 4; i += kThreads)
    ops[i] = hash32((uint32_t)i * 2654435761u + blockIdx.x) & mask;
  // scale blocks: 1.0 (UE8M0 127, E4M3 0x38)
  const uint32_t one = KIND == SITU_TC_MXF4NVF4 ? 0x38383838u : 0x7F7F7F7Fu;
  uint32_t* sf = reinterpret_cast<uint32_t*>(smem + kOffSf);
  for (int i = tid; i < 3 * kSfBlock / 4; i += kThreads) sf[i] = one;
  if (tid == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the MMAs and the scale copies read shared memory through the async proxy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
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
    const bool leader = elect_one();
    if (leader) {
      const uint32_t sfa = tmem + kSfaCol, sfb = tmem + kSfbCol;
      if (KIND != SITU_TC_BF16) {
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfa), "l"(sf_desc(sbase + kOffSf))
                     : "memory");
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfb),
                     "l"(sf_desc(sbase + kOffSf + kSfBlock))
                     : "memory");
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfb + 4),
                     "l"(sf_desc(sbase + kOffSf + 2 * kSfBlock))
                     : "memory");
      }
      const uint64_t ad = sdesc(sbase + kOffA), bd = sdesc(sbase + kOffB);
      constexpr uint32_t kId = idesc_of<KIND>();
      // four MMAs walk the 128-byte rows (32 bytes each), as one K stage of a GEMM
      for (long i = 0; i < mmas; i += 4) {
#pragma unroll
        for (uint32_t k4 = 0; k4 < 4; ++k4) {
          // block-scaled mxf8f6f4 picks scale byte k4 of each word; mxf4nvf4
          // (4X) reads a whole word per MMA; its columns stay 4-aligned
          const uint32_t id = KIND == SITU_TC_MXF8F6F4 ? (kId | (k4 << 4) | (k4 << 29)) : kId;
          mma<KIND>(tmem, ad + 2 * k4, bd + 2 * k4, id, sfa, sfb, (i | (long)k4) != 0);
        }
      }
      mma_commit(bar);
    }
    __syncwarp();
    mbar_wait_warp(bar, 0, err, kWaitCode);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int KIND>
cudaError_t launch_t(long mmas, int* err, int sms, cudaStream_t st) {
  static int set_for[64];
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (dev >= 64 || set_for[dev] == 0) {
      cudaError_t e = cudaFuncSetAttribute(tc_peak_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      if (e != cudaSuccess) return e;
      if (dev < 64) set_for[dev] = 1;
    }
  }
  tc_peak_kernel<KIND><<<sms, kThreads, kSmem, st>>>(mmas, err);
  return cudaGetLastError();
}

}  // namespace
}  // namespace situ

extern "C" situ_status situ_tc_peak(int32_t kind, int32_t mmas_per_sm, int32_t* device_status, double* flops,
                                    void* stream) {
  using namespace situ;
  if (!device_status || !flops) return SITU_ERR_NULL_ARG;
  if ((reinterpret_cast<uintptr_t>(device_status) & 3) != 0) return SITU_ERR_MISALIGNED;
  if (kind != SITU_TC_MXF8F6F4 && kind != SITU_TC_MXF4NVF4 && kind != SITU_TC_BF16) return SITU_ERR_UNSUPPORTED;
  if (mmas_per_sm < 4 || mmas_per_sm % 4 != 0) return SITU_ERR_BAD_SHAPE;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return SITU_ERR_CUDA;
  *flops = 2.0 * kM * kN * (double)k_per_mma(kind) * (double)mmas_per_sm * (double)sms;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = kind == SITU_TC_MXF8F6F4   ? launch_t<SITU_TC_MXF8F6F4>(mmas_per_sm, device_status, sms, st)
                  : kind == SITU_TC_MXF4NVF4 ? launch_t<SITU_TC_MXF4NVF4>(mmas_per_sm, device_status, sms, st)
                                             : launch_t<SITU_TC_BF16>(mmas_per_sm, device_status, sms, st);
  return e == cudaSuccess ? SITU_OK : SITU_ERR_CUDA;
}
