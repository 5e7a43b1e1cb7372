// quant_combine.cu -- the two HBM-bound elementwise steps of the layer.
//
// quant_mxfp8: bf16 activations -> MXFP8 (E4M3 + one UE8M0 scale per token
// per 32 hidden elements; TokenSpeed SiTU, "Supported contract").  Four
// lanes share one 32-element block: each lane loads 8 bf16 with one 128-bit
// load (a warp reads 512 contiguous bytes), the block amax is reduced with
// two shuffles, and each lane stores its 8 E4M3 codes with one 64-bit store.
//
// combine: the top-k-weighted un-permute sum out[t] = sum_j w[t,j] * Y[row]
// over the kept slots in ascending j, from the FC2 output (fp32 rows, or f16
// rows with a power-of-two scale per 32 columns), accumulated in fp32 and
// rounded to bf16 once (the golden loop of TensorRT-LLM PR #17865 adds
// weight * expert output per slot); a token with no kept slot gets 0.  Each
// thread owns one 16-byte piece of the rows and has all K slots' loads in
// flight at once, so each row of Y is read fully coalesced.
#include "../../include/situ_moe.h"
#include "situ_internal.h"

namespace situ {

__global__ void __launch_bounds__(256)
quant_mxfp8_kernel(const uint4* __restrict__ x, long n_lanes, uint2* __restrict__ q,
                   uint8_t* __restrict__ s) {
  long gid = (long)blockIdx.x * blockDim.x + threadIdx.x;
  bool valid = gid < n_lanes;
  uint4 v = valid ? __ldg(x + gid) : make_uint4(0, 0, 0, 0);
  float f[8];
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) { f[2 * i] = bf16_lo(w[i]); f[2 * i + 1] = bf16_hi(w[i]); }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  int e = mxfp8_exponent(amax);
  float sc = exp2i(-e);
  uint32_t c01 = f32x2_to_e4m3x2(f[0] * sc, f[1] * sc);
  uint32_t c23 = f32x2_to_e4m3x2(f[2] * sc, f[3] * sc);
  uint32_t c45 = f32x2_to_e4m3x2(f[4] * sc, f[5] * sc);
  uint32_t c67 = f32x2_to_e4m3x2(f[6] * sc, f[7] * sc);
  if (valid) {
    q[gid] = make_uint2(c01 | (c23 << 16), c45 | (c67 << 16));
    if ((gid & 3) == 0) s[gid >> 2] = (uint8_t)(e + 127);
  }
}

cudaError_t launch_quant_mxfp8(const void* x, int T, int H, uint8_t* q, uint8_t* s,
                               cudaStream_t st) {
  long n_lanes = (long)T * H / 8;
  long blocks = (n_lanes + 255) / 256;
  quant_mxfp8_kernel<<<(unsigned)blocks, 256, 0, st>>>((const uint4*)x, n_lanes, (uint2*)q, s);
  return cudaGetLastError();
}

// One thread owns 16 bytes of one token's Y rows (4 fp32 or 8 f16 columns)
// and issues the loads of all K slots before the first multiply-add, so a
// thread keeps K 16-byte loads in flight; the sums still run in ascending j.
// F16: Y rows are f16 mantissas with a scale byte per 32 columns
// (y16_exponent), block-major (byte of row r, block b at b * ys_rows + r).
// Threads per CTA: 64 for f16 rows, 128 for fp32 rows (the Kimi-K3 row of
// 3584 columns is then exactly 7 CTAs of 16-byte pieces either way).
template <bool F16>
__host__ __device__ constexpr int combine_threads() { return F16 ? 64 : 128; }

template <bool F16>
__global__ void __launch_bounds__(combine_threads<F16>())
combine_kernel(const uint4* __restrict__ y, const uint8_t* __restrict__ ys, long ys_rows,
               const int32_t* __restrict__ slot_to_row, const float* __restrict__ w, int K, int n16,
               uint4* __restrict__ out) {
  griddep_wait();   // Y is the predecessor's output
  const int t = blockIdx.x;
  const int c = blockIdx.y * combine_threads<F16>() + threadIdx.x;   // 16-byte column piece
  if (c >= n16) return;
  int r[SITU_MAX_TOP_K];
  float wt[SITU_MAX_TOP_K];
  uint4 v[SITU_MAX_TOP_K];
  uint32_t sb[SITU_MAX_TOP_K];
#pragma unroll
  for (int j = 0; j < SITU_MAX_TOP_K; ++j) {
    r[j] = j < K ? __ldg(slot_to_row + (size_t)t * K + j) : -1;
    wt[j] = r[j] >= 0 ? (w ? __ldg(w + (size_t)t * K + j) : 1.f) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < SITU_MAX_TOP_K; ++j) {
    v[j] = r[j] >= 0 ? __ldg(y + (size_t)r[j] * n16 + c) : make_uint4(0u, 0u, 0u, 0u);
    if (F16) sb[j] = r[j] >= 0 ? __ldg(ys + (size_t)(c >> 2) * ys_rows + r[j]) : 127u;
  }
  if (!F16) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < SITU_MAX_TOP_K; ++j) {
      if (r[j] >= 0) {
        acc.x = fmaf(wt[j], __uint_as_float(v[j].x), acc.x);
        acc.y = fmaf(wt[j], __uint_as_float(v[j].y), acc.y);
        acc.z = fmaf(wt[j], __uint_as_float(v[j].z), acc.z);
        acc.w = fmaf(wt[j], __uint_as_float(v[j].w), acc.w);
      }
    }
    // 4 bf16 of this thread's 4 columns: 8 bytes (two threads fill 16)
    reinterpret_cast<uint2*>(out)[(size_t)t * n16 + c] =
        make_uint2(f32x2_to_bf16x2(acc.x, acc.y), f32x2_to_bf16x2(acc.z, acc.w));
  } else {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < SITU_MAX_TOP_K; ++j) {
      if (r[j] >= 0) {
        const float s = wt[j] * exp2i((int)sb[j] - 127);
        const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] = fmaf(s, f16_to_f32(u[q] & 0xFFFFu), acc[2 * q]);
          acc[2 * q + 1] = fmaf(s, f16_to_f32(u[q] >> 16), acc[2 * q + 1]);
        }
      }
    }
    out[(size_t)t * n16 + c] = make_uint4(f32x2_to_bf16x2(acc[0], acc[1]), f32x2_to_bf16x2(acc[2], acc[3]),
                                          f32x2_to_bf16x2(acc[4], acc[5]), f32x2_to_bf16x2(acc[6], acc[7]));
  }
}

cudaError_t launch_combine16(const void* y16, const uint8_t* ys, long ys_rows, const int32_t* slot_to_row,
                             const float* w, int T, int K, int H, void* out, cudaStream_t st) {
  const int n16 = H / 8;   // 16-byte pieces of an f16 row (H is a multiple of 32)
  constexpr int nt = combine_threads<true>();
  dim3 grid(T, (n16 + nt - 1) / nt);
  return launch_pdl(combine_kernel<true>, grid, dim3(nt), 0, st, (const uint4*)y16, ys, ys_rows,
                    slot_to_row, w, K, n16, (uint4*)out);
}

cudaError_t launch_combine(const void* y, const int32_t* slot_to_row, const float* w, int T, int K,
                           int H, void* out, cudaStream_t st) {
  const int n16 = H / 4;   // 16-byte pieces of an fp32 row
  constexpr int nt = combine_threads<false>();
  dim3 grid(T, (n16 + nt - 1) / nt);
  return launch_pdl(combine_kernel<false>, grid, dim3(nt), 0, st, (const uint4*)y,
                    (const uint8_t*)nullptr, 0L, slot_to_row, w, K, n16, (uint4*)out);
}

// ---------------------------------------------------------------------------
// Per-token NVFP4 activation quantisation: row global scale gs = amax / 2688
// (6 * 448; 1 for an all-zero row), E4M3 scale per 16 elements
// s = E4M3(amax16 / (6 gs)), elements E2M1(x / (value(s) gs)), every step one
// fp32 operation rounded to nearest even.  One CTA per token row.
// ---------------------------------------------------------------------------

// eight fp32 values -> eight E2M1 codes in one word, element 2i in the low
// nibble of byte i (the first operand of each pair conversion is the high
// nibble); nearest even, saturating to +-6
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float* y) {
  uint32_t d;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(d)
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
  return d;
}

__global__ void __launch_bounds__(128) quant_nvfp4_kernel(const uint4* __restrict__ x, int H,
                                                          uint2* __restrict__ q, uint8_t* __restrict__ s,
                                                          float* __restrict__ gs) {
  __shared__ float red[4];
  const long t = blockIdx.x;
  const int tid = threadIdx.x;
  const uint4* xr = x + (size_t)t * (H / 8);
  float amax = 0.f;
  for (int i = tid; i < H / 8; i += 128) {
    const uint4 v = __ldg(xr + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  float g = __fdiv_rn(amax, 2688.f);
  if (!(g > 0.f)) g = 1.f;
  if (tid == 0) gs[t] = g;
  const float den6 = __fmul_rn(6.f, g);
  for (int b = tid; b < H / 16; b += 128) {
    float v[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 u = __ldg(xr + 2 * b + h);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * h + 2 * j] = bf16_lo(w[j]);
        v[8 * h + 2 * j + 1] = bf16_hi(w[j]);
      }
    }
    float ab = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[i]));
    const uint32_t s8 = f32x2_to_e4m3x2(__fdiv_rn(ab, den6), 0.f) & 0xFFu;
    const float denom = __fmul_rn(e4m3_code_to_f32(s8), g);
    uint2 out = make_uint2(0u, 0u);
    if (denom > 0.f) {
      float y[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = __fdiv_rn(v[i], denom);
      out = make_uint2(f32x8_to_e2m1x8(y), f32x8_to_e2m1x8(y + 8));
    }
    q[(size_t)t * (H / 16) + b] = out;
    s[(size_t)t * (H / 16) + b] = (uint8_t)s8;
  }
}

cudaError_t launch_quant_nvfp4(const void* x, int T, int H, uint8_t* q, uint8_t* s, float* gs, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  quant_nvfp4_kernel<<<(unsigned)T, 128, 0, st>>>((const uint4*)x, H, (uint2*)q, s, gs);
  return cudaGetLastError();
}

// The bf16 H1 rows in expert order requantised to NVFP4 per row, with the
// rule of quant_nvfp4_kernel (the NVFP4 chain's opt-in H1 requantisation).
// One warp per row: the row maximum, then lane c takes the 64-element chunks
// c, c + 32, ...: four E4M3 scales and 32 bytes of codes each.  The scales
// go out as rows [S, I/16] or as one 16-byte chunk per 64 elements (its four
// bytes first, the rest 0), the token-side layout of the NVFP4 tiles.
__global__ void __launch_bounds__(128) requant_h1_nvfp4_kernel(const uint4* __restrict__ h, int I, long S,
                                                               const int32_t* __restrict__ meta, uint4* __restrict__ q,
                                                               uint8_t* __restrict__ s, float* __restrict__ gs,
                                                               int chunked) {
  griddep_wait();   // H1 is the predecessor's output
  const long r = (long)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= S || r >= __ldg(meta)) return;
  const uint4* hr = h + (size_t)r * (I / 8);
  float amax = 0.f;
  for (int i = lane; i < I / 8; i += 32) {
    const uint4 v = hr[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  float g = __fdiv_rn(amax, 2688.f);
  if (!(g > 0.f)) g = 1.f;
  if (lane == 0) gs[r] = g;
  const float den6 = __fmul_rn(6.f, g);
  for (int c = lane; c < I / 64; c += 32) {
    uint32_t sw = 0;
#pragma unroll
    for (int b4 = 0; b4 < 4; ++b4) {   // the chunk's four 16-element blocks
      float v[16];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint4 u = hr[8 * c + 2 * b4 + hh];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * hh + 2 * j] = bf16_lo(w[j]);
          v[8 * hh + 2 * j + 1] = bf16_hi(w[j]);
        }
      }
      float ab = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[i]));
      const uint32_t s8 = f32x2_to_e4m3x2(__fdiv_rn(ab, den6), 0.f) & 0xFFu;
      const float denom = __fmul_rn(e4m3_code_to_f32(s8), g);
      uint2 out = make_uint2(0u, 0u);
      if (denom > 0.f) {
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = __fdiv_rn(v[i], denom);
        out = make_uint2(f32x8_to_e2m1x8(y), f32x8_to_e2m1x8(y + 8));
      }
      reinterpret_cast<uint2*>(q)[(size_t)r * (I / 16) + 4 * c + b4] = out;
      sw |= s8 << (8 * b4);
      if (!chunked) s[(size_t)r * (I / 16) + 4 * c + b4] = (uint8_t)s8;
    }
    if (chunked) reinterpret_cast<uint4*>(s)[(size_t)r * (I / 64) + c] = make_uint4(sw, 0u, 0u, 0u);
  }
}

cudaError_t launch_requant_h1_nvfp4(const uint16_t* h, int I, long S, const int32_t* meta, uint8_t* q, uint8_t* s,
                                    float* gs, int chunked, cudaStream_t st) {
  if (S <= 0) return cudaSuccess;
  if (I % 64 != 0) return cudaErrorInvalidValue;
  return launch_pdl(requant_h1_nvfp4_kernel, dim3((unsigned)((S + 3) / 4)), dim3(128), 0, st, (const uint4*)h, I, S,
                    meta, (uint4*)q, s, gs, chunked);
}

__global__ void __launch_bounds__(256) zero_f32_kernel(float4* __restrict__ a, long n4) {
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long)gridDim.x * blockDim.x)
    a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(256) acc_to_bf16_kernel(const float4* __restrict__ acc, long n4,
                                                          uint2* __restrict__ out) {
  griddep_wait();   // the accumulator is the predecessor's output
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long)gridDim.x * blockDim.x) {
    const float4 v = acc[i];
    out[i] = make_uint2(f32x2_to_bf16x2(v.x, v.y), f32x2_to_bf16x2(v.z, v.w));
  }
}

static unsigned grid_for(long n4) {
  const long b = (n4 + 255) / 256;
  return (unsigned)(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

cudaError_t launch_zero_f32(float* a, long n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  zero_f32_kernel<<<grid_for(n / 4), 256, 0, st>>>((float4*)a, n / 4);
  return cudaGetLastError();
}

cudaError_t launch_acc_to_bf16(const float* acc, long n, void* out, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(acc_to_bf16_kernel, dim3(grid_for(n / 4)), dim3(256), 0, st, (const float4*)acc, n / 4,
                    (uint2*)out);
}

}  // namespace situ
