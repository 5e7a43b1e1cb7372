// gemm.cu -- grouped FC1 (gate/up + SiTU) and FC2 GEMMs over local experts.
//
// FC1: for each local expert e and its rows r (pairs routed to e),
//   gate_i = alpha_g * <x_r, W1[e, i]>,  up_i = alpha_u * <x_r, W1[e, I+i]>,
//   h_ri   = SiTU(gate_i, up_i; beta_e, beta_lin_e)
// with beta / linear beta from gemm1_alpha / gemm1_beta and the up half's
// net scale g1_alphas_up (FlashInfer 0.6.18 SM100a+SM103a MoE-LoRA AOT
// release notes, "Changes since 875b7d7"; SiTU formula: golden `_situ_act`,
// TensorRT-LLM PR #17865).  FC2: y_r = alpha2 * H1_r W2[e]^T.
//
// Tiling ("swap AB"): the weight rows are the MMA M side and the expert's
// tokens the N side, so a decode expert with one or two tokens still fills
// the 16-row MMA.  A CTA owns one (token tile, 128 weight rows) unit; FC1's
// 128 rows are 64 gate rows and the 64 matching up rows, arranged so that a
// thread's accumulator holds gate and up of the same (i, token) and SiTU
// runs in registers.  Units come from the token-tile prefix sum the permute
// writes on the device (no host synchronisation); CTAs past the last unit
// exit at once.  K runs in chunks of 128 with no power-of-two assumption on
// the hidden size (Kimi-K3's 3584 = 28 * 128), so the "hidden % 1024 != 0"
// hang of the FlashInfer release notes cannot arise.
//
// Operands: each thread loads 16 bytes (32 E2M1 codes = one MXFP4 scale
// block, or two NVFP4 blocks) of each of its two weight rows straight from
// HBM with 128-bit non-allocating loads, one chunk ahead of use, and turns
// them into exact bf16 in registers (PRMT table lookup, then a bf16x2
// multiply by the power-of-two or E4M3 block scale).  The K order inside a
// thread's 32-element block is permuted consistently in the weight and
// activation fragments, which is what lets one 128-bit load feed eight
// m16n8k16 steps; the contraction is unchanged.  Activations are the
// expert-ordered bf16 rows, staged per chunk with cp.async into a swizzled
// shared tile (conflict-free 128-bit fragment loads), double buffered.
#include "situ_internal.h"

namespace situ {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

__device__ __forceinline__ void sts128_zero(uint32_t dst) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0));
}
__device__ __forceinline__ void lds128(uint32_t* d, uint32_t addr) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
               : "r"(addr));
}
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Physical 16-byte slot of logical slot s16 (0..15) of token row `tok` in a
// 256-byte activation row: the 8 lanes of a quarter warp (2 tokens x 4
// k-blocks) land on 8 distinct bank groups.
__device__ __forceinline__ int swz(int s16, int tok) {
  return s16 ^ (((s16 >> 3) & 1) << 1) ^ (tok & 1);
}

// E4M3 scale byte as a bf16 pair (exact).
__device__ __forceinline__ uint32_t e4m3_to_bf16x2(uint32_t b) {
  uint32_t h = __float_as_uint(e4m3_to_f32(b)) >> 16;
  return h | (h << 16);
}

// 32 E2M1 codes + block scale(s) -> 16 bf16 pairs (pair p = elements 2p, 2p+1).
template <bool NV>
__device__ __forceinline__ void dequant32(uint4 w, uint32_t sc, uint32_t* out) {
  e2m1x8_to_bf16x8(w.x, out + 0);
  e2m1x8_to_bf16x8(w.y, out + 4);
  e2m1x8_to_bf16x8(w.z, out + 8);
  e2m1x8_to_bf16x8(w.w, out + 12);
  if (NV) {
    uint32_t s0 = e4m3_to_bf16x2(sc & 0xFFu), s1 = e4m3_to_bf16x2((sc >> 8) & 0xFFu);
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = bf16x2_mul(out[i], s0);
#pragma unroll
    for (int i = 8; i < 16; ++i) out[i] = bf16x2_mul(out[i], s1);
  } else {
    uint32_t s = ue8m0_to_bf16x2(sc);
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = bf16x2_mul(out[i], s);
  }
}

constexpr int kFcThreads = 256;
constexpr int kKC = 128;   // K chunk (elements)

template <int NS, bool FC1, bool NV>
__global__ void __launch_bounds__(kFcThreads, 2) fc_kernel(const FcParams p) {
  constexpr int NT = 8 * NS;
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int mt = blockIdx.x % p.n_mtiles;
  const int tile = blockIdx.x / p.n_mtiles;
  const int total = __ldg(p.tile_offsets + p.E_loc);
  if (tile >= total) return;
  const int2 ti = __ldg(p.tile_info + tile);   // (local expert, first row)
  const int e = ti.x;
  const int row0 = ti.y;
  const int nrows = min(NT, __ldg(p.offsets + e + 1) - row0);

  // the two weight rows this thread feeds (MMA rows g and g+8)
  int ra, rb;
  bool va, vb;
  if (FC1) {
    int i = mt * 64 + warp * 8 + g;
    va = vb = i < p.I;
    ra = i;
    rb = p.I + i;
  } else {
    ra = mt * 128 + warp * 16 + g;
    rb = ra + 8;
    va = ra < p.Mtot;
    vb = rb < p.Mtot;
  }
  const int bs = NV ? 16 : 32;
  const size_t wrow = (size_t)p.K / 2, srow = (size_t)p.K / bs;
  const uint8_t* wa = p.w + ((size_t)e * p.Mtot + (va ? ra : 0)) * wrow;
  const uint8_t* wb = p.w + ((size_t)e * p.Mtot + (vb ? rb : 0)) * wrow;
  const uint8_t* sa = p.ws + ((size_t)e * p.Mtot + (va ? ra : 0)) * srow;
  const uint8_t* sb = p.ws + ((size_t)e * p.Mtot + (vb ? rb : 0)) * srow;
  const int nchunks = (p.K + kKC - 1) / kKC;
  const uint32_t sx = smem_u32(smem);

  auto stage = [&](int kc, int buf) {
    for (int idx = tid; idx < NT * 16; idx += kFcThreads) {
      int tok = idx >> 4, s16 = idx & 15;
      int k = kc * kKC + s16 * 8;
      uint32_t dst = sx + (uint32_t)(((buf * NT + tok) * 16 + swz(s16, tok)) * 16);
      if (tok < nrows && k < p.K) cp_async16(dst, p.x + (size_t)(row0 + tok) * p.K + k);
      else sts128_zero(dst);
    }
    cp_async_commit();
  };
  auto fetch = [&](int kc, uint4& a, uint4& b, uint32_t& sca, uint32_t& scb) {
    int kb = kc * 4 + c;
    bool kv = kb * 32 < p.K;
    a = (va && kv) ? ldg_stream(wa + kb * 16) : make_uint4(0, 0, 0, 0);
    b = (vb && kv) ? ldg_stream(wb + kb * 16) : make_uint4(0, 0, 0, 0);
    if (NV) {
      sca = (va && kv) ? __ldg((const uint16_t*)(sa + kb * 2)) : 0u;
      scb = (vb && kv) ? __ldg((const uint16_t*)(sb + kb * 2)) : 0u;
    } else {
      sca = (va && kv) ? __ldg(sa + kb) : 0u;
      scb = (vb && kv) ? __ldg(sb + kb) : 0u;
    }
  };

  float acc[NS][4];
#pragma unroll
  for (int j = 0; j < NS; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  uint4 ca, cb;
  uint32_t csa, csb;
  stage(0, 0);
  fetch(0, ca, cb, csa, csb);
  for (int kc = 0; kc < nchunks; ++kc) {
    uint4 na = make_uint4(0, 0, 0, 0), nb = na;
    uint32_t nsa = 0, nsb = 0;
    const bool more = kc + 1 < nchunks;
    if (more) {
      stage(kc + 1, (kc + 1) & 1);
      fetch(kc + 1, na, nb, nsa, nsb);
    }
    uint32_t A0[16], A1[16];
    dequant32<NV>(ca, csa, A0);
    dequant32<NV>(cb, csb, A1);
    if (more) cp_async_wait<1>(); else cp_async_wait<0>();
    __syncthreads();
    const int buf = kc & 1;
#pragma unroll
    for (int j = 0; j < NS; ++j) {
      const int tok = 8 * j + g;
      uint32_t B[16];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        lds128(B + 4 * q, sx + (uint32_t)(((buf * NT + tok) * 16 + swz(4 * c + q, tok)) * 16));
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        uint32_t a[4] = {A0[2 * s], A1[2 * s], A0[2 * s + 1], A1[2 * s + 1]};
        uint32_t b[2] = {B[2 * s], B[2 * s + 1]};
        mma_bf16_16816(acc[j], a, b);
      }
    }
    __syncthreads();
    ca = na; cb = nb; csa = nsa; csb = nsb;
  }

  if (FC1) {
    // SiTU in registers, staged through shared memory for coalesced stores
    float* sH = reinterpret_cast<float*>(smem);   // [NT][64]
    const int il = warp * 8 + g;
    if (va) {
      const float ag = p.alpha_g ? __ldg(p.alpha_g + e) : 1.f;
      const float au = p.alpha_u ? __ldg(p.alpha_u + e) : 1.f;
      const float bt = __ldg(p.beta + e), btl = __ldg(p.beta_lin + e);
      const float gg = NV ? __ldg(p.w1_gs + 2 * e) : 1.f, gu = NV ? __ldg(p.w1_gs + 2 * e + 1) : 1.f;
#pragma unroll
      for (int j = 0; j < NS; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int tok = 8 * j + 2 * c + h;
          if (tok < nrows) {
            const float xs = p.xg ? __ldg(p.xg + row0 + tok) : 1.f;
            const float gate = acc[j][h] * (ag * gg * xs);
            const float up = acc[j][2 + h] * (au * gu * xs);
            sH[tok * 64 + il] = situ_f(gate, up, bt, btl);
          }
        }
      }
    }
    __syncthreads();
    for (int idx = tid; idx < NT * 2; idx += kFcThreads) {
      const int tok = idx >> 1, blk = idx & 1;
      const int i0 = mt * 64 + blk * 32;
      if (tok >= nrows || i0 >= p.I) continue;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = sH[tok * 64 + blk * 32 + i];
      if (p.mxfp8_h) {
        // FC1 output as MXFP8 per 32 along I, dequantised for FC2 (exact)
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        const int ex = mxfp8_exponent(amax);
        const float sc = exp2i(-ex), back = exp2i(ex);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          uint32_t cc = f32x2_to_e4m3x2(v[i] * sc, v[i + 1] * sc);
          v[i] = e4m3_to_f32(cc & 0xFFu) * back;
          v[i + 1] = e4m3_to_f32(cc >> 8) * back;
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(p.h_out + (size_t)(row0 + tok) * p.I + i0);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        dst[q] = make_uint4(f32x2_to_bf16x2(v[8 * q + 0], v[8 * q + 1]), f32x2_to_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                            f32x2_to_bf16x2(v[8 * q + 4], v[8 * q + 5]), f32x2_to_bf16x2(v[8 * q + 6], v[8 * q + 7]));
    }
  } else {
    float* sY = reinterpret_cast<float*>(smem);   // [NT][128] fp32
    const float scale = (p.alpha2 ? __ldg(p.alpha2 + e) : 1.f) * (NV ? __ldg(p.w2_gs + e) : 1.f);
    const int nl = warp * 16 + g;
#pragma unroll
    for (int j = 0; j < NS; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int tok = 8 * j + 2 * c + h;
        sY[tok * 128 + nl] = acc[j][h] * scale;
        sY[tok * 128 + nl + 8] = acc[j][2 + h] * scale;
      }
    }
    __syncthreads();
    for (int idx = tid; idx < NT * 32; idx += kFcThreads) {
      const int tok = idx >> 5, ch = idx & 31;
      const int n0 = mt * 128 + ch * 4;
      if (tok >= nrows || n0 >= p.Mtot) continue;
      const float4 v = *reinterpret_cast<const float4*>(sY + tok * 128 + ch * 4);
      *reinterpret_cast<float4*>(p.y_out + (size_t)(row0 + tok) * p.Mtot + n0) = v;
    }
  }
}

template <int NS, bool FC1, bool NV>
static cudaError_t launch_fc_t(const FcParams& p, long max_tiles, cudaStream_t st) {
  const size_t smem = (size_t)2 * 8 * NS * 256;   // two [NT][128] bf16 buffers
  const long grid = max_tiles * p.n_mtiles;
  if (grid <= 0) return cudaSuccess;
  fc_kernel<NS, FC1, NV><<<(unsigned)grid, kFcThreads, smem, st>>>(p);
  return cudaGetLastError();
}

template <bool FC1, bool NV>
static cudaError_t launch_fc_ns(const FcParams& p, int ns, long max_tiles, cudaStream_t st) {
  switch (ns) {
    case 1: return launch_fc_t<1, FC1, NV>(p, max_tiles, st);
    case 2: return launch_fc_t<2, FC1, NV>(p, max_tiles, st);
    case 4: return launch_fc_t<4, FC1, NV>(p, max_tiles, st);
    default: return launch_fc_t<8, FC1, NV>(p, max_tiles, st);
  }
}

cudaError_t launch_fc(const FcParams& p, bool fc1, bool nvfp4, int ns, long max_tiles,
                      cudaStream_t st) {
  if (fc1) return nvfp4 ? launch_fc_ns<true, true>(p, ns, max_tiles, st)
                        : launch_fc_ns<true, false>(p, ns, max_tiles, st);
  return nvfp4 ? launch_fc_ns<false, true>(p, ns, max_tiles, st)
               : launch_fc_ns<false, false>(p, ns, max_tiles, st);
}

// ---------------------------------------------------------------------------
// gather: expert-ordered bf16 activation rows
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) gather_kernel(const GatherParams p) {
  const long r = blockIdx.x;
  const int h8 = blockIdx.y * blockDim.x + threadIdx.x;
  const int R = __ldg(p.meta);
  if (r >= R || h8 >= p.H / 8) return;
  const int t = __ldg(p.permuted_src + r) / p.top_k;
  uint4 out;
  if (p.act == 0) {
    out = __ldg(reinterpret_cast<const uint4*>(p.x_bf16) + (size_t)t * (p.H / 8) + h8);
  } else if (p.act == 1) {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(p.x_q + (size_t)t * p.H) + h8);
    const float sc = exp2i((int)__ldg(p.x_s + (size_t)t * (p.H / 32) + h8 / 4) - 127);
    uint32_t w[2] = {q.x, q.y}, o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t wd = w[i >> 1] >> (16 * (i & 1));
      o[i] = f32x2_to_bf16x2(e4m3_to_f32(wd & 0xFFu) * sc, e4m3_to_f32((wd >> 8) & 0xFFu) * sc);
    }
    out = make_uint4(o[0], o[1], o[2], o[3]);
  } else {
    const uint32_t q = __ldg(reinterpret_cast<const uint32_t*>(p.x_q + (size_t)t * (p.H / 2)) + h8);
    const float sc = e4m3_to_f32(__ldg(p.x_s + (size_t)t * (p.H / 16) + h8 / 2));
    uint32_t d[4];
    e2m1x8_to_bf16x8(q, d);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = f32x2_to_bf16x2(bf16_lo(d[i]) * sc, bf16_hi(d[i]) * sc);
    out = make_uint4(d[0], d[1], d[2], d[3]);
  }
  reinterpret_cast<uint4*>(p.x_perm + (size_t)r * p.H)[h8] = out;
  if (p.xg_perm && h8 == 0) p.xg_perm[r] = __ldg(p.x_gs + t);
}

cudaError_t launch_gather(const GatherParams& p, cudaStream_t st) {
  if (p.S <= 0) return cudaSuccess;
  dim3 grid((unsigned)p.S, (p.H / 8 + 255) / 256);
  gather_kernel<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace situ
