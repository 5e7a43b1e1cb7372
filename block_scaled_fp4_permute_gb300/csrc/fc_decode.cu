// fc_decode.cu -- FC1 (gate/up + SiTU) and FC2 for decode-sized token tiles.
//
// Decode streams every touched expert's FP4 weights once and has one or two
// tokens per expert, so the bound is HBM bandwidth plus the ALU work of
// turning FP4 into MMA operands.  This path keeps the latter small:
//   * E2M1 codes become f16 pairs with the hardware conversion
//     (cvt.rn.f16x2.e2m1x2, exact), one instruction per two weights;
//   * weight block scales are applied in fp32 after each block's MMAs
//     (acc += scale * partial), the way a block-scaled MMA applies them,
//     instead of rescaling every weight;
//   * activations arrive as "f16 block rows" (mantissa * per-32-block fp32
//     scale), built once per row: gather16 converts the token-major input
//     in expert order (bf16 rows take one power-of-two scale per 32-element
//     block that puts the block maximum in [2^14, 2^15), exact for every
//     element within 2^-28 of it; MXFP8 rows convert exactly and keep their
//     block scales;
//     NVFP4 rows convert exactly with the E4M3 block scales folded in and
//     the per-token fp32 scale as the row scale), and FC1's epilogue writes
//     H1 the same way for FC2.
// A CTA stages its 8-row token tile for the whole K with one cp.async pass,
// after it has started its weight stream.  Each warp streams its own 16
// weight rows, and their block scales, through a kST-stage shared ring with
// cp.async copies (full sectors, asynchronous); the stream runs on across
// the m-tiles a CTA owns, so the next m-tile's loads overlap an epilogue.
//
// Fragment mapping (m16n8k16, A = weights, B = tokens): within a 32-element
// MXFP4 block lane (g, c) owns elements 8c..8c+7 of rows g and g+8, so one
// 4-byte read per row feeds both k16 steps of the block; for NVFP4 the lane
// owns elements 16s + 4c..+3 of step s, which keeps each step inside one
// 16-element scale block.  The K order is permuted identically in A and B,
// so the contraction is unchanged.
#include "situ_internal.h"

namespace situ {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kNT = 8;                  // tokens per CTA
constexpr int kST = 5;                  // weight-ring stages per warp (128-element chunks)
constexpr int kStageW = 16 * 64;        // one chunk of the warp's 16 rows
constexpr int kStageBytes = kStageW + 16 * 8;   // + their block scales (8 bytes per row)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// four E2M1 pairs (one 32-bit word, byte j = elements 2j, 2j+1) -> f16 pairs
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t* d) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(w));
}

// two E2M1 pairs in the low 16 bits -> f16 pairs
__device__ __forceinline__ void e2m1x4_to_f16x4(uint32_t w, uint32_t* d) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %2;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n}"
      : "=r"(d[0]), "=r"(d[1])
      : "r"(w));
}

// two E4M3 codes (low byte -> low half) -> f16 pair, exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)v));
  return d;
}

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void mma_f16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// first MMA of a block: C = 0
__device__ __forceinline__ void mma_f16_z(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ uint32_t ldg8(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(ok ? 16 : 0));
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(ok ? 8 : 0));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(ok ? 4 : 0));
}

// UE8M0 byte in [1, 254] as an fp32 power of two (byte 0, reserved for
// all-zero blocks, gives 0)
__device__ __forceinline__ float ue8m0_f32(uint32_t b) { return __uint_as_float(b << 23); }

// Row stride of the staged activation tile, in bytes: 2K padded so that the
// fragment loads of a quarter warp (LDS.128, MXFP4 mapping) or half warp
// (LDS.64, NVFP4 mapping) hit distinct banks.
__host__ __device__ __forceinline__ int x_stride(int K, bool nv) {
  int s = 2 * ((K + 127) / 128 * 128);   // rows zero-padded to whole 128-element chunks
  int want = nv ? 32 : 64;
  return s + ((want - (s % 128)) % 128 + 128) % 128;
}

}  // namespace

// ABLK: activation scales per (token, 32-block) (MXFP8 rows); otherwise one
// scale per token.
template <bool FC1, bool WNV, bool ABLK>
__global__ void __launch_bounds__(kThreads, 2) fcd_kernel(const FcdParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float s_tok[kNT];       // per-token activation scale (rows without block scales)
  __shared__ float s_w[kNT];         // routing weight of each row when it scales H1
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int K = p.K;
  const int nkb = K / 32;
  const int stride = x_stride(K, WNV);
  uint8_t* sX = smem;                                               // [kNT][stride]
  float* sS = reinterpret_cast<float*>(smem + kNT * stride);        // [kNT][nkb4]
  const int nkb4 = (nkb + 3) / 4 * 4;                               // blocks incl. zero padding
  float* sE = sS + nkb4 * kNT;                                      // epilogue [kNT][128]
  uint8_t* sWw = reinterpret_cast<uint8_t*>(sE + kNT * 128) + warp * kST * kStageBytes;

  const int ngroups = (p.n_mtiles + p.mg - 1) / p.mg;
  const int grp = blockIdx.x % ngroups;
  const int tile = blockIdx.x / ngroups;
  const int total = __ldg(p.tile_offsets + p.E_loc);
  if (tile >= total) return;
  const int2 ti = __ldg(p.tile_info + tile);
  const int e = ti.x;
  const int row0 = ti.y;
  const int nrows = min(kNT, __ldg(p.offsets + e + 1) - row0);
  const int mt0 = grp * p.mg;
  const int mcount = min(p.mg, p.n_mtiles - mt0);
  const int nch = (nkb + 3) / 4;
  const int steps = mcount * nch;
  const int bsz = WNV ? 16 : 32;
  const size_t wrow = (size_t)(K / 2), srow = (size_t)(K / bsz);
  const uint8_t* wexp = p.w + (size_t)e * p.Mtot * wrow;
  const uint8_t* sexp = p.ws + (size_t)e * p.Mtot * srow;

  // weight row r16 (0..15 of the warp's 16) of m-tile mt
  auto row_of = [&](int mt, int r16, bool& v) -> int {
    if (FC1) {
      const int i = mt * 64 + warp * 8 + (r16 & 7);
      v = i < p.I;
      return r16 < 8 ? i : p.I + i;
    }
    const int r = mt * 128 + warp * 16 + r16;
    v = r < p.Mtot;
    return r;
  };

  // ---- weight ring: per stage, piece p of row r at r*64 + 16*(p ^ ((r>>1)&3)),
  // then the 16 rows' scale bytes for the chunk, 8 bytes per row ----
  const uint32_t sw_u = smem_addr(sWw);
  // scale bytes per row per chunk: 4 (MXFP4) or 8 (NVFP4); cp.async needs
  // them aligned, which whole-128 rows give; otherwise plain loads
  const int sc_bytes = WNV ? 8 : 4;
  const bool sc_async = ((srow % sc_bytes) == 0) && ((reinterpret_cast<uintptr_t>(p.ws) % sc_bytes) == 0) &&
                        (nkb % 4 == 0);
  int ld_mi = -1, ld_cc = nch - 1;        // position of the last issued chunk
  const uint8_t *cpA = wexp, *cpB = wexp, *cpS = sexp;
  bool cvA = false, cvB = false, cvS = false;
  auto issue = [&](int u, int slot) {
    if (++ld_cc == nch) {   // next m-tile: recompute the row pointers once
      ld_cc = 0;
      ++ld_mi;
      const int mt = mt0 + ld_mi;
      int r;
      r = row_of(mt, lane >> 2, cvA);
      cpA = wexp + (size_t)(cvA ? r : 0) * wrow;
      r = row_of(mt, (lane >> 2) + 8, cvB);
      cpB = wexp + (size_t)(cvB ? r : 0) * wrow;
      r = row_of(mt, lane & 15, cvS);
      cpS = sexp + (size_t)(cvS ? r : 0) * srow;
    }
    const bool live = u < steps;
    const int cc = ld_cc;
    const int piece = lane & 3, rc = lane >> 2;
    const int b = cc * 4 + piece;
    const bool kb = live && b < nkb;
    const uint32_t st = sw_u + slot * kStageBytes;
    cp_async16(st + rc * 64 + 16 * (piece ^ ((rc >> 1) & 3)), cpA + (kb && cvA ? b * 16 : 0), kb && cvA);
    cp_async16(st + (rc + 8) * 64 + 16 * (piece ^ (((rc + 8) >> 1) & 3)), cpB + (kb && cvB ? b * 16 : 0),
               kb && cvB);
    if (lane < 16) {
      const uint32_t sdst = st + kStageW + lane * 8;
      const bool sv = live && cvS;
      if (sc_async) {
        if (WNV) cp_async8(sdst, cpS + (sv ? cc * 8 : 0), sv);
        else cp_async4(sdst, cpS + (sv ? cc * 4 : 0), sv);
      } else {
        // rows whose scales are not 4/8-byte aligned, or a partial last chunk
        uint32_t lo = 0u, hi = 0u;
#pragma unroll
        for (int q = 0; q < (WNV ? 8 : 4); ++q) {
          const int idx = cc * (WNV ? 8 : 4) + q;
          const uint32_t v = (sv && idx < (int)srow) ? ldg8(cpS + idx) : 0u;
          if (q < 4) lo |= v << (8 * q); else hi |= v << (8 * (q - 4));
        }
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(sdst), "r"(lo), "r"(hi));
      }
    }
    asm volatile("cp.async.commit_group;");
  };

  // start the weight stream (kST - 1 chunks) before staging the activations
  for (int i = 0; i < kST - 1; ++i) issue(i, i);

  // ---- stage the token tile: f16 block rows in expert order ----
  {
    const int kpad = nkb4 * 32;
    const int k8n = kpad / 8;            // 16-byte mantissa pieces per row
    const int s4n = nkb4 / 4;            // 16-byte scale pieces per row
    const uint32_t sx_u = smem_addr(sX), ss_u = smem_addr(sS);
    for (int it = tid; it < kNT * (k8n + s4n); it += kThreads) {
      if (it < kNT * k8n) {
        const int tok = it / k8n, k8 = it - tok * k8n;
        const bool v = tok < nrows && k8 < K / 8;   // columns past K are zero-filled
        cp_async16(sx_u + tok * stride + k8 * 16,
                   p.x16 + (size_t)(v ? row0 + tok : 0) * kpad + k8 * 8, v);
      } else {
        const int j2 = it - kNT * k8n;
        const int tok = j2 / s4n, s4 = j2 - tok * s4n;
        const bool v = tok < nrows;
        cp_async16(ss_u + (tok * nkb4 + s4 * 4) * 4, p.xs + (size_t)(v ? row0 + tok : 0) * nkb4 + s4 * 4, v);
      }
    }
    asm volatile("cp.async.commit_group;");
    // this group was committed after the weight prologue's groups, so
    // waiting for all but none of them is the simple, correct choice
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    // the scales of blocks past K are zero whatever the source row holds there
    for (int it = tid; it < kNT * (nkb4 - nkb); it += kThreads) {
      const int tok = it / (nkb4 - nkb), b = nkb + it % (nkb4 - nkb);
      sS[tok * nkb4 + b] = 0.f;
    }
    __syncthreads();
    if (tid < kNT) {
      s_tok[tid] = (tid < nrows && !ABLK) ? sS[tid * nkb4] : (tid < nrows ? 1.f : 0.f);
      s_w[tid] = (FC1 && p.topk_fc1 && tid < nrows) ? __ldg(p.topk_weights + __ldg(p.permuted_src + row0 + tid))
                                                     : 1.f;
    }
  }
  __syncthreads();

  const uint32_t sx_base = smem_addr(sX);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};

  // ---- epilogue of m-tile mt ----
  auto epilogue = [&](int mt) {
    const float t0 = s_tok[2 * c], t1 = s_tok[2 * c + 1];
    if (FC1) {
      float* sH = sE;   // [kNT][64]
      const int il = warp * 8 + g;
      if (mt * 64 + il < p.I) {
        const float ag = p.alpha_g ? __ldg(p.alpha_g + e) : 1.f;
        const float au = p.alpha_u ? __ldg(p.alpha_u + e) : 1.f;
        const float bt = __ldg(p.beta + e), btl = __ldg(p.beta_lin + e);
        const float gg = WNV ? __ldg(p.w1_gs + 2 * e) : 1.f, gu = WNV ? __ldg(p.w1_gs + 2 * e + 1) : 1.f;
        with_act(p.act_kind, bt, btl, [&](auto act) {
          sH[(2 * c) * 64 + il] = act(acc[0] * (ag * gg * t0), acc[2] * (au * gu * t0)) * s_w[2 * c];
          sH[(2 * c + 1) * 64 + il] = act(acc[1] * (ag * gg * t1), acc[3] * (au * gu * t1)) * s_w[2 * c + 1];
        });
      }
      __syncthreads();
      if (tid < kNT * 2) {
        const int tok = tid >> 1, blk = tid & 1;
        const int i0 = mt * 64 + blk * 32;
        if (tok < nrows && i0 < p.I) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = sH[tok * 64 + blk * 32 + i];
          const size_t r = (size_t)(row0 + tok);
          // H1 as FC2 consumes it: the MXFP8 round trip of h (w4a8) or h
          // rounded to bf16, held exactly as f16 mantissas x 2^ex
          uint32_t o[16];
          float scale;
          if (p.h_mxfp8) {
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
            const int ex = mxfp8_exponent(amax);
            const float sc = exp2i(-ex);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = e4m3x2_to_f16x2(f32x2_to_e4m3x2(v[2 * i] * sc, v[2 * i + 1] * sc));
            scale = exp2i(ex);
          } else {
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v[i] = bf16_lo(f32x2_to_bf16x2(v[i], 0.f));
              amax = fmaxf(amax, fabsf(v[i]));
            }
            int ex = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 14 : 0;
            ex = ex < -126 ? -126 : ex;
            const float inv = exp2i(-ex);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = f32x2_to_f16x2(v[2 * i] * inv, v[2 * i + 1] * inv);
            scale = exp2i(ex);
          }
          const int ipad = pad128(p.I);
          uint4* dst = reinterpret_cast<uint4*>(p.h16 + r * ipad + i0);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          p.hs[r * (ipad / 32) + i0 / 32] = scale;
        }
      }
      __syncthreads();
    } else {
      const float scale = (p.alpha2 ? __ldg(p.alpha2 + e) : 1.f) * (WNV ? __ldg(p.w2_gs + e) : 1.f);
      const int nl = warp * 16 + g;
      sE[(2 * c) * 128 + nl] = acc[0] * (scale * t0);
      sE[(2 * c + 1) * 128 + nl] = acc[1] * (scale * t1);
      sE[(2 * c) * 128 + nl + 8] = acc[2] * (scale * t0);
      sE[(2 * c + 1) * 128 + nl + 8] = acc[3] * (scale * t1);
      __syncthreads();
      {
        const int tok = tid >> 5, ch = tid & 31;   // 8 tokens x 32 float4
        const int n0 = mt * 128 + ch * 4;
        if (tok < nrows && n0 < p.Mtot)
          *reinterpret_cast<float4*>(p.y_out + (size_t)(row0 + tok) * p.Mtot + n0) =
              *reinterpret_cast<const float4*>(sE + tok * 128 + ch * 4);
      }
      __syncthreads();
    }
  };

  // ---- the (m-tile, chunk) stream: kST - 1 chunks in flight, across
  // m-tile boundaries, so the next m-tile's loads overlap an epilogue ----
  const int f = (g >> 1) & 3;
  const uint32_t off0 = 16 * (0 ^ f), off1 = 16 * (1 ^ f), off2 = 16 * (2 ^ f), off3 = 16 * (3 ^ f);
  const uint8_t* xrowp = sX + g * stride;
  int mi = 0, cc = 0, slot = 0;
  for (int u = 0; u < steps; ++u) {
    // refill the stage freed last step, then wait for chunk u
    issue(u + kST - 1, slot == 0 ? kST - 1 : slot - 1);
    asm volatile("cp.async.wait_group %0;" ::"n"(kST - 1) : "memory");
    __syncwarp();
    const uint8_t* stg = sWw + slot * kStageBytes;
    const uint8_t* rowA = stg + g * 64;
    const uint8_t* rowB = stg + (g + 8) * 64;
    // this lane's rows' scale bytes for the chunk
    const uint2 scA = *reinterpret_cast<const uint2*>(stg + kStageW + g * 8);
    const uint2 scB = *reinterpret_cast<const uint2*>(stg + kStageW + (g + 8) * 8);
    const uint32_t scA0 = scA.x, scA1 = scA.y, scB0 = scB.x, scB1 = scB.y;
    const uint8_t* xb = xrowp + cc * 256;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t off = q == 0 ? off0 : q == 1 ? off1 : q == 2 ? off2 : off3;
      float2 as = make_float2(1.f, 1.f);
      if (ABLK) as = make_float2(sS[(2 * c) * nkb4 + cc * 4 + q], sS[(2 * c + 1) * nkb4 + cc * 4 + q]);
      if (WNV) {
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const uint16_t ha = *reinterpret_cast<const uint16_t*>(rowA + off + 8 * s2 + 2 * c);
          const uint16_t hb = *reinterpret_cast<const uint16_t*>(rowB + off + 8 * s2 + 2 * c);
          uint32_t fa[2], fb[2];
          e2m1x4_to_f16x4((uint32_t)ha, fa);
          e2m1x4_to_f16x4((uint32_t)hb, fb);
          const uint2 bb = *reinterpret_cast<const uint2*>(xb + q * 64 + s2 * 32 + c * 8);
          const uint32_t b0 = bb.x, b1 = bb.y;
          float t4[4];
          mma_f16_z(t4, fa[0], fb[0], fa[1], fb[1], b0, b1);
          // scale of 16-block 2q+s2: byte (2q+s2) of the row's 8 scale bytes
          const int sb = 2 * q + s2;
          const uint32_t wa = sb < 4 ? scA0 : scA1, wb = sb < 4 ? scB0 : scB1;
          const float swa = e4m3_to_f32((wa >> (8 * (sb & 3))) & 0xFFu);
          const float swb = e4m3_to_f32((wb >> (8 * (sb & 3))) & 0xFFu);
          if (ABLK) {
            acc[0] = fmaf(t4[0], swa * as.x, acc[0]);
            acc[1] = fmaf(t4[1], swa * as.y, acc[1]);
            acc[2] = fmaf(t4[2], swb * as.x, acc[2]);
            acc[3] = fmaf(t4[3], swb * as.y, acc[3]);
          } else {
            acc[0] = fmaf(t4[0], swa, acc[0]);
            acc[1] = fmaf(t4[1], swa, acc[1]);
            acc[2] = fmaf(t4[2], swb, acc[2]);
            acc[3] = fmaf(t4[3], swb, acc[3]);
          }
        }
      } else {
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(rowA + off + 4 * c);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(rowB + off + 4 * c);
        uint32_t fa[4], fb[4];
        e2m1x8_to_f16x8(wa, fa);
        e2m1x8_to_f16x8(wb, fb);
        const uint4 bv = *reinterpret_cast<const uint4*>(xb + q * 64 + c * 16);
        const uint32_t bx[4] = {bv.x, bv.y, bv.z, bv.w};
        float t4[4];
        mma_f16_z(t4, fa[0], fb[0], fa[1], fb[1], bx[0], bx[1]);
        mma_f16(t4, fa[2], fb[2], fa[3], fb[3], bx[2], bx[3]);
        const float swa = ue8m0_f32((scA0 >> (8 * q)) & 0xFFu);
        const float swb = ue8m0_f32((scB0 >> (8 * q)) & 0xFFu);
        if (ABLK) {
          acc[0] = fmaf(t4[0], swa * as.x, acc[0]);
          acc[1] = fmaf(t4[1], swa * as.y, acc[1]);
          acc[2] = fmaf(t4[2], swb * as.x, acc[2]);
          acc[3] = fmaf(t4[3], swb * as.y, acc[3]);
        } else {
          acc[0] = fmaf(t4[0], swa, acc[0]);
          acc[1] = fmaf(t4[1], swa, acc[1]);
          acc[2] = fmaf(t4[2], swb, acc[2]);
          acc[3] = fmaf(t4[3], swb, acc[3]);
        }
      }
    }
    __syncwarp();   // every lane is done with this stage before it is refilled
    slot = slot == kST - 1 ? 0 : slot + 1;
    if (++cc == nch) {
      epilogue(mt0 + mi);
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
      cc = 0;
      ++mi;
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------
// gather16: expert-ordered f16 block rows from the token-major input
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(128) gather16_kernel(const Gather16Params p) {
  __shared__ float red[4];
  const long r = blockIdx.x;
  if (r >= __ldg(p.meta)) return;
  const int tid = threadIdx.x;
  const int K = p.K, kpad = pad128(K), nkb4 = kpad / 32, nkb = K / 32, k8n = K / 8;
  const int t = p.permuted_src ? __ldg(p.permuted_src + r) / p.top_k : (int)r;
  uint4* orow = reinterpret_cast<uint4*>(p.x16 + (size_t)r * kpad);
  float* srow = p.xs + (size_t)r * nkb4;
  float row_scale = 0.f;
  if (p.act == 0 && !p.row_scale) {
    // one power-of-two scale per 32-element block, putting the block maximum
    // in [2^14, 2^15): exact for every element within 2^-28 of its block's
    // maximum, whatever the other blocks of the row hold.  Lanes 4b..4b+3 of
    // a warp hold block b; every thread runs the same number of iterations,
    // so the shuffles see the whole warp.
    const uint4* xrow = reinterpret_cast<const uint4*>(p.x_bf16) + (size_t)t * k8n;
    for (int base = 0; base < k8n; base += 128) {
      const int k8 = base + tid;
      const bool valid = k8 < k8n;
      const uint4 v = valid ? __ldg(xrow + k8) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      // clamped at -126 so that 2^-ex stays an fp32 normal: a block whose
      // maximum is below 2^-112 then maps into [2^-14, 2^14), where every
      // bf16 value, subnormals included, is an exact f16
      int ex = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 14 : 0;
      ex = ex < -126 ? -126 : ex;
      const float inv = exp2i(-ex);
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = f32x2_to_f16x2(bf16_lo(w[i]) * inv, bf16_hi(w[i]) * inv);
      if (valid) {
        orow[k8] = make_uint4(o[0], o[1], o[2], o[3]);
        if ((k8 & 3) == 0) srow[k8 >> 2] = exp2i(ex);
      }
    }
  } else if (p.act == 0) {
    const uint4* xrow = reinterpret_cast<const uint4*>(p.x_bf16) + (size_t)t * k8n;
    float amax = 0.f;
    for (int k8 = tid; k8 < k8n; k8 += 128) {
      const uint4 v = __ldg(xrow + k8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    // row exponent: amax * 2^-ex in [2^14, 2^15)
    int ex = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 14 : 0;
    ex = ex < -126 ? -126 : ex;
    const float inv = exp2i(-ex);
    row_scale = exp2i(ex);
    for (int k8 = tid; k8 < k8n; k8 += 128) {
      const uint4 v = __ldg(xrow + k8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = f32x2_to_f16x2(bf16_lo(w[i]) * inv, bf16_hi(w[i]) * inv);
      orow[k8] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  } else if (p.act == 1) {
    const uint2* xrow = reinterpret_cast<const uint2*>(p.x_q + (size_t)t * K);
    int smax = 0;
    if (p.row_scale) {   // fold the block scales into the mantissas, relative to the row's largest
      for (int b = tid; b < nkb; b += 128) smax = max(smax, (int)__ldg(p.x_s + (size_t)t * nkb + b));
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) smax = max(smax, __shfl_xor_sync(0xffffffffu, smax, d));
      if ((tid & 31) == 0) red[tid >> 5] = (float)smax;
      __syncthreads();
      smax = (int)fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
      row_scale = exp2i(smax - 127);
    }
    for (int k8 = tid; k8 < k8n; k8 += 128) {
      const uint2 q = __ldg(xrow + k8);
      uint4 o = make_uint4(e4m3x2_to_f16x2(q.x & 0xFFFFu), e4m3x2_to_f16x2(q.x >> 16),
                           e4m3x2_to_f16x2(q.y & 0xFFFFu), e4m3x2_to_f16x2(q.y >> 16));
      if (p.row_scale) {
        // 2^(s_b - s_max) as an f16 pair: exact while the block is within
        // 2^15 of the row's largest block scale
        const int k = (int)__ldg(p.x_s + (size_t)t * nkb + k8 / 4) - smax;
        const uint32_t hk = k >= -14 ? (uint32_t)(k + 15) << 10 : (k >= -24 ? 1u << (k + 24) : 0u);
        const uint32_t f2 = hk | (hk << 16);
        o = make_uint4(hmul2_f16(o.x, f2), hmul2_f16(o.y, f2), hmul2_f16(o.z, f2), hmul2_f16(o.w, f2));
      }
      orow[k8] = o;
    }
  } else {
    const uint32_t* xrow = reinterpret_cast<const uint32_t*>(p.x_q + (size_t)t * (K / 2));
    for (int k8 = tid; k8 < k8n; k8 += 128) {
      uint32_t o[4];
      e2m1x8_to_f16x8(__ldg(xrow + k8), o);
      const uint32_t sb = __ldg(p.x_s + (size_t)t * (K / 16) + k8 / 2);
      const uint32_t s2 = e4m3x2_to_f16x2(sb | (sb << 8));
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = hmul2_f16(o[i], s2);
      orow[k8] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    row_scale = __ldg(p.x_gs + t);
  }
  for (int k8 = k8n + tid; k8 < kpad / 8; k8 += 128) orow[k8] = make_uint4(0, 0, 0, 0);
  const bool block_scaled_bf16 = p.act == 0 && !p.row_scale;   // written above, per block
  for (int b = tid; b < nkb4; b += 128) {
    if (block_scaled_bf16 && b < nkb) continue;
    float v = 0.f;
    if (b < nkb) v = (p.act == 1 && !p.row_scale) ? exp2i((int)__ldg(p.x_s + (size_t)t * nkb + b) - 127) : row_scale;
    srow[b] = v;
  }
}

cudaError_t launch_gather16(const Gather16Params& p, cudaStream_t st) {
  if (p.S <= 0) return cudaSuccess;
  gather16_kernel<<<(unsigned)p.S, 128, 0, st>>>(p);
  return cudaGetLastError();
}

size_t fcd_smem_bytes(int K, bool nvfp4) {
  return (size_t)kNT * x_stride(K, nvfp4) + (size_t)((K / 32 + 3) / 4 * 4) * kNT * 4 +
         (size_t)kNT * 128 * 4 + (size_t)kWarps * kST * kStageBytes;
}

template <bool FC1, bool WNV, bool ABLK>
static cudaError_t launch_fcd_t(const FcdParams& p, long max_tiles, cudaStream_t st) {
  const size_t smem = fcd_smem_bytes(p.K, WNV);
  static int set_for[64];
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (smem > 48 * 1024 && (dev >= 64 || set_for[dev] < (int)smem)) {
      cudaError_t err = cudaFuncSetAttribute(fcd_kernel<FC1, WNV, ABLK>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      if (dev < 64) set_for[dev] = (int)smem;
    }
  }
  const long ngroups = (p.n_mtiles + p.mg - 1) / p.mg;
  const long grid = max_tiles * ngroups;
  if (grid <= 0) return cudaSuccess;
  fcd_kernel<FC1, WNV, ABLK><<<(unsigned)grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fcd(const FcdParams& p, bool fc1, bool nvfp4, long max_tiles, cudaStream_t st) {
  const bool ablk = p.ablk != 0;
  if (fc1) {
    if (nvfp4) return ablk ? launch_fcd_t<true, true, true>(p, max_tiles, st) : launch_fcd_t<true, true, false>(p, max_tiles, st);
    return ablk ? launch_fcd_t<true, false, true>(p, max_tiles, st) : launch_fcd_t<true, false, false>(p, max_tiles, st);
  }
  if (nvfp4) return ablk ? launch_fcd_t<false, true, true>(p, max_tiles, st) : launch_fcd_t<false, true, false>(p, max_tiles, st);
  return ablk ? launch_fcd_t<false, false, true>(p, max_tiles, st) : launch_fcd_t<false, false, false>(p, max_tiles, st);
}

}  // namespace situ
