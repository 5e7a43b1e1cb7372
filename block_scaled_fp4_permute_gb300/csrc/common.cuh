// common.cuh -- device helpers shared by the SiTU MoE kernels (sm_103a).
//
// Number formats (OCP Microscaling): E2M1 codes (sign in bit 3, two
// exponent bits with bias 1, one mantissa bit), E4M3 "fn" (bias 7, max 448),
// UE8M0 (2^(b-127)).  bf16 values are handled as raw 16-bit patterns packed
// in pairs (low half = even element).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace situ {

constexpr int kWarp = 32;

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialisation attribute may start while its predecessor on the
// stream is still running; griddep_wait blocks until the predecessor has
// completed and its writes are visible (a no-op for a normal launch), and
// griddep_launch_dependents lets the successor start launching once every
// CTA of this grid has issued it.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Eight E2M1 codes (one 32-bit word, element 0 in bits 0..3) to eight bf16
// values, exactly: out[q] holds elements (2q, 2q+1).  The bf16 bit patterns
// of the eight magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} are split into a
// high-byte table {00 3F 3F 3F 40 40 40 40} and a low-byte table
// {00 00 80 C0 00 40 80 C0}; PRMT looks four magnitudes up at a time, a
// second PRMT interleaves the bytes into bf16 pairs and the sign bits are
// moved to bit 15 / 31.
__device__ __forceinline__ void e2m1x8_to_bf16x8(uint32_t w, uint32_t out[4]) {
  const uint32_t kHiA = 0x3F3F3F00u, kHiB = 0x40404040u;
  const uint32_t kLoA = 0xC0800000u, kLoB = 0xC0804000u;
  uint32_t sel_lo = w & 0x7777u;
  uint32_t sel_hi = (w >> 16) & 0x7777u;
  uint32_t h0 = prmt(kHiA, kHiB, sel_lo), l0 = prmt(kLoA, kLoB, sel_lo);
  uint32_t h1 = prmt(kHiA, kHiB, sel_hi), l1 = prmt(kLoA, kLoB, sel_hi);
  out[0] = prmt(l0, h0, 0x5140u) | ((w << 12) & 0x00008000u) | ((w << 24) & 0x80000000u);
  out[1] = prmt(l0, h0, 0x7362u) | ((w << 4) & 0x00008000u) | ((w << 16) & 0x80000000u);
  out[2] = prmt(l1, h1, 0x5140u) | ((w >> 4) & 0x00008000u) | ((w << 8) & 0x80000000u);
  out[3] = prmt(l1, h1, 0x7362u) | ((w >> 12) & 0x00008000u) | (w & 0x80000000u);
}

// bf16x2 multiply (round to nearest even; exact when the product is a bf16).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// E4M3 code to fp32, exactly (finite codes).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float v = (e == 0) ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (b & 0x80u) ? -v : v;
}

// 2^k as fp32 for k in [-149, 127] (exact, including the subnormal range).
__device__ __forceinline__ float exp2i(int k) {
  if (k >= -126) return __uint_as_float((uint32_t)(k + 127) << 23);
  return __uint_as_float(1u << (k + 149));
}

// UE8M0 scale byte in [1, 254] as a bf16 pair (both halves 2^(b-127)).
__device__ __forceinline__ uint32_t ue8m0_to_bf16x2(uint32_t b) {
  return (b << 7) | (b << 23);
}

// fp32 pair -> bf16 pair, round to nearest even; lo in the low half.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

// E4M3 codes of two fp32 values, nearest even with saturation to +-448;
// returns lo in bits 0..7 and hi in bits 8..15.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return (uint32_t)d;
}

// fp32 pair -> f16 pair, round to nearest even; lo in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float f16_to_f32(uint32_t h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"((uint16_t)h));
  return f;
}

// Y rows of the block-scaled prefill path: f16 mantissas with one
// power-of-two scale per 32 elements, 2^(byte - 127), chosen so that the
// block maximum lies in [2^14, 2^15): 11 significant bits for every element
// within 2^-28 of the block maximum.
__device__ __forceinline__ int y16_exponent(float amax) {
  const int k = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  if (k == 0) return 0;                 // zero (or an fp32 subnormal block)
  const int ex = k - 127 - 14;
  return ex < -127 ? -127 : (ex > 127 ? 127 : ex);
}

// Two E4M3 codes (low byte = first) to fp32, exactly, through the hardware
// E4M3 -> f16 conversion (every finite E4M3 value is an f16).
__device__ __forceinline__ void e4m3x2_to_f32x2(uint32_t codes, float& lo, float& hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)codes));
  asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"((uint16_t)(h2 & 0xFFFFu)));
  asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"((uint16_t)(h2 >> 16)));
}
__device__ __forceinline__ float e4m3_code_to_f32(uint32_t code) {
  float lo, hi;
  e4m3x2_to_f32x2(code & 0xFFu, lo, hi);
  return lo;
}

// The MXFP8 block exponent: the smallest e in [-127, 127] with
// amax * 2^-e <= 448, from the fp32 bits of amax (amax = m * 2^k with
// m in [1, 2); 448 = 1.75 * 2^8, so e = k - 8 + (m > 1.75)).
__device__ __forceinline__ int mxfp8_exponent(float amax) {
  uint32_t bits = __float_as_uint(amax);
  int k = (int)((bits >> 23) & 0xFFu) - 127;
  if (((bits >> 23) & 0xFFu) == 0) return -127;   // zero or fp32 subnormal
  int e = k - 8 + (((bits & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// A block of 32 values held exactly in fp32 (bf16 values) as two MXFP8
// blocks, hi + lo: hi is the block rounded to E4M3 under its MXFP8 scale 2^e
// (mxfp8_exponent), lo the remainder rounded to E4M3 under 2^(e - c),
// c = min(4, e + 127).  hi carries the leading four significant bits of an
// element and lo the next four, so the pair represents every element whose
// exponent is within 2^-14 of the block maximum exactly, and any other with
// an absolute error below 2^-22 of the maximum.  Codes go to hi[0..7] and
// lo[0..7] (element 4j + u in byte u of word j); returns the two scale bytes
// (hi in bits 0..7, lo in bits 8..15).
__device__ __forceinline__ uint32_t split_hl32(const float* v, uint32_t* hi, uint32_t* lo) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const int e = mxfp8_exponent(amax);
  const int c = min(4, e + 127);
  const float s = exp2i(-e), sl = exp2i(c);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float x[4], r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = v[4 * j + u] * s;
    const uint32_t h01 = f32x2_to_e4m3x2(x[0], x[1]), h23 = f32x2_to_e4m3x2(x[2], x[3]);
    float f[4];
    e4m3x2_to_f32x2(h01, f[0], f[1]);
    e4m3x2_to_f32x2(h23, f[2], f[3]);
#pragma unroll
    for (int u = 0; u < 4; ++u) r[u] = x[u] - f[u];
    hi[j] = h01 | (h23 << 16);
    lo[j] = f32x2_to_e4m3x2(r[0] * sl, r[1] * sl) | (f32x2_to_e4m3x2(r[2] * sl, r[3] * sl) << 16);
  }
  return (uint32_t)(e + 127) | ((uint32_t)(e - c + 127) << 8);
}

// SiTU: [b*tanh(g/b)*sigmoid(g)] * [bl*tanh(u/bl)], a cap <= 0 meaning the
// factor's limit (g*sigmoid(g), u).  With E(y) = exp(-y):
//   sigmoid(g) = 1 / (1 + E(g)),  tanh(y) = (1 - E(2y)) / (1 + E(2y)),
// so the whole product is one fraction and takes three fast exponentials and
// one division.  Each E is 2^z with z = -y * log2(e), log2(e) folded into
// the constants, and z clamped at 25 log2(e) (y >= -25), where tanh is -1
// and sigmoid 0 to within 1.4e-11 absolute; larger y only drives E to 0, so
// the product of the three denominators stays below 4e32.  The error is a
// few fp32 ulps of the factors' magnitudes (absolute, not relative, near 0).
// k0 = -2 log2(e)/b and k1 = -2 log2(e)/bl are the expert's constants, 0
// for a cap that is off; the body has no branches, so that the element loops
// of the epilogues interleave many independent chains.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float exp2_approx(float z) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(z));
  return r;
}
// 2^min(z, 25 log2 e)
__device__ __forceinline__ float exp2_clamped(float z) { return exp2_approx(fminf(z, 25.f * kLog2e)); }
__device__ __forceinline__ float situ_k(float g, float u, float b, float k0, float bl, float k1) {
  const float e0 = exp2_clamped(-kLog2e * g);
  const float e1 = exp2_clamped(k0 * g);
  const float e2 = exp2_clamped(k1 * u);
  const float ng = k0 < 0.f ? b * (1.f - e1) : g;
  const float dg = k0 < 0.f ? 1.f + e1 : 1.f;
  const float nu = k1 < 0.f ? bl * (1.f - e2) : u;
  const float du = k1 < 0.f ? 1.f + e2 : 1.f;
  return __fdividef(ng * nu, ((1.f + e0) * dg) * du);
}
__device__ __forceinline__ float situ_cap_k(float b) { return b > 0.f ? -2.f * kLog2e / b : 0.f; }

// SwigluBias g * sigmoid(alpha * g) * (u + beta), the exponent argument
// clamped to [-80, 80], where sigmoid is 0 or 1 to fp32 precision.
__device__ __forceinline__ float swiglu_bias_f(float g, float u, float alpha, float beta) {
  return __fdividef(g * (u + beta), 1.f + __expf(-fminf(fmaxf(alpha * g, -80.f), 80.f)));
}

// FC1's gated activation: kind 0 is SiTU (caps p0 = b, p1 = bl), kind 1
// SwigluBias (p0 = alpha, p1 = beta).  with_act(kind, p0, p1, body) picks
// the kind once and runs body(act), act(g, u) being the activation of that
// kind, so the element loops inside body carry no per-element branch.
constexpr int kActSitu = 0, kActSwigluBias = 1;
template <class Body>
__device__ __forceinline__ void with_act(int kind, float p0, float p1, Body&& body) {
  if (kind == kActSwigluBias) {
    body([=](float g, float u) { return swiglu_bias_f(g, u, p0, p1); });
  } else {
    const float k0 = situ_cap_k(p0), k1 = situ_cap_k(p1);
    body([=](float g, float u) { return situ_k(g, u, p0, k0, p1, k1); });
  }
}

}  // namespace situ
