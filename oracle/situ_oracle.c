/*
 * situ_oracle.c -- plain, slow CPU oracle for the SiTU routed-MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline / reference leg use it.  It shares no code, header, table or
 * helper with the CUDA library; its format tables are written out here from
 * the format definitions themselves.
 *
 * What it computes (each function names the passage it follows):
 *   - the block-scaled number formats the layer consumes: E2M1 (FP4) values,
 *     UE8M0 power-of-two block scales and E4M3 ("fn") values;
 *   - the per-token NVFP4 activation quantisation of the NVFP4 variant
 *     (FlashInfer 0.6.18 MoE-LoRA AOT release notes, Summary: the NVFP4
 *     path scales its activations per token; the rule itself is a reading,
 *     see below);
 *   - the per-token MXFP8 activation quantisation of the w4a8 chain
 *     (TokenSpeed SiTU, "Activation precision (w4a16 vs w4a8)" and
 *     "Supported contract": MXFP8 activations with a per-token
 *     hidden_states_scale block-scale tensor);
 *   - the routing step upstream of the layer, top-k of router logits with
 *     softmax weights (the golden reference MoE of TensorRT-LLM PR #17865
 *     applies a routing method to router logits; the method is a reading);
 *   - the expert permute with local-shard filtering (TokenSpeed SiTU,
 *     "Supported contract": top-k IDs stay global, experts outside the rank's
 *     contiguous shard are filtered, the output is a partial sum);
 *   - the routed-MoE forward: the golden per-token/per-slot loop of the
 *     SiTU reference MoE (TensorRT-LLM PR #17865, review comment on
 *     test_kimi_k3_situ_moe.py, `_reference_moe` / `_situ_act`), with the
 *     per-expert beta / linear beta taken from gemm1_alpha / gemm1_beta and
 *     the up half rescaled by g1_alphas_up / g1_alphas before the tanh
 *     (FlashInfer 0.6.18 SM100a+SM103a MoE-LoRA AOT release notes,
 *     "Changes since 875b7d7").
 *
 * Arithmetic is fp64 on exactly-dequantised operands.  Where a float value
 * decides a stored code (rounding the FC1 output to bf16, or to MXFP8 in the
 * w4a8 chain) the value is first rounded to fp32, the precision in which the
 * device takes the same decision.
 *
 * Readings of points the pages leave open:
 *   - E2M1 packing: element 2i in the low nibble of byte i.
 *   - W1 rows: gate rows 0..I-1, then up rows I..2I-1.
 *   - A cap (beta or linear beta) <= 0 switches that factor to its
 *     beta -> infinity limit: gate g*sigmoid(g), up u.
 *   - MXFP8 scale: the smallest power of two 2^e, e in [-127,127], with
 *     amax * 2^-e <= 448; elements round to nearest even E4M3, saturating.
 *   - The routing weight is applied after FC2, in the un-permute sum.
 *   - NVFP4: per-tensor fp32 global scales (w1 gate half, w1 up half, w2,
 *     per-token activation) multiply the dot products they belong to.
 *
 * Build: gcc -O2 -shared -fPIC -pthread situ_oracle.c -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------ */
/* Formats (OCP Microscaling formats: E2M1, E4M3, E8M0; bfloat16)      */
/* ------------------------------------------------------------------ */

/* E2M1: 1 sign bit (bit 3), 2 exponent bits (bias 1), 1 mantissa bit.
 * Exponent field 0 is subnormal: value = m * 0.5. */
double oracle_e2m1_value(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return s ? -mag : mag;
}

/* E4M3 "fn": 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinities; exponent 15 with mantissa 7 is NaN.  Exponent field 0 is
 * subnormal: value = m/8 * 2^-6. */
double oracle_e4m3_value(unsigned code) {
  unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  double mag;
  if (e == 15u && m == 7u) return NAN;
  if (e == 0) mag = ldexp((double)m / 8.0, -6);
  else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return s ? -mag : mag;
}

/* UE8M0: an unsigned biased exponent, value 2^(b-127); 255 is NaN. */
double oracle_ue8m0_value(unsigned b) {
  if (b == 255u) return NAN;
  return ldexp(1.0, (int)b - 127);
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round an fp32 value to bfloat16, nearest-even (finite inputs). */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* Round a finite value to E4M3 by searching the table of non-negative
 * finite codes 0x00..0x7E (values increase with the code): nearest value,
 * ties to the even code, magnitudes above 448 saturate to 448.  The sign is
 * kept, so negative values that round to zero give 0x80. */
unsigned oracle_e4m3_encode(double v) {
  unsigned sign = signbit(v) ? 0x80u : 0u;
  double a = fabs(v);
  if (a >= 448.0) return sign | 0x7Eu;
  unsigned lo = 0, hi = 0x7E; /* invariant: value(lo) <= a < value(hi) */
  while (hi - lo > 1) {
    unsigned mid = (lo + hi) / 2;
    if (oracle_e4m3_value(mid) <= a) lo = mid; else hi = mid;
  }
  double dlo = a - oracle_e4m3_value(lo), dhi = oracle_e4m3_value(hi) - a;
  unsigned code;
  if (dlo < dhi) code = lo;
  else if (dhi < dlo) code = hi;
  else code = (lo & 1u) ? hi : lo;
  return sign | code;
}

/* MXFP8 block exponent: the smallest e in [-127, 127] with
 * amax * 2^-e <= 448 (448 = largest finite E4M3). */
int oracle_mxfp8_exponent(double amax) {
  if (!(amax > 0.0)) return -127;
  int p;
  frexp(amax, &p);          /* amax = f * 2^p, f in [0.5, 1) */
  int e = p - 10;           /* amax * 2^-e = f * 1024 > 448 */
  while (ldexp(amax, -e) > 448.0) e++;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* Quantise one block of n fp32 values to MXFP8: returns the UE8M0 scale
 * byte and writes n E4M3 codes. */
static unsigned mxfp8_block(const float* v, int n, uint8_t* q) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i) if (fabs((double)v[i]) > amax) amax = fabs((double)v[i]);
  int e = oracle_mxfp8_exponent(amax);
  for (int i = 0; i < n; ++i) q[i] = (uint8_t)oracle_e4m3_encode(ldexp((double)v[i], -e));
  return (unsigned)(e + 127);
}

/* ------------------------------------------------------------------ */
/* A small parallel-for (pthreads, static interleave) for the slow loops */
/* ------------------------------------------------------------------ */

typedef void (*range_fn)(void* ctx, long i);
typedef struct { range_fn fn; void* ctx; long n; int nthreads; int tid; } worker_arg;

static void* worker(void* p) {
  worker_arg* w = (worker_arg*)p;
  for (long i = w->tid; i < w->n; i += w->nthreads) w->fn(w->ctx, i);
  return NULL;
}

static int g_threads = 0;
void oracle_set_threads(int n) { g_threads = n; }
int oracle_get_threads(void) {
  if (g_threads > 0) return g_threads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static void parallel_for(long n, range_fn fn, void* ctx) {
  int nt = oracle_get_threads();
  if (nt > n) nt = (int)n;
  if (nt <= 1) { for (long i = 0; i < n; ++i) fn(ctx, i); return; }
  pthread_t th[256];
  worker_arg args[256];
  if (nt > 256) nt = 256;
  for (int t = 0; t < nt; ++t) {
    args[t].fn = fn; args[t].ctx = ctx; args[t].n = n; args[t].nthreads = nt; args[t].tid = t;
    pthread_create(&th[t], NULL, worker, &args[t]);
  }
  for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* MXFP8 activation quantisation (w4a8 chain)                           */
/* ------------------------------------------------------------------ */

typedef struct { const uint16_t* x; int H; uint8_t* q; uint8_t* s; } quant_ctx;

static void quant_row(void* p, long t) {
  quant_ctx* c = (quant_ctx*)p;
  float buf[32];
  for (int b = 0; b < c->H / 32; ++b) {
    for (int i = 0; i < 32; ++i) buf[i] = (float)oracle_bf16_value(c->x[(size_t)t * c->H + b * 32 + i]);
    c->s[(size_t)t * (c->H / 32) + b] =
        (uint8_t)mxfp8_block(buf, 32, c->q + (size_t)t * c->H + b * 32);
  }
}

/* x: bf16 [T,H] row-major; q: E4M3 [T,H]; s: UE8M0 [T,H/32] (one scale per
 * token per 32 consecutive hidden elements).  Requires H % 32 == 0 and
 * finite inputs. */
void oracle_quant_mxfp8(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* s) {
  quant_ctx c = {x, H, q, s};
  parallel_for(T, quant_row, &c);
}

/* ------------------------------------------------------------------ */
/* NVFP4 activation quantisation (per-token)                            */
/* ------------------------------------------------------------------ */

/* Round a value to E2M1 by searching the eight magnitudes: nearest value,
 * ties to the even code, magnitudes above 6 saturate to 6.  The sign is
 * kept (bit 3), so a negative value that rounds to zero gives code 8. */
unsigned oracle_e2m1_encode(double v) {
  unsigned sign = signbit(v) ? 8u : 0u;
  double a = fabs(v);
  if (a >= 6.0) return sign | 7u;
  unsigned lo = 0;
  while (lo < 7 && oracle_e2m1_value(lo + 1) <= a) ++lo;   /* value(lo) <= a < value(lo + 1) */
  unsigned hi = lo + 1;
  double dlo = a - oracle_e2m1_value(lo), dhi = oracle_e2m1_value(hi) - a;
  unsigned code;
  if (dlo < dhi) code = lo;
  else if (dhi < dlo) code = hi;
  else code = (lo & 1u) ? hi : lo;
  return sign | code;
}

typedef struct { const uint16_t* x; int H; uint8_t* q; uint8_t* s; float* gs; } nvq_ctx;

/* The per-token NVFP4 rule of the layer's NVFP4 activations (a reading:
 * the FlashInfer notes name per-token NVFP4 activation scaling, and the
 * pages fix no rule).  Every step is one fp32 operation, rounded to
 * nearest even, as the device performs it:
 *   gs     = amax_row / 2688   (2688 = 6 * 448; 1 when the row is all zero)
 *   s      = E4M3(amax_block16 / (6 * gs))   (round to nearest even)
 *   denom  = value(s) * gs
 *   code_i = E2M1(x_i / denom), or 0 when denom is 0. */
static void nvq_one_row(const uint16_t* xr, int H, uint8_t* q, uint8_t* s, float* gs_out) {
  float amax = 0.0f;
  for (int i = 0; i < H; ++i) {
    float a = fabsf((float)oracle_bf16_value(xr[i]));
    if (a > amax) amax = a;
  }
  float gs = amax / 2688.0f;
  if (!(gs > 0.0f)) gs = 1.0f;
  *gs_out = gs;
  for (int b = 0; b < H / 16; ++b) {
    float ab = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float a = fabsf((float)oracle_bf16_value(xr[b * 16 + i]));
      if (a > ab) ab = a;
    }
    float den6 = 6.0f * gs;
    float qv = ab / den6;
    unsigned s8 = oracle_e4m3_encode((double)qv);
    float denom = (float)oracle_e4m3_value(s8) * gs;
    s[b] = (uint8_t)s8;
    for (int i = 0; i < 16; i += 2) {
      unsigned c0 = 0, c1 = 0;
      if (denom > 0.0f) {
        float y0 = (float)oracle_bf16_value(xr[b * 16 + i]) / denom;
        float y1 = (float)oracle_bf16_value(xr[b * 16 + i + 1]) / denom;
        c0 = oracle_e2m1_encode((double)y0);
        c1 = oracle_e2m1_encode((double)y1);
      }
      q[(b * 16 + i) / 2] = (uint8_t)(c0 | (c1 << 4));
    }
  }
}

static void nvq_row(void* p, long t) {
  nvq_ctx* c = (nvq_ctx*)p;
  nvq_one_row(c->x + (size_t)t * c->H, c->H, c->q + (size_t)t * (c->H / 2), c->s + (size_t)t * (c->H / 16),
              c->gs + t);
}

/* x: bf16 [T,H]; q: packed E2M1 [T,H/2] (element 2i in the low nibble);
 * s: E4M3 [T,H/16]; gs: fp32 [T].  Requires H % 16 == 0, finite inputs. */
void oracle_quant_nvfp4(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* s, float* gs) {
  nvq_ctx c = {x, H, q, s, gs};
  parallel_for(T, nvq_row, &c);
}

/* ------------------------------------------------------------------ */
/* Expert permute with local-shard filtering                            */
/* ------------------------------------------------------------------ */

/* topk_ids: int32 [T,K] global expert IDs.  Slot t*K+j is kept when
 * off <= id < off + E_loc.  Outputs:
 *   counts[E_loc]         kept slots per local expert;
 *   offsets[E_loc+1]      exclusive prefix sum of counts (offsets[E_loc] = R);
 *   permuted_src[T*K]     for row r < R, the slot t*K+j it came from; rows
 *                         are grouped by local expert and, within an expert,
 *                         in ascending slot order; entries >= R are -1;
 *   slot_to_row[T*K]      the row of each kept slot, -1 for dropped slots.
 * Returns R. */
int oracle_permute(const int32_t* ids, int T, int K, int E_total, int E_loc, int off,
                   int32_t* counts, int32_t* offsets, int32_t* permuted_src,
                   int32_t* slot_to_row) {
  (void)E_total;
  long S = (long)T * K;
  for (int e = 0; e < E_loc; ++e) counts[e] = 0;
  for (long i = 0; i < S; ++i) {
    int id = ids[i];
    if (id >= off && id < off + E_loc) counts[id - off]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E_loc; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)calloc((size_t)(E_loc > 0 ? E_loc : 1), sizeof(int32_t));
  for (long i = 0; i < S; ++i) { permuted_src[i] = -1; slot_to_row[i] = -1; }
  for (long i = 0; i < S; ++i) { /* ascending slot order: a stable scatter */
    int id = ids[i];
    if (id >= off && id < off + E_loc) {
      int e = id - off;
      int row = offsets[e] + fill[e]++;
      permuted_src[row] = (int32_t)i;
      slot_to_row[i] = row;
    }
  }
  free(fill);
  return offsets[E_loc];
}

/* ------------------------------------------------------------------ */
/* Routing from router logits                                          */
/* ------------------------------------------------------------------ */

/* The routing step upstream of the layer: the golden reference MoE of
 * TensorRT-LLM PR #17865 (`_reference_moe`) starts from router logits and
 * `routing_method.apply(router_logits)`, and TokenSpeed SiTU ("Supported
 * contract") takes the resulting top-k.  The pages name no routing method;
 * the reading taken is the one the workloads' routing weights follow:
 *   ids[t, 0..K-1]  the K largest logits of token t, in descending order of
 *                   logit, ties taken by the lower expert ID first;
 *   w[t, j]         renormalize = 1: exp(l_j) / sum over the K selected of
 *                   exp(l_i) (a softmax over the selected logits);
 *                   renormalize = 0: exp(l_j) / sum over all E logits (the
 *                   softmax probabilities of the selected experts).
 * Logits are finite fp32.  The weights are computed in fp64 with the
 * maximum subtracted first and rounded once to fp32.  Returns 0, or -1 for
 * bad sizes (K < 1 or K > E). */
int oracle_route_topk(const float* logits, int T, int E, int K, int renormalize, int32_t* ids, float* w) {
  if (T < 0 || E < 1 || K < 1 || K > E) return -1;
  char* taken = (char*)malloc((size_t)E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * E;
    memset(taken, 0, (size_t)E);
    /* K rounds of "the largest logit not taken yet, lowest ID among equals" */
    for (int j = 0; j < K; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;   /* strict: an equal later ID loses */
      }
      taken[best] = 1;
      ids[(size_t)t * K + j] = best;
    }
    const double m = l[ids[(size_t)t * K]];   /* the largest logit of the row */
    double den = 0.0;
    if (renormalize) {
      for (int j = 0; j < K; ++j) den += exp((double)l[ids[(size_t)t * K + j]] - m);
    } else {
      for (int e = 0; e < E; ++e) den += exp((double)l[e] - m);
    }
    for (int j = 0; j < K; ++j)
      w[(size_t)t * K + j] = (float)(exp((double)l[ids[(size_t)t * K + j]] - m) / den);
  }
  free(taken);
  return 0;
}

/* ------------------------------------------------------------------ */
/* SiTU gated activation                                                */
/* ------------------------------------------------------------------ */

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* [beta * tanh(g/beta) * sigmoid(g)] * [beta_lin * tanh(u/beta_lin)]
 * (TensorRT-LLM PR #17865, golden `_situ_act`).  A cap <= 0 takes the
 * factor's beta -> infinity limit (g*sigmoid(g) resp. u). */
/* CUTLASS SwigluBias, the variant printed beside SiTU in the golden
 * reference of TensorRT-LLM PR #17865 (`_swiglu_bias_act`):
 * gate * sigmoid(gate * alpha) * (linear + beta).  With alpha = 1 and
 * beta = 0 it is SwiGLU. */
double oracle_swiglu_bias(double g, double u, double alpha, double beta) {
  return g * sigmoid(g * alpha) * (u + beta);
}

double oracle_situ(double g, double u, double beta, double beta_lin) {
  double gate = (beta > 0.0) ? beta * tanh(g / beta) * sigmoid(g) : g * sigmoid(g);
  double up = (beta_lin > 0.0) ? beta_lin * tanh(u / beta_lin) : u;
  return gate * up;
}

/* ------------------------------------------------------------------ */
/* Routed-MoE forward                                                   */
/* ------------------------------------------------------------------ */

enum { ACT_BF16 = 0, ACT_MXFP8 = 1, ACT_NVFP4 = 2 };
enum { W_MXFP4 = 0, W_NVFP4 = 1 };
enum { ACT_FN_SITU = 0, ACT_FN_SWIGLU_BIAS = 1 };

typedef struct {
  int T, H, I, E_total, E_loc, off, K, act, wt;
  const uint16_t* x_bf16;   /* [T,H] bf16 (ACT_BF16) */
  const uint8_t* x_q;       /* [T,H] E4M3 (ACT_MXFP8) or [T,H/2] packed E2M1 (ACT_NVFP4) */
  const uint8_t* x_s;       /* [T,H/32] UE8M0 (ACT_MXFP8) or [T,H/16] E4M3 (ACT_NVFP4) */
  const float* x_gs;        /* [T] fp32 per-token global scale (ACT_NVFP4) */
  const int32_t* ids;       /* [T,K] global expert IDs */
  const float* wts;         /* [T,K] routing weights */
  const uint8_t* w1;        /* [E_loc, 2I, H/2] packed E2M1 */
  const uint8_t* w1s;       /* [E_loc, 2I, H/32] UE8M0 (MXFP4) or [E_loc, 2I, H/16] E4M3 (NVFP4) */
  const float* w1_gs;       /* [E_loc, 2] fp32 (NVFP4): gate half, up half */
  const uint8_t* w2;        /* [E_loc, H, I/2] packed E2M1 */
  const uint8_t* w2s;       /* [E_loc, H, I/32] UE8M0 or [E_loc, H, I/16] E4M3 */
  const float* w2_gs;       /* [E_loc] fp32 (NVFP4) */
  const float* beta;        /* gemm1_alpha [E_loc] */
  const float* beta_lin;    /* gemm1_beta  [E_loc] */
  const float* alpha_g;     /* g1_alphas    [E_loc] or NULL (1) */
  const float* alpha_u;     /* g1_alphas_up [E_loc] or NULL (1) */
  const float* alpha2;      /* g2_alphas    [E_loc] or NULL (1) */
  int activation;           /* ACT_FN_SITU (beta, beta_lin) or ACT_FN_SWIGLU_BIAS (alpha, beta) */
  int topk_in_fc1;          /* 1: the routing weight scales H1 instead of the FC2 output */
  int h1_nvfp4;             /* 1 (NVFP4 weights): H1 requantised per token to NVFP4 before FC2 */
} oracle_args;

/* Dequantise one packed FP4 matrix row (n elements) with its block scales:
 * MXFP4 = E2M1 * UE8M0 per 32, NVFP4 = E2M1 * E4M3 per 16 (the per-tensor
 * fp32 global scale is applied to the dot product, not here). */
static void dequant_fp4_row(const uint8_t* packed, const uint8_t* scales, int n, int nvfp4,
                            float* out) {
  int bs = nvfp4 ? 16 : 32;
  for (int k = 0; k < n; ++k) {
    unsigned byte = packed[k / 2];
    unsigned code = (k & 1) ? (byte >> 4) : (byte & 15u);
    double sc = nvfp4 ? oracle_e4m3_value(scales[k / bs]) : oracle_ue8m0_value(scales[k / bs]);
    out[k] = (float)(oracle_e2m1_value(code) * sc); /* exact in fp32 */
  }
}

/* The dequantised activation row of token t (fp32 holds it exactly). */
static void dequant_act_row(const oracle_args* a, int t, float* out) {
  int H = a->H;
  for (int k = 0; k < H; ++k) {
    double v;
    if (a->act == ACT_BF16) {
      v = oracle_bf16_value(a->x_bf16[(size_t)t * H + k]);
    } else if (a->act == ACT_MXFP8) {
      v = oracle_e4m3_value(a->x_q[(size_t)t * H + k]) *
          oracle_ue8m0_value(a->x_s[(size_t)t * (H / 32) + k / 32]);
    } else {
      unsigned byte = a->x_q[(size_t)t * (H / 2) + k / 2];
      unsigned code = (k & 1) ? (byte >> 4) : (byte & 15u);
      v = oracle_e2m1_value(code) * oracle_e4m3_value(a->x_s[(size_t)t * (H / 16) + k / 16]);
    }
    out[k] = (float)v;
  }
}

typedef struct {
  const oracle_args* a;
  int R;                      /* kept pairs in the subset */
  const int32_t* pair_tok;    /* [R] token of each pair */
  const float* pair_w;        /* [R] routing weight of each pair */
  const int32_t* exp_start;   /* [E_loc+1] pairs grouped by expert */
  double* y;                  /* [R, H] FC2 output per pair */
} expert_ctx;

/* One local expert: dequantise its W1/W2, then for each of its pairs run
 * FC1 -> SiTU -> (bf16 | MXFP8 round trip) -> FC2. */
static void run_expert(void* p, long e) {
  expert_ctx* c = (expert_ctx*)p;
  const oracle_args* a = c->a;
  int H = a->H, I = a->I;
  int p0 = c->exp_start[e], p1 = c->exp_start[e + 1];
  if (p0 == p1) return;
  int nv = (a->wt == W_NVFP4);
  int bs = nv ? 16 : 32;
  float* W1 = (float*)malloc(sizeof(float) * (size_t)2 * I * H);
  float* W2 = (float*)malloc(sizeof(float) * (size_t)H * I);
  float* x = (float*)malloc(sizeof(float) * (size_t)H);
  float* hf = (float*)malloc(sizeof(float) * (size_t)I);
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  for (int n = 0; n < 2 * I; ++n)
    dequant_fp4_row(a->w1 + ((size_t)e * 2 * I + n) * (H / 2),
                    a->w1s + ((size_t)e * 2 * I + n) * (H / bs), H, nv, W1 + (size_t)n * H);
  for (int n = 0; n < H; ++n)
    dequant_fp4_row(a->w2 + ((size_t)e * H + n) * (I / 2),
                    a->w2s + ((size_t)e * H + n) * (I / bs), I, nv, W2 + (size_t)n * I);
  double ag = a->alpha_g ? a->alpha_g[e] : 1.0;
  double au = a->alpha_u ? a->alpha_u[e] : 1.0;
  double a2 = a->alpha2 ? a->alpha2[e] : 1.0;
  double g1g = nv ? a->w1_gs[2 * e] : 1.0, g1u = nv ? a->w1_gs[2 * e + 1] : 1.0;
  double g2 = nv ? a->w2_gs[e] : 1.0;
  for (int pi = p0; pi < p1; ++pi) {
    int t = c->pair_tok[pi];
    double xg = (a->act == ACT_NVFP4) ? a->x_gs[t] : 1.0;
    dequant_act_row(a, t, x);
    /* FC1: gate row i and up row I+i, then SiTU. */
    for (int i = 0; i < I; ++i) {
      double accg = 0.0, accu = 0.0;
      const float* wg = W1 + (size_t)i * H;
      const float* wu = W1 + (size_t)(I + i) * H;
      for (int k = 0; k < H; ++k) { accg += (double)x[k] * wg[k]; accu += (double)x[k] * wu[k]; }
      double g = ag * g1g * xg * accg;
      double u = au * g1u * xg * accu;
      double h_act = (a->activation == ACT_FN_SWIGLU_BIAS) ? oracle_swiglu_bias(g, u, a->beta[e], a->beta_lin[e])
                                                           : oracle_situ(g, u, a->beta[e], a->beta_lin[e]);
      /* apply_topk_in_fc1: the slot's routing weight scales H1 before it is
       * rounded for FC2, and the un-permute sum is unweighted */
      if (a->topk_in_fc1) h_act *= (double)c->pair_w[pi];
      hf[i] = (float)h_act;
    }
    /* The FC1 output as FC2 consumes it. */
    if (nv && a->h1_nvfp4) {
      /* the NVFP4 chain with H1 requantised: H1 rounded to bf16, then the
       * per-token NVFP4 quantisation of that row (the rule of
       * oracle_quant_nvfp4) and its exact dequantisation code * scale * gs */
      uint16_t* hb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
      uint8_t* q = (uint8_t*)malloc((size_t)I / 2);
      uint8_t* sc = (uint8_t*)malloc((size_t)I / 16);
      float gs = 1.0f;
      for (int i = 0; i < I; ++i) hb[i] = oracle_f32_to_bf16(hf[i]);
      nvq_one_row(hb, I, q, sc, &gs);
      for (int i = 0; i < I; ++i) {
        unsigned code = (i & 1) ? (q[i / 2] >> 4) : (q[i / 2] & 15u);
        h[i] = oracle_e2m1_value(code) * oracle_e4m3_value(sc[i / 16]) * (double)gs;
      }
      free(hb); free(q); free(sc);
    } else if (a->act == ACT_MXFP8) {
      uint8_t q[32];
      for (int b = 0; b < I / 32; ++b) {
        double sc = oracle_ue8m0_value(mxfp8_block(hf + b * 32, 32, q));
        for (int i = 0; i < 32; ++i) h[b * 32 + i] = oracle_e4m3_value(q[i]) * sc;
      }
    } else {
      for (int i = 0; i < I; ++i) h[i] = oracle_bf16_value(oracle_f32_to_bf16(hf[i]));
    }
    /* FC2 */
    double* y = c->y + (size_t)pi * H;
    for (int n = 0; n < H; ++n) {
      const float* w = W2 + (size_t)n * I;
      double acc = 0.0;
      for (int i = 0; i < I; ++i) acc += h[i] * w[i];
      y[n] = a2 * g2 * acc;
    }
  }
  free(W1); free(W2); free(x); free(hf); free(h);
}

typedef struct {
  const oracle_args* a; const int32_t* toks; const int32_t* slot_pair;
  const double* y; double* out;
} combine_ctx;

/* Un-permute: out[t] = sum over kept slots j (ascending) of w[t,j] * y. */
static void combine_token(void* p, long ti) {
  combine_ctx* c = (combine_ctx*)p;
  const oracle_args* a = c->a;
  int H = a->H, K = a->K;
  int t = c->toks ? c->toks[ti] : (int)ti;
  double* o = c->out + (size_t)ti * H;
  for (int n = 0; n < H; ++n) o[n] = 0.0;
  for (int j = 0; j < K; ++j) {
    int pi = c->slot_pair[(size_t)ti * K + j];
    if (pi < 0) continue;
    double w = a->topk_in_fc1 ? 1.0 : a->wts[(size_t)t * K + j];
    const double* y = c->y + (size_t)pi * H;
    for (int n = 0; n < H; ++n) o[n] += w * y[n];
  }
}

/* Forward for a subset of tokens (toks[n_tok], or all T when toks is NULL).
 * out: fp64 [n_tok, H].  Rows of tokens with no kept slot are 0.
 * Returns the number of kept pairs in the subset, or -1 on a bad argument. */
int oracle_moe_forward(const oracle_args* a, int n_tok, const int32_t* toks, double* out) {
  if (!a || a->H % 32 || a->I % 32 || !a->beta || !a->beta_lin) return -1;
  int K = a->K, E = a->E_loc;
  int32_t* slot_pair = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_tok > 0 ? n_tok : 1) * K);
  int32_t* exp_start = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
  for (int ti = 0; ti < n_tok; ++ti) {       /* pairs per expert over the subset */
    int t = toks ? toks[ti] : ti;
    for (int j = 0; j < K; ++j) {
      int id = a->ids[(size_t)t * K + j];
      if (id >= a->off && id < a->off + E) exp_start[id - a->off + 1]++;
    }
  }
  for (int e = 0; e < E; ++e) exp_start[e + 1] += exp_start[e];
  int R = exp_start[E];
  int32_t* pair_tok = (int32_t*)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
  float* pair_w = (float*)malloc(sizeof(float) * (size_t)(R > 0 ? R : 1));
  int32_t* fill = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
  for (int ti = 0; ti < n_tok; ++ti) {
    int t = toks ? toks[ti] : ti;
    for (int j = 0; j < K; ++j) {
      int id = a->ids[(size_t)t * K + j];
      int pi = -1;
      if (id >= a->off && id < a->off + E) {
        int e = id - a->off;
        pi = exp_start[e] + fill[e]++;
        pair_tok[pi] = t;
        pair_w[pi] = a->wts[(size_t)t * K + j];
      }
      slot_pair[(size_t)ti * K + j] = pi;
    }
  }
  double* y = (double*)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1) * a->H);
  expert_ctx ec = {a, R, pair_tok, pair_w, exp_start, y};
  parallel_for(E, run_expert, &ec);
  combine_ctx cc = {a, toks, slot_pair, y, out};
  parallel_for(n_tok, combine_token, &cc);
  free(slot_pair); free(exp_start); free(pair_tok); free(pair_w); free(fill); free(y);
  return R;
}
