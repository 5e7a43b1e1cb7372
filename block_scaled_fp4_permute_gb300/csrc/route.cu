// route.cu -- top-k routing from router logits (the step upstream of the
// permute).
//
// The golden reference MoE of TensorRT-LLM PR #17865 starts from router
// logits and applies a routing method; TokenSpeed SiTU ("Supported
// contract") takes the resulting top-k.  Per token: the K largest logits,
// in descending order with ties to the lower expert ID, and fp32 weights
// that are a softmax over the K selected logits (renormalize = 1), or the
// selected experts' probabilities under a softmax over all E (0).
//
// One warp per token.  Each lane streams its strided share of the row
// (coalesced 128-byte warp loads) into a sorted list of its own K best
// (value, id) pairs held in registers; then K rounds of a warp-wide arg-max
// over the lanes' list heads pick the row's top-k in order, the winning
// lane popping its head.  The comparison is (value descending, id
// ascending) on the fp32 logits themselves, so the selection is exact.
#include "../../include/situ_moe.h"
#include "situ_internal.h"

#include <utility>

namespace situ {

namespace {

constexpr int kRouteWarps = 8;

// (va, ia) ranks before (vb, ib): the larger logit, or the lower ID of two
// equal logits
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// K is a template parameter so that every list index is a constant and the
// lists stay in registers
template <int K>
__global__ void __launch_bounds__(kRouteWarps * kWarp)
route_topk_kernel(const float* __restrict__ logits, int T, int E, int renorm, int32_t* __restrict__ ids,
                  float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const long t = (long)blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;
  // this lane's best K, sorted; sentinels rank after every finite logit
  float lv[K];
  int li[K];
#pragma unroll
  for (int p = 0; p < K; ++p) {
    lv[p] = -INFINITY;
    li[p] = 0x7FFFFFFF;
  }
  // (thv, thi): the list's K-th entry, the bar a new logit has to pass
  float thv = -INFINITY;
  int thi = 0x7FFFFFFF;
  for (int e = lane; e < E; e += kWarp) {
    float cv = __ldg(row + e);
    int ci = e;
    if (!before(cv, ci, thv, thi)) continue;
    // insertion by swaps keeps the list sorted; entries past K fall off
#pragma unroll
    for (int p = 0; p < K; ++p) {
      if (before(cv, ci, lv[p], li[p])) {
        const float tv = lv[p];
        const int ti = li[p];
        lv[p] = cv;
        li[p] = ci;
        cv = tv;
        ci = ti;
      }
    }
    thv = lv[K - 1];
    thi = li[K - 1];
  }
  // K rounds: the warp's best head is the row's next expert
  float my_v = -INFINITY;
  int my_i = 0;
#pragma unroll 1
  for (int j = 0; j < K; ++j) {
    float bv = lv[0];
    int bi = li[0];
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, d);
      if (before(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (li[0] == bi) {   // the winner pops its head (IDs are unique, sentinels never win)
#pragma unroll
      for (int p = 0; p < K - 1; ++p) {
        lv[p] = lv[p + 1];
        li[p] = li[p + 1];
      }
      lv[K - 1] = -INFINITY;
      li[K - 1] = 0x7FFFFFFF;
    }
    if (lane == j) {
      my_v = bv;
      my_i = bi;
    }
  }
  // weights: exp(l - max) over the selected (or all) logits, fp32
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < K ? expf(my_v - m) : 0.f;
  float den = 0.f;
  if (renorm) {
    den = ex;
  } else {
    for (int e = lane; e < E; e += kWarp) den += expf(__ldg(row + e) - m);
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) den += __shfl_xor_sync(0xffffffffu, den, d);
  if (lane < K) {
    ids[(size_t)t * K + lane] = my_i;
    w[(size_t)t * K + lane] = ex / den;
  }
}

template <int K>
void launch_k(const float* l, int T, int E, int renorm, int32_t* ids, float* w, cudaStream_t st) {
  const long blocks = ((long)T + kRouteWarps - 1) / kRouteWarps;
  route_topk_kernel<K><<<(unsigned)blocks, kRouteWarps * kWarp, 0, st>>>(l, T, E, renorm, ids, w);
}

template <int... Ks>
void launch_any(int K, const float* l, int T, int E, int renorm, int32_t* ids, float* w, cudaStream_t st,
                std::integer_sequence<int, Ks...>) {
  ((K == Ks + 1 ? launch_k<Ks + 1>(l, T, E, renorm, ids, w, st) : void()), ...);
}

}  // namespace

}  // namespace situ

extern "C" situ_status situ_moe_route_topk(const float* router_logits, int32_t T, int32_t num_experts_total,
                                           int32_t top_k, int32_t renormalize, int32_t* topk_ids,
                                           float* topk_weights, void* stream) {
  using namespace situ;
  if (T < 0 || num_experts_total < 1 || top_k < 1 || top_k > SITU_MAX_TOP_K || top_k > num_experts_total)
    return SITU_ERR_BAD_SHAPE;
  if (renormalize != 0 && renormalize != 1) return SITU_ERR_UNSUPPORTED;
  if (T == 0) return SITU_OK;
  if (!router_logits || !topk_ids || !topk_weights) return SITU_ERR_NULL_ARG;
  const void* ptrs[] = {router_logits, topk_ids, topk_weights};
  for (const void* p : ptrs)
    if ((reinterpret_cast<uintptr_t>(p) & 3u) != 0) return SITU_ERR_MISALIGNED;
  launch_any(top_k, router_logits, T, num_experts_total, renormalize, topk_ids, topk_weights, (cudaStream_t)stream,
             std::make_integer_sequence<int, SITU_MAX_TOP_K>{});
  return cudaGetLastError() == cudaSuccess ? SITU_OK : SITU_ERR_CUDA;
}
