// permute_noalloc.cu -- situ_moe_permute for callers that cannot allocate.
//
// Same kernels, inputs and outputs as situ_moe_permute; the only scratch the
// permute needs (the per-chunk expert counts, ceil(T*top_k/4096) x E_loc
// int32) lives in a fixed array compiled into the library instead of in a
// caller-provided workspace.  Nothing here calls cudaMalloc, cudaFree or any
// other allocating routine.
#include <mutex>

#include "../../include/situ_moe.h"
#include "situ_internal.h"

namespace {

// The scratch itself.  Host code must not pass this name to a kernel: on
// the host it is only a stand-in symbol, and its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) int32_t g_permute_scratch[SITU_NOALLOC_SCRATCH_INTS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_addr[kMaxDevices];   // device address of the array, per device

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev >= 0 && dev < kMaxDevices && g_scratch_addr[dev]) {
    *out = g_scratch_addr[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  err = cudaGetSymbolAddress(&p, g_permute_scratch);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < kMaxDevices) g_scratch_addr[dev] = (int32_t*)p;
  *out = (int32_t*)p;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" situ_status situ_moe_permute_noalloc(const int32_t* topk_ids, int32_t T, int32_t top_k,
                                                int32_t num_experts_total,
                                                int32_t num_local_experts,
                                                int32_t local_expert_offset,
                                                int32_t* expert_counts, int32_t* expert_offsets,
                                                int32_t* permuted_src, int32_t* slot_to_row,
                                                void* stream) {
  if (T < 0 || top_k < 1 || top_k > SITU_MAX_TOP_K) return SITU_ERR_BAD_SHAPE;
  if (num_local_experts < 1 || num_local_experts > SITU_MAX_LOCAL_EXPERTS ||
      local_expert_offset < 0 || num_experts_total < 1 ||
      (int64_t)local_expert_offset + num_local_experts > (int64_t)num_experts_total)
    return SITU_ERR_BAD_SHAPE;
  if ((int64_t)T * top_k > (int64_t)0x7FFFFFFF) return SITU_ERR_BAD_SHAPE;
  if (T == 0) return SITU_OK;
  if (!topk_ids || !expert_counts || !expert_offsets || !permuted_src || !slot_to_row)
    return SITU_ERR_NULL_ARG;
  const void* ptrs[] = {topk_ids, expert_counts, expert_offsets, permuted_src, slot_to_row};
  for (const void* p : ptrs)
    if (!aligned16(p)) return SITU_ERR_MISALIGNED;
  // the fixed scratch must hold ceil(T*top_k / 4096) x num_local_experts counts
  if (situ::permute_scratch_bytes(T, top_k, num_local_experts) >
      sizeof(int32_t) * (size_t)SITU_NOALLOC_SCRATCH_INTS)
    return SITU_ERR_WORKSPACE_TOO_SMALL;
  int32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SITU_ERR_CUDA;
  // Every count the scan reads is written by the count kernel of this call,
  // so no part of the scratch has to be cleared first.
  cudaError_t err = situ::launch_permute(topk_ids, T, top_k, num_local_experts,
                                         local_expert_offset, 1, expert_counts, expert_offsets,
                                         nullptr, nullptr, permuted_src, slot_to_row, nullptr,
                                         scratch,
                                         (cudaStream_t)stream);
  return err == cudaSuccess ? SITU_OK : SITU_ERR_CUDA;
}
