// permute_noalloc.cu -- situ_moe_permute for callers that cannot allocate.
//
// Same kernels, inputs and outputs as situ_moe_permute; the only scratch the
// permute needs (the per-chunk expert counts, ceil(T*top_k/4096) x E_loc
// int32) lives in a fixed array compiled into the library instead of in a
// caller-provided workspace.  Nothing here calls cudaMalloc, cudaFree or any
// other allocating routine.
#include <cuda.h>

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
// per device: the device address of the array and the ID of the context it
// was looked up in (0: none yet)
int32_t* g_scratch_addr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];

// The driver's cuCtxGetCurrent / cuCtxGetId, looked up once through the
// runtime (the library links only the runtime).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
template <class F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

// ID of the calling thread's current context (0 if there is none yet).
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch in the current device's context, looked up
// once per device and context (with that device current) and cached.  A
// context created anew on a device (after cudaDeviceReset, say) has a new
// ID, so its first call looks the address up again.
cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long ctx = current_context_id();
  const bool cacheable = dev >= 0 && dev < kMaxDevices;
  if (cacheable && ctx != 0 && g_scratch_ctx[dev] == ctx && g_scratch_addr[dev]) {
    *out = g_scratch_addr[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  err = cudaGetSymbolAddress(&p, g_permute_scratch);   // also makes the primary context current
  if (err != cudaSuccess) return err;
  if (ctx == 0) ctx = current_context_id();
  if (cacheable) {
    g_scratch_addr[dev] = (int32_t*)p;
    g_scratch_ctx[dev] = ctx;   // 0 (unknown) is never matched above
  }
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
