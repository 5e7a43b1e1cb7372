// permute.cu -- expert histogram, prefix scan and stable scatter.
//
// Groups the (token, slot) pairs of a global top-k routing by local expert,
// dropping IDs outside the rank's contiguous shard (TokenSpeed SiTU,
// "Supported contract": top-k IDs stay global and the routing filters the
// experts outside the current shard).  The row order inside an expert is the
// ascending slot order, so the result is deterministic and bit-exact.
//
// Up to kPermChunk slots (decode) one CTA does everything in one launch
// (permute_small_kernel).  Beyond that, three launches over chunks of
// kPermChunk slots (the second and third with programmatic dependent launch,
// waiting for their predecessor before they read its output):
//   count   -- per-chunk histogram in shared memory (block-local atomics);
//   scan    -- one block: per-expert prefix over chunks, then an exclusive
//              scan over experts of the counts and of the GEMM token tiles
//              (ceil(count / tile_n)), with a table tile -> (expert, first
//              row) for the GEMMs; clears the unused permuted_src tail;
//   scatter -- per chunk: per-warp counts, a prefix over warps, then each
//              warp walks its slots 32 at a time; __match_any_sync groups the
//              lanes that hit the same expert and a popcount of the lower
//              peers gives each lane its rank, so equal experts keep slot
//              order without any global atomics.
// Scratch: blk_counts [n_chunks, E_loc] int32.
#include "situ_internal.h"

namespace situ {

// count and scatter take 1024 threads per chunk (4 slots each; 128 per warp
// in the scatter), or 256 when 32 warps' counts of E_loc experts would not
// fit in shared memory
constexpr int kPermThreads = 1024;
constexpr int kPermThreadsFew = 256;
constexpr size_t kPermMaxSmem = 160 * 1024;

__device__ __forceinline__ int local_expert(int id, int off, int E_loc) {
  int e = id - off;
  return (id >= off && e < E_loc) ? e : -1;
}

__global__ void __launch_bounds__(kPermThreads)
permute_count_kernel(const int32_t* __restrict__ ids, long S, int E_loc, int off,
                     int32_t* __restrict__ blk_counts) {
  extern __shared__ int32_t hist[];
  griddep_launch_dependents();   // the scan may start launching
  for (int e = threadIdx.x; e < E_loc; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  long base = (long)blockIdx.x * kPermChunk;
  for (int i = threadIdx.x; i < kPermChunk; i += blockDim.x) {
    long s = base + i;
    if (s < S) {
      int e = local_expert(__ldg(ids + s), off, E_loc);
      if (e >= 0) atomicAdd(&hist[e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E_loc; e += blockDim.x)
    blk_counts[(size_t)blockIdx.x * E_loc + e] = hist[e];
}

// Exclusive scan of one int per thread across the block; returns the
// thread's prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* total) {
  __shared__ int warp_sums[32];
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += y;
    }
    warp_sums[lane] = w;   // inclusive prefix over warps
  }
  __syncthreads();
  int warp_prefix = warp ? warp_sums[warp - 1] : 0;
  *total = warp_sums[nwarps - 1];
  __syncthreads();
  return warp_prefix + x - v;
}

__global__ void __launch_bounds__(1024)
permute_scan_kernel(int32_t* __restrict__ blk_counts, int nblk, int E_loc, long S, int tile_n,
                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ tile_offsets, int2* __restrict__ tile_info,
                    int32_t* __restrict__ permuted_src, int32_t* __restrict__ meta) {
  griddep_wait();   // the chunk counts
  griddep_launch_dependents();
  // 1. per expert: prefix over chunks (becomes each chunk's base), total
  // count; the chunk counts are loaded 16 at a time, so that each batch costs
  // one memory round trip instead of one per chunk
  constexpr int kScanBatch = 16;
  for (int e = threadIdx.x; e < E_loc; e += blockDim.x) {
    int run = 0;
    for (int b0 = 0; b0 < nblk; b0 += kScanBatch) {
      int v[kScanBatch];
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j)
        v[j] = b0 + j < nblk ? blk_counts[(size_t)(b0 + j) * E_loc + e] : 0;
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j) {
        if (b0 + j < nblk) blk_counts[(size_t)(b0 + j) * E_loc + e] = run;
        run += v[j];
      }
    }
    counts[e] = run;
  }
  __syncthreads();
  // 2. exclusive scans over experts: each thread owns a contiguous segment
  int per = (E_loc + blockDim.x - 1) / blockDim.x;
  int e0 = min(E_loc, (int)threadIdx.x * per), e1 = min(E_loc, e0 + per);
  int sc = 0, st = 0;
  for (int e = e0; e < e1; ++e) {
    int c = counts[e];
    sc += c;
    st += (c + tile_n - 1) / tile_n;
  }
  int R, tiles;
  int pc = block_exclusive_scan(sc, &R);
  int pt = block_exclusive_scan(st, &tiles);
  for (int e = e0; e < e1; ++e) {
    int c = counts[e];
    offsets[e] = pc;
    if (tile_offsets) {
      tile_offsets[e] = pt;
      const int nt = (c + tile_n - 1) / tile_n;
      if (tile_info)
        for (int k = 0; k < nt; ++k) tile_info[pt + k] = make_int2(e, pc + k * tile_n);
      pt += nt;
    }
    pc += c;
  }
  if (threadIdx.x == 0) {
    offsets[E_loc] = R;
    if (tile_offsets) tile_offsets[E_loc] = tiles;
    if (meta) { meta[0] = R; meta[1] = tiles; meta[2] = 0; meta[3] = 0; }
  }
  // 3. rows >= R of permuted_src hold -1
  for (long r = R + threadIdx.x; r < S; r += blockDim.x) permuted_src[r] = -1;
}

__global__ void __launch_bounds__(kPermThreads)
permute_scatter_kernel(const int32_t* __restrict__ ids, long S, int E_loc, int off,
                       const int32_t* __restrict__ blk_base, const int32_t* __restrict__ offsets,
                       int32_t* __restrict__ permuted_src, int32_t* __restrict__ slot_to_row) {
  extern __shared__ int32_t wcnt[];   // [warps][E_loc]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5, per_warp = kPermChunk / nwarps;
  for (int i = threadIdx.x; i < nwarps * E_loc; i += blockDim.x) wcnt[i] = 0;
  const long wbase = (long)blockIdx.x * kPermChunk + (long)warp * per_warp;
  // the lane's slots' local experts, loaded once for the counts and the
  // scatter (4 per lane on 1,024 threads, 16 on 256) while the scan runs:
  // the routing is the caller's input, which the count kernel (launched
  // after everything before this call) has already read
  constexpr int kMaxPerLane = kPermChunk / kPermThreadsFew;
  const int n_lane = per_warp / kWarp;
  int le[kMaxPerLane];
#pragma unroll
  for (int u = 0; u < kMaxPerLane; ++u) {
    const long s = wbase + u * kWarp + lane;
    le[u] = (u < n_lane && s < S) ? local_expert(__ldg(ids + s), off, E_loc) : -1;
  }
  griddep_wait();   // the chunk bases and the offsets
  griddep_launch_dependents();
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kMaxPerLane; ++u)
    if (le[u] >= 0) atomicAdd(&wcnt[warp * E_loc + le[u]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E_loc; e += blockDim.x) {
    int run = offsets[e] + blk_base[(size_t)blockIdx.x * E_loc + e];
    for (int w = 0; w < nwarps; ++w) {
      int v = wcnt[w * E_loc + e];
      wcnt[w * E_loc + e] = run;
      run += v;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  int32_t* my = wcnt + warp * E_loc;
#pragma unroll
  for (int u = 0; u < kMaxPerLane; ++u) {
    if (u >= n_lane) break;   // warp-uniform
    const long s = wbase + u * kWarp + lane;
    const int e = le[u];
    unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      int row = my[e] + __popc(peers & lt);
      permuted_src[row] = (int32_t)s;
      slot_to_row[s] = row;
    } else if (s < S) {
      slot_to_row[s] = -1;
    }
    __syncwarp();
    if (e >= 0 && (peers & lt) == 0) my[e] += __popc(peers);
    __syncwarp();
  }
}

// One CTA for routings of at most kPermChunk slots: histogram, scans and
// scatter in shared memory with no global scratch and a single launch.
// Warp w owns slots [128w, 128w + 128), so the per-warp prefix keeps slot
// order exactly as the three-launch path does.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / kWarp;
constexpr int kSmallMaxExperts = 1024;

__global__ void __launch_bounds__(kSmallThreads)
permute_small_kernel(const int32_t* __restrict__ ids, int S, int E_loc, int off, int tile_n,
                     int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                     int32_t* __restrict__ tile_offsets, int2* __restrict__ tile_info,
                     int32_t* __restrict__ permuted_src, int32_t* __restrict__ slot_to_row,
                     int32_t* __restrict__ meta) {
  extern __shared__ int32_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kPerWarp = kPermChunk / kSmallWarps;   // 128
  // only the warps that own slots keep counts (8 of 32 at 1,024 slots), and
  // the launch sizes shared memory for them alone
  const int nw = (S + kPerWarp - 1) / kPerWarp;
  int32_t* wcnt = sm;                  // [nw][E_loc]
  int32_t* cnt = sm + nw * E_loc;      // [E_loc]
  int32_t* offs = cnt + E_loc;         // [E_loc]
  // the lane's slots' local experts, loaded once (all four loads in flight
  // while the counts are cleared) for both the histogram and the scatter
  constexpr int kPerLane = kPerWarp / kWarp;   // 4
  int le[kPerLane];
#pragma unroll
  for (int u = 0; u < kPerLane; ++u) {
    const int s = warp * kPerWarp + u * kWarp + lane;
    le[u] = s < S ? local_expert(__ldg(ids + s), off, E_loc) : -1;
  }
  for (int i = threadIdx.x; i < nw * E_loc; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kPerLane; ++u)
    if (le[u] >= 0) atomicAdd(&wcnt[warp * E_loc + le[u]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E_loc; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < nw; ++w) {
      const int v = wcnt[w * E_loc + e];
      wcnt[w * E_loc + e] = run;
      run += v;
    }
    cnt[e] = run;
    counts[e] = run;
  }
  __syncthreads();
  const int per = (E_loc + blockDim.x - 1) / blockDim.x;
  const int e0 = min(E_loc, (int)threadIdx.x * per), e1 = min(E_loc, e0 + per);
  int sc = 0, st = 0;
  for (int e = e0; e < e1; ++e) {
    sc += cnt[e];
    st += (cnt[e] + tile_n - 1) / tile_n;
  }
  // one scan of both prefixes: slots in the low 16 bits, tiles in the high
  // (at most kPermChunk slots and kPermChunk + kSmallMaxExperts tiles)
  int both;
  const int pb = block_exclusive_scan(sc | (st << 16), &both);
  const int R = both & 0xFFFF, tiles = both >> 16;
  int pc = pb & 0xFFFF, pt = pb >> 16;
  for (int e = e0; e < e1; ++e) {
    offs[e] = pc;
    offsets[e] = pc;
    if (tile_offsets) {
      tile_offsets[e] = pt;
      const int nt = (cnt[e] + tile_n - 1) / tile_n;
      if (tile_info)
        for (int k = 0; k < nt; ++k) tile_info[pt + k] = make_int2(e, pc + k * tile_n);
      pt += nt;
    }
    pc += cnt[e];
  }
  if (threadIdx.x == 0) {
    offsets[E_loc] = R;
    if (tile_offsets) tile_offsets[E_loc] = tiles;
    if (meta) { meta[0] = R; meta[1] = tiles; meta[2] = 0; meta[3] = 0; }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  int32_t* my = wcnt + warp * E_loc;
#pragma unroll
  for (int u = 0; u < kPerLane; ++u) {
    const int s = warp * kPerWarp + u * kWarp + lane;
    const int e = le[u];
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int row = offs[e] + my[e] + __popc(peers & lt);
      permuted_src[row] = s;
      slot_to_row[s] = row;
    } else if (s < S) {
      slot_to_row[s] = -1;
    }
    __syncwarp();
    if (e >= 0 && (peers & lt) == 0) my[e] += __popc(peers);
    __syncwarp();
  }
  for (int r = R + threadIdx.x; r < S; r += blockDim.x) permuted_src[r] = -1;
}

// A second GEMM tile table over the same expert-ordered rows, for a GEMM
// whose token tiles are tile_n rows (offsets from the permute): one block,
// each thread a contiguous run of experts, an exclusive scan of their tile
// counts, then tile_info[t] = (expert, first row).
__global__ void __launch_bounds__(1024)
tile_table_kernel(const int32_t* __restrict__ offsets, int E_loc, int tile_n, int32_t* __restrict__ tile_offsets,
                  int2* __restrict__ tile_info) {
  const int per = (E_loc + blockDim.x - 1) / blockDim.x;
  const int e0 = min(E_loc, (int)threadIdx.x * per), e1 = min(E_loc, e0 + per);
  int st = 0;
  for (int e = e0; e < e1; ++e) st += (__ldg(offsets + e + 1) - __ldg(offsets + e) + tile_n - 1) / tile_n;
  int tiles;
  int pt = block_exclusive_scan(st, &tiles);
  for (int e = e0; e < e1; ++e) {
    const int r0 = __ldg(offsets + e);
    const int nt = (__ldg(offsets + e + 1) - r0 + tile_n - 1) / tile_n;
    tile_offsets[e] = pt;
    for (int k = 0; k < nt; ++k) tile_info[pt + k] = make_int2(e, r0 + k * tile_n);
    pt += nt;
  }
  if (threadIdx.x == 0) tile_offsets[E_loc] = tiles;
}

cudaError_t launch_tile_table(const int32_t* offsets, int E_loc, int tile_n, int32_t* tile_offsets, int2* tile_info,
                              cudaStream_t st) {
  tile_table_kernel<<<1, 1024, 0, st>>>(offsets, E_loc, tile_n, tile_offsets, tile_info);
  return cudaGetLastError();
}

static int g_scatter_smem_set[64];
static int g_small_smem_set[64];

cudaError_t launch_permute(const int32_t* ids, int T, int K, int E_loc, int off, int tile_n,
                           int32_t* counts, int32_t* offsets, int32_t* tile_offsets,
                           int2* tile_info, int32_t* permuted_src, int32_t* slot_to_row,
                           int32_t* meta, int32_t* blk_counts, cudaStream_t st) {
  long S = (long)T * K;
  int nblk = (int)((S + kPermChunk - 1) / kPermChunk);
  size_t hist_smem = sizeof(int32_t) * (size_t)E_loc;
  const int sthreads = sizeof(int32_t) * (size_t)(kPermThreads / kWarp) * E_loc <= kPermMaxSmem ? kPermThreads
                                                                                                : kPermThreadsFew;
  size_t wcnt_smem = sizeof(int32_t) * (size_t)(sthreads / kWarp) * E_loc;
  int dev = 0;
  cudaGetDevice(&dev);
  if (nblk == 1 && E_loc <= kSmallMaxExperts) {
    // per-warp counts of the warps that own slots, counts and offsets; a
    // small request keeps the SM's shared-memory split as it is
    const long nw = (S + kPermChunk / kSmallWarps - 1) / (kPermChunk / kSmallWarps);
    const size_t smem = sizeof(int32_t) * (size_t)(nw + 2) * E_loc;
    {
      std::lock_guard<std::mutex> lock(attr_mutex());
      if (dev < 0 || dev >= 64 || g_small_smem_set[dev] < (int)smem) {
        cudaError_t err = cudaFuncSetAttribute(permute_small_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < 64) g_small_smem_set[dev] = (int)smem;
      }
    }
    permute_small_kernel<<<1, kSmallThreads, smem, st>>>(ids, (int)S, E_loc, off, tile_n, counts,
                                                         offsets, tile_offsets, tile_info,
                                                         permuted_src, slot_to_row, meta);
    return cudaGetLastError();
  }
  {
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (dev >= 0 && dev < 64 && g_scatter_smem_set[dev] < (int)wcnt_smem) {
      cudaError_t err = cudaFuncSetAttribute(permute_scatter_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)wcnt_smem);
      if (err != cudaSuccess) return err;
      g_scatter_smem_set[dev] = (int)wcnt_smem;
    }
  }
  permute_count_kernel<<<nblk, kPermThreads, hist_smem, st>>>(ids, S, E_loc, off, blk_counts);
  cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess)
    err = launch_pdl(permute_scan_kernel, dim3(1), dim3(1024), 0, st, blk_counts, nblk, E_loc, S, tile_n, counts,
                     offsets, tile_offsets, tile_info, permuted_src, meta);
  if (err == cudaSuccess)
    err = launch_pdl(permute_scatter_kernel, dim3(nblk), dim3(sthreads), wcnt_smem, st, (const int32_t*)ids, S, E_loc,
                     off, (const int32_t*)blk_counts, (const int32_t*)offsets, permuted_src, slot_to_row);
  return err;
}

int permute_launches(int T, int K, int E_loc) {
  const long S = (long)T * K;
  return (S <= kPermChunk && E_loc <= kSmallMaxExperts) ? 1 : 3;
}

size_t permute_scratch_bytes(int T, int K, int E_loc) {
  long S = (long)T * K;
  long nblk = (S + kPermChunk - 1) / kPermChunk;
  return sizeof(int32_t) * (size_t)(nblk > 0 ? nblk : 1) * (size_t)(E_loc > 0 ? E_loc : 1);
}

}  // namespace situ
