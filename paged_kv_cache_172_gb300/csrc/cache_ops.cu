// cache_ops.cu -- the two copy kernels of the paged cache (sm_103a).
//
// kv_cache_write: scatter each new token's K/V row (H * D fp16) into its
//   slot of the [num_blocks * block_size, H, D] pool view; the slot is the
//   physical block the sequence's block table maps its position to, times
//   block_size, plus the offset (tutorial "4. PagedAttention机制：vLLM的核心创新",
//   section "Block管理策略": the cache grows into newly mapped blocks).
// block_copy: copy whole physical blocks (copy-on-write of a block shared by
//   several sequences; study notes "DataWhale组队学习笔记--llm-algo-leetcode(五)",
//   "4. PagedAttention 带来的核心红利").
//
// Both are pure HBM copies: 16-byte vector loads and stores, several loads
// in flight per thread before the stores, grid sized so every SM has many
// CTAs.  Bounds are checked against the pool on the device; bad entries set
// a status bit and are skipped.
#include "pk_common.cuh"
#include "pk_internal.h"

namespace pk {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Copy `nvec` 16-byte vectors from src to dst, this CTA's share being the
// vectors [chunk0, chunk0 + chunk) of the row.
__device__ __forceinline__ void copy_vectors(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                             long long begin, long long end) {
  for (long long base = begin + threadIdx.x; base < end; base += (long long)kCopyThreads * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = base + (long long)u * kCopyThreads;
      if (i < end) v[u] = ld_stream(src + i);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = base + (long long)u * kCopyThreads;
      if (i < end) st_stream(dst + i, v[u]);
    }
  }
}

// grid = (T, 2): blockIdx.y selects K (0) or V (1).
__global__ void __launch_bounds__(kCopyThreads)
    kv_cache_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                          const int64_t* __restrict__ slots, long long row_vecs, long long n_slots,
                          uint4* __restrict__ kc, uint4* __restrict__ vc, int32_t* status) {
  pdl_launch_dependents();  // a following decode may be scheduled; it waits for this grid
  const int t = blockIdx.x;
  const long long slot = slots[t];
  if (slot < 0) return;  // padding token
  if (slot >= n_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0) flag_status(status, PA_DEV_BAD_SLOT);
    return;
  }
  const uint4* src = (blockIdx.y == 0 ? k : v) + (long long)t * row_vecs;
  uint4* dst = (blockIdx.y == 0 ? kc : vc) + slot * row_vecs;
  copy_vectors(src, dst, 0, row_vecs);
}

// grid = (chunks, N, 2): chunk c of pair n of pool K (0) or V (1).
__global__ void __launch_bounds__(kCopyThreads)
    block_copy_kernel(uint4* __restrict__ kc, uint4* __restrict__ vc,
                      const int64_t* __restrict__ pairs, long long block_vecs, long long chunk_vecs,
                      int num_blocks, int32_t* status) {
  const int n = blockIdx.y;
  const long long src = pairs[2 * n], dst = pairs[2 * n + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0)
      flag_status(status, PA_DEV_BAD_PAIR);
    return;
  }
  if (src == dst) return;
  uint4* pool = blockIdx.z == 0 ? kc : vc;
  const long long begin = (long long)blockIdx.x * chunk_vecs;
  const long long end = min(begin + chunk_vecs, block_vecs);
  copy_vectors(pool + src * block_vecs, pool + dst * block_vecs, begin, end);
}

}  // namespace

cudaError_t launch_kv_cache_write(const __half* k, const __half* v, const int64_t* slots, int T,
                                  int H, int D, long long n_slots, __half* kc, __half* vc,
                                  int32_t* status, cudaStream_t stream) {
  const long long row_vecs = (long long)H * D / 8;
  dim3 grid(T, 2);
  kv_cache_write_kernel<<<grid, kCopyThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), slots, row_vecs,
      n_slots, reinterpret_cast<uint4*>(kc), reinterpret_cast<uint4*>(vc), status);
  return cudaGetLastError();
}

cudaError_t launch_block_copy(__half* kc, __half* vc, const int64_t* pairs, int N,
                              long long block_elems, int num_blocks, int32_t* status,
                              cudaStream_t stream) {
  const long long block_vecs = block_elems / 8;
  const long long chunk_vecs = (long long)kCopyThreads * kUnroll * 4;  // 64 KB per CTA
  const long long chunks = (block_vecs + chunk_vecs - 1) / chunk_vecs;
  dim3 grid((unsigned)chunks, N, 2);
  block_copy_kernel<<<grid, kCopyThreads, 0, stream>>>(
      reinterpret_cast<uint4*>(kc), reinterpret_cast<uint4*>(vc), pairs, block_vecs, chunk_vecs,
      num_blocks, status);
  return cudaGetLastError();
}

}  // namespace pk
