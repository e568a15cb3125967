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
#include <cuda_fp8.h>

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

// Copy the 16-byte vectors [begin, end) from src to dst; thread x takes
// begin + x, begin + x + kCopyThreads, ... with kUnroll loads in flight.
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

// Quantizing write into e4m3 pools: one warp per (token, head) row; lane l
// owns D/32 consecutive dims.  scale = max|row| / 448 (1 for a zero row),
// code = e4m3(x / scale) rounded to nearest even (both divisions correctly
// rounded single precision).  grid = (T, 2, ceil(H / 8)): token, K (0) or V
// (1), group of eight heads; every warp has one row, so a token's rows are
// read at once instead of one after another.
template <int D>
__global__ void __launch_bounds__(kCopyThreads)
    kv_cache_write_fp8_kernel(const __half* __restrict__ k, const __half* __restrict__ v,
                              const int64_t* __restrict__ slots, int H, int bs, long long n_slots,
                              uint8_t* __restrict__ k8, uint8_t* __restrict__ v8,
                              float* __restrict__ ks, float* __restrict__ vs, int32_t* status) {
  constexpr int EPL = D / 32;
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const long long slot = slots[t];
  if (slot < 0) return;
  if (slot >= n_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) flag_status(status, PA_DEV_BAD_SLOT);
    return;
  }
  const long long blk = slot / bs, off = slot % bs;
  const __half* src_pool = blockIdx.y == 0 ? k : v;
  uint8_t* dst_pool = blockIdx.y == 0 ? k8 : v8;
  float* scl = blockIdx.y == 0 ? ks : vs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.z * (kCopyThreads / 32) + warp;
  if (h < H) {
    const __half* src = src_pool + ((long long)t * H + h) * D + lane * EPL;
    float x[EPL];
#pragma unroll
    for (int e = 0; e < EPL; e += 2) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(src + e));
      x[e] = f.x;
      x[e + 1] = f.y;
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(x[e], sc), __NV_SATFINITE,
                                                         __NV_E4M3);
      packed |= (uint32_t)c << (8 * e);
    }
    uint8_t* dst = dst_pool + (slot * H + h) * D + lane * EPL;
    if constexpr (EPL == 4) {
      *reinterpret_cast<uint32_t*>(dst) = packed;
    } else {
      *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
    }
    if (lane == 0) scl[(blk * H + h) * bs + off] = sc;
  }
}

}  // namespace

cudaError_t launch_kv_cache_write_fp8(const __half* k, const __half* v, const int64_t* slots,
                                      int T, int H, int D, int block_size, long long n_slots,
                                      uint8_t* k8, uint8_t* v8, float* k_scale, float* v_scale,
                                      int32_t* status, cudaStream_t stream) {
  dim3 grid(T, 2, (H + kCopyThreads / 32 - 1) / (kCopyThreads / 32));
  if (D == 128)
    kv_cache_write_fp8_kernel<128><<<grid, kCopyThreads, 0, stream>>>(
        k, v, slots, H, block_size, n_slots, k8, v8, k_scale, v_scale, status);
  else
    kv_cache_write_fp8_kernel<64><<<grid, kCopyThreads, 0, stream>>>(
        k, v, slots, H, block_size, n_slots, k8, v8, k_scale, v_scale, status);
  return cudaGetLastError();
}

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
