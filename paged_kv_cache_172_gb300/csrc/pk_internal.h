// pk_internal.h -- declarations shared between the C-ABI layer and the kernel
// translation units (host side only).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "pagedkv.h"

namespace pk {

// Sets Kern's dynamic shared-memory limit on the current device the first
// time it is launched there.  The attribute belongs to the function as loaded
// on one device, so it is tracked per device; two threads that race on a
// device's first launch may both set it, which is harmless.
template <auto Kern>
cudaError_t ensure_dynamic_smem(int bytes) {
  static std::atomic<unsigned long long> done{0};  // bit d: set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Multiprocessor count of the current device (cached per device; 0 when the
// query fails).
int sm_count();

// Makes `e` the value pa_last_cuda_error() reports on this thread.
void record_cuda_error(cudaError_t e);

struct DecodeArgs {
  const __half* q;
  const __half* k_new;  // [B, H, D] token appended at position ctx-1, or null
  const __half* v_new;
  __half* k_cache;      // pools, written only when appending
  __half* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  __half* out;
  float* ws_o;    // [B, H, num_parts, D] unnormalised partition outputs
  float* ws_ml;   // [B, H, num_parts, 2] partition (max, normaliser), log2 domain
  int32_t* status;
  int B, H, D, block_size, num_blocks, max_blocks, max_context_len;
  int part_tokens, num_parts;
  float scale_log2;  // scale * log2(e)
  // Shared-prefix decode (null otherwise): group of each sequence (-1: none),
  // and per group the tokens its members share; partitions lying entirely
  // inside the shared prefix are computed once per group by the prefix kernel.
  const int32_t* seq_group;
  const int32_t* group_prefix_len;
  const int32_t* group_offsets;  // [G+1] into group_seqs
  const int32_t* group_seqs;     // member sequence indices, the first one's table is read
  int num_groups, max_group_size, max_prefix_parts;
  // FP8 (e4m3) pools: per-(token, head) fp32 scales laid out [num_blocks, H, bs].
  bool fp8;
  const float* k_scale;
  const float* v_scale;
};

// The four tensor maps of a decode launch (scale maps used by FP8 pools only).
struct DecodeMaps {
  CUtensorMap k, v, ks, vs;
  CUtensorMap ksw, vsw;  // 64-dim halves, 128-byte swizzle (grouped calls' shared prefix)
};

// Encodes the [num_blocks * block_size, H, D] view of a cache pool as a 3-D
// TMA tensor map with a box of (D, box_heads, box_tokens).
cudaError_t make_pool_map(CUtensorMap* map, const void* base, long long rows, int H, int D,
                          int box_heads, int box_tokens);

// General 3-D tiled tensor map over fp16 data: dims innermost first, byte
// strides of dims 1 and 2, box extents; swizzle128 selects the 128-byte
// shared-memory swizzle (the inner box must then be 64 fp16 = 128 bytes).
cudaError_t make_map_3d(CUtensorMap* map, const void* base, const unsigned long long dims[3],
                        const unsigned long long strides[2], const unsigned box[3],
                        bool swizzle128,
                        CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_FLOAT16);

// 5-D tiled tensor map over fp16 data (same conventions, strides of dims 1..4
// in bytes, in any order).
cudaError_t make_map_5d(CUtensorMap* map, const void* base, const unsigned long long dims[5],
                        const unsigned long long strides[4], const unsigned box[5],
                        bool swizzle128);

// Launch the partition kernel then the combine kernel on `stream`.  When
// a.seq_group is set, the partition grid also computes the groups' shared-
// prefix partitions (multi-query, from maps.ksw / maps.vsw).
cudaError_t launch_decode(const DecodeArgs& a, const DecodeMaps& maps, cudaStream_t stream);
bool decode_supported(int D, int block_size);
// Heads per warp of the decode partition kernel (2: e4m3 pools with an even
// head count, whose K/V and scale boxes then span two adjacent heads).
int decode_heads_per_warp(bool fp8, int H);
// Tokens per TMA box of the decode partition kernel's stages (the box of the
// K/V and scale maps must match it).
int decode_box_tokens(bool fp8, int block_size, int heads_per_warp);
bool prefix_supported(int D, int block_size, int max_group_size);

cudaError_t launch_kv_cache_write(const __half* k, const __half* v, const int64_t* slots, int T,
                                  int H, int D, long long n_slots, __half* kc, __half* vc,
                                  int32_t* status, cudaStream_t stream);

cudaError_t launch_kv_cache_write_fp8(const __half* k, const __half* v, const int64_t* slots,
                                      int T, int H, int D, int block_size, long long n_slots,
                                      uint8_t* k8, uint8_t* v8, float* k_scale, float* v_scale,
                                      int32_t* status, cudaStream_t stream);

cudaError_t launch_block_copy(__half* kc, __half* vc, const int64_t* pairs, int N,
                              long long block_elems, int num_blocks, int32_t* status,
                              cudaStream_t stream);

struct PrefillArgs {
  const __half* q;
  // Tail split (set by launch_prefill): CTAs [0, full_units) are whole units
  // (one per (sequence, head, 256-query pair), in that order, units gx * H * B);
  // each later unit's key tiles are split into `split` parts whose partials
  // (D + 4 floats per query row: o[D], m, l, pad) go to ws and are merged by
  // a combine kernel.
  float* ws;
  size_t ws_floats;
  int gx, full_units, split;
  const __half* k_cache;  // the pools (set by launch_prefill; read directly by
  const __half* v_cache;  // the cp.async gather of blocks under 8 tokens)
  const int32_t* block_tables;
  const int32_t* context_lens;
  // [B] new queries per sequence (<= Lq; rows past it are written as zeros),
  // or null: Lq for every sequence
  const int32_t* q_lens;
  __half* out;
  int32_t* status;
  int B, H, Lq, D, block_size, num_blocks, max_blocks;
  float scale_log2;
};
bool prefill_supported(int D, int block_size);
// Bytes of workspace the tail split needs on the current device (0: none).
size_t prefill_workspace_bytes(int B, int H, int Lq, int D);
cudaError_t launch_prefill(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                           cudaStream_t stream);

}  // namespace pk
