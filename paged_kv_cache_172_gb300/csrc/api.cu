// api.cu -- the extern "C" entry points of libpagedkv (declared in
// include/pagedkv.h): argument validation, the decode partition plan, TMA
// tensor-map encoding, and the launches.  No entry point allocates memory or
// synchronises.
#include <cudaTypedefs.h>
#include <math.h>

#include <string.h>

#include <mutex>

#include "pk_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

pa_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return PA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool block_size_ok(int bs) { return bs == 4 || bs == 8 || bs == 16 || bs == 32; }

// Largest pool the kernels address with 32-bit row coordinates.
bool pool_ok(int num_blocks, int block_size, int H, int D) {
  if (num_blocks <= 0 || H <= 0 || D <= 0) return false;
  const long long rows = (long long)num_blocks * block_size;
  if (rows >= (1LL << 31)) return false;
  const long long elems = rows * H * D;
  return elems / rows == (long long)H * D && elems < (1LL << 46);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

namespace pk {

void record_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

int sm_count() {
  static std::atomic<int> cached[64];  // per device; 0 = not queried yet
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const bool slot = dev >= 0 && dev < 64;
  if (slot && (n = cached[dev].load(std::memory_order_relaxed)) > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (slot) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t make_pool_map(CUtensorMap* map, const void* base, long long rows, int H, int D,
                          int box_heads, int box_tokens) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)box_heads, (cuuint32_t)box_tokens};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_map_3d(CUtensorMap* map, const void* base, const unsigned long long dims[3],
                        const unsigned long long strides[2], const unsigned box[3],
                        bool swizzle128, CUtensorMapDataType dtype) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, 3, const_cast<void*>(base), d, st, bx,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_map_5d(CUtensorMap* map, const void* base, const unsigned long long dims[5],
                        const unsigned long long strides[4], const unsigned box[5],
                        bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < 5; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i < 4) st[i] = strides[i];
  }
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, const_cast<void*>(base), d, st, bx,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace pk

extern "C" {

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID: bad pointer, size or alignment";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: no kernel for this head_dim/block_size";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA launch error";
  }
  return "unknown pa_status";
}

int pa_last_cuda_error(void) { return g_last_cuda_error; }

int pa_version(void) { return 100; }

pa_status pa_host_device_pointer(const void* host_ptr, void** device_ptr) {
  if (device_ptr == nullptr) return PA_ERR_INVALID;
  *device_ptr = nullptr;
  if (host_ptr == nullptr) return PA_ERR_INVALID;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, host_ptr) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of the query
    return PA_ERR_INVALID;
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return PA_ERR_INVALID;
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, const_cast<void*>(host_ptr), 0) != cudaSuccess || !d) {
    cudaGetLastError();
    return PA_ERR_INVALID;
  }
  *device_ptr = d;
  return PA_OK;
}

// ---------------------------------------------------------------------------
// decode
// ---------------------------------------------------------------------------
int pa_decode_partition_tokens(int B, int H, int block_size, int max_context_len) {
  if (B <= 0 || H <= 0 || !block_size_ok(block_size) || max_context_len <= 0) return block_size;
  // Aim for at least ~8192 warp work items (152 SMs x 4-warp CTAs x several
  // waves), without partitions shorter than 8 blocks or longer than 32.
  const long long pairs = (long long)B * H;
  const long long want_parts = (8192 + pairs - 1) / pairs;
  long long tokens = (max_context_len + want_parts - 1) / want_parts;
  const long long lo = 8LL * block_size, hi = 32LL * block_size;
  if (tokens < lo) tokens = lo;
  if (tokens > hi) tokens = hi;
  tokens = (tokens + block_size - 1) / block_size * block_size;
  return (int)tokens;
}

static int resolve_partition(int B, int H, int block_size, int max_context_len,
                             int partition_tokens) {
  return partition_tokens > 0
             ? partition_tokens
             : pa_decode_partition_tokens(B, H, block_size, max_context_len);
}

size_t pa_decode_workspace_size(int B, int H, int D, int block_size, int max_context_len,
                                int partition_tokens) {
  if (B <= 0 || H <= 0 || D <= 0 || !block_size_ok(block_size) || max_context_len <= 0) return 0;
  const int pt = resolve_partition(B, H, block_size, max_context_len, partition_tokens);
  if (pt <= 0) return 0;
  const long long parts = (max_context_len + pt - 1) / pt;
  if (parts <= 1) return 0;
  return (size_t)B * H * parts * (size_t)(D + 2) * sizeof(float);
}

// Optional shared-prefix description for decode_impl.
struct PrefixGroups {
  const int32_t* seq_group = nullptr;
  const int32_t* group_offsets = nullptr;
  const int32_t* group_seqs = nullptr;
  const int32_t* group_prefix_len = nullptr;
  int num_groups = 0, max_group_size = 0, max_prefix_len = 0;
};

// Optional FP8 (e4m3) pools with per-(token, head) scales [num_blocks, H, bs].
struct Fp8Pools {
  const uint8_t* k8 = nullptr;
  const uint8_t* v8 = nullptr;
  const float* k_scale = nullptr;
  const float* v_scale = nullptr;
};

// Shared body of pa_decode, pa_decode_append (k_new/v_new non-null),
// pa_decode_shared_prefix (groups non-null) and pa_decode_fp8 (fp8 non-null,
// k_cache/v_cache then unused).
static pa_status decode_impl(const pa_half* q, const pa_half* k_new, const pa_half* v_new,
                             const pa_half* k_cache, const pa_half* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens, int B,
                             int H, int D, int block_size, int num_blocks,
                             int max_blocks_per_seq, int max_context_len, int partition_tokens,
                             float scale, pa_half* out, void* workspace, size_t workspace_bytes,
                             int32_t* status, pa_stream_t stream,
                             const PrefixGroups* groups = nullptr,
                             const Fp8Pools* fp8 = nullptr) {
  if (B < 0 || H <= 0 || H > 65535 || max_blocks_per_seq <= 0 || max_context_len < 0 ||
      !isfinite(scale))
    return PA_ERR_INVALID;
  if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
  if (!block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (B == 0) return PA_OK;
  if (fp8 != nullptr) {
    if (!fp8->k8 || !fp8->v8 || !fp8->k_scale || !fp8->v_scale || k_new) return PA_ERR_INVALID;
    if (!aligned16(fp8->k8) || !aligned16(fp8->v8) || !aligned16(fp8->k_scale) ||
        !aligned16(fp8->v_scale))
      return PA_ERR_INVALID;
    if (groups != nullptr) return PA_ERR_UNSUPPORTED;
    k_cache = reinterpret_cast<const pa_half*>(fp8->k8);  // non-null placeholders below
    v_cache = reinterpret_cast<const pa_half*>(fp8->v8);
  }
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_INVALID;
  if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_INVALID;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_INVALID;
  if (!pool_ok(num_blocks, block_size, H, D)) return PA_ERR_INVALID;
  if ((long long)max_context_len > (long long)max_blocks_per_seq * block_size)
    return PA_ERR_INVALID;
  if (max_context_len == 0) max_context_len = 1;  // every row is empty: one partition
  const int pt = resolve_partition(B, H, block_size, max_context_len, partition_tokens);
  if (pt <= 0 || pt % block_size != 0 || pt > 32 * block_size) return PA_ERR_INVALID;
  const long long parts = (max_context_len + pt - 1) / pt;
  if (parts > 65535) return PA_ERR_INVALID;
  const size_t need = pa_decode_workspace_size(B, H, D, block_size, max_context_len, pt);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return PA_ERR_WORKSPACE;
  if (need > 0 && !aligned16(workspace)) return PA_ERR_INVALID;
  int prefix_parts = 0;
  if (groups != nullptr && groups->num_groups > 0) {
    if (!groups->seq_group || !groups->group_offsets || !groups->group_seqs ||
        !groups->group_prefix_len || groups->max_prefix_len < 0 ||
        groups->max_prefix_len > max_context_len || groups->num_groups > 2147483647)
      return PA_ERR_INVALID;
    if (!pk::prefix_supported(D, block_size, groups->max_group_size)) return PA_ERR_UNSUPPORTED;
    prefix_parts = groups->max_prefix_len / pt;
    if (prefix_parts > 65535) return PA_ERR_INVALID;
  }

  const long long rows = (long long)num_blocks * block_size;
  pk::DecodeMaps maps;
  memset(&maps, 0, sizeof(maps));
  // e4m3 boxes span the heads of a warp (two adjacent ones for an even head
  // count), fp16 boxes one head.
  const int hpw = pk::decode_heads_per_warp(fp8 != nullptr, H);
  const int box_tokens = pk::decode_box_tokens(fp8 != nullptr, block_size, hpw);
  cudaError_t e;
  if (fp8 == nullptr) {
    e = pk::make_pool_map(&maps.k, k_cache, rows, H, D, 1, box_tokens);
    if (e == cudaSuccess) e = pk::make_pool_map(&maps.v, v_cache, rows, H, D, 1, box_tokens);
  } else {
    const unsigned long long dims[3] = {(unsigned long long)D, (unsigned long long)H,
                                        (unsigned long long)rows};
    const unsigned long long strides[2] = {(unsigned long long)D,
                                           (unsigned long long)H * D};
    const unsigned box[3] = {(unsigned)D, (unsigned)hpw, (unsigned)box_tokens};
    e = pk::make_map_3d(&maps.k, fp8->k8, dims, strides, box, false,
                        CU_TENSOR_MAP_DATA_TYPE_UINT8);
    if (e == cudaSuccess)
      e = pk::make_map_3d(&maps.v, fp8->v8, dims, strides, box, false,
                          CU_TENSOR_MAP_DATA_TYPE_UINT8);
    const unsigned long long sdims[3] = {(unsigned long long)block_size, (unsigned long long)H,
                                         (unsigned long long)num_blocks};
    const unsigned long long sstrides[2] = {(unsigned long long)block_size * 4,
                                            (unsigned long long)H * block_size * 4};
    const unsigned sbox[3] = {(unsigned)box_tokens, (unsigned)hpw, 1};
    if (e == cudaSuccess)
      e = pk::make_map_3d(&maps.ks, fp8->k_scale, sdims, sstrides, sbox, false,
                          CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
    if (e == cudaSuccess)
      e = pk::make_map_3d(&maps.vs, fp8->v_scale, sdims, sstrides, sbox, false,
                          CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
  }
  if (e != cudaSuccess) return PA_ERR_INVALID;

  pk::DecodeArgs a;
  a.q = reinterpret_cast<const __half*>(q);
  a.k_new = reinterpret_cast<const __half*>(k_new);
  a.v_new = reinterpret_cast<const __half*>(v_new);
  a.k_cache = reinterpret_cast<__half*>(const_cast<pa_half*>(k_cache));
  a.v_cache = reinterpret_cast<__half*>(const_cast<pa_half*>(v_cache));
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = reinterpret_cast<__half*>(out);
  float* ws = reinterpret_cast<float*>(workspace);
  a.ws_o = need ? ws : nullptr;
  a.ws_ml = need ? ws + (size_t)B * H * parts * D : nullptr;
  a.status = status;
  a.B = B;
  a.H = H;
  a.D = D;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks_per_seq;
  a.max_context_len = max_context_len;
  a.part_tokens = pt;
  a.num_parts = (int)parts;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  a.seq_group = nullptr;
  a.group_prefix_len = nullptr;
  a.group_offsets = nullptr;
  a.group_seqs = nullptr;
  a.num_groups = 0;
  a.max_group_size = 0;
  a.max_prefix_parts = 0;
  a.fp8 = fp8 != nullptr;
  a.k_scale = fp8 ? fp8->k_scale : nullptr;
  a.v_scale = fp8 ? fp8->v_scale : nullptr;
  if (prefix_parts > 0) {
    a.seq_group = groups->seq_group;
    a.group_prefix_len = groups->group_prefix_len;
    a.group_offsets = groups->group_offsets;
    a.group_seqs = groups->group_seqs;
    a.num_groups = groups->num_groups;
    a.max_group_size = groups->max_group_size;
    a.max_prefix_parts = prefix_parts;
    // 64-dim halves in 128-byte swizzle for the shared-prefix ldmatrix reads
    const unsigned long long dims[3] = {(unsigned long long)D, (unsigned long long)H,
                                        (unsigned long long)rows};
    const unsigned long long strides[2] = {(unsigned long long)D * 2,
                                           (unsigned long long)H * D * 2};
    // one block's rows per box below 16 tokens (4-token blocks are copied by
    // the lanes and never use these maps)
    const unsigned box[3] = {64, 1, (unsigned)(block_size < 16 ? block_size : 16)};
    if (pk::make_map_3d(&maps.ksw, k_cache, dims, strides, box, true) != cudaSuccess ||
        pk::make_map_3d(&maps.vsw, v_cache, dims, strides, box, true) != cudaSuccess)
      return PA_ERR_INVALID;
  }
  e = pk::launch_decode(a, maps, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_decode(const pa_half* q, const pa_half* k_cache, const pa_half* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens, int B, int H, int D,
                    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len,
                    int partition_tokens, float scale, pa_half* out, void* workspace,
                    size_t workspace_bytes, int32_t* status, pa_stream_t stream) {
  return decode_impl(q, nullptr, nullptr, k_cache, v_cache, block_tables, context_lens, B, H, D,
                     block_size, num_blocks, max_blocks_per_seq, max_context_len,
                     partition_tokens, scale, out, workspace, workspace_bytes, status, stream);
}

pa_status pa_decode_shared_prefix(const pa_half* q, const pa_half* k_cache,
                                  const pa_half* v_cache, const int32_t* block_tables,
                                  const int32_t* context_lens, const int32_t* seq_group,
                                  const int32_t* group_offsets, const int32_t* group_seqs,
                                  const int32_t* group_prefix_len, int num_groups,
                                  int max_group_size, int max_prefix_len, int B, int H, int D,
                                  int block_size, int num_blocks, int max_blocks_per_seq,
                                  int max_context_len, int partition_tokens, float scale,
                                  pa_half* out, void* workspace, size_t workspace_bytes,
                                  int32_t* status, pa_stream_t stream) {
  if (num_groups < 0) return PA_ERR_INVALID;
  PrefixGroups g;
  g.seq_group = seq_group;
  g.group_offsets = group_offsets;
  g.group_seqs = group_seqs;
  g.group_prefix_len = group_prefix_len;
  g.num_groups = num_groups;
  g.max_group_size = max_group_size;
  g.max_prefix_len = max_prefix_len;
  return decode_impl(q, nullptr, nullptr, k_cache, v_cache, block_tables, context_lens, B, H, D,
                     block_size, num_blocks, max_blocks_per_seq, max_context_len,
                     partition_tokens, scale, out, workspace, workspace_bytes, status, stream,
                     &g);
}

pa_status pa_decode_fp8(const pa_half* q, const uint8_t* k_cache8, const uint8_t* v_cache8,
                        const float* k_scale, const float* v_scale, const int32_t* block_tables,
                        const int32_t* context_lens, int B, int H, int D, int block_size,
                        int num_blocks, int max_blocks_per_seq, int max_context_len,
                        int partition_tokens, float scale, pa_half* out, void* workspace,
                        size_t workspace_bytes, int32_t* status, pa_stream_t stream) {
  Fp8Pools p;
  p.k8 = k_cache8;
  p.v8 = v_cache8;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  if (B > 0 && (!k_cache8 || !v_cache8 || !k_scale || !v_scale)) return PA_ERR_INVALID;
  return decode_impl(q, nullptr, nullptr, nullptr, nullptr, block_tables, context_lens, B, H, D,
                     block_size, num_blocks, max_blocks_per_seq, max_context_len,
                     partition_tokens, scale, out, workspace, workspace_bytes, status, stream,
                     nullptr, &p);
}

pa_status pa_kv_cache_write_fp8(const pa_half* k, const pa_half* v, const int64_t* slot_mapping,
                                int T, int H, int D, int block_size, int num_blocks,
                                uint8_t* k_cache8, uint8_t* v_cache8, float* k_scale,
                                float* v_scale, int32_t* status, pa_stream_t stream) {
  if (T < 0 || H <= 0 || H > 65535 || D <= 0) return PA_ERR_INVALID;
  if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
  if (!block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (T == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache8 || !v_cache8 || !k_scale || !v_scale)
    return PA_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache8) || !aligned16(v_cache8) ||
      !aligned16(k_scale) || !aligned16(v_scale))
    return PA_ERR_INVALID;
  if (!pool_ok(num_blocks, block_size, H, D)) return PA_ERR_INVALID;
  cudaError_t e = pk::launch_kv_cache_write_fp8(
      reinterpret_cast<const __half*>(k), reinterpret_cast<const __half*>(v), slot_mapping, T, H,
      D, block_size, (long long)num_blocks * block_size, k_cache8, v_cache8, k_scale, v_scale,
      status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_decode_append(const pa_half* q, const pa_half* k_new, const pa_half* v_new,
                           pa_half* k_cache, pa_half* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, int B, int H, int D, int block_size,
                           int num_blocks, int max_blocks_per_seq, int max_context_len,
                           int partition_tokens, float scale, pa_half* out, void* workspace,
                           size_t workspace_bytes, int32_t* status, pa_stream_t stream) {
  if (B > 0 && (!k_new || !v_new)) return PA_ERR_INVALID;
  return decode_impl(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, B, H, D,
                     block_size, num_blocks, max_blocks_per_seq, max_context_len,
                     partition_tokens, scale, out, workspace, workspace_bytes, status, stream);
}

// ---------------------------------------------------------------------------
// chunked prefill
// ---------------------------------------------------------------------------
size_t pa_prefill_workspace_size(int B, int H, int Lq, int D) {
  return pk::prefill_workspace_bytes(B, H, Lq, D);
}

// Shared body of pa_prefill_chunk (q_lens null: Lq queries per sequence) and
// pa_prefill_chunk_varlen.
static pa_status prefill_impl(const pa_half* q, const pa_half* k_cache, const pa_half* v_cache,
                              const int32_t* block_tables, const int32_t* context_lens,
                              const int32_t* q_lens, int B, int H, int Lq, int D, int block_size,
                              int num_blocks, int max_blocks_per_seq, float scale, pa_half* out,
                              void* workspace, size_t workspace_bytes, int32_t* status,
                              pa_stream_t stream) {
  if (B < 0 || H <= 0 || Lq < 0 || max_blocks_per_seq <= 0 || !isfinite(scale) ||
      !(scale > 0.f))
    return PA_ERR_INVALID;
  if (!pk::prefill_supported(D, block_size)) return PA_ERR_UNSUPPORTED;
  if (B == 0 || Lq == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_INVALID;
  if (!pool_ok(num_blocks, block_size, H, D)) return PA_ERR_INVALID;
  // the prefill kernel addresses the pool by (slot, head) rows
  if ((long long)num_blocks * block_size * H >= (1LL << 31)) return PA_ERR_INVALID;
  if ((long long)Lq > (long long)max_blocks_per_seq * block_size) return PA_ERR_INVALID;
  const size_t need = pk::prefill_workspace_bytes(B, H, Lq, D);
  if (workspace != nullptr && need > 0 && workspace_bytes < need) return PA_ERR_WORKSPACE;
  if (workspace != nullptr && !aligned16(workspace)) return PA_ERR_INVALID;
  pk::PrefillArgs a;
  a.q = reinterpret_cast<const __half*>(q);
  a.ws = reinterpret_cast<float*>(workspace);
  a.ws_floats = workspace != nullptr ? workspace_bytes / sizeof(float) : 0;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.q_lens = q_lens;
  a.out = reinterpret_cast<__half*>(out);
  a.status = status;
  a.B = B;
  a.H = H;
  a.Lq = Lq;
  a.D = D;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks_per_seq;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  cudaError_t e = pk::launch_prefill(a, k_cache, v_cache, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return PA_ERR_INVALID;
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_prefill_chunk(const pa_half* q, const pa_half* k_cache, const pa_half* v_cache,
                           const int32_t* block_tables, const int32_t* context_lens, int B, int H,
                           int Lq, int D, int block_size, int num_blocks, int max_blocks_per_seq,
                           float scale, pa_half* out, void* workspace, size_t workspace_bytes,
                           int32_t* status, pa_stream_t stream) {
  return prefill_impl(q, k_cache, v_cache, block_tables, context_lens, nullptr, B, H, Lq, D,
                      block_size, num_blocks, max_blocks_per_seq, scale, out, workspace,
                      workspace_bytes, status, stream);
}

pa_status pa_prefill_chunk_varlen(const pa_half* q, const pa_half* k_cache,
                                  const pa_half* v_cache, const int32_t* block_tables,
                                  const int32_t* context_lens, const int32_t* q_lens, int B,
                                  int H, int Lq_max, int D, int block_size, int num_blocks,
                                  int max_blocks_per_seq, float scale, pa_half* out,
                                  void* workspace, size_t workspace_bytes, int32_t* status,
                                  pa_stream_t stream) {
  if (q_lens == nullptr && B > 0 && Lq_max > 0) return PA_ERR_INVALID;
  return prefill_impl(q, k_cache, v_cache, block_tables, context_lens, q_lens, B, H, Lq_max, D,
                      block_size, num_blocks, max_blocks_per_seq, scale, out, workspace,
                      workspace_bytes, status, stream);
}

// ---------------------------------------------------------------------------
// cache write / block copy
// ---------------------------------------------------------------------------
pa_status pa_kv_cache_write(const pa_half* k, const pa_half* v, const int64_t* slot_mapping, int T,
                            int H, int D, int block_size, int num_blocks, pa_half* k_cache,
                            pa_half* v_cache, int32_t* status, pa_stream_t stream) {
  if (T < 0 || H <= 0 || D <= 0) return PA_ERR_INVALID;
  if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
  if (!block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (T == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID;
  if (!pool_ok(num_blocks, block_size, H, D)) return PA_ERR_INVALID;
  cudaError_t e = pk::launch_kv_cache_write(
      reinterpret_cast<const __half*>(k), reinterpret_cast<const __half*>(v), slot_mapping, T, H,
      D, (long long)num_blocks * block_size, reinterpret_cast<__half*>(k_cache),
      reinterpret_cast<__half*>(v_cache), status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_block_copy(pa_half* k_cache, pa_half* v_cache, const int64_t* pairs, int N, int H,
                        int D, int block_size, int num_blocks, int32_t* status,
                        pa_stream_t stream) {
  if (N < 0 || H <= 0 || D <= 0) return PA_ERR_INVALID;
  if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
  if (!block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (N == 0) return PA_OK;
  if (!k_cache || !v_cache || !pairs) return PA_ERR_INVALID;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID;
  if (!pool_ok(num_blocks, block_size, H, D)) return PA_ERR_INVALID;
  const long long block_elems = (long long)block_size * H * D;
  for (int first = 0; first < N; first += 65535) {
    const int n = N - first < 65535 ? N - first : 65535;
    cudaError_t e = pk::launch_block_copy(
        reinterpret_cast<__half*>(k_cache), reinterpret_cast<__half*>(v_cache),
        pairs + 2LL * first, n, block_elems, num_blocks, status,
        reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return PA_OK;
}

}  // extern "C"
