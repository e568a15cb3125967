/*
 * pagedkv.h -- C ABI of libpagedkv: attention over a paged KV cache on one
 * NVIDIA GB300 (sm_103a), plus the two cache-maintenance copies.
 *
 * The problem statement these calls implement comes from three pages:
 *  - blog "PagedAttention origin and evolution" (PagedAttention的起源与演进),
 *    sec. 3.2.1 (K and V pools of shape [num_blocks, block_size, num_heads,
 *    head_dim], fp16) and sec. 3.2.2 (forward pass: per request, gather K/V
 *    through block_tables[batch, max_num_blocks], cut to context_lens,
 *    Q K^T / sqrt(head_dim), softmax, weighted sum of V);
 *  - tutorial chapter "4. PagedAttention机制：vLLM的核心创新", sections
 *    "PagedAttention的核心思想" (fixed-size blocks of 16 or 32 tokens, not
 *    contiguous, mapped by a Block Table), "Block管理策略" (blocks taken and
 *    returned through a free list as the cache grows) and
 *    "PagedAttention的注意力计算" (per logical block: physical =
 *    block_table[logical], score every token, softmax, weighted V);
 *  - study notes "DataWhale组队学习笔记--llm-algo-leetcode(五)", sections
 *    "3. PagedAttention 的工作机制" (the lookup is transparent to the model)
 *    and "4. PagedAttention 带来的核心红利" (sequences sharing a prompt point
 *    at the same physical blocks; a block is copied when one of them writes).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - fp16 data (pa_half) is IEEE binary16, passed as raw 16-bit patterns.
 *  - Every pointer argument except the host-side scalars is a DEVICE pointer
 *    of the current CUDA device, row-major and contiguous.  Where a call says
 *    so, an argument may instead be the device address of mapped page-locked
 *    host memory (pa_host_device_pointer): the kernel then reads or writes
 *    it across the host link itself.  The caller owns all memory; the
 *    library allocates nothing and never synchronises.
 *  - Every call is asynchronous on `stream` (0 = the legacy default stream).
 *  - Argument errors are reported synchronously, before anything is
 *    launched: PA_ERR_INVALID for a bad pointer, size or alignment,
 *    PA_ERR_UNSUPPORTED for a head_dim / block_size pair with no kernel,
 *    PA_ERR_WORKSPACE for a workspace that is too small, PA_ERR_CUDA when a
 *    launch fails (pa_last_cuda_error() then holds the cudaError_t value).
 *  - Errors in device-resident data (a block id outside [0, num_blocks), a
 *    context length out of range, a slot outside the pool, a copy pair out
 *    of range) are detected by the kernels: the affected work is skipped or
 *    clamped, never read or written out of bounds, and the PA_DEV_* bit is
 *    OR-ed into `*status` when `status` (a device int32) is not NULL.  The
 *    caller zeroes *status before the call and reads it afterwards.
 *  - Buffers that a call reads must not be written by the same call
 *    (no aliasing between inputs and outputs).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pa_half;               /* IEEE binary16 bit pattern */
typedef struct CUstream_st *pa_stream_t; /* same type as cudaStream_t */

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID = 1,
    PA_ERR_UNSUPPORTED = 2,
    PA_ERR_WORKSPACE = 3,
    PA_ERR_CUDA = 4
} pa_status;

/* Bits OR-ed into the device status word. */
#define PA_DEV_BAD_BLOCK_ID 0x1   /* a needed block-table entry is outside [0, num_blocks) */
#define PA_DEV_BAD_CONTEXT 0x2    /* context length < 0, > max_context_len or > table capacity */
#define PA_DEV_BAD_SLOT 0x4       /* a slot >= num_blocks * block_size */
#define PA_DEV_BAD_PAIR 0x8       /* a copy pair outside [0, num_blocks) */
#define PA_DEV_TIMEOUT 0x10       /* a bounded wait inside a kernel gave up */

/* Human-readable name of a status code (static storage). */
const char *pa_status_string(pa_status s);

/* cudaError_t value behind the last PA_ERR_CUDA returned on this thread. */
int pa_last_cuda_error(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int pa_version(void);

/* Device address of page-locked host memory: memory from cudaHostAlloc /
 * cudaMallocHost, or registered with cudaHostRegister, that is mapped into
 * the current device's address space (always so with unified addressing).
 * The device address lets a kernel load and store that memory directly,
 * with no staging copy.  host_ptr may point anywhere inside the
 * allocation.  Returns PA_ERR_INVALID, with *device_ptr set to NULL, when
 * host_ptr is NULL or is not mapped page-locked memory; device_ptr must not
 * be NULL.  Synchronous, launches nothing. */
pa_status pa_host_device_pointer(const void *host_ptr, void **device_ptr);

/* ---------------------------------------------------------------------------
 * Decode attention (one query token per sequence).
 *
 * Definition (blog sec. 3.2.2, tutorial "PagedAttention的注意力计算"): for each
 * sequence b and head h, with n = context_lens[b] and key j stored in
 * physical block block_tables[b][j / block_size], token slot j % block_size,
 *     s_j   = scale * sum_d q[b,h,d] * k_cache[blk(j), j % bs, h, d]
 *     p_j   = exp(s_j - max_k s_k) / sum_k exp(s_k - max_k s_k)
 *     out[b,h,:] = sum_j p_j * v_cache[blk(j), j % bs, h, :]
 * for j in [0, n).  n == 0 gives a zero row.  Only the first
 * ceil(n / block_size) entries of a table row are read; later entries may
 * hold anything (conventionally -1).  Pool slots past a sequence's length
 * (the tail of its last block, unreferenced blocks) may hold anything, NaN
 * included, without changing the result.
 *
 * q            [B, H, D] fp16
 * k_cache      [num_blocks, block_size, H, D] fp16 (v_cache alike)
 * block_tables [B, max_blocks_per_seq] int32
 * context_lens [B] int32, each in [0, min(max_context_len,
 *              max_blocks_per_seq * block_size)]
 * out          [B, H, D] fp16, written with round-to-nearest-even from an
 *              fp32 accumulation
 * D in {64, 128}; block_size in {4, 8, 16, 32}; q, k_cache, v_cache and out
 * 16-byte aligned.  q, out, block_tables and context_lens may be mapped
 * page-locked host memory (pa_host_device_pointer); the caches and the
 * workspace are device memory.
 *
 * Long contexts are split into partitions of `partition_tokens` keys (a
 * multiple of block_size, at most 32 blocks; 0 picks one from B, H and
 * max_context_len); each partition's running max, normaliser and
 * unnormalised output go to `workspace` and a second kernel merges them by
 * log-sum-exp.  max_context_len is a host-side bound on every
 * context_lens[b] so the split plan never reads device memory.
 * workspace: device memory of at least
 * pa_decode_workspace_size(B, H, D, block_size, max_context_len,
 * partition_tokens) bytes, 16-byte aligned, owned by the caller, contents
 * need not be initialised; may be NULL when that size is 0.
 * ------------------------------------------------------------------------- */
int pa_decode_partition_tokens(int B, int H, int block_size, int max_context_len);

size_t pa_decode_workspace_size(int B, int H, int D, int block_size,
                                int max_context_len, int partition_tokens);

pa_status pa_decode(const pa_half *q, const pa_half *k_cache,
                    const pa_half *v_cache, const int32_t *block_tables,
                    const int32_t *context_lens, int B, int H, int D,
                    int block_size, int num_blocks, int max_blocks_per_seq,
                    int max_context_len, int partition_tokens, float scale,
                    pa_half *out, void *workspace, size_t workspace_bytes,
                    int32_t *status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Decode for groups of sequences that share a prefix of physical blocks.
 *
 * Sequences forked from one prompt point at the same physical blocks until
 * they diverge (study notes "4. PagedAttention 带来的核心红利": shared blocks,
 * copy-on-write).  Same result as pa_decode (same arguments, workspace and
 * errors), but every partition of partition_tokens keys that lies entirely
 * inside a group's shared prefix is read from HBM once for the whole group
 * and attended by all its members' queries together; the remaining
 * partitions run per sequence, and all are merged by log-sum-exp.
 *
 * Groups (CSR): members of group g are group_seqs[group_offsets[g] ..
 * group_offsets[g+1]) (sequence indices, at most max_group_size <= 16 per
 * group); group_prefix_len[g] is the number of leading tokens whose blocks
 * all its members share; seq_group[b] is the group of sequence b or -1.  The
 * caller guarantees that members' block tables agree on the shared blocks
 * (the first member's table is read for them) and that every member's
 * context holds the prefix.  max_prefix_len bounds group_prefix_len on the
 * host.  Only whole partitions are shared: choose partition_tokens dividing
 * the shared prefix for the full benefit; partitions are shared only when
 * partition_tokens is a multiple of 16 (with other sizes every member reads
 * its own, same result).  D in {64, 128}, block_size in {4, 8, 16, 32}
 * (4-token blocks are copied by the lanes, the slower path).
 * ------------------------------------------------------------------------- */
pa_status pa_decode_shared_prefix(const pa_half *q, const pa_half *k_cache,
                                  const pa_half *v_cache,
                                  const int32_t *block_tables,
                                  const int32_t *context_lens,
                                  const int32_t *seq_group,
                                  const int32_t *group_offsets,
                                  const int32_t *group_seqs,
                                  const int32_t *group_prefix_len,
                                  int num_groups, int max_group_size,
                                  int max_prefix_len, int B, int H, int D,
                                  int block_size, int num_blocks,
                                  int max_blocks_per_seq, int max_context_len,
                                  int partition_tokens, float scale,
                                  pa_half *out, void *workspace,
                                  size_t workspace_bytes, int32_t *status,
                                  pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Groups for pa_decode_shared_prefix, derived from the block tables (host).
 *
 * Sequences share logical block i when their tables hold the same physical
 * id at position i and at every earlier position (study notes "4.
 * PagedAttention 带来的核心红利": forked sequences map their common prompt
 * to the same blocks).  A prefix tree over each sequence's full blocks
 * (floor(min(context_lens[b], max_blocks_per_seq*block_size) / block_size)
 * leading entries, stopping at the first negative id) groups the sequences:
 * where the sequences below a node part ways, at depth d blocks, they form
 * one group sharing d*block_size tokens; a node holding more than
 * max_group_size sequences first groups those of its children that hold two
 * or more (they share more) and cuts the rest into groups of at most
 * max_group_size at depth d.  No group shares fewer than min_shared_tokens
 * (pass partition_tokens: shorter prefixes hold no whole shared partition).
 * Each group has >= 2 members in increasing index order, groups in increasing
 * order of their first member; the shared prefix is the exact longest common
 * prefix of the members' full blocks.
 *
 * All pointers are HOST memory, row-major [B, max_blocks_per_seq] tables.
 * Outputs, caller-allocated: seq_group[B] (group of b or -1),
 * group_offsets[B/2 + 1], group_seqs[B], group_prefix_len[B/2] (tokens), and
 * *num_groups.  Pass them straight to pa_decode_shared_prefix after copying
 * to the device.  Errors: PA_ERR_INVALID for a null pointer, B < 0,
 * max_blocks_per_seq or block_size <= 0, min_shared_tokens < 0 or
 * max_group_size < 2 (outputs untouched except *num_groups = 0).  Host code
 * only: no CUDA call, thread-safe, O(total full blocks * log) time.
 * ------------------------------------------------------------------------- */
pa_status pa_shared_prefix_groups(const int32_t *block_tables,
                                  const int32_t *context_lens, int B,
                                  int max_blocks_per_seq, int block_size,
                                  int min_shared_tokens, int max_group_size,
                                  int32_t *seq_group, int32_t *group_offsets,
                                  int32_t *group_seqs,
                                  int32_t *group_prefix_len, int *num_groups);

/* ---------------------------------------------------------------------------
 * Decode with append: cache write of the new token fused into decode.
 *
 * Each decode step appends one token per sequence (tutorial "Block管理策略": the
 * cache grows into the sequence's mapped blocks) and attends with it.  For
 * every sequence b with n = context_lens[b] >= 1, the new token sits at
 * position n-1: its K/V rows k_new[b], v_new[b] ([B, H, D] fp16) are stored
 * to slot block_tables[b][(n-1)/bs] * bs + (n-1) % bs of k_cache/v_cache
 * (bit-exact, as pa_kv_cache_write would), and the query attends to keys
 * 0..n-1 exactly as pa_decode, the new key included.  One launch replaces
 * pa_kv_cache_write + pa_decode.  Every other argument, the workspace and
 * the errors are as for pa_decode; a block id outside [0, num_blocks) for
 * the new token's block skips its store and sets PA_DEV_BAD_BLOCK_ID.
 * k_new and v_new must not alias the caches; like q, out, block_tables
 * and context_lens they may be mapped page-locked host memory (16-byte
 * aligned).
 * ------------------------------------------------------------------------- */
pa_status pa_decode_append(const pa_half *q, const pa_half *k_new,
                           const pa_half *v_new, pa_half *k_cache,
                           pa_half *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, int B, int H, int D,
                           int block_size, int num_blocks,
                           int max_blocks_per_seq, int max_context_len,
                           int partition_tokens, float scale, pa_half *out,
                           void *workspace, size_t workspace_bytes,
                           int32_t *status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * FP8 (e4m3) KV storage: quantizing cache write and decode over it.
 *
 * The blog's sec. 2.3 lists mixed-precision KV storage; this is its reading
 * here.  Each (token, head) row of K and of V is stored as D e4m3 codes
 * (1 sign, 4 exponent bits with bias 7, 3 fraction bits, largest finite
 * value 448) plus one fp32 scale: value = code * scale, with
 * scale = max|row| / 448 (1 for an all-zero row) and code = e4m3(x / scale)
 * rounded to nearest even (both divisions correctly rounded fp32).  A row is
 * D + 4 bytes instead of 2D, so decode reads about half the bytes.
 *
 * k_cache8, v_cache8  [num_blocks, block_size, H, D] uint8 (e4m3 codes)
 * k_scale, v_scale    [num_blocks, H, block_size] float32
 * pa_kv_cache_write_fp8 takes the same tokens and slots as
 * pa_kv_cache_write (fp16 k, v [T, H, D]) and writes codes and scales;
 * H at most 65535 (as for decode), else PA_ERR_INVALID.
 * pa_decode_fp8 computes pa_decode's result on the dequantized cache
 * (fp32 accumulation, fp16 output), same arguments, workspace and errors.
 * ------------------------------------------------------------------------- */
pa_status pa_kv_cache_write_fp8(const pa_half *k, const pa_half *v,
                                const int64_t *slot_mapping, int T, int H,
                                int D, int block_size, int num_blocks,
                                uint8_t *k_cache8, uint8_t *v_cache8,
                                float *k_scale, float *v_scale,
                                int32_t *status, pa_stream_t stream);

pa_status pa_decode_fp8(const pa_half *q, const uint8_t *k_cache8,
                        const uint8_t *v_cache8, const float *k_scale,
                        const float *v_scale, const int32_t *block_tables,
                        const int32_t *context_lens, int B, int H, int D,
                        int block_size, int num_blocks, int max_blocks_per_seq,
                        int max_context_len, int partition_tokens, float scale,
                        pa_half *out, void *workspace, size_t workspace_bytes,
                        int32_t *status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Decode attention with no workspace and no allocation.
 *
 * This entry point has no counterpart on the pages; it exists for callers
 * that cannot allocate device memory for a call -- a host runtime that has
 * handed the whole device heap to its own pool, a plugin inside another
 * engine that forbids allocations outside that engine's allocator, or a
 * latency-critical loop that cannot pay for cudaMalloc's implicit device
 * synchronisation.  It computes exactly what pa_decode computes, with the
 * same arguments minus the workspace: the split-KV partition scratch lives
 * in a fixed device array inside the library (PA_DECODE_STATIC_SCRATCH_BYTES,
 * held on every GPU that loads the library until the process exits).
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Arguments are checked as pa_decode checks them, with the same codes;
 *    then a plan needing more scratch than the array holds, i.e.
 *    pa_decode_workspace_size(...) > PA_DECODE_STATIC_SCRATCH_BYTES, is
 *    refused with PA_ERR_WORKSPACE before anything is launched; a smaller
 *    partition count (larger partition_tokens) or batch fits.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make
 *    that first call before any stream capture.  A failed look-up returns
 *    PA_ERR_CUDA.  The cached address belongs to the device's current
 *    context: after cudaDeviceReset on a device, do not call this entry
 *    point on that device again in the same process.
 *  - All calls share the one array and it keeps the last call's contents;
 *    nothing in it needs to start at zero.  Calls whose kernels overlap on
 *    the GPU (different streams without ordering) race on it: serialise them.
 * ------------------------------------------------------------------------- */
#define PA_DECODE_STATIC_SCRATCH_BYTES (8u << 20)

pa_status pa_decode_static(const pa_half *q, const pa_half *k_cache,
                           const pa_half *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, int B, int H, int D,
                           int block_size, int num_blocks,
                           int max_blocks_per_seq, int max_context_len,
                           int partition_tokens, float scale, pa_half *out,
                           int32_t *status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Chunked prefill attention (Lq new query tokens per sequence).
 *
 * The Lq queries of sequence b are its last Lq positions: query i sits at
 * position n - Lq + i, n = context_lens[b] (which counts the chunk, whose
 * K/V must already be in the cache), and attends to keys
 * 0 .. n - Lq + i (causal mask aligned to the end of the context; with
 * Lq == n this is the lower-triangular mask of the blog's sec. 3.2.2, with
 * Lq == 1 it is decode).  Same per-row arithmetic as pa_decode; pool slots
 * past a sequence's length may hold anything, NaN included.
 *
 * q   [B, H, Lq, D] fp16 (the blog's [batch, heads, seq_len, head_dim])
 * out [B, H, Lq, D] fp16
 * context_lens[b] in [Lq, max_blocks_per_seq * block_size]; scale > 0.
 * D in {64, 128} and block_size in {4, 8, 16, 32}, all on the tcgen05
 * tensor-core kernel (blocks of 8 or more tokens arrive by TMA; 4-token
 * blocks are gathered with 16-byte copies, the slower path); any other
 * (D, block_size) returns PA_ERR_UNSUPPORTED.  The pool must hold fewer
 * than 2^31 (slot, head) rows (num_blocks * block_size * H; under 512 GiB
 * per pool at D = 128), else PA_ERR_INVALID.
 *
 * workspace (device, 16-byte aligned, caller-owned, may be NULL): with at
 * least pa_prefill_workspace_size(B, H, Lq, D) bytes, the work units of the
 * grid's last, partial round (one CTA per SM) are each split into key ranges
 * whose partial results are merged by log-sum-exp, so that round fills the
 * GPU; with NULL every unit runs whole (same result up to rounding).  A
 * non-NULL workspace smaller than that returns PA_ERR_WORKSPACE.  The size
 * depends on the SM count of the current device.
 * ------------------------------------------------------------------------- */
size_t pa_prefill_workspace_size(int B, int H, int Lq, int D);

pa_status pa_prefill_chunk(const pa_half *q, const pa_half *k_cache,
                           const pa_half *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, int B, int H, int Lq,
                           int D, int block_size, int num_blocks,
                           int max_blocks_per_seq, float scale, pa_half *out,
                           void *workspace, size_t workspace_bytes,
                           int32_t *status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Chunked prefill with a chunk length per sequence.
 *
 * The same computation as pa_prefill_chunk for sequence b's q_lens[b] new
 * queries, which sit in rows 0 .. q_lens[b]-1 of its [H, Lq_max, D] slice
 * of q: query i is at position n - q_lens[b] + i (n = context_lens[b]) and
 * attends to keys 0 .. n - q_lens[b] + i (the blog's sec. 3.2.2 forward pass
 * takes each request's queries on their own).  Rows q_lens[b] .. Lq_max-1
 * of out are written as zeros.  q_lens is [B] int32 on the device (or in
 * mapped page-locked host memory), each in [0, Lq_max] and at most
 * context_lens[b]; a sequence breaking that is flagged PA_DEV_BAD_CONTEXT in
 * *status and its rows are zeros.  q_lens NULL (with B, Lq_max > 0) returns
 * PA_ERR_INVALID.  Every other argument, the workspace rule (with
 * pa_prefill_workspace_size(B, H, Lq_max, D)) and the error behaviour are
 * those of pa_prefill_chunk with Lq = Lq_max.
 * ------------------------------------------------------------------------- */
pa_status pa_prefill_chunk_varlen(const pa_half *q, const pa_half *k_cache,
                                  const pa_half *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, const int32_t *q_lens,
                                  int B, int H, int Lq_max, int D, int block_size,
                                  int num_blocks, int max_blocks_per_seq, float scale,
                                  pa_half *out, void *workspace, size_t workspace_bytes,
                                  int32_t *status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Cache write (scatter new tokens' K/V into their slots).
 *
 * With the caches viewed as [num_blocks * block_size, H, D], for each token
 * t with slot_mapping[t] >= 0:  k_cache[slot] = k[t], v_cache[slot] = v[t]
 * (bit-exact copies).  slot = physical_block * block_size + offset, the
 * address a sequence's block table gives its position (tutorial, "Block管理
 * 策略": the cache grows into newly mapped blocks).  Negative slots are
 * padding and are skipped.  Two tokens with the same slot: undefined which
 * one lands.
 *
 * k, v          [T, H, D] fp16
 * slot_mapping  [T] int64
 * k_cache, v_cache as for pa_decode, written in place.
 * ------------------------------------------------------------------------- */
pa_status pa_kv_cache_write(const pa_half *k, const pa_half *v,
                            const int64_t *slot_mapping, int T, int H, int D,
                            int block_size, int num_blocks, pa_half *k_cache,
                            pa_half *v_cache, int32_t *status,
                            pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Block copy (copy-on-write of shared blocks; study notes sec. 4).
 *
 * For each pair i: physical block pairs[i][1] of k_cache and of v_cache
 * becomes a bit-exact copy of block pairs[i][0] (all block_size * H * D
 * values).  Destinations must be distinct and no destination may be the
 * source of another pair in the same call (otherwise the result is
 * undefined); src == dst is a no-op.
 *
 * pairs [N, 2] int64 (src, dst).
 * ------------------------------------------------------------------------- */
pa_status pa_block_copy(pa_half *k_cache, pa_half *v_cache,
                        const int64_t *pairs, int N, int H, int D,
                        int block_size, int num_blocks, int32_t *status,
                        pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
