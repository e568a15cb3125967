// decode.cu -- paged decode attention for sm_103a.
//
// Definition (blog "PagedAttention origin and evolution", sec. 3.2.2, and the
// tutorial "4. PagedAttention机制：vLLM的核心创新", section
// "PagedAttention的注意力计算"): one query per (sequence, head) attends to all
// context_lens[b] keys, each key found through block_tables[b][j / bs].
//
// Design (GB300):
//  * Work unit = one warp = one (sequence b, head h, partition of
//    part_tokens keys).  A CTA holds WARPS warps for WARPS consecutive heads
//    of the same (b, partition), so all its warps stream the same number of
//    blocks.  Grid = (B, ceil(H / WARPS), num_parts) with b fastest: the
//    sequences that share prompt blocks are scheduled together, so shared
//    blocks are read from HBM once and served from L2 to the sharers.
//  * Each warp runs its own NSTAGE-deep TMA pipeline: lane 0 issues one 3-D
//    tensor load per stage for K and one for V (box = min(block_size, 16)
//    token rows of one head, H*D*2 bytes apart in the pool; a 32-token block
//    is two stages), completing on a per-stage mbarrier.  The block-table entries of the
//    partition are loaded once, one per lane, so address generation never
//    waits on a dependent global load.
//  * Scores: lane l owns D/32 consecutive dims; every lane forms partial dot
//    products for all block_size tokens of the block, then a transposing
//    butterfly (offsets 16, 8, ...) halves the number of live values per step
//    so that after log2(block_size) shuffle rounds each lane holds the full
//    score of token lane / (32 / block_size): block_size + ... + 1 shuffles
//    instead of 5 per token.
//  * Online softmax in the log2 domain (scale * log2(e) folded into one
//    multiply), fp32 accumulation of P V with the lane's D/32 dims.
//  * e4m3 pools (pa_decode_fp8) with an even head count: a warp takes two
//    adjacent heads (boxes of 2 D contiguous bytes per token), eight lanes
//    per (token, head) row, and the two warps of a pair split the
//    partition's stages and merge their softmax states at the end.
//  * Optional append (pa_decode_append): the warp whose partition holds
//    position ctx-1 stores the new token's K/V (its head's slice) to the
//    cache slot the block table gives and scores it from registers-to-smem,
//    so the cache write and the attention are one launch.  No other warp
//    reads that slot.
//  * A sequence that fits in one partition writes fp16 output directly;
//    otherwise each partition writes (max, normaliser, unnormalised output)
//    to the workspace and a combine kernel merges them by log-sum-exp.
#include <math.h>

#include <cuda_fp8.h>

#include "pk_common.cuh"
#include "pk_internal.h"
#include "pk_prefix.cuh"

namespace pk {

namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int EPL>
struct LaneVec;  // EPL fp16 values of one lane
template <>
struct LaneVec<4> {
  uint2 raw;
  __device__ __forceinline__ void load(const __half* p) { raw = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ void to_float(float* f) const {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  }
};
template <>
struct LaneVec<2> {
  uint32_t raw;
  __device__ __forceinline__ void load(const __half* p) { raw = *reinterpret_cast<const uint32_t*>(p); }
  __device__ __forceinline__ void to_float(float* f) const {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw));
    f[0] = a.x; f[1] = a.y;
  }
};

// Sum of a.lo*b.lo + a.hi*b.hi + c for fp16 pairs a, b: products exact in fp32,
// each addition rounded once, in this order (the same value as converting a
// and b to float and chaining fmaf).
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t.reg .f32 t;\n\t"
      "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
      "fma.rn.f32.f16 t, a0, b0, %3;\n\tfma.rn.f32.f16 %0, a1, b1, t;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

// N consecutive 32-bit words from p (4 N bytes, aligned to min(16, 4 N)).
template <int N>
__device__ __forceinline__ void load_words(uint32_t* w, const void* p) {
  if constexpr (N == 1) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  } else if constexpr (N == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y;
  } else {
    static_assert(N % 4 == 0, "whole 16-byte chunks");
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      const uint4 v = reinterpret_cast<const uint4*>(p)[i];
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  }
}

// Four e4m3 codes (one word) as two fp16 pairs; exact.
__device__ __forceinline__ void e4m3x4_to_half2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const __half2_raw l = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  lo = *reinterpret_cast<const uint32_t*>(&l);
  hi = *reinterpret_cast<const uint32_t*>(&h);
}

// Lane partial of q . k for EPL e4m3 codes of k (EPL / 4 words w; fp16 query
// pairs qh); from 16 dims on, two interleaved sums shorten the dependent chain.
template <int EPL>
__device__ __forceinline__ float dot_e4m3(const uint32_t* qh, const uint32_t* w) {
  static_assert(EPL % 4 == 0, "whole words of codes");
  constexpr int NW = EPL / 4, NACC = EPL >= 16 ? 2 : 1;
  float t[NACC];
#pragma unroll
  for (int k = 0; k < NACC; ++k) t[k] = 0.f;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    uint32_t lo, hi;
    e4m3x4_to_half2x2(w[i], lo, hi);
    t[i % NACC] = fma2_f16_f32(qh[2 * i], lo, t[i % NACC]);
    t[i % NACC] = fma2_f16_f32(qh[2 * i + 1], hi, t[i % NACC]);
  }
  if constexpr (NACC == 2) return t[0] + t[1];
  return t[0];
}

// o[e] += w * v[e] for EPL e4m3 codes v (EPL / 4 words wd; exact in fp16),
// products exact in fp32, one rounding per addition.
template <int EPL>
__device__ __forceinline__ void axpy_e4m3(float* o, __half w, const uint32_t* wd) {
  static_assert(EPL % 4 == 0, "whole words of codes");
  constexpr int NW = EPL / 4;
  const uint16_t wb = __half_as_ushort(w);
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    uint32_t lo, hi;
    e4m3x4_to_half2x2(wd[i], lo, hi);
    asm("{\n\t.reg .f16 w, b0, b1, b2, b3;\n\tmov.b16 w, %4;\n\t"
        "mov.b32 {b0, b1}, %5;\n\tmov.b32 {b2, b3}, %6;\n\t"
        "fma.rn.f32.f16 %0, w, b0, %0;\n\tfma.rn.f32.f16 %1, w, b1, %1;\n\t"
        "fma.rn.f32.f16 %2, w, b2, %2;\n\tfma.rn.f32.f16 %3, w, b3, %3;\n\t}"
        : "+f"(o[4 * i]), "+f"(o[4 * i + 1]), "+f"(o[4 * i + 2]), "+f"(o[4 * i + 3])
        : "h"(wb), "r"(lo), "r"(hi));
  }
}

// Warp maximum of a float (NaN-free inputs; -inf allowed), one instruction.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

template <int EPL>
__device__ __forceinline__ void store_half_row(__half* dst, const float* v) {
  uint32_t w[EPL / 2];
#pragma unroll
  for (int i = 0; i < EPL / 2; ++i) {
    __half2 h2 = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h2);
  }
  if constexpr (EPL % 8 == 0) {
#pragma unroll
    for (int i = 0; i < EPL / 8; ++i)
      reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  } else if constexpr (EPL == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = w[0];
  }
}

// Context length of sequence b clamped to what the launch can address.
__device__ __forceinline__ int checked_ctx(const DecodeArgs& a, int b, bool report) {
  int ctx = a.context_lens[b];
  const int cap = min(a.max_context_len, a.max_blocks * a.block_size);
  if (ctx < 0 || ctx > cap) {
    if (report) flag_status(a.status, PA_DEV_BAD_CONTEXT);
    ctx = ctx < 0 ? 0 : cap;
  }
  return ctx;
}

#ifndef PK_DECODE_FP8_RL
#define PK_DECODE_FP8_RL 8
#endif
#ifndef PK_DECODE_FP8_TB
#define PK_DECODE_FP8_TB 32  // e4m3 rows per stage at block size >= 16
#endif
#ifndef PK_DECODE_FP8_HPW
#define PK_DECODE_FP8_HPW 2  // heads per e4m3 warp when the head count is even
#endif

// Tokens per pipeline stage: 16 fp16 rows, or PK_DECODE_FP8_TB / hpw e4m3
// tokens (hpw heads each) at block size >= 16; below 16, one block.
constexpr int stage_tokens_for(bool fp8, int bs, int hpw) {
  return fp8 ? (bs >= 16 ? PK_DECODE_FP8_TB / hpw : bs) : (bs < 16 ? bs : 16);
}
// Tokens per TMA box of a stage (the maps' box): a stage's tokens, at most
// one block.
constexpr int box_tokens_for(bool fp8, int bs, int hpw) {
  return stage_tokens_for(fp8, bs, hpw) < bs ? stage_tokens_for(fp8, bs, hpw) : bs;
}

// Copy each stage to registers before its arithmetic and refill it at once
// (bit 0: fp16 pools, bit 1: e4m3 pools).
#ifndef PK_DECODE_STAGE_REGS
#define PK_DECODE_STAGE_REGS 0
#endif

// HPW: heads per warp.  An e4m3 row of one (token, head) is D bytes (128 at
// D = 128), and HBM serves such 128-byte pieces about 7 % slower than 256-byte
// ones, so with an even head count each e4m3 warp takes two adjacent heads:
// its boxes read both heads' rows of a token, 2 D contiguous bytes.  The two
// warps of a pair then split the partition's stages (even and odd ones) and
// merge their results at the end, so a warp still streams one head's worth
// of a partition and the grid keeps its number of work units.
template <int D, int BS, int WARPS, int NSTAGE, bool FP8, int HPW = 1>
struct PartitionCfg {
  static_assert(HPW == 1 || (FP8 && HPW == 2), "two heads per warp for e4m3 pools only");
  // Tokens per pipeline stage: 16 fp16 tokens (4 KB per head at D = 128), or
  // 32 / HPW e4m3 tokens at block size >= 16 -- the same bytes per stage, and
  // every lane then holds a distinct row's score, so the per-stage reductions
  // cost half as much per row.  A row is one (token, head), HPW rows per token.
  // A TMA box never spans blocks: TBX tokens, BPS per stage.
  static constexpr int TB = stage_tokens_for(FP8, BS, HPW);
  static constexpr int ROWS = TB * HPW;               // rows per stage
  // Lanes covering one row's D dims: 32 for fp16; 8 for e4m3 (four rows per
  // warp instruction, 16 codes per lane: one 16-byte shared-memory read per
  // row and lane, eight lanes per 128-byte row, so no bank conflicts; three
  // butterfly rounds per stage instead of four at 16 lanes), at least 32 / ROWS
  // so that a stage still fills one warp instruction.
  static constexpr int RL =
      !FP8 ? 32 : (PK_DECODE_FP8_RL * ROWS >= 32 ? PK_DECODE_FP8_RL : 32 / ROWS);
  static constexpr int NT = 32 / RL;                  // rows per warp instruction
  // Row it * NT + lane / RL of a stage is head (lane / RL) % HPW of its token:
  // a lane stays on one head.
  static_assert(NT % HPW == 0, "each lane keeps one head");
  static constexpr int EPL = D / RL;                  // dims per lane
  static constexpr int TBX = TB < BS ? TB : BS;       // tokens per TMA box
  static_assert(TBX == box_tokens_for(FP8, BS, HPW), "the maps' box is one stage box");
  static constexpr int BPS = TB / TBX;                // boxes per tensor per stage
  static constexpr int SUB = BS / TBX;                // boxes per physical block
  static constexpr int ELEM = FP8 ? 1 : 2;            // bytes per stored K/V element
  static constexpr int TILE_BYTES = ROWS * D * ELEM;  // the rows of one stage
  static constexpr int SCALE_BYTES = FP8 ? ROWS * 4 : 0;  // per-row scales of one stage
  // Scales of one tensor and stage: box k ([HPW heads][TBX tokens]) at byte
  // k * 128 (a TMA destination in shared memory must be 128-byte aligned).
  static constexpr int SCALE_SLOT = FP8 ? BPS * 128 : 0;
  static_assert(!FP8 || TBX * HPW * 4 <= 128, "one box of scales per 128-byte slot");
  // Float index of row r's scale inside a scale slot.
  static __device__ __forceinline__ int scale_index(int r) {
    const int t = r / HPW;
    return (t / TBX) * 32 + (r % HPW) * TBX + t % TBX;
  }
  // stage = [K rows][V rows][K scales][V scales]; TX_BYTES actually land
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES + 2 * SCALE_SLOT;
  static constexpr int TX_BYTES = 2 * TILE_BYTES + 2 * SCALE_BYTES;
  static_assert(TILE_BYTES % 128 == 0 && STAGE_BYTES % 128 == 0, "TMA destinations 128-B aligned");
  static constexpr int LANES_PER_ROW = 32 / ROWS > 1 ? 32 / ROWS : 1;  // lanes sharing a score
  static constexpr int SMEM_BYTES = WARPS * NSTAGE * STAGE_BYTES + WARPS * NSTAGE * 8;
};

// GRP: grouped call (a.seq_group set) that also runs shared-prefix partitions;
// a separate instantiation so plain decode keeps its small register budget.
// HPW: heads per warp (two: e4m3 pools with an even head count).
template <int D, int BS, int WARPS, int NSTAGE, bool FP8, bool GRP = false, int HPW = 1>
__global__ void __launch_bounds__(WARPS * 32)
    partition_kernel(const __grid_constant__ DecodeMaps maps, const DecodeArgs a) {
  using Cfg = PartitionCfg<D, BS, WARPS, NSTAGE, FP8, HPW>;
  constexpr int EPL = Cfg::EPL;
  constexpr int TB = Cfg::TB;
  constexpr int SUB = Cfg::SUB;
  constexpr int LPR = Cfg::LANES_PER_ROW;
  constexpr int RL = Cfg::RL, NT = Cfg::NT;
  constexpr int ITER = Cfg::ROWS / NT;  // warp instructions per stage (one row per RL lanes each)
  static_assert(ITER >= 1 && RL % ITER == 0, "stage rows vs row lanes");
  constexpr int KWORDS = EPL * Cfg::ELEM / 4;  // 32-bit words of a lane's slice of one row
  constexpr bool kStageRegs = ((FP8 ? 2 : 1) & PK_DECODE_STAGE_REGS) != 0;
  static_assert(BS >= 1 && BS <= 32 && (32 % BS) == 0, "block_size must divide 32");

  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  static_assert(WARPS % HPW == 0, "whole warp pairs");
  const int th = warp % HPW;                         // the pair's stages this warp takes
  const int h0 = blockIdx.y * WARPS + warp - th;     // the warp's first head (WARPS per CTA)
  const int h = h0 + (lane / RL) % HPW;              // the head of this lane's rows
  const int part = blockIdx.z;
  pdl_wait();             // inputs may come from the previous kernel on the stream
  if (h0 >= a.H) return;  // idle warp of a ragged head group (no CTA-wide sync below)

  uint8_t* wbase = smem + warp * NSTAGE * Cfg::STAGE_BYTES;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + WARPS * NSTAGE * Cfg::STAGE_BYTES) + warp * NSTAGE;

  const int tok0 = part * a.part_tokens;
  const int lb0 = tok0 / BS;
  // The partition's block-table entries (one per lane, at most 32) are read
  // together with the context length, before it is known, so that the first
  // copies wait for one round trip to memory instead of two; entries past the
  // context are never looked at.
  int tab = 0;
  if (lane < min(a.part_tokens / BS, a.max_blocks - lb0))
    tab = a.block_tables[(size_t)b * a.max_blocks + lb0 + lane];
  const int ctx = checked_ctx(a, b, lane == 0 && part == 0);
  const size_t row_bh = (size_t)b * a.H + h;
  // Partitions inside a group's shared prefix (partitions of whole 16-token
  // stages; with other partition sizes every member computes its own).
  if (a.seq_group != nullptr && a.part_tokens % pfx::kTB == 0) {
    const int g = a.seq_group[b];
    if (g >= 0 && g < a.num_groups) {
      const int shared = min(a.group_prefix_len[g], ctx) / a.part_tokens * a.part_tokens;
      if (tok0 + a.part_tokens <= shared) {
        if constexpr (GRP && !FP8) {
          // The group's first member computes this partition for every member.
          if (a.group_seqs[a.group_offsets[g]] == b) {
            const uint32_t sa = smem_u32(smem);
            pfx::prefix_partition<D, BS, WARPS>(maps.ksw, maps.vsw, a, g, part,
                                                smem + ((1024u - (sa & 1023u)) & 1023u));
          }
        }
        return;
      }
    }
  }
  if (tok0 >= ctx) {
    if (part == 0 && th == 0 && lane < RL * HPW) {  // empty sequence: zero rows
      float z[EPL] = {};
      store_half_row<EPL>(a.out + row_bh * D + (lane % RL) * EPL, z);
    }
    return;
  }
  const int tok1 = min(ctx, tok0 + a.part_tokens);
  const int nblk = (tok1 - tok0 + BS - 1) / BS;  // <= 32 by construction of part_tokens
  const int nunit = (tok1 - tok0 + TB - 1) / TB; // pipeline stages (TB-token sub-blocks)
  // Stages of this warp: units th, th + HPW, ... of the partition.
  const int nmine = (nunit - th + HPW - 1) / HPW;

  // Block-table entries of this partition, one per lane.
  int phys = 0;
  if (lane < nblk) {
    phys = tab;
    if (phys < 0 || phys >= a.num_blocks) {
      flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
      phys = a.num_blocks;  // entirely outside the tensor map: TMA fills zeros
    }
  }

  // Dims [dl, dl + EPL) of this lane; lane / RL picks the row of an instruction.
  const int dl = (lane % RL) * EPL;

  if (lane == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Prologue: fill the pipeline.  Unit u is tokens [u*TB, u*TB+TB) of the
  // partition; its box k holds tokens u*TB + k*TBX + [0, TBX), inside logical
  // block lb0 + (u*TB + k*TBX) / BS, for the warp's HPW heads ([token][head]
  // rows; scales [head][token]).
  auto issue = [&](int u, int s) {  // all lanes (shuffle), lane 0 issues
    uint8_t* st = wbase + s * Cfg::STAGE_BYTES;
    if (lane == 0) mbar_arrive_expect_tx(&bars[s], Cfg::TX_BYTES);
#pragma unroll
    for (int k = 0; k < Cfg::BPS; ++k) {
      const int tt = u * TB + k * Cfg::TBX;  // first token of the box in the partition
      const int pb = __shfl_sync(kFull, phys, tt / BS);
      if (lane == 0) {
        const int row = pb * BS + tt % BS;
        constexpr int kBoxBytes = Cfg::TBX * HPW * D * Cfg::ELEM;
        tma_load_3d(st + k * kBoxBytes, &maps.k, 0, h0, row, &bars[s]);
        tma_load_3d(st + Cfg::TILE_BYTES + k * kBoxBytes, &maps.v, 0, h0, row, &bars[s]);
        if constexpr (FP8) {  // scales [num_blocks, H, bs]: box of HPW x TBX
          tma_load_3d(st + 2 * Cfg::TILE_BYTES + k * 128, &maps.ks, tt % BS, h0, pb, &bars[s]);
          tma_load_3d(st + 2 * Cfg::TILE_BYTES + Cfg::SCALE_SLOT + k * 128, &maps.vs, tt % BS,
                      h0, pb, &bars[s]);
        }
      }
    }
  };
  for (int i = 0; i < NSTAGE && i < nmine; ++i) issue(i * HPW + th, i);

  // Query slice of this lane (and, for e4m3 pools, its fp16 pairs), read once
  // the first stages are in flight so that its latency overlaps the K/V copies.
  float qf[FP8 ? 1 : EPL];
  uint32_t qh[FP8 ? EPL / 2 : 1];
  if constexpr (FP8) {
    load_words<EPL / 2>(qh, a.q + row_bh * D + dl);
  } else {
    LaneVec<EPL> qv;
    qv.load(a.q + row_bh * D + dl);
    qv.to_float(qf);
  }

  float m = -INFINITY, l = 0.f;
  float o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = 0.f;

  // Row whose score this lane holds after the butterfly (lane / LPR for RL =
  // 32); it is a row of the lane's own head.
  const int my_tok = ((lane % RL) / (RL / ITER)) * NT + lane / RL;
  int i = 0;
  for (; i < nmine; ++i) {
    const int u = i * HPW + th;  // unit of the partition
    const int s = i % NSTAGE;
    const uint32_t parity = (i / NSTAGE) & 1;
    const bool got = mbar_wait(&bars[s], parity);
    if (!__all_sync(kFull, got)) break;

    uint8_t* kst = wbase + s * Cfg::STAGE_BYTES;
    __half* ks = reinterpret_cast<__half*>(kst);
    __half* vs = reinterpret_cast<__half*>(kst + Cfg::TILE_BYTES);
    const float* kscl = reinterpret_cast<const float*>(kst + 2 * Cfg::TILE_BYTES);
    const float* vscl = reinterpret_cast<const float*>(kst + 2 * Cfg::TILE_BYTES + Cfg::SCALE_SLOT);
    const int valid = min(TB, tok1 - (tok0 + u * TB));  // tokens of this unit inside the partition
    const int valid_rows = valid * HPW;  // rows are [token][head]

    // Appending: the new token (position ctx-1) is scored from k_new/v_new,
    // copied over the stage row TMA brought in, and stored to its cache slot.
    if constexpr (!FP8) {
      const int t_new = ctx - 1 - (tok0 + u * TB);
      if (a.k_new != nullptr && t_new >= 0 && t_new < TB) {
        const int pb = __shfl_sync(kFull, phys, u / SUB);
        const size_t src = row_bh * D + lane * EPL;
        LaneVec<EPL> kn, vn;
        kn.load(a.k_new + src);
        vn.load(a.v_new + src);
        *reinterpret_cast<decltype(kn.raw)*>(ks + t_new * D + lane * EPL) = kn.raw;
        *reinterpret_cast<decltype(vn.raw)*>(vs + t_new * D + lane * EPL) = vn.raw;
        if (pb < a.num_blocks) {
          const size_t slot = (size_t)pb * BS + (u % SUB) * TB + t_new;
          const size_t dst = (slot * a.H + h) * D + lane * EPL;
          *reinterpret_cast<decltype(kn.raw)*>(a.k_cache + dst) = kn.raw;
          *reinterpret_cast<decltype(vn.raw)*>(a.v_cache + dst) = vn.raw;
        }
        __syncwarp();
      }
    }

    // This lane's K and V data of the stage: its dims of the rows of every
    // warp instruction (EPL fp16 values or EPL e4m3 codes each) and, for e4m3
    // pools, the scales of the row whose score it will hold.  With kStageRegs
    // they are copied to registers first and the stage is refilled at once,
    // so the copy of unit i + NSTAGE overlaps this unit's arithmetic instead
    // of waiting for it.
    uint32_t kw[ITER][KWORDS], vw[ITER][KWORDS];
    auto load_k = [&](int it) {
      const int t = it * NT + lane / RL;
      load_words<KWORDS>(kw[it], kst + (t * D + dl) * Cfg::ELEM);
    };
    auto load_v = [&](int it) {
      const int t = it * NT + lane / RL;
      load_words<KWORDS>(vw[it], kst + Cfg::TILE_BYTES + (t * D + dl) * Cfg::ELEM);
    };
    [[maybe_unused]] float ksc = 1.f, vsc = 1.f;
    if constexpr (kStageRegs) {
#pragma unroll
      for (int it = 0; it < ITER; ++it) {
        load_k(it);
        load_v(it);
      }
      if constexpr (FP8) {
        ksc = kscl[Cfg::scale_index(my_tok)];
        vsc = vscl[Cfg::scale_index(my_tok)];
      }
      __syncwarp();
      const int nxt = i + NSTAGE;
      if (nxt < nmine) {
        if (lane == 0) fence_proxy_async_smem();
        issue(nxt * HPW + th, s);
      }
    }

    // Partial dot products: instruction it covers row it * NT + lane / RL.
    float part_dot[ITER];
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      if constexpr (!kStageRegs) load_k(it);
      if constexpr (FP8) {
        part_dot[it] = dot_e4m3<EPL>(qh, kw[it]);
      } else {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < EPL / 2; ++e) {
          const float2 kf = __half22float2(*reinterpret_cast<const __half2*>(&kw[it][e]));
          acc = fmaf(qf[2 * e], kf.x, acc);
          acc = fmaf(qf[2 * e + 1], kf.y, acc);
        }
        part_dot[it] = acc;
      }
    }
    // Transposing butterfly over the RL lanes of a row: after round r,
    // lanes keep half of the remaining instructions' rows.
#pragma unroll
    for (int cnt = ITER, off = RL / 2; cnt > 1; cnt >>= 1, off >>= 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int k = 0; k < cnt / 2; ++k) {
        const float send = upper ? part_dot[k] : part_dot[k + cnt / 2];
        const float keep = upper ? part_dot[k + cnt / 2] : part_dot[k];
        part_dot[k] = keep + __shfl_xor_sync(kFull, send, off);
      }
    }
    // Remaining lanes of the same row hold disjoint dim ranges: sum them.
#pragma unroll
    for (int off = RL / ITER / 2; off >= 1; off >>= 1)
      part_dot[0] += __shfl_xor_sync(kFull, part_dot[0], off);

    float dot = part_dot[0];
    if constexpr (FP8) {  // per-(token, head) scale
      if constexpr (!kStageRegs) ksc = kscl[Cfg::scale_index(my_tok)];
      dot *= ksc;
    }
    float sc = (my_tok < valid_rows) ? dot * a.scale_log2 : -INFINITY;
    float mx;  // this stage's maximum of the lane's head
    if constexpr (HPW == 1) {
      mx = warp_max(sc);
    } else {
      const bool second = ((lane / RL) & 1) != 0;
      const float m0 = warp_max(second ? -INFINITY : sc);
      const float m1 = warp_max(second ? sc : -INFINITY);
      mx = second ? m1 : m0;
    }
    const float m_new = fmaxf(m, mx);
    const float alpha = fast_exp2(m - m_new);
    const float pr = (my_tok < valid_rows) ? fast_exp2(sc - m_new) : 0.f;
    // Each lane keeps the sum of its own rows' weights (alpha is uniform over
    // the lanes of a head); the lanes are summed once, after the last stage.
    l = l * alpha + pr;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] *= alpha;
    // e4m3 pools: the weight p * v_scale goes to fp16 (relative error 2^-11)
    // times 2^8, which keeps it in the normal fp16 range; o carries the 2^8
    // until the partition writes it.  The lane holding a row's score forms
    // its weight; instruction it broadcasts the weights of its NT rows.
    float wv = pr;
    if constexpr (FP8) {
      if constexpr (!kStageRegs) vsc = vscl[Cfg::scale_index(my_tok)];
      wv = __uint_as_float((uint32_t)__half_as_ushort(__float2half_rn(pr * 256.f * vsc)));
    }
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      const int t = it * NT + lane / RL;
      const float pt = __shfl_sync(kFull, wv, (lane / RL) * RL + it * (RL / ITER));
      if (t < valid_rows) {
        if constexpr (!kStageRegs) load_v(it);
        if constexpr (FP8) {
          axpy_e4m3<EPL>(o, __ushort_as_half((unsigned short)__float_as_uint(pt)), vw[it]);
        } else {
#pragma unroll
          for (int e = 0; e < EPL / 2; ++e) {
            const float2 vf = __half22float2(*reinterpret_cast<const __half2*>(&vw[it][e]));
            o[2 * e] = fmaf(pt, vf.x, o[2 * e]);
            o[2 * e + 1] = fmaf(pt, vf.y, o[2 * e + 1]);
          }
        }
      }
    }
    m = m_new;

    if constexpr (!kStageRegs) {  // refill this stage with unit i + NSTAGE
      __syncwarp();
      const int nxt = i + NSTAGE;
      if (nxt < nmine) {
        if (lane == 0) fence_proxy_async_smem();
        issue(nxt * HPW + th, s);
      }
    }
  }

  pdl_launch_dependents();  // the combine kernel may be scheduled now
  bool ok = i >= nmine;
  if (!ok) {
    // A bounded wait gave up: report, drain what is still in flight (again
    // bounded) so no copy lands after the CTA exits, and write nothing.
    if (lane == 0) flag_status(a.status, PA_DEV_TIMEOUT);
    for (int j = i; j < nmine && j < i + NSTAGE; ++j) mbar_wait(&bars[j % NSTAGE], (j / NSTAGE) & 1);
  }
  if constexpr (HPW == 2) {
    // Merge the pair's two halves lane by lane (the same head and dims): the
    // odd-stage warp leaves (m, l, o) in its own, now idle, stage room.  Both
    // warps always reach the barrier, so a wait that gave up in one of them
    // cannot leave the other waiting.
    float* xch = reinterpret_cast<float*>(smem + (warp - th + 1) * NSTAGE * Cfg::STAGE_BYTES) +
                 lane * (EPL + 2);
    if (th == 1 && ok) {
      xch[0] = m;
      xch[1] = l;
#pragma unroll
      for (int e = 0; e < EPL; ++e) xch[2 + e] = o[e];
    }
    ok = named_bar_and(1 + warp / 2, 64, ok);
    if (th == 1) return;
    if (ok) {
      const float m1 = xch[0];
      const float mm = fmaxf(m, m1);  // finite: the even warp has at least one stage
      const float w0 = fast_exp2(m - mm), w1 = fast_exp2(m1 - mm);
      l = l * w0 + xch[1] * w1;
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[e] = o[e] * w0 + xch[2 + e] * w1;
      m = mm;
    }
  }
  if (!ok) return;

  if constexpr (FP8) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] *= 1.f / 256.f;  // exact
  }
  // Lanes whose rows differ (of the lane's own head): their weight sums, and
  // (e4m3: several rows per instruction) their o rows for the same dims.
#pragma unroll
  for (int off = LPR; off <= 16; off <<= 1)
    if (HPW == 1 || off != RL) l += __shfl_xor_sync(kFull, l, off);  // lanes of one head
#pragma unroll
  for (int off = RL * HPW; off < 32; off <<= 1)
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] += __shfl_xor_sync(kFull, o[e], off);
  const int n_parts = (ctx + a.part_tokens - 1) / a.part_tokens;
  if (n_parts == 1) {
    const float inv = 1.f / l;
    float r[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) r[e] = o[e] * inv;
    if (lane < RL * HPW) store_half_row<EPL>(a.out + row_bh * D + dl, r);
  } else {
    const size_t row = row_bh * a.num_parts + part;
    float* dst = a.ws_o + row * D + dl;
    if (lane < RL * HPW) {
      if constexpr (EPL % 4 == 0) {
#pragma unroll
        for (int i = 0; i < EPL / 4; ++i)
          reinterpret_cast<float4*>(dst)[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(o[0], o[1]);
      }
    }
    if (lane % RL == 0 && lane < RL * HPW)
      *reinterpret_cast<float2*>(a.ws_ml + row * 2) = make_float2(m, l);
  }
}

// Log-sum-exp merge of the partitions of one (b, h):
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  out = sum_s 2^(m_s - M) o_s / L.
// Up to kFastParts parts: combine_fast_kernel, one warp per (b, h).  More:
// combine_kernel, one CTA of W = blockDim.x / 32 warps per (b, h); warp w
// takes partitions w, w + W, ...; lane l owns dims [l * D/32, (l+1) * D/32).
// W grows with the partition count so a 1M-token context (thousands of
// partitions) still keeps many loads in flight.
constexpr int kMaxCombineWarps = 16;
constexpr int kFastParts = 16;  // combine: parts merged from registers by one warp

constexpr int kCombineHeads = 4;  // fast combine: heads (one warp each) per CTA

// At most kFastParts parts: one warp per (b, h), kCombineHeads heads per CTA
// (one wave of CTAs even for a few thousand (b, h) pairs).  Every part's
// (m, l) and output slice are loaded at once (slots past the sequence's
// parts hold stale data and are masked), so the merge waits on one round
// trip to L2 instead of two.
template <int D>
__global__ void __launch_bounds__(kCombineHeads * 32) combine_fast_kernel(const DecodeArgs a) {
  constexpr int EPL = D / 32;
  pdl_wait();  // partitions come from the partition kernel just before
  const int b = blockIdx.x;
  const int h = blockIdx.y * kCombineHeads + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (h >= a.H) return;  // idle warp of a ragged head group (no CTA-wide sync)
  const size_t row0 = ((size_t)b * a.H + h) * a.num_parts;
  const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + row0;
  float2 mlv = make_float2(-INFINITY, 0.f);
  if (lane < a.num_parts) mlv = ml[lane];
  float ov[kFastParts][EPL];
#pragma unroll
  for (int s = 0; s < kFastParts; ++s) {
    if (s < a.num_parts) {
      const float* src = a.ws_o + (row0 + s) * D + lane * EPL;
      if constexpr (EPL == 4) {
        const float4 t = *reinterpret_cast<const float4*>(src);
        ov[s][0] = t.x; ov[s][1] = t.y; ov[s][2] = t.z; ov[s][3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(src);
        ov[s][0] = t.x; ov[s][1] = t.y;
      }
    }
  }
  const int n = (checked_ctx(a, b, false) + a.part_tokens - 1) / a.part_tokens;
  if (n <= 1) return;  // the partition kernel wrote the row itself
  if (lane >= n) mlv = make_float2(-INFINITY, 0.f);
  float mx = mlv.x;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
  const float wl = lane < n ? fast_exp2(mlv.x - mx) : 0.f;  // weight of part `lane`
  float lsum = wl * mlv.y;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) lsum += __shfl_xor_sync(kFull, lsum, off);
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
#pragma unroll
  for (int s = 0; s < kFastParts; ++s) {
    const float w = __shfl_sync(kFull, wl, s);
    if (s < n) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, ov[s][e], acc[e]);
    }
  }
  const float inv = 1.f / lsum;
  float r[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) r[e] = acc[e] * inv;
  store_half_row<EPL>(a.out + ((size_t)b * a.H + h) * D + lane * EPL, r);
}

// More parts: one CTA of W = blockDim.x / 32 warps per (b, h).
template <int D>
__global__ void __launch_bounds__(kMaxCombineWarps * 32) combine_kernel(const DecodeArgs a) {
  constexpr int EPL = D / 32;
  pdl_wait();  // partitions come from the partition kernel just before
  const int b = blockIdx.x;
  const int h = blockIdx.y;
  const int W = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row0 = ((size_t)b * a.H + h) * a.num_parts;
  const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + row0;
  const int ctx = checked_ctx(a, b, false);
  const int n = (ctx + a.part_tokens - 1) / a.part_tokens;
  if (n <= 1) return;

  __shared__ float red_m[kMaxCombineWarps];
  __shared__ float red_l[kMaxCombineWarps];
  __shared__ float red_o[kMaxCombineWarps][D];

  float mx = -INFINITY;
  for (int s = threadIdx.x; s < n; s += blockDim.x) mx = fmaxf(mx, ml[s].x);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
  if (W > 1) {
    if (lane == 0) red_m[warp] = mx;
    __syncthreads();
    mx = red_m[0];
    for (int w = 1; w < W; ++w) mx = fmaxf(mx, red_m[w]);
  }

  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float lsum = 0.f;
#pragma unroll 4
  for (int s = warp; s < n; s += W) {
    const float2 p = ml[s];
    const float w = fast_exp2(p.x - mx);
    lsum = fmaf(p.y, w, lsum);
    const float* src = a.ws_o + (row0 + s) * D + lane * EPL;
    if constexpr (EPL == 4) {
      const float4 t = *reinterpret_cast<const float4*>(src);
      acc[0] = fmaf(w, t.x, acc[0]); acc[1] = fmaf(w, t.y, acc[1]);
      acc[2] = fmaf(w, t.z, acc[2]); acc[3] = fmaf(w, t.w, acc[3]);
    } else {
      const float2 t = *reinterpret_cast<const float2*>(src);
      acc[0] = fmaf(w, t.x, acc[0]); acc[1] = fmaf(w, t.y, acc[1]);
    }
  }
  if (W > 1) {
    if (lane == 0) red_l[warp] = lsum;
#pragma unroll
    for (int e = 0; e < EPL; ++e) red_o[warp][lane * EPL + e] = acc[e];
    __syncthreads();
    if (warp != 0) return;
    lsum = 0.f;
    for (int w = 0; w < W; ++w) lsum += red_l[w];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      float t = 0.f;
      for (int w = 0; w < W; ++w) t += red_o[w][lane * EPL + e];
      acc[e] = t;
    }
  }
  const float inv = 1.f / lsum;
  float r[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) r[e] = acc[e] * inv;
  store_half_row<EPL>(a.out + ((size_t)b * a.H + h) * D + lane * EPL, r);
}

// Launch shape: WARPS heads per CTA, each warp with ~PK_DECODE_STAGE_BYTES of
// K+V in flight (2..8 stages).  Both can be overridden at compile time.
#ifndef PK_DECODE_WARPS
#define PK_DECODE_WARPS 4
#endif
#ifndef PK_DECODE_INFLIGHT_BYTES
#define PK_DECODE_INFLIGHT_BYTES 16384
#endif

#ifndef PK_DECODE_FP8_NSTAGE
#define PK_DECODE_FP8_NSTAGE 2
#endif

template <int D, int BS, bool FP8, int HPW = 1>
struct DecodeTuning {
  static constexpr int WARPS = PK_DECODE_WARPS;
  static constexpr int STAGE = 2 * (BS < 16 ? BS : 16) * D * 2;
#ifdef PK_DECODE_NSTAGE
  static constexpr int NSTAGE16 = PK_DECODE_NSTAGE;
#else
  static constexpr int RAW = PK_DECODE_INFLIGHT_BYTES / STAGE;
  static constexpr int NSTAGE16 = RAW < 2 ? 2 : (RAW > 8 ? 8 : RAW);
#endif
  // e4m3 stages of 32 rows hold as many bytes as 16 fp16 tokens: two per
  // warp, as for fp16, keeps three CTAs per SM (three stages leave two).
  // Below block size 16 a stage is one block (HPW heads): enough of them for
  // the bytes.
  static constexpr int STAGE8 = 2 * BS * HPW * D;
  static constexpr int RAW8 = PK_DECODE_INFLIGHT_BYTES / STAGE8;
  static constexpr int NSTAGE = !FP8 ? NSTAGE16
                                     : (BS >= 16 ? PK_DECODE_FP8_NSTAGE
                                                 : (RAW8 < 2 ? 2 : (RAW8 > 8 ? 8 : RAW8)));
};

// Programmatic stream serialisation: the kernel may be scheduled before its
// predecessor on the stream finishes; it calls griddepcontrol.wait before
// touching any input, so ordering is preserved while the launch latency hides
// behind the predecessor's tail.
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The partition grid of an ungrouped call with HPW heads per warp.
template <int D, int BS, bool FP8, int HPW>
cudaError_t launch_partitions(const DecodeArgs& a, const DecodeMaps& maps, cudaStream_t stream) {
  using T = DecodeTuning<D, BS, FP8, HPW>;
  using Cfg = PartitionCfg<D, BS, T::WARPS, T::NSTAGE, FP8, HPW>;
  constexpr auto kern = partition_kernel<D, BS, T::WARPS, T::NSTAGE, FP8, false, HPW>;
  cudaError_t e = ensure_dynamic_smem<kern>(Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // WARPS heads per CTA either way (with HPW = 2, two pairs of two warps)
  return launch_pdl(kern, dim3(a.B, (a.H + T::WARPS - 1) / T::WARPS, a.num_parts),
                    dim3(T::WARPS * 32), Cfg::SMEM_BYTES, stream, maps, a);
}

template <int D, int BS, bool FP8>
cudaError_t launch_decode_t(const DecodeArgs& a, const DecodeMaps& maps, cudaStream_t stream) {
  using T = DecodeTuning<D, BS, FP8>;
  using Cfg = PartitionCfg<D, BS, T::WARPS, T::NSTAGE, FP8>;
  dim3 grid(a.B, (a.H + T::WARPS - 1) / T::WARPS, a.num_parts);
  cudaError_t e;
  bool grouped = false;
  if constexpr (!FP8) grouped = a.seq_group != nullptr;
  if (!grouped) {
    if constexpr (FP8) {
      e = decode_heads_per_warp(true, a.H) == 2 ? launch_partitions<D, BS, true, 2>(a, maps, stream)
                                                : launch_partitions<D, BS, true, 1>(a, maps, stream);
    } else {
      e = launch_partitions<D, BS, false, 1>(a, maps, stream);
    }
  } else if constexpr (!FP8) {
    // The grouped grid also runs the shared-prefix partitions.
    constexpr int kPfxSmem = pfx::PrefixCfg<D, T::WARPS>::SMEM;
    constexpr int kSmem = Cfg::SMEM_BYTES > kPfxSmem ? Cfg::SMEM_BYTES : kPfxSmem;
    constexpr auto kern = partition_kernel<D, BS, T::WARPS, T::NSTAGE, FP8, true>;
    e = ensure_dynamic_smem<kern>(kSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, grid, dim3(T::WARPS * 32), kSmem, stream, maps, a);
  }
  if (e != cudaSuccess) return e;
  if (a.num_parts > 1 && a.num_parts <= kFastParts) {
    e = launch_pdl(combine_fast_kernel<D>, dim3(a.B, (a.H + kCombineHeads - 1) / kCombineHeads),
                   dim3(32 * kCombineHeads), 0, stream, a);
  } else if (a.num_parts > 1) {
    int w = a.num_parts / 8;
    w = w < 1 ? 1 : (w > kMaxCombineWarps ? kMaxCombineWarps : w);
    e = launch_pdl(combine_kernel<D>, dim3(a.B, a.H), dim3(32 * w), 0, stream, a);
  }
  return e;
}

}  // namespace

bool prefix_supported(int D, int block_size, int max_group_size) {
  return (D == 64 || D == 128) &&
         (block_size == 4 || block_size == 8 || block_size == 16 || block_size == 32) &&
         max_group_size >= 1 && max_group_size <= pfx::kMaxMembers;
}

int decode_heads_per_warp(bool fp8, int H) {
  return fp8 && PK_DECODE_FP8_HPW == 2 && H % 2 == 0 ? 2 : 1;
}

int decode_box_tokens(bool fp8, int block_size, int heads_per_warp) {
  return box_tokens_for(fp8, block_size, heads_per_warp);
}

bool decode_supported(int D, int block_size) {
  return (D == 64 || D == 128) &&
         (block_size == 4 || block_size == 8 || block_size == 16 || block_size == 32);
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodeMaps& maps, cudaStream_t stream) {
#define PK_CASE(DD, BB)                                              \
  if (a.D == DD && a.block_size == BB)                               \
    return a.fp8 ? launch_decode_t<DD, BB, true>(a, maps, stream)    \
                 : launch_decode_t<DD, BB, false>(a, maps, stream);
  PK_CASE(128, 16) PK_CASE(128, 32) PK_CASE(128, 8) PK_CASE(128, 4)
  PK_CASE(64, 16) PK_CASE(64, 32) PK_CASE(64, 8) PK_CASE(64, 4)
#undef PK_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pk
