// pk_prefix.cuh -- shared-prefix partitions of paged decode (device code included
// by decode.cu: the partition kernel runs them in place of the partitions it skips).
//
// Sequences that share a prompt point at the same physical blocks (study
// notes "DataWhale组队学习笔记--llm-algo-leetcode(五)", "4. PagedAttention 带来的
// 核心红利": the members of a group reference the same blocks until they
// diverge).  Plain decode reads those blocks once per member.  Here the
// partitions lying entirely inside a group's shared prefix are computed once
// per group: a warp streams the shared blocks of one (group, head, partition)
// and attends with every member's query at once, writing each member's
// partition partial (max, normaliser, unnormalised output) to the decode
// workspace.  In the partition kernel's grid, the CTA of the group's first
// member for such a partition does this work for the whole group and the
// other members' CTAs return; the combine kernel merges all partials of a
// sequence by log-sum-exp as usual.  One launch, so the group-wide
// partitions overlap the members' private partitions.
//
// With up to 16 member queries the per-block work is a small dense product
// (16 x 16 scores over D dims, then 16 x D outputs over 16 keys), done with
// warp-level m16n8k16 MMAs (fp16 in, fp32 accumulate) so that it stays far
// below the HBM time of the block: Q fragments stay in registers, K and V
// stages arrive by TMA in 128-byte-swizzled 64-dim halves (conflict-free
// ldmatrix), and the score fragments become the P fragments of the second
// product in registers.
#pragma once
#include "pk_common.cuh"
#include "pk_internal.h"

namespace pk {
namespace pfx {

constexpr unsigned kPfxFull = 0xffffffffu;
constexpr int kMaxMembers = 16;  // rows of one m16n8k16 tile
constexpr int kTB = 16;          // tokens per pipeline stage
constexpr int kStages = 2;

template <int D, int WARPS>
struct PrefixCfg {
  static constexpr int SLABS = D / 64;             // 64-dim halves, 128-byte rows
  static constexpr int SLAB_BYTES = kTB * 128;     // 16 rows x 128 B
  static constexpr int TILE = SLABS * SLAB_BYTES;  // K (or V) of one stage
  static constexpr int STAGE = 2 * TILE;
  // per-warp stages, barriers, and slack to align the base to 1024 B
  static constexpr int SMEM = WARPS * kStages * STAGE + WARPS * kStages * 8 + 1024;
  static constexpr int KSTEPS = D / 16;  // k-steps of the score product
  static constexpr int NT_O = D / 8;     // n-tiles of the output product
};

// Byte offset of (row r, 16-byte chunk c) in a stage tile made of 64-dim
// slabs of 16 rows x 128 B with the 128-byte swizzle (chunk ^ row % 8).
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return (uint32_t)((c >> 3) * (kTB * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16-byte asynchronous global -> shared copy in the thread's current cp.async
// group; commit the group; wait until at most N groups are pending.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_pfx() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ int seq_ctx(const DecodeArgs& a, int b) {  // clamped, silent
  int ctx = a.context_lens[b];
  const int cap = min(a.max_context_len, a.max_blocks * a.block_size);
  return ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
}

// One (group, head group, shared partition) unit: warp w of the CTA takes
// head blockIdx.y * WARPS + w; smem is 1024-byte aligned, PrefixCfg::SMEM - 1024
// bytes long.
// A 16-token stage is a 16-row box of one block (block size 16 or 32), two
// 8-row boxes of two blocks (block size 8: each box fills one 1 KB swizzle
// atom), or, with 4-token blocks (half an atom), 16-byte cp.async copies by
// the lanes into the same swizzled rows.  part_tokens is a multiple of 16
// (the caller runs other partitions as private ones).
template <int D, int BS, int WARPS>
__device__ __forceinline__ void prefix_partition(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                                 const DecodeArgs& a, int grp, int part,
                                                 uint8_t* smem) {
  using Cfg = PrefixCfg<D, WARPS>;
  constexpr int SUB = BS >= kTB ? BS / kTB : 1;  // stages per block
  constexpr int BPS = BS >= kTB ? 1 : kTB / BS;  // blocks per stage
  constexpr bool kGatherCp = BS < 8;
  static_assert(BS % kTB == 0 || kTB % BS == 0, "block size divides 16 or 16 divides it");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * WARPS + warp;
  if (h >= a.H) return;
  const int m0 = a.group_offsets[grp];
  const int mcount = a.group_offsets[grp + 1] - m0;
  if (mcount <= 0) return;
  if (mcount > kMaxMembers) {
    if (lane == 0 && part == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
    return;
  }
  const int first = a.group_seqs[m0];
  if (first < 0 || first >= a.B) return;
  // Partition [tok0, tok1) must lie inside the prefix the members share.
  const int shared =
      min(a.group_prefix_len[grp], seq_ctx(a, first)) / a.part_tokens * a.part_tokens;
  const int tok0 = part * a.part_tokens;
  if (tok0 + a.part_tokens > shared) return;
  const int lb0 = tok0 / BS;
  const int nblk = a.part_tokens / BS;        // <= 32
  const int nunit = a.part_tokens / kTB;

  uint8_t* wbase = smem + warp * kStages * Cfg::STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + WARPS * kStages * Cfg::STAGE) +
                   warp * kStages;

  // Shared block ids from the first member's table, one per lane.
  int phys = 0;
  if (lane < nblk) {
    phys = a.block_tables[(size_t)first * a.max_blocks + lb0 + lane];
    if (phys < 0 || phys >= a.num_blocks) {
      flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
      phys = a.num_blocks;  // outside the tensor map: zero fill
    }
  }

  // Query fragments: rows g and g+8 of the 16-row tile are members g, g+8.
  const int gq = lane >> 2, tq = lane & 3;
  int seq_r[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = gq + 8 * i;
    int sb = -1;
    if (r < mcount) {
      sb = a.group_seqs[m0 + r];
      if (sb < 0 || sb >= a.B || seq_ctx(a, sb) < tok0 + a.part_tokens) sb = -1;
    }
    seq_r[i] = sb;
  }
  uint32_t qa[Cfg::KSTEPS][4];
#pragma unroll
  for (int ks = 0; ks < Cfg::KSTEPS; ++ks) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int sb = seq_r[j & 1];
      const int dim = ks * 16 + 2 * tq + ((j >> 1) << 3);
      qa[ks][j] = sb >= 0 ? *reinterpret_cast<const uint32_t*>(
                                a.q + ((size_t)sb * a.H + h) * D + dim)
                          : 0u;
    }
  }

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  auto issue = [&](int u, int s) {
    uint8_t* st = wbase + s * Cfg::STAGE;
    if constexpr (kGatherCp) {
      // Row r of the stage is token u * 16 + r of the partition; every lane
      // takes (row, 16-byte chunk) pairs of K and of V; one cp.async group
      // per stage.  Rows of an out-of-range block read as zeros.
      constexpr int kChunks = D / 8;
#pragma unroll
      for (int i = lane; i < kTB * kChunks; i += 32) {
        const int r = i / kChunks, c = i % kChunks;
        const int pb = __shfl_sync(kPfxFull, phys, (u * kTB + r) / BS);
        const size_t src = (((size_t)pb * BS + r % BS) * a.H + h) * D + c * 8;
        uint8_t* dk = st + sw_off(r, c);
        if (pb < a.num_blocks) {
          cp_async16(dk, a.k_cache + src);
          cp_async16(dk + Cfg::TILE, a.v_cache + src);
        } else {
          *reinterpret_cast<uint4*>(dk) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(dk + Cfg::TILE) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      cp_async_commit();
    } else {
      int pb[BPS];
#pragma unroll
      for (int k = 0; k < BPS; ++k) pb[k] = __shfl_sync(kPfxFull, phys, (u * BPS + k) / SUB);
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[s], Cfg::STAGE);
#pragma unroll
        for (int k = 0; k < BPS; ++k) {
          const int row = pb[k] * BS + (u % SUB) * kTB;  // first row of the box
          const int r0 = k * (kTB / BPS);                 // its row in the stage
#pragma unroll
          for (int sl = 0; sl < Cfg::SLABS; ++sl) {
            tma_load_3d(st + sl * Cfg::SLAB_BYTES + r0 * 128, &kmap, sl * 64, h, row, &bars[s]);
            tma_load_3d(st + Cfg::TILE + sl * Cfg::SLAB_BYTES + r0 * 128, &vmap, sl * 64, h,
                        row, &bars[s]);
          }
        }
      }
    }
  };
  // (cp.async gathers: one group per stage, an empty one past the end, so
  // that waiting for all but the last kStages - 1 groups completes stage u.)
  for (int u = 0; u < kStages; ++u) {
    if (u < nunit)
      issue(u, u);
    else if constexpr (kGatherCp)
      cp_async_commit();
  }

  float o[Cfg::NT_O][4];
#pragma unroll
  for (int nt = 0; nt < Cfg::NT_O; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const float sl2 = a.scale_log2;
  // ldmatrix row/chunk owned by this lane: matrix lane >> 3, row lane & 7
  const int mi = lane >> 3, rr = lane & 7;

  int u = 0;
  for (; u < nunit; ++u) {
    const int s = u % kStages;
    if constexpr (kGatherCp) {
      cp_async_wait_pfx<kStages - 1>();  // this lane's copies of stage u landed
      __syncwarp();                       // ... and every other lane's
    } else {
      if (!__all_sync(kPfxFull, mbar_wait(&bars[s], (u / kStages) & 1))) break;
    }
    const uint32_t kb = smem_u32(wbase + s * Cfg::STAGE);
    const uint32_t vb = kb + Cfg::TILE;

    // scores: 16 rows (members) x 16 keys, two n-tiles of 8 keys
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < Cfg::KSTEPS; ++ks) {
      uint32_t b00, b01, b10, b11;
      ldsm_x4(kb + sw_off(((mi >> 1) << 3) + rr, 2 * ks + (mi & 1)), b00, b01, b10, b11);
      mma16816(sc[0], qa[ks], b00, b01);
      mma16816(sc[1], qa[ks], b10, b11);
    }
    // online softmax for rows g (elements 0, 1) and g+8 (elements 2, 3)
    float alpha[2], pr[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float mx = fmaxf(fmaxf(sc[0][2 * i], sc[0][2 * i + 1]), fmaxf(sc[1][2 * i], sc[1][2 * i + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(kPfxFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kPfxFull, mx, 2));
      const float m_new = fmaxf(mrow[i], mx * sl2);
      alpha[i] = fast_exp2(mrow[i] - m_new);
      mrow[i] = m_new;
      float sum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float p = fast_exp2(fmaf(sc[nt][2 * i + e], sl2, -m_new));
          pr[nt][2 * i + e] = p;
          sum += p;
        }
      sum += __shfl_xor_sync(kPfxFull, sum, 1);
      sum += __shfl_xor_sync(kPfxFull, sum, 2);
      lrow[i] = lrow[i] * alpha[i] + sum;
    }
#pragma unroll
    for (int nt = 0; nt < Cfg::NT_O; ++nt) {
      o[nt][0] *= alpha[0];
      o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1];
      o[nt][3] *= alpha[1];
    }
    // P as the A fragment of the second product (keys = k)
    uint32_t pa[4];
    pa[0] = pack_half2(pr[0][0], pr[0][1]);
    pa[1] = pack_half2(pr[0][2], pr[0][3]);
    pa[2] = pack_half2(pr[1][0], pr[1][1]);
    pa[3] = pack_half2(pr[1][2], pr[1][3]);
#pragma unroll
    for (int nt = 0; nt < Cfg::NT_O; nt += 2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vb + sw_off(((mi & 1) << 3) + rr, nt + (mi >> 1)), b0, b1, b2, b3);
      mma16816(o[nt], pa, b0, b1);
      mma16816(o[nt + 1], pa, b2, b3);
    }
    __syncwarp();
    const int nxt = u + kStages;
    if (nxt < nunit) {
      if (!kGatherCp && lane == 0) fence_proxy_async_smem();
      issue(nxt, s);
    } else if constexpr (kGatherCp) {
      cp_async_commit();
    }
  }
  if constexpr (kGatherCp) cp_async_wait_pfx<0>();
  if (u < nunit) {
    if (lane == 0) flag_status(a.status, PA_DEV_TIMEOUT);
    for (int j = u; j < nunit && j < u + kStages; ++j)
      mbar_wait(&bars[j % kStages], (j / kStages) & 1);
    return;
  }

  // Each member's partial for this partition (or its final row when the
  // whole context is this one partition).
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int sb = seq_r[i];
    if (sb < 0) continue;
    const int n_parts = (seq_ctx(a, sb) + a.part_tokens - 1) / a.part_tokens;
    const size_t row_bh = (size_t)sb * a.H + h;
    if (n_parts == 1) {
      const float inv = 1.f / lrow[i];
#pragma unroll
      for (int nt = 0; nt < Cfg::NT_O; ++nt)
        *reinterpret_cast<uint32_t*>(a.out + row_bh * D + nt * 8 + 2 * tq) =
            pack_half2(o[nt][2 * i] * inv, o[nt][2 * i + 1] * inv);
    } else {
      const size_t row = row_bh * a.num_parts + part;
#pragma unroll
      for (int nt = 0; nt < Cfg::NT_O; ++nt)
        *reinterpret_cast<float2*>(a.ws_o + row * D + nt * 8 + 2 * tq) =
            make_float2(o[nt][2 * i], o[nt][2 * i + 1]);
      if (tq == 0) *reinterpret_cast<float2*>(a.ws_ml + row * 2) = make_float2(mrow[i], lrow[i]);
    }
  }
}


}  // namespace pfx
}  // namespace pk
