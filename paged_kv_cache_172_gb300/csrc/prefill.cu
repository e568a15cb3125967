// prefill.cu -- chunked prefill attention over a paged KV cache on the sm_103a
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Definition (blog "PagedAttention origin and evolution", sec. 3.2.2: per
// request gather K/V through the block table, Q K^T / sqrt(d), causal mask,
// softmax, P V; the mask is read as aligned to the END of the context, so the
// Lq chunk queries sit at positions n-Lq .. n-1 and query i sees keys
// 0 .. n-Lq+i).
//
// One CTA = 256 queries (two 128-row tiles A and B) of one (sequence, head);
// it walks the visible keys in tiles of 128 (128 / block_size blocks):
//   warps 0-3   softmax of tile A, one query row per thread (TMEM lane = row);
//   warps 4-7   softmax of tile B;
//   warp 8      producer: Q (boxes of 128 rows x 64 dims, 128-byte swizzle),
//               then per key tile one 5-D TMA box per block (all its tokens,
//               every 64-dim half) for K and for V, gathered through the
//               block table, into a ring in first-use order K_0, K_1, V_0,
//               K_2, V_1, ...  With 4-token blocks (half of an 8-row swizzle
//               atom) the lanes gather the rows with 16-byte cp.async copies
//               into the same layout instead;
//   warp 9      S issuer (one thread) and tensor-memory owner;
//   warp 10     P V issuer (one thread).
// Head dims 128 and 64 are instantiations of the same kernel (D / 64 halves
// of 64 dims; 128-byte swizzle rows of 64 fp16).
// Tensor memory: S [0,128) shared by the two tiles, P_A [128,192) and P_B
// [192,256) (fp16 pairs: column c holds keys 2c, 2c+1), O_A and O_B from
// column 256 (D columns each).  Q stays in shared memory where TMA put it
// (the A operand of S = Q K^T) and P lives in tensor memory (the A operand
// of O += P V): per key tile the shared memory then serves 64 KB of TMA
// fills, Q and K reads of the two S products and the V reads of the two
// P V products (~256 KB) where P in shared memory cost another 64 KB of P
// stores and 64 KB of P reads (~320 KB); its bandwidth, not the tensor pipe,
// bounded that layout.
// Softmax of tile X, key tile j: wait for S_X(j), load the whole row into
// registers and release S at once, so the tensor core computes the other
// tile's S while this softmax still works on j.  Row max: returned by the
// loads themselves (tcgen05.ld.red) on tiles with no masked key, taken over
// the unmasked keys on diagonal tiles; p = 2^(s*scale*log2e - m) (one FMA, one ex2)
// packed to fp16 in registers with the row sum; then wait for P_X(j-1) V_{j-1}
// (so O_X is stable and P_X free), rescale O_X only when the row max grew by
// more than 2^8 (P then stays <= 256, exact in fp16 range), store P_X to
// tensor memory (two 32-column stores).
// The S products go A(0), B(0), A(1), B(1), ..., each once the softmax
// released the previous one and its K tile landed; O_X += P_X(j) V_j once
// P_X(j) is stored and V_j landed.  The two
// kinds come from two threads, so a P V product that gates a softmax never
// queues behind S products at the issuing end.
// Operand layouts (tcgen05 shared-memory descriptors, 128-byte swizzle; the
// 16-byte chunk c of a 128-byte row r sits at chunk position c ^ (r mod 8)):
//   Q_X         : K-major, rows of 64 fp16 (128 B), 8-row atoms 1024 B
//                 apart, 64-element halves 16 KB apart (the TMA boxes'
//                 landing order; the output tile is staged the same way);
//   K_j, V_j    : key groups of 8 keys x D dims (D * 16 bytes apart), each
//                 holding the 1 KB atom of dims 0-63 then (D = 128) that of
//                 dims 64-127 (the order one box of a block lands in).  K_j
//                 is read K-major (8-key atoms one group apart along N, halves
//                 1 KB apart along K), V_j MN-major (8-key atoms one group
//                 apart along K, halves 1 KB apart along N).  Fewer, larger
//                 boxes: the TMA unit spends a fixed ~50 cycles per box besides
//                 ~2 per 128-byte row, which bounded the K/V stream at block
//                 size 16.
#include <string.h>

#include "pk_common.cuh"
#include "pk_internal.h"
#include "pk_tcgen05.cuh"

namespace pk {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kTileM = 128;                  // queries per Q tile (two per CTA)
constexpr int kTileN = 128;                  // keys per tile
constexpr int kSlabBytes = 128 * 128;        // 128 rows x 64 fp16 (half of a Q tile)
constexpr int kQTileBytes = 2 * kSlabBytes;  // a Q tile's room: 128 queries x up to 128 dims
constexpr int kThreads = 352;                // 8 softmax warps + producer + 2 MMA issuers
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;                  // S = Q K^T issuer, tensor-memory owner
constexpr int kWarpPv = 10;                  // O += P V issuer
constexpr int kTblWindow = 256;              // block-table entries staged in smem
constexpr int kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColP = 128;              // P_A, then P_B 64 columns later
constexpr uint32_t kColO = 256;              // O_A, then O_B D columns later
constexpr int kMaxStages = 8;
constexpr int kNumBars = 1 + 2 * kMaxStages + 2 + 2 + 2 + 2 + 1;

// Per head dim: the K/V tile (128 keys x D dims), its 8-key groups, and the
// ring depth that fills the shared memory the two Q tiles leave.
template <int D>
struct PfCfg {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int HALVES = D / 64;                 // 64-dim halves of a row
  static constexpr int TILE_BYTES = kTileN * D * 2;     // one K or V tile (= one Q tile)
  static constexpr int GROUP_BYTES = 8 * D * 2;         // 8 keys x D dims
  static constexpr int STAGES = D == 128 ? 5 : 8;       // K/V ring slots
  static_assert(STAGES <= kMaxStages, "barrier room");
  static constexpr int OFF_Q = 0;                       // Q_A, Q_B (then the output tiles)
  static constexpr int OFF_KV = OFF_Q + 2 * kQTileBytes;
  static constexpr int OFF_BAR = OFF_KV + STAGES * TILE_BYTES;
  static constexpr int OFF_TMEM_HOLDER = OFF_BAR + kNumBars * 8;
  static constexpr int OFF_ISSUED = OFF_TMEM_HOLDER + 4;  // [2] S products issued per tile
  static constexpr int OFF_TBL = (OFF_ISSUED + 8 + 15) / 16 * 16;
  static constexpr int SMEM_BYTES = OFF_TBL + kTblWindow * 4 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static constexpr uint32_t IDESC_S = tc::idesc_f16_f32(kTileM, kTileN, false, false);
  static constexpr uint32_t IDESC_O = tc::idesc_f16_f32(kTileM, D, false, true);
  static constexpr uint32_t TILE_DESC = TILE_BYTES >> 4;  // one K/V tile, descriptor units
  static constexpr int PARTIAL_STRIDE = D + 4;            // o[D], m, l, pad (16-byte rows)
};

constexpr uint32_t kQTileDesc = kQTileBytes >> 4;  // one Q tile, descriptor units

// Descriptor address offset of K step kk (16 elements = 32 B) of a K-major
// Q tile: inside the 64-element half kk / 4.
__device__ __forceinline__ constexpr uint32_t kmajor_off(int kk) {
  return (uint32_t)((kk >> 2) * kSlabBytes + (kk & 3) * 32) >> 4;
}
// ... of a K tile (key groups): the half's atom sits 1 KB into each group.
__device__ __forceinline__ constexpr uint32_t kgroup_off(int kk) {
  return (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
}
// ... of an MN-major V tile: keys 16*kk .. 16*kk+15 are two key groups.
template <int D>
__device__ __forceinline__ constexpr uint32_t vmn_off(int kk) {
  return (uint32_t)(kk * 2 * PfCfg<D>::GROUP_BYTES) >> 4;
}

// Wait until the S issuer has issued `n` S products of a tile (its counter
// only grows); false after kWaitLimitCycles.
__device__ __forceinline__ bool wait_issued(volatile int* cnt, int n) {
  if (*cnt >= n) return true;
  const long long t0 = clock64();
  while (*cnt < n) {
    __nanosleep(32);
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}

// Ring load index of K_t and V_t (loads go K_0, then K_{t+1}, V_t per t).
__device__ __forceinline__ int load_k(int t) { return t == 0 ? 0 : 2 * t - 1; }
__device__ __forceinline__ int load_v(int t, int n_kv) { return t + 1 < n_kv ? 2 * t + 2 : 2 * t + 1; }

// 16-byte asynchronous global -> shared copy (cached in L2 only), in the
// thread's current cp.async group.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's committed cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap omap, const PrefillArgs a) {
  using C = PfCfg<D>;
  constexpr int BPT = kTileN / BS;    // blocks per key tile
  constexpr bool kGatherCp = BS < 8;  // a block is less than one 8-row swizzle atom
  constexpr int kStages = C::STAGES;
  constexpr int kTileBytes = C::TILE_BYTES;
  constexpr int kGroupBytes = C::GROUP_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint8_t* sQ = smem + C::OFF_Q;  // Q_A, Q_B; each becomes its tile's output staging
  uint8_t* sKV = smem + C::OFF_KV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;  // [2] per Q tile: S_X(j) computed
  uint64_t* s_free = s_full + 2;          // [2]: softmax of X holds S in registers
  uint64_t* p_full = s_free + 2;          // [2]: P_X(j) stored
  uint64_t* pv_done = p_full + 2;         // [2]: O_X += P_X(j) V_j completed
  uint64_t* drain = pv_done + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_HOLDER);
  int32_t* tbl_s = reinterpret_cast<int32_t*>(smem + C::OFF_TBL);
  volatile int* s_issued = reinterpret_cast<volatile int*>(smem + C::OFF_ISSUED);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Work unit (sequence, head, 256-query pair) and, for a split unit, its part.
  int unit = blockIdx.x, part = -1;
  if (unit >= a.full_units) {
    const int t = unit - a.full_units;
    unit = a.full_units + t / a.split;
    part = t % a.split;
  }
  const int ct = unit % a.gx, h = (unit / a.gx) % a.H, b = unit / (a.gx * a.H);
  // Partial rows of this part (query row r of the unit at ws_part + r * stride).
  float* ws_part = part < 0 ? nullptr
                            : a.ws + ((size_t)(unit - a.full_units) * a.split + part) *
                                         (2 * kTileM) * C::PARTIAL_STRIDE;

  pdl_wait();  // inputs may come from the previous kernel on the stream
  const int n = a.context_lens[b];
  const int ql = a.q_lens != nullptr ? a.q_lens[b] : a.Lq;  // this sequence's new queries
  const int q0 = ct * 2 * kTileM;
  const int rows_all = min(2 * kTileM, a.Lq - q0);
  const size_t out_row0 = ((size_t)b * a.H + h) * a.Lq + q0;
  const bool bad = ql < 0 || ql > a.Lq || n < ql || n > a.max_blocks * BS;
  if (bad || q0 >= ql) {
    // A bad length (flagged), or rows past this sequence's chunk only: zero
    // rows (a whole unit) or an empty partial (a part; the combine writes
    // the zeros).
    if (bad && threadIdx.x == 0 && part <= 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
    if (part < 0) {
      uint4* o4 = reinterpret_cast<uint4*>(a.out + out_row0 * D);
      for (int i = threadIdx.x; i < rows_all * (D / 8); i += kThreads)
        o4[i] = make_uint4(0, 0, 0, 0);
    } else {  // an empty partial: the combine writes zero rows
      for (int r = threadIdx.x; r < 2 * kTileM; r += kThreads) {
        ws_part[(size_t)r * C::PARTIAL_STRIDE + D] = -INFINITY;
        ws_part[(size_t)r * C::PARTIAL_STRIDE + D + 1] = 0.f;
      }
    }
    return;
  }
  // Per Q tile (A = 0, B = 1): rows, sequence position of row 0, key tiles.
  // ntile_a <= ntile_b whenever tile B has rows.
  const int rows_a = min(kTileM, ql - q0);
  const int rows_b = max(0, min(kTileM, ql - (q0 + kTileM)));
  const int pos0_a = n - ql + q0;
  const int pos0_b = pos0_a + kTileM;
  // Key tiles of the unit, then this CTA's range [kt0, kt0 + n_kv) of them;
  // ntile_a / ntile_b count the range's tiles each Q tile reads.
  const int ntile_a_all = (pos0_a + rows_a - 1) / kTileN + 1;
  const int ntile_b_all = rows_b > 0 ? (pos0_b + rows_b - 1) / kTileN + 1 : 0;
  const int n_kv_all = max(ntile_a_all, ntile_b_all);
  int kt0 = 0, n_kv = n_kv_all;
  if (part >= 0) {
    kt0 = part * n_kv_all / a.split;
    n_kv = (part + 1) * n_kv_all / a.split - kt0;
  }
  const int ntile_a = min(max(ntile_a_all - kt0, 0), n_kv);
  const int ntile_b = min(max(ntile_b_all - kt0, 0), n_kv);
  const int nblk_seq = (n + BS - 1) / BS;

  if (threadIdx.x == 0) {
    s_issued[0] = 0;
    s_issued[1] = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);  // one arrival per softmax warp
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(drain, 2);
    fence_mbar_init();
    // Q goes out first, before tensor memory is allocated and the CTA syncs:
    // it heads the start-up path (Q -> first S product).
    const int bh = b * a.H + h;
    mbar_arrive_expect_tx(q_full, 2 * kTileBytes);
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int hf = 0; hf < C::HALVES; ++hf)
        tma_load_3d(sQ + x * kQTileBytes + hf * kSlabBytes, &qmap, 64 * hf, q0 + x * kTileM,
                    bh, q_full);
  }
  // The producer's first block-table window, in flight across the sync.
  constexpr int kPerLane = kTblWindow / 32;
  int ent0[kPerLane];
  if (warp == kWarpProducer) {
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) {
      const int lb = kt0 * BPT + lane + 32 * k;
      ent0[k] = lb < nblk_seq ? __ldg(a.block_tables + (size_t)b * a.max_blocks + lb)
                              : a.num_blocks;
    }
  }
  if (warp == kWarpMma) {
    tc::tmem_alloc(tmem_holder, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;
  int issued = 0;  // K/V tiles the producer issued into the ring by TMA

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    int win = -kTblWindow;
    if (lane == 0 && !kGatherCp) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
    }
    // Key tile t (K when v == 0, else V) into ring slot u % kStages.
    auto load_tile = [&](int t, int v, int u) {
      const int lb0 = (kt0 + t) * BPT;
      if (lb0 < win || lb0 + BPT > win + kTblWindow) {
        // K_t is requested before V_{t-1}: start the window one tile early.
        win = (v == 0 && t > 0) ? lb0 - BPT : lb0;
        __syncwarp();
        // All of the window's loads in flight at once (one round trip, not
        // one per 32 entries: this sits on the CTA's start-up path).
        int ent[kPerLane];
        if (win == kt0 * BPT && t == 0) {  // the first window, loaded before the sync
#pragma unroll
          for (int k = 0; k < kPerLane; ++k) ent[k] = ent0[k];
        } else {
#pragma unroll
          for (int k = 0; k < kPerLane; ++k) {
            const int lb = win + lane + 32 * k;
            ent[k] = lb < nblk_seq ? __ldg(a.block_tables + (size_t)b * a.max_blocks + lb)
                                   : a.num_blocks;  // past the sequence: zeros
          }
        }
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
          int phys = ent[k];
          if (phys < 0 || phys > a.num_blocks ||
              (phys == a.num_blocks && win + lane + 32 * k < nblk_seq)) {
            flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
            phys = a.num_blocks;
          }
          tbl_s[lane + 32 * k] = phys;
        }
        __syncwarp();
      }
      const int st = u % kStages;
      if (lane == 0) {
        ok = mbar_wait(&kv_empty[st], ((u / kStages) & 1) ^ 1);
        if (ok && !kGatherCp) mbar_arrive_expect_tx(&kv_full[st], kTileBytes);
      }
      ok = __shfl_sync(kFull, ok, 0);
      if constexpr (!kGatherCp) {
        // One box per lane and block: (64 dims, 8 keys, D/64 halves, BS/8 key
        // groups) at row phys*BS*H + h of the pool seen as [slot*H + head]
        // rows; past-the-sequence blocks (phys = num_blocks) fall outside the
        // map and read as zeros.
        if (ok && lane < BPT) {
          uint8_t* dst = sKV + st * kTileBytes + lane * (BS / 8) * kGroupBytes;
          tma_load_5d(dst, v ? &vmap : &kmap, 0, 0, 0, 0,
                      tbl_s[lb0 - win + lane] * BS * a.H + h, &kv_full[st]);
        }
        if (ok && lane == 0) ++issued;
      } else if (ok) {
        // Blocks of fewer than 8 tokens: 16-byte copies by the lanes, placed
        // as the TMA boxes would land them (key r at row r & 7 of group
        // r >> 3, chunk c of a 64-dim half at c ^ (r & 7)).  Keys of blocks
        // past the sequence are zero-filled.  Lane l takes keys l + 32 i.
        const __half* pool = v ? a.v_cache : a.k_cache;
        uint8_t* tile = sKV + st * kTileBytes;
#pragma unroll
        for (int i = 0; i < kTileN / 32; ++i) {
          const int r = lane + 32 * i;
          const int phys = tbl_s[lb0 - win + r / BS];
          uint8_t* grp = tile + (r >> 3) * kGroupBytes + (r & 7) * 128;
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {  // 16-byte chunks of the row
            uint8_t* dst = grp + (c >> 3) * 1024 + (((c & 7) ^ (r & 7)) * 16);
            if (phys < a.num_blocks)
              cp_async16(dst, pool + (((size_t)phys * BS + r % BS) * a.H + h) * D + c * 8);
            else
              *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        cp_async_commit();
      }
    };
    // cp.async gathers: tile u is published one load later, once this lane's
    // copies of it have completed (the group of tile u+1 may still fly); the
    // proxy fence makes the copied bytes visible to the tensor core.
    auto publish = [&](int u) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&kv_full[u % kStages]);
    };
    int u = 0;
    if (n_kv > 0) load_tile(0, 0, u++);
    for (int j = 0; j < n_kv && ok; ++j) {
      if (j + 1 < n_kv) {
        load_tile(j + 1, 0, u++);
        if constexpr (kGatherCp) {
          if (ok) {
            cp_async_wait<1>();
            publish(u - 2);
          }
        }
      }
      if (ok) {
        load_tile(j, 1, u++);
        if constexpr (kGatherCp) {
          if (ok) {
            cp_async_wait<1>();
            publish(u - 2);
          }
        }
      }
    }
    if constexpr (kGatherCp) {
      cp_async_wait<0>();  // none of this warp's copies stays in flight
      if (ok && u > 0) publish(u - 1);
    }
  } else if (warp == kWarpMma || warp == kWarpPv) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads: S_X(t) = Q_X K_t^T once the softmax of X released S_X(t-1)
    // and K_t landed; O_X (+)= P_X(t) V_t once P_X(t) is stored and V_t
    // landed.  Each thread's commits track its own MMAs, and K is read only
    // by the first, V and O only by the second.
    const int nt[2] = {ntile_a, ntile_b};
    auto landed = [&](int u) { return mbar_wait(&kv_full[u % kStages], (u / kStages) & 1); };
    if (warp == kWarpMma) {
      if (lane == 0) {
        // Base descriptors; each MMA adds a compile-time offset (a slot, a
        // tile or a K step never carries out of the 14-bit address field).
        const uint64_t dk = tc::smem_desc(smem_u32(sKV), 16, kGroupBytes, tc::kSwizzle128B);
        const uint64_t dq = tc::smem_desc(smem_u32(sQ), 16, 1024, tc::kSwizzle128B);
        bool q_landed = false;
        int last_x = -1, last_t = 0;  // the S product issued last
        for (int t = 0; t < n_kv && ok; ++t) {
          const int u = load_k(t);
          for (int x = 0; x < 2 && ok; ++x) {
            if (t >= nt[x]) continue;
            if (!q_landed && !(ok = q_landed = mbar_wait(q_full, 0))) break;
            // S is free once the softmax of the previous product loaded it
            if (last_x >= 0 && !(ok = mbar_wait(&s_free[last_x], last_t & 1))) break;
            if (!(ok = landed(u))) break;
            tc::fence_after_sync();
            const uint64_t db = dk + (u % kStages) * C::TILE_DESC;
            const uint64_t da = dq + x * kQTileDesc;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc::mma_f16(tmem + kColS, da + kmajor_off(kk), db + kgroup_off(kk), C::IDESC_S,
                          kk > 0 ? 1u : 0u);
            tc::commit(&s_full[x]);
            s_issued[x] = t + 1;  // read by the P V issuer (a scheduling hint only)
            last_x = x;
            last_t = t;
          }
          if (ok) tc::commit(&kv_empty[u % kStages]);  // K_t has no further reader
        }
      }
    } else {
      const uint64_t dv = tc::smem_desc(smem_u32(sKV), 1024, kGroupBytes, tc::kSwizzle128B);
      // Rows of the last key tile at or past the context length come from the
      // unused tail of the last block (never written: possibly NaN) and would
      // give P * V = 0 * NaN; the whole warp zeroes them once V has landed.
      const int tail_rows = n - (kt0 + n_kv - 1) * kTileN;  // valid rows of the last key tile
      auto issue_pv = [&](int t) {  // lane 0
        const int u = load_v(t, n_kv);
        for (int x = 0; x < 2 && ok; ++x) {
          if (t >= nt[x]) continue;
          if (!(ok = mbar_wait(&p_full[x], t & 1))) break;
          if (!(ok = landed(u))) break;
          // Keep the tensor core's queue in chain order: P_X(t) V_t goes in
          // behind S_X(t+1), so that S product never waits for it.  The S
          // chain does not depend on this product, so the wait ends.
          if (t + 1 < nt[x] && !(ok = wait_issued(s_issued + x, t + 2))) break;
          tc::fence_after_sync();
          const uint32_t ta = tmem + kColP + x * (kTileN / 2);
          const uint64_t db = dv + (u % kStages) * C::TILE_DESC;
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            tc::mma_f16_ts(tmem + kColO + x * D, ta + kk * 8, db + vmn_off<D>(kk), C::IDESC_O,
                           (t > 0 || kk > 0) ? 1u : 0u);
          tc::commit(&pv_done[x]);
        }
        if (ok) tc::commit(&kv_empty[u % kStages]);  // V_t has no further reader
      };
      if (lane == 0)
        for (int t = 0; t + 1 < n_kv && ok; ++t) issue_pv(t);
      ok = __shfl_sync(kFull, ok, 0);
      if (ok && n_kv > 0) {
        if (tail_rows < kTileN) {
          const int u = load_v(n_kv - 1, n_kv);
          if (lane == 0) ok = landed(u);
          ok = __shfl_sync(kFull, ok, 0);
          if (ok) {
            uint8_t* vt = sKV + (u % kStages) * kTileBytes;
            constexpr int kChunks = D / 8;  // 16-byte chunks per row
            for (int i = lane; i < (kTileN - tail_rows) * kChunks; i += 32) {
              const int r = tail_rows + i / kChunks, c = i % kChunks;
              *reinterpret_cast<uint4*>(vt + (r >> 3) * kGroupBytes + (c >> 3) * 1024 +
                                        (r & 7) * 128 + (c & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // read by the tensor core (async proxy)
          }
          __syncwarp();
        }
        if (ok && lane == 0) issue_pv(n_kv - 1);
      }
    }
    ok = __shfl_sync(kFull, ok, 0);
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;       // Q tile of this warpgroup
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_s = tmem + t_lane + kColS;
    const uint32_t t_o = tmem + t_lane + kColO + x * D;
    const int pos0 = x ? pos0_b : pos0_a;
    const int pos = pos0 + row;
    const int ntile = x ? ntile_b : ntile_a;
    const float sl2 = a.scale_log2;
    uint8_t* orow = sQ + x * kQTileBytes + row * 128;  // output staging (Q's room)
    float m = -INFINITY, l = 0.f;
    // Q lands in shared memory by TMA and is read there by the S products;
    // waiting for it here also keeps a CTA with no S product to issue from
    // leaving while its copy is in flight.
    ok = __all_sync(kFull, mbar_wait(q_full, 0));
    for (int j = 0; j < ntile && ok; ++j) {
      if (!(ok = __all_sync(kFull, mbar_wait(&s_full[x], j & 1)))) break;
      tc::fence_after_sync();
      const int kbase = (kt0 + j) * kTileN;
      const bool diag = kbase + kTileN - 1 > pos0;  // some key here is past some row
      // The whole S row in registers; S_X is then free for S_X(j+1).
      // The loads also give each 32-key chunk's maximum.
      uint32_t r[4][32];
      float cm[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::ld_32x32_max(t_s + c * 32, r[c], cm[c]);
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[x]);  // one arrival per warp
      float mt = max3f(cm[0], cm[1], fmaxf(cm[2], cm[3]));
      if (diag) {  // keys past this row's position: -inf, and the maximum of the rest
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (kbase + c * 32 + i > pos) r[c][i] = __float_as_uint(-INFINITY);
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            mx[(i >> 1) & 7] = max3f(mx[(i >> 1) & 7], __uint_as_float(r[c][i]),
                                     __uint_as_float(r[c][i + 1]));
        mt = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      }
      mt *= sl2;
      const float m_new = fmaxf(m, mt);
      const bool resc = m_new > m + 8.0f;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m - m_new);
        m = m_new;
        l *= alpha;
      }
      // P = 2^(s * scale * log2e - m) packed to fp16 pairs in place (the
      // first 16 words of each 32-key chunk), row sum.  A masked key has
      // s = -inf, so p = 0.
      // Packed pairs: one FMA and one add instruction per two keys.
      const float neg_m = -m;
      float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float y0, y1;
          fma_f32x2(y0, y1, __uint_as_float(r[c][2 * e]), __uint_as_float(r[c][2 * e + 1]), sl2,
                    sl2, neg_m, neg_m);
          const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
          const int k = 2 * (e & 3);
          add_f32x2(rs[k], rs[k + 1], rs[k], rs[k + 1], p0, p1);
          __half2 hp = __floats2half2_rn(p0, p1);
          r[c][e] = *reinterpret_cast<uint32_t*>(&hp);
        }
      l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      // P_X(j-1) V_{j-1} done: the P_X tile is free, O_X is stable.
      if (j > 0) {
        if (!(ok = __all_sync(kFull, mbar_wait(&pv_done[x], (j - 1) & 1)))) break;
        tc::fence_after_sync();
      }
      if (j > 0 && __any_sync(kFull, resc)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tc::ld_32x32(t_o + c * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tc::st_32x32(t_o + c * 32, o);
        }
        tc::wait_st();
      }
      // Store P into tensor memory: column c of P_X holds keys 2c, 2c+1 (the
      // A operand of O += P V; chunk c of the row packed in r[c][0..15]).
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pw[32];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          pw[e] = r[2 * hf][e];
          pw[16 + e] = r[2 * hf + 1][e];
        }
        tc::st_32x32(tmem + t_lane + kColP + x * (kTileN / 2) + hf * 32, pw);
      }
      tc::wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[x]);
    }
    if (ok && ntile > 0) ok = __all_sync(kFull, mbar_wait(&pv_done[x], (ntile - 1) & 1));
    // One decision for the whole tile (a wait that gave up in one warp only
    // must not leave the others at the epilogue's barrier).
    ok = named_bar_and(1 + x, 128, ok);
    if (ok && part >= 0) {
      // Part of a split unit: the unnormalised row (o, m, l) for the combine;
      // a Q tile with no key tile in this part leaves an empty partial.
      float* wrow = ws_part + (size_t)(x * kTileM + row) * C::PARTIAL_STRIDE;
      if (ntile > 0) tc::fence_after_sync();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (ntile > 0) {
          tc::ld_32x32(t_o + c * 32, o);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        float4* dst = reinterpret_cast<float4*>(wrow + c * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                               __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
      }
      wrow[D] = ntile > 0 ? m : -INFINITY;
      wrow[D + 1] = ntile > 0 ? l : 0.f;
    } else if (ok && q0 + x * kTileM < a.Lq) {
      // The output tile goes through Q_X's room (free: every S product of X
      // is done, since its last P V product is; Q_X landed before any
      // softmax started), swizzled like the TMA tiles, and leaves by TMA
      // stores: one 16 KB copy per 64-dim half instead of scattered 16-byte
      // stores per thread.  Rows past the tensor's Lq fall outside the map and
      // are not written; rows past this sequence's chunk (chunks of different
      // lengths) are written as zeros.
      const bool live = row < (x ? rows_b : rows_a);
      if (ntile > 0) tc::fence_after_sync();
      const float inv = ntile > 0 ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {  // dims 32c .. 32c+31
        uint32_t o[32];
        if (ntile > 0) {
          tc::ld_32x32(t_o + c * 32, o);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t hv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          __half2 t = __floats2half2_rn(__uint_as_float(o[2 * i]) * inv,
                                        __uint_as_float(o[2 * i + 1]) * inv);
          hv[i] = live ? *reinterpret_cast<uint32_t*>(&t) : 0u;
        }
        uint8_t* slab = orow + (c >> 1) * kSlabBytes;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = (((c & 1) << 2) + q) ^ (row & 7);
          *reinterpret_cast<uint4*>(slab + chunk * 16) =
              make_uint4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();  // read by the TMA unit (async proxy)
      named_bar_sync(1 + x, 128);
      if (quarter == 0 && lane == 0) {
        const int bh = b * a.H + h;
#pragma unroll
        for (int hf = 0; hf < C::HALVES; ++hf)
          tma_store_3d(&omap, sQ + x * kQTileBytes + hf * kSlabBytes, 64 * hf, q0 + x * kTileM,
                       bh);
        bulk_commit_group();
        bulk_wait_all();  // the shared-memory source stays valid until the CTA exits
      }
    }
  }

  // All roles meet here.  After a bounded wait gave up anywhere, the producer
  // lets the copies it still has in flight land and the MMA issuer waits for
  // its last MMAs (both bounded) before shared and tensor memory are released.
  tc::fence_before_sync();
  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) flag_status(a.status, PA_DEV_TIMEOUT);
    if (warp == kWarpProducer && lane == 0) {
      mbar_wait(q_full, 0);
      for (int u = max(0, issued - kStages); u < issued; ++u)
        mbar_wait(&kv_full[u % kStages], (u / kStages) & 1);
    }
    if ((warp == kWarpMma || warp == kWarpPv) && lane == 0) {
      tc::commit(drain);
      mbar_wait(drain, 0);
    }
    __syncthreads();
  }
  if (warp == kWarpMma) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the parts of split units by log-sum-exp (m, l in the softmax's log2
// domain): one warp per query row, lane l owns dims [l * D/32, (l+1) * D/32).
template <int D>
__global__ void __launch_bounds__(256)
    prefill_combine_kernel(const PrefillArgs a, int n_split_units) {
  constexpr int EPL = D / 32;
  constexpr int kStride = PfCfg<D>::PARTIAL_STRIDE;
  pdl_wait();  // the partials come from the prefill kernel just before
  const int w = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= n_split_units * 2 * kTileM) return;
  const int su = w / (2 * kTileM), r = w % (2 * kTileM);
  const int unit = a.full_units + su;
  const int ct = unit % a.gx, h = (unit / a.gx) % a.H, b = unit / (a.gx * a.H);
  const int qi = ct * 2 * kTileM + r;
  if (qi >= a.Lq) return;
  // rows past this sequence's chunk (chunks of different lengths): zeros
  const bool live = qi < (a.q_lens != nullptr ? a.q_lens[b] : a.Lq);
  const float* base = a.ws + (size_t)su * a.split * (2 * kTileM) * kStride + (size_t)r * kStride;
  const size_t part_stride = (size_t)(2 * kTileM) * kStride;
  // All parts' loads issued together (split <= PK_PREFILL_MAX_SPLIT <= 8).
  constexpr int kMaxParts = 8;
  float ms[kMaxParts], ls[kMaxParts];
  float ov[kMaxParts][EPL];
#pragma unroll
  for (int s = 0; s < kMaxParts; ++s) {
    if (s < a.split) {
      const float* pr = base + s * part_stride;
      ms[s] = pr[D];
      ls[s] = pr[D + 1];
      if constexpr (EPL == 4) {
        const float4 t = *reinterpret_cast<const float4*>(pr + lane * 4);
        ov[s][0] = t.x; ov[s][1] = t.y; ov[s][2] = t.z; ov[s][3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(pr + lane * 2);
        ov[s][0] = t.x; ov[s][1] = t.y;
      }
    } else {
      ms[s] = -INFINITY;
      ls[s] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) ov[s][e] = 0.f;
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < kMaxParts; ++s)
    if (ls[s] > 0.f) M = fmaxf(M, ms[s]);
  float L = 0.f, o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxParts; ++s) {
    if (ls[s] > 0.f) {  // an empty part's o is never read as a number
      const float wgt = ex2_approx(ms[s] - M);
      L += ls[s] * wgt;
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[e] += wgt * ov[s][e];
    }
  }
  const float inv = L > 0.f && live ? 1.f / L : 0.f;
  __half* dst = a.out + (((size_t)b * a.H + h) * a.Lq + qi) * D + lane * EPL;
  if constexpr (EPL == 4) {
    __half2 h0 = __floats2half2_rn(o[0] * inv, o[1] * inv);
    __half2 h1 = __floats2half2_rn(o[2] * inv, o[3] * inv);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&h0);
    u.y = *reinterpret_cast<uint32_t*>(&h1);
    *reinterpret_cast<uint2*>(dst) = u;
  } else {
    *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(o[0] * inv, o[1] * inv);
  }
}

#ifndef PK_PREFILL_MAX_SPLIT
#define PK_PREFILL_MAX_SPLIT 4  // key ranges per split unit at most (swept: 2..8)
#endif
static_assert(PK_PREFILL_MAX_SPLIT >= 1 && PK_PREFILL_MAX_SPLIT <= 8, "combine merges <= 8 parts");
// Tail split plan: the units of the last, partial round of the grid (one CTA
// per SM) are cut into `split` key ranges so that round fills the SMs.
struct SplitPlan {
  int units, full_units, split;
};
SplitPlan split_plan(int B, int H, int Lq) {
  SplitPlan p;
  const int gx = (Lq + 2 * kTileM - 1) / (2 * kTileM);
  p.units = gx * H * B;
  p.full_units = p.units;
  p.split = 1;
  const int nsm = sm_count();
  if (nsm <= 0 || p.units <= nsm) return p;
  const int rem = p.units % nsm;
  if (rem == 0) return p;
  const int s = min(PK_PREFILL_MAX_SPLIT, nsm / rem);
  if (s < 2) return p;
  p.full_units = p.units - rem;
  p.split = s;
  return p;
}

template <int D, int BS>
cudaError_t launch_prefill_t(const PrefillArgs& a_in, const void* k_cache, const void* v_cache,
                             cudaStream_t stream) {
  using C = PfCfg<D>;
  PrefillArgs a = a_in;
  a.k_cache = reinterpret_cast<const __half*>(k_cache);
  a.v_cache = reinterpret_cast<const __half*>(v_cache);
  a.gx = (a.Lq + 2 * kTileM - 1) / (2 * kTileM);
  SplitPlan plan = split_plan(a.B, a.H, a.Lq);
  const size_t need = (size_t)(plan.units - plan.full_units) * plan.split * (2 * kTileM) *
                      C::PARTIAL_STRIDE;
  if (plan.split > 1 && (a.ws == nullptr || a.ws_floats < need)) {
    plan.full_units = plan.units;  // no workspace: every unit whole
    plan.split = 1;
  }
  a.full_units = plan.full_units;
  a.split = plan.split;
  CUtensorMap qmap, kmap, vmap, omap;
  const long long rows = (long long)a.num_blocks * BS;
  cudaError_t e;
  {
    unsigned long long dims[3] = {(unsigned long long)D, (unsigned long long)a.Lq,
                                  (unsigned long long)a.B * a.H};
    unsigned long long strides[2] = {(unsigned long long)D * 2,
                                     (unsigned long long)a.Lq * D * 2};
    unsigned box[3] = {64, kTileM, 1};
    e = make_map_3d(&qmap, a.q, dims, strides, box, true);
    if (e != cudaSuccess) return e;
    e = make_map_3d(&omap, a.out, dims, strides, box, true);  // same layout as q
    if (e != cudaSuccess) return e;
  }
  memset(&kmap, 0, sizeof(kmap));  // unused by the cp.async gather of 4-token blocks
  memset(&vmap, 0, sizeof(vmap));
  if constexpr (BS >= 8) {
    // The pool as rows r = slot * H + head of D fp16, and inside a block
    // (rows r, r + H, ..., r + (BS-1) H from its first slot) the box order
    // (64 dims, 8 keys, D/64 halves, BS/8 key groups).
    const unsigned long long row = (unsigned long long)D * 2, tok = row * a.H;
    unsigned long long dims[5] = {64, 8, (unsigned long long)C::HALVES,
                                  (unsigned long long)BS / 8, (unsigned long long)rows * a.H};
    unsigned long long strides[4] = {tok, 128, 8 * tok, row};
    unsigned box[5] = {64, 8, (unsigned)C::HALVES, (unsigned)BS / 8, 1};
    e = make_map_5d(&kmap, k_cache, dims, strides, box, true);
    if (e != cudaSuccess) return e;
    e = make_map_5d(&vmap, v_cache, dims, strides, box, true);
    if (e != cudaSuccess) return e;
  }
  constexpr auto kern = prefill_kernel<D, BS>;
  e = ensure_dynamic_smem<kern>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.full_units + (plan.units - plan.full_units) * plan.split);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, qmap, kmap, vmap, omap, a);
  if (e != cudaSuccess || plan.split == 1) return e;
  const int n_split = plan.units - plan.full_units;
  cudaLaunchConfig_t cc = {};
  cc.gridDim = dim3((n_split * 2 * kTileM * 32 + 255) / 256);
  cc.blockDim = dim3(256);
  cc.stream = stream;
  cc.attrs = attr;
  cc.numAttrs = 1;
  return cudaLaunchKernelEx(&cc, prefill_combine_kernel<D>, a, n_split);
}

}  // namespace

size_t prefill_workspace_bytes(int B, int H, int Lq, int D) {
  if (B <= 0 || H <= 0 || Lq <= 0 || (D != 64 && D != 128)) return 0;
  const SplitPlan p = split_plan(B, H, Lq);
  return (size_t)(p.units - p.full_units) * p.split * (2 * kTileM) * (D + 4) * sizeof(float);
}

bool prefill_supported(int D, int block_size) {
  return (D == 64 || D == 128) &&
         (block_size == 4 || block_size == 8 || block_size == 16 || block_size == 32);
}

cudaError_t launch_prefill(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                           cudaStream_t stream) {
  if (a.H > 65535 || a.B > 65535) return cudaErrorInvalidValue;
#define PK_PF_CASE(DD, BB) \
  if (a.D == DD && a.block_size == BB) return launch_prefill_t<DD, BB>(a, k_cache, v_cache, stream);
  PK_PF_CASE(128, 16) PK_PF_CASE(128, 32) PK_PF_CASE(128, 8) PK_PF_CASE(128, 4)
  PK_PF_CASE(64, 16) PK_PF_CASE(64, 32) PK_PF_CASE(64, 8) PK_PF_CASE(64, 4)
#undef PK_PF_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pk
