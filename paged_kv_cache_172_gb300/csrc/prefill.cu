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
// it walks the visible keys in tiles of 128 (8 blocks of 16 or 4 of 32):
//   warps 0-3   softmax of tile A, one query row per thread (TMEM lane = row);
//   warps 4-7   softmax of tile B;
//   warp 8      TMA producer: Q (4 boxes of 128 rows x 64 dims, 128-byte
//               swizzle), then per key tile one box per (block, 64-dim half)
//               for K and for V, gathered through the block table, into a
//               5-stage ring shared by both Q tiles (two key tiles ahead);
//   warp 9      MMA issuer (one thread) and tensor-memory owner, in ping-pong
//               order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): while one tile's
//               softmax runs the tensor core works on the other tile.
// Tensor memory: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512);
// P_X (fp16 pairs packed per 32-bit column) overwrites the first 64 columns
// of S_X once the softmax holds S_X in registers, and the P V MMA reads it
// from tensor memory.  Because tcgen05 operations of one thread complete in
// issue order, "S_X(j+1) done" implies "P_X(j) V_j done": the softmax may
// then rescale O_X without any further barrier.
// Softmax per tile: two tensor-memory round trips over the S row, one for
// the row max (keys past the row's position skipped on diagonal tiles), one
// for p = 2^(s*scale*log2e - m) (one FMA and one ex2 per element); between
// them the output accumulator is rescaled, only when the row max grew by more
// than 2^8 (P then stays <= 256, exact in fp16 range).  The row is summed and
// P (fp16) stored to tensor memory.
// Operand layouts (tcgen05 shared-memory descriptors, 128-byte swizzle):
//   Q, K_j      : K-major, rows of 64 fp16 (128 B), 8-row atoms 1024 B apart,
//                 the two 64-element halves 16 KB apart;
//   V_j         : MN-major (dims contiguous): 8-key atoms 1024 B apart along
//                 K, the two 64-dim halves 16 KB apart along N.
#include "pk_common.cuh"
#include "pk_internal.h"
#include "pk_tcgen05.cuh"

namespace pk {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kTileM = 128;                  // queries per Q tile (two per CTA)
constexpr int kTileN = 128;                  // keys per tile
constexpr int kD = 128;                      // head dim
constexpr int kSlabBytes = 128 * 128;        // 128 rows x 64 fp16
constexpr int kTileBytes = 2 * kSlabBytes;   // 128 rows x 128 fp16
constexpr int kStages = 5;                   // K/V ring (K and V tiles alternate)
constexpr int kThreads = 320;                // 8 softmax warps + producer + MMA
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kTblWindow = 256;              // block-table entries staged in smem
constexpr int kTmemCols = 512;
constexpr uint32_t kColO = 256;

constexpr int kOffQ = 0;                                // Q_A, Q_B
constexpr int kOffKV = kOffQ + 2 * kTileBytes;
constexpr int kOffBar = kOffKV + kStages * kTileBytes;
constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 2 + 1;
constexpr int kOffTmemHolder = kOffBar + kNumBars * 8;
constexpr int kOffTbl = (kOffTmemHolder + 4 + 15) / 16 * 16;
constexpr int kSmemBytes = kOffTbl + kTblWindow * 4 + 1024;  // + alignment slack

constexpr uint32_t kIdescS = tc::idesc_f16_f32(kTileM, kTileN, false, false);
constexpr uint32_t kIdescO = tc::idesc_f16_f32(kTileM, kD, false, true);

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_addr, int kk) {
  // K step kk (16 elements = 32 B) inside the 64-element half kk / 4.
  return tc::smem_desc(tile_addr + (kk >> 2) * kSlabBytes + (kk & 3) * 32, 16, 1024,
                       tc::kSwizzle128B);
}

__device__ __forceinline__ uint64_t vmn_desc(uint32_t tile_addr, int kk) {
  // keys 16*kk .. 16*kk+15: two 8-key atoms starting 2048 B * kk into the tile.
  return tc::smem_desc(tile_addr + kk * 2048, kSlabBytes, 1024, tc::kSwizzle128B);
}

template <int BS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  constexpr int BPT = kTileN / BS;  // blocks per key tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint8_t* sQ = smem + kOffQ;
  uint8_t* sKV = smem + kOffKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;  // [2]: per Q tile
  uint64_t* p_full = s_full + 2;          // [2]
  uint64_t* o_done = p_full + 2;          // [2]
  uint64_t* drain = o_done + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffTmemHolder);
  int32_t* tbl_s = reinterpret_cast<int32_t*>(smem + kOffTbl);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ct = blockIdx.x, h = blockIdx.y, b = blockIdx.z;

  pdl_wait();  // inputs may come from the previous kernel on the stream
  const int n = a.context_lens[b];
  const int q0 = ct * 2 * kTileM;
  const int rows_all = min(2 * kTileM, a.Lq - q0);
  const size_t out_row0 = ((size_t)b * a.H + h) * a.Lq + q0;
  if (n < a.Lq || n > a.max_blocks * BS) {
    if (threadIdx.x == 0) flag_status(a.status, PA_DEV_BAD_CONTEXT);
    uint4* o4 = reinterpret_cast<uint4*>(a.out + out_row0 * kD);
    for (int i = threadIdx.x; i < rows_all * (kD / 8); i += kThreads)
      o4[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  // Per Q tile (A = 0, B = 1): rows, sequence position of row 0, key tiles.
  const int rows_a = min(kTileM, a.Lq - q0);
  const int rows_b = max(0, min(kTileM, a.Lq - (q0 + kTileM)));
  const int pos0_a = n - a.Lq + q0;
  const int pos0_b = pos0_a + kTileM;
  const int ntile_a = (pos0_a + rows_a - 1) / kTileN + 1;
  const int ntile_b = rows_b > 0 ? (pos0_b + rows_b - 1) / kTileN + 1 : 0;
  const int n_kv = max(ntile_a, ntile_b);
  const int nblk_seq = (n + BS - 1) / BS;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
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
  int issued = 0;  // K/V tiles the producer issued into the ring

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ TMA producer
    int win = -kTblWindow;
    if (lane == 0) {
      const int bh = b * a.H + h;
      mbar_arrive_expect_tx(q_full, 2 * kTileBytes);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        tma_load_3d(sQ + x * kTileBytes, &qmap, 0, q0 + x * kTileM, bh, q_full);
        tma_load_3d(sQ + x * kTileBytes + kSlabBytes, &qmap, 64, q0 + x * kTileM, bh, q_full);
      }
    }
    for (int j = 0; j < n_kv && ok; ++j) {
      const int lb0 = j * BPT;
      if (lb0 + BPT > win + kTblWindow) {
        win = lb0;
        __syncwarp();
        for (int i = lane; i < kTblWindow; i += 32) {
          const int lb = win + i;
          int phys = a.num_blocks;  // past the sequence: outside the map, TMA fills zeros
          if (lb < nblk_seq) {
            phys = a.block_tables[(size_t)b * a.max_blocks + lb];
            if (phys < 0 || phys >= a.num_blocks) {
              flag_status(a.status, PA_DEV_BAD_BLOCK_ID);
              phys = a.num_blocks;
            }
          }
          tbl_s[i] = phys;
        }
        __syncwarp();
      }
      for (int half = 0; half < 2 && ok; ++half) {  // K tile, then V tile
        const int u = 2 * j + half;
        const int st = u % kStages;
        if (lane == 0) {
          ok = mbar_wait(&kv_empty[st], ((u / kStages) & 1) ^ 1);
          if (ok) {
            uint8_t* dst = sKV + st * kTileBytes;
            const CUtensorMap* map = half ? &vmap : &kmap;
            mbar_arrive_expect_tx(&kv_full[st], kTileBytes);
#pragma unroll
            for (int i = 0; i < BPT; ++i) {
              const int row = tbl_s[lb0 - win + i] * BS;
              tma_load_3d(dst + i * BS * 128, map, 0, h, row, &kv_full[st]);
              tma_load_3d(dst + kSlabBytes + i * BS * 128, map, 64, h, row, &kv_full[st]);
            }
            ++issued;
          }
        }
        ok = __shfl_sync(kFull, ok, 0);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t kv_addr = smem_u32(sKV);
      // S_X(j) = Q_X K_j^T; releases K_j when X is its last user.
      auto issue_s = [&](int x, int j, bool release) -> bool {
        const int u = 2 * j;
        const int st = u % kStages;
        if (!mbar_wait(&kv_full[st], (u / kStages) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t qa = q_addr + x * kTileBytes;
        const uint32_t kb = kv_addr + st * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          tc::mma_f16(tmem + x * kTileN, kmajor_desc(qa, kk), kmajor_desc(kb, kk), kIdescS,
                      kk > 0);
        tc::commit(&s_full[x]);
        if (release) tc::commit(&kv_empty[st]);
        return true;
      };
      // O_X += P_X V_j once the softmax of X has written P_X for tile j.
      auto issue_pv = [&](int x, int j, int ntile) -> bool {
        if (!mbar_wait(&p_full[x], j & 1)) return false;
        const int u = 2 * j + 1;
        const int st = u % kStages;
        if (!mbar_wait(&kv_full[st], (u / kStages) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t vb = kv_addr + st * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)  // P columns: 16 keys = 8 packed columns
          tc::mma_f16_ts(tmem + kColO + x * kD, tmem + x * kTileN + kk * 8, vmn_desc(vb, kk),
                         kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        if (j == ntile - 1) tc::commit(&o_done[x]);
        return true;
      };
      ok = mbar_wait(q_full, 0);
      if (ok) {
        tc::fence_after_sync();
        ok = issue_s(0, 0, ntile_b == 0);
        if (ok && ntile_b > 0) ok = issue_s(1, 0, true);
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        if (j < ntile_a && !(ok = issue_pv(0, j, ntile_a))) break;
        if (j + 1 < ntile_a && !(ok = issue_s(0, j + 1, j + 1 >= ntile_b))) break;
        if (j < ntile_b && !(ok = issue_pv(1, j, ntile_b))) break;
        tc::commit(&kv_empty[(2 * j + 1) % kStages]);  // V_j has no further reader
        if (j + 1 < ntile_b && !(ok = issue_s(1, j + 1, true))) break;
      }
    }
    ok = __shfl_sync(kFull, ok, 0);
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;       // Q tile of this warpgroup
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_s = tmem + t_lane + x * kTileN;
    const uint32_t t_o = tmem + t_lane + kColO + x * kD;
    const int pos0 = x ? pos0_b : pos0_a;
    const int pos = pos0 + row;
    const int ntile = x ? ntile_b : ntile_a;
    const int rows = x ? rows_b : rows_a;
    const float sl2 = a.scale_log2;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < ntile && ok; ++j) {
      if (!(ok = __all_sync(kFull, mbar_wait(&s_full[x], j & 1)))) break;
      tc::fence_after_sync();
      const int kbase = j * kTileN;
      const bool diag = kbase + kTileN - 1 > pos0;  // some key here is past some row
      // Row max: the whole S row in one tensor-memory round trip (4 loads, one
      // wait); keys past this row's position are skipped on diagonal tiles.
      float mx[8];
      {
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::ld_32x32(t_s + c * 32, r[c]);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
        if (diag) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (kbase + c * 32 + i <= pos) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(r[c][i]));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(r[c][i]));
        }
      }
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
      const float m_new = fmaxf(m, mt);
      const bool resc = m_new > m + 8.0f;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m - m_new);
        m = m_new;
        l *= alpha;
      }
      if (j > 0 && __any_sync(kFull, resc)) {
        // S_X(j) has completed, hence so has P_X(j-1) V_{j-1}: rescale O_X.
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tc::ld_32x32(t_o + c * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tc::st_32x32(t_o + c * 32, o);
        }
        tc::wait_st();
      }
      // P = 2^(s * scale * log2e - m) in fp16, row sum: S reloaded 32 columns
      // at a time, P stored over the first 64 columns of S_X.
      const float neg_m = -m;
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 32 keys -> 16 packed columns per store
        uint32_t r[32];
        tc::ld_32x32(t_s + c * 32, r);
        tc::wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int i0 = 2 * e;
          float p0 = ex2_approx(fmaf(__uint_as_float(r[i0]), sl2, neg_m));
          float p1 = ex2_approx(fmaf(__uint_as_float(r[i0 + 1]), sl2, neg_m));
          if (diag) {
            if (kbase + c * 32 + i0 > pos) p0 = 0.f;
            if (kbase + c * 32 + i0 + 1 > pos) p1 = 0.f;
          }
          rs[e & 3] += p0 + p1;
          __half2 hp = __floats2half2_rn(p0, p1);
          pk[e] = *reinterpret_cast<uint32_t*>(&hp);
        }
        // P columns [16c, 16c+16) lie below S columns [32c, ...) not yet read.
        tc::st_32x16(t_s + c * 16, pk);
      }
      tc::wait_st();
      l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      tc::fence_before_sync();
      mbar_arrive(&p_full[x]);
    }
    if (ok && ntile > 0) ok = __all_sync(kFull, mbar_wait(&o_done[x], 0));
    if (ok && ntile > 0) {
      tc::fence_after_sync();
      const float inv = 1.f / l;
      __half* orow = a.out + (out_row0 + x * kTileM + row) * kD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tc::ld_32x32(t_o + c * 32, o);
        tc::wait_ld();
        uint32_t hv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          __half2 t = __floats2half2_rn(__uint_as_float(o[2 * i]) * inv,
                                        __uint_as_float(o[2 * i + 1]) * inv);
          hv[i] = *reinterpret_cast<uint32_t*>(&t);
        }
        if (row < rows) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
        }
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
    if (warp == kWarpMma && lane == 0) {
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

template <int BS>
cudaError_t launch_prefill_t(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                             cudaStream_t stream) {
  CUtensorMap qmap, kmap, vmap;
  const long long rows = (long long)a.num_blocks * BS;
  cudaError_t e;
  {
    unsigned long long dims[3] = {(unsigned long long)kD, (unsigned long long)a.Lq,
                                  (unsigned long long)a.B * a.H};
    unsigned long long strides[2] = {(unsigned long long)kD * 2,
                                     (unsigned long long)a.Lq * kD * 2};
    unsigned box[3] = {64, kTileM, 1};
    e = make_map_3d(&qmap, a.q, dims, strides, box, true);
    if (e != cudaSuccess) return e;
  }
  {
    unsigned long long dims[3] = {(unsigned long long)kD, (unsigned long long)a.H,
                                  (unsigned long long)rows};
    unsigned long long strides[2] = {(unsigned long long)kD * 2,
                                     (unsigned long long)a.H * kD * 2};
    unsigned box[3] = {64, 1, (unsigned)BS};
    e = make_map_3d(&kmap, k_cache, dims, strides, box, true);
    if (e != cudaSuccess) return e;
    e = make_map_3d(&vmap, v_cache, dims, strides, box, true);
    if (e != cudaSuccess) return e;
  }
  auto kern = prefill_kernel<BS>;
  static bool attr_done = false;
  if (!attr_done) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.Lq + 2 * kTileM - 1) / (2 * kTileM), a.H, a.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, qmap, kmap, vmap, a);
}

}  // namespace

bool prefill_supported(int D, int block_size) {
  return D == kD && (block_size == 16 || block_size == 32);
}

cudaError_t launch_prefill(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                           cudaStream_t stream) {
  if (a.H > 65535 || a.B > 65535) return cudaErrorInvalidValue;
  if (a.block_size == 16) return launch_prefill_t<16>(a, k_cache, v_cache, stream);
  if (a.block_size == 32) return launch_prefill_t<32>(a, k_cache, v_cache, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pk
