// Grouped GEMM on CTA pairs: one tcgen05 MMA of M = 256 weight rows spans two
// SMs (cta_group::2). Each CTA of a cluster pair stages its own 128 weight rows
// and half of the token rows, and keeps its 128 accumulator lanes in its own
// TMEM. So each SM stages fewer bytes per FLOP than in moe_gemm_tc: 131 FLOPs
// per byte with 256-token tiles, with the accumulator double-buffered.
//
//   plain mode (GEMM2): the pair's 256 rows are 256 consecutive output rows.
//                       Optionally the epilogue writes token column p to out
//                       row out_rows[p], times out_scale[p] (the weighted
//                       un-permute of an EP expert rank).
//   SiLU mode (GEMM1):  a pair tile covers 128 intermediate indices. Each CTA
//                       stages 64 gate rows and the 64 up rows of the same
//                       indices (two 64-row boxes), so its accumulator holds
//                       gate in lanes 0..63 and up in lanes 64..127. The warps
//                       on the up lanes pass their values through shared
//                       memory to the warps on the gate lanes, in 32-column
//                       chunks over two slots; those apply SiLU(gate)*up and
//                       store. Both CTAs store half of the pair's outputs.
//
// Roles per CTA (persistent, 320 threads), as in moe_gemm_tc:
//   warp 0      TMA producer of this CTA's rows. The bytes of both CTAs are
//               counted on rank 0's full barrier (rank 0 declares them).
//   warp 1      TMEM allocation (both CTAs, cta_group::2). On rank 0 also the
//               MMA issuer. Its commits arrive on the stage-free and
//               accumulator-full barriers of both CTAs.
//   warps 2..9  epilogue on this CTA's 128 accumulator lanes (two warps per
//               lane quarter, each on one 16-column half of a 32-column
//               chunk). Each warp then arrives once on rank 0's
//               accumulator-free barrier.
// Work units (one 256-row pair tile x one token tile) are ordered as in
// moe_gemm_tc: expert by expert.
#include <cuda_bf16.h>

#include "act.cuh"
#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
[[maybe_unused]] constexpr DbgFile kDbgFileCode = kDbgGemmPair;
namespace {

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kABytes = 128 * 128;
constexpr int kChunk = 32;                       // columns per SiLU exchange chunk
constexpr int kHalfCols = kChunk / 2;            // columns of a chunk per epilogue warp
constexpr int kXSlotBytes = 64 * kChunk * 4;     // one chunk of up values, fp32

// A pipeline stage holds KPS consecutive K blocks (128 bytes of K each): one
// SM's TMA engine completes stages at a roughly fixed rate whatever their size
// (measured: ~2 per us), so its throughput grows with the bytes per stage,
// not with the number of stages in flight.
template <int MODE, int NMAX, int KPS>
struct PairShape {
  static constexpr int kBRows = NMAX / 2;  // token rows staged per CTA
  static constexpr int kBBytes = kBRows * 128;
  static constexpr int kSubBytes = kABytes + kBBytes;  // one K block: A, then B
  static constexpr int kStageBytes = KPS * kSubBytes;
  static constexpr int kXBytes = (MODE == kGemmSiluUp) ? 2 * kXSlotBytes : 0;
  // output staging: per column half, two buffers of 16 token rows of this
  // CTA's output columns (64 of h in SiLU mode, 128 of y in plain mode)
  static constexpr int kOutRowBytes = (MODE == kGemmSiluUp) ? 64 * 2 : 128 * 2;
  static constexpr int kOutBufBytes = 16 * kOutRowBytes;
  static constexpr int kOutBytes = 2 * 2 * kOutBufBytes;
  static constexpr int kStages0 = (216 * 1024 - kXBytes - kOutBytes) / kStageBytes;
  static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
  static constexpr int kAccCols = NMAX;
  static constexpr int kNAcc = 2;
  static constexpr int kTmemCols = kAccCols * kNAcc <= 256 ? 256 : 512;
  static constexpr int kMaxGroups = 1024;
  // + xfull[2], xempty[2], ofull[2 halves][2 buffers]
  static constexpr int kNBars = 2 * kStages + 2 * kNAcc + 1 + 4 + 4;
  static constexpr int kBarBytes = 8 * kNBars + 16 + 4 * (kMaxGroups + 1);
  static constexpr int kSmemBytes =
      1024 + kStages * kStageBytes + kXBytes + kOutBytes + kBarBytes;
  static_assert(kAccCols * kNAcc <= 512, "TMEM overflow");
  static_assert(kStages >= 2, "need at least two stages");
  static_assert(NMAX % 32 == 0 && NMAX <= 256, "bad NMAX");
};


__device__ __forceinline__ void decode_unit(int u, const int* gstart, int n_groups, int m_tiles,
                                            int& tile, int& m) {
  int lo = 0, hi = n_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (gstart[mid] * m_tiles <= u) lo = mid;
    else hi = mid - 1;
  }
  const int n = gstart[lo + 1] - gstart[lo];
  const int r = u - gstart[lo] * m_tiles;
  m = r / n;
  tile = gstart[lo] + (r - m * n);
}

// Spin for about `ns` of %globaltimer (lets in-flight copies land when a
// kernel unwinds after a timeout).
__device__ __forceinline__ void settle(uint64_t ns) {
  const uint64_t t0 = ptx::globaltimer();
  while (ptx::globaltimer() - t0 < ns) {
  }
}

template <int MODE, int NMAX, int KPS>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_pair(const __grid_constant__ CUtensorMap mapA,
                  const __grid_constant__ CUtensorMap mapB, const Tile* __restrict__ tiles,
                  const int* __restrict__ group_start, int n_groups, int dense_T, int m_tiles,
                  int k_blocks, int a_rows_per_expert, int a_up_offset, int b_from_out,
                  __nv_bfloat16* __restrict__ out, long out_ld,
                  const int32_t* __restrict__ out_rows, const float* __restrict__ out_scale,
                  int b_cap, unsigned* status, const GemmBounds bnd) {
  using S = PairShape<MODE, NMAX, KPS>;
  const int n_st = k_blocks / KPS;  // stages per unit (k_blocks is a multiple of KPS)
  const uint32_t rank = ptx::cluster_rank();
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  // Dense problems (shared experts: every token of dense_T for each of
  // n_groups weight slabs) pass no tile table; their tiles are implicit.
  const int dense_per = (dense_T + NMAX - 1) / NMAX;
  const int total = (tiles ? group_start[n_groups] : n_groups * dense_per) * m_tiles;
  if (pair >= total) return;  // both CTAs of the pair leave together

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t xbase = sbase + S::kStages * S::kStageBytes;  // SiLU exchange slots
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + S::kStages * S::kStageBytes + S::kXBytes + S::kOutBytes);
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S::kStages;
  const uint32_t tfull0 = empty0 + 8 * S::kStages;
  const uint32_t tempty0 = tfull0 + 8 * S::kNAcc;
  const uint32_t drain = tempty0 + 8 * S::kNAcc;
  const uint32_t xfull0 = drain + 8;     // the up warps wrote a chunk
  const uint32_t xempty0 = xfull0 + 16;  // the gate warps consumed a chunk
  const uint32_t ofull0 = xempty0 + 16;  // [half][buffer]: a chunk's outputs are staged
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + S::kNBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* gstart = reinterpret_cast<int*>(tmem_slot + 4);
  for (int i = threadIdx.x; i <= n_groups; i += kThreads)
    gstart[i] = tiles ? group_start[i] : i * dense_per;
  auto tile_at = [&](int ti) -> Tile {
    if (tiles) return tiles[MOE_DCHECK(ti, bnd.max_tiles) ? ti : 0];
    const int sl = ti / dense_per, t0 = (ti - sl * dense_per) * NMAX;
    return make_int4(sl, t0, sl * dense_T + t0, min(NMAX, dense_T - t0));
  };
  // A tile table entry every role can act on: a valid width and, when the
  // row count b_cap of the position space is given, rows inside it. Every
  // role skips the same entries (and flags them), so their pipelines stay
  // in step. The debug build also checks the entry against the buffers'
  // extents.
  auto tile_ok = [&](const Tile& tl) {
    return tl.w >= 1 && tl.w <= NMAX && tl.x >= 0 && tl.y >= 0 && tl.z >= 0 &&
           (b_cap <= 0 || (tl.y <= b_cap - tl.w && tl.z <= b_cap - tl.w)) &&
           MOE_DCHECK(tl.x, n_groups) &&
           MOE_DCHECK(b_from_out ? tl.z : tl.y, bnd.b_rows - tl.w + 1) &&
           MOE_DCHECK(tl.z, (out_rows ? bnd.out_map : bnd.out_rows) - tl.w + 1);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);   // rank 0's producer expects both CTAs' bytes
      ptx::mbar_init(empty0 + 8 * s, 1);  // the pair MMA commit
    }
    for (int b = 0; b < S::kNAcc; ++b) {
      ptx::mbar_init(tfull0 + 8 * b, 1);
      ptx::mbar_init(tempty0 + 8 * b, 2 * kEpiWarps);  // one per epilogue warp of each CTA
    }
    ptx::mbar_init(drain, 1);
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(xfull0 + 8 * x, kEpiWarps / 2);   // the four up warps
      ptx::mbar_init(xempty0 + 8 * x, kEpiWarps / 2);  // the four gate warps
    }
    // the epilogue warps that stage a half's chunk: two gate warps (SiLU
    // mode) or the four lane-quarter warps (plain mode)
    for (int x = 0; x < 4; ++x)
      ptx::mbar_init(ofull0 + 8 * x, MODE == kGemmSiluUp ? 2 : 4);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async();
    ptx::tma_prefetch_map(&mapA);
    ptx::tma_prefetch_map(&mapB);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), S::kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // barriers of both CTAs exist before any cross-CTA arrive
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t full_r0 = ptx::map_to_rank(full0, 0);  // rank 0's full barriers
      // this CTA's weight rows of unit (tile, m) for K block kb: SiLU mode
      // loads 64 gate and the matching 64 up rows, plain mode 128 rows
      auto load_a = [&](uint32_t dst, uint32_t fb, int kb, const Tile& tl, int m) {
        if constexpr (MODE == kGemmSiluUp) {
          const int g_row = tl.x * a_rows_per_expert + m * 128 + static_cast<int>(rank) * 64;
          ptx::tma_load_2d_pair(dst, &mapA, fb, kb * 64, g_row);
          ptx::tma_load_2d_pair(dst + kABytes / 2, &mapA, fb, kb * 64, g_row + a_up_offset);
        } else {
          ptx::tma_load_2d_pair(dst, &mapA, fb, kb * 64,
                                tl.x * a_rows_per_expert + m * 256 + static_cast<int>(rank) * 128);
        }
      };
      // Operand A (weights) of the first kStages stages before the
      // dependency wait; operand B (token rows) only after it.
      int pre = 0;
      for (int u = pair; u < total && pre < S::kStages; u += n_pairs) {
        int ti, m;
        decode_unit(u, gstart, n_groups, m_tiles, ti, m);
        const Tile tl = tile_at(ti);
        if (!tile_ok(tl)) continue;
        for (int j = 0; j < n_st && pre < S::kStages; ++j, ++pre) {
          if (rank == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * pre, 2 * S::kStageBytes);
#pragma unroll
          for (int p = 0; p < KPS; ++p)
            load_a(sbase + pre * S::kStageBytes + p * S::kSubBytes, full_r0 + 8 * pre,
                   j * KPS + p, tl, m);
        }
      }
      pdl_enter();
      int it = 0;
      bool ok = true;
      for (int u = pair; u < total && ok; u += n_pairs) {
        int ti, m;
        decode_unit(u, gstart, n_groups, m_tiles, ti, m);
        const Tile tl = tile_at(ti);
        if (!tile_ok(tl)) {
          if (rank == 0) atomicOr(status, MOE_DEV_BAD_SEGMENT);
          continue;
        }
        const int n_mma = (tl.w + 31) & ~31;
        const int b_row = (b_from_out ? tl.z : tl.y) + static_cast<int>(rank) * (n_mma >> 1);
        (void)MOE_DCHECK(tl.x * static_cast<long>(a_rows_per_expert) +
                             m * (MODE == kGemmSiluUp ? 128 : 256) +
                             (MODE == kGemmSiluUp ? a_up_offset : 0),
                         bnd.a_rows);
        for (int j = 0; j < n_st; ++j, ++it) {
          const int s = it % S::kStages;
          const uint32_t ph = (it / S::kStages) & 1;
          const uint32_t st = sbase + s * S::kStageBytes;
          const uint32_t fb = full_r0 + 8 * s;
          if (it >= pre) {  // stages of the early loads are fresh: no empty wait
            if (!ptx::mbar_wait_cluster(empty0 + 8 * s, ph ^ 1, abort_flag, status)) {
              ok = false;
              break;
            }
            // Rank 0 declares the bytes of both CTAs on its own barrier; the
            // peer's copies only complete transactions on it. The peer loads
            // stage s again only after rank 0's MMAs freed it, so its bytes
            // never land in an older phase.
            if (rank == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * s, 2 * S::kStageBytes);
#pragma unroll
            for (int p = 0; p < KPS; ++p) load_a(st + p * S::kSubBytes, fb, j * KPS + p, tl, m);
          }
#pragma unroll
          for (int p = 0; p < KPS; ++p)
            ptx::tma_load_2d_pair(st + p * S::kSubBytes + kABytes, &mapB, fb,
                                  (j * KPS + p) * 64, b_row);
        }
      }
      if (!ok) settle(200000);
    } else {
      pdl_enter();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    pdl_enter();
    if (lane == 0 && rank == 0) {
      int it = 0, ai = 0;
      bool ok = true;
      for (int u = pair; u < total && ok; u += n_pairs) {
        int ti, m;
        decode_unit(u, gstart, n_groups, m_tiles, ti, m);
        const Tile tl = tile_at(ti);
        if (!tile_ok(tl)) continue;
        const int n_mma = (tl.w + 31) & ~31;
        const uint32_t idesc = ptx::idesc_make(1u, 256, n_mma);
        const int b = ai % S::kNAcc;
        const uint32_t aph = (ai / S::kNAcc) & 1;
        if (!ptx::mbar_wait_cluster(tempty0 + 8 * b, aph ^ 1, abort_flag, status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + b * S::kAccCols;
        for (int j = 0; j < n_st; ++j, ++it) {
          const int s = it % S::kStages;
          const uint32_t ph = (it / S::kStages) & 1;
          if (!ptx::mbar_wait_cluster(full0 + 8 * s, ph, abort_flag, status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int p = 0; p < KPS; ++p) {
            const uint32_t st = sbase + s * S::kStageBytes + p * S::kSubBytes;
            const uint64_t da = ptx::sdesc_sw128(st);
            const uint64_t db = ptx::sdesc_sw128(st + kABytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::tc_mma_pair(d, da + 2 * kk, db + 2 * kk, idesc, (j | p | kk) ? 1u : 0u);
          }
          ptx::tc_commit_pair(empty0 + 8 * s);
        }
        if (!ok) break;
        ptx::tc_commit_pair(tfull0 + 8 * b);
        ++ai;
      }
      if (!ok) {
        ptx::tc_commit_pair(drain);
        ptx::mbar_wait_drain(drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Each 16-column piece of the accumulator goes through a staging buffer
    // in shared memory, so that the global stores are whole 16-byte vectors
    // along output rows instead of 2-byte values down a column.
    pdl_enter();
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t tempty_r0 = ptx::map_to_rank(tempty0, 0);
    const int row_l = q * 32 + lane;  // accumulator lane of this thread
    uint8_t* const stg =
        smem + S::kStages * S::kStageBytes + S::kXBytes + half * 2 * S::kOutBufBytes;
    const uint32_t ofull = ofull0 + 16 * half;
    int ai = 0, cc = 0;
    bool ok = true;
    for (int u = pair; u < total && ok; u += n_pairs) {
      int ti, m;
      decode_unit(u, gstart, n_groups, m_tiles, ti, m);
      const Tile tl = tile_at(ti);
      if (!tile_ok(tl)) continue;
      const int b = ai % S::kNAcc;
      const uint32_t aph = (ai / S::kNAcc) & 1;
      if (!ptx::mbar_wait_cluster(tfull0 + 8 * b, aph, abort_flag, status)) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + b * S::kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (MODE == kGemmSiluUp) {
        // lanes 0..63: gate, 64..127: up, of the CTA's 64 intermediate indices
        const bool up_warp = q >= 2;
        const int r64 = (q & 1) * 32 + lane;
        const long h_col0 = static_cast<long>(m) * 128 + static_cast<int>(rank) * 64;
        for (int c0 = 0; c0 < tl.w; c0 += kChunk, ++cc) {
          const int slot = cc & 1;
          const uint32_t xph = (cc >> 1) & 1;
          const int col = c0 + kHalfCols * half;
          // slot layout [column group of 4][row of 64][4 floats]: a warp's
          // 16-byte accesses cover 512 contiguous bytes, free of bank conflicts
          float4* xs = reinterpret_cast<float4*>(smem + (xbase - sbase) + slot * kXSlotBytes) +
                       (kHalfCols / 4) * half * 64 + r64;
          float v[kHalfCols];
          ptx::tmem_ld16(tb + col, v);
          if (up_warp) {
            if (!ptx::mbar_wait(xempty0 + 8 * slot, xph ^ 1, abort_flag, status)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int j = 0; j < kHalfCols; j += 4)
              xs[(j / 4) * 64] = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(xfull0 + 8 * slot);
            continue;
          }
          if (!ptx::mbar_wait(xfull0 + 8 * slot, xph, abort_flag, status)) {
            ok = false;
            break;
          }
          // staging [16 columns][64 indices] bf16: h of this lane's index
          __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(stg + (cc & 1) * S::kOutBufBytes);
#pragma unroll
          for (int j = 0; j < kHalfCols; j += 4) {
            const float4 u4 = xs[(j / 4) * 64];
            const float uj[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int t = 0; t < 4; ++t)
              sb[(j + t) * 64 + r64] = __float2bfloat16_rn(silu(v[j + t]) * uj[t]);
          }
          __syncwarp();
          if (lane == 0) {
            ptx::mbar_arrive(xempty0 + 8 * slot);
            ptx::mbar_arrive(ofull + 8 * (cc & 1));
          }
          if (!ptx::mbar_wait(ofull + 8 * (cc & 1), (cc >> 1) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
          // 16 rows of 128 bytes: the two gate warps of this half store 16
          // bytes per lane, 4 rows per warp per pass
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int t = k * 8 + (r64 >> 3);
            if (col + t < tl.w && MOE_DCHECK(h_col0 + (r64 & 7) * 8 + 7, out_ld)) {
              const uint4 val = *reinterpret_cast<const uint4*>(sb + t * 64 + (r64 & 7) * 8);
              *reinterpret_cast<uint4*>(out + static_cast<long>(tl.z + col + t) * out_ld +
                                        h_col0 + (r64 & 7) * 8) = val;
            }
          }
        }
        if (!ok) break;
      } else {
        // columns c0 = 16*half + 32*it of the tile; per piece, staging
        // [16 columns][128 rows] bf16, written out as 16 rows of 256 bytes
        const long y_col0 = static_cast<long>(m) * 256 + static_cast<int>(rank) * 128;
        const int t_out = row_l >> 4;     // this lane's first output row in a piece
        const int c8 = (row_l & 15) * 8;  // and its 8 columns of that row
        // with out_rows: each lane's destination rows and, lane j < 16, the
        // scales of column j of every piece, fetched once per unit
        int dst[8][2];
        float scl[8];
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int c0 = 16 * half + 32 * it;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int t = c0 + k * 8 + t_out;
            dst[it][k] = t < tl.w ? (out_rows ? out_rows[tl.z + t] : tl.z + t) : -1;
            if (dst[it][k] >= 0 && !MOE_DCHECK(dst[it][k], bnd.out_rows)) dst[it][k] = -1;
          }
          scl[it] = (out_scale && (lane & 15) + c0 < tl.w) ? out_scale[tl.z + c0 + (lane & 15)]
                                                           : 1.f;
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int c0 = 16 * half + 32 * it;
          if (c0 >= tl.w) break;
          float v[16];
          ptx::tmem_ld16(tb + c0, v);
          __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(stg + (cc & 1) * S::kOutBufBytes);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float f = __shfl_sync(0xffffffffu, scl[it], j);
            sb[j * 128 + row_l] = __float2bfloat16_rn(v[j] * f);
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(ofull + 8 * (cc & 1));
          if (!ptx::mbar_wait(ofull + 8 * (cc & 1), (cc >> 1) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (dst[it][k] >= 0 && MOE_DCHECK(y_col0 + c8 + 7, out_ld)) {
              const uint4 val =
                  *reinterpret_cast<const uint4*>(sb + (k * 8 + t_out) * 128 + c8);
              *reinterpret_cast<uint4*>(out + static_cast<long>(dst[it][k]) * out_ld + y_col0 +
                                        c8) = val;
            }
          }
          ++cc;
        }
        if (!ok) break;
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(tempty_r0 + 8 * b);
      ++ai;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // no CTA leaves while its peer may still touch its memory
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, S::kTmemCols);
  }
}

template <int MODE, int NMAX, int KPS>
cudaError_t launch_pair_variant(const GemmArgs& a, int num_sms, cudaStream_t st) {
  using S = PairShape<MODE, NMAX, KPS>;
  auto kern = moe_gemm_pair<MODE, NMAX, KPS>;
  static std::atomic<unsigned long long> smem_set{0};  // devices, one bit each
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(kern), S::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((num_sms / 2) * 2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return counted(cudaLaunchKernelEx(&cfg, kern, *a.mapA, *a.mapB, a.tiles, a.group_start, a.n_groups,
                            a.dense_T, a.m_tiles, a.k_blocks, a.a_rows_per_expert, a.a_up_offset,
                            a.b_from_out, static_cast<__nv_bfloat16*>(a.out), a.out_ld,
                            a.out_rows, a.out_scale, a.b_cap, a.status, a.bnd));
}

}  // namespace

cudaError_t launch_gemm_pair(GemmMode mode, int nmax, const GemmArgs& a, int num_sms,
                             cudaStream_t st) {
  if ((a.tiles == nullptr && a.dense_T <= 0) || a.k_split != 1) return cudaErrorInvalidValue;
  if (a.out_rows && mode != kGemmPlain) return cudaErrorInvalidValue;
  if (MOE_DEBUG_BUILD && (a.bnd.a_rows <= 0 || a.bnd.b_rows <= 0 || a.bnd.out_rows <= 0 ||
                          (a.tiles && a.bnd.max_tiles <= 0) || (a.out_rows && a.bnd.out_map <= 0)))
    return cudaErrorInvalidValue;
  const bool two = a.k_blocks % 2 == 0;  // two K blocks per stage when they pair up
  if (nmax == 256 && mode == kGemmPlain)
    return two ? launch_pair_variant<kGemmPlain, 256, 2>(a, num_sms, st)
               : launch_pair_variant<kGemmPlain, 256, 1>(a, num_sms, st);
  if (nmax == 256 && mode == kGemmSiluUp)
    return two ? launch_pair_variant<kGemmSiluUp, 256, 2>(a, num_sms, st)
               : launch_pair_variant<kGemmSiluUp, 256, 1>(a, num_sms, st);
  return cudaErrorInvalidValue;
}

MOE_WAIT_LIMIT_SETTER(set_wait_limit_gemm_pair)
MOE_DEBUG_TAKER(take_dbg_gemm_pair)

}  // namespace moe
