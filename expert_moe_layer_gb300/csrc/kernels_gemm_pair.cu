// Grouped GEMM on CTA pairs: one tcgen05 MMA of M = 256 weight rows spans two
// SMs (cta_group::2). Each CTA of a cluster pair stages its own 128 weight rows
// and half of the token rows, and keeps its 128 accumulator lanes in its own
// TMEM. So each SM stages fewer bytes per FLOP than in moe_gemm_tc: 131 FLOPs
// per byte with 256-token tiles, with the accumulator double-buffered.
//
//   plain mode (GEMM2): the pair's 256 rows are 256 consecutive output rows.
//   SiLU mode (GEMM1):  rank 0 holds 128 gate rows and rank 1 the matching
//                       128 up rows, so the pair computes gate and up for the
//                       same 128 intermediate indices. Rank 1's epilogue sends
//                       its up values to rank 0 over distributed shared memory
//                       in 16-column chunks. Two slots alternate: st.async
//                       completes bytes on rank 0's full barrier, and rank 0
//                       frees a slot with a relaxed arrive. Rank 0 then applies
//                       SiLU(gate)*up and stores.
//
// Roles per CTA (persistent, 320 threads), as in moe_gemm_tc:
//   warp 0      TMA producer of this CTA's rows. The bytes of both CTAs are
//               counted on rank 0's full barrier (rank 0 declares them).
//   warp 1      TMEM allocation (both CTAs, cta_group::2). On rank 0 also the
//               MMA issuer. Its commits arrive on the stage-free and
//               accumulator-full barriers of both CTAs.
//   warps 2..9  epilogue on this CTA's 128 accumulator lanes (two warps per
//               lane quarter: 8 columns each of a 16-column SiLU chunk, or
//               alternate 16-column blocks in plain mode). Each warp
//               then arrives once on rank 0's accumulator-free barrier.
// Work units (one 256-row pair tile x one token tile) are ordered as in
// moe_gemm_tc: expert by expert.
#include <cuda_bf16.h>

#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kABytes = 128 * 128;
constexpr int kChunk = 16;                       // columns per SiLU exchange chunk
constexpr int kHalfCols = kChunk / 2;            // columns of a chunk per epilogue warp
constexpr int kXSlotBytes = 128 * kChunk * 4;    // one chunk of up values, fp32

template <int MODE, int NMAX>
struct PairShape {
  static constexpr int kBRows = NMAX / 2;  // token rows staged per CTA
  static constexpr int kBBytes = kBRows * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kXBytes = (MODE == kGemmSiluUp) ? 2 * kXSlotBytes : 0;
  static constexpr int kStages0 = (216 * 1024 - kXBytes) / kStageBytes;
  static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
  static constexpr int kAccCols = NMAX;
  static constexpr int kNAcc = 2;
  static constexpr int kTmemCols = kAccCols * kNAcc <= 256 ? 256 : 512;
  static constexpr int kMaxGroups = 1024;
  static constexpr int kNBars = 2 * kStages + 2 * kNAcc + 1 + 4;  // + xfull[2], xempty[2]
  static constexpr int kBarBytes = 8 * kNBars + 16 + 4 * (kMaxGroups + 1);
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kXBytes + kBarBytes;
  static_assert(kAccCols * kNAcc <= 512, "TMEM overflow");
  static_assert(kStages >= 2, "need at least two stages");
  static_assert(NMAX % 32 == 0 && NMAX <= 256, "bad NMAX");
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

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

template <int MODE, int NMAX>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_pair(const __grid_constant__ CUtensorMap mapA,
                  const __grid_constant__ CUtensorMap mapB, const Tile* __restrict__ tiles,
                  const int* __restrict__ group_start, int n_groups, int dense_T, int m_tiles,
                  int k_blocks, int a_rows_per_expert, int a_up_offset, int b_from_out,
                  __nv_bfloat16* __restrict__ out, long out_ld, unsigned* status) {
  using S = PairShape<MODE, NMAX>;
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
      reinterpret_cast<uint64_t*>(smem + S::kStages * S::kStageBytes + S::kXBytes);
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S::kStages;
  const uint32_t tfull0 = empty0 + 8 * S::kStages;
  const uint32_t tempty0 = tfull0 + 8 * S::kNAcc;
  const uint32_t drain = tempty0 + 8 * S::kNAcc;
  const uint32_t xfull0 = drain + 8;     // on rank 0: rank 1 wrote a chunk
  const uint32_t xempty0 = xfull0 + 16;  // on rank 1: rank 0 consumed a chunk
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + S::kNBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* gstart = reinterpret_cast<int*>(tmem_slot + 4);
  for (int i = threadIdx.x; i <= n_groups; i += kThreads)
    gstart[i] = tiles ? group_start[i] : i * dense_per;
  auto tile_at = [&](int ti) -> Tile {
    if (tiles) return tiles[ti];
    const int sl = ti / dense_per, t0 = (ti - sl * dense_per) * NMAX;
    return make_int4(sl, t0, sl * dense_T + t0, min(NMAX, dense_T - t0));
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
      ptx::mbar_init(xfull0 + 8 * x, 1);          // rank 0 arms it with the chunk's bytes
      ptx::mbar_init(xempty0 + 8 * x, kEpiWarps);
    }
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
      // Operand A (weights) of the first kStages stages before the
      // dependency wait; operand B (token rows) only after it.
      int pre = 0;
      for (int u = pair; u < total && pre < S::kStages; u += n_pairs) {
        int ti, m;
        decode_unit(u, gstart, n_groups, m_tiles, ti, m);
        const Tile tl = tile_at(ti);
        const int a_row =
            MODE == kGemmSiluUp
                ? tl.x * a_rows_per_expert + static_cast<int>(rank) * a_up_offset + m * 128
                : tl.x * a_rows_per_expert + m * 256 + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < k_blocks && pre < S::kStages; ++kb, ++pre) {
          if (rank == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * pre, 2 * S::kStageBytes);
          ptx::tma_load_2d_pair(sbase + pre * S::kStageBytes, &mapA, full_r0 + 8 * pre,
                                kb * 64, a_row);
        }
      }
      pdl_enter();
      int it = 0;
      bool ok = true;
      for (int u = pair; u < total && ok; u += n_pairs) {
        int ti, m;
        decode_unit(u, gstart, n_groups, m_tiles, ti, m);
        const Tile tl = tile_at(ti);
        const int n_mma = (tl.w + 31) & ~31;
        const int b_row = (b_from_out ? tl.z : tl.y) + static_cast<int>(rank) * (n_mma >> 1);
        const int a_row =
            MODE == kGemmSiluUp
                ? tl.x * a_rows_per_expert + static_cast<int>(rank) * a_up_offset + m * 128
                : tl.x * a_rows_per_expert + m * 256 + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < k_blocks; ++kb, ++it) {
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
            ptx::tma_load_2d_pair(st, &mapA, fb, kb * 64, a_row);
          }
          ptx::tma_load_2d_pair(st + kABytes, &mapB, fb, kb * 64, b_row);
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
      for (int u = pair; u < total && ok; u += n_pairs, ++ai) {
        int ti, m;
        decode_unit(u, gstart, n_groups, m_tiles, ti, m);
        const Tile tl = tile_at(ti);
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
        for (int kb = 0; kb < k_blocks; ++kb, ++it) {
          const int s = it % S::kStages;
          const uint32_t ph = (it / S::kStages) & 1;
          if (!ptx::mbar_wait_cluster(full0 + 8 * s, ph, abort_flag, status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t st = sbase + s * S::kStageBytes;
          const uint64_t da = ptx::sdesc_sw128(st);
          const uint64_t db = ptx::sdesc_sw128(st + kABytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::tc_mma_pair(d, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
          ptx::tc_commit_pair(empty0 + 8 * s);
        }
        if (!ok) break;
        ptx::tc_commit_pair(tfull0 + 8 * b);
      }
      if (!ok) {
        ptx::tc_commit_pair(drain);
        ptx::mbar_wait_drain(drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_enter();
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t tempty_r0 = ptx::map_to_rank(tempty0, 0);
    const uint32_t xfull_r0 = ptx::map_to_rank(xfull0, 0);
    const uint32_t xempty_r1 = ptx::map_to_rank(xempty0, 1);
    const int row_l = q * 32 + lane;  // accumulator lane of this thread
    int ai = 0, cc = 0;
    bool ok = true;
    for (int u = pair; u < total && ok; u += n_pairs, ++ai) {
      int ti, m;
      decode_unit(u, gstart, n_groups, m_tiles, ti, m);
      const Tile tl = tile_at(ti);
      const int b = ai % S::kNAcc;
      const uint32_t aph = (ai / S::kNAcc) & 1;
      if (!ptx::mbar_wait_cluster(tfull0 + 8 * b, aph, abort_flag, status)) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + b * S::kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (MODE == kGemmSiluUp) {
        const int i = m * 128 + row_l;
        __nv_bfloat16* orow = out + static_cast<long>(tl.z) * out_ld + i;
        for (int c0 = 0; c0 < tl.w; c0 += kChunk, ++cc) {
          const int slot = cc & 1;
          const uint32_t xph = (cc >> 1) & 1;
          const int col = c0 + kHalfCols * half;
          // slot layout [column group of 4][row][4]: eight lanes' 16-byte
          // accesses cover 128 contiguous bytes, free of bank conflicts
          const uint32_t xg = xbase + slot * kXSlotBytes + (2 * half * 128 + row_l) * 16;
          float v[kHalfCols];
          ptx::tmem_ld8(tb + col, v);
          if (rank == 1) {
            // up values -> rank 0's slot, once rank 0 has drained it; the
            // asynchronous stores complete bytes on rank 0's xfull barrier
            if (!ptx::mbar_wait_cluster(xempty0 + 8 * slot, xph ^ 1, abort_flag, status)) {
              ok = false;
              break;
            }
            const uint32_t dst = ptx::map_to_rank(xg, 0);
#pragma unroll
            for (int j = 0; j < kHalfCols; j += 4)
              ptx::st_async_v4(dst + (j / 4) * 128 * 16, v[j], v[j + 1], v[j + 2], v[j + 3],
                               xfull_r0 + 8 * slot);
          } else {
            if (warp == 2 && lane == 0) ptx::mbar_arrive_expect_tx(xfull0 + 8 * slot, kXSlotBytes);
            if (!ptx::mbar_wait_cluster(xfull0 + 8 * slot, xph, abort_flag, status)) {
              ok = false;
              break;
            }
            const float4* up = reinterpret_cast<const float4*>(smem + (xg - sbase));
#pragma unroll
            for (int j = 0; j < kHalfCols; j += 4) {
              const float4 u4 = up[(j / 4) * 128];
              const float uj[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                if (col + j + t < tl.w)
                  orow[static_cast<long>(col + j + t) * out_ld] =
                      __float2bfloat16_rn(silu_f(v[j + t]) * uj[t]);
              }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster_relaxed(xempty_r1 + 8 * slot);
          }
        }
        if (!ok) break;
      } else {
        const int row = m * 256 + static_cast<int>(rank) * 128 + row_l;
        __nv_bfloat16* orow = out + static_cast<long>(tl.z) * out_ld + row;
        for (int c0 = 16 * half; c0 < tl.w; c0 += 32) {
          float v[16];
          ptx::tmem_ld16(tb + c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < tl.w) orow[static_cast<long>(c0 + j) * out_ld] = __float2bfloat16_rn(v[j]);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(tempty_r0 + 8 * b);
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

template <int MODE, int NMAX>
cudaError_t launch_pair_variant(const GemmArgs& a, int num_sms, cudaStream_t st) {
  using S = PairShape<MODE, NMAX>;
  auto kern = moe_gemm_pair<MODE, NMAX>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         S::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
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
                            a.status));
}

}  // namespace

cudaError_t launch_gemm_pair(GemmMode mode, int nmax, const GemmArgs& a, int num_sms,
                             cudaStream_t st) {
  if ((a.tiles == nullptr && a.dense_T <= 0) || a.k_split != 1) return cudaErrorInvalidValue;
  if (nmax == 256 && mode == kGemmPlain)
    return launch_pair_variant<kGemmPlain, 256>(a, num_sms, st);
  if (nmax == 256 && mode == kGemmSiluUp)
    return launch_pair_variant<kGemmSiluUp, 256>(a, num_sms, st);
  return cudaErrorInvalidValue;
}

}  // namespace moe
