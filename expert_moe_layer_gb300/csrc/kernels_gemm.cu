// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Orientation: the weight rows are the MMA's M side (128 rows per tile) and
// the token rows of one expert segment are the N side (16..nmax per tile).
// The accumulator holds D[w_row, token] = sum_k W[w_row, k] * X[token, k].
// The same kernel serves prefill (segments of hundreds of rows, nmax = 128)
// and decode (a few rows per expert, nmax = 32). Only the N of the
// instruction changes.
//
// Per CTA (persistent, one per SM, 576 threads):
//   warp 0      TMA producer: weights (A) and token rows (B) into a ring of
//               shared-memory stages with the 128-byte swizzle (when the
//               kernel gathers its token rows itself, A only)
//   warp 1      TMEM allocator and MMA issuer (one thread): 4 MMAs of
//               K = 128 bytes per stage; in SiLU mode a second accumulator for
//               the "up" rows shares the same B stage
//   warps 2..9  epilogue: tcgen05.ld of the accumulator (two warps per 32-lane
//               TMEM quarter, alternating 16-column chunks), SiLU(gate)*up or
//               plain, store to global. bf16 outputs go through a staging
//               buffer in shared memory per 16-column chunk, so the stores
//               are 16-byte vectors along output rows.
//   warps 10-17 with gathered token rows: copy each stage's rows of x by the
//               permutation (per-lane cp.async into the swizzled layout);
//               otherwise idle
// Accumulators are double-buffered in TMEM, so the epilogue of one work unit
// overlaps the main loop of the next.
//
// The producer takes the CTA's units in turn (blockIdx.x, + gridDim.x, ... or,
// with a grid-wide counter, whichever unit is next) and passes each to the
// MMA issuer and the epilogue through a ring of unit slots in shared memory.
//
// A GEMM1 with `publish` adds 1 per epilogue warp and unit to its tile's
// counter once the warp's h rows are stored. A GEMM2 given those counters
// (`ready`) starts before GEMM1 has finished: it skips the launch dependency
// wait, takes its units from the grid-wide counter (CTAs that start on SMs
// GEMM1 has left take more of them), and loads a tile's h rows only once the
// tile's count is complete. GEMM1's CTAs are all resident before GEMM2 can
// launch and never wait on it, so every count completes. GEMM2 waits for
// GEMM1's completion at its end, before it lets the next kernel launch.
//
// A GEMM1 given x and the sorted item ids gathers its token rows itself: the
// row warps copy row sorted_ids[p] / K of x for segment position p straight
// into the stage, so no permuted copy of x is written and read back. It waits
// for the kernel before it (which wrote the tile table and the ids) at its
// start and reads what that kernel wrote through L2: a CTA launched early by
// the dependent launch may otherwise read stale lines through the read-only
// path even after the wait.
//
// Work units are ordered group by group (a group = one expert's tiles, or one
// shared-expert slab), then by weight tile m, then by token tile. CTAs running
// at the same time therefore work on one expert. The 128-row weight tiles of
// that expert are read from DRAM once and shared by its token tiles through
// L2. The expert's token rows stay resident in L2 while all its weight tiles
// stream past them.
#include <cuda_bf16.h>

#include "act.cuh"
#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
[[maybe_unused]] constexpr DbgFile kDbgFileCode = kDbgGemm;
namespace {

constexpr bool kWeightEvictFirst = true;  // L2 policy of grouped weight boxes
constexpr int kRowWarps = 8;        // warps 10..17: gathered token rows
constexpr int kThreads = 320 + 32 * kRowWarps;
constexpr int kEpiThreads = 256;    // warps 2..9
static_assert(kEpiThreads / 32 == kGemmEpiWarps, "tile counts assume one add per epilogue warp");
constexpr int kABytes = 128 * 128;  // one 128-row x 128-byte weight box

// A pipeline stage holds KPS consecutive K blocks (128 bytes of K each), each
// with its weight box(es), then its token-row box. One SM's TMA engine
// completes stages at a roughly fixed rate whatever their size, so its
// throughput follows the bytes per stage rather than the number of stages.
template <int MODE, int NMAX, bool STG, int KPS = 1>
struct GemmShape {
  static constexpr int kNA = (MODE == kGemmSiluUp) ? 2 : 1;  // weight boxes per K block
  static constexpr int kBBytes = NMAX * 128;
  static constexpr int kSubBytes = kNA * kABytes + kBBytes;  // one K block
  static constexpr int kStageBytes = KPS * kSubBytes;
  // output staging (bf16 outputs): per column half, two buffers of 16 token
  // rows x 128 output columns
  static constexpr int kOutBufBytes = 16 * 128 * 2;
  static constexpr int kOutBytes = STG ? 2 * 2 * kOutBufBytes : 0;
  static constexpr int kStages0 =
      STG ? (216 * 1024 - kOutBytes) / kStageBytes : (200 * 1024) / kStageBytes;
  static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
  static constexpr int kAccCols = kNA * NMAX;            // fp32 columns per buffer
  static constexpr int kNAcc = kAccCols <= 256 ? 2 : 1;  // TMEM accumulator buffers
  static constexpr int kTmemNeed = kAccCols * kNAcc;
  static constexpr int kTmemCols = kTmemNeed <= 32    ? 32
                                   : kTmemNeed <= 64  ? 64
                                   : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256
                                                      : 512;
  static constexpr int kMaxGroups = 1024;
  static constexpr int kUnitRing = 8;  // unit slots from the producer to the other roles
  // full/empty per stage, tfull/tempty per accumulator, drain, ofull[2 halves][2 bufs],
  // ufull/uempty per unit slot
  static constexpr int kNBars = 2 * kStages + 2 * kNAcc + 1 + 4 + 2 * kUnitRing;
  static constexpr int kBarBytes = 8 * kNBars + 16 + 4 * kUnitRing + 4 * (kMaxGroups + 1);
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kOutBytes + kBarBytes;
  static_assert(kTmemNeed <= 512, "TMEM overflow");
  static_assert(kStages >= 2, "need at least two stages");
  static_assert(NMAX % 16 == 0 && NMAX <= 256, "bad NMAX");
};

template <typename T>
__device__ __forceinline__ T to_out(float v);
template <>
__device__ __forceinline__ float to_out<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}


// Unit u -> (tile index, weight tile m). gstart (shared memory) holds the
// first tile of each group and the total at [n_groups]; group g owns units
// [gstart[g]*m_tiles, gstart[g+1]*m_tiles), ordered m-major inside the group.
__device__ __forceinline__ void decode_unit(int u, const int* gstart, int n_groups, int m_tiles,
                                            int& tile, int& m) {
  int lo = 0, hi = n_groups - 1;
  while (lo < hi) {  // last group whose first unit is <= u (skips empty groups)
    const int mid = (lo + hi + 1) >> 1;
    if (gstart[mid] * m_tiles <= u) lo = mid;
    else hi = mid - 1;
  }
  const int n = gstart[lo + 1] - gstart[lo];
  const int r = u - gstart[lo] * m_tiles;
  m = r / n;
  tile = gstart[lo] + (r - m * n);
}

template <int MODE, bool TF32, typename TOut, int NMAX, int KPS>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_tc(const __grid_constant__ CUtensorMap mapA,
                const __grid_constant__ CUtensorMap mapB, const Tile* __restrict__ tiles,
                const int* __restrict__ group_start, int n_groups, int dense_T, int m_tiles,
                int k_blocks, int k_split, int a_rows_per_expert, int a_up_offset,
                int b_from_out, TOut* __restrict__ out, long out_ld, long split_stride,
                float* __restrict__ part, int m_valid, unsigned* status,
                const GemmBounds bnd, int* __restrict__ sched, const int* __restrict__ ready,
                int ready_target, int* __restrict__ publish, int* __restrict__ published,
                const void* __restrict__ gx, const int32_t* __restrict__ gids, int gdiv,
                long gld, long gitems) {
  constexpr bool kStaged = sizeof(TOut) == 2;
  const bool early = ready != nullptr;  // GEMM2 overlapping the GEMM1 before it
  const bool gather = gx != nullptr;    // token rows fetched by this kernel from x
  // the tile table of a gathering GEMM1 (and the ids it gathers by) come from
  // the kernel just before: wait first, and read them through laundered
  // pointers so that no load moves above the wait
  if (gather) {
    pdl_enter();
    tiles = fresh(tiles);
    group_start = fresh(group_start);
    gids = fresh(gids);
  }
  using S = GemmShape<MODE, NMAX, kStaged, KPS>;
  constexpr uint32_t kAB = TF32 ? 2u : 1u;   // operand type code
  constexpr int kKe = TF32 ? 32 : 64;         // K elements per 128-byte row

  // With k_split > 1 a unit covers one K range and writes its raw fp32
  // accumulator to the slab part + ks * split_stride (row stride out_ld; in
  // SiLU mode gate at column i and up at column a_up_offset + i). The caller
  // sums the slabs in order and applies the epilogue.
  // Dense problems (router, shared experts: every token of T for each of
  // n_groups weight slabs) pass no tile table; their tiles are implicit.
  const int dense_per = (dense_T + NMAX - 1) / NMAX;
  // A gathering GEMM1 may have started before the kernel that wrote its tile
  // table and ids finished; it reads them from L2 (not through the read-only
  // path), after its dependency wait.
  auto ld_group = [&](int i) -> int { return gather ? __ldcg(group_start + i) : group_start[i]; };
  const int total = (tiles ? ld_group(n_groups) : n_groups * dense_per) * m_tiles * k_split;
  const int kb_per = (k_blocks + k_split - 1) / k_split;
  if (static_cast<int>(blockIdx.x) >= total) return;  // uniform across the CTA

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kStages * S::kStageBytes + S::kOutBytes);
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S::kStages;
  const uint32_t tfull0 = empty0 + 8 * S::kStages;
  const uint32_t tempty0 = tfull0 + 8 * S::kNAcc;
  const uint32_t drain = tempty0 + 8 * S::kNAcc;
  const uint32_t ofull0 = drain + 8;  // [half][buffer]: a chunk's outputs are staged
  const uint32_t ufull0 = ofull0 + 32;  // [slot]: the unit in the slot is posted
  const uint32_t uempty0 = ufull0 + 8 * S::kUnitRing;  // [slot]: every role has read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + S::kNBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* uslot = reinterpret_cast<volatile int*>(tmem_slot + 4);
  int* gstart = reinterpret_cast<int*>(tmem_slot + 4 + S::kUnitRing);
  for (int i = threadIdx.x; i <= n_groups; i += kThreads)
    gstart[i] = tiles ? ld_group(i) : i * dense_per;
  // The debug build checks every entry and clamps a bad one into range, so
  // that all roles still walk the same pipeline.
  auto tile_at = [&](int ti) -> Tile {
    Tile tl;
    if (tiles) {
      const int tj = MOE_DCHECK(ti, bnd.max_tiles) ? ti : 0;
      tl = gather ? __ldcg(tiles + tj) : tiles[tj];
    } else {
      const int s = ti / dense_per, t0 = (ti - s * dense_per) * NMAX;
      tl = make_int4(s, t0, s * dense_T + t0, min(NMAX, dense_T - t0));
    }
#if MOE_DEBUG_BUILD
    if (!MOE_DCHECK(tl.x, n_groups)) tl.x = 0;
    if (!MOE_DCHECK(tl.w - 1, NMAX)) tl.w = 1;
    if (!b_from_out && !MOE_DCHECK(tl.y, bnd.b_rows - tl.w + 1)) tl.y = 0;
    if (!MOE_DCHECK(tl.z, (b_from_out ? min(bnd.b_rows, bnd.out_rows) : bnd.out_rows) - tl.w + 1))
      tl.z = 0;
#endif
    return tl;
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      // gathering: the weights' bytes, and one arrival per producer lane
      // once its copies of the token rows have landed
      ptx::mbar_init(full0 + 8 * s, gather ? 1 + 32 * kRowWarps : 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < S::kNAcc; ++b) {
      ptx::mbar_init(tfull0 + 8 * b, 1);
      ptx::mbar_init(tempty0 + 8 * b, kEpiThreads);
    }
    ptx::mbar_init(drain, 1);
    for (int x = 0; x < 4; ++x) ptx::mbar_init(ofull0 + 8 * x, 4);  // the half's 4 warps
    for (int x = 0; x < S::kUnitRing; ++x) {
      ptx::mbar_init(ufull0 + 8 * x, 1);
      // read by the MMA thread, the epilogue warps and, gathering, the row warps
      ptx::mbar_init(uempty0 + 8 * x, 1 + kEpiThreads / 32 + (gather ? kRowWarps : 0));
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async();
    ptx::tma_prefetch_map(&mapA);
    ptx::tma_prefetch_map(&mapB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), S::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // A grouped GEMM reads each weight box once, or again only for the other
  // token tiles of the same expert, which run at the same time: its weights
  // go into L2 first in line for eviction, so that they do not push out the
  // activations the next kernels read back. The router and shared-expert
  // weights (used by every token tile) keep the default priority.
  const uint64_t wpol =
      (kWeightEvictFirst && tiles) ? ptx::policy_evict_first() : ptx::policy_evict_normal();

  if (warp == 0 && gather) {
    // ---------------------------------------- weight producer (gathering)
    // Lane 0 takes the units, passes them on and issues each stage's weight
    // boxes with TMA; the row warps fill the stage's token rows.
    if (lane == 0) {
      int it = 0, posted = 0;
      bool ok = true;
      for (int j = 0;; ++j) {
        int u = static_cast<int>(blockIdx.x) + j * static_cast<int>(gridDim.x);
        u = u < total ? u : total;
        const int slot = posted % S::kUnitRing;
        if (posted >= S::kUnitRing &&
            !ptx::mbar_wait(uempty0 + 8 * slot, ((posted / S::kUnitRing) & 1) ^ 1, abort_flag,
                            status)) {
          ok = false;
          break;
        }
        uslot[slot] = u;
        ptx::mbar_arrive(ufull0 + 8 * slot);
        ++posted;
        if (u >= total) break;
        int ti, m;
        const int ks = u % k_split;
        decode_unit(u / k_split, gstart, n_groups, m_tiles, ti, m);
        const Tile tl = tile_at(ti);
        const int a_row = tl.x * a_rows_per_expert + m * 128;
        const int kb1 = min(k_blocks, (ks + 1) * kb_per);
        for (int kb = ks * kb_per; kb < kb1; kb += KPS, ++it) {
          const int s = it % S::kStages;
          const uint32_t ph = (it / S::kStages) & 1;
          if (!ptx::mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, status)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(full0 + 8 * s, KPS * S::kNA * kABytes);
#pragma unroll
          for (int p = 0; p < KPS; ++p) {
            const uint32_t st = sbase + s * S::kStageBytes + p * S::kSubBytes;
            ptx::tma_load_2d_hint(st, &mapA, full0 + 8 * s, (kb + p) * kKe, a_row, wpol);
            if (MODE == kGemmSiluUp)
              ptx::tma_load_2d_hint(st + kABytes, &mapA, full0 + 8 * s, (kb + p) * kKe,
                                    a_row + a_up_offset, wpol);
          }
        }
        if (!ok) break;
      }
      if (!ok) {
        // unwinding: let the weight boxes issued land before exit
        const int n = it < S::kStages ? it : S::kStages;
        for (int i = 0; i < n; ++i) {
          const int jj = it - 1 - i;
          ptx::mbar_wait_drain(full0 + 8 * (jj % S::kStages), (jj / S::kStages) & 1);
        }
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int taken = 0, posted = 0;
      // With the grid-wide counter, the next unit's ticket is drawn one unit
      // ahead, so the atomic's round trip overlaps the current unit's loads.
      int ticket = sched ? atomicAdd(sched, 1) : 0;
      // the CTA's next unit, or total when none is left
      auto take_unit = [&]() -> int {
        int u;
        if (sched) {
          u = ticket;
          if (u < total) ticket = atomicAdd(sched, 1);
        } else {
          u = static_cast<int>(blockIdx.x) + taken * static_cast<int>(gridDim.x);
        }
        ++taken;
        return u < total ? u : total;
      };
      // unit u into the next slot of the ring, for the MMA issuer and the epilogue
      auto post_unit = [&](int u) -> bool {
        const int slot = posted % S::kUnitRing;
        if (posted >= S::kUnitRing &&
            !ptx::mbar_wait(uempty0 + 8 * slot, ((posted / S::kUnitRing) & 1) ^ 1, abort_flag,
                            status))
          return false;
        uslot[slot] = u;
        ptx::mbar_arrive(ufull0 + 8 * slot);
        ++posted;
        return true;
      };
      // Operand A (weights) of the first kStages stages before the
      // dependency wait; operand B (token rows) only after it. These units
      // (at most kStages, so the ring does not fill) stay in their slots.
      int pre = 0, n_pre = 0;
      while (pre < S::kStages) {
        const int u = take_unit();
        post_unit(u);
        ++n_pre;
        if (u >= total) break;
        int ti, m;
        const int ks = u % k_split;
        decode_unit(u / k_split, gstart, n_groups, m_tiles, ti, m);
        const Tile tl = tile_at(ti);
        const int a_row = tl.x * a_rows_per_expert + m * 128;
        const int kb1 = min(k_blocks, (ks + 1) * kb_per);
        for (int kb = ks * kb_per; kb < kb1 && pre < S::kStages; kb += KPS, ++pre) {
          ptx::mbar_arrive_expect_tx(full0 + 8 * pre, S::kStageBytes);
#pragma unroll
          for (int p = 0; p < KPS; ++p) {
            const uint32_t st = sbase + pre * S::kStageBytes + p * S::kSubBytes;
            ptx::tma_load_2d_hint(st, &mapA, full0 + 8 * pre, (kb + p) * kKe, a_row, wpol);
            if (MODE == kGemmSiluUp)
              ptx::tma_load_2d_hint(st + kABytes, &mapA, full0 + 8 * pre, (kb + p) * kKe,
                                    a_row + a_up_offset, wpol);
          }
        }
      }
      if (!early) pdl_enter();
      int it = 0;
      bool ok = true;
      // every tile published (GEMM1 has stored all its rows): from then on no
      // unit needs its own acquire and proxy fence
      bool all_ready = false;
      const int all_target = (tiles ? gstart[n_groups] : 0) * ready_target;
      for (int j = 0;; ++j) {
        // after a failure only the stages whose weights went out before the
        // wait still get their token rows, so that their copies complete
        if (!ok && it >= pre) break;
        int u;
        if (j < n_pre) {
          u = uslot[j % S::kUnitRing];
        } else {
          if (!ok) break;
          u = take_unit();
          if (!post_unit(u)) {
            ok = false;
            break;
          }
        }
        if (u >= total) break;
        int ti, m;
        const int ks = u % k_split;
        decode_unit(u / k_split, gstart, n_groups, m_tiles, ti, m);
        const Tile tl = tile_at(ti);
        const int b_row = b_from_out ? tl.z : tl.y;
        const int kb1 = min(k_blocks, (ks + 1) * kb_per);
        (void)MOE_DCHECK(tl.x * static_cast<long>(a_rows_per_expert) + m * 128 +
                             (MODE == kGemmSiluUp ? a_up_offset : 0),
                         bnd.a_rows);
        if (ok && early && !all_ready) {
          // the tile's h rows: every GEMM1 epilogue warp of every weight tile
          if (ptx::ld_acquire(published) >= all_target) {
            all_ready = true;
            ptx::fence_proxy_async_global();
          } else if (ptx::wait_count(ready + ti, ready_target, abort_flag, status)) {
            ptx::fence_proxy_async_global();
          } else {
            ok = false;
          }
        }
        for (int kb = ks * kb_per; kb < kb1; kb += KPS, ++it) {
          const int s = it % S::kStages;
          const uint32_t ph = (it / S::kStages) & 1;
          const uint32_t st0 = sbase + s * S::kStageBytes;
          if (it >= pre) {  // stages of the early loads are fresh: no empty wait
            if (!ok) break;
            if (!ptx::mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, status)) {
              ok = false;
              break;
            }
            ptx::mbar_arrive_expect_tx(full0 + 8 * s, S::kStageBytes);
            const int a_row = tl.x * a_rows_per_expert + m * 128;
#pragma unroll
            for (int p = 0; p < KPS; ++p) {
              const uint32_t st = st0 + p * S::kSubBytes;
              ptx::tma_load_2d_hint(st, &mapA, full0 + 8 * s, (kb + p) * kKe, a_row, wpol);
              if (MODE == kGemmSiluUp)
                ptx::tma_load_2d_hint(st + kABytes, &mapA, full0 + 8 * s, (kb + p) * kKe,
                                      a_row + a_up_offset, wpol);
            }
          }
#pragma unroll
          for (int p = 0; p < KPS; ++p)
            ptx::tma_load_2d(st0 + p * S::kSubBytes + S::kNA * kABytes, &mapB, full0 + 8 * s,
                             (kb + p) * kKe, b_row);
        }
      }
      if (!ok) {
        // unwinding: let every load this thread issued land before exit (every
        // stage below `it` has both operands; none at or above it was issued)
        const int n = it < S::kStages ? it : S::kStages;
        for (int i = 0; i < n; ++i) {
          const int jj = it - 1 - i;
          ptx::mbar_wait_drain(full0 + 8 * (jj % S::kStages), (jj / S::kStages) & 1);
        }
      }
    } else if (!early) {
      pdl_enter();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (!early) pdl_enter();
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int ai = 0; ok; ++ai) {
        const int slot = ai % S::kUnitRing;
        if (!ptx::mbar_wait(ufull0 + 8 * slot, (ai / S::kUnitRing) & 1, abort_flag, status)) {
          ok = false;
          break;
        }
        const int u = uslot[slot];
        ptx::mbar_arrive(uempty0 + 8 * slot);
        if (u >= total) break;
        int ti, m;
        const int ks = u % k_split;
        decode_unit(u / k_split, gstart, n_groups, m_tiles, ti, m);
        const Tile tl = tile_at(ti);
        const int n_mma = (tl.w + 15) & ~15;
        const int kb0 = ks * kb_per, kb1 = min(k_blocks, kb0 + kb_per);
        const uint32_t idesc = ptx::idesc_make(kAB, 128, n_mma);
        const int b = ai % S::kNAcc;
        const uint32_t aph = (ai / S::kNAcc) & 1;
        if (!ptx::mbar_wait(tempty0 + 8 * b, aph ^ 1, abort_flag, status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + b * S::kAccCols;
        for (int kb = kb0; kb < kb1; kb += KPS, ++it) {
          const int s = it % S::kStages;
          const uint32_t ph = (it / S::kStages) & 1;
          if (!ptx::mbar_wait(full0 + 8 * s, ph, abort_flag, status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          // gathered token rows were written through the generic proxy
          if (gather) ptx::fence_proxy_async();
#pragma unroll
          for (int p = 0; p < KPS; ++p) {
            const uint32_t st = sbase + s * S::kStageBytes + p * S::kSubBytes;
            const uint64_t da = ptx::sdesc_sw128(st);
            const uint64_t db = ptx::sdesc_sw128(st + S::kNA * kABytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc = (kb + p > kb0 || kk > 0) ? 1u : 0u;
              ptx::tc_mma<TF32>(d, da + 2 * kk, db + 2 * kk, idesc, acc);
              if (MODE == kGemmSiluUp) {
                const uint64_t du = ptx::sdesc_sw128(st + kABytes);
                ptx::tc_mma<TF32>(d + NMAX, du + 2 * kk, db + 2 * kk, idesc, acc);
              }
            }
          }
          ptx::tc_commit(empty0 + 8 * s);
        }
        if (!ok) break;
        ptx::tc_commit(tfull0 + 8 * b);
      }
      if (!ok) {
        // unwinding: wait for the MMAs already issued
        ptx::tc_commit(drain);
        ptx::mbar_wait_drain(drain, 0);
      }
    }
  } else if (warp <= 9) {
    // ------------------------------------------------------------ epilogue
    if (!early) pdl_enter();
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;    // two warps per quarter split the columns
    int cc = 0;
    for (int ai = 0;; ++ai) {
      const int slot = ai % S::kUnitRing;
      if (!ptx::mbar_wait(ufull0 + 8 * slot, (ai / S::kUnitRing) & 1, abort_flag, status)) break;
      const int u = uslot[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(uempty0 + 8 * slot);
      if (u >= total) break;
      int ti, m;
      const int ks = u % k_split;
      decode_unit(u / k_split, gstart, n_groups, m_tiles, ti, m);
      const Tile tl = tile_at(ti);
      const int b = ai % S::kNAcc;
      const uint32_t aph = (ai / S::kNAcc) & 1;
      if (!ptx::mbar_wait(tfull0 + 8 * b, aph, abort_flag, status)) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + b * S::kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      const int row = m * 128 + q * 32 + lane;
      const bool row_ok = row < m_valid;
      if (k_split > 1) {
        float* prow = part + ks * split_stride + static_cast<long>(tl.z) * out_ld + row;
        for (int c0 = 16 * half; c0 < tl.w; c0 += 32) {
          float v[16];
          if constexpr (MODE == kGemmSiluUp) {
            float w[16];
            ptx::tmem_ld16x2(tb + c0, tb + NMAX + c0, v, w);
            if (row_ok && MOE_DCHECK(row + a_up_offset, out_ld)) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if (c0 + j < tl.w) {
                  prow[static_cast<long>(c0 + j) * out_ld] = v[j];
                  prow[static_cast<long>(c0 + j) * out_ld + a_up_offset] = w[j];
                }
              }
            }
          } else {
            ptx::tmem_ld16(tb + c0, v);
            if (row_ok && MOE_DCHECK(row, out_ld)) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < tl.w) prow[static_cast<long>(c0 + j) * out_ld] = v[j];
            }
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(tempty0 + 8 * b);
        continue;
      }
      if constexpr (kStaged) {
        // staging [16 columns][128 rows] bf16 per chunk, written out as 16
        // rows of 256 bytes, 16 bytes per lane
        uint8_t* const stg = smem + S::kStages * S::kStageBytes + half * 2 * S::kOutBufBytes;
        const uint32_t ofull = ofull0 + 16 * half;
        const int row_l = q * 32 + lane;
        const int t_out = row_l >> 4, c8 = (row_l & 15) * 8;
        const bool cols_ok = m * 128 + c8 < m_valid;
        bool ok = true;
        for (int c0 = 16 * half; c0 < tl.w; c0 += 32, ++cc) {
          float v[16];
          if constexpr (MODE == kGemmSiluUp) {
            float w[16];
            ptx::tmem_ld16x2(tb + c0, tb + NMAX + c0, v, w);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = silu(v[j]) * w[j];
          } else {
            ptx::tmem_ld16(tb + c0, v);
          }
          __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(stg + (cc & 1) * S::kOutBufBytes);
#pragma unroll
          for (int j = 0; j < 16; ++j) sb[j * 128 + row_l] = __float2bfloat16_rn(v[j]);
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(ofull + 8 * (cc & 1));
          if (!ptx::mbar_wait(ofull + 8 * (cc & 1), (cc >> 1) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int t = k * 8 + t_out;
            if (c0 + t < tl.w && cols_ok && MOE_DCHECK(m * 128 + c8 + 7, out_ld)) {
              const uint4 val = *reinterpret_cast<const uint4*>(sb + t * 128 + c8);
              *reinterpret_cast<uint4*>(out + static_cast<long>(tl.z + c0 + t) * out_ld +
                                        m * 128 + c8) = val;
            }
          }
        }
        if (!ok) break;
        ptx::tc_fence_before();
        ptx::mbar_arrive(tempty0 + 8 * b);
        if (publish) ptx::publish_rows(publish + ti, published, lane);
        continue;
      }
      TOut* orow = out + static_cast<long>(tl.z) * out_ld + row;
      for (int c0 = 16 * half; c0 < tl.w; c0 += 32) {
        float v[16];
        if constexpr (MODE == kGemmSiluUp) {
          float w[16];
          ptx::tmem_ld16x2(tb + c0, tb + NMAX + c0, v, w);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = silu(v[j]) * w[j];
        } else {
          ptx::tmem_ld16(tb + c0, v);
        }
        if (row_ok && MOE_DCHECK(row, out_ld)) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < tl.w) orow[static_cast<long>(c0 + j) * out_ld] = to_out<TOut>(v[j]);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty0 + 8 * b);
      if (publish) ptx::publish_rows(publish + ti, published, lane);
    }
  } else if (gather) {
    // ----------------------------------------------------------- row warps
    // Copy each stage's token rows from x, 16 bytes per lane and copy,
    // straight into the 128-byte-swizzled layout the MMA reads (chunk c of
    // row r at r * 128 + ((c ^ (r & 7)) * 16)). Row warp w takes the groups
    // of four rows g = w, w + kRowWarps, ...; in a group, lanes 8i..8i+7 take
    // row 4g + i, one chunk each, so each warp-wide copy fills four whole
    // rows. Each lane's copies of a stage arrive on the stage's barrier once
    // they have landed (it expects the weights' bytes and every row-warp
    // lane); the MMA thread then fences the rows for the async proxy.
    constexpr int kBOff = S::kNA * kABytes;
    constexpr int kPer = NMAX / (4 * kRowWarps);  // row groups per warp
    static_assert(kPer >= 1 && kPer * 4 * kRowWarps == NMAX, "row groups per warp");
    const int rw = warp - 10;
    const int rsub = lane >> 3, chunk = lane & 7;
    const char* xb = static_cast<const char*>(gx);
    const long row_bytes = gld * (TF32 ? 4 : 2);
    int it = 0;
    for (int ai = 0;; ++ai) {
      const int slot = ai % S::kUnitRing;
      if (!ptx::mbar_wait(ufull0 + 8 * slot, (ai / S::kUnitRing) & 1, abort_flag, status)) break;
      const int u = uslot[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(uempty0 + 8 * slot);
      if (u >= total) break;
      int ti, m;
      const int ks = u % k_split;
      decode_unit(u / k_split, gstart, n_groups, m_tiles, ti, m);
      const Tile tl = tile_at(ti);
      const int kb1 = min(k_blocks, (ks + 1) * kb_per);
      // this lane's rows and their tokens; rows past the segment repeat its
      // first row (their columns of the accumulator are never stored). An
      // item id outside [0, gitems), possible only in caller-made segments,
      // reads row 0: its output row is garbage, as from an unwritten x_perm.
      long src[kPer];
      int dst[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int r = 4 * (i * kRowWarps + rw) + rsub;
        const int id = __ldcg(gids + tl.y + (r < tl.w ? r : 0));
        int tok = (id >= 0 && id < gitems) ? id / gdiv : 0;
        if (!MOE_DCHECK(tok, bnd.x_rows)) tok = 0;
        src[i] = static_cast<long>(tok) * row_bytes + chunk * 16;
        dst[i] = r * 128 + ((chunk ^ (r & 7)) << 4);
      }
      bool ok = true;
      for (int kb = ks * kb_per; kb < kb1; kb += KPS, ++it) {
        const int s = it % S::kStages;
        const uint32_t ph = (it / S::kStages) & 1;
        int w_ok = 1;
        if (lane == 0) w_ok = ptx::mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, status) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        const uint32_t st0 = sbase + s * S::kStageBytes;
#pragma unroll
        for (int p = 0; p < KPS; ++p) {
          const uint32_t bdst = st0 + p * S::kSubBytes + kBOff;
          const long kbyte = static_cast<long>(kb + p) * 128;
#pragma unroll
          for (int i = 0; i < kPer; ++i) ptx::cp_async16(bdst + dst[i], xb + src[i] + kbyte);
        }
        ptx::cp_async_arrive_noinc(full0 + 8 * s);
      }
      if (!ok) break;
    }
    ptx::cp_async_wait_all();  // nothing of this warp is in flight when the CTA exits
  } else if (!early) {
    pdl_enter();  // the row warps idle when the token rows come through mapB
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, S::kTmemCols);
  }
  // overlapping GEMM2: the GEMM1 before it has completed before the next
  // kernel may launch
  if (early) pdl_enter();
}

template <int MODE, bool TF32, typename TOut, int NMAX, int KPS = 1>
cudaError_t launch_variant(const GemmArgs& a, int num_sms, cudaStream_t st) {
  using S = GemmShape<MODE, NMAX, sizeof(TOut) == 2, KPS>;
  auto kern = moe_gemm_tc<MODE, TF32, TOut, NMAX, KPS>;
  static std::atomic<unsigned long long> smem_set{0};  // devices, one bit each
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(kern), S::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(num_sms), dim3(kThreads), S::kSmemBytes, st, *a.mapA, *a.mapB,
                    a.tiles, a.group_start, a.n_groups, a.dense_T, a.m_tiles, a.k_blocks, a.k_split,
                    a.a_rows_per_expert, a.a_up_offset, a.b_from_out, static_cast<TOut*>(a.out),
                    a.out_ld, a.split_stride, a.part, a.m_valid, a.status, a.bnd, a.sched,
                    a.ready, a.ready_target, a.publish, a.published, a.gather_x,
                    a.gather_ids, a.gather_div, a.gather_ld, a.gather_items);
}

}  // namespace

cudaError_t launch_gemm(GemmMode mode, bool tf32, int nmax, const GemmArgs& a, int num_sms,
                        cudaStream_t st) {
  if (a.k_split < 1 || (a.k_split > 1 && a.part == nullptr)) return cudaErrorInvalidValue;
  // the overlap needs the tile table (and one K range: the tile's count is
  // of whole units)
  if ((a.ready || a.publish) && (!a.tiles || a.k_split != 1)) return cudaErrorInvalidValue;
  if ((a.ready || a.publish) && !a.published) return cudaErrorInvalidValue;
  // gathering needs the tile table, whole token tiles and one K range per unit
  if (a.gather_x && (!a.tiles || !a.gather_ids || a.gather_div < 1 || a.gather_ld <= 0 ||
                     a.gather_items <= 0 || a.ready))
    return cudaErrorInvalidValue;
  if (a.ready && (!a.sched || a.ready_target <= 0)) return cudaErrorInvalidValue;
  if (MOE_DEBUG_BUILD && (a.bnd.a_rows <= 0 || a.bnd.b_rows <= 0 || a.bnd.out_rows <= 0 ||
                          (a.tiles && a.bnd.max_tiles <= 0)))
    return cudaErrorInvalidValue;
  if (nmax != 32 && nmax != 128 && nmax != 256) return cudaErrorInvalidValue;
  if (nmax == 256) {  // prefill-sized segments, bf16 only
    if (tf32) return cudaErrorInvalidValue;
    if (mode == kGemmSiluUp)
      return launch_variant<kGemmSiluUp, false, __nv_bfloat16, 256>(a, num_sms, st);
    if (mode == kGemmPlain)
      return launch_variant<kGemmPlain, false, __nv_bfloat16, 256>(a, num_sms, st);
    return cudaErrorInvalidValue;
  }
  const bool big = nmax == 128;
  // bf16 plain GEMMs with whole K ranges and an even K block count take two K
  // blocks per stage (three or more stages still fit). The SiLU mode's
  // stages carry two weight boxes: doubled, only two fit, and that measured
  // slower (EP-shard GEMM1 99.5 against 93.8 us).
  const bool two = a.k_split == 1 && a.k_blocks % 2 == 0;
  static_assert(GemmShape<kGemmPlain, 128, true, 2>::kStages >= 3 &&
                    GemmShape<kGemmPlain, 32, true, 2>::kStages >= 3 &&
                    GemmShape<kGemmPlain, 128, false, 2>::kStages >= 3,
                "two K blocks per stage keep at least three stages");
  switch (mode) {
    case kGemmSiluUp:
      if (tf32)
        return big ? launch_variant<kGemmSiluUp, true, float, 128>(a, num_sms, st)
                   : launch_variant<kGemmSiluUp, true, float, 32>(a, num_sms, st);
      return big ? launch_variant<kGemmSiluUp, false, __nv_bfloat16, 128>(a, num_sms, st)
                 : launch_variant<kGemmSiluUp, false, __nv_bfloat16, 32>(a, num_sms, st);
    case kGemmPlain:
      if (tf32)
        return big ? launch_variant<kGemmPlain, true, float, 128>(a, num_sms, st)
                   : launch_variant<kGemmPlain, true, float, 32>(a, num_sms, st);
      if (two)
        return big ? launch_variant<kGemmPlain, false, __nv_bfloat16, 128, 2>(a, num_sms, st)
                   : launch_variant<kGemmPlain, false, __nv_bfloat16, 32, 2>(a, num_sms, st);
      return big ? launch_variant<kGemmPlain, false, __nv_bfloat16, 128>(a, num_sms, st)
                 : launch_variant<kGemmPlain, false, __nv_bfloat16, 32>(a, num_sms, st);
    case kGemmLogits: {
      if (tf32) return cudaErrorInvalidValue;
      // router logits split over K: two K blocks per stage where every K
      // range holds an even number of blocks
      const int kb_per = (a.k_blocks + a.k_split - 1) / a.k_split;
      const bool two_split = a.k_blocks % 2 == 0 && kb_per % 2 == 0;
      if ((two || two_split) && big)
        return launch_variant<kGemmPlain, false, float, 128, 2>(a, num_sms, st);
      return big ? launch_variant<kGemmPlain, false, float, 128>(a, num_sms, st)
                 : launch_variant<kGemmPlain, false, float, 32>(a, num_sms, st);
    }
  }
  return cudaErrorInvalidValue;
}

MOE_WAIT_LIMIT_SETTER(set_wait_limit_gemm)
MOE_DEBUG_TAKER(take_dbg_gemm)

}  // namespace moe
