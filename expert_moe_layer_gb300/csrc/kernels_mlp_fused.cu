// Both expert GEMMs of a decode-sized batch in one persistent tcgen05 kernel.
//
// The routed expert MLP (MixtralMoE expert forward: w2(silu(w1 x) * w3 x)) is
// two grouped GEMMs: h = silu(gate) * up over w13, then y = h w2^T. Launched
// one after the other, the second waits for the first one's slowest CTA. At
// decode sizes both are short and bound by weight reads, so that wait, plus
// the wave quantisation of the first GEMM's units and the launches around
// them, costs a sizeable share of the layer. Here one grid walks a single
// unit list:
//
//   units [0, U1)        GEMM1: (tile, 128 rows of w13's gate and up halves,
//                        K range ks of ks1)
//   units [U1, U1 + U2)  GEMM2: (tile, 128 rows of w2)
//
// Token rows are TMA boxes of x_perm, gathered by the kernel before this one.
// The tile table is therefore two kernels old, so the weight boxes of each
// CTA's first stages are issued before the dependency wait and stream in
// while the gather runs.
//
// Each CTA takes units blockIdx.x, blockIdx.x + gridDim.x, ... in order.
// With ks1 = 1 the epilogue warps of a GEMM1 unit store their block of h and
// add 1 to the tile's ready counter. With ks1 > 1 they store raw fp32 gate and
// up partials. The last of the ks1 warps that cover the same 32 rows x 16
// columns (a counter per block) sums the partials in slab order, applies
// SiLU*up, stores h and adds 1 to the ready counter. A GEMM2 unit's producer
// streams its w2 tiles first, then waits (bounded) until the counter reaches
// 8 blocks x I/128, then loads the h rows. All GEMM1 units precede all GEMM2
// units in every CTA's sequence, so GEMM1 work never waits and no wait can
// deadlock once every CTA is resident (one CTA per SM; a wait that runs out
// sets MOE_DEV_TIMEOUT). The grid is one CTA per SM that the current context
// may use, and the caller takes this kernel only where one CTA fits on an SM
// (mlp_fused_fits); otherwise it runs the two GEMM kernels. Kernels of other
// streams that hold SMs only delay some CTAs: they finish without waiting on
// this one. A cooperative launch would also guarantee residency, but measured
// 1.8 us slower per decode step (T = 1 and 8) with the same kernel time, so
// the launch stays a plain dependent launch. The counters are zeroed before
// the kernel.
//
// Stage layout (40 KB): two 128-row weight boxes and two token-row boxes of
// 32 rows, each box 128 bytes of K with the 128-byte swizzle.
//   GEMM1 stage: A0 = gate rows, A1 = up rows, B0 = x rows (one K block);
//                gate accumulates in columns [0, 32), up in [32, 64)
//   GEMM2 stage: A0/B0 = K block 2j, A1/B1 = K block 2j+1, one accumulator
// Warp roles as in moe_gemm_tc: warp 0 TMA producer, warp 1 TMEM owner and
// MMA issuer, warps 2..9 epilogue (two per TMEM lane quarter).
#include <cuda_bf16.h>

#include "act.cuh"
#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
[[maybe_unused]] constexpr DbgFile kDbgFileCode = kDbgMlpFused;
namespace {

constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kEpiWarps = 8;
constexpr int kABytes = 128 * 128;
constexpr int kNmax = 32;                          // token rows per tile
constexpr int kBBytes = kNmax * 128;
constexpr int kStageBytes = 2 * kABytes + 2 * kBBytes;
constexpr int kStages = 5;
constexpr int kAccCols = 2 * kNmax;                // gate + up
constexpr int kNAcc = 2;
constexpr int kTmemCols = 128;
constexpr int kMaxGroups = 1024;
constexpr int kMaxSplit = 8;                       // K ranges of GEMM1 at most
constexpr int kBarBytes = 8 * (2 * kStages + 2 * kNAcc + 1) + 16 + 4 * (kMaxGroups + 1);
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes;
static_assert(kAccCols * kNAcc <= kTmemCols, "TMEM overflow");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");


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

struct UnitInfo {
  bool g2;      // GEMM2 unit
  int ti, m;    // tile index, weight tile
  int ks;       // K range (GEMM1)
  int kb0;      // first K block (GEMM1)
  int n_st;     // pipeline stages of the unit
};

__device__ __forceinline__ UnitInfo unit_info(int u, int U1, const int* gstart, int n_groups,
                                              int m1, int m2, int kb1, int kb2, int ks1,
                                              int kb_per) {
  UnitInfo r;
  r.g2 = u >= U1;
  if (!r.g2) {
    r.ks = u % ks1;
    decode_unit(u / ks1, gstart, n_groups, m1, r.ti, r.m);
    r.kb0 = r.ks * kb_per;
    r.n_st = min(kb1, r.kb0 + kb_per) - r.kb0;
  } else {
    r.ks = 0;
    r.kb0 = 0;
    decode_unit(u - U1, gstart, n_groups, m2, r.ti, r.m);
    r.n_st = (kb2 + 1) >> 1;
  }
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
    moe_mlp_fused(const __grid_constant__ CUtensorMap mapW13,
                  const __grid_constant__ CUtensorMap mapW2,
                  const __grid_constant__ CUtensorMap mapH,
                  const __grid_constant__ CUtensorMap mapX, const Tile* __restrict__ tiles,
                  const int* __restrict__ group_start, int n_groups, int H, int I,
                  int ks1, float* __restrict__ part, long part_stride,
                  int* __restrict__ split_cnt, int* __restrict__ ready,
                  __nv_bfloat16* __restrict__ h_out, __nv_bfloat16* __restrict__ y_out,
                  unsigned* status, const GemmBounds bnd) {
  const int m1 = I / 128, m2 = H / 128;
  const int kb1 = H / 64, kb2 = I / 64;
  const int kb_per = (kb1 + ks1 - 1) / ks1;
  const int ready_target = kEpiWarps * m1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kStages;
  const uint32_t tfull0 = empty0 + 8 * kStages;
  const uint32_t tempty0 = tfull0 + 8 * kNAcc;
  const uint32_t drain = tempty0 + 8 * kNAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 2 * kNAcc + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* gstart = reinterpret_cast<int*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < kNAcc; ++b) {
      ptx::mbar_init(tfull0 + 8 * b, 1);
      ptx::mbar_init(tempty0 + 8 * b, kEpiThreads);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async();
    ptx::tma_prefetch_map(&mapW13);
    ptx::tma_prefetch_map(&mapW2);
    ptx::tma_prefetch_map(&mapH);
    ptx::tma_prefetch_map(&mapX);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  // the tile table is two kernels old: read before the dependency wait
  for (int i = threadIdx.x; i <= n_groups; i += kThreads) gstart[i] = group_start[i];
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int n_tiles = gstart[n_groups];
  const int U1 = n_tiles * m1 * ks1;
  const int total = U1 + n_tiles * m2;
  // A unit's tile. The debug build checks the tile index and the entry (the
  // rows of x_perm, h and y are b_rows = out_rows) and clamps a bad one, so
  // that every role still walks the same pipeline.
  auto unit_tile = [&](UnitInfo& ui) -> Tile {
    if (!MOE_DCHECK(ui.ti, bnd.max_tiles)) ui.ti = 0;
    Tile tl = tiles[ui.ti];
#if MOE_DEBUG_BUILD
    if (!MOE_DCHECK(tl.x, n_groups)) tl.x = 0;
    if (!MOE_DCHECK(tl.w - 1, kNmax)) tl.w = 1;
    if (!MOE_DCHECK(tl.y, bnd.b_rows - tl.w + 1)) tl.y = 0;
    if (!MOE_DCHECK(tl.z, bnd.out_rows - tl.w + 1)) tl.z = 0;
#endif
    return tl;
  };

  // weight boxes of the first stages before the wait
  int pre = 0;
  {
    if (warp == 0 && lane == 0) {
      for (int u = blockIdx.x; u < U1 && pre < kStages; u += gridDim.x) {
        UnitInfo ui = unit_info(u, U1, gstart, n_groups, m1, m2, kb1, kb2, ks1, kb_per);
        const Tile tl = unit_tile(ui);
        const int arow = tl.x * 2 * I + ui.m * 128;
        for (int j = 0; j < ui.n_st && pre < kStages; ++j, ++pre) {
          const uint32_t st = sbase + pre * kStageBytes, fb = full0 + 8 * pre;
          const int kx = (ui.kb0 + j) * 64;
          ptx::mbar_arrive_expect_tx(fb, 2 * kABytes + kBBytes);
          ptx::tma_load_2d(st, &mapW13, fb, kx, arow);
          ptx::tma_load_2d(st + kABytes, &mapW13, fb, kx, arow + I);
        }
      }
    }
    pre = __shfl_sync(0xffffffffu, pre, 0);
    pdl_enter();
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // lane 0 issues; the warp keeps the unit walk and the status in step
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      UnitInfo ui = unit_info(u, U1, gstart, n_groups, m1, m2, kb1, kb2, ks1, kb_per);
      const Tile tl = unit_tile(ui);
      if (!ui.g2) {
        // token rows from x_perm (segment rows tl.y ..) with TMA
        if (lane == 0) {
          const int arow = tl.x * 2 * I + ui.m * 128;
          for (int j = 0; j < ui.n_st; ++j) {
            const int i2 = it + j;
            const int s = i2 % kStages;
            const uint32_t ph = (i2 / kStages) & 1;
            const uint32_t st = sbase + s * kStageBytes, fb = full0 + 8 * s;
            const int kx = (ui.kb0 + j) * 64;
            if (i2 >= pre) {  // stages of the early loads are fresh: no empty wait
              if (!ptx::mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, status)) {
                ok = false;
                break;
              }
              ptx::mbar_arrive_expect_tx(fb, 2 * kABytes + kBBytes);
              ptx::tma_load_2d(st, &mapW13, fb, kx, arow);
              ptx::tma_load_2d(st + kABytes, &mapW13, fb, kx, arow + I);
            }
            ptx::tma_load_2d(st + 2 * kABytes, &mapX, fb, kx, tl.y);
          }
        }
        it += ui.n_st;
        ok = __shfl_sync(0xffffffffu, ok, 0);
      } else {
        // GEMM2: the unit's first weight boxes, then wait for its h rows
        if (lane == 0) {
          const int arow = tl.x * H + ui.m * 128;
          const int n_a = min(ui.n_st, kStages);
          int j = 0;
          for (; j < n_a; ++j) {
            const int i2 = it + j;
            const int s = i2 % kStages;
            const uint32_t ph = (i2 / kStages) & 1;
            if (!ptx::mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, status)) {
              ok = false;
              break;
            }
            const uint32_t st = sbase + s * kStageBytes, fb = full0 + 8 * s;
            const bool two = 2 * j + 1 < kb2;
            ptx::mbar_arrive_expect_tx(fb, two ? 2 * (kABytes + kBBytes) : kABytes + kBBytes);
            ptx::tma_load_2d(st, &mapW2, fb, 2 * j * 64, arow);
            if (two) ptx::tma_load_2d(st + kABytes, &mapW2, fb, (2 * j + 1) * 64, arow);
          }
          // on failure the issued weight boxes still land; their stages never fill
          if (ok && !ptx::wait_count(ready + ui.ti, ready_target, abort_flag, status)) ok = false;
          if (ok) ptx::fence_proxy_async_global();
          for (j = 0; j < ui.n_st && ok; ++j) {
            const int i2 = it + j;
            const int s = i2 % kStages;
            const uint32_t ph = (i2 / kStages) & 1;
            const uint32_t st = sbase + s * kStageBytes, fb = full0 + 8 * s;
            const bool two = 2 * j + 1 < kb2;
            if (j >= n_a) {
              if (!ptx::mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, status)) {
                ok = false;
                break;
              }
              ptx::mbar_arrive_expect_tx(fb, two ? 2 * (kABytes + kBBytes) : kABytes + kBBytes);
              ptx::tma_load_2d(st, &mapW2, fb, 2 * j * 64, arow);
              if (two) ptx::tma_load_2d(st + kABytes, &mapW2, fb, (2 * j + 1) * 64, arow);
            }
            ptx::tma_load_2d(st + 2 * kABytes, &mapH, fb, 2 * j * 64, tl.z);
            if (two) ptx::tma_load_2d(st + 2 * kABytes + kBBytes, &mapH, fb, (2 * j + 1) * 64, tl.z);
          }
        }
        it += ui.n_st;
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
    if (!ok) {
      // unwinding: give in-flight copies time to land before the CTA exits
      const uint64_t t0 = ptx::globaltimer();
      while (ptx::globaltimer() - t0 < 200000) {
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, ai = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++ai) {
        UnitInfo ui = unit_info(u, U1, gstart, n_groups, m1, m2, kb1, kb2, ks1, kb_per);
        const Tile tl = unit_tile(ui);
        const int n_mma = (tl.w + 15) & ~15;
        const uint32_t idesc = ptx::idesc_make(1u, 128, n_mma);
        const int b = ai % kNAcc;
        const uint32_t aph = (ai / kNAcc) & 1;
        if (!ptx::mbar_wait(tempty0 + 8 * b, aph ^ 1, abort_flag, status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + b * kAccCols;
        for (int j = 0; j < ui.n_st; ++j, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!ptx::mbar_wait(full0 + 8 * s, ph, abort_flag, status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t st = sbase + s * kStageBytes;
          const uint64_t da0 = ptx::sdesc_sw128(st);
          const uint64_t da1 = ptx::sdesc_sw128(st + kABytes);
          const uint64_t db0 = ptx::sdesc_sw128(st + 2 * kABytes);
          const uint64_t db1 = ptx::sdesc_sw128(st + 2 * kABytes + kBBytes);
          if (!ui.g2) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
              ptx::tc_mma<false>(d, da0 + 2 * kk, db0 + 2 * kk, idesc, acc);
              ptx::tc_mma<false>(d + kNmax, da1 + 2 * kk, db0 + 2 * kk, idesc, acc);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::tc_mma<false>(d, da0 + 2 * kk, db0 + 2 * kk, idesc,
                                 (j > 0 || kk > 0) ? 1u : 0u);
            if (2 * j + 1 < kb2) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                ptx::tc_mma<false>(d, da1 + 2 * kk, db1 + 2 * kk, idesc, 1u);
            }
          }
          ptx::tc_commit(empty0 + 8 * s);
        }
        if (!ok) break;
        ptx::tc_commit(tfull0 + 8 * b);
      }
      if (!ok) {
        ptx::tc_commit(drain);
        ptx::mbar_wait_drain(drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int blk = warp - 2;                     // this warp's 32 x 16 block of a unit
    int ai = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++ai) {
      UnitInfo ui = unit_info(u, U1, gstart, n_groups, m1, m2, kb1, kb2, ks1, kb_per);
      const Tile tl = unit_tile(ui);
      const int b = ai % kNAcc;
      const uint32_t aph = (ai / kNAcc) & 1;
      if (!ptx::mbar_wait(tfull0 + 8 * b, aph, abort_flag, status)) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + b * kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      const int row = ui.m * 128 + q * 32 + lane;  // h column (GEMM1) or y column (GEMM2)
      const int c0 = 16 * half;                     // this warp's 16 token columns
      float v[16];
      if (ui.g2) {
        ptx::tmem_ld16(tb + c0, v);
        ptx::tc_fence_before();
        ptx::mbar_arrive(tempty0 + 8 * b);
        __nv_bfloat16* orow = y_out + static_cast<long>(tl.z) * H + row;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < tl.w) orow[static_cast<long>(c0 + j) * H] = __float2bfloat16_rn(v[j]);
        continue;
      }
      float w[16];
      ptx::tmem_ld16x2(tb + c0, tb + kNmax + c0, v, w);
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty0 + 8 * b);
      __nv_bfloat16* hrow = h_out + static_cast<long>(tl.z) * I + row;
      if (ks1 == 1) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < tl.w) hrow[static_cast<long>(c0 + j) * I] = __float2bfloat16_rn(silu(v[j]) * w[j]);
        ptx::publish_rows(ready + ui.ti, nullptr, lane);
        continue;
      }
      // K split: raw partials of this slab ([row][gate I | up I] fp32), then
      // the last of the ks1 warps on this block finishes it
      float* prow = part + ui.ks * part_stride + static_cast<long>(tl.z) * 2 * I + row;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (c0 + j < tl.w) {
          prow[static_cast<long>(c0 + j) * 2 * I] = v[j];
          prow[static_cast<long>(c0 + j) * 2 * I + I] = w[j];
        }
      }
      __syncwarp();
      int old = 0;
      if (lane == 0) old = ptx::add_acq_rel(split_cnt + (ui.ti * m1 + ui.m) * kEpiWarps + blk, 1);
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old != ks1 - 1) continue;
      // every slab's value is loaded before the sum, which runs in slab order;
      // the other slabs were written by other CTAs before their counter add
      const float* qrow = fresh(part) + static_cast<long>(tl.z) * 2 * I + row;
      for (int j = 0; j < 16 && c0 + j < tl.w; ++j) {
        const float* pc = qrow + static_cast<long>(c0 + j) * 2 * I;
        float gs[kMaxSplit], us[kMaxSplit];
#pragma unroll
        for (int s = 0; s < kMaxSplit; ++s) {
          gs[s] = s < ks1 ? __ldcg(pc + s * part_stride) : 0.f;
          us[s] = s < ks1 ? __ldcg(pc + s * part_stride + I) : 0.f;
        }
        float g = gs[0], up = us[0];
#pragma unroll
        for (int s = 1; s < kMaxSplit; ++s) {
          if (s < ks1) {
            g += gs[s];
            up += us[s];
          }
        }
        hrow[static_cast<long>(c0 + j) * I] = __float2bfloat16_rn(silu(g) * up);
      }
      ptx::publish_rows(ready + ui.ti, nullptr, lane);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

std::atomic<unsigned long long> g_smem_set{0};  // devices with the shared memory opt-in

}  // namespace

size_t mlp_fused_smem_bytes() { return kSmemBytes; }

bool mlp_fused_fits() {
  static std::atomic<unsigned long long> checked{0}, fits{0};  // devices, one bit each
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (checked.load(std::memory_order_acquire) & bit))
    return (fits.load(std::memory_order_acquire) & bit) != 0;
  int n = 0;
  const bool ok =
      opt_in_smem(reinterpret_cast<const void*>(moe_mlp_fused), kSmemBytes, g_smem_set) ==
          cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, moe_mlp_fused, kThreads, kSmemBytes) ==
          cudaSuccess &&
      n >= 1;
  if (bit) {
    if (ok) fits.fetch_or(bit, std::memory_order_acq_rel);
    checked.fetch_or(bit, std::memory_order_acq_rel);
  }
  return ok;
}

cudaError_t launch_mlp_fused(const MlpFusedArgs& a, int num_sms, cudaStream_t st) {
  const cudaError_t e =
      opt_in_smem(reinterpret_cast<const void*>(moe_mlp_fused), kSmemBytes, g_smem_set);
  if (e != cudaSuccess) return e;
  if (a.H % 128 != 0 || a.I % 128 != 0 || a.n_groups > kMaxGroups || a.ks1 < 1 ||
      a.ks1 > kMaxSplit || (a.ks1 > 1 && (!a.part || !a.split_cnt)))
    return cudaErrorInvalidValue;
  if (MOE_DEBUG_BUILD && (a.bnd.b_rows <= 0 || a.bnd.out_rows <= 0 || a.bnd.max_tiles <= 0))
    return cudaErrorInvalidValue;
  return launch_pdl(moe_mlp_fused, dim3(num_sms), dim3(kThreads), kSmemBytes, st, *a.mapW13,
                    *a.mapW2, *a.mapH, *a.mapX, a.tiles, a.group_start, a.n_groups, a.H, a.I,
                    a.ks1, a.part, a.part_stride, a.split_cnt, a.ready,
                    static_cast<__nv_bfloat16*>(a.h), static_cast<__nv_bfloat16*>(a.y), a.status,
                    a.bnd);
}

MOE_WAIT_LIMIT_SETTER(set_wait_limit_mlp_fused)
MOE_DEBUG_TAKER(take_dbg_mlp_fused)

}  // namespace moe
