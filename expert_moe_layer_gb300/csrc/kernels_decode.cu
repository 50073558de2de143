// The routed MoE layer of a decode-sized batch (T <= 16 tokens) in one
// persistent tcgen05 kernel, followed by a small combine kernel.
//
// MixtralMoE.forward at decode: router logits, fp32 softmax, top-k and
// renormalise (FusedMoE select_experts arguments), then for every chosen
// local expert w2(silu(w1 x) * w3 x), weighted and summed per token. At a
// handful of tokens the layer is a read of the touched experts' weights; any
// step that is not streaming those bytes (a kernel boundary, a serial
// routing chain on one SM, a gather, a wait between the two GEMMs) shows up
// directly in the layer time. So one grid does everything:
//
//   1. every CTA loads the batch's token rows x (at most 16) into shared
//      memory, once, as the B operand of all its MMAs (rows >= T are zero),
//      and computes the router logits of its share of the experts
//      (e = blockIdx.x, blockIdx.x + gridDim.x, ...) on CUDA cores;
//   2. a grid barrier (one counter, bounded wait): every logit is written;
//   3. every CTA takes the routing decision of all T tokens itself (one warp
//      per token, topk_warp) and builds the list of touched local experts in
//      ascending order. No CTA waits on another after this point;
//   4. units (touched expert j, 64-index slice m of I) are dealt round robin
//      over the CTAs. A unit computes h = silu(x Wg^T) * (x Wu^T) for its 64
//      intermediate indices (GEMM1, M = 64 gate + 64 up weight rows, N = 16
//      tokens), keeps h in shared memory and multiplies it by the matching
//      64 columns of w2 (GEMM2, H/128 tiles of M = 128 output rows). The
//      result is a partial of y over that slice: for every token routed to
//      the expert, weight * partial goes to its own fp32 row of `part`.
//      Units share nothing, so the weights stream without any cross-CTA
//      wait; GEMM1 of unit i+1 is issued before GEMM2 of unit i, so the
//      SiLU epilogue of unit i overlaps the next unit's weight reads.
//   5. the combine kernel sums, per token, the partial rows of its local
//      slots in a fixed order (slot k, then slice m), times
//      routed_scaling_factor, into the bf16 output.
// The last CTA (which holds the fewest units) also writes the routing arrays
// of the workspace after its units: topk_ids, topk_w, and the stable
// counting sort (counts, offsets, sorted_ids, inv_pos) that the other paths
// produce, with segments unpadded.
//
// Every wait is bounded; the grid barrier and the cross-CTA reads assume that
// all CTAs are resident (one per SM), as the launch guarantees when the GPU
// is not shared. A wait that runs out sets MOE_DEV_TIMEOUT.
//
// Warp roles after the routing phase (6 warps):
//   warp 0      TMA producer: 16 KB stages (GEMM1: 64 gate + 64 up rows of
//               one 64-column K block; GEMM2: 128 w2 rows x 64 columns)
//   warp 1      TMEM owner and MMA issuer (one thread)
//   warps 2..5  epilogue, one per 32-lane TMEM quarter. GEMM1 accumulators
//               hold gate rows in lanes 0-63 and up rows in lanes 64-127; the
//               up warps hand their values to the gate warps through shared
//               memory (two mbarriers), which write h (bf16, 128-byte
//               swizzled, the B operand of GEMM2).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "align_block.cuh"
#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"
#include "topk_warp.cuh"

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int kWarps = kThreads / 32;
constexpr int kEpiThreads = 128;                 // warps 2..5
constexpr int kTokN = kDecodeMaxTokens;          // MMA N: the batch's token rows
constexpr int kSlice = 64;                       // intermediate indices per unit
constexpr int kStageBytes = 16384;
constexpr int kXBlk = kTokN * 128;               // 16 token rows x one 64-element K block
constexpr int kHBytes = kTokN * 128;             // h of one unit: 16 x 64 bf16
constexpr int kMaxItems = kDecodeMaxItems;
constexpr int kMaxWords = kDecodeMaxLocal / 32;  // touched-expert bit mask
constexpr int kMaxStages = 10;
constexpr int kMaxChunks = kDecodeMaxHidden / 8 / 32;  // router row, 16-byte pieces per lane
constexpr int kTmemCols = 64;                    // D1 x 2 + D2 x 2, 16 columns each
constexpr int kSmemLimit = 227 * 1024;

// Shared memory after the stages and the token rows (bytes), 1024-aligned
// start of the h buffers first.
constexpr int kFixedBytes = 2 * kHBytes + kTokN * kSlice * 4 + 3 * kMaxItems * 4 +
                            kMaxWords * 4 + kMaxItems * 4 + 8 * (2 * kMaxStages + 16) + 64;

__host__ __device__ constexpr int x_bytes(int H) { return (H / 64) * kXBlk; }

int stages_for(int H) {
  const int s = (kSmemLimit - 1024 - kFixedBytes - x_bytes(H)) / kStageBytes;
  return s > kMaxStages ? kMaxStages : s;
}
int smem_for(int H) { return 1024 + stages_for(H) * kStageBytes + x_bytes(H) + kFixedBytes; }

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until *p >= target, bounded like the mbarrier waits.
__device__ __forceinline__ bool wait_count(const int* p, int target, volatile int* abort,
                                           unsigned* status) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (ld_acquire(p) >= target) return true;
    if ((n & 15u) == 0) {
      if (*abort) return false;
      if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
        *abort = 1;
        if (status) atomicOr(status, MOE_DEV_TIMEOUT);
        return false;
      }
    }
    __nanosleep(32);
  }
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& r, float (&v)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

struct DecodeParams {
  const __nv_bfloat16* wg;
  const float* bias;
  int T, E, H, I, K, renorm, flags, n_group, topk_group;
  float* logits;
  int* grid_bar;
  int32_t* ids;
  float* w;
  const int32_t* emap;
  int R, E_l, ep_start;
  float* part;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_ids;
  int32_t* inv_pos;
  unsigned* status;
  int stages;
};

template <int VPL>
__global__ void __launch_bounds__(kThreads, 1)
    moe_decode_layer(const __grid_constant__ CUtensorMap mapX,
                     const __grid_constant__ CUtensorMap mapW13,
                     const __grid_constant__ CUtensorMap mapW2, const DecodeParams p) {
  const int T = p.T, E = p.E, H = p.H, K = p.K, nst = p.stages;
  const int G = gridDim.x;
  const int kbx = H / 64;         // K blocks of GEMM1
  const int n_mt = H / 128;       // output tiles of GEMM2
  const int S = p.I / kSlice;     // slices per expert
  const int n_items = T * K;
  const bool book = blockIdx.x == static_cast<unsigned>(G - 1);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  uint8_t* xs = smem + nst * kStageBytes;
  uint8_t* hs = xs + x_bytes(H);
  float* xchg = reinterpret_cast<float*>(hs + 2 * kHBytes);     // [16 tokens][64]
  int* s_ids = reinterpret_cast<int*>(xchg + kTokN * kSlice);   // [T*K]
  float* s_w = reinterpret_cast<float*>(s_ids + kMaxItems);     // [T*K]
  int* s_le = reinterpret_cast<int*>(s_w + kMaxItems);          // [T*K] local expert or -1
  unsigned* s_mask = reinterpret_cast<unsigned*>(s_le + kMaxItems);
  int* s_touched = reinterpret_cast<int*>(s_mask + kMaxWords);  // touched local experts
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_touched + kMaxItems);
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * nst;
  const uint32_t d1full0 = empty0 + 8 * nst;   // [2]
  const uint32_t d1empty0 = d1full0 + 16;      // [2]
  const uint32_t d2full0 = d1empty0 + 16;      // [2]
  const uint32_t d2empty0 = d2full0 + 16;      // [2]
  const uint32_t hfull0 = d2empty0 + 16;       // [2]
  const uint32_t hempty0 = hfull0 + 16;        // [2]
  const uint32_t xfull = hempty0 + 16;
  const uint32_t xempty = xfull + 8;
  const uint32_t drain = xempty + 8;
  const uint32_t xbar = drain + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * nst + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_ntouched = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(d1full0 + 8 * b, 1);
      ptx::mbar_init(d1empty0 + 8 * b, kEpiThreads);
      ptx::mbar_init(d2full0 + 8 * b, 1);
      ptx::mbar_init(d2empty0 + 8 * b, kEpiThreads);
      ptx::mbar_init(hfull0 + 8 * b, 64);   // the two gate warps
      ptx::mbar_init(hempty0 + 8 * b, 1);
    }
    ptx::mbar_init(xfull, 64);              // the two up warps
    ptx::mbar_init(xempty, 64);             // the two gate warps
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(xbar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async();
    ptx::tma_prefetch_map(&mapX);
    ptx::tma_prefetch_map(&mapW13);
    ptx::tma_prefetch_map(&mapW2);
  }
  for (int i = threadIdx.x; i < kMaxWords; i += kThreads) s_mask[i] = 0u;
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // ---------------------------------------------------------------- 1. logits
  // (expert j of this CTA, token t) pairs, j-major, a contiguous run per warp.
  // A lane holds 16-byte pieces lane, lane + 32, ... of the router row
  // (never written by the library: loaded before the dependency wait).
  const int n_my = static_cast<int>(blockIdx.x) < E ? (E - 1 - blockIdx.x) / G + 1 : 0;
  const int n_pairs = n_my * T;
  const int per_warp = (n_pairs + kWarps - 1) / kWarps;
  const int p0 = min(n_pairs, warp * per_warp), p1 = min(n_pairs, p0 + per_warp);
  const int n_chunk = H / 8;
  uint4 wr[kMaxChunks];
  int cur_j = -1;
  auto load_row = [&](int j) {
    const uint4* row =
        reinterpret_cast<const uint4*>(p.wg + static_cast<long>(blockIdx.x + j * G) * H);
#pragma unroll
    for (int i = 0; i < kMaxChunks; ++i) {
      const int g = lane + 32 * i;
      wr[i] = g < n_chunk ? __ldg(row + g) : make_uint4(0u, 0u, 0u, 0u);
    }
    cur_j = j;
  };
  if (p0 < p1) load_row(p0 / T);

  pdl_wait();
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(x_bytes(H)));
    for (int kb = 0; kb < kbx; ++kb)
      ptx::tma_load_2d(ptx::smem_u32(xs + kb * kXBlk), &mapX, xbar, kb * 64, 0);
  }
  pdl_launch_dependents();
  bool ok = ptx::mbar_wait(xbar, 0, abort_flag, p.status);
  if (!ok && threadIdx.x == 0) ptx::mbar_wait_drain(xbar, 0);  // let late copies land
  ok = __syncthreads_and(ok);
  if (ok) {
    for (int q = p0; q < p1; ++q) {
      const int j = q / T, t = q - j * T;
      if (j != cur_j) load_row(j);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxChunks; ++i) {
        const int g = lane + 32 * i;
        if (g < n_chunk) {
          // token row t, 16-byte piece g: K block g/8, swizzled chunk (g%8)^(t%8)
          const uint4 xr = *reinterpret_cast<const uint4*>(
              xs + (g >> 3) * kXBlk + t * 128 + (((g & 7) ^ (t & 7)) << 4));
          float xv[8], wv[8];
          bf16x8_to_f32(xr, xv);
          bf16x8_to_f32(wr[i], wv);
#pragma unroll
          for (int k = 0; k < 8; ++k) acc = fmaf(xv[k], wv[k], acc);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) p.logits[static_cast<long>(t) * E + blockIdx.x + j * G] = acc;
    }
  }

  // ---------------------------------------------------------------- 2. grid barrier
  __syncthreads();
  if (threadIdx.x == 0) {
    red_release_add(p.grid_bar, 1);
    if (!wait_count(p.grid_bar, G, abort_flag, p.status)) *abort_flag = 1;
  }
  ok = __syncthreads_and(ok && !*abort_flag);

  // ---------------------------------------------------------------- 3. routing
  int n_units = 0;
  if (ok) {
    const float* lg = fresh(p.logits);  // written by every CTA before the barrier
    const bool sel = p.flags & kRouteBiasSelect;
    for (int t = warp; t < T; t += kWarps) {
      float pv[VPL], sb[VPL];
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int e = lane + 32 * j;
        const float b = (p.bias && e < E) ? __ldg(p.bias + e) : 0.f;
        pv[j] = e < E ? __ldcg(lg + static_cast<long>(t) * E + e) + (sel ? 0.f : b)
                      : -CUDART_INF_F;
        sb[j] = sel ? b : 0.f;
      }
      topk_warp<VPL>(pv, sb, lane, E, K, p.renorm, p.flags, p.n_group, p.topk_group,
                     s_ids + t * K, s_w + t * K);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_items; i += kThreads) {
      const int le = local_expert(s_ids[i], i / K, p.emap, p.R, E, p.E_l, p.ep_start,
                                  book ? p.status : nullptr);
      s_le[i] = le;
      if (le >= 0) atomicOr(s_mask + (le >> 5), 1u << (le & 31));
    }
    __syncthreads();
    if (warp == 0) {
      // touched local experts in ascending order
      unsigned m = lane < (p.E_l + 31) / 32 ? s_mask[lane] : 0u;
      const int c = __popc(m);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      int pos = incl - c;
      while (m) {
        const int b = __ffs(m) - 1;
        s_touched[pos++] = lane * 32 + b;
        m &= m - 1;
      }
      if (lane == 31) *s_ntouched = incl;
    }
    __syncthreads();
    n_units = *s_ntouched * S;
  }
  const int n_mine =
      static_cast<int>(blockIdx.x) < n_units ? (n_units - 1 - blockIdx.x) / G + 1 : 0;
  // unit i of this CTA: u = blockIdx.x + i*G -> touched expert u / S, slice u % S
  auto unit_le = [&](int i) { return s_touched[(blockIdx.x + i * G) / S]; };
  auto unit_m = [&](int i) { return static_cast<int>((blockIdx.x + i * G) % S); };

  // ---------------------------------------------------------------- 4. units
  // Phase order: G1(0), then G1(i), G2(i-1) for i = 1 .. n-1, then G2(n-1).
  if (ok && n_mine > 0) {
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        int it = 0;
        bool pok = true;
        for (int i = 0; i <= n_mine && pok; ++i) {
          if (i < n_mine) {
            const int le = unit_le(i), m = unit_m(i);
            const int rg = le * 2 * p.I + m * kSlice;
            for (int kb = 0; kb < kbx; ++kb, ++it) {
              const int s = it % nst;
              const uint32_t ph = (it / nst) & 1;
              if (!ptx::mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, p.status)) {
                pok = false;
                break;
              }
              const uint32_t st = sbase + s * kStageBytes, fb = full0 + 8 * s;
              ptx::mbar_arrive_expect_tx(fb, kStageBytes);
              ptx::tma_load_2d(st, &mapW13, fb, kb * 64, rg);
              ptx::tma_load_2d(st + kStageBytes / 2, &mapW13, fb, kb * 64, rg + p.I);
            }
          }
          if (i >= 1 && pok) {
            const int le = unit_le(i - 1), m = unit_m(i - 1);
            for (int mt = 0; mt < n_mt; ++mt, ++it) {
              const int s = it % nst;
              const uint32_t ph = (it / nst) & 1;
              if (!ptx::mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, p.status)) {
                pok = false;
                break;
              }
              const uint32_t st = sbase + s * kStageBytes, fb = full0 + 8 * s;
              ptx::mbar_arrive_expect_tx(fb, kStageBytes);
              ptx::tma_load_2d(st, &mapW2, fb, m * kSlice, le * H + mt * 128);
            }
          }
        }
        if (!pok) {
          // unwinding: let every load this thread issued land before exit
          const int n = it < nst ? it : nst;
          for (int k = 0; k < n; ++k) {
            const int j = it - 1 - k;
            ptx::mbar_wait_drain(full0 + 8 * (j % nst), (j / nst) & 1);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        const uint32_t idesc = ptx::idesc_make(1u, 128, kTokN);
        int it = 0, d2i = 0;
        bool mok = true;
        for (int i = 0; i <= n_mine && mok; ++i) {
          if (i < n_mine) {
            const int b = i & 1;
            if (!ptx::mbar_wait(d1empty0 + 8 * b, ((i >> 1) & 1) ^ 1, abort_flag, p.status)) {
              mok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t d = tmem_base + b * kTokN;
            for (int kb = 0; kb < kbx; ++kb, ++it) {
              const int s = it % nst;
              if (!ptx::mbar_wait(full0 + 8 * s, (it / nst) & 1, abort_flag, p.status)) {
                mok = false;
                break;
              }
              ptx::tc_fence_after();
              const uint64_t da = ptx::sdesc_sw128(sbase + s * kStageBytes);
              const uint64_t db = ptx::sdesc_sw128(ptx::smem_u32(xs + kb * kXBlk));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                ptx::tc_mma<false>(d, da + 2 * kk, db + 2 * kk, idesc,
                                   (kb > 0 || kk > 0) ? 1u : 0u);
              ptx::tc_commit(empty0 + 8 * s);
            }
            if (!mok) break;
            ptx::tc_commit(d1full0 + 8 * b);
          }
          if (i >= 1) {
            const int j = i - 1, bh = j & 1;
            if (!ptx::mbar_wait(hfull0 + 8 * bh, (j >> 1) & 1, abort_flag, p.status)) {
              mok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t db = ptx::sdesc_sw128(ptx::smem_u32(hs + bh * kHBytes));
            for (int mt = 0; mt < n_mt; ++mt, ++it, ++d2i) {
              const int s = it % nst, b2 = d2i & 1;
              if (!ptx::mbar_wait(full0 + 8 * s, (it / nst) & 1, abort_flag, p.status) ||
                  !ptx::mbar_wait(d2empty0 + 8 * b2, ((d2i >> 1) & 1) ^ 1, abort_flag,
                                  p.status)) {
                mok = false;
                break;
              }
              ptx::tc_fence_after();
              const uint64_t da = ptx::sdesc_sw128(sbase + s * kStageBytes);
              const uint32_t d = tmem_base + 2 * kTokN + b2 * kTokN;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                ptx::tc_mma<false>(d, da + 2 * kk, db + 2 * kk, idesc, kk > 0 ? 1u : 0u);
              ptx::tc_commit(empty0 + 8 * s);
              // h[bh] is free once this unit's last MMA is done; committed
              // before the accumulator, so that no arrive is still pending
              // when the epilogue has seen the last tile and the CTA exits
              if (mt == n_mt - 1) ptx::tc_commit(hempty0 + 8 * bh);
              ptx::tc_commit(d2full0 + 8 * b2);
            }
            if (!mok) break;
          }
        }
        if (!mok) {
          // unwinding: wait for the MMAs already issued
          ptx::tc_commit(drain);
          ptx::mbar_wait_drain(drain, 0);
        }
      }
    } else {
      // ------------------------------------------------------------ epilogue
      const int q = warp & 3;  // TMEM lane quarter: 0, 1 gate rows; 2, 3 up rows
      int d2i = 0;
      bool eok = true;
      for (int i = 0; i <= n_mine && eok; ++i) {
        if (i < n_mine) {
          const int b = i & 1;
          if (!ptx::mbar_wait(d1full0 + 8 * b, (i >> 1) & 1, abort_flag, p.status)) break;
          ptx::tc_fence_after();
          float v[16];
          ptx::tmem_ld16(tmem_base + b * kTokN + (static_cast<uint32_t>(q * 32) << 16), v);
          ptx::tc_fence_before();
          ptx::mbar_arrive(d1empty0 + 8 * b);
          if (q >= 2) {
            // up rows: hand them to the gate warp of the same 32 indices
            if (!ptx::mbar_wait(xempty, (i & 1) ^ 1, abort_flag, p.status)) break;
#pragma unroll
            for (int t = 0; t < kTokN; ++t) xchg[t * kSlice + (q - 2) * 32 + lane] = v[t];
            ptx::mbar_arrive(xfull);
          } else {
            if (!ptx::mbar_wait(xfull, i & 1, abort_flag, p.status)) break;
            float u[16];
#pragma unroll
            for (int t = 0; t < kTokN; ++t) u[t] = xchg[t * kSlice + q * 32 + lane];
            ptx::mbar_arrive(xempty);
            // h buffer b was last read by GEMM2 of unit i - 2
            if (!ptx::mbar_wait(hempty0 + 8 * b, ((i >> 1) & 1) ^ 1, abort_flag, p.status))
              break;
            // h[t][il] (il = q*32 + lane) into the 128-byte swizzled K-major
            // tile: row t at t*128, 16-byte chunk il/8 at (il/8) ^ (t % 8)
            uint8_t* hb = hs + b * kHBytes;
            const int il = q * 32 + lane;
#pragma unroll
            for (int t = 0; t < kTokN; ++t) {
              const __nv_bfloat16 hv = __float2bfloat16_rn(silu_f(v[t]) * u[t]);
              *reinterpret_cast<__nv_bfloat16*>(hb + t * 128 + (((il >> 3) ^ (t & 7)) << 4) +
                                                (il & 7) * 2) = hv;
            }
            ptx::fence_proxy_async();
            ptx::mbar_arrive(hfull0 + 8 * b);
          }
        }
        if (i >= 1) {
          // GEMM2 of unit i - 1: each token routed to its expert gets
          // weight * partial over this slice in its own fp32 row
          const int j = i - 1;
          const int le = unit_le(j), m = unit_m(j);
          int tk[kTokN];
          float cf[kTokN];
#pragma unroll
          for (int t = 0; t < kTokN; ++t) {
            tk[t] = -1;
            cf[t] = 0.f;
            if (t < T) {
              for (int k = 0; k < K; ++k) {
                if (s_le[t * K + k] == le) {
                  tk[t] = t * K + k;
                  cf[t] = s_w[t * K + k];
                }
              }
            }
          }
          for (int mt = 0; mt < n_mt; ++mt, ++d2i) {
            const int b2 = d2i & 1;
            if (!ptx::mbar_wait(d2full0 + 8 * b2, (d2i >> 1) & 1, abort_flag, p.status)) {
              eok = false;
              break;
            }
            ptx::tc_fence_after();
            float v[16];
            ptx::tmem_ld16(tmem_base + 2 * kTokN + b2 * kTokN +
                               (static_cast<uint32_t>(q * 32) << 16),
                           v);
            ptx::tc_fence_before();
            ptx::mbar_arrive(d2empty0 + 8 * b2);
            const int r = mt * 128 + q * 32 + lane;
#pragma unroll
            for (int t = 0; t < kTokN; ++t)
              if (tk[t] >= 0)
                p.part[(static_cast<long>(tk[t]) * S + m) * H + r] = cf[t] * v[t];
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }

  // ---------------------------------------------------------------- bookkeeping
  // The last CTA writes the routing arrays of the workspace: ids and weights,
  // then a stable counting sort of the items over the local experts with
  // unpadded segments (counts, offsets, sorted_ids with the sentinel T*K past
  // the last segment, inv_pos = -1 for items of other ranks).
  if (!book || !ok || *abort_flag) return;
  for (int i = threadIdx.x; i < n_items; i += kThreads) {
    p.ids[i] = s_ids[i];
    p.w[i] = s_w[i];
  }
  int* cnt = reinterpret_cast<int*>(smem);  // the stages are free now
  for (int e = threadIdx.x; e < p.E_l; e += kThreads) cnt[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n_items; i += kThreads)
    if (s_le[i] >= 0) atomicAdd(cnt + s_le[i], 1);
  __syncthreads();
  // exclusive scan of cnt over E_l: a contiguous run of entries per thread
  int* warp_sums = cnt + kDecodeMaxLocal;  // 32 ints of scan scratch
  const int per = (p.E_l + kThreads - 1) / kThreads;
  const int e0 = min(p.E_l, static_cast<int>(threadIdx.x) * per), e1 = min(p.E_l, e0 + per);
  int run = 0;
  for (int e = e0; e < e1; ++e) run += cnt[e];
  int total = 0;
  int base = block_exclusive_scan(run, warp_sums, total);
  for (int e = e0; e < e1; ++e) {
    const int c = cnt[e];
    p.counts[e] = c;
    p.offsets[e] = base;
    cnt[e] = base;
    base += c;
  }
  if (threadIdx.x == 0) p.offsets[p.E_l] = total;
  __syncthreads();
  for (int i = threadIdx.x; i < n_items; i += kThreads) {
    const int le = s_le[i];
    int pos = -1;
    if (le >= 0) {
      int rank = 0;
      for (int j = 0; j < i; ++j) rank += s_le[j] == le;
      pos = cnt[le] + rank;
      p.sorted_ids[pos] = i;
    }
    p.inv_pos[i] = pos;
    if (i >= total) p.sorted_ids[i] = n_items;  // cap = T*K rows
  }
}

// out[t] = rsf * sum over local slots k (inv_pos >= 0), then slices m, of the
// partial rows, in that order; bf16. One thread per 4 output columns.
__global__ void __launch_bounds__(64, 8) decode_combine_kernel(const float* __restrict__ part,
                                                            const int32_t* __restrict__ inv_pos,
                                                            int T, int K, int S, int H,
                                                            float rsf,
                                                            __nv_bfloat16* __restrict__ out) {
  pdl_enter();
  part = fresh(part);
  inv_pos = fresh(inv_pos);
  const long idx = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int c4 = H / 4;
  if (idx >= static_cast<long>(T) * c4) return;
  const int t = static_cast<int>(idx / c4), c = static_cast<int>(idx - static_cast<long>(t) * c4);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < K; ++k) {
    if (__ldcg(inv_pos + t * K + k) < 0) continue;
    const float4* row =
        reinterpret_cast<const float4*>(part + static_cast<long>(t * K + k) * S * H) + c;
    for (int m = 0; m < S; ++m) {
      const float4 v = __ldcg(row + static_cast<long>(m) * c4);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
  }
  const __nv_bfloat162 lo = __floats2bfloat162_rn(rsf * acc.x, rsf * acc.y);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(rsf * acc.z, rsf * acc.w);
  uint2 pk;
  pk.x = static_cast<uint32_t>(__bfloat16_as_ushort(lo.x)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(lo.y)) << 16);
  pk.y = static_cast<uint32_t>(__bfloat16_as_ushort(hi.x)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(hi.y)) << 16);
  *reinterpret_cast<uint2*>(out + static_cast<long>(t) * H + 4 * c) = pk;
}

template <int VPL>
cudaError_t decode_launch(const DecodeArgs& a, const DecodeParams& prm, int smem, int num_sms,
                          cudaStream_t st) {
  auto kern = moe_decode_layer<VPL>;
  static std::atomic<unsigned long long> smem_set{0};  // devices, one bit each
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(kern), smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(num_sms), dim3(kThreads), smem, st, *a.mapX, *a.mapW13,
                    *a.mapW2, prm);
}

}  // namespace

bool decode_layer_ok(int T, int E, int H, int I, int K, int E_l) {
  return T >= 1 && T <= kDecodeMaxTokens && static_cast<long>(T) * K <= kDecodeMaxItems &&
         E >= 1 && E <= 512 && E_l >= 1 && E_l <= kDecodeMaxLocal && H % 128 == 0 &&
         H <= kDecodeMaxHidden && I % kSlice == 0 && stages_for(H) >= 4;
}

size_t decode_part_floats(int T, int K, int H, int I) {
  return static_cast<size_t>(T) * K * (I / kSlice) * H;
}

cudaError_t launch_decode_layer(const DecodeArgs& a, int num_sms, cudaStream_t st) {
  if (!decode_layer_ok(a.T, a.E, a.H, a.I, a.K, a.E_l) || num_sms < 1)
    return cudaErrorInvalidValue;
  DecodeParams prm;
  prm.wg = static_cast<const __nv_bfloat16*>(a.wg);
  prm.bias = a.bias;
  prm.T = a.T;
  prm.E = a.E;
  prm.H = a.H;
  prm.I = a.I;
  prm.K = a.K;
  prm.renorm = a.renorm;
  prm.flags = a.flags;
  prm.n_group = a.n_group;
  prm.topk_group = a.topk_group;
  prm.logits = a.logits;
  prm.grid_bar = a.grid_bar;
  prm.ids = a.ids;
  prm.w = a.w;
  prm.emap = a.emap;
  prm.R = a.R;
  prm.E_l = a.E_l;
  prm.ep_start = a.ep_start;
  prm.part = a.part;
  prm.counts = a.counts;
  prm.offsets = a.offsets;
  prm.sorted_ids = a.sorted_ids;
  prm.inv_pos = a.inv_pos;
  prm.status = a.status;
  prm.stages = stages_for(a.H);
  const int smem = smem_for(a.H);
  const int vpl = (a.E + 31) / 32;
  cudaError_t e;
  if (vpl <= 1) e = decode_launch<1>(a, prm, smem, num_sms, st);
  else if (vpl <= 2) e = decode_launch<2>(a, prm, smem, num_sms, st);
  else if (vpl <= 4) e = decode_launch<4>(a, prm, smem, num_sms, st);
  else if (vpl <= 8) e = decode_launch<8>(a, prm, smem, num_sms, st);
  else e = decode_launch<16>(a, prm, smem, num_sms, st);
  return e;
}

cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t st) {
  const long threads = static_cast<long>(a.T) * (a.H / 4);
  return launch_pdl(decode_combine_kernel, dim3(static_cast<unsigned>((threads + 63) / 64)),
                    dim3(64), 0, st, static_cast<const float*>(a.part),
                    static_cast<const int32_t*>(a.inv_pos), a.T, a.K, a.I / kSlice, a.H,
                    a.rsf, static_cast<__nv_bfloat16*>(a.out));
}

}  // namespace moe
