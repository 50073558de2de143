// Routing: router logits, fp32 softmax, plain or group-limited top-k,
// renormalise (MixtralMoE.forward; FusedMoE select_experts arguments).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "align_block.cuh"
#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
[[maybe_unused]] constexpr DbgFile kDbgFileCode = kDbgRoute;  // before topk_warp.cuh, which checks ids
}  // namespace moe

#include "topk_warp.cuh"

namespace moe {
namespace {

// --------------------------------------------------------------- logits
// CTA = 8 warps; warp w computes expert e = blockIdx.x*8 + w for kTok tokens.
// A lane walks H in 8-element chunks (16-byte loads for bf16) and keeps one
// fp32 partial per token. A butterfly reduction then finishes each dot.
constexpr int kTok = 8;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 r = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename TX, typename TW>
__global__ void __launch_bounds__(256) router_logits_kernel(const TX* __restrict__ x,
                                                            const TW* __restrict__ wg,
                                                            float* __restrict__ logits, int T,
                                                            int E, int H) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  const int t0 = blockIdx.y * kTok;
  if (e >= E) return;
  float acc[kTok];
#pragma unroll
  for (int j = 0; j < kTok; ++j) acc[j] = 0.f;
  const TW* wrow = wg + static_cast<long>(e) * H;
#pragma unroll 4
  for (int h = lane * 8; h < H; h += 256) {
    float w[8];
    load8(wrow + h, w);
#pragma unroll
    for (int j = 0; j < kTok; ++j) {
      if (t0 + j < T) {
        float xv[8];
        load8(x + static_cast<long>(t0 + j) * H + h, xv);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j] = fmaf(xv[i], w[i], acc[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kTok; ++j) {
    float v = acc[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    acc[j] = v;
  }
  if (lane < kTok && t0 + lane < T) {
    float v = 0.f;
#pragma unroll
    for (int j = 0; j < kTok; ++j)
      if (j == lane) v = acc[j];
    logits[static_cast<long>(t0 + lane) * E + e] = v;
  }
}

// Split-H variant for small E (<= 32). A CTA covers one kRouterSplitCols-wide
// slice of H (blockIdx.x) and up to 8 experts (blockIdx.z picks the expert
// octet). Each lane keeps its 8 columns of those experts' router rows in
// registers, loaded once per CTA. The CTA's warps then stream token batches
// (blockIdx.y*8 + warp, then every gridDim.y*8-th batch): each lane copies its
// own 16-byte pieces of x with cp.async, kSplitDepth batches ahead, into a
// per-warp ring in shared memory and reads them back once its own copy group
// has landed, so a few KB per warp stay in flight with few registers. The
// grid is sized for two CTAs per SM. The slice sums go to partial slab
// blockIdx.x; the top-k kernel adds the slabs in slab order.
constexpr int kSplitDepth = 4;                     // token batches in flight per warp
template <typename TX>  // tokens per batch
__host__ __device__ constexpr int split_batch() { return sizeof(TX) == 2 ? 4 : 2; }
template <typename TX>
constexpr int split_smem_bytes() {                 // 8 warps x depth x batch x 32 lanes
  return 8 * kSplitDepth * split_batch<TX>() * 32 * 8 * static_cast<int>(sizeof(TX));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(ptx::smem_u32(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void unpack8(const uint4* s, __nv_bfloat16, float (&v)[8]) {
  const uint4 r = s[0];
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void unpack8(const uint4* s, float, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(s)[0];
  const float4 b = reinterpret_cast<const float4*>(s)[32];  // second piece, 32 lanes on
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Sum acc[0..7] over the 32 lanes; lane l ends up with the total of entry
// (l >> 2) & 7. Each halving step keeps half of the entries and hands the
// other half to the partner lane: 4 + 2 + 1 + 1 + 1 shuffles.
__device__ __forceinline__ float warp_sum8(const float (&acc)[8], int lane) {
  float r[4], s[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 16;
    const float keep = hi ? acc[i + 4] : acc[i];
    const float give = hi ? acc[i] : acc[i + 4];
    r[i] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 8;
    const float keep = hi ? r[i + 2] : r[i];
    const float give = hi ? r[i] : r[i + 2];
    s[i] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
  }
  const bool hi = lane & 4;
  float u = (hi ? s[1] : s[0]) + __shfl_xor_sync(0xffffffffu, hi ? s[0] : s[1], 4);
  u += __shfl_xor_sync(0xffffffffu, u, 2);
  u += __shfl_xor_sync(0xffffffffu, u, 1);
  return u;
}

template <typename TX, typename TW>
__global__ void __launch_bounds__(256, 2) router_logits_split_kernel(const TX* __restrict__ x,
                                                                     const TW* __restrict__ wg,
                                                                     float* __restrict__ logits,
                                                                     int T, int E, int H) {
  constexpr int kTB = split_batch<TX>();
  constexpr int kPieces = static_cast<int>(sizeof(TX)) / 2;  // 16-byte pieces per lane and token
  extern __shared__ uint4 xs[];  // [warp][depth][kTB][kPieces][32 lanes]
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * kRouterSplitCols + lane * 8;
  const bool hv = h < H;  // H is a multiple of 128
  const int e0 = blockIdx.z * 8;
  float w[8][8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (hv && e0 + j < E) {
      load8(wg + static_cast<long>(e0 + j) * H + h, w[j]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[j][i] = 0.f;
    }
  }
  float* slab = logits + static_cast<long>(blockIdx.x) * T * E;
  const int ex = (lane >> 2) & 7;
  uint4* ring = xs + warp * (kSplitDepth * kTB * kPieces * 32) + lane;
  const long nb = (T + kTB - 1) / kTB;
  const long stride = static_cast<long>(gridDim.y) * 8;
  const long b0 = static_cast<long>(blockIdx.y) * 8 + warp;
  // every call commits one group (possibly empty), so group i is batch i
  auto issue = [&](long b, int slot) {
    if (hv && b < nb) {
#pragma unroll
      for (int i = 0; i < kTB; ++i) {
        const long t = b * kTB + i;
        if (t < T) {
          const uint4* src = reinterpret_cast<const uint4*>(x + t * H + h);
#pragma unroll
          for (int q = 0; q < kPieces; ++q)
            cp_async16(ring + ((slot * kTB + i) * kPieces + q) * 32, src + q);
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int d = 0; d < kSplitDepth - 1; ++d) issue(b0 + d * stride, d);
  int slot = 0;
  for (long b = b0; b < nb; b += stride) {
    issue(b + (kSplitDepth - 1) * stride, (slot + kSplitDepth - 1) % kSplitDepth);
    cp_async_wait<kSplitDepth - 1>();  // this lane's copies of batch b have landed
#pragma unroll
    for (int i = 0; i < kTB; ++i) {
      const long t = b * kTB + i;
      if (t >= T) break;  // uniform over the warp
      float xv[8];
      if (hv) {
        unpack8(ring + (slot * kTB + i) * kPieces * 32, TX(), xv);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) xv[k] = 0.f;
      }
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float d = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) d = fmaf(xv[k], w[j][k], d);
        acc[j] = d;
      }
      const float v = warp_sum8(acc, lane);
      if ((lane & 3) == 0 && e0 + ex < E) slab[t * E + e0 + ex] = v;
    }
    slot = (slot + 1) % kSplitDepth;
  }
  cp_async_wait<0>();
}

// --------------------------------------------------------------- top-k
// One warp per token (large batches): logits = sum of n_part partial slabs.
template <int VPL, bool PART>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits,
                                                   int n_part, long partial_stride,
                                                   const float* __restrict__ bias, int T,
                                                   int E, int K, int renorm, int flags,
                                                   int n_group, int topk_group,
                                                   int32_t* __restrict__ ids,
                                                   float* __restrict__ wout) {
  pdl_enter();
  logits = fresh(logits);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float* row = logits + static_cast<long>(t) * E;
  float p[VPL], sb[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    p[j] = e < E ? row[e] : 0.f;
  }
  // The partial slabs of a router split over K (PART: n_part > 1) are added
  // in slab order, four slabs at a time: their loads are all issued before
  // the first add, so a token waits for one L2 round trip per four slabs, not
  // one per slab. Without slabs the variant keeps the registers of one row.
  if constexpr (PART) {
    for (int s0 = 1; s0 < n_part; s0 += 4) {
      float v[4][VPL];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const int e = lane + 32 * j;
          v[q][j] = (s0 + q < n_part && e < E) ? row[(s0 + q) * partial_stride + e] : 0.f;
        }
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int j = 0; j < VPL; ++j)
          if (s0 + q < n_part) p[j] += v[q][j];
    }
  }
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    float l = e < E ? p[j] : -CUDART_INF_F;
    sb[j] = 0.f;
    if (e < E) {
      const float b = bias ? bias[e] : 0.f;
      if (flags & kRouteBiasSelect) sb[j] = b;
      else l += b;
    }
    p[j] = l;
  }
  topk_warp<VPL>(p, sb, lane, E, K, renorm, flags, n_group, topk_group,
                 ids + static_cast<long>(t) * K, wout + static_cast<long>(t) * K);
}

// One CTA per token (small batches): all threads sum the partial slabs into
// shared memory in parallel, then warp 0 takes the decision.
template <int VPL>
__global__ void __launch_bounds__(256) topk_cta_kernel(const float* __restrict__ logits,
                                                       int n_part, long partial_stride,
                                                       const float* __restrict__ bias, int T,
                                                       int E, int K, int renorm, int flags,
                                                       int n_group, int topk_group,
                                                       int32_t* __restrict__ ids,
                                                       float* __restrict__ wout) {
  pdl_enter();
  logits = fresh(logits);
  __shared__ float sl[32 * VPL];
  const long t = blockIdx.x;
  const float* row = logits + t * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float l = row[e];
#pragma unroll 8
    for (int s = 1; s < n_part; ++s) l += row[s * partial_stride + e];
    sl[e] = l + ((bias && !(flags & kRouteBiasSelect)) ? bias[e] : 0.f);
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  float p[VPL], sb[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    p[j] = e < E ? sl[e] : -CUDART_INF_F;
    sb[j] = (e < E && bias && (flags & kRouteBiasSelect)) ? bias[e] : 0.f;
  }
  topk_warp<VPL>(p, sb, lane, E, K, renorm, flags, n_group, topk_group, ids + t * K,
                 wout + t * K);
}

// ------------------------------------------------- small batches: fused
// Routing and alignment of a small batch in one launch (T <= kRouteSmallTokens
// and the single-CTA align applies). Grid (E/8 expert octets, T/16 token
// blocks), CTAs of 1024 threads.
//   phase 1, every CTA: logits of its 8 experts x 16 tokens. Thread 0 bulk
//     copies the 8 router rows and 16 token rows (in chunks of kHC columns,
//     rows padded by 16 bytes) into shared memory, all in flight at once on
//     one mbarrier. bf16 x bf16: each warp takes a share of the 16-column K
//     steps on mma.sync m16n8k16 (fp32 accumulation) and the 32 partial
//     16x8 tiles are summed in warp order. Otherwise warp w takes expert
//     w & 7 and tokens 4*(w >> 3) .. +3 with fp32 FMA and a butterfly sum.
//   the last CTA of a token block (ticket per block) takes the decision for
//     its 16 tokens (topk_warp, one warp per token); the last of those
//     (block ticket) runs the single-CTA alignment and tile table. Each
//     ticket is reset by the CTA that drew the last number. A ticket is drawn
//     after a __syncthreads by one thread with an acquire-release atomic, so
//     the CTA's writes are published and the other CTAs' writes observed.
// A copy that does not complete in time sets MOE_DEV_TIMEOUT; the CTA still
// draws its tickets, so the tables downstream are always well formed.
constexpr int kRouteTokBlock = 16;

template <typename TX, typename TW>
struct RouteSmem {
  static constexpr int kHC = sizeof(TX) == 4 ? 1024 : 2048;  // columns per chunk
  static constexpr int kRW = kHC + 16 / static_cast<int>(sizeof(TW));  // padded row strides
  static constexpr int kRX = kHC + 16 / static_cast<int>(sizeof(TX));
  static constexpr int kW = 8 * kRW * static_cast<int>(sizeof(TW));
  static constexpr int kX = kRouteTokBlock * kRX * static_cast<int>(sizeof(TX));
  static constexpr int kHist = 4 * 32 * kSmallExperts;  // align counts, or MMA partials
  static constexpr int kBytes = kW + kX + kHist + 4 * 32 + 16 + 128;
  static constexpr bool kMma = sizeof(TX) == 2 && sizeof(TW) == 2;
};

__device__ __forceinline__ int ticket_acq_rel(int* p) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <typename TX, typename TW, int VPL>
__global__ void __launch_bounds__(1024) route_align_small_kernel(
    const TX* __restrict__ x, const TW* __restrict__ wg, const float* __restrict__ bias, int T,
    int E, int H, int K, int renorm, int flags, int n_group, int topk_group,
    float* __restrict__ logits,
    int* __restrict__ tickets, int32_t* __restrict__ ids, float* __restrict__ wout,
    const int32_t* __restrict__ emap, int R, int E_l, int ep_start, int block_m,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ sorted_ids, int32_t* __restrict__ inv_pos, int cap,
    unsigned* status, Tile* __restrict__ tiles, int* __restrict__ group_start, int nmax,
    int max_tiles) {
  using S = RouteSmem<TX, TW>;
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  TW* wbuf = reinterpret_cast<TW*>(smem);
  TX* xbuf = reinterpret_cast<TX*>(smem + S::kW);
  int* hist = reinterpret_cast<int*>(smem + S::kW + S::kX);
  int* warp_sums = hist + 32 * kSmallExperts;
  uint64_t* bar = reinterpret_cast<uint64_t*>(warp_sums + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 1);
  __shared__ int is_last;
  const uint32_t bar_a = ptx::smem_u32(bar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * 8, tb0 = blockIdx.y * kRouteTokBlock;
  const int ne = min(8, E - e0), nt = min(kRouteTokBlock, T - tb0);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_a, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();

  // the router bias of the decision warps, fetched while the logits are made
  float bv[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int ex = lane + 32 * j;
    bv[j] = (bias && warp < nt && ex < E) ? bias[ex] : 0.f;
  }

  const int el = warp & 7, ta = 4 * (warp >> 3);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  bool ok = true;
  uint32_t phase = 0;
  for (int hc0 = 0; hc0 < H && ok; hc0 += S::kHC, phase ^= 1) {
    const int hc = min(S::kHC, H - hc0);
    if (threadIdx.x == 0) {
      const uint32_t wrow = hc * sizeof(TW), xrow = hc * sizeof(TX);
      ptx::mbar_arrive_expect_tx(bar_a, ne * wrow + nt * xrow);
      for (int j = 0; j < ne; ++j)
        ptx::bulk_load(ptx::smem_u32(wbuf + j * S::kRW), wg + static_cast<long>(e0 + j) * H + hc0,
                       wrow, bar_a);
      for (int a = 0; a < nt; ++a)
        ptx::bulk_load(ptx::smem_u32(xbuf + a * S::kRX), x + static_cast<long>(tb0 + a) * H + hc0,
                       xrow, bar_a);
    }
    ok = __syncthreads_and(ptx::mbar_wait(bar_a, phase, abort_flag, status));
    if (ok) {
      if constexpr (S::kMma) {
        // acc = this warp's partial D[token][expert] over its K steps
        const uint32_t xa = ptx::smem_u32(xbuf) +
                            ((lane & 15) * S::kRX + (lane >> 4) * 8) * 2;
        const uint32_t wa = ptx::smem_u32(wbuf) + ((lane & 7) * S::kRW + ((lane >> 3) & 1) * 8) * 2;
        for (int ks = warp; ks < hc / 16; ks += 32) {
          uint32_t a[4], b[2];
          ldsm_x4(xa + ks * 32, a);
          ldsm_x2(wa + ks * 32, b);
          mma_bf16_16816(acc, a, b);
        }
      } else if (el < ne && ta < nt) {
        const TW* wr = wbuf + el * S::kRW;
        for (int h = lane * 8; h < hc; h += 256) {
          float wv[8], xv[8];
          load8(wr + h, wv);
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            if (ta + a < nt) {
              load8(xbuf + (ta + a) * S::kRX + h, xv);
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[a] = fmaf(xv[i], wv[i], acc[a]);
            }
          }
        }
      }
    }
    __syncthreads();  // the next chunk overwrites the buffers
  }
  if (!ok && threadIdx.x == 0) ptx::mbar_wait_drain(bar_a, phase);  // let late copies land
  if (ok) {
    if constexpr (S::kMma) {
      // partial tiles -> shared memory (the align counts area), then a fixed
      // order sum over the 32 warps; lane holds D rows g, g+8, columns 2c, 2c+1
      float* red = reinterpret_cast<float*>(hist);
      const int g = lane >> 2, c = 2 * (lane & 3);
      red[warp * 128 + g * 8 + c] = acc[0];
      red[warp * 128 + g * 8 + c + 1] = acc[1];
      red[warp * 128 + (g + 8) * 8 + c] = acc[2];
      red[warp * 128 + (g + 8) * 8 + c + 1] = acc[3];
      __syncthreads();
      if (threadIdx.x < 128) {
        const int r = threadIdx.x >> 3, col = threadIdx.x & 7;
        float v = 0.f;
        for (int w2 = 0; w2 < 32; ++w2) v += red[w2 * 128 + threadIdx.x];
        if (r < nt && col < ne) logits[static_cast<long>(tb0 + r) * E + e0 + col] = v;
      }
    } else if (el < ne && ta < nt) {
#pragma unroll
      for (int a = 0; a < 4; ++a) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[a] += __shfl_xor_sync(0xffffffffu, acc[a], o);
      }
      if (lane < 4 && ta + lane < nt) {
        float v = acc[0];
#pragma unroll
        for (int a = 1; a < 4; ++a)
          if (lane == a) v = acc[a];
        logits[static_cast<long>(tb0 + ta + lane) * E + e0 + el] = v;
      }
    }
  }

  // last CTA of this token block: the routing decisions of its tokens
  __syncthreads();
  if (threadIdx.x == 0) {
    is_last = ticket_acq_rel(tickets + blockIdx.y) == static_cast<int>(gridDim.x) - 1;
    if (is_last) tickets[blockIdx.y] = 0;
  }
  __syncthreads();
  if (!is_last) return;
  logits = fresh(logits);  // written by the other CTAs of this token block
  if (warp < nt) {
    const int t = tb0 + warp;
    float p[VPL], sb[VPL];
    const bool sel = flags & kRouteBiasSelect;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int ex = lane + 32 * j;
      p[j] = ex < E ? __ldcg(logits + static_cast<long>(t) * E + ex) + (sel ? 0.f : bv[j])
                    : -CUDART_INF_F;
      sb[j] = sel ? bv[j] : 0.f;
    }
    topk_warp<VPL>(p, sb, lane, E, K, renorm, flags, n_group, topk_group,
                   ids + static_cast<long>(t) * K, wout + static_cast<long>(t) * K);
  }

  // last token block: alignment of all T*K items (a single token block is
  // its own last one)
  __syncthreads();
  if (gridDim.y > 1) {
    int* block_ticket = tickets + gridDim.y;
    if (threadIdx.x == 0) {
      is_last = ticket_acq_rel(block_ticket) == static_cast<int>(gridDim.y) - 1;
      if (is_last) *block_ticket = 0;
    }
    __syncthreads();
    if (!is_last) return;
  }
  align_small_block(ids, T * K, K, emap, R, E, E_l, ep_start, block_m, counts, offsets,
                    sorted_ids, inv_pos, cap, status, tiles, group_start, nmax, max_tiles, hist,
                    warp_sums);
}

}  // namespace

template <typename TX, typename TW>
cudaError_t logits_launch(const void* x, const void* wg, float* logits, int T, int E, int H,
                          cudaStream_t st) {
  const TX* xp = static_cast<const TX*>(x);
  const TW* wp = static_cast<const TW*>(wg);
  if (E <= 32) {
    auto kern = router_logits_split_kernel<TX, TW>;
    constexpr int kSmem = split_smem_bytes<TX>();
    static std::atomic<unsigned long long> smem_set{0};  // devices, one bit each
    const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(kern), kSmem, smem_set);
    if (e != cudaSuccess) return e;
    // two CTAs per SM over (slices x token groups x expert octets)
    const long slices = router_split_slabs(H), octets = (E + 7) / 8;
    const long batches = (T + split_batch<TX>() - 1) / split_batch<TX>();
    long groups = (2L * 152) / (slices * octets);
    if (groups > (batches + 7) / 8) groups = (batches + 7) / 8;
    if (groups < 1) groups = 1;
    return launch_pdl(kern, dim3(static_cast<unsigned>(slices), static_cast<unsigned>(groups),
                                 static_cast<unsigned>(octets)),
                      dim3(256), kSmem, st, xp, wp, logits, T, E, H);
  }
  return launch_pdl(router_logits_kernel<TX, TW>, dim3((E + 7) / 8, (T + kTok - 1) / kTok),
                    dim3(256), 0, st, xp, wp, logits, T, E, H);
}

cudaError_t launch_router_logits(bool act_bf16, bool router_bf16, const void* x,
                                 const void* wg, float* logits, int T, int E, int H,
                                 cudaStream_t st) {
  if (act_bf16 && router_bf16)
    return logits_launch<__nv_bfloat16, __nv_bfloat16>(x, wg, logits, T, E, H, st);
  if (act_bf16) return logits_launch<__nv_bfloat16, float>(x, wg, logits, T, E, H, st);
  return logits_launch<float, float>(x, wg, logits, T, E, H, st);
}

template <int V>
cudaError_t topk_launch(const float* logits, int n_part, long partial_stride, const float* bias,
                        int T, int E, int K, int renorm, int flags, int n_group,
                        int topk_group, int32_t* ids, float* w, cudaStream_t st) {
  if (T < 256)
    return launch_pdl(topk_cta_kernel<V>, dim3(T), dim3(256), 0, st, logits, n_part,
                      partial_stride, bias, T, E, K, renorm, flags, n_group, topk_group, ids,
                      w);
  if (n_part > 1)
    return launch_pdl(topk_kernel<V, true>, dim3((T + 7) / 8), dim3(256), 0, st, logits, n_part,
                      partial_stride, bias, T, E, K, renorm, flags, n_group, topk_group, ids,
                      w);
  return launch_pdl(topk_kernel<V, false>, dim3((T + 7) / 8), dim3(256), 0, st, logits, n_part,
                    partial_stride, bias, T, E, K, renorm, flags, n_group, topk_group, ids, w);
}

template <typename TX, typename TW, int VPL>
cudaError_t route_align_launch(const RouteAlignArgs& a, cudaStream_t st) {
  using S = RouteSmem<TX, TW>;
  auto kern = route_align_small_kernel<TX, TW, VPL>;
  static std::atomic<unsigned long long> smem_set{0};  // devices, one bit each
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(kern), S::kBytes, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((a.E + 7) / 8, (a.T + kRouteTokBlock - 1) / kRouteTokBlock),
                    dim3(1024), S::kBytes, st, static_cast<const TX*>(a.x),
                    static_cast<const TW*>(a.wg), a.bias, a.T,
                    a.E, a.H, a.K, a.renorm, a.flags, a.n_group, a.topk_group, a.logits,
                    a.tickets, a.ids,
                    a.w, a.emap, a.R, a.E_l, a.ep_start, a.block_m, a.counts, a.offsets,
                    a.sorted_ids, a.inv_pos, a.cap, a.status, a.tiles, a.group_start, a.nmax,
                    a.max_tiles);
}

template <typename TX, typename TW>
cudaError_t route_align_vpl(const RouteAlignArgs& a, cudaStream_t st) {
  const int vpl = (a.E + 31) / 32;
  if (vpl <= 1) return route_align_launch<TX, TW, 1>(a, st);
  if (vpl <= 2) return route_align_launch<TX, TW, 2>(a, st);
  if (vpl <= 4) return route_align_launch<TX, TW, 4>(a, st);
  if (vpl <= 8) return route_align_launch<TX, TW, 8>(a, st);
  if (vpl <= 16) return route_align_launch<TX, TW, 16>(a, st);
  return cudaErrorInvalidValue;
}

bool route_align_small_ok(int T, int K, int E_l) {
  return T >= 1 && T <= kRouteSmallTokens && static_cast<long>(T) * K <= kSmallItems &&
         E_l <= kSmallExperts;
}

cudaError_t launch_route_align_small(const RouteAlignArgs& a, bool act_bf16, bool router_bf16,
                                     cudaStream_t st) {
  if (!route_align_small_ok(a.T, a.K, a.E_l)) return cudaErrorInvalidValue;
  if (act_bf16 && router_bf16) return route_align_vpl<__nv_bfloat16, __nv_bfloat16>(a, st);
  if (act_bf16) return route_align_vpl<__nv_bfloat16, float>(a, st);
  return route_align_vpl<float, float>(a, st);
}

cudaError_t launch_topk(const float* logits, int n_part, long partial_stride,
                        const float* bias, int T, int E, int K, int renorm, int flags,
                        int n_group, int topk_group, int32_t* ids, float* w,
                        unsigned* /*status*/, cudaStream_t st) {
  const int vpl = (E + 31) / 32;
  if (vpl <= 1) return topk_launch<1>(logits, n_part, partial_stride, bias, T, E, K, renorm,
                                      flags, n_group, topk_group, ids, w, st);
  if (vpl <= 2) return topk_launch<2>(logits, n_part, partial_stride, bias, T, E, K, renorm,
                                      flags, n_group, topk_group, ids, w, st);
  if (vpl <= 4) return topk_launch<4>(logits, n_part, partial_stride, bias, T, E, K, renorm,
                                      flags, n_group, topk_group, ids, w, st);
  if (vpl <= 8) return topk_launch<8>(logits, n_part, partial_stride, bias, T, E, K, renorm,
                                      flags, n_group, topk_group, ids, w, st);
  if (vpl <= 16) return topk_launch<16>(logits, n_part, partial_stride, bias, T, E, K, renorm,
                                        flags, n_group, topk_group, ids, w, st);
  return cudaErrorInvalidValue;
}

MOE_WAIT_LIMIT_SETTER(set_wait_limit_route)
MOE_DEBUG_TAKER(take_dbg_route)

}  // namespace moe
