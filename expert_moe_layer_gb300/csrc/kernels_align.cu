// Token alignment / permutation by local expert, GEMM tile tables, row gather
// and the weighted combine.
//
// Work item i = t*K + k (token t, slot k) is the flattening of
// ep_fused_moe_patch.py _ep_forward step 2. Segments are a stable counting
// sort of the items by local expert id. A warp owns kItemsPerWarp
// consecutive items. Pass 1 counts them per expert (match_any groups the
// lanes with equal keys). Pass 2 turns the counts into padded offsets and
// into a base row per (warp, expert). Pass 3 replays the same walk in the
// same order and writes each item to base + rank, so the order inside a
// segment is ascending item order with no atomics on global memory.
#include <cuda_bf16.h>

#include "align_block.cuh"
#include "act.cuh"
#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
[[maybe_unused]] constexpr DbgFile kDbgFileCode = kDbgAlign;
namespace {

constexpr int kItemsPerWarp = 256;
constexpr int kWarpsPerBlock = 8;

// Pass 1: per-warp expert counts; also fills sorted_ids with the sentinel.
__global__ void __launch_bounds__(256) align_count_kernel(
    const int32_t* __restrict__ ids, long n_items, int K, const int32_t* __restrict__ emap, int R,
    int E, int E_l, int ep_start, int* __restrict__ hist, int n_warps,
    int32_t* __restrict__ sorted_ids, int cap, unsigned* status) {
  pdl_enter();
  ids = fresh(ids);
  extern __shared__ int cnt[];  // [kWarpsPerBlock][E_l]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (long r = blockIdx.x * 256L + threadIdx.x; r < cap; r += 256L * gridDim.x)
    sorted_ids[r] = static_cast<int32_t>(n_items);
  for (int i = threadIdx.x; i < kWarpsPerBlock * E_l; i += 256) cnt[i] = 0;
  __syncthreads();
  const int gw = blockIdx.x * kWarpsPerBlock + warp;
  if (gw >= n_warps) return;
  int* my = cnt + warp * E_l;
  const long base = static_cast<long>(gw) * kItemsPerWarp;
  int idv[kItemsPerWarp / 32];  // all of this lane's ids in flight at once
#pragma unroll
  for (int i = 0; i < kItemsPerWarp / 32; ++i) {
    const long item = base + 32 * i + lane;
    idv[i] = item < n_items ? ids[item] : 0;
  }
#pragma unroll
  for (int i = 0; i < kItemsPerWarp / 32; ++i) {
    const long item = base + 32 * i + lane;
    int le = -1;
    if (item < n_items)
      le = local_expert(idv[i], static_cast<int>(item / K), emap, R, E, E_l, ep_start, status);
    const unsigned peers = __match_any_sync(0xffffffffu, le);
    if (le >= 0 && lane == __ffs(peers) - 1) my[le] += __popc(peers);
    __syncwarp();
  }
  for (int e = lane; e < E_l; e += 32) hist[static_cast<long>(gw) * E_l + e] = my[e];
}

// Pass 2 (one CTA): counts, padded exclusive offsets, and per-warp base rows
// written back into hist. G = 1024 / E_l threads share each expert's column
// of hist: thread (g, e) sums warps [g*R, (g+1)*R), the partial sums are
// turned into per-group prefixes, and each thread then rewrites its own range.
__global__ void __launch_bounds__(1024) align_scan_kernel(int* __restrict__ hist, int n_warps,
                                                          int E_l, int block_m,
                                                          int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets,
                                                          int cap, unsigned* status,
                                                          Tile* __restrict__ tiles,
                                                          int* __restrict__ group_start,
                                                          int nmax, int max_tiles) {
  pdl_enter();
  hist = fresh(hist);
  __shared__ int warp_sums[32];
  __shared__ int part[1024];   // per-(group, expert) sums, then their exclusive prefixes
  __shared__ int sbase[1024];  // each expert's first row
  const int G = E_l >= 1024 ? 1 : 1024 / E_l;
  const bool active = threadIdx.x < G * E_l;
  const int ge = active ? threadIdx.x % E_l : 0, g = active ? threadIdx.x / E_l : 0;
  const int R = (n_warps + G - 1) / G;
  const int w0 = min(n_warps, g * R), w1 = min(n_warps, w0 + R);
  int sum = 0;
  if (active) {
#pragma unroll 8
    for (int w = w0; w < w1; ++w) sum += hist[static_cast<long>(w) * E_l + ge];
    part[threadIdx.x] = sum;
  }
  __syncthreads();
  const int e = threadIdx.x;
  int c = 0;
  if (e < E_l) {
    for (int gg = 0; gg < G; ++gg) {
      const int v = part[gg * E_l + e];
      part[gg * E_l + e] = c;
      c += v;
    }
  }
  const int padded = e < E_l ? ((c + block_m - 1) / block_m) * block_m : 0;
  // block-wide inclusive scan of padded
  int v = padded;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int s2 = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, s2, o);
      if (lane >= o) s2 += n;
    }
    warp_sums[lane] = s2;
  }
  __syncthreads();
  const int incl = v + (wid > 0 ? warp_sums[wid - 1] : 0);
  if (e < E_l) {
    const int start = incl - padded;
    counts[e] = c;
    offsets[e] = start;
    sbase[e] = start;
    if (e == E_l - 1) {
      offsets[E_l] = incl;
      if (incl > cap && status) atomicOr(status, MOE_DEV_CAP_OVERFLOW);
    }
  }
  __syncthreads();
  if (active) {
    int run = sbase[ge] + part[threadIdx.x];
#pragma unroll 8
    for (int w = w0; w < w1; ++w) {
      const long idx = static_cast<long>(w) * E_l + ge;
      const int h = hist[idx];
      hist[idx] = run;
      run += h;
    }
  }
  if (tiles)
    write_tile_table(e, E_l, e < E_l ? c : 0, incl - padded, nmax, tiles, group_start,
                     max_tiles, warp_sums, status);
}

// Pass 3: stable scatter of item ids into their segments.
__global__ void __launch_bounds__(256) align_scatter_kernel(
    const int32_t* __restrict__ ids, long n_items, int K, const int32_t* __restrict__ emap, int R,
    int E, int E_l, int ep_start, const int* __restrict__ hist, int n_warps,
    int32_t* __restrict__ sorted_ids, int32_t* __restrict__ inv_pos, int cap,
    unsigned* status) {
  pdl_enter();
  ids = fresh(ids);
  hist = fresh(hist);
  extern __shared__ int run[];  // [kWarpsPerBlock][E_l]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kWarpsPerBlock + warp;
  if (gw >= n_warps) return;
  int* my = run + warp * E_l;
  const long base = static_cast<long>(gw) * kItemsPerWarp;
  int idv[kItemsPerWarp / 32];  // all of this lane's ids in flight at once
#pragma unroll
  for (int i = 0; i < kItemsPerWarp / 32; ++i) {
    const long item = base + 32 * i + lane;
    idv[i] = item < n_items ? ids[item] : 0;
  }
  for (int e = lane; e < E_l; e += 32) my[e] = hist[static_cast<long>(gw) * E_l + e];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < kItemsPerWarp / 32; ++i) {
    const long item = base + 32 * i + lane;
    int le = -1;
    // status already recorded by pass 1 for bad ids
    if (item < n_items)
      le = local_expert(idv[i], static_cast<int>(item / K), emap, R, E, E_l, ep_start, nullptr);
    const unsigned peers = __match_any_sync(0xffffffffu, le);
    if (item < n_items) {
      int pos = -1;
      if (le >= 0) {
        pos = my[le] + __popc(peers & lt);
        if (pos < cap) {
          sorted_ids[pos] = static_cast<int32_t>(item);
        } else {
          if (status) atomicOr(status, MOE_DEV_CAP_OVERFLOW);
          pos = -1;
        }
      }
      inv_pos[item] = pos;
    }
    __syncwarp();
    if (le >= 0 && lane == __ffs(peers) - 1) my[le] += __popc(peers);
    __syncwarp();
  }
}

// Two passes, where E_l <= 256 and the per-CTA counts are few (at most
// kFoldHist entries): CTAs of kFoldWarps warps x kFoldItemsPerWarp items.
// The count pass writes one row of expert counts per CTA. In the second pass
// every CTA sums each expert's column itself (all rows for the count, the
// rows before its own for its base), so no single-CTA scan runs between two
// grid-wide passes; it counts its own warps' items again in shared memory for
// their bases and places them. CTA 0 writes counts, offsets and the tile
// table. The order of the items is that of the three passes.
constexpr long kFoldHist = 32768;
constexpr int kFoldItemsPerWarp = 64;
constexpr int kFoldWarps = 8;
constexpr int kFoldItems = kFoldItemsPerWarp * kFoldWarps;  // per CTA

__global__ void __launch_bounds__(256) align_fold_count_kernel(
    const int32_t* __restrict__ ids, long n_items, int K, const int32_t* __restrict__ emap, int R,
    int E, int E_l, int ep_start, int* __restrict__ bhist, int32_t* __restrict__ sorted_ids,
    int cap, unsigned* status) {
  pdl_enter();
  ids = fresh(ids);
  __shared__ int cnt[256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (long r = blockIdx.x * 256L + threadIdx.x; r < cap; r += 256L * gridDim.x)
    sorted_ids[r] = static_cast<int32_t>(n_items);
  if (threadIdx.x < E_l) cnt[threadIdx.x] = 0;
  __syncthreads();
  const long base = static_cast<long>(blockIdx.x) * kFoldItems + warp * kFoldItemsPerWarp;
  int idv[kFoldItemsPerWarp / 32];
#pragma unroll
  for (int i = 0; i < kFoldItemsPerWarp / 32; ++i) {
    const long item = base + 32 * i + lane;
    idv[i] = item < n_items ? ids[item] : 0;
  }
#pragma unroll
  for (int i = 0; i < kFoldItemsPerWarp / 32; ++i) {
    const long item = base + 32 * i + lane;
    int le = -1;
    if (item < n_items)
      le = local_expert(idv[i], static_cast<int>(item / K), emap, R, E, E_l, ep_start, status);
    const unsigned peers = __match_any_sync(0xffffffffu, le);
    if (le >= 0 && lane == __ffs(peers) - 1) atomicAdd(&cnt[le], __popc(peers));
  }
  __syncthreads();
  if (threadIdx.x < E_l)
    bhist[static_cast<long>(blockIdx.x) * E_l + threadIdx.x] = cnt[threadIdx.x];
}

__global__ void __launch_bounds__(256) align_fold_scatter_kernel(
    const int32_t* __restrict__ ids, long n_items, int K, const int32_t* __restrict__ emap, int R,
    int E, int E_l, int ep_start, const int* __restrict__ bhist, int n_blocks, int block_m,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ sorted_ids, int32_t* __restrict__ inv_pos, int cap, unsigned* status,
    Tile* __restrict__ tiles, int* __restrict__ group_start, int nmax, int max_tiles) {
  pdl_enter();
  ids = fresh(ids);
  bhist = fresh(bhist);
  __shared__ int run[kFoldWarps][256];  // per-warp counts, then the warps' next rows
  __shared__ int warp_sums[32];
  __shared__ int part_c[256], part_b[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = threadIdx.x;
  for (int i = threadIdx.x; i < kFoldWarps * 256; i += 256) (&run[0][0])[i] = 0;
  const long base = static_cast<long>(blockIdx.x) * kFoldItems + warp * kFoldItemsPerWarp;
  int idv[kFoldItemsPerWarp / 32];  // this lane's ids, loaded before the column sums
#pragma unroll
  for (int i = 0; i < kFoldItemsPerWarp / 32; ++i) {
    const long item = base + 32 * i + lane;
    idv[i] = item < n_items ? ids[item] : 0;
  }
  // G = 256 / E_l threads share each expert's column of the per-CTA counts:
  // thread (g, e') sums the rows b = g, g + G, ... (all of them for the
  // count, those before this CTA for its base); the G partial sums are then
  // added in order
  {
    const int G = 256 / E_l;
    const int ge = threadIdx.x % E_l, g = threadIdx.x / E_l;
    int pc = 0, pb = 0;
    if (g < G) {
#pragma unroll 16
      for (int b = g; b < n_blocks; b += G) {
        const int h = bhist[static_cast<long>(b) * E_l + ge];
        if (b < static_cast<int>(blockIdx.x)) pb += h;
        pc += h;
      }
    }
    part_c[threadIdx.x] = pc;
    part_b[threadIdx.x] = pb;
  }
  __syncthreads();  // run zeroed, partial sums in
  // this CTA's items: their local experts, and each warp's count per expert
  int lev[kFoldItemsPerWarp / 32];
  unsigned pev[kFoldItemsPerWarp / 32];
#pragma unroll
  for (int i = 0; i < kFoldItemsPerWarp / 32; ++i) {
    const long item = base + 32 * i + lane;
    int le = -1;
    // status already recorded by the count pass for bad ids
    if (item < n_items)
      le = local_expert(idv[i], static_cast<int>(item / K), emap, R, E, E_l, ep_start, nullptr);
    const unsigned peers = __match_any_sync(0xffffffffu, le);
    lev[i] = le;
    pev[i] = peers;
    if (le >= 0 && lane == __ffs(peers) - 1) run[warp][le] += __popc(peers);
    __syncwarp();
  }
  int c = 0, before = 0;
  if (e < E_l) {
    for (int g = 0; g < 256 / E_l; ++g) {
      c += part_c[g * E_l + e];
      before += part_b[g * E_l + e];
    }
  }
  const int padded = e < E_l ? ((c + block_m - 1) / block_m) * block_m : 0;
  int total = 0;
  // (the scan's barriers also make every warp's counts visible below)
  const int start = block_exclusive_scan(padded, warp_sums, total);
  if (blockIdx.x == 0) {
    if (e < E_l) {
      counts[e] = c;
      offsets[e] = start;
    }
    if (threadIdx.x == 0) {
      offsets[E_l] = total;
      if (total > cap && status) atomicOr(status, MOE_DEV_CAP_OVERFLOW);
    }
    if (tiles)
      write_tile_table(e, E_l, e < E_l ? c : 0, start, nmax, tiles, group_start, max_tiles,
                       warp_sums, status);
  }
  if (e < E_l) {
    int r = start + before;
    for (int wi = 0; wi < kFoldWarps; ++wi) {
      const int n = run[wi][e];
      run[wi][e] = r;
      r += n;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < kFoldItemsPerWarp / 32; ++i) {
    const long item = base + 32 * i + lane;
    const int le = lev[i];
    const unsigned peers = pev[i];
    if (item < n_items) {
      int pos = -1;
      if (le >= 0) {
        pos = run[warp][le] + __popc(peers & lt);
        if (pos < cap) {
          sorted_ids[pos] = static_cast<int32_t>(item);
        } else {
          if (status) atomicOr(status, MOE_DEV_CAP_OVERFLOW);
          pos = -1;
        }
      }
      inv_pos[item] = pos;
    }
    __syncwarp();
    if (le >= 0 && lane == __ffs(peers) - 1) run[warp][le] += __popc(peers);
    __syncwarp();
  }
}

// Small inputs (n_items <= kSmallItems, E_l <= kSmallExperts): the three
// passes above in one CTA of 32 warps (align_small_block).
__global__ void __launch_bounds__(1024) align_small_kernel(
    const int32_t* __restrict__ ids, int n_items, int K, const int32_t* __restrict__ emap, int R,
    int E, int E_l, int ep_start, int block_m, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
    int32_t* __restrict__ inv_pos, int cap, unsigned* status, Tile* __restrict__ tiles,
    int* __restrict__ group_start, int nmax, int max_tiles) {
  pdl_enter();
  ids = fresh(ids);
  __shared__ int hist[32 * kSmallExperts];
  __shared__ int warp_sums[32];
  align_small_block(ids, n_items, K, emap, R, E, E_l, ep_start, block_m, counts, offsets,
                    sorted_ids, inv_pos, cap, status, tiles, group_start, nmax, max_tiles, hist,
                    warp_sums);
}

// Tile table of the routed experts: each segment's rows in chunks of nmax.
__global__ void __launch_bounds__(1024) build_tiles_kernel(const int32_t* __restrict__ counts,
                                                           const int32_t* __restrict__ offsets,
                                                           int E_l, int nmax, Tile* __restrict__ tiles,
                                                           int* __restrict__ group_start,
                                                           int max_tiles, int cap,
                                                           unsigned* status) {
  pdl_enter();
  counts = fresh(counts);
  offsets = fresh(offsets);
  __shared__ int warp_sums[32];
  const int e = threadIdx.x;
  int n = 0, c = 0, off = 0;
  if (e < E_l) {
    c = counts[e];
    off = offsets[e];
    // a segment must lie inside [0, cap) and end before the next one starts
    if (c < 0 || off < 0 || off > cap - c || off + c > offsets[e + 1]) {
      if (status) atomicOr(status, MOE_DEV_BAD_SEGMENT);
      c = 0;
    }
    n = (c + nmax - 1) / nmax;
  }
  int v = n;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += x;
  }
  if (lane == 31) warp_sums[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += x;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int incl = v + (wid > 0 ? warp_sums[wid - 1] : 0);
  const int start = incl - n;
  for (int j = 0; j < n; ++j) {
    const int idx = start + j;
    if (idx < max_tiles) {
      const int r0 = off + j * nmax;
      const int rows = c - j * nmax < nmax ? c - j * nmax : nmax;
      tiles[idx] = make_int4(e, r0, r0, rows);
    }
  }
  if (e < E_l) group_start[e] = start < max_tiles ? start : max_tiles;
  if (threadIdx.x == blockDim.x - 1) {
    const int total = incl;
    if (total > max_tiles && status) atomicOr(status, MOE_DEV_CAP_OVERFLOW);
    group_start[E_l] = total < max_tiles ? total : max_tiles;
  }
}

// x_perm[r] = x[sorted_ids[r] / K], one warp per row, 16-byte vectors; with
// w_perm also w_perm[r] = w_items[sorted_ids[r]].
template <typename TE>
__global__ void __launch_bounds__(256) gather_kernel(const TE* __restrict__ x,
                                                     const int32_t* __restrict__ sorted_ids,
                                                     const int32_t* __restrict__ offsets_end,
                                                     int cap, long n_items, int K, int H,
                                                     TE* __restrict__ x_perm,
                                                     const float* __restrict__ w_items,
                                                     float* __restrict__ w_perm) {
  pdl_enter();
  sorted_ids = fresh(sorted_ids);
  offsets_end = fresh(offsets_end);
  w_items = fresh(w_items);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int rows = *offsets_end;
  if (rows > cap) rows = cap;
  constexpr int kVec = 16 / sizeof(TE);
  for (long r = blockIdx.x * 8L + warp; r < rows; r += 8L * gridDim.x) {
    const int id = sorted_ids[r];
    if (id < 0 || id >= n_items) continue;
    if (!MOE_DCHECK(r, cap) || !MOE_DCHECK(id / K, n_items / K)) continue;
    if (w_perm && lane == 0) w_perm[r] = w_items[id];
    const uint4* src = reinterpret_cast<const uint4*>(x + (id / K) * static_cast<long>(H));
    uint4* dst = reinterpret_cast<uint4*>(x_perm + r * H);
    for (int c = lane; c < H / kVec; c += 32) dst[c] = src[c];
  }
}

// 8 consecutive fp32 values (two 16-byte loads) and 8 outputs in one store.
__device__ __forceinline__ void ld8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 r;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = r;
}
__device__ __forceinline__ void st8(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// The SiLU*up epilogue of a GEMM1 split over K: sums the fp32 partial gate
// and up accumulators in slab order. One warp per (row, 256-column chunk).
template <typename TE>
__global__ void __launch_bounds__(256) silu_finalize_kernel(const float* __restrict__ part,
                                                            int n_part, long part_stride,
                                                            const int32_t* __restrict__ rows_dev,
                                                            int cap, int I, TE* __restrict__ h) {
  pdl_enter();
  part = fresh(part);
  rows_dev = fresh(rows_dev);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int rows = *rows_dev;
  if (rows > cap) rows = cap;
  const int chunks = (I + 255) / 256;
  const long tasks = static_cast<long>(rows) * chunks;
  for (long task = blockIdx.x * 8L + warp; task < tasks; task += 8L * gridDim.x) {
    const long r = task / chunks;
    const int c = static_cast<int>(task - r * chunks) * 256 + lane * 8;
    if (c >= I) continue;
    float g[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float u[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < n_part; ++s) {
      const float* src = part + s * part_stride + r * (2L * I) + c;
      float a[8], b[8];
      ld8(src, a);
      ld8(src + I, b);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        g[i] += a[i];
        u[i] += b[i];
      }
    }
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = silu(g[i]) * u[i];
    st8(h + r * I + c, o);
  }
}

// A CTA takes tpc consecutive tokens (at most kCombTok). Its warps first
// stage each token's slots into shared memory: position and weight of the
// slots whose row is local, compacted in slot order so the accumulation keeps
// the fixed order k = 0..K-1. Then one warp step = one token x U consecutive
// 256-column chunks (8 columns per lane per chunk), U = 4 / KB for KB < 4:
// the rows of up to KB slots for all U chunks (plus, with U = 1, up to two
// shared experts) are loaded together as raw 16-byte vectors, so at least
// four loads per lane are in flight whatever top_k is, then summed in slot
// order.
constexpr int kCombTok = 8;

__device__ __forceinline__ void raw8_add(float (&acc)[8], const uint4& r, float w) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
  }
}
__device__ __forceinline__ void raw8_add(float (&acc)[8], const float4 (&r)[2], float w) {
  acc[0] = fmaf(w, r[0].x, acc[0]); acc[1] = fmaf(w, r[0].y, acc[1]);
  acc[2] = fmaf(w, r[0].z, acc[2]); acc[3] = fmaf(w, r[0].w, acc[3]);
  acc[4] = fmaf(w, r[1].x, acc[4]); acc[5] = fmaf(w, r[1].y, acc[5]);
  acc[6] = fmaf(w, r[1].z, acc[6]); acc[7] = fmaf(w, r[1].w, acc[7]);
}
template <typename TE> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
  uint4 v;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void add_to(float (&acc)[8], float w) const { raw8_add(acc, v, w); }
};
template <> struct Raw8<float> {
  float4 v[2];
  __device__ __forceinline__ void load(const float* p) {
    v[0] = *reinterpret_cast<const float4*>(p);
    v[1] = *reinterpret_cast<const float4*>(p + 4);
  }
  __device__ __forceinline__ void add_to(float (&acc)[8], float w) const { raw8_add(acc, v, w); }
};

// CTAs per SM from the registers a variant holds: fp32 rows take twice the
// registers of bf16 ones; KB = 1 keeps four column chunks in flight.
template <typename TE, int KB>
constexpr int combine_ctas_per_sm() {
  return sizeof(TE) == 4 ? 2 : (KB > 4 || KB == 1) ? 3 : 4;
}

template <typename TE, int KB>
__global__ void __launch_bounds__(256, (combine_ctas_per_sm<TE, KB>())) combine_kernel(
    const TE* __restrict__ y_perm, int cap, const int32_t* __restrict__ inv_pos,
    const float* __restrict__ topk_w, int K, const TE* __restrict__ shared, int n_shared,
    long shared_stride, float rsf, TE* __restrict__ out, int T, int H, int tpc,
    int slots_early, unsigned* status) {
  constexpr int U = KB >= 4 ? 1 : 4 / KB;  // chunks per warp step
  // slots_early: inv_pos and topk_w were written at least two kernels back,
  // so they are staged before the dependency wait, while the kernel before
  // finishes; the rows of y_perm and shared are read only after it.
  if (!slots_early) {
    pdl_enter();
    inv_pos = fresh(inv_pos);
    topk_w = fresh(topk_w);
  }
  __shared__ int s_pos[kCombTok][32];
  __shared__ float s_w[kCombTok][32];
  __shared__ int s_n[kCombTok];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long t0 = static_cast<long>(blockIdx.x) * tpc;
  for (int tt = warp; tt < tpc; tt += 8) {
    const long t = t0 + tt;
    int p = -1;
    float w = 0.f;
    if (t < T && lane < K) {
      p = inv_pos[t * K + lane];
      w = topk_w ? topk_w[t * K + lane] : 1.f;
      if (p >= cap) {
        if (status) atomicOr(status, MOE_DEV_BAD_SEGMENT);
        p = -1;
      }
    }
    const unsigned local = __ballot_sync(0xffffffffu, p >= 0);
    if (p >= 0) {
      const int j = __popc(local & ((1u << lane) - 1u));
      s_pos[tt][j] = p;
      s_w[tt][j] = w;
    }
    if (lane == 0) s_n[tt] = __popc(local);
  }
  if (slots_early) pdl_enter();
  y_perm = fresh(y_perm);
  shared = fresh(shared);
  __syncthreads();
  const int chunks = (H + 255) / 256;
  const int steps = (chunks + U - 1) / U;  // warp steps per token
  for (int task = warp; task < tpc * steps; task += 8) {
    const int tt = task / steps;
    const long t = t0 + tt;
    if (t >= T) continue;
    const int cb = (task - tt * steps) * U * 256 + lane * 8;
    const int n = s_n[tt];
    Raw8<TE> sh[2];
    const int ns0 = U == 1 ? (n_shared < 2 ? n_shared : 2) : 0;
    if (cb < H)
      for (int s = 0; s < ns0; ++s) sh[s].load(shared + s * shared_stride + t * H + cb);
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
    for (int j0 = 0; j0 < n; j0 += KB) {
      Raw8<TE> y[KB][U];
#pragma unroll
      for (int j = 0; j < KB; ++j) {
        if (j0 + j < n) {
          const int pos = s_pos[tt][j0 + j];
          const TE* row = y_perm + static_cast<long>(MOE_DCHECK(pos, cap) ? pos : 0) * H;
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (cb + u * 256 < H) y[j][u].load(row + cb + u * 256);
        }
      }
#pragma unroll
      for (int j = 0; j < KB; ++j) {
        if (j0 + j < n) {
          const float w = s_w[tt][j0 + j];
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (cb + u * 256 < H) y[j][u].add_to(acc[u], w);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = cb + u * 256;
      if (c >= H) continue;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[u][i] *= rsf;
      for (int s = 0; s < ns0; ++s) sh[s].add_to(acc[u], 1.f);
      for (int s = ns0; s < n_shared; ++s) {
        Raw8<TE> r;
        r.load(shared + s * shared_stride + t * H + c);
        r.add_to(acc[u], 1.f);
      }
      st8(out + t * H + c, acc[u]);
    }
  }
}

// Expert-parallel dispatch (ep_fused_moe_patch.py _ep_forward step 2):
// destination rank of each work item, -1 for an id outside [0, E).
__global__ void __launch_bounds__(256) ep_dest_kernel(const int32_t* __restrict__ ids,
                                                      long n, int E, int n_local,
                                                      int32_t* __restrict__ dest,
                                                      int32_t* __restrict__ phys,
                                                      const int32_t* __restrict__ phys_map,
                                                      int R, int K, int E_phys) {
  pdl_enter();
  ids = fresh(ids);
  for (long i = blockIdx.x * 256L + threadIdx.x; i < n; i += 256L * gridDim.x) {
    const int id = ids[i];
    int p = -1;
    if (id >= 0 && id < E) {
      if (phys_map) {
        // replica t mod n_e of the id's replicas (a prefix of its row)
        const int32_t* row = phys_map + static_cast<long>(id) * R;
        int nrep = 0;
        while (nrep < R && row[nrep] != -2) ++nrep;
        if (nrep > 0) {
          const int q = row[(i / K) % nrep];
          if (q >= 0 && q < E_phys) p = q;
        }
      } else {
        p = id;
      }
    }
    phys[i] = p;
    dest[i] = p >= 0 ? p / n_local : -1;
  }
}

// Rows of items that the align step dropped (inv_pos < 0) are zeroed; the
// others were written by the scattering GEMM2. Row bytes are a multiple of 16.
__global__ void __launch_bounds__(256) zero_dropped_rows_kernel(const int32_t* __restrict__ inv_pos,
                                                                long n, long row_bytes,
                                                                uint8_t* __restrict__ y) {
  pdl_enter();
  inv_pos = fresh(inv_pos);
  for (long i = blockIdx.x * 256L + threadIdx.x; i < n; i += 256L * gridDim.x) {
    if (inv_pos[i] >= 0) continue;
    int4* row = reinterpret_cast<int4*>(y + i * row_bytes);
    for (long c = 0; c < row_bytes / 16; ++c) row[c] = make_int4(0, 0, 0, 0);
  }
}

// Send buffers in destination order: row r holds item sorted_ids[r] (one
// warp per row, 16-byte vectors for the hidden row).
template <typename TE>
__global__ void __launch_bounds__(256) ep_pack_kernel(
    const TE* __restrict__ x, const int32_t* __restrict__ ids, const float* __restrict__ w,
    const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ rows_dev, long n_items,
    int K, int H, TE* __restrict__ send_x, int32_t* __restrict__ send_ids,
    float* __restrict__ send_w, int32_t* __restrict__ send_tok) {
  pdl_enter();
  x = fresh(x);
  ids = fresh(ids);
  w = fresh(w);
  sorted_ids = fresh(sorted_ids);
  rows_dev = fresh(rows_dev);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long rows = *rows_dev;
  if (rows > n_items) rows = n_items;
  constexpr int kVec = 16 / sizeof(TE);
  for (long r = blockIdx.x * 8L + warp; r < rows; r += 8L * gridDim.x) {
    const int item = sorted_ids[r];
    if (item < 0 || item >= n_items) continue;
    const long t = item / K;
    if (lane == 0) {
      send_ids[r] = ids[item];
      send_w[r] = w[item];
      send_tok[r] = static_cast<int32_t>(t);
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    uint4* dst = reinterpret_cast<uint4*>(send_x + r * H);
    for (int c = lane; c < H / kVec; c += 32) dst[c] = src[c];
  }
}

// ------------------------------------------------------------ ring combine
// The same combine for prefill-sized batches, with the rows streamed through
// shared memory. Each CTA (one per SM) takes a contiguous range of tokens.
// Warp 0 stages the slot positions and weights of up to kRingMetaTok tokens at
// a time, then for each token copies its local rows of y_perm and its shared
// expert rows with bulk copies (one row per lane) into a ring of row slots,
// kRingEntries tokens ahead of the reducers. Warps 1..8 wait for a token's
// rows, sum them across the columns (8 per thread and pass) in the same order
// and with the same roundings as combine_kernel, store the output row and
// release the token's slots. Up to kRingBytes of rows per SM are in flight,
// against a few KB per warp for register loads.
constexpr int kRingThreads = 288;           // warp 0 copies, warps 1..8 sum
constexpr int kRingEntries = 32;            // tokens in the ring at most
constexpr int kRingMetaTok = 64;            // tokens whose slots are staged at once
constexpr int kRingBytes = 192 * 1024;      // row slots
constexpr int kRingMinTokens = 1024;        // fewer tokens: combine_kernel
// Bulk copies complete at about two per microsecond per SM whatever their
// size, so the ring pays only where a token brings many bytes (its expected
// local rows and the shared rows): DeepSeek-V2's eight 10 KB rows, not an EP
// shard's two 4 KB rows.
constexpr long kRingMinTokenBytes = 48 * 1024;
constexpr int kRingCtas = 152;              // one per SM
struct RingEntry {
  int n;          // local rows (weighted), then the shared rows
  int slot0;      // first row slot (the token's rows wrap around the ring)
  int tok;
  int pad;
  float w[32];    // weights of the local rows, in slot order
};
constexpr int kRingSmem = kRingBytes + kRingMetaTok * 32 * 8 + kRingEntries * sizeof(RingEntry) +
                          2 * kRingEntries * 8 + 16 + 128;

template <typename TE>
__global__ void __launch_bounds__(kRingThreads, 1) combine_ring_kernel(
    const TE* __restrict__ y_perm, int cap, const int32_t* __restrict__ inv_pos,
    const float* __restrict__ topk_w, int K, const TE* __restrict__ shared, int n_shared,
    long shared_stride, float rsf, TE* __restrict__ out, int T, int H, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* rows = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  int* meta_p = reinterpret_cast<int*>(rows + kRingBytes);      // [kRingMetaTok][K]
  float* meta_w = reinterpret_cast<float*>(meta_p + kRingMetaTok * 32);
  RingEntry* ent = reinterpret_cast<RingEntry*>(meta_w + kRingMetaTok * 32);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ent + kRingEntries);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kRingEntries);
  const uint32_t full0 = ptx::smem_u32(bars);           // [entry]: the token's rows landed
  const uint32_t empty0 = full0 + 8 * kRingEntries;     // [entry]: the reducers are done
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t row_bytes = static_cast<uint32_t>(H) * sizeof(TE);
  const int n_slots = kRingBytes / static_cast<int>(row_bytes);  // >= K + n_shared (host)
  if (threadIdx.x == 0) {
    for (int e = 0; e < kRingEntries; ++e) {
      ptx::mbar_init(full0 + 8 * e, 1);
      ptx::mbar_init(empty0 + 8 * e, kRingThreads / 32 - 1);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  pdl_enter();
  inv_pos = fresh(inv_pos);
  topk_w = fresh(topk_w);
  y_perm = fresh(y_perm);
  shared = fresh(shared);
  const int per = (T + gridDim.x - 1) / gridDim.x;
  const int t_begin = static_cast<int>(blockIdx.x) * per;
  const int n_tok = max(0, min(T, t_begin + per) - t_begin);

  if (warp == 0) {
    // ------------------------------------------------------------ copier
    int head = 0, freed = 0, rel = 0, issued = 0;
    bool ok = true;
    for (int i = 0; i < n_tok && ok; ++i) {
      const int mi = i % kRingMetaTok;
      if (mi == 0) {  // stage the next batch's slots (all loads in flight together)
        const int nb = min(kRingMetaTok, n_tok - i);
        const long base = static_cast<long>(t_begin + i) * K;
        for (int x = lane; x < nb * K; x += 32) {
          meta_p[x] = inv_pos[base + x];
          meta_w[x] = topk_w ? topk_w[base + x] : 1.f;
        }
        __syncwarp();
      }
      const int t = t_begin + i;
      const int e = i % kRingEntries;
      int p = -1;
      float w = 0.f;
      if (lane < K) {
        p = meta_p[mi * K + lane];
        w = meta_w[mi * K + lane];
        if (p >= cap) {
          if (status) atomicOr(status, MOE_DEV_BAD_SEGMENT);
          p = -1;
        }
      }
      const unsigned local = __ballot_sync(0xffffffffu, p >= 0);
      const int n = __popc(local);
      const int rows_t = n + n_shared;
      // the entry's previous token, and older ones while the ring lacks room
      while (rel <= i - kRingEntries || head + rows_t - freed > n_slots) {
        const int er = rel % kRingEntries;
        int w_ok = 1;
        if (lane == 0)
          w_ok = ptx::mbar_wait(empty0 + 8 * er, (rel / kRingEntries) & 1, abort_flag, status);
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        freed += ent[er].n;
        ++rel;
      }
      if (!ok) break;
      const int j = __popc(local & ((1u << lane) - 1u));
      if (p >= 0) ent[e].w[j] = w;
      if (lane == 0) {
        ent[e].n = rows_t;
        ent[e].slot0 = head % n_slots;
        ent[e].tok = t;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * e, rows_t * row_bytes);
      __syncwarp();
      if (p >= 0) {  // 0 <= p < cap, checked above
        const int slot = (head + j) % n_slots;
        ptx::bulk_load(ptx::smem_u32(rows + static_cast<long>(slot) * row_bytes),
                       y_perm + static_cast<long>(p) * H, row_bytes, full0 + 8 * e);
      }
      if (lane < n_shared) {
        const int slot = (head + n + lane) % n_slots;
        ptx::bulk_load(ptx::smem_u32(rows + static_cast<long>(slot) * row_bytes),
                       shared + lane * shared_stride + static_cast<long>(t) * H, row_bytes,
                       full0 + 8 * e);
      }
      head += rows_t;
      issued = i + 1;
    }
    if (!ok && lane == 0) {
      // unwinding: let the copies already issued land before the CTA exits
      for (int k = rel; k < issued; ++k)
        ptx::mbar_wait_drain(full0 + 8 * (k % kRingEntries), (k / kRingEntries) & 1);
    }
  } else {
    // ------------------------------------------------------------ reducers
    const int ct = threadIdx.x - 32;
    for (int i = 0; i < n_tok; ++i) {
      const int e = i % kRingEntries;
      if (!ptx::mbar_wait(full0 + 8 * e, (i / kRingEntries) & 1, abort_flag, status)) break;
      const int rows_t = ent[e].n, slot0 = ent[e].slot0;
      const int n = rows_t - n_shared;
      const long t = ent[e].tok;
      for (int c = ct * 8; c < H; c += (kRingThreads - 32) * 8) {
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
        int slot = slot0;
        for (int r = 0; r < rows_t; ++r) {
          if (r == n) {
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] *= rsf;
          }
          Raw8<TE> y;
          y.load(reinterpret_cast<const TE*>(rows + static_cast<long>(slot) * row_bytes) + c);
          y.add_to(acc, r < n ? ent[e].w[r] : 1.f);
          slot = slot + 1 == n_slots ? 0 : slot + 1;
        }
        if (n == rows_t) {
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] *= rsf;
        }
        st8(out + t * H + c, acc);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(empty0 + 8 * e);
    }
  }
}

int grid_for(long work, int per_block, int cap_blocks) {
  long g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > cap_blocks) g = cap_blocks;
  return static_cast<int>(g);
}

}  // namespace

namespace {
// Every scatter CTA of the fold sums the count rows of all CTAs, so its work
// grows with the square of the CTA count: past kFoldWork row entries in all
// (about 64 MB of L2 reads) the three passes cost less.
constexpr long kFoldWork = 1L << 24;
bool align_fold(long n_items, int E_l) {
  const long fb = (n_items + kFoldItems - 1) / kFoldItems;
  return E_l <= 256 && fb * E_l <= kFoldHist && fb * fb * E_l <= kFoldWork;
}

}  // namespace

bool combine_uses_ring(bool bf16, int T, int K, int k_local, int n_shared, int H) {
  const long row_bytes = static_cast<long>(H) * (bf16 ? 2 : 4);
  const int kl = k_local < 1 ? 1 : k_local > K ? K : k_local;
  return T >= kRingMinTokens && K <= 32 && (K + n_shared) * row_bytes <= kRingBytes &&
         (kl + n_shared) * row_bytes >= kRingMinTokenBytes;
}

int align_kernel_count(long n_items, int E_l) {
  if (n_items <= kSmallItems && E_l <= kSmallExperts) return 1;
  return align_fold(n_items, E_l) ? 2 : 3;
}

int align_warps(long n_items) {
  long w = (n_items + kItemsPerWarp - 1) / kItemsPerWarp;
  return static_cast<int>(w < 1 ? 1 : w);
}

cudaError_t launch_align(const int32_t* ids, long n_items, const int32_t* emap, int E, int E_l,
                         int ep_start, int block_m, int* hist, int32_t* counts,
                         int32_t* offsets, int32_t* sorted_ids, int32_t* inv_pos, int cap,
                         unsigned* status, cudaStream_t st, Tile* tiles, int* group_start,
                         int nmax, int max_tiles, int K, int R) {
  if (n_items <= kSmallItems && E_l <= kSmallExperts) {
    return launch_pdl(align_small_kernel, dim3(1), dim3(1024), 0, st, ids,
                      static_cast<int>(n_items), K, emap, R, E, E_l, ep_start, block_m, counts,
                      offsets, sorted_ids, inv_pos, cap, status, tiles, group_start, nmax,
                      max_tiles);
  }
  if (align_fold(n_items, E_l)) {
    // per-CTA counts: (n_items / kFoldItems) x E_l ints, within hist's
    // align_warps(n_items) x E_l
    const int fb = static_cast<int>((n_items + kFoldItems - 1) / kFoldItems);
    cudaError_t e = launch_pdl(align_fold_count_kernel, dim3(fb), dim3(256), 0, st, ids, n_items,
                               K, emap, R, E, E_l, ep_start, hist, sorted_ids, cap, status);
    if (e != cudaSuccess) return e;
    return launch_pdl(align_fold_scatter_kernel, dim3(fb), dim3(256), 0, st, ids, n_items, K,
                      emap, R, E, E_l, ep_start, static_cast<const int*>(hist), fb, block_m,
                      counts, offsets, sorted_ids, inv_pos, cap, status, tiles, group_start,
                      nmax, max_tiles);
  }
  const int n_warps = align_warps(n_items);
  const int blocks = (n_warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const size_t smem = sizeof(int) * kWarpsPerBlock * E_l;
  cudaError_t e = launch_pdl(align_count_kernel, dim3(blocks), dim3(256), smem, st, ids, n_items,
                             K, emap, R, E, E_l, ep_start, hist, n_warps, sorted_ids, cap,
                             status);
  if (e != cudaSuccess) return e;
  e = launch_pdl(align_scan_kernel, dim3(1), dim3(1024), 0, st, hist, n_warps, E_l, block_m,
                 counts, offsets, cap, status, tiles, group_start, nmax, max_tiles);
  if (e != cudaSuccess) return e;
  return launch_pdl(align_scatter_kernel, dim3(blocks), dim3(256), smem, st, ids, n_items, K,
                    emap, R, E, E_l, ep_start, static_cast<const int*>(hist), n_warps, sorted_ids,
                    inv_pos, cap, status);
}

cudaError_t launch_build_tiles(const int32_t* counts, const int32_t* offsets, int E_l, int nmax,
                               Tile* tiles, int* group_start, int max_tiles, int cap,
                               unsigned* status, cudaStream_t st) {
  return launch_pdl(build_tiles_kernel, dim3(1), dim3(1024), 0, st, counts, offsets, E_l, nmax,
                    tiles, group_start, max_tiles, cap, status);
}

cudaError_t launch_gather(bool bf16, const void* x, const int32_t* sorted_ids,
                          const int32_t* offsets_end, int cap, long n_items, int K, int H,
                          void* x_perm, cudaStream_t st, const float* w_items,
                          float* w_perm) {
  const int grid = grid_for(cap, 8, 8 * 152);
  if (bf16)
    return launch_pdl(gather_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st,
                      static_cast<const __nv_bfloat16*>(x), sorted_ids, offsets_end, cap, n_items,
                      K, H, static_cast<__nv_bfloat16*>(x_perm), w_items, w_perm);
  return launch_pdl(gather_kernel<float>, dim3(grid), dim3(256), 0, st,
                    static_cast<const float*>(x), sorted_ids, offsets_end, cap, n_items, K, H,
                    static_cast<float*>(x_perm), w_items, w_perm);
}

cudaError_t launch_silu_finalize(bool bf16, const float* part, int n_part, long part_stride,
                                 const int32_t* rows_dev, int cap, int I, void* h,
                                 cudaStream_t st) {
  const int grid = grid_for(static_cast<long>(cap) * ((I + 255) / 256), 8, 16 * 152);
  if (bf16)
    return launch_pdl(silu_finalize_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st, part,
                      n_part, part_stride, rows_dev, cap, I, static_cast<__nv_bfloat16*>(h));
  return launch_pdl(silu_finalize_kernel<float>, dim3(grid), dim3(256), 0, st, part, n_part,
                    part_stride, rows_dev, cap, I, static_cast<float*>(h));
}

cudaError_t launch_ep_dest(const int32_t* ids, long n, int E, int n_local, int32_t* dest,
                           int32_t* phys, const int32_t* phys_map, int R, int K, int E_phys,
                           cudaStream_t st) {
  if (phys_map && (R < 1 || K < 1)) return cudaErrorInvalidValue;
  return launch_pdl(ep_dest_kernel, dim3(grid_for(n, 256, 8 * 152)), dim3(256), 0, st, ids, n,
                    E, n_local, dest, phys, phys_map, R, K, E_phys);
}

cudaError_t launch_zero_dropped_rows(const int32_t* inv_pos, long n, long row_bytes, void* y,
                                     cudaStream_t st) {
  return launch_pdl(zero_dropped_rows_kernel, dim3(grid_for(n, 256, 8 * 152)), dim3(256), 0, st,
                    inv_pos, n, row_bytes, static_cast<uint8_t*>(y));
}

cudaError_t launch_ep_pack(bool bf16, const void* x, const int32_t* ids, const float* w,
                           const int32_t* sorted_ids, const int32_t* rows_dev, long n_items,
                           int K, int H, void* send_x, int32_t* send_ids, float* send_w,
                           int32_t* send_tok, cudaStream_t st) {
  const int grid = grid_for(n_items, 8, 8 * 152);
  if (bf16)
    return launch_pdl(ep_pack_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st,
                      static_cast<const __nv_bfloat16*>(x), ids, w, sorted_ids, rows_dev,
                      n_items, K, H, static_cast<__nv_bfloat16*>(send_x), send_ids, send_w,
                      send_tok);
  return launch_pdl(ep_pack_kernel<float>, dim3(grid), dim3(256), 0, st,
                    static_cast<const float*>(x), ids, w, sorted_ids, rows_dev, n_items, K, H,
                    static_cast<float*>(send_x), send_ids, send_w, send_tok);
}

cudaError_t launch_combine(bool bf16, const void* y_perm, int cap, const int32_t* inv_pos,
                           const float* topk_w, int K, int k_local, const void* shared,
                           int n_shared, long shared_stride, float rsf, void* out, int T, int H,
                           unsigned* status, cudaStream_t st, bool slots_early) {
  // Prefill-sized batches whose rows per token fit the ring and bring enough
  // bytes: the ring combine, one CTA per SM.
  const int ns = shared ? n_shared : 0;
  if (combine_uses_ring(bf16, T, K, k_local, ns, H)) {
    const int grid = T < kRingCtas ? T : kRingCtas;
#define MOE_RING(TE)                                                                         \
  do {                                                                                       \
    static std::atomic<unsigned long long> smem_set{0};                                      \
    const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(combine_ring_kernel<TE>), \
                                      kRingSmem, smem_set);                                  \
    if (e != cudaSuccess) return e;                                                          \
    return launch_pdl(combine_ring_kernel<TE>, dim3(grid), dim3(kRingThreads), kRingSmem, st, \
                      static_cast<const TE*>(y_perm), cap, inv_pos, topk_w, K,               \
                      static_cast<const TE*>(shared), ns, shared_stride, rsf,                \
                      static_cast<TE*>(out), T, H, status);                                  \
  } while (0)
    if (bf16) MOE_RING(__nv_bfloat16);
    MOE_RING(float);
#undef MOE_RING
  }
  // Rows loaded together (KB) follow the expected number of local rows per
  // token, not K: on an EP shard most slots are elsewhere, and a narrower
  // batch over more column chunks keeps more bytes in flight per warp. A
  // token with more local rows takes several batches, in slot order.
  // Up to kCombTok tokens per CTA, about four warp steps per warp, and at
  // least two CTAs per SM where the batch allows.
  const int kl = k_local < 1 ? 1 : k_local > K ? K : k_local;
  const int kb = bf16 ? (kl <= 1 ? 1 : kl <= 2 ? 2 : kl <= 4 ? 4 : 8) : (kl <= 2 ? 2 : 8);
  const int chunks = (H + 255) / 256;
  const int u = kb >= 4 ? 1 : 4 / kb;
  const int steps = (chunks + u - 1) / u;
  int tpc = 32 / steps;
  if (tpc > T / 304) tpc = T / 304;
  tpc = tpc < 1 ? 1 : tpc > kCombTok ? kCombTok : tpc;
  const int grid = (T + tpc - 1) / tpc;
#define MOE_COMBINE(TE, KB)                                                                \
  return launch_pdl(combine_kernel<TE, KB>, dim3(grid), dim3(256), 0, st,                  \
                    static_cast<const TE*>(y_perm), cap, inv_pos, topk_w, K,               \
                    static_cast<const TE*>(shared), n_shared, shared_stride, rsf,          \
                    static_cast<TE*>(out), T, H, tpc, slots_early ? 1 : 0, status)
  if (bf16) {
    if (kb == 1) MOE_COMBINE(__nv_bfloat16, 1);
    else if (kb == 2) MOE_COMBINE(__nv_bfloat16, 2);
    else if (kb == 4) MOE_COMBINE(__nv_bfloat16, 4);
    else MOE_COMBINE(__nv_bfloat16, 8);
  } else {
    if (kb == 2) MOE_COMBINE(float, 2);
    else MOE_COMBINE(float, 8);
  }
#undef MOE_COMBINE
  return cudaGetLastError();
}

MOE_DEBUG_TAKER(take_dbg_align)
MOE_WAIT_LIMIT_SETTER(set_wait_limit_align)

}  // namespace moe
