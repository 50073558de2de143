// Block-level pieces of token alignment shared by the align kernels and the
// fused small-batch route kernel: expert-id mapping, a block-wide exclusive
// scan, the routed tile table and the single-CTA counting sort.
#pragma once

#include <cuda_runtime.h>

#include "internal.h"

namespace moe {

// Local slot of a work item of global expert id and token t, or -1 (not on
// this rank, or flagged as bad). emap: NULL (contiguous shard from
// ep_start), the plain map [E], or with R > 0 a replica map [E, R]: the item
// goes to replica t mod n of the n replicas listed in row id (entries -1 for
// another rank, padded with -2).
__device__ __forceinline__ int local_expert(int id, int t, const int32_t* __restrict__ emap,
                                            int R, int E, int E_l, int ep_start,
                                            unsigned* status) {
  if (id < 0 || id >= E) {
    if (status) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
    return -1;
  }
  int le;
  if (emap && R > 0) {
    const int32_t* row = emap + static_cast<long>(id) * R;
    int n = 0;
    while (n < R && row[n] != -2) ++n;
    le = n > 0 ? row[t % n] : -3;
    if (le < -1 || le >= E_l) {
      if (status) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
      return -1;
    }
  } else if (emap) {
    le = emap[id];
    if (le < -1 || le >= E_l) {
      if (status) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
      return -1;
    }
  } else {
    le = id - ep_start;
    if (le < 0 || le >= E_l) le = -1;
  }
  return le;
}

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  __syncthreads();  // warp_sums may still be read by a previous scan
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = lane < (blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int incl = x + (wid > 0 ? warp_sums[wid - 1] : 0);
  total = warp_sums[(blockDim.x >> 5) - 1];
  return incl - v;
}

// Block-wide: the routed tile table from each expert's count c and first
// row off (thread e < E_l; other threads pass c = 0). Called by every thread.
__device__ __forceinline__ void write_tile_table(int e, int E_l, int c, int off, int nmax,
                                                 Tile* __restrict__ tiles,
                                                 int* __restrict__ group_start, int max_tiles,
                                                 int* warp_sums, unsigned* status) {
  const int n = e < E_l ? (c + nmax - 1) / nmax : 0;
  int total = 0;
  const int start = block_exclusive_scan(n, warp_sums, total);
  for (int j = 0; j < n; ++j) {
    const int idx = start + j;
    if (idx < max_tiles) {
      const int r0 = off + j * nmax;
      tiles[idx] = make_int4(e, r0, r0, min(nmax, c - j * nmax));
    }
  }
  if (e < E_l) group_start[e] = min(start, max_tiles);
  if (threadIdx.x == 0) {
    group_start[E_l] = min(total, max_tiles);
    if (total > max_tiles && status) atomicOr(status, MOE_DEV_CAP_OVERFLOW);
  }
}

// Single-CTA alignment for n_items <= kSmallItems and E_l <= kSmallExperts,
// run by a CTA of exactly 1024 threads (32 warps). A warp owns a run of
// consecutive items; per-warp counts live in hist ([warp][expert], 32*E_l
// ints of shared memory), which then become each warp's base rows, and the
// walk is replayed in the same order, so the order inside a segment is
// ascending item order (a stable counting sort). warp_sums: 32 ints of
// shared memory. ids may have been written by this CTA before a
// __syncthreads().
constexpr int kSmallItems = 32 * 256;
constexpr int kSmallExperts = 256;

// Up to kTinyItems items: one CTA of 1024 threads, G = 1024 / E_l threads per
// local expert. The local ids sit in shared memory; thread (g, e) counts expert e
// in the g-th range of items, the counts become padded offsets (one scan),
// and the same thread writes its range's items of expert e in item order
// (a stable counting sort without per-warp histograms). Each thread walks
// n/G items twice, so this only pays below a few dozen items (decode
// batches of a token or a few), where it skips the per-warp passes.
constexpr int kTinyItems = 64;

__device__ __forceinline__ void align_tiny_block(
    const int32_t* __restrict__ ids, int n_items, int K, const int32_t* __restrict__ emap, int R,
    int E, int E_l, int ep_start, int block_m, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
    int32_t* __restrict__ inv_pos, int cap, unsigned* status, Tile* __restrict__ tiles,
    int* __restrict__ group_start, int nmax, int max_tiles, int* smem, int* warp_sums) {
  int* le_s = smem;            // [kTinyItems] local expert of each item
  int* part = smem + 1024;     // [G][E_l] counts, then bases
  int* off_s = smem + 2048;    // [E_l] first row of each expert
  const int tid = threadIdx.x;
  for (int r = tid; r < cap; r += 1024) sorted_ids[r] = n_items;
  if (tid < n_items)
    le_s[tid] = local_expert(ids[tid], tid / K, emap, R, E, E_l, ep_start, status);
  __syncthreads();
  const int G = 1024 / E_l;  // E_l <= 256: at least 4
  const int g = tid / E_l, e = tid - g * E_l;
  const bool active = g < G;
  const int per = (n_items + G - 1) / G;  // items of each range
  const int i0 = min(n_items, g * per), i1 = min(n_items, i0 + per);
  if (active) {
    int c = 0;
    for (int i = i0; i < i1; ++i) c += le_s[i] == e;
    part[tid] = c;
  }
  __syncthreads();
  int c = 0;
  if (tid < E_l) {
    for (int gg = 0; gg < G; ++gg) {
      const int v = part[gg * E_l + tid];
      part[gg * E_l + tid] = c;
      c += v;
    }
  }
  const int padded = tid < E_l ? ((c + block_m - 1) / block_m) * block_m : 0;
  int total = 0;
  const int start = block_exclusive_scan(padded, warp_sums, total);
  if (tid < E_l) {
    counts[tid] = c;
    offsets[tid] = start;
    off_s[tid] = start;
  }
  if (tid == 0) {
    offsets[E_l] = total;
    if (total > cap && status) atomicOr(status, MOE_DEV_CAP_OVERFLOW);
  }
  if (tiles)
    write_tile_table(tid, E_l, tid < E_l ? c : 0, start, nmax, tiles, group_start, max_tiles,
                     warp_sums, status);
  __syncthreads();
  if (active) {
    int pos = off_s[e] + part[tid];
    for (int i = i0; i < i1; ++i) {
      if (le_s[i] != e) continue;
      if (pos < cap) {
        sorted_ids[pos] = i;
        inv_pos[i] = pos;
      } else {
        if (status) atomicOr(status, MOE_DEV_CAP_OVERFLOW);
        inv_pos[i] = -1;
      }
      ++pos;
    }
  }
  if (tid < n_items && le_s[tid] < 0) inv_pos[tid] = -1;
}

__device__ __forceinline__ void align_small_block(
    const int32_t* __restrict__ ids, int n_items, int K, const int32_t* __restrict__ emap, int R,
    int E, int E_l, int ep_start, int block_m, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
    int32_t* __restrict__ inv_pos, int cap, unsigned* status, Tile* __restrict__ tiles,
    int* __restrict__ group_start, int nmax, int max_tiles, int* hist, int* warp_sums) {
  if (n_items <= kTinyItems) {
    align_tiny_block(ids, n_items, K, emap, R, E, E_l, ep_start, block_m, counts, offsets,
                     sorted_ids, inv_pos, cap, status, tiles, group_start, nmax, max_tiles, hist,
                     warp_sums);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ipw = ((n_items + 31) / 32 + 31) / 32 * 32;  // items per warp, multiple of 32
  for (int r = threadIdx.x; r < cap; r += 1024) sorted_ids[r] = n_items;
  for (int i = threadIdx.x; i < 32 * E_l; i += 1024) hist[i] = 0;
  __syncthreads();
  int* my = hist + warp * E_l;
  const int base = warp * ipw;
  // this lane's items (at most 8): ids loaded together, local ids kept for
  // the second walk
  constexpr int kRuns = kSmallItems / 32 / 32;
  int lev[kRuns];
#pragma unroll
  for (int i = 0; i < kRuns; ++i) {
    const int item = base + 32 * i + lane;
    lev[i] = (32 * i < ipw && item < n_items) ? ids[item] : -1;
  }
#pragma unroll
  for (int i = 0; i < kRuns; ++i) {
    if (32 * i >= ipw) break;
    const int item = base + 32 * i + lane;
    lev[i] = item < n_items ? local_expert(lev[i], item / K, emap, R, E, E_l, ep_start, status)
                            : -1;
    const int le = lev[i];
    const unsigned peers = __match_any_sync(0xffffffffu, le);
    if (le >= 0 && lane == __ffs(peers) - 1) my[le] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // counts, padded offsets, per-warp base rows
  const int e = threadIdx.x;
  int c = 0;
  if (e < E_l)
    for (int w = 0; w < 32; ++w) c += hist[w * E_l + e];
  const int padded = e < E_l ? ((c + block_m - 1) / block_m) * block_m : 0;
  int total = 0;
  const int start = block_exclusive_scan(padded, warp_sums, total);
  if (e < E_l) {
    counts[e] = c;
    offsets[e] = start;
    int run = start;
    for (int w = 0; w < 32; ++w) {
      const int h = hist[w * E_l + e];
      hist[w * E_l + e] = run;
      run += h;
    }
  }
  if (threadIdx.x == 0) {
    offsets[E_l] = total;
    if (total > cap && status) atomicOr(status, MOE_DEV_CAP_OVERFLOW);
  }
  if (tiles)
    write_tile_table(e, E_l, e < E_l ? c : 0, start, nmax, tiles, group_start, max_tiles,
                     warp_sums, status);
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < kRuns; ++i) {
    if (32 * i >= ipw) break;
    const int item = base + 32 * i + lane;
    const int le = lev[i];
    const unsigned peers = __match_any_sync(0xffffffffu, le);
    if (item < n_items) {
      int pos = -1;
      if (le >= 0) {
        pos = my[le] + __popc(peers & lt);
        if (pos < cap) {
          sorted_ids[pos] = item;
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


}  // namespace moe
