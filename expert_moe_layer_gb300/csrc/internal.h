// Host-side launch helpers shared between the translation units of libmoe.
// All launches are asynchronous on `st` and return cudaGetLastError().
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "dbg.cuh"
#include "moe.h"

namespace moe {

// One GEMM work tile: `count` token rows of one expert's segment.
//   x = expert (weight slab index), y = first B row, z = first output row,
//   w = rows (1..nmax).
using Tile = int4;

// Extents of the buffers a GEMM kernel touches. Only the debug build reads
// them (its checks of the kernels' derived indices); launches there refuse
// zero extents, so every call site fills them in.
struct GemmBounds {
  long a_rows = 0;    // rows behind the weight tensor map
  long b_rows = 0;    // rows behind the token-row tensor map
  long out_rows = 0;  // rows of out (and of each split-K slab of part)
  long out_map = 0;   // CTA-pair plain mode with out_rows: entries of out_rows /
                      //   out_scale (0 without them)
  int max_tiles = 0;  // entries of the tile table (0 for dense problems)
  long x_rows = 0;    // gathered token rows: rows of x
};

struct GemmArgs {
  const CUtensorMap* mapA;     // weights, 2-D [slabs*rows_per_slab, K]
  const CUtensorMap* mapB;     // token rows, 2-D [rows, K]
  const Tile* tiles;           // tile table, grouped (one group per expert), or nullptr:
                               //   dense tiles over dense_T tokens per slab, implicit
  const int* group_start;      // [n_groups+1] first tile of each group; [n_groups] = total
  int n_groups;                // <= 1024 (experts, or dense slabs)
  int dense_T = 0;             // tokens per slab when tiles == nullptr
  int m_tiles;                 // 128-row weight tiles per expert
  int k_blocks;                // K / (128 bytes of K)
  int k_split = 1;             // K ranges per tile; with k_split > 1 the raw fp32
  long split_stride = 0;       //   accumulators go to part + ks * split_stride
  float* part = nullptr;
  int a_rows_per_expert;       // weight rows per expert slab
  int a_up_offset;             // row offset of the "up" half (SiLU mode)
  int b_from_out;              // 1: B row = tile.z instead of tile.y
  void* out;                   // output rows
  long out_ld;                 // output row stride (elements)
  const int32_t* out_rows = nullptr;  // CTA-pair plain mode: token column p (a segment
  const float* out_scale = nullptr;   //   position) goes to out row out_rows[p], times
                                      //   out_scale[p]
  int b_cap = 0;                      // CTA-pair: rows of the position space (tile entries
                                      //   past it are skipped and flagged); 0: unchecked
  int m_valid;                 // weight rows with an output (router: E)
  unsigned* status;
  GemmBounds bnd;
  // grouped GEMM (single CTAs) only, routed tiles and one K range:
  int* publish = nullptr;      // GEMM1: per-tile counters; each epilogue warp adds 1 per
                               //   unit once its rows are stored
  const int* ready = nullptr;  // GEMM2: those counters; it then starts before GEMM1 ends
                               //   and loads a tile's rows once its count is ready_target
  int ready_target = 0;
  int* sched = nullptr;        // grid-wide unit counter (zeroed); nullptr: each CTA takes
                               //   units blockIdx.x, + gridDim.x, ...
  int* published = nullptr;    // with publish / ready: the adds over all tiles (zeroed);
                               //   GEMM2 stops checking tiles once it is complete
  // Token rows gathered by the kernel itself (routed tiles): B row r of a
  // tile is row gather_ids[tile.y + r] / gather_div of gather_x (row stride
  // gather_ld elements), fetched with per-lane copies instead of mapB (which
  // must still be a valid map). The tile table may then come from the kernel
  // just before.
  const void* gather_x = nullptr;
  const int32_t* gather_ids = nullptr;
  int gather_div = 1;
  long gather_ld = 0;
  long gather_items = 0;       // ids outside [0, gather_items) read row 0 of gather_x
};

enum GemmMode { kGemmSiluUp = 0, kGemmPlain = 1, kGemmLogits = 2 };

// Epilogue warps of the grouped GEMM: with `publish`, each adds 1 to its
// unit's tile counter, so a tile of GEMM1 is complete at m_tiles * this.
constexpr int kGemmEpiWarps = 8;

// tcgen05 grouped GEMM, D[w_row, token] = sum_k W[w_row, k] * B[token, k].
//   kGemmSiluUp: W = w13 rows, out = silu(gate) * up (act dtype)
//   kGemmPlain : W = w2 rows,  out = D (act dtype)
//   kGemmLogits: W = router rows (bf16), out = D (fp32)
cudaError_t launch_gemm(GemmMode mode, bool tf32, int nmax, const GemmArgs& a,
                        int num_sms, cudaStream_t st);

// The same grouped GEMM on CTA pairs (cta_group::2, M = 256 weight rows per
// pair unit, 128 per CTA): bf16, nmax = 256 token tiles, routed tile table,
// m_tiles counted in 256-row tiles, B tensor map boxes of nmax/2 rows.
cudaError_t launch_gemm_pair(GemmMode mode, int nmax, const GemmArgs& a, int num_sms,
                             cudaStream_t st);

// Router logits on CUDA cores: logits[t,e] = x[t].Wg[e] (fp32 accumulation).
// For E <= 32 the sum over H is split into slices of kRouterSplitCols
// columns, each written to its own partial slab (T*E floats apart); larger E
// writes one slab.
constexpr int kRouterSplitCols = 256;
inline int router_split_slabs(int H) { return (H + kRouterSplitCols - 1) / kRouterSplitCols; }
inline int router_cuda_core_slabs(int E, int H) { return E <= 32 ? router_split_slabs(H) : 1; }
cudaError_t launch_router_logits(bool act_bf16, bool router_bf16, const void* x,
                                 const void* wg, float* logits, int T, int E, int H,
                                 cudaStream_t st);

// Softmax + (grouped) top-k + renormalise on fp32 logits (+ bias if given).
// logits = sum of n_part partial slabs, partial_stride floats apart.
// flags: kRouteSigmoid / kRouteBiasSelect (topk_warp.cuh); bias, if given, is
// added to the logits, or with kRouteBiasSelect to the scores for the choice.
cudaError_t launch_topk(const float* logits, int n_part, long partial_stride,
                        const float* bias, int T, int E, int K,
                        int renorm, int flags, int n_group, int topk_group, int32_t* ids,
                        float* w, unsigned* status, cudaStream_t st);

// Routing and single-CTA alignment of a small batch in one kernel: router
// logits ([T, E] fp32 into logits), fp32 softmax, (grouped) top-k and
// renormalise into ids / w, then the counting sort into segments and the
// routed tile table, as launch_topk + launch_align would. tickets:
// kRouteTickets ints, zero before the call (the kernel leaves them zero).
constexpr int kRouteSmallTokens = 128;
constexpr int kRouteTickets = kRouteSmallTokens / 16 + 1;
struct RouteAlignArgs {
  const void* x;
  const void* wg;
  const float* bias;
  int T, E, H, K, renorm, flags, n_group, topk_group;
  float* logits;
  int* tickets;
  int32_t* ids;
  float* w;
  const int32_t* emap;
  int R;                      // replica map width (0: plain map or contiguous shard)
  int E_l, ep_start, block_m;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_ids;
  int32_t* inv_pos;
  int cap;
  unsigned* status;
  Tile* tiles;
  int* group_start;
  int nmax, max_tiles;
};
bool route_align_small_ok(int T, int K, int E_l);
cudaError_t launch_route_align_small(const RouteAlignArgs& a, bool act_bf16, bool router_bf16,
                                     cudaStream_t st);

// Alignment / permutation. hist has n_warps*E_l ints, n_warps = align_warps(T*K).
// Small inputs run as one fused kernel (hist unused), larger ones as three.
int align_kernel_count(long n_items, int E_l);
int align_warps(long n_items);
// With tiles != nullptr the align kernels also write the routed tile table
// (token chunks of nmax per local expert) and its group_start, as
// launch_build_tiles would.
cudaError_t launch_align(const int32_t* ids, long n_items, const int32_t* emap, int E,
                         int E_l, int ep_start, int block_m, int* hist, int32_t* counts,
                         int32_t* offsets, int32_t* sorted_ids, int32_t* inv_pos, int cap,
                         unsigned* status, cudaStream_t st, Tile* tiles = nullptr,
                         int* group_start = nullptr, int nmax = 0, int max_tiles = 0,
                         int K = 1, int R = 0);

// Routed tile table: group_start gets E_l+1 ints, one group per local expert.
// (Dense problems need no table: the GEMM derives their tiles from T.) A
// segment outside [0, cap) or past the next one's start is dropped and flagged
// (MOE_DEV_BAD_SEGMENT).
cudaError_t launch_build_tiles(const int32_t* counts, const int32_t* offsets, int E_l,
                               int nmax, Tile* tiles, int* group_start, int max_tiles, int cap,
                               unsigned* status, cudaStream_t st);
inline int dense_tile_count(int T, int S, int nmax) { return S * ((T + nmax - 1) / nmax); }
inline long routed_tile_bound(long n_items, int E_l, int nmax) {
  return n_items / nmax + E_l + 1;
}

// h[r][i] = silu(sum_s g_s[r][i]) * sum_s u_s[r][i] over n_part fp32 slabs
// (gate at column i, up at column I + i, row stride 2I), rows below
// min(*rows_dev, cap).
cudaError_t launch_silu_finalize(bool bf16, const float* part, int n_part, long part_stride,
                                 const int32_t* rows_dev, int cap, int I, void* h,
                                 cudaStream_t st);

// x_perm[r] = x[sorted_ids[r] / K] for rows holding an item.
// x_perm rows in segment order; with w_perm also the items' weights in that
// order (w_perm[r] = w_items[sorted_ids[r]]).
cudaError_t launch_gather(bool bf16, const void* x, const int32_t* sorted_ids,
                          const int32_t* offsets_end, int cap, long n_items, int K, int H,
                          void* x_perm, cudaStream_t st, const float* w_items = nullptr,
                          float* w_perm = nullptr);

// Both routed GEMMs of a decode-sized batch (32-token tiles, bf16) in one
// persistent kernel: h = silu(x W_gate^T) * (x W_up^T) per tile, then
// y = h W2^T, GEMM2 units
// waiting on per-tile ready counters. GEMM1 may be split over K (ks1 > 1):
// fp32 partial slabs in part, finished by the last warp of each block
// (split_cnt). ready and split_cnt must be zero before the launch.
struct MlpFusedArgs {
  const CUtensorMap* mapW13;  // [E_l*2I, H], box 128 x 64
  const CUtensorMap* mapW2;   // [E_l*H, I], box 128 x 64
  const CUtensorMap* mapH;    // h_perm [cap, I], box 32 x 64
  const CUtensorMap* mapX;    // x_perm [cap, H], box 32 x 64 (gathered rows)
  const Tile* tiles;
  const int* group_start;
  int n_groups;
  int H, I;
  int ks1;                    // K ranges of GEMM1
  float* part;                // ks1 slabs of [cap, 2I] fp32 (ks1 > 1)
  long part_stride;           // floats per slab
  int* split_cnt;             // max tiles x I/128 x 8 counters (ks1 > 1)
  int* ready;                 // one counter per tile
  void* h;                    // h_perm
  void* y;                    // y_perm
  unsigned* status;
  GemmBounds bnd;             // a_rows: w13 rows; b_rows = out_rows = cap; max_tiles
};
cudaError_t launch_mlp_fused(const MlpFusedArgs& a, int num_sms, cudaStream_t st);
size_t mlp_fused_smem_bytes();
// One CTA of the fused kernel fits on an SM of the current device (checked
// once per device).
bool mlp_fused_fits();

// Expert-parallel dispatch: the physical id of each item (the global id, or
// with a global replica map [E, R] replica (i / K) mod n of the id's row,
// -1 when invalid or outside [0, E_phys)) and dest[i] = phys[i] / n_local
// (-1 when invalid); then, after an align over the destination ranks, the
// send buffers in destination order (row r = item sorted_ids[r], rows_dev[0]
// valid rows).
cudaError_t launch_ep_dest(const int32_t* ids, long n, int E, int n_local, int32_t* dest,
                           int32_t* phys, const int32_t* phys_map, int R, int K, int E_phys,
                           cudaStream_t st);
// Zero y rows [i] with inv_pos[i] < 0 (row_bytes a multiple of 16).
cudaError_t launch_zero_dropped_rows(const int32_t* inv_pos, long n, long row_bytes, void* y,
                                     cudaStream_t st);
cudaError_t launch_ep_pack(bool bf16, const void* x, const int32_t* ids, const float* w,
                           const int32_t* sorted_ids, const int32_t* rows_dev, long n_items,
                           int K, int H, void* send_x, int32_t* send_ids, float* send_w,
                           int32_t* send_tok, cudaStream_t st);

// out[t] = rsf * sum_k w[t,k] y_perm[inv_pos[t,k]] + sum_s shared[s][t]
// (topk_w may be null: unit weights). k_local: the expected number of local
// rows per token (K, or about K/ep on an EP shard); it only picks the kernel
// variant. slots_early: inv_pos and topk_w were written by a kernel at least
// two launches back on this stream (true only inside moe_forward), so the
// kernel may read them before its dependency wait.
// Whether launch_combine streams the rows through the shared-memory ring
// (n_shared: the shared-expert outputs it adds, 0 without them).
bool combine_uses_ring(bool bf16, int T, int K, int k_local, int n_shared, int H);
cudaError_t launch_combine(bool bf16, const void* y_perm, int cap, const int32_t* inv_pos,
                           const float* topk_w, int K, int k_local, const void* shared,
                           int n_shared, long shared_stride, float rsf, void* out, int T, int H,
                           unsigned* status, cudaStream_t st, bool slots_early = false);

// The pipeline-wait limit of each translation unit with bounded waits (ns of
// %globaltimer), set on the current device.
cudaError_t set_wait_limit_gemm(unsigned long long ns);
cudaError_t set_wait_limit_gemm_pair(unsigned long long ns);
cudaError_t set_wait_limit_mlp_fused(unsigned long long ns);
cudaError_t set_wait_limit_route(unsigned long long ns);
cudaError_t set_wait_limit_align(unsigned long long ns);

// Debug build: each translation unit's record of failed bounds checks, read
// and cleared (all zero in the release build).
cudaError_t take_dbg_api(DbgRecord* out);
cudaError_t take_dbg_gemm(DbgRecord* out);
cudaError_t take_dbg_gemm_pair(DbgRecord* out);
cudaError_t take_dbg_mlp_fused(DbgRecord* out);
cudaError_t take_dbg_route(DbgRecord* out);
cudaError_t take_dbg_align(DbgRecord* out);

}  // namespace moe
