// C ABI of the fused MoE layer forward: host validation, workspace layout,
// TMA tensor maps and the stream-ordered launch sequence. See include/moe.h
// for the contract of each entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "launch.cuh"

namespace moe {
[[maybe_unused]] constexpr DbgFile kDbgFileCode = kDbgApi;  // before topk_warp.cuh
}  // namespace moe

#include "topk_warp.cuh"
#include "moe.h"

namespace moe {
namespace {

constexpr int kMaxT = 1 << 18;
// 256-token tiles from this many GEMM1 units (single CTAs below 512, CTA
// pairs from 512)
constexpr long kTile256MinUnits = 256;
constexpr int kForwardBlock = 1;    // moe_forward leaves segments unpadded (the GEMMs
                                    // read past a segment's end but never store there)
constexpr size_t kAlignBytes = 256;

// The failure behind the calling thread's latest MOE_ERR_CUDA, reported by
// moe_last_cuda_error: a cudaError_t, or kEncodeErrorBase + the CUresult of a
// tensor-map encoding that failed.
constexpr int kEncodeErrorBase = 10000;
thread_local int g_last_cuda_error = 0;

int fail_cuda(int code) {
  g_last_cuda_error = code;
  return MOE_ERR_CUDA;
}
int cuda_ok(cudaError_t e) { return e == cudaSuccess ? MOE_OK : fail_cuda(static_cast<int>(e)); }

#define MOE_TRY(x)              \
  do {                          \
    const int _rc = (x);        \
    if (_rc != MOE_OK) return _rc; \
  } while (0)

size_t rup(size_t v) { return (v + kAlignBytes - 1) / kAlignBytes * kAlignBytes; }
int ebytes(moe_dtype d) { return d == MOE_BF16 ? 2 : 4; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate_cfg(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->router_dtype != MOE_F32 && c->router_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  const int E = c->num_experts, K = c->top_k, H = c->hidden_size, I = c->intermediate_size;
  if (E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
  if (H < 128 || H % 128 != 0 || I < 128 || I % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (c->num_redundant_experts < 0 || (c->num_redundant_experts > 0 && c->max_replicas < 1))
    return MOE_ERR_INVALID_ARG;
  if (c->ep_size < 1 || (E + c->num_redundant_experts) % c->ep_size != 0)
    return MOE_ERR_INVALID_ARG;
  if (c->ep_rank < 0 || c->ep_rank >= c->ep_size) return MOE_ERR_INVALID_ARG;
  if (c->use_grouped_topk) {
    const int g = c->num_expert_group, tg = c->topk_group;
    if (g < 1 || E % g != 0 || tg < 1 || tg > g) return MOE_ERR_INVALID_ARG;
    if (static_cast<long>(K) > static_cast<long>(tg) * (E / g)) return MOE_ERR_INVALID_ARG;
  }
  if (c->num_shared_experts < 0) return MOE_ERR_INVALID_ARG;
  if (c->num_shared_experts > 0) {
    const int Is = c->shared_intermediate_size;
    if (Is < 128 || Is % 128 != 0) return MOE_ERR_INVALID_ARG;
  }
  if (!std::isfinite(c->routed_scaling_factor)) return MOE_ERR_INVALID_ARG;
  if (c->scoring_func != MOE_SCORE_SOFTMAX && c->scoring_func != MOE_SCORE_SIGMOID)
    return MOE_ERR_INVALID_ARG;
  if (c->bias_mode != MOE_BIAS_LOGIT && c->bias_mode != MOE_BIAS_SELECT)
    return MOE_ERR_INVALID_ARG;
  if (c->max_replicas < 0 || c->max_replicas > 16) return MOE_ERR_INVALID_ARG;
  // kernel coverage
  if (E > 512 || K > 32) return MOE_ERR_UNSUPPORTED;
  if (c->use_grouped_topk && c->num_expert_group > 32) return MOE_ERR_UNSUPPORTED;
  if ((E + c->num_redundant_experts) / c->ep_size > 1024) return MOE_ERR_UNSUPPORTED;
  if (c->num_shared_experts > 1024) return MOE_ERR_UNSUPPORTED;
  if (c->act_dtype == MOE_F32 && c->router_dtype == MOE_BF16) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int validate_T(int T) { return (T < 0 || T > kMaxT) ? MOE_ERR_INVALID_ARG : MOE_OK; }

// Local weight slots: the rank's share of the logical experts plus the
// redundant replicas.
int n_local(const moe_config* c) {
  return (c->num_experts + c->num_redundant_experts) / c->ep_size;
}

// Expected local rows per token: each of the K slots lands on this rank with
// probability about 1/ep_size.
int local_rows(const moe_config* c) { return (c->top_k + c->ep_size - 1) / c->ep_size; }

// Token tile (MMA N) of the routed GEMMs, from the average segment length:
// 256 (bf16) from 192 rows when that still leaves >= 256 GEMM1 work units
// (CTA pairs from 512, single CTAs below), 128 from 48 rows, else 32. A larger N means more FLOPs
// per byte staged into shared memory; more units mean better balance.
// GEMM1 units on 256-token tiles (weight tiles x full token tiles)
long units256(const moe_config* c, int T) {
  const long local_items = static_cast<long>(T) * c->top_k / c->ep_size;
  return (local_items / 256) * (c->intermediate_size / 128);
}
int routed_nmax(const moe_config* c, int T) {
  const long avg = static_cast<long>(T) * c->top_k / c->num_experts;
  if (avg >= 192 && c->act_dtype == MOE_BF16 && units256(c, T) >= kTile256MinUnits) return 256;
  return avg >= 48 ? 128 : 32;
}
int dense_nmax(int T) { return T >= 64 ? 128 : 32; }

// The router runs as a tcgen05 GEMM whenever x and the router weights are
// bf16 (fp32 routers run on CUDA cores, split over H into 256-column slices
// when E <= 32). Tensor-core routers whose units (expert tiles x token tiles)
// fill less than half the SMs split K = H into ranges, as many as still fit
// the units into one wave; the top-k kernel sums the fp32 partials in slab
// order.
int route_flags(const moe_config* c) {
  return (c->scoring_func == MOE_SCORE_SIGMOID ? kRouteSigmoid : 0) |
         (c->bias_mode == MOE_BIAS_SELECT ? kRouteBiasSelect : 0);
}

bool router_on_tensor_cores(const moe_config* c, int /*T*/) {
  return c->act_dtype == MOE_BF16 && c->router_dtype == MOE_BF16;
}
int router_nmax(int T) { return T >= 256 ? 128 : 32; }
int router_ksplit(const moe_config* c, int T) {
  if (!router_on_tensor_cores(c, T)) return router_cuda_core_slabs(c->num_experts, c->hidden_size);
  const int k_blocks = c->hidden_size / 64;
  const long base = static_cast<long>((c->num_experts + 127) / 128) *
                    dense_tile_count(T, 1, router_nmax(T));
  if (2 * base >= 152) return 1;  // fills half the SMs: fp32 partials would cost more
  // one wave of units on the 152 SMs: each unit pays a pipeline fill and an
  // epilogue, so fewer, longer units beat two waves of short ones
  long ks = 152 / base;
  if (ks > 16) ks = 16;
  if (ks > k_blocks) ks = k_blocks;
  if (ks < 1) ks = 1;
  const long kb_per = (k_blocks + ks - 1) / ks;
  return static_cast<int>((k_blocks + kb_per - 1) / kb_per);
}

// Decode batches leave few GEMM1 units (token tiles x I/128): split K = H
// into as many ranges as still fit the units into one wave on the SMs (a
// second wave adds a full DRAM round trip and partial-sum chain). Estimate
// tiles as one per touched expert.
int gemm1_ksplit(const moe_config* c, int T) {
  const long local_items = static_cast<long>(T) * c->top_k / c->ep_size;
  long tiles = local_items < n_local(c) ? local_items : n_local(c);
  if (tiles < 1) tiles = 1;
  const long units = tiles * (c->intermediate_size / 128);
  if (units >= 152) return 1;
  const int k_blocks = c->hidden_size * (c->act_dtype == MOE_BF16 ? 2 : 4) / 128;
  long ks = 152 / units;
  if (ks < 1) ks = 1;
  if (ks > 8) ks = 8;
  if (ks > k_blocks) ks = k_blocks;
  const long kb_per = (k_blocks + ks - 1) / ks;
  return static_cast<int>((k_blocks + kb_per - 1) / kb_per);
}

long max_routed_tiles(const moe_config* c, int T) {
  return routed_tile_bound(static_cast<long>(T) * c->top_k, n_local(c), routed_nmax(c, T));
}

// Decode-sized bf16 batches (32-token tiles) run both routed GEMMs in one
// persistent kernel that gathers its token rows from x itself.
bool mlp_fused(const moe_config* c, int T) {
  return c->act_dtype == MOE_BF16 && routed_nmax(c, T) == 32 && n_local(c) <= 1024;
}

bool gemm2_early(const moe_config* c, int T);

// Zeroed at the start of every call (one memset): the status word, the
// small-batch route tickets and, on the fused MLP path, its per-tile ready
// counters and per-block split counters; where GEMM2 overlaps GEMM1, GEMM2's
// unit counter, the count of tile publishes and the per-tile ready counters.
// Offsets from the start of ws.
struct SyncRegion {
  size_t bytes, ready, split, sched;
};
SyncRegion sync_region(const moe_config* c, int T) {
  SyncRegion r;
  size_t off = 4 + 4 * static_cast<size_t>(kRouteTickets);
  r.ready = r.split = r.sched = off;
  const size_t tiles = static_cast<size_t>(max_routed_tiles(c, T));
  if (mlp_fused(c, T)) {
    off += 4 * tiles;
    r.split = off;
    if (gemm1_ksplit(c, T) > 1) off += 4 * tiles * (c->intermediate_size / 128) * 8;
  } else if (gemm2_early(c, T)) {
    off += 16;
    r.ready = off;
    off += 4 * tiles;
  }
  r.bytes = off;
  return r;
}

// With 256-token tiles both GEMMs run on CTA pairs: one M = 256 MMA over two
// SMs, each SM staging half of the token rows. In GEMM1 each CTA holds 64 gate
// rows and the matching 64 up rows of a 128-index slice of I (two
// accumulators of the double buffer fit in TMEM); GEMM2 puts 256 consecutive
// output rows on the pair.
bool gemms_on_pairs(const moe_config* c, int T) {
  return routed_nmax(c, T) == 256 && c->hidden_size % 256 == 0 && units256(c, T) >= 512;
}

// GEMM2 starts while GEMM1's last units run, on the SMs GEMM1 has left, when
// both run on single CTAs with one K range: GEMM1 publishes each tile's h rows
// and GEMM2 takes its units from a counter, loading a tile's rows once they
// are all published. The fused decode kernel and the CTA-pair GEMMs keep
// their own schedules.
bool gemm2_early(const moe_config* c, int T) {
  return !mlp_fused(c, T) && !gemms_on_pairs(c, T) && gemm1_ksplit(c, T) == 1;
}

// Shared experts over at least two 256-token tiles per slab run on CTA pairs
// like the long routed segments.
bool shared_on_pairs(const moe_config* c, int T) {
  return c->act_dtype == MOE_BF16 && T >= 512 && c->hidden_size % 256 == 0;
}

// SMs of the current context's SM resource (a green context holds part of
// the device), or 0 where the driver reports none.
int context_sms() {
  static PFN_cuCtxGetCurrent_v4000 get_ctx = nullptr;
  static PFN_cuCtxGetDevResource_v12040 get_res = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_ctx = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetDevResource", &p, 12040, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_res = reinterpret_cast<PFN_cuCtxGetDevResource_v12040>(p);
  });
  CUcontext ctx = nullptr;
  if (!get_ctx || !get_res || get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  CUdevResource r;
  std::memset(&r, 0, sizeof(r));
  if (get_res(ctx, &r, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS) return 0;
  return static_cast<int>(r.sm.smCount);
}

// SMs the persistent grids run on: those of the current context where it
// has fewer than the device (the fused decode kernel's CTAs wait on one
// another, so its grid must fit), else the device's. Not cached: one device
// may run under several contexts.
int sm_count() {
  int dev = 0;
  if (cuda_ok(cudaGetDevice(&dev)) != MOE_OK) return 0;
  int n = 0;
  if (cuda_ok(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != MOE_OK)
    return 0;
  const int c = context_sms();
  return (c > 0 && c < n) ? c : n;
}

// -------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D row-major [rows, cols] map; box = 128 bytes of a row x box_rows rows,
// 128-byte swizzle, zero fill out of bounds. MOE_OK or MOE_ERR_CUDA.
int make_map(CUtensorMap* m, const void* base, moe_dtype dt, long rows, long cols,
             int box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail_cuda(static_cast<int>(cudaErrorSymbolNotFound));
  const int eb = ebytes(dt);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * eb};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType t =
      dt == MOE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUresult r = fn(m, t, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : fail_cuda(kEncodeErrorBase + static_cast<int>(r));
}

// Output extents of a GEMM launch for the debug build's checks: rows of out,
// entries of the tile table, entries of an out_rows map.
GemmBounds out_bounds(long out_rows, int max_tiles = 0, long out_map = 0) {
  GemmBounds b;
  b.out_rows = out_rows;
  b.max_tiles = max_tiles;
  b.out_map = out_map;
  return b;
}

// One grouped GEMM launch. A = weights [slabs*rows_per_slab, Kdim]; B = token
// rows [b_rows, Kdim].
int run_gemm(GemmMode mode, moe_dtype dt, int nmax, const void* A, long a_rows, const void* B,
             long b_rows, int Kdim, const Tile* tiles, const int* group_start, int n_groups,
             int m_tiles, int rows_per_slab, int up_off, int b_from_out, void* out, long out_ld,
             int m_valid, unsigned* status, cudaStream_t st, int k_split = 1,
             long split_stride = 0, int dense_T = 0, bool pair = false,
             float* part = nullptr, const int32_t* out_rows = nullptr,
             const float* out_scale = nullptr, int b_cap = 0, GemmBounds bnd = {},
             int* publish = nullptr, const int* ready = nullptr, int ready_target = 0,
             int* sched = nullptr, int* published = nullptr, const void* gather_x = nullptr,
             const int32_t* gather_ids = nullptr, int gather_div = 1, long gather_rows = 0) {
  CUtensorMap ma, mb;
  // CTA pairs in SiLU mode stage 64 gate and 64 up rows per CTA: 64-row boxes
  const int a_box = (pair && mode == kGemmSiluUp) ? 64 : 128;
  MOE_TRY(make_map(&ma, A, dt, a_rows, Kdim, a_box));
  // a kernel that gathers its token rows reads no B map; it gets a valid one
  // over x
  MOE_TRY(make_map(&mb, gather_x ? gather_x : B, dt, gather_x ? gather_rows : b_rows, Kdim,
                   pair ? nmax / 2 : nmax));
  GemmArgs g;
  g.mapA = &ma;
  g.mapB = &mb;
  g.tiles = tiles;
  g.group_start = group_start;
  g.n_groups = n_groups;
  g.m_tiles = m_tiles;
  g.k_blocks = Kdim * ebytes(dt) / 128;
  g.k_split = k_split;
  g.split_stride = split_stride;
  g.dense_T = dense_T;
  g.part = part;
  g.a_rows_per_expert = rows_per_slab;
  g.a_up_offset = up_off;
  g.b_from_out = b_from_out;
  g.out = out;
  g.out_ld = out_ld;
  g.out_rows = out_rows;
  g.out_scale = out_scale;
  g.b_cap = b_cap;
  g.m_valid = m_valid;
  g.status = status;
  bnd.a_rows = a_rows;
  bnd.b_rows = b_rows;
  g.bnd = bnd;
  g.publish = publish;
  g.ready = ready;
  g.ready_target = ready_target;
  g.sched = sched;
  g.published = published;
  if (gather_x) {
    g.gather_x = gather_x;
    g.gather_ids = gather_ids;
    g.gather_div = gather_div;
    g.gather_ld = Kdim;
    g.gather_items = gather_rows * gather_div;
    g.bnd.x_rows = gather_rows;
  }
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  if (pair) return cuda_ok(launch_gemm_pair(mode, nmax, g, sms, st));
  return cuda_ok(launch_gemm(mode, dt == MOE_F32, nmax, g, sms, st));
}

// -------------------------------------------------------------- layouts
struct Carver {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off = rup(off + bytes);
    return o;
  }
};

struct RouteLayout {
  size_t status, logits, total;
};
RouteLayout route_layout(const moe_config* c, int T) {
  Carver cv;
  RouteLayout L;
  L.status = cv.take(4);
  L.logits = cv.take(sizeof(float) * static_cast<size_t>(router_ksplit(c, T)) * T *
                     c->num_experts);
  L.total = cv.off;
  return L;
}

struct AlignLayout {
  size_t status, hist, total;
};
AlignLayout align_layout(const moe_config* c, int T) {
  Carver cv;
  AlignLayout L;
  L.status = cv.take(4);
  L.hist = cv.take(sizeof(int) * static_cast<size_t>(align_warps(static_cast<long>(T) * c->top_k)) *
                   n_local(c));
  L.total = cv.off;
  return L;
}

struct MlpLayout {
  size_t status, tiles, groups, x_perm, h_perm, part1, total;
  SyncRegion sync;
};
MlpLayout mlp_layout(const moe_config* c, int T, int cap) {
  Carver cv;
  MlpLayout L;
  const size_t eb = ebytes(c->act_dtype);
  L.sync = sync_region(c, T);
  L.status = cv.take(L.sync.bytes);
  L.tiles = cv.take(sizeof(Tile) * static_cast<size_t>(max_routed_tiles(c, T)));
  L.groups = cv.take(sizeof(int) * static_cast<size_t>(n_local(c) + 1));
  L.x_perm = cv.take(eb * static_cast<size_t>(cap) * c->hidden_size);
  L.h_perm = cv.take(eb * static_cast<size_t>(cap) * c->intermediate_size);
  L.part1 = cv.take(gemm1_ksplit(c, T) > 1 ? sizeof(float) * gemm1_ksplit(c, T) * cap * 2 *
                                                 static_cast<size_t>(c->intermediate_size)
                                           : 0);
  L.total = cv.off;
  return L;
}

struct FwdLayout {
  size_t status, topk_ids, topk_w, logits, hist, counts, offsets, sorted_ids, inv_pos;
  size_t tiles, groups, x_perm, h_perm, y_perm, h_sh, y_sh, part1, total;
  int cap;
  SyncRegion sync;
};
FwdLayout fwd_layout(const moe_config* c, int T) {
  Carver cv;
  FwdLayout L;
  const size_t eb = ebytes(c->act_dtype);
  const size_t TK = static_cast<size_t>(T) * c->top_k;
  const int El = n_local(c);
  const int S = c->num_shared_experts;
  L.cap = static_cast<int>(TK + static_cast<size_t>(El) * (kForwardBlock - 1));
  L.sync = sync_region(c, T);
  L.status = cv.take(L.sync.bytes);
  L.topk_ids = cv.take(4 * TK);
  L.topk_w = cv.take(4 * TK);
  L.logits = cv.take(sizeof(float) * static_cast<size_t>(router_ksplit(c, T)) * T *
                     c->num_experts);
  L.hist = cv.take(sizeof(int) * static_cast<size_t>(align_warps(TK)) * El);
  L.counts = cv.take(4 * static_cast<size_t>(El));
  L.offsets = cv.take(4 * static_cast<size_t>(El + 1));
  L.sorted_ids = cv.take(4 * static_cast<size_t>(L.cap));
  L.inv_pos = cv.take(4 * TK);
  L.tiles = cv.take(sizeof(Tile) * static_cast<size_t>(max_routed_tiles(c, T)));
  L.groups = cv.take(sizeof(int) * static_cast<size_t>(El + 1));
  L.x_perm = cv.take(eb * L.cap * c->hidden_size);
  L.h_perm = cv.take(eb * L.cap * c->intermediate_size);
  L.y_perm = cv.take(eb * L.cap * c->hidden_size);
  L.h_sh = cv.take(eb * static_cast<size_t>(S) * T * (S ? c->shared_intermediate_size : 0));
  L.y_sh = cv.take(eb * static_cast<size_t>(S) * T * c->hidden_size);
  L.part1 = cv.take(gemm1_ksplit(c, T) > 1 ? sizeof(float) * gemm1_ksplit(c, T) * L.cap * 2 *
                                                 static_cast<size_t>(c->intermediate_size)
                                           : 0);
  L.total = cv.off;
  return L;
}

// Workspace of moe_ep_dispatch.
struct EpLayout {
  size_t status, dest, phys, hist, sorted, total;
};
EpLayout ep_layout(const moe_config* c, int T) {
  Carver cv;
  EpLayout L;
  const size_t n = static_cast<size_t>(T) * c->top_k;
  L.status = cv.take(4);
  L.dest = cv.take(4 * n);
  L.phys = cv.take(4 * n);
  L.hist = cv.take(sizeof(int) * static_cast<size_t>(align_warps(static_cast<long>(n))) *
                   c->ep_size);
  L.sorted = cv.take(4 * n);
  L.total = cv.off;
  return L;
}

// The configuration an expert-parallel rank computes its received items with:
// top_k 1 over its own shard, seen as a layer of E_l experts on one rank, so
// that the tile-size and split heuristics count every item as local: one
// slot per item, no routing, no shared experts, no scaling. The align step
// still maps the global ids with the caller's E and rank.
moe_config ep_item_config(const moe_config* c) {
  moe_config c1 = *c;
  c1.num_experts = n_local(c);
  c1.num_redundant_experts = 0;
  c1.ep_size = 1;
  c1.ep_rank = 0;
  c1.top_k = 1;
  c1.use_grouped_topk = 0;
  c1.num_expert_group = 0;
  c1.topk_group = 0;
  c1.num_shared_experts = 0;
  c1.shared_intermediate_size = 0;
  c1.routed_scaling_factor = 1.0f;
  c1.scoring_func = MOE_SCORE_SOFTMAX;
  c1.bias_mode = MOE_BIAS_LOGIT;
  return c1;
}


template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}


// Record a caller's timing event on `st`. Under stream capture the event
// becomes an event-record node, so a replayed graph still timestamps stages.
int record_event(void* ev, cudaStream_t st) {
  if (!ev) return MOE_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  MOE_TRY(cuda_ok(cudaStreamIsCapturing(st, &cs)));
  const cudaError_t e =
      cs == cudaStreamCaptureStatusActive
          ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), st, cudaEventRecordExternal)
          : cudaEventRecord(static_cast<cudaEvent_t>(ev), st);
  return cuda_ok(e);
}


// ------------------------------------------------------------- stage bodies
int do_route(const moe_config* c, int T, const void* x, const void* router_w,
             const float* bias, int32_t* ids, float* w, float* logits,
             unsigned* status, cudaStream_t st) {
  const int E = c->num_experts, H = c->hidden_size;
  int n_part = 1;
  if (router_on_tensor_cores(c, T)) {
    const int nm = router_nmax(T);
    n_part = router_ksplit(c, T);
    MOE_TRY(run_gemm(kGemmLogits, MOE_BF16, nm, router_w, E, x, T, H, nullptr, nullptr, 1,
                     (E + 127) / 128, 0, 0, 0, logits, E, E, status, st, n_part,
                     static_cast<long>(T) * E, T, false, logits, nullptr, nullptr, 0,
                     out_bounds(T)));
  } else {
    n_part = router_ksplit(c, T);
    MOE_TRY(cuda_ok(launch_router_logits(c->act_dtype == MOE_BF16, c->router_dtype == MOE_BF16,
                                         x, router_w, logits, T, E, H, st)));
  }
  return cuda_ok(launch_topk(logits, n_part, static_cast<long>(T) * E, bias, T, E, c->top_k,
                             c->renormalize ? 1 : 0, route_flags(c),
                             c->use_grouped_topk ? c->num_expert_group : 0,
                             c->use_grouped_topk ? c->topk_group : 0, ids, w, status, st));
}

int do_mlp(const moe_config* c, int T, const void* x, const int32_t* sorted_ids,
           const int32_t* counts, const int32_t* offsets, int cap, const void* w13,
           const void* w2, void* y_perm, Tile* tiles, int* groups, const SyncRegion& sync,
           void* x_perm, void* h_perm, float* part1, unsigned* status, cudaStream_t st,
           void* const* ev = nullptr, bool tiles_ready = false,
           const int32_t* y_rows = nullptr, const float* w_items = nullptr,
           float* w_perm = nullptr) {
  const int El = n_local(c), H = c->hidden_size, I = c->intermediate_size, K = c->top_k;
  const int nmax = routed_nmax(c, T);
  const long n_items = static_cast<long>(T) * K;
  const bool pairs = gemms_on_pairs(c, T);
  // the fused kernel needs one CTA resident on every SM of its grid; where
  // one does not fit, the two GEMM kernels run on the same tile table
  const bool fused = mlp_fused(c, T) && mlp_fused_fits();
  const int max_tiles = static_cast<int>(max_routed_tiles(c, T));
  if (!tiles_ready)
    MOE_TRY(cuda_ok(launch_build_tiles(counts, offsets, El, nmax, tiles, groups, max_tiles,
                                       cap, status, st)));
  // GEMM1 on single CTAs fetches its token rows from x itself; the CTA-pair
  // and fused kernels read them from x_perm
  const bool self_gather = !pairs && !fused;
  if (!self_gather)
    MOE_TRY(cuda_ok(launch_gather(c->act_dtype == MOE_BF16, x, sorted_ids, offsets + El, cap,
                                  n_items, K, H, x_perm, st, y_rows ? w_items : nullptr,
                                  y_rows ? w_perm : nullptr)));
  if (ev) MOE_TRY(record_event(ev[0], st));
  if (fused) {
    const int ks = gemm1_ksplit(c, T);
    CUtensorMap m13, m2, mh, mx;
    MOE_TRY(make_map(&m13, w13, c->act_dtype, static_cast<long>(El) * 2 * I, H, 128));
    MOE_TRY(make_map(&m2, w2, c->act_dtype, static_cast<long>(El) * H, I, 128));
    MOE_TRY(make_map(&mh, h_perm, c->act_dtype, cap, I, 32));
    MOE_TRY(make_map(&mx, x_perm, c->act_dtype, cap, H, 32));
    MlpFusedArgs a;
    a.mapW13 = &m13;
    a.mapW2 = &m2;
    a.mapH = &mh;
    a.mapX = &mx;
    a.tiles = tiles;
    a.group_start = groups;
    a.n_groups = El;
    a.H = H;
    a.I = I;
    a.ks1 = ks;
    a.part = ks > 1 ? part1 : nullptr;
    a.part_stride = static_cast<long>(cap) * 2 * I;
    a.split_cnt = reinterpret_cast<int*>(reinterpret_cast<char*>(status) + sync.split);
    a.ready = reinterpret_cast<int*>(reinterpret_cast<char*>(status) + sync.ready);
    a.h = h_perm;
    a.y = y_perm;
    a.status = status;
    a.bnd = out_bounds(cap, max_tiles);
    a.bnd.a_rows = static_cast<long>(El) * 2 * I;
    a.bnd.b_rows = cap;
    const int sms = sm_count();
    if (sms <= 0) return MOE_ERR_CUDA;
    MOE_TRY(cuda_ok(launch_mlp_fused(a, sms, st)));
    if (ev) MOE_TRY(record_event(ev[1], st));  // GEMM1 and GEMM2 share one kernel
    return MOE_OK;
  }
  const int ks1 = pairs ? 1 : gemm1_ksplit(c, T);  // pairs: long segments, never split
  // GEMM2 overlapping GEMM1's last units (counters zeroed with the status word)
  const bool early = ks1 == 1 && gemm2_early(c, T);
  int* ready = reinterpret_cast<int*>(reinterpret_cast<char*>(status) + sync.ready);
  int* sched = reinterpret_cast<int*>(reinterpret_cast<char*>(status) + sync.sched);
  if (ks1 > 1) {
    // split over K: raw gate/up partials, then the SiLU*up epilogue
    MOE_TRY(run_gemm(kGemmSiluUp, c->act_dtype, nmax, w13, static_cast<long>(El) * 2 * I, x_perm,
                     cap, H, tiles, groups, El, I / 128, 2 * I, I, 0, h_perm, 2 * I, I, status,
                     st, ks1, static_cast<long>(cap) * 2 * I, 0, false, part1, nullptr, nullptr,
                     0, out_bounds(cap, max_tiles), nullptr, nullptr, 0, nullptr, nullptr,
                     self_gather ? x : nullptr, sorted_ids, K, T));
    MOE_TRY(cuda_ok(launch_silu_finalize(c->act_dtype == MOE_BF16, part1, ks1,
                                         static_cast<long>(cap) * 2 * I, offsets + El, cap, I,
                                         h_perm, st)));
  } else {
    MOE_TRY(run_gemm(kGemmSiluUp, c->act_dtype, nmax, w13, static_cast<long>(El) * 2 * I, x_perm,
                     cap, H, tiles, groups, El, I / 128, 2 * I, I, 0, h_perm, I, I, status, st,
                     1, 0, 0, pairs, nullptr, nullptr, nullptr, pairs ? cap : 0,
                     out_bounds(cap, max_tiles), early ? ready : nullptr, nullptr, 0, nullptr,
                     early ? sched + 1 : nullptr, self_gather ? x : nullptr, sorted_ids, K, T));
  }
  if (ev) MOE_TRY(record_event(ev[1], st));
  // with y_rows (CTA pairs only) GEMM2 writes segment position p to row
  // y_rows[p] of y_perm, times the item weight w_perm[p] (from the gather)
  MOE_TRY(run_gemm(kGemmPlain, c->act_dtype, nmax, w2, static_cast<long>(El) * H, h_perm, cap, I,
                   tiles, groups, El, H / (pairs ? 256 : 128), H, 0, 0, y_perm, H, H, status, st,
                   1, 0, 0, pairs, nullptr, pairs ? y_rows : nullptr,
                   pairs && y_rows ? w_perm : nullptr, pairs ? cap : 0,
                   pairs && y_rows ? out_bounds(n_items, max_tiles, cap)
                                   : out_bounds(cap, max_tiles),
                   nullptr, early ? ready : nullptr, (I / 128) * kGemmEpiWarps,
                   early ? sched : nullptr, early ? sched + 1 : nullptr));
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_strerror(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace or capacity too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_STATUS: return "device status flag set";
    case MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
    default: return "unknown status";
  }
}

int moe_validate_config(const moe_config* cfg) { return validate_cfg(cfg); }

size_t moe_align_cap(const moe_config* cfg, int T, int block_m) {
  if (validate_cfg(cfg) != MOE_OK || validate_T(T) != MOE_OK || block_m < 1) return 0;
  return static_cast<size_t>(T) * cfg->top_k +
         static_cast<size_t>(n_local(cfg)) * (block_m - 1);
}

size_t moe_route_workspace_size(const moe_config* cfg, int T) {
  if (validate_cfg(cfg) != MOE_OK || validate_T(T) != MOE_OK) return 0;
  return route_layout(cfg, T).total;
}

int moe_route(const moe_config* cfg, int T, const void* x, const void* router_w,
              const float* router_bias, int32_t* topk_ids, float* topk_w, void* ws,
              size_t ws_bytes, void* stream) {
  MOE_TRY(validate_cfg(cfg));
  MOE_TRY(validate_T(T));
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(router_w)) return MOE_ERR_INVALID_ARG;
  const RouteLayout L = route_layout(cfg, T);
  if (!ws || ws_bytes < L.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = at<unsigned>(ws, L.status);
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, 4, st)));
  return do_route(cfg, T, x, router_w, router_bias, topk_ids, topk_w, at<float>(ws, L.logits),
                  status, st);
}

size_t moe_align_workspace_size(const moe_config* cfg, int T) {
  if (validate_cfg(cfg) != MOE_OK || validate_T(T) != MOE_OK) return 0;
  return align_layout(cfg, T).total;
}

int moe_align_permute(const moe_config* cfg, int T, const int32_t* topk_ids,
                      const int32_t* expert_map, int block_m, int32_t* counts, int32_t* offsets,
                      int32_t* sorted_ids, int32_t* inv_pos, int cap, void* ws, size_t ws_bytes,
                      void* stream) {
  MOE_TRY(validate_cfg(cfg));
  MOE_TRY(validate_T(T));
  if (block_m < 1 || block_m > 4096) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !counts || !offsets || !sorted_ids || !inv_pos) return MOE_ERR_INVALID_ARG;
  if (cfg->max_replicas > 0 && !expert_map) return MOE_ERR_INVALID_ARG;
  if (cap < 0 || static_cast<size_t>(cap) < moe_align_cap(cfg, T, block_m))
    return MOE_ERR_WORKSPACE;
  const AlignLayout L = align_layout(cfg, T);
  if (!ws || ws_bytes < L.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = at<unsigned>(ws, L.status);
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, 4, st)));
  const int El = n_local(cfg);
  return cuda_ok(launch_align(topk_ids, static_cast<long>(T) * cfg->top_k, expert_map,
                              cfg->num_experts, El, cfg->ep_rank * El, block_m,
                              at<int>(ws, L.hist), counts, offsets, sorted_ids, inv_pos, cap,
                              status, st, nullptr, nullptr, 0, 0, cfg->top_k,
                              cfg->max_replicas));
}

size_t moe_grouped_mlp_workspace_size(const moe_config* cfg, int T, int cap) {
  if (validate_cfg(cfg) != MOE_OK || validate_T(T) != MOE_OK || cap < 0) return 0;
  return mlp_layout(cfg, T, cap).total;
}

int moe_grouped_mlp(const moe_config* cfg, int T, const void* x, const int32_t* sorted_ids,
                    const int32_t* counts, const int32_t* offsets, int cap, const void* w13,
                    const void* w2, void* y_perm, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(validate_cfg(cfg));
  MOE_TRY(validate_T(T));
  if (T == 0) return MOE_OK;
  if (!x || !sorted_ids || !counts || !offsets || !w13 || !w2 || !y_perm)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13) || !aligned16(w2) || !aligned16(y_perm))
    return MOE_ERR_INVALID_ARG;
  if (cap < 1) return MOE_ERR_WORKSPACE;
  const MlpLayout L = mlp_layout(cfg, T, cap);
  if (!ws || ws_bytes < L.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = at<unsigned>(ws, L.status);
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, L.sync.bytes, st)));
  return do_mlp(cfg, T, x, sorted_ids, counts, offsets, cap, w13, w2, y_perm,
                at<Tile>(ws, L.tiles), at<int>(ws, L.groups), L.sync, at<void>(ws, L.x_perm),
                at<void>(ws, L.h_perm), at<float>(ws, L.part1), status, st);
}

int moe_combine(const moe_config* cfg, int T, const void* y_perm, int cap, const int32_t* inv_pos,
                const float* topk_w, const void* shared_out, void* out, void* ws,
                size_t ws_bytes, void* stream) {
  MOE_TRY(validate_cfg(cfg));
  MOE_TRY(validate_T(T));
  if (T == 0) return MOE_OK;
  if (!y_perm || !inv_pos || !topk_w || !out || cap < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(out) || (shared_out && !aligned16(shared_out)))
    return MOE_ERR_INVALID_ARG;
  if (ws && ws_bytes < 4) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = ws ? static_cast<unsigned*>(ws) : nullptr;
  if (status) MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, 4, st)));
  return cuda_ok(launch_combine(cfg->act_dtype == MOE_BF16, y_perm, cap, inv_pos, topk_w,
                                cfg->top_k, local_rows(cfg), shared_out, shared_out ? 1 : 0,
                                0, cfg->routed_scaling_factor, out, T, cfg->hidden_size,
                                status, st));
}

// ------------------------------------------------------ expert parallel
size_t moe_ep_dispatch_workspace_size(const moe_config* cfg, int T) {
  if (validate_cfg(cfg) != MOE_OK || validate_T(T) != MOE_OK) return 0;
  return ep_layout(cfg, T).total;
}

int moe_ep_dispatch(const moe_config* cfg, int T, const void* x, const int32_t* topk_ids,
                    const float* topk_w, const int32_t* phys_map, int32_t* send_counts,
                    int32_t* send_offsets, int32_t* send_pos, void* send_x, int32_t* send_ids,
                    float* send_w, int32_t* send_tok, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(validate_cfg(cfg));
  // the global placement goes with replicas, and only with them
  if ((cfg->max_replicas > 0) != (phys_map != nullptr)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(validate_T(T));
  if (!send_counts || !send_offsets) return MOE_ERR_INVALID_ARG;
  const int ep = cfg->ep_size;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    MOE_TRY(cuda_ok(cudaMemsetAsync(send_counts, 0, 4 * static_cast<size_t>(ep), st)));
    return cuda_ok(cudaMemsetAsync(send_offsets, 0, 4 * static_cast<size_t>(ep + 1), st));
  }
  if (!x || !topk_ids || !topk_w || !send_pos || !send_x || !send_ids || !send_w || !send_tok)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(send_x)) return MOE_ERR_INVALID_ARG;
  const EpLayout L = ep_layout(cfg, T);
  if (!ws || ws_bytes < L.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  unsigned* status = at<unsigned>(ws, L.status);
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, 4, st)));
  const long n = static_cast<long>(T) * cfg->top_k;
  int32_t* dest = at<int32_t>(ws, L.dest);
  int32_t* phys = at<int32_t>(ws, L.phys);
  int32_t* sorted = at<int32_t>(ws, L.sorted);
  MOE_TRY(cuda_ok(launch_ep_dest(topk_ids, n, cfg->num_experts, n_local(cfg), dest, phys,
                                 phys_map, cfg->max_replicas, cfg->top_k,
                                 cfg->num_experts + cfg->num_redundant_experts, st)));
  // a stable counting sort of the items over the destination ranks
  MOE_TRY(cuda_ok(launch_align(dest, n, nullptr, ep, ep, 0, 1, at<int>(ws, L.hist), send_counts,
                               send_offsets, sorted, send_pos, static_cast<int>(n), status, st)));
  return cuda_ok(launch_ep_pack(cfg->act_dtype == MOE_BF16, x, phys, topk_w, sorted,
                                send_offsets + ep, n, cfg->top_k, cfg->hidden_size, send_x,
                                send_ids, send_w, send_tok, st));
}

size_t moe_ep_expert_compute_workspace_size(const moe_config* cfg, int R) {
  if (validate_cfg(cfg) != MOE_OK || validate_T(R) != MOE_OK) return 0;
  const moe_config c1 = ep_item_config(cfg);
  // the forward's layout, then the items' weights in segment order
  return fwd_layout(&c1, R).total + rup(4 * static_cast<size_t>(R));
}

int moe_ep_expert_compute(const moe_config* cfg, int R, const void* recv_x,
                          const int32_t* recv_ids, const float* recv_w, const void* w13,
                          const void* w2, void* y, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(validate_cfg(cfg));
  MOE_TRY(validate_T(R));
  if (R == 0) return MOE_OK;
  if (!recv_x || !recv_ids || !recv_w || !w13 || !w2 || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(recv_x) || !aligned16(w13) || !aligned16(w2) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  const moe_config c1 = ep_item_config(cfg);
  const FwdLayout L = fwd_layout(&c1, R);
  if (!ws || ws_bytes < moe_ep_expert_compute_workspace_size(cfg, R) || !aligned16(ws))
    return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = at<unsigned>(ws, L.status);
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, L.sync.bytes, st)));
  const int El = n_local(&c1);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* sorted_ids = at<int32_t>(ws, L.sorted_ids);
  int32_t* inv_pos = at<int32_t>(ws, L.inv_pos);
  // ids are global, or physical with replicas: slot = id - ep_rank * E_local
  MOE_TRY(cuda_ok(launch_align(recv_ids, R, nullptr,
                               cfg->num_experts + cfg->num_redundant_experts, El,
                               cfg->ep_rank * El,
                               kForwardBlock, at<int>(ws, L.hist), counts, offsets, sorted_ids,
                               inv_pos, L.cap, status, st, at<Tile>(ws, L.tiles),
                               at<int>(ws, L.groups), routed_nmax(&c1, R),
                               static_cast<int>(max_routed_tiles(&c1, R)))));
  if (gemms_on_pairs(&c1, R)) {
    // GEMM2 writes each item's row straight to y, weighted; dropped items
    // (ids outside the shard) get zero rows
    MOE_TRY(do_mlp(&c1, R, recv_x, sorted_ids, counts, offsets, L.cap, w13, w2, y,
                   at<Tile>(ws, L.tiles), at<int>(ws, L.groups), L.sync, at<void>(ws, L.x_perm),
                   at<void>(ws, L.h_perm), at<float>(ws, L.part1), status, st, nullptr, true,
                   sorted_ids, recv_w, at<float>(ws, L.total)));
    return cuda_ok(launch_zero_dropped_rows(inv_pos, R,
                                            static_cast<long>(c1.hidden_size) * ebytes(c1.act_dtype),
                                            y, st));
  }
  MOE_TRY(do_mlp(&c1, R, recv_x, sorted_ids, counts, offsets, L.cap, w13, w2,
                 at<void>(ws, L.y_perm), at<Tile>(ws, L.tiles), at<int>(ws, L.groups), L.sync,
                 at<void>(ws, L.x_perm), at<void>(ws, L.h_perm), at<float>(ws, L.part1), status,
                 st, nullptr, true));
  return cuda_ok(launch_combine(c1.act_dtype == MOE_BF16, at<void>(ws, L.y_perm), L.cap,
                                inv_pos, recv_w, 1, 1, nullptr, 0, 0, 1.0f, y, R,
                                c1.hidden_size, status, st));
}

int moe_ep_combine(const moe_config* cfg, int T, const void* ret, const int32_t* send_pos,
                   const void* shared_out, void* out, void* ws, size_t ws_bytes,
                   void* stream) {
  MOE_TRY(validate_cfg(cfg));
  MOE_TRY(validate_T(T));
  if (T == 0) return MOE_OK;
  if (!ret || !send_pos || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ret) || !aligned16(out) || (shared_out && !aligned16(shared_out)))
    return MOE_ERR_INVALID_ARG;
  if (ws && ws_bytes < 4) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = ws ? static_cast<unsigned*>(ws) : nullptr;
  if (status) MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, 4, st)));
  return cuda_ok(launch_combine(cfg->act_dtype == MOE_BF16, ret, T * cfg->top_k, send_pos,
                                nullptr, cfg->top_k, cfg->top_k, shared_out,
                                shared_out ? 1 : 0, 0, cfg->routed_scaling_factor, out, T,
                                cfg->hidden_size, status, st));
}

size_t moe_workspace_size(const moe_config* cfg, int T) {
  if (validate_cfg(cfg) != MOE_OK || validate_T(T) != MOE_OK) return 0;
  return fwd_layout(cfg, T).total;
}

int moe_workspace_layout(const moe_config* cfg, int T, moe_workspace_offsets* out) {
  MOE_TRY(validate_cfg(cfg));
  MOE_TRY(validate_T(T));
  if (!out) return MOE_ERR_INVALID_ARG;
  const FwdLayout L = fwd_layout(cfg, T);
  out->status = L.status;
  out->topk_ids = L.topk_ids;
  out->topk_w = L.topk_w;
  out->counts = L.counts;
  out->offsets = L.offsets;
  out->sorted_ids = L.sorted_ids;
  out->inv_pos = L.inv_pos;
  out->total = L.total;
  out->cap = L.cap;
  out->block_m = kForwardBlock;
  return MOE_OK;
}

int moe_forward_plan(const moe_config* cfg, int T, moe_plan* out) {
  MOE_TRY(validate_cfg(cfg));
  MOE_TRY(validate_T(T));
  if (!out) return MOE_ERR_INVALID_ARG;
  moe_plan p;
  p.fused_route = route_align_small_ok(T, cfg->top_k, n_local(cfg)) ? 1 : 0;
  p.router_tensor_cores = !p.fused_route && router_on_tensor_cores(cfg, T) ? 1 : 0;
  p.router_partials = p.fused_route ? 1 : router_ksplit(cfg, T);
  p.align_kernels =
      p.fused_route ? 0 : align_kernel_count(static_cast<long>(T) * cfg->top_k, n_local(cfg));
  p.tile_rows = routed_nmax(cfg, T);
  p.fused_mlp = mlp_fused(cfg, T) ? 1 : 0;
  p.gemm1_k_split = gemm1_ksplit(cfg, T);
  p.cta_pairs = gemms_on_pairs(cfg, T) ? 1 : 0;
  p.gemm2_overlap = gemm2_early(cfg, T) ? 1 : 0;
  p.combine_ring = T > 0 && combine_uses_ring(cfg->act_dtype == MOE_BF16, T, cfg->top_k,
                                              local_rows(cfg), cfg->num_shared_experts,
                                              cfg->hidden_size)
                       ? 1
                       : 0;
  p.kernels = 0;
  if (T > 0) {
    // logits + top-k and align (or the fused route kernel), the routed MLP
    // (gather + fused kernel; gather + GEMMs on CTA pairs; GEMMs on single
    // CTAs, which gather their token rows themselves, with a finalize kernel
    // when GEMM1 is split over K), shared GEMMs, combine
    p.kernels = (p.fused_route ? 1 : 2 + p.align_kernels) +
                (p.fused_mlp ? 2 : p.cta_pairs ? 3 : p.gemm1_k_split > 1 ? 3 : 2) +
                (cfg->num_shared_experts > 0 ? 2 : 0) + 1;
  }
  *out = p;
  return MOE_OK;
}

static int forward_impl(const moe_config* cfg, int T, const void* x, const void* router_w,
                        const float* router_bias, const void* w13, const void* w2,
                        const void* shared_w13, const void* shared_w2,
                        const int32_t* expert_map, void* out, void* ws, size_t ws_bytes,
                        void* stream, void* const* events, int* kernels) {
  MOE_TRY(validate_cfg(cfg));
  MOE_TRY(validate_T(T));
  if (kernels) *kernels = 0;
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !w13 || !w2 || !out) return MOE_ERR_INVALID_ARG;
  if (cfg->max_replicas > 0 && !expert_map) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(w13) || !aligned16(w2) ||
      !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  const bool with_shared = cfg->num_shared_experts > 0 && shared_w13 && shared_w2;
  if (with_shared && (!aligned16(shared_w13) || !aligned16(shared_w2)))
    return MOE_ERR_INVALID_ARG;
  const FwdLayout L = fwd_layout(cfg, T);
  if (!ws || ws_bytes < L.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto mark = [&](int i) -> int { return events ? record_event(events[i], st) : MOE_OK; };
  const int El = n_local(cfg), H = cfg->hidden_size, K = cfg->top_k;
  unsigned* status = at<unsigned>(ws, L.status);
  int32_t* ids = at<int32_t>(ws, L.topk_ids);
  float* w = at<float>(ws, L.topk_w);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* sorted_ids = at<int32_t>(ws, L.sorted_ids);
  int32_t* inv_pos = at<int32_t>(ws, L.inv_pos);
  const long launches0 = g_kernel_launches;

  MOE_TRY(mark(0));
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, L.sync.bytes, st)));
  if (route_align_small_ok(T, K, El)) {
    RouteAlignArgs a;
    a.x = x;
    a.wg = router_w;
    a.bias = router_bias;
    a.T = T;
    a.E = cfg->num_experts;
    a.H = H;
    a.K = K;
    a.renorm = cfg->renormalize ? 1 : 0;
    a.flags = route_flags(cfg);
    a.n_group = cfg->use_grouped_topk ? cfg->num_expert_group : 0;
    a.topk_group = cfg->use_grouped_topk ? cfg->topk_group : 0;
    a.logits = at<float>(ws, L.logits);
    a.tickets = reinterpret_cast<int*>(status + 1);
    a.ids = ids;
    a.w = w;
    a.emap = expert_map;
    a.R = cfg->max_replicas;
    a.E_l = El;
    a.ep_start = cfg->ep_rank * El;
    a.block_m = kForwardBlock;
    a.counts = counts;
    a.offsets = offsets;
    a.sorted_ids = sorted_ids;
    a.inv_pos = inv_pos;
    a.cap = L.cap;
    a.status = status;
    a.tiles = at<Tile>(ws, L.tiles);
    a.group_start = at<int>(ws, L.groups);
    a.nmax = routed_nmax(cfg, T);
    a.max_tiles = static_cast<int>(max_routed_tiles(cfg, T));
    MOE_TRY(cuda_ok(launch_route_align_small(a, cfg->act_dtype == MOE_BF16,
                                             cfg->router_dtype == MOE_BF16, st)));
    MOE_TRY(mark(1));  // routing and align share one kernel
  } else {
    MOE_TRY(do_route(cfg, T, x, router_w, router_bias, ids, w, at<float>(ws, L.logits),
                     status, st));
    MOE_TRY(mark(1));
    MOE_TRY(cuda_ok(launch_align(ids, static_cast<long>(T) * K, expert_map, cfg->num_experts,
                                 El, cfg->ep_rank * El, kForwardBlock, at<int>(ws, L.hist),
                                 counts, offsets, sorted_ids, inv_pos, L.cap, status, st,
                                 at<Tile>(ws, L.tiles), at<int>(ws, L.groups),
                                 routed_nmax(cfg, T),
                                 static_cast<int>(max_routed_tiles(cfg, T)), K,
                                 cfg->max_replicas)));
  }
  MOE_TRY(mark(2));
  MOE_TRY(do_mlp(cfg, T, x, sorted_ids, counts, offsets, L.cap, w13, w2,
                 at<void>(ws, L.y_perm), at<Tile>(ws, L.tiles), at<int>(ws, L.groups),
                 L.sync, at<void>(ws, L.x_perm), at<void>(ws, L.h_perm),
                 at<float>(ws, L.part1), status, st, events ? events + 3 : nullptr, true));
  MOE_TRY(mark(5));
  const void* shared_y = nullptr;
  int S = 0;
  if (with_shared) {
    S = cfg->num_shared_experts;
    const int Is = cfg->shared_intermediate_size;
    const bool sp = shared_on_pairs(cfg, T);
    const int nm = sp ? 256 : dense_nmax(T);
    void* h_sh = at<void>(ws, L.h_sh);
    void* y_sh = at<void>(ws, L.y_sh);
    MOE_TRY(run_gemm(kGemmSiluUp, cfg->act_dtype, nm, shared_w13, static_cast<long>(S) * 2 * Is,
                     x, T, H, nullptr, nullptr, S, Is / 128, 2 * Is, Is, 0, h_sh, Is, Is, status,
                     st, 1, 0, T, sp, nullptr, nullptr, nullptr, 0,
                     out_bounds(static_cast<long>(S) * T)));
    MOE_TRY(run_gemm(kGemmPlain, cfg->act_dtype, nm, shared_w2, static_cast<long>(S) * H, h_sh,
                     static_cast<long>(S) * T, Is, nullptr, nullptr, S, H / (sp ? 256 : 128), H,
                     0, 1, y_sh, H, H, status, st, 1, 0, T, sp, nullptr, nullptr, nullptr, 0,
                     out_bounds(static_cast<long>(S) * T)));
    shared_y = y_sh;
  }
  MOE_TRY(mark(6));
  MOE_TRY(cuda_ok(launch_combine(cfg->act_dtype == MOE_BF16, at<void>(ws, L.y_perm), L.cap,
                                 inv_pos, w, K, local_rows(cfg), shared_y, S,
                                 static_cast<long>(T) * H,
                                 cfg->routed_scaling_factor, out, T, H, status, st,
                                 /*slots_early=*/true)));  // ids, weights, inv_pos: >= 3 back
  MOE_TRY(mark(7));
  if (kernels) *kernels = static_cast<int>(g_kernel_launches - launches0);
  return MOE_OK;
}

int moe_forward(const moe_config* cfg, int T, const void* x, const void* router_w,
                const float* router_bias, const void* w13, const void* w2,
                const void* shared_w13, const void* shared_w2, const int32_t* expert_map,
                void* out, void* ws, size_t ws_bytes, void* stream) {
  return forward_impl(cfg, T, x, router_w, router_bias, w13, w2, shared_w13, shared_w2,
                      expert_map, out, ws, ws_bytes, stream, nullptr, nullptr);
}

int moe_forward_timed(const moe_config* cfg, int T, const void* x, const void* router_w,
                      const float* router_bias, const void* w13, const void* w2,
                      const void* shared_w13, const void* shared_w2,
                      const int32_t* expert_map, void* out, void* ws, size_t ws_bytes,
                      void* stream, void* const* events, int* kernels_launched) {
  return forward_impl(cfg, T, x, router_w, router_bias, w13, w2, shared_w13, shared_w2,
                      expert_map, out, ws, ws_bytes, stream, events, kernels_launched);
}

int moe_set_wait_limit_ns(uint64_t ns) {
  const unsigned long long v = ns ? ns : 1000000000ull;  // 0: the default, 1 s
  cudaError_t (*const setters[])(unsigned long long) = {
      set_wait_limit_gemm, set_wait_limit_gemm_pair, set_wait_limit_mlp_fused,
      set_wait_limit_route, set_wait_limit_align};
  for (auto set : setters)
    MOE_TRY(cuda_ok(set(v)));
  return MOE_OK;
}

int moe_last_cuda_error(void) { return g_last_cuda_error; }

int moe_get_status(const void* ws, void* stream, uint32_t* flags) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  MOE_TRY(cuda_ok(cudaMemcpyAsync(&v, ws, 4, cudaMemcpyDeviceToHost, st)));
  MOE_TRY(cuda_ok(cudaStreamSynchronize(st)));
  if (flags) *flags = v;
  if (v == 0) return MOE_OK;
  return (v & MOE_DEV_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE_STATUS;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Debug build (MOE_DEBUG): the bounds-check records of every translation unit.
namespace moe {
namespace {

// One failed check and no memory access, so that a test can see the record
// path of the debug build work.
__global__ void dbg_selftest_kernel(int i, int n) {
  if (threadIdx.x == 0 && blockIdx.x == 0) (void)MOE_DCHECK(i, n);
}

}  // namespace

MOE_DEBUG_TAKER(take_dbg_api)

}  // namespace moe

extern "C" int moe_debug_build(void) { return MOE_DEBUG_BUILD; }

extern "C" int moe_debug_take(moe_debug_record* rec) {
  if (!rec) return MOE_ERR_INVALID_ARG;
  std::memset(rec, 0, sizeof(*rec));
  if (!MOE_DEBUG_BUILD) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(cuda_ok(cudaDeviceSynchronize()));
  cudaError_t (*const takers[])(DbgRecord*) = {take_dbg_api,       take_dbg_gemm,
                                               take_dbg_gemm_pair, take_dbg_mlp_fused,
                                               take_dbg_route,     take_dbg_align};
  for (auto take : takers) {
    DbgRecord r = {};
    MOE_TRY(cuda_ok(take(&r)));
    if (r.count && !rec->count) {
      rec->site = r.site;
      rec->index = r.index;
      rec->bound = r.bound;
    }
    rec->count += r.count;
  }
  return MOE_OK;
}

extern "C" int moe_debug_selftest(void* stream) {
  if (!MOE_DEBUG_BUILD) return MOE_ERR_UNSUPPORTED;
  dbg_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(5, 4);
  return cuda_ok(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// moe_align_permute_noalloc: the align/permute launch with its scratch in a
// static device array instead of a caller workspace (see include/moe.h).
static __device__ __align__(256) unsigned char moe_align_noalloc_scratch
    [MOE_ALIGN_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the static scratch in the current context. The host-side
// name of the array is only a stand-in, so the address is looked up with the
// caller's device current, on every call: a cached address would go stale
// once the module is loaded again (after cudaDeviceReset, or in another
// context made current on the same device). The lookup allocates nothing;
// the first one in a context loads the library's device code, which is why
// that first call belongs before any stream capture.
int noalloc_scratch(void** out) {
  void* p = nullptr;
  MOE_TRY(cuda_ok(cudaGetSymbolAddress(&p, moe_align_noalloc_scratch)));
  if (!p) return fail_cuda(static_cast<int>(cudaErrorInvalidSymbol));
  *out = p;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_align_permute_noalloc(const moe_config* cfg, int T, const int32_t* topk_ids,
                                         const int32_t* expert_map, int block_m,
                                         int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                                         int32_t* inv_pos, int cap, void* stream) {
  MOE_TRY(validate_cfg(cfg));
  MOE_TRY(validate_T(T));
  if (block_m < 1 || block_m > 4096) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !counts || !offsets || !sorted_ids || !inv_pos) return MOE_ERR_INVALID_ARG;
  if (cfg->max_replicas > 0 && !expert_map) return MOE_ERR_INVALID_ARG;
  if (cap < 0 || static_cast<size_t>(cap) < moe_align_cap(cfg, T, block_m))
    return MOE_ERR_WORKSPACE;
  const AlignLayout L = align_layout(cfg, T);
  if (L.total > MOE_ALIGN_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  MOE_TRY(noalloc_scratch(&scratch));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = at<unsigned>(scratch, L.status);
  MOE_TRY(cuda_ok(cudaMemsetAsync(status, 0, 4, st)));
  // the per-warp counts need no clearing: pass 1 writes every entry it reads
  const int El = n_local(cfg);
  return cuda_ok(launch_align(topk_ids, static_cast<long>(T) * cfg->top_k, expert_map,
                              cfg->num_experts, El, cfg->ep_rank * El, block_m,
                              at<int>(scratch, L.hist), counts, offsets, sorted_ids, inv_pos,
                              cap, status, st, nullptr, nullptr, 0, 0, cfg->top_k,
                              cfg->max_replicas));
}
