/*
 * moe.h -- C ABI of the fused Mixture-of-Experts layer forward for sm_103a.
 *
 * One layer forward is:
 *   route         router GEMM, fp32 softmax, (grouped) top-k, renormalise
 *   align/permute expert_map mask, per-local-expert padded segments
 *   grouped MLP   GEMM1 with the SiLU(gate)*up epilogue on the token rows
 *                 gathered by expert, GEMM2
 *   combine       weighted gather back to token order, routed_scaling_factor,
 *                 plus the shared-expert output
 * Each stage is a hand-written CUDA kernel. moe_forward runs all of them.
 *
 * Sources of the semantics (the web pages this library restates):
 *   - SGLang issue "[Feature] Expert parallelism support", MixtralMoE:
 *     gate = bias-free linear over all experts, softmax in fp32, topk,
 *     renormalise, sum over experts of weight * expert MLP.
 *   - ep_fused_moe_patch.py (EP-aware FusedMoE override): _ep_init
 *     (num_experts % ep_size == 0; local experts [r*E/ep, (r+1)*E/ep)),
 *     _ep_forward (global routing, flatten (token, slot) work items, local
 *     expert compute, weighted scatter-add back to tokens).
 *   - vLLM docs, MoEMixin.recursive_replace: top_k, moe_intermediate_size,
 *     renormalize = norm_topk_prob, routed_scaling_factor, n_group /
 *     topk_group (use_grouped_topk), n_shared_experts, router dtype,
 *     activation "silu", gate_up_proj (E, 2I, H).
 *   - vllm-omni "Expert Parallel": shared experts are added unweighted on
 *     every rank; EP size divisibility; contiguous local expert ranges.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers of the current CUDA device.
 *     They are row-major and contiguous, with 16-byte-aligned bases. The
 *     caller owns every buffer. The library allocates no device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All work is enqueued asynchronously on it. Only
 *     moe_get_status synchronises, and only that stream.
 *   - `ws` is caller-owned device scratch of at least the size reported by
 *     the matching *_workspace_size call. Its first 4 bytes are the device
 *     status word (MOE_DEV_* flags). Each call that takes `ws` clears that
 *     word first, so it reports on the latest call only. Read it with
 *     moe_get_status.
 *   - Arguments are validated on the host before any CUDA call. Invalid
 *     ones return MOE_ERR_INVALID_ARG (or MOE_ERR_UNSUPPORTED, or
 *     MOE_ERR_WORKSPACE) and enqueue nothing. A launch failure returns
 *     MOE_ERR_CUDA. Data-dependent faults found on the device (an expert id
 *     out of range, a full segment buffer, a pipeline wait that timed out)
 *     never trap. They set a MOE_DEV_* flag and skip the offending access.
 *   - T == 0 is a valid no-op that returns MOE_OK. T (and the received row
 *     count R of moe_ep_expert_compute) may be at most 262144 (2^18);
 *     larger or negative values return MOE_ERR_INVALID_ARG, and the
 *     workspace queries return 0 for them.
 *   - Calls that share a `ws` buffer must be ordered, as on one stream.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The entry points below are the library's only exported symbols; it is
 * compiled with hidden visibility, so that two builds loaded in one process
 * (libmoe.so and libmoe_debug.so) share no internal state. */
#if defined(__GNUC__) || defined(__clang__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* bad config, size, pointer or alignment     */
  MOE_ERR_UNSUPPORTED = 2,   /* valid, but outside what the kernels cover  */
  MOE_ERR_WORKSPACE = 3,     /* ws too small / NULL, or cap too small      */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed          */
  MOE_ERR_DEVICE_STATUS = 5, /* moe_get_status: a MOE_DEV_* flag is set    */
  MOE_ERR_TIMEOUT = 6        /* moe_get_status: MOE_DEV_TIMEOUT is set     */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Device status flags (bit OR, first 4 bytes of ws). */
#define MOE_DEV_BAD_EXPERT_ID 0x1u /* topk id not in [0,E) or expert_map value
                                      not in [-1,E_local): item dropped      */
#define MOE_DEV_CAP_OVERFLOW 0x2u  /* padded segments exceed cap or a tile
                                      table overflowed: rows dropped        */
#define MOE_DEV_TIMEOUT 0x4u       /* a GEMM pipeline wait passed its time
                                      limit; that kernel stopped early      */
#define MOE_DEV_BAD_SEGMENT 0x8u   /* offsets/counts inconsistent          */

/* Layer description. The field names follow the FusedMoE arguments the
 * pages pass (num_experts, top_k, hidden_size, intermediate_size,
 * renormalize, use_grouped_topk, num_expert_group, topk_group,
 * routed_scaling_factor, shared experts, ep_size / ep_rank). */
typedef struct {
  int num_experts;           /* E: global routed experts (router width)      */
  int top_k;                 /* K: experts per token, 1 <= K <= min(E, 32)   */
  int hidden_size;           /* H: multiple of 128                           */
  int intermediate_size;     /* I: per routed expert, multiple of 128        */
  int renormalize;           /* 1: topk_w /= sum(topk_w) per token           */
  int use_grouped_topk;      /* 1: group-limited top-k (reading below)       */
  int num_expert_group;      /* n_group: E % n_group == 0, n_group <= 32     */
  int topk_group;            /* groups kept per token, 1..n_group            */
  float routed_scaling_factor; /* rsf: multiplies the routed sum; 1 = off    */
  int num_shared_experts;    /* S >= 0 shared experts, added unweighted      */
  int shared_intermediate_size; /* I_s of each shared expert (x128)          */
  int ep_size;               /* expert-parallel size; (E + redundant) % ep_size
                                == 0                                         */
  int ep_rank;               /* this shard, 0 <= ep_rank < ep_size           */
  moe_dtype act_dtype;       /* x, expert weights, y_perm, out               */
  moe_dtype router_dtype;    /* router weight storage (logits are fp32)      */
  int scoring_func;          /* MOE_SCORE_SOFTMAX (0) or MOE_SCORE_SIGMOID (1) */
  int bias_mode;             /* role of router_bias: MOE_BIAS_LOGIT (0) or
                                MOE_BIAS_SELECT (1), reading below          */
  int max_replicas;          /* 0: expert_map is the plain map [E]; R in 1..16:
                                expert_map is a replica map [E, R] (redundant
                                experts, reading below)                      */
  int num_redundant_experts; /* extra physical replicas over all ranks (needs
                                max_replicas > 0); each rank holds
                                E_local = (E + this) / ep_size weight slots  */
} moe_config;

/* Redundant experts (max_replicas = R > 0). The pages name redundant experts
 * (num_redundant_experts, physical and logical experts) without a placement
 * policy. Row e of the replica map lists the physical replicas of logical
 * expert e in one global order: the local slot in [0, E_l) of a replica on
 * this rank, -1 for a replica on another rank, then -2 padding. The reading
 * taken: work item (t, k) of expert e goes to replica t mod n_e (n_e = the
 * replicas listed), so a hot expert's tokens are spread round robin and each
 * item lands on exactly one replica across the ranks; the slot's weights are
 * w13[slot], w2[slot]. A row without replicas, or with a value outside
 * [-2, E_l), drops the item and sets MOE_DEV_BAD_EXPERT_ID.
 *
 * Routing scores p: fp32 softmax over the E logits (MixtralMoE.forward), or,
 * with MOE_SCORE_SIGMOID, 1 / (1 + exp(-logit)) per expert. The pages name a
 * non-softmax scoring_func among the FusedMoE routing arguments without
 * defining it; the elementwise logistic is the reading taken.
 *
 * router_bias (nullable, fp32 [E]): with MOE_BIAS_LOGIT it is added to the
 * logits before scoring (a skew input of this library). With MOE_BIAS_SELECT
 * it is the per-expert score correction the pages name as
 * e_score_correction_bias: it is added to p only to choose the groups and
 * the top-k, and the weights are the uncorrected p of the chosen experts.
 *
 * Grouped top-k reading: the E experts form n_group contiguous groups of
 * E/n_group. A group's score is the max selection score of its members.
 * The topk_group best groups are kept (ties to the lower group id). Top-k
 * then runs over the kept experts (ties to the lower expert id), and the
 * weights are the scores p of the chosen experts. */
#define MOE_SCORE_SOFTMAX 0
#define MOE_SCORE_SIGMOID 1
#define MOE_BIAS_LOGIT 0
#define MOE_BIAS_SELECT 1

/* Human-readable name of a moe_status. Never NULL. */
MOE_API const char* moe_strerror(int status);

/* Host-only validation of a config (no CUDA call). Returns MOE_OK,
 * MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED. Checks: E % ep_size == 0 and
 * 0 <= ep_rank < ep_size (ep_fused_moe_patch.py _ep_init assert), E_local >= 1
 * (MixtralMoE "has no experts" error), 1 <= K <= E, grouped constraints
 * (E % n_group == 0, 1 <= topk_group <= n_group, K <= topk_group*E/n_group),
 * H and I multiples of 128, S >= 0 with I_s a multiple of 128 when S > 0.
 * Kernel limits (MOE_ERR_UNSUPPORTED): E <= 512, K <= 32, n_group <= 32,
 * E_local <= 1024, S <= 1024, and act_dtype F32 needs router_dtype F32. */
MOE_API int moe_validate_config(const moe_config* cfg);

/* Rows of the padded permutation buffers for T tokens and segment padding
 * block_m: T*K + E_local*(block_m-1). Returns 0 on an invalid config. */
MOE_API size_t moe_align_cap(const moe_config* cfg, int T, int block_m);

/* ------------------------------------------------------------------------ */
/* moe_route: router logits, fp32 softmax over E, top-k, renormalise.
 * MixtralMoE.forward (gate, F.softmax(dtype=float), torch.topk, divide by
 * the sum); ep_fused_moe_patch.py _ep_forward step 1 (global routing: all E
 * experts on every rank).
 *   x           [T, H]  act_dtype
 *   router_w    [E, H]  router_dtype
 *   router_bias [E]     fp32, nullable. It is added to the logits before the
 *                       softmax (a per-expert skew of the load).
 *   topk_ids    [T, K]  int32 out: global expert ids in descending
 *                       probability, ties to the lower id.
 *   topk_w      [T, K]  fp32 out: softmax probabilities of those experts
 *                       (renormalised to sum 1 when cfg->renormalize).
 *                       routed_scaling_factor is NOT applied here.
 * ws: moe_route_workspace_size(cfg, T) bytes (status word + fp32 logits). */
MOE_API size_t moe_route_workspace_size(const moe_config* cfg, int T);
MOE_API int moe_route(const moe_config* cfg, int T, const void* x, const void* router_w,
                      const float* router_bias, int32_t* topk_ids, float* topk_w,
                      void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* moe_align_permute: keep local experts, sort work items by local expert.
 * Work item i = t*K + k is (token t, slot k), the flattening in
 * ep_fused_moe_patch.py _ep_forward step 2. expert_map turns global ids
 * into local ids (-1 = not on this rank: the item is dropped, as step 3
 * keeps only local ids).
 *   topk_ids    [T, K] int32 global ids
 *   expert_map  [E] int32 (values in [-1, E_local)), or NULL for the
 *               contiguous shard of cfg->ep_rank: id - ep_rank*E/ep_size;
 *               with cfg->max_replicas = R > 0 a replica map [E, R]
 *               (required; see the redundant-experts reading above).
 *   block_m     segment padding (>= 1). The grouped MLP accepts any value.
 *   counts      [E_local]   out: items per local expert (unpadded)
 *   offsets     [E_local+1] out: exclusive prefix of counts, each rounded
 *               up to a multiple of block_m
 *   sorted_ids  [cap] out: rows offsets[e] .. offsets[e]+counts[e]-1 hold
 *               expert e's items in ascending item order (a stable sort).
 *               Every other row holds the sentinel T*K.
 *   inv_pos     [T*K] out: row of each item, -1 if dropped
 *   cap         rows of sorted_ids. Must be >= moe_align_cap(cfg,T,block_m),
 *               else MOE_ERR_WORKSPACE.
 * ws: moe_align_workspace_size(cfg, T) bytes. */
MOE_API size_t moe_align_workspace_size(const moe_config* cfg, int T);
MOE_API int moe_align_permute(const moe_config* cfg, int T, const int32_t* topk_ids,
                              const int32_t* expert_map, int block_m, int32_t* counts,
                              int32_t* offsets, int32_t* sorted_ids, int32_t* inv_pos,
                              int cap, void* ws, size_t ws_bytes, void* stream);

/* moe_align_permute_noalloc: moe_align_permute for callers that cannot
 * allocate device memory. The source pages have no counterpart to this entry
 * point; it exists for integration. Some hosts own every byte of device memory
 * through their own pool and forbid side allocations. Some serving loops must
 * not pay the implicit synchronisation of cudaMalloc. Some embedded callers
 * fix their memory budget at start-up. None of them can supply `ws`.
 *
 * The per-warp counts and the status word live instead in one scratch array
 * of MOE_ALIGN_NOALLOC_SCRATCH_BYTES, compiled into the library as a static
 * device array. Every GPU that loads the library holds that array until the
 * process exits. This call allocates nothing, on the host or on the device.
 *   - Arguments and outputs are as moe_align_permute, minus ws/ws_bytes.
 *   - Results are identical to moe_align_permute.
 *   - It returns MOE_ERR_WORKSPACE, before any CUDA call, when the scratch
 *     that (T, top_k, E_local) need, moe_align_workspace_size(cfg, T), exceeds
 *     MOE_ALIGN_NOALLOC_SCRATCH_BYTES. At 256 local experts that is about
 *     260k (token, slot) items.
 *   - Every call looks up the array's device address in the current context
 *     (cudaGetSymbolAddress with the caller's device current), so an address
 *     never outlives a cudaDeviceReset or a context switch. The first lookup
 *     in a context loads the library's device code: make the first call on
 *     each device before any stream capture.
 *   - All calls share the one array, and it keeps the last call's contents.
 *     Each call clears the status word it uses, and every count it reads is
 *     rewritten first. Calls that can overlap on the GPU (different streams
 *     without ordering, or several host threads) race on the array and must
 *     be serialised by the caller.
 *   - Device flags (MOE_DEV_*) land in the shared array and are not reported.
 *     Out-of-range expert ids are still dropped, exactly as moe_align_permute
 *     drops them. */
#define MOE_ALIGN_NOALLOC_SCRATCH_BYTES (1u << 20)
MOE_API int moe_align_permute_noalloc(const moe_config* cfg, int T, const int32_t* topk_ids,
                                      const int32_t* expert_map, int block_m, int32_t* counts,
                                      int32_t* offsets, int32_t* sorted_ids, int32_t* inv_pos,
                                      int cap, void* stream);

/* ------------------------------------------------------------------------ */
/* moe_grouped_mlp: the local experts' SiLU-gated MLPs on permuted rows.
 * For every row r of segment e with sorted_ids[r] < T*K:
 *   y_perm[r] = W2[e] . ( silu(W13[e][0:I] . x_t) * (W13[e][I:2I] . x_t) ),
 *   t = sorted_ids[r] / K.
 * The expert MLP is MixtralMLP with activation "silu" (MoEMixin); w1 = w13,
 * w2 as passed to fused_experts (ep_fused_moe_patch.py _ep_forward step 3).
 *   x        [T, H] act_dtype
 *   sorted_ids, counts, offsets: as produced by moe_align_permute (any
 *            block_m); cap = rows of sorted_ids and y_perm.
 *   w13      [E_local, 2*I, H] act_dtype: gate rows [0,I), up rows [I,2I).
 *   w2       [E_local, H, I]   act_dtype ([out, in]).
 *   y_perm   [cap, H] act_dtype out. Only rows holding items are written.
 * Both GEMMs run on the tcgen05 tensor cores (bf16: kind::f16, fp32:
 * kind::tf32), with fp32 accumulation. The SiLU*up product is rounded to
 * act_dtype between them.
 * ws: moe_grouped_mlp_workspace_size(cfg, T, cap) bytes. */
MOE_API size_t moe_grouped_mlp_workspace_size(const moe_config* cfg, int T, int cap);
MOE_API int moe_grouped_mlp(const moe_config* cfg, int T, const void* x,
                            const int32_t* sorted_ids, const int32_t* counts,
                            const int32_t* offsets, int cap, const void* w13,
                            const void* w2, void* y_perm, void* ws, size_t ws_bytes,
                            void* stream);

/* ------------------------------------------------------------------------ */
/* moe_combine: weighted gather back to token order.
 *   out[t] = rsf * sum_{k : inv_pos[t*K+k] >= 0} topk_w[t,k] * y_perm[inv_pos]
 *            + shared_out[t]
 * This is the scatter_add_ by token of ep_fused_moe_patch.py _ep_forward
 * step 4, done as a deterministic per-token gather in slot order with fp32
 * accumulation. rsf = routed_scaling_factor (MoEMixin). The shared output is
 * added unweighted (vllm-omni "Expert Parallel", Step 5).
 *   y_perm     [cap, H] act_dtype
 *   inv_pos    [T*K] int32; entries outside [-1, cap) count as dropped
 *   topk_w     [T, K] fp32
 *   shared_out [T, H] act_dtype, nullable
 *   out        [T, H] act_dtype out
 * ws: NULL, or >= 4 bytes for the status word. */
MOE_API int moe_combine(const moe_config* cfg, int T, const void* y_perm, int cap,
                        const int32_t* inv_pos, const float* topk_w,
                        const void* shared_out, void* out, void* ws, size_t ws_bytes,
                        void* stream);

/* ------------------------------------------------------------------------ */
/* moe_forward: the whole layer (route -> align/permute -> grouped MLP of the
 * local experts and of the shared experts -> combine), stream-ordered with no
 * host synchronisation.
 *   x, router_w, router_bias: as moe_route
 *   w13, w2:     local experts, as moe_grouped_mlp ([E_local, ...]).
 *   shared_w13   [S, 2*I_s, H], shared_w2 [S, H, I_s]: nullable. When NULL
 *                (or S == 0) no shared output is added. With EP, pass them on
 *                one rank only if the partial outputs are to be summed.
 *   expert_map   as moe_align_permute (NULL = contiguous shard).
 *   out          [T, H] act_dtype. With ep_size > 1 this is the partial sum
 *                over this rank's experts. No collective is made.
 * Segments are padded to 16 rows. After the call, ws holds topk_ids,
 * topk_w, counts, offsets, sorted_ids and inv_pos at the byte offsets given
 * by moe_workspace_layout.
 * ws: moe_workspace_size(cfg, T) bytes. */
typedef struct {
  size_t status, topk_ids, topk_w, counts, offsets, sorted_ids, inv_pos;
  size_t total;   /* == moe_workspace_size */
  int cap;        /* rows of sorted_ids */
  int block_m;    /* segment padding used by moe_forward */
} moe_workspace_offsets;

MOE_API size_t moe_workspace_size(const moe_config* cfg, int T);
MOE_API int moe_workspace_layout(const moe_config* cfg, int T, moe_workspace_offsets* out);
MOE_API int moe_forward(const moe_config* cfg, int T, const void* x,
                        const void* router_w, const float* router_bias,
                        const void* w13, const void* w2, const void* shared_w13,
                        const void* shared_w2, const int32_t* expert_map, void* out,
                        void* ws, size_t ws_bytes, void* stream);

/* moe_forward plus instrumentation. No page counterpart: this entry point is
 * there so that each kernel's duration can be measured live on the stream that
 * runs it. events: 8 caller-created cudaEvent_t (as void*; any may be NULL),
 * recorded on `stream` at the stage boundaries:
 *   [0] start  [1] after routing  [2] after align/permute
 *   [3] after the tile table (and the row gather kernel on the CTA-pair and
 *       fused paths; on single CTAs GEMM1 gathers its rows itself)
 *   [4] after GEMM1 (SiLU*up)
 *   [5] after GEMM2  [6] after the shared experts  [7] after combine.
 * kernels_launched (nullable): number of kernels this call launched. The
 * results are identical to moe_forward. When `stream` is being captured into a
 * CUDA graph, the events are recorded as external event nodes
 * (cudaEventRecordExternal), so every replay timestamps the stages. */
MOE_API int moe_forward_timed(const moe_config* cfg, int T, const void* x,
                              const void* router_w, const float* router_bias,
                              const void* w13, const void* w2, const void* shared_w13,
                              const void* shared_w2, const int32_t* expert_map, void* out,
                              void* ws, size_t ws_bytes, void* stream,
                              void* const* events, int* kernels_launched);

/* ------------------------------------------------------------------------ */
/* Expert-parallel dispatch and combine: the rank-local halves of
 * ep_fused_moe_patch.py _ep_forward steps 2-4. The exchange between ranks
 * (all_to_all_single of the send buffers with the counts as split sizes, and
 * back) is the caller's: this library runs no collective.
 *
 * Redundant experts (cfg->max_replicas > 0; MoEMixin num_redundant_experts,
 * physical vs logical experts): each rank holds E_local =
 * (E + num_redundant_experts) / ep_size weight slots, and the physical expert
 * id of slot s on rank r is r * E_local + s. The sender picks the replica, so
 * moe_ep_dispatch takes the global placement: phys_map [E, max_replicas]
 * int32, row e listing the physical ids of logical expert e's replicas in
 * their global order, padded with -2 (the same order the per-rank replica
 * maps of moe_forward use). Item (t, k) goes to replica t mod n_e of its n_e
 * replicas, and the physical id is what it carries.
 *
 * moe_ep_dispatch (step 2). Work item i = t*K + k goes to rank
 * topk_ids[i] / (E / ep_size), or with replicas to rank phys / E_local of the
 * replica chosen above. The items are sorted by destination rank and packed.
 * The page's argsort leaves the order inside a destination open; here it is
 * stable (ascending i).
 *   x        [T, H] act_dtype
 *   topk_ids [T, K] int32 global (logical) ids, topk_w [T, K] fp32 (from
 *            moe_route)
 *   phys_map NULL without replicas; [E, max_replicas] as above with them
 *            (MOE_ERR_INVALID_ARG if given without, or missing with)
 *   send_counts  [ep_size] int32 out: rows for each destination rank
 *   send_offsets [ep_size + 1] int32 out: exclusive prefix of send_counts
 *   send_pos [T*K] int32 out: row of item i in the send buffers (-1 for an id
 *            outside [0, E), or a replica row with no entry or an entry
 *            outside the physical ids, which also sets MOE_DEV_BAD_EXPERT_ID)
 *   send_x   [T*K, H] act_dtype out, send_ids [T*K] int32 out (global ids, or
 *            physical ids with replicas), send_w [T*K] fp32 out, send_tok
 *            [T*K] int32 out (token index); rows past send_offsets[ep_size]
 *            are left untouched.
 * ws: moe_ep_dispatch_workspace_size(cfg, T) bytes. */
MOE_API size_t moe_ep_dispatch_workspace_size(const moe_config* cfg, int T);
MOE_API int moe_ep_dispatch(const moe_config* cfg, int T, const void* x, const int32_t* topk_ids,
                            const float* topk_w, const int32_t* phys_map, int32_t* send_counts,
                            int32_t* send_offsets, int32_t* send_pos, void* send_x, int32_t* send_ids,
                            float* send_w, int32_t* send_tok, void* ws, size_t ws_bytes, void* stream);

/* moe_ep_expert_compute (step 3): the R items this rank received, each run
 * through its expert with top_k = 1 and weighted, as the page's call to
 * fused_experts does:
 *   y[r] = recv_w[r] * f_{recv_ids[r] - ep_rank*E_local}(recv_x[r]).
 * Rows whose id is not one of this rank's experts come back as zeros. With
 * replicas the ids are physical (as moe_ep_dispatch sends them) and the slot
 * is recv_ids[r] - ep_rank*E_local in the same way.
 *   recv_x [R, H] act_dtype, recv_ids [R] int32 global ids, recv_w [R] fp32
 *   w13, w2: this rank's experts, as for moe_forward
 *   y      [R, H] act_dtype out
 * cfg's top_k, shared experts, routed_scaling_factor and routing fields are
 * not used. ws: moe_ep_expert_compute_workspace_size(cfg, R) bytes. */
MOE_API size_t moe_ep_expert_compute_workspace_size(const moe_config* cfg, int R);
MOE_API int moe_ep_expert_compute(const moe_config* cfg, int R, const void* recv_x,
                                  const int32_t* recv_ids, const float* recv_w, const void* w13,
                                  const void* w2, void* y, void* ws, size_t ws_bytes, void* stream);

/* moe_ep_combine (step 4): the rows returned to this rank (in its send
 * order) are added back by token, unweighted (the expert-holding rank applied
 * the weights), then scaled by rsf; the shared output is added:
 *   out[t] = rsf * sum_{k : send_pos[t*K+k] >= 0} ret[send_pos[t*K+k]]
 *            + shared_out[t]
 *   ret [T*K, H] act_dtype, send_pos [T*K] int32 (from moe_ep_dispatch),
 *   shared_out [T, H] nullable, out [T, H] act_dtype out.
 * ws: NULL, or >= 4 bytes for the status word. */
MOE_API int moe_ep_combine(const moe_config* cfg, int T, const void* ret, const int32_t* send_pos,
                           const void* shared_out, void* out, void* ws, size_t ws_bytes,
                           void* stream);

/* The kernel plan moe_forward follows for (cfg, T): which variant runs each
 * stage. No page counterpart; it describes this library's own kernels, for
 * instrumentation and tests. Host-only (no device work); returns the
 * validation status of (cfg, T). The plan assumes shared-expert weights are
 * passed when cfg->num_shared_experts > 0. */
typedef struct {
  int kernels;             /* kernels one moe_forward call launches           */
  int fused_route;         /* 1: logits, top-k and align in one kernel        */
  int router_tensor_cores; /* 1: router GEMM on tcgen05, 0: CUDA cores        */
  int router_partials;     /* partial logit slabs the top-k kernel sums       */
  int align_kernels;       /* 0 (fused route), 1 (one CTA), 2 (per-CTA counts,
                              then scan and scatter) or 3 (three passes)     */
  int tile_rows;           /* token rows per routed GEMM tile: 32, 128 or 256 */
  int gemm1_k_split;       /* 1, or K ranges of GEMM1 whose fp32 partials are
                              summed by a finalize kernel or, fused, in-kernel */
  int cta_pairs;           /* 1: routed GEMMs on CTA pairs (cta_group::2)     */
  int fused_mlp;           /* 1: GEMM1 and GEMM2 in one persistent kernel,
                              one CTA per SM of the current context; where
                              one CTA does not fit on an SM, the call runs
                              the two GEMM kernels instead                   */
  int gemm2_overlap;       /* 1: GEMM2 starts on the SMs GEMM1 has left and
                              takes each token tile once GEMM1 has published
                              its rows (single-CTA GEMMs, one K range)       */
  int combine_ring;        /* 1: the combine streams each token's rows through
                              a shared-memory ring (from 1024 tokens whose
                              expected routed and shared rows bring >= 48 KB) */
} moe_plan;
MOE_API int moe_forward_plan(const moe_config* cfg, int T, moe_plan* out);

/* Sets the time limit of the library's pipeline waits on the current device,
 * in ns of the GPU's global timer; 0 restores the default of 1 s. No page
 * counterpart: it exists so that a test can make a bounded device wait run
 * out. Every wait on a barrier or a cross-CTA counter inside the kernels gives
 * up after this limit; the kernel then sets MOE_DEV_TIMEOUT, lets its own
 * copies and MMAs land (those waits keep 1 s), frees its tensor memory and
 * exits, and moe_get_status returns MOE_ERR_TIMEOUT. Outputs of such a call
 * are unusable. The setting applies to every kernel launched after this call
 * returns (it synchronises with the device) until it is set again; a process
 * with several host threads must not change it while others launch. Returns
 * MOE_ERR_CUDA if a copy to the device fails. */
MOE_API int moe_set_wait_limit_ns(uint64_t ns);

/* The failure behind the calling host thread's latest MOE_ERR_CUDA: the
 * cudaError_t of the CUDA call that failed, or 10000 + the CUresult of a TMA
 * tensor-map encoding that failed; 0 if no call of this thread has failed.
 * Not cleared by later successful calls. No CUDA call. */
MOE_API int moe_last_cuda_error(void);

/* ------------------------------------------------------------------------ */
/* Synchronises `stream` and reads the device status word at the start of
 * `ws`. Writes the raw MOE_DEV_* bits to *flags (nullable). Returns MOE_OK if
 * no flag is set, MOE_ERR_TIMEOUT if MOE_DEV_TIMEOUT is set, else
 * MOE_ERR_DEVICE_STATUS. MOE_ERR_CUDA if the synchronisation fails. */
MOE_API int moe_get_status(const void* ws, void* stream, uint32_t* flags);

/* ------------------------------------------------------------------------ */
/* Debug build. No page counterpart: it stands in for a memory checker.
 * libmoe_debug.so is this library compiled with MOE_DEBUG. Its kernels also
 * check the indices they derive themselves and trust in libmoe.so: tile-table
 * entries (index, expert, first row, row count) against the tile table and
 * the permuted buffers, output rows and columns against the output, weight
 * rows against the weight tensor, the sorted positions read by the gather
 * and the combine, the token rows GEMM1's row warps copy from x, and the
 * top-k ids against E. A failed check skips the
 * access or clamps the value into range (the outputs are then unusable) and
 * is counted in a device record, which also keeps the site, index and bound
 * of the first failure. Same entry points and results otherwise; slower. */
typedef struct {
  uint32_t count; /* failed check evaluations since the last take (one bad
                     value may be checked, and counted, several times)      */
  uint32_t site;  /* first failure: file code * 65536 + source line; file
                     codes 1 moe_api.cu, 2 kernels_gemm.cu,
                     3 kernels_gemm_pair.cu, 4 kernels_mlp_fused.cu,
                     5 kernels_route.cu (and topk_warp.cuh there),
                     6 kernels_align.cu                                     */
  int64_t index;  /* first failure: the index checked                       */
  int64_t bound;  /* first failure: the bound; 0 <= index < bound failed    */
} moe_debug_record;

/* 1 in libmoe_debug.so, 0 in libmoe.so. No CUDA call. */
MOE_API int moe_debug_build(void);

/* Synchronises the current device, then reads and clears the records of
 * the device code's translation units: *rec gets the sum of their counts
 * and the first failure of the first unit with one, in file-code order.
 * MOE_ERR_UNSUPPORTED (and *rec zeroed, no CUDA call) in libmoe.so;
 * MOE_ERR_INVALID_ARG if rec is NULL; MOE_ERR_CUDA if a copy fails. */
MOE_API int moe_debug_take(moe_debug_record* rec);

/* libmoe_debug.so: enqueues one kernel on `stream` that fails one check
 * (index 5 against bound 4) and touches no memory, so that a test can see a
 * record arrive. MOE_ERR_UNSUPPORTED in libmoe.so. */
MOE_API int moe_debug_selftest(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
