// Routing: router logits, fp32 softmax, plain or group-limited top-k,
// renormalise (MixtralMoE.forward; FusedMoE select_experts arguments).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "internal.h"
#include "launch.cuh"

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

// Split-H variant for small E (<= 32). A CTA covers 64 tokens (8 per warp),
// one kRouterSplitCols-wide slice of H and up to 8 experts (blockIdx.z picks
// the expert octet). Each lane keeps its 8 columns of those experts' router
// rows in registers, so the router weights are read once per warp and every
// token row once per octet. The slice sums go to partial slab blockIdx.y; the
// top-k kernel adds the slabs in slab order.
constexpr int kSplitTokWarp = 8;

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
__global__ void __launch_bounds__(256) router_logits_split_kernel(const TX* __restrict__ x,
                                                                  const TW* __restrict__ wg,
                                                                  float* __restrict__ logits,
                                                                  int T, int E, int H) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kRouterSplitCols + lane * 8;
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
  float* slab = logits + static_cast<long>(blockIdx.y) * T * E;
  const long tw = (static_cast<long>(blockIdx.x) * 8 + warp) * kSplitTokWarp;
  const int ex = (lane >> 2) & 7;
#pragma unroll
  for (int a = 0; a < kSplitTokWarp; a += 4) {
    float xv[4][8];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      if (hv && tw + a + b < T) {
        load8(x + (tw + a + b) * H + h, xv[b]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xv[b][i] = 0.f;
      }
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) d = fmaf(xv[b][i], w[j][i], d);
        acc[j] = d;
      }
      const float v = warp_sum8(acc, lane);
      const long t = tw + a + b;
      if ((lane & 3) == 0 && t < T && e0 + ex < E) slab[t * E + e0 + ex] = v;
    }
  }
}

// --------------------------------------------------------------- top-k
// One warp per token. Lane l holds experts e = l + 32*j (j < VPL).
// Ordering: larger value first, equal values -> lower index first.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// The warp-level routing decision for one token. p[j] holds the logit (with
// bias) of expert lane + 32*j, or -inf beyond E. Softmax, the optional group
// limit, K rounds of argmax and the renormalisation all run on this warp.
template <int VPL>
__device__ __forceinline__ void topk_warp(float (&p)[VPL], int lane, int E, int K, int renorm,
                                          int n_group, int topk_group,
                                          int32_t* __restrict__ ids_row,
                                          float* __restrict__ w_row) {
  float mx = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < VPL; ++j) mx = fmaxf(mx, p[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    p[j] = (e < E) ? expf(p[j] - mx) : 0.f;
    sum += p[j];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
#pragma unroll
  for (int j = 0; j < VPL; ++j) p[j] = (lane + 32 * j < E) ? p[j] / sum : -CUDART_INF_F;

  // candidate values: p, or -inf outside the kept groups
  float c[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) c[j] = p[j];
  if (n_group > 0) {
    const int gs = E / n_group;
    float my_score = -CUDART_INF_F;  // lane g holds the score of group g
    for (int g = 0; g < n_group; ++g) {
      float m = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int e = lane + 32 * j;
        if (e < E && e / gs == g) m = fmaxf(m, p[j]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == g) my_score = m;
    }
    bool taken = false;
    for (int r = 0; r < topk_group; ++r) {
      float v = (lane < n_group && !taken) ? my_score : -CUDART_INF_F;
      int i = (lane < n_group && !taken) ? lane : 0x7fffffff;
      warp_argmax(v, i);
      if (lane == i) taken = true;
    }
    const unsigned keep = __ballot_sync(0xffffffffu, taken);
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      if (e < E && !((keep >> (e / gs)) & 1u)) c[j] = -CUDART_INF_F;
    }
  }

  float my_w = 0.f;
  int my_id = 0;
  float wsum = 0.f;
  for (int k = 0; k < K; ++k) {
    float v = -CUDART_INF_F;
    int i = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      if (e < E && better(c[j], e, v, i)) {
        v = c[j];
        i = e;
      }
    }
    warp_argmax(v, i);
    // owner lane marks the winner as taken and publishes its probability
    float pw = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      if (lane + 32 * j == i) {
        pw = p[j];
        c[j] = -CUDART_INF_F;
      }
    }
    pw = __shfl_sync(0xffffffffu, pw, i & 31);
    wsum += pw;
    if (lane == k) {
      my_w = pw;
      my_id = i;
    }
  }
  if (lane < K) {
    ids_row[lane] = my_id;
    w_row[lane] = renorm ? my_w / wsum : my_w;
  }
}

// One warp per token (large batches): logits = sum of n_part partial slabs.
template <int VPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits,
                                                   int n_part, long partial_stride,
                                                   const float* __restrict__ bias, int T,
                                                   int E, int K, int renorm, int n_group,
                                                   int topk_group, int32_t* __restrict__ ids,
                                                   float* __restrict__ wout) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float* row = logits + static_cast<long>(t) * E;
  float p[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    p[j] = -CUDART_INF_F;
    if (e < E) {
      float l = row[e];
#pragma unroll 8
      for (int s = 1; s < n_part; ++s) l += row[s * partial_stride + e];
      p[j] = l + (bias ? bias[e] : 0.f);
    }
  }
  topk_warp<VPL>(p, lane, E, K, renorm, n_group, topk_group, ids + static_cast<long>(t) * K,
                 wout + static_cast<long>(t) * K);
}

// One CTA per token (small batches): all threads sum the partial slabs into
// shared memory in parallel, then warp 0 takes the decision.
template <int VPL>
__global__ void __launch_bounds__(256) topk_cta_kernel(const float* __restrict__ logits,
                                                       int n_part, long partial_stride,
                                                       const float* __restrict__ bias, int T,
                                                       int E, int K, int renorm, int n_group,
                                                       int topk_group,
                                                       int32_t* __restrict__ ids,
                                                       float* __restrict__ wout) {
  pdl_enter();
  __shared__ float sl[32 * VPL];
  const long t = blockIdx.x;
  const float* row = logits + t * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float l = row[e];
#pragma unroll 8
    for (int s = 1; s < n_part; ++s) l += row[s * partial_stride + e];
    sl[e] = l + (bias ? bias[e] : 0.f);
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  float p[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    p[j] = e < E ? sl[e] : -CUDART_INF_F;
  }
  topk_warp<VPL>(p, lane, E, K, renorm, n_group, topk_group, ids + t * K, wout + t * K);
}

}  // namespace

template <typename TX, typename TW>
cudaError_t logits_launch(const void* x, const void* wg, float* logits, int T, int E, int H,
                          cudaStream_t st) {
  const TX* xp = static_cast<const TX*>(x);
  const TW* wp = static_cast<const TW*>(wg);
  if (E <= 32)
    return launch_pdl(router_logits_split_kernel<TX, TW>,
                      dim3((T + 8 * kSplitTokWarp - 1) / (8 * kSplitTokWarp),
                           router_split_slabs(H), (E + 7) / 8),
                      dim3(256), 0, st, xp, wp, logits, T, E, H);
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
                        int T, int E, int K, int renorm, int n_group, int topk_group,
                        int32_t* ids, float* w, cudaStream_t st) {
  if (T < 256)
    return launch_pdl(topk_cta_kernel<V>, dim3(T), dim3(256), 0, st, logits, n_part,
                      partial_stride, bias, T, E, K, renorm, n_group, topk_group, ids, w);
  return launch_pdl(topk_kernel<V>, dim3((T + 7) / 8), dim3(256), 0, st, logits, n_part,
                    partial_stride, bias, T, E, K, renorm, n_group, topk_group, ids, w);
}

cudaError_t launch_topk(const float* logits, int n_part, long partial_stride,
                        const float* bias, int T, int E, int K, int renorm, int n_group,
                        int topk_group, int32_t* ids, float* w, unsigned* /*status*/,
                        cudaStream_t st) {
  const int vpl = (E + 31) / 32;
  if (vpl <= 1) return topk_launch<1>(logits, n_part, partial_stride, bias, T, E, K, renorm,
                                      n_group, topk_group, ids, w, st);
  if (vpl <= 2) return topk_launch<2>(logits, n_part, partial_stride, bias, T, E, K, renorm,
                                      n_group, topk_group, ids, w, st);
  if (vpl <= 4) return topk_launch<4>(logits, n_part, partial_stride, bias, T, E, K, renorm,
                                      n_group, topk_group, ids, w, st);
  if (vpl <= 8) return topk_launch<8>(logits, n_part, partial_stride, bias, T, E, K, renorm,
                                      n_group, topk_group, ids, w, st);
  if (vpl <= 16) return topk_launch<16>(logits, n_part, partial_stride, bias, T, E, K, renorm,
                                        n_group, topk_group, ids, w, st);
  return cudaErrorInvalidValue;
}

}  // namespace moe
