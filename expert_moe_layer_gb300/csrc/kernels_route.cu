// Routing: router logits, fp32 softmax, plain or group-limited top-k,
// renormalise (MixtralMoE.forward; FusedMoE select_experts arguments).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "internal.h"

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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  const int t0 = blockIdx.y * kTok;
  if (e >= E) return;
  float acc[kTok];
#pragma unroll
  for (int j = 0; j < kTok; ++j) acc[j] = 0.f;
  const TW* wrow = wg + static_cast<long>(e) * H;
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

// Token-major variant for small E (<= 32): warp = one token, all experts in
// chunks of 8. The token's row is read once per chunk (once for E <= 8); the
// router rows stay in L1/L2.
template <typename TX, typename TW>
__global__ void __launch_bounds__(256) router_logits_token_kernel(const TX* __restrict__ x,
                                                                  const TW* __restrict__ wg,
                                                                  float* __restrict__ logits,
                                                                  int T, int E, int H) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long t = blockIdx.x * 8L + warp;
  if (t >= T) return;
  const TX* xrow = x + t * H;
  for (int e0 = 0; e0 < E; e0 += 8) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (int h = lane * 8; h < H; h += 256) {
      float xv[8];
      load8(xrow + h, xv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (e0 + j < E) {
          float w[8];
          load8(wg + static_cast<long>(e0 + j) * H + h, w);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[j] = fmaf(xv[i], w[i], acc[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float v = acc[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[j] = v;
    }
    if (lane < 8 && e0 + lane < E) {
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j == lane) v = acc[j];
      logits[t * E + e0 + lane] = v;
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

template <int VPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits,
                                                   const float* __restrict__ bias, int T,
                                                   int E, int K, int renorm, int n_group,
                                                   int topk_group, int32_t* __restrict__ ids,
                                                   float* __restrict__ wout) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float* row = logits + static_cast<long>(t) * E;

  float p[VPL];
  float mx = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    p[j] = -CUDART_INF_F;
    if (e < E) {
      p[j] = row[e] + (bias ? bias[e] : 0.f);
      mx = fmaxf(mx, p[j]);
    }
  }
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
    if (((i & 31) != lane)) pw = 0.f;
    pw = __shfl_sync(0xffffffffu, pw, i & 31);
    wsum += pw;
    if (lane == k) {
      my_w = pw;
      my_id = i;
    }
  }
  if (lane < K) {
    ids[static_cast<long>(t) * K + lane] = my_id;
    wout[static_cast<long>(t) * K + lane] = renorm ? my_w / wsum : my_w;
  }
}

}  // namespace

cudaError_t launch_router_logits(bool act_bf16, bool router_bf16, const void* x,
                                 const void* wg, float* logits, int T, int E, int H,
                                 cudaStream_t st) {
  if (E <= 32) {
    const int grid = (T + 7) / 8;
    if (act_bf16 && router_bf16)
      router_logits_token_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                                        static_cast<const __nv_bfloat16*>(wg),
                                                        logits, T, E, H);
    else if (act_bf16)
      router_logits_token_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                                        static_cast<const float*>(wg), logits,
                                                        T, E, H);
    else
      router_logits_token_kernel<<<grid, 256, 0, st>>>(static_cast<const float*>(x),
                                                        static_cast<const float*>(wg), logits,
                                                        T, E, H);
    return cudaGetLastError();
  }
  dim3 grid((E + 7) / 8, (T + kTok - 1) / kTok);
  if (act_bf16 && router_bf16)
    router_logits_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                                static_cast<const __nv_bfloat16*>(wg), logits,
                                                T, E, H);
  else if (act_bf16)
    router_logits_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                                static_cast<const float*>(wg), logits, T, E,
                                                H);
  else
    router_logits_kernel<<<grid, 256, 0, st>>>(static_cast<const float*>(x),
                                                static_cast<const float*>(wg), logits, T, E,
                                                H);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int K,
                        int renorm, int n_group, int topk_group, int32_t* ids, float* w,
                        unsigned* /*status*/, cudaStream_t st) {
  const int grid = (T + 7) / 8;
  const int vpl = (E + 31) / 32;
#define MOE_TOPK(V) \
  topk_kernel<V><<<grid, 256, 0, st>>>(logits, bias, T, E, K, renorm, n_group, topk_group, ids, w)
  if (vpl <= 1) MOE_TOPK(1);
  else if (vpl <= 2) MOE_TOPK(2);
  else if (vpl <= 4) MOE_TOPK(4);
  else if (vpl <= 8) MOE_TOPK(8);
  else if (vpl <= 16) MOE_TOPK(16);
  else return cudaErrorInvalidValue;
#undef MOE_TOPK
  return cudaGetLastError();
}

}  // namespace moe
