// The per-token routing decision on one warp: fp32 scores over the logits
// (softmax, or per-expert sigmoid), the optional selection-only score
// correction and group limit, top-k and renormalisation (MixtralMoE.forward;
// FusedMoE select_experts / grouped_topk / scoring_func /
// e_score_correction_bias arguments).
//
// Order: larger selection score first, equal scores -> lower expert id.
// Every argmax is two single-instruction warp reductions (redux.sync) on an
// order-preserving 32-bit key of the float: the largest key, then the lowest
// expert id among the lanes that hold it. Each lane first sorts its VPL
// candidates (expert lane + 32*j in slot j) with a bitonic network on 64-bit
// values key << 32 | (16 - j), so that equal keys keep the lower slot (the
// lower id) first and an emptied entry (0) sorts below every real one. A
// round then offers each lane's first entry, and the owner of the winner
// drops it (a shift of its list), instead of every lane scanning its
// remaining slots every round.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "dbg.cuh"  // the including unit declares moe::kDbgFileCode first

namespace moe {

// flags of the routing kernels
constexpr int kRouteSigmoid = 1;     // scores = sigmoid(logit) instead of softmax
constexpr int kRouteBiasSelect = 2;  // the per-expert bias corrects the selection only

// Unsigned key with key(a) > key(b) <=> a > b for non-NaN floats (-0 sorts
// just below +0; probabilities are never -0). NaN maps to 0, below every
// number, so it is never chosen over one.
__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t b = __float_as_uint(v);
  if (v != v) return 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Warp argmax of (key, id) with ties to the lower id; every lane gets both.
__device__ __forceinline__ void warp_argmax_key(uint32_t& key, int& id) {
  const uint32_t m = __reduce_max_sync(0xffffffffu, key);
  const uint32_t cand = key == m ? static_cast<uint32_t>(id) : 0x7fffffffu;
  id = static_cast<int>(__reduce_min_sync(0xffffffffu, cand));
  key = m;
}

// The warp-level routing decision for one token. p[j] holds the logit of
// expert lane + 32*j, or -inf beyond E; sb[j] its selection-only correction
// (0 without one). Scoring, the optional group limit, K selections and the
// renormalisation all run on this warp. Lane k < K writes ids_row[k] and
// w_row[k].
template <int VPL>
__device__ __forceinline__ void topk_warp(float (&p)[VPL], const float (&sb)[VPL], int lane,
                                          int E, int K, int renorm, int flags, int n_group,
                                          int topk_group, int32_t* __restrict__ ids_row,
                                          float* __restrict__ w_row) {
  // A division per score would serialise this warp: the IEEE quotient takes a
  // checked path per element, which costs some hundreds of cycles each on a
  // single warp's dependency chain. Softmax divides by one reciprocal of the
  // sum instead, the logistic uses the fast quotient; both agree with the
  // IEEE quotients to a few ulp, far inside the routing weights' tolerance
  // and below the score gaps the routing decisions see.
  if (flags & kRouteSigmoid) {
    // per-expert logistic in fp32
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      p[j] = (lane + 32 * j < E) ? __fdividef(1.0f, 1.0f + expf(-p[j])) : -CUDART_INF_F;
  } else {
    // softmax in fp32: max, exp, sum, divide
    float lmx = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < VPL; ++j) lmx = fmaxf(lmx, p[j]);
    const float mx = fkey_inv(__reduce_max_sync(0xffffffffu, fkey(lmx)));
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      p[j] = (e < E) ? expf(p[j] - mx) : 0.f;
      sum += p[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float inv = 1.0f / sum;
#pragma unroll
    for (int j = 0; j < VPL; ++j) p[j] = (lane + 32 * j < E) ? p[j] * inv : -CUDART_INF_F;
  }

  // candidate keys: p + correction, or -inf outside the kept groups (group
  // score = the largest corrected score in the group; topk_group groups by
  // score, ties to lower group)
  uint32_t ck[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) ck[j] = fkey(lane + 32 * j < E ? p[j] + sb[j] : -CUDART_INF_F);
  if (n_group > 0) {
    // each slot's group, from one integer quotient per slot (not one per
    // slot and group)
    const int gs = E / n_group;
    int gj[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      gj[j] = e < E ? e / gs : -1;
    }
    uint32_t my_score = 0;  // lane g holds the key of group g's score
    for (int g = 0; g < n_group; ++g) {
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (gj[j] == g) m = max(m, ck[j]);
      m = __reduce_max_sync(0xffffffffu, m);
      if (lane == g) my_score = m;
    }
    bool taken = false;
    for (int r = 0; r < topk_group; ++r) {
      uint32_t key = (lane < n_group && !taken) ? my_score : 0u;
      int id = (lane < n_group && !taken) ? lane : 0x7fffffff;
      warp_argmax_key(key, id);
      if (lane == id) taken = true;
    }
    const unsigned keep = __ballot_sync(0xffffffffu, taken);
    const uint32_t ninf = fkey(-CUDART_INF_F);
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (gj[j] >= 0 && !((keep >> gj[j]) & 1u)) ck[j] = ninf;
  }

  static_assert(VPL >= 1 && VPL <= 16 && (VPL & (VPL - 1)) == 0, "VPL: a power of two <= 16");
  // this lane's candidates, sorted: larger key first, then lower slot (slots
  // beyond E hold -inf keys with ids >= E: they never win while a real expert
  // remains; a NaN score has key 0)
  uint64_t v[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j)
    v[j] = (static_cast<uint64_t>(ck[j]) << 32) | static_cast<uint32_t>(16 - j);
#pragma unroll
  for (int kk = 2; kk <= VPL; kk <<= 1) {
#pragma unroll
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int l = i ^ jj;
        if (l > i) {
          const bool desc = (i & kk) == 0;
          const uint64_t a = v[i], b = v[l];
          const bool sw = desc ? (a < b) : (a > b);
          v[i] = sw ? b : a;
          v[l] = sw ? a : b;
        }
      }
    }
  }

  float my_w = 0.f;
  int my_id = 0;
  float wsum = 0.f;
  for (int k = 0; k < K; ++k) {
    // this lane's best remaining candidate, or id 0x7fffffff when none is left
    const uint32_t low = static_cast<uint32_t>(v[0]) & 31u;
    uint32_t key = low ? static_cast<uint32_t>(v[0] >> 32) : 0u;
    int id = low ? lane + 32 * (16 - static_cast<int>(low)) : 0x7fffffff;
    warp_argmax_key(key, id);
    // the winner's score: the key itself, or with a selection correction the
    // uncorrected score from the lane that holds it (picked by a bit mask,
    // not a select, so that p stays in registers and is not indexed in local
    // memory)
    const int ws = id >> 5;
    float pw = fkey_inv(key);
    if (flags & kRouteBiasSelect) {
      uint32_t mine = 0u;
#pragma unroll
      for (int j = 0; j < VPL; ++j) mine |= __float_as_uint(p[j]) & (0u - (ws == j));
      pw = __shfl_sync(0xffffffffu, __uint_as_float(mine), id & 31);
    }
    if (id != 0x7fffffff && lane == (id & 31)) {  // the owner drops its first entry
#pragma unroll
      for (int j = 0; j + 1 < VPL; ++j) v[j] = v[j + 1];
      v[VPL - 1] = 0;
    }
    wsum += pw;
    if (lane == k) {
      my_w = pw;
      my_id = id;
    }
  }
  if (lane < K) {
    (void)MOE_DCHECK(my_id, E);
    ids_row[lane] = my_id;
    w_row[lane] = renorm ? my_w / wsum : my_w;
  }
}

}  // namespace moe
