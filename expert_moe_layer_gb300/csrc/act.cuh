// The activation of the expert MLP (MixtralMoE expert forward:
// w2(silu(w1 x) * w3 x); MoEMixin activation "silu").
#pragma once

#include <cuda_runtime.h>

namespace moe {

// silu(g) = g / (1 + e^-g) with the fast single-precision quotient. The IEEE
// quotient takes a checked path per value, which serialises an epilogue's
// chain of dependent values; the fast one differs from it by a few ulp. For g
// below about -87, where 1 + e^-g passes 2^126, it returns zero, the limit.
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

}  // namespace moe
