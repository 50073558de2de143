// Bounds checks of the debug build.
//
// The release kernels check what a caller hands them (expert ids, segment
// offsets, the capacity of the permuted buffers) and flag it in the device
// status word. Indices they derive themselves from those checked values (a
// tile-table entry, a unit's weight rows, an output row, a TMA coordinate)
// they trust. Compiled with -DMOE_DEBUG (libmoe_debug.so), MOE_DCHECK(i, n)
// tests 0 <= i < n for such a derived index:
//   - a failed check adds 1 to a device record of its translation unit and,
//     if it is the first since the record was last taken, stores its site
//     (file code * 65536 + source line), index and bound;
//   - it evaluates to false, so the caller skips the access or clamps the
//     value into range (tile-table entries are clamped, so that every warp
//     role of a kernel still walks the same pipeline).
// In the release build MOE_DCHECK is the constant true and its arguments are
// not evaluated: they must have no side effects. TMA coordinates are checked
// for the logic only; the copy engine itself fills boxes outside the tensor.
#pragma once

#include <cuda_runtime.h>

namespace moe {

struct DbgRecord {
  unsigned count;   // failed check evaluations (one bad value may fail several)
  unsigned site;    // first failure: file code * 65536 + line
  long long index;  // first failure: the index
  long long bound;  // first failure: the bound (0 <= index < bound failed)
};

// File codes of the sites.
enum DbgFile : unsigned {
  kDbgApi = 1,
  kDbgGemm = 2,
  kDbgGemmPair = 3,
  kDbgMlpFused = 4,
  kDbgRoute = 5,
  kDbgAlign = 6,
};

}  // namespace moe

#ifdef MOE_DEBUG

namespace moe {
namespace dbg {

// One record per translation unit (internal linkage), read and cleared by the
// unit's MOE_DEBUG_TAKER function.
static __device__ DbgRecord g_record;

static __device__ __noinline__ void fail(unsigned site, long long i, long long n) {
  if (atomicAdd(&g_record.count, 1u) == 0u) {
    g_record.site = site;
    g_record.index = i;
    g_record.bound = n;
  }
}

static __device__ __forceinline__ bool in_range(unsigned site, long long i, long long n) {
  if (i >= 0 && i < n) return true;
  fail(site, i, n);
  return false;
}

}  // namespace dbg
}  // namespace moe

#define MOE_DEBUG_BUILD 1
#define MOE_DCHECK(i, n)                                                             \
  (::moe::dbg::in_range(static_cast<unsigned>(kDbgFileCode) * 65536u + __LINE__, \
                        static_cast<long long>(i), static_cast<long long>(n)))
#define MOE_DEBUG_TAKER(fn)                                                     \
  cudaError_t fn(DbgRecord* out) {                                              \
    cudaError_t e = cudaMemcpyFromSymbol(out, ::moe::dbg::g_record, sizeof(*out)); \
    if (e != cudaSuccess) return e;                                             \
    const DbgRecord zero = {};                                                  \
    return cudaMemcpyToSymbol(::moe::dbg::g_record, &zero, sizeof(zero));       \
  }

#else

#define MOE_DEBUG_BUILD 0
#define MOE_DCHECK(i, n) true
#define MOE_DEBUG_TAKER(fn)         \
  cudaError_t fn(DbgRecord* out) {  \
    *out = DbgRecord{};             \
    return cudaSuccess;             \
  }

#endif
