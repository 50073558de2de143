// Programmatic dependent launch (PDL) for every kernel of the library.
//
// Kernels are launched with programmatic stream serialisation, so the next
// kernel of the layer can be scheduled while the current one finishes. Each
// kernel's first statement is pdl_enter(): it waits until the preceding grid
// has completed and its memory is visible, then allows the following grid to
// launch. Consumers never read a producer's output before that wait.
//
// Since every kernel allows its dependents only after its own wait, a kernel
// that has launched may assume that the kernel two places before it has
// completed. The GEMM kernels use this: their tile tables (written at least
// two kernels earlier) and their weight operands (never written by the
// library) are read before the wait, so the first weight tiles stream in
// while the preceding kernel finishes.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <utility>

namespace moe {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_launch_dependents();
}

// The same pointer, with a value the compiler cannot know before this point.
// Kernel pointer parameters are restrict-qualified, so the compiler may assume
// that an asm statement (the dependency wait, an acquire atomic) does not
// write through them and move their loads above it. A kernel reads data that
// the preceding kernel, or another CTA, has just written through pointers
// passed through this after the wait. The unknown value is a zero offset
// rather than the pointer itself: passing the pointer through the asm made
// the compiler keep small per-thread arrays of the same kernel in local
// memory.
template <typename T>
__device__ __forceinline__ T* fresh(T* p) {
  long off = 0;
  asm volatile("" : "+l"(off));
  return p + off;
}

// Kernels this host thread has launched (successfully) through the library;
// moe_forward_timed reports the difference across one call.
inline thread_local long g_kernel_launches = 0;

inline cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) ++g_kernel_launches;
  return e;
}

// Allow a kernel more than 48 KB of dynamic shared memory on the current
// device. Function attributes belong to each device's context, so `done` (one
// per kernel) records the device ordinals already set, one bit each; an
// ordinal past 63 is set on every call. Two host threads that race here both
// set the attribute, which is harmless.
inline cudaError_t opt_in_smem(const void* kern, int bytes,
                               std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return counted(cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...));
}

}  // namespace moe
