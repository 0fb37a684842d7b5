// Kernel launch with programmatic dependent launch (PDL).
//
// Every kernel of the library starts with griddep_wait() before it touches
// global memory, which blocks until the preceding kernel in the stream has
// completed and its writes are visible; so letting the next kernel launch
// early (PDL) only overlaps its launch and prologue with the predecessor's
// tail, and never changes a result.  Kernels call griddep_launch() once their
// remaining work no longer needs the SM resources a waiting successor would
// take.
#pragma once
#include <cuda_runtime.h>

#include <atomic>
#include <utility>

namespace gp {

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Whether launches made by this thread may overlap their predecessor (set by
// the step executor; default on).
bool pdl_enabled();
void set_pdl_enabled(bool on);

// heavy = true: the kernel holds most of an SM's shared memory / tensor
// memory; it is never launched early, so a waiting copy cannot keep those from
// kernels of other streams.
// Every launch carries its stream's priority as a launch attribute, so that a
// kernel captured into a graph (instantiated with node priorities) keeps the
// priority of the stream it was issued to: the step's critical-path streams
// get SMs before its weight-gradient streams.
inline void set_priority_attr(cudaLaunchAttribute& a, cudaStream_t s) {
  int prio = 0;
  if (cudaStreamGetPriority(s, &prio) != cudaSuccess) prio = 0;
  a.id = cudaLaunchAttributePriority;
  a.val.priority = prio;
}

template <bool heavy = false, typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = (!heavy && pdl_enabled()) ? 1 : 0;
  set_priority_attr(attr[1], s);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Run f (a per-device setup such as a kernel attribute, which CUDA keeps per
// device) once for each device it succeeds on; devices >= 64 run it every time.
template <typename F>
int once_per_device(std::atomic<unsigned long long>& done, F&& f) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return f();
  const unsigned long long bit = 1ull << dev;
  if (done.load(std::memory_order_acquire) & bit) return 0;
  const int rc = f();
  if (rc == 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return rc;
}

}  // namespace gp
