// Host <-> device copies by a kernel (sm_103a).
//
// A decode step that starts from host buffers moves its inputs to the device
// and its output back.  Done by the copy engines (stream-ordered DMA copies),
// each copy sits between two kernels of the stream, so the kernel after it
// can no longer be launched while the one before it finishes: it starts cold,
// and a step pays for the copy's own latency on top.  Here the copies are
// kernels in the same chain of programmatic launches as the decode and merge
// kernels: the threads read mapped pinned host memory (or device memory) and
// write device memory (or mapped pinned host memory) directly.
//
// A host-to-device copy reads its source before griddepcontrol.wait (host
// inputs are complete when the call is made, and no kernel writes them), so
// the reads over the host link overlap the end of the previous kernel; the
// stores into the device staging come after the wait, once the kernels that
// read the previous step's staging have finished.  A device-to-host copy
// reads only after the wait (its source is the previous kernel's output).
//
// The work is a list of runs, each cut into units of 16 bytes (source,
// destination and length 16-byte aligned) or else 4 bytes; consecutive
// threads take consecutive units (coalesced on both sides).
#pragma once

#include <cstdint>

namespace pkv {

constexpr int kMaxCopyRuns = 6;
constexpr int kCopyThreads = 256;
constexpr int kCopyUnitsPerThread = 4;  // units held in registers across the wait

struct CopyRun {
  const uint8_t* src;
  uint8_t* dst;
  int64_t first;  // index of the run's first unit in the whole list
  int32_t shift;  // log2 of the unit size: 4 (16 bytes) or 2 (4 bytes)
};

struct CopyList {
  CopyRun run[kMaxCopyRuns];
  int64_t total;  // units over all runs
  int32_t n;
};

__device__ __forceinline__ int copy_run_of(const CopyList& l, int64_t u) {
  int r = 0;
#pragma unroll
  for (int i = 1; i < kMaxCopyRuns; ++i)
    if (i < l.n && u >= l.run[i].first) r = i;
  return r;
}

__device__ __forceinline__ uint4 copy_load(const CopyList& l, int64_t u) {
  const CopyRun& c = l.run[copy_run_of(l, u)];
  const int64_t off = (u - c.first) << c.shift;
  if (c.shift == 4) return *reinterpret_cast<const uint4*>(c.src + off);
  return make_uint4(*reinterpret_cast<const uint32_t*>(c.src + off), 0u, 0u, 0u);
}

__device__ __forceinline__ void copy_store(const CopyList& l, int64_t u, const uint4& v) {
  const CopyRun& c = l.run[copy_run_of(l, u)];
  const int64_t off = (u - c.first) << c.shift;
  if (c.shift == 4)
    *reinterpret_cast<uint4*>(c.dst + off) = v;
  else
    *reinterpret_cast<uint32_t*>(c.dst + off) = v.x;
}

// kSrcBeforeWait: the sources are host inputs that no earlier kernel writes.
template <bool kSrcBeforeWait>
__global__ void __launch_bounds__(kCopyThreads) stage_copy_kernel(const __grid_constant__ CopyList l) {
  // The next kernel may launch now; it waits for this grid to complete
  // before it reads what this grid writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kCopyThreads;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * kCopyThreads + threadIdx.x;
  uint4 r[kCopyUnitsPerThread];
  if (kSrcBeforeWait) {
#pragma unroll
    for (int k = 0; k < kCopyUnitsPerThread; ++k)
      if (u0 + k * stride < l.total) r[k] = copy_load(l, u0 + k * stride);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!kSrcBeforeWait) {
#pragma unroll
    for (int k = 0; k < kCopyUnitsPerThread; ++k)
      if (u0 + k * stride < l.total) r[k] = copy_load(l, u0 + k * stride);
  }
#pragma unroll
  for (int k = 0; k < kCopyUnitsPerThread; ++k)
    if (u0 + k * stride < l.total) copy_store(l, u0 + k * stride, r[k]);
  // Lists longer than the grid holds in registers: the rest, unit by unit.
  for (int64_t u = u0 + kCopyUnitsPerThread * stride; u < l.total; u += stride) copy_store(l, u, copy_load(l, u));
}

}  // namespace pkv
