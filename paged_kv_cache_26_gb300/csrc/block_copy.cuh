// Copy-on-write of shared blocks (sm_103a).
//
// kasblo.com "vLLMとは？LLMサーバーを高速化する仕組み", section "block共有とAutomatic
// Prefix Caching": a physical block carries a reference count, several
// sequences may hold it, and it is duplicated only when one of them must write
// into it (parallel sampling, a shared prefix that ends inside a block).  The
// host allocator decides the copies; this kernel performs them: for each
// (src, dst) pair, block dst of the K pool and of the V pool becomes a copy of
// block src (all KV heads and slots), before the step that writes into dst.
//
// A pure HBM copy.  Consecutive threads take consecutive 16-byte chunks of a
// block (coalesced), grid-stride; each thread loads kCopyUnroll chunks of K
// and of V before it stores any, so that 2 * kCopyUnroll loads are in flight
// per thread (one chunk at a time left the copy waiting on DRAM latency).
#pragma once

#include "pkv_device.cuh"

namespace pkv {

constexpr int kCopyUnroll = 4;

__global__ void copy_blocks_kernel(const int32_t* __restrict__ pairs, int32_t num_pairs, int64_t chunks_per_block,
                                   int32_t num_blocks, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache) {
  const int64_t total = chunks_per_block * num_pairs;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; base < total;
       base += stride * kCopyUnroll) {
    uint4 kv[kCopyUnroll], vv[kCopyUnroll];
    int64_t dst_off[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      dst_off[u] = -1;
      const int64_t idx = base + u * stride;
      if (idx >= total) continue;
      const int64_t p = idx / chunks_per_block;
      const int64_t c = idx - p * chunks_per_block;
      const int32_t src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
      if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (c == 0) flag_error(kErrBlockId);
        continue;
      }
      kv[u] = k_cache[src * chunks_per_block + c];
      vv[u] = v_cache[src * chunks_per_block + c];
      dst_off[u] = dst * chunks_per_block + c;
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      if (dst_off[u] < 0) continue;
      k_cache[dst_off[u]] = kv[u];
      v_cache[dst_off[u]] = vv[u];
    }
  }
}

// Self-test of the bounded waits: one warp waits on an mbarrier that nothing
// ever arrives on.  The wait gives up after kWaitLimitNs, flags kErrTimeout
// and the kernel returns; the context stays usable.
__global__ void wait_selftest_kernel() {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0);
}

}  // namespace pkv
