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
// A pure HBM copy: every thread moves one 16-byte chunk of K and one of V,
// consecutive threads consecutive chunks of a block (coalesced), grid-stride.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

__global__ void copy_blocks_kernel(const int32_t* __restrict__ pairs, int32_t num_pairs, int64_t chunks_per_block,
                                   int32_t num_blocks, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache) {
  const int64_t total = chunks_per_block * num_pairs;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = idx / chunks_per_block;
    const int64_t c = idx - p * chunks_per_block;
    const int32_t src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (c == 0) flag_error(kErrBlockId);
      continue;
    }
    const uint4 kv = k_cache[src * chunks_per_block + c];
    const uint4 vv = v_cache[src * chunks_per_block + c];
    k_cache[dst * chunks_per_block + c] = kv;
    v_cache[dst * chunks_per_block + c] = vv;
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
