// Kernels of the paged decode path (sm_103a).
//
//  append_kernel            -- slot-mapped copy of each new token's K/V into the
//                              pool ("How to Scale Your Model, Part 7: Inference",
//                              section "Transformer 推論の基礎: Prefill と
//                              Generation": the new token's K/V projection is
//                              appended to the cache).
//  decode_persistent_kernel -- the automatic path.  One CTA per SM; the flattened
//                              (sequence, KV head, block) space is cut into equal
//                              contiguous ranges, one per warp, so every warp
//                              streams the same number of K/V blocks whatever the
//                              length mix.  A unit (sequence, KV head) cut across
//                              warps is merged by the last warp to finish it.
//  decode_split_kernel      -- explicit sequence partitioning: one CTA per
//                              (split, KV head, sequence), followed by
//  merge_split_kernel       -- the log-sum-exp merge of the split partials.
//
// Both decode kernels walk the block table (kasblo.com "vLLMとは？", section
// "PagedAttentionはKV Cacheをblockで管理する": the attention kernel reads the K/V
// it needs through the table), stream each 16-token K/V block once through a TMA
// ring in shared memory, and serve the whole GQA query group from that one read
// with an fp32 online softmax (design.babushkai.com "GPU推論の内部構造", section
// "カーネル: FlashAttentionとメモリ階層": tiled attention with a running softmax, so
// the score matrix never reaches HBM).
//
// Cache layout: T[num_blocks][Hkv][16][D].  The (block, KV head) tile of 16
// tokens x D is contiguous; the TMA tensor map views the pool as a 2-D array of
// rows = num_blocks * Hkv * 16 and D columns and loads a tile as D/64 boxes of
// 16 rows x 64 elements (128 bytes) with the 128-byte swizzle, which makes the
// fragment loads below free of shared-memory bank conflicts.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

constexpr int kBlockSize = 16;
constexpr int kMaxGroup = 8;  // query heads per KV head served by one mma tile

// ===================================================================== append

// One thread copies one 16-byte chunk of one token's K row and the same chunk
// of its V row for one KV head.  C = chunks per row = D * sizeof(T) / 16.
__global__ void append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                              const int32_t* __restrict__ slots, int32_t num_tokens, int32_t num_kv_heads,
                              int32_t chunks_per_row, int64_t num_slots, uint4* __restrict__ k_cache,
                              uint4* __restrict__ v_cache) {
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * chunks_per_row;
  const int64_t total = per_token * num_tokens;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t token = idx / per_token;
    const int64_t within = idx - token * per_token;  // head * C + chunk
    const int32_t slot = slots[token];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      flag_error(kErrSlot);
      continue;
    }
    const int64_t blk = slot / kBlockSize;
    const int64_t off = slot % kBlockSize;
    const int64_t head = within / chunks_per_row;
    const int64_t chunk = within - head * chunks_per_row;
    const int64_t dst = ((blk * num_kv_heads + head) * kBlockSize + off) * chunks_per_row + chunk;
    k_cache[dst] = k_new[idx];
    v_cache[dst] = v_new[idx];
  }
}

// ===================================================================== warp math

template <int D>
struct TileShape {
  static constexpr int kBoxes = D / 64;                  // 64-element TMA boxes per row
  static constexpr int kTileBytes = kBlockSize * D * 2;  // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;     // K + V of one block
  static constexpr int kQChunks = D / 32;                // 16-byte chunks of q per lane
  static constexpr int kMTiles = D / 16;                 // m-tiles of O^T
};

// One warp's attention state for one (sequence, KV head) unit.
//
// Per 16-token block:  S^T = K Q^T  (mma rows = the 16 tokens, mma columns =
// the <= 8 query heads of the group, k = head_dim), online softmax per head,
// then O^T += V^T P^T  (mma rows = head_dim, columns = heads, k = tokens).
// Lane (gid = lane/4, c = lane%4):
//  * owns the 16-byte chunks {2c, 2c+1} (+{2c+8, 2c+9} when D = 128) of q row
//    gid and of K rows gid, gid+8; k-step j uses half j%2 of chunk j/2 (the
//    order of the head_dim sum is permuted the same way for q and K);
//  * holds scores for tokens gid, gid+8 and heads 2c, 2c+1;
//  * holds O^T for heads 2c, 2c+1 and head_dim entries in chunks gid (and
//    gid+8 when D = 128), reading V rows 2c, 2c+1, 2c+8, 2c+9.
template <typename T, int D>
struct WarpAttn {
  using Shape = TileShape<D>;
  uint4 qf[Shape::kQChunks];
  float acc[Shape::kMTiles][4];
  float m0, m1, l0, l1;  // running max (log2 units) and sum for heads 2c, 2c+1

  __device__ __forceinline__ void reset() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int i = 0; i < Shape::kMTiles; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  }

  // q rows of the group's heads start at q_group (row h at q_group + h * D).
  __device__ __forceinline__ void load_q(const T* q_group, int group, int lane) {
    const int gid = lane >> 2, c = lane & 3;
#pragma unroll
    for (int qc = 0; qc < Shape::kQChunks; ++qc) {
      const int chunk = 2 * c + (qc & 1) + 8 * (qc >> 1);
      qf[qc] = gid < group ? __ldg(reinterpret_cast<const uint4*>(q_group + gid * D) + chunk) : make_uint4(0, 0, 0, 0);
    }
  }

  // Accumulate one block whose K and V tiles sit (swizzled) at ks / vs; the
  // first `valid` of its 16 tokens belong to the context.
  __device__ __forceinline__ void block(const uint8_t* ks, const uint8_t* vs, int valid, float scale_log2,
                                        int lane) {
    const int gid = lane >> 2, c = lane & 3;
    float s[4] = {0.f, 0.f, 0.f, 0.f}, t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int qc = 0; qc < Shape::kQChunks; ++qc) {
      const int off = (qc >> 1) * 2048 + (((2 * c + (qc & 1)) ^ gid) << 4);
      const uint4 k0 = *reinterpret_cast<const uint4*>(ks + off + gid * 128);
      const uint4 k1 = *reinterpret_cast<const uint4*>(ks + off + (gid + 8) * 128);
      mma16816<T>(s, k0.x, k1.x, k0.y, k1.y, qf[qc].x, qf[qc].y);
      mma16816<T>(t, k0.z, k1.z, k0.w, k1.w, qf[qc].z, qf[qc].w);
    }
    float x0 = (s[0] + t[0]) * scale_log2, x1 = (s[1] + t[1]) * scale_log2;  // token gid
    float x2 = (s[2] + t[2]) * scale_log2, x3 = (s[3] + t[3]) * scale_log2;  // token gid + 8
    if (valid < kBlockSize) {
      if (gid >= valid) x0 = x1 = -INFINITY;
      if (gid + 8 >= valid) x2 = x3 = -INFINITY;
    }
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: token 0 is valid
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    const uint32_t plo = pack2<T>(exp2f(x0 - mn0), exp2f(x1 - mn1));  // token gid, heads 2c, 2c+1
    const uint32_t phi = pack2<T>(exp2f(x2 - mn0), exp2f(x3 - mn1));  // token gid + 8
    const float2 fl = unpack2<T>(plo), fh = unpack2<T>(phi);
    l0 = l0 * al0 + (fl.x + fh.x);  // sums of the rounded weights the P V product uses
    l1 = l1 * al1 + (fl.y + fh.y);
    // P^T as the B operand: tokens 2c, 2c+1 (and 2c+8, 2c+9) of head gid.
    const uint32_t b0 = movmatrix_trans(plo);
    const uint32_t b1 = movmatrix_trans(phi);

    uint4 vr[4][Shape::kBoxes];  // V rows 2c, 2c+1, 2c+8, 2c+9; chunk gid of each box
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int row = 2 * c + (rr & 1) + 8 * (rr >> 1);
#pragma unroll
      for (int a = 0; a < Shape::kBoxes; ++a)
        vr[rr][a] = *reinterpret_cast<const uint4*>(vs + a * 2048 + row * 128 + ((gid ^ (row & 7)) << 4));
      if (valid < kBlockSize && row >= valid) {
#pragma unroll
        for (int a = 0; a < Shape::kBoxes; ++a) vr[rr][a] = make_uint4(0, 0, 0, 0);  // never 0 * NaN
      }
    }
#pragma unroll
    for (int mt = 0; mt < Shape::kMTiles; ++mt) {
      acc[mt][0] *= al0;
      acc[mt][1] *= al1;
      acc[mt][2] *= al0;
      acc[mt][3] *= al1;
    }
    // m-tile mt, row r: head_dim index 8 * gid + mt (rows 0-7) and, for rows
    // 8-15, 8 * (gid + 8) + mt when D = 128 or 8 * gid + 4 + mt when D = 64.
#pragma unroll
    for (int mt = 0; mt < Shape::kMTiles; ++mt) {
      const uint32_t sel = (mt & 1) ? 0x7632u : 0x5410u;
      const int w0 = mt >> 1;
      const int bx1 = Shape::kBoxes == 2 ? 1 : 0;
      const int w1 = Shape::kBoxes == 2 ? (mt >> 1) : 2 + (mt >> 1);
      const uint32_t a0 = __byte_perm(word_of(vr[0][0], w0), word_of(vr[1][0], w0), sel);
      const uint32_t a1 = __byte_perm(word_of(vr[0][bx1], w1), word_of(vr[1][bx1], w1), sel);
      const uint32_t a2 = __byte_perm(word_of(vr[2][0], w0), word_of(vr[3][0], w0), sel);
      const uint32_t a3 = __byte_perm(word_of(vr[2][bx1], w1), word_of(vr[3][bx1], w1), sel);
      mma16816<T>(acc[mt], a0, a1, a2, a3, b0, b1);
    }
  }

  // Complete the row sums (each lane summed tokens gid and gid + 8 only).
  __device__ __forceinline__ void finish_sums() {
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
  }

  // The 8 values of chunk `k` (0: chunk gid, 1: chunk gid + 8 when D = 128)
  // of head 2c + e, scaled by `mul`.
  __device__ __forceinline__ void chunk_values(int e, int k, float mul, float (&v)[8]) const {
    if constexpr (D == 128) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) v[mt] = acc[mt][2 * k + e] * mul;
    } else {
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        v[mt] = acc[mt][e] * mul;
        v[4 + mt] = acc[mt][2 + e] * mul;
      }
    }
  }

  // Head-dim offset of chunk k of this lane.
  __device__ __forceinline__ static int chunk_dim(int lane, int k) { return 8 * ((lane >> 2) + 8 * k); }
  static constexpr int kChunks = D / 64;
};

template <typename T>
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  return make_uint4(pack2<T>(v[0], v[1]), pack2<T>(v[2], v[3]), pack2<T>(v[4], v[5]), pack2<T>(v[6], v[7]));
}

// ===================================================================== shared argument block

struct DecodeArgs {
  const void* q;              // T[B][Hq][D]
  void* out;                  // T[B][Hq][D]
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_o;              // split: f32[B][Hq][splits][D]; persistent: f32[warps][2][8][D]
  float* part_lse;            // split: f32[B][Hq][splits];    persistent: f32[warps][2][8]
  int32_t* counters;          // persistent: int32[B][Hkv], zero between calls
  float scale_log2;           // scale * log2(e)
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;              // Hq / Hkv, 1..8
  int32_t max_blocks;
  int32_t num_blocks;
  int32_t num_splits;         // split path only
  int32_t split_blocks;       // split path only
};

// Context length as the kernels see it: clamped to [0, max_blocks * 16].
__device__ __forceinline__ int clamped_context(const int32_t* lens, int b, int max_blocks, bool flag) {
  int ctx = lens[b];
  const int cap = max_blocks * kBlockSize;
  if (ctx < 0 || ctx > cap) {
    if (flag) flag_error(kErrContext);
    ctx = ctx < 0 ? 0 : cap;
  }
  return ctx;
}

// Pool row of (physical block, KV head); a block id outside the pool is
// flagged and mapped to a row range entirely outside the tensor (reads zeros).
__device__ __forceinline__ int tile_row(int phys, int kvh, const DecodeArgs& a) {
  if (phys < 0 || phys >= a.num_blocks) {
    flag_error(kErrBlockId);
    return -kBlockSize;
  }
  return (phys * a.num_kv_heads + kvh) * kBlockSize;
}

template <int D>
__device__ __forceinline__ void issue_block(uint32_t stage, uint32_t bar, const CUtensorMap* mk,
                                            const CUtensorMap* mv, int row, uint64_t policy) {
  using Shape = TileShape<D>;
  mbar_arrive_expect_tx(bar, Shape::kStageBytes);
#pragma unroll
  for (int bx = 0; bx < Shape::kBoxes; ++bx) {
    tma_load_2d(stage + bx * 2048, mk, bx * 64, row, bar, policy);
    tma_load_2d(stage + Shape::kTileBytes + bx * 2048, mv, bx * 64, row, bar, policy);
  }
}

// ===================================================================== persistent kernel

template <int D>
struct PersistentShape {
  static constexpr int kWarps = 8;
  static constexpr int kStages = D == 128 ? 3 : 6;  // per warp
  static constexpr int kRingBytes = kWarps * kStages * TileShape<D>::kStageBytes;
};

// Dynamic shared memory: [ring][prefix P[B+1]][context ctx[B]] (+1 KB alignment slack).
template <int D>
constexpr size_t persistent_smem_bytes(int num_seqs) {
  return PersistentShape<D>::kRingBytes + (2 * static_cast<size_t>(num_seqs) + 1) * 4 + 1024;
}

template <typename T, int D>
__global__ void __launch_bounds__(PersistentShape<D>::kWarps * 32, 1)
    decode_persistent_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                             const DecodeArgs a) {
  using Shape = TileShape<D>;
  constexpr int NW = PersistentShape<D>::kWarps;
  constexpr int SW = PersistentShape<D>::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[NW][SW];
  __shared__ int s_warp_sum[NW];

  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* s_P = reinterpret_cast<int*>(ring + PersistentShape<D>::kRingBytes);
  int* s_ctx = s_P + a.num_seqs + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.num_seqs, Hkv = a.num_kv_heads, g = a.group;

  // ---- context lengths and the exclusive prefix P[b] of blocks per sequence
  {
    const int per = (B + NW * 32 - 1) / (NW * 32);
    const int lo = min(B, tid * per), hi = min(B, lo + per);
    int local = 0;
    for (int b = lo; b < hi; ++b) {
      const int ctx = clamped_context(a.context_lens, b, a.max_blocks, blockIdx.x == 0);
      s_ctx[b] = ctx;
      local += (ctx + kBlockSize - 1) / kBlockSize;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp_sum[warp] = incl;
    if (lane == 0) {
      for (int s = 0; s < SW; ++s) mbar_init(smem_u32(&full_bar[warp][s]), 1);
      fence_mbar_init();
    }
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += s_warp_sum[w];
    for (int b = lo; b < hi; ++b) {
      s_P[b] = run;
      run += (s_ctx[b] + kBlockSize - 1) / kBlockSize;
    }
    if (tid == NW * 32 - 1) s_P[B] = run;
    __syncthreads();
  }

  // Empty contexts produce zero rows (CTA 0 writes them).
  if (blockIdx.x == 0) {
    for (int b = 0; b < B; ++b) {
      if (s_ctx[b] != 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(a.out) + static_cast<int64_t>(b) * a.num_q_heads * D);
      for (int i = tid; i < a.num_q_heads * D / 8; i += NW * 32) dst[i] = make_uint4(0, 0, 0, 0);
    }
  }

  const int total = Hkv * s_P[B];                       // blocks of all units
  const int nwarps = gridDim.x * NW;
  const int R = (total + nwarps - 1) / nwarps;          // blocks per warp
  const int gw = blockIdx.x * NW + warp;
  const int start = min(total, gw * R);
  const int n = min(total, start + R) - start;

  // Unit (b, kvh) and block j of flattened block f: units are ordered
  // (b, kvh) and unit (b, kvh) holds blocks [Hkv*P[b] + kvh*nb, +nb).
  auto locate = [&](int f, int& b, int& kvh, int& j) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (Hkv * s_P[mid] <= f) lo = mid; else hi = mid - 1;
    }
    b = lo;
    const int nb = (s_ctx[b] + kBlockSize - 1) / kBlockSize;
    const int rem = f - Hkv * s_P[b];
    kvh = rem / nb;
    j = rem - kvh * nb;
  };

  if (warp == 0 && lane == 0 && n > 0) {
    // Warm L2 with the query rows this CTA will read (contiguous: units are in q order).
    const int cta_lo = min(total, blockIdx.x * NW * R), cta_hi = min(total, (blockIdx.x + 1) * NW * R);
    if (cta_hi > cta_lo) {
      int b0, h0, j0, b1, h1, j1;
      locate(cta_lo, b0, h0, j0);
      locate(cta_hi - 1, b1, h1, j1);
      const int64_t u0 = static_cast<int64_t>(b0) * Hkv + h0, u1 = static_cast<int64_t>(b1) * Hkv + h1;
      prefetch_l2_bulk(static_cast<const T*>(a.q) + u0 * g * D,
                       static_cast<uint32_t>((u1 - u0 + 1) * g * D * sizeof(T)));
    }
  }

  if (n > 0) {
    uint8_t* wring = ring + warp * SW * Shape::kStageBytes;
    const uint64_t policy = l2_evict_first_policy();
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    // Per-lane block info for a 32-block chunk of this warp's range: lane i
    // describes block base + i (unit id, block index j, pool row).
    auto chunk_info = [&](int base, int& u, int& jj, int& row) {
      u = -1; jj = 0; row = -kBlockSize;
      if (base + lane < n) {
        int b, kvh, j;
        locate(start + base + lane, b, kvh, j);
        u = b * Hkv + kvh;
        jj = j;
        row = tile_row(__ldg(a.block_tables + static_cast<int64_t>(b) * a.max_blocks + j), kvh, a);
      }
    };
    int cu, cj, crow, nu = -1, nj = 0, nrow = -kBlockSize;
    chunk_info(0, cu, cj, crow);
    if (n > 32) chunk_info(32, nu, nj, nrow);

    // Fill the ring.
    for (int k = 0; k < min(SW, n); ++k) {
      const int row = __shfl_sync(0xffffffffu, crow, k);
      if (lane == 0)
        issue_block<D>(smem_u32(wring + k * Shape::kStageBytes), smem_u32(&full_bar[warp][k]), &tmap_k, &tmap_v,
                       row, policy);
    }

    WarpAttn<T, D> at;
    bool first_unit = true;
    int unit_first_j = 0;
    for (int k = 0; k < n; ++k) {
      if ((k & 31) == 0 && k > 0) {  // advance the chunk window
        cu = nu; cj = nj; crow = nrow;
        if (k + 32 < n) chunk_info(k + 32, nu, nj, nrow);
      }
      const int st = k % SW;
      if (!mbar_wait(smem_u32(&full_bar[warp][st]), (k / SW) & 1)) break;  // timed out: flagged
      const int u = __shfl_sync(0xffffffffu, cu, k & 31);
      const int j = __shfl_sync(0xffffffffu, cj, k & 31);
      const int b = u / Hkv, kvh = u - b * Hkv;
      const int ctx = s_ctx[b];
      const int nb = (ctx + kBlockSize - 1) / kBlockSize;
      if (k == 0 || j == 0) {
        unit_first_j = j;
        at.load_q(static_cast<const T*>(a.q) + (static_cast<int64_t>(b) * a.num_q_heads + kvh * g) * D, g, lane);
        at.reset();
      }
      const uint8_t* ks = wring + st * Shape::kStageBytes;
      at.block(ks, ks + Shape::kTileBytes, min(kBlockSize, ctx - j * kBlockSize), a.scale_log2, lane);

      // Refill this stage with block k + SW.
      const int kn = k + SW;
      const int src = kn & 31;
      const int r_cur = __shfl_sync(0xffffffffu, crow, src);
      const int r_nxt = __shfl_sync(0xffffffffu, nrow, src);
      __syncwarp();
      if (lane == 0 && kn < n) {
        fence_proxy_async_smem();
        issue_block<D>(smem_u32(wring + st * Shape::kStageBytes), smem_u32(&full_bar[warp][st]), &tmap_k, &tmap_v,
                       (kn & ~31) == (k & ~31) ? r_cur : r_nxt, policy);
      }

      if (j == nb - 1 || k == n - 1) {
        // ---- the unit ends in this warp's range: write it out or hand it to the merge
        at.finish_sums();
        const int gid = lane >> 2, c = lane & 3;
        if (unit_first_j == 0 && j == nb - 1) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = 2 * c + e;
            if (h >= g) continue;
            T* orow = static_cast<T*>(a.out) + (static_cast<int64_t>(b) * a.num_q_heads + kvh * g + h) * D;
            const float inv = 1.0f / (e ? at.l1 : at.l0);
#pragma unroll
            for (int kk = 0; kk < WarpAttn<T, D>::kChunks; ++kk) {
              float v[8];
              at.chunk_values(e, kk, inv, v);
              *reinterpret_cast<uint4*>(orow + WarpAttn<T, D>::chunk_dim(lane, kk)) = pack8<T>(v);
            }
          }
        } else {
          const int slot = first_unit ? 0 : 1;
          const int64_t pbase = (static_cast<int64_t>(gw) * 2 + slot) * kMaxGroup;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = 2 * c + e;
            const float l = e ? at.l1 : at.l0;
            float* prow = a.part_o + (pbase + h) * D;
#pragma unroll
            for (int kk = 0; kk < WarpAttn<T, D>::kChunks; ++kk) {
              float v[8];
              at.chunk_values(e, kk, 1.0f / l, v);
              float4* dst = reinterpret_cast<float4*>(prow + WarpAttn<T, D>::chunk_dim(lane, kk));
              dst[0] = make_float4(v[0], v[1], v[2], v[3]);
              dst[1] = make_float4(v[4], v[5], v[6], v[7]);
            }
            if (gid == 0) a.part_lse[pbase + h] = (e ? at.m1 : at.m0) + log2f(l);
          }
          // Count this piece; the warp that completes the unit merges it.
          const int U = Hkv * s_P[b] + kvh * nb;
          const int r0 = U / R, r1 = (U + nb - 1) / R;
          __threadfence();
          __syncwarp();
          int last = 0;
          if (lane == 0) last = atomicAdd(a.counters + u, 1) == r1 - r0;
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) {
            __threadfence();
            // lane: head lane / 4, head_dim quarter lane % 4
            const int h = lane >> 2;
            if (h < g) {
              constexpr int kQ = D / 4;
              const int d0 = (lane & 3) * kQ;
              float M = -INFINITY;
              for (int r = r0; r <= r1; ++r) {
                const int sl = (r == r0 && U > r0 * R) ? 1 : 0;
                M = fmaxf(M, __ldcg(a.part_lse + (static_cast<int64_t>(r) * 2 + sl) * kMaxGroup + h));
              }
              float o[kQ];
#pragma unroll
              for (int i = 0; i < kQ; ++i) o[i] = 0.f;
              float L = 0.f;
              for (int r = r0; r <= r1; ++r) {
                const int sl = (r == r0 && U > r0 * R) ? 1 : 0;
                const int64_t pr = (static_cast<int64_t>(r) * 2 + sl) * kMaxGroup + h;
                const float w = exp2f(__ldcg(a.part_lse + pr) - M);
                L += w;
                const float4* src4 = reinterpret_cast<const float4*>(a.part_o + pr * D + d0);
#pragma unroll
                for (int i = 0; i < kQ / 4; ++i) {
                  const float4 x = __ldcg(src4 + i);
                  o[4 * i] += w * x.x;
                  o[4 * i + 1] += w * x.y;
                  o[4 * i + 2] += w * x.z;
                  o[4 * i + 3] += w * x.w;
                }
              }
              const float inv = 1.0f / L;
              T* orow = static_cast<T*>(a.out) + (static_cast<int64_t>(b) * a.num_q_heads + kvh * g + h) * D + d0;
#pragma unroll
              for (int i = 0; i < kQ / 8; ++i) {
                float v[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) v[x] = o[8 * i + x] * inv;
                *reinterpret_cast<uint4*>(orow + 8 * i) = pack8<T>(v);
              }
            }
            if (lane == 0) a.counters[u] = 0;  // ready for the next call
          }
        }
        first_unit = false;
      }
    }
  }
}

// ===================================================================== split kernel

// Warp roles: warps [0, NC) consume, warp NC produces (TMA).  Block i of the
// split lives in ring stage i % S and is consumed by warp i % NC; S is a
// multiple of NC so each stage always belongs to the same consumer warp, which
// therefore observes every phase of that stage's barriers in order.
template <typename T, int D, int NC, int S>
__global__ void __launch_bounds__((NC + 1) * 32)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        const DecodeArgs args) {
  using Shape = TileShape<D>;
  static_assert(S % NC == 0, "ring depth must be a multiple of the consumer warps");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[S];
  __shared__ __align__(8) uint64_t empty_bar[S];
  __shared__ int s_abort;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = args.group;

  const int ctx = clamped_context(args.context_lens, b, args.max_blocks, threadIdx.x == 0 && split == 0);
  const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
  const int blk0 = split * args.split_blocks;
  const int nb = min(nblk, blk0 + args.split_blocks) - blk0;

  if (nb <= 0) {
    // Empty split.  In one pass this is an empty context: write a zero row.
    if (args.num_splits == 1) {
      T* out = static_cast<T*>(args.out) + (static_cast<int64_t>(b) * args.num_q_heads + kvh * g) * D;
      for (int i = threadIdx.x; i < g * D; i += blockDim.x) out[i] = T(0.0f);
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  WarpAttn<T, D> at;
  at.reset();

  if (warp == NC) {
    // ------------------------------------------------------------ producer
    const int32_t* trow = args.block_tables + static_cast<int64_t>(b) * args.max_blocks + blk0;
    const uint64_t policy = l2_evict_first_policy();
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    int issued = 0;
    bool ok = true;
    for (int base = 0; base < nb && ok; base += 32) {
      const int j = base + lane;
      const int row = j < nb ? tile_row(trow[j], kvh, args) : 0;
      const int cnt = min(32, nb - base);
      for (int k = 0; k < cnt; ++k) {
        const int r = __shfl_sync(0xffffffffu, row, k);
        if (lane == 0 && ok) {
          const int i = base + k;
          const int st = i % S;
          if (i >= S && !mbar_wait(smem_u32(&empty_bar[st]), ((i / S) & 1) ^ 1)) {
            ok = false;
            s_abort = 1;
          } else if (*reinterpret_cast<volatile int*>(&s_abort)) {
            ok = false;
          } else {
            issue_block<D>(smem_u32(smem + st * Shape::kStageBytes), smem_u32(&full_bar[st]), &tmap_k, &tmap_v, r,
                           policy);
            ++issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
    // No copy may still be landing in shared memory when the CTA moves on.
    if (lane == 0) {
      for (int i = max(0, issued - S); i < issued; ++i) mbar_wait(smem_u32(&full_bar[i % S]), (i / S) & 1);
    }
  } else {
    // ------------------------------------------------------------ consumers
    at.load_q(static_cast<const T*>(args.q) + (static_cast<int64_t>(b) * args.num_q_heads + kvh * g) * D, g, lane);
    for (int i = warp; i < nb; i += NC) {
      if (*reinterpret_cast<volatile int*>(&s_abort)) break;
      const int st = i % S;
      if (!mbar_wait(smem_u32(&full_bar[st]), (i / S) & 1)) {
        s_abort = 1;
        break;
      }
      const uint8_t* ks = smem + st * Shape::kStageBytes;
      at.block(ks, ks + Shape::kTileBytes, min(kBlockSize, ctx - (blk0 + i) * kBlockSize), args.scale_log2, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));  // stage may be refilled
    }
    at.finish_sums();
  }

  // ---------------------------------------------------------------- merge warps
  __syncthreads();  // ring drained: reuse it for the cross-warp merge
  float* red_o = reinterpret_cast<float*>(smem);  // [NC][8][D]
  float* red_m = red_o + NC * kMaxGroup * D;      // [NC][8]
  float* red_l = red_m + NC * kMaxGroup;          // [NC][8]
  if (warp < NC) {
    const int gid = lane >> 2, c = lane & 3;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = 2 * c + e;
      if (gid == 0) {
        red_m[warp * kMaxGroup + h] = e ? at.m1 : at.m0;
        red_l[warp * kMaxGroup + h] = e ? at.l1 : at.l0;
      }
      float* dst = red_o + (warp * kMaxGroup + h) * D;
#pragma unroll
      for (int kk = 0; kk < WarpAttn<T, D>::kChunks; ++kk) {
        float v[8];
        at.chunk_values(e, kk, 1.0f, v);
        float4* d4 = reinterpret_cast<float4*>(dst + WarpAttn<T, D>::chunk_dim(lane, kk));
        d4[0] = make_float4(v[0], v[1], v[2], v[3]);
        d4[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  }
  __syncthreads();
  if (*reinterpret_cast<volatile int*>(&s_abort)) return;

  constexpr int kQuads = D / 4;
  for (int idx = threadIdx.x; idx < g * kQuads; idx += blockDim.x) {
    const int row = idx / kQuads;
    const int d4 = (idx - row * kQuads) * 4;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NC; ++w) M = fmaxf(M, red_m[w * kMaxGroup + row]);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NC; ++w) {
      const float wt = exp2f(red_m[w * kMaxGroup + row] - M);  // 0 for a warp that saw no block
      L += red_l[w * kMaxGroup + row] * wt;
      const float4 v = *reinterpret_cast<const float4*>(red_o + (w * kMaxGroup + row) * D + d4);
      o.x += v.x * wt;
      o.y += v.y * wt;
      o.z += v.z * wt;
      o.w += v.w * wt;
    }
    const float inv = 1.0f / L;
    const int hq = kvh * g + row;
    if (args.num_splits == 1) {
      T* out = static_cast<T*>(args.out) + (static_cast<int64_t>(b) * args.num_q_heads + hq) * D + d4;
      uint2 pk;
      pk.x = pack2<T>(o.x * inv, o.y * inv);
      pk.y = pack2<T>(o.z * inv, o.w * inv);
      *reinterpret_cast<uint2*>(out) = pk;
    } else {
      const int64_t prow = (static_cast<int64_t>(b) * args.num_q_heads + hq) * args.num_splits + split;
      *reinterpret_cast<float4*>(args.part_o + prow * D + d4) = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
      if (d4 == 0) args.part_lse[prow] = M + log2f(L);
    }
  }
}

// One warp per (sequence, query head): out = sum_s w_s o_s / sum_s w_s with
// w_s = 2^(lse_s - max lse), over the splits that hold at least one token.
template <typename T, int D>
__global__ void __launch_bounds__(128) merge_split_kernel(const float* __restrict__ o_part,
                                                          const float* __restrict__ lse_part,
                                                          const int32_t* __restrict__ context_lens,
                                                          T* __restrict__ out, int32_t num_seqs, int32_t num_q_heads,
                                                          int32_t num_splits, int32_t split_blocks,
                                                          int32_t max_blocks) {
  constexpr int kPer = D / 32;  // outputs per lane
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= num_seqs * num_q_heads) return;
  const int b = row / num_q_heads;
  const int ctx = clamped_context(context_lens, b, max_blocks, false);
  const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
  const int nvalid = (nblk + split_blocks - 1) / split_blocks;
  T* dst = out + static_cast<int64_t>(row) * D + lane * kPer;
  float o[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) o[k] = 0.f;
  if (nvalid > 0) {
    const float* lse = lse_part + static_cast<int64_t>(row) * num_splits;
    float M = -INFINITY;
    for (int s = 0; s < nvalid; ++s) M = fmaxf(M, lse[s]);
    float L = 0.f;
    for (int s = 0; s < nvalid; ++s) {
      const float w = exp2f(lse[s] - M);
      L += w;
      const float* src = o_part + (static_cast<int64_t>(row) * num_splits + s) * D + lane * kPer;
#pragma unroll
      for (int k = 0; k < kPer; k += 2) {
        const float2 v = *reinterpret_cast<const float2*>(src + k);
        o[k] += w * v.x;
        o[k + 1] += w * v.y;
      }
    }
    const float inv = 1.0f / L;
#pragma unroll
    for (int k = 0; k < kPer; ++k) o[k] *= inv;
  }
#pragma unroll
  for (int k = 0; k < kPer; k += 2) *reinterpret_cast<uint32_t*>(dst + k) = pack2<T>(o[k], o[k + 1]);
}

}  // namespace pkv
