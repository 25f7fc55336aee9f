// Kernels of the paged decode path (sm_103a).
//
//  append_kernel  -- slot-mapped copy of each new token's K/V into the pool
//                    ("How to Scale Your Model, Part 7: Inference", section
//                    "Transformer 推論の基礎: Prefill と Generation": the new
//                    token's K/V projection is appended to the cache).
//  decode_kernel  -- one CTA per (split, KV head, sequence): walks the block
//                    table (kasblo.com "vLLMとは？", section
//                    "PagedAttentionはKV Cacheをblockで管理する"), streams each
//                    K/V block once through a TMA ring in shared memory, and
//                    serves the whole GQA query group from that one read with
//                    an fp32 online softmax (design.babushkai.com
//                    "GPU推論の内部構造", section "カーネル: FlashAttentionとメモリ階層").
//  merge_kernel   -- log-sum-exp merge of the normalised split partials.
//
// Cache layout: T[num_blocks][Hkv][16][D].  The (block, KV head) tile of
// 16 tokens x D is contiguous; the TMA tensor map views the pool as a 2-D
// array of rows = num_blocks * Hkv * 16 and D columns and loads the tile as
// D/64 boxes of 16 rows x 64 elements (128 bytes) with the 128-byte swizzle,
// so the fragment loads below are free of shared-memory bank conflicts.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

constexpr int kBlockSize = 16;

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

// ===================================================================== decode

struct DecodeArgs {
  const void* q;              // T[B][Hq][D]
  void* out;                  // T[B][Hq][D]          (single pass)
  float* o_part;              // f32[B][Hq][splits][D] (split pass, normalised)
  float* lse_part;            // f32[B][Hq][splits]    (log2-domain log-sum-exp)
  const int32_t* block_tables;
  const int32_t* context_lens;
  float scale_log2;           // scale * log2(e)
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;              // Hq / Hkv, 1..8
  int32_t max_blocks;
  int32_t num_blocks;
  int32_t num_splits;
  int32_t split_blocks;       // blocks per split
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

template <int D>
struct DecodeShape {
  static constexpr int kBoxes = D / 64;                  // 64-element boxes per row
  static constexpr int kTileBytes = kBlockSize * D * 2;  // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;     // K + V
  static constexpr int kQChunks = D / 32;                // 16-byte chunks of q per lane
  static constexpr int kNTiles = D / 8;                  // n-tiles of the P*V product
};

// Warp roles: warps [0, NC) consume, warp NC produces (TMA).  Block i of the
// split lives in ring stage i % S and is consumed by warp i % NC; S is a
// multiple of NC so each stage always belongs to the same consumer warp,
// which therefore observes every phase of that stage's barriers in order.
template <typename T, int D, int NC, int S>
__global__ void __launch_bounds__((NC + 1) * 32)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeArgs args) {
  using Shape = DecodeShape<D>;
  static_assert(S % NC == 0, "ring depth must be a multiple of the consumer warps");
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");

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

  float m_run = -INFINITY, l_run = 0.0f;
  float acc[Shape::kNTiles][4];
#pragma unroll
  for (int i = 0; i < Shape::kNTiles; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

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
      int row = 0;
      if (j < nb) {
        const int phys = trow[j];
        if (phys < 0 || phys >= args.num_blocks) {
          flag_error(kErrBlockId);
          row = -kBlockSize;  // entirely outside the tensor: the box reads zeros
        } else {
          row = (phys * args.num_kv_heads + kvh) * kBlockSize;
        }
      }
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
            const uint32_t fb = smem_u32(&full_bar[st]);
            const uint32_t ks = smem_u32(smem + st * Shape::kStageBytes);
            mbar_arrive_expect_tx(fb, Shape::kStageBytes);
#pragma unroll
            for (int bx = 0; bx < Shape::kBoxes; ++bx) {
              tma_load_2d(ks + bx * 2048, &tmap_k, bx * 64, r, fb, policy);
              tma_load_2d(ks + Shape::kTileBytes + bx * 2048, &tmap_v, bx * 64, r, fb, policy);
            }
            ++issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
    // Make sure no copy is still landing in shared memory when the CTA moves on.
    if (lane == 0) {
      for (int i = max(0, issued - S); i < issued; ++i) mbar_wait(smem_u32(&full_bar[i % S]), (i / S) & 1);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int gid = lane >> 2;  // row of the query group (mma row), token row of K
    const int c = lane & 3;     // quad position
    const bool row_ok = gid < g;
    const T* qrow = static_cast<const T*>(args.q) + (static_cast<int64_t>(b) * args.num_q_heads + kvh * g + gid) * D;

    // q fragments: lane owns 16-byte chunks {2c, 2c+1, 2c+8, 2c+9} (D = 128)
    // or {2c, 2c+1} (D = 64) of its row; k-step j uses half j & 1 of chunk j / 2.
    uint4 qf[Shape::kQChunks];
#pragma unroll
    for (int qc = 0; qc < Shape::kQChunks; ++qc) {
      const int chunk = 2 * c + (qc & 1) + 8 * (qc >> 1);
      qf[qc] = row_ok ? __ldg(reinterpret_cast<const uint4*>(qrow) + chunk) : make_uint4(0, 0, 0, 0);
    }

    for (int i = warp; i < nb; i += NC) {
      if (*reinterpret_cast<volatile int*>(&s_abort)) break;
      const int st = i % S;
      if (!mbar_wait(smem_u32(&full_bar[st]), (i / S) & 1)) {
        s_abort = 1;
        break;
      }
      const uint8_t* ks = smem + st * Shape::kStageBytes;
      const uint8_t* vs = ks + Shape::kTileBytes;

      // S = Q K^T for this block's 16 tokens: n-tile nt covers token rows
      // 8nt..8nt+7; this lane supplies K row gid + 8nt.
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int row = gid + 8 * nt;
#pragma unroll
        for (int qc = 0; qc < Shape::kQChunks; ++qc) {
          const int cb = 2 * c + (qc & 1);  // chunk within the 64-element box
          const uint4 kv =
              *reinterpret_cast<const uint4*>(ks + (qc >> 1) * 2048 + row * 128 + ((cb ^ gid) << 4));
          mma16816<T>(s[nt], qf[qc].x, 0u, qf[qc].y, 0u, kv.x, kv.y);
          mma16816<T>(s[nt], qf[qc].z, 0u, qf[qc].w, 0u, kv.z, kv.w);
        }
      }

      // Online softmax (log2 domain) over tokens 2c, 2c+1, 8+2c, 9+2c of the block.
      const int tok0 = (blk0 + i) * kBlockSize;
      float x0 = s[0][0] * args.scale_log2, x1 = s[0][1] * args.scale_log2;
      float x2 = s[1][0] * args.scale_log2, x3 = s[1][1] * args.scale_log2;
      const bool tail = tok0 + kBlockSize > ctx;
      if (tail) {
        if (tok0 + 2 * c >= ctx) x0 = -INFINITY;
        if (tok0 + 2 * c + 1 >= ctx) x1 = -INFINITY;
        if (tok0 + 8 + 2 * c >= ctx) x2 = -INFINITY;
        if (tok0 + 9 + 2 * c >= ctx) x3 = -INFINITY;
      }
      float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);  // finite: the block holds a valid token
      const float alpha = exp2f(m_run - m_new);
      const uint32_t pa0 = pack2<T>(exp2f(x0 - m_new), exp2f(x1 - m_new));
      const uint32_t pa2 = pack2<T>(exp2f(x2 - m_new), exp2f(x3 - m_new));
      const float2 p01 = unpack2<T>(pa0), p23 = unpack2<T>(pa2);
      l_run = l_run * alpha + ((p01.x + p01.y) + (p23.x + p23.y));
      m_run = m_new;

      // V rows 2c, 2c+1, 2c+8, 2c+9; chunks gid (+8) of each row.
      uint4 vr[4][Shape::kBoxes];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int row = 2 * c + (rr & 1) + 8 * (rr >> 1);
#pragma unroll
        for (int a = 0; a < Shape::kBoxes; ++a)
          vr[rr][a] = *reinterpret_cast<const uint4*>(vs + a * 2048 + row * 128 + ((gid ^ (row & 7)) << 4));
      }
      if (tail) {
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int row = 2 * c + (rr & 1) + 8 * (rr >> 1);
          if (tok0 + row >= ctx) {
#pragma unroll
            for (int a = 0; a < Shape::kBoxes; ++a) vr[rr][a] = make_uint4(0, 0, 0, 0);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));  // stage may be refilled

#pragma unroll
      for (int t = 0; t < Shape::kNTiles; ++t) {
        acc[t][0] *= alpha;
        acc[t][1] *= alpha;
      }
      // O += P V: n-tile t = 8a + e holds output column 8 * (n + 8a) + e for
      // mma column n; this lane supplies column n = gid, i.e. element e of chunk gid + 8a.
#pragma unroll
      for (int a = 0; a < Shape::kBoxes; ++a) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t sel = (e & 1) ? 0x7632u : 0x5410u;
          const uint32_t b0 = __byte_perm(word_of(vr[0][a], e >> 1), word_of(vr[1][a], e >> 1), sel);
          const uint32_t b1 = __byte_perm(word_of(vr[2][a], e >> 1), word_of(vr[3][a], e >> 1), sel);
          mma16816<T>(acc[8 * a + e], pa0, 0u, pa2, 0u, b0, b1);
        }
      }
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  }

  // ---------------------------------------------------------------- merge warps
  __syncthreads();  // ring drained: reuse it for the cross-warp merge
  float* red_o = reinterpret_cast<float*>(smem);  // [NC][8][D]
  float* red_m = red_o + NC * 8 * D;              // [NC][8]
  float* red_l = red_m + NC * 8;                  // [NC][8]
  if (warp < NC) {
    const int gid = lane >> 2, c = lane & 3;
    if (c == 0) {
      red_m[warp * 8 + gid] = m_run;
      red_l[warp * 8 + gid] = l_run;
    }
    float* dst = red_o + (warp * 8 + gid) * D;
#pragma unroll
    for (int a = 0; a < Shape::kBoxes; ++a) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        dst[8 * (2 * c + 8 * a) + e] = acc[8 * a + e][0];
        dst[8 * (2 * c + 1 + 8 * a) + e] = acc[8 * a + e][1];
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
    for (int w = 0; w < NC; ++w) M = fmaxf(M, red_m[w * 8 + row]);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NC; ++w) {
      const float wt = exp2f(red_m[w * 8 + row] - M);  // 0 for a warp that saw no block
      L += red_l[w * 8 + row] * wt;
      const float4 v = *reinterpret_cast<const float4*>(red_o + (w * 8 + row) * D + d4);
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
      *reinterpret_cast<float4*>(args.o_part + prow * D + d4) = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
      if (d4 == 0) args.lse_part[prow] = M + log2f(L);
    }
  }
}

// ===================================================================== merge

// One warp per (sequence, query head): out = sum_s w_s o_s / sum_s w_s with
// w_s = 2^(lse_s - max lse), over the splits that hold at least one token.
template <typename T, int D>
__global__ void __launch_bounds__(128) merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                                                    const int32_t* __restrict__ context_lens, T* __restrict__ out,
                                                    int32_t num_seqs, int32_t num_q_heads, int32_t num_splits,
                                                    int32_t split_blocks, int32_t max_blocks) {
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
