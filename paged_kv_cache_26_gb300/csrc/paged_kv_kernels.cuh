// Kernels of the paged decode path (sm_103a).
//
//  append_kernel            -- slot-mapped copy of each new token's K/V into the
//                              pool ("How to Scale Your Model, Part 7: Inference",
//                              section "Transformer 推論の基礎: Prefill と
//                              Generation": the new token's K/V projection is
//                              appended to the cache).
//  decode_persistent_kernel -- the automatic path.  One CTA per SM; the flattened
//                              (sequence, KV head, block) space is cut into equal
//                              shares, one per warp, whatever the length mix.  A
//                              warp streams the head of its share, then claims
//                              tail chunks of any share from a counter, so SMs
//                              with more memory bandwidth take more work.
//  merge_persistent_kernel  -- log-sum-exp merge of the units it left in pieces.
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
//
// FP8 cache: the same kernels over a pool of E4M3 codes, uint8[num_blocks][Hkv]
// [16][D] with one float32 scale per KV head for K and one for V (value =
// code * scale; design.babushkai.com "GPU推論の内部構造", section "KVキャッシュの
// 台帳": an FP8 cache halves the bytes per token).  A tile row is then 128
// bytes for D = 128 and a tile one 2 KB box.
#pragma once

#include <type_traits>

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
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// The same copy with each sequence's slot derived from its table: token b goes
// to position context_lens[b] - 1 (nothing when the context is empty).
__global__ void append_at_end_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                     const int32_t* __restrict__ block_tables,
                                     const int32_t* __restrict__ context_lens, int32_t num_seqs,
                                     int32_t max_blocks, int32_t num_kv_heads, int32_t chunks_per_row,
                                     int32_t num_blocks, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * chunks_per_row;
  const int64_t total = per_token * num_seqs;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = idx / per_token;
    const int L = context_lens[b];
    if (L <= 0) continue;
    if (L > max_blocks * kBlockSize) {
      flag_error(kErrContext);
      continue;
    }
    const int pos = L - 1;
    const int32_t blk = block_tables[b * max_blocks + pos / kBlockSize];
    if (blk < 0 || blk >= num_blocks) {
      flag_error(kErrBlockId);
      continue;
    }
    const int64_t within = idx - b * per_token;
    const int64_t head = within / chunks_per_row;
    const int64_t chunk = within - head * chunks_per_row;
    const int64_t dst =
        ((static_cast<int64_t>(blk) * num_kv_heads + head) * kBlockSize + pos % kBlockSize) * chunks_per_row + chunk;
    k_cache[dst] = k_new[idx];
    v_cache[dst] = v_new[idx];
  }
}

// E4M3 codes of 8 fp16/bf16 values divided by `scale` (IEEE fp32 division,
// then round to nearest even with saturation to +-448).
template <typename T>
__device__ __forceinline__ uint2 quantize8(const uint4& v, float scale) {
  uint32_t out[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float2 a = unpack2<T>(word_of(v, 2 * h)), b = unpack2<T>(word_of(v, 2 * h + 1));
    const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(a.x, scale), __fdiv_rn(a.y, scale));
    const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(b.x, scale), __fdiv_rn(b.y, scale));
    out[h] = lo | (hi << 16);
  }
  return make_uint2(out[0], out[1]);
}

// Slot-mapped append into an E4M3 pool: one thread quantises 8 consecutive
// elements of one token's K row and of its V row for one KV head (C = D / 8
// groups per row) with that head's scales.
template <typename T>
__global__ void append_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                  const int32_t* __restrict__ slots, int32_t num_tokens, int32_t num_kv_heads,
                                  int32_t groups_per_row, int64_t num_slots, uint2* __restrict__ k_cache,
                                  uint2* __restrict__ v_cache, const float* __restrict__ k_scale,
                                  const float* __restrict__ v_scale) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * groups_per_row;
  const int64_t total = per_token * num_tokens;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t token = idx / per_token;
    const int64_t within = idx - token * per_token;  // head * C + group
    const int32_t slot = slots[token];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      flag_error(kErrSlot);
      continue;
    }
    const int64_t blk = slot / kBlockSize;
    const int64_t off = slot % kBlockSize;
    const int64_t head = within / groups_per_row;
    const int64_t grp = within - head * groups_per_row;
    const int64_t dst = ((blk * num_kv_heads + head) * kBlockSize + off) * groups_per_row + grp;
    k_cache[dst] = quantize8<T>(k_new[idx], __ldg(k_scale + head));
    v_cache[dst] = quantize8<T>(v_new[idx], __ldg(v_scale + head));
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
    uint32_t b0, b1, c0 = 0, c1 = 0;
    weights(exp2f(x0 - mn0), exp2f(x1 - mn1), exp2f(x2 - mn0), exp2f(x3 - mn1), al0, al1, b0, b1, c0, c1);

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
      if constexpr (MmaKind<T>::kBf16) mma16816<T>(acc[mt], a0, a1, a2, a3, c0, c1);
    }
  }

  // Softmax weights of tokens gid (e0: head 2c, e1: head 2c+1) and gid + 8
  // (e2, e3) as the B operand of O^T += V^T P^T (b0 / b1: tokens 2c, 2c+1 and
  // 2c+8, 2c+9 of head gid, via movmatrix), and the running sums.  fp16 keeps
  // 11 bits of each weight, enough for the output bound; bf16 keeps 8, which
  // short contexts with cancelling values would feel (about 2^-9 of |V|), so
  // for bf16 the weights go in as two bf16 terms, p = hi + lo (c0 / c1 = lo),
  // good to about 2^-17.  l sums the weights as fp32 (what the product uses,
  // to that precision).
  __device__ __forceinline__ void weights(float e0, float e1, float e2, float e3, float al0, float al1, uint32_t& b0,
                                          uint32_t& b1, uint32_t& c0, uint32_t& c1) {
    const uint32_t plo = pack2<T>(e0, e1);
    const uint32_t phi = pack2<T>(e2, e3);
    b0 = movmatrix_trans(plo);
    b1 = movmatrix_trans(phi);
    if constexpr (MmaKind<T>::kBf16) {
      const float2 fl = unpack2<T>(plo), fh = unpack2<T>(phi);
      c0 = movmatrix_trans(pack2<T>(e0 - fl.x, e1 - fl.y));
      c1 = movmatrix_trans(pack2<T>(e2 - fh.x, e3 - fh.y));
      l0 = l0 * al0 + (e0 + e2);
      l1 = l1 * al1 + (e1 + e3);
    } else {
      const float2 fl = unpack2<T>(plo), fh = unpack2<T>(phi);
      l0 = l0 * al0 + (fl.x + fh.x);  // sums of the rounded weights the P V product uses
      l1 = l1 * al1 + (fl.y + fh.y);
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

// One warp's attention state for one unit whose K and V tiles hold E4M3
// codes (D = 128: a tile row is 128 bytes, one TMA box with the 128-byte
// swizzle).  Every E4M3 value is exactly an fp16 value, so the products run as
// fp16 mma with fp32 accumulation, the query converted to fp16 at load and
// the weights P rounded to fp16.  The per-KV-head scales stay outside the mma:
// K's is folded into the logit scale, V's into the final normalisation.
// Lane (gid = lane/4, c = lane%4):
//  * S^T = K Q^T: k-step j (0..7) covers head_dim entries 32c + 4j .. 32c + 4j + 3
//    (byte word j of chunks {2c, 2c+1} of K rows gid and gid + 8, and the same
//    entries of q row gid);
//  * O^T += V^T P^T: row m of m-tile mt is head_dim entry 16 gid + mt (m = gid)
//    or 16 gid + 8 + mt (m = gid + 8), so the lane reads chunk gid of V rows
//    2c, 2c+1, 2c+8, 2c+9 and ends up holding output entries
//    [16 gid, 16 gid + 16) of heads 2c and 2c + 1.
template <typename T>
struct WarpAttnE4M3 {
  static constexpr int D = 128;
  uint32_t qf[16];  // q row gid as fp16 pairs; k-step j uses qf[2j], qf[2j + 1]
  float acc[8][4];
  float m0, m1, l0, l1;

  __device__ __forceinline__ void reset() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  }

  // Entries [32c, 32c + 32) of query row gid.  A bf16 query beyond the fp16
  // range would become infinite: that is flagged (kErrQuery).
  __device__ __forceinline__ void load_q(const T* q_group, int group, int lane) {
    const int gid = lane >> 2, c = lane & 3;
    bool big = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 raw =
          gid < group ? __ldg(reinterpret_cast<const uint4*>(q_group + gid * D + 32 * c) + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t x = word_of(raw, w);
        if constexpr (MmaKind<T>::kBf16) {
          const float2 f = unpack2<T>(x);
          big |= fabsf(f.x) > 65504.f || fabsf(f.y) > 65504.f;
          qf[4 * i + w] = pack2<__half>(f.x, f.y);
        } else {
          qf[4 * i + w] = x;
        }
      }
    }
    if (__any_sync(0xffffffffu, big) && lane == 0) flag_error(kErrQuery);
  }

  // Scores of one 16-token K tile against the group: s[0..1] token gid and
  // s[2..3] token gid + 8 (heads 2c, 2c+1), unscaled; two interleaved mma
  // chains.
  __device__ __forceinline__ void scores(const uint8_t* ks, int lane, float (&x)[4]) const {
    const int gid = lane >> 2, c = lane & 3;
    const uint8_t* kr0 = ks + gid * 128;
    const uint8_t* kr1 = ks + (gid + 8) * 128;  // same swizzle phase: (gid + 8) & 7 == gid
    const uint4 ka0 = *reinterpret_cast<const uint4*>(kr0 + (((2 * c) ^ gid) << 4));
    const uint4 ka1 = *reinterpret_cast<const uint4*>(kr0 + (((2 * c + 1) ^ gid) << 4));
    const uint4 kb0 = *reinterpret_cast<const uint4*>(kr1 + (((2 * c) ^ gid) << 4));
    const uint4 kb1 = *reinterpret_cast<const uint4*>(kr1 + (((2 * c + 1) ^ gid) << 4));
    float s[4] = {0.f, 0.f, 0.f, 0.f}, t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t wa = word_of(j < 4 ? ka0 : ka1, j & 3);  // row gid: entries 32c + 4j .. + 3
      const uint32_t wb = word_of(j < 4 ? kb0 : kb1, j & 3);  // row gid + 8
      const uint32_t a0 = e4m3x2_to_f16x2(wa), a2 = e4m3x2_to_f16x2(wa >> 16);
      const uint32_t a1 = e4m3x2_to_f16x2(wb), a3 = e4m3x2_to_f16x2(wb >> 16);
      if (j & 1)
        mma16816<__half>(t, a0, a1, a2, a3, qf[2 * j], qf[2 * j + 1]);
      else
        mma16816<__half>(s, a0, a1, a2, a3, qf[2 * j], qf[2 * j + 1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = s[i] + t[i];
  }

  // Chunk gid of V rows 2c, 2c+1, 2c+8, 2c+9 of one tile; rows at or past
  // `valid` read as zeros (never 0 * NaN).
  __device__ __forceinline__ static void load_v(const uint8_t* vs, int valid, int lane, uint4 (&vr)[4]) {
    const int gid = lane >> 2, c = lane & 3;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int row = 2 * c + (rr & 1) + 8 * (rr >> 1);
      vr[rr] = *reinterpret_cast<const uint4*>(vs + row * 128 + ((gid ^ (row & 7)) << 4));
      if (valid < kBlockSize && row >= valid) vr[rr] = make_uint4(0, 0, 0, 0);
    }
  }

  // acc += V^T P^T for one tile.  m-tiles 2p and 2p + 1 read bytes 2p, 2p + 1
  // (rows m = gid) and 8 + 2p, 9 + 2p (rows m = gid + 8) of the chunks;
  // interleaving the byte pairs of two token rows puts each mma operand's two
  // tokens side by side.
  __device__ __forceinline__ void pv(const uint4 (&vr)[4], uint32_t b0, uint32_t b1) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int w = p >> 1;
      const uint32_t sel = (p & 1) ? 0x7362u : 0x5140u;
      const uint32_t x0 = __byte_perm(word_of(vr[0], w), word_of(vr[1], w), sel);
      const uint32_t x1 = __byte_perm(word_of(vr[0], w + 2), word_of(vr[1], w + 2), sel);
      const uint32_t x2 = __byte_perm(word_of(vr[2], w), word_of(vr[3], w), sel);
      const uint32_t x3 = __byte_perm(word_of(vr[2], w + 2), word_of(vr[3], w + 2), sel);
      mma16816<__half>(acc[2 * p], e4m3x2_to_f16x2(x0), e4m3x2_to_f16x2(x1), e4m3x2_to_f16x2(x2),
                       e4m3x2_to_f16x2(x3), b0, b1);
      mma16816<__half>(acc[2 * p + 1], e4m3x2_to_f16x2(x0 >> 16), e4m3x2_to_f16x2(x1 >> 16),
                       e4m3x2_to_f16x2(x2 >> 16), e4m3x2_to_f16x2(x3 >> 16), b0, b1);
    }
  }

  __device__ __forceinline__ void rescale(float al0, float al1) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      acc[mt][0] *= al0;
      acc[mt][1] *= al1;
      acc[mt][2] *= al0;
      acc[mt][3] *= al1;
    }
  }

  // Scores of tokens at or past `valid` in one tile become -inf.
  __device__ __forceinline__ static void mask(float (&x)[4], int valid, int lane) {
    const int gid = lane >> 2;
    if (valid < kBlockSize) {
      if (gid >= valid) x[0] = x[1] = -INFINITY;
      if (gid + 8 >= valid) x[2] = x[3] = -INFINITY;
    }
  }

  // Accumulate one block whose K and V tiles sit (swizzled) at ks / vs; the
  // first `valid` (1..16) of its 16 tokens belong to the context.
  __device__ __forceinline__ void block(const uint8_t* ks, const uint8_t* vs, int valid, float scale_log2,
                                        int lane) {
    float x[4];
    scores(ks, lane, x);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] *= scale_log2;
    mask(x, valid, lane);
    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: token 0 is valid
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    const uint32_t plo = pack2<__half>(exp2f(x[0] - mn0), exp2f(x[1] - mn1));  // token gid
    const uint32_t phi = pack2<__half>(exp2f(x[2] - mn0), exp2f(x[3] - mn1));  // token gid + 8
    const float2 fl = unpack2<__half>(plo), fh = unpack2<__half>(phi);
    l0 = l0 * al0 + (fl.x + fh.x);  // sums of the rounded weights the P V product uses
    l1 = l1 * al1 + (fl.y + fh.y);
    uint4 vr[4];
    load_v(vs, valid, lane, vr);
    rescale(al0, al1);
    pv(vr, movmatrix_trans(plo), movmatrix_trans(phi));
  }

  // Two consecutive blocks of one unit (tiles kA/vA, then kB/vB) as one
  // 32-token softmax step; `valid` (1..32) tokens belong to the context.
  __device__ __forceinline__ void block2(const uint8_t* kA, const uint8_t* vA, const uint8_t* kB, const uint8_t* vB,
                                         int valid, float scale_log2, int lane) {
    if (valid <= kBlockSize) {  // the second block is not part of this stage
      block(kA, vA, valid, scale_log2, lane);
      return;
    }
    float xa[4], xb[4];
    scores(kA, lane, xa);
    scores(kB, lane, xb);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xa[i] *= scale_log2;
      xb[i] *= scale_log2;
    }
    mask(xb, valid - kBlockSize, lane);
    float mx0 = fmaxf(fmaxf(xa[0], xa[2]), fmaxf(xb[0], xb[2]));
    float mx1 = fmaxf(fmaxf(xa[1], xa[3]), fmaxf(xb[1], xb[3]));
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    const uint32_t pal = pack2<__half>(exp2f(xa[0] - mn0), exp2f(xa[1] - mn1));
    const uint32_t pah = pack2<__half>(exp2f(xa[2] - mn0), exp2f(xa[3] - mn1));
    const uint32_t pbl = pack2<__half>(exp2f(xb[0] - mn0), exp2f(xb[1] - mn1));
    const uint32_t pbh = pack2<__half>(exp2f(xb[2] - mn0), exp2f(xb[3] - mn1));
    const float2 f0 = unpack2<__half>(pal), f1 = unpack2<__half>(pah);
    const float2 f2 = unpack2<__half>(pbl), f3 = unpack2<__half>(pbh);
    l0 = l0 * al0 + ((f0.x + f1.x) + (f2.x + f3.x));
    l1 = l1 * al1 + ((f0.y + f1.y) + (f2.y + f3.y));
    uint4 va[4], vb[4];
    load_v(vA, kBlockSize, lane, va);
    load_v(vB, valid - kBlockSize, lane, vb);
    rescale(al0, al1);
    pv(va, movmatrix_trans(pal), movmatrix_trans(pah));
    pv(vb, movmatrix_trans(pbl), movmatrix_trans(pbh));
  }

  __device__ __forceinline__ void finish_sums() {
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
  }

  // Entries chunk_dim(lane, k) .. + 7 of head 2c + e, scaled by `mul`.
  __device__ __forceinline__ void chunk_values(int e, int k, float mul, float (&v)[8]) const {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) v[mt] = acc[mt][2 * k + e] * mul;
  }
  __device__ __forceinline__ static int chunk_dim(int lane, int k) { return 16 * (lane >> 2) + 8 * k; }
  static constexpr int kChunks = 2;
};

// ===================================================================== shared argument block

struct DecodeArgs {
  const void* q;              // T[B][Hq][D]
  void* out;                  // T[B][Hq][D]
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_o;              // split: f32[B][Hq][splits][D]; persistent: f32[segments][2][8][D]
  float* part_lse;            // split: f32[B][Hq][splits];    persistent: f32[segments][2][8]
  int32_t* sched;             // persistent: int32[2] chunk counter and finished-warp counter, zero between calls
  int32_t* pub;               // persistent: [epoch][context B][prefix B + 1]: the decode grid's validated
                              // lengths, published (release) for the merge of the same call
  uint32_t epoch;             // persistent: this call's publication tag; 0 = none (the merge re-reads)
  const int32_t* pre_context_lens;  // persistent: where the decode and merge prologues (before their grid
  const int32_t* pre_block_tables;  // wait) read the lengths and tables; null: context_lens / block_tables.
                                    // The host-buffer step points them at the mapped host inputs that a copy
                                    // kernel, still running, is staging into context_lens / block_tables.
  const void* k_new;          // fused append (persistent only): T[B][Hkv][D], or null for no append
  const void* v_new;
  void* k_cache_w;            // the pool, for the appended rows
  void* v_cache_w;
  const float* k_scale;       // E4M3 pool only: f32[Hkv] scales of K and V codes
  const float* v_scale;
  float scale_log2;           // scale * log2(e)
  int32_t recheck;            // persistent: 1 = the lengths / tables read before the grid wait may be stale
                              // (device inputs a previous kernel may still write) and are read again after
                              // it; 0 = they are final when the kernel starts (written by the host)
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
__device__ __forceinline__ int clamp_context(int ctx, int max_blocks, bool flag) {
  const int cap = max_blocks * kBlockSize;
  if (ctx < 0 || ctx > cap) {
    if (flag) flag_error(kErrContext);
    ctx = ctx < 0 ? 0 : cap;
  }
  return ctx;
}
__device__ __forceinline__ int clamped_context(const int32_t* lens, int b, int max_blocks, bool flag) {
  return clamp_context(lens[b], max_blocks, flag);
}

// Pool row of (physical block, KV head); a block id outside the pool maps to
// a row range entirely outside the tensor (reads zeros) and, with `flag`, is
// flagged.
__device__ __forceinline__ int tile_row(int phys, int kvh, const DecodeArgs& a, bool flag = true) {
  if (phys < 0 || phys >= a.num_blocks) {
    if (flag) flag_error(kErrBlockId);
    return -kBlockSize;
  }
  return (phys * a.num_kv_heads + kvh) * kBlockSize;
}

// Byte geometry of one (block, KV head) K or V tile: 16 rows of D elements
// (2 bytes for fp16 / bf16, 1 for E4M3), loaded as 128-byte-wide TMA boxes of
// 16 rows (2 KB each) with the 128-byte swizzle.
template <int D, bool F8>
struct KvTile {
  static constexpr int kRowBytes = F8 ? D : 2 * D;
  static constexpr int kBoxes = kRowBytes / 128;
  static constexpr int kBoxElems = F8 ? 128 : 64;
  static constexpr int kTileBytes = kBlockSize * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
};

// TMA loads of one block's K and V tiles into a stage, completing on `bar`
// (whose transaction count the caller has set).
template <int D, bool F8 = false>
__device__ __forceinline__ void issue_tiles(uint32_t stage, uint32_t bar, const CUtensorMap* mk,
                                            const CUtensorMap* mv, int row, uint64_t policy) {
  using Tile = KvTile<D, F8>;
#pragma unroll
  for (int bx = 0; bx < Tile::kBoxes; ++bx) {
    tma_load_2d(stage + bx * 2048, mk, bx * Tile::kBoxElems, row, bar, policy);
    tma_load_2d(stage + Tile::kTileBytes + bx * 2048, mv, bx * Tile::kBoxElems, row, bar, policy);
  }
}

template <int D, bool F8 = false>
__device__ __forceinline__ void issue_block(uint32_t stage, uint32_t bar, const CUtensorMap* mk,
                                            const CUtensorMap* mv, int row, uint64_t policy) {
  mbar_arrive_expect_tx(bar, KvTile<D, F8>::kStageBytes);
  issue_tiles<D, F8>(stage, bar, mk, mv, row, policy);
}

// ===================================================================== persistent kernel

// 24 KB of K/V in flight per warp.  A stage holds one block (fp16/bf16: 3
// stages of 8 KB for D = 128, 6 of 4 KB for D = 64) or, for E4M3, two
// consecutive blocks of one unit (3 stages of 2 x 4 KB): 32 tokens per softmax
// step halve the per-block bookkeeping and give each warp two independent
// score chains.
template <int D, bool F8 = false>
struct PersistentShape {
  static constexpr int kWarps = F8 ? 12 : 8;
  static constexpr int kBlocksPerStage = F8 ? 2 : 1;
  static constexpr int kStageBytes = kBlocksPerStage * KvTile<D, F8>::kStageBytes;
  static constexpr int kStages = (F8 ? 16384 : 24576) / kStageBytes;  // per warp
  static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
};
constexpr int kMaxPersistentWarps = 12;  // sizes the workspace

// Dynamic shared memory: [ring][appended-token rows (fp16/bf16, K and V)]
// [prefix P[B+1]][context ctx[B]] (+1 KB alignment slack).
template <int D, bool F8 = false>
constexpr size_t persistent_smem_bytes(int num_seqs) {
  return PersistentShape<D, F8>::kRingBytes +
         PersistentShape<D, F8>::kWarps * PersistentShape<D, F8>::kStages * 4 * D +
         (2 * static_cast<size_t>(num_seqs) + 1) * 4 + 1024;
}

// Largest batch whose prefix arrays fit beside the ring in 227 KB of shared
// memory (1.5 KB kept for the static arrays, which take 1.2 KB), at most 2048.
template <int D, bool F8 = false>
constexpr int persistent_max_seqs() {
  constexpr long long room = 232448LL - 1536 - static_cast<long long>(persistent_smem_bytes<D, F8>(0));
  return room / 8 < 2048 ? static_cast<int>(room / 8) : 2048;
}

// Work partition of the persistent kernel.  The flattened block space
// [0, total) is cut into equal shares of R blocks, one per warp.  Each share
// is a static head, processed by its own warp, followed by tail chunks that
// warps claim in order from a counter once their head is done, so SMs with
// more memory bandwidth take more of the tails.  The tail is cut into four
// chunks (4/10, 3/10, 2/10, 1/10) for shares of 200 blocks or more, three
// (7/10, 2/10, 1/10) from 100, two (8/10, 2/10) below, with the head 4/5 of
// the share for three or four chunks and 17/20 for two: every segment
// boundary inside a unit leaves a piece for the merge, and fewer, larger
// chunks keep those few where a share is short.  Shares under
// kMinDynamicShare blocks are all head, with nothing to claim (the chunks
// would be too small to pay for their hand-over).  Chunk k of share w is
// segment nwarps + k * nwarps + w.  Every segment is a contiguous block
// range; the decode and merge kernels derive all boundaries from
// (total, nwarps) alone.
struct Partition {
  static constexpr int kMaxTailChunks = 4;
  static constexpr int kMinDynamicShare = 48;
  static constexpr int kThreeChunkShare = 100;
  static constexpr int kFourChunkShare = 200;
  int total, nwarps, R, nchunks;

  __device__ __forceinline__ Partition(int total_, int nwarps_)
      : total(total_), nwarps(nwarps_), R(total_ > 0 ? (total_ + nwarps_ - 1) / nwarps_ : 1),
        nchunks(R < kMinDynamicShare ? 0 : R < kThreeChunkShare ? 2 : R < kFourChunkShare ? 3 : 4) {}
  // Cumulative tenths of the tail before chunk k.
  __device__ __forceinline__ int cum(int k) const {
    if (nchunks == 2) return k == 0 ? 0 : k == 1 ? 8 : 10;
    if (nchunks == 3) return k == 0 ? 0 : k == 1 ? 7 : k == 2 ? 9 : 10;
    return k == 0 ? 0 : k == 1 ? 4 : k == 2 ? 7 : k == 3 ? 9 : 10;
  }
  __device__ __forceinline__ void head(int w, int& s, int& e) const {
    s = min(total, w * R);
    const int len = min(total, (w + 1) * R) - s;
    e = s + (nchunks == 0 ? len : nchunks == 2 ? len * 17 / 20 : len * 4 / 5);
  }
  __device__ __forceinline__ void chunk(int k, int w, int& s, int& e) const {
    int hs, he;
    head(w, hs, he);
    const int tail = min(total, (w + 1) * R) - he;
    s = he + tail * cum(k) / 10;
    e = he + tail * cum(k + 1) / 10;
  }
  __device__ __forceinline__ int num_chunks() const { return nwarps * nchunks; }
  __device__ __forceinline__ int seg_per_share() const { return 1 + nchunks; }
  __device__ __forceinline__ int num_segments() const { return nwarps * (1 + nchunks); }
  // Segment holding block p (0 <= p < total): its id and [s, e).
  __device__ __forceinline__ int segment_of(int p, int& s, int& e) const {
    const int w = p / R;
    head(w, s, e);
    if (p < e) return w;
    for (int k = 0; k < nchunks; ++k) {
      chunk(k, w, s, e);
      if (p < e) return nwarps + k * nwarps + w;
    }
    return -1;  // unreachable for p < total
  }
};

// Exclusive prefix of blocks per sequence into s_P[0..B] and clamped contexts
// into s_ctx[0..B), computed by the whole CTA (nthreads threads) from `lens`.
// Loads go to L2 (ld.global.cg), never to a per-SM cache that an earlier
// read before the grid wait could have filled.
__device__ __forceinline__ void context_prefix(const DecodeArgs& a, const int32_t* lens, int* s_P, int* s_ctx,
                                               int* s_warp_sum, int nthreads, bool flag) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, B = a.num_seqs;
  const int per = (B + nthreads - 1) / nthreads;
  const int lo = min(B, tid * per), hi = min(B, lo + per);
  int local = 0;
  for (int b = lo; b < hi; ++b) {
    const int ctx = clamp_context(__ldcg(lens + b), a.max_blocks, flag);
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
  __syncthreads();
  int run = incl - local;
  for (int w = 0; w < warp; ++w) run += s_warp_sum[w];
  for (int b = lo; b < hi; ++b) {
    s_P[b] = run;
    run += (s_ctx[b] + kBlockSize - 1) / kBlockSize;
  }
  if (tid == nthreads - 1) s_P[B] = run;
  __syncthreads();
}

// context_prefix from the staged lengths, for the rare rebuild after the grid
// wait: kept out of line so that it costs the kernels no registers.
__device__ __noinline__ void context_prefix_again(const DecodeArgs& a, int* s_P, int* s_ctx, int* s_warp_sum,
                                                  int nthreads) {
  context_prefix(a, a.context_lens, s_P, s_ctx, s_warp_sum, nthreads, false);
}

// After the grid wait: do the lengths this CTA read before the wait (s_ctx)
// still hold?  Each thread re-reads its share of context_lens from L2 (the
// previous kernels' writes are visible now) and the CTA votes; the result is
// the same in every thread.  With `flag`, out-of-range lengths are flagged
// here, from the values the kernel finally uses.
__device__ __forceinline__ bool context_changed(const DecodeArgs& a, const int* s_ctx, int nthreads, bool flag) {
  const int tid = threadIdx.x, B = a.num_seqs;
  const int per = (B + nthreads - 1) / nthreads;
  const int lo = min(B, tid * per), hi = min(B, lo + per);
  int diff = 0;
  for (int b = lo; b < hi; ++b) diff |= clamp_context(__ldcg(a.context_lens + b), a.max_blocks, flag) != s_ctx[b];
  return __syncthreads_or(diff) != 0;
}

// F8: the pool holds E4M3 codes (D = 128 only); the query, output and the
// appended token's K/V stay fp16/bf16 and the append quantises in-kernel.
// Registers are capped so that two 4-warp merge CTAs (64 registers a thread)
// fit beside a decode CTA (8 warps x 192 registers) on an SM.
template <typename T, int D, bool F8 = false>
__global__ void __maxnreg__(F8 ? 168 : 192)
    decode_persistent_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                             const DecodeArgs a) {
  static_assert(!F8 || D == 128, "the E4M3 path is built for head_dim 128");
  using Tile = KvTile<D, F8>;
  using Shape = PersistentShape<D, F8>;
  using Attn = std::conditional_t<F8, WarpAttnE4M3<T>, WarpAttn<T, D>>;
  constexpr int NW = Shape::kWarps;
  constexpr int SW = Shape::kStages;
  constexpr int NPS = Shape::kBlocksPerStage;
  constexpr int kRowBytes = D * 2;  // one appended token's K (or V) row for one KV head (fp16/bf16)
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[NW][SW];
  __shared__ int4 s_desc[NW][SW];  // per stage: sequence, KV head, first block j, segment id | flags << 28
  __shared__ int s_prow[NW][SW];   // per stage: pool row of its last block (the fused append's target)
  __shared__ int s_warp_sum[NW];

  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* side = ring + Shape::kRingBytes;  // [NW][SW][K row, V row] of appended tokens
  int* s_P = reinterpret_cast<int*>(side + NW * SW * 2 * kRowBytes);
  int* s_ctx = s_P + a.num_seqs + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.num_seqs, Hkv = a.num_kv_heads, g = a.group;
  const bool fused_append = a.k_new != nullptr;

  // The merge kernel may launch now; it waits for this grid to complete.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (lane == 0) {
    for (int s = 0; s < SW; ++s) mbar_init(smem_u32(&full_bar[warp][s]), 1);
    fence_mbar_init();
  }
  // Inputs only (context lengths, and below the block tables and query rows)
  // are read before the wait for the previous kernel in the stream.  What is
  // read there is a guess: a previous kernel may still be writing the lengths
  // or tables (a serving loop that advances context_lens on the GPU), and
  // nothing makes its writes visible before the wait.  After the wait both
  // are read again and everything derived from them is rebuilt if they
  // changed (see below), so the guess only decides how early the first loads
  // can start.  Errors are flagged from the values read after the wait.
  context_prefix(a, a.pre_context_lens ? a.pre_context_lens : a.context_lens, s_P, s_ctx, s_warp_sum, NW * 32,
                 !a.recheck && blockIdx.x == 0);

  Partition part(Hkv * s_P[B], gridDim.x * NW);
  const int gw = blockIdx.x * NW + warp;

  // Sequence b, KV head kvh and block j of flattened block f: units are
  // ordered (b, kvh) and unit (b, kvh) holds blocks [Hkv*P[b] + kvh*nb, +nb).
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

  uint8_t* wring = ring + warp * SW * Shape::kStageBytes;
  uint8_t* wside = side + warp * SW * 2 * kRowBytes;
  const uint64_t policy = l2_evict_first_policy();
  if (lane == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }

  // Block tables: the prologue's source until the grid wait, then the staged
  // ones.  Read through L2 only (ld.global.cg), like the lengths.
  const int32_t* tables = a.pre_block_tables ? a.pre_block_tables : a.block_tables;
  bool after_wait = !a.recheck;  // block ids are flagged only from values known to be final

  // ---- issue side: current segment [seg_s, seg_e) and a 32-block window of it,
  // lane i describing block win_s + i (sequence, KV head, block j, table entry,
  // pool row).
  int seg, seg_s, seg_e;
  int win_s, win_e, ip;
  int wb = -1, wkvh = -1, wj = 0, wphys = -1, wrow = -kBlockSize;
  bool more = true;
  auto fill_window = [&]() {
    win_s = ip;
    win_e = min(seg_e, ip + 32);
    wb = -1; wkvh = -1; wj = 0; wphys = -1; wrow = -kBlockSize;
    if (win_s + lane < win_e) {
      int b, kvh, j;
      locate(win_s + lane, b, kvh, j);
      wb = b;
      wkvh = kvh;
      wj = j;
      wphys = __ldcg(tables + static_cast<int64_t>(b) * a.max_blocks + j);
      wrow = tile_row(wphys, kvh, a, after_wait);
      if (j == 0 || lane == 0)  // a unit starts here: bring its query rows into L2
        prefetch_l2_bulk(static_cast<const T*>(a.q) + (static_cast<int64_t>(b) * Hkv + kvh) * g * D,
                         static_cast<uint32_t>(g * D * sizeof(T)));
    }
  };
  // Start on this warp's static head segment.
  auto start_head = [&]() {
    part.head(gw, seg_s, seg_e);
    seg = gw;
    ip = win_s = win_e = seg_s;
    more = true;
    if (ip < seg_e) fill_window();
  };
  // Next window: the rest of this segment, else the next claimed chunk.
  auto advance = [&]() {
    if (ip < seg_e) {
      fill_window();
      return;
    }
    if (part.nchunks == 0) {  // all head: nothing to claim, the counters stay untouched
      more = false;
      return;
    }
    while (true) {
      int q = 0;
      if (lane == 0) q = atomicAdd(a.sched, 1);
      q = __shfl_sync(0xffffffffu, q, 0);
      if (q >= part.num_chunks()) {
        more = false;
        // The last warp to run out of chunks resets the counters for the next call.
        if (lane == 0 && atomicAdd(a.sched + 1, 1) == part.nwarps - 1) {
          a.sched[0] = 0;
          a.sched[1] = 0;
        }
        return;
      }
      int s, e;
      part.chunk(q / part.nwarps, q % part.nwarps, s, e);
      if (e > s) {
        seg = part.nwarps + q;
        seg_s = s;
        seg_e = e;
        ip = s;
        fill_window();
        return;
      }
    }
  };

  int issued = 0, consumed = 0;
  int st_i = 0;                  // stage the next issue fills
  int st_c = 0, ph_c = 0;        // stage the next consume reads, and its phase parity
  // Fill free stages of the ring.  With may_advance false the issue stops at
  // the end of the current window: no chunk is claimed from the counter.
  auto issue_stages = [&](bool may_advance) {
    while (more && issued - consumed < SW) {
      if (ip == win_e) {
        if (!may_advance) break;
        advance();
        if (!more) break;
      }
      const int src = ip - win_s;
      const int b = __shfl_sync(0xffffffffu, wb, src);
      const int kvh = __shfl_sync(0xffffffffu, wkvh, src);
      const int j = __shfl_sync(0xffffffffu, wj, src);
      const int row = __shfl_sync(0xffffffffu, wrow, src);
      int n = 1, row2 = row;
      if constexpr (NPS == 2) {
        // Take the next block too when it is in this window (so in this
        // segment) and belongs to the same unit.
        const int src2 = src + 1 < 32 ? src + 1 : src;
        const int b2 = __shfl_sync(0xffffffffu, wb, src2);
        const int kvh2 = __shfl_sync(0xffffffffu, wkvh, src2);
        const int r2 = __shfl_sync(0xffffffffu, wrow, src2);
        if (ip + 1 < win_e && b2 == b && kvh2 == kvh) {
          n = 2;
          row2 = r2;
        }
      }
      if (lane == 0) {
        const bool unit_last = j + n == (s_ctx[b] + kBlockSize - 1) / kBlockSize;
        const int flags = (ip == seg_s ? 1 : 0) | (ip + n == seg_e ? 2 : 0) | ((n - 1) << 2);
        s_desc[warp][st_i] = make_int4(b, kvh, j, seg | (flags << 28));
        s_prow[warp][st_i] = row2;
        fence_proxy_async_smem();  // earlier generic accesses of this stage come before the refill
        const uint32_t bar = smem_u32(&full_bar[warp][st_i]);
        const uint32_t stage = smem_u32(wring + st_i * Shape::kStageBytes);
        const int64_t unit = static_cast<int64_t>(b) * Hkv + kvh;
        if (fused_append && unit_last) {
          // The block that receives this step's token: fetch the token's K and V rows too.
          mbar_arrive_expect_tx(bar, n * Tile::kStageBytes + 2 * kRowBytes);
          const uint32_t sd = smem_u32(wside + st_i * 2 * kRowBytes);
          bulk_load(sd, static_cast<const T*>(a.k_new) + unit * D, kRowBytes, bar);
          bulk_load(sd + kRowBytes, static_cast<const T*>(a.v_new) + unit * D, kRowBytes, bar);
        } else {
          mbar_arrive_expect_tx(bar, n * Tile::kStageBytes);
        }
        issue_tiles<D, F8>(stage, bar, &tmap_k, &tmap_v, row, policy);
        if (NPS == 2 && n == 2) issue_tiles<D, F8>(stage + Tile::kStageBytes, bar, &tmap_k, &tmap_v, row2, policy);
      }
      ++issued;
      ip += n;
      st_i = st_i + 1 == SW ? 0 : st_i + 1;
    }
  };
  // Wait for every issued stage and drop it (bounded; false on a timeout).
  auto drain = [&]() -> bool {
    for (; consumed < issued; ++consumed) {
      if (!mbar_wait(smem_u32(&full_bar[warp][st_c]), ph_c)) return false;
      if (++st_c == SW) {
        st_c = 0;
        ph_c ^= 1;
      }
    }
    return true;
  };

  // First window of the head (block-table and query inputs only), then wait:
  // from here on this grid reads the cache and writes the workspace and out,
  // which the previous kernels in the stream (append, merge) touch.  Before
  // the wait, the tiles of the first stages are only prefetched into L2: a
  // prefetch moves no data into this grid's view, and the loads after the
  // wait see every earlier write, so they just find the lines in L2.
  start_head();
  if (lane < SW * NPS && win_s + lane < win_e && wrow >= 0) {
    constexpr int kCacheRowBytes = F8 ? D : 2 * D;
    const int64_t off = static_cast<int64_t>(wrow) * kCacheRowBytes;
    prefetch_l2_bulk(static_cast<const uint8_t*>(a.k_cache_w) + off, Tile::kTileBytes);
    prefetch_l2_bulk(static_cast<const uint8_t*>(a.v_cache_w) + off, Tile::kTileBytes);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  tables = a.block_tables;
  after_wait = true;

  // The first stages go out on the prologue's reading of the inputs; then the
  // lengths (CTA vote) and this warp's first window of table entries are read
  // again.  If either changed, the stages are dropped and the partition and
  // window are rebuilt from the values read now: all CTAs then agree, since
  // they all read the same values after the wait.  Otherwise the first
  // window's block ids are checked (flagged) here.
  //
  // With at most kWarpChecked sequences every warp re-reads all the lengths
  // itself (lane-strided) and compares them once its first stage has landed,
  // so their latency hides under that load and no CTA barrier is needed: all
  // warps read the same values, so they all reach the same verdict.  Larger
  // batches compare at once with a CTA vote.
  issue_stages(false);
  bool ok = true;
  if (a.recheck) {
    constexpr int kHeld = 4;
    constexpr int kWarpChecked = 32 * kHeld;
    const bool warp_check = B <= kWarpChecked;
    int held[kHeld];
#pragma unroll
    for (int k = 0; k < kHeld; ++k)
      held[k] = warp_check && lane + 32 * k < B ? __ldcg(a.context_lens + lane + 32 * k) : 0;
    const bool in_window = win_s + lane < win_e;
    const int tv = in_window ? __ldcg(tables + static_cast<int64_t>(wb) * a.max_blocks + wj) : wphys;
    if (warp_check && issued > consumed) ok = mbar_wait(smem_u32(&full_bar[warp][st_c]), ph_c);
    bool lens_changed;
    if (warp_check) {
      bool d = false;
      const bool flag = blockIdx.x == 0 && warp == 0;
#pragma unroll
      for (int k = 0; k < kHeld; ++k)
        if (lane + 32 * k < B) d |= clamp_context(held[k], a.max_blocks, flag) != s_ctx[lane + 32 * k];
      lens_changed = __any_sync(0xffffffffu, d);
    } else {
      lens_changed = context_changed(a, s_ctx, NW * 32, blockIdx.x == 0);
    }
    const bool table_changed = __any_sync(0xffffffffu, !lens_changed && in_window && tv != wphys);
    if (lens_changed || table_changed) {
      if (ok) ok = drain();
      if (lens_changed) {
        // CTA-uniform: every warp takes this branch.  The barrier keeps the
        // rebuild from changing s_ctx while another warp still compares.
        __syncthreads();
        context_prefix_again(a, s_P, s_ctx, s_warp_sum, NW * 32);
        part = Partition(Hkv * s_P[B], gridDim.x * NW);
      }
      start_head();
    } else if (in_window) {
      tile_row(wphys, wkvh, a, true);
    }
  }

  // The lengths and block prefix this grid partitioned (known final now) go
  // to the merge of the same call: the grid's last warp, whose share (the
  // last one, often partial) leaves it time to spare, writes them and
  // releases the call's tag, which the merge acquires instead of reading the
  // lengths again after its own wait.
  if (a.epoch != 0 && blockIdx.x == gridDim.x - 1 && warp == NW - 1) {
    for (int b = lane; b < B; b += 32) a.pub[1 + b] = s_ctx[b];
    for (int b = lane; b <= B; b += 32) a.pub[1 + B + b] = s_P[b];
    __syncwarp();  // the lanes' stores come before lane 0's (cumulative) release
    if (lane == 0) st_release_gpu(a.pub, static_cast<int32_t>(a.epoch));
  }

  // ---- consume side
  Attn at;
  float unit_sl2 = a.scale_log2, unit_vs = 1.f;  // logit scale (log2 units) and output factor of the unit
  int unit_first_j = 0;
  bool seg_first_flush = true;
  while (ok) {
    issue_stages(true);
    __syncwarp();  // the descriptors written by lane 0 are visible to the warp
    if (consumed == issued) break;

    if (!mbar_wait(smem_u32(&full_bar[warp][st_c]), ph_c)) {  // timed out: flagged
      ok = false;
      break;
    }
    const int4 dsc = s_desc[warp][st_c];
    const int b = dsc.x, kvh = dsc.y, j = dsc.z, sid = dsc.w & 0x0FFFFFFF;
    const int flags = dsc.w >> 28;
    const bool first_of_seg = flags & 1, last_of_seg = flags & 2;
    const int n = 1 + ((flags >> 2) & 1);
    const int ctx = s_ctx[b];
    const int nb = (ctx + kBlockSize - 1) / kBlockSize;
    const int jl = j + n - 1;  // the stage's last block
    uint8_t* ks = wring + st_c * Shape::kStageBytes;
    if (fused_append && jl == nb - 1) {
      // Append: the token at position ctx - 1 goes into row r of block jl, in
      // the staged tile (for this step's attention) and in the pool.
      const int r = (ctx - 1) % kBlockSize;
      const int prow = s_prow[warp][st_c];
      uint8_t* lt = ks + (n - 1) * Tile::kStageBytes;  // K tile of block jl; its V tile follows
      const uint8_t* sd = wside + st_c * 2 * kRowBytes;
      constexpr int kChunksPerRow = D / 8;
      if constexpr (F8) {
        // Lanes 0-15 quantise 8 entries each of the K row, lanes 16-31 of the V row.
        const int v = lane >> 4, c8 = lane & 15;
        const uint4 val = *reinterpret_cast<const uint4*>(sd + v * kRowBytes + c8 * 16);
        const uint2 code = quantize8<T>(val, __ldg((v ? a.v_scale : a.k_scale) + kvh));
        uint8_t* tile = lt + v * Tile::kTileBytes;
        *reinterpret_cast<uint2*>(tile + r * 128 + (((c8 >> 1) ^ (r & 7)) << 4) + 8 * (c8 & 1)) = code;
        if (prow >= 0) {
          uint8_t* cache = static_cast<uint8_t*>(v ? a.v_cache_w : a.k_cache_w);
          *reinterpret_cast<uint2*>(cache + (static_cast<int64_t>(prow) + r) * D + 8 * c8) = code;
        }
      } else if (lane < 2 * kChunksPerRow) {
        const int v = lane / kChunksPerRow, c16 = lane % kChunksPerRow;
        const uint4 val = *reinterpret_cast<const uint4*>(sd + v * kRowBytes + c16 * 16);
        uint8_t* tile = lt + v * Tile::kTileBytes;
        *reinterpret_cast<uint4*>(tile + (c16 >> 3) * 2048 + r * 128 + (((c16 & 7) ^ (r & 7)) << 4)) = val;
        if (prow >= 0) {
          T* cache = static_cast<T*>(v ? a.v_cache_w : a.k_cache_w);
          *reinterpret_cast<uint4*>(cache + (static_cast<int64_t>(prow) + r) * D + c16 * 8) = val;
        }
      }
      __syncwarp();
    }
    if (first_of_seg || j == 0) {
      if (first_of_seg) seg_first_flush = true;
      unit_first_j = j;
      at.load_q(static_cast<const T*>(a.q) + (static_cast<int64_t>(b) * a.num_q_heads + kvh * g) * D, g, lane);
      at.reset();
      if constexpr (F8) {
        unit_sl2 = a.scale_log2 * __ldg(a.k_scale + kvh);
        unit_vs = __ldg(a.v_scale + kvh);
      }
    }
    const int valid = min(n * kBlockSize, ctx - j * kBlockSize);
    if constexpr (NPS == 2)
      at.block2(ks, ks + Tile::kTileBytes, ks + Tile::kStageBytes, ks + Tile::kStageBytes + Tile::kTileBytes, valid,
                unit_sl2, lane);
    else
      at.block(ks, ks + Tile::kTileBytes, valid, unit_sl2, lane);
    ++consumed;
    if (++st_c == SW) {
      st_c = 0;
      ph_c ^= 1;
    }

    if (jl == nb - 1 || last_of_seg) {
      // ---- the unit ends here or the segment does: write it out, or leave a piece for the merge
      at.finish_sums();
      const int gid = lane >> 2, c = lane & 3;
      const bool complete = unit_first_j == 0 && jl == nb - 1;
      const int64_t pbase = (static_cast<int64_t>(sid) * 2 + (seg_first_flush ? 0 : 1)) * kMaxGroup;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * c + e;
        if (h >= g) continue;
        const float l = e ? at.l1 : at.l0;
        if (complete) {
          T* orow = static_cast<T*>(a.out) + (static_cast<int64_t>(b) * a.num_q_heads + kvh * g + h) * D;
#pragma unroll
          for (int kk = 0; kk < Attn::kChunks; ++kk) {
            float v[8];
            at.chunk_values(e, kk, unit_vs / l, v);
            *reinterpret_cast<uint4*>(orow + Attn::chunk_dim(lane, kk)) = pack8<T>(v);
          }
        } else {
          float* prow = a.part_o + (pbase + h) * D;
#pragma unroll
          for (int kk = 0; kk < Attn::kChunks; ++kk) {
            float v[8];
            at.chunk_values(e, kk, unit_vs / l, v);
            float4* dst = reinterpret_cast<float4*>(prow + Attn::chunk_dim(lane, kk));
            dst[0] = make_float4(v[0], v[1], v[2], v[3]);
            dst[1] = make_float4(v[4], v[5], v[6], v[7]);
          }
          if (gid == 0) a.part_lse[pbase + h] = (e ? at.m1 : at.m0) + log2f(l);
        }
      }
      seg_first_flush = false;
    }
  }
  if (!ok && lane == 0) {
    // A wait gave up: let this warp's copies in flight land before the CTA exits.
    for (int i = consumed; i < issued; ++i) {
      mbar_wait(smem_u32(&full_bar[warp][st_c]), ph_c);
      if (++st_c == SW) {
        st_c = 0;
        ph_c ^= 1;
      }
    }
  }
}

// Merge of the pieces the persistent kernel left.  A CTA of kMergeWarps warps
// takes kMergeWarps (sequence, query head) rows at a time, one warp per row;
// or, COOP, one row at a time, its warps splitting the row's pieces between
// them and combining their partial results through shared memory (for long
// units cut into many pieces, which one warp would fold in a long serial
// chain).
// Units wholly inside one segment were written by the decode kernel; an empty
// context gives a zero row.  Everything that depends only on the inputs (the
// block prefix of the contexts, and the plan of the CTA's first row with its
// first batch of candidate pieces) is computed before griddepcontrol.wait,
// while the decode grid is still running; after it, unpublished lengths are
// checked again and the partials are read.  The unit's blocks [U, U+nb)
// overlap shares w0..w1 of 5 segments each; lanes test those candidates in
// parallel, the overlapping ones are compacted into a list, and their rows
// are accumulated with independent loads, up to kBatch pieces per round trip
// (6 in the small warp-per-row CTAs, which then need no spills).  Small CTAs
// (4 warps at <= 64 registers, 80 for COOP) fit two beside a decode CTA.
// WIDE (a warp per row, 16 pieces per round trip, <= 128 registers, one
// beside a decode CTA) is for units cut into many pieces, whose rows would
// otherwise take two round trips.
constexpr int kMergeWarps = 4;

template <typename T, int D, bool COOP, bool WIDE = false>
__global__ void __launch_bounds__(kMergeWarps * 32, COOP ? 6 : WIDE ? 4 : 8)
    merge_persistent_kernel(const DecodeArgs a, int32_t nwarps) {
  static_assert(!(COOP && WIDE), "WIDE is a warp-per-row variant");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kPer = D / 32;

  extern __shared__ int merge_smem[];
  __shared__ int s_warp_sum[kMergeWarps];
  __shared__ int64_t s_row[kMergeWarps][32];
  __shared__ float s_w[kMergeWarps][32];
  __shared__ float s_ml[COOP ? kMergeWarps : 1][2];
  __shared__ __align__(16) float s_o[COOP ? kMergeWarps : 1][COOP ? D : 4];
  int* s_P = merge_smem;
  int* s_ctx = s_P + a.num_seqs + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kThreads = kMergeWarps * 32;
  // Before its wait the merge needs the lengths and the block prefix the
  // decode grid partitioned.  When the decode grid publishes them (device
  // inputs, tag != 0) every thread acquires the call's tag, then takes the
  // published values: final by construction, so nothing is read again after
  // the wait.  Otherwise the lengths are read before the wait (host-written
  // inputs are final; device inputs are then checked again after the wait and
  // the prefix rebuilt if they changed).
  bool published = false;
  if (a.recheck && a.epoch != 0) {
    // One thread polls, backing off so that the merge CTAs waiting beside the
    // decode grid do not load the memory system; its acquire and the CTA
    // barrier after it order every thread's reads of the published values.
    const int32_t tag = static_cast<int32_t>(a.epoch);
    __shared__ int s_got;
    if (threadIdx.x == 0) {
      const unsigned long long t0 = global_ns();
      bool got = ld_acquire_gpu(a.pub) == tag;
      while (!got && global_ns() - t0 < kWaitLimitNs) {
        __nanosleep(256);
        got = ld_acquire_gpu(a.pub) == tag;
      }
      s_got = got;
    }
    __syncthreads();
    published = s_got != 0;
  }
  if (published) {
    for (int b = threadIdx.x; b < a.num_seqs; b += kThreads) s_ctx[b] = __ldcg(a.pub + 1 + b);
    for (int b = threadIdx.x; b <= a.num_seqs; b += kThreads) s_P[b] = __ldcg(a.pub + 1 + a.num_seqs + b);
    __syncthreads();
  } else {
    context_prefix(a, a.pre_context_lens ? a.pre_context_lens : a.context_lens, s_P, s_ctx, s_warp_sum, kThreads,
                   false);
  }

  constexpr int rows_per_cta = COOP ? 1 : kMergeWarps;
  constexpr int wpr = kMergeWarps / rows_per_cta;  // warps per row
  const int sub = warp % wpr;                      // this warp's part of its row
  const int Hkv = a.num_kv_heads;
  const int rows = a.num_seqs * a.num_q_heads;
  // What the lengths fix for one row: its unit's blocks [U, Uend), whether
  // the decode kernel left it in pieces (work: the unit spans two or more
  // segments) or it is empty (zero_row), and its candidate segments, shares
  // w0.. of seg_per_share() segments each.
  struct RowPlan {
    int b, kvh, h, U, Uend, w0, ncand;
    bool work, zero_row;
  };
  auto plan_row = [&](const Partition& part, int row) -> RowPlan {
    RowPlan r{0, 0, 0, 0, 0, 0, 0, row < rows, false};
    int nb = 0;
    if (r.work) {
      r.b = row / a.num_q_heads;
      const int hq = row - r.b * a.num_q_heads;
      r.kvh = hq / a.group;
      r.h = hq - r.kvh * a.group;
      nb = (s_ctx[r.b] + kBlockSize - 1) / kBlockSize;
    }
    r.zero_row = r.work && nb == 0;
    if (r.zero_row) r.work = false;
    if (r.work) {
      r.U = Hkv * s_P[r.b] + r.kvh * nb;
      r.Uend = r.U + nb;
      int s, e;
      part.segment_of(r.U, s, e);
      if (e >= r.Uend) r.work = false;  // one segment: the decode kernel wrote it
    }
    if (r.work) {
      r.w0 = r.U / part.R;
      r.ncand = ((r.Uend - 1) / part.R - r.w0 + 1) * part.seg_per_share();
    }
    return r;
  };
  // Candidate c of a row: the row of its piece in the partials, or -1 when
  // that segment does not overlap the unit.
  auto piece = [&](const Partition& part, const RowPlan& r, int c) -> int64_t {
    const int kSegPerShare = part.seg_per_share();
    const int w = r.w0 + c / kSegPerShare, k = c % kSegPerShare;
    int s, e, sid;
    if (k == 0) {
      part.head(w, s, e);
      sid = w;
    } else {
      part.chunk(k - 1, w, s, e);
      sid = part.nwarps + (k - 1) * part.nwarps + w;
    }
    if (e <= s || e <= r.U || s >= r.Uend) return -1;
    return (static_cast<int64_t>(sid) * 2 + (r.U > s ? 1 : 0)) * kMaxGroup + r.h;
  };
  // Batch k of this warp's candidates, one per lane: candidate
  // sub + wpr * (32 k + lane), so that the row's warps (COOP) share even a
  // short candidate list.  The overlapping ones are compacted into
  // s_row[warp] (the result: their lanes).
  auto gather = [&](const Partition& part, const RowPlan& r, int k) -> unsigned {
    const int c = sub + wpr * (32 * k + lane);
    const int64_t pr = c < r.ncand ? piece(part, r, c) : -1;
    const unsigned valid = __ballot_sync(0xffffffffu, pr >= 0);
    if (pr >= 0) s_row[warp][__popc(valid & ((1u << lane) - 1))] = pr;
    return valid;
  };

  // The CTA's first row and its first batch of candidates depend on the
  // lengths only: planned before the wait (the partition arithmetic then runs
  // while the decode grid drains), so that after it the loads go out at once.
  // Device inputs without publication are checked after the wait and the plan
  // rebuilt if they changed.  Only the first batch's lane mask stays in a
  // register across the wait; each lane finds its own piece in s_row again.
  const int first_base = blockIdx.x * rows_per_cta;
  RowPlan r{};
  unsigned valid0 = 0;
  auto plan_first = [&]() {
    const Partition part(Hkv * s_P[a.num_seqs], nwarps);
    r = plan_row(part, first_base + warp / wpr);
    valid0 = r.work && sub < r.ncand ? gather(part, r, 0) : 0u;
  };
  plan_first();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!published && a.recheck && context_changed(a, s_ctx, kThreads, false)) {
    context_prefix(a, a.context_lens, s_P, s_ctx, s_warp_sum, kThreads, false);
    __syncwarp();
    plan_first();
  }

  // Every warp of the CTA runs the same number of iterations (barriers inside).
  for (int base_row = first_base; base_row < rows; base_row += gridDim.x * rows_per_cta) {
    const int row = base_row + warp / wpr;
    const bool first = base_row == first_base;
    const Partition part(Hkv * s_P[a.num_seqs], nwarps);
    if (!first) r = plan_row(part, row);
    const bool work = r.work, zero_row = r.zero_row;
    T* dst = static_cast<T*>(a.out) + static_cast<int64_t>(row) * D + lane * kPer;
    float m = -INFINITY, L = 0.f, o[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) o[k] = 0.f;
    if (work) {
      // Pieces are folded in with a running log-sum-exp, in batches of up to
      // 32 candidates (this warp's share of them); within a batch the
      // log-sum-exps and the partial rows are loaded together (one round
      // trip), at most kBatch rows in flight.
      constexpr int kBatch = WIDE ? 16 : COOP ? 8 : 6;
      for (int k = 0; sub + wpr * 32 * k < r.ncand; ++k) {
        unsigned valid;
        int rank;
        int64_t pr;
        if (first && k == 0) {
          valid = valid0;
          rank = __popc(valid & ((1u << lane) - 1));
          pr = (valid >> lane) & 1u ? s_row[warp][rank] : -1;
        } else {
          valid = gather(part, r, k);
          rank = __popc(valid & ((1u << lane) - 1));
          pr = (valid >> lane) & 1u ? s_row[warp][rank] : -1;
        }
        const float lse = pr >= 0 ? __ldcg(a.part_lse + pr) : -INFINITY;
        __syncwarp();
        const int cnt = __popc(valid);
        for (int i0 = 0; i0 < cnt; i0 += kBatch) {
          float v[kBatch][kPer];
#pragma unroll
          for (int i = 0; i < kBatch; ++i) {
            if (i0 + i < cnt) {
              const float* src = a.part_o + s_row[warp][i0 + i] * D + lane * kPer;
#pragma unroll
              for (int k = 0; k < kPer; k += 2) {
                const float2 x = __ldcg(reinterpret_cast<const float2*>(src + k));
                v[i][k] = x.x;
                v[i][k + 1] = x.y;
              }
            }
          }
          if (i0 == 0 && pr >= 0) s_w[warp][rank] = lse;  // the batch's log-sum-exps, by rank
          __syncwarp();
          float mb = m;
#pragma unroll
          for (int i = 0; i < kBatch; ++i)
            if (i0 + i < cnt) mb = fmaxf(mb, s_w[warp][i0 + i]);
          const float sc = exp2f(m - mb);  // m == mb == -inf cannot happen: a batch has a piece
          L *= sc;
#pragma unroll
          for (int k = 0; k < kPer; ++k) o[k] *= sc;
#pragma unroll
          for (int i = 0; i < kBatch; ++i) {
            if (i0 + i < cnt) {
              const float w = exp2f(s_w[warp][i0 + i] - mb);
              L += w;
#pragma unroll
              for (int k = 0; k < kPer; ++k) o[k] += w * v[i][k];
            }
          }
          m = mb;
        }
        __syncwarp();
      }
    }
    if (zero_row && sub == 0) {
#pragma unroll
      for (int k = 0; k < kPer; k += 2) *reinterpret_cast<uint32_t*>(dst + k) = 0u;
    }
    if constexpr (COOP) {
      // Combine the row's warps: (m, L, o) of each through shared memory.
      if (lane == 0) {
        s_ml[warp][0] = m;
        s_ml[warp][1] = L;
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) s_o[warp][lane * kPer + k] = o[k];
      __syncthreads();
      if (work && sub == 0) {
        float mt = m;
        for (int w = 1; w < wpr; ++w) mt = fmaxf(mt, s_ml[warp + w][0]);
        float Lt = 0.f, ot[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) ot[k] = 0.f;
        for (int w = 0; w < wpr; ++w) {
          const float mw = s_ml[warp + w][0];
          if (mw == -INFINITY) continue;  // that warp had no pieces
          const float sc = exp2f(mw - mt);
          Lt += sc * s_ml[warp + w][1];
#pragma unroll
          for (int k = 0; k < kPer; ++k) ot[k] += sc * s_o[warp + w][lane * kPer + k];
        }
        const float inv = 1.0f / Lt;
#pragma unroll
        for (int k = 0; k < kPer; k += 2)
          *reinterpret_cast<uint32_t*>(dst + k) = pack2<T>(ot[k] * inv, ot[k + 1] * inv);
      }
      __syncthreads();
    } else if (work) {
      const float inv = 1.0f / L;
#pragma unroll
      for (int k = 0; k < kPer; k += 2) *reinterpret_cast<uint32_t*>(dst + k) = pack2<T>(o[k] * inv, o[k + 1] * inv);
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
// w_s = 2^(lse_s - max lse), over the splits that hold at least one token.  A
// row no split saw (lse = -inf everywhere: a new token before position 0 of
// a multi-token call) is zero.
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
  const float* lse = lse_part + static_cast<int64_t>(row) * num_splits;
  float M = -INFINITY;
  for (int s = 0; s < nvalid; ++s) M = fmaxf(M, lse[s]);
  if (M > -INFINITY) {
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
