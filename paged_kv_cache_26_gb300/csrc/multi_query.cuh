// Paged decode attention for several new tokens per sequence (sm_103a).
//
// Speculative verification checks q_len draft tokens in one pass
// (youngju.dev "LLM サービング最適化完全ガイド", speculative decoding section), and
// chunked decode feeds several tokens of one sequence at once
// (design.babushkai.com "GPU推論の内部構造", section "KVキャッシュの台帳").  The
// q_len new tokens of sequence b sit at positions L - q_len .. L - 1 of its
// context (L = context_lens[b] counts them); token i attends to positions
// [0, L - q_len + i]: the cache before it plus the new tokens up to itself.
//
//  append_multi_kernel      -- each sequence's q_len new K/V rows into the slots
//                              of positions L - q_len .. L - 1 of its table.
//  decode_multi_query_kernel-- one CTA per (split, KV head, sequence).  A TMA
//                              producer warp streams the split's blocks through
//                              a ring; the consumer warps each own 16 (or, for
//                              at most 8 rows in all, 8) of the unit's
//                              g * q_len query rows and all of them read every
//                              staged block, so K/V leave HBM once for all the
//                              new tokens of the group.  Rows are ordered
//                              token-major (row r = token r / g, head r % g),
//                              the order of q in memory.  With more than 8 rows
//                              the query rows are the mma M dimension (16 per
//                              warp), unlike the one-token kernels.
// The split partials are combined by merge_split_kernel with q_len * Hq rows
// per sequence.
#pragma once

#include "paged_kv_kernels.cuh"

namespace pkv {

constexpr int kMaxQueryLen = 8;
constexpr int kQueryRowsPerWarp = 16;
constexpr int kMaxQueryWarps = kMaxGroup * kMaxQueryLen / kQueryRowsPerWarp;  // 4 consumer warps
constexpr int kMultiStages = 4;

// Token (b, i) of k_new / v_new ([B][q_len][Hkv][D]) goes to position
// context_lens[b] - q_len + i through the block table (nothing for a negative
// position).  One thread per 16-byte chunk of one row.
__global__ void append_multi_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                    const int32_t* __restrict__ block_tables,
                                    const int32_t* __restrict__ context_lens, int32_t num_seqs, int32_t q_len,
                                    int32_t max_blocks, int32_t num_kv_heads, int32_t chunks_per_row,
                                    int32_t num_blocks, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * chunks_per_row;
  const int64_t total = per_token * num_seqs * q_len;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = idx / per_token;  // b * q_len + i
    const int b = static_cast<int>(tok / q_len), i = static_cast<int>(tok - static_cast<int64_t>(b) * q_len);
    const int L = context_lens[b];
    if (L > max_blocks * kBlockSize) {
      flag_error(kErrContext);
      continue;
    }
    const int pos = L - q_len + i;
    if (pos < 0) continue;
    const int32_t blk = block_tables[static_cast<int64_t>(b) * max_blocks + pos / kBlockSize];
    if (blk < 0 || blk >= num_blocks) {
      flag_error(kErrBlockId);
      continue;
    }
    const int64_t within = idx - tok * per_token;
    const int64_t head = within / chunks_per_row;
    const int64_t chunk = within - head * chunks_per_row;
    const int64_t dst =
        ((static_cast<int64_t>(blk) * num_kv_heads + head) * kBlockSize + pos % kBlockSize) * chunks_per_row + chunk;
    k_cache[dst] = k_new[idx];
    v_cache[dst] = v_new[idx];
  }
}

// WarpAttn with one query row per mma column taken from anywhere (the rows of
// a warp are (token, head) pairs, not consecutive heads) and a causal limit per
// column: column 2c (2c + 1) sees the first vc0 (vc1) tokens of a block.  A
// column with no visible token so far keeps m = -inf and l = 0.
template <typename T, int D>
struct WarpAttnCausal : WarpAttn<T, D> {
  using Base = WarpAttn<T, D>;
  using Shape = typename Base::Shape;
  using Base::acc;
  using Base::l0;
  using Base::l1;
  using Base::m0;
  using Base::m1;
  using Base::qf;

  // This lane's share of query row gid, whose first element is at rowp (null:
  // a padding row of zeros).
  __device__ __forceinline__ void load_q_row(const T* rowp, int lane) {
    const int c = lane & 3;
#pragma unroll
    for (int qc = 0; qc < Shape::kQChunks; ++qc) {
      const int chunk = 2 * c + (qc & 1) + 8 * (qc >> 1);
      qf[qc] = rowp ? __ldg(reinterpret_cast<const uint4*>(rowp) + chunk) : make_uint4(0, 0, 0, 0);
    }
  }

  // One block: V rows at or past valid_v read as zeros; token t of the block
  // is visible to column 2c (2c + 1) when t < vc0 (vc1).
  __device__ __forceinline__ void block_causal(const uint8_t* ks, const uint8_t* vs, int valid_v, int vc0, int vc1,
                                               float scale_log2, int lane) {
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
    if (gid >= vc0) x0 = -INFINITY;
    if (gid >= vc1) x1 = -INFINITY;
    if (gid + 8 >= vc0) x2 = -INFINITY;
    if (gid + 8 >= vc1) x3 = -INFINITY;
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float r0 = mn0 == -INFINITY ? 0.f : mn0, r1 = mn1 == -INFINITY ? 0.f : mn1;  // nothing visible yet
    const float al0 = exp2f(m0 - r0), al1 = exp2f(m1 - r1);
    m0 = mn0;
    m1 = mn1;
    uint32_t b0, b1, c0 = 0, c1 = 0;
    this->weights(exp2f(x0 - r0), exp2f(x1 - r1), exp2f(x2 - r0), exp2f(x3 - r1), al0, al1, b0, b1, c0, c1);

    uint4 vr[4][Shape::kBoxes];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int row = 2 * c + (rr & 1) + 8 * (rr >> 1);
#pragma unroll
      for (int a = 0; a < Shape::kBoxes; ++a)
        vr[rr][a] = *reinterpret_cast<const uint4*>(vs + a * 2048 + row * 128 + ((gid ^ (row & 7)) << 4));
      if (row >= valid_v) {
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
};

// ldmatrix: four 8x8 matrices of 16-bit elements from shared memory; lane l
// supplies the address of row l % 8 of matrix l / 8, and r[m] receives this
// lane's part of matrix m (row lane / 4, elements 2 (lane % 4) and + 1; with
// .trans, of the transposed matrix).
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// One warp's attention state for 16 query rows (rows gid and gid + 8 of the
// mma layout, gid = lane / 4, c = lane % 4) over the blocks of one unit.
//  * S = Q K^T per block: M = the 16 rows, N = 2 tiles of 8 tokens, K = head_dim
//    in steps of 16; K fragments come from the swizzled tile with ldmatrix.
//  * The score accumulators are already the A fragments of P V (rows gid,
//    gid + 8; tokens 2c, 2c+1 and 2c+8, 2c+9), so P never leaves registers.
//  * O = P V: M = the 16 rows, N = head_dim in tiles of 8, K = the 16 tokens;
//    V fragments come with ldmatrix.trans.  The lane holds O for rows gid and
//    gid + 8, columns 8 nd + 2c and + 1.
//  * Each row has its own causal limit: the first vc0 (vc1) tokens of a block
//    are visible to row gid (gid + 8).  A row with nothing visible so far keeps
//    m = -inf and l = 0; O is rescaled only when a row's maximum grows.
//  * bf16 weights enter P V as two bf16 terms, p = hi + lo (fp16: one term).
template <typename T, int D>
struct WarpAttnRows {
  static constexpr int kKSteps = D / 16;
  static constexpr int kNTiles = D / 8;
  uint32_t qa[kKSteps][4];
  float o[kNTiles][4];
  float m0, m1, l0, l1;

  __device__ __forceinline__ void reset() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int i = 0; i < kNTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  }

  // rows gid (row0) and gid + 8 (row1) of q; null: a padding row of zeros.
  __device__ __forceinline__ void load_q(const T* row0, const T* row1, int lane) {
    const int c = lane & 3;
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk) {
      const int d = 16 * kk + 2 * c;
      qa[kk][0] = row0 ? __ldg(reinterpret_cast<const uint32_t*>(row0 + d)) : 0u;
      qa[kk][1] = row1 ? __ldg(reinterpret_cast<const uint32_t*>(row1 + d)) : 0u;
      qa[kk][2] = row0 ? __ldg(reinterpret_cast<const uint32_t*>(row0 + d + 8)) : 0u;
      qa[kk][3] = row1 ? __ldg(reinterpret_cast<const uint32_t*>(row1 + d + 8)) : 0u;
    }
  }

  __device__ __forceinline__ void block(uint32_t ks, uint32_t vs, int valid_v, int vc0, int vc1, float scale_log2,
                                        int lane) {
    const int c = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;  // the matrix and row this lane addresses
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk) {
      // matrices: (tokens 0-7, d lo), (tokens 0-7, d hi), (tokens 8-15, d lo), (tokens 8-15, d hi)
      const int token = 8 * (mi >> 1) + rr;
      const int chunk = 2 * (kk & 3) + (mi & 1);
      uint32_t kb[4];
      ldmatrix_x4(ks + (kk >> 2) * 2048 + token * 128 + ((chunk ^ rr) << 4), kb);
      mma16816<T>(s[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], kb[0], kb[1]);
      mma16816<T>(s[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], kb[2], kb[3]);
    }
    float x[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 8 * nt + 2 * c + e;
        x[nt][e] = t < vc0 ? s[nt][e] * scale_log2 : -INFINITY;
        x[nt][2 + e] = t < vc1 ? s[nt][2 + e] * scale_log2 : -INFINITY;
      }
    }
    float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
    float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    if (__any_sync(0xffffffffu, mn0 > m0 || mn1 > m1)) {
      const float al0 = mn0 > m0 ? exp2f(m0 - mn0) : 1.f, al1 = mn1 > m1 ? exp2f(m1 - mn1) : 1.f;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int nd = 0; nd < kNTiles; ++nd) {
        o[nd][0] *= al0;
        o[nd][1] *= al0;
        o[nd][2] *= al1;
        o[nd][3] *= al1;
      }
      m0 = mn0;
      m1 = mn1;
    }
    const float r0 = m0 == -INFINITY ? 0.f : m0, r1 = m1 == -INFINITY ? 0.f : m1;  // nothing visible yet
    float p[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      p[nt][0] = exp2f(x[nt][0] - r0);
      p[nt][1] = exp2f(x[nt][1] - r0);
      p[nt][2] = exp2f(x[nt][2] - r1);
      p[nt][3] = exp2f(x[nt][3] - r1);
    }
    uint32_t ph[4], pl[4] = {0u, 0u, 0u, 0u};
    ph[0] = pack2<T>(p[0][0], p[0][1]);  // row gid, tokens 2c, 2c+1
    ph[1] = pack2<T>(p[0][2], p[0][3]);  // row gid + 8
    ph[2] = pack2<T>(p[1][0], p[1][1]);  // row gid, tokens 2c+8, 2c+9
    ph[3] = pack2<T>(p[1][2], p[1][3]);
    if constexpr (MmaKind<T>::kBf16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 h = unpack2<T>(ph[i]);
        const int nt = i >> 1, e = (i & 1) * 2;
        pl[i] = pack2<T>(p[nt][e] - h.x, p[nt][e + 1] - h.y);
      }
      l0 += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
      l1 += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
    } else {
      const float2 a = unpack2<T>(ph[0]), b = unpack2<T>(ph[1]), cc = unpack2<T>(ph[2]), dd = unpack2<T>(ph[3]);
      l0 += (a.x + a.y) + (cc.x + cc.y);  // the rounded weights the product uses
      l1 += (b.x + b.y) + (dd.x + dd.y);
    }
    // V rows at or past valid_v read as zeros (never 0 * NaN).
    const uint32_t keep0 = (2 * c < valid_v ? 0x0000FFFFu : 0u) | (2 * c + 1 < valid_v ? 0xFFFF0000u : 0u);
    const uint32_t keep1 = (2 * c + 8 < valid_v ? 0x0000FFFFu : 0u) | (2 * c + 9 < valid_v ? 0xFFFF0000u : 0u);
#pragma unroll
    for (int pr = 0; pr < kNTiles / 2; ++pr) {
      // matrices: (tokens 0-7, d tile 2pr), (tokens 8-15, 2pr), (0-7, 2pr+1), (8-15, 2pr+1)
      const int nd = 2 * pr + (mi >> 1);
      const int token = 8 * (mi & 1) + rr;
      uint32_t vb[4];
      ldmatrix_x4_trans(vs + (nd >> 3) * 2048 + token * 128 + (((nd & 7) ^ rr) << 4), vb);
      if (valid_v < kBlockSize) {
        vb[0] &= keep0;
        vb[1] &= keep1;
        vb[2] &= keep0;
        vb[3] &= keep1;
      }
      mma16816<T>(o[2 * pr], ph[0], ph[1], ph[2], ph[3], vb[0], vb[1]);
      mma16816<T>(o[2 * pr + 1], ph[0], ph[1], ph[2], ph[3], vb[2], vb[3]);
      if constexpr (MmaKind<T>::kBf16) {
        mma16816<T>(o[2 * pr], pl[0], pl[1], pl[2], pl[3], vb[0], vb[1]);
        mma16816<T>(o[2 * pr + 1], pl[0], pl[1], pl[2], pl[3], vb[2], vb[3]);
      }
    }
  }

  // Complete the row sums (each lane summed its own columns).
  __device__ __forceinline__ void finish_sums() {
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }
};

// args.num_q_heads = Hq; q / out are T[B][q_len][Hq][D]; split partials are
// indexed by row = (b * q_len + i) * Hq + h (args.num_splits, args.split_blocks).
// ROWS: query rows in the mma M dimension, 16 per warp (WarpAttnRows), for
// more than 8 rows per KV head; else 8 rows per warp in the N dimension
// (WarpAttnCausal), which pads less when the rows are few.
template <typename T, int D, int S, bool ROWS>
__global__ void __launch_bounds__((ROWS ? kMaxQueryWarps : 1) * 32 + 32)
    decode_multi_query_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                              const DecodeArgs args, int32_t q_len) {
  using Shape = TileShape<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[S];
  __shared__ __align__(8) uint64_t empty_bar[S];
  __shared__ int s_abort;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int NQ = static_cast<int>(blockDim.x >> 5) - 1;  // consumer warps; warp NQ produces
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = args.group, Hq = args.num_q_heads, n = q_len;
  const int nrows = g * n;  // query rows of this (sequence, KV head)

  const int ctx = clamped_context(args.context_lens, b, args.max_blocks, threadIdx.x == 0 && split == 0);
  const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
  const int blk0 = split * args.split_blocks;
  const int nb = min(nblk, blk0 + args.split_blocks) - blk0;
  auto row_index = [&](int r) -> int64_t {  // output row of query row r
    return (static_cast<int64_t>(b) * n + r / g) * Hq + kvh * g + r % g;
  };

  if (nb <= 0) {
    // Empty split.  In one pass this is an empty context: zero rows.
    if (args.num_splits == 1) {
      for (int idx = threadIdx.x; idx < nrows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx - r * D;
        static_cast<T*>(args.out)[row_index(r) * D + d] = T(0.0f);
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), NQ);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NQ) {
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
    // No copy may still be landing in shared memory when the CTA exits.
    if (lane == 0) {
      for (int i = max(0, issued - S); i < issued; ++i) mbar_wait(smem_u32(&full_bar[i % S]), (i / S) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int gid = lane >> 2, c = lane & 3;
  if constexpr (ROWS) {
    const int ra = kQueryRowsPerWarp * warp + gid, rb = ra + 8;  // this lane's two rows
    WarpAttnRows<T, D> at;
    {
      const T* q = static_cast<const T*>(args.q);
      at.load_q(ra < nrows ? q + row_index(ra) * D : nullptr, rb < nrows ? q + row_index(rb) * D : nullptr, lane);
    }
    at.reset();
    // Last position each row attends to (-1: a padding row).
    const int lim_a = ra < nrows ? ctx - n + ra / g : -1;
    const int lim_b = rb < nrows ? ctx - n + rb / g : -1;
    for (int i = 0; i < nb; ++i) {
      if (*reinterpret_cast<volatile int*>(&s_abort)) return;
      const int st = i % S;
      if (!mbar_wait(smem_u32(&full_bar[st]), (i / S) & 1)) {
        s_abort = 1;
        return;
      }
      const int t0 = (blk0 + i) * kBlockSize;
      const int vc0 = max(0, min(kBlockSize, lim_a + 1 - t0));
      const int vc1 = max(0, min(kBlockSize, lim_b + 1 - t0));
      const uint32_t ks = smem_u32(smem + st * Shape::kStageBytes);
      at.block(ks, ks + Shape::kTileBytes, min(kBlockSize, ctx - t0), vc0, vc1, args.scale_log2, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));  // this warp is done with the stage
    }
    at.finish_sums();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = half ? rb : ra;
      if (r >= nrows) continue;
      const float l = half ? at.l1 : at.l0;
      const float inv = l > 0.f ? 1.0f / l : 0.f;  // no visible token: a zero row
      const int64_t orow = row_index(r);
      if (args.num_splits == 1) {
        T* dst = static_cast<T*>(args.out) + orow * D + 2 * c;
#pragma unroll
        for (int nd = 0; nd < WarpAttnRows<T, D>::kNTiles; ++nd)
          *reinterpret_cast<uint32_t*>(dst + 8 * nd) =
              pack2<T>(at.o[nd][2 * half] * inv, at.o[nd][2 * half + 1] * inv);
      } else {
        const int64_t prow = orow * args.num_splits + split;
        float* dst = args.part_o + prow * D + 2 * c;
#pragma unroll
        for (int nd = 0; nd < WarpAttnRows<T, D>::kNTiles; ++nd)
          *reinterpret_cast<float2*>(dst + 8 * nd) =
              make_float2(at.o[nd][2 * half] * inv, at.o[nd][2 * half + 1] * inv);
        if (c == 0) args.part_lse[prow] = l > 0.f ? (half ? at.m1 : at.m0) + log2f(l) : -INFINITY;
      }
    }
  } else {
    WarpAttnCausal<T, D> at;
    {
      const int rq = 8 * warp + gid;  // the query row this lane loads
      at.load_q_row(rq < nrows ? static_cast<const T*>(args.q) + row_index(rq) * D : nullptr, lane);
    }
    at.reset();
    // Last position each of this lane's two columns attends to (-1: padding row).
    const int r0 = 8 * warp + 2 * c, r1 = r0 + 1;
    const int lim0 = r0 < nrows ? ctx - n + r0 / g : -1;
    const int lim1 = r1 < nrows ? ctx - n + r1 / g : -1;
    for (int i = 0; i < nb; ++i) {
      if (*reinterpret_cast<volatile int*>(&s_abort)) return;
      const int st = i % S;
      if (!mbar_wait(smem_u32(&full_bar[st]), (i / S) & 1)) {
        s_abort = 1;
        return;
      }
      const int t0 = (blk0 + i) * kBlockSize;
      const int vc0 = max(0, min(kBlockSize, lim0 + 1 - t0));
      const int vc1 = max(0, min(kBlockSize, lim1 + 1 - t0));
      const uint8_t* ks = smem + st * Shape::kStageBytes;
      at.block_causal(ks, ks + Shape::kTileBytes, min(kBlockSize, ctx - t0), vc0, vc1, args.scale_log2, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));  // this warp is done with the stage
    }
    at.finish_sums();
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = r0 + e;
      if (r >= nrows) continue;
      const float l = e ? at.l1 : at.l0;
      const float inv = l > 0.f ? 1.0f / l : 0.f;  // no visible token: a zero row
      const int64_t orow = row_index(r);
      if (args.num_splits == 1) {
        T* dst = static_cast<T*>(args.out) + orow * D;
#pragma unroll
        for (int kk = 0; kk < WarpAttn<T, D>::kChunks; ++kk) {
          float v[8];
          at.chunk_values(e, kk, inv, v);
          *reinterpret_cast<uint4*>(dst + WarpAttn<T, D>::chunk_dim(lane, kk)) = pack8<T>(v);
        }
      } else {
        const int64_t prow = orow * args.num_splits + split;
        float* dst = args.part_o + prow * D;
#pragma unroll
        for (int kk = 0; kk < WarpAttn<T, D>::kChunks; ++kk) {
          float v[8];
          at.chunk_values(e, kk, inv, v);
          float4* d4 = reinterpret_cast<float4*>(dst + WarpAttn<T, D>::chunk_dim(lane, kk));
          d4[0] = make_float4(v[0], v[1], v[2], v[3]);
          d4[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
        if (gid == 0) args.part_lse[prow] = l > 0.f ? (e ? at.m1 : at.m0) + log2f(l) : -INFINITY;
      }
    }
  }
}

}  // namespace pkv
