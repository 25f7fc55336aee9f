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
//  decode_multi_rows_kernel -- more than 8 query rows per KV head: one CTA per
//                              (split, KV head, sequence); a TMA producer warp
//                              streams the split's blocks through a ring and
//                              each consumer warp owns 16 of the unit's
//                              g * q_len query rows in the mma M dimension, so
//                              K/V leave HBM once for all the new tokens of
//                              the group.  Rows are ordered token-major (row
//                              r = token r / g, head r % g), the order of q in
//                              memory.
//  decode_multi_query_kernel-- at most 8 rows: one consumer warp with the rows
//                              in the mma N dimension, as in the one-token
//                              kernels.
// The split partials are combined by merge_split_kernel with q_len * Hq rows
// per sequence.
#pragma once

#include "paged_kv_kernels.cuh"

namespace pkv {

constexpr int kMaxQueryLen = 8;
constexpr int kQueryRowsPerWarp = 16;
constexpr int kMaxQueryWarps = kMaxGroup * kMaxQueryLen / kQueryRowsPerWarp;  // 4 consumer warps
constexpr int kMultiStages = 4;   // ring stages of one block
constexpr int kRowStages2 = 3;    // ring stages of two blocks (the 64-row kernel)

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


// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32: relative error
// about 2^-22; 2^-inf = 0; results below 2^-126 flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// mma.sync m16n8k16 (fp32 accumulate) as a plain register operation, free to
// be interleaved with the shared-memory loads around it.
template <typename T>
__device__ __forceinline__ void mma_rr(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                       uint32_t b0, uint32_t b1) {
  if constexpr (MmaKind<T>::kBf16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// One warp's attention state for 16 query rows (rows gid and gid + 8 of the
// mma layout, gid = lane / 4, c = lane % 4) over the blocks of one unit, NSUB
// consecutive 16-token blocks per softmax step.
//  * S = Q K^T per step: M = the 16 rows, N = 8-token tiles, K = head_dim in
//    steps of 16 (2 NSUB independent accumulator chains).  Q fragments are
//    staged once in shared memory (one 16-byte load per k-step, so they cost
//    no registers); K fragments come from the swizzled tile with ldmatrix.
//  * The score accumulators are already the A fragments of P V (rows gid,
//    gid + 8; tokens 2c, 2c+1 and 2c+8, 2c+9 of each block), so P never
//    leaves registers.  O = P V: M = the rows, N = head_dim in tiles of 8,
//    K = the tokens; V fragments come with ldmatrix.trans.  The lane holds O
//    for rows gid and gid + 8, columns 8 nd + 2c and + 1.
//  * Each row has its own causal limit: the first vc0 (vc1) tokens of a step
//    are visible to row gid (gid + 8); masks are applied only on steps that
//    some row of the warp does not see whole.  A row with nothing visible so
//    far keeps m = -inf and l = 0.
//  * Lazy reference maximum: a row's reference m (log2 units) moves only when
//    a step's maximum exceeds it by more than kLazy, so weights stay below
//    2^kLazy and O is rescaled in a few steps per unit; out = O / l and
//    lse = m + log2 l hold for any reference.
//  * Weights: hi = the weight rounded to T always enters P V.  For bf16 the
//    remainder lo = bf16(p - hi) enters as well in each step whose weights
//    carry more than kLoShare of a row's running sum after the step (any row
//    of the warp): every token holding more than that share of its row's
//    final weight is exact to about 2^-17, the others carry a rounding error
//    below 2^-9 of their own weight.  l sums the unrounded weights (bf16) or
//    the rounded ones (fp16, one term, 2^-11).  l is kept as the full row sum
//    (reduced over the lane quad every step).
template <typename T, int D, int NSUB>
struct WarpAttnRows {
  static constexpr int kKSteps = D / 16;
  static constexpr int kNTiles = D / 8;
  static constexpr int kTok = 16 * NSUB;
  static constexpr float kLazy = 8.f;
  static constexpr float kLoShare = 0.25f;
  float o[kNTiles][4];
  float m0, m1, l0, l1;

  __device__ __forceinline__ void reset() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int i = 0; i < kNTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  }

  // Store this lane's A fragments of rows gid (row0) and gid + 8 (row1) at
  // qs[kk * 32] (qs already offset by the lane); a null row is zeros.  With
  // `negate` the rows are stored negated (an exact sign flip), which lets a
  // negative softmax scale use the same maximum as a positive one.
  __device__ __forceinline__ static void stage_q(uint4* qs, const T* row0, const T* row1, bool negate, int lane) {
    const int c = lane & 3;
    const uint32_t flip = negate ? 0x80008000u : 0u;
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk) {
      const int d = 16 * kk + 2 * c;
      uint4 f;
      f.x = (row0 ? __ldg(reinterpret_cast<const uint32_t*>(row0 + d)) : 0u) ^ flip;
      f.y = (row1 ? __ldg(reinterpret_cast<const uint32_t*>(row1 + d)) : 0u) ^ flip;
      f.z = (row0 ? __ldg(reinterpret_cast<const uint32_t*>(row0 + d + 8)) : 0u) ^ flip;
      f.w = (row1 ? __ldg(reinterpret_cast<const uint32_t*>(row1 + d + 8)) : 0u) ^ flip;
      qs[kk * 32] = f;
    }
  }

  // O += P V over the step's blocks (block j's V tile at vs + j * sub_stride);
  // with LO the remainder weights too.  MASK: V rows at or past valid_v read
  // as zeros (never 0 * NaN).
  template <bool MASK, bool LO>
  __device__ __forceinline__ void pv(uint32_t vs, uint32_t sub_stride, const uint32_t (&ph)[NSUB][4],
                                     const uint32_t (&pl)[NSUB][4], int valid_v, int lane) {
    const int c = lane & 3, mi = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int pr = 0; pr < kNTiles / 2; ++pr) {
      // matrices: (tokens 0-7, d tile 2pr), (tokens 8-15, 2pr), (0-7, 2pr+1), (8-15, 2pr+1)
      const int nd = 2 * pr + (mi >> 1);
      const int token = 8 * (mi & 1) + rr;
#pragma unroll
      for (int j = 0; j < NSUB; ++j) {
        uint32_t vb[4];
        ldmatrix_x4_trans(vs + j * sub_stride + (nd >> 3) * 2048 + token * 128 + (((nd & 7) ^ rr) << 4), vb);
        if constexpr (MASK) {
          const int vv = valid_v - 16 * j;
          const uint32_t keep0 = (2 * c < vv ? 0x0000FFFFu : 0u) | (2 * c + 1 < vv ? 0xFFFF0000u : 0u);
          const uint32_t keep1 = (2 * c + 8 < vv ? 0x0000FFFFu : 0u) | (2 * c + 9 < vv ? 0xFFFF0000u : 0u);
          vb[0] &= keep0;
          vb[1] &= keep1;
          vb[2] &= keep0;
          vb[3] &= keep1;
        }
        mma_rr<T>(o[2 * pr], ph[j][0], ph[j][1], ph[j][2], ph[j][3], vb[0], vb[1]);
        mma_rr<T>(o[2 * pr + 1], ph[j][0], ph[j][1], ph[j][2], ph[j][3], vb[2], vb[3]);
        if constexpr (LO) {
          mma_rr<T>(o[2 * pr], pl[j][0], pl[j][1], pl[j][2], pl[j][3], vb[0], vb[1]);
          mma_rr<T>(o[2 * pr + 1], pl[j][0], pl[j][1], pl[j][2], pl[j][3], vb[2], vb[3]);
        }
      }
    }
  }

  // One step: block j's K tile at ks + j * sub_stride.  c2 = |scale| / ln 2.
  template <bool MASK>
  __device__ __forceinline__ void step(uint32_t ks, uint32_t vs, uint32_t sub_stride, const uint4* qs, int valid_v,
                                       int vc0, int vc1, float c2, int lane) {
    const int c = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    float s[2 * NSUB][4];
#pragma unroll
    for (int a = 0; a < 2 * NSUB; ++a) s[a][0] = s[a][1] = s[a][2] = s[a][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk) {
      const uint4 qf = qs[kk * 32];
      // matrices: (tokens 0-7, d lo), (tokens 0-7, d hi), (tokens 8-15, d lo), (tokens 8-15, d hi)
      const int token = 8 * (mi >> 1) + rr;
      const int chunk = 2 * (kk & 3) + (mi & 1);
#pragma unroll
      for (int j = 0; j < NSUB; ++j) {
        uint32_t kb[4];
        ldmatrix_x4(ks + j * sub_stride + (kk >> 2) * 2048 + token * 128 + ((chunk ^ rr) << 4), kb);
        mma_rr<T>(s[2 * j], qf.x, qf.y, qf.z, qf.w, kb[0], kb[1]);
        mma_rr<T>(s[2 * j + 1], qf.x, qf.y, qf.z, qf.w, kb[2], kb[3]);
      }
    }
    if constexpr (MASK) {
#pragma unroll
      for (int nt = 0; nt < 2 * NSUB; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 8 * nt + 2 * c + e;
          if (t >= vc0) s[nt][e] = -INFINITY;
          if (t >= vc1) s[nt][2 + e] = -INFINITY;
        }
    }
    float mx0 = fmaxf(s[0][0], s[0][1]), mx1 = fmaxf(s[0][2], s[0][3]);
#pragma unroll
    for (int nt = 1; nt < 2 * NSUB; ++nt) {
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    mx0 *= c2;  // c2 >= 0: the maximum of the scaled scores
    mx1 *= c2;
    const bool up0 = mx0 > m0 + kLazy, up1 = mx1 > m1 + kLazy;
    if (__any_sync(0xffffffffu, up0 || up1)) {
      const float al0 = up0 ? ex2(m0 - mx0) : 1.f, al1 = up1 ? ex2(m1 - mx1) : 1.f;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int nd = 0; nd < kNTiles; ++nd) {
        o[nd][0] *= al0;
        o[nd][1] *= al0;
        o[nd][2] *= al1;
        o[nd][3] *= al1;
      }
      if (up0) m0 = mx0;
      if (up1) m1 = mx1;
    }
    const float nr0 = m0 == -INFINITY ? 0.f : -m0, nr1 = m1 == -INFINITY ? 0.f : -m1;  // nothing visible yet
    float p[NSUB][2][4];
    uint32_t ph[NSUB][4], pl[NSUB][4];
    float ps0 = 0.f, ps1 = 0.f;  // this lane's part of the step's row sums
#pragma unroll
    for (int j = 0; j < NSUB; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        p[j][h][0] = ex2(fmaf(s[2 * j + h][0], c2, nr0));
        p[j][h][1] = ex2(fmaf(s[2 * j + h][1], c2, nr0));
        p[j][h][2] = ex2(fmaf(s[2 * j + h][2], c2, nr1));
        p[j][h][3] = ex2(fmaf(s[2 * j + h][3], c2, nr1));
      }
      ph[j][0] = pack2<T>(p[j][0][0], p[j][0][1]);  // row gid, tokens 2c, 2c+1
      ph[j][1] = pack2<T>(p[j][0][2], p[j][0][3]);  // row gid + 8
      ph[j][2] = pack2<T>(p[j][1][0], p[j][1][1]);  // row gid, tokens 2c+8, 2c+9
      ph[j][3] = pack2<T>(p[j][1][2], p[j][1][3]);
      pl[j][0] = pl[j][1] = pl[j][2] = pl[j][3] = 0u;
      if constexpr (MmaKind<T>::kBf16) {
        ps0 += (p[j][0][0] + p[j][0][1]) + (p[j][1][0] + p[j][1][1]);
        ps1 += (p[j][0][2] + p[j][0][3]) + (p[j][1][2] + p[j][1][3]);
      } else {
        const float2 a = unpack2<T>(ph[j][0]), b = unpack2<T>(ph[j][1]), cc = unpack2<T>(ph[j][2]),
                     dd = unpack2<T>(ph[j][3]);
        ps0 += (a.x + a.y) + (cc.x + cc.y);  // the rounded weights the product uses
        ps1 += (b.x + b.y) + (dd.x + dd.y);
      }
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, off);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, off);
    }
    bool lo = false;
    if constexpr (MmaKind<T>::kBf16)
      lo = __any_sync(0xffffffffu, ps0 > kLoShare * (l0 + ps0) || ps1 > kLoShare * (l1 + ps1));
    l0 += ps0;
    l1 += ps1;
    if (lo) {
#pragma unroll
      for (int j = 0; j < NSUB; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 hh = unpack2<T>(ph[j][i]);
          const int h = i >> 1, e = (i & 1) * 2;
          pl[j][i] = pack2<T>(p[j][h][e] - hh.x, p[j][h][e + 1] - hh.y);
        }
      pv<MASK, true>(vs, sub_stride, ph, pl, valid_v, lane);
    } else {
      pv<MASK, false>(vs, sub_stride, ph, pl, valid_v, lane);
    }
  }
};

// More than 8 query rows per KV head: one CTA per (split, KV head, sequence),
// NQ = ceil(rows / 16) consumer warps of 16 rows each (WarpAttnRows) and one
// TMA warp that streams the split's blocks, NSUB per ring stage, so that K/V
// leave HBM once for all the new tokens of the group.  Rows are ordered
// token-major (row r = token r / g, head r % g), the order of q in memory.
// Stages hold NSUB blocks of the same split; a step at the end of a split
// with fewer blocks masks the rest.  split_major: the grid is (sequence, KV
// head, split), so that every unit's first split is dispatched before any
// later one (the later splits of short sequences are empty and exit at the
// tail); otherwise (split, KV head, sequence).
template <typename T, int D, int S, int NSUB>
__global__ void __launch_bounds__(kMaxQueryWarps * 32 + 32, 3)
    decode_multi_rows_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                             const DecodeArgs args, int32_t q_len, int32_t split_major) {
  using Shape = TileShape<D>;
  using Attn = WarpAttnRows<T, D, NSUB>;
  constexpr int kStep = NSUB * Shape::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[S];
  __shared__ __align__(8) uint64_t empty_bar[S];
  __shared__ int s_abort;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint4* qsm = reinterpret_cast<uint4*>(smem + S * kStep);  // Q fragments: [warp][k-step][lane]

  const int split = split_major ? blockIdx.z : blockIdx.x, kvh = blockIdx.y;
  const int b = split_major ? blockIdx.x : blockIdx.z;
  const int NQ = static_cast<int>(blockDim.x >> 5) - 1;  // consumer warps; warp NQ produces
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = args.group, Hq = args.num_q_heads, n = q_len;
  const int nrows = g * n;  // query rows of this (sequence, KV head)

  const int ctx = clamped_context(args.context_lens, b, args.max_blocks, threadIdx.x == 0 && split == 0);
  const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
  const int blk0 = split * args.split_blocks;
  const int nb = min(nblk, blk0 + args.split_blocks) - blk0;
  const int nsteps = (nb + NSUB - 1) / NSUB;
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
    // Table entries in windows of 32 blocks (a multiple of NSUB: no step straddles two).
    for (int base = 0; base < nb && ok; base += 32) {
      const int jb = base + lane;
      const int row = jb < nb ? tile_row(trow[jb], kvh, args) : 0;
      const int cnt = min(32, nb - base);
      for (int k = 0; k < cnt; k += NSUB) {
        int r[NSUB];
#pragma unroll
        for (int j = 0; j < NSUB; ++j) r[j] = __shfl_sync(0xffffffffu, row, k + j);
        if (lane == 0 && ok) {
          const int i = (base + k) / NSUB;
          const int st = i % S;
          const int here = min(NSUB, nb - base - k);
          if (i >= S && !mbar_wait(smem_u32(&empty_bar[st]), ((i / S) & 1) ^ 1)) {
            ok = false;
            s_abort = 1;
          } else if (*reinterpret_cast<volatile int*>(&s_abort)) {
            ok = false;
          } else {
            const uint32_t sa = smem_u32(smem + st * kStep), fb = smem_u32(&full_bar[st]);
            mbar_arrive_expect_tx(fb, here * Shape::kStageBytes);
#pragma unroll
            for (int j = 0; j < NSUB; ++j)
              if (j < here) issue_tiles<D, false>(sa + j * Shape::kStageBytes, fb, &tmap_k, &tmap_v, r[j], policy);
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
  const int ra = kQueryRowsPerWarp * warp + (lane >> 2), rb = ra + 8;  // this lane's two rows
  uint4* qs = qsm + warp * Attn::kKSteps * 32 + lane;
  {
    const T* q = static_cast<const T*>(args.q);
    Attn::stage_q(qs, ra < nrows ? q + row_index(ra) * D : nullptr, rb < nrows ? q + row_index(rb) * D : nullptr,
                  args.scale_log2 < 0.f, lane);
    __syncwarp();
  }
  Attn at;
  at.reset();
  // Last position each row attends to (padding rows: the last of the context).
  const int lim_a = ra < nrows ? ctx - n + ra / g : ctx - 1;
  const int lim_b = rb < nrows ? ctx - n + rb / g : ctx - 1;
  // Every row of this warp sees a whole step of this split starting at t0 when
  // t0 + kTok <= full_end (its first row has the smallest limit).
  const int full_end = ctx - n + (kQueryRowsPerWarp * warp) / g + 1;
  const float c2 = fabsf(args.scale_log2);
  for (int i = 0; i < nsteps; ++i) {
    if (*reinterpret_cast<volatile int*>(&s_abort)) return;
    const int st = i % S;
    if (!mbar_wait(smem_u32(&full_bar[st]), (i / S) & 1)) {
      s_abort = 1;
      return;
    }
    const int t0 = (blk0 + NSUB * i) * kBlockSize;
    const int here_tok = min(NSUB, nb - NSUB * i) * kBlockSize;  // tokens of this split in the step
    const uint32_t ks = smem_u32(smem + st * kStep);
    if (here_tok == Attn::kTok && t0 + Attn::kTok <= full_end) {
      at.template step<false>(ks, ks + Shape::kTileBytes, Shape::kStageBytes, qs, Attn::kTok, Attn::kTok, Attn::kTok,
                              c2, lane);
    } else {
      const int valid = min(here_tok, ctx - t0);
      const int vc0 = max(0, min(valid, lim_a + 1 - t0));
      const int vc1 = max(0, min(valid, lim_b + 1 - t0));
      at.template step<true>(ks, ks + Shape::kTileBytes, Shape::kStageBytes, qs, valid, vc0, vc1, c2, lane);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));  // this warp is done with the stage
  }
  const int c = lane & 3;
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
      for (int nd = 0; nd < Attn::kNTiles; ++nd)
        *reinterpret_cast<uint32_t*>(dst + 8 * nd) = pack2<T>(at.o[nd][2 * half] * inv, at.o[nd][2 * half + 1] * inv);
    } else {
      const int64_t prow = orow * args.num_splits + split;
      float* dst = args.part_o + prow * D + 2 * c;
#pragma unroll
      for (int nd = 0; nd < Attn::kNTiles; ++nd)
        *reinterpret_cast<float2*>(dst + 8 * nd) = make_float2(at.o[nd][2 * half] * inv, at.o[nd][2 * half + 1] * inv);
      if (c == 0) args.part_lse[prow] = l > 0.f ? (half ? at.m1 : at.m0) + log2f(l) : -INFINITY;
    }
  }
}

// args.num_q_heads = Hq; q / out are T[B][q_len][Hq][D]; split partials are
// indexed by row = (b * q_len + i) * Hq + h (args.num_splits, args.split_blocks).
// At most 8 query rows per KV head: one consumer warp with the rows in the
// mma N dimension (WarpAttnCausal), which pads less than 16-row M tiles.
template <typename T, int D, int S>
__global__ void __launch_bounds__(64)
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
  {
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
