// Multi-token paged decode for 64 query rows per KV head on the fifth-
// generation tensor cores (sm_103a), run by paged_decode_step_multi_tc.  Same
// result as decode_multi_rows_kernel (youngju.dev "LLM サービング最適化完全ガイド",
// speculative decoding section: several draft tokens checked in one pass),
// with the products as tcgen05 MMAs whose accumulators and A operands live in
// tensor memory.  Its 448 TMEM columns hold it to one CTA per SM, which leaves
// each CTA's start, pipeline ramp and tensor-memory latencies exposed; the
// mma.sync row kernel stays the default until this one overtakes it.
//
// Every mbarrier wait below is on a phase at most one ahead of the barrier's
// last completed phase: a parity wait cannot tell phase k from k + 2, so each
// wait names the barrier whose progress the waiter bounds (for instance the
// softmax warps wait for P V of tile t - 1 on its P buffer's barrier, which
// they themselves held back until P V of t - 3 was done).
//
// One CTA per (split, pair of KV heads, sequence): the two heads 2p and 2p+1
// of a sequence share its block table and length, so the CTA streams both
// heads' tiles of the same blocks and fills the MMA's 128 rows with two
// units of 64 query rows.  Q is block-diagonal over the two heads (rows 0-63
// hold head 2p's queries in K entries 0-127, rows 64-127 head 2p+1's in K
// entries 128-255), so
//   S = Q K^T   M = 128, N = 32 tokens (two blocks), K = 256: each row meets
//               only its own head's keys (head 2p's in K entries 0-127);
//   O += P V    M = 128, N = 128 (head_dim), K = 64: tokens 0-31 of head 2p
//               then of head 2p+1, P zero outside a row's own head.
// Warps: 0-3 softmax (TMEM lane r = MMA row r, one thread per row), 4 TMA
// producer, 5 TMEM allocation and the MMA issuer (one thread).
// TMEM columns: Q 0-127, S 128-191 (two buffers), P hi 192-255 and P lo
// 256-319 (two buffers each; their zero halves are written once), O 384-511.
// bf16 weights enter as hi + lo (two MMAs per k-step), fp16 as one term.
#pragma once

#include "multi_query.cuh"
#include "tcgen05.cuh"

namespace pkv {

struct Tc2 {
  static constexpr int D = 128;
  static constexpr int kTok = 32;                               // tokens per tile: two blocks
  static constexpr int kAtomBytes = kTok * 128;                 // 32 rows x 128 B
  static constexpr int kKBytes = 4 * kAtomBytes;                // K atoms [head][dim half]
  static constexpr int kVHalfBytes = 2 * kTok * 128;            // V rows [head][token] of one dim half
  static constexpr int kVBytes = 2 * kVHalfBytes;               // V [dim half][head][token]
  static constexpr int kStageBytes = kKBytes + kVBytes;         // 32 KB
  static constexpr int kStages = 4;
  static constexpr int kSmem = kStages * kStageBytes + 1024;
  static constexpr int kQCol = 0, kSCol = 128, kPhCol = 192, kPlCol = 256, kOCol = 384;
  static constexpr int kTmemCols = 512;
  static constexpr int kThreads = 192;
  static constexpr int kRows = 64;                              // query rows per unit
};

template <typename T>
__global__ void __launch_bounds__(Tc2::kThreads, 1)
    decode_multi_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                           const DecodeArgs args, int32_t q_len) {
  constexpr int D = Tc2::D;
  constexpr int NST = Tc2::kStages;
  constexpr bool kBf16 = MmaKind<T>::kBf16;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t kv_full[NST];
  __shared__ __align__(8) uint64_t kv_empty[NST];
  __shared__ __align__(8) uint64_t s_full[2];
  __shared__ __align__(8) uint64_t s_free[2];
  __shared__ __align__(8) uint64_t p_full[2];
  __shared__ __align__(8) uint64_t p_free[2];
  __shared__ __align__(8) uint64_t q_ready;
  __shared__ __align__(8) uint64_t mma_fin;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int split = blockIdx.x, pair = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = args.group, Hq = args.num_q_heads, n = q_len;

  const int ctx = clamped_context(args.context_lens, b, args.max_blocks, threadIdx.x == 0 && split == 0 && pair == 0);
  const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
  const int blk0 = split * args.split_blocks;
  const int nb = min(nblk, blk0 + args.split_blocks) - blk0;
  auto row_index = [&](int u, int r) -> int64_t {  // output row of query row r of head 2 pair + u
    return (static_cast<int64_t>(b) * n + r / g) * Hq + (2 * pair + u) * g + r % g;
  };

  if (nb <= 0) {
    if (args.num_splits == 1) {  // an empty context: zero rows
      for (int idx = threadIdx.x; idx < 2 * Tc2::kRows * D; idx += blockDim.x) {
        const int ur = idx / D, d = idx - ur * D;
        static_cast<T*>(args.out)[row_index(ur / Tc2::kRows, ur % Tc2::kRows) * D + d] = T(0.0f);
      }
    }
    return;
  }
  const int ntiles = (nb + 1) / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&kv_full[s]), 1);
      mbar_init(smem_u32(&kv_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&s_free[s]), 4);
      mbar_init(smem_u32(&p_full[s]), 4);
      mbar_init(smem_u32(&p_free[s]), 1);
    }
    mbar_init(smem_u32(&q_ready), 4);
    mbar_init(smem_u32(&mma_fin), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(smem_u32(&s_tmem), Tc2::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = s_tmem;
  volatile int* abort_flag = &s_abort;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    const int32_t* trow = args.block_tables + static_cast<int64_t>(b) * args.max_blocks + blk0;
    const uint64_t policy = l2_evict_first_policy();
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    int issued = 0;
    int win = 0;  // lane i holds the table entry of block win + i
    int wphys = lane < nb ? __ldg(trow + lane) : 0;
    for (int t = 0; t < ntiles; ++t) {
      const int first = 2 * t;
      if (first >= win + 32) {
        win = first;
        wphys = win + lane < nb ? __ldg(trow + win + lane) : 0;
      }
      const int here = min(2, nb - first);
      int phys[2];
      phys[0] = __shfl_sync(0xffffffffu, wphys, first - win);
      phys[1] = __shfl_sync(0xffffffffu, wphys, first - win + 1);
      const int st = t % NST;
      bool ok = true;
      if (lane == 0 && t >= NST) ok = mbar_wait(smem_u32(&kv_empty[st]), ((t / NST) & 1) ^ 1);
      ok = __shfl_sync(0xffffffffu, ok, 0) && !*abort_flag;
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      if (lane == 0) {
        const uint32_t bar = smem_u32(&kv_full[st]);
        const uint32_t kst = smem_u32(ring + st * Tc2::kStageBytes);
        const uint32_t vst = kst + Tc2::kKBytes;
        mbar_arrive_expect_tx(bar, here * 2 * 2 * 2 * 2048);
        for (int i = 0; i < here; ++i) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int row = tile_row(phys[i], 2 * pair + u, args);
#pragma unroll
            for (int d = 0; d < 2; ++d) {
              tma_load_2d(kst + (2 * u + d) * Tc2::kAtomBytes + i * 2048, &tmap_k, 64 * d, row, bar, policy);
              tma_load_2d(vst + d * Tc2::kVHalfBytes + (u * Tc2::kTok + i * kBlockSize) * 128, &tmap_v, 64 * d, row,
                          bar, policy);
            }
          }
        }
      }
      issued = t + 1;
    }
    // After an abort no copy may still be landing in shared memory at exit.
    if (lane == 0 && *abort_flag) {
      for (int t = max(0, issued - NST); t < issued; ++t) mbar_wait(smem_u32(&kv_full[t % NST]), (t / NST) & 1);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = tc::idesc_f16(kBf16, 128, Tc2::kTok, false);
      constexpr uint32_t kIdescPV = tc::idesc_f16(kBf16, 128, D, true);
      bool ok = mbar_wait(smem_u32(&q_ready), 0);
      tc::fence_after_sync();
      int nq = 0, np = 0;  // next tile for S = Q K^T, next tile for O += P V
      unsigned long long idle_since = 0;
      uint32_t spins = 0;
      while (ok && np < ntiles) {
        bool progressed = false;
        // S = Q K^T of tile nq once its tiles have landed and the softmax has
        // read S of tile nq - 2 out of the same buffer.
        if (nq < ntiles && nq <= np + 2) {
          const int st = nq % NST;
          if (tc::mbar_test_wait(smem_u32(&kv_full[st]), (nq / NST) & 1) &&
              (nq < 2 || tc::mbar_test_wait(smem_u32(&s_free[nq & 1]), ((nq - 2) >> 1) & 1))) {
            tc::fence_after_sync();
            const uint32_t kst = smem_u32(ring + st * Tc2::kStageBytes);
            const uint32_t sb = tbase + Tc2::kSCol + (nq & 1) * Tc2::kTok;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              // K entries 16 kk .. + 15: Q columns 8 kk .. + 7; K atom kk / 4 (head kk / 8), 32 bytes (kk % 4) in.
              const uint64_t bdesc = tc::smem_desc_sw128(kst + (kk >> 2) * Tc2::kAtomBytes + (kk & 3) * 32, 16, 1024);
              tc::mma_ts(sb, tbase + Tc2::kQCol + 8 * kk, bdesc, kIdescQK, kk > 0 ? 1u : 0u);
            }
            tc::mma_commit(smem_u32(&s_full[nq & 1]));
            ++nq;
            progressed = true;
          }
        }
        // O += P V of tile np once the softmax has written its weights.
        if (np < nq && tc::mbar_test_wait(smem_u32(&p_full[np & 1]), (np >> 1) & 1)) {
          tc::fence_after_sync();
          const int st = np % NST;
          const uint32_t vst = smem_u32(ring + st * Tc2::kStageBytes) + Tc2::kKBytes;
          const uint32_t ph = tbase + Tc2::kPhCol + (np & 1) * 32, pl = tbase + Tc2::kPlCol + (np & 1) * 32;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // K entries 16 i .. + 15 = V rows 16 i .. + 15 (head i / 2, tokens 16 (i % 2) ..); P columns 8 i .. + 7.
            const uint64_t vdesc = tc::smem_desc_sw128(vst + i * 2048, Tc2::kVHalfBytes, 1024);
            tc::mma_ts(tbase + Tc2::kOCol, ph + 8 * i, vdesc, kIdescPV, (np > 0 || i > 0) ? 1u : 0u);
            if constexpr (kBf16) tc::mma_ts(tbase + Tc2::kOCol, pl + 8 * i, vdesc, kIdescPV, 1u);
          }
          tc::mma_commit(smem_u32(&kv_empty[st]));
          tc::mma_commit(smem_u32(&p_free[np & 1]));
          ++np;
          progressed = true;
        }
        if (progressed) {
          spins = 0;
        } else if ((++spins & 63u) == 0) {
          const unsigned long long now = global_ns();
          if (spins == 64) idle_since = now;
          if (now - idle_since > kWaitLimitNs || *abort_flag) {
            if (!*abort_flag) flag_error(kErrTimeout);
            ok = false;
          }
        }
      }
      if (!ok) *abort_flag = 1;
      // No MMA may still be running when the CTA frees its TMEM.
      tc::mma_commit(smem_u32(&mma_fin));
      mbar_wait(smem_u32(&mma_fin), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 0-3
    const int r = 32 * warp + lane;  // MMA row = TMEM lane
    const int u = r >> 6, lr = r & 63;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    const int limit = ctx - n + lr / g;  // last position this row attends to
    const float c2 = fabsf(args.scale_log2);
    // Q row into its half of the block-diagonal A operand (negated for a
    // negative scale, an exact sign flip, so that max(s) * |scale| is the
    // maximum of the scaled scores); the other half and every P buffer are
    // zeros.
    {
      const uint32_t flip = args.scale_log2 < 0.f ? 0x80008000u : 0u;
      const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const T*>(args.q) + row_index(u, lr) * D);
      uint32_t z[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) z[k] = 0u;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t qw[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = __ldg(qrow + 8 * h + c);
          qw[4 * c] = v.x ^ flip;
          qw[4 * c + 1] = v.y ^ flip;
          qw[4 * c + 2] = v.z ^ flip;
          qw[4 * c + 3] = v.w ^ flip;
        }
        tc::tmem_st32(tbase + lane_base + Tc2::kQCol + 64 * u + 32 * h, qw);
        tc::tmem_st32(tbase + lane_base + Tc2::kQCol + 64 * (1 - u) + 32 * h, z);
      }
      tc::tmem_st32(tbase + lane_base + Tc2::kPhCol, z);
      tc::tmem_st32(tbase + lane_base + Tc2::kPhCol + 32, z);
      tc::tmem_st32(tbase + lane_base + Tc2::kPlCol, z);
      tc::tmem_st32(tbase + lane_base + Tc2::kPlCol + 32, z);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&q_ready));
    }

    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[t & 1]), (t >> 1) & 1) && !*abort_flag);
      if (!ok) break;
      tc::fence_after_sync();
      uint32_t sv[32];
      tc::tmem_ld32(tbase + lane_base + Tc2::kSCol + (t & 1) * Tc2::kTok, sv);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_free[t & 1]));  // S buffer t & 1 may take tile t + 2

      const int t0 = (blk0 + 2 * t) * kBlockSize;
      const int here_tok = min(2, nb - 2 * t) * kBlockSize;
      const int valid = min(here_tok, ctx - t0);                 // tokens of the tile in the context
      const int vis = max(0, min(valid, limit - t0 + 1));        // tokens this row sees
      float x[32];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        x[c] = c < vis ? __uint_as_float(sv[c]) : -INFINITY;
        mx = fmaxf(mx, x[c]);
      }
      mx *= c2;
      const bool up = mx > m + 8.f;  // lazy reference maximum (2^8)
      if (__any_sync(0xffffffffu, up)) {
        const float al = up ? ex2(m - mx) : 1.f;
        if (t > 0) {
          // O holds P V of tiles up to t - 1: wait for the last of them (its
          // p_free phase is never two away: this warp waited for P V of
          // t - 3 before writing P of t - 1), then rescale this warp's rows.
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&p_free[(t - 1) & 1]), ((t - 1) >> 1) & 1));
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int j = 0; j < D / 32; ++j) {
            uint32_t o[32];
            const uint32_t oa = tbase + lane_base + Tc2::kOCol + 32 * j;
            tc::tmem_ld32(oa, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * al);
            tc::tmem_st32(oa, o);
          }
          tc::tmem_wait_st();
        }
        l *= al;
        if (up) m = mx;
      }
      const float nr = m == -INFINITY ? 0.f : -m;
      uint32_t hi[16], lo[16];
      float ls = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float p0 = ex2(fmaf(x[2 * k], c2, nr)), p1 = ex2(fmaf(x[2 * k + 1], c2, nr));
        hi[k] = pack2<T>(p0, p1);
        const float2 h = unpack2<T>(hi[k]);
        if constexpr (kBf16) {
          lo[k] = pack2<T>(p0 - h.x, p1 - h.y);
          ls += p0 + p1;
        } else {
          lo[k] = 0u;
          ls += h.x + h.y;  // the rounded weights the product uses
        }
      }
      l += ls;
      // P buffer t & 1 is free once P V of tile t - 2 is done.
      if (t >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&p_free[t & 1]), ((t - 2) >> 1) & 1));
        if (!ok) break;
        tc::fence_after_sync();
      }
      // The tile's V rows past the context (a partly filled last block, or a
      // block beyond the split) must be zeros: a weight of 0 times a NaN
      // sentinel is NaN.  The tiles have landed (S of this tile was computed).
      if (valid < Tc2::kTok && (warp & 1) == 0) {
        uint8_t* v = ring + (t % NST) * Tc2::kStageBytes + Tc2::kKBytes;
        const int zrows = Tc2::kTok - valid;
        for (int idx = lane; idx < 2 * zrows * 8; idx += 32) {
          const int d = idx / (zrows * 8), rem = idx - d * zrows * 8;
          *reinterpret_cast<uint4*>(v + d * Tc2::kVHalfBytes + (u * Tc2::kTok + valid + rem / 8) * 128 +
                                    (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      const uint32_t pcol = (t & 1) * 32 + 16 * u;
      uint32_t h8[8], l8[8];
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          h8[k] = hi[8 * hlf + k];
          l8[k] = lo[8 * hlf + k];
        }
        tc::tmem_st8(tbase + lane_base + Tc2::kPhCol + pcol + 8 * hlf, h8);
        if constexpr (kBf16) tc::tmem_st8(tbase + lane_base + Tc2::kPlCol + pcol + 8 * hlf, l8);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full[t & 1]));
    }
    // Epilogue: after the last P V, O / l is the output row.
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&p_free[(ntiles - 1) & 1]), ((ntiles - 1) >> 1) & 1));
    if (!ok) *abort_flag = 1;
    tc::fence_after_sync();
    const bool aborted = __any_sync(0xffffffffu, *abort_flag != 0);
    if (!aborted) {
      const float inv = l > 0.f ? 1.0f / l : 0.f;  // no visible token: a zero row
      const int64_t orow = row_index(u, lr);
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        uint32_t o[32];
        tc::tmem_ld32(tbase + lane_base + Tc2::kOCol + 32 * j, o);
        tc::tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(o[k]) * inv;
        if (args.num_splits == 1) {
          T* dst = static_cast<T*>(args.out) + orow * D + 32 * j;
#pragma unroll
          for (int k = 0; k < 32; k += 8)
            *reinterpret_cast<uint4*>(dst + k) =
                make_uint4(pack2<T>(v[k], v[k + 1]), pack2<T>(v[k + 2], v[k + 3]), pack2<T>(v[k + 4], v[k + 5]),
                           pack2<T>(v[k + 6], v[k + 7]));
        } else {
          float* dst = args.part_o + (orow * args.num_splits + split) * D + 32 * j;
#pragma unroll
          for (int k = 0; k < 32; k += 4) *reinterpret_cast<float4*>(dst + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
        }
      }
      if (args.num_splits != 1)
        args.part_lse[orow * args.num_splits + split] = l > 0.f ? m + log2f(l) : -INFINITY;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, Tc2::kTmemCols);
  }
}

}  // namespace pkv
