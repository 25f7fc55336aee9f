// C ABI of libpagedkv.so: argument validation, split selection, TMA tensor
// maps and kernel launches.  The declarations and their contracts are in
// include/paged_kv.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "paged_kv.h"
#include "block_copy.cuh"
#include "host_copy.cuh"
#include "multi_query.cuh"
#include "multi_query_tc.cuh"
#include "paged_kv_kernels.cuh"
#include "pkv_errors.h"
#include "pkv_internal.h"

namespace {

constexpr int kConsumerWarps = 4;   // split kernel
constexpr int kStages = 8;          // split kernel ring depth
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kAutoSplitBlocks = 32;  // 512-token splits when the split path is chosen automatically
constexpr int kMaxDevices = 64;

int device_sms() {
  static int sms[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= kMaxDevices) dev = kMaxDevices - 1;
  if (sms[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = v > 0 ? v : 1;
  }
  return sms[dev];
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Per-call tags of the decode grid's publication to its merge (never 0).
uint32_t next_epoch() {
  static std::atomic<uint32_t> counter{0};
  uint32_t e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  if (e == 0) e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  return e;
}

int cuda_fail(cudaError_t e, const char* what) {
  return pkv_fail(PKV_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_dims(const pkv_dims* d, bool need_q_heads) {
  if (!d) return pkv_fail(PKV_ERR_INVALID_ARG, "dims is NULL");
  if (d->num_seqs < 0 || d->num_kv_heads <= 0 || d->num_blocks <= 0 || d->max_blocks_per_seq < 0)
    return pkv_fail(PKV_ERR_INVALID_ARG, "dims: negative or zero size");
  if (d->dtype != PKV_DTYPE_FP16 && d->dtype != PKV_DTYPE_BF16)
    return pkv_fail(PKV_ERR_UNSUPPORTED, "dims: dtype must be fp16 or bf16");
  if (d->head_dim != 64 && d->head_dim != 128) return pkv_fail(PKV_ERR_UNSUPPORTED, "dims: head_dim must be 64 or 128");
  if (d->block_size != pkv::kBlockSize) return pkv_fail(PKV_ERR_UNSUPPORTED, "dims: block_size must be 16");
  if (static_cast<int64_t>(d->num_blocks) * d->num_kv_heads * pkv::kBlockSize >= (int64_t(1) << 31))
    return pkv_fail(PKV_ERR_UNSUPPORTED, "dims: num_blocks * num_kv_heads * 16 must be < 2^31");
  if (need_q_heads) {
    if (d->num_q_heads <= 0 || d->num_q_heads % d->num_kv_heads != 0)
      return pkv_fail(PKV_ERR_INVALID_ARG, "dims: num_kv_heads must divide num_q_heads");
    if (d->num_q_heads / d->num_kv_heads > 8)
      return pkv_fail(PKV_ERR_UNSUPPORTED, "dims: at most 8 query heads per KV head");
  }
  return PKV_OK;
}

// ------------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The pool as a 2-D tensor: rows = num_blocks * Hkv * 16 of head_dim elements;
// boxes of 16 rows x 128 bytes (64 fp16/bf16 elements or 128 E4M3 codes) with
// the 128-byte swizzle.
int make_cache_map(CUtensorMap* map, const void* cache, const pkv_dims* d, bool f8) {
  auto fn = encode_fn();
  if (!fn) return pkv_fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d->head_dim),
                              static_cast<cuuint64_t>(d->num_blocks) * d->num_kv_heads * pkv::kBlockSize};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d->head_dim) * (f8 ? 1 : 2)};
  const cuuint32_t box[2] = {f8 ? 128u : 64u, static_cast<cuuint32_t>(pkv::kBlockSize)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = f8                           ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : d->dtype == PKV_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(map, dt, 2, const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return pkv_fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string(r) + ")");
  return PKV_OK;
}

// Small cache of encoded maps keyed by (address, shape, dtype): a decode loop
// reuses the same pool every step.
struct MapCache {
  struct Entry {
    const void* ptr = nullptr;
    int32_t nb = 0, hkv = 0, hd = 0, dt = -1;
    CUtensorMap map;
  };
  static constexpr int kEntries = 16;
  Entry e[kEntries];
  int next = 0;
  std::mutex mu;

  int get(const void* ptr, const pkv_dims* d, bool f8, CUtensorMap* out) {
    const int32_t dt = f8 ? -2 : d->dtype;
    std::lock_guard<std::mutex> lock(mu);
    for (auto& x : e)
      if (x.ptr == ptr && x.nb == d->num_blocks && x.hkv == d->num_kv_heads && x.hd == d->head_dim && x.dt == dt) {
        *out = x.map;
        return PKV_OK;
      }
    Entry& n = e[next];
    int rc = make_cache_map(&n.map, ptr, d, f8);
    if (rc != PKV_OK) return rc;
    n.ptr = ptr;
    n.nb = d->num_blocks;
    n.hkv = d->num_kv_heads;
    n.hd = d->head_dim;
    n.dt = dt;
    next = (next + 1) % kEntries;
    *out = n.map;
    return PKV_OK;
  }
};
MapCache g_maps;

// ------------------------------------------------------------------ splits

struct SplitPlan {
  bool persistent;        // balanced persistent kernel (no fixed split)
  int32_t num_splits;     // split kernel: splits per sequence
  int32_t split_blocks;   // split kernel: blocks per split
};

// Largest batch of the persistent kernel: its prefix sums live in shared
// memory beside the ring (2048 sequences for every pool format built).
int max_persistent_seqs(const pkv_dims* d, bool f8) {
  if (f8) return pkv::persistent_max_seqs<128, true>() / 256 * 256;
  return d->head_dim == 128 ? pkv::persistent_max_seqs<128>() : pkv::persistent_max_seqs<64>();
}

bool persistent_eligible(const pkv_dims* d, bool f8 = false) {
  return d->num_seqs <= max_persistent_seqs(d, f8) &&
         static_cast<int64_t>(d->num_seqs) * d->num_kv_heads * d->max_blocks_per_seq < (int64_t(1) << 31);
}

int plan_splits(const pkv_dims* d, int32_t requested, SplitPlan* plan) {
  if (requested < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "num_splits must be >= 0");
  const int32_t mb = d->max_blocks_per_seq;
  if (requested == 0 && persistent_eligible(d)) {
    *plan = {true, 0, 0};
    return PKV_OK;
  }
  if (mb <= 1) {
    *plan = {false, 1, mb > 0 ? mb : 1};
    return PKV_OK;
  }
  int32_t n = requested == 0 ? (mb + kAutoSplitBlocks - 1) / kAutoSplitBlocks : requested;
  if (n > mb) n = mb;
  if (n < 1) n = 1;
  const int32_t per = (mb + n - 1) / n;
  *plan = {false, (mb + per - 1) / per, per};
  return PKV_OK;
}

// Workspace regions: [partial outputs][partial log-sum-exps][publication of
// the decode grid's lengths to its merge][scheduler counters].
struct WorkspaceLayout {
  size_t o_bytes = 0, lse_bytes = 0, sched_bytes = 0, pub_bytes = 0;
  size_t total() const { return o_bytes + lse_bytes + sched_bytes + pub_bytes; }
};

// Segments of the persistent partition for the largest grid (one CTA per SM).
size_t persistent_segments() {
  return static_cast<size_t>(device_sms()) * pkv::kMaxPersistentWarps * (1 + pkv::Partition::kMaxTailChunks);
}

WorkspaceLayout workspace_layout(const pkv_dims* d, const SplitPlan& p) {
  WorkspaceLayout w;
  if (p.persistent) {
    const size_t seg = persistent_segments();
    w.o_bytes = align256(seg * 2 * pkv::kMaxGroup * d->head_dim * sizeof(float));
    w.lse_bytes = align256(seg * 2 * pkv::kMaxGroup * sizeof(float));
    w.sched_bytes = 256;
    // The decode grid's validated lengths and block prefix, for the merge:
    // [epoch][context B][prefix B + 1] int32.
    w.pub_bytes = align256((2 * static_cast<size_t>(d->num_seqs) + 2) * sizeof(int32_t));
  } else if (p.num_splits > 1) {
    const size_t rows = static_cast<size_t>(d->num_seqs) * d->num_q_heads * p.num_splits;
    w.o_bytes = align256(rows * d->head_dim * sizeof(float));
    w.lse_bytes = align256(rows * sizeof(float));
  }
  return w;
}

// ------------------------------------------------------------------ launches

// Raise a kernel's dynamic shared-memory limit once per device (and ask for
// the largest shared-memory carveout).  The kernel is a template argument so
// that every kernel instantiation keeps its own flags.
template <auto kern>
cudaError_t configure_smem(int bytes) {
  static bool done[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < kMaxDevices && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && dev < kMaxDevices) done[dev] = true;
  return e;
}

// Persistent decode + merge.  Both are programmatic dependent launches: each
// may start while the kernel before it in the stream finishes, and waits
// in-kernel (griddepcontrol.wait) before touching anything that kernel writes.
template <typename T, int D, bool F8>
int launch_persistent(const CUtensorMap& mk, const CUtensorMap& mv, const pkv::DecodeArgs& args,
                      const pkv_dims* d, int max_seqs, cudaStream_t stream, bool pdl = true) {
  using PS = pkv::PersistentShape<D, F8>;
  constexpr auto kern = pkv::decode_persistent_kernel<T, D, F8>;
  cudaError_t e = configure_smem<kern>(static_cast<int>(pkv::persistent_smem_bytes<D, F8>(max_seqs)));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_persistent_kernel)");
  const int64_t upper_blocks = static_cast<int64_t>(d->num_seqs) * d->num_kv_heads * d->max_blocks_per_seq;
  int64_t grid = (upper_blocks + PS::kWarps - 1) / PS::kWarps;
  if (grid > device_sms()) grid = device_sms();
  if (grid < 1) grid = 1;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(PS::kWarps * 32);
  cfg.dynamicSmemBytes = pkv::persistent_smem_bytes<D, F8>(d->num_seqs);
  cfg.stream = stream;
  cfg.attrs = attr;
  // !pdl: the kernel before this one wrote its inputs (block tables, lengths,
  // query), which it reads before griddepcontrol.wait: no early launch.
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, mk, mv, args);
  if (e != cudaSuccess) return cuda_fail(e, "decode_persistent_kernel launch");
  cfg.numAttrs = 1;
  // Long units cut into many pieces (on average 8 or more warp shares per
  // unit): a CTA per row, its warps splitting the row's pieces; otherwise a
  // warp per row (measured: at 7.1 shares, the E4M3 pool at B=32, a warp per
  // row 0.741 against 0.703; at 9.5, bf16 at B=16, a CTA per row 0.784
  // against 0.770).
  const int32_t nwarps = static_cast<int32_t>(grid) * PS::kWarps;
  const int64_t units = static_cast<int64_t>(d->num_seqs) * d->num_kv_heads;
  const bool coop = nwarps >= 8 * units;
  // Two or more warp shares per unit on average: rows have many pieces, so
  // fold up to 16 per round trip (fewer registers leave room for more merge
  // CTAs beside the decode grid, which pays when rows are many and short).
  const bool wide = !coop && nwarps >= 2 * units;
  const int merge_smem = static_cast<int>((2 * static_cast<size_t>(max_persistent_seqs(d, false)) + 1) * 4);
  const int rows = d->num_seqs * d->num_q_heads;
  const int rows_per_cta = coop ? 1 : pkv::kMergeWarps;
  cfg.gridDim = dim3(static_cast<unsigned>((rows + rows_per_cta - 1) / rows_per_cta));
  cfg.blockDim = dim3(pkv::kMergeWarps * 32);
  cfg.dynamicSmemBytes = (2 * static_cast<size_t>(d->num_seqs) + 1) * 4;
  if (coop) {
    constexpr auto merge = pkv::merge_persistent_kernel<T, D, true>;
    e = configure_smem<merge>(merge_smem);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, merge, args, nwarps);
  } else if (wide) {
    constexpr auto merge = pkv::merge_persistent_kernel<T, D, false, true>;
    e = configure_smem<merge>(merge_smem);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, merge, args, nwarps);
  } else {
    constexpr auto merge = pkv::merge_persistent_kernel<T, D, false>;
    e = configure_smem<merge>(merge_smem);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, merge, args, nwarps);
  }
  if (e != cudaSuccess) return cuda_fail(e, "merge_persistent_kernel launch");
  return PKV_OK;
}

template <typename T, int D>
int launch_decode(const CUtensorMap& mk, const CUtensorMap& mv, const pkv::DecodeArgs& args, const SplitPlan& plan,
                  const pkv_dims* d, cudaStream_t stream, bool pdl) {
  using Shape = pkv::TileShape<D>;
  if (plan.persistent)
    return launch_persistent<T, D, false>(mk, mv, args, d, max_persistent_seqs(d, false), stream, pdl);
  constexpr int kSmem = kStages * Shape::kStageBytes + 1024;
  constexpr auto kern = pkv::decode_split_kernel<T, D, kConsumerWarps, kStages>;
  cudaError_t e = configure_smem<kern>(kSmem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_split_kernel)");
  dim3 grid(plan.num_splits, d->num_kv_heads, d->num_seqs);
  kern<<<grid, kThreads, kSmem, stream>>>(mk, mv, args);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode_split_kernel launch");
  if (plan.num_splits > 1) {
    const int rows = d->num_seqs * d->num_q_heads;
    pkv::merge_split_kernel<T, D><<<(rows + 3) / 4, 128, 0, stream>>>(
        args.part_o, args.part_lse, args.context_lens, static_cast<T*>(args.out), d->num_seqs, d->num_q_heads,
        plan.num_splits, plan.split_blocks, args.max_blocks);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "merge_split_kernel launch");
  }
  return PKV_OK;
}

int append_at_end_impl(const void* k_new, const void* v_new, const int32_t* block_tables,
                       const int32_t* context_lens, void* k_cache, void* v_cache, const pkv_dims* d,
                       cudaStream_t stream);

// Attention, optionally preceded by the append of each sequence's token at
// position context_lens[b] - 1 (k_new / v_new non-null): fused into the
// persistent kernel when that path runs, else a separate append launch.
//
// f8: the pool holds E4M3 codes with per-KV-head scales k_scale / v_scale
// (head_dim 128, persistent path only).
int decode_impl(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                const int32_t* block_tables, const int32_t* context_lens, float scale, void* out,
                int32_t num_splits, void* workspace, size_t workspace_bytes, const pkv_dims* d,
                cudaStream_t stream, bool f8 = false, const float* k_scale = nullptr,
                const float* v_scale = nullptr, bool pdl = true, const int32_t* pre_lens = nullptr,
                const int32_t* pre_tables = nullptr, bool recheck = true, bool publish = true) {
  int rc = check_dims(d, true);
  if (rc != PKV_OK) return rc;
  if (f8) {
    if (d->head_dim != 128) return pkv_fail(PKV_ERR_UNSUPPORTED, "fp8 cache: head_dim must be 128");
    if (!persistent_eligible(d, true))
      return pkv_fail(PKV_ERR_UNSUPPORTED, "fp8 cache: at most " + std::to_string(max_persistent_seqs(d, true)) +
                                               " sequences per call");
    if (!k_scale || !v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4))
      return pkv_fail(PKV_ERR_INVALID_ARG, "fp8 cache: k_scale / v_scale missing or misaligned");
  }
  if (d->num_seqs == 0) return PKV_OK;
  // A zero-width table means every context is empty (contexts are clamped to
  // the table): the table pointer is then never read.
  if (!q || !k_cache || !v_cache || (!block_tables && d->max_blocks_per_seq > 0) || !context_lens || !out)
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_attention: NULL pointer");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_attention: misaligned pointer (q/out/caches need 16 bytes)");
  if (!std::isfinite(scale)) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_attention: scale is not finite");
  SplitPlan plan;
  rc = plan_splits(d, num_splits, &plan);
  if (rc != PKV_OK) return rc;
  const WorkspaceLayout wl = workspace_layout(d, plan);
  const size_t need = wl.total();
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_attention: workspace missing, too small (" +
                                             std::to_string(need) + " bytes needed) or not 256-byte aligned");
  const bool append = k_new != nullptr;
  if (append != (v_new != nullptr))
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_step: k_new and v_new must both be given");
  if (append && (!aligned(k_new, 16) || !aligned(v_new, 16)))
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_step: k_new / v_new must be 16-byte aligned");
  if (append && !plan.persistent) {
    rc = append_at_end_impl(k_new, v_new, block_tables, context_lens, k_cache, v_cache, d, stream);
    if (rc != PKV_OK) return rc;
  }
  CUtensorMap mk, mv;
  if ((rc = g_maps.get(k_cache, d, f8, &mk)) != PKV_OK) return rc;
  if ((rc = g_maps.get(v_cache, d, f8, &mv)) != PKV_OK) return rc;

  pkv::DecodeArgs args;
  args.k_new = append && plan.persistent ? k_new : nullptr;
  args.v_new = append && plan.persistent ? v_new : nullptr;
  args.k_cache_w = k_cache;
  args.v_cache_w = v_cache;
  args.k_scale = k_scale;
  args.v_scale = v_scale;
  args.q = q;
  args.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  args.part_o = need ? reinterpret_cast<float*>(ws) : nullptr;
  args.part_lse = need ? reinterpret_cast<float*>(ws + wl.o_bytes) : nullptr;
  // [partials][log-sum-exps][publication][scheduler counters]
  args.pub = wl.pub_bytes ? reinterpret_cast<int32_t*>(ws + wl.o_bytes + wl.lse_bytes) : nullptr;
  args.sched = wl.sched_bytes ? reinterpret_cast<int32_t*>(ws + wl.o_bytes + wl.lse_bytes + wl.pub_bytes) : nullptr;
  args.epoch = 0;
  if (recheck && publish && plan.persistent && args.pub) {
    // A new tag per call, so that a merge never takes an earlier call's
    // publication for its own; 0 (no publication: the merge re-reads the
    // lengths itself) while the stream is being captured, since a graph
    // replays the tag it captured.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
      cudaGetLastError();
      cap = cudaStreamCaptureStatusActive;
    }
    if (cap == cudaStreamCaptureStatusNone) args.epoch = next_epoch();
  }
  args.block_tables = block_tables;
  args.context_lens = context_lens;
  args.pre_context_lens = pre_lens;
  args.pre_block_tables = pre_tables;
  args.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  args.recheck = recheck ? 1 : 0;
  args.num_seqs = d->num_seqs;
  args.num_q_heads = d->num_q_heads;
  args.num_kv_heads = d->num_kv_heads;
  args.group = d->num_q_heads / d->num_kv_heads;
  args.max_blocks = d->max_blocks_per_seq;
  args.num_blocks = d->num_blocks;
  args.num_splits = plan.num_splits;
  args.split_blocks = plan.split_blocks;

  const bool bf16 = d->dtype == PKV_DTYPE_BF16;
  if (f8) {
    const int mx = max_persistent_seqs(d, true);
    return bf16 ? launch_persistent<__nv_bfloat16, 128, true>(mk, mv, args, d, mx, stream, pdl)
                : launch_persistent<__half, 128, true>(mk, mv, args, d, mx, stream, pdl);
  }
  if (d->head_dim == 128)
    return bf16 ? launch_decode<__nv_bfloat16, 128>(mk, mv, args, plan, d, stream, pdl)
                : launch_decode<__half, 128>(mk, mv, args, plan, d, stream, pdl);
  return bf16 ? launch_decode<__nv_bfloat16, 64>(mk, mv, args, plan, d, stream, pdl)
              : launch_decode<__half, 64>(mk, mv, args, plan, d, stream, pdl);
}

int append_at_end_impl(const void* k_new, const void* v_new, const int32_t* block_tables,
                       const int32_t* context_lens, void* k_cache, void* v_cache, const pkv_dims* d,
                       cudaStream_t stream) {
  if (d->num_seqs == 0 || d->max_blocks_per_seq == 0) return PKV_OK;
  const int32_t chunks = d->head_dim * 2 / 16;
  const int64_t total = static_cast<int64_t>(d->num_seqs) * d->num_kv_heads * chunks;
  const int threads = 256;
  const int64_t blocks64 = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(blocks64 < 65536 ? blocks64 : 65536);
  pkv::append_at_end_kernel<<<blocks, threads, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), block_tables, context_lens, d->num_seqs,
      d->max_blocks_per_seq, d->num_kv_heads, chunks, d->num_blocks, static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "append_at_end_kernel launch");
  return PKV_OK;
}

int append_impl(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t num_tokens,
                void* k_cache, void* v_cache, const pkv_dims* d, cudaStream_t stream) {
  int rc = check_dims(d, false);
  if (rc != PKV_OK) return rc;
  if (num_tokens < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "append: num_tokens < 0");
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache)
    return pkv_fail(PKV_ERR_INVALID_ARG, "append: NULL pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 4))
    return pkv_fail(PKV_ERR_INVALID_ARG, "append: misaligned pointer (values need 16 bytes)");
  const int32_t chunks = d->head_dim * 2 / 16;
  const int64_t total = static_cast<int64_t>(num_tokens) * d->num_kv_heads * chunks;
  const int threads = 256;
  const int64_t blocks64 = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(blocks64 < 65536 ? blocks64 : 65536);
  pkv::append_kernel<<<blocks, threads, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, num_tokens, d->num_kv_heads,
      chunks, static_cast<int64_t>(d->num_blocks) * pkv::kBlockSize, static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "append_kernel launch");
  return PKV_OK;
}

// Slot-mapped append into an E4M3 pool (head_dim 128 or 64: any multiple of 8
// works for the copy; the attention side needs 128).
int append_fp8_impl(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t num_tokens,
                    void* k_cache, void* v_cache, const float* k_scale, const float* v_scale, const pkv_dims* d,
                    cudaStream_t stream) {
  int rc = check_dims(d, false);
  if (rc != PKV_OK) return rc;
  if (num_tokens < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "append_fp8: num_tokens < 0");
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
    return pkv_fail(PKV_ERR_INVALID_ARG, "append_fp8: NULL pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 8) || !aligned(v_cache, 8) ||
      !aligned(slot_mapping, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return pkv_fail(PKV_ERR_INVALID_ARG, "append_fp8: misaligned pointer (values 16 bytes, caches 8)");
  const int32_t groups = d->head_dim / 8;
  const int64_t total = static_cast<int64_t>(num_tokens) * d->num_kv_heads * groups;
  const int threads = 256;
  const int64_t blocks64 = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(blocks64 < 65536 ? blocks64 : 65536);
  const int64_t slots = static_cast<int64_t>(d->num_blocks) * pkv::kBlockSize;
  auto kv = [&](auto kern) {
    kern<<<blocks, threads, 0, stream>>>(static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                                         slot_mapping, num_tokens, d->num_kv_heads, groups, slots,
                                         static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), k_scale,
                                         v_scale);
  };
  if (d->dtype == PKV_DTYPE_BF16)
    kv(pkv::append_fp8_kernel<__nv_bfloat16>);
  else
    kv(pkv::append_fp8_kernel<__half>);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "append_fp8_kernel launch");
  return PKV_OK;
}

// ------------------------------------------------------------------ several new tokens per sequence

// Splits of the multi-token kernels: 512-token splits, at least 2 blocks per
// query row of a (sequence, KV head) unit with more than 8 rows (its split
// partials, 8 bytes per row and dimension written and read back, then stay
// under 1/16 of the K/V bytes the split reads), more splits when the units
// alone would not give two CTAs per SM.
void multi_plan(const pkv_dims* d, int32_t q_len, int32_t requested, int32_t* splits, int32_t* split_blocks) {
  const int32_t mb = d->max_blocks_per_seq;
  const int32_t rows = d->num_kv_heads > 0 ? d->num_q_heads / d->num_kv_heads * q_len : 1;
  const int32_t min_per = rows > 8 ? std::max<int32_t>(kAutoSplitBlocks, 2 * rows) : kAutoSplitBlocks;
  if (mb <= 1) {
    *splits = 1;
    *split_blocks = mb > 0 ? mb : 1;
    return;
  }
  int64_t n = requested;
  if (n == 0) {
    const int64_t units = static_cast<int64_t>(d->num_seqs) * d->num_kv_heads;
    n = (mb + min_per - 1) / min_per;
    const int64_t fill = (2 * static_cast<int64_t>(device_sms()) + units - 1) / units;
    if (fill > n) n = fill;
  }
  if (n > mb) n = mb;
  if (n < 1) n = 1;
  const int32_t per = static_cast<int32_t>((mb + n - 1) / n);
  *split_blocks = per;
  *splits = (mb + per - 1) / per;
}

size_t multi_workspace(const pkv_dims* d, int32_t q_len, int32_t splits) {
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(d->num_seqs) * q_len * d->num_q_heads * splits;
  return align256(rows * d->head_dim * sizeof(float)) + align256(rows * sizeof(float));
}

int check_multi(const pkv_dims* d, int32_t q_len, int32_t num_splits) {
  int rc = check_dims(d, true);
  if (rc != PKV_OK) return rc;
  if (q_len < 1 || q_len > pkv::kMaxQueryLen)
    return pkv_fail(PKV_ERR_UNSUPPORTED, "multi-token decode: q_len must be 1.." + std::to_string(pkv::kMaxQueryLen));
  if (num_splits < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "num_splits must be >= 0");
  if (static_cast<int64_t>(d->num_seqs) * q_len * d->num_q_heads >= (int64_t(1) << 31))
    return pkv_fail(PKV_ERR_UNSUPPORTED, "multi-token decode: too many query rows");
  return PKV_OK;
}

// Attention for q_len new tokens per sequence, optionally preceded by the
// append of their K/V (k_new / v_new non-null) at positions L - q_len .. L - 1.
int decode_multi_impl(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, int32_t q_len, float scale,
                      void* out, int32_t num_splits, void* workspace, size_t workspace_bytes, const pkv_dims* d,
                      cudaStream_t stream, bool tensor_cores = false) {
  int rc = check_multi(d, q_len, num_splits);
  if (rc != PKV_OK) return rc;
  if (tensor_cores && (d->num_kv_heads < 1 || d->num_q_heads / d->num_kv_heads * q_len != pkv::Tc2::kRows ||
                       d->head_dim != 128 || d->num_kv_heads % 2 != 0))
    return pkv_fail(PKV_ERR_UNSUPPORTED,
                    "decode_step_multi_tc: needs 64 query rows per KV head (group x q_len), head_dim 128 and an even "
                    "number of KV heads");
  if (d->num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || (!block_tables && d->max_blocks_per_seq > 0) || !context_lens || !out)
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_attention_multi: NULL pointer");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_attention_multi: misaligned pointer (q/out/caches need 16 bytes)");
  if (!std::isfinite(scale)) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_attention_multi: scale is not finite");
  const bool append = k_new != nullptr;
  if (append != (v_new != nullptr))
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_step_multi: k_new and v_new must both be given");
  if (append && (!aligned(k_new, 16) || !aligned(v_new, 16)))
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_step_multi: k_new / v_new must be 16-byte aligned");
  int32_t splits, split_blocks;
  multi_plan(d, q_len, num_splits, &splits, &split_blocks);
  const size_t need = multi_workspace(d, q_len, splits);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_attention_multi: workspace missing, too small (" +
                                             std::to_string(need) + " bytes needed) or not 256-byte aligned");
  const bool bf16 = d->dtype == PKV_DTYPE_BF16;
  cudaError_t e;
  if (append && d->max_blocks_per_seq > 0) {
    const int32_t chunks = d->head_dim * 2 / 16;
    const int64_t total = static_cast<int64_t>(d->num_seqs) * q_len * d->num_kv_heads * chunks;
    const int64_t blocks64 = (total + 255) / 256;
    pkv::append_multi_kernel<<<static_cast<int>(blocks64 < 65536 ? blocks64 : 65536), 256, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), block_tables, context_lens,
        d->num_seqs, q_len, d->max_blocks_per_seq, d->num_kv_heads, chunks, d->num_blocks,
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache));
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "append_multi_kernel launch");
  }
  CUtensorMap mk, mv;
  if ((rc = g_maps.get(k_cache, d, false, &mk)) != PKV_OK) return rc;
  if ((rc = g_maps.get(v_cache, d, false, &mv)) != PKV_OK) return rc;
  pkv::DecodeArgs args = {};
  args.q = q;
  args.out = out;
  args.block_tables = block_tables;
  args.context_lens = context_lens;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t rows = static_cast<size_t>(d->num_seqs) * q_len * d->num_q_heads;
  args.part_o = need ? reinterpret_cast<float*>(ws) : nullptr;
  args.part_lse = need ? reinterpret_cast<float*>(ws + align256(rows * splits * d->head_dim * sizeof(float)))
                       : nullptr;
  args.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  args.recheck = 0;  // the multi-token kernels are stream-ordered: no early reads
  args.num_seqs = d->num_seqs;
  args.num_q_heads = d->num_q_heads;
  args.num_kv_heads = d->num_kv_heads;
  args.group = d->num_q_heads / d->num_kv_heads;
  args.max_blocks = d->max_blocks_per_seq;
  args.num_blocks = d->num_blocks;
  args.num_splits = splits;
  args.split_blocks = split_blocks;
  // More than 8 query rows per KV head: 16 rows per warp in the mma M
  // dimension, two blocks per step for 64 rows (one otherwise, which keeps
  // more CTAs resident for fewer rows); else one warp with the rows in N.
  const bool rows_in_m = args.group * q_len > 8;
  const int nq = rows_in_m ? (args.group * q_len + pkv::kQueryRowsPerWarp - 1) / pkv::kQueryRowsPerWarp : 1;
  const bool two_blocks = nq == pkv::kMaxQueryWarps;
  const dim3 grid(splits, d->num_kv_heads, d->num_seqs);
  // The row kernel dispatches every unit's first split before any later one
  // when the units alone give at least 8 CTAs per SM (measured, Llama-70B tail
  // q_len 8: 0.540 -> 0.560 of the copy peak; with 512 units, Llama-8B B=64,
  // interleaved splits balance the tail better: 0.745 against 0.735).
  const int64_t units = static_cast<int64_t>(d->num_seqs) * d->num_kv_heads;
  const int32_t split_major = splits > 1 && units >= 8 * static_cast<int64_t>(device_sms()) ? 1 : 0;
  const dim3 rgrid = split_major ? dim3(d->num_seqs, d->num_kv_heads, splits) : grid;
  auto launch_rows = [&](auto kern, int smem, auto merge, auto typed_out) -> int {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute(decode_multi_rows_kernel)");
    kern<<<rgrid, (nq + 1) * 32, smem, stream>>>(mk, mv, args, q_len, split_major);
    err = cudaGetLastError();
    if (err != cudaSuccess) return cuda_fail(err, "decode_multi_rows_kernel launch");
    if (splits > 1) {
      merge<<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(
          args.part_o, args.part_lse, context_lens, static_cast<decltype(typed_out)>(out), d->num_seqs,
          q_len * d->num_q_heads, splits, split_blocks, d->max_blocks_per_seq);
      err = cudaGetLastError();
      if (err != cudaSuccess) return cuda_fail(err, "merge_split_kernel launch");
    }
    return PKV_OK;
  };
  auto launch = [&](auto kern, int smem, auto merge, auto typed_out) -> int {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute(multi-token decode kernel)");
    kern<<<grid, (nq + 1) * 32, smem, stream>>>(mk, mv, args, q_len);
    err = cudaGetLastError();
    if (err != cudaSuccess) return cuda_fail(err, "multi-token decode kernel launch");
    if (splits > 1) {
      merge<<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(
          args.part_o, args.part_lse, context_lens, static_cast<decltype(typed_out)>(out), d->num_seqs,
          q_len * d->num_q_heads, splits, split_blocks, d->max_blocks_per_seq);
      err = cudaGetLastError();
      if (err != cudaSuccess) return cuda_fail(err, "merge_split_kernel launch");
    }
    return PKV_OK;
  };
  // Dynamic shared memory: the ring (1024-byte aligned) and, for the row
  // kernel, each consumer warp's Q fragments (16 rows x head_dim x 2 bytes).
  auto pick = [&](auto kern_rows1, auto kern_rows2, auto kern_cols, auto merge, int stage_bytes,
                  auto typed_out) -> int {
    if (!rows_in_m) return launch(kern_cols, pkv::kMultiStages * stage_bytes + 1024, merge, typed_out);
    if (tensor_cores) {
      // One CTA per (split, pair of KV heads, sequence) on the tensor-core kernel.
      const void* kern = bf16 ? reinterpret_cast<const void*>(pkv::decode_multi_tc_kernel<__nv_bfloat16>)
                              : reinterpret_cast<const void*>(pkv::decode_multi_tc_kernel<__half>);
      cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pkv::Tc2::kSmem);
      if (err != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute(decode_multi_tc_kernel)");
      const dim3 tgrid(splits, d->num_kv_heads / 2, d->num_seqs);
      if (bf16)
        pkv::decode_multi_tc_kernel<__nv_bfloat16>
            <<<tgrid, pkv::Tc2::kThreads, pkv::Tc2::kSmem, stream>>>(mk, mv, args, q_len);
      else
        pkv::decode_multi_tc_kernel<__half><<<tgrid, pkv::Tc2::kThreads, pkv::Tc2::kSmem, stream>>>(mk, mv, args, q_len);
      err = cudaGetLastError();
      if (err != cudaSuccess) return cuda_fail(err, "decode_multi_tc_kernel launch");
      if (splits > 1) {
        merge<<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(
            args.part_o, args.part_lse, context_lens, static_cast<decltype(typed_out)>(out), d->num_seqs,
            q_len * d->num_q_heads, splits, split_blocks, d->max_blocks_per_seq);
        err = cudaGetLastError();
        if (err != cudaSuccess) return cuda_fail(err, "merge_split_kernel launch");
      }
      return PKV_OK;
    }
    const int qbytes = nq * pkv::kQueryRowsPerWarp * d->head_dim * 2;
    if (two_blocks)
      return launch_rows(kern_rows2, pkv::kRowStages2 * 2 * stage_bytes + 1024 + qbytes, merge, typed_out);
    return launch_rows(kern_rows1, pkv::kMultiStages * stage_bytes + 1024 + qbytes, merge, typed_out);
  };
  if (d->head_dim == 128) {
    if (bf16)
      return pick(pkv::decode_multi_rows_kernel<__nv_bfloat16, 128, pkv::kMultiStages, 1>,
                  pkv::decode_multi_rows_kernel<__nv_bfloat16, 128, pkv::kRowStages2, 2>,
                  pkv::decode_multi_query_kernel<__nv_bfloat16, 128, pkv::kMultiStages>,
                  pkv::merge_split_kernel<__nv_bfloat16, 128>, pkv::TileShape<128>::kStageBytes,
                  static_cast<__nv_bfloat16*>(nullptr));
    return pick(pkv::decode_multi_rows_kernel<__half, 128, pkv::kMultiStages, 1>,
                pkv::decode_multi_rows_kernel<__half, 128, pkv::kRowStages2, 2>,
                pkv::decode_multi_query_kernel<__half, 128, pkv::kMultiStages>, pkv::merge_split_kernel<__half, 128>,
                pkv::TileShape<128>::kStageBytes, static_cast<__half*>(nullptr));
  }
  if (bf16)
    return pick(pkv::decode_multi_rows_kernel<__nv_bfloat16, 64, pkv::kMultiStages, 1>,
                pkv::decode_multi_rows_kernel<__nv_bfloat16, 64, pkv::kRowStages2, 2>,
                pkv::decode_multi_query_kernel<__nv_bfloat16, 64, pkv::kMultiStages>,
                pkv::merge_split_kernel<__nv_bfloat16, 64>, pkv::TileShape<64>::kStageBytes,
                static_cast<__nv_bfloat16*>(nullptr));
  return pick(pkv::decode_multi_rows_kernel<__half, 64, pkv::kMultiStages, 1>,
              pkv::decode_multi_rows_kernel<__half, 64, pkv::kRowStages2, 2>,
              pkv::decode_multi_query_kernel<__half, 64, pkv::kMultiStages>, pkv::merge_split_kernel<__half, 64>,
              pkv::TileShape<64>::kStageBytes, static_cast<__half*>(nullptr));
}

}  // namespace

// ---- host <-> device copies of a host-buffer step

namespace {

// A host range and its device counterpart.
struct HostRange {
  void* dev;
  const void* host;
  size_t n;
};

// Device address of a host range that a kernel may access: both ends in
// pinned, device-mapped host memory (cudaHostAlloc / cudaHostRegister), at
// device addresses n - 1 apart.  False for pageable memory.
bool mapped_host_range(const void* p, size_t n, const uint8_t** dev) {
  if (!p || n == 0) return false;
  cudaPointerAttributes a, b;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return false;
  if (cudaPointerGetAttributes(&b, static_cast<const uint8_t*>(p) + (n - 1)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (b.type != cudaMemoryTypeHost ||
      static_cast<const uint8_t*>(b.devicePointer) != static_cast<const uint8_t*>(a.devicePointer) + (n - 1))
    return false;
  *dev = static_cast<const uint8_t*>(a.devicePointer);
  return true;
}

// Copies host -> device (to_dev) or device -> host.  Ranges that continue one
// another on both sides are merged first.  A merged run in mapped pinned host
// memory, 4-byte aligned on both sides, goes into one stage_copy_kernel launch
// (a programmatic launch in the stream's chain of kernels); any other run is
// a cudaMemcpyAsync, issued before that launch.  *kernel_copied tells whether
// the kernel ran.
int copy_host_ranges(const HostRange* r, int count, bool to_dev, cudaStream_t stream, bool* kernel_copied) {
  *kernel_copied = false;
  HostRange run[8];
  int nrun = 0;
  for (int i = 0; i < count; ++i) {
    if (r[i].n == 0) continue;
    if (nrun > 0) {
      HostRange& last = run[nrun - 1];
      if (static_cast<const uint8_t*>(last.host) + last.n == r[i].host &&
          static_cast<uint8_t*>(last.dev) + last.n == r[i].dev) {
        last.n += r[i].n;
        continue;
      }
    }
    run[nrun++] = r[i];
  }
  pkv::CopyList list = {};
  for (int i = 0; i < nrun; ++i) {
    const HostRange& c = run[i];
    const uint8_t* hdev = nullptr;
    const bool mapped = mapped_host_range(c.host, c.n, &hdev);
    const uintptr_t bits = reinterpret_cast<uintptr_t>(hdev) | reinterpret_cast<uintptr_t>(c.dev) | c.n;
    if (mapped && (bits & 3) == 0 && list.n < pkv::kMaxCopyRuns) {
      pkv::CopyRun& k = list.run[list.n++];
      k.src = to_dev ? hdev : static_cast<const uint8_t*>(c.dev);
      k.dst = to_dev ? static_cast<uint8_t*>(c.dev) : const_cast<uint8_t*>(hdev);
      k.shift = (bits & 15) == 0 ? 4 : 2;
      k.first = list.total;
      list.total += static_cast<int64_t>(c.n >> k.shift);
      continue;
    }
    const cudaError_t e = to_dev ? cudaMemcpyAsync(c.dev, c.host, c.n, cudaMemcpyHostToDevice, stream)
                                 : cudaMemcpyAsync(const_cast<void*>(c.host), c.dev, c.n, cudaMemcpyDeviceToHost,
                                                   stream);
    if (e != cudaSuccess) return cuda_fail(e, to_dev ? "step: host-to-device copy" : "step: device-to-host copy");
  }
  if (list.total == 0) return PKV_OK;
  constexpr int64_t per_cta = static_cast<int64_t>(pkv::kCopyThreads) * pkv::kCopyUnitsPerThread;
  int64_t grid = (list.total + per_cta - 1) / per_cta;
  if (grid > 4 * static_cast<int64_t>(device_sms())) grid = 4 * static_cast<int64_t>(device_sms());
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(pkv::kCopyThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = to_dev ? cudaLaunchKernelEx(&cfg, pkv::stage_copy_kernel<true>, list)
                               : cudaLaunchKernelEx(&cfg, pkv::stage_copy_kernel<false>, list);
  if (e != cudaSuccess) return cuda_fail(e, "stage_copy_kernel launch");
  *kernel_copied = true;
  return PKV_OK;
}

// One step from host buffers.  q_len new tokens per sequence (1: the
// one-token step; more: the multi-token step); k_scale / v_scale set: the
// pools hold E4M3 codes (one token only).
int step_from_host(const pkv_step_buffers* s, int32_t q_len, void* k_cache, void* v_cache, const float* k_scale,
                   const float* v_scale, float scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                   const pkv_dims* d, cudaStream_t stream) {
  int rc = check_dims(d, true);
  if (rc != PKV_OK) return rc;
  if (!s) return pkv_fail(PKV_ERR_INVALID_ARG, "step: buffers is NULL");
  if (q_len < 1 || q_len > pkv::kMaxQueryLen)
    return pkv_fail(PKV_ERR_UNSUPPORTED, "step: q_len must be 1.." + std::to_string(pkv::kMaxQueryLen));
  const size_t elem = 2;
  const size_t B = d->num_seqs;
  const size_t q_bytes = B * q_len * d->num_q_heads * d->head_dim * elem;
  const size_t kv_bytes = B * q_len * d->num_kv_heads * d->head_dim * elem;
  const size_t tbl_bytes = B * d->max_blocks_per_seq * sizeof(int32_t);
  const HostRange h2d[] = {{s->q_dev, s->q_host, q_bytes},
                           {s->k_new_dev, s->k_new_host, kv_bytes},
                           {s->v_new_dev, s->v_new_host, kv_bytes},
                           {s->block_tables_dev, s->block_tables_host, tbl_bytes},
                           {s->context_lens_dev, s->context_lens_host, B * sizeof(int32_t)}};
  for (const auto& c : h2d)
    if (c.n > 0 && (!c.dev || !c.host)) return pkv_fail(PKV_ERR_INVALID_ARG, "step: NULL staging or host buffer");
  bool kernel_copied = false;
  if ((rc = copy_host_ranges(h2d, 5, true, stream, &kernel_copied)) != PKV_OK) return rc;
  if (B == 0) return PKV_OK;
  if (!s->out_host || !s->out_dev) return pkv_fail(PKV_ERR_INVALID_ARG, "step: out_host or out_dev is NULL");
  if (q_len > 1) {
    // The multi-token launches are stream-ordered after the copy kernel.
    rc = decode_multi_impl(s->q_dev, s->k_new_dev, s->v_new_dev, k_cache, v_cache, s->block_tables_dev,
                           s->context_lens_dev, q_len, scale, s->out_dev, num_splits, workspace, workspace_bytes, d,
                           stream);
  } else {
    // After a copy kernel the decode kernel reads the lengths and tables
    // before its griddepcontrol.wait while the copy may still be staging them.
    // With the host inputs mapped, those early reads go to the host buffers
    // (the same values) and the decode kernel launches early, as in a chain
    // of device steps; otherwise it waits for the copy to finish.
    const uint8_t* pre_lens = nullptr;
    const uint8_t* pre_tables = nullptr;
    bool early = !kernel_copied;
    if (kernel_copied && mapped_host_range(s->context_lens_host, B * sizeof(int32_t), &pre_lens) &&
        (tbl_bytes == 0 || mapped_host_range(s->block_tables_host, tbl_bytes, &pre_tables)))
      early = true;
    else
      pre_lens = pre_tables = nullptr;
    const bool f8 = k_scale != nullptr;
    // The host buffers hold their final values before this call (the caller
    // wrote them), so the early reads need no re-check after the grid wait.
    rc = decode_impl(s->q_dev, s->k_new_dev, s->v_new_dev, k_cache, v_cache, s->block_tables_dev,
                     s->context_lens_dev, scale, s->out_dev, num_splits, workspace, workspace_bytes, d, stream, f8,
                     k_scale, v_scale, early, reinterpret_cast<const int32_t*>(pre_lens),
                     reinterpret_cast<const int32_t*>(pre_tables), pre_lens == nullptr);
  }
  if (rc != PKV_OK) return rc;
  const HostRange d2h[] = {{s->out_dev, s->out_host, q_bytes}};
  return copy_host_ranges(d2h, 1, false, stream, &kernel_copied);
}

}  // namespace

int decode_step_host_written(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const float* k_scale, const float* v_scale, const int32_t* block_tables,
                             const int32_t* context_lens, float scale, void* out, void* workspace,
                             size_t workspace_bytes, const pkv_dims* dims, void* stream) {
  if (!k_new || !v_new) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_step: NULL k_new / v_new");
  return decode_impl(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out, 0, workspace,
                     workspace_bytes, dims, static_cast<cudaStream_t>(stream), k_scale != nullptr, k_scale, v_scale,
                     true, nullptr, nullptr, false);
}

extern "C" {

int paged_decode_attention_multi(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, const int32_t* context_lens, int32_t q_len,
                                 float scale, void* out, int32_t num_splits, void* workspace,
                                 size_t workspace_bytes, const pkv_dims* dims, void* stream) {
  return decode_multi_impl(q, nullptr, nullptr, const_cast<void*>(k_cache), const_cast<void*>(v_cache), block_tables,
                           context_lens, q_len, scale, out, num_splits, workspace, workspace_bytes, dims,
                           static_cast<cudaStream_t>(stream));
}

int paged_decode_step_multi(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens, int32_t q_len, float scale,
                            void* out, int32_t num_splits, void* workspace, size_t workspace_bytes,
                            const pkv_dims* dims, void* stream) {
  if (!k_new || !v_new) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_step_multi: NULL k_new / v_new");
  return decode_multi_impl(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, q_len, scale, out,
                           num_splits, workspace, workspace_bytes, dims, static_cast<cudaStream_t>(stream));
}

int paged_decode_step_multi_tc(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens, int32_t q_len, float scale,
                               void* out, int32_t num_splits, void* workspace, size_t workspace_bytes,
                               const pkv_dims* dims, void* stream) {
  if (!k_new || !v_new) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_step_multi_tc: NULL k_new / v_new");
  return decode_multi_impl(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, q_len, scale, out,
                           num_splits, workspace, workspace_bytes, dims, static_cast<cudaStream_t>(stream), true);
}

size_t paged_decode_multi_workspace_bytes(const pkv_dims* dims, int32_t q_len, int32_t num_splits) {
  if (check_multi(dims, q_len, num_splits) != PKV_OK) return 0;
  int32_t splits, split_blocks;
  multi_plan(dims, q_len, num_splits, &splits, &split_blocks);
  return multi_workspace(dims, q_len, splits);
}

int32_t paged_decode_multi_resolve_splits(const pkv_dims* dims, int32_t q_len, int32_t num_splits) {
  int rc = check_multi(dims, q_len, num_splits);
  if (rc != PKV_OK) return rc;
  int32_t splits, split_blocks;
  multi_plan(dims, q_len, num_splits, &splits, &split_blocks);
  return splits;
}

int paged_kv_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs, int32_t num_pairs,
                         const pkv_dims* d, int32_t cache_elem_bytes, void* stream_v) {
  if (!d) return pkv_fail(PKV_ERR_INVALID_ARG, "copy_blocks: dims is NULL");
  if (num_pairs < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "copy_blocks: num_pairs < 0");
  if (num_pairs == 0) return PKV_OK;
  if (cache_elem_bytes != 1 && cache_elem_bytes != 2)
    return pkv_fail(PKV_ERR_INVALID_ARG, "copy_blocks: cache_elem_bytes must be 1 (E4M3) or 2 (fp16/bf16)");
  if (d->num_kv_heads <= 0 || d->num_blocks <= 0 || d->head_dim <= 0 || d->head_dim % 16 != 0 ||
      d->block_size != pkv::kBlockSize)
    return pkv_fail(PKV_ERR_INVALID_ARG, "copy_blocks: bad dims");
  if (!k_cache || !v_cache || !block_pairs) return pkv_fail(PKV_ERR_INVALID_ARG, "copy_blocks: NULL pointer");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_pairs, 4))
    return pkv_fail(PKV_ERR_INVALID_ARG, "copy_blocks: misaligned pointer (caches need 16 bytes)");
  const int64_t chunks = static_cast<int64_t>(d->num_kv_heads) * pkv::kBlockSize * d->head_dim * cache_elem_bytes / 16;
  const int64_t total = chunks * num_pairs;
  const int64_t blocks64 = (total + 255) / 256;
  const int cap = 8 * device_sms();
  pkv::copy_blocks_kernel<<<static_cast<int>(blocks64 < cap ? blocks64 : cap), 256, 0,
                            static_cast<cudaStream_t>(stream_v)>>>(block_pairs, num_pairs, chunks, d->num_blocks,
                                                                   static_cast<uint4*>(k_cache),
                                                                   static_cast<uint4*>(v_cache));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks_kernel launch");
  return PKV_OK;
}

int paged_kv_selftest_wait(void* stream) {
  pkv::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "wait_selftest_kernel launch");
  return PKV_OK;
}

int paged_kv_selftest_stale_prologue(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                                     const int32_t* stale_block_tables, const int32_t* stale_context_lens,
                                     float scale, void* out, void* workspace, size_t workspace_bytes,
                                     int32_t publish, const pkv_dims* dims, void* stream) {
  if (!stale_block_tables || !stale_context_lens || !aligned(stale_block_tables, 4) ||
      !aligned(stale_context_lens, 4))
    return pkv_fail(PKV_ERR_INVALID_ARG, "selftest_stale_prologue: stale inputs missing or misaligned");
  return decode_impl(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out, 0, workspace,
                     workspace_bytes, dims, static_cast<cudaStream_t>(stream), false, nullptr, nullptr, true,
                     stale_context_lens, stale_block_tables, true, publish != 0);
}

int paged_kv_append_fp8(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t num_tokens,
                        void* k_cache, void* v_cache, const float* k_scale, const float* v_scale,
                        const pkv_dims* dims, void* stream) {
  return append_fp8_impl(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, k_scale, v_scale, dims,
                         static_cast<cudaStream_t>(stream));
}

int paged_decode_attention_fp8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                               const float* v_scale, const int32_t* block_tables, const int32_t* context_lens,
                               float scale, void* out, void* workspace, size_t workspace_bytes,
                               const pkv_dims* dims, void* stream) {
  return decode_impl(q, nullptr, nullptr, const_cast<void*>(k_cache), const_cast<void*>(v_cache), block_tables,
                     context_lens, scale, out, 0, workspace, workspace_bytes, dims,
                     static_cast<cudaStream_t>(stream), true, k_scale, v_scale);
}

int paged_decode_step_fp8(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                          const float* k_scale, const float* v_scale, const int32_t* block_tables,
                          const int32_t* context_lens, float scale, void* out, void* workspace,
                          size_t workspace_bytes, const pkv_dims* dims, void* stream) {
  if (!k_new || !v_new) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_step_fp8: NULL k_new / v_new");
  return decode_impl(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out, 0, workspace,
                     workspace_bytes, dims, static_cast<cudaStream_t>(stream), true, k_scale, v_scale);
}

int paged_kv_append(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t num_tokens,
                    void* k_cache, void* v_cache, const pkv_dims* dims, void* stream) {
  return append_impl(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, dims,
                     static_cast<cudaStream_t>(stream));
}

int paged_decode_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, float scale, void* out, int32_t num_splits, void* workspace,
                           size_t workspace_bytes, const pkv_dims* dims, void* stream) {
  return decode_impl(q, nullptr, nullptr, const_cast<void*>(k_cache), const_cast<void*>(v_cache), block_tables,
                     context_lens, scale, out, num_splits, workspace, workspace_bytes, dims,
                     static_cast<cudaStream_t>(stream));
}

int paged_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, float scale, void* out,
                      int32_t num_splits, void* workspace, size_t workspace_bytes, const pkv_dims* dims,
                      void* stream) {
  if (!k_new || !v_new) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_step: NULL k_new / v_new");
  return decode_impl(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out, num_splits,
                     workspace, workspace_bytes, dims, static_cast<cudaStream_t>(stream));
}

int32_t paged_decode_resolve_splits(const pkv_dims* dims, int32_t num_splits) {
  int rc = check_dims(dims, true);
  if (rc != PKV_OK) return rc;
  SplitPlan p;
  rc = plan_splits(dims, num_splits, &p);
  return rc != PKV_OK ? rc : (p.persistent ? 0 : p.num_splits);
}

size_t paged_decode_workspace_bytes(const pkv_dims* dims, int32_t num_splits) {
  if (check_dims(dims, true) != PKV_OK) return 0;
  SplitPlan p;
  if (plan_splits(dims, num_splits, &p) != PKV_OK) return 0;
  return workspace_layout(dims, p).total();
}

int paged_decode_step_from_host(const pkv_step_buffers* s, void* k_cache, void* v_cache, float scale,
                                int32_t num_splits, void* workspace, size_t workspace_bytes, const pkv_dims* d,
                                void* stream_v) {
  return step_from_host(s, 1, k_cache, v_cache, nullptr, nullptr, scale, num_splits, workspace, workspace_bytes, d,
                        static_cast<cudaStream_t>(stream_v));
}

int paged_decode_step_multi_from_host(const pkv_step_buffers* s, int32_t q_len, void* k_cache, void* v_cache,
                                      float scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                      const pkv_dims* d, void* stream_v) {
  return step_from_host(s, q_len, k_cache, v_cache, nullptr, nullptr, scale, num_splits, workspace, workspace_bytes,
                        d, static_cast<cudaStream_t>(stream_v));
}

int paged_decode_step_fp8_from_host(const pkv_step_buffers* s, void* k_cache, void* v_cache, const float* k_scale,
                                    const float* v_scale, float scale, void* workspace, size_t workspace_bytes,
                                    const pkv_dims* d, void* stream_v) {
  if (!k_scale || !v_scale) return pkv_fail(PKV_ERR_INVALID_ARG, "step_fp8_from_host: NULL k_scale / v_scale");
  return step_from_host(s, 1, k_cache, v_cache, k_scale, v_scale, scale, 0, workspace, workspace_bytes, d,
                        static_cast<cudaStream_t>(stream_v));
}

int paged_kv_check_status(void* stream_v) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "check_status: stream synchronize");
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_pkv_error_word, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e, "check_status: read error word");
  if (word == 0) return PKV_OK;
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_pkv_error_word, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "check_status: clear error word");
  std::string msg = "kernel reported:";
  if (word & pkv::kErrBlockId) msg += " block id out of range;";
  if (word & pkv::kErrSlot) msg += " append slot out of range;";
  if (word & pkv::kErrContext) msg += " context length out of range;";
  if (word & pkv::kErrTimeout) msg += " a bounded wait gave up;";
  if (word & pkv::kErrQuery) msg += " a query value exceeds the fp16 range (fp8 cache path);";
  return pkv_fail((word & pkv::kErrTimeout) ? PKV_ERR_TIMEOUT : PKV_ERR_OUT_OF_RANGE, msg);
}

const char* paged_kv_last_error(void) { return pkv_error_slot().c_str(); }

}  // extern "C"

// ------------------------------------------------------------------ scratch without allocation
//
// Some callers cannot allocate device memory at the moment they run attention:
// plugin hosts that hand a kernel a fixed context and forbid allocation while
// enqueuing work, processes whose device memory is already reserved in full by
// another allocator (so a raw cudaMalloc would fail or break that allocator's
// budget), and latency-critical paths where cudaMalloc's implicit device
// synchronisation is not acceptable.  paged_decode_attention_no_alloc serves
// them: its scratch is a fixed array in this library's device memory, so the
// call allocates nothing.  Every GPU that loads the library holds the array
// until the process exits.

namespace {
constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB per device
}  // namespace

static __device__ __align__(256) unsigned char g_pkv_static_scratch[kStaticScratchBytes];

namespace {

// Device address of the scratch array for the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and kept.  The stream must
// belong to the current device: the address is that device's, and kernels on
// another device's stream would write to the wrong GPU.
int static_scratch(cudaStream_t stream, void** ptr) {
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "no_alloc: cudaGetDevice");
  if (dev >= kMaxDevices) return pkv_fail(PKV_ERR_UNSUPPORTED, "no_alloc: device index too large");
  int stream_dev = dev;
  e = cudaStreamGetDevice(stream, &stream_dev);
  if (e != cudaSuccess) return cuda_fail(e, "no_alloc: cudaStreamGetDevice");
  if (stream_dev != dev)
    return pkv_fail(PKV_ERR_INVALID_ARG, "no_alloc: the stream belongs to device " + std::to_string(stream_dev) +
                                             " but device " + std::to_string(dev) + " is current");
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pkv_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "no_alloc: cudaGetSymbolAddress(scratch)");
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" int paged_decode_attention_no_alloc(const void* q, const void* k_cache, const void* v_cache,
                                               const int32_t* block_tables, const int32_t* context_lens,
                                               float scale, void* out, int32_t num_splits, const pkv_dims* dims,
                                               void* stream) {
  int rc = check_dims(dims, true);
  if (rc != PKV_OK) return rc;
  if (num_splits < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "no_alloc: num_splits must be >= 0");
  // Always the split kernels: 0 picks 512-token splits.
  int32_t n = num_splits;
  if (n == 0) {
    n = (dims->max_blocks_per_seq + kAutoSplitBlocks - 1) / kAutoSplitBlocks;
    if (n < 1) n = 1;
  }
  SplitPlan plan;
  rc = plan_splits(dims, n, &plan);
  if (rc != PKV_OK) return rc;
  const size_t need = workspace_layout(dims, plan).total();
  if (need > kStaticScratchBytes)
    return pkv_fail(PKV_ERR_INVALID_ARG,
                    "no_alloc: this batch needs " + std::to_string(need) +
                        " bytes of split scratch; the library's static scratch holds " +
                        std::to_string(kStaticScratchBytes) + " (use fewer splits or paged_decode_attention)");
  void* scratch = nullptr;
  rc = static_scratch(static_cast<cudaStream_t>(stream), &scratch);
  if (rc != PKV_OK) return rc;
  return decode_impl(q, nullptr, nullptr, const_cast<void*>(k_cache), const_cast<void*>(v_cache), block_tables,
                     context_lens, scale, out, n, scratch, kStaticScratchBytes, dims,
                     static_cast<cudaStream_t>(stream));
}
