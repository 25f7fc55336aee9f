/*
 * paged_kv.h -- C ABI of libpagedkv.so: single-token decode attention over a
 * paged KV cache, the per-step slot-mapped KV append, and the host block
 * allocator that produces block tables.  One GPU, sm_103a (GB300).
 *
 * The method (vLLM-style PagedAttention) is stated on these pages:
 *  - kasblo.com "vLLMとは？LLMサーバーを高速化する仕組み", section
 *    "PagedAttentionはKV Cacheをblockで管理する": logical blocks of a request
 *    map to non-contiguous physical blocks through a per-request block table,
 *    and the attention kernel reads K/V through that table;
 *    section "blockはrequestの成長に合わせて割り当てる": blocks come from a pool,
 *    one more is added when the current block fills, and they return to the
 *    pool when the request ends; section "block共有とAutomatic Prefix Caching":
 *    blocks carry a reference count and can be shared by several sequences.
 *  - youngju.dev "LLM サービング最適化完全ガイド": the AttentionWithKVCache
 *    listing (one new query token against all cached K/V:
 *    softmax(Q K^T / sqrt(d_k)) V) and the PagedAttention memory-layout figure
 *    (fixed 16-token physical blocks, virtual slot -> block table -> physical block).
 *  - notes on "How to Scale Your Model, Part 7: Inference": section
 *    "Transformer 推論の基礎: Prefill と Generation" (each generated token's K/V
 *    is appended to the cache) and the GQA figure in section
 *    "生成スループット/レイテンシ改善のテクニック" (groups of query heads share one KV head).
 *
 * Layouts (all row-major, T = fp16 or bf16 as given by pkv_dims.dtype):
 *   k_cache, v_cache : T[num_blocks][num_kv_heads][block_size][head_dim]
 *                      token slot s lives in block s / block_size at offset
 *                      s % block_size.
 *   q, out           : T[num_seqs][num_q_heads][head_dim]
 *   k_new, v_new     : T[num_tokens][num_kv_heads][head_dim]
 *   block_tables     : int32[num_seqs][max_blocks_per_seq]; entry j of row b is
 *                      the physical block of sequence b's logical block j.
 *                      Entries at or past ceil(context_lens[b] / block_size) are
 *                      never read.
 *   context_lens     : int32[num_seqs], tokens attended by each sequence
 *                      (including the token appended this step).
 * Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *
 * Ownership: the caller allocates and owns every buffer.  Functions marked
 * "device" take device pointers; the library allocates no device memory.
 * Kernels run asynchronously on the given stream (a cudaStream_t passed as
 * void*, NULL = the legacy default stream).  Argument errors are reported
 * synchronously by the return value; errors found by the kernels themselves
 * (an out-of-range block id or slot, a context longer than its table, a device
 * wait that gave up) set a per-device error word that paged_kv_check_status()
 * reads and clears.
 *
 * Every function returns PKV_OK (0) or a negative PKV_ERR_* code;
 * paged_kv_last_error() gives a message for the calling thread's last failure.
 *
 * The automatic (persistent) attention path launches its kernels as
 * programmatic dependents of the kernel before them in the stream: they may
 * start while that kernel finishes.  Before waiting for it they read
 * block_tables and context_lens (and prefetch q) only as a guess, to start
 * their first loads early; after the wait they read the lengths and the
 * tables they started on again and rebuild everything derived from them if
 * anything changed, and only then use them.  So inputs written on the GPU
 * right before the call (a serving loop advancing context_lens, a new block
 * id stored into block_tables) are always seen, whether or not the kernel
 * that writes them signals programmatic launch completion early.  The cache,
 * the workspace, q and out are touched only after the wait.
 */
#ifndef PAGED_KV_H_
#define PAGED_KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, bad shape, Hkv does not divide Hq */
  PKV_ERR_UNSUPPORTED = -2,   /* head_dim, block_size, group size or dtype not compiled in */
  PKV_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed (message kept) */
  PKV_ERR_TIMEOUT = -4,       /* a kernel's bounded wait gave up */
  PKV_ERR_NO_BLOCKS = -5,     /* block allocator has too few free blocks */
  PKV_ERR_OUT_OF_RANGE = -6,  /* a kernel met a block id, slot or length outside its buffers */
  PKV_ERR_SHARED_BLOCK = -7   /* a write would land in a block other sequences share */
};

enum { PKV_DTYPE_FP16 = 0, PKV_DTYPE_BF16 = 1 };

typedef struct pkv_dims {
  int32_t num_seqs;            /* batch size B (also num_tokens for the append) */
  int32_t num_q_heads;         /* Hq */
  int32_t num_kv_heads;        /* Hkv; must divide Hq */
  int32_t head_dim;            /* D: 64 or 128 */
  int32_t block_size;          /* tokens per physical block: 16 */
  int32_t num_blocks;          /* physical blocks in each of k_cache / v_cache */
  int32_t max_blocks_per_seq;  /* width of block_tables */
  int32_t dtype;               /* PKV_DTYPE_FP16 or PKV_DTYPE_BF16 */
} pkv_dims;

/*
 * KV append (device).  Passage: "How to Scale Your Model, Part 7: Inference",
 * section "Transformer 推論の基礎: Prefill と Generation" (each generated token's
 * K/V is stored in the cache for later steps), through the slot of youngju.dev's
 * PagedAttention layout figure (virtual slot -> block table -> physical block).
 * For each token i in [0, num_tokens) with
 * slot_mapping[i] >= 0, copies k_new[i][:][:] into k_cache at slot
 * slot_mapping[i] (block slot / block_size, offset slot % block_size, every KV
 * head) and v_new[i] into v_cache likewise.  A negative slot skips the token.
 * Bit-exact copy.  Uses dims->num_kv_heads, head_dim, block_size, num_blocks,
 * dtype.  A slot >= num_blocks * block_size is skipped and flagged
 * (PKV_ERR_OUT_OF_RANGE from paged_kv_check_status).  All value pointers must
 * be 16-byte aligned.
 */
int paged_kv_append(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                    int32_t num_tokens, void* k_cache, void* v_cache,
                    const pkv_dims* dims, void* stream);

/*
 * Paged decode attention (device).  Passages: youngju.dev "LLM サービング最適化
 * 完全ガイド", AttentionWithKVCache listing (one query token: softmax(q K^T /
 * sqrt(d_k)) V); kasblo.com "vLLMとは？", section "PagedAttentionはKV Cacheを
 * blockで管理する" (K/V read through the block table); the GQA figure of "How to
 * Scale Your Model, Part 7", section "生成スループット/レイテンシ改善のテクニック".
 * For every sequence b and query head h,
 *   out[b][h] = sum_t softmax_t(scale * q[b][h] . K_t) V_t,  t in [0, context_lens[b]),
 * where K_t / V_t is token t of sequence b for KV head h / g, read from
 * physical block block_tables[b][t / block_size] at offset t % block_size.
 * Softmax and accumulation run in fp32 (online softmax); out is rounded once
 * to T.  context_lens[b] == 0 gives an all-zero row.
 *
 * num_splits: 0 = automatic: when num_seqs <= 2048 a persistent kernel (one
 * CTA per SM) cuts the batch's (sequence, KV head, block) space into equal
 * contiguous ranges, one per warp, whatever the length mix, and merges a
 * sequence cut across warps in the same launch; larger batches use 512-token
 * splits.  1 = one pass per (sequence, KV head).  n > 1 = each sequence is cut
 * into splits of ceil(max_blocks_per_seq / n) blocks, each split writes a
 * normalised fp32 partial and its log-sum-exp into the workspace, and a merge
 * kernel combines them.
 * The workspace (device) must hold paged_decode_workspace_bytes(dims,
 * num_splits) bytes, be 256-byte aligned, and be zero-filled before its first
 * use (and again after a call that reported an error); the kernels leave the
 * counters in it at zero (on the automatic path it also carries, from the
 * decode kernel to the merge of the same call, the lengths the decode kernel
 * used, under a per-call tag).  It may be NULL when that size is 0.  Calls
 * that share a workspace must not run concurrently.
 *
 * Requirements: head_dim 64 or 128, block_size 16, 1 <= Hq/Hkv <= 8,
 * caches and q/out 16-byte aligned, num_blocks * num_kv_heads * 16 < 2^31.
 * A block id outside [0, num_blocks) reads zeros and is flagged; a context
 * longer than max_blocks_per_seq * block_size is clamped and flagged.
 */
int paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* context_lens,
                           float scale, void* out, int32_t num_splits,
                           void* workspace, size_t workspace_bytes,
                           const pkv_dims* dims, void* stream);

/*
 * One decode step (device): the append of each sequence's new token followed
 * by paged decode attention.  Sequence b's token (k_new[b], v_new[b]:
 * T[num_seqs][num_kv_heads][head_dim]) is stored at position
 * context_lens[b] - 1, i.e. slot block_tables[b][(L-1)/16] * 16 + (L-1) % 16
 * with L = context_lens[b] (nothing for an empty context), and the attention
 * over positions [0, L) sees it.  Same results as paged_kv_append with that
 * slot mapping followed by paged_decode_attention.  On the automatic path
 * (num_splits = 0) the append runs inside the attention kernel, so a step is
 * one decode launch plus the merge; otherwise it is a separate append launch.
 * Arguments and requirements otherwise as paged_decode_attention.
 */
int paged_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, float scale, void* out,
                      int32_t num_splits, void* workspace, size_t workspace_bytes,
                      const pkv_dims* dims, void* stream);

/* The split count paged_decode_attention will use for this num_splits
 * argument: 0 for the persistent balanced kernel, >= 1 for the split kernel,
 * or a PKV_ERR_* code. */
int32_t paged_decode_resolve_splits(const pkv_dims* dims, int32_t num_splits);

/* Workspace bytes paged_decode_attention needs for these dims and num_splits
 * (0 when it runs in one pass). */
size_t paged_decode_workspace_bytes(const pkv_dims* dims, int32_t num_splits);

/*
 * One whole decode step from host memory: copies q, k_new, v_new,
 * block_tables and context_lens from host buffers into the caller's device
 * staging buffers, runs paged_decode_step on `stream`, and copies out back to
 * out_host.  The step is complete when the stream is; host inputs must stay
 * unchanged and out_host unread until then.  Inputs laid out back to back
 * (q, k_new, v_new, block_tables, context_lens) in one host buffer and one
 * device region, each at the same offsets, travel in a single copy.
 * Copies whose host side lies in pinned, device-mapped memory (cudaHostAlloc,
 * cudaHostRegister) and whose addresses and length are 4-byte aligned are made
 * by a copy kernel in the stream's chain of programmatic launches: it reads
 * the host inputs over the host link while the previous step's last kernel
 * finishes, and the output is written back by the same kernel after the
 * merge.  Other copies (pageable memory) are cudaMemcpyAsync calls.  When
 * context_lens_host and block_tables_host are mapped, the attention kernels
 * read them there (the same values the copy stages) before their grid wait,
 * so the decode kernel starts while the copy still runs; otherwise it starts
 * after the copy.  Every buffer stays the caller's; the kernels use them
 * until the stream reaches the end of the step.
 * Errors: PKV_ERR_INVALID_ARG for a NULL bufs, a NULL host or staging pointer
 * of a non-empty input, or NULL out pointers (nothing is launched for
 * num_seqs = 0 beyond the copies); PKV_ERR_CUDA for a failed copy or launch;
 * otherwise those of paged_decode_step.
 */
typedef struct pkv_step_buffers {
  const void* q_host;  const void* k_new_host;  const void* v_new_host;
  const int32_t* block_tables_host;  const int32_t* context_lens_host;  void* out_host;
  void* q_dev;  void* k_new_dev;  void* v_new_dev;
  int32_t* block_tables_dev;  int32_t* context_lens_dev;  void* out_dev;
} pkv_step_buffers;

int paged_decode_step_from_host(const pkv_step_buffers* bufs, void* k_cache, void* v_cache,
                                float scale, int32_t num_splits,
                                void* workspace, size_t workspace_bytes,
                                const pkv_dims* dims, void* stream);

/* paged_decode_step_multi from host memory: the same buffers and copies as
 * paged_decode_step_from_host with q_len new tokens per sequence (q, k_new,
 * v_new and out hold q_len rows per sequence: [B][q_len][...]); workspace as
 * paged_decode_multi_workspace_bytes gives for num_splits.  The multi-token
 * kernels start after the copy.  q_len outside 1..8 gives PKV_ERR_UNSUPPORTED;
 * other errors as paged_decode_step_from_host and paged_decode_step_multi. */
int paged_decode_step_multi_from_host(const pkv_step_buffers* bufs, int32_t q_len, void* k_cache, void* v_cache,
                                      float scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                      const pkv_dims* dims, void* stream);

/* paged_decode_step_fp8 from host memory: the same buffers and copies as
 * paged_decode_step_from_host (q, k_new, v_new and out fp16/bf16 per
 * dims->dtype), over E4M3 pools with the per-KV-head scales k_scale / v_scale
 * (device float32[num_kv_heads]); num_splits is 0 (the persistent path). */
int paged_decode_step_fp8_from_host(const pkv_step_buffers* bufs, void* k_cache, void* v_cache,
                                    const float* k_scale, const float* v_scale, float scale,
                                    void* workspace, size_t workspace_bytes,
                                    const pkv_dims* dims, void* stream);

/*
 * Paged decode attention that allocates nothing (device).  There is no
 * counterpart on the pages: this is a convenience of this library.  It is for
 * callers that cannot allocate device memory when they run attention: plugin
 * hosts that forbid allocation while enqueuing work, processes whose device
 * memory another allocator already holds in full, and latency-critical paths
 * that cannot take cudaMalloc's implicit synchronisation.  Same inputs, output
 * and result as paged_decode_attention with the split kernels (num_splits 0 =
 * 512-token splits, n >= 1 = n splits), but the split scratch is a fixed
 * 16 MiB array in the library's device memory, held on every GPU that loads
 * the library until the process exits.
 *  - A batch needing more than 16 MiB of scratch (num_seqs * num_q_heads *
 *    splits * (head_dim + 1) * 4 bytes, each region rounded up to 256) is
 *    rejected with PKV_ERR_INVALID_ARG and a message giving both sizes.
 *  - The first call on a device looks up the array's device address (with that
 *    device current); make that first call before any stream capture.  The
 *    stream must belong to the current device (PKV_ERR_INVALID_ARG
 *    otherwise).  The address is kept for the life of the process: calls made
 *    after a cudaDeviceReset of that device are not supported.
 *  - Every call on a device shares the one array and nothing in it needs to
 *    start at zero, but calls that overlap on the GPU (other streams, other
 *    host threads) race on it: serialise them, e.g. on one stream.
 */
int paged_decode_attention_no_alloc(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, const int32_t* context_lens,
                                    float scale, void* out, int32_t num_splits,
                                    const pkv_dims* dims, void* stream);

/* ------------------------------------------------------------------------
 * FP8 (E4M3) KV cache.  design.babushkai.com "GPU推論の内部構造", section
 * "KVキャッシュの台帳", and the quantisation section of youngju.dev "LLM
 * サービング最適化完全ガイド": storing K/V in FP8 halves the cache's bytes per
 * token, so decode attention -- bound by reading the cache -- moves half the
 * bytes.  The pages fix neither the FP8 format nor the scaling; this library
 * takes E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, S.1111.111 = NaN, largest finite 448) with one float32 scale per
 * KV head for K and one for V:  value = E4M3(code) * scale.
 *
 * Layouts: k_cache, v_cache : uint8[num_blocks][num_kv_heads][block_size][head_dim]
 *                             (E4M3 codes, same slot rule as above)
 *          k_scale, v_scale : float32[num_kv_heads] (device), finite and > 0
 *          q, out, k_new, v_new: T as above (pkv_dims.dtype is their type).
 * Quantisation (append): code = E4M3(float32(x) / scale) -- IEEE float32
 * division, round to nearest even, magnitudes past 448 saturate to 448.
 * Attention: the plain attention of the dequantised cache, as
 * paged_decode_attention computes it for fp16/bf16 caches.  The products run
 * as fp16 tensor-core mma (E4M3 values are exact in fp16), so a bf16 query is
 * converted to fp16: a query entry beyond +-65504 sets the error word
 * (PKV_ERR_OUT_OF_RANGE from paged_kv_check_status).
 * Limits: head_dim 128 for attention; at most 2048 sequences per call; only
 * the automatic persistent path (its workspace is
 * paged_decode_workspace_bytes(dims, 0) bytes, zero-filled once, as above).
 * Bad shapes and pointers return PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED.
 * ---------------------------------------------------------------------- */

/* Slot-mapped append of num_tokens tokens into an E4M3 pool (device).  Same
 * slot rule and error behaviour as paged_kv_append; caches 8-byte aligned,
 * k_new / v_new 16-byte aligned. */
int paged_kv_append_fp8(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                        int32_t num_tokens, void* k_cache, void* v_cache, const float* k_scale,
                        const float* v_scale, const pkv_dims* dims, void* stream);

/* Decode attention over an E4M3 pool (device); arguments as
 * paged_decode_attention with the automatic path. */
int paged_decode_attention_fp8(const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, const int32_t* context_lens,
                               float scale, void* out, void* workspace, size_t workspace_bytes,
                               const pkv_dims* dims, void* stream);

/* One decode step over an E4M3 pool (device): quantise and append each
 * sequence's token at position context_lens[b] - 1, then attend, in one fused
 * launch; arguments as paged_decode_step with the automatic path. */
int paged_decode_step_fp8(const void* q, const void* k_new, const void* v_new, void* k_cache,
                          void* v_cache, const float* k_scale, const float* v_scale,
                          const int32_t* block_tables, const int32_t* context_lens, float scale,
                          void* out, void* workspace, size_t workspace_bytes,
                          const pkv_dims* dims, void* stream);

/* ------------------------------------------------------------------------
 * Several new tokens per sequence (speculative verification, chunked decode):
 * youngju.dev "LLM サービング最適化完全ガイド", speculative decoding section (the
 * target model checks several draft tokens in one pass) and
 * design.babushkai.com "GPU推論の内部構造", section "KVキャッシュの台帳" (chunked
 * prefill).  The pages give no kernel; the masking is the causal rule of
 * decoding itself.
 *
 * q, out       : T[num_seqs][q_len][num_q_heads][head_dim], 1 <= q_len <= 8
 * k_new, v_new : T[num_seqs][q_len][num_kv_heads][head_dim] (step only)
 * context_lens[b] = L counts the q_len new tokens, which sit at positions
 * L - q_len .. L - 1; new token i attends to positions [0, L - q_len + i]
 * (the cache before it and the new tokens up to itself).  A token whose
 * position would be negative (L < q_len) gets a zero row.  num_splits: 0 =
 * automatic (512-token splits, more when the batch alone would not fill the
 * GPU), n >= 1 = n splits.  Workspace: paged_decode_multi_workspace_bytes
 * bytes (0 for one split), 256-byte aligned; its contents need no
 * initialisation.  Errors as paged_decode_attention; q_len outside 1..8 gives
 * PKV_ERR_UNSUPPORTED.
 * ---------------------------------------------------------------------- */
int paged_decode_attention_multi(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, const int32_t* context_lens,
                                 int32_t q_len, float scale, void* out, int32_t num_splits,
                                 void* workspace, size_t workspace_bytes, const pkv_dims* dims,
                                 void* stream);

/* Append the q_len new tokens' K/V of every sequence (at positions
 * L - q_len .. L - 1 through its table; nothing for negative positions), then
 * paged_decode_attention_multi (device). */
int paged_decode_step_multi(const void* q, const void* k_new, const void* v_new, void* k_cache,
                            void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                            int32_t q_len, float scale, void* out, int32_t num_splits, void* workspace,
                            size_t workspace_bytes, const pkv_dims* dims, void* stream);

/* paged_decode_step_multi on the fifth-generation tensor cores (tcgen05
 * MMAs with accumulators in tensor memory), for 64 query rows per KV head:
 * group x q_len == 64 (for example 64 query heads over 8 KV heads at q_len 8),
 * head_dim 128, an even number of KV heads.  Defining passage as
 * paged_decode_step_multi (youngju.dev "LLM サービング最適化完全ガイド",
 * speculative decoding section).  Same arguments, layouts, ownership,
 * workspace and results (within the attention tolerance: both kernels
 * accumulate in fp32 with the same weight rounding); other shapes give
 * PKV_ERR_UNSUPPORTED before any launch.  One CTA per pair of KV heads of a
 * sequence; the default paged_decode_step_multi is faster on GB300 for now. */
int paged_decode_step_multi_tc(const void* q, const void* k_new, const void* v_new, void* k_cache,
                               void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                               int32_t q_len, float scale, void* out, int32_t num_splits, void* workspace,
                               size_t workspace_bytes, const pkv_dims* dims, void* stream);

/* Workspace bytes, and the number of splits, a multi-token call with these
 * arguments uses (0 bytes / a negative error code for invalid arguments). */
size_t paged_decode_multi_workspace_bytes(const pkv_dims* dims, int32_t q_len, int32_t num_splits);
int32_t paged_decode_multi_resolve_splits(const pkv_dims* dims, int32_t q_len, int32_t num_splits);

/* Host helper: slots of each sequence's q_len newest tokens, slot_mapping[b][i]
 * for position L - q_len + i (-1 when negative).  Host pointers;
 * slot_mapping holds num_seqs * q_len entries. */
int paged_kv_slot_mapping_multi(const int32_t* block_tables, const int32_t* context_lens,
                                int32_t num_seqs, int32_t max_blocks, int32_t block_size,
                                int32_t q_len, int32_t* slot_mapping);

/* ------------------------------------------------------------------------
 * Copy-on-write of shared blocks: kasblo.com "vLLMとは？", section
 * "block共有とAutomatic Prefix Caching" (a block carries a reference count, is
 * shared by several sequences, and is duplicated only when one of them must
 * write into it: parallel sampling, a shared prefix that ends inside a block).
 * The allocator (block_allocator_fork / _append_slot_cow / _step_batch_cow
 * below) decides the copies; this call performs them (device): for each pair
 * block_pairs[i] = {src, dst} (int32[num_pairs][2], device), physical block
 * dst of k_cache and of v_cache becomes a copy of block src.  Destinations
 * must be distinct and not among the sources (the allocator's are fresh
 * blocks).  cache_elem_bytes: 2 for fp16/bf16 pools, 1 for E4M3 pools
 * (dims.dtype is not used).  Enqueue it before the append that writes into the
 * copies.  A pair outside [0, num_blocks) is skipped and flagged
 * (PKV_ERR_OUT_OF_RANGE from paged_kv_check_status).
 * ---------------------------------------------------------------------- */
int paged_kv_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs, int32_t num_pairs,
                         const pkv_dims* dims, int32_t cache_elem_bytes, void* stream);

/* Self-test of the kernels' bounded waits (device); no counterpart on the
 * pages.  Launches one warp that waits on a barrier nothing ever signals: the
 * wait gives up after its limit (1.5 s), sets the timeout bit of the error
 * word and the kernel returns, so the next paged_kv_check_status(stream)
 * returns PKV_ERR_TIMEOUT and the device stays usable.  Lets a caller (and the
 * tests) check the failure path without a real hang. */
int paged_kv_selftest_wait(void* stream);

/* Self-test of the kernels' re-check of their early inputs (device); no
 * counterpart on the pages.  paged_decode_step on the automatic path, except
 * that the decode and merge prologues -- which run before the grid wait, while
 * the previous kernel in the stream may still be writing the inputs -- read
 * stale_block_tables / stale_context_lens (same shapes as block_tables /
 * context_lens, device or mapped host memory) instead of the real inputs.
 * Such a read stands in for inputs whose latest writes are not yet visible.
 * After their wait the kernels read block_tables / context_lens again and
 * rebuild what they derived from the stale values, so out and the caches must
 * be exactly what paged_decode_step gives on the real inputs.  publish != 0:
 * the decode grid hands its validated lengths to the merge, as a
 * paged_decode_step outside stream capture does; 0: it does not, as under
 * capture, and the merge plans from the stale lengths before its own wait and
 * plans again after it.  Arguments and errors otherwise as paged_decode_step
 * with num_splits = 0. */
int paged_kv_selftest_stale_prologue(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                                     const int32_t* stale_block_tables, const int32_t* stale_context_lens,
                                     float scale, void* out, void* workspace, size_t workspace_bytes,
                                     int32_t publish, const pkv_dims* dims, void* stream);

/* Synchronises `stream`, then reads and clears this device's error word.
 * Returns PKV_OK, PKV_ERR_OUT_OF_RANGE, PKV_ERR_TIMEOUT or PKV_ERR_CUDA. */
int paged_kv_check_status(void* stream);

/* Message for the calling thread's last non-OK return (never NULL). */
const char* paged_kv_last_error(void);

/* Host helper: slot of each sequence's newest token,
 * slot_mapping[b] = block_tables[b][(L-1) / block_size] * block_size + (L-1) % block_size
 * with L = context_lens[b]; -1 when L == 0.  Host pointers. */
int paged_kv_slot_mapping(const int32_t* block_tables, const int32_t* context_lens,
                          int32_t num_seqs, int32_t max_blocks, int32_t block_size,
                          int32_t* slot_mapping);

/* ------------------------------------------------------------------------
 * Host block allocator (no device memory).  A pool of num_blocks physical
 * blocks of block_size tokens.  Free blocks are handed out in a seeded random
 * order so that a sequence's blocks are scattered through the pool.  Each
 * block has a reference count; a sequence may share whole leading blocks of
 * another (a common prefix).  Not thread-safe: one allocator per thread.
 * ---------------------------------------------------------------------- */
typedef struct pkv_block_allocator pkv_block_allocator;

/* A pool of num_blocks free blocks (kasblo.com "vLLMとは？", section
 * "blockはrequestの成長に合わせて割り当てる": blocks come from a pool).
 * Returns NULL if num_blocks <= 0 or block_size <= 0. */
pkv_block_allocator* block_allocator_create(int32_t num_blocks, int32_t block_size, uint64_t seed);
void block_allocator_destroy(pkv_block_allocator* a);

/* New sequence holding num_tokens tokens: ceil(num_tokens / block_size) blocks
 * (kasblo.com "vLLMとは？", section "blockはrequestの成長に合わせて割り当てる").
 * PKV_ERR_NO_BLOCKS (and no change) if the pool is short. */
int block_allocator_add_seq(pkv_block_allocator* a, int32_t num_tokens, int32_t* seq_id);

/* New sequence of num_tokens tokens whose first prefix_tokens tokens are the
 * blocks of src_seq (reference counts raised, nothing copied; kasblo.com
 * "vLLMとは？", section "block共有とAutomatic Prefix Caching").  prefix_tokens
 * must be a multiple of block_size and <= the length of src_seq. */
int block_allocator_fork_prefix(pkv_block_allocator* a, int32_t src_seq, int32_t prefix_tokens,
                                int32_t num_tokens, int32_t* seq_id);

/* A new sequence holding the first prefix_tokens tokens of src_seq (any
 * count 0..length; kasblo.com "vLLMとは？", section "block共有とAutomatic
 * Prefix Caching": shared blocks with reference counts): it shares the ceil(prefix_tokens / block_size) blocks that
 * hold them (their reference counts rise), the last possibly partly filled.
 * Parallel sampling forks the whole prompt; a request reusing part of
 * another's context forks that part.  Its writes go through the _cow calls
 * below, which copy a shared block before writing into it. */
int block_allocator_fork(pkv_block_allocator* a, int32_t src_seq, int32_t prefix_tokens, int32_t* seq_id);

/* append_slot with copy-on-write (kasblo.com "vLLMとは？", section "block共有と
 * Automatic Prefix Caching": a shared block is copied when one holder writes
 * into it): if the block that receives the token is shared, the sequence gets a fresh block in its place (the old block loses a
 * reference) and *num_copies = 1 with copy_pair = {old, fresh}: the caller
 * copies the block (paged_kv_copy_blocks) before writing the token.  Else
 * *num_copies = 0.  PKV_ERR_NO_BLOCKS (nothing changed) if a block is needed
 * and the pool is empty. */
int block_allocator_append_slot_cow(pkv_block_allocator* a, int32_t seq_id, int32_t* slot,
                                    int32_t* copy_pair, int32_t* num_copies);

/* step_batch with copy-on-write (the same passage): as block_allocator_step_batch, but a
 * sequence whose next token lands in a shared block gets a private copy
 * instead of an error.  copy_pairs (int32[n][2], host) receives the
 * *num_copies {src, dst} block copies to perform before this step's append;
 * when several sequences of the batch write into the same shared block, the
 * last of them keeps the original.  All or nothing: on an error nothing
 * changes. */
int block_allocator_step_batch_cow(pkv_block_allocator* a, const int32_t* slot_seq_ids, int32_t n,
                                   int32_t max_blocks, int32_t* tables, int32_t* context_lens,
                                   int32_t* copy_pairs, int32_t* num_copies);

/* Grow seq_id by one token and return its slot (block * block_size + offset).
 * Takes a new block when the last one is full (kasblo.com "vLLMとは？", section
 * "blockはrequestの成長に合わせて割り当てる": one more block when the current
 * one fills).  PKV_ERR_SHARED_BLOCK if the
 * token would land in a partly filled block that another sequence shares. */
int block_allocator_append_slot(pkv_block_allocator* a, int32_t seq_id, int32_t* slot);

/* One decode step's growth for a batch (the same passage): block_allocator_append_slot for each
 * of seq_ids[0..n), slots[i] receiving sequence i's new slot.  All or nothing:
 * PKV_ERR_NO_BLOCKS / PKV_ERR_SHARED_BLOCK / PKV_ERR_INVALID_ARG (a sequence
 * not live or listed twice) leave the allocator unchanged. */
int block_allocator_append_slots(pkv_block_allocator* a, const int32_t* seq_ids, int32_t n, int32_t* slots);

/* The host side of one continuous-batching decode step (magi "Inference
 * Batching", continuous batching; kasblo.com section "blockはrequestの成長に
 * 合わせて割り当てる"), in one call: for a
 * batch of n slots (slot_seq_ids[i] = a live sequence, or -1 for an empty
 * slot) grow every listed sequence by one token and write row i of
 * tables (int32[n][max_blocks], -1 padded) and context_lens[i] (0 for an empty
 * slot).  All or nothing, like block_allocator_append_slots; also
 * PKV_ERR_INVALID_ARG if a sequence would outgrow max_blocks. */
int block_allocator_step_batch(pkv_block_allocator* a, const int32_t* slot_seq_ids, int32_t n, int32_t max_blocks,
                               int32_t* tables, int32_t* context_lens);

/* Drop seq_id; blocks whose count reaches zero return to the pool (kasblo.com
 * "vLLMとは？", section "blockはrequestの成長に合わせて割り当てる": a finished
 * request's blocks go back to the pool). */
int block_allocator_free_seq(pkv_block_allocator* a, int32_t seq_id);

/* The block tables themselves (kasblo.com "vLLMとは？", section
 * "PagedAttentionはKV Cacheをblockで管理する": logical block j -> physical
 * block).  Export rows for seq_ids[0..n): tables int32[n][max_blocks] (-1 padded) and
 * context_lens int32[n].  PKV_ERR_INVALID_ARG if a sequence needs more than
 * max_blocks blocks. */
int block_allocator_block_tables(const pkv_block_allocator* a, const int32_t* seq_ids, int32_t n,
                                 int32_t max_blocks, int32_t* tables, int32_t* context_lens);

/* Free blocks left in the pool. */
int32_t block_allocator_num_free(const pkv_block_allocator* a);
/* Reference count of a physical block (0 = free; kasblo.com section "block共有と
 * Automatic Prefix Caching"); -1 if out of range. */
int32_t block_allocator_refcount(const pkv_block_allocator* a, int32_t block);
/* Tokens held by a live sequence; -1 if seq_id is not live. */
int32_t block_allocator_seq_len(const pkv_block_allocator* a, int32_t seq_id);

/* ------------------------------------------------------------------------
 * Continuous-batching decode engine (host; the kernels it launches are the
 * ones above).  A fixed number of batch slots over one block allocator: a
 * sequence is admitted with its prompt's K/V, grows by one token per step
 * (a new block when its last one fills), and frees its blocks when its
 * generation budget is spent, so later sequences reuse them (kasblo.com
 * "vLLMとは？" section "blockはrequestの成長に合わせて割り当てる"; magi "Inference
 * Batching", continuous batching).  One call does a step's host work: growth
 * of every active sequence, export of every table row, and the launch of
 * paged_decode_step.  The tables, context lengths, copy-on-write pairs and
 * prompt slot mappings are written into mapped pinned host memory that the
 * engine owns, and the kernels read them there in place: no host-to-device
 * copy is issued.  The engine allocates that host memory only; the caches,
 * q / k_new / v_new / out and the workspace are the caller's.  Not
 * thread-safe; one stream per engine.
 * ---------------------------------------------------------------------- */
typedef struct pkv_decode_engine pkv_decode_engine;

/* alloc stays owned by the caller and must outlive the engine.  Returns NULL
 * on a bad argument or if pinned host staging cannot be allocated. */
pkv_decode_engine* decode_engine_create(pkv_block_allocator* alloc, int32_t max_batch, int32_t max_blocks_per_seq);
void decode_engine_destroy(pkv_decode_engine* e);

/* Admit a sequence whose prompt_tokens K/V rows (prompt_k, prompt_v: device,
 * T[prompt_tokens][Hkv][D]) are written into the cache through a slot-mapped
 * append (its slot mapping is read from the engine's mapped host staging), and
 * which will take gen_tokens decode steps.  *batch_slot receives the slot (-1
 * and PKV_ERR_NO_BLOCKS when no slot or too few blocks are free). */
int decode_engine_admit(pkv_decode_engine* e, int32_t prompt_tokens, int32_t gen_tokens, const void* prompt_k,
                        const void* prompt_v, void* k_cache, void* v_cache, const pkv_dims* dims, void* stream,
                        int32_t* batch_slot);

/* E4M3 pools: with k_scale / v_scale (float32[num_kv_heads], device, owned by
 * the caller) set, the engine's pools hold E4M3 codes: admission appends
 * with paged_kv_append_fp8, steps run paged_decode_step_fp8, and
 * copy-on-write copies 1-byte elements.  NULL for both: fp16/bf16 pools. */
int decode_engine_set_kv_scales(pkv_decode_engine* e, const float* k_scale, const float* v_scale);

/* Parallel sampling: a new sequence in a free batch slot that shares every
 * block of the sequence in src_slot (its whole context so far; reference
 * counts rise, nothing is copied now) and runs gen_tokens steps.  The shared
 * block that a step writes into is copied first (copy-on-write, see
 * decode_engine_step).  PKV_ERR_NO_BLOCKS if no batch slot is free. */
int decode_engine_fork(pkv_decode_engine* e, int32_t src_slot, int32_t gen_tokens, int32_t* batch_slot);

/* One decode step for every active slot.  Blocks shared by forked sequences
 * that this step writes into are first copied (paged_kv_copy_blocks); then
 * paged_decode_step (paged_decode_step_fp8 with kv scales set) runs with
 * q / k_new / v_new / out covering all max_batch slots (empty slots: context
 * 0, zero output, nothing appended) and num_splits 0.  The step's block
 * tables, lengths and copy pairs come from a ring of three mapped pinned host
 * buffers; an entry is rewritten only after the kernels that read it have
 * finished (the call waits for them if the host is that far ahead).
 * dims->num_seqs must be max_batch and dims->max_blocks_per_seq the engine's
 * table width. */
int decode_engine_step(pkv_decode_engine* e, const void* q, const void* k_new, const void* v_new, void* k_cache,
                       void* v_cache, float scale, void* out, void* workspace, size_t workspace_bytes,
                       const pkv_dims* dims, void* stream);

/* The block tables (int32[max_batch][max_blocks_per_seq], -1 padded) and
 * context lengths (int32[max_batch]) the last step ran with, copied into
 * host arrays.  PKV_ERR_INVALID_ARG before the first step. */
int decode_engine_last_step(const pkv_decode_engine* e, int32_t* tables, int32_t* context_lens);

/* Totals over the steps since creation or the last reset. */
typedef struct pkv_engine_stats {
  int64_t steps;              /* decode_engine_step calls that launched */
  int64_t sequence_steps;     /* active sequences summed over steps = tokens generated */
  int64_t context_tokens;     /* context lengths summed over steps = tokens attended */
  int64_t unused_tail_slots;  /* unused slots of each active sequence's last block, summed over steps */
  int64_t copied_blocks;      /* copy-on-write block copies */
} pkv_engine_stats;
int decode_engine_get_stats(const pkv_decode_engine* e, pkv_engine_stats* stats);
int decode_engine_reset_stats(pkv_decode_engine* e);

/* Count the step against every active sequence; those that spent their
 * budget free their blocks.  freed_slots (host, max_batch entries) receives
 * their slots, *num_freed how many. */
int decode_engine_finish(pkv_decode_engine* e, int32_t* freed_slots, int32_t* num_freed);

/* Host view: sequence id (or -1) and current context length of every slot. */
int decode_engine_state(const pkv_decode_engine* e, int32_t* slot_seq_ids, int32_t* context_lens);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_H_ */
