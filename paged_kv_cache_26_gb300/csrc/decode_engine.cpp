// Native continuous-batching decode engine: the host side of a decode loop
// over the paged KV cache, so that one call per step does all host work.
//
// Lifecycle after kasblo.com "vLLMとは？LLMサーバーを高速化する仕組み", section
// "blockはrequestの成長に合わせて割り当てる" (blocks for the prompt, one more when
// the current block fills, the blocks returned when the request ends and reused)
// and magi "Inference Batching", continuous batching (finished sequences leave
// and waiting ones enter at every iteration).
//
// The engine owns only host memory: pinned staging for the block tables, the
// copy-on-write block pairs and the prompts' slot mappings (two table / pair
// buffers, a ring of four slot buffers), each reused only after an event shows
// that the copy reading it finished.  Device buffers are the caller's.
//
// Parallel sampling (kasblo.com "vLLMとは？", section "block共有とAutomatic
// Prefix Caching"): decode_engine_fork starts a sequence that shares all of
// another's blocks; each step grows the batch with copy-on-write and copies
// the shared blocks that are about to be written before the step's append.
#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "paged_kv.h"
#include "pkv_errors.h"

namespace {
constexpr int kSlotRing = 4;
constexpr int kBlockSize = 16;
}  // namespace

struct pkv_decode_engine {
  pkv_block_allocator* alloc = nullptr;  // not owned
  int32_t max_batch = 0, max_blocks = 0;
  std::vector<int32_t> seq;              // sequence id per batch slot, -1 = empty
  std::vector<int64_t> remaining;        // tokens still to generate
  int32_t* tables_h[2] = {nullptr, nullptr};
  int32_t* lens_h[2] = {nullptr, nullptr};
  int32_t* pairs_h[2] = {nullptr, nullptr};
  cudaEvent_t copied[2] = {nullptr, nullptr};
  bool pending[2] = {false, false};
  int parity = 0;
  int last = -1;                         // table buffer of the last step
  int32_t* slots_h[kSlotRing] = {};
  const float* k_scale = nullptr;        // set: the pools hold E4M3 codes with these per-KV-head scales
  const float* v_scale = nullptr;
  cudaEvent_t adm_ev[kSlotRing] = {};
  bool adm_pending[kSlotRing] = {};
  int adm_i = 0;
  std::vector<int32_t> row;

  ~pkv_decode_engine() {
    for (int i = 0; i < 2; ++i) {
      if (copied[i]) cudaEventSynchronize(copied[i]), cudaEventDestroy(copied[i]);
      if (tables_h[i]) cudaFreeHost(tables_h[i]);
      if (lens_h[i]) cudaFreeHost(lens_h[i]);
      if (pairs_h[i]) cudaFreeHost(pairs_h[i]);
    }
    for (int i = 0; i < kSlotRing; ++i) {
      if (adm_ev[i]) cudaEventSynchronize(adm_ev[i]), cudaEventDestroy(adm_ev[i]);
      if (slots_h[i]) cudaFreeHost(slots_h[i]);
    }
  }
};

namespace {
int cuda_err(cudaError_t e, const char* what) {
  return pkv_fail(PKV_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}
}  // namespace

extern "C" {

pkv_decode_engine* decode_engine_create(pkv_block_allocator* alloc, int32_t max_batch, int32_t max_blocks_per_seq) {
  if (!alloc || max_batch <= 0 || max_blocks_per_seq <= 0) {
    pkv_set_error("decode_engine_create: bad argument");
    return nullptr;
  }
  auto* e = new pkv_decode_engine();
  e->alloc = alloc;
  e->max_batch = max_batch;
  e->max_blocks = max_blocks_per_seq;
  e->seq.assign(max_batch, -1);
  e->remaining.assign(max_batch, 0);
  e->row.resize(max_blocks_per_seq);
  const size_t tbl = static_cast<size_t>(max_batch) * max_blocks_per_seq * sizeof(int32_t);
  const size_t cap = static_cast<size_t>(max_blocks_per_seq) * kBlockSize * sizeof(int32_t);
  bool ok = true;
  for (int i = 0; i < 2 && ok; ++i) {
    ok = cudaHostAlloc(reinterpret_cast<void**>(&e->tables_h[i]), tbl, cudaHostAllocDefault) == cudaSuccess &&
         cudaHostAlloc(reinterpret_cast<void**>(&e->lens_h[i]), max_batch * sizeof(int32_t),
                       cudaHostAllocDefault) == cudaSuccess &&
         cudaHostAlloc(reinterpret_cast<void**>(&e->pairs_h[i]), 2 * max_batch * sizeof(int32_t),
                       cudaHostAllocDefault) == cudaSuccess &&
         cudaEventCreateWithFlags(&e->copied[i], cudaEventDisableTiming) == cudaSuccess;
  }
  for (int i = 0; i < kSlotRing && ok; ++i)
    ok = cudaHostAlloc(reinterpret_cast<void**>(&e->slots_h[i]), cap, cudaHostAllocDefault) == cudaSuccess &&
         cudaEventCreateWithFlags(&e->adm_ev[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    pkv_set_error("decode_engine_create: pinned host staging or event creation failed");
    delete e;
    return nullptr;
  }
  return e;
}

void decode_engine_destroy(pkv_decode_engine* e) { delete e; }

int decode_engine_admit(pkv_decode_engine* e, int32_t prompt_tokens, int32_t gen_tokens, const void* prompt_k,
                        const void* prompt_v, void* k_cache, void* v_cache, int32_t* slot_staging_dev,
                        const pkv_dims* dims, void* stream, int32_t* batch_slot) {
  if (!e || !batch_slot || !dims || prompt_tokens < 0 || gen_tokens < 1 ||
      (prompt_tokens > 0 && (!prompt_k || !prompt_v || !slot_staging_dev)))
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_admit: bad argument");
  *batch_slot = -1;
  if (static_cast<int64_t>(prompt_tokens) + gen_tokens > static_cast<int64_t>(e->max_blocks) * kBlockSize)
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_admit: prompt + generation exceed max_blocks_per_seq");
  int32_t slot = -1;
  for (int32_t i = 0; i < e->max_batch; ++i)
    if (e->seq[i] < 0) {
      slot = i;
      break;
    }
  if (slot < 0) return pkv_fail(PKV_ERR_NO_BLOCKS, "decode_engine_admit: no free batch slot");
  int32_t sid;
  int rc = block_allocator_add_seq(e->alloc, prompt_tokens, &sid);
  if (rc != PKV_OK) return rc;
  if (prompt_tokens > 0) {
    int32_t len;
    block_allocator_block_tables(e->alloc, &sid, 1, e->max_blocks, e->row.data(), &len);
    const int i = e->adm_i;
    e->adm_i = (i + 1) % kSlotRing;
    if (e->adm_pending[i]) cudaEventSynchronize(e->adm_ev[i]);
    int32_t* host = e->slots_h[i];
    for (int32_t p = 0; p < prompt_tokens; ++p) host[p] = e->row[p / kBlockSize] * kBlockSize + p % kBlockSize;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* dev = slot_staging_dev + static_cast<int64_t>(i) * e->max_blocks * kBlockSize;
    cudaError_t ce = cudaMemcpyAsync(dev, host, prompt_tokens * sizeof(int32_t), cudaMemcpyHostToDevice, s);
    if (ce != cudaSuccess) {
      block_allocator_free_seq(e->alloc, sid);
      return cuda_err(ce, "decode_engine_admit: slot copy");
    }
    cudaEventRecord(e->adm_ev[i], s);
    e->adm_pending[i] = true;
    rc = e->k_scale ? paged_kv_append_fp8(prompt_k, prompt_v, dev, prompt_tokens, k_cache, v_cache, e->k_scale,
                                          e->v_scale, dims, stream)
                    : paged_kv_append(prompt_k, prompt_v, dev, prompt_tokens, k_cache, v_cache, dims, stream);
    if (rc != PKV_OK) {
      block_allocator_free_seq(e->alloc, sid);
      return rc;
    }
  }
  e->seq[slot] = sid;
  e->remaining[slot] = gen_tokens;
  *batch_slot = slot;
  return PKV_OK;
}

int decode_engine_fork(pkv_decode_engine* e, int32_t src_slot, int32_t gen_tokens, int32_t* batch_slot) {
  if (!e || !batch_slot || gen_tokens < 1 || src_slot < 0 || src_slot >= e->max_batch || e->seq[src_slot] < 0)
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_fork: bad argument");
  *batch_slot = -1;
  const int32_t src = e->seq[src_slot];
  const int32_t len = block_allocator_seq_len(e->alloc, src);
  if (static_cast<int64_t>(len) + gen_tokens > static_cast<int64_t>(e->max_blocks) * kBlockSize)
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_fork: length + generation exceed max_blocks_per_seq");
  int32_t slot = -1;
  for (int32_t i = 0; i < e->max_batch; ++i)
    if (e->seq[i] < 0) {
      slot = i;
      break;
    }
  if (slot < 0) return pkv_fail(PKV_ERR_NO_BLOCKS, "decode_engine_fork: no free batch slot");
  int32_t sid;
  const int rc = block_allocator_fork(e->alloc, src, len, &sid);
  if (rc != PKV_OK) return rc;
  e->seq[slot] = sid;
  e->remaining[slot] = gen_tokens;
  *batch_slot = slot;
  return PKV_OK;
}

int decode_engine_step(pkv_decode_engine* e, int32_t* tables_dev, int32_t* lens_dev, int32_t* copy_pairs_dev,
                       const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache, float scale,
                       void* out, void* workspace, size_t workspace_bytes, const pkv_dims* dims, void* stream) {
  if (!e || !tables_dev || !lens_dev || !dims) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_step: bad argument");
  if (dims->num_seqs != e->max_batch || dims->max_blocks_per_seq != e->max_blocks)
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_step: dims must match the engine's batch and table width");
  const int i = e->parity;
  if (e->pending[i]) cudaEventSynchronize(e->copied[i]);  // the copies that last read these buffers are done
  int32_t ncopy = 0;
  int rc = block_allocator_step_batch_cow(e->alloc, e->seq.data(), e->max_batch, e->max_blocks, e->tables_h[i],
                                          e->lens_h[i], e->pairs_h[i], &ncopy);
  if (rc != PKV_OK) return rc;
  if (ncopy > 0 && !copy_pairs_dev)
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_step: shared blocks need copying but copy_pairs_dev is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t tbl = static_cast<size_t>(e->max_batch) * e->max_blocks * sizeof(int32_t);
  cudaError_t ce = cudaMemcpyAsync(tables_dev, e->tables_h[i], tbl, cudaMemcpyHostToDevice, s);
  if (ce == cudaSuccess)
    ce = cudaMemcpyAsync(lens_dev, e->lens_h[i], e->max_batch * sizeof(int32_t), cudaMemcpyHostToDevice, s);
  if (ce == cudaSuccess && ncopy > 0)
    ce = cudaMemcpyAsync(copy_pairs_dev, e->pairs_h[i], 2 * ncopy * sizeof(int32_t), cudaMemcpyHostToDevice, s);
  if (ce == cudaSuccess) ce = cudaEventRecord(e->copied[i], s);
  if (ce != cudaSuccess) return cuda_err(ce, "decode_engine_step: table copy");
  e->pending[i] = true;
  e->last = i;
  e->parity ^= 1;
  if (ncopy > 0) {
    rc = paged_kv_copy_blocks(k_cache, v_cache, copy_pairs_dev, ncopy, dims, e->k_scale ? 1 : 2, stream);
    if (rc != PKV_OK) return rc;
  }
  if (e->k_scale)
    return paged_decode_step_fp8(q, k_new, v_new, k_cache, v_cache, e->k_scale, e->v_scale, tables_dev, lens_dev,
                                 scale, out, workspace, workspace_bytes, dims, stream);
  return paged_decode_step(q, k_new, v_new, k_cache, v_cache, tables_dev, lens_dev, scale, out, 0, workspace,
                           workspace_bytes, dims, stream);
}

int decode_engine_set_kv_scales(pkv_decode_engine* e, const float* k_scale, const float* v_scale) {
  if (!e || (k_scale == nullptr) != (v_scale == nullptr))
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_set_kv_scales: give both scales or neither");
  e->k_scale = k_scale;
  e->v_scale = v_scale;
  return PKV_OK;
}

int decode_engine_finish(pkv_decode_engine* e, int32_t* freed_slots, int32_t* num_freed) {
  if (!e || !freed_slots || !num_freed) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_finish: bad argument");
  int32_t n = 0;
  for (int32_t i = 0; i < e->max_batch; ++i) {
    if (e->seq[i] < 0) continue;
    if (--e->remaining[i] <= 0) {
      block_allocator_free_seq(e->alloc, e->seq[i]);
      e->seq[i] = -1;
      e->remaining[i] = 0;
      freed_slots[n++] = i;
    }
  }
  *num_freed = n;
  return PKV_OK;
}

int decode_engine_state(const pkv_decode_engine* e, int32_t* slot_seq_ids, int32_t* context_lens) {
  if (!e || !slot_seq_ids || !context_lens) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_state: bad argument");
  for (int32_t i = 0; i < e->max_batch; ++i) {
    slot_seq_ids[i] = e->seq[i];
    context_lens[i] = e->seq[i] >= 0 ? block_allocator_seq_len(e->alloc, e->seq[i]) : 0;
  }
  return PKV_OK;
}

}  // extern "C"
