// Native continuous-batching decode engine: the host side of a decode loop
// over the paged KV cache, so that one call per step does all host work.
//
// Lifecycle after kasblo.com "vLLMとは？LLMサーバーを高速化する仕組み", section
// "blockはrequestの成長に合わせて割り当てる" (blocks for the prompt, one more when
// the current block fills, the blocks returned when the request ends and reused)
// and magi "Inference Batching", continuous batching (finished sequences leave
// and waiting ones enter at every iteration).
//
// The engine owns only host memory: mapped pinned staging for the block
// tables, context lengths and copy-on-write block pairs of a step (a ring of
// three) and for the prompts' slot mappings (a ring of four).  The kernels of
// a step read that staging in place through its device mapping, so a step
// issues no host-to-device copy: a stream-ordered copy between two decode
// steps would cost more than the table it moves, since the next step's kernel
// could then no longer launch while the previous one finishes.  A staging
// buffer is rewritten only after an event shows that the kernels reading it
// have finished.
//
// Parallel sampling (kasblo.com "vLLMとは？", section "block共有とAutomatic
// Prefix Caching"): decode_engine_fork starts a sequence that shares all of
// another's blocks; each step grows the batch with copy-on-write and copies
// the shared blocks that are about to be written before the step's append.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <string>
#include <vector>

#include "paged_kv.h"
#include "pkv_errors.h"
#include "pkv_internal.h"

namespace {
constexpr int kSlotRing = 4;
constexpr int kStepRing = 3;
constexpr int kBlockSize = 16;

// One mapped pinned allocation: host address and the address kernels use.
struct Mapped {
  int32_t* h = nullptr;
  int32_t* d = nullptr;
  bool alloc(size_t entries) {
    if (cudaHostAlloc(reinterpret_cast<void**>(&h), entries * sizeof(int32_t), cudaHostAllocMapped) != cudaSuccess) {
      h = nullptr;
      return false;
    }
    return cudaHostGetDevicePointer(reinterpret_cast<void**>(&d), h, 0) == cudaSuccess;
  }
  void release() {
    if (h) cudaFreeHost(h);
    h = d = nullptr;
  }
};
}  // namespace

struct pkv_decode_engine {
  pkv_block_allocator* alloc = nullptr;  // not owned
  int32_t max_batch = 0, max_blocks = 0;
  std::vector<int32_t> seq;              // sequence id per batch slot, -1 = empty
  std::vector<int64_t> remaining;        // tokens still to generate
  // Step staging, per ring entry: [tables: max_batch * max_blocks][lens: max_batch][pairs: 2 * max_batch].
  Mapped step_buf[kStepRing];
  cudaEvent_t step_ev[kStepRing] = {};
  bool step_pending[kStepRing] = {};
  int step_i = 0;
  int last = -1;                         // ring entry of the last step
  Mapped slots[kSlotRing];
  cudaEvent_t adm_ev[kSlotRing] = {};
  bool adm_pending[kSlotRing] = {};
  int adm_i = 0;
  const float* k_scale = nullptr;        // set: the pools hold E4M3 codes with these per-KV-head scales
  const float* v_scale = nullptr;
  std::vector<int32_t> row;
  pkv_engine_stats stats = {};

  int32_t* tables(int i, bool dev) { return dev ? step_buf[i].d : step_buf[i].h; }
  int32_t* lens(int i, bool dev) { return tables(i, dev) + static_cast<int64_t>(max_batch) * max_blocks; }
  int32_t* pairs(int i, bool dev) { return lens(i, dev) + max_batch; }

  ~pkv_decode_engine() {
    for (int i = 0; i < kStepRing; ++i) {
      if (step_ev[i]) cudaEventSynchronize(step_ev[i]), cudaEventDestroy(step_ev[i]);
      step_buf[i].release();
    }
    for (int i = 0; i < kSlotRing; ++i) {
      if (adm_ev[i]) cudaEventSynchronize(adm_ev[i]), cudaEventDestroy(adm_ev[i]);
      slots[i].release();
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
  const size_t step_entries = static_cast<size_t>(max_batch) * max_blocks_per_seq + 3 * static_cast<size_t>(max_batch);
  const size_t slot_entries = static_cast<size_t>(max_blocks_per_seq) * kBlockSize;
  bool ok = true;
  for (int i = 0; i < kStepRing && ok; ++i)
    ok = e->step_buf[i].alloc(step_entries) &&
         cudaEventCreateWithFlags(&e->step_ev[i], cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; i < kSlotRing && ok; ++i)
    ok = e->slots[i].alloc(slot_entries) &&
         cudaEventCreateWithFlags(&e->adm_ev[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    pkv_set_error("decode_engine_create: mapped pinned host staging or event creation failed");
    delete e;
    return nullptr;
  }
  return e;
}

void decode_engine_destroy(pkv_decode_engine* e) { delete e; }

int decode_engine_admit(pkv_decode_engine* e, int32_t prompt_tokens, int32_t gen_tokens, const void* prompt_k,
                        const void* prompt_v, void* k_cache, void* v_cache, const pkv_dims* dims, void* stream,
                        int32_t* batch_slot) {
  if (!e || !batch_slot || !dims || prompt_tokens < 0 || gen_tokens < 1 ||
      (prompt_tokens > 0 && (!prompt_k || !prompt_v)))
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
    if (e->adm_pending[i]) cudaEventSynchronize(e->adm_ev[i]);  // the append that last read this buffer is done
    int32_t* host = e->slots[i].h;
    for (int32_t p = 0; p < prompt_tokens; ++p) host[p] = e->row[p / kBlockSize] * kBlockSize + p % kBlockSize;
    rc = e->k_scale ? paged_kv_append_fp8(prompt_k, prompt_v, e->slots[i].d, prompt_tokens, k_cache, v_cache,
                                          e->k_scale, e->v_scale, dims, stream)
                    : paged_kv_append(prompt_k, prompt_v, e->slots[i].d, prompt_tokens, k_cache, v_cache, dims,
                                      stream);
    if (rc != PKV_OK) {
      block_allocator_free_seq(e->alloc, sid);
      return rc;
    }
    const cudaError_t ce = cudaEventRecord(e->adm_ev[i], static_cast<cudaStream_t>(stream));
    if (ce != cudaSuccess) return cuda_err(ce, "decode_engine_admit: event record");
    e->adm_pending[i] = true;
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

int decode_engine_step(pkv_decode_engine* e, const void* q, const void* k_new, const void* v_new, void* k_cache,
                       void* v_cache, float scale, void* out, void* workspace, size_t workspace_bytes,
                       const pkv_dims* dims, void* stream) {
  if (!e || !dims) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_step: bad argument");
  if (dims->num_seqs != e->max_batch || dims->max_blocks_per_seq != e->max_blocks)
    return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_step: dims must match the engine's batch and table width");
  const int i = e->step_i;
  if (e->step_pending[i]) cudaEventSynchronize(e->step_ev[i]);  // the kernels that last read this entry are done
  int32_t ncopy = 0;
  int rc = block_allocator_step_batch_cow(e->alloc, e->seq.data(), e->max_batch, e->max_blocks, e->tables(i, false),
                                          e->lens(i, false), e->pairs(i, false), &ncopy);
  if (rc != PKV_OK) return rc;
  e->last = i;
  e->step_i = (i + 1) % kStepRing;
  if (ncopy > 0) {
    rc = paged_kv_copy_blocks(k_cache, v_cache, e->pairs(i, true), ncopy, dims, e->k_scale ? 1 : 2, stream);
    if (rc != PKV_OK) return rc;
  }
  // The tables and lengths were written by the host above and no kernel writes
  // them: the kernels may trust what they read before their grid wait.
  rc = decode_step_host_written(q, k_new, v_new, k_cache, v_cache, e->k_scale, e->v_scale, e->tables(i, true),
                                e->lens(i, true), scale, out, workspace, workspace_bytes, dims, stream);
  // Recorded even after a failed launch, so that the entry is never reused
  // while an earlier kernel (the block copy) may still read it.
  const cudaError_t ce = cudaEventRecord(e->step_ev[i], static_cast<cudaStream_t>(stream));
  e->step_pending[i] = ce == cudaSuccess;
  if (ce != cudaSuccess) cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (rc != PKV_OK) return rc;
  if (ce != cudaSuccess) return cuda_err(ce, "decode_engine_step: event record");
  const int32_t* L = e->lens(i, false);
  auto& st = e->stats;
  ++st.steps;
  st.copied_blocks += ncopy;
  for (int32_t b = 0; b < e->max_batch; ++b)
    if (L[b] > 0) {
      ++st.sequence_steps;
      st.context_tokens += L[b];
      st.unused_tail_slots += (L[b] + kBlockSize - 1) / kBlockSize * kBlockSize - L[b];
    }
  return PKV_OK;
}

int decode_engine_last_step(const pkv_decode_engine* e, int32_t* tables, int32_t* context_lens) {
  if (!e || !tables || !context_lens) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_last_step: bad argument");
  if (e->last < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_last_step: no step has run");
  auto* me = const_cast<pkv_decode_engine*>(e);
  std::memcpy(tables, me->tables(e->last, false), sizeof(int32_t) * static_cast<size_t>(e->max_batch) * e->max_blocks);
  std::memcpy(context_lens, me->lens(e->last, false), sizeof(int32_t) * static_cast<size_t>(e->max_batch));
  return PKV_OK;
}

int decode_engine_get_stats(const pkv_decode_engine* e, pkv_engine_stats* stats) {
  if (!e || !stats) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_get_stats: bad argument");
  *stats = e->stats;
  return PKV_OK;
}

int decode_engine_reset_stats(pkv_decode_engine* e) {
  if (!e) return pkv_fail(PKV_ERR_INVALID_ARG, "decode_engine_reset_stats: bad argument");
  e->stats = pkv_engine_stats{};
  return PKV_OK;
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
