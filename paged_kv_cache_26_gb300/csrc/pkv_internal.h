// Library-internal entry points shared by the translation units of
// libpagedkv.so (not part of the C ABI in paged_kv.h).
#pragma once
#include <cstddef>
#include <cstdint>

#include "paged_kv.h"

// paged_decode_step (k_scale / v_scale null) or paged_decode_step_fp8 on the
// automatic path, for block tables and context lengths that the host wrote
// into mapped pinned memory before the call and that no kernel writes: the
// values the kernels read before their grid wait are final, so they are not
// read again after it.
int decode_step_host_written(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const float* k_scale, const float* v_scale, const int32_t* block_tables,
                             const int32_t* context_lens, float scale, void* out, void* workspace,
                             size_t workspace_bytes, const pkv_dims* dims, void* stream);
