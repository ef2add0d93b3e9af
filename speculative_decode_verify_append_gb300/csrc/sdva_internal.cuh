// sdva_internal.cuh -- the launch functions behind the C entry points, shared
// between the library's translation units (verify_step chains them).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sdva.h"

namespace sdva {

// Each returns SDVA_OK or the call's SDVA_ERR_*; with check_only it validates
// the arguments the same way and enqueues nothing.

// kv_append_quant / kv_append_quant_ragged (n_lane null: every lane writes n_new).
int append_launch(const sdva_kv_cache* cache, const void* k_new, const void* v_new, int num_lanes, int n_new,
                  const int32_t* n_lane, const int32_t* page_table, int max_pages_per_lane, const int32_t* seq_lens,
                  int32_t* status, sdva_stream_t stream, bool check_only = false);

// verify_attn / _tree / _ragged.  after_append: the kernel enqueued just
// before on the stream writes nothing but the cache, so the split kernel may
// be launched as its programmatic dependent (it waits before reading pages).
int verify_launch(const sdva_kv_cache* cache, const void* q, int num_q_heads, int num_lanes, int window,
                  const int32_t* parent, const int32_t* n_lane, const int32_t* page_table, int max_pages_per_lane,
                  const int32_t* seq_lens, int max_context, float sm_scale, void* out, void* workspace,
                  size_t workspace_bytes, int32_t* status, sdva_stream_t stream, bool after_append,
                  bool check_only = false);

// spec_accept.  after_verify: the kernel enqueued just before on the stream is
// verify_attn's merge, which writes nothing the argmax reads; the argmax is
// launched as its programmatic dependent and waits for it before finishing.
int accept_launch(const float* logits, int num_lanes, int window, int vocab, const int32_t* drafts,
                  int32_t* accept_len, int32_t* out_tokens, int32_t* seq_lens_inout, int32_t* status,
                  sdva_stream_t stream, bool after_verify, bool check_only = false);

}  // namespace sdva
