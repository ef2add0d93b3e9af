// verify_step.cu -- the three calls of one verify step, enqueued as a chain of
// programmatic dependent launches.
//
// A speculative round ends with one verify pass of the main model over the
// window of 1 + d tokens (Baseten talk summary, section "추측 디코드"):
// append the window's K/V, attend, accept.  verify_step enqueues exactly
// kv_append_quant, verify_attn and spec_accept on one stream, with the same
// results, but lets each kernel start while its predecessor drains:
//   * the append is launched normally (it waits for all earlier work on the
//     stream) and lets its dependent be scheduled at once;
//   * the split kernel of verify_attn is its programmatic dependent: its
//     prologue (lane lengths, cost partition, page ids, the Q split, tensor
//     memory) runs under the append; it waits for the append before reading
//     any page or page scale;
//   * verify_attn's merge is the split kernel's dependent (as in verify_attn)
//     and lets the acceptance start at once;
//   * the argmax of spec_accept reads only the logits, written before the
//     append started, so it runs beside the merge; it waits for the merge
//     before it finishes, and the finalize kernel (the commit of seq_lens,
//     which every earlier kernel reads) waits for the argmax.
// Only kernels of this library come between the append and the commit, which
// is what makes the early reads safe; the separate entry points keep strict
// stream order with whatever the caller enqueues between them.
#include "sdva_common.cuh"
#include "sdva_internal.cuh"

extern "C" int verify_step(const sdva_kv_cache* cache, const void* k_new, const void* v_new, const void* q,
                           int num_q_heads, int num_lanes, int window, const int32_t* page_table,
                           int max_pages_per_lane, int32_t* seq_lens, int max_context, float sm_scale, void* out,
                           void* workspace, size_t workspace_bytes, const float* logits, int vocab,
                           const int32_t* drafts, int32_t* accept_len, int32_t* out_tokens, int commit,
                           int32_t* status, sdva_stream_t stream) {
  if (seq_lens == nullptr) return SDVA_ERR_INVALID;
  // the checks of all three calls before anything is enqueued, then the launches
  for (int pass = 0; pass < 2; ++pass) {
    const bool check = pass == 0;
    if (const int rc = sdva::append_launch(cache, k_new, v_new, num_lanes, window, nullptr, page_table,
                                           max_pages_per_lane, seq_lens, status, stream, check))
      return rc;
    if (const int rc = sdva::verify_launch(cache, q, num_q_heads, num_lanes, window, nullptr, nullptr, page_table,
                                           max_pages_per_lane, seq_lens, max_context, sm_scale, out, workspace,
                                           workspace_bytes, status, stream, true, check))
      return rc;
    if (const int rc = sdva::accept_launch(logits, num_lanes, window, vocab, drafts, accept_len, out_tokens,
                                           commit ? seq_lens : nullptr, status, stream, true, check))
      return rc;
  }
  return SDVA_OK;
}
