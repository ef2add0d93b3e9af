// verify_attn_tc.cuh -- internal interface between the verify_attn entry
// points and the tcgen05 kernels of verify_attn_tc.cu.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sdva.h"

namespace sdva {
namespace tc {

constexpr int kMaxLanesTc = 1024;  // lanes per call handled by the tcgen05 path

struct TcArgs {
  const uint16_t* q;        // bf16 [B][W][Hq][128]
  const uint8_t* k_codes;   // INT4 / INT8 pools (the FP8 pools are read through tensor maps)
  const uint8_t* v_codes;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* parent;  // draft tree [B][W] (slot 0 unused) or null for the causal window
  const int32_t* n_lane;  // window rows per lane (1 + d_b) or null for all `window` rows
  const void* k_scales;  // FP8: f32 [pages][Hkv]; INT4: f16 [pages][Hkv][64][4];
                         // INT8: f16 [pages][Hkv][64][2]; FP8 row: f32 [pages][Hkv][64]
  const void* v_scales;
  float2* ws_ml;  // [lanes * Hkv + ctas][R]
  float* ws_o;    // [lanes * Hkv + ctas][R][128]
  uint16_t* out;  // bf16 [B][W][Hq][128]
  int32_t* status;
  int num_pages, B, Hkv, Hq, G, W, R, max_pages, max_context;
  long long wait_limit;  // clock cycles a device wait may take before the CTA gives up
  int unit_cost;         // price of a unit's start in the partition, in pages (unit_cost_of)
  float sm_scale_log2;
};

// The partition's price of starting a unit, in pages of the cache format.
int unit_cost_of(int dtype);
// Scratch bytes of the tcgen05 path (split-K partials, one slot per unit and per CTA).
size_t tc_workspace_bytes(int B, int W, int Hq, int Hkv, int num_sms);
// Whether the tcgen05 path handles this call (<= 128 rows per kv head, ...).
bool tc_supported(const sdva_kv_cache* cache, int B, int W, int Hq, int max_pages, int num_sms);
// Enqueue the split and merge kernels on `stream`; with after_append the split
// kernel is a programmatic dependent of the kernel enqueued just before it,
// which must write nothing but the cache (verify_step's append).
int launch_verify_tc(const sdva_kv_cache* cache, const TcArgs& args, int num_sms, cudaStream_t stream,
                     bool after_append);

}  // namespace tc
}  // namespace sdva
