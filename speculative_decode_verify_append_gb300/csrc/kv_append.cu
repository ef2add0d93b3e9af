// kv_append.cu -- kv_append_quant: write the verify window's new K/V rows into
// the paged, quantised KV cache.
//
// FP8 E4M3 cache with one fp32 scale per (page, kv head): the KV format the
// NInfer review names in section "성능과 평가" ("FP8 E4M3" KV).  INT4 cache with
// an fp16 scale per token and group of 32 head dims: the 4-bit KV setting of
// the MegaCapybara announcement, item 2.  INT8 with an fp16 scale per token
// and group of 64 dims, and FP8 E4M3 with an fp32 scale per token row: the
// "INT8 group-64" and "FP8 E4M3 row-256" records of the same review section.
// The scale rules (a page's FP8 scale only grows while it fills; growth
// re-encodes the page's earlier tokens; the per-token formats never
// re-encode) are the reading this library takes; they are spelled out in sdva.h.
//
// The kernels are launch-bound (a verify window is at most 16 tokens, 64 KB
// of bf16 input at 12 lanes): one CTA per (touched page, lane[, kv head, K|V]),
// 16-byte vector loads and stores, fp32 arithmetic through explicitly rounded
// intrinsics (__fdiv_rn / __fmul_rn) so that no contraction or approximate
// division can change a code.
#include "sdva_common.cuh"
#include "sdva_internal.cuh"

namespace sdva {
namespace {

struct AppendArgs {
  const uint16_t* k_new;  // bf16 [B][n_new][Hkv][128]
  const uint16_t* v_new;
  uint8_t* k_codes;
  uint8_t* v_codes;
  void* k_scales;
  void* v_scales;
  const int32_t* page_table;
  const int32_t* seq_lens;
  int32_t* status;
  const int32_t* n_lane;  // nullable [B]: tokens lane b writes (<= n_new); NULL: n_new each
  int num_pages, num_kv_heads, n_new, max_pages;
};

constexpr int kAppendThreads = 256;

// Tokens lane b writes: its own count when per-lane counts are given (a
// padded window whose lanes drafted different numbers of tokens), else n_new.
// A count outside [0, n_new] skips the lane and is flagged (once).
__device__ __forceinline__ int lane_tokens(const AppendArgs& a, int b, bool report) {
  if (a.n_lane == nullptr) return a.n_new;
  const int n = a.n_lane[b];
  if (n < 0 || n > a.n_new) {
    if (report && threadIdx.x == 0) raise_status(a.status, SDVA_STATUS_BAD_COUNT);
    return 0;
  }
  return n;
}

// Lane admission shared by both kernels: the lane's token range [L, L + n)
// must fit its page-table row and every touched page id must be valid;
// otherwise the lane is skipped and flagged (once, by the lane's first CTA).
__device__ bool lane_admitted(const AppendArgs& a, int b, int L, int n, bool report) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const long long end = (long long)L + n;
  if (L < 0 || end > (long long)a.max_pages * kPage) {
    if (report && threadIdx.x == 0) raise_status(a.status, SDVA_STATUS_OVERFLOW);
    return false;
  }
  const int32_t* row = a.page_table + (size_t)b * a.max_pages;
  const int first = L / kPage, last = (int)((end - 1) / kPage);
  for (int p = first + (int)threadIdx.x; p <= last; p += blockDim.x) {
    const int id = row[p];
    if (id < 0 || id >= a.num_pages) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (report && threadIdx.x == 0) raise_status(a.status, SDVA_STATUS_BAD_PAGE);
    return false;
  }
  return true;
}

__device__ __forceinline__ float block_max(float v) {
  __shared__ float s_part[kAppendThreads / 32];
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = s_part[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, s_part[w]);
  return r;
}

// grid: (touched-page slot, lane, kv_head * 2 + {0: K, 1: V})
__global__ void __launch_bounds__(kAppendThreads) append_fp8_kernel(AppendArgs a) {
  // a kernel launched as this one's programmatic dependent may be scheduled
  // now; it waits (griddepcontrol.wait) before it reads the cache
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int slot = blockIdx.x, b = blockIdx.y;
  const int hk = blockIdx.z >> 1, is_v = blockIdx.z & 1;
  const bool report = slot == 0 && blockIdx.z == 0;
  const int n = lane_tokens(a, b, report);
  if (n == 0) return;  // nothing to write: the lane is not examined
  const int L = a.seq_lens[b];
  if (!lane_admitted(a, b, L, n, report)) return;
  const int lp = L / kPage + slot;
  if ((long long)lp * kPage >= (long long)L + n) return;
  const int pid = a.page_table[(size_t)b * a.max_pages + lp];
  const int t0 = max(L, lp * kPage), t1 = min(L + n, lp * kPage + kPage);
  const int start = t0 - lp * kPage, count = t1 - t0;
  const size_t token_stride = (size_t)a.num_kv_heads * kHeadDim;
  const uint16_t* src = (is_v ? a.v_new : a.k_new) + ((size_t)b * a.n_new + (t0 - L)) * token_stride +
                        (size_t)hk * kHeadDim;
  uint8_t* codes = (is_v ? a.v_codes : a.k_codes) + ((size_t)pid * a.num_kv_heads + hk) * kPage * kHeadDim;
  float* scale = reinterpret_cast<float*>(is_v ? a.v_scales : a.k_scales) + (size_t)pid * a.num_kv_heads + hk;

  // items: (token, 8 consecutive dims) -> one 16-byte load each, <= 4 per thread
  constexpr int kMaxItems = kPage * kHeadDim / 8 / kAppendThreads;
  uint4 x[kMaxItems];
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < kMaxItems; ++k) {
    const int it = threadIdx.x + k * kAppendThreads;
    if (it < count * (kHeadDim / 8)) {
      const int t = it >> 4, g = it & 15;
      x[k] = *reinterpret_cast<const uint4*>(src + (size_t)t * token_stride + g * 8);
      const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    }
  }
  amax = block_max(amax);
  const float s_old = *scale;  // read by every thread before the barrier below
  const float s_cand = __fdiv_rn(amax, 448.0f);
  const float s_new = (start == 0) ? s_cand : (s_cand > s_old ? s_cand : s_old);

  if (start > 0 && s_new > s_old) {
    // earlier tokens of the page move to the larger scale: 4 codes per item
    uint32_t* old = reinterpret_cast<uint32_t*>(codes);
    for (int it = threadIdx.x; it < start * (kHeadDim / 4); it += blockDim.x) {
      const uint32_t c = old[it];
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __fdiv_rn(__fmul_rn(e4m3_to_f32((c >> (8 * j)) & 0xFFu), s_old), s_new);
      old[it] = (uint32_t)e4m3x2_from_f32(v[0], v[1]) | ((uint32_t)e4m3x2_from_f32(v[2], v[3]) << 16);
    }
  }
#pragma unroll
  for (int k = 0; k < kMaxItems; ++k) {
    const int it = threadIdx.x + k * kAppendThreads;
    if (it < count * (kHeadDim / 8)) {
      const int t = it >> 4, g = it & 15;
      uint2 out = make_uint2(0u, 0u);
      if (s_new != 0.0f) {
        const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
        uint32_t p[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          p[j] = e4m3x2_from_f32(__fdiv_rn(bf16_lo(w[j]), s_new), __fdiv_rn(bf16_hi(w[j]), s_new));
        out.x = p[0] | (p[1] << 16);
        out.y = p[2] | (p[3] << 16);
      }
      *reinterpret_cast<uint2*>(codes + (size_t)(start + t) * kHeadDim + g * 8) = out;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) *scale = s_new;
}

// grid: (touched-page slot, lane).  One thread per (token, kv head, K|V,
// group of 32 dims): 64 bytes in, 16 bytes of codes and one fp16 scale out.
__global__ void __launch_bounds__(kAppendThreads) append_int4_kernel(AppendArgs a) {
  // a kernel launched as this one's programmatic dependent may be scheduled
  // now; it waits (griddepcontrol.wait) before it reads the cache
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int slot = blockIdx.x, b = blockIdx.y;
  const int n = lane_tokens(a, b, slot == 0);
  if (n == 0) return;  // nothing to write: the lane is not examined
  const int L = a.seq_lens[b];
  if (!lane_admitted(a, b, L, n, slot == 0)) return;
  const int lp = L / kPage + slot;
  if ((long long)lp * kPage >= (long long)L + n) return;
  const int pid = a.page_table[(size_t)b * a.max_pages + lp];
  const int t0 = max(L, lp * kPage), t1 = min(L + n, lp * kPage + kPage);
  const int count = t1 - t0;
  const int H = a.num_kv_heads;
  const size_t token_stride = (size_t)H * kHeadDim;
  for (int it = threadIdx.x; it < count * H * 8; it += blockDim.x) {
    const int g = it & 3, is_v = (it >> 2) & 1, rest = it >> 3;
    const int hk = rest % H, t = rest / H;
    const int off = t0 + t - lp * kPage;
    const uint16_t* src = (is_v ? a.v_new : a.k_new) + ((size_t)b * a.n_new + (t0 - L + t)) * token_stride +
                          (size_t)hk * kHeadDim + g * 32;
    float x[32];
    float amax = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = reinterpret_cast<const uint4*>(src)[q];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[q * 8 + 2 * j] = bf16_lo(w[j]);
        x[q * 8 + 2 * j + 1] = bf16_hi(w[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(x[j]));
    const __half s16 = __float2half_rn(fminf(__fdiv_rn(amax, 7.0f), 65504.0f));
    const float sf = __half2float(s16);
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
    if (sf != 0.0f) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        int qv = __float2int_rn(__fdiv_rn(x[j], sf));
        qv = max(-7, min(7, qv));
        packed[j >> 3] |= (uint32_t)(qv & 0xF) << (4 * (j & 7));
      }
    }
    const size_t ph = (size_t)pid * H + hk;
    uint8_t* codes = (is_v ? a.v_codes : a.k_codes) + (ph * kPage + off) * (kHeadDim / 2) + g * 16;
    *reinterpret_cast<uint4*>(codes) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    __half* scales = reinterpret_cast<__half*>(is_v ? a.v_scales : a.k_scales);
    scales[(ph * kPage + off) * (kHeadDim / 32) + g] = s16;
  }
}

// grid: (touched-page slot, lane).  INT8 group-64 and FP8 row formats: every
// token carries its own scales, so each row is quantised on its own.  Eight
// threads per (token, kv head, K|V) row, 16 dims each (two 16-byte loads, one
// 16-byte store of codes); the amax of the row (FP8 row) or of each 64-dim
// group (INT8) is reduced over the row's threads with shuffles.
template <bool kFp8Row>
__global__ void __launch_bounds__(kAppendThreads) append_rowscaled_kernel(AppendArgs a) {
  // a kernel launched as this one's programmatic dependent may be scheduled
  // now; it waits (griddepcontrol.wait) before it reads the cache
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int slot = blockIdx.x, b = blockIdx.y;
  const int n = lane_tokens(a, b, slot == 0);
  if (n == 0) return;  // nothing to write: the lane is not examined
  const int L = a.seq_lens[b];
  if (!lane_admitted(a, b, L, n, slot == 0)) return;
  const int lp = L / kPage + slot;
  if ((long long)lp * kPage >= (long long)L + n) return;
  const int pid = a.page_table[(size_t)b * a.max_pages + lp];
  const int t0 = max(L, lp * kPage), t1 = min(L + n, lp * kPage + kPage);
  const int count = t1 - t0;
  const int H = a.num_kv_heads;
  const size_t token_stride = (size_t)H * kHeadDim;
  // The item count is a multiple of 8 and a row's 8 items are 8 aligned
  // lanes of one warp, so a row's threads enter and leave the loop together.
  const unsigned row_mask = 0xFFu << (threadIdx.x & 24);
  for (int it = threadIdx.x; it < count * H * 16; it += blockDim.x) {
    const int sub = it & 7, is_v = (it >> 3) & 1, rest = it >> 4;
    const int hk = rest % H, t = rest / H;
    const int off = t0 + t - lp * kPage;
    const uint16_t* src = (is_v ? a.v_new : a.k_new) + ((size_t)b * a.n_new + (t0 - L + t)) * token_stride +
                          (size_t)hk * kHeadDim + sub * 16;
    float x[16];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 v = reinterpret_cast<const uint4*>(src)[q];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[q * 8 + 2 * j] = bf16_lo(w[j]);
        x[q * 8 + 2 * j + 1] = bf16_hi(w[j]);
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(x[j]));
    // over the 4 threads of a 64-dim group, then (FP8 row) over both groups
    amax = fmaxf(amax, __shfl_xor_sync(row_mask, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(row_mask, amax, 2));
    if (kFp8Row) amax = fmaxf(amax, __shfl_xor_sync(row_mask, amax, 4));
    const size_t row = ((size_t)pid * H + hk) * kPage + off;  // (page, kv head, token) row
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
    if constexpr (kFp8Row) {
      const float s = __fdiv_rn(amax, 448.0f);
      if (s != 0.0f) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          packed[j] = e4m3x2_from_f32(__fdiv_rn(x[4 * j], s), __fdiv_rn(x[4 * j + 1], s)) |
                      ((uint32_t)e4m3x2_from_f32(__fdiv_rn(x[4 * j + 2], s), __fdiv_rn(x[4 * j + 3], s)) << 16);
      }
      if (sub == 0) reinterpret_cast<float*>(is_v ? a.v_scales : a.k_scales)[row] = s;
    } else {
      const __half s16 = __float2half_rn(fminf(__fdiv_rn(amax, 127.0f), 65504.0f));
      const float sf = __half2float(s16);
      if (sf != 0.0f) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          int qv = __float2int_rn(__fdiv_rn(x[j], sf));
          qv = max(-127, min(127, qv));
          packed[j >> 2] |= (uint32_t)(qv & 0xFF) << (8 * (j & 3));
        }
      }
      if ((sub & 3) == 0) reinterpret_cast<__half*>(is_v ? a.v_scales : a.k_scales)[row * 2 + (sub >> 2)] = s16;
    }
    *reinterpret_cast<uint4*>((is_v ? a.v_codes : a.k_codes) + row * kHeadDim + sub * 16) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

}  // namespace
}  // namespace sdva

using namespace sdva;

int sdva::append_launch(const sdva_kv_cache* cache, const void* k_new, const void* v_new, int num_lanes, int n_new,
                       const int32_t* n_lane, const int32_t* page_table, int max_pages_per_lane,
                       const int32_t* seq_lens, int32_t* status, sdva_stream_t stream, bool check_only) {
  if (cache == nullptr || k_new == nullptr || v_new == nullptr || page_table == nullptr || seq_lens == nullptr)
    return SDVA_ERR_INVALID;
  if (cache->k_codes == nullptr || cache->v_codes == nullptr || cache->k_scales == nullptr ||
      cache->v_scales == nullptr)
    return SDVA_ERR_INVALID;
  if (num_lanes <= 0 || n_new <= 0 || max_pages_per_lane <= 0 || cache->num_pages <= 0 ||
      cache->num_kv_heads <= 0)
    return SDVA_ERR_INVALID;
  if (cache->page_size != kPage || cache->head_dim != kHeadDim) return SDVA_ERR_UNSUPPORTED;
  if (cache->dtype < SDVA_KV_FP8_E4M3 || cache->dtype > SDVA_KV_FP8_ROW) return SDVA_ERR_UNSUPPORTED;
  if (!cache_aligned(cache)) return SDVA_ERR_INVALID;
  if (num_lanes > 65535 || cache->num_kv_heads > 32767) return SDVA_ERR_UNSUPPORTED;
  if (check_only) return SDVA_OK;
  AppendArgs a;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k_codes = static_cast<uint8_t*>(cache->k_codes);
  a.v_codes = static_cast<uint8_t*>(cache->v_codes);
  a.k_scales = cache->k_scales;
  a.v_scales = cache->v_scales;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.status = status;
  a.n_lane = n_lane;
  a.num_pages = cache->num_pages;
  a.num_kv_heads = cache->num_kv_heads;
  a.n_new = n_new;
  a.max_pages = max_pages_per_lane;
  const int slots = (n_new + kPage - 1) / kPage + 1;  // pages a range of n_new tokens can touch
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cache->dtype == SDVA_KV_FP8_E4M3) {
    append_fp8_kernel<<<dim3(slots, num_lanes, cache->num_kv_heads * 2), kAppendThreads, 0, s>>>(a);
  } else if (cache->dtype == SDVA_KV_INT4_G32) {
    append_int4_kernel<<<dim3(slots, num_lanes), kAppendThreads, 0, s>>>(a);
  } else if (cache->dtype == SDVA_KV_INT8_G64) {
    append_rowscaled_kernel<false><<<dim3(slots, num_lanes), kAppendThreads, 0, s>>>(a);
  } else {
    append_rowscaled_kernel<true><<<dim3(slots, num_lanes), kAppendThreads, 0, s>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? SDVA_OK : SDVA_ERR_CUDA;
}

extern "C" int kv_append_quant(const sdva_kv_cache* cache, const void* k_new, const void* v_new, int num_lanes,
                               int n_new, const int32_t* page_table, int max_pages_per_lane,
                               const int32_t* seq_lens, int32_t* status, sdva_stream_t stream) {
  return sdva::append_launch(cache, k_new, v_new, num_lanes, n_new, nullptr, page_table, max_pages_per_lane, seq_lens,
                     status, stream);
}

extern "C" int kv_append_quant_ragged(const sdva_kv_cache* cache, const void* k_new, const void* v_new,
                                      int num_lanes, int n_new, const int32_t* n_lane, const int32_t* page_table,
                                      int max_pages_per_lane, const int32_t* seq_lens, int32_t* status,
                                      sdva_stream_t stream) {
  if (n_lane == nullptr) return SDVA_ERR_INVALID;
  return sdva::append_launch(cache, k_new, v_new, num_lanes, n_new, n_lane, page_table, max_pages_per_lane, seq_lens,
                     status, stream);
}
