// verify_attn.cu -- batched verify attention over the paged, quantised cache.
//
// What it computes: every window row (lane b, window position i, q head h)
// attends over keys 0 .. L_b + i of its kv head h / (Hq / Hkv): the lane's
// cached context plus the window's own, already appended tokens (causal inside
// the window).  Sources: Baseten talk summary, section "추측 디코드" (the main
// model checks all drafts in one forward pass); NInfer review, section
// "아키텍처 ③" (windows of 1 + 1..15 drafts) and the 240,000-token FP8-KV
// example config of section "설치·실행·서빙".
//
// How (flash-decoding split-K, GB300 layout):
//   * work unit = (lane, kv head); its R = window * G query rows share every
//     K/V page, so one CTA holds all R rows (<= 128) and streams a contiguous
//     range of the unit's pages; the unit's pages are cut into equal splits
//     so that the grid fills the GPU for any mix of context lengths.
//   * page loads: 16-byte cp.async into a 2-stage ring; the FP8 codes are
//     re-read as fp16 (value * 2^-8, exact) and the INT4 codes are scaled to
//     fp16, both into XOR-swizzled shared tiles for ldmatrix.
//   * S = Q K^T and O += P V on the tensor cores (m16n8k16, fp32 accumulate);
//     online softmax in the log2 domain with the per-page FP8 K scale folded
//     into the logit scale and the per-page V scale folded into the softmax
//     shift (weights stay <= 1 in fp16, the normaliser carries 1/scale).
//   * each split writes (m, l, O) partials to the caller's workspace; a second
//     kernel merges them by log-sum-exp and writes bf16 rows.
#include <math.h>

#include <atomic>

#include "sdva_common.cuh"
#include "sdva_internal.cuh"
#include "verify_attn_tc.cuh"

namespace sdva {
namespace {

constexpr int kRowsPerCta = 128;  // rows of one unit handled by one CTA (8 m16 tiles)
constexpr int kTileBytes16 = kPage * kHeadDim * 2;  // one page of one head as fp16

struct VerifyPlan {
  int R;           // rows per unit: window * (Hq / Hkv)
  int row_blocks;  // ceil(R / 128)
  int warps;       // m16 tiles per CTA
  int pps;         // pages per split
  int max_splits;  // splits per unit at max_context
  int units;       // lanes * kv heads
  size_t ml_offset, o_offset, bytes;
};

bool make_plan(int B, int W, int Hq, int Hkv, int max_context, int num_sms, VerifyPlan* p) {
  if (B <= 0 || W <= 0 || W > kMaxWindow || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_context < 0 ||
      num_sms <= 0)
    return false;
  const int G = Hq / Hkv;
  p->R = W * G;
  p->row_blocks = (p->R + kRowsPerCta - 1) / kRowsPerCta;
  p->warps = (min(p->R, kRowsPerCta) + 15) / 16;
  p->units = B * Hkv;
  const long long max_pages = ((long long)max_context + W + kPage - 1) / kPage;
  // aim for ~4 CTAs per SM over the whole grid at the upper-bound length
  const long long target = (long long)num_sms * 4;
  long long pps = ((long long)p->units * p->row_blocks * max_pages + target - 1) / target;
  pps = max(2LL, pps);
  p->pps = (int)pps;
  p->max_splits = (int)((max_pages + pps - 1) / pps);
  const size_t rows_total = (size_t)p->units * p->max_splits * p->R;
  p->ml_offset = 0;
  p->o_offset = ((rows_total * sizeof(float2)) + 255) / 256 * 256;
  p->bytes = p->o_offset + rows_total * kHeadDim * sizeof(float);
  return true;
}

struct VerifyArgs {
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  const void* k_scales;
  const void* v_scales;
  const uint16_t* q;  // bf16 [B][W][Hq][128]
  const int32_t* page_table;
  const int32_t* seq_lens;
  float2* ws_ml;  // [units][max_splits][R] (m in log2 units, l)
  float* ws_o;    // [units][max_splits][R][128]
  uint16_t* out;  // bf16 [B][W][Hq][128]
  int32_t* status;
  int num_pages, Hkv, Hq, G, W, R, max_pages, max_context, pps, max_splits;
  float sm_scale_log2;  // sm_scale * log2(e)
};

// Lane admission (same rule in both kernels): length range and, for the
// merge, every page id of the lane.
__device__ __forceinline__ bool lane_len_ok(const VerifyArgs& a, int L) {
  return L >= 0 && L <= a.max_context && (long long)L + a.W <= (long long)a.max_pages * kPage;
}

// byte offset of 16-byte chunk `c` (0..15) of key row `j` in a swizzled fp16 tile
__device__ __forceinline__ uint32_t swz(int j, int c) { return (uint32_t)(j * 256 + ((c ^ (j & 7)) << 4)); }

template <int KVT>
struct PageBytes;
template <>
struct PageBytes<SDVA_KV_FP8_E4M3> {
  static constexpr int codes = kPage * kHeadDim;  // 8192
  static constexpr int scales = 0;
};
template <>
struct PageBytes<SDVA_KV_INT4_G32> {
  static constexpr int codes = kPage * kHeadDim / 2;       // 4096
  static constexpr int scales = kPage * kHeadDim / 32 * 2;  // 512
};

template <int KVT>
__device__ __forceinline__ void issue_page_load(const VerifyArgs& a, int pid, int hk, uint8_t* stage) {
  constexpr int CB = PageBytes<KVT>::codes, SB = PageBytes<KVT>::scales;
  const size_t ph = (size_t)pid * a.Hkv + hk;
  const uint8_t* kc = a.k_codes + ph * CB;
  const uint8_t* vc = a.v_codes + ph * CB;
  const uint32_t base = smem_u32(stage);
  for (int c = threadIdx.x; c < CB / 16; c += blockDim.x) {
    cp_async_16(base + c * 16, kc + c * 16);
    cp_async_16(base + CB + c * 16, vc + c * 16);
  }
  if (SB > 0) {
    const uint8_t* ks = reinterpret_cast<const uint8_t*>(a.k_scales) + ph * SB;
    const uint8_t* vs = reinterpret_cast<const uint8_t*>(a.v_scales) + ph * SB;
    for (int c = threadIdx.x; c < SB / 16; c += blockDim.x) {
      cp_async_16(base + 2 * CB + c * 16, ks + c * 16);
      cp_async_16(base + 2 * CB + SB + c * 16, vs + c * 16);
    }
  }
}

// Codes of one page (stage) -> fp16 tiles Kh, Vh (swizzled).  FP8: value *
// 2^-8 exactly; INT4: code * scale rounded to fp16.
template <int KVT>
__device__ __forceinline__ void dequant_page(const uint8_t* stage, uint8_t* kh, uint8_t* vh) {
  constexpr int CB = PageBytes<KVT>::codes;
  if constexpr (KVT == SDVA_KV_FP8_E4M3) {
    // item: (tile, key j, 16 codes) -> 2 chunks of 8 halves
    for (int it = threadIdx.x; it < 2 * kPage * 8; it += blockDim.x) {
      const int tile = it >> 9, j = (it >> 3) & 63, cg = it & 7;
      const uint4 c = *reinterpret_cast<const uint4*>(stage + tile * CB + j * kHeadDim + cg * 16);
      uint4 h0, h1;
      e4m3x4_to_f16x4_scaled(c.x, h0.x, h0.y);
      e4m3x4_to_f16x4_scaled(c.y, h0.z, h0.w);
      e4m3x4_to_f16x4_scaled(c.z, h1.x, h1.y);
      e4m3x4_to_f16x4_scaled(c.w, h1.z, h1.w);
      uint8_t* dst = tile ? vh : kh;
      *reinterpret_cast<uint4*>(dst + swz(j, 2 * cg)) = h0;
      *reinterpret_cast<uint4*>(dst + swz(j, 2 * cg + 1)) = h1;
    }
  } else {
    constexpr int SB = PageBytes<KVT>::scales;
    // item: (tile, key j, 16 dims = 8 code bytes) -> 2 chunks of 8 halves
    for (int it = threadIdx.x; it < 2 * kPage * 8; it += blockDim.x) {
      const int tile = it >> 9, j = (it >> 3) & 63, cg = it & 7;
      const uint2 c = *reinterpret_cast<const uint2*>(stage + tile * CB + j * (kHeadDim / 2) + cg * 8);
      const __half s = reinterpret_cast<const __half*>(stage + 2 * CB + tile * SB)[j * 4 + (cg >> 1)];
      const __half2 s2 = __halves2half2(s, s);
      const __half2 bias = __floats2half2_rn(1032.0f, 1032.0f);
      uint32_t h[8];
      const uint32_t words[2] = {c.x, c.y};
#pragma unroll
      for (int w = 0; w < 2; ++w) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // two nibbles (dims 2k, 2k+1 of this word) -> fp16 pair of exact small ints:
          // 1024 + (u ^ 8) - 1032 = two's-complement value of the nibble u
          const uint32_t byte = (words[w] >> (8 * k)) & 0xFFu;
          const uint32_t spread = ((byte & 0xFu) | ((byte & 0xF0u) << 12)) ^ 0x00080008u;
          const uint32_t biased = spread | 0x64006400u;
          __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&biased), bias);
          v = __hmul2(v, s2);
          h[w * 4 + k] = *reinterpret_cast<uint32_t*>(&v);
        }
      }
      uint8_t* dst = tile ? vh : kh;
      *reinterpret_cast<uint4*>(dst + swz(j, 2 * cg)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(dst + swz(j, 2 * cg + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
}

template <int KVT>
__global__ void __launch_bounds__(256) verify_split_kernel(VerifyArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int STAGE = 2 * PageBytes<KVT>::codes + 2 * PageBytes<KVT>::scales;
  uint8_t* stages = smem;                  // 2 stages
  uint8_t* kh = smem + 2 * STAGE;          // fp16 [64][128] swizzled
  uint8_t* vh = kh + kTileBytes16;

  const int split = blockIdx.x, unit = blockIdx.y, rb = blockIdx.z;
  const int b = unit / a.Hkv, hk = unit % a.Hkv;
  const int L = a.seq_lens[b];
  if (!lane_len_ok(a, L)) return;
  const int n_pages = (L + a.W + kPage - 1) / kPage;
  const int p_begin = split * a.pps;
  if (p_begin >= n_pages) return;
  const int p_end = min(n_pages, p_begin + a.pps);
  const int32_t* prow = a.page_table + (size_t)b * a.max_pages;
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  for (int p = p_begin + threadIdx.x; p < p_end; p += blockDim.x) {
    const int id = prow[p];
    if (id < 0 || id >= a.num_pages) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) return;  // the merge flags the lane and zeroes its rows

  issue_page_load<KVT>(a, prow[p_begin], hk, stages);
  cp_async_commit();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = rb * kRowsPerCta + warp * 16;
  const bool active = row0 < a.R;
  const int rA = row0 + g, rB = row0 + g + 8;
  // window position of each row (padding rows behave like the last one)
  const int iA = min(rA / a.G, a.W - 1), iB = min(rB / a.G, a.W - 1);
  const int limA = L + iA, limB = L + iB;  // last visible key position

  // Q fragments for this warp's 16 rows, fp16, all 128 dims (8 k16 steps)
  uint32_t qa[8][4];
  {
    const uint32_t* qA = nullptr;
    const uint32_t* qB = nullptr;
    if (rA < a.R)
      qA = reinterpret_cast<const uint32_t*>(
          a.q + (((size_t)b * a.W + rA / a.G) * a.Hq + hk * a.G + rA % a.G) * kHeadDim);
    if (rB < a.R)
      qB = reinterpret_cast<const uint32_t*>(
          a.q + (((size_t)b * a.W + rB / a.G) * a.Hq + hk * a.G + rB % a.G) * kHeadDim);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int w0 = (ks * 16 + 2 * t) / 2, w1 = (ks * 16 + 8 + 2 * t) / 2;
      qa[ks][0] = qA ? bf16x2_to_f16x2(qA[w0]) : 0u;
      qa[ks][1] = qB ? bf16x2_to_f16x2(qB[w0]) : 0u;
      qa[ks][2] = qA ? bf16x2_to_f16x2(qA[w1]) : 0u;
      qa[ks][3] = qB ? bf16x2_to_f16x2(qB[w1]) : 0u;
    }
  }

  float o[16][4];
#pragma unroll
  for (int dt = 0; dt < 16; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.0f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.0f, lB = 0.0f;

  const uint32_t kh_base = smem_u32(kh), vh_base = smem_u32(vh);
  for (int p = p_begin; p < p_end; ++p) {
    const int st = (p - p_begin) & 1;
    if (p + 1 < p_end) {
      issue_page_load<KVT>(a, prow[p + 1], hk, stages + (st ^ 1) * STAGE);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    dequant_page<KVT>(stages + st * STAGE, kh, vh);
    __syncthreads();

    if (active) {
      const int pid = prow[p];
      float kscale, shift, inv_f;
      if constexpr (KVT == SDVA_KV_FP8_E4M3) {
        const size_t ph = (size_t)pid * a.Hkv + hk;
        const float sk = reinterpret_cast<const float*>(a.k_scales)[ph];
        const float sv = reinterpret_cast<const float*>(a.v_scales)[ph];
        kscale = sk * 256.0f * a.sm_scale_log2;
        const float f = sv > 0.0f ? sv * 256.0f : 1.0f;  // Vh holds value / f
        shift = log2f(f);
        inv_f = 1.0f / f;
      } else {
        kscale = a.sm_scale_log2;
        shift = 0.0f;
        inv_f = 1.0f;
      }
      // ---- S = Q K^T for the 64 keys of this page ----
      float s[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int key = np * 16 + (mi >> 1) * 8 + rr;
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4(kh_base + swz(key, 2 * ks + (mi & 1)), r0, r1, r2, r3);
          mma_f16_16816(s[2 * np], qa[ks], r0, r1);
          mma_f16_16816(s[2 * np + 1], qa[ks], r2, r3);
        }
      }
      // ---- mask, online softmax (log2 domain) ----
      const int kbase = p * kPage;
      float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kp = kbase + nt * 8 + 2 * t + (e & 1);
          const int lim = e < 2 ? limA : limB;
          const float x = kp <= lim ? fmaf(s[nt][e], kscale, shift) : -INFINITY;
          s[nt][e] = x;
          if (e < 2)
            mxA = fmaxf(mxA, x);
          else
            mxB = fmaxf(mxB, x);
        }
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, off));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, off));
      }
      const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
      const float uA = nA == -INFINITY ? 0.0f : nA, uB = nB == -INFINITY ? 0.0f : nB;
      const float alA = fast_exp2(mA - uA), alB = fast_exp2(mB - uB);
      mA = nA;
      mB = nB;
      float sumA = 0.0f, sumB = 0.0f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = fast_exp2(s[nt][0] - uA);
        s[nt][1] = fast_exp2(s[nt][1] - uA);
        s[nt][2] = fast_exp2(s[nt][2] - uB);
        s[nt][3] = fast_exp2(s[nt][3] - uB);
        sumA += s[nt][0] + s[nt][1];
        sumB += s[nt][2] + s[nt][3];
      }
      lA = lA * alA + sumA * inv_f;
      lB = lB * alB + sumB * inv_f;
#pragma unroll
      for (int dt = 0; dt < 16; ++dt) {
        o[dt][0] *= alA;
        o[dt][1] *= alA;
        o[dt][2] *= alB;
        o[dt][3] *= alB;
      }
      // ---- O += P V ----
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_f16x2(s[2 * kk][0], s[2 * kk][1]);
        pa[1] = pack_f16x2(s[2 * kk][2], s[2 * kk][3]);
        pa[2] = pack_f16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        pa[3] = pack_f16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          const int key = kk * 16 + (mi & 1) * 8 + rr;
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(vh_base + swz(key, 2 * dp + (mi >> 1)), r0, r1, r2, r3);
          mma_f16_16816(o[2 * dp], pa, r0, r1);
          mma_f16_16816(o[2 * dp + 1], pa, r2, r3);
        }
      }
    }
    __syncthreads();  // Kh/Vh and this stage are rewritten next iteration
  }

  if (!active) return;
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, off);
    lB += __shfl_xor_sync(0xffffffffu, lB, off);
  }
  const size_t base_row = ((size_t)unit * a.max_splits + split) * a.R;
  if (rA < a.R) {
    if (t == 0) a.ws_ml[base_row + rA] = make_float2(mA, lA);
    float* dst = a.ws_o + (base_row + rA) * kHeadDim;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt)
      *reinterpret_cast<float2*>(dst + dt * 8 + 2 * t) = make_float2(o[dt][0], o[dt][1]);
  }
  if (rB < a.R) {
    if (t == 0) a.ws_ml[base_row + rB] = make_float2(mB, lB);
    float* dst = a.ws_o + (base_row + rB) * kHeadDim;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt)
      *reinterpret_cast<float2*>(dst + dt * 8 + 2 * t) = make_float2(o[dt][2], o[dt][3]);
  }
}

// grid: units; block 256.  Each warp merges rows r = warp, warp + 8, ...
// out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, rounded to bf16.
__global__ void __launch_bounds__(256) verify_merge_kernel(VerifyArgs a) {
  const int unit = blockIdx.x;
  const int b = unit / a.Hkv, hk = unit % a.Hkv;
  const int L = a.seq_lens[b];
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  int n_pages = 0;
  if (!lane_len_ok(a, L)) {
    if (threadIdx.x == 0) {
      s_bad = SDVA_STATUS_OVERFLOW;
    }
  } else {
    n_pages = (L + a.W + kPage - 1) / kPage;
    const int32_t* prow = a.page_table + (size_t)b * a.max_pages;
    for (int p = threadIdx.x; p < n_pages; p += blockDim.x) {
      const int id = prow[p];
      if (id < 0 || id >= a.num_pages) s_bad = SDVA_STATUS_BAD_PAGE;
    }
  }
  __syncthreads();
  const int bad = s_bad;
  if (bad && threadIdx.x == 0 && hk == 0) raise_status(a.status, bad);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_splits = (n_pages + a.pps - 1) / a.pps;
  for (int r = warp; r < a.R; r += blockDim.x >> 5) {
    const int i = r / a.G, h = hk * a.G + r % a.G;
    uint16_t* dst = a.out + (((size_t)b * a.W + i) * a.Hq + h) * kHeadDim + lane * 4;
    if (bad) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
      continue;
    }
    const size_t base_row = (size_t)unit * a.max_splits * a.R + r;
    float M = -INFINITY;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, a.ws_ml[base_row + (size_t)s * a.R].x);
    float den = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int s = 0; s < n_splits; ++s) {
      const float2 ml = a.ws_ml[base_row + (size_t)s * a.R];
      if (ml.x == -INFINITY) continue;
      const float w = exp2f(ml.x - M);
      den += w * ml.y;
      const float4 v = *reinterpret_cast<const float4*>(a.ws_o + (base_row + (size_t)s * a.R) * kHeadDim + lane * 4);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    }
    const float inv = 1.0f / den;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  }
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int KVT>
constexpr int split_smem_bytes() {
  return 2 * (2 * PageBytes<KVT>::codes + 2 * PageBytes<KVT>::scales) + 2 * kTileBytes16;
}

}  // namespace
}  // namespace sdva

using namespace sdva;

extern "C" size_t verify_attn_workspace_size(int num_lanes, int window, int num_q_heads, int num_kv_heads,
                                             int max_context, int num_sms) {
  if (num_sms == 0) num_sms = device_sm_count();
  VerifyPlan plan;
  if (!make_plan(num_lanes, window, num_q_heads, num_kv_heads, max_context, num_sms, &plan)) return 0;
  // enough for either kernel family (the cache dtype is not an argument here)
  return max(plan.bytes, tc::tc_workspace_bytes(num_lanes, window, num_q_heads, num_kv_heads, num_sms));
}

namespace sdva {

constexpr long long kDefaultWaitLimit = 4000000000LL;  // clock cycles, about two seconds
std::atomic<long long> g_wait_limit{kDefaultWaitLimit};

// verify_attn, verify_attn_tree and verify_attn_ragged: `parent` null selects
// the causal window; `n_lane` null, `window` rows for every lane.
int verify_launch(const sdva_kv_cache* cache, const void* q, int num_q_heads, int num_lanes, int window,
                  const int32_t* parent, const int32_t* n_lane, const int32_t* page_table, int max_pages_per_lane,
                  const int32_t* seq_lens, int max_context, float sm_scale, void* out, void* workspace,
                  size_t workspace_bytes, int32_t* status, sdva_stream_t stream, bool after_append,
                  bool check_only) {
  if (cache == nullptr || q == nullptr || page_table == nullptr || seq_lens == nullptr || out == nullptr)
    return SDVA_ERR_INVALID;
  // q and out are read and written in 16-byte vectors (and q by bulk copies)
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u) return SDVA_ERR_INVALID;
  if (cache->k_codes == nullptr || cache->v_codes == nullptr || cache->k_scales == nullptr ||
      cache->v_scales == nullptr)
    return SDVA_ERR_INVALID;
  if (num_lanes <= 0 || window <= 0 || num_q_heads <= 0 || cache->num_kv_heads <= 0 || cache->num_pages <= 0 ||
      max_pages_per_lane <= 0 || max_context < 0 || num_q_heads % cache->num_kv_heads != 0)
    return SDVA_ERR_INVALID;
  if (!(sm_scale > 0.0f) || !isfinite(sm_scale)) return SDVA_ERR_INVALID;
  if (cache->page_size != kPage || cache->head_dim != kHeadDim || window > kMaxWindow) return SDVA_ERR_UNSUPPORTED;
  if (cache->dtype < SDVA_KV_FP8_E4M3 || cache->dtype > SDVA_KV_FP8_ROW) return SDVA_ERR_UNSUPPORTED;
  if (!cache_aligned(cache)) return SDVA_ERR_INVALID;
  const int num_sms = device_sm_count();
  VerifyPlan plan;
  if (num_sms <= 0) return SDVA_ERR_CUDA;
  if (!make_plan(num_lanes, window, num_q_heads, cache->num_kv_heads, max_context, num_sms, &plan))
    return SDVA_ERR_INVALID;
  if (plan.units > 65535 || plan.row_blocks > 65535) return SDVA_ERR_UNSUPPORTED;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return SDVA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (tc::tc_supported(cache, num_lanes, window, num_q_heads, max_pages_per_lane, num_sms)) {
    // <= 128 rows per kv head: tcgen05 kernels (every cache format)
    if (workspace_bytes < tc::tc_workspace_bytes(num_lanes, window, num_q_heads, cache->num_kv_heads, num_sms))
      return SDVA_ERR_WORKSPACE;
    if (check_only) return SDVA_OK;
    const size_t slots = (size_t)num_lanes * cache->num_kv_heads + num_sms;
    tc::TcArgs t;
    t.q = static_cast<const uint16_t*>(q);
    t.k_codes = static_cast<const uint8_t*>(cache->k_codes);
    t.v_codes = static_cast<const uint8_t*>(cache->v_codes);
    t.page_table = page_table;
    t.seq_lens = seq_lens;
    t.parent = parent;
    t.n_lane = n_lane;
    t.k_scales = cache->k_scales;
    t.v_scales = cache->v_scales;
    t.ws_ml = reinterpret_cast<float2*>(workspace);
    t.ws_o = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                      (slots * plan.R * sizeof(float2) + 255) / 256 * 256);
    t.out = static_cast<uint16_t*>(out);
    t.status = status;
    t.num_pages = cache->num_pages;
    t.B = num_lanes;
    t.Hkv = cache->num_kv_heads;
    t.Hq = num_q_heads;
    t.G = num_q_heads / cache->num_kv_heads;
    t.W = window;
    t.R = plan.R;
    t.max_pages = max_pages_per_lane;
    t.max_context = max_context;
    t.sm_scale_log2 = sm_scale * 1.4426950408889634f;
    t.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
    t.unit_cost = tc::unit_cost_of(cache->dtype);
    return tc::launch_verify_tc(cache, t, num_sms, s, after_append);
  }
  // the mma.sync kernels (more than 128 rows per kv head) know only the
  // causal window and the FP8 page-scale and INT4 formats
  if (parent != nullptr || n_lane != nullptr) return SDVA_ERR_UNSUPPORTED;
  if (cache->dtype != SDVA_KV_FP8_E4M3 && cache->dtype != SDVA_KV_INT4_G32) return SDVA_ERR_UNSUPPORTED;
  if (workspace_bytes < plan.bytes) return SDVA_ERR_WORKSPACE;
  if (check_only) return SDVA_OK;

  VerifyArgs a;
  a.k_codes = static_cast<const uint8_t*>(cache->k_codes);
  a.v_codes = static_cast<const uint8_t*>(cache->v_codes);
  a.k_scales = cache->k_scales;
  a.v_scales = cache->v_scales;
  a.q = static_cast<const uint16_t*>(q);
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.ws_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + plan.ml_offset);
  a.ws_o = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.o_offset);
  a.out = static_cast<uint16_t*>(out);
  a.status = status;
  a.num_pages = cache->num_pages;
  a.Hkv = cache->num_kv_heads;
  a.Hq = num_q_heads;
  a.G = num_q_heads / cache->num_kv_heads;
  a.W = window;
  a.R = plan.R;
  a.max_pages = max_pages_per_lane;
  a.max_context = max_context;
  a.pps = plan.pps;
  a.max_splits = plan.max_splits;
  a.sm_scale_log2 = sm_scale * 1.4426950408889634f;

  const dim3 grid(plan.max_splits, plan.units, plan.row_blocks);
  const int threads = plan.warps * 32;
  if (cache->dtype == SDVA_KV_FP8_E4M3) {
    constexpr int smem = split_smem_bytes<SDVA_KV_FP8_E4M3>();
    // the shared-memory limit is a per-device attribute of the function: set
    // it on every call, for the device current now
    if (cudaFuncSetAttribute(verify_split_kernel<SDVA_KV_FP8_E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return SDVA_ERR_CUDA;
    verify_split_kernel<SDVA_KV_FP8_E4M3><<<grid, threads, smem, s>>>(a);
  } else {
    constexpr int smem = split_smem_bytes<SDVA_KV_INT4_G32>();
    if (cudaFuncSetAttribute(verify_split_kernel<SDVA_KV_INT4_G32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return SDVA_ERR_CUDA;
    verify_split_kernel<SDVA_KV_INT4_G32><<<grid, threads, smem, s>>>(a);
  }
  if (cudaGetLastError() != cudaSuccess) return SDVA_ERR_CUDA;
  verify_merge_kernel<<<plan.units, 256, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? SDVA_OK : SDVA_ERR_CUDA;
}

}  // namespace sdva

extern "C" long long sdva_debug_set_wait_limit(long long cycles) {
  return sdva::g_wait_limit.exchange(cycles < 0 ? sdva::kDefaultWaitLimit : cycles);
}

extern "C" int verify_attn(const sdva_kv_cache* cache, const void* q, int num_q_heads, int num_lanes, int window,
                           const int32_t* page_table, int max_pages_per_lane, const int32_t* seq_lens,
                           int max_context, float sm_scale, void* out, void* workspace, size_t workspace_bytes,
                           int32_t* status, sdva_stream_t stream) {
  return sdva::verify_launch(cache, q, num_q_heads, num_lanes, window, nullptr, nullptr, page_table,
                                max_pages_per_lane, seq_lens, max_context, sm_scale, out, workspace, workspace_bytes,
                                status, stream, false);
}

extern "C" int verify_attn_ragged(const sdva_kv_cache* cache, const void* q, int num_q_heads, int num_lanes,
                                  int window, const int32_t* n_lane, const int32_t* page_table,
                                  int max_pages_per_lane, const int32_t* seq_lens, int max_context, float sm_scale,
                                  void* out, void* workspace, size_t workspace_bytes, int32_t* status,
                                  sdva_stream_t stream) {
  if (n_lane == nullptr) return SDVA_ERR_INVALID;
  return sdva::verify_launch(cache, q, num_q_heads, num_lanes, window, nullptr, n_lane, page_table,
                                max_pages_per_lane, seq_lens, max_context, sm_scale, out, workspace, workspace_bytes,
                                status, stream, false);
}

extern "C" int verify_attn_tree(const sdva_kv_cache* cache, const void* q, int num_q_heads, int num_lanes,
                                int window, const int32_t* parent, const int32_t* page_table, int max_pages_per_lane,
                                const int32_t* seq_lens, int max_context, float sm_scale, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* status, sdva_stream_t stream) {
  if (parent == nullptr && window > 1) return SDVA_ERR_INVALID;
  // a window of one slot is the root alone: the causal kernels
  return sdva::verify_launch(cache, q, num_q_heads, num_lanes, window, window > 1 ? parent : nullptr, nullptr,
                                page_table,
                                max_pages_per_lane, seq_lens, max_context, sm_scale, out, workspace, workspace_bytes,
                                status, stream, false);
}

// ---------------------------------------------------------------------------
// verify_attn_noalloc: the same verify_attn launches, with the split-K scratch
// taken from a fixed array that is part of this library's device image instead
// of a caller-provided workspace.  For callers that cannot allocate device
// memory at call time: runtimes that plan every byte of device memory once at
// start-up (a fixed pool with nothing left for per-call scratch), plugin hosts
// that hand an operator only its own input and output tensors, and
// latency-critical loops that must not pay for an allocator's implicit device
// synchronisation.  The array is 256-byte aligned, holds
// SDVA_NOALLOC_SCRATCH_BYTES, and lives on every GPU that loads the library
// until the process exits.
// ---------------------------------------------------------------------------
namespace sdva {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[SDVA_NOALLOC_SCRATCH_BYTES];

// Host code must not pass the array's name to a kernel: on the host it is a
// stand-in symbol, not a device address.  The address is looked up on every
// call, for the device current at that call (a host-side query, no
// allocation), so no address outlives the context that produced it.
int noalloc_scratch_for_current_device(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SDVA_ERR_CUDA;
  *out = p;
  return SDVA_OK;
}

}  // namespace
}  // namespace sdva

extern "C" int verify_attn_noalloc(const sdva_kv_cache* cache, const void* q, int num_q_heads, int num_lanes,
                                   int window, const int32_t* page_table, int max_pages_per_lane,
                                   const int32_t* seq_lens, int max_context, float sm_scale, void* out,
                                   int32_t* status, sdva_stream_t stream) {
  if (cache == nullptr || cache->num_kv_heads <= 0) return SDVA_ERR_INVALID;
  // reject sizes beyond the fixed scratch before touching the device
  const size_t need = verify_attn_workspace_size(num_lanes, window, num_q_heads, cache->num_kv_heads, max_context,
                                                 sdva::device_sm_count());
  if (need > SDVA_NOALLOC_SCRATCH_BYTES) return SDVA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = sdva::noalloc_scratch_for_current_device(&scratch);
  if (rc != SDVA_OK) return rc;
  // Nothing in the scratch needs to start at zero: every partial the merge
  // reads is written earlier in the same call.
  return verify_attn(cache, q, num_q_heads, num_lanes, window, page_table, max_pages_per_lane, seq_lens,
                     max_context, sm_scale, out, scratch, SDVA_NOALLOC_SCRATCH_BYTES, status, stream);
}
