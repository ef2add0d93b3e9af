// verify_attn_tc.cu -- verify attention over the paged, quantised cache (FP8
// E4M3 with page or row scales, INT4 group-32, INT8 group-64) on the
// 5th-generation tensor cores (tcgen05, tensor memory, TMA).
//
// Computes the same thing as the mma.sync path in verify_attn.cu (see there
// and sdva.h): every window row attends over keys 0 .. L_b + i of its kv head.
//
// Design (one persistent CTA of 16 warps per SM; 20 for INT8):
//   * Work = the flattened list of (lane, kv head, page) triples, cut into one
//     contiguous range per CTA by cost (a unit's pages plus a fixed start cost,
//     see Partition), computed on the device from seq_lens, so the launch
//     shape depends only on host arguments.  A maximal run of one (lane, kv
//     head) inside a range is a "segment"; a segment that is a whole unit
//     writes the final bf16 rows, otherwise it writes (m, l, O) partials that
//     verify_merge_tc_kernel combines.
//   * Pages alternate between two softmax warpgroups by the parity of their
//     position in the CTA's range.  Each warpgroup has its own S, P and O in
//     tensor memory and its own running (m, l); at the end of a segment
//     warpgroup 0 combines both halves.
//   * Warp 8 (producer): TMA-loads each page's K and V tiles (8 KB each,
//     128-byte swizzle) into a ring of shared-memory stages, and stages the
//     page's scale terms (FP8 formats; the row scales by bulk copies); the
//     INT4 and INT8 codes and scales arrive by 1-D bulk copies.
//   * Warps 12-15, 12-19 for INT8 (converters; for FP8 page scales at R <= 64
//     the softmax warps without rows on sub-partitions 2-3 take this role
//     instead): widen each page's V codes to fp16 (exact for
//     E4M3; FP8 row: times s_j / s_max; INT4 and INT8: times the group scale)
//     into a second ring, laid out as the MN-major operand of the PV MMA; for
//     INT4 and INT8 also the K codes, into a third ring.
//   * Warps 9-11 issue tcgen05.mma, one thread each:
//       warp 9 + j: S_j  = Q_hi K^T + Q_lo K^T  (kind::f8f6f4; A = Q from shared
//                                                memory, B = the page's K tile)
//       warp 11:    O_j += P_j V                (kind::f16; A = P_j from tensor
//                                                memory, B = the fp16 V tile)
//     A thread waits on the order of a hundred cycles per tcgen05.mma it
//     issues, whatever the tile's N, so a page's twelve instructions are
//     spread over three issuing warps; the tensor core interleaves their
//     streams.  FP8 formats: Q is carried as the sum of two E4M3 terms (hi +
//     lo, 8 significant bits, like bf16) and the K codes feed the tensor core
//     as they are stored.  INT4 and INT8: the QK is kind::f16 with fp16 Q
//     and the converters' fp16 K.
//   * Warps 0-3 / 4-7 (softmax warpgroup 0 / 1): thread t owns TMEM lane t =
//     query row t.  Per page it reads its 64 scores, applies the page's K
//     scale (FP8 row: each key's) and the row's Q scale, masks the window's
//     future keys (or, for a draft tree, the keys outside the row's ancestor
//     set), runs the
//     online softmax in the log2 domain (the page's V scale folded into the
//     shift), rescales its O in tensor memory only when the running max
//     outgrows a lag of kTau, and writes P as fp16 back to tensor memory.
//     It releases S as soon as the scores are in registers, so the QK of its
//     next page overlaps the rest of the softmax.
//   * Every wait is bounded; on timeout the CTA raises SDVA_STATUS_TIMEOUT,
//     drains its own copies and MMAs, frees tensor memory and returns.
#include <string.h>

#include "tc_primitives.cuh"
#include "verify_attn_tc.cuh"

namespace sdva {
namespace tc {
namespace {

constexpr int kStages = 8;            // code stages, at most (INT8 holds fewer)
constexpr int kTileBytes = 8192;     // FP8: 64 rows x 128 E4M3 codes
constexpr int kRowScaleBytes = 512;  // FP8 row: 64 fp32 K scales | 64 fp32 V scales
constexpr int kV16Stages = 3;
constexpr int kQBytes = 32768;       // Q operand: FP8 Q_hi | Q_lo (128 rows x 128 B each), or fp16 (dims 0-63 | 64-127)
constexpr int kV16Bytes = 16384;     // fp16 K or V of one page: dims 0-63 | dims 64-127, 64 rows x 128 B each
constexpr int kProducerWarp = 8;
constexpr int kQkWarp = 9;           // + warpgroup index
constexpr int kPvWarp = 11;
constexpr int kConvWarp = 12;        // converters: warps 12 .. 12 + Smem<KVT>::kConvWarps - 1
constexpr int kThreads = 16 * 32;    // the block of the formats with four converter warps
// Shared memory: the fp16 V ring, the fp16 K ring (INT4 and INT8), the K/V
// code stages, the row-scale stages (FP8 row), then Ctl.  A stage holds one
// (page, kv head): FP8 K and V tiles (TMA, 128-byte swizzle, 1024-byte
// aligned), or INT4 / INT8 K codes, V codes, K scales, V scales as stored.
template <int KVT>
struct Smem {
  static constexpr bool kInt4 = KVT == SDVA_KV_INT4_G32;
  static constexpr bool kInt8 = KVT == SDVA_KV_INT8_G64;
  static constexpr bool kRow = KVT == SDVA_KV_FP8_ROW;
  // K and V widened to fp16 (code * scale) by the converters; the QK MMA is
  // then kind::f16 against fp16 Q
  static constexpr bool kDeq = kInt4 || kInt8;
  static constexpr uint32_t kCodeBytes = kInt4 ? 4096 : 8192;  // per K or V page: 64 rows of codes
  static constexpr uint32_t kScaleBytes = kInt4 ? 512 : 256;   // INT4 / INT8: 64 rows of fp16 group scales
  static constexpr uint32_t kStageBytes = kDeq ? 2 * kCodeBytes + 2 * kScaleBytes : 2 * kTileBytes;
  static constexpr int kNumStages = kInt8 ? 5 : kStages;
  // converter warps 12 .. 12 + kConvWarps - 1: eight (two per sub-partition)
  // for INT8, whose widening of K and V is on the page's critical path (eight
  // measured 120.3 against 125.5 us multi-lane; INT4 gained nothing)
  static constexpr int kConvWarps = kInt8 ? 8 : 4;
  // threads per block: softmax, producer and issuers, converters
  static constexpr int kThreads = (12 + kConvWarps) * 32;
  static constexpr uint32_t kOffV16 = 0;
  static constexpr uint32_t kOffK16 = kOffV16 + kV16Stages * kV16Bytes;
  static constexpr uint32_t kOffQ = kOffK16 + (kDeq ? kV16Stages * kV16Bytes : 0);
  static constexpr uint32_t kOffStages = kOffQ + kQBytes;
  static constexpr uint32_t kOffRowSc = kOffStages + kNumStages * kStageBytes;
  static constexpr uint32_t kOffCtl = kOffRowSc + (kRow ? kNumStages * kRowScaleBytes : 0);
};
// Register split: launched at 128 per thread (65536 for the block); the two
// softmax warpgroups grow to kRegsSoftmax, the other two shrink to kRegsOther.
constexpr int kRegsSoftmax = 176;
constexpr int kRegsOther = 80;
static_assert(2 * 128 * kRegsSoftmax + 2 * 128 * kRegsOther <= kThreads * 128, "register split");
// INT8 (20 warps, launched at 96 registers: 61,440 for the block): softmax
// 160, producer and issuers 56, the eight converter warps 48
constexpr int kRegsSoftmax20 = 160, kRegsIss20 = 56, kRegsConv20 = 48;
static_assert(256 * kRegsSoftmax20 + 128 * kRegsIss20 + 256 * kRegsConv20 <= 640 * 96, "register split (20 warps)");
// tensor memory columns
// S buffer x of warpgroup j: 64 fp32 columns of scores; once they are in
// registers the warpgroup writes its P (64 keys of fp16 = 32 columns) over
// the buffer's first half, where the PV MMA reads it
__host__ __device__ constexpr uint32_t col_s(int j, int x) { return 128u * j + 64u * x; }
__host__ __device__ constexpr uint32_t col_o(int j) { return 256u + 128u * j; }  // 128 fp32 cols
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescQK = idesc_e4m3(128, 64, 0);
constexpr uint32_t kIdescQK16 = idesc_f16(128, 64, 0);
constexpr uint32_t kIdescPV = idesc_f16(128, 128, 1);
constexpr float kTau = 8.0f;       // allowed lag of the running max (log2 units)
constexpr float kPScale = 128.0f;  // P' = softmax weight * 2^(15 - kTau) <= 2^15 (fp16)
constexpr int kBadPage = 1 << 30;  // marks a page whose id was out of range (bit free in a (page, head) index)
constexpr int kBarWg1Done = 1;    // named barriers between the two softmax warpgroups
constexpr int kBarWg0Done = 2;

struct Ctl {
  uint64_t full[kStages];   // TMA bytes of the stage landed
  uint64_t empty[kStages];  // the stage's K was used by QK, its V converted, its scales read
  uint64_t v16_full[kV16Stages];   // fp16 V written (one arrival per converter warp)
  uint64_t v16_empty[kV16Stages];  // the PV that read it completed
  uint64_t k16_full[kV16Stages];   // INT4 / INT8: fp16 K written (one arrival per converter warp)
  uint64_t k16_empty[kV16Stages];  // INT4 / INT8: the QK that read it completed
  uint64_t s_full[2][2];    // [warpgroup j][buffer x]: QK of the buffer's page is in it
  uint64_t p_full[2][2];    // the warpgroup wrote P over the buffer
  uint64_t pv_done[2][2];   // the PV that read that P has completed (the buffer is free)
  uint64_t q_full;          // warpgroup 0 wrote the segment's Q
  uint64_t q_free;          // both QK issuers are done with the segment (2 arrivals)
  float sk[kStages];        // K scale of the page in stage s
  int bad[kStages];         // the page id in stage s was out of range (page 0 was loaded instead)
  int bad1;                 // warpgroup 1 met such a page in the current segment
  float shift[kStages];     // log2 of its V scale (0 when the scale is 0)
  float inv_v[kStages];     // 1 / V scale (1 when the scale is 0)
  int nv[kStages];          // FP8 row: rows of the page written (the lane's tokens in it)
  float m1[128];            // warpgroup 1's running max / sum at the end of a segment
  float l1[128];
  uint32_t tmem_base;
  int abort;
  int stop;                   // set by warpgroup 0 at a segment end when the CTA gives up
  int pref[kMaxLanesTc + 1];  // pages per kv head of lanes < b (prefix)
  int cp[kMaxLanesTc + 1];    // cost per kv head of lanes < b (see Partition)
  long long range[2];         // this CTA's pages [start, end) of the flattened list
  int lens[kMaxLanesTc];      // L_b
};

template <int KVT>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)Smem<KVT>::kOffCtl + sizeof(Ctl);
}
static_assert(smem_bytes<SDVA_KV_FP8_E4M3>() <= 232448, "shared memory budget");
static_assert(smem_bytes<SDVA_KV_INT4_G32>() <= 232448, "shared memory budget");
static_assert(smem_bytes<SDVA_KV_INT8_G64>() <= 232448, "shared memory budget");
static_assert(smem_bytes<SDVA_KV_FP8_ROW>() <= 232448, "shared memory budget");
static_assert(Smem<SDVA_KV_FP8_ROW>::kOffStages % 1024 == 0 && Smem<SDVA_KV_FP8_E4M3>::kOffStages % 1024 == 0,
              "TMA tiles with the 128-byte swizzle start on 1024-byte boundaries");

// Partition of the flattened (lane, kv head, page) list over the CTAs.  Each
// unit (lane, kv head) costs its pages plus a unit cost uc: a CTA that starts
// a new unit inside its range pays a segment end and a segment start (an
// output epilogue, a Q row load and a pipeline refill), so equal shares of
// cost, not of pages, end together.  uc is that price in pages of the format
// (measured: 20 for FP8 page scales, 16 for the formats whose pages take
// longer: FP8 row scales, INT4, INT8).  CTA c owns the cost interval [c T / Ce, (c + 1) T / Ce), T the
// total cost and Ce = min(CTAs, T), mapped to real pages: the cost of a
// unit's start maps to its first page.
struct Partition {
  const int* pref;  // [B + 1] pages per kv head of lanes < b
  const int* cp;    // [B + 1] cost per kv head of lanes < b (pages + uc per lane with pages)
  int B, Hkv, uc;
  __device__ long long total_pages() const { return (long long)Hkv * pref[B]; }
  __device__ long long total_cost() const { return (long long)Hkv * cp[B]; }
  __device__ long long ctas(int C) const { return min((long long)C, total_cost()); }
  // real flattened page position of cost position y (0 <= y <= total cost).
  // The offset inside a lane, below Hkv * (pages + uc), fits in 32
  // bits: this path requires num_pages * Hkv * 64 < 2^31.
  __device__ long long real_of(long long y) const {
    if (y >= total_cost()) return total_pages();
    int lo = 0, hi = B - 1;  // the lane of y: the last b with cost prefix <= y (it has pages)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)Hkv * cp[mid] <= y)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int nb = pref[lo + 1] - pref[lo];
    const uint32_t r = (uint32_t)(y - (long long)Hkv * cp[lo]);
    const uint32_t span = (uint32_t)(nb + uc);
    const uint32_t q = r / span, v = r - q * span;
    return (long long)Hkv * pref[lo] + (long long)q * nb + max(0, (int)v - uc);
  }
  // floor(c T / Ce), 0 <= c <= Ce <= 1024, in 32-bit arithmetic (T < 2^31):
  // c T / Ce = c (T / Ce) + c (T % Ce) / Ce
  __device__ long long cost_begin(long long c, long long Ce) const {
    const uint32_t T = (uint32_t)total_cost(), ce = (uint32_t)Ce, cc = (uint32_t)c;
    const uint32_t qT = T / ce, rT = T - qT * ce;
    return (long long)(cc * qT + (cc * rT) / ce);
  }
  // first real position of CTA c of Ce (c = Ce: the end)
  __device__ long long cta_begin(long long c, long long Ce) const { return real_of(cost_begin(c, Ce)); }
  // the CTA of Ce whose cost interval holds cost position y (0 <= y < total
  // cost).  The page at cost position y belongs to that CTA's page range:
  // real_of is monotone and maps y back to the page.  An fp32 estimate, then
  // exact steps.
  __device__ long long cta_of_cost(long long y, long long Ce) const {
    long long c = (long long)((float)y * (float)Ce / (float)total_cost());
    c = max(0LL, min(c, Ce - 1));
    while (c > 0 && cost_begin(c, Ce) > y) --c;
    while (c + 1 < Ce && cost_begin(c + 1, Ce) <= y) ++c;
    return c;
  }
};

// Warp-wide prefix over lanes (one warp, all lanes): pref[b] = pages per kv
// head of lanes < b and cp[b] = their cost (pages + unit_cost per lane with
// pages), b = 0 .. B; lens[b] = L_b when lens is not null.
__device__ __forceinline__ void partition_prefix(const int32_t* seq_lens, int B, int W, int max_context, int max_pages,
                                                 int unit_cost,
                                                 int lane, int* pref, int* cp, int* lens) {
  int carry = 0, carry_c = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    int n = 0;
    if (b < B) {
      const int L = seq_lens[b];
      if (lens) lens[b] = L;
      const bool ok = L >= 0 && L <= max_context && (long long)L + W <= (long long)max_pages * kPage;
      n = ok ? (L + W + kPage - 1) / kPage : 0;
    }
    const int cost = n > 0 ? n + unit_cost : 0;
    int incl = n, incl_c = cost;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      const int yc = __shfl_up_sync(0xffffffffu, incl_c, o);
      if (lane >= o) {
        incl += y;
        incl_c += yc;
      }
    }
    if (b < B) {
      pref[b] = carry + incl - n;
      cp[b] = carry_c + incl_c - cost;
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
    carry_c += __shfl_sync(0xffffffffu, incl_c, 31);
  }
  if (lane == 0) {
    pref[B] = carry;
    cp[B] = carry_c;
  }
}

// Walks the flattened (lane, kv head, page) list in order.
struct PageIter {
  int b, hk, p, nb;
  __device__ void seek(long long x, const int* pref, int B, int Hkv) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)Hkv * pref[mid] <= x)
        lo = mid;
      else
        hi = mid - 1;
    }
    b = lo;
    nb = pref[b + 1] - pref[b];
    const long long r = x - (long long)Hkv * pref[b];
    hk = (int)(r / nb);
    p = (int)(r % nb);
  }
  __device__ void next(const int* pref, int B, int Hkv) {
    if (++p < nb) return;
    p = 0;
    if (++hk < Hkv) return;
    hk = 0;
    do {
      ++b;
    } while (b < B && pref[b + 1] == pref[b]);
    if (b < B) nb = pref[b + 1] - pref[b];
  }
  // from any page of a segment to the first page of the next unit
  __device__ void next_unit(const int* pref, int B, int Hkv) {
    p = nb - 1;
    next(pref, B, Hkv);
  }
};

__device__ __forceinline__ void fail(Ctl* ctl, int32_t* status) {
  if (atomicExch(&ctl->abort, 1) == 0) raise_status(status, SDVA_STATUS_TIMEOUT);
}

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void named_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// first position >= g of warpgroup j's pages (positions of parity j)
__device__ __forceinline__ long long first_own(long long g, int j) { return g + ((g ^ (long long)j) & 1); }

// Row exponent e of a Q row: 2^e * max|q| lies in [128, 256).
__device__ __forceinline__ int q_row_exponent(const uint16_t* qrow) {
  const uint4* qp = reinterpret_cast<const uint4*>(qrow);
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint4 v = qp[k];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[t])), fabsf(bf16_hi(w[t]))));
  }
  if (!(amax > 0.0f)) return 0;
  int k2;
  frexpf(amax, &k2);  // amax < 2^k2
  return max(-100, min(100, 8 - k2));
}

// The Q row scaled by 2^e as fp16, stored to row `row` of the two 64-dim
// halves of the shared-memory operand (16384 bytes apart; 128-byte swizzle:
// 8-dim chunk c of row r at r * 128 + ((c ^ (r & 7)) << 4)).  A null row
// stores zeros.
__device__ __forceinline__ void store_q16_row_smem(const uint16_t* qrow, int e, uint8_t* q, int row) {
  const float up = ldexpf(1.0f, e);
#pragma unroll 1
  for (int c = 0; c < 16; ++c) {  // 8 dims per 16-byte chunk
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (qrow) v = reinterpret_cast<const uint4*>(qrow)[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) h[t] = pack_f16x2(bf16_lo(w[t]) * up, bf16_hi(w[t]) * up);
    const uint32_t off = 16384u * (uint32_t)(c >> 3) + (uint32_t)row * 128u + ((uint32_t)((c & 7) ^ (row & 7)) << 4);
    *reinterpret_cast<uint4*>(q + off) = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

// As q_row_exponent, for the FP8 path: the loads go through the
// non-coherent cache, so that store_q_row_smem re-reads the row from L1.
__device__ __forceinline__ int q_row_exponent_ldg(const uint16_t* qrow) {
  if (qrow == nullptr) return 0;
  uint4 v[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) v[k] = __ldg(reinterpret_cast<const uint4*>(qrow) + k);
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int t = 0; t < 4; ++t) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[t])), fabsf(bf16_hi(w[t]))));
  }
  if (!(amax > 0.0f)) return 0;
  int k2;
  frexpf(amax, &k2);  // amax < 2^k2
  return max(-100, min(100, 8 - k2));
}

// The Q row scaled by 2^e, split into hi + lo E4M3 codes and stored to row
// `row` of the two shared-memory operand tiles (128-byte swizzle: 16-byte
// chunk c of row r at r * 128 + ((c ^ (r & 7)) << 4)).  A null row stores
// zeros.  The row is re-read (an L1 hit after q_row_exponent) four chunks at
// a time, the loads of a group in flight together.
__device__ __forceinline__ void store_q_row_smem(const uint16_t* qrow, int e, uint8_t* qhi, uint8_t* qlo, int row) {
  const float up = ldexpf(1.0f, e);
#pragma unroll 1
  for (int c0 = 0; c0 < 8; c0 += 4) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      v[k] = qrow ? __ldg(reinterpret_cast<const uint4*>(qrow) + c0 * 2 + k) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {  // 16 elements per 16-byte chunk
      const int c = c0 + cc;
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint4 x = v[cc * 2 + k];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int t = 0; t < 4; t += 2) {
          const float x0 = bf16_lo(w[t]) * up, x1 = bf16_hi(w[t]) * up;
          const float x2 = bf16_lo(w[t + 1]) * up, x3 = bf16_hi(w[t + 1]) * up;
          const uint32_t h01 = e4m3x2_from_f32(x0, x1), h23 = e4m3x2_from_f32(x2, x3);
          const float2 d01 = f32x2_from_e4m3x2(h01), d23 = f32x2_from_e4m3x2(h23);
          const uint32_t l01 = e4m3x2_from_f32(x0 - d01.x, x1 - d01.y),
                         l23 = e4m3x2_from_f32(x2 - d23.x, x3 - d23.y);
          hw[2 * k + (t >> 1)] = h01 | (h23 << 16);
          lw[2 * k + (t >> 1)] = l01 | (l23 << 16);
        }
      }
      const uint32_t off = (uint32_t)row * 128u + ((uint32_t)(c ^ (row & 7)) << 4);
      *reinterpret_cast<uint4*>(qhi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(qlo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
}

// 16 bytes of INT4 codes (32 dims of one key, dims 2i / 2i + 1 in the low /
// high nibble of byte i, two's complement) times their group's fp16 scale ->
// 32 fp16 values as 4 x 16-byte chunks (chunk k = dims 8k .. 8k + 7).  A
// nibble u becomes the exact fp16 1024 + (u ^ 8) by bit placement; minus 1032
// that is its signed value, then one rounding by the scale.
__device__ __forceinline__ void int4_group_to_f16(uint4 codes, uint32_t scale_bits, uint4 (&out)[4]) {
  const __half2 s2 = __halves2half2(__ushort_as_half((unsigned short)scale_bits),
                                    __ushort_as_half((unsigned short)scale_bits));
  // nibble n with its sign bit flipped is the byte q + 8; placed under the
  // fp16 exponent of 1024 (0x64 high byte) it reads 1032 + q, exactly
  const __half2 bias = __floats2half2_rn(1032.0f, 1032.0f);
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t lo = (cw[k] & 0x0F0F0F0Fu) ^ 0x08080808u, hi = ((cw[k] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    const uint32_t d03 = __byte_perm(lo, hi, 0x5140);  // bytes: dims 0, 1, 2, 3 of this word
    const uint32_t d47 = __byte_perm(lo, hi, 0x7362);  // dims 4, 5, 6, 7
    uint32_t h[4];
    const uint32_t src[2] = {d03, d47};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t biased = __byte_perm(src[q >> 1], 0x64646464u, (q & 1) ? 0x4342 : 0x4140);  // two dims
      __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&biased), bias);
      v = __hmul2(v, s2);
      h[q] = *reinterpret_cast<const uint32_t*>(&v);
    }
    out[k] = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

// Sixteen INT8 codes (dims 16c .. 16c + 15 of a row, one 64-dim group) times
// the group's fp16 scale -> fp16, dims in order two per word.  The int8 ->
// fp16 step is exact: with its sign bit flipped a code q is the byte q + 128,
// placed under the fp16 exponent of 1024 (0x6400 | byte) it reads 1152 + q,
// and subtracting 1152 leaves q.  The product is the one rounding.
__device__ __forceinline__ void int8x16_to_f16(uint4 codes, uint32_t scale_bits, uint32_t (&out)[8]) {
  const __half2 s2 = __halves2half2(__ushort_as_half((unsigned short)scale_bits),
                                    __ushort_as_half((unsigned short)scale_bits));
  const __half2 bias = __floats2half2_rn(1152.0f, 1152.0f);
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t ob = cw[k] ^ 0x80808080u;
    const uint32_t lo = __byte_perm(ob, 0x64646464u, 0x4140);  // dims 4k, 4k + 1
    const uint32_t hi = __byte_perm(ob, 0x64646464u, 0x4342);  // dims 4k + 2, 4k + 3
    const __half2 v0 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&lo), bias), s2);
    const __half2 v1 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&hi), bias), s2);
    out[2 * k] = *reinterpret_cast<const uint32_t*>(&v0);
    out[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&v1);
  }
}

// FP8 row format: the largest V row scale among the first nv rows of a
// stage's page (zero when there is none), computed by a whole warp from the
// row-scale stage (V scales at entries 64 .. 127).
__device__ __forceinline__ float row_vscale_max(const float* rs, int nv, int lane) {
  float m = fmaxf(lane < nv ? rs[64 + lane] : 0.0f, lane + 32 < nv ? rs[96 + lane] : 0.0f);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// kMode: bit 0 -- draft-tree window (a.parent); bit 1 -- a window row count
// per lane (a.n_lane).  Mode 0, the causal window, is the common case.
constexpr int kModeTree = 1, kModeRagged = 2;
template <int KVT, int kMode>
__global__ void __launch_bounds__(Smem<KVT>::kThreads, 1) verify_split_tc_kernel(const __grid_constant__ CUtensorMap map_k,
                                                                    const __grid_constant__ CUtensorMap map_v,
                                                                    TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  using SM = Smem<KVT>;
  constexpr bool kDeq = SM::kDeq, kRow = SM::kRow;
  constexpr int kNS = SM::kNumStages;
  // A CTA's page positions are below 2^31, so ring slots and phases are taken
  // in 32-bit unsigned arithmetic: a 64-bit division by 5 (INT8 stages) or 3
  // (fp16 rings) on every page cost the INT8 call 3%.
  constexpr bool kTree = (kMode & kModeTree) != 0, kRagged = (kMode & kModeRagged) != 0;
  constexpr bool kSpinWait = !kDeq;  // see mbar_wait (the converters need the issue slots)
  constexpr uint32_t kStageBytes = SM::kStageBytes;
  Ctl* ctl = reinterpret_cast<Ctl*>(base_ptr + SM::kOffCtl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = gridDim.x, c = blockIdx.x;
  volatile int* abort_flag = &ctl->abort;

  // ---- partition: pages and cost per kv head of every lane, prefix over lanes ----
  if (warp == 0) {
    partition_prefix(a.seq_lens, a.B, a.W, a.max_context, a.max_pages, a.unit_cost, lane, ctl->pref, ctl->cp,
                     ctl->lens);
    __syncwarp();
    if (lane < 2) {
      // this CTA's page range [start, end): start on lane 0, end on lane 1
      const Partition part{ctl->pref, ctl->cp, a.B, a.Hkv, a.unit_cost};
      const long long Ce = part.ctas(C);
      ctl->range[lane] = c < Ce ? part.cta_begin(c + lane, Ce) : 0;
    }
  }
  // only the softmax warps that own query rows take part in the page protocol
  const uint32_t row_threads = 32u * (uint32_t)min(4, (a.R + 31) / 32);
  if (threadIdx.x == 32) {
    for (int s = 0; s < kNS; ++s) {
      // FP8 formats: the copies' expect_tx arrival, then the scale terms;
      // INT4 / INT8: the copies' arrival (the scales are inside the stage)
      mbar_init(smem_u32(&ctl->full[s]), kDeq ? 1 : 2);
      // FP8 formats: QK commit (K tile), converters (V tile), softmax warps
      // (scales); INT4 / INT8: converters (K and V codes), softmax warps
      mbar_init(smem_u32(&ctl->empty[s]), (kDeq ? 0 : 1) + SM::kConvWarps + row_threads / 32);
    }
    for (int t = 0; t < kV16Stages; ++t) {
      mbar_init(smem_u32(&ctl->v16_full[t]), SM::kConvWarps);
      mbar_init(smem_u32(&ctl->v16_empty[t]), 1);
      mbar_init(smem_u32(&ctl->k16_full[t]), SM::kConvWarps);
      mbar_init(smem_u32(&ctl->k16_empty[t]), 1);
    }
    for (int j = 0; j < 2; ++j)
      for (int x = 0; x < 2; ++x) {
        mbar_init(smem_u32(&ctl->s_full[j][x]), 1);
        mbar_init(smem_u32(&ctl->p_full[j][x]), row_threads);
        mbar_init(smem_u32(&ctl->pv_done[j][x]), 1);
      }
    mbar_init(smem_u32(&ctl->q_full), row_threads);
    mbar_init(smem_u32(&ctl->q_free), 2);
    ctl->abort = 0;
    ctl->stop = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const long long start = ctl->range[0], end = ctl->range[1];
  const long long n_local = end - start;
  // uniform for the whole CTA (a range inside a unit's start cost has no pages)
  if (n_local <= 0) return;

  if (warp == kProducerWarp) tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  const uint32_t stages = base + SM::kOffStages;
  const uint32_t v16 = base + SM::kOffV16;
  const uint32_t k16 = base + SM::kOffK16;
  const uint32_t qsm = base + SM::kOffQ;
  // The V (and INT K) widening of every page, run by converter thread u
  // (0 .. 32 * kConvWarps - 1) of the warps that take the converter role.
  auto convert = [&](const int u) {
    // ------------------------------------------------------------------
    // converters: page g's V codes (TMA tile, 128-byte swizzle, row = key)
    // -> fp16 in V16 slot g % kV16Stages: dims 0-63 and 64-127 as two
    // 64-row x 128-byte regions, each with the 128-byte swizzle (16-byte
    // chunk c of row r at r * 128 + ((c ^ (r & 7)) << 4)).  E4M3 -> fp16 is
    // exact.  Converter thread u handles the items u, u + kCT, ... of a page
    // (kCT converter threads; the row and chunk of an item follow below).
    // ------------------------------------------------------------------
    constexpr int kCT = 32 * SM::kConvWarps;  // converter threads
    // Shared memory serves a warp's 16-byte accesses a quarter-warp (8
    // lanes) at a time, and the two 8 KB halves of an fp16 tile share banks:
    // each quarter-warp takes two rows whose stores land in 8 distinct
    // 16-byte bank groups (as do its loads).  Lane l of a warp covering rows
    // r0 .. : row offset rof, 16-dim chunk c8 (FP8, INT8) or group g4 (INT4).
    const int q8 = lane >> 3, rr = (lane >> 2) & 1;
    const int c8 = (lane & 3) + 4 * (rr ^ (q8 & 1));                        // rows r0 + rof, 4 per warp
    const int rof8 = 2 * (q8 >> 1) + rr;
    const int hb = (lane >> 2) & 1, r4 = (lane >> 1) & 1;                   // INT4: 8 rows per warp
    const int g4 = (lane & 1) + 2 * (hb ^ (q8 & 1));
    const int rof4 = 4 * (q8 >> 1) + 2 * hb + r4;
    bool ok = true;
    for (long long h = 0; h < n_local && ok; ++h) {
      const int s = (int)((uint32_t)h % (uint32_t)kNS), t = (int)((uint32_t)h % (uint32_t)kV16Stages);
      if (!(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->full[s]), (uint32_t)(((uint32_t)h / (uint32_t)kNS) & 1), abort_flag, a.wait_limit))) break;
      if (h >= kV16Stages &&
          !(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->v16_empty[t]), (uint32_t)(((uint32_t)h / (uint32_t)kV16Stages - 1) & 1), abort_flag, a.wait_limit)))
        break;
      if (kDeq && h >= kV16Stages &&
          !(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->k16_empty[t]), (uint32_t)(((uint32_t)h / (uint32_t)kV16Stages - 1) & 1), abort_flag, a.wait_limit)))
        break;
      const uint8_t* stage = base_ptr + SM::kOffStages + s * kStageBytes;
      uint8_t* dst = base_ptr + SM::kOffV16 + t * kV16Bytes;
      if constexpr (SM::kInt8) {
        // INT8: K and V, 64 rows x 8 chunks of 16 dims each; chunk (tk, r, c)
        // -> 2 chunks of 8 dims in the swizzled fp16 layout (K: the K-major
        // operand of the QK MMA; V: the MN-major operand of the PV MMA)
        uint8_t* kdst = base_ptr + SM::kOffK16 + t * kV16Bytes;
#pragma unroll 4
        for (int q = 0; q < 1024 / kCT; ++q) {
          const int item = u + kCT * q;  // 1024 chunks per page, 32 per warp: 4 rows x 8 chunks
          const int tk = item >> 9, r = 4 * ((item & 511) >> 5) + rof8, c = c8;
          const uint4 codes = *reinterpret_cast<const uint4*>(stage + tk * SM::kCodeBytes + r * 128 + c * 16);
          const uint32_t sc = *reinterpret_cast<const uint16_t*>(stage + 2 * SM::kCodeBytes + tk * SM::kScaleBytes +
                                                                 r * 4 + (c >> 2) * 2);
          uint32_t h16[8];
          int8x16_to_f16(codes, sc, h16);
          // dims 16c .. 16c + 15 -> region c >> 2, 8-dim chunks 2 (c & 3) and 2 (c & 3) + 1
          uint8_t* reg = (tk ? dst : kdst) + (c >> 2) * 8192 + r * 128;
          const int c0 = 2 * (c & 3);
          *reinterpret_cast<uint4*>(reg + ((c0 ^ (r & 7)) << 4)) = make_uint4(h16[0], h16[1], h16[2], h16[3]);
          *reinterpret_cast<uint4*>(reg + (((c0 + 1) ^ (r & 7)) << 4)) = make_uint4(h16[4], h16[5], h16[6], h16[7]);
        }
      } else if constexpr (kDeq) {
        // INT4: K and V, 64 rows x 4 groups of 32 dims each; group (tk, r, gi)
        // -> 4 chunks of 8 dims in the same swizzled fp16 layout as V (for K
        // it is the K-major operand of the QK MMA)
        uint8_t* kdst = base_ptr + SM::kOffK16 + t * kV16Bytes;
        constexpr int kQ = 512 / kCT;
        uint4 codes4[kQ];
        uint32_t sc4[kQ];
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          const int item = u + kCT * q;
          const int tk = item >> 8, r = 8 * ((item & 255) >> 5) + rof4, gi = g4;
          codes4[q] = *reinterpret_cast<const uint4*>(stage + tk * SM::kCodeBytes + r * 64 + gi * 16);
          sc4[q] = *reinterpret_cast<const uint16_t*>(stage + 2 * SM::kCodeBytes + tk * SM::kScaleBytes + r * 8 + gi * 2);
        }
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          const int item = u + kCT * q;  // 512 groups per page, 32 per warp: 8 rows x 4 groups
          const int tk = item >> 8, r = 8 * ((item & 255) >> 5) + rof4, gi = g4;
          uint4 ch[4];
          int4_group_to_f16(codes4[q], sc4[q], ch);
          // dims 32gi .. 32gi + 31 -> region gi >> 1, 8-dim chunks 4 (gi & 1) .. + 3
          uint8_t* reg = (tk ? dst : kdst) + (gi >> 1) * 8192 + r * 128;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(reg + (((4 * (gi & 1) + k) ^ (r & 7)) << 4)) = ch[k];
        }
      } else {
        const uint8_t* src = stage + kTileBytes;
        // FP8 row: row r is widened as code * (s_r / s_max) (zero past the
        // page's written rows); the softmax folds s_max into its shift
        const float* rs = reinterpret_cast<const float*>(base_ptr + SM::kOffRowSc + s * kRowScaleBytes);
        int nv = 0;
        float inv_max = 0.0f;
        if constexpr (kRow) {
          nv = ctl->nv[s];
          const float vmax = row_vscale_max(rs, nv, lane);
          inv_max = vmax > 0.0f ? __fdividef(1.0f, vmax) : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
        const int item = u + 128 * q;  // 512 chunks per page, 32 per warp: 4 rows x 8 chunks
        const int r = 4 * (item >> 5) + rof8, c = c8;  // key row, 16-dim chunk
        const uint4 w = *reinterpret_cast<const uint4*>(src + r * 128 + ((c ^ (r & 7)) << 4));
        const uint32_t b[4] = {w.x, w.y, w.z, w.w};
        uint32_t h16[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          h16[2 * k] = f16x2_from_e4m3x2(b[k] & 0xFFFFu);
          h16[2 * k + 1] = f16x2_from_e4m3x2(b[k] >> 16);
        }
        if constexpr (kRow) {
          const __half2 f2 = __float2half2_rn(r < nv ? rs[64 + r] * inv_max : 0.0f);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h16[k]), f2);
            h16[k] = *reinterpret_cast<const uint32_t*>(&v);
          }
        }
        // dims 16c .. 16c + 15 -> region c >> 2, 8-dim chunks 2 (c & 3) and 2 (c & 3) + 1
        uint8_t* reg = dst + (c >> 2) * 8192 + r * 128;
        const int c0 = 2 * (c & 3);
        *reinterpret_cast<uint4*>(reg + (((c0) ^ (r & 7)) << 4)) = make_uint4(h16[0], h16[1], h16[2], h16[3]);
        *reinterpret_cast<uint4*>(reg + (((c0 + 1) ^ (r & 7)) << 4)) = make_uint4(h16[4], h16[5], h16[6], h16[7]);
        }
      }
      // generic-proxy writes -> visible to the tensor core
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&ctl->v16_full[t]));
        if (kDeq) mbar_arrive(smem_u32(&ctl->k16_full[t]));
        mbar_arrive(smem_u32(&ctl->empty[s]));
      }
    }
    if (!ok) fail(ctl, a.status);
  };
  // FP8 page scales with at most 64 rows per kv head: the softmax warps that own
  // no rows (sub-partitions 2-3) convert, so the converters' issue load leaves
  // the sub-partitions that run the row warps; warps 12-15 then stand aside
  const bool conv_on_idle = KVT == SDVA_KV_FP8_E4M3 && a.R <= 64;
  // Each warpgroup changes its register budget as a whole, before its warps
  // take their roles.
  if (warp >= 8) {
  if constexpr (SM::kConvWarps == 8) {
    if (warp >= kConvWarp) regs_decrease<kRegsConv20>(); else regs_decrease<kRegsIss20>();
  } else {
    regs_decrease<kRegsOther>();
  }
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------
    // producer: page ids and scales prefetched 32 pages at a time, two
    // batches ahead; lane 0 issues the TMA loads.
    // ------------------------------------------------------------------
    if constexpr (!kDeq) {
      prefetch_tmap(&map_k);
      prefetch_tmap(&map_v);
    }
    // Launched as a programmatic dependent of the append (verify_step), the
    // kernel got here while the append may still be writing the cache: wait
    // for it before the first read of a page or a page scale.  (Q, seq_lens
    // and the page table are not written by the append.)  A no-op otherwise.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // (page, kv head) index of position g of this CTA's range, -1 past its
    // end; an out-of-range page id loads page 0 instead and is marked with
    // kBadPage (the lane's rows are then written as zeros and flagged)
    auto locate = [&](long long g) -> int {
      if (g >= n_local) return -1;
      PageIter it;
      it.seek(start + g, ctl->pref, a.B, a.Hkv);
      const int pid = a.page_table[(size_t)it.b * a.max_pages + it.p];
      if (pid < 0 || pid >= a.num_pages) return it.hk | kBadPage;
      return pid * a.Hkv + it.hk;
    };
    // the page's scale terms for the softmax (INT4 and INT8 scales are applied
    // by the converters; FP8 row scales travel in the row-scale stage)
    auto k_scale_of = [&](int ph) -> float {
      return (kDeq || kRow) ? 1.0f : (ph >= 0 ? static_cast<const float*>(a.k_scales)[ph & ~kBadPage] : 0.0f);
    };
    auto v_scale_of = [&](int ph) -> float {
      return (kDeq || kRow) ? 1.0f : (ph >= 0 ? static_cast<const float*>(a.v_scales)[ph & ~kBadPage] : 0.0f);
    };
    // FP8 row: rows of the page at position g that hold the lane's tokens (up
    // to L_b + the lane's window rows); the other rows' scales are not read
    auto written_of = [&](long long g) -> int {
      if (g >= n_local) return 0;
      PageIter it;
      it.seek(start + g, ctl->pref, a.B, a.Hkv);
      int rows = a.W;
      if constexpr (kRagged) rows = min(max(a.n_lane[it.b], 0), a.W);
      const long long end = (long long)ctl->lens[it.b] + rows - (long long)it.p * kPage;
      return (int)max(0LL, min((long long)kPage, end));
    };
    long long issued = 0;
    bool ok = true;
    if constexpr (kDeq) {
      // INT4 / INT8: the scales travel inside the stage (applied by the converters)
      int ph_a = locate(lane), ph_b = locate(32 + lane);
      for (long long g0 = 0; g0 < n_local && ok; g0 += 32) {
        const int ph_c = locate(g0 + 64 + lane);
        for (int i = 0; i < 32 && g0 + i < n_local; ++i) {
          const long long g = g0 + i;
          const int ph_m = __shfl_sync(0xffffffffu, ph_a, i);
          const int ph = ph_m & ~kBadPage;
          const int s = (int)((uint32_t)g % (uint32_t)kNS);
          if (g >= kNS &&
              !(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->empty[s]), (uint32_t)(((uint32_t)g / (uint32_t)kNS - 1) & 1), abort_flag, a.wait_limit)))
            break;
          if (lane == 0) {
            const int page_bad = (ph_m & kBadPage) ? 1 : 0;
            if (page_bad) raise_status(a.status, SDVA_STATUS_BAD_PAGE);
            ctl->bad[s] = page_bad;
            ctl->sk[s] = 1.0f;
            ctl->shift[s] = 0.0f;
            ctl->inv_v[s] = 1.0f;
            const uint32_t bar = smem_u32(&ctl->full[s]);
            const uint32_t dst = stages + s * kStageBytes;
            mbar_arrive_expect_tx(bar, kStageBytes);
            // K codes | V codes | K scales | V scales, each contiguous per (page, kv head)
            constexpr uint32_t kC = SM::kCodeBytes, kS = SM::kScaleBytes;
            bulk_load(dst, a.k_codes + (size_t)ph * kC, kC, bar);
            bulk_load(dst + kC, a.v_codes + (size_t)ph * kC, kC, bar);
            bulk_load(dst + 2 * kC, static_cast<const uint8_t*>(a.k_scales) + (size_t)ph * kS, kS, bar);
            bulk_load(dst + 2 * kC + kS, static_cast<const uint8_t*>(a.v_scales) + (size_t)ph * kS, kS, bar);
          }
          __syncwarp();
          issued = g + 1;
        }
        ph_a = ph_b;
        ph_b = ph_c;
      }
    } else {
      // FP8: page ids and scales prefetched 32 pages at a time, two batches ahead
      int ph_a = locate(lane), ph_b = locate(32 + lane);
      float sk_a = k_scale_of(ph_a), sv_a = v_scale_of(ph_a);
      for (long long g0 = 0; g0 < n_local && ok; g0 += 32) {
        const int ph_c = locate(g0 + 64 + lane);
        const float sk_b = k_scale_of(ph_b), sv_b = v_scale_of(ph_b);
        const int nv_a = kRow ? written_of(g0 + lane) : 0;
        for (int i = 0; i < 32 && g0 + i < n_local; ++i) {
          const long long g = g0 + i;
          const int ph_m = __shfl_sync(0xffffffffu, ph_a, i);
          const int ph = ph_m & ~kBadPage;
          const int s = (int)((uint32_t)g % (uint32_t)kNS);
          if (g >= kNS && !(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->empty[s]), (uint32_t)(((uint32_t)g / (uint32_t)kNS - 1) & 1), abort_flag, a.wait_limit)))
            break;
          const uint32_t bar = smem_u32(&ctl->full[s]);
          if (lane == 0) {
            // the copies go out as soon as the page id is known; the stage's
            // scale terms follow with the barrier's second arrival
            const uint32_t dst = stages + s * kStageBytes;
            mbar_arrive_expect_tx(bar, kStageBytes + (kRow ? kRowScaleBytes : 0));
            tma_load_2d(dst, &map_k, 0, ph * kPage, bar);
            tma_load_2d(dst + kTileBytes, &map_v, 0, ph * kPage, bar);
            if constexpr (kRow) {
              // the page's 64 K and 64 V row scales (256 bytes each per (page, kv head))
              const uint32_t rs = base + SM::kOffRowSc + s * kRowScaleBytes;
              bulk_load(rs, static_cast<const uint8_t*>(a.k_scales) + (size_t)ph * 256, 256, bar);
              bulk_load(rs + 256, static_cast<const uint8_t*>(a.v_scales) + (size_t)ph * 256, 256, bar);
            }
          }
          const float sk = __shfl_sync(0xffffffffu, sk_a, i);
          const float sv = __shfl_sync(0xffffffffu, sv_a, i);
          const int nv = __shfl_sync(0xffffffffu, nv_a, i);
          if (lane == 0) {
            const int page_bad = (ph_m & kBadPage) ? 1 : 0;
            if (page_bad) raise_status(a.status, SDVA_STATUS_BAD_PAGE);
            ctl->bad[s] = page_bad;
            ctl->nv[s] = nv;
            ctl->sk[s] = sk;
            ctl->shift[s] = sv > 0.0f ? log2f(sv) : 0.0f;
            ctl->inv_v[s] = sv > 0.0f ? 1.0f / sv : 1.0f;
            mbar_arrive(bar);
          }
          __syncwarp();
          issued = g + 1;
        }
        ph_a = ph_b;
        sk_a = sk_b;
        sv_a = sv_b;
        ph_b = ph_c;
      }
    }
    if (!ok) {
      fail(ctl, a.status);
      // drain this CTA's own copies still in flight (bounded)
      for (long long g = max(0LL, issued - kNS); g < issued; ++g) {
        int dummy = 0;
        mbar_wait<kSpinWait>(smem_u32(&ctl->full[(uint32_t)g % (uint32_t)kNS]), (uint32_t)(((uint32_t)g / (uint32_t)kNS) & 1), &dummy, 400000000LL);
      }
    }
  } else if (warp == kQkWarp || warp == kQkWarp + 1) {
    // ------------------------------------------------------------------
    // QK issuer of warpgroup j: S = Q K^T for the warpgroup's pages into its
    // two S buffers in turn, each as soon as the page's K has landed and the
    // PV that read the buffer's previous P (two own pages back) has completed.
    // ------------------------------------------------------------------
    const int j = warp - kQkWarp;
    PageIter it;
    it.seek(start, ctl->pref, a.B, a.Hkv);
    uint32_t q_phase = 0;
    bool ok = true;
    long long last = -1;
    long long g = 0;
    while (g < n_local && ok) {
      const long long seg_len = min((long long)(it.nb - it.p), n_local - g);
      if (!(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->q_full), q_phase, abort_flag, a.wait_limit))) break;
      q_phase ^= 1u;
      for (long long h = first_own(g, j); h < g + seg_len; h += 2) {
        const int s = (int)((uint32_t)h % (uint32_t)kNS), t = (int)((uint32_t)h % (uint32_t)kV16Stages);
        // FP8 formats: the page's K tile as loaded; INT4 / INT8: its fp16 K from the converters
        if (!(ok = kDeq ? mbar_wait<kSpinWait>(smem_u32(&ctl->k16_full[t]), (uint32_t)(((uint32_t)h / (uint32_t)kV16Stages) & 1), abort_flag, a.wait_limit)
                         : mbar_wait<kSpinWait>(smem_u32(&ctl->full[s]), (uint32_t)(((uint32_t)h / (uint32_t)kNS) & 1), abort_flag, a.wait_limit)))
          break;
        const long long n = h >> 1;  // the warpgroup's own page index
        const int x = (int)(n & 1);
        if (n >= 2 &&
            !(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->pv_done[j][x]), (uint32_t)(((n >> 1) - 1) & 1), abort_flag, a.wait_limit)))
          break;
        fence_after_sync();
        if (lane == 0) {
          const uint32_t d = tmem + col_s(j, x);
          if constexpr (kDeq) {
            // kind::f16: Q and K as fp16 rows of 128 bytes per 64-dim half
            // (Q halves 16384 bytes apart, K halves 8192)
            const uint32_t kt = k16 + t * kV16Bytes;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_f16_ss(d, sdesc_sw128(qsm + 16384 * (k >> 2) + 32 * (k & 3), 1024, 1024),
                         sdesc_sw128(kt + 8192 * (k >> 2) + 32 * (k & 3), 1024, 1024), kIdescQK16, k == 0 ? 0u : 1u);
            mma_commit(smem_u32(&ctl->s_full[j][x]));
            mma_commit(smem_u32(&ctl->k16_empty[t]));
          } else {
            // kind::f8f6f4: Q_hi and Q_lo (16384 bytes apart) against the K tile as loaded
            const uint32_t ktile = stages + s * kStageBytes;
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_e4m3_ss(d, sdesc_sw128(qsm + 16384 * half + 32 * k, 1024, 1024),
                            sdesc_sw128(ktile + 32 * k, 1024, 1024), kIdescQK, (half == 0 && k == 0) ? 0u : 1u);
            mma_commit(smem_u32(&ctl->s_full[j][x]));
            mma_commit(smem_u32(&ctl->empty[s]));
          }
        }
        __syncwarp();
        last = h;
      }
      if (!ok) break;
      // every QK of this segment is issued: warpgroup 0 may store the next Q
      // once the other issuer is done too (and the softmax has consumed S)
      if (lane == 0) mbar_arrive(smem_u32(&ctl->q_free));
      __syncwarp();
      g += seg_len;
      it.next_unit(ctl->pref, a.B, a.Hkv);
    }
    if (!ok) {
      fail(ctl, a.status);
      // let the tensor core finish what this thread issued before tensor memory is freed
      if (last >= 0) {
        int dummy = 0;
        const long long n = last >> 1;
        mbar_wait<kSpinWait>(smem_u32(&ctl->s_full[j][n & 1]), (uint32_t)((n >> 1) & 1), &dummy, 400000000LL);
      }
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------------
    // PV issuer: O_j += P_j V for every page in order (j = its warpgroup);
    // a warpgroup's first page of a segment starts its O_j afresh.
    // ------------------------------------------------------------------
    PageIter it;
    it.seek(start, ctl->pref, a.B, a.Hkv);
    bool ok = true;
    long long last = -1;
    long long g = 0;
    while (g < n_local && ok) {
      const long long seg_len = min((long long)(it.nb - it.p), n_local - g);
      bool fresh0 = true, fresh1 = true;
      for (long long h = g; h < g + seg_len; ++h) {
        const int j = (int)(h & 1), t = (int)((uint32_t)h % (uint32_t)kV16Stages);
        const long long n = h >> 1;  // the page's index among its warpgroup's pages
        const int x = (int)(n & 1);
        const bool fresh = j ? fresh1 : fresh0;
        if (!(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->p_full[j][x]), (uint32_t)((n >> 1) & 1), abort_flag, a.wait_limit))) break;
        if (!(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->v16_full[t]), (uint32_t)(((uint32_t)h / (uint32_t)kV16Stages) & 1), abort_flag, a.wait_limit))) break;
        fence_after_sync();
        if (lane == 0) {
          const uint32_t vt = v16 + t * kV16Bytes;
          // B: 16 keys per instruction (2048 bytes of both dim halves), the
          // two 64-dim halves 8192 bytes apart (leading byte offset), 8-key
          // groups 1024 bytes apart (stride byte offset)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16_ts(tmem + col_o(j), tmem + col_s(j, x) + 8 * k, sdesc_sw128(vt + 2048 * k, 8192, 1024), kIdescPV,
                       (fresh && k == 0) ? 0u : 1u);
          mma_commit(smem_u32(&ctl->pv_done[j][x]));
          mma_commit(smem_u32(&ctl->v16_empty[t]));
        }
        __syncwarp();
        (j ? fresh1 : fresh0) = false;
        last = h;
      }
      g += seg_len;
      it.next_unit(ctl->pref, a.B, a.Hkv);
    }
    if (!ok) {
      fail(ctl, a.status);
      if (last >= 0) {
        int dummy = 0;
        mbar_wait<kSpinWait>(smem_u32(&ctl->v16_empty[(uint32_t)last % (uint32_t)kV16Stages]), (uint32_t)(((uint32_t)last / (uint32_t)kV16Stages) & 1), &dummy,
                  400000000LL);
      }
    }
  } else if (warp >= kConvWarp) {
    if (!conv_on_idle) convert(threadIdx.x - kConvWarp * 32);
  }
  } else {
    regs_increase<SM::kConvWarps == 8 ? kRegsSoftmax20 : kRegsSoftmax>();
    // ------------------------------------------------------------------
    // softmax warpgroups: wg 0 = warps 0-3 (even positions), wg 1 = warps
    // 4-7 (odd positions); thread = query row = TMEM lane
    // ------------------------------------------------------------------
  if ((warp & 3) * 32 >= a.R) {
    // a softmax warp that owns no query rows
    if (conv_on_idle && (warp & 3) >= 2) convert(((warp >> 2) * 2 + (warp & 3) - 2) * 32 + lane);
  } else {
    const int wg = warp >> 2;
    const int row = threadIdx.x & 127;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const bool warp_active = (warp & 3) * 32 < a.R;
    const bool row_valid = row < a.R;
    const int i_row = row_valid ? row / a.G : a.W - 1;
    PageIter it;
    it.seek(start, ctl->pref, a.B, a.Hkv);
    long long g = 0;
    uint32_t seg_count = 0;
    bool ok = true;
    while (g < n_local) {
      // ---- segment setup ----
      int seg_bad = 0;  // the segment met an out-of-range page id, or the lane's draft tree is invalid
      const int b = it.b, hk = it.hk, nb = it.nb, p0 = it.p;
      const int L = ctl->lens[b];
      const long long g_first = g;
      const long long seg_len = min((long long)(nb - p0), n_local - g);
      const bool whole_unit = (p0 == 0) && seg_len == nb;
      const int u = b * a.Hkv + hk;
      const int h = hk * a.G + (row_valid ? row % a.G : 0);
      const uint16_t* qrow = a.q + (((size_t)b * a.W + i_row) * a.Hq + h) * kHeadDim;
      const int e = kDeq ? (row_valid ? q_row_exponent(qrow) : 0) : q_row_exponent_ldg(row_valid ? qrow : nullptr);
      if (ok && wg == 0 && warp_active) {
        // the previous segment's QKs are all issued (and, through the
        // segment-end handshake, complete): Q may be overwritten
        if (seg_count > 0) ok = mbar_wait<kSpinWait>(smem_u32(&ctl->q_free), (seg_count - 1) & 1u, abort_flag, a.wait_limit);
        if (ok) {
          // Q into the shared-memory A operand of the QK MMAs
          uint8_t* qb = base_ptr + SM::kOffQ;
          if constexpr (kDeq)
            store_q16_row_smem(row_valid ? qrow : nullptr, e, qb, row);
          else
            store_q_row_smem(row_valid ? qrow : nullptr, e, qb, qb + 16384, row);
          fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
          mbar_arrive(smem_u32(&ctl->q_full));
        }
      }
      ++seg_count;
      const float row_scale = ldexpf(a.sm_scale_log2, -e);
      // Draft tree: the window keys L + d this row sees are the set bits d of
      // `vis` -- its own slot and its ancestors, found by walking the parent
      // links, held one per lane of the warp (slot k's parent on lane k).  A
      // parent outside [0, k) makes the lane invalid: its rows are zeroed and
      // SDVA_STATUS_BAD_TREE is raised.
      uint32_t vis = 0u;
      if constexpr (kTree) {
        const int pk = (lane >= 1 && lane < a.W) ? a.parent[(size_t)b * a.W + lane] : 0;
        const bool tree_bad = __any_sync(0xffffffffu, lane >= 1 && lane < a.W && (pk < 0 || pk >= lane));
        int jj = i_row;
#pragma unroll 1
        for (int t = 0; t < kMaxWindow; ++t) {
          vis |= 1u << jj;
          const int up = __shfl_sync(0xffffffffu, pk, jj);
          jj = (jj > 0 && !tree_bad) ? up : 0;
        }
        if (tree_bad) {
          seg_bad = 1;
          if (wg == 0 && row == 0) raise_status(a.status, SDVA_STATUS_BAD_TREE);
        }
      }
      // a row whose visible window keys are slots 0 .. i (a chain) is masked
      // exactly like the causal window
      const bool vis_prefix = !kTree || vis == (2u << i_row) - 1u;
      // per-lane window: rows past the lane's count n_b are written as zeros
      // (a count outside [0, W] zeroes the lane and raises SDVA_STATUS_BAD_COUNT)
      bool row_zero = false;
      if constexpr (kRagged) {
        const int nb_rows = a.n_lane[b];
        if (nb_rows < 0 || nb_rows > a.W) {
          seg_bad = 1;
          if (wg == 0 && row == 0) raise_status(a.status, SDVA_STATUS_BAD_COUNT);
        }
        row_zero = i_row >= nb_rows;
      }

      float m = -INFINITY, l = 0.0f;
      bool had_page = false;
      for (long long k = 0; k < seg_len && ok; ++k, ++g) {
        if ((int)(g & 1) != wg) continue;
        had_page = true;
        if (!warp_active) continue;
        const int j = wg;
        const int p = p0 + (int)k;
        const int s = (int)((uint32_t)g % (uint32_t)kNS);
        const long long n = g >> 1;  // this warpgroup's own page index
        const int xb = (int)(n & 1);  // its S buffer
        if (!(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->s_full[j][xb]), (uint32_t)((n >> 1) & 1), abort_flag, a.wait_limit))) break;
        // the producer staged the page's scale terms before completing full[s]
        if (!(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->full[s]), (uint32_t)(((uint32_t)g / (uint32_t)kNS) & 1), abort_flag, a.wait_limit))) break;
        fence_after_sync();
        const float kscale = ctl->sk[s] * row_scale;
        float shift = ctl->shift[s], inv_f = ctl->inv_v[s];
        seg_bad |= ctl->bad[s];
        if constexpr (!kRow) {
          // the stage's scale terms are in registers: this warp's share of releasing the stage
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->empty[s]));
        }
        uint32_t x[64];
        tmem_ld32(lane_base + col_s(j, xb), *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
        tmem_ld32(lane_base + col_s(j, xb) + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
        tmem_wait_ld();
        if constexpr (kRow) {
          // FP8 row: score j times key j's K scale; the page's largest V row
          // scale is the V scale folded into the shift (the converters
          // divided it out of the fp16 V)
          const float* rs = reinterpret_cast<const float*>(base_ptr + SM::kOffRowSc + s * kRowScaleBytes);
          const float vmax = row_vscale_max(rs, ctl->nv[s], lane);
          shift = vmax > 0.0f ? __log2f(vmax) : 0.0f;
          inv_f = vmax > 0.0f ? __fdividef(1.0f, vmax) : 1.0f;
#pragma unroll
          for (int q = 0; q < 64; q += 4) {
            const float4 k4 = reinterpret_cast<const float4*>(rs)[q >> 2];
            const float2 a = f2_unpack(fmul2(f2_pack(__uint_as_float(x[q]), __uint_as_float(x[q + 1])), f2_pack(k4.x, k4.y)));
            const float2 b = f2_unpack(fmul2(f2_pack(__uint_as_float(x[q + 2]), __uint_as_float(x[q + 3])), f2_pack(k4.z, k4.w)));
            x[q] = __float_as_uint(a.x);
            x[q + 1] = __float_as_uint(a.y);
            x[q + 2] = __float_as_uint(b.x);
            x[q + 3] = __float_as_uint(b.y);
          }
          // the row scales are used: this warp's share of releasing the stage
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->empty[s]));
        }
        const int kbase = p * kPage;
        const int lim = L + i_row;  // causal window: last visible key position of this row
        // a draft tree masks every page that holds window keys key by key:
        // bit q of vm = key kbase + q is visible (cached context, or a window
        // key whose bit is set in vis)
        const int d0 = kbase - L;
        const bool partial = kbase + kPage - 1 > lim || (!vis_prefix && d0 + kPage - 1 >= 0);
        uint64_t vm = 0;
        if (kTree && partial) {
          const int n_ctx = max(0, -d0);  // < 64 on such a page
          vm = d0 <= 0 ? (((1ull << n_ctx) - 1ull) | ((uint64_t)vis << n_ctx)) : ((uint64_t)vis >> min(d0, 63));
        }
        float smax = -INFINITY;
        if (!partial) {
          float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
          for (int q = 0; q < 64; q += 8) {
            m0 = fmax3(m0, __uint_as_float(x[q]), __uint_as_float(x[q + 1]));
            m1 = fmax3(m1, __uint_as_float(x[q + 2]), __uint_as_float(x[q + 3]));
            m2 = fmax3(m2, __uint_as_float(x[q + 4]), __uint_as_float(x[q + 5]));
            m3 = fmax3(m3, __uint_as_float(x[q + 6]), __uint_as_float(x[q + 7]));
          }
          smax = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
        } else {
#pragma unroll
          for (int q = 0; q < 64; ++q)
            if (kTree ? ((vm >> q) & 1ull) != 0 : kbase + q <= lim) smax = fmaxf(smax, __uint_as_float(x[q]));
        }
        const float xmax = smax == -INFINITY ? -INFINITY : fmaf(smax, kscale, shift);
        // The running max may lag the true one by up to kTau (log2 units):
        // weights then reach 2^kTau and P' = w * 2^(15 - kTau) stays <= 2^15,
        // inside fp16.  O is rescaled only when some row of the warp outgrows that.
        const bool need = m != -INFINITY && xmax > m + kTau;
        if (__any_sync(0xffffffffu, need)) {
          // O_j: the PV of the warpgroup's previous page (the latest issued)
          // must have completed
          if (n >= 1 && !(ok = mbar_wait<kSpinWait>(smem_u32(&ctl->pv_done[j][xb ^ 1]), (uint32_t)(((n - 1) >> 1) & 1),
                                         abort_flag, a.wait_limit)))
            break;
          fence_after_sync();
          const float m_new = m == -INFINITY ? m : fmaxf(m, xmax);
          const float alpha = (m == -INFINITY || m_new == m) ? 1.0f : fast_exp2(m - m_new);
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            tmem_ld32(lane_base + col_o(j) + 32 * cc, o);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
            tmem_st32(lane_base + col_o(j) + 32 * cc, o);
          }
          tmem_wait_st();
          l *= alpha;
          m = m_new;
        }
        if (m == -INFINITY) m = xmax;  // first visible key of this row in the segment
        const float bias = shift - (m == -INFINITY ? 0.0f : m) + (15.0f - kTau);
        // P' = 2^(s * kscale + bias) as fp16; P_j column w holds keys 2w, 2w + 1
        float sum = 0.0f;
        const unsigned long long k2 = f2_pack(kscale, kscale), b2 = f2_pack(bias, bias);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t ph[16];
          if (!partial) {
            unsigned long long acc = f2_pack(0.0f, 0.0f);
#pragma unroll
            for (int q = 32 * hf; q < 32 * hf + 32; q += 4) {
              const float2 y01 = f2_unpack(ffma2(f2_pack(__uint_as_float(x[q]), __uint_as_float(x[q + 1])), k2, b2));
              const float2 y23 =
                  f2_unpack(ffma2(f2_pack(__uint_as_float(x[q + 2]), __uint_as_float(x[q + 3])), k2, b2));
              const float w0 = fast_exp2(y01.x), w1 = fast_exp2(y01.y), w2 = fast_exp2(y23.x), w3 = fast_exp2(y23.y);
              acc = fadd2(acc, fadd2(f2_pack(w0, w1), f2_pack(w2, w3)));
              ph[(q & 31) >> 1] = pack_f16x2(w0, w1);
              ph[((q & 31) >> 1) + 1] = pack_f16x2(w2, w3);
            }
            const float2 a2 = f2_unpack(acc);
            sum += a2.x + a2.y;
          } else {
#pragma unroll
            for (int q = 32 * hf; q < 32 * hf + 32; q += 2) {
              const bool v0 = kTree ? ((vm >> q) & 1ull) != 0 : kbase + q <= lim;
              const bool v1 = kTree ? ((vm >> (q + 1)) & 1ull) != 0 : kbase + q + 1 <= lim;
              const float w0 = v0 ? fast_exp2(fmaf(__uint_as_float(x[q]), kscale, bias)) : 0.0f;
              const float w1 = v1 ? fast_exp2(fmaf(__uint_as_float(x[q + 1]), kscale, bias)) : 0.0f;
              sum += w0 + w1;
              ph[(q & 31) >> 1] = pack_f16x2(w0, w1);
            }
          }
          // over the S buffer's first half: its scores are in registers
          tmem_st16(lane_base + col_s(j, xb) + 16 * hf, ph);
        }
        l += sum * (1.0f / kPScale) * inv_f;
        tmem_wait_st();
        fence_before_sync();
        mbar_arrive(smem_u32(&ctl->p_full[j][xb]));
      }
      g = g_first + seg_len;
      it.next_unit(ctl->pref, a.B, a.Hkv);
      // ---- segment end: this warpgroup's last PV must have completed ----
      if (ok && had_page && warp_active) {
        long long g_last = g - 1;
        if ((int)(g_last & 1) != wg) --g_last;
        const long long n_last = g_last >> 1;
        ok = mbar_wait<kSpinWait>(smem_u32(&ctl->pv_done[wg][n_last & 1]), (uint32_t)((n_last >> 1) & 1), abort_flag, a.wait_limit);
        fence_after_sync();
      }
      if (!ok) fail(ctl, a.status);
      // Both warpgroups meet here once per segment, whatever happened, so
      // neither waits on a named barrier the other never reaches.
      if (wg == 1) {
        ctl->m1[row] = (had_page && warp_active) ? m : -INFINITY;
        ctl->l1[row] = (had_page && warp_active) ? l : 0.0f;
        if (row == 0) ctl->bad1 = seg_bad;
        named_arrive(kBarWg1Done, 2 * row_threads);
        named_sync(kBarWg0Done, 2 * row_threads);  // warpgroup 0 has read this warpgroup's O
        fence_after_sync();
        if (ctl->stop) break;
        continue;
      }
      named_sync(kBarWg1Done, 2 * row_threads);
      fence_after_sync();
      const bool stop = !ok || *abort_flag;
      const bool had0 = seg_len > 1 || (g_first & 1) == 0;  // warpgroup 0 owned a page of this segment
      const bool had1 = seg_len > 1 || (g_first & 1) == 1;  // warpgroup 1 owned a page of this segment
      // a page id out of range anywhere in the segment: zero rows for a whole
      // unit, a NaN max marks the partial for the merge
      const bool bad = (seg_bad | ctl->bad1) != 0;
      if (warp_active && !stop && (bad || row_zero) && row_valid) {
        if (whole_unit) {
          uint4* dst = reinterpret_cast<uint4*>(a.out + (((size_t)b * a.W + i_row) * a.Hq + h) * kHeadDim);
#pragma unroll 4
          for (int t = 0; t < 16; ++t) dst[t] = make_uint4(0u, 0u, 0u, 0u);
        } else {
          a.ws_ml[((size_t)(u + c)) * a.R + row] = make_float2(__int_as_float(0x7fc00000), 0.0f);
        }
      }
      // (warp-uniform: the tensor-memory loads below are warp collectives)
      if (warp_active && !stop && !bad) {
        const float m0 = had0 ? m : -INFINITY, l0 = had0 ? l : 0.0f;
        const float mm1 = ctl->m1[row], ll1 = ctl->l1[row];
        const float M = fmaxf(m0, mm1);
        const float a0 = m0 == -INFINITY ? 0.0f : fast_exp2(m0 - M);
        const float a1 = mm1 == -INFINITY ? 0.0f : fast_exp2(mm1 - M);
        const float lt = a0 * l0 + a1 * ll1;
        const size_t slot_row = ((size_t)(u + c)) * a.R + row;
        const float inv = (row_valid && lt > 0.0f) ? 1.0f / (kPScale * lt) : 0.0f;
        uint16_t* orow = nullptr;
        float* prow = nullptr;
        if (row_valid && !row_zero) {
          if (whole_unit)
            orow = a.out + (((size_t)b * a.W + i_row) * a.Hq + h) * kHeadDim;
          else {
            prow = a.ws_o + slot_row * kHeadDim;
            a.ws_ml[slot_row] = make_float2(M, lt);
          }
        }
        const float f0 = had0 ? a0 : 0.0f, f1 = had1 ? a1 : 0.0f;
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t o0[16], o1[16];
          if (had0) tmem_ld16(lane_base + col_o(0) + 16 * cc, o0);
          if (had1) tmem_ld16(lane_base + col_o(1) + 16 * cc, o1);
          tmem_wait_ld();
          if (!had0) {
#pragma unroll
            for (int t = 0; t < 16; ++t) o0[t] = 0u;
          }
          if (!had1) {
#pragma unroll
            for (int t = 0; t < 16; ++t) o1[t] = 0u;
          }
#pragma unroll
          for (int t = 0; t < 16; ++t)
            o0[t] = __float_as_uint(fmaf(f0, __uint_as_float(o0[t]), f1 * __uint_as_float(o1[t])));
          if (orow) {
            uint32_t pk[8];
#pragma unroll
            for (int t = 0; t < 8; ++t)
              pk[t] = pack_bf16x2(__uint_as_float(o0[2 * t]) * inv, __uint_as_float(o0[2 * t + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(orow + 16 * cc);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          } else if (prow) {
            float4* dst = reinterpret_cast<float4*>(prow + 16 * cc);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              dst[t] = make_float4(__uint_as_float(o0[4 * t]) * (1.0f / kPScale),
                                   __uint_as_float(o0[4 * t + 1]) * (1.0f / kPScale),
                                   __uint_as_float(o0[4 * t + 2]) * (1.0f / kPScale),
                                   __uint_as_float(o0[4 * t + 3]) * (1.0f / kPScale));
          }
        }
      }
      if (threadIdx.x == 0) ctl->stop = stop ? 1 : 0;
      fence_before_sync();
      named_arrive(kBarWg0Done, 2 * row_threads);
      if (stop) break;
    }
  }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == kProducerWarp) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge prologue, run by warp 0 of a block: whether lane b's length fits, and
// the first and last CTA whose page range holds part of unit (b, hk) (the
// split kernel's partition, from the same prefix arrays).  pref and cp are
// shared-memory arrays of B + 1 entries.
__device__ __forceinline__ bool merge_locate(const TcArgs& a, int C, int b, int hk, int warp, int lane, int* pref,
                                             int* cp, long long* s_first, long long* s_last) {
  const int L = a.seq_lens[b];
  const bool len_ok = L >= 0 && L <= a.max_context && (long long)L + a.W <= (long long)a.max_pages * kPage;
  if (warp == 0) {
    partition_prefix(a.seq_lens, a.B, a.W, a.max_context, a.max_pages, a.unit_cost, lane, pref, cp, nullptr);
    __syncwarp();
    if (lane == 0 && len_ok) {
      const Partition part{pref, cp, a.B, a.Hkv, a.unit_cost};
      const int nb = pref[b + 1] - pref[b];
      // cost position of the unit's first page (after its start cost)
      const long long y0 = (long long)a.Hkv * cp[b] + (long long)hk * (nb + a.unit_cost) + a.unit_cost;
      const long long Ce = part.ctas(C);
      *s_first = part.cta_of_cost(y0, Ce);
      *s_last = part.cta_of_cost(y0 + nb - 1, Ce);
    }
  }
  return len_ok;
}

// grid: (units, ceil(R / 8)); block 256 = one warp per row, for units that
// span few CTAs.  Same duties as verify_merge_tc_kernel below.
__global__ void __launch_bounds__(256) verify_merge_rows_tc_kernel(TcArgs a, int C) {
  // a following acceptance launched as a programmatic dependent (verify_step)
  // may start now: it reads only the logits
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int u = blockIdx.x;
  const int b = u / a.Hkv, hk = u % a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ long long s_first, s_last;
  __shared__ int s_pref[kMaxLanesTc + 1], s_cp[kMaxLanesTc + 1];
  const bool len_ok = merge_locate(a, C, b, hk, warp, lane, s_pref, s_cp, &s_first, &s_last);
  __syncthreads();
  // programmatic dependent of the split kernel (see verify_merge_tc_kernel)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int r = blockIdx.y * 8 + warp;
  if (r >= a.R) return;
  const int i = r / a.G, h = hk * a.G + r % a.G;
  uint16_t* dst = a.out + (((size_t)b * a.W + i) * a.Hq + h) * kHeadDim + lane * 4;
  if (!len_ok) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
    if (lane == 0 && r == 0 && hk == 0) raise_status(a.status, SDVA_STATUS_OVERFLOW);
    return;
  }
  const long long c_first = s_first, c_last = s_last;
  if (c_first == c_last) return;  // one segment: the split kernel wrote the row
  const int nseg = (int)(c_last - c_first + 1);
  const size_t row0 = (size_t)(u + c_first) * a.R + r;  // segment k's partial row: row0 + k * R
  float M = -INFINITY;
  int bad = 0;
  for (int k = lane; k < nseg; k += 32) {
    const float mk = a.ws_ml[row0 + (size_t)k * a.R].x;
    if (isnan(mk))
      bad = 1;
    else
      M = fmaxf(M, mk);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  }
  if (bad) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
    return;
  }
  // Segments in groups of 32: lane k holds the weight of segment s0 + k; the
  // partial rows are read 8 at a time so their loads are in flight together.
  float den = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int s0 = 0; s0 < nseg; s0 += 32) {
    float wk = 0.0f;
    if (s0 + lane < nseg) {
      const float2 ml = a.ws_ml[row0 + (size_t)(s0 + lane) * a.R];
      wk = ml.x == -INFINITY ? 0.0f : exp2f(ml.x - M);
      den += wk * ml.y;
    }
    const int n = min(32, nseg - s0);
    for (int q = 0; q < n; q += 8) {
      float w[8];
      float4 v[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        w[t] = __shfl_sync(0xffffffffu, wk, (q + t) & 31);
        v[t] = q + t < n ? *reinterpret_cast<const float4*>(a.ws_o + (row0 + (size_t)(s0 + q + t) * a.R) * kHeadDim +
                                                             lane * 4)
                         : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        acc[0] += w[t] * v[t].x;
        acc[1] += w[t] * v[t].y;
        acc[2] += w[t] * v[t].z;
        acc[3] += w[t] * v[t].w;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const float inv = 1.0f / den;
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
}

// grid: (units, R); block 256 = 8 warps on one row, for units that span
// many CTAs (the warps divide the unit's segments).  Zeroes the rows of
// lanes whose length does not fit (and flags them) and of units whose split
// met an out-of-range page id (the split flagged those); merges by
// log-sum-exp the partials of units that span several CTAs.
constexpr int kMergeThreads = 256;
constexpr int kMaxSegments = 1024;  // >= CTAs of the split kernel (one per SM)

__global__ void __launch_bounds__(kMergeThreads) verify_merge_tc_kernel(TcArgs a, int C) {
  // a following acceptance launched as a programmatic dependent (verify_step)
  // may start now: it reads only the logits
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int u = blockIdx.x, r = blockIdx.y;
  const int b = u / a.Hkv, hk = u % a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ long long s_first, s_last;
  __shared__ float2 s_ml[kMaxSegments];
  __shared__ float s_M, s_inv;
  __shared__ int s_bad;
  __shared__ float4 s_acc[kMergeThreads / 32][32];
  __shared__ int s_pref[kMaxLanesTc + 1], s_cp[kMaxLanesTc + 1];
  const bool len_ok = merge_locate(a, C, b, hk, warp, lane, s_pref, s_cp, &s_first, &s_last);
  __syncthreads();
  // launched as a programmatic dependent of the split kernel: everything
  // above overlapped its tail; its partials and rows are visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int i = r / a.G, h = hk * a.G + r % a.G;
  uint16_t* dst = a.out + (((size_t)b * a.W + i) * a.Hq + h) * kHeadDim;
  if (!len_ok) {
    if (threadIdx.x < 32) *reinterpret_cast<uint2*>(dst + 4 * threadIdx.x) = make_uint2(0u, 0u);
    if (threadIdx.x == 0 && r == 0 && hk == 0) raise_status(a.status, SDVA_STATUS_OVERFLOW);
    return;
  }
  const long long c_first = s_first, c_last = s_last;
  if (c_first == c_last) return;  // one segment: the split kernel wrote the row
  const int nseg = (int)(c_last - c_first + 1);
  const size_t row0 = (size_t)(u + c_first) * a.R + r;  // segment k's partial row: row0 + k * R
  for (int k = threadIdx.x; k < nseg; k += kMergeThreads) s_ml[k] = a.ws_ml[row0 + (size_t)k * a.R];
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
    int bad = 0;
    for (int k = lane; k < nseg; k += 32) {
      const float mk = s_ml[k].x;
      if (isnan(mk))
        bad = 1;
      else
        M = fmaxf(M, mk);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    float den = 0.0f;
    for (int k = lane; k < nseg; k += 32) {
      const float2 ml = s_ml[k];
      if (ml.x != -INFINITY) den += exp2f(ml.x - M) * ml.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane == 0) {
      s_M = M;
      s_bad = bad;
      s_inv = 1.0f / den;
    }
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x < 32) *reinterpret_cast<uint2*>(dst + 4 * threadIdx.x) = make_uint2(0u, 0u);
    return;
  }
  // warp w: segments w, w + 8, ...; lane: dims 4 lane .. 4 lane + 3
  const float M = s_M;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
  for (int k = warp; k < nseg; k += kMergeThreads / 32) {
    const float2 ml = s_ml[k];
    const float w = ml.x == -INFINITY ? 0.0f : exp2f(ml.x - M);
    const float4 v = *reinterpret_cast<const float4*>(a.ws_o + (row0 + (size_t)k * a.R) * kHeadDim + lane * 4);
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  s_acc[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float4 t = s_acc[0][lane];
#pragma unroll
    for (int w2 = 1; w2 < kMergeThreads / 32; ++w2) {
      const float4 q = s_acc[w2][lane];
      t.x += q.x;
      t.y += q.y;
      t.z += q.z;
      t.w += q.w;
    }
    const float inv = s_inv;
    *reinterpret_cast<uint2*>(dst + lane * 4) =
        make_uint2(pack_bf16x2(t.x * inv, t.y * inv), pack_bf16x2(t.z * inv, t.w * inv));
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// One (page, kv head) of FP8 codes is 64 rows of 128 bytes; the whole pool is
// a 2-D tensor [num_pages * Hkv * 64][128] bytes, loaded in 64-row boxes with
// the 128-byte swizzle the MMA descriptors expect.
bool encode_pool_map(CUtensorMap* m, const void* pool, long long rows) {
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, 64};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The split kernel, one CTA per SM; with after_append, as a programmatic
// dependent of the kernel before it on the stream (the append of verify_step).
cudaError_t launch_split(void (*kern)(CUtensorMap, CUtensorMap, TcArgs), const CUtensorMap& mk,
                         const CUtensorMap& mv, const TcArgs& args, int num_sms, size_t smem, int threads,
                         cudaStream_t stream, bool after_append) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_append ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, mk, mv, args);
}

int unit_cost_of(int dtype) {
  return dtype == SDVA_KV_FP8_E4M3 ? 20 : 16;
}

size_t tc_workspace_bytes(int B, int W, int Hq, int Hkv, int num_sms) {
  const int R = W * (Hq / Hkv);
  const size_t slots = (size_t)B * Hkv + (size_t)num_sms;
  const size_t ml = (slots * R * sizeof(float2) + 255) / 256 * 256;
  return ml + slots * R * kHeadDim * sizeof(float);
}

bool tc_supported(const sdva_kv_cache* cache, int B, int W, int Hq, int max_pages, int num_sms) {
  const int Hkv = cache->num_kv_heads;
  const int R = W * (Hq / Hkv);
  // the FP8 formats read their code tiles through tensor maps
  const bool dtype_ok = cache->dtype == SDVA_KV_INT4_G32 || cache->dtype == SDVA_KV_INT8_G64 ||
                        ((cache->dtype == SDVA_KV_FP8_E4M3 || cache->dtype == SDVA_KV_FP8_ROW) && encoder() != nullptr);
  // the partition's cost arithmetic is 32-bit (see Partition)
  const bool cost_ok = (long long)B * (max_pages + unit_cost_of(cache->dtype)) * Hkv < (1LL << 31);
  return dtype_ok && cost_ok && R <= 128 && B <= kMaxLanesTc && num_sms > 0 && num_sms <= kMaxSegments &&
         (long long)cache->num_pages * Hkv * kPage < (1LL << 31);
}

// The split kernel for cache format KVT, in the mode the arguments select.
template <int KVT>
int launch_split_kvt(const sdva_kv_cache* cache, const TcArgs& args, int num_sms, cudaStream_t stream,
                     bool after_append) {
  CUtensorMap mk, mv;
  if constexpr (Smem<KVT>::kDeq) {
    // the INT4 and INT8 pools are read with 1-D bulk copies: no tensor maps
    memset(&mk, 0, sizeof(mk));
    memset(&mv, 0, sizeof(mv));
  } else {
    const long long rows = (long long)cache->num_pages * cache->num_kv_heads * kPage;
    if (!encode_pool_map(&mk, cache->k_codes, rows) || !encode_pool_map(&mv, cache->v_codes, rows))
      return SDVA_ERR_CUDA;
  }
  auto kern = args.parent   ? verify_split_tc_kernel<KVT, kModeTree>
              : args.n_lane ? verify_split_tc_kernel<KVT, kModeRagged>
                            : verify_split_tc_kernel<KVT, 0>;
  // the shared-memory limit is a per-device attribute of the function: set it
  // on every call, for the device current now
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<KVT>()) != cudaSuccess)
    return SDVA_ERR_CUDA;
  if (launch_split(kern, mk, mv, args, num_sms, smem_bytes<KVT>(), Smem<KVT>::kThreads, stream, after_append) !=
      cudaSuccess)
    return SDVA_ERR_CUDA;
  return SDVA_OK;
}

int launch_verify_tc(const sdva_kv_cache* cache, const TcArgs& args, int num_sms, cudaStream_t stream,
                     bool after_append) {
  int rc;
  switch (cache->dtype) {
    case SDVA_KV_FP8_E4M3: rc = launch_split_kvt<SDVA_KV_FP8_E4M3>(cache, args, num_sms, stream, after_append); break;
    case SDVA_KV_INT4_G32: rc = launch_split_kvt<SDVA_KV_INT4_G32>(cache, args, num_sms, stream, after_append); break;
    case SDVA_KV_INT8_G64: rc = launch_split_kvt<SDVA_KV_INT8_G64>(cache, args, num_sms, stream, after_append); break;
    case SDVA_KV_FP8_ROW: rc = launch_split_kvt<SDVA_KV_FP8_ROW>(cache, args, num_sms, stream, after_append); break;
    default: return SDVA_ERR_UNSUPPORTED;
  }
  if (rc != SDVA_OK) return rc;
  if (cudaGetLastError() != cudaSuccess) return SDVA_ERR_CUDA;
  // A unit spans about num_sms / units + 1 CTAs: few -> one warp per row, many
  // -> one block of 8 warps per row.
  const bool many = (long long)args.B * args.Hkv * 8 < (long long)num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = many ? dim3(args.B * args.Hkv, args.R, 1) : dim3(args.B * args.Hkv, (args.R + 7) / 8, 1);
  cfg.blockDim = dim3(many ? kMergeThreads : 256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, many ? verify_merge_tc_kernel : verify_merge_rows_tc_kernel, args, num_sms) !=
      cudaSuccess)
    return SDVA_ERR_CUDA;
  return SDVA_OK;
}

}  // namespace tc
}  // namespace sdva
