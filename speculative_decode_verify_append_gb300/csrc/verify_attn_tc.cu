// verify_attn_tc.cu -- verify attention over the FP8 E4M3 paged cache on the
// 5th-generation tensor cores (tcgen05, tensor memory, TMA).
//
// Computes the same thing as the mma.sync path in verify_attn.cu (see there
// and sdva.h): every window row attends over keys 0 .. L_b + i of its kv head.
//
// Design (one persistent CTA of 6 warps per SM):
//   * Work = the flattened list of (lane, kv head, page) triples, cut into
//     one equal contiguous range per CTA (computed on the device from
//     seq_lens, so the launch shape depends only on host arguments).  A
//     maximal run of one (lane, kv head) inside a range is a "segment"; a
//     segment that is a whole unit writes the final bf16 rows, otherwise it
//     writes (m, l, O) partials that verify_merge_tc_kernel combines.  A
//     segment is processed in blocks of up to 4 pages (256 keys).
//   * Warp 4 (producer): TMA-loads each page's K tile into a ring of 4-page
//     blocks (so a block is one contiguous 256-row operand) and its V tile
//     into a ring of page slots (128-byte swizzle), and stages the page's
//     scale terms.
//   * Warp 5 (MMA): one thread issues tcgen05.mma kind::f8f6f4:
//       S[256 keys] = Q_hi K^T + Q_lo K^T   (A = Q from shared memory,
//                                            B = the block's K tiles, N = 256)
//       O += P_hi V + P_lo V                (A = P from tensor memory,
//                                            B = the page's V tile, MN-major)
//     The tensor core streams the 128 rows of A once per instruction, so
//     S is computed 4 pages per instruction; the K/V codes feed it as they
//     are stored, and Q and P are each carried as the sum of two E4M3 terms
//     (hi + lo, 8 significant bits, like bf16).
//   * Warps 0-3 (softmax): thread t owns query row t (TMEM lane t).  Per page
//     it reads its 64 scores, applies the page's K scale and the row's Q
//     scale, masks the window's future keys, runs the online softmax in the
//     log2 domain (the page's V scale folded into the shift), rescales O in
//     tensor memory only when the running max outgrows a lag of kTau, and
//     writes P (hi, lo) to the page's tensor-memory slot.  It releases S as
//     soon as the block's last scores are in registers, so the next block's
//     QK overlaps the rest of the softmax and the PVs.
//   * Every wait is bounded; on timeout the CTA raises SDVA_STATUS_TIMEOUT,
//     drains its own copies, frees tensor memory and returns.
#include "tc_primitives.cuh"
#include "verify_attn_tc.cuh"

namespace sdva {
namespace tc {
namespace {

constexpr int kPagesPerBlock = 4;
constexpr int kKBlocks = 3;    // K ring: blocks of 4 page tiles
constexpr int kVStages = 10;   // V ring: page tiles
constexpr int kTileBytes = 8192;  // one (page, kv head) of FP8 codes: 64 rows x 128 B
constexpr int kKBlockBytes = kPagesPerBlock * kTileBytes;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;
// shared memory (offsets from the 1024-byte aligned base)
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kKBlocks * kKBlockBytes;
constexpr uint32_t kOffQ = kOffV + kVStages * kTileBytes;
constexpr uint32_t kQTermBytes = 128 * 128;  // 128 rows x 128 E4M3 codes, 128-byte swizzle
constexpr uint32_t kOffCtl = kOffQ + 2 * kQTermBytes;
// tensor memory columns
constexpr uint32_t kColS = 0;  // S: 256 fp32 columns (4 pages x 64 keys)
__host__ __device__ constexpr uint32_t col_p(int k) { return 256u + 32u * k; }  // P slot k: hi 16 + lo 16 cols
constexpr uint32_t kColO = 384;  // O: 128 fp32 columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescPV = idesc_e4m3(128, 128, 1);
constexpr float kTau = 2.0f;      // allowed lag of the running max (log2 units)
constexpr float kPScale = 64.0f;  // P' = softmax weight * 2^(8 - kTau) <= 256

struct Ctl {
  uint64_t kfull[kKBlocks];
  uint64_t kempty[kKBlocks];
  uint64_t vfull[kVStages];
  uint64_t vempty[kVStages];
  uint64_t s_full;  // QK of the current block is in S
  uint64_t s_free;  // the softmax has copied the block's S to registers
  uint64_t p_full[kPagesPerBlock];   // P slot k written
  uint64_t pv_done[kPagesPerBlock];  // PV that read P slot k has completed
  uint64_t q_full;
  float sk[kVStages];     // K scale of the page in V slot s
  float shift[kVStages];  // log2 of its V scale (0 when the scale is 0)
  float inv_v[kVStages];  // 1 / V scale (1 when the scale is 0)
  uint32_t tmem_base;
  int abort;
  int pref[kMaxLanesTc + 1];  // pages per kv head of lanes < b (prefix)
  int lens[kMaxLanesTc];      // L_b
};

constexpr size_t kSmemBytes = 1024 + (size_t)kOffCtl + sizeof(Ctl);
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ long long cta_start(long long c, long long C, long long total) { return c * total / C; }

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
  // from the first page of a segment to the first page of the next unit
  __device__ void next_unit(const int* pref, int B, int Hkv) {
    p = nb - 1;
    next(pref, B, Hkv);
  }
};

__device__ __forceinline__ void fail(Ctl* ctl, int32_t* status) {
  if (atomicExch(&ctl->abort, 1) == 0) raise_status(status, SDVA_STATUS_TIMEOUT);
}

__device__ __forceinline__ int block_pages(long long seg_len, int t) {
  return (int)min((long long)kPagesPerBlock, seg_len - (long long)kPagesPerBlock * t);
}

// Two weights -> the hi and lo E4M3 bytes of each (P' = hi + lo to ~8 bits).
__device__ __forceinline__ void split_pair(float w0, float w1, uint32_t& hi2, uint32_t& lo2) {
  const uint32_t h = pack_f16x2(w0, w1);
  hi2 = e4m3x2_from_f16x2(h);
  lo2 = e4m3x2_from_f16x2(hsub2_u32(h, f16x2_from_e4m3x2(hi2)));
}

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

// The Q row scaled by 2^e, split into hi + lo E4M3 codes and stored to row
// `row` of the two shared-memory operand tiles (128-byte swizzle: 16-byte
// chunk c of row r at r * 128 + ((c ^ (r & 7)) << 4)).  A null row stores zeros.
__device__ __forceinline__ void store_q_row_smem(const uint16_t* qrow, int e, uint8_t* qhi, uint8_t* qlo, int row) {
  const float up = ldexpf(1.0f, e);
#pragma unroll 1
  for (int c = 0; c < 8; ++c) {  // 16 elements per 16-byte chunk
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (qrow) v = reinterpret_cast<const uint4*>(qrow)[c * 2 + k];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int t = 0; t < 4; t += 2) {
        const float x0 = bf16_lo(w[t]) * up, x1 = bf16_hi(w[t]) * up;
        const float x2 = bf16_lo(w[t + 1]) * up, x3 = bf16_hi(w[t + 1]) * up;
        const uint32_t h01 = e4m3x2_from_f32(x0, x1), h23 = e4m3x2_from_f32(x2, x3);
        const float2 d01 = f32x2_from_e4m3x2(h01), d23 = f32x2_from_e4m3x2(h23);
        const uint32_t l01 = e4m3x2_from_f32(x0 - d01.x, x1 - d01.y), l23 = e4m3x2_from_f32(x2 - d23.x, x3 - d23.y);
        hw[2 * k + (t >> 1)] = h01 | (h23 << 16);
        lw[2 * k + (t >> 1)] = l01 | (l23 << 16);
      }
    }
    const uint32_t off = (uint32_t)row * 128u + ((uint32_t)(c ^ (row & 7)) << 4);
    *reinterpret_cast<uint4*>(qhi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(qlo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

__global__ void __launch_bounds__(kThreads, 1) verify_split_tc_kernel(const __grid_constant__ CUtensorMap map_k,
                                                                    const __grid_constant__ CUtensorMap map_v,
                                                                    TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  Ctl* ctl = reinterpret_cast<Ctl*>(base_ptr + kOffCtl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = gridDim.x, c = blockIdx.x;
  volatile int* abort_flag = &ctl->abort;

  // ---- partition: pages per kv head of every lane, prefix over lanes ----
  if (warp == 0) {
    int carry = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < a.B) {
        const int L = a.seq_lens[b];
        ctl->lens[b] = L;
        const bool ok = L >= 0 && L <= a.max_context && (long long)L + a.W <= (long long)a.max_pages * kPage;
        n = ok ? (L + a.W + kPage - 1) / kPage : 0;
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (b < a.B) ctl->pref[b] = carry + incl - n;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) ctl->pref[a.B] = carry;
  }
  const uint32_t row_threads = 32u * (uint32_t)min(4, (a.R + 31) / 32);  // softmax threads that own rows
  if (threadIdx.x == 32) {
    for (int s = 0; s < kKBlocks; ++s) {
      mbar_init(smem_u32(&ctl->kfull[s]), 1);
      mbar_init(smem_u32(&ctl->kempty[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&ctl->vfull[s]), 1);
      mbar_init(smem_u32(&ctl->vempty[s]), 1);
    }
    mbar_init(smem_u32(&ctl->s_full), 1);
    mbar_init(smem_u32(&ctl->s_free), row_threads);
    for (int k = 0; k < kPagesPerBlock; ++k) {
      mbar_init(smem_u32(&ctl->p_full[k]), row_threads);
      mbar_init(smem_u32(&ctl->pv_done[k]), 1);
    }
    mbar_init(smem_u32(&ctl->q_full), row_threads);
    ctl->abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const long long total = (long long)a.Hkv * ctl->pref[a.B];
  const long long start = cta_start(c, C, total), end = cta_start(c + 1, C, total);
  const long long n_local = end - start;
  if (n_local <= 0) return;  // uniform for the whole CTA

  if (warp == kMmaWarp) tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------
    // producer: page ids and scales prefetched 32 pages at a time, two
    // batches ahead; lane 0 issues the TMA loads.
    // ------------------------------------------------------------------
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
    auto locate = [&](long long g, int& row_coord, int& ph_out) {
      row_coord = 0;
      ph_out = -1;
      if (g < n_local) {
        PageIter it;
        it.seek(start + g, ctl->pref, a.B, a.Hkv);
        int pid = a.page_table[(size_t)it.b * a.max_pages + it.p];
        if (pid < 0 || pid >= a.num_pages) pid = 0;  // the merge zeroes lanes with bad ids
        ph_out = pid * a.Hkv + it.hk;
        row_coord = ph_out * kPage;
      }
    };
    int rc_a, ph_a, rc_b, ph_b;
    locate(lane, rc_a, ph_a);
    locate(32 + lane, rc_b, ph_b);
    float sk_a = ph_a >= 0 ? a.k_scales[ph_a] : 0.0f;
    float sv_a = ph_a >= 0 ? a.v_scales[ph_a] : 0.0f;
    PageIter it;
    it.seek(start, ctl->pref, a.B, a.Hkv);
    long long seg_left = 0, bi = 0;
    int blk_left = 0, kk = 0;
    long long issued = 0;
    bool ok = true;
    for (long long g0 = 0; g0 < n_local && ok; g0 += 32) {
      int rc_c, ph_c;
      locate(g0 + 64 + lane, rc_c, ph_c);
      const float sk_b = ph_b >= 0 ? a.k_scales[ph_b] : 0.0f;
      const float sv_b = ph_b >= 0 ? a.v_scales[ph_b] : 0.0f;
      const float shift_a = sv_a > 0.0f ? log2f(sv_a) : 0.0f;
      const float inv_a = sv_a > 0.0f ? 1.0f / sv_a : 1.0f;
      for (int i = 0; i < 32 && g0 + i < n_local; ++i) {
        const long long g = g0 + i;
        const int rc = __shfl_sync(0xffffffffu, rc_a, i);
        const float sk = __shfl_sync(0xffffffffu, sk_a, i);
        const float sh = __shfl_sync(0xffffffffu, shift_a, i);
        const float iv = __shfl_sync(0xffffffffu, inv_a, i);
        if (seg_left == 0) seg_left = min((long long)(it.nb - it.p), n_local - g);
        const int bs = (int)(bi % kKBlocks);
        if (blk_left == 0) {
          // a new block of up to 4 pages of this segment
          blk_left = (int)min((long long)kPagesPerBlock, seg_left);
          kk = 0;
          if (bi >= kKBlocks &&
              !(ok = mbar_wait(smem_u32(&ctl->kempty[bs]), (uint32_t)((bi / kKBlocks - 1) & 1), abort_flag)))
            break;
          if (lane == 0) mbar_arrive_expect_tx(smem_u32(&ctl->kfull[bs]), (uint32_t)blk_left * kTileBytes);
        }
        const int vs = (int)(g % kVStages);
        if (g >= kVStages &&
            !(ok = mbar_wait(smem_u32(&ctl->vempty[vs]), (uint32_t)((g / kVStages - 1) & 1), abort_flag)))
          break;
        if (lane == 0) {
          ctl->sk[vs] = sk;
          ctl->shift[vs] = sh;
          ctl->inv_v[vs] = iv;
          const uint32_t vbar = smem_u32(&ctl->vfull[vs]);
          mbar_arrive_expect_tx(vbar, kTileBytes);
          tma_load_2d(base + kOffV + vs * kTileBytes, &map_v, 0, rc, vbar);
          tma_load_2d(base + kOffK + bs * kKBlockBytes + kk * kTileBytes, &map_k, 0, rc,
                      smem_u32(&ctl->kfull[bs]));
        }
        __syncwarp();
        issued = g + 1;
        ++kk;
        --seg_left;
        if (--blk_left == 0) ++bi;
        it.next(ctl->pref, a.B, a.Hkv);
      }
      rc_a = rc_b;
      sk_a = sk_b;
      sv_a = sv_b;
      rc_b = rc_c;
      ph_b = ph_c;
    }
    if (!ok) {
      fail(ctl, a.status);
      // drain this CTA's own copies still in flight (bounded)
      for (long long g = max(0LL, issued - kVStages); g < issued; ++g) {
        int dummy = 0;
        mbar_wait(smem_u32(&ctl->vfull[g % kVStages]), (uint32_t)((g / kVStages) & 1), &dummy, 400000000LL);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------
    // MMA issuer.  Per block: the PVs of the pages before its last pair,
    // then (within a segment) the next block's QK as soon as S is free, then
    // the PVs of the last pair.  All PVs of a segment are issued before the
    // next segment's Q is awaited.
    // ------------------------------------------------------------------
    PageIter it;
    it.seek(start, ctl->pref, a.B, a.Hkv);
    uint32_t q_phase = 0;
    uint32_t slot_use[kPagesPerBlock] = {0u, 0u, 0u, 0u};
    bool ok = true;
    long long last_pv = -1;
    const uint32_t qhi = base + kOffQ, qlo = base + kOffQ + kQTermBytes;
    auto issue_qk = [&](long long b, int npg) -> bool {
      const int bs = (int)(b % kKBlocks);
      if (!mbar_wait(smem_u32(&ctl->kfull[bs]), (uint32_t)((b / kKBlocks) & 1), abort_flag)) return false;
      if (b > 0 && !mbar_wait(smem_u32(&ctl->s_free), (uint32_t)((b - 1) & 1), abort_flag)) return false;
      fence_after_sync();
      if (lane == 0) {
        const uint32_t kblk = base + kOffK + bs * kKBlockBytes;
        const uint32_t idesc = idesc_e4m3(128, 64 * npg, 0);
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_e4m3_ss(tmem + kColS, sdesc_sw128((half ? qlo : qhi) + 32 * k, 1024, 1024),
                        sdesc_sw128(kblk + 32 * k, 1024, 1024), idesc, (half == 0 && k == 0) ? 0u : 1u);
        mma_commit(smem_u32(&ctl->s_full));
        mma_commit(smem_u32(&ctl->kempty[bs]));
      }
      __syncwarp();
      return true;
    };
    auto issue_pv = [&](long long gp, int k, bool first_of_seg) -> bool {
      const int vs = (int)(gp % kVStages);
      if (!mbar_wait(smem_u32(&ctl->vfull[vs]), (uint32_t)((gp / kVStages) & 1), abort_flag)) return false;
      if (!mbar_wait(smem_u32(&ctl->p_full[k]), slot_use[k] & 1u, abort_flag)) return false;
      fence_after_sync();
      if (lane == 0) {
        const uint32_t vtile = base + kOffV + vs * kTileBytes;
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_e4m3_ts(tmem + kColO, tmem + col_p(k) + 16 * half + 8 * kk,
                        sdesc_sw128(vtile + 4096 * kk, 1024, 1024), kIdescPV,
                        (first_of_seg && half == 0 && kk == 0) ? 0u : 1u);
        mma_commit(smem_u32(&ctl->pv_done[k]));
        mma_commit(smem_u32(&ctl->vempty[vs]));
      }
      __syncwarp();
      ++slot_use[k];
      last_pv = gp;
      return true;
    };
    long long g = 0, bi = 0;
    while (g < n_local && ok) {
      const long long s0 = g, seg_len = min((long long)(it.nb - it.p), n_local - g);
      const int nblk = (int)((seg_len + kPagesPerBlock - 1) / kPagesPerBlock);
      if (!(ok = mbar_wait(smem_u32(&ctl->q_full), q_phase, abort_flag))) break;
      q_phase ^= 1u;
      if (!(ok = issue_qk(bi, block_pages(seg_len, 0)))) break;
      for (int t = 0; t < nblk && ok; ++t, ++bi) {
        const int npg = block_pages(seg_len, t);
        const long long g0 = s0 + (long long)kPagesPerBlock * t;
        const int last_pair = npg > 2 ? 2 : 0;
        for (int k = 0; k < last_pair && ok; ++k) ok = issue_pv(g0 + k, k, g0 + k == s0);
        if (ok && t + 1 < nblk) ok = issue_qk(bi + 1, block_pages(seg_len, t + 1));
        for (int k = last_pair; k < npg && ok; ++k) ok = issue_pv(g0 + k, k, g0 + k == s0);
      }
      it.next_unit(ctl->pref, a.B, a.Hkv);
      g = s0 + seg_len;
    }
    if (!ok) {
      fail(ctl, a.status);
      // let the tensor core finish what this thread issued before tensor memory is freed
      if (last_pv >= 0) {
        int dummy = 0;
        mbar_wait(smem_u32(&ctl->vempty[last_pv % kVStages]), (uint32_t)((last_pv / kVStages) & 1), &dummy,
                  400000000LL);
      }
    }
  } else if (warp < 4 && warp * 32 < a.R) {
    // ------------------------------------------------------------------
    // softmax: thread = query row = TMEM lane (warps without rows idle)
    // ------------------------------------------------------------------
    const int row = threadIdx.x;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const bool row_valid = row < a.R;
    const int i_row = row_valid ? row / a.G : a.W - 1;
    uint8_t* qhi = base_ptr + kOffQ;
    uint8_t* qlo = base_ptr + kOffQ + kQTermBytes;
    PageIter it;
    it.seek(start, ctl->pref, a.B, a.Hkv);
    uint32_t slot_use[kPagesPerBlock] = {0u, 0u, 0u, 0u};
    long long g = 0, bi = 0;
    int last_slot = -1;
    uint32_t last_use = 0;
    bool ok = true;
    while (g < n_local && ok) {
      // ---- segment setup: Q of this (lane, kv head) into shared memory ----
      const int b = it.b, hk = it.hk, nb = it.nb, p0 = it.p;
      const int L = ctl->lens[b];
      const long long seg_len = min((long long)(nb - p0), n_local - g);
      const bool whole_unit = (p0 == 0) && seg_len == nb;
      const int u = b * a.Hkv + hk;
      const int h = hk * a.G + (row_valid ? row % a.G : 0);
      const uint16_t* qrow = a.q + (((size_t)b * a.W + i_row) * a.Hq + h) * kHeadDim;
      const int e = row_valid ? q_row_exponent(qrow) : 0;
      store_q_row_smem(row_valid ? qrow : nullptr, e, qhi, qlo, row);
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&ctl->q_full));
      const float row_scale = ldexpf(a.sm_scale_log2, -e);

      float m = -INFINITY, l = 0.0f;
      const int nblk = (int)((seg_len + kPagesPerBlock - 1) / kPagesPerBlock);
      for (int t = 0; t < nblk && ok; ++t, ++bi) {
        const int npg = block_pages(seg_len, t);
        const long long g0 = g + (long long)kPagesPerBlock * t;
        if (!(ok = mbar_wait(smem_u32(&ctl->s_full), (uint32_t)(bi & 1), abort_flag))) break;
        fence_after_sync();
        for (int pair = 0; pair * 2 < npg && ok; ++pair) {
          // the scores of up to two pages in registers
          uint32_t xs[2][64];
          const int k0 = 2 * pair;
          tmem_ld32(lane_base + kColS + 64 * k0, *reinterpret_cast<uint32_t(*)[32]>(&xs[0][0]));
          tmem_ld32(lane_base + kColS + 64 * k0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&xs[0][32]));
          if (k0 + 1 < npg) {
            tmem_ld32(lane_base + kColS + 64 * (k0 + 1), *reinterpret_cast<uint32_t(*)[32]>(&xs[1][0]));
            tmem_ld32(lane_base + kColS + 64 * (k0 + 1) + 32, *reinterpret_cast<uint32_t(*)[32]>(&xs[1][32]));
          }
          tmem_wait_ld();
          if (k0 + 2 >= npg) {
            // the block's last scores are in registers: the MMA may compute the next block's S
            fence_before_sync();
            mbar_arrive(smem_u32(&ctl->s_free));
          }
          for (int kp = 0; kp < 2 && k0 + kp < npg && ok; ++kp) {
            const int k = k0 + kp;
            const long long gp = g0 + k;
            const int vs = (int)(gp % kVStages);
            // the producer staged this page's scale terms before completing vfull
            if (!(ok = mbar_wait(smem_u32(&ctl->vfull[vs]), (uint32_t)((gp / kVStages) & 1), abort_flag))) break;
            const float kscale = ctl->sk[vs] * row_scale, shift = ctl->shift[vs], inv_f = ctl->inv_v[vs];
            const uint32_t* x = xs[kp];
            const int kbase = (p0 + kPagesPerBlock * t + k) * kPage;
            const int lim = L + i_row;  // last visible key position of this row
            const bool partial = kbase + kPage - 1 > lim;
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
                if (kbase + q <= lim) smax = fmaxf(smax, __uint_as_float(x[q]));
            }
            const float xmax = smax == -INFINITY ? -INFINITY : fmaf(smax, kscale, shift);
            // The running max may lag the true one by up to kTau (log2 units):
            // weights then reach 2^kTau and P' = w * 2^(8 - kTau) stays <= 256.
            // O is rescaled only when some row of the warp outgrows that.
            const bool need = m != -INFINITY && xmax > m + kTau;
            if (__any_sync(0xffffffffu, need)) {
              // every PV of this segment so far must be complete
              if (!(ok = mbar_wait(smem_u32(&ctl->pv_done[last_slot]), last_use & 1u, abort_flag))) break;
              fence_after_sync();
              const float m_new = m == -INFINITY ? m : fmaxf(m, xmax);
              const float alpha = (m == -INFINITY || m_new == m) ? 1.0f : fast_exp2(m - m_new);
#pragma unroll 1
              for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
                tmem_ld32(lane_base + kColO + 32 * cc, o);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
                tmem_st32(lane_base + kColO + 32 * cc, o);
              }
              tmem_wait_st();
              l *= alpha;
              m = m_new;
            }
            if (m == -INFINITY) m = xmax;  // first visible key of this row in the segment
            const float bias = shift - (m == -INFINITY ? 0.0f : m) + (8.0f - kTau);
            uint32_t phi[16], plo[16];
            float sum;
            if (!partial) {
              const unsigned long long k2 = f2_pack(kscale, kscale), b2 = f2_pack(bias, bias);
              unsigned long long acc = f2_pack(0.0f, 0.0f);
#pragma unroll
              for (int q = 0; q < 64; q += 4) {
                const float2 y01 = f2_unpack(ffma2(f2_pack(__uint_as_float(x[q]), __uint_as_float(x[q + 1])), k2, b2));
                const float2 y23 =
                    f2_unpack(ffma2(f2_pack(__uint_as_float(x[q + 2]), __uint_as_float(x[q + 3])), k2, b2));
                const float w0 = fast_exp2(y01.x), w1 = fast_exp2(y01.y), w2 = fast_exp2(y23.x), w3 = fast_exp2(y23.y);
                acc = fadd2(acc, fadd2(f2_pack(w0, w1), f2_pack(w2, w3)));
                uint32_t h01, l01, h23, l23;
                split_pair(w0, w1, h01, l01);
                split_pair(w2, w3, h23, l23);
                phi[q >> 2] = __byte_perm(h01, h23, 0x5410);
                plo[q >> 2] = __byte_perm(l01, l23, 0x5410);
              }
              const float2 a2 = f2_unpack(acc);
              sum = a2.x + a2.y;
            } else {
              sum = 0.0f;
#pragma unroll
              for (int q = 0; q < 64; q += 4) {
                float w[4];
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4)
                  w[r4] = kbase + q + r4 <= lim ? fast_exp2(fmaf(__uint_as_float(x[q + r4]), kscale, bias)) : 0.0f;
                sum += (w[0] + w[1]) + (w[2] + w[3]);
                uint32_t h01, l01, h23, l23;
                split_pair(w[0], w[1], h01, l01);
                split_pair(w[2], w[3], h23, l23);
                phi[q >> 2] = __byte_perm(h01, h23, 0x5410);
                plo[q >> 2] = __byte_perm(l01, l23, 0x5410);
              }
            }
            l += sum * (1.0f / kPScale) * inv_f;
            // P slot k is free once the PV of its previous use has completed
            if (slot_use[k] > 0 &&
                !(ok = mbar_wait(smem_u32(&ctl->pv_done[k]), (slot_use[k] - 1u) & 1u, abort_flag)))
              break;
            tmem_st16(lane_base + col_p(k), phi);
            tmem_st16(lane_base + col_p(k) + 16, plo);
            tmem_wait_st();
            fence_before_sync();
            mbar_arrive(smem_u32(&ctl->p_full[k]));
            last_slot = k;
            last_use = slot_use[k]++;
          }
        }
      }
      if (!ok) break;
      // ---- segment epilogue: every PV of the segment must have completed ----
      if (!(ok = mbar_wait(smem_u32(&ctl->pv_done[last_slot]), last_use & 1u, abort_flag))) break;
      fence_after_sync();
      const size_t slot_row = ((size_t)(u + c)) * a.R + row;
      const float inv = (row_valid && l > 0.0f) ? 1.0f / (kPScale * l) : 0.0f;
      uint16_t* orow = nullptr;
      float* prow = nullptr;
      if (row_valid) {
        if (whole_unit)
          orow = a.out + (((size_t)b * a.W + i_row) * a.Hq + h) * kHeadDim;
        else {
          prow = a.ws_o + slot_row * kHeadDim;
          a.ws_ml[slot_row] = make_float2(m, l);
        }
      }
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        tmem_ld32(lane_base + kColO + 32 * cc, o);
        tmem_wait_ld();
        if (orow) {
#pragma unroll
          for (int q = 0; q < 32; q += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[q]) * inv, __uint_as_float(o[q + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[q + 2]) * inv, __uint_as_float(o[q + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[q + 4]) * inv, __uint_as_float(o[q + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[q + 6]) * inv, __uint_as_float(o[q + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + 32 * cc + q) = w;
          }
        } else if (prow) {
#pragma unroll
          for (int q = 0; q < 32; q += 4)
            *reinterpret_cast<float4*>(prow + 32 * cc + q) =
                make_float4(__uint_as_float(o[q]) * (1.0f / kPScale), __uint_as_float(o[q + 1]) * (1.0f / kPScale),
                            __uint_as_float(o[q + 2]) * (1.0f / kPScale), __uint_as_float(o[q + 3]) * (1.0f / kPScale));
        }
      }
      g += seg_len;
      it.next_unit(ctl->pref, a.B, a.Hkv);
    }
    if (!ok) fail(ctl, a.status);
  }

  fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// grid: (units, ceil(R / 8)); block 256 = one warp per row.  Zeroes the rows
// of invalid lanes (and flags them); merges the partials of units that span
// several CTAs by log-sum-exp.
__global__ void __launch_bounds__(256) verify_merge_tc_kernel(TcArgs a, int C) {
  const int u = blockIdx.x;
  const int b = u / a.Hkv, hk = u % a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int s_bad;
  __shared__ long long s_first, s_last, s_total;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const int L = a.seq_lens[b];
  const bool len_ok = L >= 0 && L <= a.max_context && (long long)L + a.W <= (long long)a.max_pages * kPage;
  const int nb = len_ok ? (L + a.W + kPage - 1) / kPage : 0;
  if (!len_ok) {
    if (threadIdx.x == 0) s_bad = SDVA_STATUS_OVERFLOW;
  } else {
    const int32_t* prow = a.page_table + (size_t)b * a.max_pages;
    for (int p = threadIdx.x; p < nb; p += blockDim.x) {
      const int id = prow[p];
      if (id < 0 || id >= a.num_pages) s_bad = SDVA_STATUS_BAD_PAGE;
    }
  }
  if (warp == 0) {
    // pages before this lane and in total (same rule as the split kernel)
    long long before = 0, all = 0;
    for (int bb = lane; bb < a.B; bb += 32) {
      const int Lb = a.seq_lens[bb];
      const bool ok = Lb >= 0 && Lb <= a.max_context && (long long)Lb + a.W <= (long long)a.max_pages * kPage;
      const int n = ok ? (Lb + a.W + kPage - 1) / kPage : 0;
      all += n;
      if (bb < b) before += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    if (lane == 0 && len_ok) {
      const long long total = (long long)a.Hkv * all;
      const long long Pu = (long long)a.Hkv * before + (long long)hk * nb;
      auto locate = [&](long long x) {
        long long cc = x * C / total;
        while (cc + 1 < C && cta_start(cc + 1, C, total) <= x) ++cc;
        while (cc > 0 && cta_start(cc, C, total) > x) --cc;
        return cc;
      };
      s_first = locate(Pu);
      s_last = locate(Pu + nb - 1);
      s_total = total;
    }
  }
  __syncthreads();
  const int bad = s_bad;
  const int r = blockIdx.y * 8 + warp;
  if (bad) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && hk == 0) raise_status(a.status, bad);
    if (r < a.R) {
      const int i = r / a.G, h = hk * a.G + r % a.G;
      uint16_t* dst = a.out + (((size_t)b * a.W + i) * a.Hq + h) * kHeadDim + lane * 4;
      *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
    }
    return;
  }
  const long long c_first = s_first, c_last = s_last, total = s_total;
  if (c_first == c_last || r >= a.R) return;  // one segment: the split kernel wrote the rows
  const int nseg = (int)(c_last - c_first + 1);
  float M = -INFINITY;
  for (int sgi = lane; sgi < nseg; sgi += 32) {
    const long long cc = c_first + sgi;
    if (cta_start(cc, C, total) == cta_start(cc + 1, C, total)) continue;
    M = fmaxf(M, a.ws_ml[(size_t)(u + cc) * a.R + r].x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float den = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
  for (int sgi = 0; sgi < nseg; ++sgi) {
    const long long cc = c_first + sgi;
    if (cta_start(cc, C, total) == cta_start(cc + 1, C, total)) continue;
    const size_t slot_row = (size_t)(u + cc) * a.R + r;
    const float2 ml = a.ws_ml[slot_row];
    const float4 v = *reinterpret_cast<const float4*>(a.ws_o + slot_row * kHeadDim + lane * 4);
    const float w = ml.x == -INFINITY ? 0.0f : exp2f(ml.x - M);
    den += w * ml.y;
    acc[0] += w * v.x;
    acc[1] += w * v.y;
    acc[2] += w * v.z;
    acc[3] += w * v.w;
  }
  const float inv = 1.0f / den;
  const int i = r / a.G, h = hk * a.G + r % a.G;
  uint16_t* dst = a.out + (((size_t)b * a.W + i) * a.Hq + h) * kHeadDim + lane * 4;
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
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

size_t tc_workspace_bytes(int B, int W, int Hq, int Hkv, int num_sms) {
  const int R = W * (Hq / Hkv);
  const size_t slots = (size_t)B * Hkv + (size_t)num_sms;
  const size_t ml = (slots * R * sizeof(float2) + 255) / 256 * 256;
  return ml + slots * R * kHeadDim * sizeof(float);
}

bool tc_supported(const sdva_kv_cache* cache, int B, int W, int Hq, int num_sms) {
  const int Hkv = cache->num_kv_heads;
  const int R = W * (Hq / Hkv);
  return cache->dtype == SDVA_KV_FP8_E4M3 && R <= 128 && B <= kMaxLanesTc && num_sms > 0 &&
         (long long)cache->num_pages * Hkv * kPage < (1LL << 31) && encoder() != nullptr;
}

int launch_verify_tc(const sdva_kv_cache* cache, const TcArgs& args, int num_sms, cudaStream_t stream) {
  CUtensorMap mk, mv;
  const long long rows = (long long)cache->num_pages * cache->num_kv_heads * kPage;
  if (!encode_pool_map(&mk, cache->k_codes, rows) || !encode_pool_map(&mv, cache->v_codes, rows)) return SDVA_ERR_CUDA;
  cudaFuncSetAttribute(verify_split_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  verify_split_tc_kernel<<<num_sms, kThreads, kSmemBytes, stream>>>(mk, mv, args);
  if (cudaGetLastError() != cudaSuccess) return SDVA_ERR_CUDA;
  verify_merge_tc_kernel<<<dim3(args.B * args.Hkv, (args.R + 7) / 8), 256, 0, stream>>>(args, num_sms);
  return cudaGetLastError() == cudaSuccess ? SDVA_OK : SDVA_ERR_CUDA;
}

}  // namespace tc
}  // namespace sdva
