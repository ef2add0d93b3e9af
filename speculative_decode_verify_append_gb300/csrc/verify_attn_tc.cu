// verify_attn_tc.cu -- verify attention over the FP8 E4M3 paged cache on the
// 5th-generation tensor cores (tcgen05, tensor memory, TMA).
//
// Computes the same thing as the mma.sync path in verify_attn.cu (see there
// and sdva.h): every window row attends over keys 0 .. L_b + i of its kv head.
//
// Design (one persistent CTA per SM):
//   * Work = the flattened list of (lane, kv head, page) triples, cut into
//     one equal contiguous range per CTA (computed on the device from
//     seq_lens, so the launch shape depends only on host arguments).  A
//     maximal run of one (lane, kv head) inside a range is a "segment"; a
//     segment that is a whole unit writes the final bf16 rows, otherwise it
//     writes (m, l, O) partials that verify_merge_tc_kernel combines.
//   * Warp 4 (producer): TMA-loads each page's K and V tiles (8 KB each,
//     128-byte swizzle) into a ring of shared-memory stages.
//   * Warp 5 (MMA): one thread issues tcgen05.mma kind::f8f6f4:
//       S = Q_hi K^T + Q_lo K^T        (A = Q from tensor memory, B = K tile)
//       O += P_hi V + P_lo V           (A = P from tensor memory, B = V tile,
//                                       MN-major)
//     The K/V codes feed the tensor cores as they are stored; Q and P are
//     each carried as the sum of two E4M3 terms (hi + lo, 8 significant
//     bits, like bf16), so no dequantisation pass touches shared memory.
//   * Warps 0-3 (softmax): thread t owns TMEM lane t = query row t.  It reads
//     its 64 scores of a page, applies the page's K scale and the row's Q
//     scale, masks the window's future keys, runs the online softmax in the
//     log2 domain (the page's V scale folded into the shift), rescales O in
//     tensor memory only when the running max grows, and writes P (hi, lo)
//     back to tensor memory for the next MMA.
//   * Every wait is bounded; on timeout the CTA raises SDVA_STATUS_TIMEOUT,
//     drains its own copies, frees tensor memory and returns.
#include "tc_primitives.cuh"
#include "verify_attn_tc.cuh"

namespace sdva {
namespace tc {
namespace {

constexpr int kStages = 10;
constexpr int kStageBytes = 16384;  // K tile + V tile of one (page, kv head)
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;
constexpr uint32_t kColQ = 0;    // Q hi: 32 cols, Q lo: 32 cols
constexpr uint32_t kColP = 64;   // P buffer j at 64 + 32 j: hi 16 cols, lo 16 cols
constexpr uint32_t kColS = 128;  // S buffer j at 128 + 64 j: 64 fp32 cols
constexpr uint32_t kColO = 256;  // O: 128 fp32 cols
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescQK = idesc_e4m3(128, 64, 0);
constexpr uint32_t kIdescPV = idesc_e4m3(128, 128, 1);

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t q_full;
  float sk[kStages];
  float sv[kStages];
  uint32_t tmem_base;
  int abort;
  int pref[kMaxLanesTc + 1];  // pages per kv head of lanes < b (prefix)
  int lens[kMaxLanesTc];      // L_b
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + sizeof(Ctl);

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
};

__device__ __forceinline__ void fail(Ctl* ctl, int32_t* status) {
  if (atomicExch(&ctl->abort, 1) == 0) raise_status(status, SDVA_STATUS_TIMEOUT);
}

__global__ void __launch_bounds__(kThreads, 1) verify_split_tc_kernel(const __grid_constant__ CUtensorMap map_k,
                                                                    const __grid_constant__ CUtensorMap map_v,
                                                                    TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  Ctl* ctl = reinterpret_cast<Ctl*>(base_ptr + (size_t)kStages * kStageBytes);
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
  if (threadIdx.x == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_u32(&ctl->s_full[j]), 1);
      mbar_init(smem_u32(&ctl->p_full[j]), 128);
      mbar_init(smem_u32(&ctl->o_done[j]), 1);
    }
    mbar_init(smem_u32(&ctl->q_full), 128);
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
  const uint32_t stages = base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------
    // producer: page ids and scales prefetched 32 pages at a time, two
    // batches ahead; lane 0 issues the TMA loads.
    // ------------------------------------------------------------------
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
    auto locate = [&](long long g, int& row_coord, int& pid_out) {
      row_coord = 0;
      pid_out = -1;
      if (g < n_local) {
        PageIter it;
        it.seek(start + g, ctl->pref, a.B, a.Hkv);
        int pid = a.page_table[(size_t)it.b * a.max_pages + it.p];
        if (pid < 0 || pid >= a.num_pages) pid = 0;  // the merge zeroes lanes with bad ids
        pid_out = pid * a.Hkv + it.hk;
        row_coord = pid_out * kPage;
      }
    };
    int rc_a, ph_a, rc_b, ph_b;
    locate(lane, rc_a, ph_a);
    locate(32 + lane, rc_b, ph_b);
    float sk_a = ph_a >= 0 ? a.k_scales[ph_a] : 0.0f;
    float sv_a = ph_a >= 0 ? a.v_scales[ph_a] : 0.0f;
    long long issued = 0;
    bool ok = true;
    for (long long g0 = 0; g0 < n_local && ok; g0 += 32) {
      int rc_c, ph_c;
      locate(g0 + 64 + lane, rc_c, ph_c);
      const float sk_b = ph_b >= 0 ? a.k_scales[ph_b] : 0.0f;
      const float sv_b = ph_b >= 0 ? a.v_scales[ph_b] : 0.0f;
      for (int i = 0; i < 32 && g0 + i < n_local; ++i) {
        const long long g = g0 + i;
        const int rc = __shfl_sync(0xffffffffu, rc_a, i);
        const float sk = __shfl_sync(0xffffffffu, sk_a, i);
        const float sv = __shfl_sync(0xffffffffu, sv_a, i);
        const int s = (int)(g % kStages);
        if (g >= kStages && !mbar_wait(smem_u32(&ctl->empty[s]), (uint32_t)((g / kStages - 1) & 1), abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          ctl->sk[s] = sk;
          ctl->sv[s] = sv;
          const uint32_t bar = smem_u32(&ctl->full[s]);
          mbar_arrive_expect_tx(bar, kStageBytes);
          tma_load_2d(stages + s * kStageBytes, &map_k, 0, rc, bar);
          tma_load_2d(stages + s * kStageBytes + 8192, &map_v, 0, rc, bar);
        }
        __syncwarp();
        issued = g + 1;
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
      for (long long g = max(0LL, issued - kStages); g < issued; ++g) {
        int dummy = 0;
        mbar_wait(smem_u32(&ctl->full[g % kStages]), (uint32_t)((g / kStages) & 1), &dummy, 400000000LL);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------
    // MMA issuer
    // ------------------------------------------------------------------
    PageIter it;
    it.seek(start, ctl->pref, a.B, a.Hkv);
    uint32_t q_phase = 0;
    bool prev_first = false, ok = true;
    long long last_committed = -1;
    auto issue_pv = [&](long long h, bool first_of_seg) -> bool {
      const int jh = (int)(h & 1), sh = (int)(h % kStages);
      if (!mbar_wait(smem_u32(&ctl->p_full[jh]), (uint32_t)((h >> 1) & 1), abort_flag)) return false;
      fence_after_sync();
      if (lane == 0) {
        const uint32_t vtile = stages + sh * kStageBytes + 8192;
        const uint32_t pcol = tmem + kColP + 32 * jh;
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int k = 0; k < 2; ++k)
            mma_e4m3_ts(tmem + kColO, pcol + 16 * half + 8 * k, sdesc_sw128(vtile + 4096 * k, 1024, 1024), kIdescPV,
                        (first_of_seg && half == 0 && k == 0) ? 0u : 1u);
        mma_commit(smem_u32(&ctl->o_done[jh]));
        mma_commit(smem_u32(&ctl->empty[sh]));
      }
      __syncwarp();
      return true;
    };
    for (long long g = 0; g < n_local && ok; ++g) {
      const bool first = (g == 0) || it.p == 0;
      const int s = (int)(g % kStages), j = (int)(g & 1);
      if (first && g > 0) {
        if (!(ok = issue_pv(g - 1, prev_first))) break;
      }
      if (first) {
        if (!(ok = mbar_wait(smem_u32(&ctl->q_full), q_phase, abort_flag))) break;
        q_phase ^= 1u;
      }
      if (!(ok = mbar_wait(smem_u32(&ctl->full[s]), (uint32_t)((g / kStages) & 1), abort_flag))) break;
      if (g >= 2 && !(ok = mbar_wait(smem_u32(&ctl->p_full[j]), (uint32_t)(((g - 2) >> 1) & 1), abort_flag))) break;
      fence_after_sync();
      if (lane == 0) {
        const uint32_t ktile = stages + s * kStageBytes;
        const uint32_t scol = tmem + kColS + 64 * j;
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_e4m3_ts(scol, tmem + kColQ + 32 * half + 8 * k, sdesc_sw128(ktile + 32 * k, 1024, 1024), kIdescQK,
                        (half == 0 && k == 0) ? 0u : 1u);
        mma_commit(smem_u32(&ctl->s_full[j]));
      }
      __syncwarp();
      if (!first && g > 0) {
        if (!(ok = issue_pv(g - 1, prev_first))) break;
      }
      prev_first = first;
      last_committed = g;
      it.next(ctl->pref, a.B, a.Hkv);
    }
    if (ok && n_local > 0) ok = issue_pv(n_local - 1, prev_first);
    if (!ok) {
      fail(ctl, a.status);
      // let the tensor core finish what this thread issued before tensor memory is freed
      if (last_committed >= 0) {
        int dummy = 0;
        mbar_wait(smem_u32(&ctl->s_full[last_committed & 1]), (uint32_t)((last_committed >> 1) & 1), &dummy,
                  400000000LL);
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------------
    // softmax warps: thread = query row = TMEM lane
    // ------------------------------------------------------------------
    const int row = threadIdx.x;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const bool warp_active = warp * 32 < a.R;
    const bool row_valid = row < a.R;
    const int i_row = row_valid ? row / a.G : a.W - 1;
    PageIter it;
    it.seek(start, ctl->pref, a.B, a.Hkv);
    long long g = 0;
    bool ok = true;
    while (g < n_local && ok) {
      // ---- segment setup ----
      const int b = it.b, hk = it.hk, nb = it.nb, p0 = it.p;
      const int L = ctl->lens[b];
      const long long seg_len = min((long long)(nb - p0), n_local - g);
      const bool whole_unit = (p0 == 0) && seg_len == nb;
      const int u = b * a.Hkv + hk;
      const int h = hk * a.G + (row_valid ? row % a.G : 0);
      float row_scale = 0.0f;
      if (warp_active) {
        uint32_t hi[32], lo[32];
        int e = 0;
        if (row_valid) {
          const uint4* qp = reinterpret_cast<const uint4*>(a.q + (((size_t)b * a.W + i_row) * a.Hq + h) * kHeadDim);
          uint4 qv[16];
          float amax = 0.0f;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            qv[k] = qp[k];
            const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
            for (int t = 0; t < 4; ++t) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[t])), fabsf(bf16_hi(w[t]))));
          }
          if (amax > 0.0f) {
            int k2;
            frexpf(amax, &k2);  // amax < 2^k2
            e = max(-100, min(100, 8 - k2));
          }
          const float up = ldexpf(1.0f, e);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
            uint32_t hw[2], lw[2];
#pragma unroll
            for (int t = 0; t < 4; t += 2) {
              const float x0 = bf16_lo(w[t]) * up, x1 = bf16_hi(w[t]) * up;
              const float x2 = bf16_lo(w[t + 1]) * up, x3 = bf16_hi(w[t + 1]) * up;
              const uint32_t h01 = e4m3x2_from_f32(x0, x1), h23 = e4m3x2_from_f32(x2, x3);
              const float2 d01 = f32x2_from_e4m3x2(h01), d23 = f32x2_from_e4m3x2(h23);
              const uint32_t l01 = e4m3x2_from_f32(x0 - d01.x, x1 - d01.y), l23 = e4m3x2_from_f32(x2 - d23.x, x3 - d23.y);
              hw[t >> 1] = h01 | (h23 << 16);
              lw[t >> 1] = l01 | (l23 << 16);
            }
            hi[2 * k] = hw[0];
            hi[2 * k + 1] = hw[1];
            lo[2 * k] = lw[0];
            lo[2 * k + 1] = lw[1];
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) hi[k] = lo[k] = 0u;
        }
        row_scale = ldexpf(a.sm_scale_log2, -e);
        tmem_st32(lane_base + kColQ, hi);
        tmem_st32(lane_base + kColQ + 32, lo);
        tmem_wait_st();
      }
      fence_before_sync();
      mbar_arrive(smem_u32(&ctl->q_full));

      float m = -INFINITY, l = 0.0f;
      const long long g_first = g;
      for (long long k = 0; k < seg_len; ++k, ++g) {
        const int p = p0 + (int)k;
        const int s = (int)(g % kStages), j = (int)(g & 1);
        if (!(ok = mbar_wait(smem_u32(&ctl->s_full[j]), (uint32_t)((g >> 1) & 1), abort_flag))) break;
        fence_after_sync();
        if (warp_active) {
          // full[s] completed before the MMA that filled S_j was issued: the
          // page's scales written by the producer are visible through it
          if (!(ok = mbar_wait(smem_u32(&ctl->full[s]), (uint32_t)((g / kStages) & 1), abort_flag))) break;
          const float sk = ctl->sk[s], sv = ctl->sv[s];
          uint32_t x0[32], x1[32];
          tmem_ld32(lane_base + kColS + 64 * j, x0);
          tmem_ld32(lane_base + kColS + 64 * j + 32, x1);
          tmem_wait_ld();
          const float kscale = sk * row_scale;
          const float shift = sv > 0.0f ? log2f(sv) : 0.0f;
          const float inv_f = sv > 0.0f ? 1.0f / sv : 1.0f;
          const int kbase = p * kPage;
          const int lim = L + i_row;  // last visible key position of this row
          const bool partial = kbase + kPage - 1 > lim;
          float smax = -INFINITY;
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const bool v0 = !partial || kbase + t <= lim, v1 = !partial || kbase + 32 + t <= lim;
            if (v0) smax = fmaxf(smax, __uint_as_float(x0[t]));
            if (v1) smax = fmaxf(smax, __uint_as_float(x1[t]));
          }
          const float xmax = smax == -INFINITY ? -INFINITY : fmaf(smax, kscale, shift);
          const float m_new = fmaxf(m, xmax);
          const bool grow = m != -INFINITY && m_new > m;
          if (__any_sync(0xffffffffu, grow)) {
            // O must hold every earlier page of this segment before it is rescaled
            if (!(ok = mbar_wait(smem_u32(&ctl->o_done[(g - 1) & 1]), (uint32_t)(((g - 1) >> 1) & 1), abort_flag)))
              break;
            fence_after_sync();
            const float alpha = grow ? fast_exp2(m - m_new) : 1.0f;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
              uint32_t o[32];
              tmem_ld32(lane_base + kColO + 32 * cc, o);
              tmem_wait_ld();
#pragma unroll
              for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
              tmem_st32(lane_base + kColO + 32 * cc, o);
            }
            tmem_wait_st();
            l *= alpha;
          }
          m = m_new;
          const float mu = m == -INFINITY ? 0.0f : m;
          const float bias = shift - mu + 8.0f;  // weights scaled by 2^8 for the E4M3 range
          float sum = 0.0f;
          uint32_t phi[16], plo[16];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t* xs = half ? x1 : x0;
#pragma unroll
            for (int t = 0; t < 32; t += 4) {
              float w[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const bool vis = !partial || kbase + 32 * half + t + q <= lim;
                w[q] = vis ? fast_exp2(fmaf(__uint_as_float(xs[t + q]), kscale, bias)) : 0.0f;
                sum += w[q];
              }
              const uint32_t h01 = pack_f16x2(w[0], w[1]), h23 = pack_f16x2(w[2], w[3]);
              const uint32_t e01 = e4m3x2_from_f16x2(h01), e23 = e4m3x2_from_f16x2(h23);
              const uint32_t f01 = e4m3x2_from_f16x2(hsub2_u32(h01, f16x2_from_e4m3x2(e01)));
              const uint32_t f23 = e4m3x2_from_f16x2(hsub2_u32(h23, f16x2_from_e4m3x2(e23)));
              phi[(32 * half + t) >> 2] = e01 | (e23 << 16);
              plo[(32 * half + t) >> 2] = f01 | (f23 << 16);
            }
          }
          l += sum * (1.0f / 256.0f) * inv_f;
          // P buffer j is free once the PV of page g - 2 has completed
          if (g >= 2 && !(ok = mbar_wait(smem_u32(&ctl->o_done[j]), (uint32_t)(((g - 2) >> 1) & 1), abort_flag)))
            break;
          tmem_st16(lane_base + kColP + 32 * j, phi);
          tmem_st16(lane_base + kColP + 32 * j + 16, plo);
          tmem_wait_st();
        }
        fence_before_sync();
        mbar_arrive(smem_u32(&ctl->p_full[j]));
        it.next(ctl->pref, a.B, a.Hkv);
      }
      if (!ok) break;
      // ---- segment epilogue: every PV of the segment must have completed ----
      const long long g_last = g - 1;
      if (!(ok = mbar_wait(smem_u32(&ctl->o_done[g_last & 1]), (uint32_t)((g_last >> 1) & 1), abort_flag))) break;
      fence_after_sync();
      (void)g_first;
      if (warp_active) {
        const size_t slot_row = ((size_t)(u + c)) * a.R + row;
        const float inv = (row_valid && l > 0.0f) ? 1.0f / (256.0f * l) : 0.0f;
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
            for (int t = 0; t < 32; t += 8) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(o[t]) * inv, __uint_as_float(o[t + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(o[t + 2]) * inv, __uint_as_float(o[t + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(o[t + 4]) * inv, __uint_as_float(o[t + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(o[t + 6]) * inv, __uint_as_float(o[t + 7]) * inv);
              *reinterpret_cast<uint4*>(orow + 32 * cc + t) = v;
            }
          } else if (prow) {
#pragma unroll
            for (int t = 0; t < 32; t += 4) {
              *reinterpret_cast<float4*>(prow + 32 * cc + t) =
                  make_float4(__uint_as_float(o[t]) * (1.0f / 256.0f), __uint_as_float(o[t + 1]) * (1.0f / 256.0f),
                              __uint_as_float(o[t + 2]) * (1.0f / 256.0f), __uint_as_float(o[t + 3]) * (1.0f / 256.0f));
            }
          }
        }
      }
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

// grid: units; block 128.  Zeroes the rows of invalid lanes (and flags them);
// merges the partials of units that span several CTAs.
__global__ void __launch_bounds__(128) verify_merge_tc_kernel(TcArgs a, int C) {
  const int u = blockIdx.x;
  const int b = u / a.Hkv, hk = u % a.Hkv;
  __shared__ int s_bad;
  __shared__ long long s_sum[4];
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
  // pages before this lane and in total (same rule as the split kernel)
  long long before = 0, all = 0;
  for (int bb = threadIdx.x; bb < a.B; bb += blockDim.x) {
    const int Lb = a.seq_lens[bb];
    const bool ok = Lb >= 0 && Lb <= a.max_context && (long long)Lb + a.W <= (long long)a.max_pages * kPage;
    const int n = ok ? (Lb + a.W + kPage - 1) / kPage : 0;
    all += n;
    if (bb < b) before += n;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    all += __shfl_xor_sync(0xffffffffu, all, o);
  }
  __shared__ long long s_all[4];
  if (lane == 0) {
    s_sum[warp] = before;
    s_all[warp] = all;
  }
  __syncthreads();
  const int bad = s_bad;
  if (bad && threadIdx.x == 0 && hk == 0) raise_status(a.status, bad);
  if (bad) {
    for (int r = warp; r < a.R; r += 4) {
      const int i = r / a.G, h = hk * a.G + r % a.G;
      uint16_t* dst = a.out + (((size_t)b * a.W + i) * a.Hq + h) * kHeadDim + lane * 4;
      *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
    }
    return;
  }
  before = s_sum[0] + s_sum[1] + s_sum[2] + s_sum[3];
  all = s_all[0] + s_all[1] + s_all[2] + s_all[3];
  const long long total = (long long)a.Hkv * all;
  const long long Pu = (long long)a.Hkv * before + (long long)hk * nb;
  auto locate = [&](long long x) {
    long long cc = x * C / total;
    while (cc + 1 < C && cta_start(cc + 1, C, total) <= x) ++cc;
    while (cc > 0 && cta_start(cc, C, total) > x) --cc;
    return cc;
  };
  const long long c_first = locate(Pu), c_last = locate(Pu + nb - 1);
  if (c_first == c_last) return;  // one segment: the split kernel wrote the rows
  for (int r = warp; r < a.R; r += 4) {
    float M = -INFINITY;
    for (long long cc = c_first; cc <= c_last; ++cc) {
      if (cta_start(cc, C, total) == cta_start(cc + 1, C, total)) continue;
      M = fmaxf(M, a.ws_ml[(size_t)(u + cc) * a.R + r].x);
    }
    float den = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (long long cc = c_first; cc <= c_last; ++cc) {
      if (cta_start(cc, C, total) == cta_start(cc + 1, C, total)) continue;
      const size_t slot_row = (size_t)(u + cc) * a.R + r;
      const float2 ml = a.ws_ml[slot_row];
      if (ml.x == -INFINITY) continue;
      const float w = exp2f(ml.x - M);
      den += w * ml.y;
      const float4 v = *reinterpret_cast<const float4*>(a.ws_o + slot_row * kHeadDim + lane * 4);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    }
    const float inv = 1.0f / den;
    const int i = r / a.G, h = hk * a.G + r % a.G;
    uint16_t* dst = a.out + (((size_t)b * a.W + i) * a.Hq + h) * kHeadDim + lane * 4;
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                pack_bf16x2(acc[2] * inv, acc[3] * inv));
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
  verify_merge_tc_kernel<<<args.B * args.Hkv, 128, 0, stream>>>(args, num_sms);
  return cudaGetLastError() == cudaSuccess ? SDVA_OK : SDVA_ERR_CUDA;
}

}  // namespace tc
}  // namespace sdva
