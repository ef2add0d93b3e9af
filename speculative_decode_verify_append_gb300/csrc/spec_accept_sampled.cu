// spec_accept_sampled.cu -- lossless stochastic acceptance of a verify window.
//
// DFlash2 keeps the draft model's real conditional distribution q (NInfer
// review, section "아키텍처 ③"), which is what an acceptance that preserves
// the target distribution needs: with p_i = softmax(logits row i), draft i
// is accepted when u_i * q_i(x_i) < p_i(x_i); at the first rejection a, one
// token is drawn from max(0, p_a - q_a) (normalised), and from p_d when every
// draft is accepted.  The uniforms are inputs; the draw is the inverse CDF in
// index order at u_sample * Z: the smallest k whose running sum exceeds it,
// else the last k of positive weight; a residual of zero mass falls back to
// p_a.
//
// Kernel 1 (row statistics): one cluster of up to 8 CTAs per logits row; each
// CTA reduces its slice to (running max, sum of exp) with 16-byte streaming
// loads, four in flight per thread and the next four requested into L2, the
// cluster combines the slices in rank
// order through distributed shared memory, and rank 0 stores (M, S) of the
// row in the workspace.  All rows are reduced at once over the whole GPU (the
// acceptance needs S of every row up to the first rejection).
// Kernel 2 (the draw, a programmatic dependent of kernel 1): up to 64 CTAs per
// lane.  Every CTA evaluates the ratio tests of the lane's drafts identically,
// so all agree on a.  Each CTA walks its slice of row a in tiles of 4 x 256
// consecutive logits (the loads of four tiles issued before the first is
// scanned), a block scan giving the running sum of the weights in index
// order, stores the slice's totals and counts itself in a per-lane counter
// (zeroed by kernel 1).  The lane's last CTA adds the totals in slice order,
// finds the slice whose running range holds the target, walks that slice
// again with the same arithmetic and stops inside the tile and the 4-logit
// group where the running sum crosses it.  No CTA waits for another.  (One
// cluster of 8 CTAs per lane, the first design, spent most of its time
// pulling a whole row through 8 SMs; a separate kernel for the walk to the
// crossing cost one more dependent launch.)
#include <cooperative_groups.h>

#include "sdva_common.cuh"

namespace cg = cooperative_groups;

namespace sdva {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxCluster = 8;
constexpr int kTile = 4 * kThreads;  // logits per tile of the walk
constexpr int kSampleSlice = 4096;   // minimum logits per CTA of the draw
constexpr int kMaxSlices = 64;       // CTAs per lane of the draw
constexpr float kLog2e = 1.4426950408889634f;

struct Stat {
  float m, s;  // running max, sum of exp(x - m)
};

__device__ __forceinline__ Stat combine(Stat a, Stat b) {
  if (a.s == 0.0f) return b;
  if (b.s == 0.0f) return a;
  const float m = fmaxf(a.m, b.m);
  return {m, a.s * fast_exp2((a.m - m) * kLog2e) + b.s * fast_exp2((b.m - m) * kLog2e)};
}

__device__ __forceinline__ Stat add4(Stat st, float4 v) {
  const float m4 = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
  const float m = st.s == 0.0f ? m4 : fmaxf(st.m, m4);
  float s = st.s == 0.0f ? 0.0f : st.s * fast_exp2((st.m - m) * kLog2e);
  s += fast_exp2((v.x - m) * kLog2e) + fast_exp2((v.y - m) * kLog2e) + fast_exp2((v.z - m) * kLog2e) +
       fast_exp2((v.w - m) * kLog2e);
  return {m, s};
}

// four consecutive values starting at index i of x (i % 4 == 0 when kVec);
// entries at or past `end` read as `fill`
template <bool kVec>
__device__ __forceinline__ float4 load4(const float* x, int i, int end, float fill) {
  if (kVec && i + 3 < end) return __ldcs(reinterpret_cast<const float4*>(x + i));
  return make_float4(i < end ? x[i] : fill, i + 1 < end ? x[i + 1] : fill, i + 2 < end ? x[i + 2] : fill,
                     i + 3 < end ? x[i + 3] : fill);
}

// grid (parts, rows), cluster (parts, 1, 1); stats[row] = (M, S)
template <bool kVec>
__global__ void __launch_bounds__(kThreads) row_stats_kernel(const float* logits, int vocab, int chunk,
                                                            float2* stats, int* counters, int num_lanes) {
  cg::cluster_group cluster = cg::this_cluster();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the draw kernel's per-lane arrival counters start at zero
  if (blockIdx.x == 0 && threadIdx.x == 0 && (int)blockIdx.y < num_lanes) counters[blockIdx.y] = 0;
  __shared__ Stat s_w[kThreads / 32];
  __shared__ Stat c_st[kMaxCluster];  // in rank 0: one entry per CTA of the cluster
  const int part = blockIdx.x, row = blockIdx.y;
  const float* x = logits + (size_t)row * vocab;
  const int lo = part * chunk, hi = min(vocab, lo + chunk);
  Stat st = {0.0f, 0.0f};
  const float ninf = __int_as_float(0xff800000);
  // four 16-byte loads in flight per thread, folded in index order
  int i = lo + 4 * (int)threadIdx.x;
  for (; i + 12 * kThreads < hi; i += 16 * kThreads) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = load4<kVec>(x, i + 4 * kThreads * u, hi, ninf);
    // the next four requested into L2 while these are in flight
#pragma unroll
    for (int u = 4; u < 8; ++u)
      if (i + 4 * kThreads * u + 3 < hi) asm volatile("prefetch.global.L2 [%0];" ::"l"(x + i + 4 * kThreads * u));
#pragma unroll
    for (int u = 0; u < 4; ++u) st = add4(st, v[u]);
  }
  for (; i < hi; i += 4 * kThreads) st = add4(st, load4<kVec>(x, i, hi, ninf));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const Stat o = {__shfl_xor_sync(0xffffffffu, st.m, off), __shfl_xor_sync(0xffffffffu, st.s, off)};
    st = combine(st, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_w[warp] = st;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) st = combine(st, s_w[w]);
    *cluster.map_shared_rank(&c_st[part], 0) = st;
  }
  cluster.sync();
  if (part == 0 && threadIdx.x == 0) {
    Stat t = c_st[0];
    for (int p = 1; p < (int)gridDim.x; ++p) t = combine(t, c_st[p]);
    stats[row] = make_float2(t.m, t.s);
  }
  cluster.sync();  // rank 0's shared memory must outlive the other CTAs' stores
}

// Scan of v over the block in thread order: *incl and *excl are this
// thread's inclusive and exclusive sums, the return value the block's sum.
// Each thread's exclusive sum is bitwise its predecessor's inclusive sum and
// the block's sum is bitwise the last thread's inclusive sum, so the ranges
// (excl, incl] tile (0, total] without gaps.
__device__ __forceinline__ float block_scan(float v, float* s_part, float* incl, float* excl) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  const float prev = __shfl_up_sync(0xffffffffu, v, 1);
  if (lane == 31) s_part[warp] = v;
  __syncthreads();
  float before = 0.0f, all = 0.0f;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) before += s_part[w];
    all += s_part[w];
  }
  __syncthreads();  // s_part is reused by the next call
  *incl = before + v;
  *excl = lane > 0 ? before + prev : before;
  return all;
}

struct Row {
  const float* l;   // logits row
  const float* q;   // draft row (residual) or nullptr (draw from p)
  float m, inv_s;   // p(x) = exp(l[x] - m) * inv_s
};

__device__ __forceinline__ float weight(const Row& r, float lx, float qx) {
  const float p = fast_exp2((lx - r.m) * kLog2e) * r.inv_s;
  if (r.q == nullptr) return p;
  const float w = p - qx;
  return w > 0.0f ? w : 0.0f;
}

// Walk [lo, hi) in tiles of kTile logits, keeping the running sum of the
// weights in index order; each thread's loads for kGroup tiles are issued
// before the first of them is scanned.  search == false: returns the slice's
// total (.x), and with `both` also the total of p alone (.y, the same
// arithmetic as a walk with q == nullptr).  search == true: stops in the
// tile, the thread and the logit where the running sum first exceeds `target`
// and stores that index in *found; when it never does (the target sits
// within rounding of the slice's end), the last index of positive weight.
// Both modes do the same arithmetic, so a target below the first mode's total
// is always crossed.
constexpr int kGroup = 4;
template <bool kVec>
__device__ float2 walk(const Row& r, int lo, int hi, bool search, bool both, float target, float* s_part, int* s_found,
                       int* found) {
  float running = 0.0f, running_p = 0.0f;
  int last_pos = -1;
  bool done = false;
  const float ninf = __int_as_float(0xff800000);
  for (int gbase = lo; gbase < hi && !done; gbase += kGroup * kTile) {
    float4 l4[kGroup], q4[kGroup];
#pragma unroll
    for (int t = 0; t < kGroup; ++t) {
      const int i = gbase + t * kTile + 4 * (int)threadIdx.x;
      l4[t] = load4<kVec>(r.l, i, hi, ninf);
      q4[t] = r.q != nullptr ? load4<kVec>(r.q, i, hi, 0.0f) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int t = 0; t < kGroup; ++t) {
      const int base = gbase + t * kTile;
      if (base >= hi) break;  // uniform
      const int i = base + 4 * (int)threadIdx.x;
      const float w[4] = {weight(r, l4[t].x, q4[t].x), weight(r, l4[t].y, q4[t].y), weight(r, l4[t].z, q4[t].z),
                          weight(r, l4[t].w, q4[t].w)};
      const float ts = (w[0] + w[1]) + (w[2] + w[3]);
      float incl, excl;
      const float tile_total = block_scan(ts, s_part, &incl, &excl);
      if (both) {
        const Row rp{r.l, nullptr, r.m, r.inv_s};
        const float wp[4] = {weight(rp, l4[t].x, 0.f), weight(rp, l4[t].y, 0.f), weight(rp, l4[t].z, 0.f),
                             weight(rp, l4[t].w, 0.f)};
        float ip, ep;
        running_p += block_scan((wp[0] + wp[1]) + (wp[2] + wp[3]), s_part, &ip, &ep);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (w[j] > 0.0f) last_pos = i + j;
      if (search && running + tile_total > target) {
        // exactly one thread's range (running + excl, running + incl] holds the target
        if (running + excl <= target && running + incl > target) {
          float cum = excl;
          int k = -1, lastj = -1;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (w[j] > 0.0f) lastj = i + j;
            cum += w[j];
            if (k < 0 && running + cum > target) k = i + j;
          }
          *s_found = k >= 0 ? k : lastj;  // lastj: the 4-term sum rounded past the target
        }
        __syncthreads();
        done = true;
        break;
      }
      running += tile_total;
    }
  }
  if (search) {
    if (*s_found < 0) atomicMax(s_found, last_pos);
    __syncthreads();
    *found = *s_found;
  }
  return make_float2(running, both ? running_p : running);
}

// The lane's accept length a: every CTA evaluates the ratio tests with the
// same fp32 arithmetic, so all CTAs of all launches agree.
__device__ int accept_count(const float* logits, const float* draft_probs, int window, int vocab, int b,
                            const int32_t* drafts, const float* u_accept, const float2* stats, int32_t* status,
                            bool report, int* s_rej) {
  const int d = window - 1;
  if (threadIdx.x == 0) *s_rej = d;
  __syncthreads();
  if ((int)threadIdx.x < d) {
    const int i = threadIdx.x, x = drafts[(size_t)b * d + i];
    bool accept = false;
    if (x < 0 || x >= vocab) {
      if (report) raise_status(status, SDVA_STATUS_BAD_DRAFT);
    } else {
      const float2 st = stats[(size_t)b * window + i];
      const float lx = logits[((size_t)b * window + i) * vocab + x];
      const float px = fast_exp2((lx - st.x) * kLog2e) / st.y;
      const float qx = draft_probs[((size_t)b * d + i) * vocab + x];
      accept = u_accept[(size_t)b * d + i] * qx < px;
    }
    if (!accept) atomicMin(s_rej, i);
  }
  __syncthreads();
  return *s_rej;
}

__device__ __forceinline__ Row draw_row(const float* logits, const float* draft_probs, int window, int vocab, int b,
                                        int a, const float2* stats) {
  const int d = window - 1;
  const float2 st = stats[(size_t)b * window + a];
  Row r;
  r.l = logits + ((size_t)b * window + a) * vocab;
  r.q = a < d ? draft_probs + ((size_t)b * d + a) * vocab : nullptr;
  r.m = st.x;
  r.inv_s = 1.0f / st.y;
  return r;
}

struct SampleArgs {
  const float* logits;
  const float* draft_probs;
  const int32_t* drafts;
  const float* u_accept;
  const float* u_sample;
  const float2* stats;  // [B][W]: (M, S) of every row
  float2* totals;       // [B][kMaxSlices]: per slice, (residual weight, p weight) of the drawn row
  int* counters;        // [B]: CTAs of the lane that have stored their slice totals
  int32_t* accept_len;
  int32_t* out_tokens;
  int32_t* seq_lens;
  int32_t* status;
  int window, vocab, chunk;
};

// grid (slices, lanes); programmatic dependent of the statistics kernel.
// Each CTA finds a and stores its slice's total weight of the drawn row (and
// the total of p_a, for a residual of zero mass); the lane's last CTA to count
// itself draws the token, writes the tokens and a, and commits seq_lens.
template <bool kVec>
__global__ void __launch_bounds__(kThreads) sample_kernel(SampleArgs g) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float s_part[kThreads / 32];
  __shared__ int s_rej;
  const int part = blockIdx.x, b = blockIdx.y;
  const int a = accept_count(g.logits, g.draft_probs, g.window, g.vocab, b, g.drafts, g.u_accept, g.stats,
                             g.status, part == 0, &s_rej);
  Row r = draw_row(g.logits, g.draft_probs, g.window, g.vocab, b, a, g.stats);
  const int lo = part * g.chunk, hi = min(g.vocab, lo + g.chunk);
  const float2 tot = walk<kVec>(r, lo, hi, false, r.q != nullptr, 0.0f, s_part, nullptr, nullptr);
  __shared__ int s_last, s_found;
  __shared__ float2 s_tot[kMaxSlices];
  if (threadIdx.x == 0) {
    g.totals[(size_t)b * kMaxSlices + part] = tot;
    __threadfence();
    s_last = atomicAdd(&g.counters[b], 1) == (int)gridDim.x - 1;
    s_found = -1;
  }
  __syncthreads();
  if (!s_last) return;
  // the lane's last CTA: every slice total is stored; find the slice whose
  // running range holds u_sample * Z and walk it to the crossing
  __threadfence();
  const int parts = gridDim.x;
  if ((int)threadIdx.x < parts) s_tot[threadIdx.x] = __ldcg(&g.totals[(size_t)b * kMaxSlices + threadIdx.x]);
  __syncthreads();
  float z = 0.0f;
  for (int p = 0; p < parts; ++p) z += s_tot[p].x;
  const bool use_p = !(z > 0.0f) && r.q != nullptr;  // a residual of zero mass falls back to p_a
  if (use_p) {
    r.q = nullptr;
    z = 0.0f;
    for (int p = 0; p < parts; ++p) z += s_tot[p].y;
  }
  const float target = g.u_sample[b] * z;
  int owner = -1, last = -1;
  float before = 0.0f, cum = 0.0f;
  for (int p = 0; p < parts; ++p) {
    const float t = use_p ? s_tot[p].y : s_tot[p].x;
    if (t > 0.0f) last = p;
    if (owner < 0 && cum + t > target) {
      owner = p;
      before = cum;
    }
    cum += t;
  }
  // no crossing (the target sits within rounding of the row's end): the last
  // slice with weight takes its last index of positive weight
  const bool crossing = owner >= 0;
  if (!crossing) owner = last;
  int32_t* tok = g.out_tokens + (size_t)b * g.window;
  int k = 0;  // no positive weight in the row (only non-finite logits give this)
  if (owner >= 0) {
    const int olo = owner * g.chunk, ohi = min(g.vocab, olo + g.chunk);
    walk<kVec>(r, olo, ohi, true, false, crossing ? target - before : __int_as_float(0x7f800000), s_part, &s_found, &k);
  }
  if (threadIdx.x == 0) {
    const int d = g.window - 1;
    for (int i = 0; i < g.window; ++i) tok[i] = i == a ? k : (i < a ? g.drafts[(size_t)b * d + i] : -1);
    g.accept_len[b] = a;
    if (g.seq_lens != nullptr) g.seq_lens[b] += 1 + a;
  }
}

bool vectorizable(const float* p, int vocab) {
  return (vocab & 3) == 0 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace
}  // namespace sdva

using namespace sdva;

namespace {
size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }
}  // namespace

// per-row statistics [B][W], per-slice totals of the drawn rows [B][kMaxSlices],
// then the draw's per-lane counters [B]
extern "C" size_t spec_accept_sampled_workspace_size(int num_lanes, int window) {
  if (num_lanes <= 0 || window <= 0) return 0;
  return align256((size_t)num_lanes * window * sizeof(float2)) +
         align256((size_t)num_lanes * kMaxSlices * sizeof(float2)) + align256((size_t)num_lanes * sizeof(int));
}

extern "C" int spec_accept_sampled(const float* logits, const float* draft_probs, int num_lanes, int window,
                                   int vocab, const int32_t* drafts, const float* u_accept, const float* u_sample,
                                   int32_t* accept_len, int32_t* out_tokens, int32_t* seq_lens_inout,
                                   void* workspace, size_t workspace_bytes, int32_t* status, sdva_stream_t stream) {
  if (logits == nullptr || u_sample == nullptr || accept_len == nullptr || out_tokens == nullptr)
    return SDVA_ERR_INVALID;
  if (num_lanes <= 0 || window <= 0 || vocab <= 0) return SDVA_ERR_INVALID;
  if (window > 1 && (draft_probs == nullptr || drafts == nullptr || u_accept == nullptr)) return SDVA_ERR_INVALID;
  if (window > kMaxWindow) return SDVA_ERR_UNSUPPORTED;
  const long long rows = (long long)num_lanes * window;
  if (rows > 65535) return SDVA_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < spec_accept_sampled_workspace_size(num_lanes, window) ||
      (reinterpret_cast<uintptr_t>(workspace) & 7u))
    return SDVA_ERR_WORKSPACE;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDVA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float2* stats = static_cast<float2*>(workspace);
  int* counters = reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                         align256((size_t)num_lanes * window * sizeof(float2)) +
                                         align256((size_t)num_lanes * kMaxSlices * sizeof(float2)));
  const bool vec = vectorizable(logits, vocab) && (window == 1 || vectorizable(draft_probs, vocab));
  {
    // CTAs per row: enough to cover every SM about four times, at most one portable cluster
    int parts = 1;
    while (parts < kMaxCluster && rows * parts < 4LL * sms) parts *= 2;
    const int chunk = (((vocab + parts - 1) / parts) + 3) & ~3;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(parts, (unsigned)rows, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = parts;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const auto kernel = vec ? row_stats_kernel<true> : row_stats_kernel<false>;
    if (cudaLaunchKernelEx(&cfg, kernel, logits, vocab, chunk, stats, counters, num_lanes) != cudaSuccess)
      return SDVA_ERR_CUDA;
  }
  SampleArgs g;
  g.logits = logits;
  g.draft_probs = draft_probs;
  g.drafts = drafts;
  g.u_accept = u_accept;
  g.u_sample = u_sample;
  g.stats = stats;
  g.totals = reinterpret_cast<float2*>(static_cast<char*>(workspace) +
                                       align256((size_t)num_lanes * window * sizeof(float2)));
  g.counters = counters;
  g.accept_len = accept_len;
  g.out_tokens = out_tokens;
  g.seq_lens = seq_lens_inout;
  g.status = status;
  g.window = window;
  g.vocab = vocab;
  const int slices = min(kMaxSlices, max(1, (vocab + kSampleSlice - 1) / kSampleSlice));
  g.chunk = (((vocab + slices - 1) / slices) + 3) & ~3;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(slices, (unsigned)num_lanes, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const auto kernel = vec ? sample_kernel<true> : sample_kernel<false>;
    if (cudaLaunchKernelEx(&cfg, kernel, g) != cudaSuccess) return SDVA_ERR_CUDA;
  }
  return SDVA_OK;
}
