// spec_accept.cu -- greedy acceptance of a verify window.
//
// The main model's argmax at window position i is compared with draft i;
// the accepted prefix is the leading run of agreements and the bonus token is
// the argmax at the first disagreement (Baseten talk summary, section
// "추측 디코드"; the commit of the new length follows the NInfer review,
// section "아키텍처 ①": state changes only once the model accepts the commit).
//
// Kernel 1 (argmax): one thread-block cluster of up to 8 CTAs per logits
// row; each CTA scans a contiguous slice of the row with 16-byte streaming
// loads, four in flight per thread and the next four requested into L2
// (32 registers, so eight 256-thread CTAs fit
// on an SM and the grid of the multi-row case is a single wave), keeps its
// best with one greater-than test per element (exact, since a thread meets
// its elements in index order; a thread that met nothing above -inf rescans
// them in the full order), reduces (value, index) in shared memory,
// and stores it into CTA rank 0's shared memory through distributed shared
// memory; rank 0 writes the row's argmax.  No global scratch.  Ties go to the
// lowest index, NaN never wins, an all-NaN row gives 0.
// Kernel 2 (finalize, one warp per lane): compares the drafts with the
// argmaxes, writes the accept length and optionally commits seq_lens += 1 + a.
// It is launched as a programmatic dependent of kernel 1 so its launch
// overlaps kernel 1's tail; it waits for kernel 1's results before reading.
//
// Lazy form (spec_accept_lazy): the accepted prefix ends at the first
// disagreement, so the rows after it decide nothing, and each lane may carry
// its own draft count d_b (at most window - 1).  Two ways to the same result:
//  - walk (many lanes): one cluster of up to 8 CTAs per lane walks the lane's
//    rows in order: each CTA reduces its slice of row i, sends its partial to
//    every CTA of the cluster through distributed shared memory, and after
//    one cluster barrier every CTA holds the same argmax and takes the same
//    decision (stop, or go on to row i + 1).  A lane reads rows 0 .. a, and
//    row a + 1 at most into L2.
//  - parallel (few lanes): kernel 1 reduces rows 0 .. d_b of every lane at
//    once and a finalize kernel takes the accept length.  A row is a serial
//    step of the walk and one SM pulls only some tens of GB/s, so a walk
//    over 8 SMs per lane costs a few microseconds per row; until the lanes
//    fill the GPU, reading the rows a lane may need all at once is faster.
#include <cooperative_groups.h>

#include "sdva_common.cuh"
#include "sdva_internal.cuh"

namespace cg = cooperative_groups;

namespace sdva {
namespace {

constexpr int kArgmaxThreads = 256;
constexpr int kMaxRowCluster = 8;
constexpr int kWalkThreads = 256;
constexpr int kWalkLoads = 8;      // 16-byte loads in flight per thread
constexpr int kWalkSlice = 4096;   // minimum logits per CTA of a walking cluster
// Below this many lanes the walk's serial chain of rows (one row per cluster
// barrier, a row split over at most 8 SMs) is slower than reducing every row
// a lane may need at once over the whole GPU.  Measured at 151,936 logits per
// row, 16 positions and drafts agreeing with probability 0.7: the walk takes
// 1.12x the parallel pass at 32 lanes, 0.95x at 48, 0.74x at 64, 0.61x at 128.
constexpr int kWalkMinLanes = SDVA_LAZY_WALK_MIN_LANES;

// true if candidate (v, i) beats the current best (bv, bi)
__device__ __forceinline__ bool beats(float v, int i, float bv, int bi) {
  const bool vn = isnan(v), bn = isnan(bv);
  if (vn != bn) return bn;  // a number beats NaN
  if (!vn && v != bv) return v > bv;
  return i < bi;  // equal values (+0 == -0) or both NaN: lower index
}

__device__ __forceinline__ void take(float v, int i, float& bv, int& bi) {
  if (beats(v, i, bv, bi)) {
    bv = v;
    bi = i;
  }
}
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void take4(const float4 v, int i, float& bv, int& bi) {
  take(v.x, i, bv, bi);
  take(v.y, i + 1, bv, bi);
  take(v.z, i + 2, bv, bi);
  take(v.w, i + 3, bv, bi);
}

// One thread meets its elements in increasing index order.  Once its best
// holds a number above -inf, "v > best" alone keeps the order of take (an
// equal value comes later and loses, NaN compares false) at a third of the
// instructions.  Scans start from (-inf, none) in that form; a thread that met
// nothing above -inf (no element, or only -inf and NaN) scans its elements
// again in the exact form.
__device__ __forceinline__ void take_gt(float v, int i, float& bv, int& bi) {
  if (v > bv) {
    bv = v;
    bi = i;
  }
}
template <bool kExact>
__device__ __forceinline__ void take4_as(const float4 v, int i, float& bv, int& bi) {
  if constexpr (kExact) {
    take4(v, i, bv, bi);
  } else {
    take_gt(v.x, i, bv, bi);
    take_gt(v.y, i + 1, bv, bi);
    take_gt(v.z, i + 2, bv, bi);
    take_gt(v.w, i + 3, bv, bi);
  }
}
constexpr int kNone = 0x7fffffff;
__device__ __forceinline__ float nan_f() { return __int_as_float(0x7fffffff); }

// float4 k, k + step, ... below kend of x4 (element index 4 k), kLoads
// 16-byte streaming loads in flight
template <bool kExact, int kLoads>
__device__ __forceinline__ void scan_vec(const float4* x4, int k, int kend, int step, float& bv, int& bi) {
  for (; k + (kLoads - 1) * step < kend; k += kLoads * step) {
    float4 v[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) v[u] = __ldcs(x4 + k + u * step);
    // the next group's lines requested into L2 while this one is in flight
#pragma unroll
    for (int u = 0; u < kLoads; ++u)
      if (k + (kLoads + u) * step < kend) asm volatile("prefetch.global.L2 [%0];" ::"l"(x4 + k + (kLoads + u) * step));
#pragma unroll
    for (int u = 0; u < kLoads; ++u) take4_as<kExact>(v[u], 4 * (k + u * step), bv, bi);
  }
  for (; k < kend; k += step) take4_as<kExact>(__ldcs(x4 + k), 4 * k, bv, bi);
}
// the argmax of one thread's elements x[k], x[k + step], ... below end, in
// the order of take
template <int kLoads>
__device__ __forceinline__ void thread_argmax_vec(const float4* x4, int k, int kend, int step, float& bv, int& bi) {
  bv = -INFINITY;
  bi = kNone;
  scan_vec<false, kLoads>(x4, k, kend, step, bv, bi);
  if (bi == kNone) {
    bv = nan_f();
    scan_vec<true, kLoads>(x4, k, kend, step, bv, bi);
  }
}
__device__ __forceinline__ void thread_argmax(const float* x, int k, int end, int step, float& bv, int& bi) {
  bv = -INFINITY;
  bi = kNone;
  for (int j = k; j < end; j += step) take_gt(x[j], j, bv, bi);
  if (bi == kNone) {
    bv = nan_f();
    for (int j = k; j < end; j += step) take(x[j], j, bv, bi);
  }
}

// grid (parts, rows), cluster (parts, 1, 1).  kVec: vocab % 4 == 0 and logits
// is 16-byte aligned, so every row starts on a 16-byte boundary.
// num_drafts (lazy form, nullable): rows past a lane's count, and every row of
// a lane whose count is invalid, are skipped (by the whole cluster of the row).
template <bool kVec>
__global__ void __launch_bounds__(kArgmaxThreads, 8) argmax_rows_kernel(const float* logits, int vocab, int chunk,
                                                                    const int32_t* num_drafts, int window,
                                                                    int32_t* out_tokens) {
  cg::cluster_group cluster = cg::this_cluster();
  // the finalize kernel may be scheduled now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int part = blockIdx.x, row = blockIdx.y;
  if (num_drafts != nullptr) {
    const int lane_b = row / window, i = row - lane_b * window, d = num_drafts[lane_b];
    if (d < 0 || d >= window || i > d) return;
  }
  const float* x = logits + (size_t)row * vocab;
  const int lo = part * chunk, hi = min(vocab, lo + chunk);
  float bv;
  int bi;
  if constexpr (kVec) {
    // chunk is a multiple of 4: every slice starts on a 16-byte boundary
    thread_argmax_vec<4>(reinterpret_cast<const float4*>(x), lo / 4 + threadIdx.x, hi / 4, blockDim.x, bv, bi);
  } else {
    thread_argmax(x, lo + threadIdx.x, hi, blockDim.x, bv, bi);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    take(ov, oi, bv, bi);
  }
  __shared__ float s_v[kArgmaxThreads / 32];
  __shared__ int s_i[kArgmaxThreads / 32];
  __shared__ float c_v[kMaxRowCluster];  // in CTA rank 0: one entry per CTA of the cluster
  __shared__ int c_i[kMaxRowCluster];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_v[warp] = bv;
    s_i[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) take(s_v[w], s_i[w], bv, bi);
    *cluster.map_shared_rank(&c_v[part], 0) = bv;
    *cluster.map_shared_rank(&c_i[part], 0) = bi;
  }
  cluster.sync();
  if (cluster.block_rank() == 0 && threadIdx.x == 0) {
    float v = __int_as_float(0x7fffffff);
    int id = 0x7fffffff;
    for (int p = 0; p < (int)gridDim.x; ++p) take(c_v[p], c_i[p], v, id);
    out_tokens[row] = id == 0x7fffffff ? 0 : id;
  }
  cluster.sync();  // rank 0's shared memory must outlive the other CTAs' stores
  // Launched as a programmatic dependent (verify_step: after verify_attn's
  // merge), this grid must not finish before that kernel has: the commit of
  // the finalize kernel, which waits for this grid, rewrites seq_lens, which
  // the verify kernels read.  A no-op otherwise.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// one warp per lane
__global__ void __launch_bounds__(128) accept_finalize_kernel(int num_lanes, int window, int vocab,
                                                              const int32_t* drafts, const int32_t* out_tokens,
                                                              int32_t* accept_len, int32_t* seq_lens,
                                                              int32_t* status) {
  // programmatic dependent launch: kernel 1's results are visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (b >= num_lanes) return;
  const int d = window - 1;
  int draft = -1, tok = -1;
  if (lane < d) {
    draft = drafts[(size_t)b * d + lane];
    tok = out_tokens[(size_t)b * window + lane];
  }
  const bool bad = lane < d && (draft < 0 || draft >= vocab);
  const unsigned mismatch = __ballot_sync(0xffffffffu, lane < d && draft != tok);
  const unsigned any_bad = __ballot_sync(0xffffffffu, bad);
  if (lane == 0) {
    const int a = mismatch ? __ffs(mismatch) - 1 : d;
    accept_len[b] = a;
    if (seq_lens != nullptr) seq_lens[b] += 1 + a;
    if (any_bad) raise_status(status, SDVA_STATUS_BAD_DRAFT);
  }
}

// Walk (lazy form, many lanes).  grid (parts, lanes), cluster (parts, 1, 1):
// the cluster of lane b walks rows 0 .. a of the lane and stops at the first
// disagreement; while row i is reduced, the CTA's slice of row i + 1 is
// prefetched into L2 whenever row i + 1 may be needed.
template <bool kVec>
__global__ void __launch_bounds__(kWalkThreads, 4)
    accept_walk_kernel(const float* logits, int window, int vocab, int chunk, const int32_t* drafts,
                       const int32_t* num_drafts, int32_t* accept_len, int32_t* out_tokens, int32_t* seq_lens,
                       int32_t* status) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ float s_v[kWalkThreads / 32];
  __shared__ int s_i[kWalkThreads / 32];
  __shared__ float c_v[2][kMaxRowCluster];  // by row parity: one partial per CTA of the cluster
  __shared__ int c_i[2][kMaxRowCluster];
  __shared__ int s_draft[kMaxWindow];
  const int part = blockIdx.x, parts = gridDim.x, b = blockIdx.y;
  const int dmax = window - 1;
  const int d = num_drafts != nullptr ? num_drafts[b] : dmax;
  const bool lead = part == 0 && threadIdx.x == 0;
  int32_t* tok = out_tokens + (size_t)b * window;
  if (d < 0 || d > dmax) {
    // every CTA of the cluster reads the same count and leaves before any exchange
    if (lead) {
      accept_len[b] = 0;
      for (int i = 0; i < window; ++i) tok[i] = -1;
      raise_status(status, SDVA_STATUS_BAD_COUNT);
    }
    return;
  }
  if ((int)threadIdx.x < d) {
    const int t = drafts[(size_t)b * dmax + threadIdx.x];
    s_draft[threadIdx.x] = t;
    if (part == 0 && (t < 0 || t >= vocab)) raise_status(status, SDVA_STATUS_BAD_DRAFT);
  }
  __syncthreads();
  const int lo = part * chunk, hi = min(vocab, lo + chunk);
  const float* rows = logits + (size_t)b * window * vocab;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int i = 0;
  for (;; ++i) {
    const float* x = rows + (size_t)i * vocab;
    float bv;
    int bi;
    if constexpr (kVec) {
      // row i + 1 is needed only if draft i agrees: start its fetch into L2 now
      if (threadIdx.x == 0 && i < d && hi > lo) prefetch_l2_bulk(x + vocab + lo, (uint32_t)(hi - lo) * 4u);
      thread_argmax_vec<kWalkLoads>(reinterpret_cast<const float4*>(x), (lo >> 2) + threadIdx.x, hi >> 2, kWalkThreads,
                                    bv, bi);
    } else {
      thread_argmax(x, lo + threadIdx.x, hi, kWalkThreads, bv, bi);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      take(ov, oi, bv, bi);
    }
    if (lane == 0) {
      s_v[warp] = bv;
      s_i[warp] = bi;
    }
    __syncthreads();
    if ((int)threadIdx.x < parts) {
      // thread r reduces the warps' partials and sends the CTA's to rank r
      float v = s_v[0];
      int id = s_i[0];
      for (int w = 1; w < kWalkThreads / 32; ++w) take(s_v[w], s_i[w], v, id);
      *cluster.map_shared_rank(&c_v[i & 1][part], threadIdx.x) = v;
      *cluster.map_shared_rank(&c_i[i & 1][part], threadIdx.x) = id;
    }
    // Every CTA's partials of row i are in place after this.  Row i + 2 reuses
    // the slot only after the next barrier, which every CTA reaches after
    // reading this row's partials.
    cluster.sync();
    float tv = __int_as_float(0x7fffffff);
    int ti = 0x7fffffff;
    for (int p = 0; p < parts; ++p) take(c_v[i & 1][p], c_i[i & 1][p], tv, ti);
    const int t = ti == 0x7fffffff ? 0 : ti;
    if (lead) tok[i] = t;
    // the same partials in the same order: every CTA takes the same branch
    if (i == d || s_draft[i] != t) break;
  }
  // no exchange follows the last barrier, so CTAs may leave in any order
  if (lead) {
    for (int j = i + 1; j < window; ++j) tok[j] = -1;
    accept_len[b] = i;
    if (seq_lens != nullptr) seq_lens[b] += 1 + i;
  }
}

// Lazy form, few lanes: the argmax kernel has reduced rows 0 .. d_b of every
// lane; one warp per lane takes the accept length, writes -1 after row a and
// optionally commits.  Programmatic dependent of the argmax kernel.
__global__ void __launch_bounds__(128) accept_lazy_finalize_kernel(int num_lanes, int window, int vocab,
                                                                   const int32_t* drafts, const int32_t* num_drafts,
                                                                   int32_t* out_tokens, int32_t* accept_len,
                                                                   int32_t* seq_lens, int32_t* status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (b >= num_lanes) return;
  const int dmax = window - 1;
  const int d = num_drafts != nullptr ? num_drafts[b] : dmax;
  int32_t* tok = out_tokens + (size_t)b * window;
  if (d < 0 || d > dmax) {
    if (lane < window) tok[lane] = -1;
    if (lane == 0) {
      accept_len[b] = 0;
      raise_status(status, SDVA_STATUS_BAD_COUNT);
    }
    return;
  }
  int draft = -1, t = -1;
  if (lane < d) {
    draft = drafts[(size_t)b * dmax + lane];
    t = tok[lane];
  }
  const unsigned mismatch = __ballot_sync(0xffffffffu, lane < d && draft != t);
  const unsigned any_bad = __ballot_sync(0xffffffffu, lane < d && (draft < 0 || draft >= vocab));
  const int a = mismatch ? __ffs(mismatch) - 1 : d;
  // each lane reads and writes only its own position
  if (lane > a && lane < window) tok[lane] = -1;
  if (lane == 0) {
    accept_len[b] = a;
    if (seq_lens != nullptr) seq_lens[b] += 1 + a;
    if (any_bad) raise_status(status, SDVA_STATUS_BAD_DRAFT);
  }
}

// Draft-tree acceptance, one warp per lane (lane i of the warp holds window
// slot i): the argmax kernel has left row i's argmax in path[b][i].  From the
// root, the walk moves to the lowest slot c whose parent is the current node
// and whose token is the current node's argmax; a = the nodes accepted, the
// bonus = the last node's argmax.  Programmatic dependent of the argmax kernel.
__global__ void __launch_bounds__(128) accept_tree_finalize_kernel(int num_lanes, int window, int vocab,
                                                                   const int32_t* tokens, const int32_t* parent,
                                                                   int32_t* path, int32_t* out_tokens,
                                                                   int32_t* accept_len, int32_t* seq_lens,
                                                                   int32_t* status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (b >= num_lanes) return;
  const bool in = lane < window;
  const size_t base = (size_t)b * window;
  const int am = in ? path[base + lane] : -1;
  const int par = in && lane > 0 ? parent[base + lane] : -1;
  const int tk = in && lane > 0 ? tokens[base + lane] : -1;
  const bool bad_parent = in && lane > 0 && (par < 0 || par >= lane);
  const bool bad_token = in && lane > 0 && (tk < 0 || tk >= vocab);
  const unsigned any_bad_parent = __ballot_sync(0xffffffffu, bad_parent);
  const unsigned any_bad_token = __ballot_sync(0xffffffffu, bad_token);
  if (any_bad_parent) {
    if (in) {
      path[base + lane] = -1;
      out_tokens[base + lane] = -1;
    }
    if (lane == 0) {
      accept_len[b] = 0;
      raise_status(status, SDVA_STATUS_BAD_TREE | (any_bad_token ? SDVA_STATUS_BAD_DRAFT : 0));
    }
    return;
  }
  int n = 0, a = 0, my_path = lane == 0 ? 0 : -1, my_tok = -1;
  for (int step = 0; step < window; ++step) {
    const int t = __shfl_sync(0xffffffffu, am, n);
    const unsigned next = __ballot_sync(0xffffffffu, in && lane > n && par == n && tk == t);
    if (next == 0u) {
      if (lane == a) my_tok = t;  // the bonus token
      break;
    }
    const int c = __ffs(next) - 1;  // the first child in slot order
    const int tc = __shfl_sync(0xffffffffu, tk, c);
    if (lane == a) my_tok = tc;  // the a-th accepted token
    ++a;
    if (lane == a) my_path = c;
    n = c;
  }
  if (in) {
    path[base + lane] = lane <= a ? my_path : -1;
    out_tokens[base + lane] = lane <= a ? my_tok : -1;
  }
  if (lane == 0) {
    accept_len[b] = a;
    if (seq_lens != nullptr) seq_lens[b] += 1 + a;
    if (any_bad_token) raise_status(status, SDVA_STATUS_BAD_DRAFT);
  }
}

}  // namespace
}  // namespace sdva

using namespace sdva;

namespace {
int check_accept_args(const float* logits, int num_lanes, int window, int vocab, const int32_t* drafts,
                      const int32_t* accept_len, const int32_t* out_tokens) {
  if (logits == nullptr || accept_len == nullptr || out_tokens == nullptr) return SDVA_ERR_INVALID;
  if (num_lanes <= 0 || window <= 0 || vocab <= 0) return SDVA_ERR_INVALID;
  if (window > 1 && drafts == nullptr) return SDVA_ERR_INVALID;
  if (window > kMaxWindow) return SDVA_ERR_UNSUPPORTED;
  if ((long long)num_lanes * window > 65535) return SDVA_ERR_UNSUPPORTED;
  return SDVA_OK;
}
// 16-byte loads are used when every row starts on a 16-byte boundary
int rows_vectorizable(const float* logits, int vocab) {
  return (vocab & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
}
int sm_count(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDVA_ERR_CUDA;
  return SDVA_OK;
}
// the argmax of every row (num_drafts: of rows 0 .. d_b of every lane)
int launch_argmax_rows(const float* logits, int num_lanes, int window, int vocab, const int32_t* num_drafts,
                       int32_t* out_tokens, cudaStream_t s, bool after_verify = false) {
  const long long rows = (long long)num_lanes * window;
  int sms = 0;
  if (const int rc = sm_count(&sms)) return rc;
  // CTAs per row: enough CTAs to cover every SM about four times, at most 8 (one portable cluster per row)
  int parts = 1;
  while (parts < kMaxRowCluster && rows * parts < 4LL * sms) parts *= 2;
  int chunk = (vocab + parts - 1) / parts;
  chunk = (chunk + 3) & ~3;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(parts, (unsigned)rows, 1);
  cfg.blockDim = dim3(kArgmaxThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = parts;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_verify ? 2 : 1;
  const auto kernel = rows_vectorizable(logits, vocab) ? argmax_rows_kernel<true> : argmax_rows_kernel<false>;
  if (cudaLaunchKernelEx(&cfg, kernel, logits, vocab, chunk, num_drafts, window, out_tokens) != cudaSuccess)
    return SDVA_ERR_CUDA;
  return SDVA_OK;
}
// a one-warp-per-lane kernel launched as a programmatic dependent of the argmax
template <typename... Args>
int launch_finalize(void (*kernel)(Args...), int num_lanes, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((num_lanes + 3) / 4, 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? SDVA_OK : SDVA_ERR_CUDA;
}
}  // namespace

int sdva::accept_launch(const float* logits, int num_lanes, int window, int vocab, const int32_t* drafts,
                       int32_t* accept_len, int32_t* out_tokens, int32_t* seq_lens_inout, int32_t* status,
                       sdva_stream_t stream, bool after_verify, bool check_only) {
  if (const int rc = check_accept_args(logits, num_lanes, window, vocab, drafts, accept_len, out_tokens)) return rc;
  if (check_only) return SDVA_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (const int rc = launch_argmax_rows(logits, num_lanes, window, vocab, nullptr, out_tokens, s, after_verify))
    return rc;
  return launch_finalize(accept_finalize_kernel, num_lanes, s, num_lanes, window, vocab, drafts,
                         (const int32_t*)out_tokens, accept_len, seq_lens_inout, status);
}

extern "C" int spec_accept(const float* logits, int num_lanes, int window, int vocab, const int32_t* drafts,
                           int32_t* accept_len, int32_t* out_tokens, int32_t* seq_lens_inout, int32_t* status,
                           sdva_stream_t stream) {
  return sdva::accept_launch(logits, num_lanes, window, vocab, drafts, accept_len, out_tokens, seq_lens_inout,
                             status, stream, false);
}

extern "C" int spec_accept_lazy(const float* logits, int num_lanes, int window, int vocab, const int32_t* drafts,
                                const int32_t* num_drafts, int32_t* accept_len, int32_t* out_tokens,
                                int32_t* seq_lens_inout, int32_t* status, sdva_stream_t stream) {
  if (const int rc = check_accept_args(logits, num_lanes, window, vocab, drafts, accept_len, out_tokens)) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (num_lanes < kWalkMinLanes) {
    if (const int rc = launch_argmax_rows(logits, num_lanes, window, vocab, num_drafts, out_tokens, s)) return rc;
    return launch_finalize(accept_lazy_finalize_kernel, num_lanes, s, num_lanes, window, vocab, drafts, num_drafts,
                           out_tokens, accept_len, seq_lens_inout, status);
  }
  // CTAs per lane: one per kWalkSlice logits of a row, at most one portable cluster
  const int parts = min(kMaxRowCluster, max(1, (vocab + kWalkSlice - 1) / kWalkSlice));
  int chunk = (vocab + parts - 1) / parts;
  chunk = (chunk + 3) & ~3;
  const auto kernel = rows_vectorizable(logits, vocab) ? accept_walk_kernel<true> : accept_walk_kernel<false>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(parts, (unsigned)num_lanes, 1);
  cfg.blockDim = dim3(kWalkThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = parts;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, logits, window, vocab, chunk, drafts, num_drafts, accept_len, out_tokens,
                         seq_lens_inout, status) != cudaSuccess)
    return SDVA_ERR_CUDA;
  return SDVA_OK;
}

extern "C" int spec_accept_tree(const float* logits, int num_lanes, int window, int vocab, const int32_t* tokens,
                                const int32_t* parent, int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                                int32_t* seq_lens_inout, int32_t* status, sdva_stream_t stream) {
  if (logits == nullptr || accept_len == nullptr || path == nullptr || out_tokens == nullptr) return SDVA_ERR_INVALID;
  if (num_lanes <= 0 || window <= 0 || vocab <= 0) return SDVA_ERR_INVALID;
  if (window > 1 && (tokens == nullptr || parent == nullptr)) return SDVA_ERR_INVALID;
  if (window > kMaxWindow) return SDVA_ERR_UNSUPPORTED;
  if ((long long)num_lanes * window > 65535) return SDVA_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the row argmaxes go to `path` first; the walk overwrites them
  if (const int rc = launch_argmax_rows(logits, num_lanes, window, vocab, nullptr, path, s)) return rc;
  return launch_finalize(accept_tree_finalize_kernel, num_lanes, s, num_lanes, window, vocab, tokens, parent, path,
                         out_tokens, accept_len, seq_lens_inout, status);
}
