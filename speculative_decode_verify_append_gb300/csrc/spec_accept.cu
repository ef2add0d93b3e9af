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
// loads, four in flight per thread (32 registers, so eight 256-thread CTAs fit
// on an SM and the grid of the multi-row case is a single wave), reduces
// (value, index) in shared memory,
// and stores it into CTA rank 0's shared memory through distributed shared
// memory; rank 0 writes the row's argmax.  No global scratch.  Ties go to the
// lowest index, NaN never wins, an all-NaN row gives 0.
// Kernel 2 (finalize, one warp per lane): compares the drafts with the
// argmaxes, writes the accept length and optionally commits seq_lens += 1 + a.
// It is launched as a programmatic dependent of kernel 1 so its launch
// overlaps kernel 1's tail; it waits for kernel 1's results before reading.
#include <cooperative_groups.h>

#include "sdva_common.cuh"

namespace cg = cooperative_groups;

namespace sdva {
namespace {

constexpr int kArgmaxThreads = 256;
constexpr int kMaxRowCluster = 8;

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
__device__ __forceinline__ void take4(const float4 v, int i, float& bv, int& bi) {
  take(v.x, i, bv, bi);
  take(v.y, i + 1, bv, bi);
  take(v.z, i + 2, bv, bi);
  take(v.w, i + 3, bv, bi);
}

// grid (parts, rows), cluster (parts, 1, 1)
__global__ void __launch_bounds__(kArgmaxThreads, 8) argmax_rows_kernel(const float* logits, int vocab, int chunk,
                                                                    int32_t* out_tokens) {
  cg::cluster_group cluster = cg::this_cluster();
  // the finalize kernel may be scheduled now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int part = blockIdx.x, row = blockIdx.y;
  const float* x = logits + (size_t)row * vocab;
  const int lo = part * chunk, hi = min(vocab, lo + chunk);
  float bv = __int_as_float(0x7fffffff);  // NaN: loses to every number
  int bi = 0x7fffffff;
  if ((vocab & 3) == 0) {
    // rows are 16-byte aligned when vocab % 4 == 0; chunk is a multiple of 4
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int step = blockDim.x;
    int k = lo / 4 + threadIdx.x;
    const int kend = hi / 4;
    for (; k + 3 * step < kend; k += 4 * step) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcs(x4 + k + u * step);
#pragma unroll
      for (int u = 0; u < 4; ++u) take4(v[u], 4 * (k + u * step), bv, bi);
    }
    for (; k < kend; k += step) take4(__ldcs(x4 + k), 4 * k, bv, bi);
  } else {
    for (int k = lo + threadIdx.x; k < hi; k += blockDim.x) take(x[k], k, bv, bi);
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

}  // namespace
}  // namespace sdva

using namespace sdva;

extern "C" int spec_accept(const float* logits, int num_lanes, int window, int vocab, const int32_t* drafts,
                           int32_t* accept_len, int32_t* out_tokens, int32_t* seq_lens_inout, int32_t* status,
                           sdva_stream_t stream) {
  if (logits == nullptr || accept_len == nullptr || out_tokens == nullptr) return SDVA_ERR_INVALID;
  if (num_lanes <= 0 || window <= 0 || vocab <= 0) return SDVA_ERR_INVALID;
  if (window > 1 && drafts == nullptr) return SDVA_ERR_INVALID;
  if (window > kMaxWindow) return SDVA_ERR_UNSUPPORTED;
  const long long rows = (long long)num_lanes * window;
  if (rows > 65535) return SDVA_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDVA_ERR_CUDA;
  // CTAs per row: enough CTAs to cover every SM about four times, at most 8 (one portable cluster per row)
  int parts = 1;
  while (parts < kMaxRowCluster && rows * parts < 4LL * sms) parts *= 2;
  int chunk = (vocab + parts - 1) / parts;
  chunk = (chunk + 3) & ~3;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(parts, (unsigned)rows, 1);
    cfg.blockDim = dim3(kArgmaxThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = parts;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, argmax_rows_kernel, logits, vocab, chunk, out_tokens) != cudaSuccess)
      return SDVA_ERR_CUDA;
  }
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((num_lanes + 3) / 4, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, accept_finalize_kernel, num_lanes, window, vocab, drafts,
                           (const int32_t*)out_tokens, accept_len, seq_lens_inout, status) != cudaSuccess)
      return SDVA_ERR_CUDA;
  }
  return SDVA_OK;
}
