// spec_accept.cu -- greedy acceptance of a verify window.
//
// The main model's argmax at window position i is compared with draft i;
// the accepted prefix is the leading run of agreements and the bonus token is
// the argmax at the first disagreement (Baseten talk summary, section
// "추측 디코드"; the commit of the new length follows the NInfer review,
// section "아키텍처 ①": state changes only once the model accepts the commit).
//
// Kernel 1 (argmax): one thread-block cluster per logits row; each CTA of the
// cluster scans a contiguous slice of the vocabulary with 16-byte loads,
// reduces (value, index) within the CTA, and CTA rank 0 reduces the cluster's
// partials through distributed shared memory -- no global scratch.  Ties go to
// the lowest index, NaN never wins, an all-NaN row gives 0.
// Kernel 2 (finalize): one thread per lane compares drafts with the argmaxes,
// writes the accept length and optionally commits seq_lens += 1 + a.
#include <cooperative_groups.h>

#include "sdva_common.cuh"

namespace cg = cooperative_groups;

namespace sdva {
namespace {

constexpr int kArgmaxThreads = 256;

// true if candidate (v, i) beats the current best (bv, bi)
__device__ __forceinline__ bool beats(float v, int i, float bv, int bi) {
  const bool vn = isnan(v), bn = isnan(bv);
  if (vn != bn) return bn;     // a number beats NaN
  if (!vn && v != bv) return v > bv;
  return i < bi;                // equal values (+0 == -0) or both NaN: lower index
}

__device__ __forceinline__ void take(float v, int i, float& bv, int& bi) {
  if (beats(v, i, bv, bi)) {
    bv = v;
    bi = i;
  }
}

__global__ void __launch_bounds__(kArgmaxThreads) argmax_cluster_kernel(const float* logits, int vocab, int chunk,
                                                                       int32_t* out_tokens) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.y;
  const float* x = logits + (size_t)row * vocab;
  const int lo = rank * chunk, hi = min(vocab, lo + chunk);
  float bv = __int_as_float(0x7fffffff);  // NaN: loses to every number
  int bi = 0x7fffffff;
  // rows are 16-byte aligned when vocab % 4 == 0; chunk is a multiple of 4
  if ((vocab & 3) == 0) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    for (int k = lo / 4 + threadIdx.x; k < hi / 4; k += blockDim.x) {
      const float4 v = __ldcs(x4 + k);  // read once: stream past L1/L2 retention
      take(v.x, 4 * k, bv, bi);
      take(v.y, 4 * k + 1, bv, bi);
      take(v.z, 4 * k + 2, bv, bi);
      take(v.w, 4 * k + 3, bv, bi);
    }
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
  __shared__ float c_v;
  __shared__ int c_i;
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    s_v[warp] = bv;
    s_i[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) take(s_v[w], s_i[w], bv, bi);
    c_v = bv;
    c_i = bi;
  }
  cluster.sync();
  if (rank == 0 && threadIdx.x == 0) {
    for (int r = 1; r < (int)cluster.num_blocks(); ++r) {
      const float* rv = cluster.map_shared_rank(&c_v, r);
      const int* ri = cluster.map_shared_rank(&c_i, r);
      take(*rv, *ri, bv, bi);
    }
    out_tokens[row] = bi == 0x7fffffff ? 0 : bi;
  }
  cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

__global__ void accept_finalize_kernel(int num_lanes, int window, int vocab, const int32_t* drafts,
                                       const int32_t* out_tokens, int32_t* accept_len, int32_t* seq_lens,
                                       int32_t* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= num_lanes) return;
  const int d = window - 1;
  int a = 0;
  bool run = true, bad = false;
  for (int i = 0; i < d; ++i) {
    const int di = drafts[(size_t)b * d + i];
    if (di < 0 || di >= vocab) bad = true;
    if (run && di == out_tokens[(size_t)b * window + i])
      ++a;
    else
      run = false;
  }
  if (bad) raise_status(status, SDVA_STATUS_BAD_DRAFT);
  accept_len[b] = a;
  if (seq_lens != nullptr) seq_lens[b] += 1 + a;
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
  const long long rows = (long long)num_lanes * window;
  if (rows > 65535) return SDVA_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDVA_ERR_CUDA;
  // cluster size: enough CTAs to cover every SM about twice, at most 8 (portable)
  int cl = 1;
  while (cl < 8 && rows * cl < 2LL * sms) cl *= 2;
  int chunk = (vocab + cl - 1) / cl;
  chunk = (chunk + 3) & ~3;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cl, (unsigned)rows, 1);
  cfg.blockDim = dim3(kArgmaxThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, argmax_cluster_kernel, logits, vocab, chunk, out_tokens) != cudaSuccess)
    return SDVA_ERR_CUDA;
  const int threads = 128;
  accept_finalize_kernel<<<(num_lanes + threads - 1) / threads, threads, 0, s>>>(
      num_lanes, window, vocab, drafts, out_tokens, accept_len, seq_lens_inout, status);
  return cudaGetLastError() == cudaSuccess ? SDVA_OK : SDVA_ERR_CUDA;
}
