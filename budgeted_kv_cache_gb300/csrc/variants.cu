// Selection variants on the score buffer.
//
//  * SnapKV pooling (the pooling / kernel options of the SnapKV baseline in
//    PASK's baseline table): each token's score becomes the average or the
//    maximum of the `kernel` scores centred on it, stride 1; outside [0, T)
//    a score counts as 0 in the average (divided by `kernel`) and is ignored
//    by the maximum.  The average is summed left to right in fp32.
//  * CommitKV Eq. 4 applies one index set to every layer and head of a
//    sequence: the shared score of a token is the sum of its units' scores
//    (unit order, fp32), and the per-sequence kept lists are copied to every
//    unit of the sequence.
// All three are HBM-bound streaming kernels (grid-stride, coalesced).
#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kTile = 1024;        // tokens per CTA in the pooling kernel

__global__ void __launch_bounds__(256) pool_kernel(const float* __restrict__ in, float* __restrict__ out,
                                                   int64_t n, int kernel, int mode) {
  __shared__ float tile[kTile + 8];
  const int h = kernel / 2;
  const int64_t row = blockIdx.y;
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kTile;
  const float* src = in + row * n;
  const float pad = mode == KVC_SCORE_POOL_MAX ? -INFINITY : 0.f;
  for (int i = threadIdx.x; i < kTile + 2 * h; i += blockDim.x) {
    const int64_t j = j0 - h + i;
    tile[i] = (j >= 0 && j < n) ? __ldg(src + j) : pad;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kTile; i += blockDim.x) {
    const int64_t j = j0 + i;
    if (j >= n) break;
    float v;
    if (mode == KVC_SCORE_POOL_MAX) {
      v = tile[i];
      for (int k = 1; k < kernel; ++k) v = fmaxf(v, tile[i + k]);
    } else {
      float sum = 0.f;
      for (int k = 0; k < kernel; ++k) sum = __fadd_rn(sum, tile[i + k]);
      v = __fdiv_rn(sum, static_cast<float>(kernel));
    }
    out[row * n + j] = v;
  }
}

__global__ void shared_sum_kernel(const float* __restrict__ scores, float* __restrict__ shared,
                                  int B, int units_per_seq, int64_t n) {
  const int64_t total = static_cast<int64_t>(B) * n;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = idx / n, j = idx % n;
    const float* src = scores + b * units_per_seq * n + j;
    float sum = 0.f;
    for (int k = 0; k < units_per_seq; ++k) sum = __fadd_rn(sum, __ldg(src + k * n));
    shared[idx] = sum;
  }
}

__global__ void broadcast_kernel(const int32_t* __restrict__ kept_seq, const int32_t* __restrict__ count_seq,
                                 int32_t* __restrict__ kept, int32_t* __restrict__ count, int B,
                                 int units_per_seq, int cap) {
  // blockIdx.y = pool * U + unit
  const int U = B * units_per_seq;
  const int pool = blockIdx.y / U, u = blockIdx.y % U, b = u / units_per_seq;
  const int c = __ldg(count_seq + pool * B + b);
  if (blockIdx.x == 0 && threadIdx.x == 0) count[pool * U + u] = c;
  const int32_t* src = kept_seq + (static_cast<int64_t>(pool) * B + b) * cap;
  int32_t* dst = kept + (static_cast<int64_t>(pool) * U + u) * cap;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < c; i += gridDim.x * blockDim.x) dst[i] = __ldg(src + i);
}

}  // namespace

cudaError_t launch_pool(const float* in, float* out, int64_t rows, int64_t n, int kernel, int mode,
                        cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>((n + kTile - 1) / kTile), static_cast<unsigned>(rows));
  pool_kernel<<<grid, 256, 0, stream>>>(in, out, n, kernel, mode);
  return cudaGetLastError();
}

cudaError_t launch_shared_sum(const float* scores, float* shared, int B, int units_per_seq, int64_t n,
                              cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(B) * n;
  const int blocks = static_cast<int>(total / 256 + 1 < 8192 ? total / 256 + 1 : 8192);
  shared_sum_kernel<<<blocks, 256, 0, stream>>>(scores, shared, B, units_per_seq, n);
  return cudaGetLastError();
}

cudaError_t launch_broadcast(const int32_t* kept_seq, const int32_t* count_seq, int32_t* kept,
                             int32_t* count, int B, int units_per_seq, int cap, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>((cap + 255) / 256), static_cast<unsigned>(KVC_N_POOLS * B * units_per_seq));
  broadcast_kernel<<<grid, 256, 0, stream>>>(kept_seq, count_seq, kept, count, B, units_per_seq, cap);
  return cudaGetLastError();
}

}  // namespace kvc
