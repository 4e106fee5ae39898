// PACE Eq. 2 foresight bonus, painted from spans.
//
// For step t, a token in span (a, b) whose next planned reader is step s*
// (computed by the caller as min{s in F : s >= t}) receives
//   beta = sigma * (1/2 + 1/2 exp(-lambda (s* - t)));
// a token in no span with a future reader receives 0, and a token in
// several spans takes the largest bonus (its soonest reference).  One CTA
// per span writes its tokens with an atomic maximum on the float bits (all
// values are >= 0, so their bit patterns order like the values), which
// makes the result independent of the order of the spans.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

__global__ void bonus_clear_kernel(float* bonus, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    bonus[i] = 0.f;
}

__global__ void bonus_paint_kernel(const BonusArgs a) {
  const int sp = blockIdx.x;
  const int next = a.span_next[sp];
  const int seq = a.span_seq[sp];
  if (next < a.step || seq < 0 || seq >= a.batch) return;      // no future reader
  const int64_t lo = a.span_a[sp] > 0 ? a.span_a[sp] : 0;
  const int64_t hi = a.span_b[sp] < a.T ? a.span_b[sp] : a.T;
  const float beta = a.sigma * (0.5f + 0.5f * expf(-a.lambda * static_cast<float>(next - a.step)));
  unsigned int* dst = reinterpret_cast<unsigned int*>(a.bonus + static_cast<int64_t>(seq) * a.T);
  const unsigned int bits = __float_as_uint(beta);
  for (int64_t j = lo + threadIdx.x; j < hi; j += blockDim.x) atomicMax(dst + j, bits);
}

}  // namespace

cudaError_t launch_bonus(const BonusArgs& a, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(a.batch) * a.T;
  const int64_t want = (n + 255) / 256;
  const int blocks = static_cast<int>(want < 4096 ? want : 4096);
  if (blocks > 0) bonus_clear_kernel<<<blocks, 256, 0, stream>>>(a.bonus, n);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || a.n_spans == 0) return err;
  bonus_paint_kernel<<<a.n_spans, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc
