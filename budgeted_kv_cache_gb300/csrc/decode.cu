// One decode-attention step over the compacted pools (the consumer check).
//
// PASK Eq. 1 over every kept row of the unit, dequantised inside the kernel
// (x = code * scale); PASK App. B.5: fp32 scores, softmax statistics and
// accumulation, bf16 output.  The kept rows of a unit (int4, int8 and bf16
// pools, concatenated) are split across `splits` CTAs; each CTA streams its
// rows in chunks of 128 once for all G query heads of the KV head and keeps
// an online (max, sum, unnormalised value sum) per head.  Partitions are
// merged with PASK Eq. 15; empty partitions contribute nothing.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kThreads = 128;
constexpr int kMaxG = 8;
constexpr float kLog2e = 1.4426950408889634f;

struct RowRef {
  const void* k;
  const void* v;
  const void* ks;
  const void* vs;
};

__device__ __forceinline__ float scale_at(const void* sp, int64_t row, int col, int d, bool row_mode) {
  const uint16_t* s = static_cast<const uint16_t*>(sp);
  if (row_mode) return __half2float(__ushort_as_half(s[row]));
  return bf16_bits_to_float(s[row * (d / 32) + col / 32]);
}

// Element `col` of row `row` of a pool, dequantised.
__device__ __forceinline__ float load_elem(int pool, const void* base, const void* sp, int64_t row,
                                           int col, int d, bool row_mode) {
  if (pool == KVC_POOL_BF16)
    return bf16_bits_to_float(static_cast<const uint16_t*>(base)[row * d + col]);
  if (pool == KVC_POOL_INT8) {
    const int8_t c = static_cast<const int8_t*>(base)[row * d + col];
    return static_cast<float>(c) * scale_at(sp, row, col, d, row_mode);
  }
  const uint8_t byte = static_cast<const uint8_t*>(base)[row * (d / 2) + col / 2];
  int c = (col & 1) ? (byte >> 4) : (byte & 0xf);
  c = c > 7 ? c - 16 : c;
  return static_cast<float>(c) * scale_at(sp, row, col, d, row_mode);
}

__global__ void __launch_bounds__(kThreads) decode_kernel(const DecodeArgs a) {
  __shared__ float qs[kMaxG][128];
  __shared__ float sc[kThreads][kMaxG + 1];
  __shared__ float cmax[kMaxG], csum[kMaxG];
  __shared__ int rpool[kThreads];
  __shared__ int64_t rrow[kThreads];
  __shared__ float accs[kThreads][kMaxG];

  const int u = blockIdx.x, split = blockIdx.y;
  const int G = a.G, d = a.d, tid = threadIdx.x;
  const bool row_mode = a.quant_mode == KVC_QUANT_ROW_FP16;
  const __nv_bfloat16* q = a.q + static_cast<int64_t>(u) * G * d;
  for (int idx = tid; idx < G * d; idx += kThreads)
    qs[idx / d][idx % d] = __bfloat162float(q[idx]);

  int cnt[KVC_N_POOLS];
  int n = 0;
  for (int p = 0; p < KVC_N_POOLS; ++p) {
    cnt[p] = (p >= a.pool_lo && p < a.pool_hi) ? a.kept_count[p * a.U + u] : 0;
    n += cnt[p];
  }
  const int per = (n + a.splits - 1) / a.splits;
  const int lo = min(n, split * per), hi = min(n, lo + per);

  // PV layout: thread = (row group rg, column c); 128 / d row groups.
  const int rgs = kThreads / d;
  const int rg = tid / d, col = tid % d;
  float m[kMaxG], l[kMaxG], acc[kMaxG];
#pragma unroll
  for (int h = 0; h < kMaxG; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
    acc[h] = 0.f;
  }
  const float cs = a.scale * kLog2e;
  __syncthreads();

  for (int base = lo; base < hi; base += kThreads) {
    const int r = base + tid;
    int pool = -1;
    int64_t row = 0;
    if (r < hi) {
      int rr = r;
      for (int p = 0; p < KVC_N_POOLS; ++p) {
        if (rr < cnt[p]) {
          pool = p;
          break;
        }
        rr -= cnt[p];
      }
      row = static_cast<int64_t>(u) * a.capacity + rr;
    }
    rpool[tid] = pool;
    rrow[tid] = row;
    // scores of this thread's row for every head
    float s[kMaxG];
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) s[h] = 0.f;
    if (pool >= 0) {
      const void* kb = pool == KVC_POOL_BF16 ? a.pools.k_bf16
                       : pool == KVC_POOL_INT8 ? a.pools.k_i8 : a.pools.k_i4;
      const void* ksp = pool == KVC_POOL_INT8 ? a.pools.k_i8_scale : a.pools.k_i4_scale;
      for (int e = 0; e < d; ++e) {
        const float kv = load_elem(pool, kb, ksp, row, e, d, row_mode);
#pragma unroll
        for (int h = 0; h < kMaxG; ++h)
          if (h < G) s[h] = fmaf(kv, qs[h][e], s[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) sc[tid][h] = pool >= 0 ? s[h] * cs : -INFINITY;
    __syncthreads();
    // chunk max per head (warp w handles heads w, w+4)
    const int warp = tid >> 5, lane = tid & 31;
    for (int h = warp; h < G; h += kThreads / 32) {
      float mx = -INFINITY;
      for (int k = lane; k < kThreads; k += 32) mx = fmaxf(mx, sc[k][h]);
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) cmax[h] = mx;
    }
    __syncthreads();
    // probabilities relative to the new running max
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) {
      if (h >= G) break;
      const float mn = fmaxf(m[h], cmax[h]);
      sc[tid][h] = (sc[tid][h] == -INFINITY) ? 0.f : exp2f(sc[tid][h] - mn);
    }
    __syncthreads();
    for (int h = warp; h < G; h += kThreads / 32) {
      float sm = 0.f;
      for (int k = lane; k < kThreads; k += 32) sm += sc[k][h];
      for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
      if (lane == 0) csum[h] = sm;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) {
      if (h >= G) break;
      const float mn = fmaxf(m[h], cmax[h]);
      const float corr = (m[h] == -INFINITY) ? 0.f : exp2f(m[h] - mn);
      l[h] = l[h] * corr + csum[h];
      acc[h] *= corr;
      m[h] = mn;
    }
    // P V for this thread's column over its row group
    for (int k = rg; k < kThreads; k += rgs) {
      const int pool_k = rpool[k];
      if (pool_k < 0) continue;
      const void* vb = pool_k == KVC_POOL_BF16 ? a.pools.v_bf16
                       : pool_k == KVC_POOL_INT8 ? a.pools.v_i8 : a.pools.v_i4;
      const void* vsp = pool_k == KVC_POOL_INT8 ? a.pools.v_i8_scale : a.pools.v_i4_scale;
      const float vv = load_elem(pool_k, vb, vsp, rrow[k], col, d, row_mode);
#pragma unroll
      for (int h = 0; h < kMaxG; ++h)
        if (h < G) acc[h] = fmaf(sc[k][h], vv, acc[h]);
    }
    __syncthreads();
  }

  // combine the row groups of each column
  if (rgs > 1) {
    for (int g = 1; g < rgs; ++g) {
      if (rg == g)
        for (int h = 0; h < G; ++h) accs[col][h] = acc[h];
      __syncthreads();
      if (rg == 0)
        for (int h = 0; h < G; ++h) acc[h] += accs[col][h];
      __syncthreads();
    }
  }
  if (rg != 0) return;
  if (a.splits == 1) {
    for (int h = 0; h < G; ++h) {
      const float o = l[h] > 0.f ? acc[h] / l[h] : 0.f;
      a.out[(static_cast<int64_t>(u) * G + h) * d + col] = __float2bfloat16_rn(o);
    }
  } else {
    for (int h = 0; h < G; ++h) {
      const int64_t slot = (static_cast<int64_t>(u) * a.splits + split) * G + h;
      a.ws_acc[slot * d + col] = acc[h];
      if (col == 0) {
        a.ws_ml[slot * 2] = m[h];
        a.ws_ml[slot * 2 + 1] = l[h];
      }
    }
  }
}

// PASK Eq. 15 over the split partitions of one (unit, head).
__global__ void __launch_bounds__(128) merge_kernel(const DecodeArgs a) {
  const int u = blockIdx.x, h = blockIdx.y, col = threadIdx.x;
  if (col >= a.d) return;
  float v = -INFINITY;
  for (int s = 0; s < a.splits; ++s) {
    const int64_t slot = (static_cast<int64_t>(u) * a.splits + s) * a.G + h;
    v = fmaxf(v, a.ws_ml[slot * 2]);
  }
  float num = 0.f, den = 0.f;
  if (v != -INFINITY) {
    for (int s = 0; s < a.splits; ++s) {
      const int64_t slot = (static_cast<int64_t>(u) * a.splits + s) * a.G + h;
      const float vj = a.ws_ml[slot * 2];
      if (vj == -INFINITY) continue;          // empty partition
      const float w = exp2f(vj - v);
      num += w * a.ws_acc[slot * a.d + col];
      den += w * a.ws_ml[slot * 2 + 1];
    }
  }
  const float o = den > 0.f ? num / den : 0.f;
  a.out[(static_cast<int64_t>(u) * a.G + h) * a.d + col] = __float2bfloat16_rn(o);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  decode_kernel<<<dim3(a.U, a.splits), kThreads, 0, stream>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || a.splits == 1) return err;
  merge_kernel<<<dim3(a.U, a.G), 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc
