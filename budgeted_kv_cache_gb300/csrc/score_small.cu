// Window-attention scoring for small windows on the CUDA cores.
//
// What it computes is kvc_score's (PASK Eq. 1 over the observation window;
// PACE Sec. 3.1's bonus; the H2O cumulative score with ACCUMULATE):
//   score[u][j] = sum_{r < R} exp(z_rj - lse_r) [+ old] + bonus[b][j],
// row r = h W + w sees keys j <= T - W + w.  With R = W G <= 16 rows (W = 1:
// one decode query per head) the contraction is too thin for the tensor
// cores: each key row meets at most 16 query rows, so the work is one HBM
// read of the keys and a few FMAs per key element.  Each warp brings 32
// consecutive key rows into shared memory, each lane one row by its own bulk
// copy into a row padded by 16 bytes, and a lane owns a key: all lanes read
// the same 16-byte chunk index of their rows, which the padding spreads over
// all banks, so the query rows (shared memory, pre-scaled to log2 units) are
// read as broadcasts.
//
//   * With the caller's row statistics one pass writes the scores.
//   * Otherwise the first pass writes each key's R logits (R floats per key,
//     a fraction of the key row) and per-split (max, sum) statistics; a merge
//     gives every row's log-sum-exp, and a second, light pass turns the stored
//     logits into scores.  The keys are read from HBM once either way.
#include <limits.h>
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kSThreads = 128;
constexpr int kSWarps = kSThreads / 32;
constexpr unsigned kAllLanes = 0xffffffffu;

// Logits of this lane's key row (in shared memory) against the RR query rows.
template <int D, int RR>
__device__ __forceinline__ void small_logits(const uint8_t* krow_bytes, const float (*qs)[D],
                                             float (&t)[RR]) {
  constexpr int CH = D * 2 / 16;
  const uint4* krow = reinterpret_cast<const uint4*>(krow_bytes);
#pragma unroll
  for (int h = 0; h < RR; ++h) t[h] = 0.f;
#pragma unroll 4
  for (int c = 0; c < CH; ++c) {
    const uint4 w = krow[c];
    const uint32_t rw[4] = {w.x, w.y, w.z, w.w};
    float x[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(rw[k] << 16);
      x[2 * k + 1] = __uint_as_float(rw[k] & 0xffff0000u);
    }
#pragma unroll
    for (int h = 0; h < RR; ++h) {
      const float4 q0 = *reinterpret_cast<const float4*>(&qs[h][c * 8]);
      const float4 q1 = *reinterpret_cast<const float4*>(&qs[h][c * 8 + 4]);
      float s = t[h];
      s = fmaf(x[0], q0.x, s);
      s = fmaf(x[1], q0.y, s);
      s = fmaf(x[2], q0.z, s);
      s = fmaf(x[3], q0.w, s);
      s = fmaf(x[4], q1.x, s);
      s = fmaf(x[5], q1.y, s);
      s = fmaf(x[6], q1.z, s);
      s = fmaf(x[7], q1.w, s);
      t[h] = s;
    }
  }
}

// The bonus and previous score of key j (loaded before the key row arrives).
__device__ __forceinline__ float small_extra(const ScoreArgs& a, int u, int b, int64_t j, bool valid) {
  if (!valid) return 0.f;
  const int64_t T = a.T;
  const float bon = a.bonus ? __ldg(a.bonus + static_cast<int64_t>(b) * T + j) : 0.f;
  const float old = a.accumulate ? a.scores[static_cast<int64_t>(u) * T + j] : 0.f;
  return bon + old;
}

// Score of key j from its mass; the page maximum over P consecutive keys
// (P lanes of the warp, the step starting on a multiple of P).
__device__ __forceinline__ void small_store(const ScoreArgs& a, int u, int64_t j, bool valid, float mass,
                                            float extra, int lane) {
  const int64_t T = a.T;
  float sc = -INFINITY;
  if (valid) {
    sc = mass + extra;
    a.scores[static_cast<int64_t>(u) * T + j] = sc;
  }
  const int P = a.page_size;
  if (P > 1) {
    float pm = sc;
    for (int o = 1; o < P; o <<= 1) pm = fmaxf(pm, __shfl_xor_sync(kAllLanes, pm, o));
    if (valid && (lane & (P - 1)) == 0) a.page_scores[static_cast<int64_t>(u) * (T / P) + j / P] = pm;
  }
}

// Pass over a split of a unit's keys.  DIRECT: the row statistics are
// given and scores are written; otherwise the logits [U][T][RR] and the
// split's (max, sum) per row are written.
template <int D, int RR, bool DIRECT>
__global__ void __launch_bounds__(kSThreads) score_small_kernel(const ScoreArgs a, float* logits,
                                                                float2* split_stats, int splits) {
  constexpr int ROWB = D * 2;
  constexpr int ROWP = ROWB + 16;                                // padded row in shared memory
  extern __shared__ __align__(128) uint8_t ssm[];                // [4 warps][32 rows][ROWP]
  __shared__ __align__(16) float qs[RR][D];
  __shared__ float lse2[RR];
  __shared__ float wm[kSWarps][RR], wl[kSWarps][RR];
  __shared__ __align__(8) uint64_t bars[kSWarps];
  __shared__ int abort_i;
  const int u = blockIdx.x, split = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = a.R;
  const int b = u / (a.L * a.Hkv);
  const int64_t T = a.T;
  if (tid < kSWarps) mbar_init(smem_u32(&bars[tid]), 1);
  if (tid == 0) abort_i = 0;
  {
    const __nv_bfloat16* q = a.q_small + static_cast<int64_t>(u) * R * D;
    for (int idx = tid; idx < RR * D; idx += kSThreads)
      qs[idx / D][idx % D] = idx / D < R ? __bfloat162float(q[idx]) * a.scale_log2 : 0.f;
    if (DIRECT && tid < RR)
      lse2[tid] = tid < R ? __ldg(a.row_lse + static_cast<int64_t>(u) * R + tid) * 1.44269504088896340736f
                          : INFINITY;
  }
  fence_barrier_init();
  // splits start on multiples of 128 keys, so every warp step starts on a
  // multiple of 32 (and of the page size)
  const int64_t per = ((T + splits - 1) / splits + 127) / 128 * 128;
  const int64_t lo = min(T, split * per), hi = min(T, lo + per);
  __syncthreads();
  volatile int* abort_flag = &abort_i;
  uint8_t* kb = ssm + warp * 32 * ROWP;
  const uint32_t bar = smem_u32(&bars[warp]);
  const uint8_t* kg = reinterpret_cast<const uint8_t*>(a.k_small) + static_cast<int64_t>(u) * T * ROWB;
  const int64_t Tq = T - a.W;                      // row w sees keys j <= Tq + w
  float m[RR], l[RR];
#pragma unroll
  for (int h = 0; h < RR; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
  }
  uint32_t phase = 0;
  bool fail = false;
#pragma unroll 1
  for (int64_t base = lo + warp * 32; base < hi; base += kSThreads) {
    const int nrow = static_cast<int>(min(static_cast<int64_t>(32), hi - base));
    const int64_t j = base + lane;
    const bool valid = lane < nrow;
    fence_proxy_async_smem();                      // the buffer's last reads precede the copies
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nrow * ROWB));
    __syncwarp();
    if (valid) bulk_copy_g2s(smem_u32(kb + lane * ROWP), kg + j * ROWB, ROWB, bar);
    const float extra = DIRECT ? small_extra(a, u, b, j, valid) : 0.f;
    const bool ok = __all_sync(kAllLanes, mbar_wait(bar, phase, abort_flag));
    if (!ok) {
      if (lane == 0) {                             // the copy lands (bounded) before the CTA leaves
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, phase) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
      __syncwarp();
      fail = true;
      break;
    }
    phase ^= 1;
    float t[RR];
    small_logits<D, RR>(kb + lane * ROWP, qs, t);
#pragma unroll
    for (int h = 0; h < RR; ++h)
      if (!valid || h >= R || j > Tq + (h % a.W)) t[h] = -INFINITY;
    if (DIRECT) {
      float mass = 0.f;
#pragma unroll
      for (int h = 0; h < RR; ++h) mass += ex2_approx(t[h] - lse2[h]);
      small_store(a, u, j, valid, mass, extra, lane);
    } else {
      if (valid) {
        float4* dst = reinterpret_cast<float4*>(logits + (static_cast<int64_t>(u) * T + j) * RR);
        if constexpr (RR >= 4) {
#pragma unroll
          for (int h = 0; h < RR; h += 4) dst[h / 4] = make_float4(t[h], t[h + 1], t[h + 2], t[h + 3]);
        } else {
#pragma unroll
          for (int h = 0; h < RR; ++h) logits[(static_cast<int64_t>(u) * T + j) * RR + h] = t[h];
        }
      }
      // online max / sum of each row over the warp's keys
#pragma unroll
      for (int h = 0; h < RR; ++h) {
        float mx = t[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kAllLanes, mx, o));
        const float mn = fmaxf(m[h], mx);
        if (mn != -INFINITY) {                     // uniform across the warp
          float e = t[h] == -INFINITY ? 0.f : ex2_approx(t[h] - mn);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(kAllLanes, e, o);
          l[h] = (m[h] == -INFINITY ? 0.f : l[h] * ex2_approx(m[h] - mn)) + e;
          m[h] = mn;
        }
      }
    }
    __syncwarp();                                  // the buffer is free for the next copy
  }
  if (fail && lane == 0 && a.unit_status) a.unit_status[u] = KVC_UNIT_TIMEOUT;
  if (!DIRECT) {
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < RR; ++h) {
        wm[warp][h] = m[h];
        wl[warp][h] = l[h];
      }
    }
    __syncthreads();
    if (tid < R) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kSWarps; ++w) M = fmaxf(M, wm[w][tid]);
      float L = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kSWarps; ++w)
          if (wm[w][tid] != -INFINITY) L += wl[w][tid] * ex2_approx(wm[w][tid] - M);
      }
      split_stats[(static_cast<int64_t>(u) * splits + split) * RR + tid] = make_float2(M, L);
    }
  }
}

// Each row's log2-domain log-sum-exp from the splits' statistics.
__global__ void __launch_bounds__(32) score_small_lse_kernel(const ScoreArgs a, const float2* split_stats,
                                                              int splits, int RR, float* lse2) {
  const int u = blockIdx.x, r = threadIdx.x;
  if (r >= RR) return;
  float M = -INFINITY, L = 0.f;
  if (r < a.R) {
    for (int s = 0; s < splits; ++s) M = fmaxf(M, split_stats[(static_cast<int64_t>(u) * splits + s) * RR + r].x);
    for (int s = 0; s < splits; ++s) {
      const float2 st = split_stats[(static_cast<int64_t>(u) * splits + s) * RR + r];
      if (st.x != -INFINITY) L += st.y * ex2_approx(st.x - M);
    }
  }
  lse2[static_cast<int64_t>(u) * RR + r] = (r < a.R && M != -INFINITY) ? M + log2f(L) : INFINITY;
}

// Scores from the stored logits: thread = key.
template <int RR>
__global__ void __launch_bounds__(256) score_small_mass_kernel(const ScoreArgs a, const float* logits,
                                                               const float* lse2) {
  const int u = blockIdx.y;
  const int b = u / (a.L * a.Hkv);
  const int64_t j = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  const bool valid = j < a.T;
  float ls[RR];
#pragma unroll
  for (int h = 0; h < RR; ++h) ls[h] = __ldg(lse2 + static_cast<int64_t>(u) * RR + h);
  float mass = 0.f;
  if (valid) {
    const float* src = logits + (static_cast<int64_t>(u) * a.T + j) * RR;
    if constexpr (RR >= 4) {
#pragma unroll
      for (int h = 0; h < RR; h += 4) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(src) + h / 4);
        mass += ex2_approx(t.x - ls[h]) + ex2_approx(t.y - ls[h + 1]) + ex2_approx(t.z - ls[h + 2]) +
                ex2_approx(t.w - ls[h + 3]);
      }
    } else {
#pragma unroll
      for (int h = 0; h < RR; ++h) mass += ex2_approx(__ldg(src + h) - ls[h]);
    }
  }
  small_store(a, u, j, valid, mass, small_extra(a, u, b, j, valid), threadIdx.x & 31);
}

}  // namespace

int small_rows(int R) { return R <= 1 ? 1 : R <= 2 ? 2 : R <= 4 ? 4 : R <= 8 ? 8 : 16; }

size_t score_small_smem_bytes(int d) { return static_cast<size_t>(kSWarps) * 32 * (d * 2 + 16); }

cudaError_t launch_score_small(const ScoreArgs& a, int splits, float* logits, float2* split_stats,
                               float* lse2, cudaStream_t stream) {
  const int RR = small_rows(a.R);
  const bool direct = a.row_lse != nullptr;
  const size_t smem = score_small_smem_bytes(a.d);
  void (*k)(const ScoreArgs, float*, float2*, int) = nullptr;
#define KVC_SMALL_PICK(DD, RV)                                                           \
  if (a.d == DD && RR == RV)                                                              \
    k = direct ? score_small_kernel<DD, RV, true> : score_small_kernel<DD, RV, false>;
  KVC_SMALL_PICK(64, 1)
  KVC_SMALL_PICK(64, 2)
  KVC_SMALL_PICK(64, 4)
  KVC_SMALL_PICK(64, 8)
  KVC_SMALL_PICK(64, 16)
  KVC_SMALL_PICK(128, 1)
  KVC_SMALL_PICK(128, 2)
  KVC_SMALL_PICK(128, 4)
  KVC_SMALL_PICK(128, 8)
  KVC_SMALL_PICK(128, 16)
#undef KVC_SMALL_PICK
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k<<<dim3(a.U, splits), kSThreads, smem, stream>>>(a, logits, split_stats, splits);
  if ((e = cudaGetLastError()) != cudaSuccess || direct) return e;
  score_small_lse_kernel<<<a.U, 32, 0, stream>>>(a, split_stats, splits, RR, lse2);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const dim3 mg(static_cast<unsigned>((a.T + 255) / 256), a.U);
  switch (RR) {
    case 1: score_small_mass_kernel<1><<<mg, 256, 0, stream>>>(a, logits, lse2); break;
    case 2: score_small_mass_kernel<2><<<mg, 256, 0, stream>>>(a, logits, lse2); break;
    case 4: score_small_mass_kernel<4><<<mg, 256, 0, stream>>>(a, logits, lse2); break;
    case 8: score_small_mass_kernel<8><<<mg, 256, 0, stream>>>(a, logits, lse2); break;
    default: score_small_mass_kernel<16><<<mg, 256, 0, stream>>>(a, logits, lse2); break;
  }
  return cudaGetLastError();
}

}  // namespace kvc
