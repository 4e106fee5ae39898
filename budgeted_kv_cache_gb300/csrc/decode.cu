// One decode-attention step over the compacted pools (the consumer check).
//
// PASK Eq. 1 over every kept row of the unit, dequantised inside the kernel
// (x = code * scale); PASK App. B.5: fp32 scores, softmax statistics and
// accumulation, bf16 output.  The kept rows of a unit (int4, int8 and bf16
// pools, concatenated in that order) are split across `splits` CTAs and the
// partitions merged with PASK Eq. 15; empty partitions contribute nothing.
//
// Layout of the work (HBM-bound: every kept row is read once for all G
// query heads of its KV head):
//   * a warp takes 32 consecutive rows per step; for the scores each lane
//     owns one key row and reads it with 16-byte loads (the query heads sit
//     in shared memory and are read as broadcasts);
//   * for P V each lane owns d / 32 adjacent columns, so every value row is
//     one coalesced warp load, and the 32 probabilities reach the lanes by
//     shuffles;
//   * each warp keeps its own online (max, sum, unnormalised value sum) per
//     head; the CTA's four warps, then the CTAs of a unit, are merged with
//     Eq. 15.
#include <math.h>

#include "kvc_internal.cuh"
#include "decode_rows.cuh"

namespace kvc {

namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

// GG: query heads per KV head rounded up to 1, 2, 4 or 8 (the loops over
// heads are unrolled for GG); BF: only the bf16 pool holds rows (token and
// page mode), so the int8 / int4 paths are not compiled in.
template <int D, int GG, bool BF>
__global__ void __launch_bounds__(kThreads, 6) decode_kernel(const DecodeArgs a) {
  constexpr int NC = D / 32;
  constexpr int VB = 16;                         // value rows whose loads are in flight together
  __shared__ __align__(16) float qs[GG][D];
  __shared__ float wm[kWarps][GG], wl[kWarps][GG];
  __shared__ float wacc[kWarps][GG][D];

  const int u = blockIdx.x, split = blockIdx.y;
  const int G = a.G, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool row_mode = a.quant_mode == KVC_QUANT_ROW_FP16;
  const float cs = a.scale * kLog2e;
  {
    const __nv_bfloat16* q = a.q + static_cast<int64_t>(u) * G * D;
    for (int idx = tid; idx < G * D; idx += kThreads) qs[idx / D][idx % D] = __bfloat162float(q[idx]) * cs;
  }
  int cnt[KVC_N_POOLS];
  int n = 0;
#pragma unroll
  for (int p = 0; p < KVC_N_POOLS; ++p) {
    // a count outside [0, capacity] is clamped, so no row past the pool is read
    cnt[p] = (p >= a.pool_lo && p < a.pool_hi) ? clamp_count(a.kept_count[p * a.U + u], a.capacity) : 0;
    n += cnt[p];
  }
  const int per = (n + a.splits - 1) / a.splits;
  const int lo = min(n, split * per), hi = min(n, lo + per);
  __syncthreads();

  float m[GG], l[GG], acc[GG][NC];
#pragma unroll
  for (int h = 0; h < GG; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[h][c] = 0.f;
  }

  for (int base = lo + warp * 32; base < hi; base += kThreads) {
    // ---- scores: lane = row
    const int r = base + lane;
    int pool = -1, rr = r;
    if (r < hi) {
#pragma unroll
      for (int p = 0; p < KVC_N_POOLS; ++p) {
        if (pool < 0) {
          if (rr < cnt[p]) pool = p;
          else rr -= cnt[p];
        }
      }
    }
    const int64_t row = static_cast<int64_t>(u) * a.capacity + rr;
    float s[GG];
#pragma unroll
    for (int h = 0; h < GG; ++h) s[h] = 0.f;
    if (pool >= 0) key_dot<D, GG, BF>(pool, pool_ptrs(a.pools, pool), row, row_mode, qs, G, s);
    // ---- online softmax per head over this step's 32 rows (log2 domain)
    float pr[GG];
#pragma unroll
    for (int h = 0; h < GG; ++h) {
      if (h < G) {
        const float sv = pool >= 0 ? s[h] : -INFINITY;
        float mx = sv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
        const float mn = fmaxf(m[h], mx);          // finite: the step has a row
        const float corr = m[h] == -INFINITY ? 0.f : exp2f(m[h] - mn);
        pr[h] = pool >= 0 ? exp2f(sv - mn) : 0.f;
        float sm = pr[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(kFull, sm, o);
        l[h] = l[h] * corr + sm;
        m[h] = mn;
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[h][c] *= corr;
      }
    }
    // ---- P V: lane = columns; the step's rows VB at a time, their loads
    // issued together; row j's pool and place come from lane j
#pragma unroll 1
    for (int j0 = 0; j0 < 32; j0 += VB) {
      if (base + j0 >= hi) break;                 // uniform across the warp
      float v[VB][NC];
#pragma unroll
      for (int k = 0; k < VB; ++k) {
        const int pk = __shfl_sync(kFull, pool, j0 + k);
        const int rk = __shfl_sync(kFull, rr, j0 + k);
#pragma unroll
        for (int c = 0; c < NC; ++c) v[k][c] = 0.f;
        if (pk >= 0)
          load_value_cols<D, BF>(pk, pool_ptrs(a.pools, pk), static_cast<int64_t>(u) * a.capacity + rk,
                                 lane, row_mode, v[k]);
      }
#pragma unroll
      for (int k = 0; k < VB; ++k) {
#pragma unroll
        for (int h = 0; h < GG; ++h) {
          if (h < G) {
            const float pj = __shfl_sync(kFull, pr[h], j0 + k);
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[h][c] = fmaf(pj, v[k][c], acc[h][c]);
          }
        }
      }
    }
  }

  // ---- merge the warps of the CTA (Eq. 15), then write out or publish
#pragma unroll
  for (int h = 0; h < GG; ++h) {
    if (h < G) {
      if (lane == 0) {
        wm[warp][h] = m[h];
        wl[warp][h] = l[h];
      }
#pragma unroll
      for (int c = 0; c < NC; ++c) wacc[warp][h][lane * NC + c] = acc[h][c];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int h = idx / D, col = idx % D;
    float v = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v = fmaxf(v, wm[w][h]);
    float num = 0.f, den = 0.f;
    if (v != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (wm[w][h] == -INFINITY) continue;       // a warp that saw no row
        const float f = exp2f(wm[w][h] - v);
        num += f * wacc[w][h][col];
        den += f * wl[w][h];
      }
    }
    if (a.splits == 1) {
      const float o = den > 0.f ? num / den : 0.f;
      a.out[(static_cast<int64_t>(u) * G + h) * D + col] = __float2bfloat16_rn(o);
    } else {
      const int64_t slot = (static_cast<int64_t>(u) * a.splits + split) * G + h;
      a.ws_acc[slot * D + col] = num;
      if (col == 0) {
        a.ws_ml[slot * 2] = v;
        a.ws_ml[slot * 2 + 1] = den;
      }
    }
  }
}

// bf16 pools only (token and page mode): each warp's 32 rows per step are
// contiguous in the pool, so bulk copies bring them into the warp's
// shared-memory buffers (the copy engine moves whole rows; no per-lane
// gathers reach L1): each lane copies one key row into a row padded by 16
// bytes, and one copy brings the 32 value rows.  Scores: lane = row, all
// lanes reading the same 16-byte chunk index (the padding puts them in
// different banks, and the query rows are read as broadcasts); P V: lane =
// d/32 columns.  Online softmax per warp and Eq. 15 merges as in
// decode_kernel.
template <int D, int GG>
__global__ void __launch_bounds__(kThreads, 3) decode_bulk_kernel(const DecodeArgs a) {
  constexpr int NC = D / 32;
  constexpr int ROWB = D * 2;                    // bytes per row
  constexpr int CH = ROWB / 16;                  // 16-byte chunks per row
  extern __shared__ __align__(128) uint8_t dsm[];
  constexpr int ROWP = ROWB + 16;                 // padded key row in shared memory
  uint8_t* kbuf0 = dsm;                          // [4 warps][32 rows][ROWP]
  uint8_t* vbuf0 = dsm + kWarps * 32 * ROWP;      // [4 warps][32 rows][ROWB]
  __shared__ __align__(16) float qs[GG][D];
  __shared__ float wm[kWarps][GG], wl[kWarps][GG];
  __shared__ float wacc[kWarps][GG][D];
  __shared__ __align__(8) uint64_t bars[kWarps];
  __shared__ int abort_i;

  const int u = blockIdx.x, split = blockIdx.y;
  const int G = a.G, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float cs = a.scale * kLog2e;
  if (tid < kWarps) mbar_init(smem_u32(&bars[tid]), 1);
  if (tid == 0) abort_i = 0;
  {
    const __nv_bfloat16* q = a.q + static_cast<int64_t>(u) * G * D;
    for (int idx = tid; idx < GG * D; idx += kThreads)
      qs[idx / D][idx % D] = idx / D < G ? __bfloat162float(q[idx]) * cs : 0.f;
  }
  fence_barrier_init();
  const int n = clamp_count(a.kept_count[KVC_POOL_BF16 * a.U + u], a.capacity);
  const int per = (n + a.splits - 1) / a.splits;
  const int lo = min(n, split * per), hi = min(n, lo + per);
  __syncthreads();
  volatile int* abort_flag = &abort_i;
  uint8_t* kb = kbuf0 + warp * 32 * ROWP;
  uint8_t* vb = vbuf0 + warp * 32 * ROWB;
  const uint32_t bar = smem_u32(&bars[warp]);
  const uint8_t* kg = static_cast<const uint8_t*>(a.pools.k_bf16) + static_cast<int64_t>(u) * a.capacity * ROWB;
  const uint8_t* vg = static_cast<const uint8_t*>(a.pools.v_bf16) + static_cast<int64_t>(u) * a.capacity * ROWB;

  float m[GG], l[GG], acc[GG][NC];
#pragma unroll
  for (int h = 0; h < GG; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[h][c] = 0.f;
  }
  uint32_t phase = 0;
  for (int base = lo + warp * 32; base < hi; base += kThreads) {
    const int nrow = min(32, hi - base);
    // key rows: one copy per lane into its padded row; value rows: one copy
    fence_proxy_async_smem();                     // the buffers' last reads precede the copies
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(2 * nrow * ROWB));
    __syncwarp();
    if (lane < nrow)
      bulk_copy_g2s(smem_u32(kb + lane * ROWP), kg + (static_cast<int64_t>(base) + lane) * ROWB, ROWB, bar);
    if (lane == 0) bulk_copy_g2s(smem_u32(vb), vg + static_cast<int64_t>(base) * ROWB, nrow * ROWB, bar);
    const bool ok = __all_sync(kFull, mbar_wait(bar, phase, abort_flag));
    if (!ok) {
      // a copy that did not land in time: wait for it (bounded) before leaving
      if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, phase) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
      __syncwarp();
      break;
    }
    phase ^= 1;
    // ---- scores: lane = row (rows >= nrow are masked)
    float s[GG];
#pragma unroll
    for (int h = 0; h < GG; ++h) s[h] = 0.f;
    const uint4* krow = reinterpret_cast<const uint4*>(kb + lane * ROWP);
#pragma unroll 4
    for (int v = 0; v < CH; ++v) {
      const int cidx = v;                       // the padding puts the lanes in different banks
      const uint4 w = krow[cidx];
      const uint32_t rw[4] = {w.x, w.y, w.z, w.w};
      float x[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(rw[k] << 16);
        x[2 * k + 1] = __uint_as_float(rw[k] & 0xffff0000u);
      }
      dot8<D, GG>(x, qs, cidx * 8, GG, s);
    }
    // ---- online softmax per head over this step's rows (log2 domain)
    const bool valid = lane < nrow;
    float pr[GG];
#pragma unroll
    for (int h = 0; h < GG; ++h) {
      const float sv = valid ? s[h] : -INFINITY;
      float mx = sv;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      const float mn = fmaxf(m[h], mx);
      const float corr = m[h] == -INFINITY ? 0.f : exp2f(m[h] - mn);
      pr[h] = valid ? exp2f(sv - mn) : 0.f;
      float sm = pr[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(kFull, sm, o);
      l[h] = l[h] * corr + sm;
      m[h] = mn;
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[h][c] *= corr;
    }
    // ---- P V: lane = columns, rows from shared memory
#pragma unroll 4
    for (int j = 0; j < nrow; ++j) {
      float vv[NC];
      if (NC == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(vb + j * ROWB + lane * 8);
        vv[0] = __uint_as_float(w.x << 16);
        vv[1] = __uint_as_float(w.x & 0xffff0000u);
        vv[2 % NC] = __uint_as_float(w.y << 16);
        vv[3 % NC] = __uint_as_float(w.y & 0xffff0000u);
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(vb + j * ROWB + lane * 4);
        vv[0] = __uint_as_float(w << 16);
        vv[1 % NC] = __uint_as_float(w & 0xffff0000u);
      }
#pragma unroll
      for (int h = 0; h < GG; ++h) {
        const float pj = __shfl_sync(kFull, pr[h], j);
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[h][c] = fmaf(pj, vv[c], acc[h][c]);
      }
    }
    __syncwarp();                                 // buffers free for the next copy
  }

  // ---- merge the warps of the CTA (Eq. 15), then write out or publish
#pragma unroll
  for (int h = 0; h < GG; ++h) {
    if (lane == 0) {
      wm[warp][h] = m[h];
      wl[warp][h] = l[h];
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) wacc[warp][h][lane * NC + c] = acc[h][c];
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int h = idx / D, col = idx % D;
    float v = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v = fmaxf(v, wm[w][h]);
    float num = 0.f, den = 0.f;
    if (v != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (wm[w][h] == -INFINITY) continue;
        const float f = exp2f(wm[w][h] - v);
        num += f * wacc[w][h][col];
        den += f * wl[w][h];
      }
    }
    if (a.splits == 1) {
      const float o = den > 0.f ? num / den : 0.f;
      a.out[(static_cast<int64_t>(u) * G + h) * D + col] = __float2bfloat16_rn(o);
    } else {
      const int64_t slot = (static_cast<int64_t>(u) * a.splits + split) * G + h;
      a.ws_acc[slot * D + col] = num;
      if (col == 0) {
        a.ws_ml[slot * 2] = v;
        a.ws_ml[slot * 2 + 1] = den;
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

cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t stream) {
  merge_kernel<<<dim3(a.U, a.G), 128, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const dim3 grid(a.U, a.splits);
  const bool bf = a.pool_lo == KVC_POOL_BF16;
  if (bf) {
    // bulk-staged kernel: 4 warps x 32 rows x (padded key row + value row) of dynamic shared memory
    const size_t smem = static_cast<size_t>(kWarps) * 32 * (a.d * 2 + 16 + a.d * 2);   // padded key rows + value rows
    const int g4 = a.G <= 1 ? 1 : a.G <= 2 ? 2 : a.G <= 4 ? 4 : 8;
    void (*k)(const DecodeArgs) = nullptr;
    if (a.d == 64) k = g4 == 1 ? decode_bulk_kernel<64, 1> : g4 == 2 ? decode_bulk_kernel<64, 2>
                     : g4 == 4 ? decode_bulk_kernel<64, 4> : decode_bulk_kernel<64, 8>;
    else k = g4 == 1 ? decode_bulk_kernel<128, 1> : g4 == 2 ? decode_bulk_kernel<128, 2>
           : g4 == 4 ? decode_bulk_kernel<128, 4> : decode_bulk_kernel<128, 8>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    k<<<grid, kThreads, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess || a.splits == 1) return e;
    merge_kernel<<<dim3(a.U, a.G), 128, 0, stream>>>(a);
    return cudaGetLastError();
  }
  const int gg = a.G <= 1 ? 1 : a.G <= 2 ? 2 : a.G <= 4 ? 4 : 8;
#define KVC_DECODE_LAUNCH(DD, GGV)                                                         \
  if (a.d == DD && gg == GGV) {                                                           \
    if (bf) decode_kernel<DD, GGV, true><<<grid, kThreads, 0, stream>>>(a);               \
    else decode_kernel<DD, GGV, false><<<grid, kThreads, 0, stream>>>(a);                 \
  }
  KVC_DECODE_LAUNCH(64, 1)
  KVC_DECODE_LAUNCH(64, 2)
  KVC_DECODE_LAUNCH(64, 4)
  KVC_DECODE_LAUNCH(64, 8)
  KVC_DECODE_LAUNCH(128, 1)
  KVC_DECODE_LAUNCH(128, 2)
  KVC_DECODE_LAUNCH(128, 4)
  KVC_DECODE_LAUNCH(128, 8)
#undef KVC_DECODE_LAUNCH
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || a.splits == 1) return err;
  merge_kernel<<<dim3(a.U, a.G), 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc
