// The engine's attention over persistent, recent and current storage.
//
// PASK App. B.5 ("Packed attention and quantization"): the kernel reads the
// disjoint high / low maps of the persistent storage (here the bf16, int8
// and int4 pools of a compaction pass, dequantised inline as code * scale),
// the recent storage and the current KV (bf16 rows), with logical positions:
// a key at position p_k is visible to a query at position p_q iff
// p_k <= p_q, whatever storage holds it, so positions and the causal mask
// survive the gaps between storages.  Query heads map to their KV head (one
// head, GQA-2, GQA-4, GQA-8); a unit's rows are split across CTAs (split-KV)
// and every partition is merged with Eq. 15.  Scores, softmax statistics and
// value sums are fp32; the output is bf16.
//
// Work layout: one unit per blockIdx.x, a split of the unit's rows (the
// storages concatenated: int4, int8, bf16 pools, recent, current) per
// blockIdx.y.  A warp takes 32 consecutive rows per step; for the scores each
// lane owns one key row (16-byte loads, the unit's query rows in shared
// memory as broadcasts) and applies the causal test of every query row; for
// P V each lane owns d / 32 columns and the step's probabilities arrive by
// shuffles.  Each warp keeps an online (max, sum, value sum) per query row;
// the warps, then the splits, are merged with Eq. 15.
#include <limits.h>
#include <math.h>

#include "decode_rows.cuh"
#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kEngThreads = 128;
constexpr int kEngWarps = kEngThreads / 32;
constexpr unsigned kAll = 0xffffffffu;
constexpr int kClasses = KVC_N_POOLS + 2;     // pools, recent, current

struct RowRef {
  PoolPtrs pp;
  int kind;          // KVC_POOL_* of the row's encoding
  int64_t row;       // row index in the storage's arrays
  const int32_t* pos;
};

__device__ __forceinline__ RowRef row_ref(const DecodeArgs& a, int u, int cls, int rr) {
  RowRef r;
  if (cls < KVC_N_POOLS) {
    r.pp = pool_ptrs(a.pools, cls);
    r.kind = cls;
    r.row = static_cast<int64_t>(u) * a.capacity + rr;
    r.pos = a.pool_pos ? a.pool_pos + (static_cast<int64_t>(cls) * a.U + u) * a.capacity + rr : nullptr;
  } else if (cls == KVC_N_POOLS) {
    r.pp = {a.rec_k, a.rec_v, nullptr, nullptr};
    r.kind = KVC_POOL_BF16;
    r.row = static_cast<int64_t>(u) * a.rec_cap + rr;
    r.pos = a.rec_pos ? a.rec_pos + r.row : nullptr;
  } else {
    r.pp = {a.cur_k, a.cur_v, nullptr, nullptr};
    r.kind = KVC_POOL_BF16;
    r.row = static_cast<int64_t>(u) * a.cur_cap + rr;
    r.pos = a.cur_pos ? a.cur_pos + r.row : nullptr;
  }
  return r;
}

// RR: query rows per unit (G heads x n_q queries) rounded up to 1, 2, 4, 8
// or 16; BF: every storage holds bf16 rows (the int8 / int4 paths are not
// compiled in).
template <int D, int RR, bool BF>
__global__ void __launch_bounds__(kEngThreads, RR >= 8 ? 2 : (RR >= 4 ? 3 : 4))
engine_attn_kernel(const DecodeArgs a) {
  constexpr int NC = D / 32;
  constexpr int VB = RR >= 16 ? 4 : (RR >= 8 ? 8 : 16);   // value rows in flight together
  __shared__ __align__(16) float qs[RR][D];
  __shared__ int qp[RR];
  __shared__ float wm[kEngWarps][RR], wl[kEngWarps][RR];
  __shared__ float wacc[kEngWarps][RR][D];

  const int u = blockIdx.x, split = blockIdx.y;
  const int R = a.G, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = u / (a.L * a.Hkv);
  const bool row_mode = a.quant_mode == KVC_QUANT_ROW_FP16;
  const float cs = a.scale * 1.4426950408889634f;
  {
    const __nv_bfloat16* q = a.q + static_cast<int64_t>(u) * R * D;
    for (int idx = tid; idx < RR * D; idx += kEngThreads)
      qs[idx / D][idx % D] = idx / D < R ? __bfloat162float(q[idx]) * cs : 0.f;
    if (tid < RR)
      qp[tid] = (tid < R && a.q_pos) ? a.q_pos[static_cast<int64_t>(b) * a.n_q + tid % a.n_q] : INT_MAX;
  }
  int cnt[kClasses];
  int n = 0;
#pragma unroll
  for (int c = 0; c < kClasses; ++c) {
    int v = 0;
    // counts outside [0, capacity] are clamped, so no row past a storage is read
    if (c < KVC_N_POOLS)
      v = (a.has_pools && c >= a.pool_lo && c < a.pool_hi) ? clamp_count(a.kept_count[c * a.U + u], a.capacity) : 0;
    else if (c == KVC_N_POOLS) v = a.rec_count ? clamp_count(a.rec_count[u], a.rec_cap) : 0;
    else v = a.cur_count ? clamp_count(a.cur_count[u], a.cur_cap) : 0;
    cnt[c] = v;
    n += v;
  }
  const int per = (n + a.splits - 1) / a.splits;
  const int lo = min(n, split * per), hi = min(n, lo + per);
  __syncthreads();

  float m[RR], l[RR], acc[RR][NC];
#pragma unroll
  for (int h = 0; h < RR; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[h][c] = 0.f;
  }

  for (int base = lo + warp * 32; base < hi; base += kEngThreads) {
    // ---- scores: lane = row; the row's storage class and index
    const int r = base + lane;
    int cls = -1, rr = r;
    if (r < hi) {
#pragma unroll
      for (int c = 0; c < kClasses; ++c) {
        if (cls < 0) {
          if (rr < cnt[c]) cls = c;
          else rr -= cnt[c];
        }
      }
    }
    float s[RR];
#pragma unroll
    for (int h = 0; h < RR; ++h) s[h] = 0.f;
    int kp = INT_MIN;
    if (cls >= 0) {
      const RowRef ref = row_ref(a, u, cls, rr);
      if (ref.pos) kp = __ldg(ref.pos);
      key_dot<D, RR, BF>(ref.kind, ref.pp, ref.row, row_mode, qs, R, s);
    }
    // ---- online softmax per query row over this step's visible keys (log2 domain)
    float pr[RR];
#pragma unroll
    for (int h = 0; h < RR; ++h) {
      pr[h] = 0.f;
      if (h < R) {
        const bool vis = cls >= 0 && kp <= qp[h];
        const float sv = vis ? s[h] : -INFINITY;
        float mx = sv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, o));
        const float mn = fmaxf(m[h], mx);
        if (mn != -INFINITY) {                     // uniform: some key so far is visible to row h
          const float corr = m[h] == -INFINITY ? 0.f : exp2f(m[h] - mn);
          pr[h] = vis ? exp2f(sv - mn) : 0.f;
          float sm = pr[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(kAll, sm, o);
          l[h] = l[h] * corr + sm;
          m[h] = mn;
#pragma unroll
          for (int c = 0; c < NC; ++c) acc[h][c] *= corr;
        }
      }
    }
    // ---- P V: lane = columns; VB rows' loads issued together; row j's
    // storage and index come from lane j
#pragma unroll 1
    for (int j0 = 0; j0 < 32; j0 += VB) {
      if (base + j0 >= hi) break;                  // uniform across the warp
      float v[VB][NC];
#pragma unroll
      for (int k = 0; k < VB; ++k) {
        const int ck = __shfl_sync(kAll, cls, j0 + k);
        const int rk = __shfl_sync(kAll, rr, j0 + k);
#pragma unroll
        for (int c = 0; c < NC; ++c) v[k][c] = 0.f;
        if (ck >= 0) {
          const RowRef ref = row_ref(a, u, ck, rk);
          load_value_cols<D, BF>(ref.kind, ref.pp, ref.row, lane, row_mode, v[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < VB; ++k) {
#pragma unroll
        for (int h = 0; h < RR; ++h) {
          if (h < R) {
            const float pj = __shfl_sync(kAll, pr[h], j0 + k);
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[h][c] = fmaf(pj, v[k][c], acc[h][c]);
          }
        }
      }
    }
  }

  // ---- merge the warps of the CTA (Eq. 15), then write out or publish
#pragma unroll
  for (int h = 0; h < RR; ++h) {
    if (h < R) {
      if (lane == 0) {
        wm[warp][h] = m[h];
        wl[warp][h] = l[h];
      }
#pragma unroll
      for (int c = 0; c < NC; ++c) wacc[warp][h][lane * NC + c] = acc[h][c];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < R * D; idx += kEngThreads) {
    const int h = idx / D, col = idx % D;
    float v = -INFINITY;
#pragma unroll
    for (int w = 0; w < kEngWarps; ++w) v = fmaxf(v, wm[w][h]);
    float num = 0.f, den = 0.f;
    if (v != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kEngWarps; ++w) {
        if (wm[w][h] == -INFINITY) continue;       // a warp that saw no visible key
        const float f = exp2f(wm[w][h] - v);
        num += f * wacc[w][h][col];
        den += f * wl[w][h];
      }
    }
    if (a.splits == 1) {
      const float o = den > 0.f ? num / den : 0.f;  // a row that sees no key outputs 0
      a.out[(static_cast<int64_t>(u) * R + h) * D + col] = __float2bfloat16_rn(o);
    } else {
      const int64_t slot = (static_cast<int64_t>(u) * a.splits + split) * R + h;
      a.ws_acc[slot * D + col] = num;
      if (col == 0) {
        a.ws_ml[slot * 2] = v;
        a.ws_ml[slot * 2 + 1] = den;
      }
    }
  }
}

// bf16 storages only (token / page mode pools, recent, current): the split's
// rows are walked storage by storage, and each warp step's 32 rows (all in
// one storage, so contiguous) reach the warp's shared-memory buffers by bulk
// copies: each lane copies one key row into a row padded by 16 bytes, one
// copy brings the value rows.  Scores: lane = row, all lanes reading the same
// 16-byte chunk index (the padding puts them in different banks, the query
// rows are read as broadcasts); P V: lane = d / 32 columns.  The buffers hold
// the warps' partial results for the final merge.
template <int D, int RR>
__global__ void __launch_bounds__(kEngThreads, RR >= 16 ? 2 : 3) engine_bulk_kernel(const DecodeArgs a) {
  constexpr int NC = D / 32;
  constexpr int ROWB = D * 2;
  constexpr int CH = ROWB / 16;
  extern __shared__ __align__(128) uint8_t esm[];
  constexpr int ROWP = ROWB + 16;                 // padded key row in shared memory
  uint8_t* kbuf0 = esm;                          // [4 warps][32 rows][ROWP]
  uint8_t* vbuf0 = esm + kEngWarps * 32 * ROWP;  // [4 warps][32 rows][ROWB]
  __shared__ __align__(16) float qs[RR][D];
  __shared__ int qp[RR];
  __shared__ float wm[kEngWarps][RR], wl[kEngWarps][RR];
  __shared__ __align__(8) uint64_t bars[kEngWarps];
  __shared__ int abort_i;

  const int u = blockIdx.x, split = blockIdx.y;
  const int R = a.G, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = u / (a.L * a.Hkv);
  const float cs = a.scale * 1.4426950408889634f;
  if (tid < kEngWarps) mbar_init(smem_u32(&bars[tid]), 1);
  if (tid == 0) abort_i = 0;
  {
    const __nv_bfloat16* q = a.q + static_cast<int64_t>(u) * R * D;
    for (int idx = tid; idx < RR * D; idx += kEngThreads)
      qs[idx / D][idx % D] = idx / D < R ? __bfloat162float(q[idx]) * cs : 0.f;
    if (tid < RR)
      qp[tid] = (tid < R && a.q_pos) ? a.q_pos[static_cast<int64_t>(b) * a.n_q + tid % a.n_q] : INT_MAX;
  }
  fence_barrier_init();
  int cnt[3];
  // counts outside [0, capacity] are clamped, so no row past a storage is read
  cnt[0] = a.has_pools ? clamp_count(a.kept_count[KVC_POOL_BF16 * a.U + u], a.capacity) : 0;
  cnt[1] = a.rec_count ? clamp_count(a.rec_count[u], a.rec_cap) : 0;
  cnt[2] = a.cur_count ? clamp_count(a.cur_count[u], a.cur_cap) : 0;
  const int n = cnt[0] + cnt[1] + cnt[2];
  const int per = (n + a.splits - 1) / a.splits;
  const int lo = min(n, split * per), hi = min(n, lo + per);
  __syncthreads();
  volatile int* abort_flag = &abort_i;
  uint8_t* kb = kbuf0 + warp * 32 * ROWP;
  uint8_t* vb = vbuf0 + warp * 32 * ROWB;
  const uint32_t bar = smem_u32(&bars[warp]);

  float m[RR], l[RR], acc[RR][NC];
#pragma unroll
  for (int h = 0; h < RR; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[h][c] = 0.f;
  }
  uint32_t phase = 0;
  bool stop = false;
  int off = 0;                                    // first concatenated row of storage c
#pragma unroll 1
  for (int c = 0; c < 3 && !stop; off += cnt[c], ++c) {
    const int s0 = max(lo, off) - off, s1 = min(hi, off + cnt[c]) - off;   // rows of storage c here
    if (s1 <= s0) continue;
    const uint8_t* kg;
    const uint8_t* vg;
    const int32_t* pg;
    if (c == 0) {
      const int64_t r0 = static_cast<int64_t>(u) * a.capacity;
      kg = static_cast<const uint8_t*>(a.pools.k_bf16) + r0 * ROWB;
      vg = static_cast<const uint8_t*>(a.pools.v_bf16) + r0 * ROWB;
      pg = a.pool_pos ? a.pool_pos + (static_cast<int64_t>(KVC_POOL_BF16) * a.U + u) * a.capacity : nullptr;
    } else if (c == 1) {
      const int64_t r0 = static_cast<int64_t>(u) * a.rec_cap;
      kg = reinterpret_cast<const uint8_t*>(a.rec_k) + r0 * ROWB;
      vg = reinterpret_cast<const uint8_t*>(a.rec_v) + r0 * ROWB;
      pg = a.rec_pos ? a.rec_pos + r0 : nullptr;
    } else {
      const int64_t r0 = static_cast<int64_t>(u) * a.cur_cap;
      kg = reinterpret_cast<const uint8_t*>(a.cur_k) + r0 * ROWB;
      vg = reinterpret_cast<const uint8_t*>(a.cur_v) + r0 * ROWB;
      pg = a.cur_pos ? a.cur_pos + r0 : nullptr;
    }
#pragma unroll 1
    for (int base = s0 + warp * 32; base < s1; base += kEngThreads) {
      const int nrow = min(32, s1 - base);
      // key rows: one copy per lane into its padded row; value rows: one copy
      fence_proxy_async_smem();                     // the buffers' last reads precede the copies
      if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(2 * nrow * ROWB));
      __syncwarp();
      if (lane < nrow)
        bulk_copy_g2s(smem_u32(kb + lane * ROWP), kg + (static_cast<int64_t>(base) + lane) * ROWB, ROWB, bar);
      if (lane == 0) bulk_copy_g2s(smem_u32(vb), vg + static_cast<int64_t>(base) * ROWB, nrow * ROWB, bar);
      const bool valid = lane < nrow;
      const int kp = (valid && pg) ? __ldg(pg + base + lane) : INT_MIN;
      const bool ok = __all_sync(kAll, mbar_wait(bar, phase, abort_flag));
      if (!ok) {
        // a copy that did not land in time: wait for it (bounded) before leaving
        if (lane == 0) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar, phase) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
        __syncwarp();
        stop = true;
        break;
      }
      phase ^= 1;
      // ---- scores: lane = row
      float s[RR];
#pragma unroll
      for (int h = 0; h < RR; ++h) s[h] = 0.f;
      const uint4* krow = reinterpret_cast<const uint4*>(kb + lane * ROWP);
#pragma unroll 4
      for (int v = 0; v < CH; ++v) {
        const int cidx = v;                     // the padding puts the lanes in different banks
        const uint4 w = krow[cidx];
        const uint32_t rw[4] = {w.x, w.y, w.z, w.w};
        float x[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[2 * k] = __uint_as_float(rw[k] << 16);
          x[2 * k + 1] = __uint_as_float(rw[k] & 0xffff0000u);
        }
        dot8<D, RR>(x, qs, cidx * 8, RR, s);
      }
      // ---- online softmax per query row over this step's visible keys
      float pr[RR];
#pragma unroll
      for (int h = 0; h < RR; ++h) {
        pr[h] = 0.f;
        const bool vis = valid && kp <= qp[h];
        const float sv = vis ? s[h] : -INFINITY;
        float mx = sv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, o));
        const float mn = fmaxf(m[h], mx);
        if (mn != -INFINITY) {                    // uniform across the warp
          const float corr = m[h] == -INFINITY ? 0.f : exp2f(m[h] - mn);
          pr[h] = vis ? exp2f(sv - mn) : 0.f;
          float sm = pr[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(kAll, sm, o);
          l[h] = l[h] * corr + sm;
          m[h] = mn;
#pragma unroll
          for (int cc = 0; cc < NC; ++cc) acc[h][cc] *= corr;
        }
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
        for (int h = 0; h < RR; ++h) {
          const float pj = __shfl_sync(kAll, pr[h], j);
#pragma unroll
          for (int cc = 0; cc < NC; ++cc) acc[h][cc] = fmaf(pj, vv[cc], acc[h][cc]);
        }
      }
      __syncwarp();                               // buffers free for the next copy
    }
  }

  // ---- merge the warps (Eq. 15); the copy buffers hold the warps' value sums
  __syncthreads();
  float* wacc = reinterpret_cast<float*>(esm);   // [4 warps][RR][D]
#pragma unroll
  for (int h = 0; h < RR; ++h) {
    if (lane == 0) {
      wm[warp][h] = m[h];
      wl[warp][h] = l[h];
    }
#pragma unroll
    for (int cc = 0; cc < NC; ++cc) wacc[(warp * RR + h) * D + lane * NC + cc] = acc[h][cc];
  }
  __syncthreads();
  for (int idx = tid; idx < R * D; idx += kEngThreads) {
    const int h = idx / D, col = idx % D;
    float v = -INFINITY;
#pragma unroll
    for (int w = 0; w < kEngWarps; ++w) v = fmaxf(v, wm[w][h]);
    float num = 0.f, den = 0.f;
    if (v != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kEngWarps; ++w) {
        if (wm[w][h] == -INFINITY) continue;
        const float f = exp2f(wm[w][h] - v);
        num += f * wacc[(w * RR + h) * D + col];
        den += f * wl[w][h];
      }
    }
    if (a.splits == 1) {
      const float o = den > 0.f ? num / den : 0.f;
      a.out[(static_cast<int64_t>(u) * R + h) * D + col] = __float2bfloat16_rn(o);
    } else {
      const int64_t slot = (static_cast<int64_t>(u) * a.splits + split) * R + h;
      a.ws_acc[slot * D + col] = num;
      if (col == 0) {
        a.ws_ml[slot * 2] = v;
        a.ws_ml[slot * 2 + 1] = den;
      }
    }
  }
}

}  // namespace

cudaError_t launch_engine(const DecodeArgs& a, cudaStream_t stream) {
  const dim3 grid(a.U, a.splits);
  const bool bf = !a.has_pools || a.pool_lo == KVC_POOL_BF16;
  const int rr = a.G <= 1 ? 1 : a.G <= 2 ? 2 : a.G <= 4 ? 4 : a.G <= 8 ? 8 : 16;
  if (bf) {
    // bulk-staged kernel: 4 warps x 32 rows x (padded key row + value row) of dynamic shared memory
    const size_t smem = static_cast<size_t>(kEngWarps) * 32 * (a.d * 2 + 16 + a.d * 2);   // padded key rows + value rows
    void (*k)(const DecodeArgs) = nullptr;
    if (a.d == 64)
      k = rr == 1 ? engine_bulk_kernel<64, 1> : rr == 2 ? engine_bulk_kernel<64, 2> : rr == 4 ? engine_bulk_kernel<64, 4>
        : rr == 8 ? engine_bulk_kernel<64, 8> : engine_bulk_kernel<64, 16>;
    else
      k = rr == 1 ? engine_bulk_kernel<128, 1> : rr == 2 ? engine_bulk_kernel<128, 2> : rr == 4 ? engine_bulk_kernel<128, 4>
        : rr == 8 ? engine_bulk_kernel<128, 8> : engine_bulk_kernel<128, 16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    k<<<grid, kEngThreads, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess || a.splits == 1) return e;
    return launch_decode_merge(a, stream);
  }
#define KVC_ENGINE_LAUNCH(DD, RRV)                                                          \
  if (a.d == DD && rr == RRV) {                                                            \
    engine_attn_kernel<DD, RRV, false><<<grid, kEngThreads, 0, stream>>>(a);               \
  }
  KVC_ENGINE_LAUNCH(64, 1)
  KVC_ENGINE_LAUNCH(64, 2)
  KVC_ENGINE_LAUNCH(64, 4)
  KVC_ENGINE_LAUNCH(64, 8)
  KVC_ENGINE_LAUNCH(64, 16)
  KVC_ENGINE_LAUNCH(128, 1)
  KVC_ENGINE_LAUNCH(128, 2)
  KVC_ENGINE_LAUNCH(128, 4)
  KVC_ENGINE_LAUNCH(128, 8)
  KVC_ENGINE_LAUNCH(128, 16)
#undef KVC_ENGINE_LAUNCH
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || a.splits == 1) return err;
  return launch_decode_merge(a, stream);
}

}  // namespace kvc
