// Window-attention scoring on the 5th-generation tensor cores (tcgen05).
//
// What it computes (PASK Eq. 1; the observation-window scorer of PASK
// App. C.3 / CommitKV Sec. 3.1; PACE Sec. 3.1 bonus): for every unit
// u = (b, l, g) and cached key j,
//   score[u][j] = sum_{h in g, w < W} exp(z_hwj - lse_hw) + bonus[b][j],
//   z_hwj = q_hw . k_j * scale over the keys row (h, w) sees causally.
//
// Design.  The R = W*G window rows of a unit against its T keys are one
// R x T x d contraction.  It is done twice per key tile, both times on
// tcgen05 with fp32 accumulators in tensor memory:
//   pass 1: D[row][token] = Q K^T  (M = 128 rows, N = 128 tokens); each
//           epilogue thread owns one row and keeps an online max / sum;
//   pass 2: D[token][row] = K Q^T  (M = 128 tokens, N = R rows); each
//           epilogue thread owns one token and sums exp(z - lse) over rows,
//           so neither pass needs a cross-thread reduction.
// A unit's T keys are split into work items of `chunk_tiles` 128-token
// tiles; one persistent CTA per SM walks the items round-robin.  After pass
// 1 of an item its row statistics are published and a per-unit counter is
// bumped; pass 2 starts once every item of the unit has published, so the
// log-sum-exp of each row is exact.  The items of a round cover a contiguous
// range of units, so the keys read by pass 1 are still in L2 for pass 2.
// Co-residency of all CTAs (needed by that wait) is guaranteed by launching
// cooperatively; every wait is bounded in time.
//
// Warp roles (12 warps): 0 = TMA producer, 1 = MMA issuer, 2 = TMEM owner,
// 3 = idle, 4..11 = epilogue (two warps per TMEM lane quarter).
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kChunkBytes = 128 * 128;   // 128 rows x 64 bf16 (one swizzle-128 K chunk)

struct Smem {
  uint8_t* q;           // n_kc chunks of q_rows x 128 B
  uint8_t* k;           // n_stages stages of n_kc chunks of 128 x 128 B
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;      // [2]
  uint64_t* tempty;     // [2]
  uint64_t* qfull;
  uint64_t* qempty;
  uint64_t* mmadone;
  uint32_t* tmem_slot;
  int* abort_flag;
  float* lam;           // [256]
  float* red;           // [128]
  float* hm;            // [128]
  float* hl;            // [128]
};

__device__ __forceinline__ Smem carve(uint8_t* base, int n_kc, int q_rows, int n_stages) {
  Smem s;
  s.q = base;
  s.k = base + n_kc * q_rows * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.k + n_stages * n_kc * kChunkBytes);
  s.full = bars;
  s.empty = bars + n_stages;
  s.tfull = bars + 2 * n_stages;
  s.tempty = bars + 2 * n_stages + 2;
  s.qfull = bars + 2 * n_stages + 4;
  s.qempty = bars + 2 * n_stages + 5;
  s.mmadone = bars + 2 * n_stages + 6;
  s.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * n_stages + 8);
  s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
  s.lam = reinterpret_cast<float*>(s.tmem_slot + 4);
  s.red = s.lam + 256;
  s.hm = s.red + 128;
  s.hl = s.hm + 128;
  return s;
}

// Wait that ignores the abort flag (used to drain work already in flight).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
score_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
             const ScoreArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int n_kc = a.d / 64;
  const Smem s = carve(base, n_kc, a.q_rows, a.n_stages);
  const uint32_t q_chunk_bytes = static_cast<uint32_t>(a.q_rows) * 128u;
  const uint32_t stage_bytes = static_cast<uint32_t>(n_kc) * kChunkBytes;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = s.abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.n_stages; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.tfull[i]), 1);
      mbar_init(smem_u32(&s.tempty[i]), kEpiThreads / 32);
    }
    mbar_init(smem_u32(s.qfull), 1);
    mbar_init(smem_u32(s.qempty), 1);
    mbar_init(smem_u32(s.mmadone), 1);
    *s.abort_flag = 0;
    fence_barrier_init();
  }
  // Q rows past R are read by the M = 128 row block of pass 1: keep them finite.
  {
    uint4* q4 = reinterpret_cast<uint4*>(s.q);
    const int n16 = n_kc * q_chunk_bytes / 16;
    for (int i = threadIdx.x; i < n16; i += kThreads) q4[i] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_q);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(s.tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s.tmem_slot;

  const int S = a.items_per_unit;
  const int n_rb = (a.R + 127) / 128;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t stream = l2_policy_evict_first();
      uint32_t jt = 0;
      int li = 0;
      int q_loads = 0;
      for (int it = blockIdx.x; it < a.n_items; it += gridDim.x, ++li) {
        const int u = it / S, c = it % S;
        const int t0 = c * a.chunk_tiles;
        const int nt = min(a.chunk_tiles, a.n_tiles - t0);
        if (li > 0 && !mbar_wait(smem_u32(s.qempty), (li - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(smem_u32(s.qfull), static_cast<uint32_t>(n_kc * a.R * 128));
        for (int kc = 0; kc < n_kc; ++kc)
          tma_load_3d(smem_u32(s.q + kc * q_chunk_bytes), &tmap_q, smem_u32(s.qfull), kc * 64, 0,
                      u, keep);
        ++q_loads;
        bool ok = true;
        for (int pass = 0; pass < 2 && ok; ++pass) {
          for (int t = 0; t < nt; ++t, ++jt) {
            const uint32_t st = jt % a.n_stages;
            const uint32_t ph = (jt / a.n_stages) & 1;
            if (!mbar_wait(smem_u32(&s.empty[st]), ph ^ 1, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(smem_u32(&s.full[st]), stage_bytes);
            for (int kc = 0; kc < n_kc; ++kc)
              tma_load_3d(smem_u32(s.k + st * stage_bytes + kc * kChunkBytes), &tmap_k,
                          smem_u32(&s.full[st]), kc * 64, (t0 + t) * kTileTokens, u,
                          pass == 0 ? keep : stream);
          }
        }
        if (!ok) break;
      }
      // Drain: every load this thread issued must land before the CTA exits.
      const uint32_t first = jt > static_cast<uint32_t>(a.n_stages) ? jt - a.n_stages : 0;
      for (uint32_t j = first; j < jt; ++j)
        mbar_drain(smem_u32(&s.full[j % a.n_stages]), (j / a.n_stages) & 1);
      if (q_loads > 0) mbar_drain(smem_u32(s.qfull), (q_loads - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc1 = mma_idesc_bf16(128, 128);
      const uint32_t idesc2 = mma_idesc_bf16(128, a.R);
      const uint32_t q_base = smem_u32(s.q);
      const int ksteps = a.d / 16;
      uint32_t jt = 0;
      int li = 0;
      for (int it = blockIdx.x; it < a.n_items; it += gridDim.x, ++li) {
        const int c = it % S;
        const int t0 = c * a.chunk_tiles;
        const int nt = min(a.chunk_tiles, a.n_tiles - t0);
        if (!mbar_wait(smem_u32(s.qfull), li & 1, abort_flag)) break;
        tc_fence_after();
        bool ok = true;
        for (int pass = 0; pass < 2 && ok; ++pass) {
          for (int t = 0; t < nt; ++t, ++jt) {
            const uint32_t st = jt % a.n_stages;
            const uint32_t ph = (jt / a.n_stages) & 1;
            const uint32_t tb = jt & 1;
            const uint32_t tph = (jt >> 1) & 1;
            if (!mbar_wait(smem_u32(&s.full[st]), ph, abort_flag) ||
                !mbar_wait(smem_u32(&s.tempty[tb]), tph ^ 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t k_base = smem_u32(s.k + st * stage_bytes);
            const uint32_t d_tmem = tmem_base + tb * 256;
            if (pass == 0) {
              for (int rb = 0; rb < n_rb; ++rb)
                for (int ks = 0; ks < ksteps; ++ks) {
                  const uint32_t kc = ks >> 2, kb = (ks & 3) * 32;
                  const uint64_t ad = sw128_desc(q_base + kc * q_chunk_bytes + rb * kChunkBytes + kb);
                  const uint64_t bd = sw128_desc(k_base + kc * kChunkBytes + kb);
                  tc_mma_bf16(d_tmem + rb * 128, ad, bd, idesc1, ks > 0);
                }
            } else {
              for (int ks = 0; ks < ksteps; ++ks) {
                const uint32_t kc = ks >> 2, kb = (ks & 3) * 32;
                const uint64_t ad = sw128_desc(k_base + kc * kChunkBytes + kb);
                const uint64_t bd = sw128_desc(q_base + kc * q_chunk_bytes + kb);
                tc_mma_bf16(d_tmem, ad, bd, idesc2, ks > 0);
              }
            }
            tc_commit(smem_u32(&s.empty[st]));
            tc_commit(smem_u32(&s.tfull[tb]));
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(s.qempty));
      }
      // All MMAs issued above must be complete before TMEM is released.
      tc_commit(smem_u32(s.mmadone));
      mbar_drain(smem_u32(s.mmadone), 0);
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    // Every named barrier below is an OR-reduction of a failure flag, and no
    // thread leaves the item loop between two of them, so a bounded wait
    // that gives up in one warp ends all epilogue warps at the same barrier.
    const int e = warp - kEpiWarp0;            // 0..7
    const int qr = warp & 3;                   // TMEM lane quarter of this warp
    const int hf = e >> 2;                     // which half of the columns
    const int et = threadIdx.x - kEpiWarp0 * 32;
    const uint32_t lane_addr = static_cast<uint32_t>(qr * 32) << 16;
    const float cs = a.scale_log2;
    const int64_t T = a.T;
    const int64_t Tq = T - a.W;                // row w sees keys j <= Tq + w
    const int n_cc = a.R / 32;
    const int cc_split = (n_cc + 1) / 2;
    const int cc_lo = hf ? cc_split : 0;
    const int cc_hi = hf ? n_cc : cc_split;
    // pass-1 geometry: which row this thread owns and which token columns
    const int row = (n_rb == 2) ? hf * 128 + qr * 32 + lane : qr * 32 + lane;
    const int tok_lo = (n_rb == 2) ? 0 : hf * 64;
    const int ntok = (n_rb == 2) ? 128 : 64;
    const int colbase = ((n_rb == 2) ? hf * 128 : 0) + tok_lo;
    const bool row_valid = row < a.R;
    const int64_t row_last = Tq + (row_valid ? row % a.W : 0);
    const bool stats_owner = ((n_rb == 2) || hf == 0) && row_valid;

    uint32_t jt = 0;
    bool fail = false;
    int cur_u = -1;
    for (int it = blockIdx.x; it < a.n_items; it += gridDim.x) {
      const int u = it / S, c = it % S;
      const int t0 = c * a.chunk_tiles;
      const int nt = min(a.chunk_tiles, a.n_tiles - t0);
      const int b = u / (a.L * a.Hkv);
      cur_u = u;

      // ---------------- pass 1: per-row online max / sum (log2 domain)
      float m = -INFINITY, l = 0.f;
      for (int t = 0; t < nt; ++t, ++jt) {
        const uint32_t tb = jt & 1, tph = (jt >> 1) & 1;
        if (fail || !mbar_wait(smem_u32(&s.tfull[tb]), tph, abort_flag)) {
          fail = true;
          continue;
        }
        tc_fence_after();
        const int64_t j0 = static_cast<int64_t>(t0 + t) * kTileTokens + tok_lo;
        const bool all_visible = (j0 + ntok - 1) <= Tq;
        for (int cc = 0; cc < ntok; cc += 32) {
          float v[32];
          tmem_ld32(tmem_base + lane_addr + tb * 256 + colbase + cc, v);
          if (!all_visible) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (j0 + cc + i > row_last) v[i] = -INFINITY;
          }
          float mx = v[0];
#pragma unroll
          for (int i = 1; i < 32; ++i) mx = fmaxf(mx, v[i]);
          const float mn = fmaxf(m, mx * cs);
          if (mn == -INFINITY) continue;
          float sum = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) sum += ex2_approx(fmaf(v[i], cs, -mn));
          l = l * ex2_approx(m - mn) + sum;
          m = mn;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.tempty[tb]));
      }
      if (n_rb == 1) {   // the two halves saw different token columns of the same row
        if (hf == 1) {
          s.hm[qr * 32 + lane] = m;
          s.hl[qr * 32 + lane] = l;
        }
        fail = named_bar_or(1, kEpiThreads, fail);
        if (hf == 0) {
          const float m2 = s.hm[qr * 32 + lane], l2 = s.hl[qr * 32 + lane];
          const float mn = fmaxf(m, m2);
          if (mn != -INFINITY) {
            l = l * ex2_approx(m - mn) + l2 * ex2_approx(m2 - mn);
            m = mn;
          }
        }
      }
      if (!fail && stats_owner)
        a.stats[(static_cast<size_t>(u) * S + c) * a.R + row] = make_float2(m, l);
      __threadfence();
      fail = named_bar_or(1, kEpiThreads, fail);
      if (fail) break;
      bool timed_out = false;
      if (et == 0) {
        atom_add_release_gpu(&a.counters[u], 1u);
        uint64_t t_start = 0;
        for (uint32_t n = 0;; ++n) {
          if (ld_acquire_gpu(&a.counters[u]) >= static_cast<uint32_t>(S)) break;
          if (*abort_flag) {
            timed_out = true;
            break;
          }
          if ((n & 63) == 0) {
            const uint64_t now = globaltimer_ns();
            if (t_start == 0) {
              t_start = now;
            } else if (now - t_start > kWaitLimitNs) {
              *abort_flag = 1;
              timed_out = true;
              break;
            }
          }
          __nanosleep(32);
        }
      }
      fail = named_bar_or(1, kEpiThreads, timed_out);
      if (fail) break;
      // log-sum-exp of every row over the whole unit
      for (int r = et; r < a.R; r += kEpiThreads) {
        float M = -INFINITY, Ls = 0.f;
        for (int cc = 0; cc < S; ++cc) {
          const float2 st = __ldcg(&a.stats[(static_cast<size_t>(u) * S + cc) * a.R + r]);
          if (st.x == -INFINITY) continue;
          if (st.x > M) {
            Ls = Ls * ex2_approx(M - st.x) + st.y;
            M = st.x;
          } else {
            Ls += st.y * ex2_approx(st.x - M);
          }
        }
        s.lam[r] = M + __log2f(Ls);
      }
      named_bar_sync(1, kEpiThreads);

      // ---------------- pass 2: per-token sum of exp2(z cs - lse) over rows
      for (int t = 0; t < nt; ++t, ++jt) {
        const uint32_t tb = jt & 1, tph = (jt >> 1) & 1;
        const int64_t tile0 = static_cast<int64_t>(t0 + t) * kTileTokens;
        const int64_t j = tile0 + qr * 32 + lane;
        float acc = 0.f;
        if (!fail && mbar_wait(smem_u32(&s.tfull[tb]), tph, abort_flag)) {
          tc_fence_after();
          const bool all_visible = (tile0 + kTileTokens - 1) <= Tq;
          for (int cc = cc_lo; cc < cc_hi; ++cc) {
            float v[32];
            tmem_ld32(tmem_base + lane_addr + tb * 256 + cc * 32, v);
            if (all_visible) {
#pragma unroll
              for (int i = 0; i < 32; ++i) acc += ex2_approx(fmaf(v[i], cs, -s.lam[cc * 32 + i]));
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int r = cc * 32 + i;
                const bool vis = j <= Tq + (r % a.W);
                acc += vis ? ex2_approx(fmaf(v[i], cs, -s.lam[r])) : 0.f;
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&s.tempty[tb]));
        } else {
          fail = true;
        }
        if (hf == 1) s.red[qr * 32 + lane] = acc;
        fail = named_bar_or(1, kEpiThreads, fail);
        if (fail) break;
        if (hf == 0) {
          acc += s.red[qr * 32 + lane];
          float sc = -INFINITY;
          if (j < T) {
            sc = acc;
            if (a.bonus) sc += a.bonus[static_cast<int64_t>(b) * T + j];
            float* dst = a.scores + static_cast<int64_t>(u) * T + j;
            if (a.accumulate) sc += *dst;
            *dst = sc;
          }
          const int P = a.page_size;
          if (P > 1) {
            float pm = sc;
            for (int o = 1; o < P; o <<= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o));
            if (j < T && (lane & (P - 1)) == 0)
              a.page_scores[static_cast<int64_t>(u) * (T / P) + j / P] = pm;
          }
        }
        named_bar_sync(1, kEpiThreads);
      }
      if (fail) break;
    }
    if (fail && et == 0 && cur_u >= 0 && a.unit_status) a.unit_status[cur_u] = KVC_UNIT_TIMEOUT;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

size_t score_smem_bytes(int d, int q_rows, int n_stages) {
  const int n_kc = d / 64;
  size_t bytes = 1024;                                   // alignment slack
  bytes += static_cast<size_t>(n_kc) * q_rows * 128;     // Q
  bytes += static_cast<size_t>(n_stages) * n_kc * kChunkBytes;
  bytes += (2 * n_stages + 8) * 8;                       // barriers
  bytes += 16;                                           // tmem slot, abort flag
  bytes += (256 + 3 * 128) * 4;                          // lam, red, hm, hl
  return bytes;
}

cudaError_t launch_score(const ScoreArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_q,
                         int grid, size_t smem_bytes, cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, score_kernel, tmap_k, tmap_q, a);
}

}  // namespace kvc
