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
// tiles (the host picks the size: few, large items when there are enough
// units, since every item carries a fixed cost); one persistent CTA per SM
// walks the items round-robin.  After pass 1 of an item its row statistics
// are published and a per-unit counter is bumped; pass 2 starts once every
// item of the unit has published, so the log-sum-exp of each row is exact.
// When the items of a round are small their keys are still in L2 for pass
// 2; whole-unit items read them from HBM again.
// Co-residency of all CTAs (needed by that wait) is guaranteed by launching
// cooperatively; every wait is bounded in time.
//
// Warp roles (18 warps): 0 = TMA producer, 1 = TMEM owner and MMA issuer,
// 2..17 = epilogue, four warpgroups that each cover the four TMEM lane
// quarters (warp w reads lanes 32 (w % 4) .. 32 (w % 4) + 31).  All four
// warpgroups work on every tile, each on a quarter of its columns, while the
// MMA warp fills the other TMEM buffer; every SM sub-partition runs four
// epilogue warps.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kThreads = 576;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiThreads = 512;
constexpr uint32_t kTmemCols = 512;
constexpr int kChunkBytes = 128 * 128;   // 128 rows x 64 bf16 (one swizzle-128 K chunk)
// Sleep between failed barrier tests of the producer and MMA threads, so
// their waits do not take issue slots from the epilogue warps.
constexpr uint32_t kProducerSleepNs = 256;
constexpr uint32_t kMmaSleepNs = 32;

struct Smem {
  uint8_t* q;           // n_kc chunks of q_rows x 128 B
  uint8_t* k;           // n_stages stages of n_kc chunks of 128 x 128 B
  uint8_t* ones;        // 128 x 16 bf16 ones, 32-byte swizzled rows (pass-2 extra K step)
  uint8_t* aug;         // q_rows x 16 bf16: -lse / scale as three parts per window row
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;      // [2]
  uint64_t* tempty;     // [2]
  uint64_t* qfull;
  uint64_t* qempty;
  uint64_t* mmadone;
  uint64_t* redfull;    // [4 slots][4 TMEM lane quarters]
  uint64_t* augfull;    // the item's aug rows are written
  uint32_t* tmem_slot;
  int* abort_flag;
  float* lam;           // [256] negated log-sum-exp of each window row
  float* red;           // [4 slots][4 groups][128] pass-2 partial sums
  float* hm;            // [4 groups][128] pass-1 partial max (+ spare)
  float* hl;            // [4 groups][128] pass-1 partial sum (+ spare)
};

__device__ __forceinline__ Smem carve(uint8_t* base, int n_kc, int q_rows, int n_stages) {
  Smem s;
  s.q = base;
  s.k = base + n_kc * q_rows * 128;
  s.ones = s.k + n_stages * n_kc * kChunkBytes;
  s.aug = s.ones + 128 * 32;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.aug + q_rows * 32);
  s.full = bars;
  s.empty = bars + n_stages;
  s.tfull = bars + 2 * n_stages;
  s.tempty = bars + 2 * n_stages + 2;
  s.qfull = bars + 2 * n_stages + 4;
  s.qempty = bars + 2 * n_stages + 5;
  s.mmadone = bars + 2 * n_stages + 6;
  s.redfull = bars + 2 * n_stages + 8;
  s.augfull = bars + 2 * n_stages + 24;
  s.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * n_stages + 26);
  s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
  s.lam = reinterpret_cast<float*>(s.tmem_slot + 4);
  s.red = s.lam + 256;
  s.hm = s.red + 2048;
  s.hl = s.hm + 1024;
  return s;
}

// First tile of slice c of a unit: the n_tiles tiles are split into S
// slices whose sizes differ by at most one.
__device__ __forceinline__ int slice_begin(const ScoreArgs& a, int c) {
  return static_cast<int>((static_cast<int64_t>(c) * a.n_tiles) / a.items_per_unit);
}

// Wait that ignores the abort flag (used to drain work already in flight).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Online max / sum update of one window row with N more raw logits
// (pass 1, log2 domain: y = z * cs).  Masked logits are -inf.  Pairs of
// logits go through packed two-lane fp32 multiply-add / add instructions.
template <int N>
__device__ __forceinline__ void row_update(const uint32_t (&r)[N], float cs, bool masked,
                                           int64_t j0, int64_t last, float& m, float& l) {
  float v[N];
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
  if (masked) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (j0 + i > last) v[i] = -INFINITY;
  }
  float mx[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) mx[k] = fmaxf(v[k], v[k + 8]);
#pragma unroll
  for (int i = 16; i < N; i += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], v[i + k], v[i + 8 + k]);
  const float mc = fmaxf(fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), mx[6]), mx[7]) * cs;
  if (mc > m) {
    l *= ex2_approx(m - mc);
    m = mc;
  }
  if (m == -INFINITY) return;
  const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(-m, -m);
  float2 s2[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x = __ffma2_rn(make_float2(v[2 * k], v[2 * k + 1]), cs2, nm2);
    s2[k] = make_float2(ex2_approx(x.x), ex2_approx(x.y));
  }
#pragma unroll
  for (int i = 8; i < N; i += 2) {
    const float2 x = __ffma2_rn(make_float2(v[i], v[i + 1]), cs2, nm2);
    s2[(i >> 1) & 3] = __fadd2_rn(s2[(i >> 1) & 3], make_float2(ex2_approx(x.x), ex2_approx(x.y)));
  }
  const float2 u2 = __fadd2_rn(__fadd2_rn(s2[0], s2[1]), __fadd2_rn(s2[2], s2[3]));
  l += u2.x + u2.y;
}

// Sum of exp2(y - m) over N raw logits y = z * cs of one row against a
// fixed reference m (pass 1 after the row's first tile): the row's running
// reference is not raised for every tile, which saves the 64-way maximum.
// Terms may exceed 1; the caller redoes the tile with its exact maximum if
// the sum leaves the range where fp32 keeps it safely (above 2^100).
template <int N>
__device__ __forceinline__ float exp_sum(const uint32_t (&r)[N], float cs, float m) {
  const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(-m, -m);
  float2 s2[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1])),
                                cs2, nm2);
    s2[k] = make_float2(ex2_approx(x.x), ex2_approx(x.y));
  }
#pragma unroll
  for (int i = 8; i < N; i += 2) {
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), cs2,
                                nm2);
    s2[(i >> 1) & 3] = __fadd2_rn(s2[(i >> 1) & 3], make_float2(ex2_approx(x.x), ex2_approx(x.y)));
  }
  const float2 u2 = __fadd2_rn(__fadd2_rn(s2[0], s2[1]), __fadd2_rn(s2[2], s2[3]));
  return u2.x + u2.y;
}

// Pass 2: add exp2(y) of N rows to the token's mass (four packed pairs of
// running sums), y = D * cs where the accumulator D = z - lse_r / cs
// already holds the row's log-sum-exp (the extra K step of the MMA).
template <int N>
__device__ __forceinline__ void mass_accum(const uint32_t (&r)[N], float cs, float2 (&acc)[4]) {
  const float2 cs2 = make_float2(cs, cs);
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    const float2 x = __fmul2_rn(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), cs2);
    const float2 y = __fmul2_rn(make_float2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])), cs2);
    const int k = (i >> 2) & 1;
    acc[2 * k] = __fadd2_rn(acc[2 * k], make_float2(ex2_approx(x.x), ex2_approx(x.y)));
    acc[2 * k + 1] = __fadd2_rn(acc[2 * k + 1], make_float2(ex2_approx(y.x), ex2_approx(y.y)));
  }
}

// Same with the causal mask of the last tiles: row r0 + i sees token j iff
// j <= Tq + (r0 + i) mod W.
template <int N>
__device__ __forceinline__ void mass_accum_masked(const uint32_t (&r)[N], float cs, int r0, int64_t j,
                                                  int64_t Tq, int W, float2 (&acc)[4]) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const bool v0 = j <= Tq + ((r0 + i) % W), v1 = j <= Tq + ((r0 + i + 1) % W);
    const float e0 = v0 ? ex2_approx(__uint_as_float(r[i]) * cs) : 0.f;
    const float e1 = v1 ? ex2_approx(__uint_as_float(r[i + 1]) * cs) : 0.f;
    acc[(i >> 1) & 3] = __fadd2_rn(acc[(i >> 1) & 3], make_float2(e0, e1));
  }
}

// kAnyR: window-row counts that are not a multiple of 32 (pass 2 padded to
// a multiple of 16 rows); a separate instantiation, so that the 16-column
// paths do not raise the register pressure of the common one.
template <int D, bool kAnyR>
__global__ void __launch_bounds__(kThreads, 1)
score_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
             const ScoreArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned start, formed by pointer arithmetic on the shared array
  // so that the compiler keeps every derived pointer in the shared space
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr int n_kc = D / 64;
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
      mbar_init(smem_u32(&s.tempty[i]), kEpiThreads / 32);   // one arrival per epilogue warp
    }
    mbar_init(smem_u32(s.qfull), 1);
    mbar_init(smem_u32(s.qempty), 1);
    mbar_init(smem_u32(s.mmadone), 1);
    mbar_init(smem_u32(s.augfull), 1);
    for (int i = 0; i < 16; ++i) mbar_init(smem_u32(&s.redfull[i]), 96);   // 3 groups x 32 threads
    *s.abort_flag = 0;
    fence_barrier_init();
  }
  // Q rows past R are read by the M = 128 row block of pass 1: keep them finite.
  {
    uint4* q4 = reinterpret_cast<uint4*>(s.q);
    const int n16 = n_kc * q_chunk_bytes / 16;
    for (int i = threadIdx.x; i < n16; i += kThreads) q4[i] = make_uint4(0, 0, 0, 0);
    // the all-ones operand of pass 2's extra K step (bf16 1.0 = 0x3f80)
    uint4* o4 = reinterpret_cast<uint4*>(s.ones);
    for (int i = threadIdx.x; i < 128 * 32 / 16; i += kThreads) o4[i] = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
  }
  fence_proxy_async_smem();
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_q);
  }
  if (warp == 1) {
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
        const int t0 = slice_begin(a, c);
        const int nt = slice_begin(a, c + 1) - t0;
        if (li > 0 && !mbar_wait_backoff(smem_u32(s.qempty), (li - 1) & 1, abort_flag, kProducerSleepNs))
          break;
        mbar_arrive_expect_tx(smem_u32(s.qfull), static_cast<uint32_t>(n_kc * a.R * 128));
        for (int kc = 0; kc < n_kc; ++kc)
          tma_load_3d(smem_u32(s.q + kc * q_chunk_bytes), &tmap_q, smem_u32(s.qfull), kc * 64, 0,
                      u, keep);
        ++q_loads;
        bool ok = true;
        for (int pass = a.row_lse ? 1 : 0; pass < 2 && ok; ++pass) {
          for (int t = 0; t < nt; ++t, ++jt) {
            const uint32_t st = jt % a.n_stages;
            const uint32_t ph = (jt / a.n_stages) & 1;
            if (!mbar_wait_backoff(smem_u32(&s.empty[st]), ph ^ 1, abort_flag, kProducerSleepNs)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(smem_u32(&s.full[st]), stage_bytes);
            for (int kc = 0; kc < n_kc; ++kc)
              tma_load_3d(smem_u32(s.k + st * stage_bytes + kc * kChunkBytes), &tmap_k,
                          smem_u32(&s.full[st]), kc * 64,
                          (t0 + (pass == 0 ? t : nt - 1 - t)) * kTileTokens, u,
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
      const uint32_t idesc2 = mma_idesc_bf16(128, a.Rp);
      // Operand descriptors: one base descriptor per buffer, every k-step and
      // stage reached by adding its byte offset / 16 to the start-address
      // field (shared addresses stay below 2^18, so the field never carries).
      // This keeps the issuing thread to a few instructions per MMA, which
      // matters because it shares its sub-partition with busy epilogue warps.
      constexpr int KS = D / 16;
      const uint64_t qdesc0 = sw128_desc(smem_u32(s.q));
      const uint64_t kdesc0 = sw128_desc(smem_u32(s.k));
      const uint64_t onesdesc = sw32_desc(smem_u32(s.ones));
      const uint64_t augdesc = sw32_desc(smem_u32(s.aug));
      const uint32_t qchunk16 = q_chunk_bytes >> 4;
      uint32_t jt = 0;
      int li = 0;
      for (int it = blockIdx.x; it < a.n_items; it += gridDim.x, ++li) {
        const int c = it % S;
        const int nt = slice_begin(a, c + 1) - slice_begin(a, c);
        if (!mbar_wait_backoff(smem_u32(s.qfull), li & 1, abort_flag, kMmaSleepNs)) break;
        tc_fence_after();
        bool ok = true;
        for (int pass = a.row_lse ? 1 : 0; pass < 2 && ok; ++pass) {
          // pass 2 adds -lse / scale through one more K step: wait for the rows
          if (pass == 1 && !mbar_wait_backoff(smem_u32(s.augfull), li & 1, abort_flag, kMmaSleepNs)) {
            ok = false;
            break;
          }
          for (int t = 0; t < nt; ++t, ++jt) {
            const uint32_t st = jt % a.n_stages;
            const uint32_t ph = (jt / a.n_stages) & 1;
            const uint32_t tb = jt & 1;
            const uint32_t tph = (jt >> 1) & 1;
            if (!mbar_wait_backoff(smem_u32(&s.full[st]), ph, abort_flag, kMmaSleepNs) ||
                !mbar_wait_backoff(smem_u32(&s.tempty[tb]), tph ^ 1, abort_flag, kMmaSleepNs)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t kd = kdesc0 + ((st * stage_bytes) >> 4);
            const uint32_t d_tmem = tmem_base + tb * 256;
            if (pass == 0) {
#pragma unroll
              for (int rb = 0; rb < 2; ++rb) {
                if (rb >= n_rb) break;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                  const uint64_t ad = qdesc0 + ((ks >> 2) * qchunk16 + rb * (kChunkBytes >> 4) + (ks & 3) * 2);
                  const uint64_t bd = kd + ((ks >> 2) * (kChunkBytes >> 4) + (ks & 3) * 2);
                  tc_mma_bf16(d_tmem + rb * 128, ad, bd, idesc1, ks > 0);
                }
              }
            } else {
#pragma unroll
              for (int ks = 0; ks < KS; ++ks) {
                const uint64_t ad = kd + ((ks >> 2) * (kChunkBytes >> 4) + (ks & 3) * 2);
                const uint64_t bd = qdesc0 + ((ks >> 2) * qchunk16 + (ks & 3) * 2);
                tc_mma_bf16(d_tmem, ad, bd, idesc2, ks > 0);
              }
              tc_mma_bf16(d_tmem, onesdesc, augdesc, idesc2, 1);
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
    // All four warpgroups process every tile, each on 64 adjacent TMEM
    // columns read by one load: in pass 1 warpgroup g takes window-row block
    // g / 2 and tokens [64 (g % 2), 64 (g % 2) + 64) of the tile; in pass 2
    // window rows [64 g, 64 g + 64).  Tile jt lives in TMEM buffer jt % 2.
    // Every named barrier is an OR-reduction of a failure flag, and no thread
    // leaves the item loop between two of them, so a bounded wait that gives
    // up in one warp ends all epilogue warps at the same barrier.
    const int e = warp - kEpiWarp0;            // 0..15
    const int qr = warp & 3;                   // TMEM lane quarter of this warp
    const int grp = e >> 2;                    // 0..3
    const int et = threadIdx.x - kEpiWarp0 * 32;
    const int lrow = qr * 32 + lane;           // TMEM lane of this thread
    const uint32_t lane_addr = static_cast<uint32_t>(qr * 32) << 16;
    const float cs = a.scale_log2;
    const int64_t T = a.T;
    const int64_t Tq = T - a.W;                // row w sees keys j <= Tq + w
    // pass 1: this thread's window row and token columns
    const int rb = grp >> 1;
    const int p1_row = lrow + 128 * rb;
    const bool p1_active = rb < n_rb;          // warp-uniform
    const bool p1_valid = p1_active && p1_row < a.R;
    const int64_t p1_last = Tq + (p1_valid ? p1_row % a.W : 0);
    const uint32_t p1_col = rb * 128 + (grp & 1) * 64;
    // pass 2: this group's window rows
    const int p2_r0 = 64 * grp;
    const int p2_n = max(0, min(64, a.Rp - p2_r0));  // 64, 48, 32, 16 or 0 (Rp: multiple of 16)

    uint32_t jt = 0;           // tile counter of both passes (TMEM buffer, phase)
    uint32_t jt2 = 0;          // pass-2 tile counter (reduction slot, phase, finalizer)
    bool fail = false;
    int cur_u = -1, cur_it = -1;
    for (int it = blockIdx.x; it < a.n_items; it += gridDim.x) {
      const int u = it / S, c = it % S;
      const int t0 = slice_begin(a, c);
      const int nt = slice_begin(a, c + 1) - t0;
      const int b = u / (a.L * a.Hkv);
      cur_u = u;
      cur_it = it;

      if (a.row_lse == nullptr) {
        // ---------------- pass 1: per-row online max / sum (log2 domain)
        float m = -INFINITY, l = 0.f;
        for (int t = 0; t < nt; ++t, ++jt) {
          const uint32_t tb = jt & 1, tph = (jt >> 1) & 1;
          if (fail || !mbar_wait(smem_u32(&s.tfull[tb]), tph, abort_flag)) {
            fail = true;
            continue;
          }
          tc_fence_after();
          // The accumulator columns are copied to registers and the buffer is
          // released at once, so the MMA of tile jt + 2 overlaps this math.
          if (p1_active) {
            uint32_t r[64];
            tmem_ld64(tmem_base + lane_addr + tb * 256 + p1_col, r);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.tempty[tb]));
            const int64_t j0 = static_cast<int64_t>(t0 + t) * kTileTokens + (grp & 1) * 64;
            const bool masked = (j0 + 63) > Tq;
            float sum = 0.f;
            if (!masked && m != -INFINITY) sum = exp_sum<64>(r, cs, m);
            if (!masked && m != -INFINITY && sum <= 0x1p100f) l += sum;
            else row_update<64>(r, cs, masked, j0, p1_last, m, l);
          } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.tempty[tb]));
          }
        }
        // merge the two warpgroups' statistics of each row
        s.hm[grp * 128 + lrow] = m;
        s.hl[grp * 128 + lrow] = l;
        fail = named_bar_or(1, kEpiThreads, fail);
        if ((grp & 1) == 0 && p1_valid && !fail) {
          const float m2 = s.hm[(grp + 1) * 128 + lrow], l2 = s.hl[(grp + 1) * 128 + lrow];
          const float mn = fmaxf(m, m2);
          float ls = 0.f;
          if (mn != -INFINITY) ls = l * ex2_approx(m - mn) + l2 * ex2_approx(m2 - mn);
          a.stats[(static_cast<size_t>(u) * S + c) * a.R + p1_row] = make_float2(mn, ls);
        }
        // Publication: the barrier orders every thread's statistics before the
        // one gpu-scope release (the counter increment) that makes them
        // visible to the unit's other CTAs.
        fail = named_bar_or(1, kEpiThreads, fail);
        if (fail) break;
        bool timed_out = false;
        if (et == 0) {
          atom_add_release_gpu(&a.counters[u], 1u);
          uint64_t t_start = 0;
          for (uint32_t n = 0;; ++n) {
            // (a.stall_unit: a test raises one unit's target to a count nothing reaches)
            if (ld_acquire_gpu(&a.counters[u]) >= static_cast<uint32_t>(S + (u == a.stall_unit))) break;
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
        // log-sum-exp of every row over the whole unit (stored negated): two
        // adjacent threads per row merge the even and the odd chunks, eight
        // loads in flight each, then combine their two partial results.
        // The loop runs over whole warps (the pair exchange is a full-warp
        // shuffle), with the threads past the last row idle inside it.
        const int n_pairs = (2 * a.R + 31) & ~31;
        for (int q = et; q < n_pairs; q += kEpiThreads) {
          const bool live = q < 2 * a.R;
          const int r = q >> 1, h = q & 1;
          float M = -INFINITY, Ls = 0.f;
          const float2* st_row = a.stats + static_cast<size_t>(u) * S * a.R + r;
          for (int c0 = h; live && c0 < S; c0 += 16) {
            float2 st[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              st[k] = (c0 + 2 * k < S) ? __ldcg(st_row + static_cast<size_t>(c0 + 2 * k) * a.R)
                                       : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (st[k].x == -INFINITY) continue;
              if (st[k].x > M) {
                Ls = Ls * ex2_approx(M - st[k].x) + st[k].y;
                M = st[k].x;
              } else {
                Ls += st[k].y * ex2_approx(st[k].x - M);
              }
            }
          }
          const float M2 = __shfl_xor_sync(0xffffffffu, M, 1);
          const float L2 = __shfl_xor_sync(0xffffffffu, Ls, 1);
          const float Mx = fmaxf(M, M2);
          const float Lt = (M == -INFINITY ? 0.f : Ls * ex2_approx(M - Mx)) +
                           (M2 == -INFINITY ? 0.f : L2 * ex2_approx(M2 - Mx));
          if (live && h == 0) s.lam[r] = -(Mx + __log2f(Lt));
        }
        // padding rows of the pass-2 MMA (R <= r < Rp) contribute nothing
        for (int r = a.R + et; r < a.Rp; r += kEpiThreads) s.lam[r] = -INFINITY;
        named_bar_sync(1, kEpiThreads);
      } else {
        // the caller's natural-log row statistics, in the log2 domain
        const float* rl = a.row_lse + static_cast<size_t>(u) * a.R;
        for (int r = et; r < a.R; r += kEpiThreads) s.lam[r] = -(__ldg(rl + r) * 1.44269504088896340736f);
        for (int r = a.R + et; r < a.Rp; r += kEpiThreads) s.lam[r] = -INFINITY;
        named_bar_sync(1, kEpiThreads);
      }
      // Pass 2's extra K step: row r of `aug` holds -lse_r / scale as the sum
      // of three bf16 parts (all 24 bits of the fp32 value; the rest of the
      // row zero), and every row of `ones` is all ones, so the MMA adds that
      // sum to z = q . k and the epilogue forms z * scale - lse_r with one
      // multiply.  A padding row gets a large negative finite value (its
      // exponentials vanish).  The previous item's pass-2 MMAs, the last
      // readers of `aug`, have completed: this epilogue consumed all of their
      // accumulators before it reached this point.
      for (int r = et; r < a.Rp; r += kEpiThreads) {
        const float lm = s.lam[r];
        float hi = -0x1p120f, mid = 0.f, lo = 0.f;
        if (lm != -INFINITY) {
          const float av = lm / cs;
          hi = __bfloat162float(__float2bfloat16_rn(av));
          const float r1 = av - hi;
          mid = __bfloat162float(__float2bfloat16_rn(r1));
          lo = __bfloat162float(__float2bfloat16_rn(r1 - mid));
        }
        uint4* row = reinterpret_cast<uint4*>(s.aug + (r >> 3) * 256 + (r & 7) * 32);
        const uint32_t w0 = static_cast<uint32_t>(float_to_bf16_bits(hi)) |
                            (static_cast<uint32_t>(float_to_bf16_bits(mid)) << 16);
        row[0] = make_uint4(w0, float_to_bf16_bits(lo), 0, 0);
        row[1] = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, kEpiThreads);
      if (et == 0) mbar_arrive(smem_u32(s.augfull));

      // ---------------- pass 2: per-token sum of exp2(z cs - lse) over rows
      // The four groups' partial sums of pass-2 tile jt2 meet in slot jt2 % 4
      // of `red`.  Group jt2 % 4 keeps its own partial in registers and, one
      // tile later (so the others have long written theirs), waits for
      // redfull[slot][quarter] and writes the token's score.  The finalizing
      // role rotates, so no group carries more work than another and no
      // CTA-wide barrier sits between tiles.  A slot is rewritten by pass-2
      // tile jt2 + 4 only after its finalize: those writers waited for that
      // tile's accumulator, whose MMA waited for every warp (the finalizer
      // too, after its finalize) to release a tile two or more behind it.
      // The finalizer loads the token's bonus and previous score when the
      // tile starts; they are consumed a tile later.
      auto finalize = [&](uint32_t jtf, float own, float bon, float old, int64_t jf) {
        const int sl = jtf & 3;
        // the give-up decision is made for the whole warp, which then either
        // leaves or reaches the page-max shuffle together
        const bool ok = !fail && mbar_wait(smem_u32(&s.redfull[sl * 4 + qr]), (jtf >> 2) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          fail = true;
          return;
        }
        const float* rs = s.red + sl * 512 + lrow;
        const float p0 = grp == 0 ? own : rs[0];
        const float p1 = grp == 1 ? own : rs[128];
        const float p2 = grp == 2 ? own : rs[256];
        const float p3 = grp == 3 ? own : rs[384];
        float sc = -INFINITY;
        if (jf < T) {
          sc = ((p0 + p1) + (p2 + p3)) + (bon + old);
          a.scores[static_cast<int64_t>(u) * T + jf] = sc;
        }
        const int P = a.page_size;
        if (P > 1) {
          float pm = sc;
          for (int o = 1; o < P; o <<= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o));
          if (jf < T && (lane & (P - 1)) == 0)
            a.page_scores[static_cast<int64_t>(u) * (T / P) + jf / P] = pm;
        }
      };
      bool pend = false;                 // this group finalizes pass-2 tile jt_p
      uint32_t jt_p = 0;
      float own_p = 0.f, bon_p = 0.f, old_p = 0.f;
      int64_t j_p = 0;
      for (int t = 0; t < nt; ++t, ++jt, ++jt2) {
        const uint32_t tb = jt & 1, tph = (jt >> 1) & 1;
        const int fg = static_cast<int>(jt2 & 3);
        // pass 2 walks the item's tiles last to first: the tiles pass 1 read
        // most recently are the likeliest to still be in L2
        const int64_t tile0 = static_cast<int64_t>(t0 + nt - 1 - t) * kTileTokens;
        const int64_t j = tile0 + lrow;
        const bool masked = (tile0 + kTileTokens - 1) > Tq;
        float bon = 0.f, old = 0.f;
        if (grp == fg && j < T) {
          if (a.bonus) bon = __ldg(a.bonus + static_cast<int64_t>(b) * T + j);
          if (a.accumulate) old = a.scores[static_cast<int64_t>(u) * T + j];
        }
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        if (!fail && mbar_wait(smem_u32(&s.tfull[tb]), tph, abort_flag)) {
          tc_fence_after();
          const uint32_t taddr = tmem_base + lane_addr + tb * 256 + p2_r0;
          // copy to registers, release the buffer, then do the math
          if (p2_n == 64) {
            uint32_t r[64];
            tmem_ld64(taddr, r);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.tempty[tb]));
            if (!masked) mass_accum<64>(r, cs, acc);
            else mass_accum_masked<64>(r, cs, p2_r0, j, Tq, a.W, acc);
          } else if (p2_n == 32 || (kAnyR && p2_n == 48)) {
            uint32_t r[32];
            tmem_ld32_issue(taddr, r);
            tmem_ld_wait(r);
            uint32_t r16[16];
            if (kAnyR && p2_n == 48) tmem_ld16(taddr + 32, r16);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.tempty[tb]));
            if (!masked) mass_accum<32>(r, cs, acc);
            else mass_accum_masked<32>(r, cs, p2_r0, j, Tq, a.W, acc);
            if (kAnyR && p2_n == 48) {
              if (!masked) mass_accum<16>(r16, cs, acc);
              else mass_accum_masked<16>(r16, cs, p2_r0 + 32, j, Tq, a.W, acc);
            }
          } else if (kAnyR && p2_n == 16) {
            uint32_t r[16];
            tmem_ld16(taddr, r);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.tempty[tb]));
            if (!masked) mass_accum<16>(r, cs, acc);
            else mass_accum_masked<16>(r, cs, p2_r0, j, Tq, a.W, acc);
          } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.tempty[tb]));
          }
        } else {
          fail = true;
        }
        const float2 a2 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
        const float part = a2.x + a2.y;
        if (grp != fg) {
          s.red[(fg * 4 + grp) * 128 + lrow] = part;
          mbar_arrive(smem_u32(&s.redfull[fg * 4 + qr]));
        }
        if (pend) {
          finalize(jt_p, own_p, bon_p, old_p, j_p);
          pend = false;
        }
        if (grp == fg) {
          pend = true;
          jt_p = jt2;
          own_p = part;
          bon_p = bon;
          old_p = old;
          j_p = j;
        }
      }
      if (pend) finalize(jt_p, own_p, bon_p, old_p, j_p);
      // the next item's pass 1 rewrites hm / hl and lam only after this barrier
      fail = named_bar_or(1, kEpiThreads, fail);
      if (fail) break;
    }
    // a CTA that gave up leaves its current item and every later one
    // unscored: all their units are marked
    if (fail && et == 0 && cur_it >= 0 && a.unit_status)
      for (int it = cur_it; it < a.n_items; it += gridDim.x) a.unit_status[it / S] = KVC_UNIT_TIMEOUT;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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
  bytes += 128 * 32 + static_cast<size_t>(q_rows) * 32;  // ones, aug
  bytes += (2 * n_stages + 26) * 8;                      // barriers
  bytes += 16;                                           // tmem slot, abort flag
  bytes += (256 + 2048 + 2 * 1024) * 4;                 // lam, red, hm, hl
  return bytes;
}

cudaError_t launch_score(const ScoreArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_q,
                         int grid, size_t smem_bytes, cudaStream_t stream) {
  const bool any_r = a.R % 32 != 0;
  void (*kern)(const CUtensorMap, const CUtensorMap, const ScoreArgs) =
      a.d == 64 ? (any_r ? score_kernel<64, true> : score_kernel<64, false>)
                : (any_r ? score_kernel<128, true> : score_kernel<128, false>);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  return cudaLaunchKernelEx(&cfg, kern, tmap_k, tmap_q, a);
}

}  // namespace kvc
