// CommitKV deletion effect and lifecycle decisions on the GPU.
//
// What it computes ("CommitKV: Lifecycle-Aware KV Cache Compression via
// Commit Transitions for Multi-Turn Agents", Sec. 3.2-3.3): for each unit
// u = (b, l, g) the R = G W window rows (query head h = g G + r / W, window
// position w = r % W at cache index T - W + w, seeing indices <= T - W + w)
// attend over the unit's T keys:
//   a_rj = softmax_j(q_r . k_j * scale),  o_r = sum_j a_rj v_j;
// and for every event page E (a span of at most 64 cache indices):
//   s_rE = sum_{j in E} a_rj,  u_rE = sum_{j in E} a_rj v_j,
//   ratio_rE = || o_r - (o_r - u_rE) / (1 - s_rE) || / || o_r ||   (Eq. 6, 7)
//            = || u_rE - s_rE o_r || / ((1 - s_rE) || o_r ||),
//   R(E; Q) = max over the layer's heads and window rows.          (Eq. 7)
// The commit kernel turns R- / R+ into percentile ranks, Eq. 9 indicators,
// Eq. 10 states and the greedy Eq. 11 retirement set; the joint effect of a
// page set is exact from the stored per-page s and u because both are sums
// over disjoint token sets.
//
// Window attention design (tcgen05, one persistent CTA per SM).  A work item
// is one unit and a chunk of its 128-token key tiles.  Pass 1 computes
// D1[m][j] = Q K^T (M = 128, N = 128) per tile: the Q block holds 128 / S
// replicas of the unit's rows (S = 32 or 64 rows), so each epilogue thread
// owns one row and S of the tile's tokens and keeps an online max / sum in
// the log2 domain; the replicas' statistics are merged once per item.  Pass 2
// recomputes D1 from the same (now L2-resident) key tiles, turns it into
// P = exp2(y - m) <= 1, splits P into a bf16 head and a bf16 tail (16
// significant bits in all) and accumulates D2[d][r] += V^T P^T with V read
// as an MN-major operand straight from its TMA tile (M = 128 = d, N = Rp,
// K = 128 tokens; two MMAs per k-step, head and tail).  D2 stays in tensor
// memory across the item's tiles and is written out as the item's (max, sum,
// value sum); a merge kernel combines the items of a unit by PASK Eq. 15.
//
// Warp roles (6 warps): 0 = TMA producer, 1 = TMEM owner and MMA issuer,
// 2..5 = epilogue (warp w reads TMEM lanes 32 (w % 4) .. + 31).  Every wait
// is bounded; a wait that gives up raises a shared abort flag, the unit is
// marked KVC_UNIT_TIMEOUT and the CTA drains its copies and MMAs before it
// frees tensor memory and returns.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kEffThreads = 192;
constexpr int kEffEpiWarp0 = 2;
constexpr int kEffEpiThreads = 128;
constexpr uint32_t kEffTmemCols = 512;       // D1: 2 x 128 columns, D2: columns 256 .. 256 + Rp
constexpr uint32_t kD2Col = 256;
constexpr int kChunk = 128 * 128;            // 128 rows x 64 bf16 (one swizzle-128 chunk)
constexpr int kTile = 2 * kChunk;            // one 128-token x 128-dim tile
constexpr uint32_t kSleepNs = 64;

struct EffSmem {
  uint8_t* q;          // 2 chunks x 128 rows x 128 B
  uint8_t* k;          // ring of n_stages tiles, key and value tiles alike
  uint8_t* p;          // [2 buffers][2 parts][2 chunks][Rp rows][128 B]
  uint64_t* kfull;     // [n_stages]
  uint64_t* kempty;    // [n_stages]
  uint64_t* tfull;     // [2]
  uint64_t* tempty;    // [2]
  uint64_t* pfull;     // [2]
  uint64_t* pempty;    // [2]
  uint64_t* qfull;
  uint64_t* qempty;
  uint64_t* d2full;
  uint64_t* d2empty;
  uint64_t* mmadone;
  uint32_t* tmem_slot;
  int* abort_flag;
  float* sm;           // [128] pass-1 maximum per TMEM lane
  float* sl;           // [128] pass-1 sum per TMEM lane
};

__device__ __forceinline__ EffSmem eff_carve(uint8_t* base, int Rp, int ns) {
  EffSmem s;
  s.q = base;
  s.k = s.q + 2 * kChunk;
  s.p = s.k + ns * kTile;
  uint64_t* b = reinterpret_cast<uint64_t*>(s.p + 8 * Rp * 128);
  s.kfull = b;
  s.kempty = b + ns;
  b += 2 * ns;
  s.tfull = b;
  s.tempty = b + 2;
  s.pfull = b + 4;
  s.pempty = b + 6;
  s.qfull = b + 8;
  s.qempty = b + 9;
  s.d2full = b + 10;
  s.d2empty = b + 11;
  s.mmadone = b + 12;
  s.tmem_slot = reinterpret_cast<uint32_t*>(b + 13);
  s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
  s.sm = reinterpret_cast<float*>(s.tmem_slot + 4);
  s.sl = s.sm + 128;
  return s;
}

__device__ __forceinline__ void eff_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Shared-memory descriptor of an MN-major bf16 operand in 128-byte swizzle:
// 64 contiguous elements along M (or N) per 128-byte row, consecutive rows
// along K; the next 8 rows along K are 1024 B further (stride byte offset)
// and the next 64 elements along M are `lbo` bytes further (leading byte
// offset).
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x (low half) = lo
  return *reinterpret_cast<const uint32_t*>(&h);
}

// S = rows per replica of the Q block (32 or 64); 128 / S replicas, each
// thread of replica k handles tokens [k S, k S + S) of every tile.
template <int S>
__global__ void __launch_bounds__(kEffThreads, 1)
effect_attn_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                   const __grid_constant__ CUtensorMap tmap_q, const EffectArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const EffSmem s = eff_carve(base, a.Rp, a.nk);
  const uint32_t NS = static_cast<uint32_t>(a.nk);
  constexpr int kRep = 128 / S;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = s.abort_flag;
  const uint32_t p_part = static_cast<uint32_t>(a.Rp) * 128u * 2u;   // one part: 2 chunks

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.nk; ++i) {
      mbar_init(smem_u32(&s.kfull[i]), 1);
      mbar_init(smem_u32(&s.kempty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.tfull[i]), 1);
      mbar_init(smem_u32(&s.tempty[i]), kEffEpiThreads / 32);
      mbar_init(smem_u32(&s.pfull[i]), kEffEpiThreads / 32);
      mbar_init(smem_u32(&s.pempty[i]), 1);
    }
    mbar_init(smem_u32(s.qfull), 1);
    mbar_init(smem_u32(s.qempty), 1);
    mbar_init(smem_u32(s.d2full), 1);
    mbar_init(smem_u32(s.d2empty), kEffEpiThreads / 32);
    mbar_init(smem_u32(s.mmadone), 1);
    *s.abort_flag = 0;
    fence_barrier_init();
  }
  // Q rows that no replica fills, and P rows past R, stay zero.
  {
    uint4* q4 = reinterpret_cast<uint4*>(s.q);
    for (int i = threadIdx.x; i < 2 * kChunk / 16; i += kEffThreads) q4[i] = make_uint4(0, 0, 0, 0);
    uint4* p4 = reinterpret_cast<uint4*>(s.p);
    for (int i = threadIdx.x; i < 8 * a.Rp * 128 / 16; i += kEffThreads) p4[i] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
    tma_prefetch_desc(&tmap_q);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s.tmem_slot), kEffTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s.tmem_slot;
  const int SP = a.splits;
  // a contiguous range of items per CTA, so that consecutive items mostly
  // share a unit and its window queries stay in shared memory
  const int it0 = static_cast<int>(static_cast<int64_t>(a.n_items) * blockIdx.x / gridDim.x);
  const int it1 = static_cast<int>(static_cast<int64_t>(a.n_items) * (blockIdx.x + 1) / gridDim.x);

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t stream = l2_policy_evict_first();
      uint32_t jr = 0;           // ring loads issued (key tiles of both passes, value tiles of pass 2)
      int q_loads = 0, prev_u = -1;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int u = it / SP, c = it % SP;
        const int t0 = c * a.chunk_tiles;
        const int nt = min(a.chunk_tiles, a.n_tiles - t0);
        if (u != prev_u) {
          // a new unit: its queries replace the previous unit's once every MMA reading them is done
          if (q_loads > 0 && !mbar_wait_backoff(smem_u32(s.qempty), (q_loads - 1) & 1, abort_flag, kSleepNs))
            break;
          mbar_arrive_expect_tx(smem_u32(s.qfull), static_cast<uint32_t>(kRep * 2 * a.R * 128));
          for (int rk = 0; rk < kRep; ++rk)
            for (int kc = 0; kc < 2; ++kc)
              tma_load_3d(smem_u32(s.q + kc * kChunk + rk * S * 128), &tmap_q, smem_u32(s.qfull),
                          kc * 64, 0, u, keep);
          ++q_loads;
          prev_u = u;
        }
        for (int pass = 0; pass < 2 && ok; ++pass) {
          for (int t = 0; t < nt && ok; ++t) {
            for (int kv = 0; kv <= pass; ++kv) {          // pass 1: the key tile; pass 2: key, value
              const uint32_t st = jr % NS, ph = (jr / NS) & 1;
              if (!mbar_wait_backoff(smem_u32(&s.kempty[st]), ph ^ 1, abort_flag, kSleepNs)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(smem_u32(&s.kfull[st]), kTile);
              for (int kc = 0; kc < 2; ++kc)
                tma_load_3d(smem_u32(s.k + st * kTile + kc * kChunk), kv ? &tmap_v : &tmap_k,
                            smem_u32(&s.kfull[st]), kc * 64, (t0 + t) * kTileTokens, u,
                            (pass == 0) ? keep : stream);
              ++jr;
            }
          }
        }
      }
      // every copy issued above lands before the CTA exits
      for (uint32_t j = jr > NS ? jr - NS : 0; j < jr; ++j) eff_drain(smem_u32(&s.kfull[j % NS]), (j / NS) & 1);
      if (q_loads > 0) eff_drain(smem_u32(s.qfull), (q_loads - 1) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc1 = mma_idesc_bf16(128, 128);
      const uint32_t idesc2 = mma_idesc_bf16(128, a.Rp) | (1u << 15);   // A (values) MN-major
      const uint64_t qdesc0 = sw128_desc(smem_u32(s.q));
      const uint64_t kdesc0 = sw128_desc(smem_u32(s.k));
      const uint64_t vdesc0 = sw128_mn_desc(smem_u32(s.k), kChunk);
      const uint64_t pdesc0 = sw128_desc(smem_u32(s.p));
      const uint32_t pchunk16 = (static_cast<uint32_t>(a.Rp) * 128u) >> 4;
      uint32_t jr = 0, jt = 0, jp = 0;
      uint32_t vslot0 = 0, vslot1 = 0;   // ring index of the value tile of even / odd pass-2 tiles
      int li = 0, q_segs = 0, prev_u = -1;
      bool ok = true;
      // MMA2 of pass-2 tile `tile` (P in buffer jp % 2, values at ring index vslot[tile % 2])
      auto mma2 = [&](int tile) -> bool {
        const uint32_t pb = jp & 1, pph = (jp >> 1) & 1;
        const uint32_t jv = (tile & 1) ? vslot1 : vslot0;
        const uint32_t sv = jv % NS, pv = (jv / NS) & 1;
        if (!mbar_wait_backoff(smem_u32(&s.pfull[pb]), pph, abort_flag, kSleepNs) ||
            !mbar_wait_backoff(smem_u32(&s.kfull[sv]), pv, abort_flag, kSleepNs))
          return false;
        if (tile == 0 && li > 0 &&
            !mbar_wait_backoff(smem_u32(s.d2empty), (li - 1) & 1, abort_flag, kSleepNs))
          return false;
        tc_fence_after();
        const uint64_t vd = vdesc0 + ((sv * kTile) >> 4);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint64_t ad = vd + ((ks * 16 * 128) >> 4);
            const uint64_t bd = pdesc0 + (((pb * 2 + part) * p_part) >> 4) + (ks >> 2) * pchunk16 +
                                (ks & 3) * 2;
            tc_mma_bf16(tmem_base + kD2Col, ad, bd, idesc2, (tile > 0 || ks > 0 || part > 0) ? 1u : 0u);
          }
        }
        tc_commit(smem_u32(&s.kempty[sv]));
        tc_commit(smem_u32(&s.pempty[pb]));
        ++jp;
        return true;
      };
      for (int it = it0; it < it1 && ok; ++it, ++li) {
        const int u = it / SP, c = it % SP;
        const int t0 = c * a.chunk_tiles;
        const int nt = min(a.chunk_tiles, a.n_tiles - t0);
        if (u != prev_u) {
          if (q_segs > 0) tc_commit(smem_u32(s.qempty));   // the previous unit's queries are done with
          if (!mbar_wait_backoff(smem_u32(s.qfull), q_segs & 1, abort_flag, kSleepNs)) break;
          ++q_segs;
          prev_u = u;
        }
        tc_fence_after();
        for (int pass = 0; pass < 2 && ok; ++pass) {
          for (int t = 0; t < nt; ++t) {
            const uint32_t sk = jr % NS, pk = (jr / NS) & 1;
            const uint32_t tb = jt & 1, tph = (jt >> 1) & 1;
            if (!mbar_wait_backoff(smem_u32(&s.kfull[sk]), pk, abort_flag, kSleepNs) ||
                !mbar_wait_backoff(smem_u32(&s.tempty[tb]), tph ^ 1, abort_flag, kSleepNs)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t kd = kdesc0 + ((sk * kTile) >> 4);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t ad = qdesc0 + ((ks >> 2) * (kChunk >> 4) + (ks & 3) * 2);
              const uint64_t bd = kd + ((ks >> 2) * (kChunk >> 4) + (ks & 3) * 2);
              tc_mma_bf16(tmem_base + tb * 128, ad, bd, idesc1, ks > 0 ? 1u : 0u);
            }
            tc_commit(smem_u32(&s.kempty[sk]));
            tc_commit(smem_u32(&s.tfull[tb]));
            ++jr;
            ++jt;
            if (pass == 1) {                         // the value tile follows its key tile in the ring
              if (t & 1) vslot1 = jr;
              else vslot0 = jr;
              ++jr;
            }
            if (pass == 1 && t > 0 && !mma2(t - 1)) ok = false;
          }
        }
        if (!ok) break;
        if (!mma2(nt - 1)) break;
        tc_commit(smem_u32(s.d2full));
      }
      // all MMAs issued above complete before tensor memory is freed
      tc_commit(smem_u32(s.mmadone));
      eff_drain(smem_u32(s.mmadone), 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int qr = warp & 3;
    const int Lq = qr * 32 + lane;             // TMEM lane of this thread
    const int rk = Lq / S;                     // Q replica
    const int r = Lq % S;                      // window row
    const bool valid = r < a.R;
    const int c0 = rk * S;                     // first token column of this thread in a tile
    const int w = r % a.W;
    const uint32_t lane_addr = static_cast<uint32_t>(qr * 32) << 16;
    const float cs = a.scale_log2;
    const int64_t last = a.T - a.W + w;        // last cache index row r sees
    const int et = threadIdx.x - kEffEpiWarp0 * 32;
    uint32_t jt = 0, jp = 0;
    int li = 0;
    bool fail = false;
    int cur_u = -1, cur_it = -1;
    for (int it = it0; it < it1; ++it, ++li) {
      const int u = it / SP, c = it % SP;
      const int t0 = c * a.chunk_tiles;
      const int nt = min(a.chunk_tiles, a.n_tiles - t0);
      cur_u = u;
      cur_it = it;
      // ---- pass 1: online max / sum of y = z * cs over this thread's tokens
      float m = -INFINITY, l = 0.f;
      for (int t = 0; t < nt; ++t, ++jt) {
        const uint32_t tb = jt & 1, tph = (jt >> 1) & 1;
        if (fail || !mbar_wait(smem_u32(&s.tfull[tb]), tph, abort_flag)) {
          fail = true;
          continue;
        }
        tc_fence_after();
        uint32_t rv[S];
        if constexpr (S == 64) tmem_ld64(tmem_base + lane_addr + tb * 128 + c0, rv);
        else tmem_ld32_issue(tmem_base + lane_addr + tb * 128 + c0, rv), tmem_ld_wait(rv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.tempty[tb]));
        const int64_t j0 = static_cast<int64_t>(t0 + t) * kTileTokens + c0;
        float y[S];
        float mc = -INFINITY;
#pragma unroll
        for (int i = 0; i < S; ++i) {
          y[i] = (j0 + i <= last) ? __uint_as_float(rv[i]) * cs : -INFINITY;
          mc = fmaxf(mc, y[i]);
        }
        if (mc > m) {
          l *= ex2_approx(m - mc);
          m = mc;
        }
        if (m != -INFINITY) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < S; ++i) acc += ex2_approx(y[i] - m);
          l += acc;
        }
      }
      // merge the replicas' statistics of each row
      s.sm[Lq] = m;
      s.sl[Lq] = l;
      fail = named_bar_or(1, kEffEpiThreads, fail);
      float M = -INFINITY, Ls = 0.f;
#pragma unroll
      for (int k = 0; k < kRep; ++k) M = fmaxf(M, s.sm[k * S + r]);
      if (M != -INFINITY) {
#pragma unroll
        for (int k = 0; k < kRep; ++k) {
          const float mk = s.sm[k * S + r];
          if (mk != -INFINITY) Ls += s.sl[k * S + r] * ex2_approx(mk - M);
        }
      }
      if (rk == 0 && valid && !fail) a.part_ml[static_cast<int64_t>(it) * a.R + r] = make_float2(M, Ls);
      // ---- pass 2: P = exp2(y - M), split into bf16 head + tail, to shared memory
      for (int t = 0; t < nt; ++t, ++jt, ++jp) {
        const uint32_t tb = jt & 1, tph = (jt >> 1) & 1;
        const uint32_t pb = jp & 1, pph = (jp >> 1) & 1;
        if (fail || !mbar_wait(smem_u32(&s.tfull[tb]), tph, abort_flag)) {
          fail = true;
          continue;
        }
        tc_fence_after();
        uint32_t rv[S];
        if constexpr (S == 64) tmem_ld64(tmem_base + lane_addr + tb * 128 + c0, rv);
        else tmem_ld32_issue(tmem_base + lane_addr + tb * 128 + c0, rv), tmem_ld_wait(rv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.tempty[tb]));
        const int64_t j0 = static_cast<int64_t>(t0 + t) * kTileTokens + c0;
        if (!mbar_wait(smem_u32(&s.pempty[pb]), pph ^ 1, abort_flag)) {
          fail = true;
          continue;
        }
        if (valid) {
          uint8_t* hi_base = s.p + (pb * 2 + 0) * p_part + (c0 >> 6) * (a.Rp * 128) + r * 128;
          uint8_t* lo_base = hi_base + p_part;
#pragma unroll
          for (int g8 = 0; g8 < S / 8; ++g8) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int h2 = 0; h2 < 4; ++h2) {
              const int i0 = g8 * 8 + 2 * h2;
              const float p0 = (j0 + i0 <= last) ? ex2_approx(__uint_as_float(rv[i0]) * cs - M) : 0.f;
              const float p1 = (j0 + i0 + 1 <= last) ? ex2_approx(__uint_as_float(rv[i0 + 1]) * cs - M) : 0.f;
              const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
              hw[h2] = *reinterpret_cast<const uint32_t*>(&h);
              lw[h2] = pack_bf16x2(p0 - __low2float(h), p1 - __high2float(h));
            }
            const int unit = (((c0 & 63) >> 3) + g8) ^ (r & 7);
            *reinterpret_cast<uint4*>(hi_base + unit * 16) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(lo_base + unit * 16) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.pfull[pb]));
      }
      // ---- the item's value sums: thread = dimension d, columns = rows
      if (!fail && mbar_wait(smem_u32(s.d2full), li & 1, abort_flag)) {
        tc_fence_after();
        const int d = Lq;
        float* dst = a.part_u + static_cast<int64_t>(it) * a.R * 128 + d;
        for (int c16 = 0; c16 < a.Rp; c16 += 16) {
          uint32_t rv[16];
          tmem_ld16(tmem_base + lane_addr + kD2Col + c16, rv);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c16 + i < a.R) dst[(c16 + i) * 128] = __uint_as_float(rv[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(s.d2empty));
      } else {
        fail = true;
      }
      fail = named_bar_or(1, kEffEpiThreads, fail);
      if (fail) break;
    }
    // a CTA that gave up leaves its current item and the rest of its range
    // unprocessed: all their units are marked
    if (fail && et == 0 && cur_it >= 0 && a.unit_status)
      for (int it = cur_it; it < it1; ++it) a.unit_status[it / SP] = KVC_UNIT_TIMEOUT;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kEffTmemCols);
  }
}

// PASK Eq. 15 over the work items of a unit: o = sum_c 2^(m_c - M) u_c /
// sum_c 2^(m_c - M) l_c, and the natural-log denominator lse = (M + log2 den) ln 2.
// One block per (unit, row); each lane owns four dimensions, the four warps
// take every fourth item and meet in shared memory.
__global__ void __launch_bounds__(128) effect_merge_kernel(const EffectArgs a) {
  __shared__ float red[4];
  __shared__ float4 part[4][32];
  __shared__ float s_M, s_den;
  const int u = blockIdx.x / a.R, r = blockIdx.x % a.R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int SP = a.splits;
  const float2* ml = a.part_ml + static_cast<int64_t>(u) * SP * a.R + r;
  float M = -INFINITY;
  for (int c = tid; c < SP; c += 128) M = fmaxf(M, ml[static_cast<int64_t>(c) * a.R].x);
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  if (tid == 0) s_M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  M = s_M;
  float den = 0.f;
  for (int c = tid; c < SP; c += 128) {
    const float2 st = ml[static_cast<int64_t>(c) * a.R];
    if (st.x != -INFINITY) den += ex2_approx(st.x - M) * st.y;   // empty partitions add nothing
  }
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o2);
  __syncthreads();
  if (lane == 0) red[warp] = den;
  const float4* pu = reinterpret_cast<const float4*>(a.part_u + (static_cast<int64_t>(u) * SP * a.R + r) * 128) + lane;
  const int64_t cstride = static_cast<int64_t>(a.R) * 32;       // float4 units between items
  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  int c = warp;
  for (; c + 12 < SP; c += 16) {
    float4 v4[4];
    float f4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float mc = ml[static_cast<int64_t>(c + 4 * i) * a.R].x;
      f4[i] = mc == -INFINITY ? 0.f : ex2_approx(mc - M);
      v4[i] = pu[(c + 4 * i) * cstride];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      num.x = fmaf(f4[i], v4[i].x, num.x);
      num.y = fmaf(f4[i], v4[i].y, num.y);
      num.z = fmaf(f4[i], v4[i].z, num.z);
      num.w = fmaf(f4[i], v4[i].w, num.w);
    }
  }
  for (; c < SP; c += 4) {
    const float mc = ml[static_cast<int64_t>(c) * a.R].x;
    if (mc == -INFINITY) continue;
    const float f = ex2_approx(mc - M);
    const float4 v = pu[c * cstride];
    num.x = fmaf(f, v.x, num.x);
    num.y = fmaf(f, v.y, num.y);
    num.z = fmaf(f, v.z, num.z);
    num.w = fmaf(f, v.w, num.w);
  }
  part[warp][lane] = num;
  __syncthreads();
  if (tid == 0) s_den = (red[0] + red[1]) + (red[2] + red[3]);
  if (warp == 0) {
    float4 t = part[0][lane];
#pragma unroll
    for (int w2 = 1; w2 < 4; ++w2) {
      t.x += part[w2][lane].x;
      t.y += part[w2][lane].y;
      t.z += part[w2][lane].z;
      t.w += part[w2][lane].w;
    }
    part[0][lane] = t;
  }
  __syncthreads();
  den = s_den;
  if (warp == 0) {
    const float4 t = part[0][lane];
    reinterpret_cast<float4*>(a.o + (static_cast<int64_t>(u) * a.R + r) * 128)[lane] =
        make_float4(t.x / den, t.y / den, t.z / den, t.w / den);
  }
  if (tid == 0) a.lse[static_cast<int64_t>(u) * a.R + r] = (M + log2f(den)) * 0.69314718055994531f;
}

// Page weights, value sums and Eq. 7 ratios: one block per (page, unit), one
// warp per window row at a time (rows r = warp, warp + 8, ...): the row's
// logits over the page's keys (lane = key), its weights and their sum, its
// value sum (lane = four dimensions) and the ratio, all inside the warp.
constexpr int kMaxPage = 64;
constexpr int kMaxRows = 64;
constexpr int kPageThreads = 256;

size_t page_smem_bytes() {
  return static_cast<size_t>(kMaxRows + 2 * kMaxPage) * 128 * 2;   // q, k, v rows (bf16)
}

__global__ void __launch_bounds__(kPageThreads) effect_page_kernel(const EffectArgs a) {
  extern __shared__ uint8_t psm_raw[];
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(psm_raw);             // [R][128]
  __nv_bfloat16* ks = qs + kMaxRows * 128;                                    // [len][128]
  __nv_bfloat16* vs = ks + kMaxPage * 128;                                    // [len][128]
  __shared__ float wmax[kPageThreads / 32];
  const int p = blockIdx.x, u = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per_b = a.L * a.Hkv;
  const int b = u / per_b, l = (u % per_b) / a.Hkv, g = u % a.Hkv;
  const int start = a.page_start[static_cast<int64_t>(b) * a.n_pages + p];
  const int len = a.page_len[static_cast<int64_t>(b) * a.n_pages + p];
  const int R = a.R;
  const int64_t row0 = (static_cast<int64_t>(b * a.L + l) * a.n_pages + p) * (a.Hkv * R) + g * R;
  const bool bad = len < 0 || len > kMaxPage || start < 0 || static_cast<int64_t>(start) + len > a.T;
  if (bad || len == 0) {
    // an empty or malformed page deletes nothing: s = 0, u = 0, no ratio
    for (int i = tid; i < R * 128; i += kPageThreads) a.u[row0 * 128 + i] = 0.f;
    if (tid < R) a.s[row0 + tid] = 0.f;
    if (bad && tid == 0 && a.unit_status) a.unit_status[u] = KVC_UNIT_BAD_INDEX;
    return;
  }
  {
    const uint4* qg = reinterpret_cast<const uint4*>(a.q + static_cast<int64_t>(u) * R * 128);
    uint4* q4 = reinterpret_cast<uint4*>(qs);
    for (int i = tid; i < R * 16; i += kPageThreads) q4[i] = __ldg(qg + i);
    const int64_t off = (static_cast<int64_t>(u) * a.T + start) * 128;
    const uint4* kg = reinterpret_cast<const uint4*>(a.k + off);
    const uint4* vg = reinterpret_cast<const uint4*>(a.v + off);
    uint4* k4 = reinterpret_cast<uint4*>(ks);
    uint4* v4 = reinterpret_cast<uint4*>(vs);
    for (int i = tid; i < len * 16; i += kPageThreads) {
      k4[i] = __ldg(kg + i);
      v4[i] = __ldg(vg + i);
    }
  }
  __syncthreads();
  const int64_t last0 = a.T - a.W;          // row w sees indices <= last0 + w
  float mx = 0.f;
  for (int r = warp; r < R; r += kPageThreads / 32) {
    const float lse2 = a.lse[static_cast<int64_t>(u) * R + r] * 1.4426950408889634f;
    const int64_t last = last0 + (r % a.W);
    const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(qs + r * 128);
    // weights of keys lane and lane + 32; each lane starts its dot product at
    // a different pair, so the 256-byte-strided key rows hit different banks
    float aw[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      if (i < len && static_cast<int64_t>(start) + i <= last) {
        const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(ks + i * 128);
        float z0 = 0.f, z1 = 0.f;
#pragma unroll 8
        for (int t = 0; t < 64; ++t) {
          const int tt = (t + lane) & 63;
          const float2 qf = __bfloat1622float2(q2[tt]);
          const float2 kf = __bfloat1622float2(k2[tt]);
          z0 = fmaf(qf.x, kf.x, z0);
          z1 = fmaf(qf.y, kf.y, z1);
        }
        aw[h] = ex2_approx((z0 + z1) * a.scale_log2 - lse2);
      }
    }
    float sr = aw[0] + aw[1];
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) sr += __shfl_xor_sync(0xffffffffu, sr, o2);
    // value sum: lane owns dimensions 4 lane .. 4 lane + 3
    float4 ur = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < len; ++i) {
      const float w = __shfl_sync(0xffffffffu, aw[i >> 5], i & 31);
      const uint2 vv = *reinterpret_cast<const uint2*>(vs + i * 128 + 4 * lane);
      const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vv.x));
      const float2 v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vv.y));
      ur.x = fmaf(w, v01.x, ur.x);
      ur.y = fmaf(w, v01.y, ur.y);
      ur.z = fmaf(w, v23.x, ur.z);
      ur.w = fmaf(w, v23.y, ur.w);
    }
    const float4 od = reinterpret_cast<const float4*>(a.o + (static_cast<int64_t>(u) * R + r) * 128)[lane];
    const float dx = ur.x - sr * od.x, dy = ur.y - sr * od.y, dz = ur.z - sr * od.z, dw = ur.w - sr * od.w;
    float nn = dx * dx + dy * dy + dz * dz + dw * dw;
    float oo = od.x * od.x + od.y * od.y + od.z * od.z + od.w * od.w;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
      nn += __shfl_xor_sync(0xffffffffu, nn, o2);
      oo += __shfl_xor_sync(0xffffffffu, oo, o2);
    }
    reinterpret_cast<float4*>(a.u + (row0 + r) * 128)[lane] = ur;
    if (lane == 0) a.s[row0 + r] = sr;
    const float om = 1.f - sr;
    float ratio;
    if (om <= 0.f) ratio = INFINITY;
    else if (oo == 0.f) ratio = nn == 0.f ? 0.f : INFINITY;
    else ratio = sqrtf(nn) / (om * sqrtf(oo));
    mx = fmaxf(mx, ratio);
  }
  if (lane == 0) wmax[warp] = mx;
  __syncthreads();
  if (tid == 0) {
    float m = 0.f;
    for (int w2 = 0; w2 < kPageThreads / 32; ++w2) m = fmaxf(m, wmax[w2]);
    // ratios are >= 0, so their bit patterns order like the values
    atomicMax(reinterpret_cast<int*>(a.effect + static_cast<int64_t>(b * a.L + l) * a.n_pages + p),
              __float_as_int(m));
  }
}

// Lifecycle states (Eqs. 8-10) and the greedy retirement set (Eq. 11) of
// one layer of one sequence per block.
constexpr int kCommitThreads = 1024;
constexpr uint8_t kStateUncertain = 0, kStateCompletion = 1, kStateDormant = 2, kStateNewlyActive = 3,
                  kStateStillActive = 4, kStateNotCompared = 255;

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(const CommitArgs a) {
  extern __shared__ float csm[];
  const int NP = a.n_pages, NR = a.Hq * a.W;
  float* rm = csm;
  float* rp = rm + NP;
  float* sd = rp + NP;            // [NR] accepted weight per row
  float* oo = sd + NR;            // [NR] ||o_r||^2
  int* order = reinterpret_cast<int*>(oo + NR);
  uint8_t* st = reinterpret_cast<uint8_t*>(order + NP);
  uint8_t* cmp = st + NP;
  __shared__ float wmax[32];
  __shared__ int s_accept;
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t rbase = (static_cast<int64_t>(b) * a.L + a.layer) * NP;
  if (tid < NP) {
    rm[tid] = a.r_minus[rbase + tid];
    rp[tid] = a.r_plus[rbase + tid];
    cmp[tid] = a.compared[static_cast<int64_t>(b) * NP + tid] != 0;
  }
  const int n_c = __syncthreads_count(tid < NP && a.compared[static_cast<int64_t>(b) * NP + tid] != 0);
  if (tid < NP) {
    uint8_t state = kStateNotCompared;
    if (cmp[tid]) {
      int cm = 0, cp = 0;
      for (int j = 0; j < NP; ++j) {
        if (!cmp[j]) continue;
        cm += rm[j] < rm[tid];
        cp += rp[j] < rp[tid];
      }
      // the percentile in double, as cm / n_c compares exactly with rho
      const double pm = static_cast<double>(cm) / n_c, pp = static_cast<double>(cp) / n_c;
      const bool hm = rm[tid] >= a.tau_use && pm >= static_cast<double>(a.rho_use);
      const bool lm = rm[tid] <= a.tau_dead && pm <= static_cast<double>(a.rho_dead);
      const bool hp = rp[tid] >= a.tau_use && pp >= static_cast<double>(a.rho_use);
      const bool lp = rp[tid] <= a.tau_dead && pp <= static_cast<double>(a.rho_dead);
      state = (hm && lp) ? kStateCompletion
            : (lm && lp) ? kStateDormant
            : (lm && hp) ? kStateNewlyActive
            : (hm && hp) ? kStateStillActive
                         : kStateUncertain;
    }
    st[tid] = state;
    a.state[static_cast<int64_t>(b) * NP + tid] = state;
    a.retire[static_cast<int64_t>(b) * NP + tid] = 0;
    if (a.joint) a.joint[static_cast<int64_t>(b) * NP + tid] = -1.f;
  }
  __syncthreads();
  // candidates by increasing R+, then decreasing R-, then lower index
  const bool cand = tid < NP && st[tid] == kStateCompletion;
  if (cand) {
    int rank = 0;
    for (int j = 0; j < NP; ++j) {
      if (st[j] != kStateCompletion || j == tid) continue;
      rank += rp[j] < rp[tid] || (rp[j] == rp[tid] && (rm[j] > rm[tid] || (rm[j] == rm[tid] && j < tid)));
    }
    order[rank] = tid;
  }
  const int n_cand = __syncthreads_count(cand);
  const int64_t obase = (static_cast<int64_t>(b) * a.L + a.layer) * NR;       // rows of o
  float* acc = a.acc + static_cast<int64_t>(b) * NR * 128;
  for (int r = warp; r < NR; r += kCommitThreads / 32) {
    const float4 o4 = reinterpret_cast<const float4*>(a.o + (obase + r) * 128)[lane];
    float x = o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o2);
    if (lane == 0) {
      oo[r] = x;
      sd[r] = 0.f;
    }
    reinterpret_cast<float4*>(acc + static_cast<int64_t>(r) * 128)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  for (int k = 0; k < n_cand; ++k) {
    const int E = order[k];
    const int64_t ebase = ((static_cast<int64_t>(b) * a.L + a.layer) * NP + E) * NR;   // rows of s / u
    float mx = 0.f;
    for (int r = warp; r < NR; r += kCommitThreads / 32) {
      const float t = sd[r] + a.s[ebase + r];
      const float4 o4 = reinterpret_cast<const float4*>(a.o + (obase + r) * 128)[lane];
      const float4 u4 = reinterpret_cast<const float4*>(a.u + (ebase + r) * 128)[lane];
      const float4 c4 = reinterpret_cast<const float4*>(acc + static_cast<int64_t>(r) * 128)[lane];
      const float dx = c4.x + u4.x - t * o4.x, dy = c4.y + u4.y - t * o4.y;
      const float dz = c4.z + u4.z - t * o4.z, dw = c4.w + u4.w - t * o4.w;
      float nn = dx * dx + dy * dy + dz * dz + dw * dw;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) nn += __shfl_xor_sync(0xffffffffu, nn, o2);
      const float om = 1.f - t;
      float ratio;
      if (om <= 0.f) ratio = INFINITY;
      else if (oo[r] == 0.f) ratio = nn == 0.f ? 0.f : INFINITY;
      else ratio = sqrtf(nn) / (om * sqrtf(oo[r]));
      mx = fmaxf(mx, ratio);
    }
    if (lane == 0) wmax[warp] = mx;
    __syncthreads();
    if (tid == 0) {
      float m = 0.f;
      for (int w2 = 0; w2 < kCommitThreads / 32; ++w2) m = fmaxf(m, wmax[w2]);
      s_accept = m <= a.tau_joint;
      if (a.joint) a.joint[static_cast<int64_t>(b) * NP + E] = m;
      if (s_accept) a.retire[static_cast<int64_t>(b) * NP + E] = 1;
    }
    __syncthreads();
    if (s_accept) {
      for (int r = warp; r < NR; r += kCommitThreads / 32) {
        const float t = sd[r] + a.s[ebase + r];
        const float4 u4 = reinterpret_cast<const float4*>(a.u + (ebase + r) * 128)[lane];
        float4* cp4 = reinterpret_cast<float4*>(acc + static_cast<int64_t>(r) * 128) + lane;
        const float4 c4 = *cp4;
        *cp4 = make_float4(c4.x + u4.x, c4.y + u4.y, c4.z + u4.z, c4.w + u4.w);
        __syncwarp();
        if (lane == 0) sd[r] = t;
      }
    }
    __syncthreads();
  }
}

// Pending pages protected by decreasing R- (ties: lower index) while the
// token count stays within B_N and the page count within max_pages (Eq. 12);
// the walk stops at the first page that does not fit.
__global__ void __launch_bounds__(kCommitThreads) protect_kernel(const ProtectArgs a) {
  extern __shared__ float psm2[];
  const int NP = a.n_pages;
  float* rm = psm2;
  int* order = reinterpret_cast<int*>(rm + NP);
  uint8_t* pend = reinterpret_cast<uint8_t*>(order + NP);
  uint8_t* prot = pend + NP;
  const int b = blockIdx.x, tid = threadIdx.x;
  if (tid < NP) {
    rm[tid] = a.r_minus[(static_cast<int64_t>(b) * a.L + a.layer) * NP + tid];
    pend[tid] = a.pending[static_cast<int64_t>(b) * NP + tid] != 0;
    prot[tid] = 0;
  }
  __syncthreads();
  const bool mine = tid < NP && pend[tid];
  if (mine) {
    int rank = 0;
    for (int j = 0; j < NP; ++j)
      if (pend[j] && j != tid) rank += rm[j] > rm[tid] || (rm[j] == rm[tid] && j < tid);
    order[rank] = tid;
  }
  const int n = __syncthreads_count(mine);
  if (tid == 0) {
    int64_t used = 0;
    int taken = 0;
    for (int k = 0; k < n; ++k) {
      const int i = order[k];
      const int len = a.page_len[static_cast<int64_t>(b) * NP + i];
      if (taken + 1 > a.max_pages || used + len > a.budget_tokens) break;
      prot[i] = 1;
      used += len;
      ++taken;
    }
  }
  __syncthreads();
  if (tid < NP) a.protect[static_cast<int64_t>(b) * NP + tid] = prot[tid];
}

// Checkpoint flags (Eq. 13): protected pages PROTECT, retired pages EXCLUDE.
__global__ void __launch_bounds__(64) flags_kernel(const FlagArgs a) {
  const int p = blockIdx.x, b = blockIdx.y;
  const int64_t idx = static_cast<int64_t>(b) * a.n_pages + p;
  const bool prot = a.protect && a.protect[idx];
  const bool ret = a.retire && a.retire[idx];
  if (!prot && !ret) return;
  const int start = a.page_start[idx], len = a.page_len[idx];
  if (len <= 0 || start < 0 || static_cast<int64_t>(start) + len > a.T) return;
  uint8_t* f = a.flags + static_cast<int64_t>(b) * a.T + start;
  for (int j = threadIdx.x; j < len; j += 64) {
    const uint8_t x = f[j];
    f[j] = prot ? static_cast<uint8_t>((x & ~KVC_FLAG_EXCLUDE) | KVC_FLAG_PROTECT)
                : static_cast<uint8_t>((x & ~KVC_FLAG_PROTECT) | KVC_FLAG_EXCLUDE);
  }
}

}  // namespace

size_t effect_smem_bytes(int Rp, int n_stages) {
  return static_cast<size_t>(2 * kChunk) + static_cast<size_t>(n_stages) * kTile +
         static_cast<size_t>(8) * Rp * 128 + static_cast<size_t>(2 * n_stages + 13) * 8 + 16 +
         2 * 128 * 4 + 1024;
}

cudaError_t launch_effect(const EffectArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                          const CUtensorMap& tmap_q, int grid, size_t smem_bytes, cudaStream_t stream) {
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const EffectArgs) =
      a.R <= 32 ? effect_attn_kernel<32> : effect_attn_kernel<64>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes));
  if (err != cudaSuccess) return err;
  kern<<<grid, kEffThreads, smem_bytes, stream>>>(tmap_k, tmap_v, tmap_q, a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  effect_merge_kernel<<<a.U * a.R, 128, 0, stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const size_t psm = page_smem_bytes();
  if ((err = cudaFuncSetAttribute(effect_page_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(psm))) != cudaSuccess)
    return err;
  if (a.n_pages > 0) effect_page_kernel<<<dim3(a.n_pages, a.U), kPageThreads, psm, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream) {
  const int NR = a.Hq * a.W;
  const size_t smem = static_cast<size_t>(a.n_pages) * (4 + 4 + 4 + 2) + static_cast<size_t>(NR) * 8 + 16;
  cudaError_t err = cudaFuncSetAttribute(commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  commit_kernel<<<a.B, kCommitThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_protect(const ProtectArgs& a, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(a.n_pages) * (4 + 4 + 2) + 16;
  protect_kernel<<<a.B, kCommitThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_flags(const FlagArgs& a, cudaStream_t stream) {
  if (a.n_pages == 0) return cudaSuccess;
  flags_kernel<<<dim3(a.n_pages, a.B), 64, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc
