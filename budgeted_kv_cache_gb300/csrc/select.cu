// Deterministic budgeted selection, one CTA per unit (1,024 threads; 256 for
// the general kernel on units of at most 16,384 items), and a multi-CTA form
// for token / page mode units of more than 32,768 items (end of the file).
//
// Token / page mode: the kept set is the forced items plus the k best
// eligible items in the order (score descending, index ascending) -- the
// "keep the top-B by the sum" rule of PACE Sec. 3.1 with CommitKV's
// |I| <= B (Eq. 4) and protected pages always kept (Eq. 13).
// Byte mode: PASK's floor-constrained allocation (App. B.4): floors are
// charged first, then the remainder promotes the longest prefix of the same
// order to bf16.
//
// Both are one weighted radix select on a 32-bit order key (1 per item in
// token mode, the upgrade cost in byte mode): four 8-bit digit passes each
// build per-warp shared-memory histograms of the items still matching the
// key prefix and locate, with a block scan, the bin where the running weight
// crosses the target (the register-resident token / page kernel stops at
// the first level whose threshold bin is taken whole).  Items above the final
// key are taken; items equal to it are taken in index order while the
// running weight still fits.  A last phase writes the kept indices in index
// order: each warp owns a contiguous range of items and the warps' offsets
// come from two 32-entry scans, so every list comes out ascending.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kThreads = 1024;
constexpr unsigned kFull = 0xffffffffu;

// Order-preserving map of a canonical fp32 score to a nonzero 32-bit key:
// -0 -> +0, NaN -> -inf; larger score -> larger key.  0 is reserved for
// "not a candidate".
__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t b = __float_as_uint(s);
  if (isnan(s)) b = 0xff800000u;          // -inf
  if (b == 0x80000000u) b = 0;            // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <typename V>
__device__ __forceinline__ V warp_incl_scan(V x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const V y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive scan over the NW warps of the block (wtot: 32 entries); `total`
// gets the sum.
template <typename V, int NW = 32>
__device__ __forceinline__ V block_excl_scan(V v, V* wtot, V& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const V incl = warp_incl_scan(v, lane);
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const V w = warp_incl_scan(lane < NW ? wtot[lane] : V(0), lane);
    wtot[lane] = w;
  }
  __syncthreads();
  const V base = warp ? wtot[warp - 1] : V(0);
  total = wtot[NW - 1];
  __syncthreads();
  return base + incl - v;
}

struct Item {
  uint32_t key;    // 0 = not a candidate
  uint8_t base;    // action if not promoted
};

struct Ctx {
  const SelectArgs* a;
  int u, b, group;
  int64_t n;
  uint32_t cost[4];
  const float* scores;
  const uint8_t* flags;
  const uint8_t* tags;
};

__device__ __forceinline__ Item eval_item(const Ctx& c, int64_t i, int& err) {
  const SelectArgs& a = *c.a;
  const bool window = i < a.sink_items || i >= c.n - a.recent_items;
  const uint8_t f = c.flags ? c.flags[i] : 0;
  const bool protect = f & KVC_FLAG_PROTECT;
  const bool exclude = f & KVC_FLAG_EXCLUDE;
  if (protect && exclude) err |= 1;
  const bool forced = window || protect;
  const bool excluded = exclude && !window;
  Item it;
  if (!a.byte_mode) {
    it.base = forced ? KVC_ACT_BF16 : KVC_ACT_RELEASE;
    it.key = (!forced && !excluded) ? order_key(c.scores[i]) : 0u;
  } else {
    const uint32_t tag = c.tags[i];
    uint32_t floor_act = KVC_ACT_RELEASE;
    if (tag >= static_cast<uint32_t>(a.n_tags)) {
      err |= 2;
    } else {
      floor_act = a.table[tag * a.n_groups + c.group];
      if (floor_act > KVC_ACT_BF16) {
        err |= 2;
        floor_act = KVC_ACT_RELEASE;
      }
    }
    it.base = forced ? KVC_ACT_BF16 : (excluded ? KVC_ACT_RELEASE : floor_act);
    it.key = (!forced && !excluded && it.base != KVC_ACT_BF16) ? order_key(c.scores[i]) : 0u;
  }
  return it;
}

__device__ __forceinline__ uint32_t item_weight(const Ctx& c, const Item& it) {
  return c.a->byte_mode ? c.cost[KVC_ACT_BF16] - c.cost[it.base] : 1u;
}

// NW warps per CTA: 32 for long units, 8 for units of at most 16,384 items
// (byte mode at T = 8,192: four times as many CTAs per SM).
template <int NW>
__global__ void __launch_bounds__(NW * 32, NW == 32 ? 1 : 1024 / (NW * 32)) select_kernel(const __grid_constant__ SelectArgs a) {
  constexpr int kT = NW * 32;               // threads of the CTA
  __shared__ uint32_t hist_w[NW * 256];     // per-warp histograms
  __shared__ unsigned long long wtot[32];
  __shared__ unsigned long long red[4];
  __shared__ int s_bin;
  __shared__ uint32_t s_kmin, s_kmax;
  __shared__ unsigned long long s_above;
  extern __shared__ uint8_t dsm[];

  const int tid = threadIdx.x, lane = tid & 31;
  Ctx c;
  c.a = &a;
  c.u = blockIdx.x;
  c.b = c.u / (a.L * a.Hkv);
  const int l = (c.u / a.Hkv) % a.L;
  c.n = a.n_items;
  c.scores = a.scores + static_cast<int64_t>(c.u) * c.n;
  c.flags = a.flags ? a.flags + static_cast<int64_t>(c.b) * c.n : nullptr;
  c.tags = a.byte_mode ? a.tags + static_cast<int64_t>(c.b) * a.T : nullptr;
  c.group = 0;
  if (a.byte_mode)
    for (int g = 0; g < a.n_groups; ++g)
      if (l >= (g * a.L + a.n_groups - 1) / a.n_groups) c.group = g;
  const uint32_t sc = a.quant_mode == KVC_QUANT_G32_BF16 ? 2u * (a.d / 32) : 2u;
  c.cost[KVC_ACT_RELEASE] = 0;
  c.cost[KVC_ACT_INT4] = 2u * (a.d / 2 + sc);
  c.cost[KVC_ACT_INT8] = 2u * (a.d + sc);
  c.cost[KVC_ACT_BF16] = 4u * a.d;

  uint32_t* ckey = reinterpret_cast<uint32_t*>(dsm);
  uint8_t* cbase = dsm + 4 * (a.cache_items ? c.n : 0);

  auto get = [&](int64_t i, int& err) -> Item {
    if (a.cache_items) {
      Item it;
      it.key = ckey[i];
      it.base = cbase[i];
      return it;
    }
    return eval_item(c, i, err);
  };

  // ---------------- phase A: classify, count, charge floors
  // Four independent items per thread per iteration keep several loads in
  // flight.  The smallest and largest candidate keys are kept too: the radix
  // passes below start at the highest bit where they differ.
  if (tid < 4) red[tid] = 0;
  if (tid == 0) {
    s_kmin = 0xffffffffu;
    s_kmax = 0u;
  }
  __syncthreads();
  unsigned long long n_forced = 0, n_cand = 0, floor_bytes = 0;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  int err = 0;
  for (int64_t i0 = tid; i0 < c.n; i0 += 4 * kT) {
    Item it[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t i = i0 + k * kT;
      it[k].key = 0;
      it[k].base = KVC_ACT_RELEASE;
      if (i < c.n) it[k] = eval_item(c, i, err);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t i = i0 + k * kT;
      if (i >= c.n) continue;
      if (a.cache_items) {
        ckey[i] = it[k].key;
        cbase[i] = it[k].base;
      }
      n_forced += (!a.byte_mode && it[k].base == KVC_ACT_BF16);
      n_cand += (it[k].key != 0);
      floor_bytes += c.cost[it[k].base];
      if (it[k].key != 0) {
        kmin = min(kmin, it[k].key);
        kmax = max(kmax, it[k].key);
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    n_forced += __shfl_xor_sync(kFull, n_forced, o);
    n_cand += __shfl_xor_sync(kFull, n_cand, o);
    floor_bytes += __shfl_xor_sync(kFull, floor_bytes, o);
    err |= __shfl_xor_sync(kFull, err, o);
    kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
  }
  if (lane == 0) {
    atomicAdd(&red[0], n_forced);
    atomicAdd(&red[1], n_cand);
    atomicAdd(&red[2], floor_bytes);
    atomicOr(reinterpret_cast<unsigned int*>(&red[3]), static_cast<unsigned int>(err));
    atomicMin(&s_kmin, kmin);
    atomicMax(&s_kmax, kmax);
  }
  __syncthreads();
  n_forced = red[0];
  n_cand = red[1];
  floor_bytes = red[2];
  err = static_cast<int>(red[3]);
  kmin = s_kmin;
  kmax = s_kmax;

  int32_t* cnt = a.kept_count;
  if (err) {
    if (tid < KVC_N_POOLS) cnt[tid * a.U + c.u] = 0;
    if (tid == 0) {
      a.unit_status[c.u] = (err & 1) ? KVC_UNIT_BAD_FLAGS : KVC_UNIT_BAD_INDEX;
      if (a.floor_excess) a.floor_excess[c.u] = 0;
    }
    return;
  }

  bool sel_none = false, sel_all = false;
  unsigned long long t = 0;      // target weight still to place
  long long excess = 0;
  if (!a.byte_mode) {
    if (n_forced > static_cast<unsigned long long>(a.budget_items)) {
      if (tid < KVC_N_POOLS) cnt[tid * a.U + c.u] = 0;
      if (tid == 0) {
        a.unit_status[c.u] = KVC_UNIT_OVER_BUDGET;
        if (a.floor_excess) a.floor_excess[c.u] = 0;
      }
      return;
    }
    const unsigned long long k =
        min(static_cast<unsigned long long>(a.budget_items) - n_forced, n_cand);
    if (k == 0) sel_none = true; else t = k - 1;
  } else {
    const long long rem = a.budget_bytes - static_cast<long long>(floor_bytes);
    if (rem < 0) {
      excess = -rem;
      sel_none = true;
    } else {
      t = static_cast<unsigned long long>(rem);
    }
  }

  // ---------------- phase B: weighted radix select of the crossing key
  // 8-bit digits, most significant first, over the bits where candidate
  // keys can differ (those above the highest bit of kmin ^ kmax are common).
  // Each warp builds a private 256-bin histogram of its own contiguous item
  // range, the 32 histograms are summed, and a block scan over the bins
  // (highest first) finds the bin where the running weight crosses t.
  uint32_t tau = 0;
  if (!sel_none && n_cand > 0) {
    const int warp = tid >> 5;
    const int64_t per_w = (c.n + NW * 32 - 1) / (NW * 32) * 32;
    const int64_t w_lo = min(c.n, static_cast<int64_t>(warp) * per_w);
    const int64_t w_hi = min(c.n, w_lo + per_w);
    uint32_t* whist = hist_w + warp * 256;
    const int top = (kmin == kmax) ? -1 : 31 - __clz(kmin ^ kmax);
    uint64_t pfx = static_cast<uint64_t>(kmax) >> (top + 1);   // common high bits
    for (int hi = top; hi >= 0; hi -= 8) {
      const int shift = max(0, hi - 7);
      const int width = hi - shift + 1;
      const uint32_t nb = 1u << width;
      for (int i = lane; i < 256; i += 32) whist[i] = 0;
      __syncwarp();
      for (int64_t i = w_lo + lane; i < w_hi; i += 32) {
        const Item it = get(i, err);
        if (it.key != 0 && (static_cast<uint64_t>(it.key) >> (hi + 1)) == pfx)
          atomicAdd(&whist[(it.key >> shift) & (nb - 1)], item_weight(c, it));
      }
      if (tid == 0) s_bin = -1;
      __syncthreads();
      // thread b < nb sums bin nb - 1 - b over the warps (descending bin order)
      unsigned long long local = 0;
      if (tid < static_cast<int>(nb)) {
        const int bn = static_cast<int>(nb) - 1 - tid;
        for (int w = 0; w < NW; ++w) local += hist_w[w * 256 + bn];
      }
      unsigned long long total;
      const unsigned long long run = block_excl_scan<unsigned long long, NW>(local, wtot, total);
      if (tid < static_cast<int>(nb) && run <= t && t < run + local) {
        s_bin = static_cast<int>(nb) - 1 - tid;
        s_above = run;
      }
      __syncthreads();
      const int bn = s_bin;
      const unsigned long long above = s_above;
      __syncthreads();
      if (bn < 0) {          // everything fits (byte mode only)
        sel_all = true;
        break;
      }
      t -= above;
      pfx = (pfx << width) | static_cast<uint32_t>(bn);
    }
    tau = static_cast<uint32_t>(pfx);
    // (one distinct key: no pass runs, every candidate is a tie at tau)
  } else if (!sel_none) {
    sel_all = true;          // no candidates: nothing to promote
  }

  // ---------------- phase C: write the kept lists in index order
  // Warp w owns the contiguous item range [w_lo, w_hi) and walks it 32 items
  // at a time, twice.  Walk 1 counts, per pool, the items whose action does
  // not depend on a tie, and the ties (items with key == tau) with their
  // weight.  Ties are taken in index order while their running weight fits,
  // so after a scan of the tie weights over the warps each warp knows how
  // many of its ties are kept (a warp straddling the cut in byte mode counts
  // its own).  A scan of the per-pool counts gives every warp its output
  // offsets; walk 2 repeats the decisions and writes each kept item.
  __shared__ unsigned long long s_tie[32];
  __shared__ uint32_t s_pool[KVC_N_POOLS][32];
  const int warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int64_t per_w = (c.n + NW * 32 - 1) / (NW * 32) * 32;
  const int64_t w_lo = min(c.n, static_cast<int64_t>(warp) * per_w);
  const int64_t w_hi = min(c.n, w_lo + per_w);
  const unsigned long long tie_slack = a.byte_mode ? 0ull : 1ull;
  const int P = a.page_size;

  auto tie_weight = [&](const Item& it) -> unsigned long long {
    const bool cand = it.key != 0 && !sel_none;
    return (cand && !sel_all && it.key == tau) ? item_weight(c, it) : 0ull;
  };
  auto decide = [&](const Item& it, unsigned long long tie_before, unsigned long long tw) -> uint32_t {
    const bool cand = it.key != 0 && !sel_none;
    const bool promoted =
        cand && (sel_all || it.key > tau || (tw > 0 && tie_before + tw <= t + tie_slack));
    return promoted ? KVC_ACT_BF16 : it.base;
  };
  auto load = [&](int64_t i) -> Item {
    Item it;
    it.key = 0;
    it.base = KVC_ACT_RELEASE;
    if (i < w_hi) it = get(i, err);
    return it;
  };

  // walk 1
  uint32_t pc[KVC_N_POOLS] = {0, 0, 0};       // tie-independent items per pool
  uint32_t tb_pc[KVC_N_POOLS] = {0, 0, 0};    // ties per pool of their unpromoted action
  uint32_t tie_n = 0;
  unsigned long long tie_w = 0;
  for (int64_t i0 = w_lo; i0 < w_hi; i0 += 32) {
    const Item it = load(i0 + lane);
    const unsigned long long tw = tie_weight(it);
    const bool tie = tw != 0;
    const uint32_t act = (i0 + lane < w_hi && !tie) ? decide(it, 0, 0) : KVC_ACT_RELEASE;
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) pc[q] += __popc(__ballot_sync(kFull, act == q + 1u));
    const unsigned tm = __ballot_sync(kFull, tie);
    if (tm) {
      tie_n += __popc(tm);
      unsigned long long ws = tw;
      for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(kFull, ws, o);
      tie_w += ws;
#pragma unroll
      for (int q = 0; q < KVC_N_POOLS; ++q) tb_pc[q] += __popc(__ballot_sync(kFull, tie && it.base == q + 1u));
    }
  }
  if (lane == 0) s_tie[warp] = a.byte_mode ? tie_w : tie_n;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long v = lane < NW ? s_tie[lane] : 0ull;
    s_tie[lane] = warp_incl_scan(v, lane) - v;     // exclusive offsets
  }
  __syncthreads();
  const unsigned long long tie_off = s_tie[warp];
  // kept ties of this warp: a prefix of its ties in index order
  const unsigned long long my_tie_total = a.byte_mode ? tie_w : tie_n;
  bool partial = false;
  uint32_t prom = 0;
  if (tie_n > 0) {
    if (tie_off + my_tie_total <= t + tie_slack) prom = tie_n;
    else if (tie_off >= t + tie_slack) prom = 0;
    else if (!a.byte_mode) prom = static_cast<uint32_t>(t + 1 - tie_off);
    else partial = true;
  }
  if (partial) {              // byte mode, the warp where the cut falls: count exactly
    unsigned long long tie_run = tie_off;
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) tb_pc[q] = 0;
    prom = 0;
    for (int64_t i0 = w_lo; i0 < w_hi; i0 += 32) {
      const Item it = load(i0 + lane);
      const unsigned long long tw = tie_weight(it);
      if (!__any_sync(kFull, tw != 0)) continue;
      const unsigned long long incl = warp_incl_scan(tw, lane);
      const uint32_t act = decide(it, tie_run + incl - tw, tw);
      tie_run += __shfl_sync(kFull, incl, 31);
      prom += __popc(__ballot_sync(kFull, tw != 0 && act == KVC_ACT_BF16));
#pragma unroll
      for (int q = 0; q < KVC_N_POOLS; ++q)
        tb_pc[q] += __popc(__ballot_sync(kFull, tw != 0 && act != KVC_ACT_BF16 && act == q + 1u));
    }
  } else if (prom == tie_n) {
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) tb_pc[q] = 0;
  } else if (prom > 0) {       // count mode: ties are never stored unpromoted
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) tb_pc[q] = 0;
  }
  if (!a.byte_mode) {
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) tb_pc[q] = 0;   // unpromoted token-mode ties are released
  }
  pc[KVC_POOL_BF16] += prom;
#pragma unroll
  for (int q = 0; q < KVC_N_POOLS; ++q) pc[q] += tb_pc[q];
  if (lane == 0) {
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) s_pool[q][warp] = pc[q];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) {
      const uint32_t v = lane < NW ? s_pool[q][lane] : 0u;
      s_pool[q][lane] = warp_incl_scan(v, lane);        // inclusive: entry 31 is the total
    }
  }
  __syncthreads();
  // walk 2: write
  uint32_t pos_run[KVC_N_POOLS];
#pragma unroll
  for (int q = 0; q < KVC_N_POOLS; ++q) pos_run[q] = warp ? s_pool[q][warp - 1] : 0u;
  unsigned long long tie_run = tie_off;
  for (int64_t i0 = w_lo; i0 < w_hi; i0 += 32) {
    const int64_t i = i0 + lane;
    const Item it = load(i);
    const unsigned long long tw = tie_weight(it);
    unsigned long long incl = 0;
    if (__any_sync(kFull, tw != 0)) incl = warp_incl_scan(a.byte_mode ? tw : (tw != 0 ? 1ull : 0ull), lane);
    const unsigned long long tb_here = a.byte_mode ? tw : (tw != 0 ? 1ull : 0ull);
    const uint32_t act = (i < w_hi) ? decide(it, tie_run + incl - tb_here, tb_here) : KVC_ACT_RELEASE;
    tie_run += __shfl_sync(kFull, incl, 31);
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) {
      const unsigned m = __ballot_sync(kFull, act == q + 1u);
      if (act == q + 1u) {
        const uint32_t pos = pos_run[q] + __popc(m & lt_mask);
        int32_t* dst = a.kept_idx + (static_cast<int64_t>(q) * a.U + c.u) * a.capacity;
        if (P == 1) {
          dst[pos] = static_cast<int32_t>(i);
        } else {
          for (int k = 0; k < P; ++k)
            dst[static_cast<int64_t>(pos) * P + k] = static_cast<int32_t>(i * P + k);
        }
      }
      pos_run[q] += __popc(m);
    }
  }
  if (tid < KVC_N_POOLS) cnt[tid * a.U + c.u] = static_cast<int32_t>(s_pool[tid][31]) * P;
  if (tid == 0) {
    a.unit_status[c.u] = KVC_UNIT_OK;
    if (a.floor_excess) a.floor_excess[c.u] = excess;
  }
}

// ----------------------------------------------------------------------------
// Token / page mode with at most 32,768 items per unit.  Item q * 1024 + t
// (q < 32) belongs to thread t, and the keys stay in registers through the
// radix passes.  With kBulk (the unit's scores 16-byte aligned and a
// multiple of 16 bytes long) the scores come into shared memory through
// bulk copies issued by one warp, which bring the unit's 128 KB in about
// half the time of 32 rounds of 4-byte loads by every thread; otherwise
// every thread requests its 32 scores before it uses any.  In index order
// the items of slab q come thread by thread, so the write-out needs one
// ballot per slab and one block scan over the 1,024 (slab, warp) counts.
// Same rule and same results as select_kernel (forced items, then the top k
// candidates by (score descending, index ascending)).
constexpr int kFastSlabs = 32;
constexpr int kFastMaxItems = kThreads * kFastSlabs;
constexpr uint32_t kFastCopyChunk = 16384;        // bytes per bulk copy (one per lane of warp 0)

template <bool kBulk>
__global__ void __launch_bounds__(kThreads, 1) select_fast_kernel(const __grid_constant__ SelectArgs a) {
  extern __shared__ __align__(16) float s_sc[];   // kBulk: the unit's scores
  __shared__ uint32_t hist_w[32 * 256];     // per-warp histograms
  __shared__ uint32_t scan_w[32];
  __shared__ uint32_t s_cnt[kFastSlabs * 32];
  __shared__ uint32_t s_red[4];
  __shared__ uint32_t s_kmin, s_kmax;
  __shared__ uint32_t s_w8[8];              // bin-scan totals of warps 0-7
  __shared__ int s_bin;
  __shared__ uint32_t s_above, s_bincnt;
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = blockIdx.x;
  const int b = u / (a.L * a.Hkv);
  const int n = static_cast<int>(a.n_items);
  const float* sc = a.scores + static_cast<int64_t>(u) * n;
  const uint8_t* fl = a.flags ? a.flags + static_cast<int64_t>(b) * n : nullptr;
  const unsigned lt_mask = (1u << lane) - 1u;
  int32_t* cnt = a.kept_count;

  // ---------------- classify
  float v[kFastSlabs];
  uint8_t f[kFastSlabs];
  if constexpr (kBulk) {
    const uint32_t bar = smem_u32(&s_bar);
    const uint32_t bytes = static_cast<uint32_t>(n) * 4u;
    if (warp == 0) {
      if (lane == 0) {
        s_abort = 0;
        mbar_init(bar, 1);
        fence_barrier_init();
        // (a.stall_unit: a test waits for 16 bytes more than the copy brings)
        mbar_arrive_expect_tx(bar, bytes + (u == a.stall_unit ? 16u : 0u));
      }
      __syncwarp();
      const uint32_t off = static_cast<uint32_t>(lane) * kFastCopyChunk;
      if (off < bytes)
        bulk_copy_g2s(smem_u32(s_sc) + off, reinterpret_cast<const char*>(sc) + off,
                      min(kFastCopyChunk, bytes - off), bar);
    }
#pragma unroll
    for (int q = 0; q < kFastSlabs; ++q) {
      const int i = q * kThreads + tid;
      f[q] = (fl != nullptr && i < n) ? __ldg(fl + i) : 0;
    }
    __syncthreads();                              // the barrier is initialised
    const bool landed = mbar_wait(bar, 0, &s_abort);
    if (__syncthreads_or(!landed)) {
      // the copy did not land within the wait bound: wait for it (bounded)
      // before the block leaves, and report the unit
      if (tid == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
        a.unit_status[u] = KVC_UNIT_TIMEOUT;
        if (a.floor_excess) a.floor_excess[u] = 0;
      }
      if (tid < KVC_N_POOLS) cnt[tid * a.U + u] = 0;
      return;
    }
  } else {
#pragma unroll
    for (int q = 0; q < kFastSlabs; ++q) {
      const int i = q * kThreads + tid;
      v[q] = i < n ? __ldg(sc + i) : 0.f;
      f[q] = (fl != nullptr && i < n) ? __ldg(fl + i) : 0;
    }
  }
  // item i < n of slab q (read from shared memory as it is classified)
  auto score = [&](int q, int i) -> float {
    if constexpr (kBulk) return s_sc[i];
    else return v[q];
  };
  uint32_t key[kFastSlabs];
  uint32_t forced_bits = 0;
  uint32_t n_forced = 0, n_cand = 0, kmin = 0xffffffffu, kmax = 0u;
  int err = 0;
  // a slab with no sink or recent item, and no flags, holds only candidates
  const int plain_lo = fl == nullptr ? (a.sink_items + kThreads - 1) / kThreads : kFastSlabs;
  const int plain_hi = fl == nullptr ? (n - a.recent_items) / kThreads : 0;   // slabs [plain_lo, plain_hi)
#pragma unroll
  for (int q = 0; q < kFastSlabs; ++q) {
    const int i = q * kThreads + tid;
    key[q] = 0;
    if (q >= plain_lo && q < plain_hi) {
      key[q] = order_key(score(q, i));
      ++n_cand;
      kmin = min(kmin, key[q]);
      kmax = max(kmax, key[q]);
    } else if (i < n) {
      const bool window = i < a.sink_items || i >= n - a.recent_items;
      const bool protect = f[q] & KVC_FLAG_PROTECT;
      const bool exclude = f[q] & KVC_FLAG_EXCLUDE;
      if (protect && exclude) err = 1;
      const bool forced = window || protect;
      const bool excluded = exclude && !window;
      if (forced) {
        forced_bits |= 1u << q;
        ++n_forced;
      } else if (!excluded) {
        key[q] = order_key(score(q, i));
        ++n_cand;
        kmin = min(kmin, key[q]);
        kmax = max(kmax, key[q]);
      }
    }
  }
  if (tid == 0) {
    s_red[0] = s_red[1] = s_red[2] = 0;
    s_kmin = 0xffffffffu;
    s_kmax = 0u;
  }
  __syncthreads();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    n_forced += __shfl_xor_sync(kFull, n_forced, o);
    n_cand += __shfl_xor_sync(kFull, n_cand, o);
    err |= __shfl_xor_sync(kFull, err, o);
    kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
  }
  if (lane == 0) {
    atomicAdd(&s_red[0], n_forced);
    atomicAdd(&s_red[1], n_cand);
    atomicOr(&s_red[2], static_cast<uint32_t>(err));
    atomicMin(&s_kmin, kmin);
    atomicMax(&s_kmax, kmax);
  }
  __syncthreads();
  n_forced = s_red[0];
  n_cand = s_red[1];
  err = static_cast<int>(s_red[2]);
  kmin = s_kmin;
  kmax = s_kmax;

  if (err || n_forced > static_cast<uint32_t>(a.budget_items)) {
    if (tid < KVC_N_POOLS) cnt[tid * a.U + u] = 0;
    if (tid == 0) {
      a.unit_status[u] = err ? KVC_UNIT_BAD_FLAGS : KVC_UNIT_OVER_BUDGET;
      if (a.floor_excess) a.floor_excess[u] = 0;
    }
    return;
  }
  const uint32_t k = min(static_cast<uint32_t>(a.budget_items) - n_forced, n_cand);

  // ---------------- radix select of the k-th largest candidate key
  // (8-bit digits over the bits where candidate keys differ; t counts the
  // candidates still to place below the prefix)
  uint32_t tau = 0xffffffffu, take_ties = 0;
  uint32_t n_tau = n_cand;                          // candidates at the threshold (key tau, or
                                                    // in tau's bin after an early exit)
  if (k > 0) {
    uint32_t t = k - 1;
    uint32_t* whist = hist_w + warp * 256;
    const int top = (kmin == kmax) ? -1 : 31 - __clz(kmin ^ kmax);
    uint64_t pfx = static_cast<uint64_t>(kmax) >> (top + 1);
    int low = 0;                                    // bits below the prefix still open
    for (int hi = top; hi >= 0; hi -= 8) {
      const int shift = max(0, hi - 7);
      const int width = hi - shift + 1;
      const uint32_t nb = 1u << width;
      // (every read of this warp's histogram and of the level's results by
      // the level before came ahead of that level's second barrier)
      for (int i = lane; i < 256; i += 32) whist[i] = 0;
      __syncwarp();
      // the bits above hi must equal the prefix: one masked 32-bit compare
      const uint32_t hmask = hi >= 31 ? 0u : ~((2u << hi) - 1u);
      const uint32_t pmask = hi >= 31 ? 0u : static_cast<uint32_t>(pfx << (hi + 1));
#pragma unroll
      for (int q = 0; q < kFastSlabs; ++q)
        if (key[q] != 0 && (key[q] & hmask) == pmask)
          atomicAdd(&whist[(key[q] >> shift) & (nb - 1)], 1u);
      __syncthreads();
      // the scan over the (at most 256) bins, highest first: warps 0-7 only
      if (tid < 256) {
        uint32_t local = 0;
        if (tid < static_cast<int>(nb)) {
          const int bn = static_cast<int>(nb) - 1 - tid;
#pragma unroll
          for (int w = 0; w < 32; ++w) local += hist_w[w * 256 + bn];
        }
        const uint32_t incl = warp_incl_scan(local, lane);
        if (lane == 31) s_w8[warp] = incl;
        named_bar_sync(1, 256);
        // candidates in the bins of the warps before this one (lanes 0-7 add
        // up the totals of warps below this one)
        uint32_t wl = lane < warp ? s_w8[lane & 7] : 0u;
        wl += __shfl_xor_sync(kFull, wl, 1);
        wl += __shfl_xor_sync(kFull, wl, 2);
        wl += __shfl_xor_sync(kFull, wl, 4);
        const uint32_t run = incl - local + __shfl_sync(kFull, wl, 0);
        if (tid < static_cast<int>(nb) && run <= t && t < run + local) {
          s_bin = static_cast<int>(nb) - 1 - tid;
          s_above = run;
          s_bincnt = local;
        }
      }
      __syncthreads();
      const int bn = s_bin;                      // always found: t < candidates under pfx
      t -= s_above;
      n_tau = s_bincnt;
      pfx = (pfx << width) | static_cast<uint32_t>(bn);
      low = shift;
      // every candidate of this bin is taken: the bin's lower edge serves as
      // the threshold (uniform: t and n_tau come from shared memory)
      if (t + 1 == n_tau) break;
    }
    tau = static_cast<uint32_t>(pfx << low);
    take_ties = t + 1;
  }

  uint32_t keep_bits = forced_bits;
  if (k > 0 && n_tau == take_ties) {
    // every candidate equal to tau is taken: no ranks needed (the common case)
#pragma unroll
    for (int q = 0; q < kFastSlabs; ++q)
      if (key[q] != 0 && key[q] >= tau) keep_bits |= 1u << q;
  } else if (k > 0) {
    // ---------------- ranks of the ties (key == tau) in index order
    uint32_t tie_bits = 0;
#pragma unroll
    for (int q = 0; q < kFastSlabs; ++q) {
      const bool tie = key[q] != 0 && key[q] == tau;
      const unsigned m = __ballot_sync(kFull, tie);
      if (tie) tie_bits |= 1u << q;
      if (lane == 0) s_cnt[q * 32 + warp] = __popc(m);
    }
    __syncthreads();
    uint32_t tot;
    const uint32_t tie_off = block_excl_scan<uint32_t>(s_cnt[tid], scan_w, tot);
    __syncthreads();
    s_cnt[tid] = tie_off;                         // exclusive offset of (slab, warp) = tid
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kFastSlabs; ++q) {
      const unsigned m = __ballot_sync(kFull, (tie_bits >> q) & 1u);
      const uint32_t rank = s_cnt[q * 32 + warp] + __popc(m & lt_mask);
      const bool keep = (key[q] != 0 && key[q] > tau) || (((tie_bits >> q) & 1u) && rank < take_ties);
      if (keep) keep_bits |= 1u << q;
    }
  }
  __syncthreads();
  // ---------------- output positions in index order, then the write
#pragma unroll
  for (int q = 0; q < kFastSlabs; ++q) {
    const unsigned m = __ballot_sync(kFull, (keep_bits >> q) & 1u);
    if (lane == 0) s_cnt[q * 32 + warp] = __popc(m);
  }
  __syncthreads();
  uint32_t kept_total;
  const uint32_t pos_off = block_excl_scan<uint32_t>(s_cnt[tid], scan_w, kept_total);
  __syncthreads();
  s_cnt[tid] = pos_off;
  __syncthreads();
  const int P = a.page_size;
  int32_t* dst = a.kept_idx + (static_cast<int64_t>(KVC_POOL_BF16) * a.U + u) * a.capacity;
#pragma unroll
  for (int q = 0; q < kFastSlabs; ++q) {
    const bool keep = (keep_bits >> q) & 1u;
    const unsigned m = __ballot_sync(kFull, keep);
    if (keep) {
      const uint32_t pos = s_cnt[q * 32 + warp] + __popc(m & lt_mask);
      const int i = q * kThreads + tid;
      if (P == 1) {
        dst[pos] = i;
      } else {
        for (int j = 0; j < P; ++j) dst[static_cast<int64_t>(pos) * P + j] = i * P + j;
      }
    }
  }
  if (tid < KVC_N_POOLS) cnt[tid * a.U + u] = tid == KVC_POOL_BF16 ? static_cast<int32_t>(kept_total) * P : 0;
  if (tid == 0) {
    a.unit_status[u] = KVC_UNIT_OK;
    if (a.floor_excess) a.floor_excess[u] = 0;
  }
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream, size_t smem_bytes) {
  if (!a.byte_mode && a.n_items <= kFastMaxItems) {
    // bulk copies need 16-byte aligned rows of whole 16-byte pieces
    const bool bulk = a.n_items > 0 && a.n_items % 4 == 0 && reinterpret_cast<uintptr_t>(a.scores) % 16 == 0;
    if (bulk) {
      const int smem = static_cast<int>(a.n_items * sizeof(float));
      cudaError_t err = cudaFuncSetAttribute(select_fast_kernel<true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
      select_fast_kernel<true><<<a.U, kThreads, smem, stream>>>(a);
    } else {
      select_fast_kernel<false><<<a.U, kThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
  }
  const bool small = a.n_items <= 16384;
  void (*kern)(const SelectArgs) = small ? select_kernel<8> : select_kernel<32>;
  if (smem_bytes > 0) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem_bytes));
    if (err != cudaSuccess) return err;
  }
  kern<<<a.U, small ? 256 : kThreads, smem_bytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc

// ----------------------------------------------------------------------------
// Token / page mode for units of more than 32,768 items: the same selection
// (forced items, then the top k candidates by (score descending, index
// ascending)) spread over many CTAs per unit.  Three histogram levels find
// the k-th largest candidate key tau digit by digit (11, 11 and 10 bits,
// most significant first): each level is one pass of all CTAs over the
// unit's items (per-CTA shared-memory histograms added into the unit's
// global one) followed by one CTA per unit that picks the digit.  Then a
// counting pass, one CTA per unit for the per-chunk output offsets, and a
// writing pass that emits the kept items of each chunk in index order.
namespace kvc {
namespace {

constexpr int kLongThreads = 256;
constexpr int kLongChunk = 8192;          // items per CTA (32 per thread)
constexpr int kLongBins = 2048;

// Per-unit state of the multi-CTA selection.
struct LongState {
  uint32_t n_forced, n_cand, err;
  uint32_t phase;          // 0 searching, 1 no candidate taken, 2 all taken, 3 nothing kept (status set)
  uint32_t prefix;         // key digits fixed so far
  uint32_t rank;           // 0-based rank of the k-th candidate inside the prefix
  uint32_t take_ties;      // candidates equal to tau taken, in index order
  uint32_t pad;
};

struct LongWs {
  LongState* st;           // [U]
  uint32_t* hist;          // [U][kLongBins]
  uint32_t* fixed;         // [U][chunks] forced + candidates above tau per chunk
  uint32_t* ties;          // [U][chunks] candidates equal to tau per chunk
  int64_t chunks;
};

__host__ __device__ inline LongWs long_ws(void* base, int64_t U, int64_t n_items) {
  LongWs w;
  uint8_t* p = static_cast<uint8_t*>(base);
  w.chunks = (n_items + kLongChunk - 1) / kLongChunk;
  w.st = reinterpret_cast<LongState*>(p);
  p += (U * sizeof(LongState) + 255) / 256 * 256;
  w.hist = reinterpret_cast<uint32_t*>(p);
  p += (U * kLongBins * 4 + 255) / 256 * 256;
  w.fixed = reinterpret_cast<uint32_t*>(p);
  p += (U * w.chunks * 4 + 255) / 256 * 256;
  w.ties = reinterpret_cast<uint32_t*>(p);
  return w;
}

// Class of item i: 0 = neither kept nor a candidate, 1 = forced, 2 = candidate
// (with its order key), from its already loaded score and flags.
__device__ __forceinline__ int long_class(const SelectArgs& a, int64_t i, float s, uint8_t f, uint32_t& key,
                                          int& err) {
  const bool window = i < a.sink_items || i >= a.n_items - a.recent_items;
  const bool protect = f & KVC_FLAG_PROTECT;
  const bool exclude = f & KVC_FLAG_EXCLUDE;
  if (protect && exclude) err = 1;
  if (window || protect) return 1;
  if (exclude) return 0;
  key = order_key(s);
  return 2;
}

// The scores (and flags) of kLongIlp items per thread, all loads issued
// before any is used: items i0 + q * kLongThreads + threadIdx.x.
constexpr int kLongIlp = 8;
__device__ __forceinline__ void long_load(const float* sc, const uint8_t* fl, int64_t i0, int64_t i1,
                                          float (&s)[kLongIlp], uint8_t (&f)[kLongIlp]) {
#pragma unroll
  for (int q = 0; q < kLongIlp; ++q) {
    const int64_t i = i0 + q * kLongThreads + threadIdx.x;
    s[q] = i < i1 ? __ldg(sc + i) : 0.f;
    f[q] = (fl && i < i1) ? __ldg(fl + i) : 0;
  }
}

// Digit `level` of a key and whether the key matches the digits fixed so far.
__device__ __forceinline__ bool long_digit(uint32_t key, int level, uint32_t prefix, uint32_t& digit) {
  if (level == 0) {
    digit = key >> 21;
    return true;
  }
  if (level == 1) {
    digit = (key >> 10) & 2047u;
    return (key >> 21) == prefix;
  }
  digit = key & 1023u;
  return (key >> 10) == prefix;
}

// One histogram level over chunk blockIdx.x of unit blockIdx.y (level 0 also
// counts forced items and candidates and checks the flags).
__global__ void __launch_bounds__(kLongThreads) select_long_hist(const __grid_constant__ SelectArgs a, int level) {
  __shared__ uint32_t h[kLongBins];
  __shared__ uint32_t s_forced, s_cand, s_err;
  const int u = blockIdx.y;
  const LongWs w = long_ws(a.long_ws, a.U, a.n_items);
  LongState* st = w.st + u;
  if (level > 0 && st->phase != 0) return;                    // block-uniform
  const uint32_t prefix = level > 0 ? st->prefix : 0u;
  for (int i = threadIdx.x; i < kLongBins; i += kLongThreads) h[i] = 0;
  if (threadIdx.x == 0) s_forced = s_cand = s_err = 0;
  __syncthreads();
  const int b = u / (a.L * a.Hkv);
  const float* sc = a.scores + static_cast<int64_t>(u) * a.n_items;
  const uint8_t* fl = a.flags ? a.flags + static_cast<int64_t>(b) * a.n_items : nullptr;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kLongChunk;
  const int64_t i1 = min(a.n_items, i0 + kLongChunk);
  uint32_t n_forced = 0, n_cand = 0;
  int err = 0;
  for (int64_t ib = i0; ib < i1; ib += kLongIlp * kLongThreads) {
    float sv[kLongIlp];
    uint8_t fv[kLongIlp];
    long_load(sc, fl, ib, i1, sv, fv);
#pragma unroll
    for (int q = 0; q < kLongIlp; ++q) {
      const int64_t i = ib + q * kLongThreads + threadIdx.x;
      uint32_t key = 0, dg = 0;
      const int cls = i < i1 ? long_class(a, i, sv[q], fv[q], key, err) : 0;
      n_forced += cls == 1;
      n_cand += cls == 2;
      if (cls == 2 && long_digit(key, level, prefix, dg)) atomicAdd(&h[dg], 1u);
    }
  }
  if (level == 0) {
    for (int o = 16; o > 0; o >>= 1) {
      n_forced += __shfl_xor_sync(kFull, n_forced, o);
      n_cand += __shfl_xor_sync(kFull, n_cand, o);
      err |= __shfl_xor_sync(kFull, err, o);
    }
    if ((threadIdx.x & 31) == 0) {
      atomicAdd(&s_forced, n_forced);
      atomicAdd(&s_cand, n_cand);
      atomicOr(&s_err, static_cast<uint32_t>(err));
    }
  }
  __syncthreads();
  uint32_t* gh = w.hist + static_cast<int64_t>(u) * kLongBins;
  for (int i = threadIdx.x; i < kLongBins; i += kLongThreads)
    if (h[i]) atomicAdd(gh + i, h[i]);
  if (level == 0 && threadIdx.x == 0) {
    if (s_forced) atomicAdd(&st->n_forced, s_forced);
    if (s_cand) atomicAdd(&st->n_cand, s_cand);
    if (s_err) atomicOr(&st->err, s_err);
  }
}

// Pick the digit of `level` for every unit (one CTA per unit): the bin where
// the descending running count of candidates passes the target rank; the
// histogram is cleared for the next level.
__global__ void __launch_bounds__(kLongThreads) select_long_pick(const __grid_constant__ SelectArgs a, int level) {
  __shared__ unsigned long long wtot[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_above;
  const int u = blockIdx.x;
  const LongWs w = long_ws(a.long_ws, a.U, a.n_items);
  LongState* st = w.st + u;
  uint32_t* gh = w.hist + static_cast<int64_t>(u) * kLongBins;
  if (level == 0 && threadIdx.x == 0) {
    // the unit's totals decide whether a search is needed at all
    const uint32_t n_forced = st->n_forced, n_cand = st->n_cand;
    uint32_t phase = 0;
    if (st->err) {
      phase = 3;
      a.unit_status[u] = KVC_UNIT_BAD_FLAGS;
    } else if (n_forced > static_cast<uint32_t>(a.budget_items)) {
      phase = 3;
      a.unit_status[u] = KVC_UNIT_OVER_BUDGET;
    } else {
      const uint32_t k = min(static_cast<uint32_t>(a.budget_items) - n_forced, n_cand);
      if (k == 0) phase = 1;
      else if (k == n_cand) phase = 2;
      else st->rank = k - 1;
    }
    st->phase = phase;
    st->prefix = 0;
  }
  __syncthreads();
  if (st->phase != 0) {
    for (int i = threadIdx.x; i < kLongBins; i += kLongThreads) gh[i] = 0;
    return;
  }
  const int nb = level == 2 ? 1024 : kLongBins;
  const uint32_t t = st->rank;
  if (threadIdx.x == 0) s_bin = -1;
  // each thread owns nb / 256 consecutive bins in descending order
  const int per = nb / kLongThreads;
  unsigned long long local = 0;
  uint32_t c[8];
  for (int k = 0; k < per; ++k) {
    c[k] = gh[nb - 1 - (threadIdx.x * per + k)];
    local += c[k];
  }
  // block exclusive scan of `local`
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = local;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  unsigned long long base = 0;
  for (int i = 0; i < warp; ++i) base += wtot[i];
  unsigned long long run = base + incl - local;
  for (int k = 0; k < per; ++k) {
    if (run <= t && t < run + c[k]) {
      s_bin = nb - 1 - (threadIdx.x * per + k);
      s_above = static_cast<uint32_t>(run);
    }
    run += c[k];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kLongBins; i += kLongThreads) gh[i] = 0;
  if (threadIdx.x == 0) {
    const int bn = s_bin;                          // always found: t < candidates in the prefix
    st->prefix = (st->prefix << (level == 2 ? 10 : 11)) | static_cast<uint32_t>(bn < 0 ? 0 : bn);
    st->rank = t - s_above;
    if (level == 2) st->take_ties = st->rank + 1;
  }
}

// Whether item (class cls, key) is kept given the unit's state; ties (key ==
// tau) are reported separately.
__device__ __forceinline__ void long_decide(const LongState& s, int cls, uint32_t key, bool& fixed, bool& tie) {
  fixed = cls == 1 || (cls == 2 && (s.phase == 2 || (s.phase == 0 && key > s.prefix)));
  tie = cls == 2 && s.phase == 0 && key == s.prefix;
}

__global__ void __launch_bounds__(kLongThreads) select_long_count(const __grid_constant__ SelectArgs a) {
  __shared__ uint32_t s_f, s_t;
  const int u = blockIdx.y;
  const LongWs w = long_ws(a.long_ws, a.U, a.n_items);
  const LongState st = w.st[u];
  if (st.phase == 3) return;
  if (threadIdx.x == 0) s_f = s_t = 0;
  __syncthreads();
  const int b = u / (a.L * a.Hkv);
  const float* sc = a.scores + static_cast<int64_t>(u) * a.n_items;
  const uint8_t* fl = a.flags ? a.flags + static_cast<int64_t>(b) * a.n_items : nullptr;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kLongChunk;
  const int64_t i1 = min(a.n_items, i0 + kLongChunk);
  uint32_t nf = 0, nt = 0;
  int err = 0;
  for (int64_t ib = i0; ib < i1; ib += kLongIlp * kLongThreads) {
    float sv[kLongIlp];
    uint8_t fv[kLongIlp];
    long_load(sc, fl, ib, i1, sv, fv);
#pragma unroll
    for (int q = 0; q < kLongIlp; ++q) {
      const int64_t i = ib + q * kLongThreads + threadIdx.x;
      if (i >= i1) continue;
      uint32_t key = 0;
      const int cls = long_class(a, i, sv[q], fv[q], key, err);
      bool fixed, tie;
      long_decide(st, cls, key, fixed, tie);
      nf += fixed;
      nt += tie;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    nf += __shfl_xor_sync(kFull, nf, o);
    nt += __shfl_xor_sync(kFull, nt, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&s_f, nf);
    atomicAdd(&s_t, nt);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    w.fixed[static_cast<int64_t>(u) * w.chunks + blockIdx.x] = s_f;
    w.ties[static_cast<int64_t>(u) * w.chunks + blockIdx.x] = s_t;
  }
}

// Per unit: output offset of every chunk (kept items in index order), the
// number of ties each chunk keeps, the kept count and the unit status.
__global__ void __launch_bounds__(32) select_long_offsets(const __grid_constant__ SelectArgs a) {
  const int u = blockIdx.x, lane = threadIdx.x;
  const LongWs w = long_ws(a.long_ws, a.U, a.n_items);
  const LongState st = w.st[u];
  int32_t* cnt = a.kept_count;
  if (st.phase == 3) {
    if (lane < KVC_N_POOLS) cnt[lane * a.U + u] = 0;
    if (lane == 0 && a.floor_excess) a.floor_excess[u] = 0;
    return;
  }
  uint32_t* fx = w.fixed + static_cast<int64_t>(u) * w.chunks;
  uint32_t* ti = w.ties + static_cast<int64_t>(u) * w.chunks;
  uint32_t out_run = 0, tie_run = 0;
  for (int64_t c0 = 0; c0 < w.chunks; c0 += 32) {
    const int64_t c = c0 + lane;
    const uint32_t f = c < w.chunks ? fx[c] : 0u, t = c < w.chunks ? ti[c] : 0u;
    // ties kept by this chunk: the part of [tie_off, tie_off + t) below take_ties
    uint32_t ti_incl = t;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, ti_incl, o);
      if (lane >= o) ti_incl += y;
    }
    const uint32_t tie_off = tie_run + ti_incl - t;
    const uint32_t take = st.phase == 0 ? st.take_ties : 0u;
    const uint32_t kt = tie_off >= take ? 0u : min(t, take - tie_off);
    const uint32_t kept = f + kt;
    uint32_t k_incl = kept;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, k_incl, o);
      if (lane >= o) k_incl += y;
    }
    if (c < w.chunks) {
      fx[c] = out_run + k_incl - kept;     // output offset of the chunk
      ti[c] = kt;                          // ties the chunk keeps
    }
    out_run += __shfl_sync(kFull, k_incl, 31);
    tie_run += __shfl_sync(kFull, ti_incl, 31);
  }
  if (lane < KVC_N_POOLS) cnt[lane * a.U + u] = lane == KVC_POOL_BF16 ? static_cast<int32_t>(out_run) * a.page_size : 0;
  if (lane == 0) {
    a.unit_status[u] = KVC_UNIT_OK;
    if (a.floor_excess) a.floor_excess[u] = 0;
  }
}

// Write the kept items of chunk blockIdx.x of unit blockIdx.y in index order
// (256 items per round: a block scan of the keep flags gives each its slot).
__global__ void __launch_bounds__(kLongThreads) select_long_write(const __grid_constant__ SelectArgs a) {
  __shared__ uint32_t wsum[kLongThreads / 32];
  const int u = blockIdx.y;
  const LongWs w = long_ws(a.long_ws, a.U, a.n_items);
  const LongState st = w.st[u];
  if (st.phase == 3) return;
  const int b = u / (a.L * a.Hkv);
  const float* sc = a.scores + static_cast<int64_t>(u) * a.n_items;
  const uint8_t* fl = a.flags ? a.flags + static_cast<int64_t>(b) * a.n_items : nullptr;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kLongChunk;
  const int64_t i1 = min(a.n_items, i0 + kLongChunk);
  uint32_t out = w.fixed[static_cast<int64_t>(u) * w.chunks + blockIdx.x];
  const uint32_t ties_kept = w.ties[static_cast<int64_t>(u) * w.chunks + blockIdx.x];
  uint32_t tie_run = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int P = a.page_size;
  int32_t* dst = a.kept_idx + (static_cast<int64_t>(KVC_POOL_BF16) * a.U + u) * a.capacity;
  int err = 0;
  float sv[kLongIlp];
  uint8_t fv[kLongIlp];
  for (int64_t base = i0, r = 0; base < i1; base += kLongThreads, ++r) {
    const int q = static_cast<int>(r % kLongIlp);
    if (q == 0) long_load(sc, fl, base, i1, sv, fv);    // the next kLongIlp rounds' items
    const int64_t i = base + threadIdx.x;
    bool fixed = false, tie = false;
    if (i < i1) {
      uint32_t key = 0;
      float s_q = sv[0];
      uint8_t f_q = fv[0];
#pragma unroll
      for (int k = 1; k < kLongIlp; ++k)
        if (q == k) {
          s_q = sv[k];
          f_q = fv[k];
        }
      const int cls = long_class(a, i, s_q, f_q, key, err);
      long_decide(st, cls, key, fixed, tie);
    }
    // a round with nothing to keep and no tie needs no ranks (the common case:
    // a chunk keeps a few of its items)
    if (!__syncthreads_or(fixed || tie)) continue;
    // rank of this tie among the chunk's ties (index order)
    const unsigned tm = __ballot_sync(kFull, tie);
    if (lane == 0) wsum[warp] = __popc(tm);
    __syncthreads();
    uint32_t tie_before = tie_run + __popc(tm & ((1u << lane) - 1u)), tie_total = 0;
    for (int k = 0; k < kLongThreads / 32; ++k) {
      if (k < warp) tie_before += wsum[k];
      tie_total += wsum[k];
    }
    __syncthreads();
    const bool keep = fixed || (tie && tie_before < ties_kept);
    const unsigned km = __ballot_sync(kFull, keep);
    if (lane == 0) wsum[warp] = __popc(km);
    __syncthreads();
    uint32_t pos = out + __popc(km & ((1u << lane) - 1u)), total = 0;
    for (int k = 0; k < kLongThreads / 32; ++k) {
      if (k < warp) pos += wsum[k];
      total += wsum[k];
    }
    __syncthreads();
    if (keep) {
      if (P == 1) {
        dst[pos] = static_cast<int32_t>(i);
      } else {
        for (int j = 0; j < P; ++j) dst[static_cast<int64_t>(pos) * P + j] = static_cast<int32_t>(i * P + j);
      }
    }
    out += total;
    tie_run += tie_total;
  }
}

// ---- Four items per load.  The same passes for units whose item count is a
// multiple of 4, with 16-byte aligned scores and 4-byte aligned flags: thread
// t takes items i0 + 4 (q kLongThreads + t) + e (q < kLongIlp, e < 4), so in
// index order a chunk is kLongIlp slabs of 1,024 items, thread by thread,
// four items each.  A chunk that holds no sink or recent item, with no
// flags, classifies every item as a candidate without the per-item tests.
__device__ __forceinline__ void long_load4(const float* sc, const uint8_t* fl, int64_t i0, int64_t i1,
                                           float4 (&s)[kLongIlp], uint32_t (&f)[kLongIlp]) {
#pragma unroll
  for (int q = 0; q < kLongIlp; ++q) {
    const int64_t i = i0 + 4 * (q * kLongThreads + threadIdx.x);
    s[q] = i < i1 ? __ldg(reinterpret_cast<const float4*>(sc + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    f[q] = (fl && i < i1) ? __ldg(reinterpret_cast<const uint32_t*>(fl + i)) : 0u;
  }
}

__device__ __forceinline__ float quad_at(const float4& v, int e) {
  return e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
}

__device__ __forceinline__ int long_class4(const SelectArgs& a, bool plain, int64_t i, float s, uint32_t f4, int e,
                                           uint32_t& key, int& err) {
  if (plain) {
    key = order_key(s);
    return 2;
  }
  return long_class(a, i, s, static_cast<uint8_t>(f4 >> (8 * e)), key, err);
}

__device__ __forceinline__ bool long_plain(const SelectArgs& a, const uint8_t* fl, int64_t i0, int64_t i1) {
  return fl == nullptr && i0 >= a.sink_items && i1 <= a.n_items - a.recent_items;
}

__global__ void __launch_bounds__(kLongThreads) select_long_hist4(const __grid_constant__ SelectArgs a, int level) {
  __shared__ uint32_t h[kLongBins];
  __shared__ uint32_t s_forced, s_cand, s_err;
  const int u = blockIdx.y;
  const LongWs w = long_ws(a.long_ws, a.U, a.n_items);
  LongState* st = w.st + u;
  if (level > 0 && st->phase != 0) return;                    // block-uniform
  const uint32_t prefix = level > 0 ? st->prefix : 0u;
  for (int i = threadIdx.x; i < kLongBins; i += kLongThreads) h[i] = 0;
  if (threadIdx.x == 0) s_forced = s_cand = s_err = 0;
  __syncthreads();
  const int b = u / (a.L * a.Hkv);
  const float* sc = a.scores + static_cast<int64_t>(u) * a.n_items;
  const uint8_t* fl = a.flags ? a.flags + static_cast<int64_t>(b) * a.n_items : nullptr;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kLongChunk;
  const int64_t i1 = min(a.n_items, i0 + kLongChunk);
  const bool plain = long_plain(a, fl, i0, i1);
  uint32_t n_forced = 0, n_cand = 0;
  int err = 0;
  float4 sv[kLongIlp];
  uint32_t fv[kLongIlp];
  long_load4(sc, fl, i0, i1, sv, fv);
#pragma unroll
  for (int q = 0; q < kLongIlp; ++q) {
    const int64_t ib = i0 + 4 * (q * kLongThreads + threadIdx.x);
    if (ib >= i1) continue;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t key = 0, dg = 0;
      const int cls = long_class4(a, plain, ib + e, quad_at(sv[q], e), fv[q], e, key, err);
      n_forced += cls == 1;
      n_cand += cls == 2;
      if (cls == 2 && long_digit(key, level, prefix, dg)) atomicAdd(&h[dg], 1u);
    }
  }
  if (level == 0) {
    for (int o = 16; o > 0; o >>= 1) {
      n_forced += __shfl_xor_sync(kFull, n_forced, o);
      n_cand += __shfl_xor_sync(kFull, n_cand, o);
      err |= __shfl_xor_sync(kFull, err, o);
    }
    if ((threadIdx.x & 31) == 0) {
      atomicAdd(&s_forced, n_forced);
      atomicAdd(&s_cand, n_cand);
      atomicOr(&s_err, static_cast<uint32_t>(err));
    }
  }
  __syncthreads();
  uint32_t* gh = w.hist + static_cast<int64_t>(u) * kLongBins;
  for (int i = threadIdx.x; i < kLongBins; i += kLongThreads)
    if (h[i]) atomicAdd(gh + i, h[i]);
  if (level == 0 && threadIdx.x == 0) {
    if (s_forced) atomicAdd(&st->n_forced, s_forced);
    if (s_cand) atomicAdd(&st->n_cand, s_cand);
    if (s_err) atomicOr(&st->err, s_err);
  }
}

__global__ void __launch_bounds__(kLongThreads) select_long_count4(const __grid_constant__ SelectArgs a) {
  __shared__ uint32_t s_f, s_t;
  const int u = blockIdx.y;
  const LongWs w = long_ws(a.long_ws, a.U, a.n_items);
  const LongState st = w.st[u];
  if (st.phase == 3) return;
  if (threadIdx.x == 0) s_f = s_t = 0;
  __syncthreads();
  const int b = u / (a.L * a.Hkv);
  const float* sc = a.scores + static_cast<int64_t>(u) * a.n_items;
  const uint8_t* fl = a.flags ? a.flags + static_cast<int64_t>(b) * a.n_items : nullptr;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kLongChunk;
  const int64_t i1 = min(a.n_items, i0 + kLongChunk);
  const bool plain = long_plain(a, fl, i0, i1);
  uint32_t nf = 0, nt = 0;
  int err = 0;
  float4 sv[kLongIlp];
  uint32_t fv[kLongIlp];
  long_load4(sc, fl, i0, i1, sv, fv);
#pragma unroll
  for (int q = 0; q < kLongIlp; ++q) {
    const int64_t ib = i0 + 4 * (q * kLongThreads + threadIdx.x);
    if (ib >= i1) continue;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t key = 0;
      const int cls = long_class4(a, plain, ib + e, quad_at(sv[q], e), fv[q], e, key, err);
      bool fixed, tie;
      long_decide(st, cls, key, fixed, tie);
      nf += fixed;
      nt += tie;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    nf += __shfl_xor_sync(kFull, nf, o);
    nt += __shfl_xor_sync(kFull, nt, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&s_f, nf);
    atomicAdd(&s_t, nt);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    w.fixed[static_cast<int64_t>(u) * w.chunks + blockIdx.x] = s_f;
    w.ties[static_cast<int64_t>(u) * w.chunks + blockIdx.x] = s_t;
  }
}

// Exclusive scan over the kLongThreads threads of the block; `total` gets the sum.
__device__ __forceinline__ uint32_t long_block_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = warp_incl_scan(v, lane);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t base = 0;
  total = 0;
#pragma unroll
  for (int k = 0; k < kLongThreads / 32; ++k) {
    if (k < warp) base += wsum[k];
    total += wsum[k];
  }
  __syncthreads();
  return base + incl - v;
}

// Write the kept items of chunk blockIdx.x of unit blockIdx.y in index order,
// one 1,024-item slab at a time (a slab with nothing to keep and no tie is
// skipped after one block-wide vote).
__global__ void __launch_bounds__(kLongThreads) select_long_write4(const __grid_constant__ SelectArgs a) {
  __shared__ uint32_t wsum[kLongThreads / 32];
  const int u = blockIdx.y;
  const LongWs w = long_ws(a.long_ws, a.U, a.n_items);
  const LongState st = w.st[u];
  if (st.phase == 3) return;
  const int b = u / (a.L * a.Hkv);
  const float* sc = a.scores + static_cast<int64_t>(u) * a.n_items;
  const uint8_t* fl = a.flags ? a.flags + static_cast<int64_t>(b) * a.n_items : nullptr;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kLongChunk;
  const int64_t i1 = min(a.n_items, i0 + kLongChunk);
  const bool plain = long_plain(a, fl, i0, i1);
  uint32_t out = w.fixed[static_cast<int64_t>(u) * w.chunks + blockIdx.x];
  const uint32_t ties_kept = w.ties[static_cast<int64_t>(u) * w.chunks + blockIdx.x];
  uint32_t tie_run = 0;
  const int P = a.page_size;
  int32_t* dst = a.kept_idx + (static_cast<int64_t>(KVC_POOL_BF16) * a.U + u) * a.capacity;
  int err = 0;
  float4 sv[kLongIlp];
  uint32_t fv[kLongIlp];
  long_load4(sc, fl, i0, i1, sv, fv);
#pragma unroll 1
  for (int q = 0; q < kLongIlp; ++q) {
    const int64_t ib = i0 + 4 * (q * kLongThreads + threadIdx.x);
    uint32_t fixed_bits = 0, tie_bits = 0;
    if (ib < i1) {
      float4 v = sv[0];
      uint32_t f4 = fv[0];
#pragma unroll
      for (int k = 1; k < kLongIlp; ++k)
        if (q == k) {
          v = sv[k];
          f4 = fv[k];
        }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t key = 0;
        const int cls = long_class4(a, plain, ib + e, quad_at(v, e), f4, e, key, err);
        bool fixed, tie;
        long_decide(st, cls, key, fixed, tie);
        fixed_bits |= static_cast<uint32_t>(fixed) << e;
        tie_bits |= static_cast<uint32_t>(tie) << e;
      }
    }
    if (!__syncthreads_or(fixed_bits | tie_bits)) continue;
    // ranks of the ties in index order, then which of them the chunk keeps
    uint32_t tie_total;
    const uint32_t tie_before = tie_run + long_block_scan(__popc(tie_bits), wsum, tie_total);
    uint32_t keep_bits = fixed_bits;
    uint32_t tr = tie_before;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if ((tie_bits >> e) & 1u) {
        if (tr < ties_kept) keep_bits |= 1u << e;
        ++tr;
      }
    uint32_t keep_total;
    uint32_t pos = out + long_block_scan(__popc(keep_bits), wsum, keep_total);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if ((keep_bits >> e) & 1u) {
        const int64_t i = ib + e;
        if (P == 1) {
          dst[pos] = static_cast<int32_t>(i);
        } else {
          for (int j = 0; j < P; ++j) dst[static_cast<int64_t>(pos) * P + j] = static_cast<int32_t>(i * P + j);
        }
        ++pos;
      }
    out += keep_total;
    tie_run += tie_total;
  }
}

}  // namespace

size_t select_long_ws_bytes(int64_t U, int64_t n_items) {
  const int64_t chunks = (n_items + kLongChunk - 1) / kLongChunk;
  return static_cast<size_t>((U * sizeof(LongState) + 255) / 256 * 256 + (U * kLongBins * 4 + 255) / 256 * 256 +
                             2 * ((U * chunks * 4 + 255) / 256 * 256));
}

cudaError_t launch_select_long(const SelectArgs& a, cudaStream_t stream) {
  const LongWs w = long_ws(a.long_ws, a.U, a.n_items);
  // state and level-0 histogram start at zero; every later level's
  // histogram is cleared by the pick of the level before
  cudaError_t err = cudaMemsetAsync(a.long_ws, 0,
                                    (a.U * sizeof(LongState) + 255) / 256 * 256 + (a.U * kLongBins * 4 + 255) / 256 * 256,
                                    stream);
  if (err != cudaSuccess) return err;
  const dim3 grid(static_cast<unsigned>(w.chunks), static_cast<unsigned>(a.U));
  // four items per load where every unit's scores (and flags) stay aligned
  const bool vec4 = a.n_items % 4 == 0 && reinterpret_cast<uintptr_t>(a.scores) % 16 == 0 &&
                    (a.flags == nullptr || reinterpret_cast<uintptr_t>(a.flags) % 4 == 0);
  for (int level = 0; level < 3; ++level) {
    if (vec4) select_long_hist4<<<grid, kLongThreads, 0, stream>>>(a, level);
    else select_long_hist<<<grid, kLongThreads, 0, stream>>>(a, level);
    select_long_pick<<<a.U, kLongThreads, 0, stream>>>(a, level);
  }
  if (vec4) select_long_count4<<<grid, kLongThreads, 0, stream>>>(a);
  else select_long_count<<<grid, kLongThreads, 0, stream>>>(a);
  select_long_offsets<<<a.U, 32, 0, stream>>>(a);
  if (vec4) select_long_write4<<<grid, kLongThreads, 0, stream>>>(a);
  else select_long_write<<<grid, kLongThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc
