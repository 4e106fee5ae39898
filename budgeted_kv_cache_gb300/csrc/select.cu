// Deterministic budgeted selection, one CTA of 1024 threads per unit.
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
// token mode, the upgrade cost in byte mode): three digit passes (11, 11,
// 10 bits) each build a warp-aggregated shared-memory histogram of the
// items still matching the key prefix and locate, with a block scan, the
// bin where the running weight crosses the target.  Items above the final
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

// Exclusive scan over the 1024 threads of the block; `total` gets the sum.
template <typename V>
__device__ __forceinline__ V block_excl_scan(V v, V* wtot, V& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const V incl = warp_incl_scan(v, lane);
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const V w = warp_incl_scan(wtot[lane], lane);
    wtot[lane] = w;
  }
  __syncthreads();
  const V base = warp ? wtot[warp - 1] : V(0);
  total = wtot[31];
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

__global__ void __launch_bounds__(kThreads, 1) select_kernel(const __grid_constant__ SelectArgs a) {
  __shared__ uint32_t hist[2048];
  __shared__ unsigned long long wtot[32];
  __shared__ unsigned long long red[4];
  __shared__ int s_bin;
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
  const int64_t n_pad = (c.n + kThreads - 1) / kThreads * kThreads;

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
  if (tid < 4) red[tid] = 0;
  __syncthreads();
  unsigned long long n_forced = 0, n_cand = 0, floor_bytes = 0;
  int err = 0;
  for (int64_t i = tid; i < c.n; i += kThreads) {
    const Item it = eval_item(c, i, err);
    if (a.cache_items) {
      ckey[i] = it.key;
      cbase[i] = it.base;
    }
    n_forced += (!a.byte_mode && it.base == KVC_ACT_BF16);
    n_cand += (it.key != 0);
    floor_bytes += c.cost[it.base];
  }
  for (int o = 16; o > 0; o >>= 1) {
    n_forced += __shfl_xor_sync(kFull, n_forced, o);
    n_cand += __shfl_xor_sync(kFull, n_cand, o);
    floor_bytes += __shfl_xor_sync(kFull, floor_bytes, o);
    err |= __shfl_xor_sync(kFull, err, o);
  }
  if (lane == 0) {
    atomicAdd(&red[0], n_forced);
    atomicAdd(&red[1], n_cand);
    atomicAdd(&red[2], floor_bytes);
    atomicOr(reinterpret_cast<unsigned int*>(&red[3]), static_cast<unsigned int>(err));
  }
  __syncthreads();
  n_forced = red[0];
  n_cand = red[1];
  floor_bytes = red[2];
  err = static_cast<int>(red[3]);

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
  uint32_t tau = 0;
  if (!sel_none) {
    uint32_t prefix = 0;
    for (int p = 0; p < 3; ++p) {
      const int shift = p == 0 ? 21 : (p == 1 ? 10 : 0);
      const int bits = p == 2 ? 10 : 11;
      const int nb = 1 << bits;
      for (int i = tid; i < nb; i += kThreads) hist[i] = 0;
      __syncthreads();
      for (int64_t i = tid; i < n_pad; i += kThreads) {
        bool active = false;
        uint32_t bin = 0, w = 0;
        if (i < c.n) {
          const Item it = get(i, err);
          active = it.key != 0 && (p == 0 || (it.key >> (shift + bits)) == prefix);
          bin = (it.key >> shift) & (nb - 1);
          w = item_weight(c, it);
        }
        const unsigned act_mask = __ballot_sync(kFull, active);
        if (active) {
          const unsigned peers = __match_any_sync(act_mask, bin);
          const uint32_t sum = a.byte_mode ? __reduce_add_sync(peers, w) : __popc(peers);
          if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], sum);
        }
      }
      if (tid == 0) s_bin = -1;
      __syncthreads();
      // bins in descending order: thread tid owns bins nb-1-(tid*per+k)
      const int per = nb / kThreads;
      unsigned long long local = 0;
      for (int k = 0; k < per; ++k) local += hist[nb - 1 - (tid * per + k)];
      unsigned long long total;
      unsigned long long run = block_excl_scan<unsigned long long>(local, wtot, total);
      for (int k = 0; k < per; ++k) {
        const int bn = nb - 1 - (tid * per + k);
        const unsigned long long h = hist[bn];
        if (run <= t && t < run + h) {
          s_bin = bn;
          s_above = run;
        }
        run += h;
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
      prefix = (prefix << bits) | static_cast<uint32_t>(bn);
    }
    tau = prefix;
  }

  // ---------------- phase C: write the kept lists in index order
  // Warp w owns the contiguous item range [w_lo, w_hi) and walks it 32 items
  // at a time: (1) total tie weight per warp, scanned across warps; (2) the
  // promotion decisions and per-pool counts, scanned across warps; (3) the
  // same decisions again, writing each kept item at its final position.
  __shared__ unsigned long long s_tie[32];
  __shared__ uint32_t s_pool[KVC_N_POOLS][32];
  const int warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int64_t per_w = (c.n + 32 * 32 - 1) / (32 * 32) * 32;
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

  // (1) tie weight per warp
  unsigned long long tie_tot = 0;
  for (int64_t i0 = w_lo; i0 < w_hi; i0 += 32) {
    unsigned long long tw = tie_weight(load(i0 + lane));
    for (int o = 16; o > 0; o >>= 1) tw += __shfl_xor_sync(kFull, tw, o);
    tie_tot += tw;
  }
  if (lane == 0) s_tie[warp] = tie_tot;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long v = s_tie[lane];
    s_tie[lane] = warp_incl_scan(v, lane) - v;
  }
  __syncthreads();
  // (2) decisions and pool counts per warp
  uint32_t pc[KVC_N_POOLS] = {0, 0, 0};
  unsigned long long tie_run = s_tie[warp];
  for (int64_t i0 = w_lo; i0 < w_hi; i0 += 32) {
    const int64_t i = i0 + lane;
    const Item it = load(i);
    const unsigned long long tw = tie_weight(it);
    const unsigned long long incl = warp_incl_scan(tw, lane);
    const uint32_t act = (i < w_hi) ? decide(it, tie_run + incl - tw, tw) : KVC_ACT_RELEASE;
    tie_run += __shfl_sync(kFull, incl, 31);
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) pc[q] += __popc(__ballot_sync(kFull, act == q + 1u));
  }
  if (lane == 0) {
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) s_pool[q][warp] = pc[q];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < KVC_N_POOLS; ++q) {
      const uint32_t v = s_pool[q][lane];
      s_pool[q][lane] = warp_incl_scan(v, lane);        // inclusive: entry 31 is the total
    }
  }
  __syncthreads();
  // (3) write
  uint32_t pos_run[KVC_N_POOLS];
#pragma unroll
  for (int q = 0; q < KVC_N_POOLS; ++q) pos_run[q] = warp ? s_pool[q][warp - 1] : 0u;
  tie_run = s_tie[warp];
  for (int64_t i0 = w_lo; i0 < w_hi; i0 += 32) {
    const int64_t i = i0 + lane;
    const Item it = load(i);
    const unsigned long long tw = tie_weight(it);
    const unsigned long long incl = warp_incl_scan(tw, lane);
    const uint32_t act = (i < w_hi) ? decide(it, tie_run + incl - tw, tw) : KVC_ACT_RELEASE;
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

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream, size_t smem_bytes) {
  if (smem_bytes > 0) {
    cudaError_t err = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem_bytes));
    if (err != cudaSuccess) return err;
  }
  select_kernel<<<a.U, kThreads, smem_bytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc
