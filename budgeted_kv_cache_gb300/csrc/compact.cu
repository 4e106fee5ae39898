// Fused gather + renumber + exact re-rotation + quantisation + store.
//
// CommitKV Eq. 4 applies the kept index set to K, V and positions; PACE
// Sec. 3.2 renumbers the kept rows to 0..n-1 in logical order and re-rotates
// each kept key by R_{p'-p} (Prop. 1), with cos/sin of (p'-p) theta_i formed
// from the engine's tables through the angle-difference identities and
// normalised to unit length; PASK App. B.5 quantises retained rows with a
// symmetric per-group scale (here bf16 scale per 32 elements, or the page's
// fp16 scale per row).
//
// One row per d/8 lanes: each lane moves 16 bytes (8 bf16) of one row with
// one 128-bit load, so a warp reads and writes two whole 256-byte rows at
// d = 128 (four at d = 64).  Key rows and value rows are handled by separate
// warps, so the rotation work of a key warp is spread over all its lanes.
// The split-half partner element (i <-> i + d/2) sits in lane ^ (d/16) and
// comes over one shuffle; the two partners split the cos/sin work.  All float operations use explicit round-to-
// nearest intrinsics (no contraction into FMA), so the stored bits are a
// fixed function of the inputs.
#include <algorithm>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ int lower_bound_i32(const int32_t* v, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
  const uint32_t r[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(r[k] << 16);
    x[2 * k + 1] = __uint_as_float(r[k] & 0xffff0000u);
  }
}

// Where this lane's 8 elements sit in the rotary pairs.  Split halves of
// the first rd elements (i with i + rd/2): lanes hl < rd/16 hold x, lanes
// rd/16 <= hl < rd/8 hold the partner y, and the two lanes of a pair
// compute four of their eight (C, S) each (table columns j0 .. j0 + 3).
// Interleaved pairs (2i, 2i + 1) lie inside one lane, which forms its own
// four (C, S).  Lanes at or past rd copy their elements.
struct LaneRot {
  bool active;
  bool inter;
  bool first_half;
  int src;         // warp lane holding the partner elements (split layout)
  int j0;          // first table column of this lane's four (C, S)
  int half;        // table width: rd / 2
};

__device__ __forceinline__ LaneRot lane_rot(int layout, int rd, int lane, int hl, int lpr) {
  LaneRot r;
  r.half = rd / 2;
  r.inter = layout == KVC_ROPE_INTERLEAVED;
  r.active = 8 * hl < rd;
  if (r.inter) {
    r.first_half = true;
    r.src = lane;
    r.j0 = 4 * hl;
  } else {
    const int q = rd / 16;                        // lanes per half
    r.first_half = hl < q;
    const int phl = !r.active ? hl : (r.first_half ? hl + q : hl - q);
    r.src = lane - hl + phl;
    r.j0 = (r.first_half ? hl : hl - q) * 8 + (r.first_half ? 0 : 4);
  }
  (void)lpr;
  return r;
}

// Normalised (C, S) of the angle difference for four pairs (see the file
// comment), from the cos / sin of the old (tab[0], tab[1]) and new
// (tab[2], tab[3]) position.
__device__ __forceinline__ void rot_cs4(const float4 (&tab)[4], float (&C4)[4], float (&S4)[4]) {
  const float cc0[4] = {tab[0].x, tab[0].y, tab[0].z, tab[0].w};
  const float ss0[4] = {tab[1].x, tab[1].y, tab[1].z, tab[1].w};
  const float cc1[4] = {tab[2].x, tab[2].y, tab[2].z, tab[2].w};
  const float ss1[4] = {tab[3].x, tab[3].y, tab[3].z, tab[3].w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float C = __fadd_rn(__fmul_rn(cc1[k], cc0[k]), __fmul_rn(ss1[k], ss0[k]));
    float S = __fsub_rn(__fmul_rn(ss1[k], cc0[k]), __fmul_rn(cc1[k], ss0[k]));
    const float nrm = __fsqrt_rn(__fadd_rn(__fmul_rn(C, C), __fmul_rn(S, S)));
    C4[k] = __fdiv_rn(C, nrm);
    S4[k] = __fdiv_rn(S, nrm);
  }
}

// General rotary layouts (interleaved pairs, or only the first rd elements
// rotated); same arithmetic and rounding as rerotate_lane.  Whole warps.
__device__ __forceinline__ void rerotate_lane_general(const LaneRot& lr, bool rotate,
                                                      const float4 (&tab)[4], float (&x)[8],
                                                      uint4& w) {
  const bool rot = rotate && lr.active;
  uint32_t rb[8];
  if (lr.inter) {
    if (!rot) return;
    float C4[4], S4[4];
    rot_cs4(tab, C4, S4);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float xr = __fsub_rn(__fmul_rn(x[2 * k], C4[k]), __fmul_rn(x[2 * k + 1], S4[k]));
      const float yr = __fadd_rn(__fmul_rn(x[2 * k + 1], C4[k]), __fmul_rn(x[2 * k], S4[k]));
      rb[2 * k] = float_to_bf16_bits(xr);
      rb[2 * k + 1] = float_to_bf16_bits(yr);
    }
  } else {
    uint4 ow;
    ow.x = __shfl_sync(kFull, w.x, lr.src);
    ow.y = __shfl_sync(kFull, w.y, lr.src);
    ow.z = __shfl_sync(kFull, w.z, lr.src);
    ow.w = __shfl_sync(kFull, w.w, lr.src);
    float y[8];
    unpack8(ow, y);
    float C4[4] = {1.f, 1.f, 1.f, 1.f}, S4[4] = {0.f, 0.f, 0.f, 0.f};
    if (rot) rot_cs4(tab, C4, S4);
    float Cx[4], Sx[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      Cx[k] = __shfl_sync(kFull, C4[k], lr.src);
      Sx[k] = __shfl_sync(kFull, S4[k], lr.src);
    }
    if (!rot) return;
    const bool fh = lr.first_half;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float Ck = k < 4 ? (fh ? C4[k] : Cx[k]) : (fh ? Cx[k - 4] : C4[k - 4]);
      const float Sk = k < 4 ? (fh ? S4[k] : Sx[k]) : (fh ? Sx[k - 4] : S4[k - 4]);
      const float r = fh ? __fsub_rn(__fmul_rn(x[k], Ck), __fmul_rn(y[k], Sk))
                         : __fadd_rn(__fmul_rn(x[k], Ck), __fmul_rn(y[k], Sk));
      rb[k] = float_to_bf16_bits(r);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = bf16_bits_to_float(static_cast<uint16_t>(rb[k]));
  w = make_uint4(rb[0] | (rb[1] << 16), rb[2] | (rb[3] << 16), rb[4] | (rb[5] << 16),
                 rb[6] | (rb[7] << 16));
}

// Re-rotation of one key row's 8 elements held by this lane (see the file
// comment): x holds them, w their packed bf16 bits; on return both hold the
// rotated row.  Called by whole warps (the shuffles need every lane).
__device__ __forceinline__ void rerotate_lane(int lpr, int hl, bool rotate, const float4 (&tab)[4],
                                              float (&x)[8], uint4& w) {
  const int px = lpr / 2;
  uint4 ow;
  ow.x = __shfl_xor_sync(kFull, w.x, px);
  ow.y = __shfl_xor_sync(kFull, w.y, px);
  ow.z = __shfl_xor_sync(kFull, w.z, px);
  ow.w = __shfl_xor_sync(kFull, w.w, px);
  float y[8];
  unpack8(ow, y);
  const bool first_half = hl < px;
  float C4[4] = {1.f, 1.f, 1.f, 1.f}, S4[4] = {0.f, 0.f, 0.f, 0.f};
  if (rotate) {
    const float cc0[4] = {tab[0].x, tab[0].y, tab[0].z, tab[0].w};
    const float ss0[4] = {tab[1].x, tab[1].y, tab[1].z, tab[1].w};
    const float cc1[4] = {tab[2].x, tab[2].y, tab[2].z, tab[2].w};
    const float ss1[4] = {tab[3].x, tab[3].y, tab[3].z, tab[3].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float C = __fadd_rn(__fmul_rn(cc1[k], cc0[k]), __fmul_rn(ss1[k], ss0[k]));
      float S = __fsub_rn(__fmul_rn(ss1[k], cc0[k]), __fmul_rn(cc1[k], ss0[k]));
      const float nrm = __fsqrt_rn(__fadd_rn(__fmul_rn(C, C), __fmul_rn(S, S)));
      C4[k] = __fdiv_rn(C, nrm);
      S4[k] = __fdiv_rn(S, nrm);
    }
  }
  float Cx[4], Sx[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    Cx[k] = __shfl_xor_sync(kFull, C4[k], px);
    Sx[k] = __shfl_xor_sync(kFull, S4[k], px);
  }
  if (rotate) {
    uint32_t rb[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float Ck = k < 4 ? (first_half ? C4[k] : Cx[k]) : (first_half ? Cx[k - 4] : C4[k - 4]);
      const float Sk = k < 4 ? (first_half ? S4[k] : Sx[k]) : (first_half ? Sx[k - 4] : S4[k - 4]);
      // first half holds x (partner y); second half holds y (partner x)
      const float r = first_half ? __fsub_rn(__fmul_rn(x[k], Ck), __fmul_rn(y[k], Sk))
                                 : __fadd_rn(__fmul_rn(x[k], Ck), __fmul_rn(y[k], Sk));
      rb[k] = float_to_bf16_bits(r);              // stored bf16 value
      x[k] = bf16_bits_to_float(static_cast<uint16_t>(rb[k]));
    }
    w = make_uint4(rb[0] | (rb[1] << 16), rb[2] | (rb[3] << 16), rb[4] | (rb[5] << 16),
                   rb[6] | (rb[7] << 16));
  }
}

// Re-rotation of this lane's part of one key row from position `from` to
// `to` (rows whose `rot` is false are left as they are); whole warps call it.
template <bool kGeneral>
__device__ __forceinline__ void rotate_row(const CompactArgs& a, const LaneRot& lr, int lpr, int hl,
                                           bool rot, int32_t from, int32_t to, uint4& w,
                                           float (&x)[8]) {
  if (!__any_sync(kFull, rot)) return;
  const int j0 = lr.j0;
  const int half = lr.half;
  float4 tab[4];
  if (rot && lr.active) {
    tab[0] = __ldg(reinterpret_cast<const float4*>(a.cos + static_cast<int64_t>(from) * half + j0));
    tab[1] = __ldg(reinterpret_cast<const float4*>(a.sin + static_cast<int64_t>(from) * half + j0));
    tab[2] = __ldg(reinterpret_cast<const float4*>(a.cos + static_cast<int64_t>(to) * half + j0));
    tab[3] = __ldg(reinterpret_cast<const float4*>(a.sin + static_cast<int64_t>(to) * half + j0));
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) tab[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (kGeneral) rerotate_lane_general(lr, rot, tab, x, w);
  else rerotate_lane(lpr, hl, rot, tab, x, w);
}

// Quantise this lane's 8 elements of one row and store codes and scales.
__device__ __forceinline__ void store_quantised(const CompactArgs& a, int pool, int is_v, int lpr,
                                                int hl, bool valid, int64_t row,
                                                const float (&x)[8]) {
  const int d = a.d;
  const bool row_mode = a.quant_mode == KVC_QUANT_ROW_FP16;
  const float qmax = pool == KVC_POOL_INT4 ? 7.f : 127.f;
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(x[k]));
  const int gl = row_mode ? lpr : 4;             // lanes per scale group
  for (int o2 = 1; o2 < gl; o2 <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o2));
  float sc = 1.f;
  uint16_t s_bits;
  if (!row_mode) {
    if (amax > 0.f) {
      sc = bf16_bits_to_float(float_to_bf16_bits(__fdiv_rn(amax, qmax)));
      sc = fmaxf(sc, __uint_as_float(0x00010000u));          // 2^-133
    }
    s_bits = float_to_bf16_bits(sc);
  } else {
    if (amax > 0.f) {
      sc = __half2float(__float2half_rn(__fdiv_rn(amax, qmax)));
      sc = fminf(sc, 65504.f);
      sc = fmaxf(sc, 5.9604644775390625e-08f);               // 2^-24
    }
    s_bits = __half_as_ushort(__float2half_rn(sc));
  }
  // one reciprocal per group, then a correctly rounded quotient per element
  // (the same bits as x / sc with IEEE division)
  const bool fast = recip_div_ok(sc);
  const float y = __fdiv_rn(1.f, sc);
  int qv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float qf = fast ? div_by_recip(x[k], sc, y) : __fdiv_rn(x[k], sc);
    int q = amax > 0.f ? __float2int_rn(qf) : 0;
    q = q > static_cast<int>(qmax) ? static_cast<int>(qmax) : q;
    q = q < -static_cast<int>(qmax) ? -static_cast<int>(qmax) : q;
    qv[k] = q;
  }
  if (!valid) return;
  if (pool == KVC_POOL_INT8) {
    uint8_t* dst = static_cast<uint8_t*>(is_v ? a.pools.v_i8 : a.pools.k_i8);
    uint2 pk;
    pk.x = (qv[0] & 0xff) | ((qv[1] & 0xff) << 8) | ((qv[2] & 0xff) << 16) | ((qv[3] & 0xff) << 24);
    pk.y = (qv[4] & 0xff) | ((qv[5] & 0xff) << 8) | ((qv[6] & 0xff) << 16) | ((qv[7] & 0xff) << 24);
    *reinterpret_cast<uint2*>(dst + row * d + hl * 8) = pk;
  } else {
    uint8_t* dst = static_cast<uint8_t*>(is_v ? a.pools.v_i4 : a.pools.k_i4);
    uint32_t pk = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      pk |= static_cast<uint32_t>((qv[2 * k] & 0xf) | ((qv[2 * k + 1] & 0xf) << 4)) << (8 * k);
    *reinterpret_cast<uint32_t*>(dst + row * (d / 2) + hl * 4) = pk;
  }
  void* sp = pool == KVC_POOL_INT8 ? (is_v ? a.pools.v_i8_scale : a.pools.k_i8_scale)
                                   : (is_v ? a.pools.v_i4_scale : a.pools.k_i4_scale);
  uint16_t* sdst = static_cast<uint16_t*>(sp);
  if (!row_mode) {
    if ((hl & 3) == 0) sdst[row * (d / 32) + hl / 4] = s_bits;
  } else {
    if (hl == 0) sdst[row] = s_bits;
  }
}

constexpr int kBatch = 512;
constexpr uint8_t kValid = 1, kRotate = 2, kChange = 4;

// Stages the kept index, old and new position and flags of rows b0 .. b0 +
// nb - 1 of one (unit, pool) stream in shared memory, one thread per row
// (all the loads of the batch in flight together).  Value streams (is_v)
// need no positions.  Returns whether this thread met a bad row.
template <bool kStore>
__device__ __forceinline__ bool stage_batch(const CompactArgs& a, int pool, int is_v, int u, int64_t slot0,
                                            int64_t b0, int nb, bool use_store, int32_t* s_t, int32_t* s_p,
                                            int32_t* s_p2, int32_t* s_pr, uint8_t* s_f) {
  const int U = a.U;
  const int cap = a.capacity;
  bool bad = false;
  for (int q = threadIdx.x; q < nb; q += kThreads) {
    const int64_t i = b0 + q;
    const int32_t t = __ldg(a.kept_idx + slot0 + i);
    uint8_t f = 0;
    int32_t p = 0, p2 = 0, pr = -1;
    if (t < 0 || t >= a.T) {
      bad = true;
    } else {
      f = kValid;
      if (!is_v) {
        p = __ldg(a.pos_in + static_cast<int64_t>(u) * a.T + t);
        p2 = p;
        if (a.renumber) {
          // rank among the kept rows of every pool (pools are disjoint, ascending)
          int rank = static_cast<int>(i);
          for (int qq = 0; qq < KVC_N_POOLS; ++qq) {
            if (qq == pool) continue;
            const int cq = clamp_count(__ldg(a.kept_count + qq * U + u), cap);
            if (cq > 0)
              rank += lower_bound_i32(a.kept_idx + (static_cast<int64_t>(qq) * U + u) * cap, cq, t);
          }
          p2 = rank;
        }
        if (p2 != p) {
          if (p < 0 || p >= a.rope_max_pos || p2 < 0 || p2 >= a.rope_max_pos) {
            f = 0;
            bad = true;
          } else {
            f |= kRotate;
          }
        }
        if (use_store && (f & kValid)) {
          pr = __ldg(a.ref.ref_pos + static_cast<int64_t>(u) * a.T + t);
          if (pr >= a.rope_max_pos) {
            f = 0;
            bad = true;
          }
        }
      }
    }
    s_t[q] = t;
    s_p[q] = p;
    s_p2[q] = p2;
    if (kStore) s_pr[q] = pr;
    s_f[q] = f;
  }
  return bad;
}

// A block works on one (unit, pool, K-or-V) stream, in batches of up to
// kBatch kept rows.  For a batch it first stages every row's kept index, old
// position, new position and status in shared memory (one thread per row,
// all loads of the batch in flight together), so the dependent chain kept
// index -> position -> rotary rows is walked once per batch instead of once
// per row.  Then each lane group moves kRows rows at a time: the row loads
// and the rotary-table loads of all of them are issued before any is used.
// The grid has up to kBatch-row batches of every stream side by side; the
// block of batch lane x takes the batches x, x + lanes, ... that lie below
// the stream's kept count.
constexpr int kRows = 2;

template <bool kStore, bool kGeneral>
__global__ void __launch_bounds__(kThreads, 4) compact_kernel(const CompactArgs a) {
  __shared__ int32_t s_t[kBatch], s_p[kBatch], s_p2[kBatch], s_pr[kStore ? kBatch : 1];
  __shared__ uint8_t s_f[kBatch];
  __shared__ int s_bad;
  const int d = a.d;
  const int lpr = d / 8;                        // lanes per row (16 B = 8 bf16 per lane)
  const int rows_per_warp = 32 / lpr;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / lpr;
  const int hl = lane % lpr;
  // blockIdx.x = (batch lane, pool, K or V) with K / V fastest, so key blocks
  // (re-rotation arithmetic) and value blocks (plain copies) run side by side
  const int n_pools = a.pool_hi - a.pool_lo;
  const int is_v = blockIdx.x & 1;              // K rows and V rows go to separate blocks
  const int pool = a.pool_lo + static_cast<int>((blockIdx.x >> 1) % n_pools);
  const int bxi = static_cast<int>((blockIdx.x >> 1) / n_pools);   // batch lane of the stream
  const int bxn = static_cast<int>(gridDim.x / (2 * n_pools));     // batch lanes per stream
  const int u = blockIdx.y;
  const int U = a.U;
  const int cap = a.capacity;
  // a count outside [0, capacity] is clamped (rows past the capacity would
  // belong to the next unit) and reported as a bad index
  const int cnt_raw = __ldg(a.kept_count + pool * U + u);
  const int cnt = clamp_count(cnt_raw, cap);
  if (cnt != cnt_raw && bxi == 0 && threadIdx.x == 0 && a.unit_status)
    a.unit_status[u] = KVC_UNIT_BAD_INDEX;
  if (static_cast<int64_t>(bxi) * kBatch >= cnt) return;    // block-uniform
  if (threadIdx.x == 0) s_bad = 0;

  const int64_t slot0 = (static_cast<int64_t>(pool) * U + u) * cap;
  const bool use_store = kStore && !is_v;                       // block-uniform
  const __nv_bfloat16* src = is_v ? a.v : a.k;
  const LaneRot lr = kGeneral ? lane_rot(a.rope_layout, a.rotary_dim, lane, hl, lpr)
                              : lane_rot(KVC_ROPE_SPLIT_HALF, d, lane, hl, lpr);
  const int j0 = lr.j0;
  const int half = lr.half;

  for (int64_t b0 = static_cast<int64_t>(bxi) * kBatch; b0 < cnt; b0 += static_cast<int64_t>(bxn) * kBatch) {
    const int nb = static_cast<int>(min(static_cast<int64_t>(kBatch), cnt - b0));
    // ---------------- stage the batch's rows (one thread per row)
    __syncthreads();                            // the previous batch is done with the arrays
    const bool bad = stage_batch<kStore>(a, pool, is_v, u, slot0, b0, nb, use_store, s_t, s_p, s_p2, s_pr, s_f);
    if (bad) s_bad = 1;
    __syncthreads();

    // ---------------- move the rows: lane group `sub` of each warp takes rows
    // q = q0 + n * rows_per_warp + sub, n < kRows
    const int step = (kThreads / 32) * rows_per_warp * kRows;
    for (int q0 = warp * rows_per_warp * kRows; q0 < nb; q0 += step) {
      bool valid[kRows], rotate[kRows], chg[kRows];
      int32_t t[kRows], p[kRows], p2[kRows], pr[kRows];
      uint4 w[kRows], wr[kRows];
#pragma unroll
      for (int n = 0; n < kRows; ++n) {
        const int q = q0 + n * rows_per_warp + sub;
        const uint8_t f = q < nb ? s_f[q] : 0;
        valid[n] = f & kValid;
        t[n] = valid[n] ? s_t[q] : 0;
        p[n] = valid[n] ? s_p[q] : 0;
        p2[n] = valid[n] ? s_p2[q] : 0;
        pr[n] = (kStore && valid[n]) ? s_pr[q] : -1;
        rotate[n] = (f & kRotate) != 0;
        w[n] = valid[n] ? __ldg(reinterpret_cast<const uint4*>(src + (static_cast<int64_t>(u) * a.T + t[n]) * d) + hl)
                        : make_uint4(0, 0, 0, 0);
        wr[n] = make_uint4(0, 0, 0, 0);
        if (use_store && valid[n] && pr[n] >= 0)
          wr[n] = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.ref.ref_k) +
                                                       (static_cast<int64_t>(u) * a.T + t[n]) * d) + hl);
      }
      // with the store, rows rotate in their own branch below (no hoisted tables)
#pragma unroll
      for (int n = 0; n < kRows; ++n) {
        chg[n] = use_store && rotate[n];
        if (use_store) rotate[n] = false;
      }
      // rotation tables: cos / sin of the old and new position for the four
      // (C, S) pairs this lane forms
      float4 tab[kRows][4];
#pragma unroll
      for (int n = 0; n < kRows; ++n) {
        if (rotate[n] && lr.active) {
          tab[n][0] = __ldg(reinterpret_cast<const float4*>(a.cos + static_cast<int64_t>(p[n]) * half + j0));
          tab[n][1] = __ldg(reinterpret_cast<const float4*>(a.sin + static_cast<int64_t>(p[n]) * half + j0));
          tab[n][2] = __ldg(reinterpret_cast<const float4*>(a.cos + static_cast<int64_t>(p2[n]) * half + j0));
          tab[n][3] = __ldg(reinterpret_cast<const float4*>(a.sin + static_cast<int64_t>(p2[n]) * half + j0));
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) tab[n][k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int n = 0; n < kRows; ++n) {
        float x[8];
        unpack8(w[n], x);
        // the branch is warp-uniform: key rows only, and only if a row rotates
        if (!is_v && __any_sync(kFull, rotate[n])) {
          if (kGeneral) rerotate_lane_general(lr, rotate[n], tab[n], x, w[n]);
          else rerotate_lane(lpr, hl, rotate[n], tab[n], x, w[n]);
        }
        const int64_t i = b0 + q0 + n * rows_per_warp + sub;
        const int64_t row = static_cast<int64_t>(u) * cap + i;
        if (use_store) {
          // PACE reference store: check the copy (re-rotated p_ref -> p, it must
          // reproduce the stored key in every lane of the row), then derive the
          // new key from it, or from the stored key if there is no valid copy
          const bool has_ref = valid[n] && pr[n] >= 0;
          uint4 chk = wr[n];
          float xc[8];
          unpack8(chk, xc);
          rotate_row<kGeneral>(a, lr, lpr, hl, chg[n] && has_ref && pr[n] != p[n], pr[n], p[n], chk, xc);
          const bool lane_ok = chk.x == w[n].x && chk.y == w[n].y && chk.z == w[n].z && chk.w == w[n].w;
          const unsigned gmask = (lpr == 32 ? kFull : ((1u << lpr) - 1u)) << (sub * lpr);
          const bool ok = (__ballot_sync(kFull, lane_ok) & gmask) == gmask;
          const bool use_ref = chg[n] && has_ref && ok;
          const bool failed = chg[n] && has_ref && !ok;
          uint4 nw = use_ref ? wr[n] : w[n];
          const int32_t from = use_ref ? pr[n] : p[n];
          float xs[8];
          unpack8(nw, xs);
          rotate_row<kGeneral>(a, lr, lpr, hl, chg[n] && from != p2[n], from, p2[n], nw, xs);
          uint4 rw = has_ref ? wr[n] : make_uint4(0, 0, 0, 0);
          int32_t rp = has_ref ? pr[n] : -1;
          if (chg[n] && !use_ref) {            // first renumber, or a failed copy: the stored key
            rw = w[n];
            rp = p[n];
          }
          if (chg[n]) {
            w[n] = nw;
#pragma unroll
            for (int k = 0; k < 8; ++k) x[k] = xs[k];
          }
          if (valid[n]) {
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.ref.ref_k_out) + (slot0 + i) * d + hl * 8) = rw;
            if (hl == 0) a.ref.ref_pos_out[slot0 + i] = rp;
          }
          if (failed && hl == 0 && a.ref.failures) atomicAdd(a.ref.failures + u, 1);
        }
        if (pool == KVC_POOL_BF16) {
          if (valid[n]) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(is_v ? a.pools.v_bf16 : a.pools.k_bf16);
            *reinterpret_cast<uint4*>(dst + row * d + hl * 8) = w[n];
          }
        } else {
          store_quantised(a, pool, is_v, lpr, hl, valid[n], row, x);
        }
        if (valid[n] && hl == 0 && !is_v) {
          a.pools.pos_out[slot0 + i] = p2[n];
          if (a.pools.orig_pos_out) a.pools.orig_pos_out[slot0 + i] = p[n];
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_bad && a.unit_status) a.unit_status[u] = KVC_UNIT_BAD_INDEX;
}

// ----------------------------------------------------------------------------
// Split-half rotation over every element and no reference store (the common
// case; any pool, blockIdx.z): keys and values of the same rows move together.
// A block takes batches of one unit's kept rows (kCopyBatch at a time, staged
// as above).  Each lane copies its 16-byte pieces of a row -- key, value and,
// for a key that changes position, the four rotary-table pieces it needs --
// into shared memory with asynchronous copies, kCopyStages - 1 steps ahead
// of the step it is working on; no registers are held by the copies in flight.
// A lane reads back only the pieces it copied itself, so no block-wide barrier
// separates the copy and the use.  Two stages and three blocks per SM: the
// 48 KB of stages per block leave most of the SM's on-chip memory to L1,
// where table rows are shared between rows and blocks, and 24 warps per SM
// hide the re-rotation arithmetic (four stages with two blocks, or two stages
// with two or four blocks, are 6-19% slower).
constexpr int kCopyStages = 2;
constexpr int kCopyRows = 1;          // rows per lane group and step
constexpr int kCopyBatch = 256;       // rows staged per block and batch
constexpr int kPieces = 6;            // key, value, cos(p), sin(p), cos(p'), sin(p')

// The same through L1 (rotary-table pieces: many rows of a block and of the
// blocks beside it on the SM share table rows).
__device__ __forceinline__ void cp_async16_l1(uint32_t saddr, const void* src, uint64_t policy) {
  asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(saddr), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(saddr), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void st_global_hint(void* dst, const uint4& w, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "r"(w.x), "r"(w.y),
               "r"(w.z), "r"(w.w), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

size_t compact_copy_smem_bytes() {
  return static_cast<size_t>(kCopyStages) * kCopyRows * kPieces * kThreads * 16;
}

__global__ void __launch_bounds__(kThreads, 3) compact_copy_kernel(const CompactArgs a) {
  extern __shared__ uint4 s_pieces[];   // [stage][row n][piece][thread]
  __shared__ int32_t s_t[kCopyBatch], s_p[kCopyBatch], s_p2[kCopyBatch];
  __shared__ uint8_t s_f[kCopyBatch];
  __shared__ int s_bad;
  const int d = a.d;
  const int lpr = d / 8;                        // lanes per row (16 B = 8 bf16 per lane)
  const int rows_per_warp = 32 / lpr;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / lpr;
  const int hl = lane % lpr;
  const int groups = (kThreads / 32) * rows_per_warp;   // lane groups of the block
  const int grp = warp * rows_per_warp + sub;
  const int per_step = groups * kCopyRows;
  const int pool = a.pool_lo + static_cast<int>(blockIdx.z);
  const int u = blockIdx.y;
  const int U = a.U;
  const int cap = a.capacity;
  const int cnt_raw = __ldg(a.kept_count + pool * U + u);
  const int cnt = clamp_count(cnt_raw, cap);
  if (cnt != cnt_raw && blockIdx.x == 0 && threadIdx.x == 0 && a.unit_status)
    a.unit_status[u] = KVC_UNIT_BAD_INDEX;
  if (static_cast<int64_t>(blockIdx.x) * kCopyBatch >= cnt) return;    // block-uniform
  if (threadIdx.x == 0) s_bad = 0;
  const int64_t slot0 = (static_cast<int64_t>(pool) * U + u) * cap;
  const LaneRot lr = lane_rot(KVC_ROPE_SPLIT_HALF, d, lane, hl, lpr);
  const int j0 = lr.j0;
  const int half = lr.half;
  const uint32_t piece0 = smem_u32(s_pieces) + threadIdx.x * 16;
  auto piece = [&](int stage, int n, int c) {
    return piece0 + static_cast<uint32_t>(((stage * kCopyRows + n) * kPieces + c) * kThreads * 16);
  };
  const int64_t row0 = static_cast<int64_t>(u) * a.T;
  // the rotary tables are read by every unit: keep them in L2 while the
  // rows stream through it once
  const uint64_t keep = l2_policy_evict_last();
  const uint64_t stream = l2_policy_evict_first();

  for (int64_t b0 = static_cast<int64_t>(blockIdx.x) * kCopyBatch; b0 < cnt;
       b0 += static_cast<int64_t>(gridDim.x) * kCopyBatch) {
    const int nb = static_cast<int>(min(static_cast<int64_t>(kCopyBatch), cnt - b0));
    __syncthreads();                            // the previous batch is done with the arrays
    const bool bad = stage_batch<false>(a, pool, 0, u, slot0, b0, nb, false, s_t, s_p, s_p2, nullptr, s_f);
    if (bad) s_bad = 1;
    __syncthreads();

    // step k: lane group g takes rows q = k * per_step + n * groups + g
    const int n_steps = (nb + per_step - 1) / per_step;
    auto issue = [&](int k) {
      const int stage = k % kCopyStages;
#pragma unroll
      for (int n = 0; n < kCopyRows; ++n) {
        const int q = k * per_step + n * groups + grp;
        const uint8_t f = (k < n_steps && q < nb) ? s_f[q] : 0;
        if (f & kValid) {
          const int64_t r = row0 + s_t[q];
          cp_async16(piece(stage, n, 0), reinterpret_cast<const uint4*>(a.k + r * d) + hl, stream);
          cp_async16(piece(stage, n, 1), reinterpret_cast<const uint4*>(a.v + r * d) + hl, stream);
          if ((f & kRotate) && lr.active) {
            const int64_t p = s_p[q], p2 = s_p2[q];
            cp_async16_l1(piece(stage, n, 2), a.cos + p * half + j0, keep);
            cp_async16_l1(piece(stage, n, 3), a.sin + p * half + j0, keep);
            cp_async16_l1(piece(stage, n, 4), a.cos + p2 * half + j0, keep);
            cp_async16_l1(piece(stage, n, 5), a.sin + p2 * half + j0, keep);
          }
        }
      }
      cp_async_commit();                        // one group per step, empty or not
    };
#pragma unroll
    for (int k = 0; k < kCopyStages - 1; ++k) issue(k);
    for (int k = 0; k < n_steps; ++k) {
      issue(k + kCopyStages - 1);
      cp_async_wait<kCopyStages - 1>();         // this thread's pieces of step k have landed
      const int stage = k % kCopyStages;
#pragma unroll
      for (int n = 0; n < kCopyRows; ++n) {
        const int q = k * per_step + n * groups + grp;
        const uint8_t f = q < nb ? s_f[q] : 0;
        const bool valid = f & kValid;
        const bool rot = (f & kRotate) != 0;
        uint4 w = make_uint4(0, 0, 0, 0), wv = w;
        float4 tab[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) tab[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w) : "r"(piece(stage, n, 0)));
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(wv.x), "=r"(wv.y), "=r"(wv.z), "=r"(wv.w) : "r"(piece(stage, n, 1)));
        }
        if (rot && lr.active) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                         : "=f"(tab[c].x), "=f"(tab[c].y), "=f"(tab[c].z), "=f"(tab[c].w)
                         : "r"(piece(stage, n, 2 + c)));
        }
        // whole warps: the rotation exchanges halves between partner lanes
        float x[8];
        unpack8(w, x);
        if (__any_sync(kFull, rot)) rerotate_lane(lpr, hl, rot, tab, x, w);
        const int64_t i = b0 + q;
        const int64_t row = static_cast<int64_t>(u) * cap + i;
        if (pool == KVC_POOL_BF16) {
          if (valid) {
            st_global_hint(static_cast<__nv_bfloat16*>(a.pools.k_bf16) + row * d + hl * 8, w, stream);
            st_global_hint(static_cast<__nv_bfloat16*>(a.pools.v_bf16) + row * d + hl * 8, wv, stream);
          }
        } else {                                  // whole warps (group maxima over lanes)
          float xv[8];
          unpack8(wv, xv);
          store_quantised(a, pool, 0, lpr, hl, valid, row, x);
          store_quantised(a, pool, 1, lpr, hl, valid, row, xv);
        }
        if (valid) {
          if (hl == 0) {
            a.pools.pos_out[slot0 + i] = s_p2[q];
            if (a.pools.orig_pos_out) a.pools.orig_pos_out[slot0 + i] = s_p[q];
          }
        }
      }
    }
    cp_async_wait<0>();
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_bad && a.unit_status) a.unit_status[u] = KVC_UNIT_BAD_INDEX;
}

}  // namespace

cudaError_t launch_compact(const CompactArgs& a, cudaStream_t stream) {
  const int n_pools = a.pool_hi - a.pool_lo;
  if (a.capacity < 1 || n_pools <= 0) return cudaSuccess;
  const bool general = a.rope_layout != KVC_ROPE_SPLIT_HALF || a.rotary_dim != a.d;
  if (a.ref.ref_pos == nullptr && !general) {
    // keys and values together; batch lanes of a (unit, pool) stream side by
    // side, as many as the capacity needs but no more than keep the grid near
    // 2,048 blocks (in byte mode the capacity is T and most of it unused)
    const int64_t streams = static_cast<int64_t>(a.U) * n_pools;
    const int64_t per_cap = (a.capacity + kCopyBatch - 1) / kCopyBatch;
    const int64_t bx = std::max<int64_t>(1, std::min<int64_t>(per_cap, (2048 + streams - 1) / streams));
    const size_t smem = compact_copy_smem_bytes();
    cudaError_t err = cudaFuncSetAttribute(compact_copy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    compact_copy_kernel<<<dim3(static_cast<unsigned>(bx), a.U, n_pools), kThreads, smem, stream>>>(a);
    return cudaGetLastError();
  }
  // batches of a stream side by side: as many as the capacity needs, but
  // no more than keep about 4,096 blocks in the grid (a block whose batches
  // all lie past the stream's kept count exits at once)
  const int64_t streams = static_cast<int64_t>(a.U) * 2 * n_pools;
  const int64_t per_cap = (a.capacity + kBatch - 1) / kBatch;
  const int64_t bx = std::max<int64_t>(1, std::min<int64_t>(per_cap, (4096 + streams - 1) / streams));
  dim3 grid(static_cast<unsigned>(bx * 2 * n_pools), a.U);            // x: (batch lane, pool, K or V)
  if (a.ref.ref_pos != nullptr) {
    if (general) compact_kernel<true, true><<<grid, kThreads, 0, stream>>>(a);
    else compact_kernel<true, false><<<grid, kThreads, 0, stream>>>(a);
  } else {
    if (general) compact_kernel<false, true><<<grid, kThreads, 0, stream>>>(a);
    else compact_kernel<false, false><<<grid, kThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kvc
