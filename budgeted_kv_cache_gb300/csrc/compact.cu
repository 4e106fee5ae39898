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
// One row pair (a K row and its V row) per 2 * d/8 lanes: each lane moves 16
// bytes (8 bf16) of one row with one 128-bit load, so a warp reads and
// writes whole 256-byte rows at d = 128 (two row pairs per warp at d = 64).
// The split-half partner element (i <-> i + d/2) sits in lane ^ (d/16) and
// comes over one shuffle.  All float operations use explicit round-to-
// nearest intrinsics (no contraction into FMA), so the stored bits are a
// fixed function of the inputs.
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

__device__ __forceinline__ uint4 pack8_bf16(const float (&x)[8]) {
  uint32_t r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    r[k] = static_cast<uint32_t>(float_to_bf16_bits(x[2 * k])) |
           (static_cast<uint32_t>(float_to_bf16_bits(x[2 * k + 1])) << 16);
  return make_uint4(r[0], r[1], r[2], r[3]);
}

__global__ void __launch_bounds__(kThreads) compact_kernel(const CompactArgs a) {
  const int d = a.d;
  const int lpr = d / 8;                        // lanes per K (or V) row
  const int pairs_per_warp = 32 / (2 * lpr);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / (2 * lpr);
  const int is_v = (lane / lpr) & 1;
  const int hl = lane % lpr;
  const int pool = a.pool_lo + blockIdx.z;
  const int u = blockIdx.y;
  const int64_t i = (static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + warp) * pairs_per_warp + sub;
  const int U = a.U;
  const int cap = a.capacity;
  const int cnt = a.kept_count[pool * U + u];
  bool valid = i < cnt;
  if (__all_sync(kFull, !valid)) return;

  const int64_t slot = (static_cast<int64_t>(pool) * U + u) * cap + i;
  int32_t t = 0, p = 0, p2 = 0;
  bool rotate = false;
  if (valid) {
    t = a.kept_idx[slot];
    if (t < 0 || t >= a.T) {
      valid = false;
      if (hl == 0 && is_v == 0 && a.unit_status) a.unit_status[u] = KVC_UNIT_BAD_INDEX;
    }
  }
  if (valid) {
    p = a.pos_in[static_cast<int64_t>(u) * a.T + t];
    p2 = p;
    if (a.renumber) {
      // rank among the kept rows of every pool (pools are disjoint, ascending)
      int rank = static_cast<int>(i);
      for (int q = 0; q < KVC_N_POOLS; ++q) {
        if (q == pool) continue;
        const int cq = a.kept_count[q * U + u];
        if (cq > 0)
          rank += lower_bound_i32(a.kept_idx + (static_cast<int64_t>(q) * U + u) * cap, cq, t);
      }
      p2 = rank;
    }
    rotate = p2 != p;
    if (rotate && (p < 0 || p >= a.rope_max_pos || p2 < 0 || p2 >= a.rope_max_pos)) {
      valid = false;
      rotate = false;
      if (hl == 0 && is_v == 0 && a.unit_status) a.unit_status[u] = KVC_UNIT_BAD_INDEX;
    }
  }

  const __nv_bfloat16* src = is_v ? a.v : a.k;
  uint4 w = make_uint4(0, 0, 0, 0);
  if (valid) w = *reinterpret_cast<const uint4*>(src + (static_cast<int64_t>(u) * a.T + t) * d + hl * 8);

  // partner half of the split-half pair lives in lane ^ (lpr / 2)
  const int px = lpr / 2;
  uint4 o;
  o.x = __shfl_xor_sync(kFull, w.x, px);
  o.y = __shfl_xor_sync(kFull, w.y, px);
  o.z = __shfl_xor_sync(kFull, w.z, px);
  o.w = __shfl_xor_sync(kFull, w.w, px);

  float x[8];
  unpack8(w, x);
  if (valid && rotate && !is_v) {
    float y[8];
    unpack8(o, y);
    const int j0 = (hl % px) * 8;                 // first pair index of this lane
    const int half = d / 2;
    const float* c0p = a.cos + static_cast<int64_t>(p) * half + j0;
    const float* s0p = a.sin + static_cast<int64_t>(p) * half + j0;
    const float* c1p = a.cos + static_cast<int64_t>(p2) * half + j0;
    const float* s1p = a.sin + static_cast<int64_t>(p2) * half + j0;
    float c0[8], s0[8], c1[8], s1[8];
#pragma unroll
    for (int k = 0; k < 8; k += 4) {
      *reinterpret_cast<float4*>(c0 + k) = *reinterpret_cast<const float4*>(c0p + k);
      *reinterpret_cast<float4*>(s0 + k) = *reinterpret_cast<const float4*>(s0p + k);
      *reinterpret_cast<float4*>(c1 + k) = *reinterpret_cast<const float4*>(c1p + k);
      *reinterpret_cast<float4*>(s1 + k) = *reinterpret_cast<const float4*>(s1p + k);
    }
    const bool first_half = hl < px;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float C = __fadd_rn(__fmul_rn(c1[k], c0[k]), __fmul_rn(s1[k], s0[k]));
      float S = __fsub_rn(__fmul_rn(s1[k], c0[k]), __fmul_rn(c1[k], s0[k]));
      const float nrm = __fsqrt_rn(__fadd_rn(__fmul_rn(C, C), __fmul_rn(S, S)));
      C = __fdiv_rn(C, nrm);
      S = __fdiv_rn(S, nrm);
      // first half holds x (partner y); second half holds y (partner x)
      x[k] = first_half ? __fsub_rn(__fmul_rn(x[k], C), __fmul_rn(y[k], S))
                        : __fadd_rn(__fmul_rn(x[k], C), __fmul_rn(y[k], S));
    }
    // round to bf16: quantisation below starts from the stored bf16 row
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = bf16_bits_to_float(float_to_bf16_bits(x[k]));
    w = pack8_bf16(x);
  }

  const int64_t row = static_cast<int64_t>(u) * cap + i;
  if (pool == KVC_POOL_BF16) {
    if (valid) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(is_v ? a.pools.v_bf16 : a.pools.k_bf16);
      *reinterpret_cast<uint4*>(dst + row * d + hl * 8) = w;
    }
  } else {
    const bool row_mode = a.quant_mode == KVC_QUANT_ROW_FP16;
    const float qmax = pool == KVC_POOL_INT4 ? 7.f : 127.f;
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(x[k]));
    const int gl = row_mode ? lpr : 4;             // lanes per scale group
    for (int o2 = 1; o2 < gl; o2 <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o2));
    float s = 1.f;
    uint16_t s_bits;
    if (!row_mode) {
      if (amax > 0.f) {
        s = bf16_bits_to_float(float_to_bf16_bits(__fdiv_rn(amax, qmax)));
        s = fmaxf(s, __uint_as_float(0x00010000u));          // 2^-133
      }
      s_bits = float_to_bf16_bits(s);
    } else {
      if (amax > 0.f) {
        s = __half2float(__float2half_rn(__fdiv_rn(amax, qmax)));
        s = fminf(s, 65504.f);
        s = fmaxf(s, 5.9604644775390625e-08f);               // 2^-24
      }
      s_bits = __half_as_ushort(__float2half_rn(s));
    }
    int qv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      int q = amax > 0.f ? __float2int_rn(__fdiv_rn(x[k], s)) : 0;
      q = q > static_cast<int>(qmax) ? static_cast<int>(qmax) : q;
      q = q < -static_cast<int>(qmax) ? -static_cast<int>(qmax) : q;
      qv[k] = q;
    }
    if (valid) {
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
  }
  if (valid && hl == 0 && !is_v) {
    a.pools.pos_out[slot] = p2;
    if (a.pools.orig_pos_out) a.pools.orig_pos_out[slot] = p;
  }
}

}  // namespace

cudaError_t launch_compact(const CompactArgs& a, cudaStream_t stream) {
  const int pairs_per_block = (kThreads / 32) * (32 / (2 * (a.d / 8)));
  const int bx = (a.capacity + pairs_per_block - 1) / pairs_per_block;
  const int n_pools = a.pool_hi - a.pool_lo;
  if (bx == 0 || n_pools <= 0) return cudaSuccess;
  dim3 grid(bx, a.U, n_pools);
  compact_kernel<<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc
