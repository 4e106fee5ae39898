// Row readers shared by the decode-attention kernels: pointers of a storage
// class, scale loads, and the per-lane key dot products and value columns
// of bf16, int8 and int4 rows (dequantised as code * scale, PASK App. B.5).
#pragma once

#include "kvc_internal.cuh"

namespace kvc {

namespace {

struct PoolPtrs {
  const void* k;
  const void* v;
  const void* ks;
  const void* vs;
};

__device__ __forceinline__ PoolPtrs pool_ptrs(const kvc_pools& p, int pool) {
  if (pool == KVC_POOL_BF16) return {p.k_bf16, p.v_bf16, nullptr, nullptr};
  if (pool == KVC_POOL_INT8) return {p.k_i8, p.v_i8, p.k_i8_scale, p.v_i8_scale};
  return {p.k_i4, p.v_i4, p.k_i4_scale, p.v_i4_scale};
}

__device__ __forceinline__ float load_scale(const void* sp, int64_t row, int group, int d,
                                            bool row_mode) {
  const uint16_t* s = static_cast<const uint16_t*>(sp);
  if (row_mode) return __half2float(__ushort_as_half(__ldg(s + row)));
  return bf16_bits_to_float(__ldg(s + row * (d / 32) + group));
}

// FMAs of 8 consecutive key elements (starting at element e0) with every
// query head; the query rows in shared memory are pre-scaled to log2 units.
template <int D, int GG>
__device__ __forceinline__ void dot8(const float (&x)[8], const float (*qs)[D], int e0, int G,
                                     float (&s)[GG]) {
#pragma unroll
  for (int h = 0; h < GG; ++h) {
    if (h < G) {
      const float4 q0 = *reinterpret_cast<const float4*>(&qs[h][e0]);
      const float4 q1 = *reinterpret_cast<const float4*>(&qs[h][e0 + 4]);
      float t = s[h];
      t = fmaf(x[0], q0.x, t);
      t = fmaf(x[1], q0.y, t);
      t = fmaf(x[2], q0.z, t);
      t = fmaf(x[3], q0.w, t);
      t = fmaf(x[4], q1.x, t);
      t = fmaf(x[5], q1.y, t);
      t = fmaf(x[6], q1.z, t);
      t = fmaf(x[7], q1.w, t);
      s[h] = t;
    }
  }
}

// Scores of key row `row` of `pool` against every query head.  All loads
// of a batch (half a bf16 row, or a whole int8 / int4 row and its scales)
// are issued before any is used.
template <int D, int GG, bool BF>
__device__ __forceinline__ void key_dot(int pool, const PoolPtrs& pp, int64_t row, bool row_mode,
                                        const float (*qs)[D], int G, float (&s)[GG]) {
  if (BF || pool == KVC_POOL_BF16) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(pp.k) + row * D);
#pragma unroll
    for (int half = 0; half < D / 64; ++half) {
      uint4 w[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) w[v] = __ldg(src + half * 8 + v);
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint32_t r[4] = {w[v].x, w[v].y, w[v].z, w[v].w};
        float x[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[2 * k] = __uint_as_float(r[k] << 16);
          x[2 * k + 1] = __uint_as_float(r[k] & 0xffff0000u);
        }
        dot8<D, GG>(x, qs, half * 64 + v * 8, G, s);
      }
    }
  } else {
    constexpr int NG = D / 32;                   // scale groups per row
    float sc[NG];
    if (row_mode) {
      const float r = load_scale(pp.ks, row, 0, D, true);
#pragma unroll
      for (int g = 0; g < NG; ++g) sc[g] = r;
    } else {
#pragma unroll
      for (int g = 0; g < NG; ++g) sc[g] = load_scale(pp.ks, row, g, D, false);
    }
    if (pool == KVC_POOL_INT8) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const int8_t*>(pp.k) + row * D);
      uint4 w[D / 16];
#pragma unroll
      for (int v = 0; v < D / 16; ++v) w[v] = __ldg(src + v);
#pragma unroll
      for (int v = 0; v < D / 16; ++v) {
        const uint32_t r[4] = {w[v].x, w[v].y, w[v].z, w[v].w};
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
          float x[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            x[k] = static_cast<float>(static_cast<int8_t>(r[2 * hlf + (k >> 2)] >> (8 * (k & 3)))) *
                   sc[(v * 16) / 32];
          dot8<D, GG>(x, qs, v * 16 + hlf * 8, G, s);
        }
      }
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(pp.k) + row * (D / 2));
      uint4 w[D / 32];
#pragma unroll
      for (int v = 0; v < D / 32; ++v) w[v] = __ldg(src + v);
#pragma unroll
      for (int v = 0; v < D / 32; ++v) {
        const uint32_t r[4] = {w[v].x, w[v].y, w[v].z, w[v].w};
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          float x[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)      // low nibble = even element; sign-extended
            x[k] = static_cast<float>(static_cast<int32_t>(r[k4] << (28 - 4 * k)) >> 28) * sc[v];
          dot8<D, GG>(x, qs, v * 32 + k4 * 8, G, s);
        }
      }
    }
  }
}

// This lane's d / 32 columns of value row `row` of `pool`, dequantised.
template <int D, bool BF>
__device__ __forceinline__ void load_value_cols(int pool, const PoolPtrs& pp, int64_t row, int lane,
                                                bool row_mode, float (&v)[D / 32]) {
  constexpr int NC = D / 32;
  const int c0 = lane * NC;
  if (BF || pool == KVC_POOL_BF16) {
    const uint16_t* src = static_cast<const uint16_t*>(pp.v) + row * D + c0;
    if (NC == 4) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
      v[0] = __uint_as_float(w.x << 16);
      v[1] = __uint_as_float(w.x & 0xffff0000u);
      v[2] = __uint_as_float(w.y << 16);
      v[3] = __uint_as_float(w.y & 0xffff0000u);
    } else {
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(src));
      v[0] = __uint_as_float(w << 16);
      v[1 % NC] = __uint_as_float(w & 0xffff0000u);
    }
  } else if (pool == KVC_POOL_INT8) {
    const float sc = load_scale(pp.vs, row, c0 / 32, D, row_mode);
    const int8_t* src = static_cast<const int8_t*>(pp.v) + row * D + c0;
    if (NC == 4) {
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(src));
#pragma unroll
      for (int k = 0; k < NC; ++k) v[k] = static_cast<float>(static_cast<int8_t>(w >> (8 * k))) * sc;
    } else {
      const uint16_t w = __ldg(reinterpret_cast<const uint16_t*>(src));
#pragma unroll
      for (int k = 0; k < NC; ++k) v[k] = static_cast<float>(static_cast<int8_t>(w >> (8 * k))) * sc;
    }
  } else {
    const float sc = load_scale(pp.vs, row, c0 / 32, D, row_mode);
    const uint8_t* src = static_cast<const uint8_t*>(pp.v) + row * (D / 2) + c0 / 2;
    uint32_t w;
    if (NC == 4) w = __ldg(reinterpret_cast<const uint16_t*>(src));
    else w = __ldg(src);
#pragma unroll
    for (int k = 0; k < NC; ++k)
      v[k] = static_cast<float>(static_cast<int32_t>(w << (28 - 4 * k)) >> 28) * sc;
  }
}

}  // namespace

}  // namespace kvc
