// Exhaustive check of div_by_recip (the compaction's quantiser division)
// against IEEE division: every finite bf16 dividend a with every bf16 or
// fp16 divisor b of the fast path such that |a| <= 256 b -- the
// quantiser's domain: a group's scale is at least its largest magnitude
// over qmax (rounded to the scale format), so every quotient it forms is at
// most about qmax (127) in magnitude.  Prints the number of mismatches of
// the rounded integer code (exit status 1 if any) and, for information, of
// the quotient's bits (normal quotients: the correction step is within one
// ulp, not always exact).
#include <cstdio>
#include "../../budgeted_kv_cache_gb300/csrc/kvc_internal.cuh"

using namespace kvc;

__global__ void check(int fp16_divisor, unsigned long long* bad_code, unsigned long long* bad_bits,
                      unsigned long long* tested) {
  const uint32_t bd = blockIdx.x;                 // divisor bits (65536 blocks)
  float b;
  if (fp16_divisor) {
    const __half h = __ushort_as_half(static_cast<unsigned short>(bd));
    b = __half2float(h);
  } else {
    b = __uint_as_float(bd << 16);
  }
  if (!(b > 0.f) || isinf(b) || !recip_div_ok(b)) return;
  const float y = __fdiv_rn(1.f, b);
  unsigned long long nc = 0, nb = 0, nt = 0;
  for (uint32_t ad = threadIdx.x; ad < 65536u; ad += blockDim.x) {
    const float a = __uint_as_float(ad << 16);
    if (isnan(a) || isinf(a) || fabsf(a) > 256.f * b) continue;
    const float q = __fdiv_rn(a, b);
    const float f = div_by_recip(a, b, y);
    ++nt;
    if (__float2int_rn(q) != __float2int_rn(f)) ++nc;
    if (fabsf(q) >= 0x1p-126f && !isinf(q) && __float_as_uint(q) != __float_as_uint(f)) ++nb;
  }
  atomicAdd(bad_code, nc);
  atomicAdd(bad_bits, nb);
  atomicAdd(tested, nt);
}

int main() {
  unsigned long long* d;
  if (cudaMalloc(&d, 3 * sizeof(unsigned long long)) != cudaSuccess) return 2;
  int rc = 0;
  for (int k = 0; k < 2; ++k) {
    cudaMemset(d, 0, 3 * sizeof(unsigned long long));
    check<<<65536, 256>>>(k, d, d + 1, d + 2);
    unsigned long long h[3];
    if (cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
    printf("%s divisors: %llu pairs, %llu code mismatches, %llu quotient mismatches\n",
           k ? "fp16" : "bf16", h[2], h[0], h[1]);
    if (h[0] || h[2] < 100000000ull) rc = 1;
  }
  return rc;
}
