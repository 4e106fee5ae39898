// Internal declarations shared by the libkvc translation units: launch
// parameter blocks, host launchers, and small device helpers (inline PTX for
// mbarriers, TMA and tcgen05; bf16 conversions).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

constexpr int kTileTokens = 128;     // tokens per scoring tile (MMA M or N)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s bound on any device wait

// ----------------------------------------------------------------------------
// launch parameter blocks
// ----------------------------------------------------------------------------

struct ScoreArgs {
  int32_t U, L, Hkv, B;
  int64_t T;
  int32_t d, W, G, R;          // R = W * G window rows per unit
  int32_t Rp;                  // R rounded up to a multiple of 16 (MMA N of pass 2)
  int32_t n_tiles;             // ceil(T / 128)
  int32_t chunk_tiles;         // tiles per work item
  int32_t items_per_unit;      // S
  int32_t n_items;             // U * S
  int32_t page_size;
  int32_t accumulate;
  int32_t n_stages;
  int32_t q_rows;              // Q rows held in shared memory (multiple of 128)
  float scale_log2;            // softmax_scale * log2(e)
  const float* row_lse;        // optional [U][R] natural-log row statistics
  const float* bonus;
  float* scores;
  float* page_scores;
  int32_t* unit_status;
  uint32_t* counters;          // [U] pass-1 chunks finished per unit
  float2* stats;               // [U][S][R] (max, sum) in the log2 domain
  int32_t stall_unit;            // test hook (-1 = none): this unit's pass-1 wait never completes
  const __nv_bfloat16* k_small;  // small-window path: keys [U][T][d]
  const __nv_bfloat16* q_small;  // small-window path: window rows [U][R][d]
};

struct SelectArgs {
  int32_t U, L, Hkv, B;
  int64_t T;
  int32_t d;
  int64_t n_items;             // T or T / page_size
  int32_t page_size;
  int32_t budget_items;        // token / page mode
  int64_t budget_bytes;        // byte mode
  int32_t sink_items, recent_items;
  int32_t capacity;
  int32_t byte_mode;
  int32_t quant_mode;
  int32_t n_tags, n_groups;
  const uint8_t* flags;
  const uint8_t* tags;
  const uint8_t* table;
  const float* scores;
  int32_t* kept_idx;
  int32_t* kept_count;
  int32_t* unit_status;
  int64_t* floor_excess;
  int32_t cache_items;         // 1: item keys staged in shared memory
  void* long_ws;               // multi-CTA selection of long units (token / page mode), or null
  int32_t stall_unit;          // test hook (-1 = none): this unit's wait for its scores never completes
};

// Workspace of the multi-CTA selection of long units (token / page mode).
size_t select_long_ws_bytes(int64_t U, int64_t n_items);

struct CompactArgs {
  int32_t U, d;
  int64_t T;
  int32_t capacity;
  int32_t renumber;
  int32_t quant_mode;
  int64_t rope_max_pos;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* pos_in;
  const int32_t* kept_idx;
  const int32_t* kept_count;
  const float* cos;
  const float* sin;
  kvc_pools pools;
  int32_t* unit_status;
  int32_t pool_lo, pool_hi;    // pools to process: [pool_lo, pool_hi)
  kvc_ref_store ref;           // reference store (ref.ref_pos == NULL: none)
  int32_t rope_layout;         // KVC_ROPE_*
  int32_t rotary_dim;          // rotated leading elements (a multiple of 16, <= d)
};

struct DecodeArgs {
  int32_t U, G, d, Hkv, L, B;
  int32_t capacity;
  int32_t quant_mode;
  int32_t splits;
  float scale;
  const __nv_bfloat16* q;
  kvc_pools pools;
  const int32_t* kept_count;
  __nv_bfloat16* out;
  float* ws_ml;                // [U][splits][G][2]
  float* ws_acc;               // [U][splits][G][d]
  int32_t pool_lo, pool_hi;
  // engine attention (PASK App. B.5): G then counts rows per unit, G_heads n_q
  int32_t n_q;                 // queries per head
  const int32_t* q_pos;        // [B][n_q] logical query positions, or null: every key visible
  const int32_t* pool_pos;     // [KVC_N_POOLS][U][capacity] key positions of the pools, or null
  bool has_pools;
  const __nv_bfloat16* rec_k;  // recent storage: bf16 [U][rec_cap][d]
  const __nv_bfloat16* rec_v;
  const int32_t* rec_pos;      // [U][rec_cap] or null
  const int32_t* rec_count;    // [U] or null (empty)
  int32_t rec_cap;
  const __nv_bfloat16* cur_k;  // current storage: bf16 [U][cur_cap][d]
  const __nv_bfloat16* cur_v;
  const int32_t* cur_pos;
  const int32_t* cur_count;
  int32_t cur_cap;
};

struct BonusArgs {
  int32_t batch;
  int64_t T;
  int32_t n_spans;
  int32_t step;
  float sigma, lambda;
  const int32_t* span_seq;     // [n_spans] sequence b of each span
  const int64_t* span_a;       // [n_spans] first token
  const int64_t* span_b;       // [n_spans] one past the last token
  const int32_t* span_next;    // [n_spans] next reading step s*, or < step: none
  float* bonus;                // [B][T]
};

// CommitKV deletion effect (Sec. 3.2): window attention of a unit's R = G W
// rows, split into work items of chunk_tiles key tiles; then the per-page
// weights and value sums.
struct EffectArgs {
  int32_t U, L, Hkv, B, G, W, R, Rp;
  int64_t T;
  int32_t n_tiles, chunk_tiles, splits, n_items;
  int32_t nk, nv;              // nk: tiles in the key / value stage ring; nv unused
  float scale_log2;            // softmax scale * log2(e)
  float* part_u;               // [n_items][R][128] unnormalised value sums of a split
  float2* part_ml;             // [n_items][R] (max, exp2-sum) of y = z * scale_log2
  float* o;                    // [U][R][128] window outputs
  float* lse;                  // [U][R] natural-log softmax denominators
  float* s;                    // [B][L][n_pages][H_q][W] page weights
  float* u;                    // [B][L][n_pages][H_q][W][128] page value sums
  const int32_t* page_start;   // [B][n_pages]
  const int32_t* page_len;     // [B][n_pages]
  int32_t n_pages;
  const __nv_bfloat16* k;      // [U][T][128]
  const __nv_bfloat16* v;      // [U][T][128]
  const __nv_bfloat16* q;      // [U][R][128]
  float* effect;               // [B][L][n_pages] (zeroed before the page kernel)
  int32_t* unit_status;        // optional [U]
};

// CommitKV Eqs. 9-11 for one layer of each sequence.
struct CommitArgs {
  int32_t B, L, Hq, W, n_pages, layer;
  float tau_use, tau_dead, rho_use, rho_dead, tau_joint;
  const float* r_minus;        // [B][L][n_pages]
  const float* r_plus;         // [B][L][n_pages]
  const uint8_t* compared;     // [B][n_pages]
  const float* o;              // record of the post-commit window: [B][L][H_q][W][128]
  const float* s;              // [B][L][n_pages][H_q][W]
  const float* u;              // [B][L][n_pages][H_q][W][128]
  float* acc;                  // workspace [B][H_q W][128]
  uint8_t* state;              // [B][n_pages]
  uint8_t* retire;             // [B][n_pages]
  float* joint;                // optional [B][n_pages]
};

struct ProtectArgs {
  int32_t B, L, n_pages, layer;
  int32_t budget_tokens, max_pages;
  const float* r_minus;        // [B][L][n_pages]
  const uint8_t* pending;      // [B][n_pages]
  const int32_t* page_len;     // [B][n_pages]
  uint8_t* protect;            // [B][n_pages]
};

struct FlagArgs {
  int32_t B, n_pages;
  int64_t T;
  const int32_t* page_start;   // [B][n_pages]
  const int32_t* page_len;     // [B][n_pages]
  const uint8_t* retire;       // optional [B][n_pages]
  const uint8_t* protect;      // optional [B][n_pages]
  uint8_t* flags;              // [B][T]
};

// host launchers (each returns a cudaError_t from the launch)
cudaError_t launch_bonus(const BonusArgs& a, cudaStream_t stream);
cudaError_t launch_pool(const float* in, float* out, int64_t rows, int64_t n, int kernel, int mode,
                        cudaStream_t stream);
cudaError_t launch_shared_sum(const float* scores, float* shared, int B, int units_per_seq, int64_t n,
                              cudaStream_t stream);
cudaError_t launch_broadcast(const int32_t* kept_seq, const int32_t* count_seq, int32_t* kept,
                             int32_t* count, int B, int units_per_seq, int cap, cudaStream_t stream);
cudaError_t launch_score(const ScoreArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_q,
                         int grid, size_t smem_bytes, cudaStream_t stream);
size_t score_smem_bytes(int d, int q_rows, int n_stages);
int small_rows(int R);
size_t score_small_smem_bytes(int d);
cudaError_t launch_score_small(const ScoreArgs& a, int splits, float* logits, float2* split_stats,
                               float* lse2, cudaStream_t stream);
cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream, size_t smem_bytes);
cudaError_t launch_select_long(const SelectArgs& a, cudaStream_t stream);
cudaError_t launch_compact(const CompactArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_engine(const DecodeArgs& a, cudaStream_t stream);
size_t effect_smem_bytes(int Rp, int n_stages);
cudaError_t launch_effect(const EffectArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                          const CUtensorMap& tmap_q, int grid, size_t smem_bytes, cudaStream_t stream);
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream);
cudaError_t launch_protect(const ProtectArgs& a, cudaStream_t stream);
cudaError_t launch_flags(const FlagArgs& a, cudaStream_t stream);

// ----------------------------------------------------------------------------
// device helpers
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// fp32 -> bf16 bits, round to nearest even (matches __float2bfloat16_rn).
__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// One test of the phase with parity `parity`.  If it has not completed, the
// thread is suspended in hardware until it completes or ~0.1 ms pass (the
// suspend-time hint), so waiting warps do not consume issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(100000)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with parity `parity` to complete.  Returns false
// (and raises *abort) if it has not completed within kWaitLimitNs, or if
// another role already raised *abort.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
}

// Bounded wait for a thread whose latency matters less than the issue slots
// it would take from busy warps on its sub-partition (a single producer or
// MMA-issuing thread): after each failed test it sleeps for `sleep_ns`.
__device__ __forceinline__ bool mbar_wait_backoff(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  uint32_t sleep_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  while (true) {
    __nanosleep(sleep_ns);
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA ----------------------------------------------------------------------

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- tcgen05 ----------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.  The load and its
// wait are one asm statement so no use of the registers can precede the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's TMEM lane (load and wait in
// one asm statement).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (load and wait in
// one asm statement).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Asynchronous half of tmem_ld32: issue the load, do not wait.  The
// registers may only be read after tmem_ld_wait() on the same array.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Asynchronous 16-column load: issue only; read the registers after
// tmem_ld_wait16() on the same array.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Wait for every outstanding tcgen05.ld of this thread.  The registers of
// `r` are tied to the wait so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),
                 "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]),
                 "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// A row count read from caller memory, limited to [0, cap] (rows past a
// pool's capacity would belong to the next unit or lie outside the pool).
__device__ __forceinline__ int clamp_count(int n, int cap) { return n < 0 ? 0 : (n > cap ? cap : n); }

// a / b from y = RN(1 / b), the reciprocal rounded to nearest: q0 = RN(a y),
// r = a - b q0 (one fused multiply-add), q = RN(q0 + r y) -- the correction
// step of Markstein's division (IA-64).  The quotient is within one ulp of
// IEEE division, not always equal to it, so it only serves where a rounded
// integer code is formed from it: the quantiser, whose codes rint(a / b)
// equal those of IEEE division for every bf16 dividend with every bf16 and
// every fp16 divisor in [2^-126, 2^125] with |a| <= 256 b (checked
// exhaustively on the GPU; a group's quotients stay below about qmax).  A
// zero quotient may come out with the other sign.
__device__ __forceinline__ float div_by_recip(float a, float b, float y) {
  const float q0 = __fmul_rn(a, y);
  const float r = __fmaf_rn(-q0, b, a);
  return __fmaf_rn(r, y, q0);
}

__device__ __forceinline__ bool recip_div_ok(float b) {
  return b >= 0x1p-126f && b <= 0x1p125f;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Shared-memory matrix descriptor of a K-major bf16 operand stored with the
// 128-byte swizzle: rows of 64 elements (128 B), 8-row atoms of 1024 B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(1) << 16;                     // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;             // stride byte offset: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                     // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                     // 128-byte swizzle
  return d;
}

// Shared-memory matrix descriptor of a K-major bf16 operand of 16 columns
// stored with the 32-byte swizzle: rows of 16 elements (32 B), 8-row atoms
// of 256 B.
__device__ __forceinline__ uint64_t sw32_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(1) << 16;                     // leading byte offset (unused)
  d |= static_cast<uint64_t>(256 >> 4) << 32;              // stride byte offset: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                     // descriptor version
  d |= static_cast<uint64_t>(6) << 61;                     // 32-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major.
__host__ __device__ constexpr uint32_t mma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier over `nthreads` threads that also ORs `pred` across them.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

}  // namespace kvc
