// C-ABI entry points of libkvc: argument validation, launch configuration,
// tensor-map encoding and workspace layout.  Every step of the pass runs in
// the kernels of score_tc.cu, select.cu, compact.cu and decode.cu.
#include <math.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "kvc_internal.cuh"

using namespace kvc;

namespace {

// Process-wide launch-plan overrides set through kvc_set_overrides (tuning
// sweeps, failure tests); 0 / -1 = the library's own choice.
std::atomic<int32_t> g_score_chunk_tiles{0};
std::atomic<int32_t> g_decode_splits{0};
std::atomic<int32_t> g_effect_chunk_tiles{0};
std::atomic<int32_t> g_score_stall_unit{-1};
std::atomic<int32_t> g_select_stall_unit{-1};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DevInfo {
  int sms = 0;
  int major = 0, minor = 0;
  int64_t l2_bytes = 0;
  bool ok = false;
};

// Properties of the current device, cached per device ordinal.
bool device_info(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  static DevInfo cache[64];
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev].ok) {
    DevInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return false;
    int l2 = 0;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return false;
    d.l2_bytes = l2;
    d.ok = true;
    cache[dev] = d;
  }
  *out = cache[dev];
  return true;
}

kvc_status check_device(DevInfo* info) {
  if (!device_info(info)) return KVC_ERR_NO_DEVICE;
  if (info->major != 10 || info->minor != 3) return KVC_ERR_NO_DEVICE;   // built for sm_103a only
  return KVC_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

kvc_status check_shape(const kvc_shape* s) {
  if (!s) return KVC_ERR_INVALID_ARG;
  if (s->batch < 1 || s->n_layers < 1 || s->n_q_heads < 1 || s->n_kv_heads < 1) return KVC_ERR_INVALID_ARG;
  if (s->n_q_heads % s->n_kv_heads) return KVC_ERR_INVALID_ARG;
  if (s->n_tokens < 1 || s->n_tokens > 0x7fffffffLL) return KVC_ERR_INVALID_ARG;
  if (s->head_dim != 64 && s->head_dim != 128) return KVC_ERR_UNSUPPORTED;
  const int64_t units = static_cast<int64_t>(s->batch) * s->n_layers * s->n_kv_heads;
  if (units > (1 << 24)) return KVC_ERR_UNSUPPORTED;
  return KVC_OK;
}

int64_t n_units(const kvc_shape* s) {
  return static_cast<int64_t>(s->batch) * s->n_layers * s->n_kv_heads;
}

// ---------------------------------------------------------------- scoring plan
struct ScorePlan {
  bool small = false;          // R <= 16: the CUDA-core path
  int small_splits = 0;
  size_t ws_logits = 0, ws_split = 0;
  int grid = 0;
  int n_tiles = 0, chunk_tiles = 0, S = 0;
  int R = 0, q_rows = 0, n_stages = 0;
  size_t smem = 0;
  size_t ws_counters = 0, ws_stats = 0, ws_total = 0;
};

kvc_status plan_score(const kvc_shape* s, int32_t window, ScorePlan* p) {
  kvc_status st = check_shape(s);
  if (st != KVC_OK) return st;
  if (window < 1 || window > s->n_tokens) return KVC_ERR_INVALID_ARG;
  const int G = s->n_q_heads / s->n_kv_heads;
  const int64_t R = static_cast<int64_t>(window) * G;
  if (R < 1 || R > 256) return KVC_ERR_UNSUPPORTED;
  DevInfo info;
  if ((st = check_device(&info)) != KVC_OK) return st;
  p->grid = info.sms;
  p->R = static_cast<int>(R);
  if (R <= 16 && n_units(s) <= 65535) {
    // a thin contraction: the CUDA-core path reads the keys once
    const int64_t U = n_units(s);
    const int RR = small_rows(p->R);
    int64_t want = (8LL * info.sms + U - 1) / U;
    want = std::min<int64_t>(want, (s->n_tokens + 2047) / 2048);
    p->small = true;
    p->small_splits = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 64)));
    p->ws_logits = (static_cast<size_t>(U) * s->n_tokens * RR * 4 + 255) / 256 * 256;
    p->ws_split = (static_cast<size_t>(U) * p->small_splits * RR * 8 + 255) / 256 * 256;
    p->ws_total = p->ws_logits + p->ws_split + (static_cast<size_t>(U) * RR * 4 + 255) / 256 * 256;
    return KVC_OK;
  }
  p->n_tiles = static_cast<int>((s->n_tokens + kTileTokens - 1) / kTileTokens);
  // Each unit's tiles are split into S slices of near-equal size, one work
  // item each.  Every item costs a fixed overhead (its queries' load, the
  // pass switch, the statistics exchange and the wait for the unit's other
  // items; measured at about 2.3 tile-times of both passes), and the items
  // run in rounds of `grid`.  Pick the split that minimises rounds x (slice
  // + overhead); a unit's items never outnumber the CTAs, because pass 2 of
  // each item waits for all of them.  (Smaller slices would let pass 2 find
  // its keys in L2, but with this kernel's epilogue the extra per-item cost
  // outweighs the saved HBM reads: measured 1.27 ms with 16 slices per unit
  // against 1.04 ms with whole units at the 32K-token workload.)
  const int64_t U = n_units(s);
  int chunk = p->n_tiles;
  double best = 1e300;
  const int s_max = std::min(p->n_tiles, p->grid);
  for (int sc = 1; sc <= s_max; ++sc) {
    const int c = (p->n_tiles + sc - 1) / sc;
    if ((p->n_tiles + c - 1) / c != sc) continue;                      // distinct chunk sizes
    const double cost = static_cast<double>((U * sc + p->grid - 1) / p->grid) * (c + 2.3);
    if (cost < best - 1e-9) {
      best = cost;
      chunk = c;
    }
  }
  if (const int v = g_score_chunk_tiles.load(std::memory_order_relaxed); v >= 1)   // override
    chunk = v;
  chunk = std::max(chunk, (p->n_tiles + p->grid - 1) / p->grid);   // S <= grid (co-resident unit)
  p->chunk_tiles = std::min(chunk, p->n_tiles);
  p->S = (p->n_tiles + p->chunk_tiles - 1) / p->chunk_tiles;
  const int64_t items = n_units(s) * p->S;
  if (items > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
  p->q_rows = static_cast<int>((R + 127) / 128 * 128);
  const size_t max_smem = 232448;       // 227 KB per block on sm_103
  const size_t stage = static_cast<size_t>(s->head_dim / 64) * 128 * 128;
  const size_t fixed = score_smem_bytes(s->head_dim, p->q_rows, 0);
  int stages = static_cast<int>((max_smem - fixed - 16 * 8) / (stage + 16));
  stages = std::min(stages, 8);
  if (stages < 2) return KVC_ERR_UNSUPPORTED;
  p->n_stages = stages;
  // at least 120 KB so that exactly one CTA (and one 512-column TMEM
  // allocation) lives on each SM
  p->smem = std::max(score_smem_bytes(s->head_dim, p->q_rows, stages), static_cast<size_t>(120 * 1024));
  p->ws_counters = (static_cast<size_t>(n_units(s)) * 4 + 255) / 256 * 256;
  p->ws_stats = static_cast<size_t>(items) * R * sizeof(float2);
  p->ws_total = p->ws_counters + (p->ws_stats + 255) / 256 * 256;
  return KVC_OK;
}

kvc_status encode_3d(CUtensorMap* map, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                     uint32_t b0, uint32_t b1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return KVC_ERR_CUDA;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KVC_OK : KVC_ERR_CUDA;
}

// ---------------------------------------------------------------- policy checks
struct SelectPlan {
  bool byte_mode = false;
  int P = 1;
  int64_t n_items = 0;
  int sink_items = 0, recent_items = 0;
  int budget_items = 0;
};

kvc_status plan_select(const kvc_shape* s, const kvc_policy* pol, SelectPlan* sp) {
  kvc_status st = check_shape(s);
  if (st != KVC_OK) return st;
  if (!pol) return KVC_ERR_INVALID_ARG;
  const bool tok = pol->budget_tokens > 0, byt = pol->budget_bytes > 0;
  if (tok == byt) return KVC_ERR_INVALID_ARG;                  // exactly one budget
  if (pol->budget_tokens < 0 || pol->budget_bytes < 0) return KVC_ERR_INVALID_ARG;
  if (pol->n_sink < 0 || pol->n_recent < 0) return KVC_ERR_INVALID_ARG;
  if (pol->quant_mode != KVC_QUANT_G32_BF16 && pol->quant_mode != KVC_QUANT_ROW_FP16)
    return KVC_ERR_INVALID_ARG;
  if (pol->renumber != 0 && pol->renumber != 1) return KVC_ERR_INVALID_ARG;
  const int64_t T = s->n_tokens;
  const int P = pol->page_size;
  if (P < 1 || P > 32 || (P & (P - 1))) return KVC_ERR_INVALID_ARG;
  sp->byte_mode = byt;
  sp->P = P;
  if (byt) {
    if (P != 1) return KVC_ERR_UNSUPPORTED;
    if (!pol->tags || !pol->action_table || pol->n_tags < 1 || pol->n_layer_groups < 1 ||
        pol->n_layer_groups > s->n_layers)
      return KVC_ERR_INVALID_ARG;
    if (pol->capacity < T) return KVC_ERR_INVALID_ARG;
    if (T * 4 * s->head_dim >= (1LL << 32)) return KVC_ERR_UNSUPPORTED;
    sp->n_items = T;
    sp->sink_items = static_cast<int>(std::min<int64_t>(pol->n_sink, T));
    sp->recent_items = static_cast<int>(std::min<int64_t>(pol->n_recent, T));
  } else {
    if (pol->capacity < pol->budget_tokens) return KVC_ERR_INVALID_ARG;
    if (P > 1 && (T % P != 0 || pol->budget_tokens % P != 0)) return KVC_ERR_INVALID_ARG;
    sp->n_items = T / P;
    sp->budget_items = pol->budget_tokens / P;
    if (P == 1) {
      sp->sink_items = static_cast<int>(std::min<int64_t>(pol->n_sink, T));
      sp->recent_items = static_cast<int>(std::min<int64_t>(pol->n_recent, T));
    } else {
      const int64_t first = (static_cast<int64_t>(pol->n_sink) + P - 1) / P;
      const int64_t rstart = std::max<int64_t>(0, T - pol->n_recent) / P;
      sp->sink_items = static_cast<int>(std::min<int64_t>(first, sp->n_items));
      sp->recent_items = static_cast<int>(sp->n_items - rstart);
    }
  }
  if (pol->capacity < 1 && (pol->budget_tokens > 0 || byt)) return KVC_ERR_INVALID_ARG;
  if (static_cast<int64_t>(KVC_N_POOLS) * n_units(s) * pol->capacity > (1LL << 40)) return KVC_ERR_UNSUPPORTED;
  return KVC_OK;
}

int decode_splits(const kvc_shape* s, const kvc_policy* pol, int sms) {
  const int64_t U = n_units(s);
  const int64_t rows = static_cast<int64_t>(pol->capacity) * (pol->budget_bytes > 0 ? 3 : 1);
  // byte mode (the register kernel): about eight CTAs (32 warps) per SM to
  // keep enough row loads in flight; bf16 pools (the bulk-staged kernel,
  // three CTAs per SM): as many splits as fit one wave of resident CTAs, so
  // that no CTA waits for a second wave and most units need no merge; no
  // split shorter than 128 rows
  int64_t want = pol->budget_bytes > 0 ? (8LL * sms + U - 1) / U : std::max<int64_t>(1, 3LL * sms / U);
  if (const int v = g_decode_splits.load(std::memory_order_relaxed); v >= 1) want = v;   // override
  const int64_t most = std::max<int64_t>(1, (rows + 127) / 128);
  want = std::min<int64_t>(std::min<int64_t>(want, most), 32);
  return static_cast<int>(std::max<int64_t>(want, 1));
}

struct EnginePlan {
  int splits = 1, rows = 0;
  bool byte_mode = false;
  size_t ws = 0;
};

kvc_status plan_engine(const kvc_shape* s, const kvc_policy* pol, int32_t n_q, bool with_pools,
                       const kvc_bf16_rows* rec, const kvc_bf16_rows* cur, EnginePlan* p) {
  kvc_status st = check_shape(s);
  if (st != KVC_OK) return st;
  if (n_q < 1) return KVC_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(s->n_q_heads / s->n_kv_heads) * n_q;
  if (rows > 16) return KVC_ERR_UNSUPPORTED;
  int64_t keys = 0;
  if (with_pools) {
    SelectPlan sp;
    if ((st = plan_select(s, pol, &sp)) != KVC_OK) return st;
    p->byte_mode = sp.byte_mode;
    keys += static_cast<int64_t>(pol->capacity) * (sp.byte_mode ? 3 : 1);
  }
  for (const kvc_bf16_rows* r : {rec, cur}) {
    if (r && r->count) {
      if (r->capacity < 1 || !r->k || !r->v) return KVC_ERR_INVALID_ARG;
      keys += r->capacity;
    }
  }
  DevInfo info;
  if ((st = check_device(&info)) != KVC_OK) return st;
  const int64_t U = n_units(s);
  // the register kernel (int8 / int4 pools): about eight CTAs per SM; the
  // bulk-staged kernel (bf16 storages): one wave of resident CTAs
  const int per_sm = rows >= 16 ? 2 : 3;
  int64_t want = p->byte_mode ? (8LL * info.sms + U - 1) / U
                              : std::max<int64_t>(1, static_cast<int64_t>(per_sm) * info.sms / U);
  want = std::min<int64_t>(std::min<int64_t>(want, std::max<int64_t>(1, (keys + 127) / 128)), 32);
  p->splits = static_cast<int>(std::max<int64_t>(want, 1));
  p->rows = static_cast<int>(rows);
  if (p->splits > 1) {
    const size_t slots = static_cast<size_t>(U) * p->splits * rows;
    p->ws = (slots * 2 * sizeof(float) + 255) / 256 * 256 + slots * s->head_dim * sizeof(float);
  }
  return KVC_OK;
}

// The address the device reads `*p` through: memory of the current device
// or managed memory as it is, page-locked host memory through its mapping
// (unregistered host memory and another device's memory are refused).
kvc_status device_view(const void** p) {
  cudaPointerAttributes at;
  int dev = -1;
  if (cudaPointerGetAttributes(&at, *p) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KVC_ERR_INVALID_ARG;
  }
  if (at.type == cudaMemoryTypeDevice) return at.device == dev ? KVC_OK : KVC_ERR_INVALID_ARG;
  if (at.type == cudaMemoryTypeManaged) return KVC_OK;
  if (at.type == cudaMemoryTypeHost && at.devicePointer) {
    *p = at.devicePointer;
    return KVC_OK;
  }
  return KVC_ERR_INVALID_ARG;
}

}  // namespace

// ---------------------------------------------------------------- CommitKV plans
struct EffectPlan {
  int R = 0, Rp = 0, n_tiles = 0, chunk = 0, splits = 0, n_items = 0, grid = 0, nk = 0, nv = 0;
  size_t smem = 0, ws_part_u = 0, ws_total = 0;
};

kvc_status plan_effect(const kvc_shape* s, int32_t window, EffectPlan* p) {
  kvc_status st = check_shape(s);
  if (st != KVC_OK) return st;
  if (s->head_dim != 128) return KVC_ERR_UNSUPPORTED;
  if (window < 1 || window > s->n_tokens) return KVC_ERR_INVALID_ARG;
  const int64_t R = static_cast<int64_t>(window) * (s->n_q_heads / s->n_kv_heads);
  if (R > 64) return KVC_ERR_UNSUPPORTED;
  DevInfo info;
  if ((st = check_device(&info)) != KVC_OK) return st;
  p->R = static_cast<int>(R);
  p->Rp = (p->R + 15) / 16 * 16;
  p->n_tiles = static_cast<int>((s->n_tokens + kTileTokens - 1) / kTileTokens);
  const int64_t U = n_units(s);
  // chunks of 2..8 tiles: the keys of all resident items stay in L2 between
  // the two passes, and there are about two items per SM
  const int64_t want = (U * p->n_tiles + 2 * info.sms - 1) / (2 * info.sms);
  p->chunk = static_cast<int>(std::min<int64_t>(std::max<int64_t>(want, 2), 8));
  if (const int v = g_effect_chunk_tiles.load(std::memory_order_relaxed); v >= 1)   // override
    p->chunk = v;
  p->chunk = std::min(p->chunk, p->n_tiles);
  p->splits = (p->n_tiles + p->chunk - 1) / p->chunk;
  const int64_t items = U * p->splits;
  if (items > 0x7fffffffLL || U * p->R > 0x7fffffffLL || U > 65535) return KVC_ERR_UNSUPPORTED;
  p->n_items = static_cast<int>(items);
  p->grid = static_cast<int>(std::min<int64_t>(items, info.sms));
  // as many 32 KB key / value stages as fit beside the queries and P buffers
  p->nk = 0;
  for (int ns = 8; ns >= 2; --ns)
    if (effect_smem_bytes(p->Rp, ns) <= 232448) {
      p->nk = ns;
      break;
    }
  if (p->nk == 0) return KVC_ERR_UNSUPPORTED;
  p->nv = 0;
  p->smem = effect_smem_bytes(p->Rp, p->nk);
  p->ws_part_u = (static_cast<size_t>(items) * p->R * 128 * 4 + 255) / 256 * 256;
  p->ws_total = p->ws_part_u + (static_cast<size_t>(items) * p->R * 8 + 255) / 256 * 256;
  return KVC_OK;
}

extern "C" {

kvc_status kvc_set_overrides(const kvc_overrides* o) {
  if (o && (o->score_chunk_tiles < 0 || o->score_chunk_tiles > (1 << 20) || o->decode_splits < 0 ||
            o->decode_splits > 32 || o->effect_chunk_tiles < 0 || o->effect_chunk_tiles > (1 << 20) ||
            o->score_stall_unit < -1 || o->select_stall_unit < -1))
    return KVC_ERR_INVALID_ARG;
  g_score_chunk_tiles.store(o ? o->score_chunk_tiles : 0);
  g_decode_splits.store(o ? o->decode_splits : 0);
  g_effect_chunk_tiles.store(o ? o->effect_chunk_tiles : 0);
  g_score_stall_unit.store(o ? o->score_stall_unit : -1);
  g_select_stall_unit.store(o ? o->select_stall_unit : -1);
  return KVC_OK;
}

const char* kvc_status_string(kvc_status status) {
  switch (status) {
    case KVC_OK: return "ok";
    case KVC_ERR_INVALID_ARG: return "invalid argument";
    case KVC_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVC_ERR_WORKSPACE: return "workspace missing or too small";
    case KVC_ERR_CUDA: return "CUDA error";
    case KVC_ERR_NO_DEVICE: return "no usable sm_103 device";
  }
  return "unknown status";
}

size_t kvc_score_workspace_bytes(const kvc_shape* shape, int32_t window) {
  ScorePlan p;
  if (plan_score(shape, window, &p) != KVC_OK) return 0;
  return p.ws_total;
}

kvc_status kvc_score(const kvc_shape* shape, const void* k_cache, const void* q_window,
                     int32_t window, float softmax_scale, const float* row_lse,
                     const float* bonus, int32_t page_size,
                     uint32_t flags, float* scores, float* page_scores, int32_t* unit_status,
                     void* workspace, size_t workspace_bytes, kvc_stream stream) {
  ScorePlan p;
  kvc_status st = plan_score(shape, window, &p);
  if (st != KVC_OK) return st;
  if (!k_cache || !q_window || !scores) return KVC_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(q_window, 16)) return KVC_ERR_INVALID_ARG;
  if (flags & ~static_cast<uint32_t>(KVC_SCORE_ACCUMULATE)) return KVC_ERR_INVALID_ARG;
  if (page_size < 1 || page_size > 32 || (page_size & (page_size - 1))) return KVC_ERR_INVALID_ARG;
  if (page_size > 1 && (shape->n_tokens % page_size != 0 || !page_scores)) return KVC_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < p.ws_total || !aligned(workspace, 256)) return KVC_ERR_WORKSPACE;
  if (!(softmax_scale > 0.f)) softmax_scale = 1.0f / sqrtf(static_cast<float>(shape->head_dim));

  ScoreArgs a = {};
  a.U = static_cast<int32_t>(n_units(shape));
  a.L = shape->n_layers;
  a.Hkv = shape->n_kv_heads;
  a.B = shape->batch;
  a.T = shape->n_tokens;
  a.d = shape->head_dim;
  a.W = window;
  a.G = shape->n_q_heads / shape->n_kv_heads;
  a.R = p.R;
  a.Rp = (p.R + 15) / 16 * 16;
  a.n_tiles = p.n_tiles;
  a.chunk_tiles = p.chunk_tiles;
  a.items_per_unit = p.S;
  a.n_items = a.U * p.S;
  a.page_size = page_size;
  a.accumulate = (flags & KVC_SCORE_ACCUMULATE) ? 1 : 0;
  a.n_stages = p.n_stages;
  a.q_rows = p.q_rows;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.row_lse = row_lse;
  a.stall_unit = g_score_stall_unit.load(std::memory_order_relaxed);   // failure test hook (-1: none)
  a.bonus = bonus;
  a.scores = scores;
  a.page_scores = page_size > 1 ? page_scores : nullptr;
  a.unit_status = unit_status;
  a.counters = static_cast<uint32_t*>(workspace);
  a.stats = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + p.ws_counters);

  if (p.small) {
    a.k_small = static_cast<const __nv_bfloat16*>(k_cache);
    a.q_small = static_cast<const __nv_bfloat16*>(q_window);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (launch_score_small(a, p.small_splits, reinterpret_cast<float*>(ws),
                           reinterpret_cast<float2*>(ws + p.ws_logits),
                           reinterpret_cast<float*>(ws + p.ws_logits + p.ws_split),
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return KVC_ERR_CUDA;
    return KVC_OK;
  }
  CUtensorMap mk, mq;
  if ((st = encode_3d(&mk, k_cache, shape->head_dim, shape->n_tokens, a.U, 64, kTileTokens)) != KVC_OK)
    return st;
  if ((st = encode_3d(&mq, q_window, shape->head_dim, p.R, a.U, 64, p.R)) != KVC_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(a.counters, 0, p.ws_counters, s) != cudaSuccess) return KVC_ERR_CUDA;
  if (launch_score(a, mk, mq, p.grid, p.smem, s) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

kvc_status kvc_foresight_bonus(int32_t batch, int64_t n_tokens, const int32_t* span_seq,
                               const int64_t* span_a, const int64_t* span_b,
                               const int32_t* span_next, int32_t n_spans, int32_t step,
                               float sigma, float lambda, float* bonus, kvc_stream stream) {
  if (batch < 1 || n_tokens < 1 || n_spans < 0 || !bonus) return KVC_ERR_INVALID_ARG;
  if (n_spans > 0 && (!span_seq || !span_a || !span_b || !span_next)) return KVC_ERR_INVALID_ARG;
  if (!(sigma > 0.f) || !(lambda >= 0.f) || !aligned(bonus, 4)) return KVC_ERR_INVALID_ARG;
  DevInfo info;
  kvc_status st;
  if ((st = check_device(&info)) != KVC_OK) return st;
  BonusArgs a = {};
  a.batch = batch;
  a.T = n_tokens;
  a.n_spans = n_spans;
  a.step = step;
  a.sigma = sigma;
  a.lambda = lambda;
  a.span_seq = span_seq;
  a.span_a = span_a;
  a.span_b = span_b;
  a.span_next = span_next;
  a.bonus = bonus;
  if (launch_bonus(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

kvc_status kvc_pool_scores(int64_t n_rows, int64_t n_tokens, const float* scores, float* pooled,
                           int32_t kernel, int32_t mode, kvc_stream stream) {
  if (n_rows < 1 || n_rows > 65535 || n_tokens < 1 || !scores || !pooled || scores == pooled)
    return KVC_ERR_INVALID_ARG;
  if (!(kernel == 1 || kernel == 3 || kernel == 5 || kernel == 7)) return KVC_ERR_INVALID_ARG;
  if (mode != KVC_SCORE_POOL_AVG && mode != KVC_SCORE_POOL_MAX) return KVC_ERR_INVALID_ARG;
  DevInfo info;
  kvc_status st;
  if ((st = check_device(&info)) != KVC_OK) return st;
  if (launch_pool(scores, pooled, n_rows, n_tokens, kernel, mode, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return KVC_ERR_CUDA;
  return KVC_OK;
}

kvc_status kvc_shared_scores(const kvc_shape* shape, const float* scores, float* shared,
                             kvc_stream stream) {
  kvc_status st = check_shape(shape);
  if (st != KVC_OK) return st;
  if (!scores || !shared) return KVC_ERR_INVALID_ARG;
  DevInfo info;
  if ((st = check_device(&info)) != KVC_OK) return st;
  if (launch_shared_sum(scores, shared, shape->batch, shape->n_layers * shape->n_kv_heads,
                        shape->n_tokens, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVC_ERR_CUDA;
  return KVC_OK;
}

kvc_status kvc_broadcast_kept(const kvc_shape* shape, const kvc_policy* policy,
                              const int32_t* kept_idx_seq, const int32_t* kept_count_seq,
                              int32_t* kept_idx, int32_t* kept_count, kvc_stream stream) {
  kvc_status st = check_shape(shape);
  if (st != KVC_OK) return st;
  if (!policy || policy->capacity < 1 || !kept_idx_seq || !kept_count_seq || !kept_idx || !kept_count)
    return KVC_ERR_INVALID_ARG;
  if (static_cast<int64_t>(KVC_N_POOLS) * n_units(shape) > 65535) return KVC_ERR_UNSUPPORTED;
  DevInfo info;
  if ((st = check_device(&info)) != KVC_OK) return st;
  if (launch_broadcast(kept_idx_seq, kept_count_seq, kept_idx, kept_count, shape->batch,
                       shape->n_layers * shape->n_kv_heads, policy->capacity,
                       static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVC_ERR_CUDA;
  return KVC_OK;
}

size_t kvc_select_workspace_bytes(const kvc_shape* shape, const kvc_policy* policy) {
  SelectPlan sp;
  if (plan_select(shape, policy, &sp) != KVC_OK) return 0;
  if (sp.byte_mode || sp.n_items <= 32768) return 0;
  return select_long_ws_bytes(n_units(shape), sp.n_items);
}

kvc_status kvc_select(const kvc_shape* shape, const kvc_policy* policy, const float* scores,
                      int32_t* kept_idx, int32_t* kept_count, int32_t* unit_status,
                      int64_t* floor_excess, void* workspace, size_t workspace_bytes,
                      kvc_stream stream) {
  SelectPlan sp;
  kvc_status st = plan_select(shape, policy, &sp);
  if (st != KVC_OK) return st;
  if (!scores || !kept_idx || !kept_count || !unit_status) return KVC_ERR_INVALID_ARG;
  DevInfo info;
  if ((st = check_device(&info)) != KVC_OK) return st;
  SelectArgs a = {};
  a.U = static_cast<int32_t>(n_units(shape));
  a.L = shape->n_layers;
  a.Hkv = shape->n_kv_heads;
  a.B = shape->batch;
  a.T = shape->n_tokens;
  a.d = shape->head_dim;
  a.n_items = sp.n_items;
  a.page_size = sp.P;
  a.budget_items = sp.budget_items;
  a.budget_bytes = policy->budget_bytes;
  a.sink_items = sp.sink_items;
  a.recent_items = sp.recent_items;
  a.capacity = policy->capacity;
  a.byte_mode = sp.byte_mode ? 1 : 0;
  a.quant_mode = policy->quant_mode;
  a.n_tags = policy->n_tags;
  a.n_groups = policy->n_layer_groups;
  a.flags = policy->flags;
  a.tags = policy->tags;
  a.table = policy->action_table;
  a.scores = scores;
  a.kept_idx = kept_idx;
  a.kept_count = kept_count;
  a.unit_status = unit_status;
  a.floor_excess = floor_excess;
  a.stall_unit = g_select_stall_unit.load(std::memory_order_relaxed);   // failure test hook (-1: none)
  // token / page mode with long units: the multi-CTA selection when the
  // caller gave its workspace (else the one-CTA-per-unit kernel, same result)
  const size_t long_bytes = kvc_select_workspace_bytes(shape, policy);
  if (long_bytes > 0 && workspace && workspace_bytes >= long_bytes) {
    if (!aligned(workspace, 256)) return KVC_ERR_WORKSPACE;
    a.long_ws = workspace;
    if (launch_select_long(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
  }
  const size_t cache_bytes = static_cast<size_t>(sp.n_items) * 5;
  a.cache_items = cache_bytes <= 190 * 1024 ? 1 : 0;   // + 34 KB static shared memory
  const size_t smem = a.cache_items ? (cache_bytes + 15) / 16 * 16 : 0;
  if (launch_select(a, static_cast<cudaStream_t>(stream), smem) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

kvc_status kvc_compact_rerotate_quant(const kvc_shape* shape, const kvc_policy* policy,
                                      const void* k_cache, const void* v_cache,
                                      const int32_t* pos_in, const int32_t* kept_idx,
                                      const int32_t* kept_count, const float* rope_cos,
                                      const float* rope_sin, int64_t rope_max_pos,
                                      const kvc_pools* pools, int32_t* unit_status,
                                      kvc_stream stream) {
  return kvc_compact_rerotate_quant_ref(shape, policy, k_cache, v_cache, pos_in, kept_idx,
                                        kept_count, rope_cos, rope_sin, rope_max_pos, nullptr,
                                        pools, unit_status, stream);
}

kvc_status kvc_compact_rerotate_quant_ref(const kvc_shape* shape, const kvc_policy* policy,
                                          const void* k_cache, const void* v_cache,
                                          const int32_t* pos_in, const int32_t* kept_idx,
                                          const int32_t* kept_count, const float* rope_cos,
                                          const float* rope_sin, int64_t rope_max_pos,
                                          const kvc_ref_store* ref, const kvc_pools* pools,
                                          int32_t* unit_status, kvc_stream stream) {
  SelectPlan sp;
  kvc_status st = plan_select(shape, policy, &sp);
  if (st != KVC_OK) return st;
  if (!k_cache || !v_cache || !pos_in || !kept_idx || !kept_count || !pools || !pools->pos_out)
    return KVC_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return KVC_ERR_INVALID_ARG;
  if (policy->renumber) {
    if (!rope_cos || !rope_sin || rope_max_pos < 1) return KVC_ERR_INVALID_ARG;
    if (!aligned(rope_cos, 16) || !aligned(rope_sin, 16)) return KVC_ERR_INVALID_ARG;
    if (rope_max_pos < policy->capacity) return KVC_ERR_INVALID_ARG;
  }
  if (!pools->k_bf16 || !pools->v_bf16 || !aligned(pools->k_bf16, 16) || !aligned(pools->v_bf16, 16))
    return KVC_ERR_INVALID_ARG;
  if (sp.byte_mode) {
    const void* need[8] = {pools->k_i8, pools->v_i8, pools->k_i8_scale, pools->v_i8_scale,
                           pools->k_i4, pools->v_i4, pools->k_i4_scale, pools->v_i4_scale};
    for (const void* q : need)
      if (!q) return KVC_ERR_INVALID_ARG;
    if (!aligned(pools->k_i8, 8) || !aligned(pools->v_i8, 8) || !aligned(pools->k_i4, 4) ||
        !aligned(pools->v_i4, 4))
      return KVC_ERR_INVALID_ARG;
  }
  if (ref) {
    if (!ref->ref_k || !ref->ref_pos || !ref->ref_k_out || !ref->ref_pos_out) return KVC_ERR_INVALID_ARG;
    if (!aligned(ref->ref_k, 16) || !aligned(ref->ref_k_out, 16)) return KVC_ERR_INVALID_ARG;
    if (!rope_cos || !rope_sin || rope_max_pos < 1 || !aligned(rope_cos, 16) || !aligned(rope_sin, 16))
      return KVC_ERR_INVALID_ARG;
  }
  if (policy->rope_layout != KVC_ROPE_SPLIT_HALF && policy->rope_layout != KVC_ROPE_INTERLEAVED)
    return KVC_ERR_INVALID_ARG;
  const int32_t rd = policy->rotary_dim ? policy->rotary_dim : shape->head_dim;
  if (rd < 16 || rd > shape->head_dim || rd % 16 != 0) return KVC_ERR_INVALID_ARG;
  DevInfo info;
  if ((st = check_device(&info)) != KVC_OK) return st;
  // the caches and positions may sit in page-locked host memory: only the
  // kept rows are read, in place, through the mapping
  if ((st = device_view(&k_cache)) != KVC_OK || (st = device_view(&v_cache)) != KVC_OK) return st;
  {
    const void* p = pos_in;
    if ((st = device_view(&p)) != KVC_OK) return st;
    pos_in = static_cast<const int32_t*>(p);
  }
  CompactArgs a = {};
  if (ref) a.ref = *ref;
  a.rope_layout = policy->rope_layout;
  a.rotary_dim = rd;
  a.U = static_cast<int32_t>(n_units(shape));
  a.d = shape->head_dim;
  a.T = shape->n_tokens;
  a.capacity = policy->capacity;
  a.renumber = policy->renumber;
  a.quant_mode = policy->quant_mode;
  a.rope_max_pos = rope_max_pos;
  a.k = static_cast<const __nv_bfloat16*>(k_cache);
  a.v = static_cast<const __nv_bfloat16*>(v_cache);
  a.pos_in = pos_in;
  a.kept_idx = kept_idx;
  a.kept_count = kept_count;
  a.cos = rope_cos;
  a.sin = rope_sin;
  a.pools = *pools;
  a.unit_status = unit_status;
  a.pool_lo = sp.byte_mode ? KVC_POOL_INT4 : KVC_POOL_BF16;
  a.pool_hi = KVC_N_POOLS;
  if (launch_compact(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

size_t kvc_decode_workspace_bytes(const kvc_shape* shape, const kvc_policy* policy) {
  SelectPlan sp;
  if (plan_select(shape, policy, &sp) != KVC_OK) return 0;
  DevInfo info;
  if (check_device(&info) != KVC_OK) return 0;
  const int splits = decode_splits(shape, policy, info.sms);
  if (splits == 1) return 0;
  const int G = shape->n_q_heads / shape->n_kv_heads;
  const size_t slots = static_cast<size_t>(n_units(shape)) * splits * G;
  const size_t ml = (slots * 2 * sizeof(float) + 255) / 256 * 256;
  return ml + slots * shape->head_dim * sizeof(float);
}

kvc_status kvc_decode_attn(const kvc_shape* shape, const kvc_policy* policy, const void* q,
                           const kvc_pools* pools, const int32_t* kept_count, float softmax_scale,
                           void* out, void* workspace, size_t workspace_bytes, kvc_stream stream) {
  SelectPlan sp;
  kvc_status st = plan_select(shape, policy, &sp);
  if (st != KVC_OK) return st;
  if (!q || !pools || !kept_count || !out) return KVC_ERR_INVALID_ARG;
  const int G = shape->n_q_heads / shape->n_kv_heads;
  if (G > 8) return KVC_ERR_UNSUPPORTED;
  if (!pools->k_bf16 || !pools->v_bf16) return KVC_ERR_INVALID_ARG;
  if (sp.byte_mode && (!pools->k_i8 || !pools->v_i8 || !pools->k_i4 || !pools->v_i4 ||
                       !pools->k_i8_scale || !pools->v_i8_scale || !pools->k_i4_scale ||
                       !pools->v_i4_scale))
    return KVC_ERR_INVALID_ARG;
  DevInfo info;
  if ((st = check_device(&info)) != KVC_OK) return st;
  const int splits = decode_splits(shape, policy, info.sms);
  const size_t need = kvc_decode_workspace_bytes(shape, policy);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
    return KVC_ERR_WORKSPACE;
  if (!(softmax_scale > 0.f)) softmax_scale = 1.0f / sqrtf(static_cast<float>(shape->head_dim));
  DecodeArgs a = {};
  a.U = static_cast<int32_t>(n_units(shape));
  a.G = G;
  a.d = shape->head_dim;
  a.Hkv = shape->n_kv_heads;
  a.L = shape->n_layers;
  a.B = shape->batch;
  a.capacity = policy->capacity;
  a.quant_mode = policy->quant_mode;
  a.splits = splits;
  a.scale = softmax_scale;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.pools = *pools;
  a.kept_count = kept_count;
  a.out = static_cast<__nv_bfloat16*>(out);
  if (splits > 1) {
    const size_t slots = static_cast<size_t>(a.U) * splits * G;
    const size_t ml = (slots * 2 * sizeof(float) + 255) / 256 * 256;
    a.ws_ml = static_cast<float*>(workspace);
    a.ws_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ml);
  }
  a.pool_lo = sp.byte_mode ? KVC_POOL_INT4 : KVC_POOL_BF16;
  a.pool_hi = KVC_N_POOLS;
  if (launch_decode(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

size_t kvc_engine_attn_workspace_bytes(const kvc_shape* shape, const kvc_policy* policy, int32_t n_q,
                                       const kvc_bf16_rows* recent, const kvc_bf16_rows* current) {
  EnginePlan p;
  if (plan_engine(shape, policy, n_q, policy != nullptr, recent, current, &p) != KVC_OK) return 0;
  return p.ws;
}

kvc_status kvc_engine_attn(const kvc_shape* shape, const kvc_policy* policy, const void* q,
                           int32_t n_q, const int32_t* q_pos, const kvc_pools* pools,
                           const int32_t* kept_count, const kvc_bf16_rows* recent,
                           const kvc_bf16_rows* current, float softmax_scale, void* out,
                           void* workspace, size_t workspace_bytes, kvc_stream stream) {
  const bool with_pools = pools != nullptr;
  if (with_pools && !policy) return KVC_ERR_INVALID_ARG;
  EnginePlan p;
  kvc_status st = plan_engine(shape, policy, n_q, with_pools, recent, current, &p);
  if (st != KVC_OK) return st;
  if (!q || !out) return KVC_ERR_INVALID_ARG;
  if (with_pools) {
    if (!kept_count || !pools->k_bf16 || !pools->v_bf16) return KVC_ERR_INVALID_ARG;
    if (p.byte_mode && (!pools->k_i8 || !pools->v_i8 || !pools->k_i4 || !pools->v_i4 ||
                        !pools->k_i8_scale || !pools->v_i8_scale || !pools->k_i4_scale ||
                        !pools->v_i4_scale))
      return KVC_ERR_INVALID_ARG;
    if (q_pos && !pools->pos_out) return KVC_ERR_INVALID_ARG;   // positions decide visibility
    if (!aligned(pools->k_bf16, 16) || !aligned(pools->v_bf16, 16)) return KVC_ERR_INVALID_ARG;
  }
  for (const kvc_bf16_rows* r : {recent, current})
    if (r && r->count && (!aligned(r->k, 16) || !aligned(r->v, 16))) return KVC_ERR_INVALID_ARG;
  if (p.ws > 0 && (!workspace || workspace_bytes < p.ws || !aligned(workspace, 256))) return KVC_ERR_WORKSPACE;
  if (!(softmax_scale > 0.f)) softmax_scale = 1.0f / sqrtf(static_cast<float>(shape->head_dim));
  DecodeArgs a = {};
  a.U = static_cast<int32_t>(n_units(shape));
  a.G = p.rows;
  a.d = shape->head_dim;
  a.Hkv = shape->n_kv_heads;
  a.L = shape->n_layers;
  a.B = shape->batch;
  a.capacity = with_pools ? policy->capacity : 0;
  a.quant_mode = with_pools ? policy->quant_mode : 0;
  a.splits = p.splits;
  a.scale = softmax_scale;
  a.q = static_cast<const __nv_bfloat16*>(q);
  if (with_pools) a.pools = *pools;
  a.kept_count = kept_count;
  a.out = static_cast<__nv_bfloat16*>(out);
  if (p.splits > 1) {
    const size_t slots = static_cast<size_t>(a.U) * p.splits * p.rows;
    a.ws_ml = static_cast<float*>(workspace);
    a.ws_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        (slots * 2 * sizeof(float) + 255) / 256 * 256);
  }
  a.pool_lo = p.byte_mode ? KVC_POOL_INT4 : KVC_POOL_BF16;
  a.pool_hi = KVC_N_POOLS;
  a.n_q = n_q;
  a.q_pos = q_pos;
  a.pool_pos = with_pools ? pools->pos_out : nullptr;
  a.has_pools = with_pools;
  if (recent && recent->count) {
    a.rec_k = static_cast<const __nv_bfloat16*>(recent->k);
    a.rec_v = static_cast<const __nv_bfloat16*>(recent->v);
    a.rec_pos = recent->pos;
    a.rec_count = recent->count;
    a.rec_cap = recent->capacity;
  }
  if (current && current->count) {
    a.cur_k = static_cast<const __nv_bfloat16*>(current->k);
    a.cur_v = static_cast<const __nv_bfloat16*>(current->v);
    a.cur_pos = current->pos;
    a.cur_count = current->count;
    a.cur_cap = current->capacity;
  }
  if (launch_engine(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

size_t kvc_deletion_effect_workspace_bytes(const kvc_shape* shape, int32_t window) {
  EffectPlan p;
  if (plan_effect(shape, window, &p) != KVC_OK) return 0;
  return p.ws_total;
}

kvc_status kvc_deletion_effect(const kvc_shape* shape, const void* k_cache, const void* v_cache,
                               const void* q_window, int32_t window, float softmax_scale,
                               const int32_t* page_start, const int32_t* page_len,
                               int32_t n_pages, float* effect, const kvc_effect_record* record,
                               int32_t* unit_status, void* workspace, size_t workspace_bytes,
                               kvc_stream stream) {
  EffectPlan p;
  kvc_status st = plan_effect(shape, window, &p);
  if (st != KVC_OK) return st;
  if (!k_cache || !v_cache || !q_window || !record || !record->o || !record->lse) return KVC_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q_window, 16)) return KVC_ERR_INVALID_ARG;
  if (n_pages < 0) return KVC_ERR_INVALID_ARG;
  if (n_pages > 0 && (!page_start || !page_len || !effect || !record->s || !record->u))
    return KVC_ERR_INVALID_ARG;
  if (!aligned(record->o, 16) || (n_pages > 0 && !aligned(record->u, 16))) return KVC_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < p.ws_total || !aligned(workspace, 256)) return KVC_ERR_WORKSPACE;
  if (!(softmax_scale > 0.f)) softmax_scale = 1.0f / sqrtf(static_cast<float>(shape->head_dim));

  EffectArgs a = {};
  a.U = static_cast<int32_t>(n_units(shape));
  a.L = shape->n_layers;
  a.Hkv = shape->n_kv_heads;
  a.B = shape->batch;
  a.G = shape->n_q_heads / shape->n_kv_heads;
  a.W = window;
  a.R = p.R;
  a.Rp = p.Rp;
  a.T = shape->n_tokens;
  a.n_tiles = p.n_tiles;
  a.chunk_tiles = p.chunk;
  a.splits = p.splits;
  a.n_items = p.n_items;
  a.nk = p.nk;
  a.nv = p.nv;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.part_u = static_cast<float*>(workspace);
  a.part_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + p.ws_part_u);
  a.o = record->o;
  a.lse = record->lse;
  a.s = record->s;
  a.u = record->u;
  a.page_start = page_start;
  a.page_len = page_len;
  a.n_pages = n_pages;
  a.k = static_cast<const __nv_bfloat16*>(k_cache);
  a.v = static_cast<const __nv_bfloat16*>(v_cache);
  a.q = static_cast<const __nv_bfloat16*>(q_window);
  a.effect = effect;
  a.unit_status = unit_status;

  CUtensorMap mk, mv, mq;
  if ((st = encode_3d(&mk, k_cache, 128, shape->n_tokens, a.U, 64, kTileTokens)) != KVC_OK) return st;
  if ((st = encode_3d(&mv, v_cache, 128, shape->n_tokens, a.U, 64, kTileTokens)) != KVC_OK) return st;
  if ((st = encode_3d(&mq, q_window, 128, p.R, a.U, 64, p.R)) != KVC_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (n_pages > 0 &&
      cudaMemsetAsync(effect, 0, static_cast<size_t>(shape->batch) * shape->n_layers * n_pages * 4, cs) !=
          cudaSuccess)
    return KVC_ERR_CUDA;
  if (launch_effect(a, mk, mv, mq, p.grid, p.smem, cs) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

size_t kvc_commit_workspace_bytes(const kvc_shape* shape, int32_t window) {
  if (check_shape(shape) != KVC_OK || window < 1) return 0;
  return (static_cast<size_t>(shape->batch) * shape->n_q_heads * window * 128 * 4 + 255) / 256 * 256;
}

kvc_status kvc_commit_transition(const kvc_shape* shape, int32_t window, int32_t layer,
                                 int32_t n_pages, const float* effect_minus,
                                 const float* effect_plus, const uint8_t* compared,
                                 const kvc_commit_thresholds* thresholds,
                                 const kvc_effect_record* record_plus, uint8_t* state,
                                 uint8_t* retire, float* joint, void* workspace,
                                 size_t workspace_bytes, kvc_stream stream) {
  kvc_status st = check_shape(shape);
  if (st != KVC_OK) return st;
  if (shape->head_dim != 128) return KVC_ERR_UNSUPPORTED;
  if (window < 1 || layer < 0 || layer >= shape->n_layers) return KVC_ERR_INVALID_ARG;
  if (n_pages < 1 || n_pages > 1024) return KVC_ERR_INVALID_ARG;
  if (static_cast<int64_t>(shape->n_q_heads) * window > 4096) return KVC_ERR_UNSUPPORTED;
  if (!effect_minus || !effect_plus || !compared || !thresholds || !record_plus || !record_plus->o ||
      !record_plus->s || !record_plus->u || !state || !retire)
    return KVC_ERR_INVALID_ARG;
  if (!aligned(record_plus->o, 16) || !aligned(record_plus->u, 16)) return KVC_ERR_INVALID_ARG;
  const size_t need = kvc_commit_workspace_bytes(shape, window);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return KVC_ERR_WORKSPACE;
  DevInfo info;
  if ((st = check_device(&info)) != KVC_OK) return st;
  CommitArgs a = {};
  a.B = shape->batch;
  a.L = shape->n_layers;
  a.Hq = shape->n_q_heads;
  a.W = window;
  a.n_pages = n_pages;
  a.layer = layer;
  a.tau_use = thresholds->tau_use;
  a.tau_dead = thresholds->tau_dead;
  a.rho_use = thresholds->rho_use;
  a.rho_dead = thresholds->rho_dead;
  a.tau_joint = thresholds->tau_joint;
  a.r_minus = effect_minus;
  a.r_plus = effect_plus;
  a.compared = compared;
  a.o = record_plus->o;
  a.s = record_plus->s;
  a.u = record_plus->u;
  a.acc = static_cast<float*>(workspace);
  a.state = state;
  a.retire = retire;
  a.joint = joint;
  if (launch_commit(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

kvc_status kvc_protect_pending(const kvc_shape* shape, int32_t layer, int32_t n_pages,
                               const float* effect_minus, const uint8_t* pending,
                               const int32_t* page_len, int32_t budget_tokens, int32_t max_pages,
                               uint8_t* protect, kvc_stream stream) {
  kvc_status st = check_shape(shape);
  if (st != KVC_OK) return st;
  if (layer < 0 || layer >= shape->n_layers || n_pages < 1 || n_pages > 1024) return KVC_ERR_INVALID_ARG;
  if (budget_tokens < 0 || max_pages < 0) return KVC_ERR_INVALID_ARG;
  if (!effect_minus || !pending || !page_len || !protect) return KVC_ERR_INVALID_ARG;
  DevInfo info;
  if ((st = check_device(&info)) != KVC_OK) return st;
  ProtectArgs a = {};
  a.B = shape->batch;
  a.L = shape->n_layers;
  a.n_pages = n_pages;
  a.layer = layer;
  a.budget_tokens = budget_tokens;
  a.max_pages = max_pages;
  a.r_minus = effect_minus;
  a.pending = pending;
  a.page_len = page_len;
  a.protect = protect;
  if (launch_protect(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

kvc_status kvc_commit_flags(int32_t batch, int64_t n_tokens, int32_t n_pages,
                            const int32_t* page_start, const int32_t* page_len,
                            const uint8_t* retire, const uint8_t* protect, uint8_t* flags,
                            kvc_stream stream) {
  if (batch < 1 || batch > 65535 || n_tokens < 1 || n_pages < 0 || n_pages > (1 << 30)) return KVC_ERR_INVALID_ARG;
  if (n_pages > 0 && (!page_start || !page_len || !flags)) return KVC_ERR_INVALID_ARG;
  DevInfo info;
  kvc_status st;
  if ((st = check_device(&info)) != KVC_OK) return st;
  FlagArgs a = {};
  a.B = batch;
  a.n_pages = n_pages;
  a.T = n_tokens;
  a.page_start = page_start;
  a.page_len = page_len;
  a.retire = retire;
  a.protect = protect;
  a.flags = flags;
  if (launch_flags(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Decode step that allocates nothing.
//
// Some callers cannot hand the library a workspace: an engine whose caching
// allocator has already reserved nearly all of HBM for its KV pools (a raw
// cudaMalloc would fail or fragment that reservation), a plug-in that only
// receives the buffers its host framework gives it and has no allocator of
// its own, or a latency-critical loop where cudaMalloc's implicit device
// synchronisation is not acceptable.  For them kvc_decode_attn_noalloc keeps
// the split-partition scratch of the decode step in the file-scope array
// below, which every device that loads this library holds until the process
// exits.
// ----------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;    // 2 MiB per device
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress (with that device current) and cached per device,
// together with the context it belongs to: after cudaDeviceReset the device
// gets a new context and module, and the address is looked up again.
kvc_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVC_ERR_NO_DEVICE;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (!get_ctx) return KVC_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return KVC_ERR_CUDA;     // NULL before the first runtime call
  static void* addr[64] = {};
  static CUcontext owner[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || !ctx || owner[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVC_ERR_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return KVC_ERR_CUDA;
    addr[dev] = p;
    owner[dev] = ctx;
  }
  *out = addr[dev];
  return KVC_OK;
}

}  // namespace

extern "C" kvc_status kvc_decode_attn_noalloc(const kvc_shape* shape, const kvc_policy* policy,
                                              const void* q, const kvc_pools* pools,
                                              const int32_t* kept_count, float softmax_scale,
                                              void* out, kvc_stream stream) {
  const size_t need = kvc_decode_workspace_bytes(shape, policy);
  if (need > kNoAllocScratchBytes) return KVC_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    kvc_status st = noalloc_scratch(&ws);
    if (st != KVC_OK) return st;
  }
  return kvc_decode_attn(shape, policy, q, pools, kept_count, softmax_scale, out, ws, need, stream);
}
