"""Python binding of libkvc (budgeted KV-cache compaction on GB300).

Argument marshalling only: every function here forwards to the C-ABI entry
point of the same name in libkvc.so (declared in include/kvc.h), passing
device pointers of torch tensors and the current CUDA stream.  There is no
fallback: if the library is missing or a call fails, a KvcError is raised.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")

KVC_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
                3: "workspace missing or too small", 4: "CUDA error", 5: "no usable sm_103 device"}
UNIT_OK, UNIT_OVER_BUDGET, UNIT_BAD_INDEX, UNIT_BAD_FLAGS, UNIT_TIMEOUT = 0, 1, 2, 3, 4
ACT_RELEASE, ACT_INT4, ACT_INT8, ACT_BF16 = 0, 1, 2, 3
POOL_INT4, POOL_INT8, POOL_BF16, N_POOLS = 0, 1, 2, 3
FLAG_PROTECT, FLAG_EXCLUDE = 1, 2
QUANT_G32_BF16, QUANT_ROW_FP16 = 0, 1
SCORE_ACCUMULATE = 1


class KvcError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)} ({code})")
        self.code = code


class kvc_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_tokens", ctypes.c_int64)]


class kvc_policy(ctypes.Structure):
    _fields_ = [("budget_tokens", ctypes.c_int32), ("budget_bytes", ctypes.c_int64),
                ("n_sink", ctypes.c_int32), ("n_recent", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("renumber", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("quant_mode", ctypes.c_int32),
                ("n_tags", ctypes.c_int32), ("n_layer_groups", ctypes.c_int32),
                ("flags", ctypes.c_void_p), ("tags", ctypes.c_void_p),
                ("action_table", ctypes.c_void_p), ("rope_layout", ctypes.c_int32),
                ("rotary_dim", ctypes.c_int32)]


class kvc_pools(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "k_bf16", "v_bf16", "k_i8", "v_i8", "k_i8_scale", "v_i8_scale",
        "k_i4", "v_i4", "k_i4_scale", "v_i4_scale", "pos_out", "orig_pos_out")]


_LIB = None


class kvc_ref_store(ctypes.Structure):
    """Reference store of kvc_compact_rerotate_quant_ref (device pointers)."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("ref_k", "ref_pos", "ref_k_out", "ref_pos_out", "failures")]


class kvc_bf16_rows(ctypes.Structure):
    """A bf16 row store of kvc_engine_attn (device pointers)."""
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("count", ctypes.c_void_p), ("capacity", ctypes.c_int32)]


class kvc_effect_record(ctypes.Structure):
    """Window record of kvc_deletion_effect (device pointers: o, lse, s, u)."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("o", "lse", "s", "u")]


class kvc_overrides(ctypes.Structure):
    """Launch-plan overrides of kvc_set_overrides (tuning and failure tests)."""
    _fields_ = [(n, ctypes.c_int32) for n in ("score_chunk_tiles", "decode_splits",
                                              "effect_chunk_tiles", "score_stall_unit",
                                              "select_stall_unit")]


class kvc_commit_thresholds(ctypes.Structure):
    """CommitKV Sec. 4.1 thresholds."""
    _fields_ = [(n, ctypes.c_float) for n in ("tau_use", "tau_dead", "rho_use", "rho_dead", "tau_joint")]


def _load():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise KvcError("load libkvc.so (not built: run budgeted_kv_cache_gb300.build.build())", -1)
        lib = ctypes.CDLL(LIB_PATH)
        P, I32, I64, U32, F32, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                     ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t)
        SH, PO, PL = ctypes.POINTER(kvc_shape), ctypes.POINTER(kvc_policy), ctypes.POINTER(kvc_pools)
        RS = ctypes.POINTER(kvc_ref_store)
        ER, CT = ctypes.POINTER(kvc_effect_record), ctypes.POINTER(kvc_commit_thresholds)
        BR = ctypes.POINTER(kvc_bf16_rows)
        sig = {
            "kvc_score_workspace_bytes": (SZ, [SH, I32]),
            "kvc_score": (ctypes.c_int, [SH, P, P, I32, F32, P, P, I32, U32, P, P, P, P, SZ, P]),
            "kvc_select_workspace_bytes": (SZ, [SH, PO]),
            "kvc_select": (ctypes.c_int, [SH, PO, P, P, P, P, P, P, SZ, P]),
            "kvc_compact_rerotate_quant": (ctypes.c_int, [SH, PO, P, P, P, P, P, P, P, I64, PL, P, P]),
            "kvc_compact_rerotate_quant_ref": (ctypes.c_int,
                                               [SH, PO, P, P, P, P, P, P, P, I64, RS, PL, P, P]),
            "kvc_decode_workspace_bytes": (SZ, [SH, PO]),
            "kvc_decode_attn": (ctypes.c_int, [SH, PO, P, PL, P, F32, P, P, SZ, P]),
            "kvc_decode_attn_noalloc": (ctypes.c_int, [SH, PO, P, PL, P, F32, P, P]),
            "kvc_foresight_bonus": (ctypes.c_int, [I32, I64, P, P, P, P, I32, I32, F32, F32, P, P]),
            "kvc_pool_scores": (ctypes.c_int, [I64, I64, P, P, I32, I32, P]),
            "kvc_shared_scores": (ctypes.c_int, [SH, P, P, P]),
            "kvc_broadcast_kept": (ctypes.c_int, [SH, PO, P, P, P, P, P]),
            "kvc_engine_attn_workspace_bytes": (SZ, [SH, PO, I32, BR, BR]),
            "kvc_engine_attn": (ctypes.c_int, [SH, PO, P, I32, P, PL, P, BR, BR, F32, P, P, SZ, P]),
            "kvc_deletion_effect_workspace_bytes": (SZ, [SH, I32]),
            "kvc_deletion_effect": (ctypes.c_int, [SH, P, P, P, I32, F32, P, P, I32, P, ER, P, P, SZ, P]),
            "kvc_commit_workspace_bytes": (SZ, [SH, I32]),
            "kvc_commit_transition": (ctypes.c_int, [SH, I32, I32, I32, P, P, P, CT, ER, P, P, P, P, SZ,
                                                     P]),
            "kvc_protect_pending": (ctypes.c_int, [SH, I32, I32, P, P, P, I32, I32, P, P]),
            "kvc_commit_flags": (ctypes.c_int, [I32, I64, I32, P, P, P, P, P, P]),
            "kvc_set_overrides": (ctypes.c_int, [ctypes.POINTER(kvc_overrides)]),
            "kvc_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype, f.argtypes = res, args
        _LIB = lib
    return _LIB


def library() -> ctypes.CDLL:
    """The loaded libkvc.so (raises KvcError if it is not built)."""
    return _load()


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, code: int):
    if code != KVC_OK:
        raise KvcError(fn, code)


# ----------------------------------------------------------------------------- structs

def make_shape(batch, n_layers, n_q_heads, n_kv_heads, head_dim, n_tokens) -> kvc_shape:
    return kvc_shape(batch, n_layers, n_q_heads, n_kv_heads, head_dim, n_tokens)


@dataclasses.dataclass
class Policy:
    budget_tokens: int = 0
    budget_bytes: int = 0
    n_sink: int = 4
    n_recent: int = 32
    page_size: int = 1
    renumber: bool = True
    capacity: int = 0
    quant_mode: int = QUANT_G32_BF16
    n_tags: int = 0
    n_layer_groups: int = 1
    flags: Optional[torch.Tensor] = None
    tags: Optional[torch.Tensor] = None
    action_table: Optional[torch.Tensor] = None
    rope_layout: int = 0          # ROPE_SPLIT_HALF or ROPE_INTERLEAVED
    rotary_dim: int = 0           # 0 = head_dim

    def c(self) -> kvc_policy:
        return kvc_policy(self.budget_tokens, self.budget_bytes, self.n_sink, self.n_recent,
                          self.page_size, int(bool(self.renumber)), self.capacity, self.quant_mode,
                          self.n_tags, self.n_layer_groups, _p(self.flags), _p(self.tags),
                          _p(self.action_table), int(self.rope_layout), int(self.rotary_dim))

    @property
    def byte_mode(self) -> bool:
        return self.budget_bytes > 0


@dataclasses.dataclass
class Pools:
    """Output arrays of kvc_compact_rerotate_quant (torch tensors)."""
    k_bf16: torch.Tensor
    v_bf16: torch.Tensor
    pos_out: torch.Tensor
    orig_pos_out: Optional[torch.Tensor] = None
    k_i8: Optional[torch.Tensor] = None
    v_i8: Optional[torch.Tensor] = None
    k_i8_scale: Optional[torch.Tensor] = None
    v_i8_scale: Optional[torch.Tensor] = None
    k_i4: Optional[torch.Tensor] = None
    v_i4: Optional[torch.Tensor] = None
    k_i4_scale: Optional[torch.Tensor] = None
    v_i4_scale: Optional[torch.Tensor] = None

    def c(self) -> kvc_pools:
        return kvc_pools(*[_p(getattr(self, n)) for n, _ in kvc_pools._fields_])

    @staticmethod
    def allocate(shape: kvc_shape, policy: Policy, device="cuda", orig_pos: bool = True) -> "Pools":
        U = shape.batch * shape.n_layers * shape.n_kv_heads
        cap, d = policy.capacity, shape.head_dim
        e = lambda *s, dt: torch.empty(s, dtype=dt, device=device)
        p = Pools(k_bf16=e(U, cap, d, dt=torch.bfloat16), v_bf16=e(U, cap, d, dt=torch.bfloat16),
                  pos_out=e(N_POOLS, U, cap, dt=torch.int32),
                  orig_pos_out=e(N_POOLS, U, cap, dt=torch.int32) if orig_pos else None)
        if policy.byte_mode:
            ns = d // 32 if policy.quant_mode == QUANT_G32_BF16 else 1
            sdt = torch.bfloat16 if policy.quant_mode == QUANT_G32_BF16 else torch.float16
            p.k_i8, p.v_i8 = e(U, cap, d, dt=torch.int8), e(U, cap, d, dt=torch.int8)
            p.k_i4, p.v_i4 = e(U, cap, d // 2, dt=torch.uint8), e(U, cap, d // 2, dt=torch.uint8)
            p.k_i8_scale, p.v_i8_scale = e(U, cap, ns, dt=sdt), e(U, cap, ns, dt=sdt)
            p.k_i4_scale, p.v_i4_scale = e(U, cap, ns, dt=sdt), e(U, cap, ns, dt=sdt)
        return p


# ----------------------------------------------------------------------------- entry points

def kvc_set_overrides(score_chunk_tiles: int = 0, decode_splits: int = 0,
                      effect_chunk_tiles: int = 0, score_stall_unit: int = -1,
                      select_stall_unit: int = -1, reset: bool = False):
    """Process-wide launch-plan overrides (tuning sweeps, failure tests); reset=True restores defaults."""
    if reset:
        _check("kvc_set_overrides", library().kvc_set_overrides(None))
        return
    o = kvc_overrides(score_chunk_tiles, decode_splits, effect_chunk_tiles, score_stall_unit,
                      select_stall_unit)
    _check("kvc_set_overrides", library().kvc_set_overrides(ctypes.byref(o)))


def kvc_status_string(code: int) -> str:
    return _load().kvc_status_string(code).decode()


def kvc_score_workspace_bytes(shape: kvc_shape, window: int) -> int:
    return _load().kvc_score_workspace_bytes(ctypes.byref(shape), window)


def kvc_score(shape, k_cache, q_window, window, softmax_scale, bonus, page_size, flags, scores,
              page_scores, unit_status, workspace, workspace_bytes=None, stream=None, row_lse=None):
    """row_lse: optional fp32 [B][L][H_q][window] natural-log row statistics (skips pass 1)."""
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check("kvc_score", _load().kvc_score(
        ctypes.byref(shape), _p(k_cache), _p(q_window), window, float(softmax_scale), _p(row_lse),
        _p(bonus), page_size, flags, _p(scores), _p(page_scores), _p(unit_status), _p(workspace),
        wb, _stream(stream)))


def kvc_select_workspace_bytes(shape: kvc_shape, policy: Policy) -> int:
    cp = policy.c()
    return _load().kvc_select_workspace_bytes(ctypes.byref(shape), ctypes.byref(cp))


def kvc_select(shape, policy: Policy, scores, kept_idx, kept_count, unit_status, floor_excess=None,
               workspace=None, workspace_bytes=0, stream=None):
    cp = policy.c()
    _check("kvc_select", _load().kvc_select(
        ctypes.byref(shape), ctypes.byref(cp), _p(scores), _p(kept_idx), _p(kept_count),
        _p(unit_status), _p(floor_excess), _p(workspace), workspace_bytes, _stream(stream)))


def kvc_compact_rerotate_quant(shape, policy: Policy, k_cache, v_cache, pos_in, kept_idx,
                               kept_count, rope_cos, rope_sin, rope_max_pos, pools: Pools,
                               unit_status=None, stream=None):
    cp, cpools = policy.c(), pools.c()
    _check("kvc_compact_rerotate_quant", _load().kvc_compact_rerotate_quant(
        ctypes.byref(shape), ctypes.byref(cp), _p(k_cache), _p(v_cache), _p(pos_in),
        _p(kept_idx), _p(kept_count), _p(rope_cos), _p(rope_sin), int(rope_max_pos),
        ctypes.byref(cpools), _p(unit_status), _stream(stream)))


def kvc_compact_rerotate_quant_ref(shape, policy: Policy, k_cache, v_cache, pos_in, kept_idx,
                                   kept_count, rope_cos, rope_sin, rope_max_pos, ref_k, ref_pos,
                                   ref_k_out, ref_pos_out, pools: Pools, failures=None,
                                   unit_status=None, stream=None):
    """kvc_compact_rerotate_quant through a key reference store (see include/kvc.h)."""
    cp, cpools = policy.c(), pools.c()
    rs = kvc_ref_store(_p(ref_k), _p(ref_pos), _p(ref_k_out), _p(ref_pos_out), _p(failures))
    _check("kvc_compact_rerotate_quant_ref", _load().kvc_compact_rerotate_quant_ref(
        ctypes.byref(shape), ctypes.byref(cp), _p(k_cache), _p(v_cache), _p(pos_in),
        _p(kept_idx), _p(kept_count), _p(rope_cos), _p(rope_sin), int(rope_max_pos),
        ctypes.byref(rs), ctypes.byref(cpools), _p(unit_status), _stream(stream)))


def kvc_foresight_bonus(batch, n_tokens, span_seq, span_a, span_b, span_next, step, sigma, lam,
                        bonus, stream=None):
    """PACE Eq. 2 bonus [batch][n_tokens] from spans (device tensors; see include/kvc.h)."""
    n = 0 if span_seq is None else int(span_seq.numel())
    _check("kvc_foresight_bonus", _load().kvc_foresight_bonus(
        int(batch), int(n_tokens), _p(span_seq), _p(span_a), _p(span_b), _p(span_next), n,
        int(step), float(sigma), float(lam), _p(bonus), _stream(stream)))


SCORE_POOL_AVG, SCORE_POOL_MAX = 0, 1
ROPE_SPLIT_HALF, ROPE_INTERLEAVED = 0, 1


def kvc_pool_scores(scores, pooled, kernel, mode, stream=None):
    """SnapKV pooling of fp32 [rows][T] scores into `pooled` (see include/kvc.h)."""
    _check("kvc_pool_scores", _load().kvc_pool_scores(
        int(scores.shape[0]), int(scores.shape[1]), _p(scores), _p(pooled), int(kernel), int(mode),
        _stream(stream)))


def kvc_shared_scores(shape, scores, shared, stream=None):
    """CommitKV Eq. 4: per-sequence sum of the units' scores, fp32 [B][T]."""
    _check("kvc_shared_scores", _load().kvc_shared_scores(ctypes.byref(shape), _p(scores),
                                                          _p(shared), _stream(stream)))


def kvc_broadcast_kept(shape, policy: Policy, kept_idx_seq, kept_count_seq, kept_idx, kept_count,
                       stream=None):
    """Copy per-sequence kept lists to every unit of the sequence."""
    cp = policy.c()
    _check("kvc_broadcast_kept", _load().kvc_broadcast_kept(
        ctypes.byref(shape), ctypes.byref(cp), _p(kept_idx_seq), _p(kept_count_seq), _p(kept_idx),
        _p(kept_count), _stream(stream)))


def kvc_decode_workspace_bytes(shape, policy: Policy) -> int:
    cp = policy.c()
    return _load().kvc_decode_workspace_bytes(ctypes.byref(shape), ctypes.byref(cp))


def kvc_decode_attn(shape, policy: Policy, q, pools: Pools, kept_count, softmax_scale, out,
                    workspace=None, workspace_bytes=None, stream=None):
    cp, cpools = policy.c(), pools.c()
    wb = 0 if workspace is None else (workspace.numel() * workspace.element_size()
                                      if workspace_bytes is None else workspace_bytes)
    _check("kvc_decode_attn", _load().kvc_decode_attn(
        ctypes.byref(shape), ctypes.byref(cp), _p(q), ctypes.byref(cpools), _p(kept_count),
        float(softmax_scale), _p(out), _p(workspace), wb, _stream(stream)))


def kvc_decode_attn_noalloc(shape, policy: Policy, q, pools: Pools, kept_count, softmax_scale,
                            out, stream=None):
    """kvc_decode_attn with the library's static scratch instead of a workspace."""
    cp, cpools = policy.c(), pools.c()
    _check("kvc_decode_attn_noalloc", _load().kvc_decode_attn_noalloc(
        ctypes.byref(shape), ctypes.byref(cp), _p(q), ctypes.byref(cpools), _p(kept_count),
        float(softmax_scale), _p(out), _stream(stream)))


# ----------------------------------------------------------------------------- CommitKV

STATE_UNCERTAIN, STATE_COMPLETION, STATE_DORMANT, STATE_NEWLY_ACTIVE, STATE_STILL_ACTIVE = 0, 1, 2, 3, 4
STATE_NOT_COMPARED = 255


class EffectRecord:
    """Device buffers of a kvc_deletion_effect record (see include/kvc.h)."""

    def __init__(self, shape: kvc_shape, window: int, n_pages: int, device="cuda"):
        B, L, Hq = shape.batch, shape.n_layers, shape.n_q_heads
        f32 = torch.float32
        self.o = torch.empty((B, L, Hq, window, 128), dtype=f32, device=device)
        self.lse = torch.empty((B, L, Hq, window), dtype=f32, device=device)
        self.s = torch.empty((B, L, max(n_pages, 1), Hq, window), dtype=f32, device=device)
        self.u = torch.empty((B, L, max(n_pages, 1), Hq, window, 128), dtype=f32, device=device)

    def c(self) -> kvc_effect_record:
        return kvc_effect_record(_p(self.o), _p(self.lse), _p(self.s), _p(self.u))


def kvc_deletion_effect_workspace_bytes(shape: kvc_shape, window: int) -> int:
    return _load().kvc_deletion_effect_workspace_bytes(ctypes.byref(shape), window)


def kvc_deletion_effect(shape, k_cache, v_cache, q_window, window, softmax_scale, page_start,
                        page_len, effect, record: EffectRecord, workspace, unit_status=None,
                        stream=None):
    """CommitKV Eqs. 6-7 per page: effect fp32 [B][L][n_pages] (see include/kvc.h)."""
    n = 0 if page_start is None else int(page_start.shape[-1])
    rec = record.c()
    _check("kvc_deletion_effect", _load().kvc_deletion_effect(
        ctypes.byref(shape), _p(k_cache), _p(v_cache), _p(q_window), int(window),
        float(softmax_scale), _p(page_start), _p(page_len), n, _p(effect), ctypes.byref(rec),
        _p(unit_status), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def kvc_commit_workspace_bytes(shape: kvc_shape, window: int) -> int:
    return _load().kvc_commit_workspace_bytes(ctypes.byref(shape), window)


def kvc_commit_transition(shape, window, layer, effect_minus, effect_plus, compared,
                          record_plus: EffectRecord, state, retire, workspace, joint=None,
                          tau_use=0.05, tau_dead=0.01, rho_use=0.75, rho_dead=0.25, tau_joint=0.01,
                          stream=None):
    """CommitKV Eqs. 8-11 on layer `layer`: lifecycle states and the retirement set."""
    th = kvc_commit_thresholds(tau_use, tau_dead, rho_use, rho_dead, tau_joint)
    rec = record_plus.c()
    _check("kvc_commit_transition", _load().kvc_commit_transition(
        ctypes.byref(shape), int(window), int(layer), int(effect_minus.shape[-1]), _p(effect_minus),
        _p(effect_plus), _p(compared), ctypes.byref(th), ctypes.byref(rec), _p(state), _p(retire),
        _p(joint), _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def kvc_protect_pending(shape, layer, effect_minus, pending, page_len, budget_tokens, max_pages,
                        protect, stream=None):
    """CommitKV Eq. 12: pending pages protected within B_N tokens and max_pages pages."""
    _check("kvc_protect_pending", _load().kvc_protect_pending(
        ctypes.byref(shape), int(layer), int(effect_minus.shape[-1]), _p(effect_minus), _p(pending),
        _p(page_len), int(budget_tokens), int(max_pages), _p(protect), _stream(stream)))


def kvc_commit_flags(batch, n_tokens, page_start, page_len, retire, protect, flags, stream=None):
    """Checkpoint flags (Eq. 13) painted over the pages' tokens, in place."""
    n = 0 if page_start is None else int(page_start.shape[-1])
    _check("kvc_commit_flags", _load().kvc_commit_flags(
        int(batch), int(n_tokens), n, _p(page_start), _p(page_len), _p(retire), _p(protect),
        _p(flags), _stream(stream)))


# ----------------------------------------------------------------------------- engine attention

def bf16_rows(k, v, pos, count) -> kvc_bf16_rows:
    """A recent / current row store: k, v bf16 [U][capacity][d], pos int32 [U][capacity] or None,
    count int32 [U]."""
    return kvc_bf16_rows(_p(k), _p(v), _p(pos), _p(count), int(k.shape[-2]))


def kvc_engine_attn_workspace_bytes(shape, policy: Optional[Policy], n_q, recent=None, current=None) -> int:
    cp = policy.c() if policy is not None else None
    return _load().kvc_engine_attn_workspace_bytes(
        ctypes.byref(shape), ctypes.byref(cp) if cp is not None else None, int(n_q),
        ctypes.byref(recent) if recent is not None else None,
        ctypes.byref(current) if current is not None else None)


def kvc_engine_attn(shape, policy: Optional[Policy], q, n_q, q_pos, pools: Optional[Pools], kept_count,
                    recent, current, softmax_scale, out, workspace=None, stream=None):
    """PASK App. B.5 attention over persistent pools, recent and current bf16 rows (see include/kvc.h)."""
    cp = policy.c() if policy is not None else None
    cpools = pools.c() if pools is not None else None
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("kvc_engine_attn", _load().kvc_engine_attn(
        ctypes.byref(shape), ctypes.byref(cp) if cp is not None else None, _p(q), int(n_q), _p(q_pos),
        ctypes.byref(cpools) if cpools is not None else None, _p(kept_count),
        ctypes.byref(recent) if recent is not None else None,
        ctypes.byref(current) if current is not None else None, float(softmax_scale), _p(out),
        _p(workspace), wb, _stream(stream)))
