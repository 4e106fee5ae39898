"""Seeded synthetic inputs for the budgeted KV-cache compaction pass.

This module only draws random numbers and lays them out; it holds none of
the pass's arithmetic (no scoring, selection, rotation or quantisation).
Both the CPU oracle and the CUDA library consume the tensors made here.

Every workload stands in for the models and traces of the three pages
(PASK, PACE, CommitKV), whose weights and datasets are not available: the
shapes follow the pages' models, the values are iid Gaussian.

Stored keys are drawn directly as N(0, 1) vectors and are *treated* as keys
already rotated at their physical positions.  A rotary rotation is
orthogonal, so an isotropic Gaussian pre-rotation key rotated to any
position is again an isotropic Gaussian with the same variance; drawing the
rotated key directly gives the same distribution as drawing the pre-rotation
key and rotating it.  The same holds for the window queries and the decode
query, and for the 3-sigma outlier keys (a scaled isotropic Gaussian).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

# action codes of a (tag, layer-group) table: release, int4, int8, bf16
ACT_RELEASE, ACT_INT4, ACT_INT8, ACT_BF16 = 0, 1, 2, 3
# per-token / per-page flag bits
FLAG_PROTECT, FLAG_EXCLUDE = 1, 2
# quantisation modes
QUANT_G32_BF16, QUANT_ROW_FP16 = 0, 1

BASE_SEED = 20261202


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_tokens: int
    window: int
    rope_theta: float
    seed: int
    budget_tokens: int = 0          # token / page mode budget (rows per unit)
    budget_bytes: int = 0           # byte mode budget per unit (K+V payload)
    n_sink: int = 4
    n_recent: int = 32
    page_size: int = 1
    renumber: bool = True
    quant_mode: int = QUANT_G32_BF16
    n_layer_groups: int = 3
    outlier_frac: float = 0.0       # fraction of tokens whose key is scaled
    outlier_scale: float = 3.0
    bonus_spans: int = 0            # planner foresight spans (same for all units)
    bonus_span_len: int = 64
    bonus_value: float = 10.0
    tag_probs: Optional[tuple] = None   # byte mode: structural tag distribution
    protect_pages: int = 0          # page mode: commit-protected pages
    retire_pages: int = 0           # page mode: retired (excluded) pages
    first_pos: int = 0              # physical position of token 0
    decode_pos: int = 0             # physical position of the decode query
    chunk: int = 0                  # session: rows appended per cycle (n_tokens = budget + chunk)
    cycles: int = 0                 # session: compaction cycles
    limit: int = 0                  # session: position limit L

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def n_units(self) -> int:
        return self.batch * self.n_layers * self.n_kv_heads

    @property
    def rows_per_unit(self) -> int:
        return self.window * self.group

    @property
    def byte_mode(self) -> bool:
        return self.budget_bytes > 0

    @property
    def max_pos(self) -> int:
        """Rows of the rotary table: every old and new position must index it."""
        return max(self.first_pos + self.n_tokens, self.decode_pos + 1,
                   self.budget_tokens + 1, self.limit)

    def capacity(self) -> int:
        """Rows per pool per unit that always suffice for this policy."""
        if self.byte_mode:
            return self.n_tokens
        return min(self.n_tokens, self.budget_tokens)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# Synthetic frozen (tag, layer-group) table for the PASK-style workload.
# Columns are layer groups 0..3 (lower .. upper); the pages print no table
# (theirs is calibrated offline), so this one is made up with a spread of
# actions per group.
PASK_TABLE = np.array([
    [ACT_RELEASE, ACT_RELEASE, ACT_RELEASE, ACT_RELEASE],   # 0 free text
    [ACT_BF16,    ACT_BF16,    ACT_BF16,    ACT_BF16],      # 1
    [ACT_INT4,    ACT_INT8,    ACT_BF16,    ACT_BF16],      # 2
    [ACT_INT4,    ACT_INT4,    ACT_INT8,    ACT_INT8],      # 3
    [ACT_RELEASE, ACT_RELEASE, ACT_RELEASE, ACT_RELEASE],   # 4
    [ACT_INT4,    ACT_INT4,    ACT_INT4,    ACT_INT4],      # 5
    [ACT_INT8,    ACT_INT8,    ACT_BF16,    ACT_BF16],      # 6
    [ACT_RELEASE, ACT_INT4,    ACT_INT4,    ACT_INT8],      # 7
], dtype=np.uint8)


def _byte_budget_third(n_tokens: int, head_dim: int) -> int:
    """One third of the full bf16 K+V payload of one unit, in bytes."""
    return (n_tokens * 4 * head_dim) // 3


def tiny() -> Workload:
    """1 layer, 4 q / 2 KV heads, d=64, T=1024, window 32, budget 256."""
    return Workload(name="tiny_T1024", batch=1, n_layers=1, n_q_heads=4, n_kv_heads=2,
                    head_dim=64, n_tokens=1024, window=32, rope_theta=1e4,
                    seed=BASE_SEED + 0, budget_tokens=256, n_sink=4, n_recent=32,
                    renumber=True, decode_pos=256)


def qwen3_8b_32k() -> Workload:
    """Qwen3-8B layout, one 32K-token session, budget 2048, bounded positions."""
    return Workload(name="qwen3_8b_T32768", batch=1, n_layers=36, n_q_heads=32, n_kv_heads=8,
                    head_dim=128, n_tokens=32768, window=64, rope_theta=1e6,
                    seed=BASE_SEED + 1, budget_tokens=2048, n_sink=4, n_recent=128,
                    renumber=True, outlier_frac=0.01, outlier_scale=3.0,
                    bonus_spans=4, bonus_span_len=64, bonus_value=10.0, decode_pos=2048)


def pask_batch16() -> Workload:
    """Llama-8B layout, batch 16, T=8192, byte budget 1/3 of full K+V."""
    return Workload(name="pask_llama8b_b16_T8192", batch=16, n_layers=32, n_q_heads=32,
                    n_kv_heads=8, head_dim=128, n_tokens=8192, window=64, rope_theta=5e5,
                    seed=BASE_SEED + 2, budget_bytes=_byte_budget_third(8192, 128),
                    n_sink=4, n_recent=64, renumber=False, n_layer_groups=4,
                    tag_probs=(0.6,) + (0.4 / 7,) * 7, decode_pos=8192)


def commitkv_pages_128k() -> Workload:
    """Qwen3-8B layout, T=131072, 16-token pages, budget 2048 tokens."""
    return Workload(name="commitkv_qwen3_8b_T131072_P16", batch=1, n_layers=36, n_q_heads=32,
                    n_kv_heads=8, head_dim=128, n_tokens=131072, window=64, rope_theta=1e6,
                    seed=BASE_SEED + 3, budget_tokens=2048, n_sink=4, n_recent=64,
                    page_size=16, renumber=False, protect_pages=16, retire_pages=819,
                    decode_pos=131072)


def million_token_8l() -> Workload:
    """8 layers of the Qwen3-8B head layout, T=1,048,576, budget 2048."""
    return Workload(name="qwen3_8b_8L_T1048576", batch=1, n_layers=8, n_q_heads=32,
                    n_kv_heads=8, head_dim=128, n_tokens=1 << 20, window=64, rope_theta=1e6,
                    seed=BASE_SEED + 4, budget_tokens=2048, n_sink=4, n_recent=128,
                    renumber=True, decode_pos=2048)


def million_token_sustained() -> Workload:
    """The million-token session in cycles (PACE Sec. 3.2 "Choosing L", Sec. 5.7):
    2,048 resident rows; each cycle appends a chunk of 4,096 rows and compacts
    the 6,144-row cache back to 2,048 rows, renumbering below L = 8,192;
    256 cycles append 1,048,576 rows."""
    return million_token_8l().replace(name="qwen3_8b_8L_sustained_4096x256", n_tokens=2048 + 4096,
                                      chunk=4096, cycles=256, limit=8192)


ALL = {w().name: w for w in (tiny, qwen3_8b_32k, pask_batch16, commitkv_pages_128k,
                             million_token_8l)}


# --------------------------------------------------------------------------
# drawing
# --------------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, g, device, chunk_rows: int = 1 << 24) -> torch.Tensor:
    """N(0,1) drawn in fp32 and rounded to bf16, in row chunks to bound memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1, shape[-1])
    rows = flat.shape[0]
    step = max(1, chunk_rows // shape[-1])
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        flat[r0:r1] = torch.randn((r1 - r0, shape[-1]), generator=g, device=device,
                                  dtype=torch.float32).to(torch.bfloat16)
    return out


def rope_tables(max_pos: int, head_dim: int, theta: float, device="cpu"):
    """The engine's split-half rotary tables, cos and sin of p * theta^(-2i/d).

    Shape [max_pos][head_dim/2] fp32, angles formed in fp64.
    """
    half = head_dim // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / head_dim)
    cos = np.empty((max_pos, half), dtype=np.float32)
    sin = np.empty((max_pos, half), dtype=np.float32)
    step = 1 << 16
    for p0 in range(0, max_pos, step):
        p1 = min(max_pos, p0 + step)
        ang = np.arange(p0, p1, dtype=np.float64)[:, None] * inv[None, :]
        cos[p0:p1] = np.cos(ang)
        sin[p0:p1] = np.sin(ang)
    return torch.from_numpy(cos).to(device), torch.from_numpy(sin).to(device)


def make_inputs(w: Workload, device="cpu", with_tables: bool = True) -> dict:
    """All inputs of one compaction pass for workload `w`, on `device`."""
    dev = torch.device(device)
    g = _gen(w.seed, dev)
    B, L, Hq, Hkv, d, T, W = (w.batch, w.n_layers, w.n_q_heads, w.n_kv_heads,
                              w.head_dim, w.n_tokens, w.window)
    U = w.n_units
    # per-sequence structure drawn on the host from its own stream
    rng = np.random.Generator(np.random.PCG64(w.seed))

    k = _randn_bf16((B, L, Hkv, T, d), g, dev)
    if w.outlier_frac > 0:
        n_out = int(round(w.outlier_frac * T))
        for b in range(B):
            idx = torch.from_numpy(rng.choice(T, size=n_out, replace=False)).to(dev)
            kb = k[b]
            kb[:, :, idx, :] = (kb[:, :, idx, :].float() * w.outlier_scale).to(torch.bfloat16)
    v = _randn_bf16((B, L, Hkv, T, d), g, dev)
    q_window = _randn_bf16((B, L, Hq, W, d), g, dev)
    q_decode = _randn_bf16((B, L, Hq, d), g, dev)

    pos = torch.arange(w.first_pos, w.first_pos + T, dtype=torch.int32, device=dev)
    pos_in = pos.view(1, T).expand(U, T).contiguous()

    out = dict(k_cache=k, v_cache=v, q_window=q_window, q_decode=q_decode, pos_in=pos_in)

    if w.bonus_spans > 0:
        bonus = np.zeros((B, T), dtype=np.float32)
        lo, hi = w.n_sink, T - w.n_recent
        span = w.bonus_span_len
        slots = (hi - lo) // span
        for b in range(B):
            pick = rng.choice(slots, size=w.bonus_spans, replace=False)
            for s in pick:
                a = lo + int(s) * span
                bonus[b, a:a + span] = w.bonus_value
        out["bonus"] = torch.from_numpy(bonus).to(dev)

    if w.tag_probs is not None:
        tags = rng.choice(len(w.tag_probs), size=(B, T), p=np.asarray(w.tag_probs))
        out["tags"] = torch.from_numpy(tags.astype(np.uint8)).to(dev)
        out["action_table"] = torch.from_numpy(PASK_TABLE.copy()).to(dev)

    if w.protect_pages > 0 or w.retire_pages > 0:
        P = w.page_size
        n_pages = T // P
        first_free = -(-w.n_sink // P)
        last_free = (T - w.n_recent) // P
        flags = np.zeros((B, n_pages), dtype=np.uint8)
        for b in range(B):
            pool = np.arange(first_free, last_free)
            pick = rng.choice(pool, size=w.protect_pages + w.retire_pages, replace=False)
            flags[b, pick[:w.protect_pages]] = FLAG_PROTECT
            flags[b, pick[w.protect_pages:]] = FLAG_EXCLUDE
        out["flags"] = torch.from_numpy(flags).to(dev)

    if with_tables:
        cos, sin = rope_tables(w.max_pos, d, w.rope_theta, dev)
        out["rope_cos"], out["rope_sin"] = cos, sin
    return out


def session_start(w: Workload, device="cpu") -> dict:
    """Resident rows before a session's first cycle: keys and values
    [B][L][H_kv][budget][d] bf16 at positions 0..budget-1, and the rotary
    tables (positions below the limit L)."""
    dev = torch.device(device)
    g = _gen(w.seed, dev)
    B, L, Hkv, d = w.batch, w.n_layers, w.n_kv_heads, w.head_dim
    k0 = _randn_bf16((B, L, Hkv, w.budget_tokens, d), g, dev)
    v0 = _randn_bf16((B, L, Hkv, w.budget_tokens, d), g, dev)
    cos, sin = rope_tables(w.max_pos, d, w.rope_theta, dev)
    return dict(k0=k0, v0=v0, rope_cos=cos, rope_sin=sin)


def session_chunk(w: Workload, c: int, device="cpu") -> dict:
    """Chunk c of a session (its own seed): keys and values
    [B][L][H_kv][chunk][d] bf16, treated as rotated at the positions the session
    assigns them, and the window queries [B][L][H_q][W][d] of its last W rows."""
    dev = torch.device(device)
    g = _gen(w.seed * 4099 + 17 * c + 1, dev)
    B, L, Hq, Hkv, d, W = w.batch, w.n_layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.window
    return dict(k=_randn_bf16((B, L, Hkv, w.chunk, d), g, dev),
                v=_randn_bf16((B, L, Hkv, w.chunk, d), g, dev),
                q_window=_randn_bf16((B, L, Hq, W, d), g, dev))


def unit_index(w: Workload, b: int, l: int, g: int) -> int:
    return (b * w.n_layers + l) * w.n_kv_heads + g


def unit_coords(w: Workload, u: int):
    g = u % w.n_kv_heads
    l = (u // w.n_kv_heads) % w.n_layers
    b = u // (w.n_kv_heads * w.n_layers)
    return b, l, g


# --------------------------------------------------------------------------
# CommitKV deletion-effect measurements
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class EffectWorkload:
    """One attention layer's window measurement over scanned event pages.

    CommitKV Sec. 4.1: query window W = 8, event pages of at most G = 16
    tokens, at most 64 pages scanned per commit.  Two windows are drawn
    over the same cache: the pre-commit one leans toward one set of "heavy"
    pages and the post-commit one toward another, partly overlapping set, so
    that all lifecycle transitions occur.
    """
    name: str
    batch: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_tokens: int
    seed: int
    window: int = 8
    n_pages: int = 64
    page_len: int = 16
    heavy_pages: int = 12        # heavy pages of each window (a third shared)
    lean: float = 7.5            # size of the shared direction added to queries / heavy keys
    away: float = 3.0            # post-commit queries lean away from the pre-commit direction
    value_mean: float = 1.0      # norm of a per-head mean added to every value, in units of sqrt(d)
    ragged_pages: bool = False   # one short page, one empty page, one over the window rows

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def n_units(self) -> int:
        return self.batch * self.n_layers * self.n_kv_heads


def commitkv_effect_128k() -> EffectWorkload:
    """Qwen3-8B layout, one layer, T=131072, W=8, 64 pages of 16 tokens."""
    return EffectWorkload(name="commitkv_effect_qwen3_8b_T131072", batch=1, n_layers=1,
                          n_q_heads=32, n_kv_heads=8, head_dim=128, n_tokens=131072,
                          seed=BASE_SEED + 5)


def commitkv_effect_small(n_q_heads=8, n_kv_heads=2, window=8, n_tokens=1000) -> EffectWorkload:
    """Two sequences, two layers, a ragged T: parity-sized."""
    return EffectWorkload(name=f"commitkv_effect_small_H{n_q_heads}_{n_kv_heads}_W{window}",
                          batch=2, n_layers=2, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads,
                          head_dim=128, n_tokens=n_tokens, seed=BASE_SEED + 6, window=window,
                          n_pages=12, heavy_pages=4, lean=6.0, ragged_pages=True)


def make_effect_inputs(w: EffectWorkload, device="cpu") -> dict:
    """K, V [B][L][H_kv][T][d], windows q_minus / q_plus [B][L][H_q][W][d] (bf16),
    pages page_start / page_len int32 [B][n_pages] (disjoint, ascending), and
    the heavy page ids of each window (host lists)."""
    dev = torch.device(device)
    g = _gen(w.seed, dev)
    rng = np.random.Generator(np.random.PCG64(w.seed))
    B, L, Hq, Hkv, d, T, W = (w.batch, w.n_layers, w.n_q_heads, w.n_kv_heads, w.head_dim,
                              w.n_tokens, w.window)
    G = w.group
    k = _randn_bf16((B, L, Hkv, T, d), g, dev).float()
    v = _randn_bf16((B, L, Hkv, T, d), g, dev).float()
    if w.value_mean > 0:
        mu = torch.randn((B, L, Hkv, 1, d), generator=g, device=dev)
        v += mu / mu.norm(dim=-1, keepdim=True) * (w.value_mean * math.sqrt(d))
    qm = _randn_bf16((B, L, Hq, W, d), g, dev).float()
    qp = _randn_bf16((B, L, Hq, W, d), g, dev).float()

    P = w.page_len
    # the ragged layout's last page covers the window rows: random pages end before it
    slots = ((T - W - 3) if w.ragged_pages else T) // P
    starts = np.zeros((B, w.n_pages), dtype=np.int32)
    lens = np.full((B, w.n_pages), P, dtype=np.int32)
    heavy_minus, heavy_plus = [], []
    for b in range(B):
        pick = np.sort(rng.choice(slots, size=w.n_pages, replace=False))
        starts[b] = pick * P
        if w.ragged_pages:
            lens[b, 1] = 5                                # a short page
            lens[b, 2] = 0                                # an empty slot
            starts[b, -1] = T - W - 3                     # over the window rows (last page)
            lens[b, -1] = min(P, W + 3)
            order = np.argsort(starts[b], kind="stable")
            starts[b], lens[b] = starts[b][order], lens[b][order]
        ids = rng.permutation(w.n_pages)
        n_h = min(w.heavy_pages, w.n_pages // 3)
        shared = n_h // 3
        hm = ids[:n_h]
        hp = np.concatenate([ids[:shared], ids[n_h:2 * n_h - shared]])
        heavy_minus.append(sorted(int(i) for i in hm))
        heavy_plus.append(sorted(int(i) for i in hp))
        # a unit direction per (layer, KV head) and window; heavy pages' keys
        # and the window's queries both lean along it, and the post-commit
        # queries lean away from the pre-commit direction
        for l in range(L):
            for gk in range(Hkv):
                dirs = []
                for q, heavy in ((qm, hm), (qp, hp)):
                    u = torch.randn(d, generator=g, device=dev)
                    u = u / u.norm()
                    dirs.append(u)
                    q[b, l, gk * G:(gk + 1) * G] += w.lean * u
                    for pid in heavy:
                        s0, n0 = int(starts[b, pid]), int(lens[b, pid])
                        k[b, l, gk, s0:s0 + n0] += w.lean * u
                qp[b, l, gk * G:(gk + 1) * G] -= w.away * dirs[0]
    return dict(k_cache=k.to(torch.bfloat16), v_cache=v.to(torch.bfloat16), q_minus=qm.to(torch.bfloat16),
                q_plus=qp.to(torch.bfloat16), page_start=torch.from_numpy(starts).to(dev),
                page_len=torch.from_numpy(lens).to(dev), heavy_minus=heavy_minus,
                heavy_plus=heavy_plus)
