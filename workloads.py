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
                   self.budget_tokens + 1)

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


def unit_index(w: Workload, b: int, l: int, g: int) -> int:
    return (b * w.n_layers + l) * w.n_kv_heads + g


def unit_coords(w: Workload, u: int):
    g = u % w.n_kv_heads
    l = (u // w.n_kv_heads) % w.n_layers
    b = u // (w.n_kv_heads * w.n_layers)
    return b, l, g
