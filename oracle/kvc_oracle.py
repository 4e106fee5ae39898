"""Plain CPU oracle of the budgeted KV-cache compaction pass.

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the CPU
baseline leg of the benchmark import this module; the library and its
Python binding never do, and nothing here calls the library.

Sources (page title, then the section / equation):
  * PASK  = "Parser Transitions Already Reveal Structural Responsibility: KV
            Persistence for Structured Generation" (arXiv 2608.28276)
  * PACE  = "PACE: Keeping the Right Tokens in the KV Cache Is Not Enough for
            Long-Horizon LLM Agents" (arXiv 2611.10240)
  * CommitKV = "CommitKV: Lifecycle-Aware KV Cache Compression via Commit
            Transitions for Multi-Turn Agents" (arXiv 2608.07855)

Floating point is fp64 except where the result decides an integer or a
stored bit pattern: re-rotation and quantisation follow a fixed fp32
operation order (each product, sum, square root and quotient rounded once,
no fused multiply-add), the precision the CUDA kernels use, so that the
stored bf16 keys and the int8/int4 codes can be compared bit for bit.

Every function below is pinned by a `-m "not gpu"` test against values the
pages print, closed forms, library routines or brute force; none is
"parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

ACT_RELEASE, ACT_INT4, ACT_INT8, ACT_BF16 = 0, 1, 2, 3
FLAG_PROTECT, FLAG_EXCLUDE = 1, 2
QUANT_G32_BF16, QUANT_ROW_FP16 = 0, 1
UNIT_OK, UNIT_OVER_BUDGET, UNIT_BAD_INDEX, UNIT_BAD_FLAGS = 0, 1, 2, 3

BF16_MIN_POSITIVE = 2.0 ** -133      # smallest bf16 subnormal
FP16_MIN_POSITIVE = 2.0 ** -24       # smallest fp16 subnormal
FP16_MAX = 65504.0

# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even; NaN stays NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint32)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, ((u >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint32), r)
    return r.astype(np.uint16)


def bf16_round(x) -> np.ndarray:
    """Round fp32 values to the nearest bf16 and return them as fp32."""
    return bf16_bits_to_f32(f32_to_bf16_bits(x))


# ----------------------------------------------------------------------------
# layer groups -- PASK, App. A.2
# ----------------------------------------------------------------------------


def layer_group_bounds(n_layers: int, n_groups: int) -> list:
    """Group boundaries b_k = floor((k*L + G - 1) / G), k = 0..G.

    For G = 3 this is PASK's b1 = floor((L+2)/3), b2 = floor((2L+2)/3); the
    same rule is used for any number of groups.
    """
    return [(k * n_layers + n_groups - 1) // n_groups if 0 < k < n_groups
            else (0 if k == 0 else n_layers) for k in range(n_groups + 1)]


def layer_group(layer: int, n_layers: int, n_groups: int) -> int:
    b = layer_group_bounds(n_layers, n_groups)
    for c in range(n_groups):
        if b[c] <= layer < b[c + 1]:
            return c
    raise ValueError("layer out of range")


# ----------------------------------------------------------------------------
# a1/a2: observation-window attention mass -- PASK Eq. 1; the SnapKV window
# scorer described in PASK App. C.3 and CommitKV Sec. 3.1; the bonus of PACE
# Sec. 3.1 is added to the score and the top-B are kept by the sum.
# ----------------------------------------------------------------------------


def window_mass(k, q, scale: float, row_block: int = 8) -> np.ndarray:
    """Attention mass that the window rows put on each cached key.

    k : [T][d] keys (already rotated at their physical positions)
    q : [G][W][d] window queries of the G query heads that share this KV
        head; row w of every head sits at cache index T - W + w and, by
        causality, sees keys j <= T - W + w.
    Returns mass[j] = sum over heads h and rows w of softmax_j(q_hw . k_j * scale),
    in fp64.
    """
    k = np.asarray(k, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    T = k.shape[0]
    G, W, d = q.shape
    rows = q.reshape(G * W, d)
    last_visible = np.tile(T - W + np.arange(W), G)          # per row
    mass = np.zeros(T, dtype=np.float64)
    j = np.arange(T)
    for r0 in range(0, G * W, row_block):
        r1 = min(G * W, r0 + row_block)
        z = (rows[r0:r1] @ k.T) * scale                        # [rb][T]
        z = np.where(j[None, :] <= last_visible[r0:r1, None], z, -np.inf)
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        a = e / e.sum(axis=1, keepdims=True)
        mass += a.sum(axis=0)
    return mass


def window_row_lse(k, q, scale: float) -> np.ndarray:
    """Natural-log log-sum-exp of each window row's visible logits, fp64.

    The softmax denominator of PASK Eq. 1 for the rows of window_mass, in
    the same row order (head-major: row h * W + w), as an attention kernel
    that ran the window would report it.
    """
    k = np.asarray(k, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    T = k.shape[0]
    G, W, d = q.shape
    rows = q.reshape(G * W, d)
    out = np.empty(G * W, dtype=np.float64)
    for r in range(G * W):
        z = (k[: T - W + (r % W) + 1] @ rows[r]) * scale
        m = z.max()
        out[r] = m + np.log(np.exp(z - m).sum())
    return out


def window_mass_given_lse(k, q, scale: float, row_lse) -> np.ndarray:
    """mass[j] = sum over visible rows of exp(q_hw . k_j * scale - row_lse[hw]), fp64.

    With the rows' own log-sum-exp this is window_mass; with any other
    per-row value it is what the scorer computes from a caller's statistics.
    """
    k = np.asarray(k, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    lse = np.asarray(row_lse, dtype=np.float64)
    T = k.shape[0]
    G, W, d = q.shape
    rows = q.reshape(G * W, d)
    mass = np.zeros(T, dtype=np.float64)
    for r in range(G * W):
        n = T - W + (r % W) + 1
        mass[:n] += np.exp((k[:n] @ rows[r]) * scale - lse[r])
    return mass


def unit_scores(k_bits, q_bits, scale: float, bonus=None, acc=None) -> np.ndarray:
    """score_j = fp32(mass_j + bonus_j + acc_j) for one unit (bf16 inputs as bits)."""
    k = bf16_bits_to_f32(k_bits)
    q = bf16_bits_to_f32(q_bits)
    s = window_mass(k, q, scale)
    if bonus is not None:
        s = s + np.asarray(bonus, dtype=np.float32).astype(np.float64)
    if acc is not None:
        s = s + np.asarray(acc, dtype=np.float32).astype(np.float64)
    return s.astype(np.float32)


def foresight_bonus(spans, t: int, n_tokens: int, sigma: float = 1e5, lam: float = 0.35) -> np.ndarray:
    """PACE Eq. 2: the foresight bonus of every token at step t, fp64 [T].

    spans: (a, b, F) with F the future steps that read tokens [a, b).  A
    token in a span whose next reference s* = min{s in F : s >= t} exists
    gets sigma * (1/2 + 1/2 exp(-lambda (s* - t))); a token with no future
    reference gets 0.  A token in several spans takes the largest bonus (its
    soonest reference).
    """
    bonus = np.zeros(n_tokens, dtype=np.float64)
    for a, b, F in spans:
        future = [s for s in F if s >= t]
        if not future:
            continue
        s_next = min(future)
        beta = sigma * (0.5 + 0.5 * math.exp(-lam * (s_next - t)))
        lo, hi = max(0, int(a)), min(n_tokens, int(b))
        if lo < hi:
            bonus[lo:hi] = np.maximum(bonus[lo:hi], beta)
    return bonus


def cumulative_decode_scores(k_bits, q_steps_bits, scale: float, bonus=None) -> np.ndarray:
    """H2O cumulative attention score of one unit after several decode steps,
    plus an optional bonus (PACE Sec. 3.1: the bonus is added to the token's
    cumulative attention score), fp32 [T].

    q_steps_bits: [n_steps][G][d] the decode queries of the G heads sharing
    the KV head, one step each; every step attends to all T cached keys
    (window 1 at the last row) and the weights are summed over heads and steps.
    """
    k = bf16_bits_to_f32(k_bits)
    acc = np.zeros(k.shape[0], dtype=np.float64)
    for q in np.asarray(q_steps_bits):
        acc += window_mass(k, bf16_bits_to_f32(q)[:, None, :], scale)
    if bonus is not None:
        acc = acc + np.asarray(bonus, dtype=np.float64)
    return acc.astype(np.float32)


def pool_scores(scores, kernel: int, mode: str) -> np.ndarray:
    """SnapKV's 1-D pooling of token scores before selection (the pooling
    and kernel options of the SnapKV baseline in PASK's baseline table):
    for each token the average or maximum over the `kernel` tokens centred on
    it, stride 1.  Positions outside [0, T) count as 0 in the average
    (divided by `kernel`) and are ignored by the maximum.  fp32 in, fp32 out
    (the average summed in fp64).
    """
    s = np.asarray(scores, dtype=np.float32)
    T = s.size
    h = kernel // 2
    out = np.empty(T, dtype=np.float32)
    for j in range(T):
        lo, hi = max(0, j - h), min(T, j + h + 1)
        if mode == "avg":
            out[j] = np.float32(s[lo:hi].astype(np.float64).sum() / kernel)
        else:
            out[j] = s[lo:hi].max()
    return out


def shared_scores(unit_scores_of_sequence) -> np.ndarray:
    """CommitKV Eq. 4 applies one index set to the keys, values and positions
    of every layer and head: the per-token score of a sequence is the sum of
    its units' scores, fp32 [T] (summed in fp64)."""
    a = np.asarray(unit_scores_of_sequence, dtype=np.float32).astype(np.float64)
    return a.sum(axis=0).astype(np.float32)


def page_max(scores, page_size: int) -> np.ndarray:
    """Page score = maximum token score over each page (max pooling)."""
    s = np.asarray(scores, dtype=np.float32)
    return s.reshape(-1, page_size).max(axis=1)


# ----------------------------------------------------------------------------
# a3/a4: masks and deterministic selection
# ----------------------------------------------------------------------------


def canonical(scores) -> np.ndarray:
    """-0 -> +0 and NaN -> -inf, so that the order of scores is total."""
    s = np.asarray(scores, dtype=np.float32).copy()
    s[np.isnan(s)] = -np.inf
    s[s == 0] = 0.0
    return s


def rank_order(scores, idx) -> np.ndarray:
    """Positions of `idx` sorted by (score descending, index ascending)."""
    s = canonical(scores).astype(np.float64)
    return np.lexsort((np.asarray(idx), -s))


def item_masks(n_items: int, sink_items: int, recent_items: int, flags):
    """forced / excluded / bad-flag masks over selection items (tokens or pages).

    Sinks (the first `sink_items`) and the recent window (the last
    `recent_items`) are always kept; PROTECT adds to the kept set (CommitKV
    Eq. 13, N is a subset of I); EXCLUDE removes an item unless it is a sink
    or recent item.  An item flagged both PROTECT and EXCLUDE is an error.
    """
    i = np.arange(n_items)
    window = (i < sink_items) | (i >= n_items - recent_items)
    fl = np.zeros(n_items, dtype=np.uint8) if flags is None else np.asarray(flags, np.uint8)
    protect = (fl & FLAG_PROTECT) != 0
    exclude = (fl & FLAG_EXCLUDE) != 0
    bad = bool((protect & exclude).any())
    forced = window | protect
    excluded = exclude & ~window
    return forced, excluded, bad


def select_top(scores, budget: int, forced, excluded):
    """Kept items (ascending) and unit status for token / page mode.

    Forced items are kept; if they alone exceed the budget the unit is
    OVER_BUDGET and nothing is kept (CommitKV Eq. 4: |I| <= B).  Otherwise
    the k = min(budget - |F|, |E|) eligible items that rank first by
    (score descending, index ascending) are added.
    """
    forced = np.asarray(forced, bool)
    excluded = np.asarray(excluded, bool)
    n_forced = int(forced.sum())
    if n_forced > budget:
        return np.zeros(0, dtype=np.int64), UNIT_OVER_BUDGET
    elig = np.nonzero(~forced & ~excluded)[0]
    k = min(budget - n_forced, elig.size)
    order = rank_order(np.asarray(scores)[elig], elig)
    take = elig[order[:k]]
    kept = np.sort(np.concatenate([np.nonzero(forced)[0], take]))
    return kept.astype(np.int64), UNIT_OK


def sink_recent_pages(n_tokens: int, page_size: int, n_sink: int, n_recent: int):
    """Pages holding any sink or recent token: (first pages, last pages)."""
    n_pages = n_tokens // page_size
    first = -(-n_sink // page_size)
    last_start = (n_tokens - n_recent) // page_size
    return first, n_pages - last_start


def select_tokens(scores, n_tokens: int, budget: int, n_sink: int, n_recent: int,
                  flags=None, page_size: int = 1):
    """Token mode (page_size = 1) or page mode (scores are page scores).

    Returns (kept token indices ascending, status).
    """
    if page_size == 1:
        forced, excluded, bad = item_masks(n_tokens, n_sink, n_recent, flags)
        if bad:
            return np.zeros(0, dtype=np.int64), UNIT_BAD_FLAGS
        return select_top(scores, budget, forced, excluded)
    n_pages = n_tokens // page_size
    sp, rp = sink_recent_pages(n_tokens, page_size, n_sink, n_recent)
    forced, excluded, bad = item_masks(n_pages, sp, rp, flags)
    if bad:
        return np.zeros(0, dtype=np.int64), UNIT_BAD_FLAGS
    pages, st = select_top(scores, budget // page_size, forced, excluded)
    toks = (pages[:, None] * page_size + np.arange(page_size)[None, :]).reshape(-1)
    return toks.astype(np.int64), st


# ----------------------------------------------------------------------------
# byte mode -- PASK App. B.3 (payload), App. B.4 (floors first, priority
# order, floor excess recorded), Sec. 3.5 (floors take precedence)
# ----------------------------------------------------------------------------


def row_bytes(action: int, head_dim: int, quant_mode: int = QUANT_G32_BF16) -> int:
    """Bytes stored for one token of one unit (its K row plus its V row)."""
    d = head_dim
    if action == ACT_RELEASE:
        return 0
    if action == ACT_BF16:
        return 2 * 2 * d
    scales = 2 * (d // 32) if quant_mode == QUANT_G32_BF16 else 2
    code = d if action == ACT_INT8 else d // 2
    return 2 * (code + scales)


def select_bytes(scores, floors, budget_bytes: int, n_sink: int, n_recent: int,
                 head_dim: int, quant_mode: int = QUANT_G32_BF16, flags=None):
    """Byte-budget selection of one unit.

    floors : per-token floor action from the (tag, layer-group) table.
    Sink/recent and PROTECT tokens are held at bf16; EXCLUDE releases.
    The remainder budget - sum(cost(floor)) is spent by promoting to bf16 the
    longest prefix of the (score desc, index asc) order of the remaining
    non-bf16 tokens whose summed upgrade costs fit.  A negative remainder is
    recorded as floor excess and nothing is promoted.
    Returns (action per token, floor_excess, status).
    """
    T = len(floors)
    forced, excluded, bad = item_masks(T, n_sink, n_recent, flags)
    if bad:
        return np.zeros(T, dtype=np.uint8), 0, UNIT_BAD_FLAGS
    act = np.asarray(floors, dtype=np.uint8).copy()
    act[forced] = ACT_BF16
    act[excluded] = ACT_RELEASE
    cost = np.array([row_bytes(a, head_dim, quant_mode) for a in range(4)], dtype=np.int64)
    rem = int(budget_bytes) - int(cost[act].sum())
    if rem < 0:
        return act, -rem, UNIT_OK
    cand = np.nonzero(~forced & ~excluded & (act != ACT_BF16))[0]
    order = cand[rank_order(np.asarray(scores)[cand], cand)]
    delta = cost[ACT_BF16] - cost[act[order]]
    n_up = int(np.searchsorted(np.cumsum(delta), rem, side="right"))
    act[order[:n_up]] = ACT_BF16
    return act, 0, UNIT_OK


# ----------------------------------------------------------------------------
# a5/a6: renumber, exact re-rotation -- PACE Sec. 3.2 (bounded positions,
# Proposition 1); CommitKV Eq. 4 (apply one index set to K, V, positions)
# ----------------------------------------------------------------------------


def rope_angles(pos, head_dim: int, theta: float) -> np.ndarray:
    """pos * theta^(-2i/d) for i < d/2, fp64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.asarray(pos, dtype=np.float64)[..., None] * theta ** (-2.0 * i / head_dim)


def rope_rotate(x, pos, head_dim: int, theta: float) -> np.ndarray:
    """Split-half rotary rotation R_pos of x in fp64 (PACE Eq. 1)."""
    x = np.asarray(x, dtype=np.float64)
    h = head_dim // 2
    a = rope_angles(pos, head_dim, theta)
    c, s = np.cos(a), np.sin(a)
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def rerotate_bits(k_bits, p: int, p_new: int, cos_tab, sin_tab, layout: str = "split",
                  rotary_dim: int = 0) -> np.ndarray:
    """Re-rotate one stored bf16 key from position p to p_new (fp32 spec).

    cos/sin of (p_new - p) theta_i come from the engine's own tables through
    the angle-difference identities and are normalised to unit length
    (PACE Sec. 3.2); every product, sum, root and quotient is rounded to fp32
    once, in this order, and the rotated elements are rounded to bf16.
    If p_new == p the stored bits are returned unchanged.

    Rotary layouts (PACE Sec. 3.2: the same rotation applied to the rotated
    dimensions only): the first `rotary_dim` elements rotate (0 = all), as
    split halves (element i pairs with i + rotary_dim/2, layout "split") or
    as adjacent pairs (2i with 2i + 1, layout "interleaved"); the tables are
    [max_pos][rotary_dim / 2]; elements past rotary_dim are copied.
    """
    k_bits = np.asarray(k_bits, dtype=np.uint16)
    if p_new == p:
        return k_bits.copy()
    f = np.float32
    d = k_bits.shape[-1]
    rd = rotary_dim or d
    c0 = np.asarray(cos_tab[p], dtype=f)
    s0 = np.asarray(sin_tab[p], dtype=f)
    c1 = np.asarray(cos_tab[p_new], dtype=f)
    s1 = np.asarray(sin_tab[p_new], dtype=f)
    C = (c1 * c0) + (s1 * s0)
    S = (s1 * c0) - (c1 * s0)
    n = np.sqrt((C * C) + (S * S))
    C = C / n
    S = S / n
    h = rd // 2
    if layout == "split":
        xi, yi = np.arange(h), h + np.arange(h)
    else:
        xi, yi = 2 * np.arange(h), 2 * np.arange(h) + 1
    x = bf16_bits_to_f32(k_bits[..., xi])
    y = bf16_bits_to_f32(k_bits[..., yi])
    xr = (x * C) - (y * S)
    yr = (y * C) + (x * S)
    out = k_bits.copy()
    out[..., xi] = f32_to_bf16_bits(xr)
    out[..., yi] = f32_to_bf16_bits(yr)
    return out


def reference_rerotate(k_bits, p: int, p_new: int, ref_bits, p_ref: int, cos_tab, sin_tab):
    """Non-compounding re-rotation of one kept key through a reference store.

    PACE Sec. 3.2 / App. D: at a key's first position-changing renumber a
    copy of the stored key is kept together with the position p_ref it is
    valid at, and every later position is derived from that copy (in fp32,
    by rerotate_bits), so the key carries about two roundings however many
    renumbers it survives.  Before use the copy is checked against the
    stored key: rotated from p_ref to the key's current position p it must
    reproduce the stored bits exactly; if it does not, the stored key is
    used and becomes the new reference.

    Returns (new key bits, reference bits, p_ref, check_failed); p_ref < 0
    means "no reference" (the key has not been renumbered yet).
    """
    k_bits = np.asarray(k_bits, dtype=np.uint16)
    if p_new == p:                                   # no renumber: carry as is
        ref = None if p_ref < 0 else np.asarray(ref_bits, dtype=np.uint16).copy()
        return k_bits.copy(), ref, p_ref, False
    if p_ref >= 0:
        ref = np.asarray(ref_bits, dtype=np.uint16)
        if np.array_equal(rerotate_bits(ref, p_ref, p, cos_tab, sin_tab), k_bits):
            return rerotate_bits(ref, p_ref, p_new, cos_tab, sin_tab), ref.copy(), p_ref, False
        failed = True
    else:
        failed = False
    return rerotate_bits(k_bits, p, p_new, cos_tab, sin_tab), k_bits.copy(), p, failed


def renumber_drift(x, positions, cos_tab, sin_tab, use_store: bool, norm: str = "max") -> float:
    """Relative error of a key renumbered along `positions` (PACE App. D).

    x: exact pre-rotation key [d] (fp64).  The stored key starts as the bf16
    rounding of x rotated (in fp64) to positions[0]; every later entry is a
    renumber, done by re-rotating the stored key (use_store False) or through
    the reference store.  Returns the relative error of the stored key at
    the last position against x rotated there in fp64: by default in the
    maximum norm, max_i |stored_i - exact_i| / max_i |exact_i| (the page's
    "relative key error"; its printed means after 23 / 71 / 240 renumbers
    are reproduced in this norm), or in the Euclidean norm (norm="l2").
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.size
    h = d // 2

    def exact(pos):
        c = np.asarray(cos_tab[pos], np.float64)
        s_ = np.asarray(sin_tab[pos], np.float64)
        return np.concatenate([x[:h] * c - x[h:] * s_, x[h:] * c + x[:h] * s_])

    k = f32_to_bf16_bits(exact(positions[0]).astype(np.float32))
    ref, p_ref = None, -1
    for p, p_new in zip(positions[:-1], positions[1:]):
        if use_store:
            k, ref, p_ref, _ = reference_rerotate(k, int(p), int(p_new), ref, p_ref, cos_tab, sin_tab)
        else:
            k = rerotate_bits(k, int(p), int(p_new), cos_tab, sin_tab)
    e = exact(positions[-1])
    diff = bf16_bits_to_f32(k).astype(np.float64) - e
    if norm == "l2":
        return float(np.linalg.norm(diff) / np.linalg.norm(e))
    return float(np.abs(diff).max() / np.abs(e).max())


def new_positions(kept_sorted, pos_in, renumber: bool) -> np.ndarray:
    """p' = rank among the kept rows in logical order if renumbering, else p."""
    kept_sorted = np.asarray(kept_sorted)
    if renumber:
        return np.arange(kept_sorted.size, dtype=np.int64)
    return np.asarray(pos_in)[kept_sorted].astype(np.int64)


def smallest_pow2_limit(budget: int, interval: int, chunk: int) -> int:
    """Smallest power of two L with L > B_max + H, B_max = budget + interval."""
    need = budget + interval + chunk
    L = 1
    while L <= need:
        L *= 2
    return L


def renumber_due(next_pos: int, limit: int, headroom: int) -> bool:
    """PACE Sec. 3.2 trigger: next physical position within H of the limit L."""
    return next_pos > limit - headroom


# ----------------------------------------------------------------------------
# quantisation -- PASK App. B.5 (symmetric, scale = max|x| / qmax rounded to
# the scale format and floored at its smallest positive value, codes rounded
# to nearest and clipped, zero groups -> zero codes and unit scale, two
# signed nibbles per byte)
# ----------------------------------------------------------------------------


def _round_scale(s32: np.ndarray, quant_mode: int) -> np.ndarray:
    if quant_mode == QUANT_G32_BF16:
        s = bf16_round(s32)
        return np.maximum(s, np.float32(BF16_MIN_POSITIVE))
    s = s32.astype(np.float16)
    s = np.minimum(s.astype(np.float32), np.float32(FP16_MAX))
    return np.maximum(s, np.float32(FP16_MIN_POSITIVE))


def quantize(x, qmax: int, quant_mode: int = QUANT_G32_BF16):
    """Quantise rows x [..., d] (fp32 values of bf16 keys/values).

    Groups are 32 consecutive elements (QUANT_G32_BF16, bf16 scale) or the
    whole row (QUANT_ROW_FP16, fp16 scale).  Returns (codes int8 [..., d],
    scales fp32 [..., n_groups]) with scales exactly representable in the
    scale format.
    """
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    gs = 32 if quant_mode == QUANT_G32_BF16 else d
    xg = x.reshape(x.shape[:-1] + (d // gs, gs))
    a = np.abs(xg).max(axis=-1)
    zero = a == 0
    s = _round_scale(a / np.float32(qmax), quant_mode)
    s = np.where(zero, np.float32(1.0), s).astype(np.float32)
    with np.errstate(over="ignore", divide="ignore", invalid="ignore"):
        r = np.rint(xg / s[..., None])
    codes = np.clip(r, -qmax, qmax).astype(np.int8)
    codes[zero] = 0
    return codes.reshape(x.shape), s


def dequantize(codes, scales, quant_mode: int = QUANT_G32_BF16) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.int8)
    d = codes.shape[-1]
    gs = 32 if quant_mode == QUANT_G32_BF16 else d
    cg = codes.reshape(codes.shape[:-1] + (d // gs, gs)).astype(np.float32)
    return (cg * np.asarray(scales, np.float32)[..., None]).reshape(codes.shape)


def pack_int4(codes) -> np.ndarray:
    """Byte j holds element 2j in its low nibble and 2j+1 in its high nibble."""
    c = np.asarray(codes, dtype=np.int8).astype(np.uint8)
    lo = c[..., 0::2] & 0xF
    hi = c[..., 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_int4(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0xF).astype(np.int8)
    hi = (p >> 4).astype(np.int8)
    lo = np.where(lo > 7, lo - 16, lo).astype(np.int8)
    hi = np.where(hi > 7, hi - 16, hi).astype(np.int8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def scale_bits(scales, quant_mode: int) -> np.ndarray:
    """Stored scale bit patterns: bf16 (g32 mode) or fp16 (row mode)."""
    s = np.asarray(scales, dtype=np.float32)
    if quant_mode == QUANT_G32_BF16:
        return f32_to_bf16_bits(s)
    return s.astype(np.float16).view(np.uint16)


# ----------------------------------------------------------------------------
# a7: consumer decode step -- PASK Eq. 1 over all kept rows; Eq. 15 merge
# ----------------------------------------------------------------------------


def attend(q, keys, values, scale: float) -> np.ndarray:
    """softmax(keys q * scale)-weighted sum of values, fp64 (one query)."""
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    if keys.shape[0] == 0:
        return np.zeros(values.shape[-1])
    z = keys @ q * scale
    m = z.max()
    e = np.exp(z - m)
    return (e[:, None] * values).sum(axis=0) / e.sum()


def partition_stats(q, keys, values, scale: float):
    """(max score v_j, exp-sum l_j, unnormalised value sum u_j) of one partition."""
    q = np.asarray(q, np.float64)
    z = np.asarray(keys, np.float64) @ q * scale
    v = z.max()
    e = np.exp(z - v)
    return v, e.sum(), (e[:, None] * np.asarray(values, np.float64)).sum(axis=0)


def merge_partitions(parts) -> np.ndarray:
    """PASK Eq. 15: o = sum_j e^{v_j - v} u_j / sum_j e^{v_j - v} l_j; empty parts skipped."""
    parts = [p for p in parts if p is not None]
    v = max(p[0] for p in parts)
    num = sum(math.exp(p[0] - v) * p[2] for p in parts)
    den = sum(math.exp(p[0] - v) * p[1] for p in parts)
    return num / den


# ----------------------------------------------------------------------------
# one unit end to end
# ----------------------------------------------------------------------------


@dataclass
class Pool:
    """Kept rows of one storage class of one unit, ascending by index."""
    action: int
    idx: np.ndarray
    pos: np.ndarray = None          # new physical position p'
    orig_pos: np.ndarray = None     # position before compaction
    k: np.ndarray = None            # bf16 bits [n][d], or codes [n][d] / packed [n][d/2]
    v: np.ndarray = None
    k_scale: np.ndarray = None      # fp32 [n][groups]
    v_scale: np.ndarray = None
    k_ref: np.ndarray = None        # reference store: bf16 bits [n][d] (zeros: none)
    p_ref: np.ndarray = None        # reference position [n] (-1: none)
    ref_failures: int = 0           # kept keys whose reference failed its check


@dataclass
class UnitResult:
    scores: np.ndarray = None
    page_scores: np.ndarray = None
    status: int = UNIT_OK
    floor_excess: int = 0
    actions: np.ndarray = None
    pools: dict = field(default_factory=dict)


@dataclass
class PassParams:
    """Policy of one compaction pass (what the C-ABI's select parameters hold)."""
    budget_tokens: int = 0
    budget_bytes: int = 0
    n_sink: int = 4
    n_recent: int = 32
    page_size: int = 1
    renumber: bool = True
    quant_mode: int = QUANT_G32_BF16
    n_layer_groups: int = 3
    softmax_scale: float = 0.0
    rope_layout: str = "split"      # "split" halves or "interleaved" pairs
    rotary_dim: int = 0             # rotated leading dimensions (0 = all)


def select_unit(scores, page_scores, n_tokens, head_dim, params: PassParams,
                flags=None, tags=None, table=None, group=0):
    """Selection of one unit: returns (actions per token, floor_excess, status)."""
    T = n_tokens
    act = np.zeros(T, dtype=np.uint8)
    if params.budget_bytes > 0:
        floors = np.asarray(table, np.uint8)[np.asarray(tags, np.int64), group]
        return select_bytes(scores, floors, params.budget_bytes, params.n_sink,
                            params.n_recent, head_dim, params.quant_mode, flags)
    src = scores if params.page_size == 1 else page_scores
    kept, st = select_tokens(src, T, params.budget_tokens, params.n_sink, params.n_recent,
                             flags, params.page_size)
    act[kept] = ACT_BF16
    return act, 0, st


def compact_unit(k_bits, v_bits, pos_in, actions, params: PassParams, cos_tab, sin_tab,
                 ref_bits=None, ref_pos=None):
    """Gather, re-rotate and quantise the kept rows of one unit into pools.

    With a reference store (ref_bits [T][d] bf16 bits, ref_pos [T], -1 = no
    reference) kept keys are re-rotated by reference_rerotate and each pool
    carries its rows' references forward (PACE Sec. 3.2: moved with the slot
    when rows are compacted).
    """
    actions = np.asarray(actions)
    kept_all = np.nonzero(actions != ACT_RELEASE)[0]
    p_new_all = new_positions(kept_all, pos_in, params.renumber)
    new_of = dict(zip(kept_all.tolist(), p_new_all.tolist()))
    pools = {}
    for a in (ACT_INT4, ACT_INT8, ACT_BF16):
        idx = np.nonzero(actions == a)[0]
        pool = Pool(action=a, idx=idx)
        pool.orig_pos = np.asarray(pos_in)[idx].astype(np.int64)
        pool.pos = np.array([new_of[int(i)] for i in idx], dtype=np.int64)
        d = k_bits.shape[-1]
        kr = np.zeros((idx.size, d), dtype=np.uint16)
        if ref_pos is None:
            for n, (i, p, p2) in enumerate(zip(idx, pool.orig_pos, pool.pos)):
                kr[n] = rerotate_bits(k_bits[i], int(p), int(p2), cos_tab, sin_tab,
                                      params.rope_layout, params.rotary_dim)
        else:
            pool.k_ref = np.zeros((idx.size, d), dtype=np.uint16)
            pool.p_ref = np.full(idx.size, -1, dtype=np.int64)
            for n, (i, p, p2) in enumerate(zip(idx, pool.orig_pos, pool.pos)):
                kr[n], ref, pr, bad = reference_rerotate(k_bits[i], int(p), int(p2), ref_bits[i],
                                                         int(ref_pos[i]), cos_tab, sin_tab)
                if pr >= 0:
                    pool.k_ref[n], pool.p_ref[n] = ref, pr
                pool.ref_failures += int(bad)
        vr = np.asarray(v_bits)[idx]
        if a == ACT_BF16:
            pool.k, pool.v = kr, vr
        else:
            qmax = 7 if a == ACT_INT4 else 127
            kc, ks = quantize(bf16_bits_to_f32(kr), qmax, params.quant_mode)
            vc, vs = quantize(bf16_bits_to_f32(vr), qmax, params.quant_mode)
            if a == ACT_INT4:
                kc, vc = pack_int4(kc), pack_int4(vc)
            pool.k, pool.v, pool.k_scale, pool.v_scale = kc, vc, ks, vs
        pools[a] = pool
    return pools


def pool_rows_f32(pool: Pool, quant_mode: int):
    """Dequantised (K, V) rows of a pool as fp32."""
    if pool.action == ACT_BF16:
        return bf16_bits_to_f32(pool.k), bf16_bits_to_f32(pool.v)
    kc, vc = pool.k, pool.v
    if pool.action == ACT_INT4:
        kc, vc = unpack_int4(kc), unpack_int4(vc)
    return (dequantize(kc, pool.k_scale, quant_mode), dequantize(vc, pool.v_scale, quant_mode))


def decode_unit(q_bits, pools: dict, scale: float, quant_mode: int) -> np.ndarray:
    """Decode-step outputs [G][d] (fp64) of the G query heads of one unit."""
    ks, vs = [], []
    for a in (ACT_INT4, ACT_INT8, ACT_BF16):
        if a in pools and pools[a].idx.size:
            k, v = pool_rows_f32(pools[a], quant_mode)
            ks.append(k)
            vs.append(v)
    q = bf16_bits_to_f32(q_bits)
    if not ks:
        return np.zeros(q.shape)
    K = np.concatenate(ks)
    V = np.concatenate(vs)
    return np.stack([attend(q[h], K, V, scale) for h in range(q.shape[0])])


def run_unit(k_bits, v_bits, q_bits, pos_in, params: PassParams, cos_tab, sin_tab,
             bonus=None, acc=None, flags=None, tags=None, table=None, group=0,
             scores=None) -> UnitResult:
    """Score, select and compact one unit.  `scores` may be given to skip scoring."""
    T, d = k_bits.shape
    scale = params.softmax_scale or 1.0 / math.sqrt(d)
    res = UnitResult()
    res.scores = unit_scores(k_bits, q_bits, scale, bonus, acc) if scores is None \
        else np.asarray(scores, np.float32)
    if params.page_size > 1:
        res.page_scores = page_max(res.scores, params.page_size)
    res.actions, res.floor_excess, res.status = select_unit(
        res.scores, res.page_scores, T, d, params, flags, tags, table, group)
    if res.status != UNIT_OK:
        res.actions = np.zeros(T, dtype=np.uint8)
    res.pools = compact_unit(k_bits, v_bits, pos_in, res.actions, params, cos_tab, sin_tab)
    return res


def session_cycle(res_k, res_v, res_pos, new_k, new_v, q_bits, params: PassParams, limit: int,
                  cos_tab, sin_tab, scores=None):
    """One cycle of a bounded-position session of one unit (PACE Sec. 3.2,
    "Bounded positions" and "Choosing L"; Sec. 5.7 runs such sessions).

    The chunk's H rows are appended after the resident rows at the next
    physical positions (one past the resident rows' largest position).  The
    cache is scored by the window queries (its last W rows), selected and
    compacted back to the budget.  The compaction renumbers iff the position
    one past the cache's last row is within H of the limit L, i.e. the next
    chunk would otherwise reach L.  `scores` may be given (stage-wise
    parity).  Returns (k_bits, v_bits, pos) of the new resident rows (the
    bf16 pool) and the cycle's UnitResult.
    """
    res_pos = np.asarray(res_pos, np.int64)
    H = np.asarray(new_k).shape[0]
    start = int(res_pos.max()) + 1 if res_pos.size else 0
    pos_in = np.concatenate([res_pos, np.arange(start, start + H, dtype=np.int64)])
    k = np.concatenate([np.asarray(res_k, np.uint16), np.asarray(new_k, np.uint16)])
    v = np.concatenate([np.asarray(res_v, np.uint16), np.asarray(new_v, np.uint16)])
    prm = PassParams(**{**params.__dict__, "renumber": renumber_due(start + H, limit, H)})
    r = run_unit(k, v, q_bits, pos_in, prm, cos_tab, sin_tab, scores=scores)
    pool = r.pools[ACT_BF16]
    return pool.k, pool.v, pool.pos, r


def cache_bytes(n_tokens: int, n_layers: int, n_kv_heads: int, head_dim: int,
                action: int = ACT_BF16, quant_mode: int = QUANT_G32_BF16) -> int:
    """Bytes of K and V payload for n_tokens tokens across all layers and KV heads."""
    return n_tokens * n_layers * n_kv_heads * row_bytes(action, head_dim, quant_mode)


# ----------------------------------------------------------------------------
# CommitKV Sec. 3.2-3.3: deletion effect of event pages, lifecycle states,
# joint validation of completion candidates, protection of pending pages.
# One layer of one sequence: k, v [H_kv][T][d]; window queries q [H_q][W][d];
# query head h reads KV head h // (H_q / H_kv).  A page is an array of cache
# indices.  The W window queries are the last W cache entries (row w at index
# T - W + w) and see indices <= T - W + w, which is the page's p_i <= p for a
# cache kept in position order.
# ----------------------------------------------------------------------------

STATE_UNCERTAIN, STATE_COMPLETION, STATE_DORMANT, STATE_NEWLY_ACTIVE, STATE_STILL_ACTIVE = 0, 1, 2, 3, 4
STATE_NOT_COMPARED = 255


def window_attention(k, v, q, scale: float):
    """Attention weights a[r][j] and outputs o[r] of the window rows r = h W + w, fp64.

    CommitKV Sec. 3.2 ("Deletion effect for event page"): a_pj is the weight
    query p gives resident token j, o_p the head output.  k, v: [T][d] of one
    KV head; q: [G][W][d] of the query heads that read it.
    """
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    q = np.asarray(q, np.float64)
    T = k.shape[0]
    G, W, d = q.shape
    rows = q.reshape(G * W, d)
    last = np.tile(T - W + np.arange(W), G)
    z = rows @ k.T * scale
    z = np.where(np.arange(T)[None, :] <= last[:, None], z, -np.inf)
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    a = e / e.sum(axis=1, keepdims=True)
    return a, a @ v


def deletion_ratio(a_row, o_row, v, tokens) -> float:
    """Relative output change of one query row when `tokens` are deleted.

    CommitKV Eq. 6: o^{\\E} = (o - sum_{i in E} a_i v_i) / (1 - sum_{i in E} a_i),
    masked tokens having a_i = 0; Eq. 7's ratio ||o - o^{\\E}|| / ||o||.
    Readings for the cases Eq. 6 leaves undefined: if the deleted tokens
    hold all of the row's weight (1 - s <= 0) nothing is left to attend to
    and the change is +inf; if ||o|| = 0 the ratio is 0 when the output does
    not change and +inf otherwise.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    o = np.asarray(o_row, np.float64)
    if tokens.size == 0:
        return 0.0
    s = float(np.asarray(a_row, np.float64)[tokens].sum())
    u = np.asarray(a_row, np.float64)[tokens] @ np.asarray(v, np.float64)[tokens]
    if 1.0 - s <= 0.0:
        return math.inf
    o_del = (o - u) / (1.0 - s)
    num = float(np.linalg.norm(o - o_del))
    den = float(np.linalg.norm(o))
    if den == 0.0:
        return 0.0 if num == 0.0 else math.inf
    return num / den


def deletion_effect(k, v, q, scale: float, token_sets) -> np.ndarray:
    """R(E; Q) of CommitKV Eq. 7 for each token set E, fp64.

    k, v: [H_kv][T][d] of one layer; q: [H_q][W][d] (the window Q of Eq. 5).
    R_h(E; Q) is the largest ratio over the window queries of head h, and
    R(E; Q) the largest over the heads.
    """
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    q = np.asarray(q, np.float64)
    Hkv = k.shape[0]
    G = q.shape[0] // Hkv
    out = np.zeros(len(token_sets), dtype=np.float64)
    for g in range(Hkv):
        a, o = window_attention(k[g], v[g], q[g * G:(g + 1) * G], scale)
        for p, E in enumerate(token_sets):
            for r in range(a.shape[0]):
                out[p] = max(out[p], deletion_ratio(a[r], o[r], v[g], E))
    return out


def page_tokens(start: int, length: int) -> np.ndarray:
    """Cache indices of the contiguous event page [start, start + length)."""
    return np.arange(start, start + length, dtype=np.int64)


def percentile_ranks(values, compared) -> np.ndarray:
    """Percentile rank of each compared page among the compared pages.

    CommitKV Sec. 3.2 ("Influence comparison across a commit"), reading:
    P(E) = |{E' in E_c : R(E') < R(E)}| / |E_c|, the fraction of the
    comparison pages that E is more influential than (0 for pages outside E_c).
    """
    values = np.asarray(values, np.float64)
    compared = np.asarray(compared, dtype=bool)
    n = int(compared.sum())
    out = np.zeros(values.shape[0], dtype=np.float64)
    if n == 0:
        return out
    pool = values[compared]
    for i in np.nonzero(compared)[0]:
        out[i] = float((pool < values[i]).sum()) / n
    return out


@dataclass
class CommitThresholds:
    """CommitKV Sec. 4.1 settings."""
    tau_use: float = 0.05
    tau_dead: float = 0.01
    rho_use: float = 0.75
    rho_dead: float = 0.25
    tau_joint: float = 0.01


def lifecycle_states(r_minus, r_plus, compared, th: CommitThresholds):
    """Eq. 9 indicators and the Eq. 10 state of each page.

    Returns (state uint8, p_minus, p_plus); pages outside E_c get
    STATE_NOT_COMPARED.
    """
    r_minus = np.asarray(r_minus, np.float64)
    r_plus = np.asarray(r_plus, np.float64)
    compared = np.asarray(compared, dtype=bool)
    p_minus = percentile_ranks(r_minus, compared)
    p_plus = percentile_ranks(r_plus, compared)
    state = np.full(r_minus.shape[0], STATE_NOT_COMPARED, dtype=np.uint8)
    for i in np.nonzero(compared)[0]:
        hm = r_minus[i] >= th.tau_use and p_minus[i] >= th.rho_use
        lm = r_minus[i] <= th.tau_dead and p_minus[i] <= th.rho_dead
        hp = r_plus[i] >= th.tau_use and p_plus[i] >= th.rho_use
        lp = r_plus[i] <= th.tau_dead and p_plus[i] <= th.rho_dead
        if hm and lp:
            state[i] = STATE_COMPLETION
        elif lm and lp:
            state[i] = STATE_DORMANT
        elif lm and hp:
            state[i] = STATE_NEWLY_ACTIVE
        elif hm and hp:
            state[i] = STATE_STILL_ACTIVE
        else:
            state[i] = STATE_UNCERTAIN
    return state, p_minus, p_plus


def candidate_order(state, r_minus, r_plus) -> list:
    """Completion candidates by increasing R+, then decreasing R- (Sec. 3.3);
    remaining ties by lower page index (reading)."""
    cands = [i for i in range(len(state)) if state[i] == STATE_COMPLETION]
    return sorted(cands, key=lambda i: (float(r_plus[i]), -float(r_minus[i]), i))


def joint_validation(order, joint_effect, tau_joint: float):
    """Greedy retirement-set construction of Eq. 11.

    order: candidate pages in test order; joint_effect(list of pages) returns
    R+ of deleting all their tokens at once.  A candidate joins D_c when the
    joint effect of D_c with it stays <= tau_joint.  Returns (accepted pages,
    the joint effect evaluated for each candidate in order).
    """
    accepted, tried = [], []
    for p in order:
        r = float(joint_effect(accepted + [p]))
        tried.append(r)
        if r <= tau_joint:
            accepted.append(p)
    return accepted, tried


def commit_transition(k_plus, v_plus, q_plus, scale: float, pages, r_minus, r_plus, compared,
                      th: CommitThresholds = CommitThresholds()):
    """Lifecycle states and retirement set of one commit (Eqs. 8-11, Alg. 1).

    pages: list of (start, length) in the post-commit cache (k_plus, v_plus,
    window q_plus); r_minus, r_plus: per-page deletion effects of the two
    windows.  The joint effect of Eq. 11 deletes the union of the pages'
    tokens and evaluates Eqs. 6-7 on the post-commit window.
    Returns (state, retire uint8, joint effects tried).
    """
    state, _, _ = lifecycle_states(r_minus, r_plus, compared, th)
    order = candidate_order(state, r_minus, r_plus)

    def joint(sel):
        toks = np.concatenate([page_tokens(*pages[p]) for p in sel])
        return deletion_effect(k_plus, v_plus, q_plus, scale, [toks])[0]

    accepted, tried = joint_validation(order, joint, th.tau_joint)
    retire = np.zeros(len(pages), dtype=np.uint8)
    retire[accepted] = 1
    return state, retire, tried


def protect_pending(r_minus, page_len, pending, budget_tokens: int, max_pages: int) -> np.ndarray:
    """Pages protected while awaiting their post-commit measurement (Eq. 12).

    Pending pages are taken by decreasing R- (ties: lower index) while the
    protected token count stays <= B_N = floor(eta B) and the page count <=
    max_pages (CommitKV Sec. 4.1: 16); reading of "protected first until":
    the walk stops at the first page that does not fit.
    """
    r_minus = np.asarray(r_minus, np.float64)
    order = sorted((i for i in range(len(r_minus)) if pending[i]), key=lambda i: (-r_minus[i], i))
    out = np.zeros(len(r_minus), dtype=np.uint8)
    used = 0
    n = 0
    for i in order:
        if n + 1 > max_pages or used + int(page_len[i]) > budget_tokens:
            break
        out[i] = 1
        used += int(page_len[i])
        n += 1
    return out


def commit_flags(n_tokens: int, pages, retire, protect, flags=None) -> np.ndarray:
    """Selection flags of a checkpoint (Alg. 1, checkpoint step; Eq. 13).

    Tokens of protected pages become PROTECT (not EXCLUDE), tokens of retired
    pages that are not protected become EXCLUDE (not PROTECT); the decision
    replaces the page's earlier protect / exclude state, other tokens keep
    their flags.
    """
    out = np.zeros(n_tokens, np.uint8) if flags is None else np.array(flags, np.uint8, copy=True)
    for p, (s, ln) in enumerate(pages):
        if protect[p]:
            out[s:s + ln] = (out[s:s + ln] & ~np.uint8(FLAG_EXCLUDE)) | FLAG_PROTECT
        elif retire[p]:
            out[s:s + ln] = (out[s:s + ln] & ~np.uint8(FLAG_PROTECT)) | FLAG_EXCLUDE
    return out


# ----------------------------------------------------------------------------
# PASK App. B.5: the engine's attention over persistent (compacted, mixed
# precision), recent and current storage
# ----------------------------------------------------------------------------


def engine_attention(q_rows, q_pos, stores, scale: float) -> np.ndarray:
    """Outputs [R][d] (fp64) of R query rows over the union of the storages.

    PASK App. B.5: each visible key appears once across persistent, recent
    and current storage, and logical positions and the causal mask survive
    storage gaps: a key at position p_k is visible to a query at position
    p_q iff p_k <= p_q.  One softmax runs over all visible keys of all
    storages (the partitions share one normalisation, Eq. 15; they are not
    normalised and averaged separately).
    q_rows: [R][d]; q_pos: [R] or None (every key visible); stores: list of
    (K [n][d], V [n][d], positions [n] or None).  A row that sees no key
    outputs 0 (reading: empty partitions contribute nothing).
    """
    q = np.asarray(q_rows, np.float64)
    R, d = q.shape
    ks, vs, ps = [], [], []
    for k, v, pos in stores:
        k = np.asarray(k, np.float64).reshape(-1, d)
        if k.shape[0] == 0:
            continue
        ks.append(k)
        vs.append(np.asarray(v, np.float64).reshape(-1, d))
        ps.append(np.full(k.shape[0], np.iinfo(np.int64).min) if pos is None
                  else np.asarray(pos, np.int64))
    out = np.zeros((R, d), dtype=np.float64)
    if not ks:
        return out
    K, V, P = np.concatenate(ks), np.concatenate(vs), np.concatenate(ps)
    for r in range(R):
        vis = np.ones(K.shape[0], dtype=bool) if q_pos is None else P <= int(q_pos[r])
        if vis.any():
            out[r] = attend(q[r], K[vis], V[vis], scale)
    return out
