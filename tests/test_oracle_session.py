"""Pins of the oracle's bounded-position session (PACE Sec. 3.2, "Bounded
positions" and "Choosing L"; Sec. 5.7 runs such sessions to a million
tokens), checked against what the page fixes rather than against the
oracle's own arithmetic:

  * positions never reach the limit L, whatever the number of cycles;
  * with renumbering never due (a large L) the session is inactive: every
    resident row is byte-identical to the row appended for it, at its
    original physical position;
  * every kept key stays the rotation of its pre-RoPE key at its current
    position (Prop. 1), within two bf16 roundings per renumber it went
    through -- which fails if the session hands the rotation the wrong old
    or new position (an off-by-one in where the chunk is appended, swapped
    positions, a renumber applied twice).
"""
import numpy as np
import pytest

import oracle as o

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

D, THETA = 16, 1e4
B, H, W = 16, 32, 8          # budget, chunk, window


def _tables(max_pos):
    half = D // 2
    inv = THETA ** (-2.0 * np.arange(half) / D)
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def _session(limit, cycles, seed=0):
    """Run the oracle session; return per cycle (resident pool, pre-RoPE keys of
    its rows, cycles each row has lived through, renumber flag)."""
    rng = np.random.default_rng(seed)
    cos, sin = _tables(limit + 4 * H)
    prm = o.PassParams(budget_tokens=B, n_sink=2, n_recent=4, renumber=True)
    pre0 = rng.standard_normal((B, D))
    pos = np.arange(B)
    k = o.f32_to_bf16_bits(o.rope_rotate(pre0, pos, D, THETA).astype(np.float32))
    v = o.f32_to_bf16_bits(rng.standard_normal((B, D)).astype(np.float32))
    pre, born = pre0, np.zeros(B, dtype=np.int64)      # pre-RoPE key and birth cycle per row
    out = []
    for c in range(cycles):
        start = int(pos.max()) + 1
        new_pos = np.arange(start, start + H)
        new_pre = rng.standard_normal((H, D))
        nk = o.f32_to_bf16_bits(o.rope_rotate(new_pre, new_pos, D, THETA).astype(np.float32))
        nv = o.f32_to_bf16_bits(rng.standard_normal((H, D)).astype(np.float32))
        qpre = rng.standard_normal((2, W, D))             # two query heads share the KV head
        q = o.f32_to_bf16_bits(o.rope_rotate(qpre.reshape(-1, D), np.tile(new_pos[-W:], 2), D,
                                             THETA).astype(np.float32)).reshape(2, W, D)
        k, v, pos, r = o.session_cycle(k, v, pos, nk, nv, q, prm, limit, cos, sin)
        idx = r.pools[o.ACT_BF16].idx                     # kept rows of the cache (resident + chunk)
        all_pre = np.concatenate([pre, new_pre])
        all_born = np.concatenate([born, np.full(H, c)])   # renumbered from this cycle on
        pre, born = all_pre[idx], all_born[idx]
        out.append(dict(k=k, v=v, pos=pos, pre=pre, born=born, idx=idx,
                        orig=r.pools[o.ACT_BF16].orig_pos))
    return out


def test_positions_stay_below_the_limit():
    limit = o.smallest_pow2_limit(B, 0, H)              # 64 for B = 16, H = 32
    assert limit == 64
    steps = _session(limit, cycles=40)
    for s in steps:
        assert s["pos"].max() < limit and s["pos"].min() >= 0
        assert s["k"].shape == (B, D)
        assert np.all(np.diff(s["pos"]) > 0)            # ascending, distinct
    # B + H + H > L: the next chunk would always pass the limit, so every cycle renumbers
    assert all(np.array_equal(s["pos"], np.arange(B)) for s in steps)


def test_inactive_session_is_token_identical():
    """PACE Sec. 5.7: when renumbering is never due the rows are untouched."""
    steps = _session(limit=1 << 20, cycles=12, seed=1)
    for c, s in enumerate(steps):
        # kept positions are the rows' original physical positions: the
        # newest chunk's recent rows end at position B + (c + 1) H - 1
        assert np.array_equal(s["pos"], s["orig"])
        assert s["pos"].max() == B + (c + 1) * H - 1
    # and the stored keys are the appended bits: rotate each row's pre-RoPE key
    # at its physical position and round once, as when it was appended
    s = steps[-1]
    exp = o.f32_to_bf16_bits(o.rope_rotate(s["pre"], s["pos"], D, THETA).astype(np.float32))
    assert np.array_equal(s["k"], exp)


def test_kept_keys_follow_their_positions_within_two_roundings_per_renumber():
    """Prop. 1: re-rotating a stored key from p to p' matches rotating its
    pre-RoPE key to p' up to the stored key's roundings (two per renumber)."""
    limit = 64
    steps = _session(limit, cycles=25, seed=2)
    u = 2.0 ** -8                                        # bf16 unit roundoff
    for c, s in enumerate(steps):
        exact = o.rope_rotate(s["pre"], s["pos"], D, THETA)
        err = np.linalg.norm(o.bf16_bits_to_f32(s["k"]) - exact, axis=1)
        lived = c + 1 - s["born"]                         # renumbers each row went through
        bound = (2 * lived + 1) * u * np.linalg.norm(s["pre"], axis=1) * 1.01
        assert np.all(err <= bound)
    # a plausible slip (rotating to p' + 1) is far outside that bound
    s = steps[5]
    wrong = o.rope_rotate(s["pre"], s["pos"] + 1, D, THETA)
    err = np.linalg.norm(o.bf16_bits_to_f32(s["k"]) - wrong, axis=1)
    assert np.median(err / np.linalg.norm(s["pre"], axis=1)) > 0.05


def test_attention_logits_depend_only_on_relative_position_across_cycles():
    """A query at position m sees a kept key at p' with the same logit as the
    original pair at m - (p' - p) ... i.e. q . k depends only on m - p' (PACE
    Sec. 3.2 relative-position identity), up to the roundings above."""
    steps = _session(64, cycles=6, seed=3)
    rng = np.random.default_rng(9)
    qpre = rng.standard_normal(D)
    s = steps[-1]
    m = 40
    got = o.rope_rotate(qpre[None], np.array([m]), D, THETA)[0] @ o.bf16_bits_to_f32(s["k"]).T
    exp = np.array([o.rope_rotate(qpre[None], np.array([m - p]), D, THETA)[0] @ s["pre"][i]
                    for i, p in enumerate(s["pos"])])
    scale = np.linalg.norm(qpre) * np.linalg.norm(s["pre"], axis=1)
    assert np.all(np.abs(got - exp) <= 0.05 * scale)


@pytest.mark.parametrize("limit", [64, 128, 256, 1 << 20])
def test_session_schedule_follows_the_oracle(limit):
    """The library session's host-side schedule (`cycle_schedule`: where each
    chunk starts and whether its compaction renumbers) against the oracle's
    session run cycle by cycle: the same renumber decisions, and the next
    chunk starts one past the largest resident position the oracle keeps.
    Limits that renumber every cycle, every few cycles and never."""
    from budgeted_kv_cache_gb300.session import cycle_schedule
    steps = _session(limit, cycles=24, seed=3)
    next_pos = B                                       # the resident rows start at 0..B-1
    for s in steps:
        ren, end, nxt = cycle_schedule(next_pos, B, H, limit)
        renumbered = not np.array_equal(s["pos"], s["orig"])
        assert ren == renumbered or (ren and np.array_equal(s["orig"], np.arange(B)))
        assert end == next_pos + H and s["pos"].max() < limit
        assert nxt == int(s["pos"].max()) + 1
        next_pos = nxt


def test_session_schedule_keeps_positions_below_the_limit():
    """From resident rows at 0..budget-1, the schedule's caches never hold a
    position at or past the limit, for every limit that holds one cache
    (budget + chunk <= L), and it renumbers exactly when the next chunk would
    otherwise reach the limit."""
    from budgeted_kv_cache_gb300.session import cycle_schedule
    # the next cache would end exactly at L (allowed) or one past it (renumber)
    assert cycle_schedule(B, B, H, B + 2 * H) == (False, B + H, B + H)
    assert cycle_schedule(B, B, H, B + 2 * H - 1) == (True, B + H, B)
    assert cycle_schedule(B + H, B, H, B + 3 * H) == (False, B + 2 * H, B + 2 * H)
    assert cycle_schedule(B + H, B, H, B + 3 * H - 1) == (True, B + 2 * H, B)
    for limit in range(B + H, B + 12 * H + 1, 7):
        next_pos = B
        for _ in range(50):
            ren, end, nxt = cycle_schedule(next_pos, B, H, limit)
            assert end <= limit                          # the cache's rows sit below L
            assert ren == (end + H > limit)              # the next chunk would pass L
            next_pos = nxt
