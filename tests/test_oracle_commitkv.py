"""Pins of the oracle's CommitKV functions (deletion effect, lifecycle states,
joint validation, pending-page protection) against brute force, closed forms
and hand-worked tables.  CPU only.

Source: "CommitKV: Lifecycle-Aware KV Cache Compression via Commit
Transitions for Multi-Turn Agents", Sec. 3.2 (Eqs. 5-10), Sec. 3.3 (Eqs.
11-13, Algorithm 1) and Sec. 4.1 (thresholds).
"""
import math

import numpy as np
import pytest

import oracle as o


def _brute_effect(k, v, q, scale, tokens):
    """Eq. 7 by deleting the tokens and re-running the softmax from scratch
    (no use of Eq. 6): largest relative output change over heads and rows."""
    Hkv, T, d = k.shape
    Hq, W, _ = q.shape
    G = Hq // Hkv
    gone = np.zeros(T, dtype=bool)
    gone[np.asarray(tokens, dtype=np.int64)] = True
    best = 0.0
    for h in range(Hq):
        g = h // G
        for w in range(W):
            vis = np.arange(T) <= T - W + w
            z = k[g] @ q[h, w] * scale
            full = np.exp(z[vis] - z[vis].max())
            o_full = (full / full.sum()) @ v[g][vis]
            keep = vis & ~gone
            zk = z[keep]
            ek = np.exp(zk - zk.max())
            o_keep = (ek / ek.sum()) @ v[g][keep]
            best = max(best, np.linalg.norm(o_full - o_keep) / np.linalg.norm(o_full))
    return best


def _case(seed, Hkv=2, G=2, W=4, T=40, d=16):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((Hkv, T, d))
    v = rng.standard_normal((Hkv, T, d))
    q = rng.standard_normal((Hkv * G, W, d))
    return k, v, q, 1.0 / math.sqrt(d)


# --------------------------------------------------------------------------- Eqs. 6-7

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_eq6_matches_deleting_and_renormalising(seed):
    k, v, q, scale = _case(seed)
    T, W = k.shape[1], q.shape[1]
    pages = [o.page_tokens(0, 4), o.page_tokens(10, 7), o.page_tokens(T - W - 2, 5),
             o.page_tokens(T - 3, 3)]                    # the last one is partly masked
    got = o.deletion_effect(k, v, q, scale, pages)
    for p, E in enumerate(pages):
        assert got[p] == pytest.approx(_brute_effect(k, v, q, scale, E), rel=1e-10)


def test_joint_deletion_of_a_page_union_matches_brute_force():
    k, v, q, scale = _case(7)
    union = np.concatenate([o.page_tokens(3, 5), o.page_tokens(20, 6)])
    got = o.deletion_effect(k, v, q, scale, [union])[0]
    assert got == pytest.approx(_brute_effect(k, v, q, scale, union), rel=1e-10)


def test_gqa_rows_read_their_own_kv_head():
    # KV head 1's page keys align with query head 2 only: the effect comes
    # from that head; a mapping other than h // G would miss it.
    k, v, q, scale = _case(3, Hkv=2, G=2, W=2, T=32, d=8)
    k[1, 5:9] = 4.0 * q[2, 0] / np.linalg.norm(q[2, 0])
    v[1, 5:9] += 5.0
    got = o.deletion_effect(k, v, q, scale, [o.page_tokens(5, 4)])[0]
    assert got == pytest.approx(_brute_effect(k, v, q, scale, o.page_tokens(5, 4)), rel=1e-10)
    assert got > 0.5


def test_uniform_attention_closed_form():
    # q = 0: every visible token gets weight 1/n.  Values e1 outside the page,
    # e2 inside (m tokens): o = ((n-m) e1 + m e2) / n, o without the page = e1,
    # so R = m sqrt(2) / sqrt((n-m)^2 + m^2).
    T, d = 8, 2
    k = np.random.default_rng(0).standard_normal((1, T, d))
    v = np.zeros((1, T, d))
    v[0, :, 0] = 1.0
    page = [2, 5]
    v[0, page] = [0.0, 1.0]
    q1 = np.zeros((1, 1, d))
    assert o.deletion_effect(k, v, q1, 1.0, [page])[0] == pytest.approx(1 / math.sqrt(5), rel=1e-12)
    # W = 2: row 0 sees n = 7 (2 sqrt2 / sqrt29), row 1 sees n = 8 (1 / sqrt5)
    q2 = np.zeros((1, 2, d))
    assert o.deletion_effect(k, v, q2, 1.0, [page])[0] == pytest.approx(
        2 * math.sqrt(2) / math.sqrt(29), rel=1e-12)
    # a page with its last token after row 0: row 0 sees one of its tokens
    # (sqrt2 / sqrt37), row 1 both (2 sqrt2 / sqrt40)
    v2 = np.zeros((1, T, d))
    v2[0, :, 0] = 1.0
    v2[0, [6, 7]] = [0.0, 1.0]
    assert o.deletion_effect(k, v2, q2, 1.0, [[6, 7]])[0] == pytest.approx(
        2 * math.sqrt(2) / math.sqrt(40), rel=1e-12)
    assert o.deletion_ratio(np.r_[np.full(7, 1 / 7), 0.0], v2[0, :7].mean(axis=0), v2[0], [6, 7]) \
        == pytest.approx(math.sqrt(2) / math.sqrt(37), rel=1e-12)


def test_undefined_cases_follow_the_stated_reading():
    k, v, q, scale = _case(5, Hkv=1, G=1, W=1, T=12, d=4)
    assert o.deletion_effect(k, v, q, scale, [np.arange(12)])[0] == math.inf   # nothing left
    assert o.deletion_effect(k, v, q, scale, [np.arange(0)])[0] == 0.0       # empty page
    zero_v = np.zeros_like(v)                                                # o = 0, no change
    assert o.deletion_effect(k, zero_v, q, scale, [np.arange(3)])[0] == 0.0


def test_effect_is_invariant_to_value_scale():
    k, v, q, scale = _case(11)
    pages = [o.page_tokens(4, 8), o.page_tokens(25, 3)]
    a = o.deletion_effect(k, v, q, scale, pages)
    b = o.deletion_effect(k, 3.7 * v, q, scale, pages)
    np.testing.assert_allclose(a, b, rtol=1e-12)


# --------------------------------------------------------------------------- Eqs. 8-10

def test_percentile_ranks_hand_example():
    r = [0.5, 0.1, 0.3, 0.3, 9.0]
    got = o.percentile_ranks(r, [1, 1, 1, 1, 0])
    np.testing.assert_array_equal(got, [3 / 4, 0.0, 1 / 4, 1 / 4, 0.0])


def test_lifecycle_states_hand_table():
    # Eight compared pages (percentile = number of compared pages below / 8)
    # and one page outside E_c whose values must not move any percentile.
    r_minus = [0.20, 0.30, 0.005, 0.002, 0.04, 0.003, 0.06, 0.001, 100.0]
    r_plus = [0.001, 0.5, 0.002, 0.3, 0.003, 0.0015, 0.2, 0.004, 0.0]
    compared = [1] * 8 + [0]
    # P-: p7 0, p3 1/8, p5 2/8, p2 3/8, p4 4/8, p6 5/8, p0 6/8, p1 7/8
    #   H- (R >= .05, P >= .75): p0, p1;  L- (R <= .01, P <= .25): p7, p3, p5
    # P+: p0 0, p5 1/8, p2 2/8, p4 3/8, p7 4/8, p6 5/8, p3 6/8, p1 7/8
    #   H+: p3, p1;  L+: p0, p5, p2
    want = [o.STATE_COMPLETION, o.STATE_STILL_ACTIVE, o.STATE_UNCERTAIN, o.STATE_NEWLY_ACTIVE,
            o.STATE_UNCERTAIN, o.STATE_DORMANT, o.STATE_UNCERTAIN, o.STATE_UNCERTAIN,
            o.STATE_NOT_COMPARED]
    state, pm, pp = o.lifecycle_states(r_minus, r_plus, compared, o.CommitThresholds())
    np.testing.assert_array_equal(state, want)
    assert pm[0] == 0.75 and pp[3] == 0.75


def test_thresholds_are_inclusive():
    # R = tau_use exactly and P = rho_use exactly count as high (Eq. 9 uses >=)
    th = o.CommitThresholds()
    r_minus = [0.05, 0.0, 0.0, 0.0]
    r_plus = [0.01, 0.02, 0.02, 0.02]
    state, pm, pp = o.lifecycle_states(r_minus, r_plus, [1, 1, 1, 1], th)
    assert pm[0] == 0.75 and pp[0] == 0.0
    assert state[0] == o.STATE_COMPLETION


# --------------------------------------------------------------------------- Eq. 11

def test_candidate_order():
    st = [o.STATE_COMPLETION] * 6 + [o.STATE_DORMANT]
    r_plus = [0.004, 0.002, 0.002, 0.001, 0.003, 0.003, 0.0]
    r_minus = [0.1, 0.2, 0.3, 0.1, 0.1, 0.1, 0.9]
    assert o.candidate_order(st, r_minus, r_plus) == [3, 2, 1, 4, 5, 0]


def test_greedy_joint_validation_hand_examples():
    eff = {3: 0.002, 2: 0.003, 1: 0.004, 0: 0.0035}
    acc, tried = o.joint_validation([3, 2, 1, 0], lambda s: sum(eff[p] for p in s), 0.01)
    assert acc == [3, 2, 1]
    np.testing.assert_allclose(tried, [0.002, 0.005, 0.009, 0.0125])
    # a rejected candidate does not stop the scan
    eff2 = {0: 0.006, 1: 0.005, 2: 0.003}
    acc2, _ = o.joint_validation([0, 1, 2], lambda s: sum(eff2[p] for p in s), 0.01)
    assert acc2 == [0, 2]


def test_commit_transition_accepts_only_sets_within_the_joint_bound():
    k, v, q, scale = _case(21, Hkv=2, G=2, W=4, T=512, d=16)
    pages = [(s, 8) for s in range(0, 500, 20)]
    toks = [o.page_tokens(*p) for p in pages]
    r_plus = o.deletion_effect(k, v, q, scale, toks)
    # pages below the median R+ are low after the commit; give them a high
    # pre-commit effect so that they are completion candidates, and set the
    # joint bound so that some but not all of them fit together
    low = r_plus <= np.median(r_plus)
    r_minus = np.where(low, 1.0, 0.0) + np.arange(len(pages)) * 1e-3
    tau_joint = 2.2 * r_plus[low].min()
    th = o.CommitThresholds(tau_use=0.5, tau_dead=float(np.median(r_plus)), rho_use=0.5,
                            rho_dead=0.5, tau_joint=float(tau_joint))
    state, retire, tried = o.commit_transition(k, v, q, scale, pages, r_minus, r_plus,
                                               np.ones(len(pages)), th)
    cands = o.candidate_order(state, r_minus, r_plus)
    assert len(cands) >= 3 and 1 <= retire.sum() < len(cands)
    accepted = []
    for p, r in zip(cands, tried):
        union = np.concatenate([toks[i] for i in accepted + [p]])
        assert r == pytest.approx(_brute_effect(k, v, q, scale, union), rel=1e-9)
        if r <= th.tau_joint:
            accepted.append(p)
    assert sorted(accepted) == list(np.nonzero(retire)[0])


# --------------------------------------------------------------------------- Eq. 12, Eq. 13

def test_protect_pending_hand_examples():
    r = np.linspace(1.0, 0.05, 20)
    lens = np.full(20, 16)
    assert list(np.nonzero(o.protect_pending(r, lens, np.ones(20), 256, 16))[0]) == list(range(16))
    assert list(np.nonzero(o.protect_pending(r, lens, np.ones(20), 100, 16))[0]) == list(range(6))
    # the walk stops at the first page that does not fit
    got = o.protect_pending([0.3, 0.2, 0.1], [16, 30, 4], [1, 1, 1], 24, 16)
    assert list(got) == [1, 0, 0]
    # pages that are not pending are never protected; ties go to the lower index
    got = o.protect_pending([0.9, 0.5, 0.5, 0.5], [4, 4, 4, 4], [0, 1, 1, 1], 8, 16)
    assert list(got) == [0, 1, 1, 0]


def test_commit_flags():
    pages = [(0, 4), (4, 4), (8, 4)]
    flags = np.zeros(14, np.uint8)
    flags[5] = o.FLAG_PROTECT
    flags[9] = o.FLAG_EXCLUDE
    flags[13] = o.FLAG_PROTECT
    got = o.commit_flags(14, pages, retire=[1, 1, 0], protect=[0, 0, 1], flags=flags)
    want = np.array([2, 2, 2, 2, 2, 2, 2, 2, 1, 1, 1, 1, 0, 1], np.uint8)
    np.testing.assert_array_equal(got, want)
