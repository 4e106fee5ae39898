"""Selection of units longer than 32,768 items over many CTAs (token and page
mode): the kept lists, counts and statuses must equal, bit for bit, those of
the one-CTA-per-unit kernel on the same scores (the same rule: forced items,
then the top k candidates by score descending, index ascending), and the
oracle's selection on sampled units."""
import numpy as np
import pytest
import torch

import oracle as o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from budgeted_kv_cache_gb300 import build
    build.build()
    import budgeted_kv_cache_gb300 as lib
    lib.library()
    return lib


def _scores(kind, U, n, g):
    if kind == "random":
        return torch.rand((U, n), generator=g, device="cuda")
    if kind == "few_values":          # heavy ties
        return torch.randint(0, 7, (U, n), generator=g, device="cuda").float() * 0.25
    if kind == "all_equal":
        return torch.full((U, n), 0.5, device="cuda")
    if kind == "special":             # -0, +0, NaN, infinities, negatives
        s = torch.randn((U, n), generator=g, device="cuda")
        idx = torch.randint(0, n, (U, 64), generator=g, device="cuda")
        vals = torch.tensor([float("nan"), float("inf"), -float("inf"), -0.0, 0.0, -3.0, 1e-38, -1e-38],
                            device="cuda").repeat(8)
        s.scatter_(1, idx, vals.expand(U, -1).contiguous())
        return s
    raise ValueError(kind)


def _run(kvc, shape, pol, scores, ws):
    U = shape.batch * shape.n_layers * shape.n_kv_heads
    kept = torch.full((3, U, pol.capacity), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((3, U), -7, dtype=torch.int32, device="cuda")
    st = torch.full((U,), -7, dtype=torch.int32, device="cuda")
    kvc.kvc_select(shape, pol, scores, kept, cnt, st, None, ws, ws.numel() if ws is not None else 0)
    torch.cuda.synchronize()
    return kept, cnt, st


def _compare(kept_a, cnt_a, st_a, kept_b, cnt_b, st_b):
    assert torch.equal(st_a, st_b)
    assert torch.equal(cnt_a, cnt_b)
    for u in range(cnt_a.shape[1]):
        n = int(cnt_a[2, u])
        assert torch.equal(kept_a[2, u, :n], kept_b[2, u, :n]), f"unit {u}"


@pytest.mark.parametrize("kind", ["random", "few_values", "all_equal", "special"])
@pytest.mark.parametrize("budget", [2048, 40000])
@pytest.mark.parametrize("n", [70001, 70000], ids=["one_item_loads", "four_item_loads"])
def test_long_selection_token_mode_matches(kvc, kind, budget, n):
    """n = 70,001: items loaded one at a time (a unit's scores are not 16-byte
    aligned); n = 70,000: four at a time.  Both with a ragged last chunk."""
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    U = 6
    shape = kvc.make_shape(1, 3, 8, 2, 128, n)
    pol = kvc.Policy(budget_tokens=budget, n_sink=4, n_recent=128, capacity=budget, renumber=False)
    need = kvc.kvc_select_workspace_bytes(shape, pol)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    scores = _scores(kind, U, n, g)
    long_ = _run(kvc, shape, pol, scores, ws)
    one = _run(kvc, shape, pol, scores, None)
    _compare(*long_, *one)
    # the oracle on two units
    for u in (0, U - 1):
        sc = scores[u].cpu().numpy()
        kept, status = o.select_tokens(sc, n, budget, 4, 128, None, 1)
        assert status == int(long_[2][u])
        assert np.array_equal(long_[0][2, u, :int(long_[1][2, u])].cpu().numpy(), np.sort(kept))


def test_long_selection_page_mode_flags_and_over_budget(kvc):
    """Page mode (16-token pages) with PROTECT / EXCLUDE flags; one sequence's
    protected pages exceed the budget (OVER_BUDGET) and one carries a page
    flagged both ways (BAD_FLAGS)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    P, pages = 16, 40000
    T = P * pages
    shape = kvc.make_shape(3, 1, 4, 2, 128, T)        # 6 units, 3 sequences
    flags = torch.zeros((3, pages), dtype=torch.uint8, device="cuda")
    flags[0, torch.randint(2, pages - 8, (30,), generator=g, device="cuda")] = 1      # protect
    flags[0, torch.randint(2, pages - 8, (4000,), generator=g, device="cuda")] |= 2   # exclude
    flags[0][flags[0] == 3] = 2
    flags[1, 10:200] = 1                               # 190 protected pages > budget
    flags[2, 500] = 3                                  # both flags
    pol = kvc.Policy(budget_tokens=2048, n_sink=4, n_recent=64, page_size=P, capacity=2048,
                     renumber=False, flags=flags)
    ws = torch.empty(kvc.kvc_select_workspace_bytes(shape, pol), dtype=torch.uint8, device="cuda")
    scores = torch.rand((6, pages), generator=g, device="cuda")
    long_ = _run(kvc, shape, pol, scores, ws)
    one = _run(kvc, shape, pol, scores, None)
    _compare(*long_, *one)
    st = long_[2].cpu().numpy()
    assert (st[2:4] == kvc.UNIT_OVER_BUDGET).all() and (st[4:6] == kvc.UNIT_BAD_FLAGS).all()
    assert (st[0:2] == kvc.UNIT_OK).all()
    sc = scores[0].cpu().numpy()
    kept, status = o.select_tokens(sc, T, 2048, 4, 64, flags[0].cpu().numpy(), P)
    assert status == o.UNIT_OK
    assert np.array_equal(long_[0][2, 0, :int(long_[1][2, 0])].cpu().numpy(), np.sort(kept))


@pytest.mark.parametrize("kind", ["random", "few_values", "all_equal", "special"])
@pytest.mark.parametrize("n", [32768, 20001, 20000])
def test_one_cta_selection_matches_oracle(kvc, kind, n):
    """Units of at most 32,768 items (one CTA each): every unit's kept list and
    status against the oracle, with heavy ties (several candidates at the
    threshold key), all-equal scores and special values, full and ragged slabs;
    20,000 items take the bulk-copy load with a short last copy, 20,001 the
    per-thread loads."""
    g = torch.Generator(device="cuda")
    g.manual_seed(12)
    U = 6
    shape = kvc.make_shape(1, 3, 8, 2, 128, n)
    budget = 2048
    pol = kvc.Policy(budget_tokens=budget, n_sink=4, n_recent=128, capacity=budget, renumber=False)
    scores = _scores(kind, U, n, g)
    kept, cnt, st = _run(kvc, shape, pol, scores, None)
    for u in range(U):
        sc = scores[u].cpu().numpy()
        ref, status = o.select_tokens(sc, n, budget, 4, 128, None, 1)
        assert status == int(st[u])
        assert np.array_equal(kept[2, u, :int(cnt[2, u])].cpu().numpy(), np.sort(ref)), f"unit {u}"


@pytest.mark.parametrize("kind", ["random", "few_values", "all_equal", "special"])
@pytest.mark.parametrize("n", [32768, 20001, 9000])
def test_many_units_selection_matches_oracle(kvc, kind, n):
    """More units than SMs (304, two waves of CTAs): every unit's kept list and
    status against the oracle, with heavy ties, all-equal scores and special
    values, full, ragged and short units."""
    g = torch.Generator(device="cuda")
    g.manual_seed(13)
    shape = kvc.make_shape(1, 38, 32, 8, 128, n)
    U = 304
    budget = 2048
    pol = kvc.Policy(budget_tokens=budget, n_sink=4, n_recent=128, capacity=budget, renumber=False)
    scores = _scores(kind, U, n, g)
    kept, cnt, st = _run(kvc, shape, pol, scores, None)
    sc_all = scores.cpu().numpy()
    cnt_h, kept_h, st_h = cnt.cpu().numpy(), kept.cpu().numpy(), st.cpu().numpy()
    for u in range(U):
        ref, status = o.select_tokens(sc_all[u], n, budget, 4, 128, None, 1)
        assert status == int(st_h[u])
        assert np.array_equal(kept_h[2, u, :int(cnt_h[2, u])], np.sort(ref)), f"unit {u}"


@pytest.mark.parametrize("extra", [0, 1, -1], ids=["bin_taken_whole", "one_more_in_bin", "one_fewer_in_bin"])
@pytest.mark.parametrize("n", [32768, 20000])
def test_threshold_bin_boundaries_match_oracle(kvc, extra, n):
    """Scores in two binades: the candidates still to take (budget minus the
    forced sink and recent items), plus `extra`, lie in [2, 4) and the rest in
    [0.5, 1).  With extra = 0 the first radix level's threshold bin holds
    exactly the candidates to take, so the levels stop there and its lower
    edge is the threshold; with one more the search goes on inside the bin;
    with one fewer the last kept candidate is the largest of the lower bin."""
    rng = np.random.default_rng(14)
    U = 4
    n_sink, n_recent, budget = 4, 128, 2048
    shape = kvc.make_shape(1, 2, 8, 2, 128, n)
    pol = kvc.Policy(budget_tokens=budget, n_sink=n_sink, n_recent=n_recent, capacity=budget,
                     renumber=False)
    need = budget - n_sink - n_recent + extra
    host = rng.uniform(0.5, 0.99, size=(U, n)).astype(np.float32)
    for u in range(U):
        cand = n_sink + rng.permutation(n - n_sink - n_recent)[:need]
        host[u, cand] = rng.uniform(2.0, 3.99, size=need).astype(np.float32)
    scores = torch.from_numpy(host).cuda()
    kept, cnt, st = _run(kvc, shape, pol, scores, None)
    for u in range(U):
        sc = scores[u].cpu().numpy()
        ref, status = o.select_tokens(sc, n, budget, n_sink, n_recent, None, 1)
        assert status == int(st[u])
        got = kept[2, u, :int(cnt[2, u])].cpu().numpy()
        assert np.array_equal(got, np.sort(ref)), f"unit {u}"
        if extra == 0:                       # exactly the high-binade candidates and the forced items
            assert np.all(sc[got[(got >= n_sink) & (got < n - n_recent)]] >= 2.0)
