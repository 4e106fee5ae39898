"""Parity of the CUDA path (through the C-ABI) with the CPU oracle.

Each workload is run through kvc_score -> kvc_select ->
kvc_compact_rerotate_quant -> kvc_decode_attn on the GPU and checked unit by
unit against the oracle on the same seeded inputs:
  * scores            within rel 1e-2 (+1e-6 absolute floor)
  * selection         bit-exact when the oracle selects from the GPU's scores;
                      with the oracle's own scores the kept sets may differ only
                      at items within the score tolerance of the threshold
  * pools             bit-exact (bf16 keys after re-rotation, values, int8/int4
                      codes, scales, positions) for the same kept set
  * decode output     max-abs 2e-2
"""
import math

import numpy as np
import pytest
import torch

import oracle as o
import workloads as wl
from helpers import (bits, DECODE_ATOL, assert_pools_equal, assert_scores_close,
                     assert_selection_consistent, bits, kept_lists, params_of, unit_inputs,
                     unit_pools_from_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from budgeted_kv_cache_gb300 import build
    build.build()
    import budgeted_kv_cache_gb300 as lib
    lib.library()
    return lib


def run_pass(w, x):
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    p = pass_for_workload(w, inputs=x)
    p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"], x["rope_sin"],
          x.get("bonus"))
    p.decode(x["q_decode"])
    torch.cuda.synchronize()
    return p


def check_unit(w, x, p, u, e2e=True):
    """All parity checks of one unit."""
    ui = unit_inputs(w, x, u)
    prm = params_of(w)
    T, d = w.n_tokens, w.head_dim
    scale = 1.0 / math.sqrt(d)
    cos, sin = x["rope_cos"].cpu().numpy(), x["rope_sin"].cpu().numpy()
    table = x["action_table"].cpu().numpy() if "action_table" in x else None

    # scores
    ref_scores = o.unit_scores(ui["k"], ui["q"], scale, ui["bonus"])
    gpu_scores = p.scores[u].cpu().numpy()
    assert_scores_close(gpu_scores, ref_scores)
    gpu_pscores = None
    if w.page_size > 1:
        gpu_pscores = p.page_scores[u].cpu().numpy()
        assert np.array_equal(gpu_pscores, o.page_max(gpu_scores, w.page_size)), "page max"

    # selection from the GPU's own scores: bit-exact
    act, excess, st = o.select_unit(gpu_scores, gpu_pscores, T, d, prm, ui["flags"], ui["tags"],
                                    table, ui["group"])
    assert int(p.unit_status[u]) == st
    if w.byte_mode:
        assert int(p.floor_excess[u]) == excess
    gk = kept_lists(p, u)
    for a in (o.ACT_INT4, o.ACT_INT8, o.ACT_BF16):
        assert np.array_equal(gk[a], np.nonzero(act == a)[0]), f"unit {u} pool {a}"

    # compaction of that kept set: bit-exact
    ref_pools = o.compact_unit(ui["k"], ui["v"], ui["pos"], act, prm, cos, sin)
    assert_pools_equal(unit_pools_from_gpu(p, u, w), ref_pools)
    assert int(p.compact_status[u]) == 0

    # decode step over the pools
    ref_out = o.decode_unit(ui["qd"], ref_pools, scale, w.quant_mode)
    gpu_out = p.out[u * w.group:(u + 1) * w.group].float().cpu().numpy()
    assert np.max(np.abs(gpu_out - ref_out)) <= DECODE_ATOL

    # end to end: the oracle's own scores and selection
    if e2e and st == o.UNIT_OK and not w.byte_mode:
        ref_src = ref_scores if w.page_size == 1 else o.page_max(ref_scores, w.page_size)
        kept_ref, _ = o.select_tokens(ref_src, T, w.budget_tokens, w.n_sink, w.n_recent,
                                      ui["flags"], w.page_size)
        if w.page_size == 1:
            forced, _, _ = o.item_masks(T, w.n_sink, w.n_recent, ui["flags"])
            sel = np.setdiff1d(kept_ref, np.nonzero(forced)[0])
            thr = float(np.min(ref_src[sel])) if sel.size else math.inf
            assert_selection_consistent(ref_src, gk[o.ACT_BF16], kept_ref, thr)
        else:
            P = w.page_size
            gp = np.unique(gk[o.ACT_BF16] // P)
            rp = np.unique(kept_ref // P)
            sp, rpg = o.sink_recent_pages(T, P, w.n_sink, w.n_recent)
            forced, _, _ = o.item_masks(T // P, sp, rpg, ui["flags"])
            sel = np.setdiff1d(rp, np.nonzero(forced)[0])
            thr = float(np.min(ref_src[sel])) if sel.size else math.inf
            assert_selection_consistent(ref_src, gp, rp, thr)


# ------------------------------------------------------------------ small workloads

def small_workloads():
    c2 = wl.qwen3_8b_32k().replace(name="qwen_small", n_layers=1, n_kv_heads=2, n_q_heads=8,
                                   n_tokens=5000, budget_tokens=512, decode_pos=512)
    c3 = wl.pask_batch16().replace(name="pask_small", batch=2, n_layers=4, n_kv_heads=2,
                                   n_q_heads=8, n_tokens=2000,
                                   budget_bytes=(2000 * 512) // 3, decode_pos=2000)
    c4 = wl.commitkv_pages_128k().replace(name="commitkv_small", n_layers=1, n_kv_heads=2,
                                          n_q_heads=8, n_tokens=8192, budget_tokens=512,
                                          protect_pages=4, retire_pages=50, decode_pos=8192)
    c1 = wl.tiny()
    c1r = wl.tiny().replace(name="tiny_ragged_d128", head_dim=128, n_tokens=1000, budget_tokens=200)
    c3row = c3.replace(name="pask_small_rowfp16", quant_mode=wl.QUANT_ROW_FP16, head_dim=64,
                       budget_bytes=(2000 * 256) // 3)
    c2w32 = c2.replace(name="qwen_small_w32", window=32, n_tokens=3001, renumber=False,
                       bonus_spans=0)
    # byte mode with renumbering: kept keys re-rotated, then quantised to int8 / int4
    c3ren = c3.replace(name="pask_small_renumber", renumber=True)
    return [c1, c1r, c2, c2w32, c3, c3row, c3ren, c4]


@pytest.mark.parametrize("w", small_workloads(), ids=lambda w: w.name)
def test_parity_small(kvc, w):
    x = wl.make_inputs(w, device="cuda")
    p = run_pass(w, x)
    assert int(p.score_status.abs().sum()) == 0
    for u in range(w.n_units):
        check_unit(w, x, p, u)


def test_score_accumulate(kvc):
    w = wl.tiny().replace(n_tokens=700)
    x = wl.make_inputs(w, device="cuda")
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    p = pass_for_workload(w, inputs=x)
    bonus = torch.linspace(0, 1, w.n_tokens, device="cuda").view(1, -1).contiguous()
    p.score(x["k_cache"], x["q_window"], bonus)
    first = p.scores.clone()
    p.score(x["k_cache"], x["q_window"], bonus, accumulate=True)
    torch.cuda.synchronize()
    for u in range(w.n_units):
        ui = unit_inputs(w, x, u)
        ref = o.unit_scores(ui["k"], ui["q"], 1 / 8, bonus[0].cpu().numpy(),
                            first[u].cpu().numpy())
        assert_scores_close(p.scores[u].cpu().numpy(), ref)


@pytest.mark.parametrize("shift", [0.0, 0.5])
def test_score_with_caller_row_lse(kvc, shift):
    """Row statistics supplied by the caller (pass 1 skipped): the oracle's
    mass given those statistics, with the true statistics (shift 0) and with
    every row's statistic raised by `shift` (the mass scales by exp(-shift))."""
    w = wl.tiny().replace(n_tokens=1100)
    x = wl.make_inputs(w, device="cuda")
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    p = pass_for_workload(w, inputs=x)
    G, W = w.group, w.window
    scale = 1.0 / math.sqrt(w.head_dim)
    lse = np.zeros((w.n_units, G * W), np.float32)
    for u in range(w.n_units):
        ui = unit_inputs(w, x, u)
        lse[u] = o.window_row_lse(o.bf16_bits_to_f32(ui["k"]), o.bf16_bits_to_f32(ui["q"]),
                                  scale) + shift
    row_lse = torch.from_numpy(lse).cuda()
    p.score(x["k_cache"], x["q_window"], x.get("bonus"), row_lse=row_lse)
    torch.cuda.synchronize()
    for u in range(w.n_units):
        ui = unit_inputs(w, x, u)
        mass = o.window_mass_given_lse(o.bf16_bits_to_f32(ui["k"]), o.bf16_bits_to_f32(ui["q"]),
                                       scale, lse[u].astype(np.float64))
        ref = mass + (ui["bonus"].astype(np.float64) if ui["bonus"] is not None else 0.0)
        assert_scores_close(p.scores[u].cpu().numpy(), ref.astype(np.float32))


# ------------------------------------------------------------------ edge cases

def test_inactive_pass_is_bytewise_identity(kvc):
    """Budget = T and no renumbering: the bf16 pool equals the input cache."""
    w = wl.tiny().replace(n_tokens=640, budget_tokens=640, renumber=False)
    x = wl.make_inputs(w, device="cuda")
    p = run_pass(w, x)
    assert torch.equal(p.kept_count[2], torch.full((w.n_units,), 640, dtype=torch.int32, device="cuda"))
    assert torch.equal(p.pools.k_bf16.view(w.n_units, 640, -1), x["k_cache"].view(w.n_units, 640, -1))
    assert torch.equal(p.pools.v_bf16.view(w.n_units, 640, -1), x["v_cache"].view(w.n_units, 640, -1))


@pytest.mark.parametrize("idx", [2, 4], ids=["token_mode", "byte_mode"])
def test_host_resident_cache_is_read_in_place(kvc, idx):
    """Keys, values and positions in page-locked host memory: compaction reads
    the kept rows through the device mapping and stores the same bytes as
    from device memory; unregistered host memory is refused before a launch."""
    import dataclasses
    w = small_workloads()[idx]
    x = wl.make_inputs(w, device="cuda")
    p = run_pass(w, x)
    pools = [getattr(p.pools, f.name) for f in dataclasses.fields(p.pools)]
    pools = [t for t in pools if t is not None]
    for t in pools:
        t.view(torch.uint8).fill_(0x5A)
    p.compact(x["k_cache"], x["v_cache"], x["pos_in"], x["rope_cos"], x["rope_sin"])
    torch.cuda.synchronize()
    ref = [t.clone() for t in pools]
    for t in pools:
        t.view(torch.uint8).fill_(0x5A)
    hk, hv, hp = (x[n].cpu().pin_memory() for n in ("k_cache", "v_cache", "pos_in"))
    p.compact(hk, hv, hp, x["rope_cos"], x["rope_sin"])
    torch.cuda.synchronize()
    for a, b in zip(pools, ref):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert int(p.compact_status.abs().sum()) == 0
    with pytest.raises(kvc.KvcError) as e:
        p.compact(x["k_cache"], x["v_cache"].cpu(), x["pos_in"], x["rope_cos"], x["rope_sin"])
    assert e.value.code == 1


def test_over_budget_and_bad_flags(kvc):
    w = wl.tiny().replace(n_tokens=512, budget_tokens=16, n_sink=10, n_recent=10)
    x = wl.make_inputs(w, device="cuda")
    p = run_pass(w, x)
    assert torch.all(p.unit_status == o.UNIT_OVER_BUDGET)
    assert int(p.kept_count.abs().sum()) == 0
    w2 = wl.tiny().replace(n_tokens=512, budget_tokens=64)
    x2 = wl.make_inputs(w2, device="cuda")
    flags = torch.zeros(1, 512, dtype=torch.uint8, device="cuda")
    flags[0, 100] = o.FLAG_PROTECT | o.FLAG_EXCLUDE
    x2["flags"] = flags
    p2 = run_pass(w2, x2)
    assert torch.all(p2.unit_status == o.UNIT_BAD_FLAGS)


def test_ties_and_special_scores_select_bit_exact(kvc):
    """Selection alone on crafted scores: ties, -0, NaN, -inf, protect/exclude flags."""
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    rng = np.random.default_rng(5)
    w = wl.tiny().replace(n_tokens=3000, budget_tokens=700, n_layers=3)
    x = wl.make_inputs(w, device="cuda", with_tables=False)
    vals = np.array([0.0, -0.0, 1.0, 0.5, np.nan, -np.inf, 2.0, 1e-30], np.float32)
    scores = rng.choice(vals, size=(w.n_units, 3000)).astype(np.float32)
    flags = rng.choice([0, 0, 0, 0, 1, 2], size=(1, 3000)).astype(np.uint8)
    x["flags"] = torch.from_numpy(flags).cuda()
    p = pass_for_workload(w, inputs=x)
    p.select(scores=torch.from_numpy(scores).cuda())
    torch.cuda.synchronize()
    for u in range(w.n_units):
        kept, st = o.select_tokens(scores[u], 3000, 700, w.n_sink, w.n_recent, flags[0])
        assert int(p.unit_status[u]) == st
        assert np.array_equal(kept_lists(p, u)[o.ACT_BF16], kept)


def test_byte_mode_floor_excess(kvc):
    """Floors above the byte budget: excess recorded, nothing promoted."""
    w = wl.pask_batch16().replace(batch=1, n_layers=4, n_kv_heads=1, n_q_heads=4, n_tokens=1024,
                                  budget_bytes=1024 * 512 // 10)
    x = wl.make_inputs(w, device="cuda")
    x["action_table"] = torch.full_like(x["action_table"], o.ACT_INT8)
    p = run_pass(w, x)
    for u in range(w.n_units):
        check_unit(w, x, p, u, e2e=False)
        assert int(p.floor_excess[u]) > 0


# ------------------------------------------------------------------ full-size workloads

def _sample_units(w, n=3):
    U = w.n_units
    return sorted({0, U // 2, U - 1} if n >= 3 else {0, U - 1})


def _round_units(U, grid=152, extra=2):
    """One unit of every round of the scoring kernel's work items (whole units
    run round-robin over the CTAs), plus the last unit and a few more."""
    us = set(range(0, U, grid)) | {U - 1}
    us |= {min(U - 1, r * grid + grid // 2) for r in range(extra)}
    return sorted(us)


@pytest.mark.parametrize("make", [wl.qwen3_8b_32k, wl.pask_batch16, wl.commitkv_pages_128k],
                         ids=lambda f: f.__name__)
def test_parity_full_size_all_units(kvc, make):
    """Full-size workloads.  Every unit: the selection from the GPU's scores
    (bit-exact against the oracle's selection of the same scores).  Every
    unit (token and page mode) or 64 spread units (byte mode, 4,096 units):
    the compaction of that kept set (bit-exact).  One unit per round of the
    scoring kernel: scores within tolerance, decode, end-to-end consistency."""
    from helpers import oracle_compact_many
    w = make()
    x = wl.make_inputs(w, device="cuda")
    p = run_pass(w, x)
    assert int(p.score_status.abs().sum()) == 0
    assert int(p.compact_status.abs().sum()) == 0
    U, T, d = w.n_units, w.n_tokens, w.head_dim
    prm = params_of(w)
    table = x["action_table"].cpu().numpy() if "action_table" in x else None
    scores = p.scores.cpu().numpy()
    pscores = p.page_scores.cpu().numpy() if w.page_size > 1 else None
    status = p.unit_status.cpu().numpy()
    excess = p.floor_excess.cpu().numpy()
    cnt = p.kept_count.cpu().numpy()
    kept = p.kept_idx.cpu().numpy()
    flags = x["flags"].cpu().numpy() if "flags" in x else None
    tags = x["tags"].cpu().numpy() if "tags" in x else None
    acts = {}
    for u in range(U):
        b, l, g = wl.unit_coords(w, u)
        grp = o.layer_group(l, w.n_layers, w.n_layer_groups) if w.byte_mode else 0
        act, exc, st = o.select_unit(scores[u], pscores[u] if pscores is not None else None, T, d, prm,
                                     flags[b] if flags is not None else None,
                                     tags[b] if tags is not None else None, table, grp)
        assert int(status[u]) == st, f"unit {u}"
        if w.byte_mode:
            assert int(excess[u]) == exc, f"unit {u}"
        for a in (o.ACT_INT4, o.ACT_INT8, o.ACT_BF16):
            n = int(cnt[a - 1, u])
            assert np.array_equal(kept[a - 1, u, :n], np.nonzero(act == a)[0]), f"unit {u} pool {a}"
        acts[u] = act
    # compaction: the kept rows only (the oracle's positions are ranks among
    # the kept rows or their old positions, so a gathered sub-problem gives
    # the same pools up to the indices, which the selection check covered)
    cu = list(range(U)) if not w.byte_mode else list(range(0, U, U // 64))
    jobs = []
    for u in cu:
        b, l, g = wl.unit_coords(w, u)
        keep = np.nonzero(acts[u] != o.ACT_RELEASE)[0]
        kt = torch.from_numpy(keep).to("cuda")
        jobs.append((bits(x["k_cache"][b, l, g].index_select(0, kt)), bits(x["v_cache"][b, l, g].index_select(0, kt)),
                     x["pos_in"][u].index_select(0, kt).cpu().numpy(), acts[u][keep], prm))
    refs = oracle_compact_many(jobs, x["rope_cos"].cpu().numpy(), x["rope_sin"].cpu().numpy())
    for u, ref_pools in zip(cu, refs):
        got = unit_pools_from_gpu(p, u, w)
        for a, rp in ref_pools.items():
            rp.idx = got[a].idx if got[a].idx.size == rp.idx.size else rp.idx
        assert_pools_equal(got, ref_pools)
    for u in _round_units(U):
        check_unit(w, x, p, u)
    del p, x
    torch.cuda.empty_cache()


def test_parity_million_token_stage_a_sampled_units(kvc):
    """The 1,048,576-row session (8 layers, 64 units, 34 GB of K/V): one
    compaction to 2,048 renumbered rows, two units checked end to end."""
    w = wl.million_token_8l()
    x = wl.make_inputs(w, device="cuda")
    p = run_pass(w, x)
    assert int(p.score_status.abs().sum()) == 0
    assert int(p.compact_status.abs().sum()) == 0
    assert torch.equal(p.kept_count[2], torch.full((w.n_units,), w.budget_tokens, dtype=torch.int32,
                                                  device="cuda"))
    for u in _sample_units(w, n=2):
        check_unit(w, x, p, u)
    del p, x
    torch.cuda.empty_cache()
