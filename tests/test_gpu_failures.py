"""Failure detection and determinism on the GPU, without faulting it.

Data-dependent failures are written per unit to `unit_status`; no kernel
traps.  A device wait that cannot complete gives up after its bound (2 s):
the test stalls one unit's cross-CTA wait through the library's test hook
(its completion target is raised to a count nothing reaches), and checks
that exactly that unit reports KVC_UNIT_TIMEOUT, that the other unit's
scores are correct, and that the GPU context stays usable.  Determinism: the
same inputs twice give identical bytes.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as o
import workloads as wl
from helpers import assert_scores_close, bits, unit_inputs

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


def _pass(w):
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    x = wl.make_inputs(w, device="cuda")
    return pass_for_workload(w, inputs=x), x


def test_a_wait_that_cannot_complete_reports_timeout(kvc):
    w = wl.tiny()                                      # 2 units, window rows on the tensor cores
    p, x = _pass(w)
    kvc.kvc_set_overrides(score_stall_unit=1)
    try:
        p.score(x["k_cache"], x["q_window"], x.get("bonus"))
        torch.cuda.synchronize()
    finally:
        kvc.kvc_set_overrides(reset=True)
    status = p.score_status.cpu().numpy()
    assert status[1] == kvc.UNIT_TIMEOUT and status[0] == kvc.UNIT_OK
    ui = unit_inputs(w, x, 0)
    ref = o.unit_scores(ui["k"], ui["q"], 1 / math.sqrt(w.head_dim), ui["bonus"])
    assert_scores_close(p.scores[0].cpu().numpy(), ref)
    # the context is still usable: the same call without the stall succeeds
    p.score_status.zero_()
    p.score(x["k_cache"], x["q_window"], x.get("bonus"))
    torch.cuda.synchronize()
    assert int(p.score_status.abs().sum()) == 0


def test_a_selection_wait_that_cannot_complete_reports_timeout(kvc):
    """The selection's wait for a unit's scores (bulk copies into shared
    memory, completing on an mbarrier) gives up after its bound: the test hook
    makes unit 1 wait for 16 bytes more than its copy brings.  That unit
    reports KVC_UNIT_TIMEOUT and keeps nothing; unit 0's kept list equals the
    oracle's; the next call without the hook selects both units."""
    w = wl.tiny()                                      # 2 units of 1,024 items: bulk-copied scores
    p, x = _pass(w)
    p.score(x["k_cache"], x["q_window"], x.get("bonus"))
    torch.cuda.synchronize()
    p.kept_count.fill_(-7)
    kvc.kvc_set_overrides(select_stall_unit=1)
    try:
        p.select()
        torch.cuda.synchronize()
    finally:
        kvc.kvc_set_overrides(reset=True)
    st = p.unit_status.cpu().numpy()
    cnt = p.kept_count.cpu().numpy()
    assert st[1] == kvc.UNIT_TIMEOUT and st[0] == kvc.UNIT_OK
    assert (cnt[:, 1] == 0).all()
    sc = p.scores.cpu().numpy()
    ref, status = o.select_tokens(sc[0], w.n_tokens, w.budget_tokens, w.n_sink, w.n_recent, None, 1)
    assert status == o.UNIT_OK
    assert np.array_equal(p.kept_idx[2, 0, :int(cnt[2, 0])].cpu().numpy(), np.sort(ref))
    # the context is still usable: the same call without the hook selects both units
    p.select()
    torch.cuda.synchronize()
    assert int(p.unit_status.abs().sum()) == 0
    cnt = p.kept_count.cpu().numpy()
    ref1, _ = o.select_tokens(sc[1], w.n_tokens, w.budget_tokens, w.n_sink, w.n_recent, None, 1)
    assert np.array_equal(p.kept_idx[2, 1, :int(cnt[2, 1])].cpu().numpy(), np.sort(ref1))


def test_kept_index_out_of_range_marks_its_unit(kvc):
    w = wl.tiny()
    p, x = _pass(w)
    p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"], x["rope_sin"],
          x.get("bonus"))
    torch.cuda.synchronize()
    assert int(p.compact_status.abs().sum()) == 0
    p.kept_idx[2, 0, 5] = w.n_tokens + 5               # bf16 pool of unit 0
    p.compact(x["k_cache"], x["v_cache"], x["pos_in"], x["rope_cos"], x["rope_sin"])
    torch.cuda.synchronize()
    st = p.compact_status.cpu().numpy()
    assert st[0] == o.UNIT_BAD_INDEX and st[1] == o.UNIT_OK


def test_kept_count_beyond_capacity_is_clamped_and_marked(kvc):
    """A kept count past the capacity (or negative) in caller memory: compaction
    marks the unit, writes no row past its capacity, and the decode and engine
    kernels read no row past the pools."""
    w = wl.tiny().replace(n_layers=2)                   # 4 units
    p, x = _pass(w)
    p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"], x["rope_sin"],
          x.get("bonus"))
    torch.cuda.synchronize()
    cap = p.policy.capacity
    good_k = p.pools.k_bf16.clone()
    ref_out = p.decode(x["q_decode"]).clone()
    kc = p.kept_count.clone()
    p.kept_count[kvc.POOL_BF16, 1] = cap + 1
    p.kept_count[kvc.POOL_BF16, 2] = -3
    p.compact_status.zero_()
    p.pools.k_bf16.fill_(0)
    p.compact(x["k_cache"], x["v_cache"], x["pos_in"], x["rope_cos"], x["rope_sin"])
    torch.cuda.synchronize()
    st = p.compact_status.cpu().numpy()
    assert st[1] == o.UNIT_BAD_INDEX and st[2] == o.UNIT_BAD_INDEX
    assert st[0] == o.UNIT_OK and st[3] == o.UNIT_OK
    # units 0 and 3 are compacted as before; unit 2 writes nothing; unit 1
    # writes at most its capacity (its own slots only)
    for u in (0, 3):
        assert torch.equal(p.pools.k_bf16[u].view(torch.int16), good_k[u].view(torch.int16))
    assert int(p.pools.k_bf16[2].view(torch.int16).abs().sum()) == 0
    # decode over the clamped counts: units with valid counts are unchanged
    p.pools.k_bf16.copy_(good_k)
    out = p.decode(x["q_decode"]).clone()
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    G = w.group
    for u in (0, 3):
        assert torch.equal(out[u * G:(u + 1) * G], ref_out[u * G:(u + 1) * G])
    assert int(out[2 * G:3 * G].float().abs().sum()) == 0     # no rows: zeros
    p.kept_count.copy_(kc)


def test_rope_table_shorter_than_the_positions_marks_the_units(kvc):
    w = wl.tiny()                                      # renumbering: kept keys rotate
    p, x = _pass(w)
    p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"], x["rope_sin"],
          x.get("bonus"))
    cap = p.policy.capacity
    # shorter than the new positions (0 .. capacity - 1): refused before any launch
    with pytest.raises(kvc.KvcError) as e:
        p.compact(x["k_cache"], x["v_cache"], x["pos_in"], x["rope_cos"][:cap - 1].contiguous(),
                  x["rope_sin"][:cap - 1].contiguous())
    assert e.value.code == 1
    # long enough for the new positions, shorter than the old ones (up to T - 1):
    # the kernel marks every unit whose kept keys it cannot rotate
    p.compact_status.zero_()
    p.compact(x["k_cache"], x["v_cache"], x["pos_in"], x["rope_cos"][:cap].contiguous(),
              x["rope_sin"][:cap].contiguous())
    torch.cuda.synchronize()
    assert (p.compact_status.cpu().numpy() == o.UNIT_BAD_INDEX).all()


def test_the_pass_and_the_deletion_effect_are_deterministic(kvc):
    w = wl.qwen3_8b_32k().replace(name="det", n_layers=2, n_kv_heads=2, n_q_heads=8, n_tokens=3000,
                                  budget_tokens=512, decode_pos=512)
    p, x = _pass(w)
    args = (x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"], x["rope_sin"],
            x.get("bonus"))
    p.run(*args)
    first = [t.clone() for t in (p.scores, p.kept_idx, p.kept_count, p.pools.k_bf16, p.pools.v_bf16,
                                 p.pools.pos_out)]
    p.run(*args)
    torch.cuda.synchronize()
    again = (p.scores, p.kept_idx, p.kept_count, p.pools.k_bf16, p.pools.v_bf16, p.pools.pos_out)
    for a, b in zip(first, again):
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)
    we = wl.commitkv_effect_small()
    xe = wl.make_effect_inputs(we, "cuda")
    es = kvc.make_shape(we.batch, we.n_layers, we.n_q_heads, we.n_kv_heads, 128, we.n_tokens)
    ws = torch.empty(kvc.kvc_deletion_effect_workspace_bytes(es, we.window), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for _ in range(2):
        rec = kvc.EffectRecord(es, we.window, we.n_pages)
        eff = torch.empty((we.batch, we.n_layers, we.n_pages), device="cuda")
        kvc.kvc_deletion_effect(es, xe["k_cache"], xe["v_cache"], xe["q_minus"], we.window, 0.0,
                                xe["page_start"], xe["page_len"], eff, rec, ws)
        torch.cuda.synchronize()
        outs.append((eff.clone(), rec.o.clone(), rec.u.clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
