"""The seeded synthetic input recipe (CPU): the same seed gives the same
bytes, units are numbered [B][L][H_kv], and each workload's structure is the
one its recipe states -- foresight bonus spans only between the sinks and the
recent window, commit flags only on pages outside them with PROTECT and
EXCLUDE on disjoint pages, structural tags drawn with the stated mix, outlier
keys at the stated fraction and scale, positions ascending from the first
physical position, rotary tables of unit modulus."""
import dataclasses

import numpy as np
import torch

import workloads as wl


def _small(w, **kw):
    """The workload's structure on a CPU-sized cache."""
    return w.replace(**kw)


def test_same_seed_same_bytes():
    w = _small(wl.qwen3_8b_32k(), n_layers=1, n_kv_heads=2, n_q_heads=8, n_tokens=1024,
               budget_tokens=256, decode_pos=256)
    a, b = wl.make_inputs(w), wl.make_inputs(w)
    assert a.keys() == b.keys()
    for name in a:
        assert torch.equal(a[name], b[name]), name
    c = wl.make_inputs(w.replace(seed=w.seed + 1))
    assert not torch.equal(a["k_cache"], c["k_cache"])


def test_unit_numbering_round_trips():
    w = wl.pask_batch16().replace(n_tokens=64)
    seen = set()
    for u in range(w.n_units):
        b, l, g = wl.unit_coords(w, u)
        assert 0 <= b < w.batch and 0 <= l < w.n_layers and 0 <= g < w.n_kv_heads
        assert wl.unit_index(w, b, l, g) == u
        seen.add((b, l, g))
    assert len(seen) == w.batch * w.n_layers * w.n_kv_heads == w.n_units


def test_bonus_spans_lie_between_sinks_and_recent_rows():
    w = _small(wl.qwen3_8b_32k(), n_layers=1, n_kv_heads=1, n_q_heads=4, n_tokens=4096,
               budget_tokens=256, decode_pos=256)
    x = wl.make_inputs(w, with_tables=False)
    bonus = x["bonus"].numpy()
    assert bonus.shape == (w.batch, w.n_tokens)
    for row in bonus:
        on = np.flatnonzero(row)
        assert on.size == w.bonus_spans * w.bonus_span_len
        assert on.min() >= w.n_sink and on.max() < w.n_tokens - w.n_recent
        assert np.all(row[on] == np.float32(w.bonus_value))
        # whole spans, aligned to span slots past the sinks
        starts = on[np.r_[True, np.diff(on) > 1]]
        assert np.all((starts - w.n_sink) % w.bonus_span_len == 0)


def test_commit_flags_on_free_pages_and_disjoint():
    w = wl.commitkv_pages_128k().replace(n_tokens=16 * 2048, n_layers=1, retire_pages=200,
                                         protect_pages=16)
    x = wl.make_inputs(w, with_tables=False)
    flags = x["flags"].numpy()
    P = w.page_size
    assert flags.shape == (w.batch, w.n_tokens // P)
    for row in flags:
        prot = np.flatnonzero(row == wl.FLAG_PROTECT)
        excl = np.flatnonzero(row == wl.FLAG_EXCLUDE)
        assert prot.size == w.protect_pages and excl.size == w.retire_pages
        assert np.all((row == 0) | (row == wl.FLAG_PROTECT) | (row == wl.FLAG_EXCLUDE))
        flagged = np.r_[prot, excl]
        assert flagged.min() * P >= w.n_sink
        assert (flagged.max() + 1) * P <= w.n_tokens - w.n_recent


def test_structural_tags_follow_the_stated_mix():
    w = wl.pask_batch16().replace(n_layers=1, n_kv_heads=1, n_q_heads=4)
    x = wl.make_inputs(w, with_tables=False)
    tags = x["tags"].numpy()
    assert tags.shape == (w.batch, w.n_tokens)
    freq = np.bincount(tags.ravel(), minlength=len(w.tag_probs)) / tags.size
    # 131,072 draws: each frequency within 5 standard deviations of its probability
    p = np.asarray(w.tag_probs)
    assert np.all(np.abs(freq - p) <= 5 * np.sqrt(p * (1 - p) / tags.size))
    assert np.array_equal(x["action_table"].numpy(), wl.PASK_TABLE)


def test_outlier_keys_at_the_stated_fraction_and_scale():
    w = _small(wl.qwen3_8b_32k(), n_layers=1, n_kv_heads=2, n_q_heads=8, n_tokens=8192,
               budget_tokens=256, decode_pos=256)
    x = wl.make_inputs(w, with_tables=False)
    k = x["k_cache"].float()[0]                            # [L][H_kv][T][d]
    norms = k.norm(dim=-1)[0, 0].numpy()
    # N(0, 1) keys have norms near sqrt(d); scaled ones near scale * sqrt(d)
    big = norms > 0.5 * (1 + w.outlier_scale) * np.sqrt(w.head_dim)
    assert big.sum() == int(round(w.outlier_frac * w.n_tokens))
    assert abs(np.median(norms[big]) / np.median(norms[~big]) - w.outlier_scale) < 0.1
    # the same rows in every head of the sequence
    norms1 = k.norm(dim=-1)[0, 1].numpy()
    assert np.array_equal(big, norms1 > 0.5 * (1 + w.outlier_scale) * np.sqrt(w.head_dim))


def test_positions_and_rotary_tables():
    w = wl.tiny().replace(first_pos=100)
    x = wl.make_inputs(w)
    pos = x["pos_in"].numpy()
    assert pos.shape == (w.n_units, w.n_tokens)
    assert np.all(pos == np.arange(100, 100 + w.n_tokens))
    cos, sin = x["rope_cos"].double(), x["rope_sin"].double()
    assert cos.shape == (w.max_pos, w.head_dim // 2) and w.max_pos >= 100 + w.n_tokens
    assert torch.all((cos * cos + sin * sin - 1).abs() < 1e-6)
    assert torch.all(cos[0] == 1) and torch.all(sin[0] == 0)


def test_workloads_are_frozen_records():
    w = wl.qwen3_8b_32k()
    assert dataclasses.is_dataclass(w)
    v = w.replace(n_tokens=10)
    assert v.n_tokens == 10 and w.n_tokens == 32768
