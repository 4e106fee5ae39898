"""Pins of the oracle's engine attention (PASK App. B.5: persistent, recent
and current storage, logical positions, causal masks, one shared softmax).
CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle as o


def _stores(rng, sizes, d, pos_start):
    out, p = [], pos_start
    for n in sizes:
        k = rng.standard_normal((n, d))
        v = rng.standard_normal((n, d))
        out.append((k, v, np.arange(p, p + n)))
        p += n + 3                                   # gaps between storages
    return out


def test_engine_attention_matches_torch_sdpa_with_a_causal_mask():
    rng = np.random.default_rng(0)
    d, R = 32, 6
    stores = _stores(rng, [40, 7, 3], d, 100)
    q = rng.standard_normal((R, d))
    # query positions inside and after the storages: some keys hidden from some rows
    q_pos = np.array([105, 139, 145, 152, 160, 1000])
    got = o.engine_attention(q, q_pos, stores, 0.2)
    K = torch.from_numpy(np.concatenate([s[0] for s in stores]))
    V = torch.from_numpy(np.concatenate([s[1] for s in stores]))
    P = torch.from_numpy(np.concatenate([s[2] for s in stores]))
    mask = P[None, :] <= torch.from_numpy(q_pos)[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], K[None], V[None], attn_mask=mask[None], scale=0.2)[0].numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_split_between_storages_does_not_change_the_output():
    # one shared normalisation: moving rows between storages (or reordering
    # them) leaves every output unchanged; averaging per-storage outputs would not
    rng = np.random.default_rng(1)
    d = 16
    (k, v, p), = _stores(rng, [50], d, 0)
    q = rng.standard_normal((3, d))
    q_pos = np.array([20, 35, 60])
    whole = o.engine_attention(q, q_pos, [(k, v, p)], 0.25)
    perm = rng.permutation(50)
    parts = [(k[perm[:10]], v[perm[:10]], p[perm[:10]]), (k[perm[10:45]], v[perm[10:45]], p[perm[10:45]]),
             (k[perm[45:]], v[perm[45:]], p[perm[45:]])]
    np.testing.assert_allclose(o.engine_attention(q, q_pos, parts, 0.25), whole, rtol=1e-12, atol=1e-14)
    avg = np.mean([o.engine_attention(q, q_pos, [s], 0.25) for s in parts], axis=0)
    assert np.abs(avg - whole).max() > 1e-3


def test_keys_after_a_query_do_not_reach_it():
    rng = np.random.default_rng(2)
    d = 8
    stores = _stores(rng, [20, 5], d, 0)
    q = rng.standard_normal((2, d))
    q_pos = np.array([10, 30])
    a = o.engine_attention(q, q_pos, stores, 1.0)
    k2, v2, p2 = stores[0]
    k2, v2 = k2.copy(), v2.copy()
    k2[11:] += 50.0
    v2[11:] -= 9.0
    b = o.engine_attention(q, q_pos, [(k2, v2, p2), stores[1]], 1.0)
    np.testing.assert_array_equal(a[0], b[0])         # row 0 sees positions <= 10 only
    assert np.abs(a[1] - b[1]).max() > 1e-3


def test_no_positions_means_every_key_and_an_empty_row_is_zero():
    rng = np.random.default_rng(3)
    d = 8
    k, v = rng.standard_normal((9, d)), rng.standard_normal((9, d))
    q = rng.standard_normal((2, d))
    got = o.engine_attention(q, None, [(k, v, None)], 0.5)
    for r in range(2):
        z = k @ q[r] * 0.5
        w = np.exp(z - z.max())
        np.testing.assert_allclose(got[r], (w / w.sum()) @ v, rtol=1e-12)
    none = o.engine_attention(q, np.array([-1, -1]), [(k, v, np.arange(9))], 0.5)
    assert (none == 0).all()
