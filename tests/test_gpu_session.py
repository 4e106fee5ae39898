"""GPU parity of the bounded-position session (PACE Sec. 3.2 "Bounded
positions" / "Choosing L", Sec. 5.7; the million-token workload in cycles).

Every cycle is checked stage-wise against the oracle's session cycle on the
same cache: scores within the score tolerance; the kept sets, the new
positions and the stored (re-rotated) keys and values bit-exact when the
oracle selects from the GPU's scores.  The oracle's own chain is carried
alongside, so after several cycles its resident rows must still equal the
GPU's byte for byte.
"""
import math

import numpy as np
import pytest
import torch

import oracle as o
import workloads as wl
from helpers import assert_scores_close, bits

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


def _small(limit):
    # G = 4, W = 16 (64 window rows), budget 256 + chunk 512: T = 768 rows
    return wl.million_token_sustained().replace(
        name="session_small", n_layers=2, n_kv_heads=2, n_q_heads=8, budget_tokens=256, chunk=512,
        n_tokens=768, window=16, n_recent=32, cycles=4, limit=limit)


def _run(kvc, w, units, cycles, check_scores=True):
    from budgeted_kv_cache_gb300.session import BoundedSession
    dev = "cuda"
    s0 = wl.session_start(w, dev)
    sess = BoundedSession(w.batch, w.n_layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.budget_tokens,
                          w.chunk, w.window, w.limit, w.n_sink, w.n_recent, device=dev)
    sess.start(s0["k0"], s0["v0"])
    cos, sin = s0["rope_cos"].cpu().numpy(), s0["rope_sin"].cpu().numpy()
    prm = o.PassParams(budget_tokens=w.budget_tokens, n_sink=w.n_sink, n_recent=w.n_recent,
                       renumber=True)
    scale = 1 / math.sqrt(w.head_dim)
    G = w.group
    # the oracle's own chain, per checked unit
    chain = {}
    k0, v0, p0 = sess.resident()
    for u in units:
        chain[u] = (bits(k0[u]), bits(v0[u]), p0[u].cpu().numpy().astype(np.int64))
    flags = []
    for c in range(cycles):
        ch = wl.session_chunk(w, c, dev)
        sess.append(ch["k"], ch["v"])
        buf = sess.passes[sess.cur].pools
        cache_k, cache_v = bits(buf.k_bf16), bits(buf.v_bf16)      # the cycle's inputs
        cache_pos = buf.pos_out[2].cpu().numpy()
        flags.append(sess.compact(ch["q_window"], s0["rope_cos"], s0["rope_sin"]))
        torch.cuda.synchronize()
        p = sess.last_pass
        assert int(p.unit_status.abs().sum()) == 0 and int(p.compact_status.abs().sum()) == 0
        kr, vr, pr = sess.resident()
        for u in units:
            b, l, g = wl.unit_coords(w, u)
            q = bits(ch["q_window"][b, l, g * G:(g + 1) * G])
            got = p.scores[u].cpu().numpy()
            if check_scores:
                assert_scores_close(got, o.unit_scores(cache_k[u], q, scale), f"cycle {c} unit {u}")
            # stage-wise: the oracle cycle from the GPU's resident rows and chunk
            rk, rv, rp = chain[u]
            assert np.array_equal(cache_k[u, :w.budget_tokens], rk)
            assert np.array_equal(cache_pos[u, :w.budget_tokens], rp)
            nk, nv = bits(ch["k"][b, l, g]), bits(ch["v"][b, l, g])
            ok_, ov_, op_, r = o.session_cycle(rk, rv, rp, nk, nv, q, prm, w.limit, cos, sin, scores=got)
            n = int(p.kept_count[2, u])
            assert n == w.budget_tokens
            assert np.array_equal(p.kept_idx[2, u, :n].cpu().numpy(), r.pools[o.ACT_BF16].idx)
            assert np.array_equal(pr[u].cpu().numpy(), op_), f"cycle {c} unit {u}: positions"
            assert np.array_equal(bits(kr[u]), ok_), f"cycle {c} unit {u}: keys"
            assert np.array_equal(bits(vr[u]), ov_), f"cycle {c} unit {u}: values"
            chain[u] = (ok_, ov_, np.asarray(op_, np.int64))
    return sess, flags


def test_session_small_renumbering_every_cycle(kvc):
    """L = 1024 < budget + 2 chunks: every compaction renumbers."""
    w = _small(limit=1024)
    sess, flags = _run(kvc, w, units=range(w.n_units), cycles=4)
    assert all(flags)
    _, _, pr = sess.resident()
    assert torch.equal(pr.cpu(), torch.arange(w.budget_tokens, dtype=torch.int32).expand(w.n_units, -1))


def test_session_small_inactive_keeps_positions(kvc):
    """A limit never reached: no renumbering, kept keys are the appended bits."""
    w = _small(limit=1 << 14)
    sess, flags = _run(kvc, w, units=range(w.n_units), cycles=3)
    assert not any(flags)
    _, _, pr = sess.resident()
    assert int(pr.max()) == w.budget_tokens + 3 * w.chunk - 1


def test_session_million_token_shape_sampled_units(kvc):
    """The million-token workload's shape (64 units, 6,144-row cache, window 64):
    three cycles, units at both ends and the middle checked in full; every
    unit keeps exactly the budget."""
    w = wl.million_token_sustained()
    _run(kvc, w, units=[0, 31, 63], cycles=3)
