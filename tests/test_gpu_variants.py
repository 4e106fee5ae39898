"""Selection variants on the GPU against the oracle.

SnapKV pooling of the score buffer (kernels 3, 5, 7; average and maximum)
and CommitKV Eq. 4's shared index set: per-sequence summed scores, one
selection per sequence, the kept lists copied to every unit and compacted.
"""
import math

import numpy as np
import pytest
import torch

import oracle as o
import workloads as wl
from helpers import bits, params_of, unit_inputs

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


@pytest.mark.parametrize("kernel", [3, 5, 7])
@pytest.mark.parametrize("mode", ["avg", "max"])
def test_pool_scores_matches_oracle(kvc, kernel, mode):
    rng = np.random.default_rng(kernel)
    s = rng.standard_normal((5, 3001)).astype(np.float32)
    s[1, 7] = np.inf                          # specials pass through the maximum
    src = torch.from_numpy(s).cuda()
    out = torch.empty_like(src)
    kvc.kvc_pool_scores(src, out, kernel, kvc.SCORE_POOL_AVG if mode == "avg" else kvc.SCORE_POOL_MAX)
    torch.cuda.synchronize()
    for r in range(5):
        ref = o.pool_scores(s[r], kernel, mode)
        got = out[r].cpu().numpy()
        if mode == "max":
            assert np.array_equal(got, ref)
        else:
            fin = np.isfinite(ref)
            np.testing.assert_allclose(got[fin], ref[fin], rtol=2e-6, atol=1e-6)
            assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_shared_index_set_end_to_end(kvc):
    w = wl.tiny().replace(batch=2, n_layers=2, n_kv_heads=2, n_q_heads=4, n_tokens=1000,
                          budget_tokens=200)
    x = wl.make_inputs(w, device="cuda")
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    p = pass_for_workload(w, inputs=x)
    p.score(x["k_cache"], x["q_window"], x.get("bonus"))
    B, T = w.batch, w.n_tokens
    shared = torch.empty(B, T, device="cuda")
    kvc.kvc_shared_scores(p.shape, p.scores, shared)
    seq_shape = kvc.make_shape(B, 1, 1, 1, w.head_dim, T)
    kept_s = torch.zeros(3, B, p.policy.capacity, dtype=torch.int32, device="cuda")
    cnt_s = torch.zeros(3, B, dtype=torch.int32, device="cuda")
    st_s = torch.zeros(B, dtype=torch.int32, device="cuda")
    kvc.kvc_select(seq_shape, p.policy, shared, kept_s, cnt_s, st_s)
    kvc.kvc_broadcast_kept(p.shape, p.policy, kept_s, cnt_s, p.kept_idx, p.kept_count)
    p.compact(x["k_cache"], x["v_cache"], x["pos_in"], x["rope_cos"], x["rope_sin"])
    torch.cuda.synchronize()
    assert int(st_s.abs().sum()) == 0 and int(p.compact_status.abs().sum()) == 0
    gsc = p.scores.cpu().numpy()
    per_seq = w.n_layers * w.n_kv_heads
    prm = params_of(w)
    cos, sin = x["rope_cos"].cpu().numpy(), x["rope_sin"].cpu().numpy()
    for b in range(B):
        ref_shared = o.shared_scores(gsc[b * per_seq:(b + 1) * per_seq])
        got_shared = shared[b].cpu().numpy()
        np.testing.assert_allclose(got_shared, ref_shared, rtol=1e-6, atol=1e-7)
        # selection on the GPU's shared scores: bit-exact, and identical for every unit
        act, _, st = o.select_unit(got_shared, None, T, w.head_dim, prm, None, None, None, 0)
        assert st == o.UNIT_OK
        kept_ref = np.nonzero(act == o.ACT_BF16)[0]
        for k in range(per_seq):
            u = b * per_seq + k
            n = int(p.kept_count[2, u])
            assert np.array_equal(p.kept_idx[2, u, :n].cpu().numpy(), kept_ref)
            ui = unit_inputs(w, x, u)
            ref_pools = o.compact_unit(ui["k"], ui["v"], ui["pos"], act, prm, cos, sin)
            assert np.array_equal(bits(p.pools.k_bf16[u, :n]), ref_pools[o.ACT_BF16].k)
            assert np.array_equal(bits(p.pools.v_bf16[u, :n]), ref_pools[o.ACT_BF16].v)


@pytest.mark.parametrize("layout,rd", [("interleaved", 0), ("split", 64), ("interleaved", 64),
                                       ("split", 0)])
def test_rotary_layouts_bit_exact(kvc, layout, rd):
    """Interleaved and partial rotary layouts (PACE Sec. 3.2: the same
    rotation on the rotated dimensions only): compacted keys bit for bit."""
    w = wl.tiny().replace(head_dim=128, n_tokens=900, budget_tokens=250)
    x = wl.make_inputs(w, device="cuda", with_tables=False)
    rdim = rd or w.head_dim
    cos, sin = wl.rope_tables(w.capacity() + w.n_tokens, rdim, 1e4, device="cuda")
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    p = pass_for_workload(w, inputs=x)
    p.policy.rope_layout = kvc.ROPE_INTERLEAVED if layout == "interleaved" else kvc.ROPE_SPLIT_HALF
    p.policy.rotary_dim = rd
    p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], cos, sin, x.get("bonus"))
    torch.cuda.synchronize()
    assert int(p.compact_status.abs().sum()) == 0
    prm = params_of(w)
    prm.rope_layout, prm.rotary_dim = layout, rd
    cos_h, sin_h = cos.cpu().numpy(), sin.cpu().numpy()
    for u in range(w.n_units):
        ui = unit_inputs(w, x, u)
        n = int(p.kept_count[2, u])
        act = np.zeros(w.n_tokens, np.int64)
        act[p.kept_idx[2, u, :n].cpu().numpy()] = o.ACT_BF16
        ref = o.compact_unit(ui["k"], ui["v"], ui["pos"], act, prm, cos_h, sin_h)[o.ACT_BF16]
        assert np.array_equal(bits(p.pools.k_bf16[u, :n]), ref.k)
        assert np.array_equal(p.pools.pos_out[2, u, :n].cpu().numpy(), ref.pos)
