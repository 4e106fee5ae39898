"""H2O cumulative scoring over decode steps and the PACE Eq. 2 bonus on the GPU.

kvc_score with window 1 (one decode query per head) and KVC_SCORE_ACCUMULATE
sums each step's attention weights into the running score (with or without
the caller's row statistics); kvc_foresight_bonus paints the bonus from
spans.  Both are compared with the oracle (scores within rel 1e-2, the
bonus within rel 1e-6), and a selection over the sum keeps every referenced
token when they fit in the budget (the sigma/2 floor of PACE Sec. 3.1).
"""
import math

import numpy as np
import pytest
import torch

import oracle as o
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


def _spans(rng, B, T, n, step):
    seq = rng.integers(0, B, n).astype(np.int32)
    a = rng.integers(0, T - 10, n).astype(np.int64)
    b = (a + rng.integers(1, 200, n)).astype(np.int64)
    F = [sorted(rng.choice(40, rng.integers(1, 4), replace=False).tolist()) for _ in range(n)]
    nxt = np.array([min([s for s in f if s >= step], default=-1) for f in F], np.int32)
    return seq, a, b, F, nxt


def test_foresight_bonus_matches_oracle(kvc):
    rng = np.random.default_rng(21)
    B, T, step = 3, 5000, 12
    seq, a, b, F, nxt = _spans(rng, B, T, 40, step)
    bonus = torch.full((B, T), -1.0, device="cuda")
    c = lambda x: torch.from_numpy(x).cuda()
    kvc.kvc_foresight_bonus(B, T, c(seq), c(a), c(b), c(nxt), step, 1e5, 0.35, bonus)
    torch.cuda.synchronize()
    for bb in range(B):
        spans = [(a[i], b[i], F[i]) for i in range(len(seq)) if seq[i] == bb]
        ref = o.foresight_bonus(spans, step, T, 1e5, 0.35)
        got = bonus[bb].cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=0)


@pytest.mark.parametrize("d,G,use_lse", [(64, 2, False), (128, 4, False), (128, 4, True)])
def test_h2o_decode_steps_accumulate_and_bonus_floor(kvc, d, G, use_lse):
    rng = np.random.default_rng(d + G)
    B, L, HKV, T, steps = 1, 2, 2, 1500, 5
    HQ = HKV * G
    U = B * L * HKV
    scale = 1 / math.sqrt(d)
    shape = kvc.make_shape(B, L, HQ, HKV, d, T)
    k = torch.randn(B, L, HKV, T, d, generator=torch.Generator().manual_seed(d)).to(torch.bfloat16).cuda()
    q = (torch.randn(steps, B, L, HQ, 1, d, generator=torch.Generator().manual_seed(d + 1)) * 2
         ).to(torch.bfloat16).cuda()
    scores = torch.zeros(U, T, device="cuda")
    status = torch.zeros(U, dtype=torch.int32, device="cuda")
    ws = torch.empty(kvc.kvc_score_workspace_bytes(shape, 1), dtype=torch.uint8, device="cuda")
    # the bonus of the last step, from two spans of sequence 0
    spans = [(100, 160, [7, 9]), (900, 950, [30])]
    c = lambda x: torch.from_numpy(np.asarray(x)).cuda()
    bonus = torch.empty(B, T, device="cuda")
    kvc.kvc_foresight_bonus(B, T, c(np.zeros(2, np.int32)), c(np.array([100, 900], np.int64)),
                            c(np.array([160, 950], np.int64)), c(np.array([7, 30], np.int32)),
                            5, 1e5, 0.35, bonus)
    for s in range(steps):
        qs = q[s].contiguous()
        lse = None
        if use_lse:
            lse_h = np.zeros((U, G), np.float32)
            for u in range(U):
                l, g = u // HKV, u % HKV
                lse_h[u] = o.window_row_lse(o.bf16_bits_to_f32(bits(k[0, l, g])),
                                            o.bf16_bits_to_f32(bits(qs[0, l, g * G:(g + 1) * G])), scale)
            lse = torch.from_numpy(lse_h).cuda()
        kvc.kvc_score(shape, k, qs, 1, scale, bonus if s == steps - 1 else None, 1,
                      kvc.SCORE_ACCUMULATE if s > 0 else 0, scores, None, status, ws, row_lse=lse)
    torch.cuda.synchronize()
    assert int(status.abs().sum()) == 0
    ref_bonus = o.foresight_bonus(spans, 5, T)
    for u in range(U):
        l, g = u // HKV, u % HKV
        qu = np.stack([bits(q[s, 0, l, g * G:(g + 1) * G, 0]) for s in range(steps)])
        ref = o.cumulative_decode_scores(bits(k[0, l, g]), qu, scale, ref_bonus)
        assert_scores_close(scores[u].cpu().numpy(), ref)
    # selection over cumulative score + bonus keeps every referenced token
    budget = 300
    pol = kvc.Policy(budget_tokens=budget, capacity=budget, n_sink=4, n_recent=16)
    kept = torch.zeros(3, U, budget, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(3, U, dtype=torch.int32, device="cuda")
    kvc.kvc_select(shape, pol, scores, kept, cnt, status)
    torch.cuda.synchronize()
    referenced = set(range(100, 160)) | set(range(900, 950))
    for u in range(U):
        got = set(kept[2, u, :int(cnt[2, u])].cpu().numpy().tolist())
        assert referenced <= got
