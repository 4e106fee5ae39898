"""kvc_score with small windows (R = W G <= 16 rows per unit: the CUDA-core
path) against the oracle: window mass (PASK Eq. 1) with the causal window,
with and without the caller's row statistics, bonus, ACCUMULATE and page
maxima, on ragged key counts."""
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


CASES = [  # d, G, W, T, page size, caller statistics
    (128, 1, 1, 1500, 1, False),
    (128, 2, 1, 1537, 1, True),
    (64, 4, 1, 2048, 16, False),
    (128, 2, 3, 999, 1, False),       # R = 6 -> 8 padded rows
    (128, 4, 3, 3000, 8, True),       # R = 12 -> 16
    (64, 1, 16, 4096, 32, False),     # R = 16, W = 16
    (128, 8, 2, 5000, 1, False),      # R = 16
]


@pytest.mark.parametrize("d,G,W,T,P,use_lse", CASES)
def test_small_window_scores_match_oracle(kvc, d, G, W, T, P, use_lse):
    B, L, HKV = 2, 1, 2
    HQ = HKV * G
    U = B * L * HKV
    scale = 1 / math.sqrt(d)
    gen = torch.Generator().manual_seed(d * 100 + G * 10 + W)
    k = torch.randn(B, L, HKV, T, d, generator=gen).to(torch.bfloat16).cuda()
    q = (torch.randn(B, L, HQ, W, d, generator=gen) * 1.5).to(torch.bfloat16).cuda()
    bonus = (torch.rand(B, T, generator=gen) * 0.01).cuda()
    first = torch.rand(U, T, generator=gen).cuda() * 0.1
    scores = first.clone()
    pages = torch.full((U, T // P), -7.0, device="cuda") if P > 1 else None
    status = torch.zeros(U, dtype=torch.int32, device="cuda")
    shape = kvc.make_shape(B, L, HQ, HKV, d, T)
    ws = torch.empty(kvc.kvc_score_workspace_bytes(shape, W), dtype=torch.uint8, device="cuda")
    lse = None
    lse_h = None
    if use_lse:
        lse_h = np.zeros((U, G * W), np.float32)
        for u in range(U):
            b, g = u // HKV, u % HKV
            lse_h[u] = o.window_row_lse(o.bf16_bits_to_f32(bits(k[b, 0, g])),
                                        o.bf16_bits_to_f32(bits(q[b, 0, g * G:(g + 1) * G])), scale)
        lse = torch.from_numpy(lse_h).cuda()
    kvc.kvc_score(shape, k, q, W, scale, bonus, P, kvc.SCORE_ACCUMULATE, scores, pages, status, ws,
                  row_lse=lse)
    torch.cuda.synchronize()
    assert int(status.abs().sum()) == 0
    for u in range(U):
        b, g = u // HKV, u % HKV
        kb = bits(k[b, 0, g])
        qb = bits(q[b, 0, g * G:(g + 1) * G])
        if use_lse:
            mass = o.window_mass_given_lse(o.bf16_bits_to_f32(kb), o.bf16_bits_to_f32(qb), scale,
                                           lse_h[u].astype(np.float64))
            ref = (mass + bonus[b].cpu().numpy().astype(np.float64)
                   + first[u].cpu().numpy().astype(np.float64)).astype(np.float32)
        else:
            ref = o.unit_scores(kb, qb, scale, bonus[b].cpu().numpy(), first[u].cpu().numpy())
        got = scores[u].cpu().numpy()
        assert_scores_close(got, ref)
        if P > 1:
            np.testing.assert_array_equal(pages[u].cpu().numpy(), got.reshape(-1, P).max(axis=1))
