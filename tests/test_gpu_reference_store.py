"""PACE reference store (kvc_compact_rerotate_quant_ref) against the oracle.

Two successive renumbering compactions of the same keys: the first creates
the references (keys equal those of plain re-rotation), the second derives
the new keys from them; a deliberately stale reference is detected and
replaced.  Keys, references, reference positions and failure counts are
compared bit for bit with oracle.compact_unit(..., ref_bits, ref_pos).
"""
import numpy as np
import pytest
import torch

import oracle as o
import workloads as wl
from helpers import bits

pytestmark = pytest.mark.gpu

B, L, HQ, HKV, D = 1, 2, 4, 2, 64
U = B * L * HKV


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from budgeted_kv_cache_gb300 import build
    build.build()
    import budgeted_kv_cache_gb300 as lib
    lib.library()
    return lib


def _kept(T, n, rng, must=None):
    """kept_idx [3][U][n] (bf16 pool only) and kept_count for n random rows per
    unit; `must` = {unit: row} rows that are kept."""
    rows = []
    for u in range(U):
        r = rng.choice(T, n, replace=False)
        if must and u in must and must[u] not in r:
            r[0] = must[u]
        rows.append(np.sort(r))
    idx = np.stack(rows).astype(np.int32)
    kept = np.zeros((3, U, n), np.int32)
    kept[2] = idx
    cnt = np.zeros((3, U), np.int32)
    cnt[2] = n
    return idx, torch.from_numpy(kept).cuda(), torch.from_numpy(cnt).cuda()


def _compact(kvc, T, cap, k, v, pos, kept, cnt, cos, sin, ref_k, ref_pos):
    shape = kvc.make_shape(B, L, HQ, HKV, D, T)
    pol = kvc.Policy(budget_tokens=cap, capacity=cap, renumber=True)
    pools = kvc.Pools.allocate(shape, pol)
    rk = torch.zeros((3, U, cap, D), dtype=torch.bfloat16, device="cuda")
    rp = torch.full((3, U, cap), -7, dtype=torch.int32, device="cuda")
    fails = torch.zeros(U, dtype=torch.int32, device="cuda")
    status = torch.zeros(U, dtype=torch.int32, device="cuda")
    kvc.kvc_compact_rerotate_quant_ref(shape, pol, k, v, pos, kept, cnt, cos, sin, cos.shape[0],
                                       ref_k, ref_pos, rk, rp, pools, fails, status)
    torch.cuda.synchronize()
    assert int(status.abs().sum()) == 0
    return pools, rk[2], rp[2], fails


def test_reference_store_two_renumbers_bit_exact(kvc):
    rng = np.random.default_rng(11)
    T1, n1, n2 = 1000, 300, 150
    cos, sin = wl.rope_tables(1024, D, 1e4, device="cuda")
    cos_h, sin_h = cos.cpu().numpy(), sin.cpu().numpy()
    # before any renumber: keys rotated at positions 0..T1-1
    k1 = (torch.randn(U, T1, D, generator=torch.Generator().manual_seed(3)) * 2).to(torch.bfloat16).cuda()
    v1 = torch.randn(U, T1, D, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16).cuda()
    pos1 = torch.arange(T1, dtype=torch.int32).repeat(U, 1).contiguous().cuda()
    ref_k1 = torch.zeros_like(k1)
    ref_p1 = torch.full((U, T1), -1, dtype=torch.int32, device="cuda")
    prm = o.PassParams(budget_tokens=n1, budget_bytes=0, n_sink=0, n_recent=0, page_size=1,
                       renumber=True, quant_mode=0, n_layer_groups=1)
    # renumber 1: creates the references
    idx1, kept1, cnt1 = _kept(T1, n1, rng)
    pools1, rk1, rp1, f1 = _compact(kvc, T1, n1, k1, v1, pos1, kept1, cnt1, cos, sin, ref_k1, ref_p1)
    k2, v2 = pools1.k_bf16, pools1.v_bf16
    pos2 = pools1.pos_out[2].contiguous()
    ref_k2, ref_p2 = rk1.contiguous(), rp1.contiguous()
    # a stale reference in unit 1: flip one bit of one referenced row
    stale_row = int(np.nonzero(rp1[1].cpu().numpy() >= 0)[0][-1])   # >= n2: its rank changes
    ref_k2_in = ref_k2.clone()
    ref_k2_in[1, stale_row, 0] = -ref_k2_in[1, stale_row, 0] if float(ref_k2_in[1, stale_row, 0]) != 0 else 1.0
    # renumber 2: from the references (the stale row is kept)
    idx2, kept2, cnt2 = _kept(n1, n2, rng, must={1: stale_row})
    pools2, rk2, rp2, f2 = _compact(kvc, n1, n2, k2, v2, pos2, kept2, cnt2, cos, sin, ref_k2_in, ref_p2)
    for u in range(U):
        # oracle, renumber 1
        act1 = np.zeros(T1, np.int64)
        act1[idx1[u]] = o.ACT_BF16
        ref1 = o.compact_unit(bits(k1[u]), bits(v1[u]), pos1[u].cpu().numpy(), act1, prm, cos_h, sin_h,
                              ref_bits=np.zeros((T1, D), np.uint16), ref_pos=np.full(T1, -1))
        p1 = ref1[o.ACT_BF16]
        assert np.array_equal(bits(pools1.k_bf16[u]), p1.k)
        plain = o.compact_unit(bits(k1[u]), bits(v1[u]), pos1[u].cpu().numpy(), act1, prm, cos_h, sin_h)
        assert np.array_equal(p1.k, plain[o.ACT_BF16].k)          # first renumber = plain re-rotation
        assert np.array_equal(bits(rk1[u]), p1.k_ref)
        assert np.array_equal(rp1[u].cpu().numpy(), p1.p_ref)
        assert int(f1[u]) == 0
        # oracle, renumber 2 (from the renumber-1 outputs as the GPU saw them)
        act2 = np.zeros(n1, np.int64)
        act2[idx2[u]] = o.ACT_BF16
        ref2 = o.compact_unit(bits(k2[u]), bits(v2[u]), pos2[u].cpu().numpy(), act2, prm, cos_h, sin_h,
                              ref_bits=bits(ref_k2_in[u]), ref_pos=ref_p2[u].cpu().numpy())
        p2 = ref2[o.ACT_BF16]
        assert np.array_equal(bits(pools2.k_bf16[u]), p2.k)
        assert np.array_equal(bits(pools2.v_bf16[u]), p2.v)
        assert np.array_equal(bits(rk2[u]), p2.k_ref)
        assert np.array_equal(rp2[u].cpu().numpy(), p2.p_ref)
        assert int(f2[u]) == p2.ref_failures
    assert int(f2[1]) == 1 and int(f2[0]) == 0
