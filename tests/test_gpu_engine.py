"""The engine attention (PASK App. B.5) on the GPU against the oracle.

Persistent storage = the pools of a compaction pass (bf16 in token mode;
int4 / int8 / bf16 in byte mode), plus recent and current bf16 rows with
logical positions that leave gaps; queries at the current positions (causal
among the current rows); one-head, GQA-2, GQA-4 and several queries per
head; split-KV.  Outputs are bf16: max-abs 2e-2, as for the decode check.
"""
import math

import numpy as np
import pytest
import torch

import oracle as o
import workloads as wl
from helpers import DECODE_ATOL, bits, unit_pools_from_gpu

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


def token_workload(hq, hkv, d=128):
    return wl.qwen3_8b_32k().replace(name=f"engine_tok_{hq}_{hkv}_{d}", n_layers=2, n_kv_heads=hkv,
                                     n_q_heads=hq, head_dim=d, n_tokens=3000, window=16,
                                     budget_tokens=512, n_recent=16, renumber=False, decode_pos=3000)


def byte_workload(hq, hkv):
    return wl.pask_batch16().replace(name=f"engine_byte_{hq}_{hkv}", batch=2, n_layers=4,
                                     n_kv_heads=hkv, n_q_heads=hq, n_tokens=2000, window=16,
                                     n_recent=16, budget_bytes=(2000 * 512) // 3, decode_pos=2000)


def run_case(kvc, w, n_q, rec_cap=40, with_pools=True, with_pos=True, blind_first=False, seed=0):
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    x = wl.make_inputs(w, "cuda")
    p = pass_for_workload(w, inputs=x)
    p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"], x["rope_sin"],
          x.get("bonus"))
    torch.cuda.synchronize()
    U, d, B = w.n_units, w.head_dim, w.batch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    rn = lambda *s: torch.randn(*s, generator=g, device="cuda").to(torch.bfloat16)
    base = w.n_tokens                                   # persistent positions are below T
    rec_k, rec_v = rn(U, rec_cap, d), rn(U, rec_cap, d)
    rec_pos = (base + 2 * torch.arange(rec_cap, device="cuda", dtype=torch.int32)).expand(U, rec_cap).contiguous()
    rec_cnt = torch.randint(0, rec_cap + 1, (U,), generator=g, device="cuda", dtype=torch.int32)
    cur_base = base + 2 * rec_cap + 5
    cur_k, cur_v = rn(U, n_q, d), rn(U, n_q, d)
    cur_pos = (cur_base + torch.arange(n_q, device="cuda", dtype=torch.int32)).expand(U, n_q).contiguous()
    cur_cnt = torch.full((U,), n_q, dtype=torch.int32, device="cuda")
    q = rn(B, w.n_layers, w.n_q_heads, n_q, d)
    q_pos = (cur_base + torch.arange(n_q, device="cuda", dtype=torch.int32)).expand(B, n_q).contiguous()
    if blind_first:
        q_pos[:, 0] = -1                                 # sees no key: output 0
    out = torch.empty_like(q)
    recent = kvc.bf16_rows(rec_k, rec_v, rec_pos if with_pos else None, rec_cnt)
    current = kvc.bf16_rows(cur_k, cur_v, cur_pos if with_pos else None, cur_cnt)
    pol = p.policy if with_pools else None
    wsb = kvc.kvc_engine_attn_workspace_bytes(p.shape, pol, n_q, recent, current)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda") if wsb else None
    kvc.kvc_engine_attn(p.shape, pol, q, n_q, q_pos if with_pos else None,
                        p.pools if with_pools else None, p.kept_count if with_pools else None,
                        recent, current, 0.0, out, ws)
    torch.cuda.synchronize()

    scale = 1.0 / math.sqrt(d)
    G = w.group
    qp = q_pos.cpu().numpy()
    rc = rec_cnt.cpu().numpy()
    worst = 0.0
    for u in range(U):
        b, l, gk = wl.unit_coords(w, u)
        stores = []
        if with_pools:
            for a, pool in unit_pools_from_gpu(p, u, w).items():
                if pool.idx.size:
                    kk, vv = o.pool_rows_f32(pool, w.quant_mode)
                    stores.append((kk, vv, pool.pos if with_pos else None))
        n = int(rc[u])
        stores.append((o.bf16_bits_to_f32(bits(rec_k[u, :n])), o.bf16_bits_to_f32(bits(rec_v[u, :n])),
                       rec_pos[u, :n].cpu().numpy() if with_pos else None))
        stores.append((o.bf16_bits_to_f32(bits(cur_k[u])), o.bf16_bits_to_f32(bits(cur_v[u])),
                       cur_pos[u].cpu().numpy() if with_pos else None))
        rows = o.bf16_bits_to_f32(bits(q[b, l, gk * G:(gk + 1) * G])).reshape(G * n_q, d)
        rpos = np.tile(qp[b], G) if with_pos else None
        ref = o.engine_attention(rows, rpos, stores, scale)
        got = out[b, l, gk * G:(gk + 1) * G].float().reshape(G * n_q, d).cpu().numpy()
        err = np.abs(got - ref).max()
        worst = max(worst, err)
        assert err <= DECODE_ATOL, f"unit {u}: max-abs {err}"
        if blind_first:
            assert (got.reshape(G, n_q, d)[:, 0] == 0).all()
    return worst


@pytest.mark.parametrize("hq,hkv,n_q", [(4, 4, 1), (8, 4, 2), (8, 2, 1), (8, 2, 4), (16, 2, 2)])
def test_engine_attention_token_pools(kvc, hq, hkv, n_q):
    run_case(kvc, token_workload(hq, hkv), n_q)


@pytest.mark.parametrize("hq,hkv,n_q", [(8, 2, 1), (8, 2, 3), (4, 2, 2)])
def test_engine_attention_byte_pools(kvc, hq, hkv, n_q):
    run_case(kvc, byte_workload(hq, hkv), n_q)


def test_engine_attention_d64_and_a_blind_query(kvc):
    run_case(kvc, token_workload(8, 2, d=64), 3, blind_first=True)


def test_engine_attention_without_positions_or_pools(kvc):
    run_case(kvc, token_workload(8, 2), 2, with_pos=False)
    run_case(kvc, token_workload(8, 2), 2, with_pools=False, rec_cap=300)


def test_engine_attention_single_query_matches_decode(kvc):
    """With no recent or current rows and one query per head, the engine
    attention is the decode check over the pools."""
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    w = token_workload(8, 2)
    x = wl.make_inputs(w, "cuda")
    p = pass_for_workload(w, inputs=x)
    p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"], x["rope_sin"],
          x.get("bonus"))
    p.decode(x["q_decode"])
    q = x["q_decode"].reshape(w.batch, w.n_layers, w.n_q_heads, 1, w.head_dim).contiguous()
    out = torch.empty_like(q)
    wsb = kvc.kvc_engine_attn_workspace_bytes(p.shape, p.policy, 1)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    kvc.kvc_engine_attn(p.shape, p.policy, q, 1, None, p.pools, p.kept_count, None, None, 0.0, out, ws)
    torch.cuda.synchronize()
    diff = (out.reshape(p.out.shape).float() - p.out.float()).abs().max().item()
    assert diff <= 1e-2
