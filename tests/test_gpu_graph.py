"""The compaction pass captured once as a CUDA graph and replayed gives the
same bytes as the pass run call by call (the bench times both): scores, kept
lists and counts, and the compacted pools with their positions."""
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

# pool tensors ([U][capacity][...]) and the pool whose kept count bounds them
POOL_TENSORS = {"k_bf16": 2, "v_bf16": 2, "k_i8": 1, "v_i8": 1, "k_i8_scale": 1, "v_i8_scale": 1,
                "k_i4": 0, "v_i4": 0, "k_i4_scale": 0, "v_i4_scale": 0}


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from budgeted_kv_cache_gb300 import build
    build.build()
    import budgeted_kv_cache_gb300 as lib
    lib.library()
    return lib


def _outputs(p):
    n = p.kept_count.clone()
    kept = [p.kept_idx[q, u, :int(n[q, u])].clone() for q in range(n.shape[0]) for u in range(n.shape[1])]
    pools = {}
    for name in POOL_TENSORS:
        t = getattr(p.pools, name, None)
        if t is not None:
            pools[name] = t.clone()
    return p.scores.clone(), n, kept, pools, p.pools.pos_out.clone()


def _clear(p):
    p.scores.zero_()
    p.kept_idx.fill_(-1)
    p.kept_count.fill_(-1)
    for name in POOL_TENSORS:
        t = getattr(p.pools, name, None)
        if t is not None:
            t.zero_()
    p.pools.pos_out.fill_(-1)


@pytest.mark.parametrize("make", [
    lambda: wl.qwen3_8b_32k().replace(name="graph_tok", n_layers=2, n_kv_heads=2, n_q_heads=8,
                                      n_tokens=5000, budget_tokens=512, decode_pos=512),
    lambda: wl.pask_batch16().replace(name="graph_byte", batch=2, n_layers=4, n_kv_heads=2,
                                      n_q_heads=8, n_tokens=2000, budget_bytes=(2000 * 512) // 3,
                                      decode_pos=2000),
], ids=["token_renumber", "byte_mode"])
def test_pass_replayed_from_a_graph_matches_eager(kvc, make):
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    w = make()
    x = wl.make_inputs(w, device="cuda")
    p = pass_for_workload(w, inputs=x)
    s = torch.cuda.Stream()
    run = lambda: p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"],
                        x["rope_sin"], x.get("bonus"), stream=s)
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    eager = _outputs(p)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        run()
    torch.cuda.synchronize()
    _clear(p)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    replay = _outputs(p)
    assert int(p.score_status.abs().sum()) == 0 and int(p.unit_status.abs().sum()) == 0
    assert torch.equal(eager[0].view(torch.int32), replay[0].view(torch.int32))
    assert torch.equal(eager[1], replay[1])
    for a, b in zip(eager[2], replay[2]):
        assert torch.equal(a, b)
    n = eager[1]
    for name, t in eager[3].items():
        r = replay[3][name]
        pool = POOL_TENSORS[name]
        for u in range(n.shape[1]):
            k = int(n[pool, u])
            assert torch.equal(t[u, :k].view(torch.uint8), r[u, :k].view(torch.uint8)), f"{name} unit {u}"
    for q in range(n.shape[0]):
        for u in range(n.shape[1]):
            k = int(n[q, u])
            assert torch.equal(eager[4][q, u, :k], replay[4][q, u, :k])
