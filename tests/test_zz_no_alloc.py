"""kvc_decode_attn_noalloc: the decode step for callers that cannot allocate.

Callers such as an engine whose allocator already owns nearly all of HBM, a
plug-in that only gets its host framework's buffers, or a latency-critical
loop that cannot pay for cudaMalloc's implicit synchronisation cannot pass
a workspace.  This entry point keeps the decode step's split-partition
scratch in a static device array inside the library instead.  The test
calls it through the C-ABI twice in a row and checks that each output is
bit-identical to kvc_decode_attn with a caller workspace: both run the same
kernels with the same split plan, so any difference would be a slip in the
scratch layout.

Collected last on purpose, so a run that stops at the first failure has
already run every other test.
"""
import pytest
import torch

import workloads as wl

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


def _workloads():
    # small unit counts and capacities above 256 rows, so the decode is split
    # across CTAs and really goes through the scratch array
    tok = wl.qwen3_8b_32k().replace(n_layers=1, n_kv_heads=2, n_q_heads=8, n_tokens=5000,
                                    budget_tokens=512)
    byt = wl.pask_batch16().replace(batch=1, n_layers=4, n_kv_heads=1, n_q_heads=4,
                                    n_tokens=2000, budget_bytes=(2000 * 512) // 3)
    return [tok, byt]


@pytest.mark.parametrize("w", _workloads(), ids=["token_mode", "byte_mode"])
def test_noalloc_decode_matches_workspace_decode(kvc, w):
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    x = wl.make_inputs(w, device="cuda")
    p = pass_for_workload(w, inputs=x)
    need = kvc.kvc_decode_workspace_bytes(p.shape, p.policy)
    if need == 0:
        pytest.skip("this device's split plan runs the unit in one partition: no scratch is used")
    assert need <= (2 << 20)
    p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"], x["rope_sin"],
          x.get("bonus"))
    ref = p.decode(x["q_decode"]).clone()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        kvc.kvc_decode_attn_noalloc(p.shape, p.policy, x["q_decode"], p.pools, p.kept_count,
                                    0.0, out)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_noalloc_rejects_sizes_beyond_its_scratch(kvc):
    """A request whose scratch would exceed 2 MiB is refused before any launch."""
    from budgeted_kv_cache_gb300 import Policy, Pools, make_shape
    shape = make_shape(1, 75, 32, 4, 128, 4096)       # 300 units, 8 query heads per KV head
    # byte mode: the register decode kernel splits each unit over several
    # CTAs (bf16-only pools run one wave and need little scratch)
    u8 = torch.zeros(16, dtype=torch.uint8, device="cuda")
    pol = Policy(budget_bytes=1 << 20, capacity=4096, n_tags=1, n_layer_groups=1, tags=u8,
                 action_table=u8)
    need = kvc.kvc_decode_workspace_bytes(shape, pol)
    if need <= (2 << 20):
        pytest.skip("this device's split count keeps the request within the scratch")
    dummy = lambda dt=torch.float32: torch.empty(16, dtype=dt, device="cuda")
    pools = Pools(k_bf16=dummy(), v_bf16=dummy(), pos_out=dummy(torch.int32))
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_decode_attn_noalloc(shape, pol, dummy(), pools, dummy(torch.int32), 0.0, dummy())
    assert e.value.code == 3
