"""Shared helpers of the GPU parity tests: unit extraction and comparisons."""
import math

import numpy as np
import torch

import oracle as o
import workloads as wl

SCORE_RTOL = 1e-2      # scores: relative 1e-2 ...
SCORE_ATOL = 1e-6      # ... with an absolute floor for near-zero mass
DECODE_ATOL = 2e-2     # decode outputs: max-abs 2e-2


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 / fp16 tensor -> uint16 bit patterns on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def unit_inputs(w, x, u):
    """Host copies of one unit's inputs (bf16 as bits)."""
    b, l, g = wl.unit_coords(w, u)
    G = w.group
    out = dict(
        k=bits(x["k_cache"][b, l, g]), v=bits(x["v_cache"][b, l, g]),
        q=bits(x["q_window"][b, l, g * G:(g + 1) * G]),
        qd=bits(x["q_decode"][b, l, g * G:(g + 1) * G]),
        pos=x["pos_in"][u].cpu().numpy(),
        bonus=x["bonus"][b].cpu().numpy() if "bonus" in x else None,
        flags=x["flags"][b].cpu().numpy() if "flags" in x else None,
        tags=x["tags"][b].cpu().numpy() if "tags" in x else None,
        group=o.layer_group(l, w.n_layers, w.n_layer_groups) if w.byte_mode else 0,
    )
    return out


def params_of(w) -> o.PassParams:
    return o.PassParams(budget_tokens=w.budget_tokens, budget_bytes=w.budget_bytes,
                        n_sink=w.n_sink, n_recent=w.n_recent, page_size=w.page_size,
                        renumber=w.renumber, quant_mode=w.quant_mode,
                        n_layer_groups=w.n_layer_groups)


def assert_scores_close(gpu, ref, what="scores"):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    bound = SCORE_RTOL * np.abs(ref) + SCORE_ATOL
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {ref.size} outside tolerance; first "
                           f"{bad[:5]} gpu={gpu[bad[:5]]} ref={ref[bad[:5]]}")


def kept_lists(pass_, u):
    """Per-pool kept token indices of unit u from a CompactionPass."""
    cnt = pass_.kept_count[:, u].cpu().numpy()
    idx = pass_.kept_idx[:, u].cpu().numpy()
    return {a: idx[a - 1, :cnt[a - 1]] for a in (o.ACT_INT4, o.ACT_INT8, o.ACT_BF16)}


def assert_selection_consistent(ref_scores, kept_gpu, kept_ref, k_th_key):
    """End-to-end selection check with independently computed scores.

    Index sets may differ only where two scores sit within the score tolerance
    of the selection threshold.
    """
    diff = np.setxor1d(kept_gpu, kept_ref)
    if diff.size == 0:
        return
    thr = float(k_th_key)
    near = np.abs(ref_scores[diff].astype(np.float64) - thr) <= 2 * (SCORE_RTOL * abs(thr) + SCORE_ATOL)
    assert near.all(), f"kept sets differ away from the threshold: {diff[~near][:10]}"


def unit_pools_from_gpu(pass_, u, w):
    """Pools of unit u read back from the device, in the oracle's format."""
    res = {}
    cnt = pass_.kept_count[:, u].cpu().numpy()
    P = pass_.pools
    for a in (o.ACT_INT4, o.ACT_INT8, o.ACT_BF16):
        pi = a - 1
        n = int(cnt[pi])
        pool = o.Pool(action=a, idx=pass_.kept_idx[pi, u, :n].cpu().numpy())
        pool.pos = P.pos_out[pi, u, :n].cpu().numpy()
        pool.orig_pos = P.orig_pos_out[pi, u, :n].cpu().numpy()
        if a == o.ACT_BF16:
            pool.k, pool.v = bits(P.k_bf16[u, :n]), bits(P.v_bf16[u, :n])
        elif n == 0:
            pool.k = pool.v = None
        else:
            kc = P.k_i8 if a == o.ACT_INT8 else P.k_i4
            vc = P.v_i8 if a == o.ACT_INT8 else P.v_i4
            ks = P.k_i8_scale if a == o.ACT_INT8 else P.k_i4_scale
            vs = P.v_i8_scale if a == o.ACT_INT8 else P.v_i4_scale
            pool.k, pool.v = kc[u, :n].cpu().numpy(), vc[u, :n].cpu().numpy()
            pool.k_scale = ks[u, :n].float().cpu().numpy()
            pool.v_scale = vs[u, :n].float().cpu().numpy()
            if a == o.ACT_INT8:
                pool.k, pool.v = pool.k.view(np.int8), pool.v.view(np.int8)
        res[a] = pool
    return res


def assert_pools_equal(gpu_pools, ref_pools):
    for a, rp in ref_pools.items():
        gp = gpu_pools[a]
        assert np.array_equal(gp.idx, rp.idx), f"pool {a}: indices differ"
        if rp.idx.size == 0:
            continue
        assert np.array_equal(gp.pos, rp.pos), f"pool {a}: positions differ"
        assert np.array_equal(gp.orig_pos, rp.orig_pos), f"pool {a}: original positions differ"
        gk = np.asarray(gp.k).view(np.uint8) if a != o.ACT_BF16 else gp.k
        rk = np.asarray(rp.k).view(np.uint8) if a != o.ACT_BF16 else rp.k
        gv = np.asarray(gp.v).view(np.uint8) if a != o.ACT_BF16 else gp.v
        rv = np.asarray(rp.v).view(np.uint8) if a != o.ACT_BF16 else rp.v
        nk = int((gk != rk).sum())
        assert nk == 0, f"pool {a}: {nk} key elements differ"
        assert np.array_equal(gv, rv), f"pool {a}: value elements differ"
        if a != o.ACT_BF16:
            assert np.array_equal(gp.k_scale, rp.k_scale), f"pool {a}: key scales differ"
            assert np.array_equal(gp.v_scale, rp.v_scale), f"pool {a}: value scales differ"


def kth_threshold(scores, kept_ref, forced_mask):
    """Smallest score among the kept non-forced items (the selection threshold)."""
    sel = np.setdiff1d(kept_ref, np.nonzero(forced_mask)[0])
    if sel.size == 0:
        return math.inf
    return float(np.min(scores[sel]))


# ------------------------------------------------------------------ oracle compaction in a process pool

_POOL_TABLES = {}


def _pool_init(cos, sin):
    _POOL_TABLES["cos"], _POOL_TABLES["sin"] = cos, sin


def _pool_compact(job):
    k, v, pos, act, prm = job
    return o.compact_unit(k, v, pos, act, prm, _POOL_TABLES["cos"], _POOL_TABLES["sin"])


def oracle_compact_many(jobs, cos, sin, processes=None):
    """oracle.compact_unit over many units in a pool of spawned processes
    (spawned, not forked: the parent has an initialised CUDA context)."""
    import multiprocessing as mp
    import os
    n = processes or max(1, min(16, os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(n, initializer=_pool_init, initargs=(cos, sin)) as pool:
        return pool.map(_pool_compact, jobs, chunksize=max(1, len(jobs) // (4 * n)))
