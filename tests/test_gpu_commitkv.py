"""CommitKV on the GPU against the oracle: deletion effects (Eqs. 6-7) and the
window record, lifecycle states (Eqs. 8-10), the greedy retirement set
(Eq. 11), pending-page protection (Eq. 12) and checkpoint flags (Eq. 13).

Tolerances.  The window outputs are sums of P v with P rounded to 16
significant bits (bf16 head + tail) and fp32 accumulation, so o_r is within
~1e-5 relative of the fp64 oracle; the page sums are fp32 over at most 64
tokens.  A page ratio ||u - s o|| / ((1 - s) ||o||) inherits about the same
relative error, so effects are compared at rel 2e-3 + abs 1e-6, record
outputs at 1e-3 of the row norm.  States, retirement and protection are
integers: states are compared exactly on identical fp32 effect inputs; the
retirement set is compared exactly after checking that no joint effect the
oracle tested lies within 1% of tau_joint (else the seed is unsuitable).
"""
import math

import numpy as np
import pytest
import torch

import oracle as o
import workloads as wl
from helpers import bits

pytestmark = pytest.mark.gpu

EFFECT_RTOL, EFFECT_ATOL = 2e-3, 1e-6
OUT_RTOL = 1e-3


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from budgeted_kv_cache_gb300 import build
    build.build()
    import budgeted_kv_cache_gb300 as lib
    lib.library()
    return lib


def f64(t):
    return o.bf16_bits_to_f32(bits(t)).astype(np.float64)


def run_effect(kvc, w, x, q):
    shape = kvc.make_shape(w.batch, w.n_layers, w.n_q_heads, w.n_kv_heads, 128, w.n_tokens)
    ws = torch.empty(kvc.kvc_deletion_effect_workspace_bytes(shape, w.window), dtype=torch.uint8,
                     device="cuda")
    rec = kvc.EffectRecord(shape, w.window, w.n_pages)
    eff = torch.full((w.batch, w.n_layers, w.n_pages), -7.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(w.n_units, dtype=torch.int32, device="cuda")
    kvc.kvc_deletion_effect(shape, x["k_cache"], x["v_cache"], q, w.window, 0.0, x["page_start"],
                            x["page_len"], eff, rec, ws, unit_status=status)
    torch.cuda.synchronize()
    return shape, eff, rec, status


def host_pages(x, b):
    st = x["page_start"][b].cpu().numpy()
    ln = x["page_len"][b].cpu().numpy()
    return [(int(s), int(n)) for s, n in zip(st, ln)]


def assert_effect_close(gpu, ref, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    both_inf = np.isinf(gpu) & np.isinf(ref)
    err = np.where(both_inf, 0.0, np.abs(gpu - ref))
    bad = np.nonzero(~(err <= EFFECT_RTOL * np.abs(ref) + EFFECT_ATOL))[0]
    assert bad.size == 0, f"{what}: pages {bad} gpu={gpu[bad]} ref={ref[bad]}"


SHAPES = [(8, 2, 8), (10, 2, 8), (16, 2, 8), (4, 1, 1), (8, 2, 4)]   # H_q, H_kv, W: R = 32, 40, 64, 4, 16


@pytest.mark.parametrize("hq,hkv,W", SHAPES)
def test_deletion_effect_and_record_match_oracle(kvc, hq, hkv, W):
    w = wl.commitkv_effect_small(hq, hkv, W)
    x = wl.make_effect_inputs(w, "cuda")
    shape, eff, rec, status = run_effect(kvc, w, x, x["q_minus"])
    assert (status.cpu().numpy() == 0).all()
    scale = 1.0 / math.sqrt(128)
    G = w.group
    for b in range(w.batch):
        pages = host_pages(x, b)
        toks = [o.page_tokens(s, n) for s, n in pages]
        for l in range(w.n_layers):
            k, v, q = f64(x["k_cache"][b, l]), f64(x["v_cache"][b, l]), f64(x["q_minus"][b, l])
            ref = o.deletion_effect(k, v, q, scale, toks)
            assert_effect_close(eff[b, l].cpu().numpy(), ref, f"effect b={b} l={l}")
            for g in range(hkv):
                a, out = o.window_attention(k[g], v[g], q[g * G:(g + 1) * G], scale)
                go = rec.o[b, l, g * G:(g + 1) * G].reshape(G * W, 128).cpu().numpy()
                nrm = np.linalg.norm(out, axis=1, keepdims=True)
                assert np.all(np.abs(go - out) <= OUT_RTOL * nrm), f"o b={b} l={l} g={g}"
                lse = o.window_row_lse(k[g], q[g * G:(g + 1) * G], scale)
                glse = rec.lse[b, l, g * G:(g + 1) * G].reshape(-1).cpu().numpy()
                np.testing.assert_allclose(glse, lse, rtol=0, atol=1e-4)
                for p, E in enumerate(toks):
                    s_ref = a[:, E].sum(axis=1)
                    u_ref = a[:, E] @ v[g][E] if len(E) else np.zeros((G * W, 128))
                    gs = rec.s[b, l, p, g * G:(g + 1) * G].reshape(-1).cpu().numpy()
                    gu = rec.u[b, l, p, g * G:(g + 1) * G].reshape(G * W, 128).cpu().numpy()
                    np.testing.assert_allclose(gs, s_ref, rtol=OUT_RTOL, atol=1e-7)
                    assert np.all(np.abs(gu - u_ref) <= OUT_RTOL * nrm + 1e-7)


def test_bad_page_marks_the_sequence(kvc):
    w = wl.commitkv_effect_small()
    x = wl.make_effect_inputs(w, "cuda")
    x["page_start"][1, 3] = w.n_tokens - 4          # runs past T
    shape, eff, rec, status = run_effect(kvc, w, x, x["q_minus"])
    st = status.cpu().numpy().reshape(w.batch, -1)
    assert (st[0] == 0).all() and (st[1] == o.UNIT_BAD_INDEX).all()
    assert (eff[1, :, 3].cpu().numpy() == 0).all()


def _thresholds_from(r_plus, r_minus):
    """Thresholds under which the small workload has completion candidates."""
    rp = np.asarray(r_plus, np.float64)
    return o.CommitThresholds(tau_use=float(np.float32(np.quantile(r_minus, 0.5))),
                              tau_dead=float(np.float32(np.median(rp))),
                              rho_use=0.5, rho_dead=0.5, tau_joint=0.0)


def run_commit(kvc, shape, w, eff_m, eff_p, compared, rec_p, th, layer):
    B, NP = w.batch, w.n_pages
    state = torch.full((B, NP), 77, dtype=torch.uint8, device="cuda")
    retire = torch.full((B, NP), 77, dtype=torch.uint8, device="cuda")
    joint = torch.empty((B, NP), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvc.kvc_commit_workspace_bytes(shape, w.window), dtype=torch.uint8, device="cuda")
    kvc.kvc_commit_transition(shape, w.window, layer, eff_m, eff_p, compared, rec_p, state, retire, ws,
                              joint=joint, tau_use=th.tau_use, tau_dead=th.tau_dead, rho_use=th.rho_use,
                              rho_dead=th.rho_dead, tau_joint=th.tau_joint)
    torch.cuda.synchronize()
    return state.cpu().numpy(), retire.cpu().numpy(), joint.cpu().numpy()


def check_commit(kvc, w, x, th_fn, layer):
    scale = 1.0 / math.sqrt(128)
    shape, eff_m, _, _ = run_effect(kvc, w, x, x["q_minus"])
    _, eff_p, rec_p, _ = run_effect(kvc, w, x, x["q_plus"])
    rng = np.random.default_rng(5)
    compared = (rng.random((w.batch, w.n_pages)) < 0.9).astype(np.uint8)
    compared_t = torch.from_numpy(compared).cuda()
    rm = eff_m[:, layer].cpu().numpy()
    rp = eff_p[:, layer].cpu().numpy()
    n_tested = 0
    for b in range(w.batch):
        th = th_fn(rp[b], rm[b], compared[b])
        # the joint bound: between the smallest candidate R+ and twice it
        state_ref, _, _ = o.lifecycle_states(rm[b].astype(np.float64), rp[b].astype(np.float64),
                                             compared[b], th)
        cands = o.candidate_order(state_ref, rm[b], rp[b])
        assert len(cands) >= 2, "workload has too few completion candidates"
        th.tau_joint = float(np.float32(2.2 * float(rp[b][cands[0]])))
        state, retire, joint = run_commit(kvc, shape, w, eff_m, eff_p, compared_t, rec_p, th, layer)
        np.testing.assert_array_equal(state[b], state_ref)
        pages = host_pages(x, b)
        k, v, q = (f64(x["k_cache"][b, layer]), f64(x["v_cache"][b, layer]), f64(x["q_plus"][b, layer]))
        _, retire_ref, tried = o.commit_transition(k, v, q, scale, pages, rm[b].astype(np.float64),
                                                   rp[b].astype(np.float64), compared[b], th)
        assert all(abs(t - th.tau_joint) > 1e-2 * th.tau_joint for t in tried), "joint effect too close to the bound"
        np.testing.assert_array_equal(retire[b], retire_ref)
        assert_effect_close(joint[b][cands], tried, "joint effects")
        assert (joint[b][[i for i in range(w.n_pages) if i not in cands]] == -1).all()
        n_tested += len(cands)
    return n_tested


def test_commit_transition_matches_oracle(kvc):
    w = wl.commitkv_effect_small()
    x = wl.make_effect_inputs(w, "cuda")

    def th_fn(rp, rm, cmp):
        return o.CommitThresholds(tau_use=float(np.float32(np.quantile(rm[cmp > 0], 0.5))),
                                  tau_dead=float(np.float32(np.median(rp[cmp > 0]))),
                                  rho_use=0.5, rho_dead=0.5, tau_joint=0.0)

    for layer in range(w.n_layers):
        assert check_commit(kvc, w, x, th_fn, layer) >= 4


def test_protect_pending_matches_oracle(kvc):
    B, L, NP = 3, 2, 300
    rng = np.random.default_rng(11)
    rm = rng.random((B, L, NP)).astype(np.float32)
    rm[0, 1, 10:20] = rm[0, 1, 5]                      # ties go to the lower index
    pending = (rng.random((B, NP)) < 0.4).astype(np.uint8)
    lens = rng.integers(1, 17, size=(B, NP)).astype(np.int32)
    shape = kvc.make_shape(B, L, 8, 2, 128, 4096)
    for budget, max_pages in ((256, 16), (100, 16), (4096, 1000), (0, 16)):
        prot = torch.empty((B, NP), dtype=torch.uint8, device="cuda")
        kvc.kvc_protect_pending(shape, 1, torch.from_numpy(rm).cuda(), torch.from_numpy(pending).cuda(),
                                torch.from_numpy(lens).cuda(), budget, max_pages, prot)
        torch.cuda.synchronize()
        for b in range(B):
            ref = o.protect_pending(rm[b, 1].astype(np.float64), lens[b], pending[b], budget, max_pages)
            np.testing.assert_array_equal(prot[b].cpu().numpy(), ref)


def test_commit_flags_match_oracle(kvc):
    B, T, NP = 2, 5000, 40
    rng = np.random.default_rng(3)
    starts = np.sort(rng.choice(T // 64, size=(B, NP), replace=True), axis=1)
    starts = np.stack([np.sort(rng.choice(T // 64, size=NP, replace=False)) for _ in range(B)]) * 64
    lens = rng.integers(0, 65, size=(B, NP)).astype(np.int32)
    retire = (rng.random((B, NP)) < 0.3).astype(np.uint8)
    protect = (rng.random((B, NP)) < 0.2).astype(np.uint8)
    flags = rng.integers(0, 3, size=(B, T)).astype(np.uint8)
    ft = torch.from_numpy(flags).cuda()
    kvc.kvc_commit_flags(B, T, torch.from_numpy(starts.astype(np.int32)).cuda(),
                         torch.from_numpy(lens).cuda(), torch.from_numpy(retire).cuda(),
                         torch.from_numpy(protect).cuda(), ft)
    torch.cuda.synchronize()
    for b in range(B):
        pages = list(zip(starts[b].tolist(), lens[b].tolist()))
        ref = o.commit_flags(T, pages, retire[b], protect[b], flags[b])
        np.testing.assert_array_equal(ft[b].cpu().numpy(), ref)


def test_full_size_effect_and_commit(kvc):
    """Qwen3-8B layout, one layer, T = 131072, W = 8, 64 pages of 16 tokens
    (the benchmark's deletion-effect workload), with the page's thresholds."""
    w = wl.commitkv_effect_128k()
    x = wl.make_effect_inputs(w, "cuda")
    shape, eff_m, _, status = run_effect(kvc, w, x, x["q_minus"])
    _, eff_p, rec_p, _ = run_effect(kvc, w, x, x["q_plus"])
    assert (status.cpu().numpy() == 0).all()
    scale = 1.0 / math.sqrt(128)
    k, v = f64(x["k_cache"][0, 0]), f64(x["v_cache"][0, 0])
    pages = host_pages(x, 0)
    toks = [o.page_tokens(s, n) for s, n in pages]
    ref_m = o.deletion_effect(k, v, f64(x["q_minus"][0, 0]), scale, toks)
    ref_p = o.deletion_effect(k, v, f64(x["q_plus"][0, 0]), scale, toks)
    assert_effect_close(eff_m[0, 0].cpu().numpy(), ref_m, "R- full size")
    assert_effect_close(eff_p[0, 0].cpu().numpy(), ref_p, "R+ full size")
    # the page's thresholds (CommitKV Sec. 4.1), on identical fp32 inputs
    th = o.CommitThresholds(*(float(np.float32(t)) for t in (0.05, 0.01, 0.75, 0.25, 0.01)))
    compared = torch.ones((1, w.n_pages), dtype=torch.uint8, device="cuda")
    state, retire, joint = run_commit(kvc, shape, w, eff_m, eff_p, compared, rec_p, th, 0)
    rm = eff_m[0, 0].cpu().numpy().astype(np.float64)
    rp = eff_p[0, 0].cpu().numpy().astype(np.float64)
    state_ref, _, _ = o.lifecycle_states(rm, rp, np.ones(w.n_pages), th)
    np.testing.assert_array_equal(state[0], state_ref)
    assert (state[0] == o.STATE_COMPLETION).sum() >= 1
    _, retire_ref, tried = o.commit_transition(k, v, f64(x["q_plus"][0, 0]), scale, pages, rm, rp,
                                               np.ones(w.n_pages), th)
    if all(abs(t - th.tau_joint) > 1e-2 * th.tau_joint for t in tried):
        np.testing.assert_array_equal(retire[0], retire_ref)
