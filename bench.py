"""Benchmark of the budgeted KV-cache compaction pass on GB300.

One step = one full compaction pass (kvc_score -> kvc_select ->
kvc_compact_rerotate_quant) over every (layer, KV head) unit of the
Qwen3-8B-shaped single-session workload: 36 layers x 8 KV heads, 32 query
heads, head_dim 128, T = 32,768 cached tokens, window 64, budget 2,048
(4 sinks + 128 recent + top-k), bounded positions (renumber + re-rotation),
foresight bonus on 4 spans.  Inputs are seeded synthetic tensors.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  Multi-GPU (torchrun, one rank per GPU): every rank
compacts its own session of the same shape (weak scaling, no collective on
the data path); the timed region is bracketed by barriers and the slowest
rank's time is reported.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "KV tokens compacted/sec per layer·head and % of roofline (HBM GB/s or TC util)"

# DRAM bytes (read + write) of one score_kernel launch, per unit: the full
# 288-unit launch of this workload captured with ncu's DRAM byte counters (one
# replay pass, the summary kept with the other profiles).  Valid while
# the kernel and its launch plan (score_tc.cu, kvc_api.cu) are the captured
# ones (the kernel's source and the plan_score function that sizes its work
# items), else reported as null.
SCORE_TRAFFIC = {"sha1": "841fba020628687e94b8620e0130905146bcd4ba", "bytes_per_unit": (4666309632 + 27208192) / 288}
UNIT = "tokens/s (summed over layer x KV-head units)"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


POOL_INT4, POOL_INT8, POOL_BF16 = 0, 1, 2


def kv_row_bytes(w, pool: int) -> int:
    """Stored bytes of one kept row's key and value in a pool (codes + scales)."""
    d = w.head_dim
    if pool == POOL_BF16:
        return 2 * 2 * d
    scales = 2 * (d // 32) if w.quant_mode == wl.QUANT_G32_BF16 else 2
    return 2 * ((d if pool == POOL_INT8 else d // 2) + scales)


def algorithmic_bytes(w, kept_rows=None) -> dict:
    """Bytes the method must move once per pass, per stage.

    kept_rows: {pool: kept rows summed over all units} (the run's kept
    counts); default: the token budget of every unit, in the bf16 pool.
      score   keys once, window queries, scores written (and page scores),
              the per-sequence bonus
      select  scores (or page scores) read, tags / flags read, kept indices
              written
      compact per kept row: its index and old position read, its bf16 key and
              value read, its pool bytes and its new / original position
              written; the rotary table rows touched (renumbering)
    """
    U, T, d, R, B = w.n_units, w.n_tokens, w.head_dim, w.rows_per_unit, w.batch
    P = w.page_size
    if kept_rows is None:
        kept_rows = {POOL_BF16: U * w.budget_tokens}
    n_kept = sum(kept_rows.values())
    n_items = T // P
    score = U * T * 2 * d + U * R * 2 * d + U * T * 4 + (U * n_items * 4 if P > 1 else 0) + \
        (B * T * 4 if w.bonus_spans else 0)
    select = U * n_items * 4 + (B * T if w.tag_probs is not None else 0) + \
        (B * n_items if (w.protect_pages or w.retire_pages) else 0) + n_kept * 4
    compact = n_kept * (4 + 4 + 2 * 2 * d + 4 + 4) + sum(n * kv_row_bytes(w, p) for p, n in kept_rows.items())
    if w.renumber:
        compact += min(w.max_pos, T) * d * 4            # cos + sin rows touched (fp32, d/2 each)
    return dict(score=score, select=select, compact=compact, total=score + select + compact)


def kept_rows_of(kept_count) -> dict:
    """{pool: rows summed over units} from a [3][U] kept-count tensor."""
    c = kept_count.sum(dim=1).tolist()
    return {POOL_INT4: int(c[0]), POOL_INT8: int(c[1]), POOL_BF16: int(c[2])}


def _code(src: str) -> str:
    """Source text without comments and blank lines (the key ignores comment edits)."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip())


def score_traffic(n_units: int):
    import hashlib
    csrc = os.path.join(ROOT, "budgeted_kv_cache_gb300", "csrc")
    h = hashlib.sha1()
    with open(os.path.join(csrc, "score_tc.cu")) as f:
        h.update(_code(f.read()).encode())
    with open(os.path.join(csrc, "kvc_api.cu")) as f:
        api = f.read()
    i = api.find("kvc_status plan_score(")
    h.update(_code(api[i:api.index("\n}\n", i) + 3]).encode() if i >= 0 else b"")
    if h.hexdigest() != SCORE_TRAFFIC["sha1"]:
        return None
    return SCORE_TRAFFIC["bytes_per_unit"] * n_units


def algorithmic_flops(w) -> int:
    return 2 * w.n_units * w.rows_per_unit * w.n_tokens * w.head_dim


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


from budgeted_kv_cache_gb300.sharding import barrier, max_over_ranks  # noqa: E402


# ---------------------------------------------------------------------------- oracle timing

def oracle_sample(w, x_host, seconds: float, max_units: int):
    """Time the CPU oracle (score + select + compact) on whole units until `seconds` pass."""
    import oracle as o
    cos, sin = x_host["rope_cos"].numpy(), x_host["rope_sin"].numpy()
    prm = o.PassParams(budget_tokens=w.budget_tokens, budget_bytes=w.budget_bytes,
                       n_sink=w.n_sink, n_recent=w.n_recent, page_size=w.page_size,
                       renumber=w.renumber, quant_mode=w.quant_mode,
                       n_layer_groups=w.n_layer_groups)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    done, t0 = 0, time.perf_counter()
    rng = np.random.default_rng(0)
    units = rng.permutation(w.n_units)
    while done < max_units:
        u = int(units[done % w.n_units])
        b, l, g = wl.unit_coords(w, u)
        G = w.group
        o.run_unit(bits(x_host["k_cache"][b, l, g]), bits(x_host["v_cache"][b, l, g]),
                   bits(x_host["q_window"][b, l, g * G:(g + 1) * G]), x_host["pos_in"][u].numpy(),
                   prm, cos, sin, bonus=x_host["bonus"][b].numpy() if "bonus" in x_host else None)
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:       # BLAS uses every host core by default
        threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return done, dt, threads


def _config(w) -> dict:
    """The workload both arms name in their JSON line."""
    return {"workload": w.name, "units": w.n_units, "n_tokens": w.n_tokens,
            "budget": w.budget_tokens, "window": w.window, "head_dim": w.head_dim,
            "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "layers": w.n_layers}


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    # the oracle's own inputs: a one-layer, one-KV-head slice of the workload
    ws = w.replace(n_layers=1, n_kv_heads=1, n_q_heads=w.group)
    x = wl.make_inputs(ws, device="cpu")
    per_step = []
    n_rows = 0
    threads = 1
    for step in range(args.warmup + args.steps):
        done, dt, threads = oracle_sample(ws, x, seconds=0.0, max_units=1)
        if step >= args.warmup:
            per_step.append(dt)
            n_rows += done * ws.n_tokens
    total = sum(per_step)
    value = n_rows / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"1 of {w.n_units} (layer, KV head) units per step, "
                                   f"score+select+compact, numpy fp64"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def commitkv_stage(dev, stream, flush, repeats: int = 10) -> dict:
    """CommitKV (Sec. 3.2-3.3): deletion effects of 64 pages over the
    post-commit window of one layer (Qwen3-8B heads, T = 131072, W = 8) and the
    commit call (states + greedy joint validation), each timed after three
    warm-ups as the mean of `repeats` calls with L2 flushed before each."""
    import budgeted_kv_cache_gb300 as kvc_mod
    ev = lambda: torch.cuda.Event(enable_timing=True)
    we = wl.commitkv_effect_128k()
    xe = wl.make_effect_inputs(we, dev)
    es = kvc_mod.make_shape(we.batch, we.n_layers, we.n_q_heads, we.n_kv_heads, 128, we.n_tokens)
    ews = torch.empty(kvc_mod.kvc_deletion_effect_workspace_bytes(es, we.window), dtype=torch.uint8,
                      device=dev)
    rec_m = kvc_mod.EffectRecord(es, we.window, we.n_pages, dev)
    rec_p = kvc_mod.EffectRecord(es, we.window, we.n_pages, dev)
    eff_m = torch.empty((we.batch, we.n_layers, we.n_pages), device=dev)
    eff_p = torch.empty_like(eff_m)
    cws = torch.empty(kvc_mod.kvc_commit_workspace_bytes(es, we.window), dtype=torch.uint8, device=dev)
    cmp_ = torch.ones((we.batch, we.n_pages), dtype=torch.uint8, device=dev)
    st_ = torch.empty((we.batch, we.n_pages), dtype=torch.uint8, device=dev)
    rt_ = torch.empty_like(st_)
    kvc_mod.kvc_deletion_effect(es, xe["k_cache"], xe["v_cache"], xe["q_minus"], we.window, 0.0,
                                xe["page_start"], xe["page_len"], eff_m, rec_m, ews, stream=stream)
    fns = {
        "commitkv_effect": lambda: kvc_mod.kvc_deletion_effect(
            es, xe["k_cache"], xe["v_cache"], xe["q_plus"], we.window, 0.0, xe["page_start"],
            xe["page_len"], eff_p, rec_p, ews, stream=stream),
        "commitkv_commit": lambda: kvc_mod.kvc_commit_transition(
            es, we.window, 0, eff_m, eff_p, cmp_, rec_p, st_, rt_, cws, stream=stream),
    }
    out = {}
    for name, fn in fns.items():
        for _ in range(3):
            fn()
        t_v = []
        for _ in range(repeats):
            flush.fill_(1)
            d0, d1 = ev(), ev()
            d0.record(stream)
            fn()
            d1.record(stream)
            torch.cuda.synchronize()
            t_v.append(d0.elapsed_time(d1))
        out[name] = statistics.mean(t_v)
    kv_bytes = 2 * we.n_units * we.n_tokens * 128 * 2
    out["commitkv_effect_gbs"] = kv_bytes / (out["commitkv_effect"] * 1e-3) / 1e9
    out["commitkv_retired_pages"] = int(rt_.sum().item())
    return out


# ---------------------------------------------------------------------------- the other workloads

def _timed(fn, stream, flush, repeats):
    """Mean ms of `repeats` calls of fn (CUDA events on `stream`, L2 flushed before each)."""
    ev = lambda: torch.cuda.Event(enable_timing=True)
    t = []
    for _ in range(repeats):
        flush.fill_(1)
        a, b = ev(), ev()
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        t.append(a.elapsed_time(b))
    return statistics.mean(t)


def _roofline(w, ab_total, flops, t_ms, hbm, tc):
    t_roof = max(ab_total / (hbm * 1e9), flops / (tc * 1e12)) * 1e3
    return {"t_roof_ms": t_roof, "frac": t_roof / t_ms,
            "bound": "hbm" if ab_total / hbm >= flops / (tc * 1e3) else "tensor",
            "algorithmic_bytes": ab_total, "algorithmic_flops": flops,
            "gbs": ab_total / (t_ms * 1e-3) / 1e9}


def time_workload(w, dev, stream, flush, steps, warmup, hbm, tc) -> dict:
    """One compaction pass of workload w (score -> select -> compact) on
    device-resident inputs: mean of `steps` passes after `warmup`, L2 flushed
    before each; per-stage times, rows/s, GB/s on the algorithmic bytes and
    the fraction of the pass roofline.  A paged workload also times one
    decode step over its compacted cache."""
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    x = wl.make_inputs(w, device=dev)
    p = pass_for_workload(w, inputs=x, device=dev)
    args = (x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"], x["rope_sin"], x.get("bonus"))
    for _ in range(warmup):
        p.run(*args, stream=stream)
    torch.cuda.synchronize()
    assert int(p.score_status.abs().sum()) == 0 and int(p.compact_status.abs().sum()) == 0
    ev = lambda: torch.cuda.Event(enable_timing=True)
    st = {"score": [], "select": [], "compact": []}
    for _ in range(steps):
        flush.fill_(1)
        m = [ev() for _ in range(4)]
        m[0].record(stream)
        p.score(x["k_cache"], x["q_window"], x.get("bonus"), stream=stream)
        m[1].record(stream)
        p.select(stream=stream)
        m[2].record(stream)
        p.compact(x["k_cache"], x["v_cache"], x["pos_in"], x["rope_cos"], x["rope_sin"], stream=stream)
        m[3].record(stream)
        torch.cuda.synchronize()
        for i, k in enumerate(st):
            st[k].append(m[i].elapsed_time(m[i + 1]))
    stages = {k: statistics.mean(v) for k, v in st.items()}
    t = sum(stages.values())
    kept = kept_rows_of(p.kept_count)
    ab = algorithmic_bytes(w, kept)
    out = {"workload": w.name, "units": w.n_units, "n_tokens": w.n_tokens, "ms_per_step": t,
           "value": w.n_units * w.n_tokens / (t * 1e-3), "unit": UNIT, "stages_ms": stages,
           "kept_rows": kept, "roofline": _roofline(w, ab["total"], algorithmic_flops(w), t, hbm, tc),
           "steps": steps, "warmup": warmup}
    if w.page_size > 1:
        out["decode_ms"] = _timed(lambda: p.decode(x["q_decode"], stream=stream), stream, flush, steps)
    del x, p
    torch.cuda.empty_cache()
    return out


def time_session(w, dev, stream, hbm, tc, warmup=3) -> dict:
    """The million-token session in cycles: each cycle appends a chunk
    (the engine's KV write, timed apart) and compacts the cache back to the
    budget; sustained rows/s = rows appended over the summed pass time."""
    from budgeted_kv_cache_gb300.session import BoundedSession
    s0 = wl.session_start(w, dev)
    sess = BoundedSession(w.batch, w.n_layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.budget_tokens,
                          w.chunk, w.window, w.limit, w.n_sink, w.n_recent, device=dev)
    sess.start(s0["k0"], s0["v0"])
    ev = lambda: torch.cuda.Event(enable_timing=True)
    marks = []
    for c in range(-warmup, w.cycles):
        ch = wl.session_chunk(w, c, dev)              # drawn outside the timed events
        m = [ev() for _ in range(3)]
        m[0].record(stream)
        sess.append(ch["k"], ch["v"], stream=stream)
        m[1].record(stream)
        sess.compact(ch["q_window"], s0["rope_cos"], s0["rope_sin"], stream=stream)
        m[2].record(stream)
        if c >= 0:
            marks.append(m)
    torch.cuda.synchronize()
    p = sess.last_pass
    assert int(p.unit_status.abs().sum()) == 0 and int(p.compact_status.abs().sum()) == 0
    t_app = sum(m[0].elapsed_time(m[1]) for m in marks)
    t_pass = sum(m[1].elapsed_time(m[2]) for m in marks)
    rows = w.n_units * w.chunk * w.cycles
    ab = algorithmic_bytes(w)                          # one cycle: a pass over budget + chunk rows
    flops = algorithmic_flops(w)
    roof = _roofline(w, ab["total"] * w.cycles, flops * w.cycles, t_pass, hbm, tc)
    out = {"workload": w.name, "units": w.n_units, "cycles": w.cycles, "chunk": w.chunk,
           "cache_rows": w.n_tokens, "budget": w.budget_tokens, "limit": w.limit,
           "value": rows / (t_pass * 1e-3), "unit": "appended rows/s (summed over layer x KV-head units)",
           "ms_per_cycle": t_pass / w.cycles, "append_ms_per_cycle": t_app / w.cycles,
           "value_with_append": rows / ((t_pass + t_app) * 1e-3),
           "renumbered_cycles": int(sum(sess.renumbered[warmup:])), "roofline": roof,
           "l2": "not flushed between cycles: each cycle's chunk is written just before its compaction"}
    del sess, s0
    torch.cuda.empty_cache()
    return out


def run_configs(dev, stream, flush, hbm, tc, steps) -> dict:
    """Every other workload of the pages, one pass each (C2 is the headline)."""
    out = {}
    for key, mk in (("C1", wl.tiny), ("C3", wl.pask_batch16), ("C4", wl.commitkv_pages_128k),
                    ("C5A", wl.million_token_8l)):
        out[key] = time_workload(mk(), dev, stream, flush, steps=steps, warmup=3, hbm=hbm, tc=tc)
    out["C1"]["us_per_step"] = 1e3 * out["C1"]["ms_per_step"]
    out["C5B"] = time_session(wl.million_token_sustained(), dev, stream, hbm, tc)
    return out


# ---------------------------------------------------------------------------- GPU arm

def run_gpu(args, w, world, rank, local):
    import budgeted_kv_cache_gb300 as kvc
    from budgeted_kv_cache_gb300 import build
    from budgeted_kv_cache_gb300.passes import pass_for_workload
    if rank == 0 or not os.path.exists(build.LIB):
        build.build()
    barrier(world)
    kvc.library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # each rank compacts its own session (different seed)
    wr = w.replace(seed=w.seed + 1000 * rank)
    x = wl.make_inputs(wr, device=dev)
    p = pass_for_workload(wr, inputs=x, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"],
              x["rope_sin"], x.get("bonus"), stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(p.unit_status.abs().sum()) == 0 and int(p.score_status.abs().sum()) == 0

    ev = lambda: torch.cuda.Event(enable_timing=True)
    marks = [[ev() for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    for s in range(args.steps):
        flush.fill_(float(s))                     # L2 flush outside the timed events
        m = marks[s]
        m[0].record(stream)
        p.score(x["k_cache"], x["q_window"], x.get("bonus"), stream=stream)
        m[1].record(stream)
        p.select(stream=stream)
        m[2].record(stream)
        p.compact(x["k_cache"], x["v_cache"], x["pos_in"], x["rope_cos"], x["rope_sin"],
                  stream=stream)
        m[3].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    t_score = [m[0].elapsed_time(m[1]) for m in marks]
    t_select = [m[1].elapsed_time(m[2]) for m in marks]
    t_compact = [m[2].elapsed_time(m[3]) for m in marks]
    t_pass = [a + b + c for a, b, c in zip(t_score, t_select, t_compact)]
    total_ms = max_over_ranks(sum(t_pass), world)

    # decode step, timed separately (consumer check, not part of the pass):
    # warm-up calls, then the mean of ten calls with L2 flushed before each
    for _ in range(3):
        p.decode(x["q_decode"], stream=stream)
    t_dec = []
    for _ in range(10):
        flush.fill_(1)
        d0, d1 = ev(), ev()
        d0.record(stream)
        p.decode(x["q_decode"], stream=stream)
        d1.record(stream)
        torch.cuda.synchronize()
        t_dec.append(d0.elapsed_time(d1))
    t_decode = statistics.mean(t_dec)

    # the engine's attention (PASK App. B.5) over the compacted pools plus 128
    # recent rows and the current rows, one and four queries per head, timed
    # separately like the decode step
    t_eng = {}
    if not w.byte_mode:
        import budgeted_kv_cache_gb300 as kvc_e
        ge = torch.Generator(device=dev)
        ge.manual_seed(7)
        Ue = w.n_units
        rec_cap = 128
        rk = torch.randn((Ue, rec_cap, w.head_dim), generator=ge, device=dev).to(torch.bfloat16)
        rv = torch.randn((Ue, rec_cap, w.head_dim), generator=ge, device=dev).to(torch.bfloat16)
        base_pos = w.n_tokens + 1
        rpos = (base_pos + torch.arange(rec_cap, device=dev, dtype=torch.int32)).expand(Ue, rec_cap).contiguous()
        rcnt = torch.full((Ue,), rec_cap, dtype=torch.int32, device=dev)
        for nq in (1, 4):
            ck = torch.randn((Ue, nq, w.head_dim), generator=ge, device=dev).to(torch.bfloat16)
            cv = torch.randn((Ue, nq, w.head_dim), generator=ge, device=dev).to(torch.bfloat16)
            cpos = (base_pos + rec_cap + torch.arange(nq, device=dev, dtype=torch.int32)).expand(Ue, nq).contiguous()
            ccnt = torch.full((Ue,), nq, dtype=torch.int32, device=dev)
            qe = torch.randn((w.batch, w.n_layers, w.n_q_heads, nq, w.head_dim), generator=ge,
                             device=dev).to(torch.bfloat16)
            qpos = (base_pos + rec_cap + torch.arange(nq, device=dev, dtype=torch.int32)).expand(w.batch, nq).contiguous()
            oute = torch.empty_like(qe)
            rec = kvc_e.bf16_rows(rk, rv, rpos, rcnt)
            cur = kvc_e.bf16_rows(ck, cv, cpos, ccnt)
            wsb = kvc_e.kvc_engine_attn_workspace_bytes(p.shape, p.policy, nq, rec, cur)
            wse = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
            fe = lambda: kvc_e.kvc_engine_attn(p.shape, p.policy, qe, nq, qpos, p.pools, p.kept_count,
                                               rec, cur, 0.0, oute, wse, stream=stream)
            for _ in range(3):
                fe()
            t_v = []
            for _ in range(10):
                flush.fill_(1)
                d0, d1 = ev(), ev()
                d0.record(stream)
                fe()
                d1.record(stream)
                torch.cuda.synchronize()
                t_v.append(d0.elapsed_time(d1))
            t_eng[f"engine_attn_{nq}q"] = statistics.mean(t_v)
        del rk, rv

    # one H2O decode step (PACE Sec. 3.1): window-1 scoring of the decode
    # query of every head over the whole cache, accumulated into the scores,
    # with the row statistics computed here (two passes) or supplied by the
    # caller's attention kernel (one pass); timed separately
    from budgeted_kv_cache_gb300 import kvc_score, kvc_score_workspace_bytes, SCORE_ACCUMULATE
    qd = x["q_decode"].reshape(w.batch, w.n_layers, w.n_q_heads, 1, w.head_dim)
    ws1 = torch.empty(kvc_score_workspace_bytes(p.shape, 1), dtype=torch.uint8, device=dev)
    lse1 = torch.full((w.n_units, w.group), 8.0, device=dev)
    t_h2o = {}
    for name, lse_arg in (("h2o_step_two_pass", None), ("h2o_step_caller_lse", lse1)):
        step1 = lambda: kvc_score(p.shape, x["k_cache"], qd, 1, 0.0, None, 1, SCORE_ACCUMULATE,
                                  p.scores, None, p.score_status, ws1, stream=stream, row_lse=lse_arg)
        for _ in range(3):
            step1()
        t_s = []
        for _ in range(10):
            flush.fill_(1)
            d0, d1 = ev(), ev()
            d0.record(stream)
            step1()
            d1.record(stream)
            torch.cuda.synchronize()
            t_s.append(d0.elapsed_time(d1))
        t_h2o[name] = statistics.mean(t_s)
    del ws1, lse1

    # selection variants, timed separately: SnapKV pooling (kernel 7, max) of
    # the score buffer, and CommitKV Eq. 4's shared index set (per-sequence
    # score sum, one selection per sequence, kept lists copied to the units)
    from budgeted_kv_cache_gb300 import (kvc_pool_scores, kvc_shared_scores, kvc_select,
                                         kvc_broadcast_kept, make_shape, SCORE_POOL_MAX)
    pooled = torch.empty_like(p.scores)
    shared = torch.empty((w.batch, w.n_tokens), device=dev)
    seq_shape = make_shape(w.batch, 1, 1, 1, w.head_dim, w.n_tokens)
    kept_s = torch.empty((3, w.batch, p.policy.capacity), dtype=torch.int32, device=dev)
    cnt_s = torch.empty((3, w.batch), dtype=torch.int32, device=dev)
    st_s = torch.empty(w.batch, dtype=torch.int32, device=dev)

    def shared_set():
        kvc_shared_scores(p.shape, p.scores, shared, stream=stream)
        kvc_select(seq_shape, p.policy, shared, kept_s, cnt_s, st_s, stream=stream)
        kvc_broadcast_kept(p.shape, p.policy, kept_s, cnt_s, p.kept_idx, p.kept_count, stream=stream)

    variants = {"pool_scores_max7": lambda: kvc_pool_scores(p.scores, pooled, 7, SCORE_POOL_MAX,
                                                            stream=stream)}
    if not w.byte_mode and w.page_size == 1:
        variants["shared_index_set"] = shared_set
    t_var = {}
    for name, fn in variants.items():
        for _ in range(3):
            fn()
        t_v = []
        for _ in range(10):
            flush.fill_(1)
            d0, d1 = ev(), ev()
            d0.record(stream)
            fn()
            d1.record(stream)
            torch.cuda.synchronize()
            t_v.append(d0.elapsed_time(d1))
        t_var[name] = statistics.mean(t_v)
    del pooled, shared
    p.select(stream=stream)             # restore the per-unit kept lists
    torch.cuda.synchronize()

    # compaction through the reference store (PACE Sec. 3.2), timed separately:
    # every cached key has a reference valid at its current position (the
    # stored key itself), so each kept key is checked and re-derived from it
    t_cref = None
    if not w.byte_mode:
        from budgeted_kv_cache_gb300 import kvc_compact_rerotate_quant_ref
        cap = p.policy.capacity
        rk_out = torch.empty((3, w.n_units, cap, w.head_dim), dtype=torch.bfloat16, device=dev)
        rp_out = torch.empty((3, w.n_units, cap), dtype=torch.int32, device=dev)
        cref = lambda: kvc_compact_rerotate_quant_ref(
            p.shape, p.policy, x["k_cache"], x["v_cache"], x["pos_in"], p.kept_idx, p.kept_count,
            x["rope_cos"], x["rope_sin"], x["rope_cos"].shape[0], x["k_cache"], x["pos_in"],
            rk_out, rp_out, p.pools, None, p.compact_status, stream=stream)
        for _ in range(3):
            cref()
        t_c = []
        for _ in range(10):
            flush.fill_(1)
            d0, d1 = ev(), ev()
            d0.record(stream)
            cref()
            d1.record(stream)
            torch.cuda.synchronize()
            t_c.append(d0.elapsed_time(d1))
        t_cref = statistics.mean(t_c)
        del rk_out, rp_out

    # the same pass captured once as a CUDA graph and replayed (launch overhead check)
    graph_ms = None
    try:
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"],
                  x["rope_sin"], x.get("bonus"), stream=gs)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs, capture_error_mode="thread_local"):
            p.run(x["k_cache"], x["v_cache"], x["q_window"], x["pos_in"], x["rope_cos"],
                  x["rope_sin"], x.get("bonus"), stream=gs)
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        t_g = []
        for _ in range(10):
            flush.fill_(1)
            d0, d1 = ev(), ev()
            d0.record()
            graph.replay()
            d1.record()
            torch.cuda.synchronize()
            t_g.append(d0.elapsed_time(d1))
        graph_ms = statistics.mean(t_g)
        del graph
    except Exception as exc:                     # reported, not fatal: the eager pass is the metric
        graph_ms = f"capture failed: {exc!r}"[:200]

    # CommitKV (Sec. 3.2-3.3), timed separately
    t_eff = None if args.no_commitkv else commitkv_stage(dev, stream, flush)

    # end to end through the C-ABI with host buffers, every step: the inputs
    # scoring reads whole (keys, window queries, bonus) and the rotary tables
    # are copied in from pinned host memory; values and positions stay in
    # pinned host memory and compaction reads their kept rows in place; the
    # compacted cache comes back.  The layers go in groups (nine by default):
    # the keys of group g + 1 are copied (side stream) while group g is
    # compacted and its results copied out, so only the last group's pass is
    # not hidden.
    e2e = None
    if not args.no_e2e:
        from budgeted_kv_cache_gb300.passes import pass_for_workload
        n_groups = args.e2e_groups if wr.batch == 1 and wr.n_layers % max(args.e2e_groups, 1) == 0 else 1
        wg = wr.replace(n_layers=wr.n_layers // n_groups)
        gpasses = [p] if n_groups == 1 else [pass_for_workload(wg, inputs=x, device=dev)
                                              for _ in range(n_groups)]
        copied = [n for n in ("k_cache", "q_window", "rope_cos", "rope_sin", "bonus") if n in x]
        in_place = ["v_cache", "pos_in"]
        host = {n: torch.empty(x[n].shape, dtype=x[n].dtype, pin_memory=True) for n in copied + in_place}
        for n in host:
            host[n].copy_(x[n])
        dev_in = {n: torch.empty_like(x[n]) for n in copied}
        Lg, Ug = wg.n_layers, wg.n_units

        def outs_of(q):
            return [q.pools.k_bf16, q.pools.v_bf16, q.pools.pos_out, q.kept_idx, q.kept_count, q.unit_status]

        host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs_of(q)]
                    for q in gpasses]
        kept_rows = sum(kept_rows_of(p.kept_count).values())
        h2d = sum(host[n].numel() * host[n].element_size() for n in copied) + \
            kept_rows * (wr.head_dim * 2 + 4)               # kept value rows and positions, read in place
        d2h = sum(t.numel() * t.element_size() for ts in host_out for t in ts)
        side = torch.cuda.Stream(dev)

        def e2e_step():
            arrived = []
            with torch.cuda.stream(side):
                side.wait_stream(stream)                  # the previous step is done with the buffers
                for n in ("rope_cos", "rope_sin", "bonus"):
                    if n in dev_in:
                        dev_in[n].copy_(host[n], non_blocking=True)
                for g in range(n_groups):
                    for n in ("k_cache", "q_window"):
                        dev_in[n][:, g * Lg:(g + 1) * Lg].copy_(host[n][:, g * Lg:(g + 1) * Lg],
                                                                non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(side)
                    arrived.append(e)
            for g, q in enumerate(gpasses):
                l0, l1, u0, u1 = g * Lg, (g + 1) * Lg, g * Ug, (g + 1) * Ug
                stream.wait_event(arrived[g])
                q.run(dev_in["k_cache"][:, l0:l1], host["v_cache"][:, l0:l1], dev_in["q_window"][:, l0:l1],
                      host["pos_in"][u0:u1], dev_in["rope_cos"], dev_in["rope_sin"], dev_in.get("bonus"),
                      stream=stream)
                for h, t in zip(host_out[g], outs_of(q)):
                    h.copy_(t, non_blocking=True)

        ref_out = []                          # the same group passes from device-resident inputs
        for g, q in enumerate(gpasses):
            l0, l1, u0, u1 = g * Lg, (g + 1) * Lg, g * Ug, (g + 1) * Ug
            q.run(x["k_cache"][:, l0:l1], x["v_cache"][:, l0:l1], x["q_window"][:, l0:l1], x["pos_in"][u0:u1],
                  x["rope_cos"], x["rope_sin"], x.get("bonus"), stream=stream)
            ref_out.append([t.clone() for t in outs_of(q)])
        e2e_step()
        torch.cuda.synchronize()
        same = all(torch.equal(h, r.cpu()) for g in range(n_groups) for h, r in zip(host_out[g], ref_out[g]))
        del ref_out
        n_e2e = max(1, min(args.steps, 5))
        barrier(world)
        e0, e1 = ev(), ev()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(e0.elapsed_time(e1), world) / n_e2e
        e2e = {"value": world * wr.n_units * wr.n_tokens / (t_e2e * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e,
               "steps": n_e2e,
               "host_resident": "v_cache and pos_in in pinned host memory, kept rows read in place",
               "layer_groups": n_groups,
               "matches_device_resident_pass": same}
        del host, dev_in, host_out, gpasses

    hbm, tc, src = _peaks()
    configs = None
    if world == 1 and not args.no_configs:
        configs = run_configs(dev, stream, flush, hbm, tc, steps=max(3, min(args.steps, 5)))
    if rank != 0:
        return
    ab = algorithmic_bytes(wr, kept_rows_of(p.kept_count))
    flops = algorithmic_flops(wr)
    ms_step = total_ms / args.steps
    score_ms = statistics.mean(t_score)
    achieved = ab["score"] / (score_ms * 1e-3) / 1e9
    t_roof = max(ab["total"] / (hbm * 1e9), flops / (tc * 1e12))
    value = world * wr.n_units * wr.n_tokens / (ms_step * 1e-3)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        ws = wr.replace(n_layers=1, n_kv_heads=1, n_q_heads=wr.group)
        xh = wl.make_inputs(ws, device="cpu")
        done, dt, threads = oracle_sample(ws, xh, seconds=args.cpu_seconds, max_units=1024)
        cpu = {"value": done * ws.n_tokens / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{done} passes over one whole (layer, KV head) unit of {wr.name} "
                         f"(score+select+compact, numpy fp64), {dt:.1f} s"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**_config(wr), "parallelism": f"replicas x{world}",
                   "l2": "256 MiB buffer written between timed steps; K/V inputs (2.4 GB each) exceed L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": score_traffic(wr.n_units),
                     "kernel": "score_kernel",
                     "peak_source": src,
                     "algorithmic_bytes_per_launch": ab["score"],
                     "tc_tflops_algorithmic": flops / (score_ms * 1e-3) / 1e12},
        "stages_ms": {"score": score_ms, "select": statistics.mean(t_select),
                      "compact": statistics.mean(t_compact), "decode": t_decode,
                      "compact_reference_store": t_cref, **t_eng, **t_h2o, **t_var, **(t_eff or {})},
        "pass_roofline": {"t_roof_ms": 1e3 * t_roof, "frac": 1e3 * t_roof / ms_step,
                          "algorithmic_bytes": ab["total"], "algorithmic_flops": flops,
                          # informational: one exponential per window logit (U R T) at the
                          # measured 30 ex2 results per clock per SM and the sampled SM clock
                          "t_exp_ms": 1e3 * wr.n_units * wr.rows_per_unit * wr.n_tokens
                                      / (30.0 * torch.cuda.get_device_properties(dev).multi_processor_count
                                         * ((clocks or {}).get("sm_mhz") or 2070.0) * 1e6)},
        # every stage on its own algorithmic bytes (HBM-bound stages)
        "stage_rooflines": {
            k: {"algorithmic_bytes": ab[k], "gbs": ab[k] / (t * 1e-3) / 1e9,
                "frac": ab[k] / (t * 1e-3) / 1e9 / hbm}
            for k, t in (("score", score_ms), ("select", statistics.mean(t_select)),
                         ("compact", statistics.mean(t_compact)))},
        "graph_ms_per_step": graph_ms,
        "configs": configs,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": 3 * args.steps, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.qwen3_8b_32k().name, choices=sorted(wl.ALL))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the passes over the pages' other workloads (C1, C3, C4, C5 A and B)")
    ap.add_argument("--e2e-groups", type=int, default=9,
                    help="layer groups of the end-to-end leg (copies of one overlap the pass of another)")
    ap.add_argument("--no-commitkv", action="store_true",
                    help="skip the CommitKV deletion-effect and commit stages")
    ap.add_argument("--commitkv-only", action="store_true",
                    help="run only the CommitKV stages (one GPU) and print their timings")
    ap.add_argument("--layers", type=int, default=0,
                    help="use only this many layers of the workload (small profiling case)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()
    w = wl.ALL[args.workload]()
    if args.layers > 0:
        w = w.replace(n_layers=min(args.layers, w.n_layers),
                      name=f"{w.name}_{min(args.layers, w.n_layers)}layers")
    if args.commitkv_only:
        # the CommitKV stages alone (a small profiling case: one layer, 0.5 GB)
        import budgeted_kv_cache_gb300 as kvc
        from budgeted_kv_cache_gb300 import build
        build.build()
        kvc.library()
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        out = commitkv_stage(dev, torch.cuda.current_stream(dev), flush, repeats=args.steps)
        if rank == 0:
            print(json.dumps({"stage": "commitkv", "workload": wl.commitkv_effect_128k().name,
                              "stages_ms": out}), flush=True)
    elif args.impl == "reference":
        run_reference(args, w, world, rank)
    else:
        run_gpu(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
