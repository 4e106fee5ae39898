"""The benchmark's JSON contract on CPU: the reference arm (the oracle on the
host cores) prints one line with the keys the driver reads, naming the same
workload as the GPU arm, and the roofline's algorithmic work of the
Qwen3-8B-shaped workload agrees with the per-unit accounting (keys read once,
window queries, score write, shared bonus; 2 R T d flops per unit)."""
import importlib.util
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    line = json.loads(lines[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 1 and line["warmup"] >= 3
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    bench = _bench()
    w = bench.wl.qwen3_8b_32k()
    assert line["config"] == bench._config(w)
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT


def test_algorithmic_work_of_the_qwen3_8b_workload():
    bench = _bench()
    w = bench.wl.qwen3_8b_32k()
    assert (w.n_units, w.n_tokens, w.head_dim, w.rows_per_unit) == (288, 32768, 128, 256)
    flops = bench.algorithmic_flops(w)
    assert flops == 618_475_290_624                       # 2 x 288 units x 256 rows x 32768 keys x 128
    ab = bench.algorithmic_bytes(w)
    keys = 288 * 32768 * 128 * 2                          # K read once: 2.416 GB
    assert ab["score"] == keys + 288 * 256 * 128 * 2 + 288 * 32768 * 4 + 32768 * 4
    assert ab["total"] == pytest.approx(3.14e9, rel=0.01)
    assert ab["score"] / ab["total"] == pytest.approx(0.786, abs=0.005)   # K dominates the pass


def test_algorithmic_bytes_of_a_byte_mode_pass():
    """PASK batch 16 (byte budget): every pool's rows are costed at their own
    width -- int4 / int8 codes plus one bf16 scale per 32 elements (PASK
    App. B.5), bf16 rows in full -- and no rotary rows are touched (no
    renumbering); tags are read by the selection."""
    bench = _bench()
    w = bench.wl.pask_batch16()
    U, T, d = 4096, 8192, 128
    assert (w.n_units, w.n_tokens, w.head_dim) == (U, T, d)
    kept = {bench.POOL_INT4: 3000 * U, bench.POOL_INT8: 2000 * U, bench.POOL_BF16: 1000 * U}
    ab = bench.algorithmic_bytes(w, kept)
    n = 6000 * U
    # per row K + V: int4 2 x (64 + 8) = 144, int8 2 x (128 + 8) = 272, bf16 512
    pools = U * (3000 * 144 + 2000 * 272 + 1000 * 512)
    assert ab["compact"] == n * (4 + 4 + 512 + 8) + pools
    assert ab["select"] == U * T * 4 + 16 * T + n * 4
    assert ab["score"] == U * T * 256 + U * 256 * 256 + U * T * 4
    # row mode (one fp16 scale per row): int4 2 x (64 + 2) = 132
    wr = w.replace(quant_mode=bench.wl.QUANT_ROW_FP16)
    assert bench.kv_row_bytes(wr, bench.POOL_INT4) == 132
    assert bench.kv_row_bytes(wr, bench.POOL_INT8) == 2 * (128 + 2)


def test_traffic_key_ignores_comments():
    bench = _bench()
    src = "int a; // note\n/* block\n comment */ int b;\n\n"
    assert bench._code(src) == bench._code("int a;\n int b;")


def test_reference_arm_under_torchrun_prints_once():
    """Launched like the driver's N = 2 run (two ranks, gloo on a CPU host):
    rank 0 alone runs the oracle and prints; the other rank exits cleanly."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2 and lines[0]["value"] > 0
