"""The compaction's quantiser divides each element by its group's scale
through one reciprocal per group and Markstein's correction step
(div_by_recip); the int8 / int4 codes must be those of IEEE division
(PASK App. B.5: q = round(x / s)).  This test compiles a small CUDA program
against the library's own helper and checks every finite bf16 dividend
against every bf16 and every fp16 divisor of the fast path, over the
quantiser's domain (|x| <= 256 s: a group's scale is at least its largest
magnitude over qmax, so its quotients stay near qmax or below)."""
import os
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_reciprocal_division_is_exact_for_every_bf16_and_fp16_operand():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "quotient_check")
        r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                            os.path.join(HERE, "cuda", "quotient_check.cu"), "-o", exe],
                           capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
        print(r.stdout)
        assert r.returncode == 0, r.stdout + r.stderr
