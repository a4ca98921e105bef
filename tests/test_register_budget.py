"""Register budget of the one-CTA-per-row register kernel (ptxas -v).

At H = 7168 a row is 896 threads at one pack per thread; two CTAs fit an
SM only at <= 32 registers a thread (registers are granted in steps of 8).
The bounded cluster wait once pushed k_fused_epilogue<3, 1> to 41
registers in launches that never ran it, halving the CTAs per SM and
taking n = 3 from 7.2 to 5.3 TB/s.  The one-CTA instantiations carry no
cluster code; this test keeps them within budget.
"""
import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _ptxas_registers(src, tmp_path):
    from allreduce_sum_residual_gb300 import _build as b
    cmd = [b.nvcc(), *b.ARCH, *b.NVCC_FLAGS, "-Xptxas", "-v", "-c", src,
           "-o", str(tmp_path / "probe.o")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    regs, entry = {}, None
    for line in (r.stdout + r.stderr).splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            entry = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and entry:
            k = re.search(r"k_fused_epilogueILi(\d+)ELi(\d+)ELb([01])ELb([01])E", entry)
            if k:
                regs[(int(k.group(1)), int(k.group(2)), k.group(3) == "1", k.group(4) == "1")] = \
                    int(m.group(1))
            entry = None
    return regs


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="needs nvcc")
def test_one_cta_register_kernel_fits_two_ctas_per_sm_at_896_threads(tmp_path):
    src = os.path.join(ROOT, "allreduce_sum_residual_gb300", "csrc", "epilogue_g0.cu")
    regs = _ptxas_registers(src, tmp_path)
    for n in (1, 2, 3):
        assert regs[(n, 1, False, False)] <= 32, (n, regs[(n, 1, False, False)])
    # 4 inputs: <= 40 keeps three 512-thread CTAs per SM (H = 4096)
    assert regs[(4, 1, False, False)] <= 40, regs[(4, 1, False, False)]
    # this translation unit holds only the one-CTA copies (16 of them)
    assert sorted(regs) == [(n, v, False, False) for n in (1, 2, 3, 4) for v in (1, 2, 4, 8)]


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="needs nvcc")
def test_late_weight_kernel_saves_registers(tmp_path):
    """Loading the weight after the sums frees its registers while the
    partials are in flight: with 4 inputs at one pack per thread the kernel
    fits 32 registers, two 896-thread CTAs per SM (H = 7168)."""
    d = os.path.join(ROOT, "allreduce_sum_residual_gb300", "csrc")
    late = _ptxas_registers(os.path.join(d, "epilogue_l0.cu"), tmp_path)
    early = _ptxas_registers(os.path.join(d, "epilogue_g0.cu"), tmp_path)
    assert sorted(late) == [(n, v, False, True) for n in (1, 2, 3, 4) for v in (1, 2, 4, 8)]
    assert late[(4, 1, False, True)] <= 32, late[(4, 1, False, True)]
    assert late[(4, 1, False, True)] < early[(4, 1, False, False)]
