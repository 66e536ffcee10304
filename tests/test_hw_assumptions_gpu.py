"""GPU probe of the hardware property the attention kernel's MMA schedule relies on:
tcgen05.mma operations issued by one thread execute in order, so an MMA that reads its A
operand from tensor memory is not disturbed by a later MMA that overwrites those columns."""

import os
import re
import subprocess

import pytest

from tiled_attention_03_gb300.build import CSRC, nvcc

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tmem_operand_read_precedes_later_mma_write(tmp_path):
    src = os.path.join(HERE, "gpu_probes", "tmem_operand_order.cu")
    exe = str(tmp_path / "tmem_operand_order")
    subprocess.check_call([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                           "-std=c++17", "-I", CSRC, src, "-o", exe])
    out = subprocess.run([exe, "2000"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    m = re.search(r"bad elements (\d+), sample O ([0-9.]+) \[(.*)\]", out.stdout)
    assert m, out.stdout
    assert m.group(3) == "no error"
    assert int(m.group(1)) == 0
    assert float(m.group(2)) == 56.0
