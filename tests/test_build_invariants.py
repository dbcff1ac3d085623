"""Build-time invariants of the CUDA sources (no GPU needed).

The fused forward kernel splits its registers between warpgroups with
setmaxnreg: the producer warpgroup gives registers back and the computing
warpgroups take them. The split adds up to the launch allocation only if
ptxas builds every instance with exactly 168 registers per thread at launch
(12 warps: three share one sub-partition's 16K). The library refuses other
instances at run time; this test pins the build itself."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dlrm_embedding_interaction_gb300", "csrc")


@pytest.mark.parametrize("source", ["fused.cu", "fused_trace.cu"])
def test_every_fused_kernel_instance_launches_with_168_registers(tmp_path, source):
    """Both translation units of the kernel: the plain instances and the ones
    with phase-trace stamps."""
    from dlrm_embedding_interaction_gb300 import build
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    cmd = [nvcc, *build.ARCH, *build.NVCC_FLAGS, "-Xptxas", "-v", "-c",
           os.path.join(CSRC, source), "-o", str(tmp_path / "fused.o")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    regs = {}
    current = None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\S*fused_forward_kernel\S*)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            regs[current] = int(m.group(1))
            current = None
    assert len(regs) == 13, regs         # every tile height and stride instance
    assert set(regs.values()) == {168}, regs
