"""Resource budgets the launch schedule depends on, checked on the compiler's
report (no GPU needed).

The combine kernel's CTAs start beside the expert kernel's (programmatic
dependent launch) only if both fit an SM together: the expert CTA at 8-pick
tiles leaves 1,152 bytes of shared memory (its 231,296 bytes of dynamic shared
memory plus each CTA's 1 KB reservation, of 233,472) and, on the SM
sub-partitions holding four of its 13 warps at 112 registers, 2048 registers:
two combine warps at 32 registers a thread.  A kernel change that crosses
either budget still computes the right result and only shows up as a slower
step, so it is checked here, for the library build and the trace build.
"""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mxfp4_mixture_experts_route_gb300", "csrc")


def _ptxas_report(src: str, defines: list[str], tmp_path) -> dict[str, tuple[int, int, int]]:
    """Kernel (mangled name) -> (registers, spill bytes, static shared memory)."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "--expt-relaxed-constexpr",
           "-I", os.path.join(ROOT, "include"), *defines, "-Xptxas", "-v", "-c", os.path.join(CSRC, src),
           "-o", str(tmp_path / "k.o")]
    out = subprocess.run(cmd, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr[-2000:]
    report, name = {}, None
    for line in out.stderr.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            name = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores", line)
        if m and name:
            report.setdefault(name, [0, 0, 0])[1] = int(m.group(1))
        m = re.search(r"Used (\d+) registers.*?(?:(\d+) bytes smem)?$", line)
        if m and name:
            r = report.setdefault(name, [0, 0, 0])
            r[0] = int(m.group(1))
            r[2] = int(m.group(2) or 0)
    return {k: tuple(v) for k, v in report.items()}


@pytest.mark.parametrize("defines", [[], ["-DMOE_TRACE"]], ids=["library", "trace"])
def test_combine_fits_beside_the_expert_kernel(defines, tmp_path):
    combine = _ptxas_report("combine.cu", defines, tmp_path)
    (regs, spill, smem), = [v for k, v in combine.items() if "k_combine" in k]
    assert regs <= 32 and smem <= 128 and spill == 0, (regs, smem, spill)
    experts = _ptxas_report("experts_mx.cu", defines, tmp_path)
    eight = [v for k, v in experts.items() if re.search(r"k_experts_mxILb[01]ELi8E", k)]
    assert len(eight) == 2
    for regs, spill, smem in eight:
        assert regs <= 112 and spill == 0 and smem == 0, (regs, spill, smem)
