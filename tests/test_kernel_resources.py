"""Register budget of the hot kernels, from ptxas's resource report.

The forward kernel runs two CTAs per SM at 168 registers per thread and the
backward kernels one CTA per SM; a spill puts local-memory traffic into the
per-tile chain (removing the forward's last 26 bytes of spill stores made
the 128K ring 1.5% faster).  nvcc cross-compiles for sm_103a without a GPU,
so this is a CPU test.
"""

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "context_causal_attention_attn_gb300", "csrc")


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    pytest.skip("nvcc not found")


def _resources(src):
    """{kernel entry (mangled): (registers, spill store bytes, spill load bytes)}"""
    with tempfile.TemporaryDirectory() as tmp:
        cmd = [_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
               "--expt-relaxed-constexpr", "-Xptxas", "-v", "-I", CSRC,
               "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src),
               "-o", os.path.join(tmp, "k.o")]
        r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out, entry, res = r.stdout + r.stderr, None, {}
    spills = None
    for line in out.splitlines():
        m = re.search(r"Compiling entry function '(\w+)'", line)
        if m:
            entry, spills = m.group(1), None
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and entry:
            spills = (int(m.group(1)), int(m.group(2)))
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and entry and spills is not None:
            res[entry] = (int(m.group(1)),) + spills
            entry = None
    return res


@pytest.fixture(scope="module")
def resources():
    with cf.ThreadPoolExecutor(2) as ex:
        fwd, bwd = ex.map(_resources, ["attn_tc.cu", "attn_bwd_tc.cu"])
    return fwd, bwd


def test_forward_kernel_fits_two_ctas_per_sm_without_spills(resources):
    fwd, _ = resources
    plain = [v for k, v in fwd.items() if "attn_fwd_tc_kernelILb0E" in k]
    assert len(plain) == 1, fwd
    regs, st, ld = plain[0]
    assert regs <= 168, regs  # 2 CTAs x 192 threads on 65536 registers
    assert st == 0 and ld == 0, (st, ld)


def test_backward_kernels_do_not_spill(resources):
    _, bwd = resources
    kernels = {k: v for k, v in bwd.items() if "attn_bwd_tc_kernel" in k}
    assert len(kernels) == 4, bwd  # dK/dV and dQ, plain and strided rows
    for name, (regs, st, ld) in kernels.items():
        assert st == 0 and ld == 0, (name, st, ld)
