"""The bounds-checked library (libcpattn_debug.so, loaded with CPATTN_DEBUG=1).

Its kernels check, per tile or row, that everything they read or write lies
inside the tensors the call describes, and report a failure through
cp_check_device_error as CP_ERR_BOUNDS.  No test here provokes a failure on
the GPU (valid calls cannot reach one, and an invalid call is rejected on
the host): the checks are run over a cross-section of the parity tests,
where every call is followed by cp_check_device_error, so a check that fired
on a valid tile would fail the test; and the checked build must reproduce
the release build's bits.
"""

import os
import subprocess
import sys
import tempfile

import pytest
import torch

from context_causal_attention_attn_gb300 import build
from context_causal_attention_attn_gb300._lib import debug_requested
from context_causal_attention_attn_gb300.inputs import make_dout, make_qkv

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REF_ENV = "CPATTN_DEBUG_REF"


@pytest.fixture(scope="module")
def cp():
    build.build(debug=debug_requested())
    import context_causal_attention_attn_gb300 as m
    m.lib()
    return m


def _cases(cp):
    """Outputs of a few calls that cover the four attention kernels: the
    one-launch ring, the per-step striped ring, the fp32 ring, and the
    two-launch ring backward."""
    res = {}
    q, k, v = (t.cuda() for t in make_qkv(2048, 4, 128, Hkv=2, dtype=torch.bfloat16, seed=5))
    res["fused"] = cp.cp_ring_forward(q, k, v, 4, "zigzag")
    res["striped"] = cp.cp_ring_forward(q, k, v, 4, "striped")
    do = make_dout(2048, 4, 128, dtype=torch.bfloat16, seed=6).cuda()
    out, lse = res["fused"]
    res["backward"] = cp.cp_ring_backward(q, k, v, out, do, lse, 4, "zigzag",
                                          grad_dtype=torch.bfloat16)
    qf, kf, vf = (t.cuda() for t in make_qkv(96, 2, 16, seed=7))
    res["fp32"] = cp.cp_ring_forward(qf, kf, vf, 3, "contiguous")
    cp.cp_check_device_error()
    return {name: tuple(t.cpu() for t in val) for name, val in res.items()}


def test_loaded_library_matches_request(cp):
    """CPATTN_DEBUG=1 loads the bounds-checked build, otherwise the release
    build is loaded."""
    assert cp.cp_debug_bounds() == debug_requested()


def test_bounds_checked_matches_release_bits(cp):
    """Inside the bounds-checked run: the checked kernels give the release
    kernels' results bit for bit (the checks read indices only)."""
    ref = os.environ.get(REF_ENV)
    if not debug_requested() or not ref:
        pytest.skip("runs inside the bounds-checked run")
    want = torch.load(ref)
    got = _cases(cp)
    for name, tensors in want.items():
        for a, b in zip(got[name], tensors):
            assert torch.equal(a, b), name


def test_parity_suite_under_bounds_checks(cp):
    """A cross-section of the parity tests (block attention, the ring in
    every layout and form, host buffers, Ulysses, USP, the backward,
    non-finite inputs) with every kernel bounds-checked: no check fires and
    the oracle still agrees; then the checked build's bits against the
    release build's."""
    if debug_requested():
        pytest.skip("already inside the bounds-checked run")
    build.build(debug=True)
    with tempfile.TemporaryDirectory() as tmp:
        ref = os.path.join(tmp, "release.pt")
        torch.save(_cases(cp), ref)
        env = dict(os.environ, CPATTN_DEBUG="1", **{REF_ENV: ref})
        files = ["tests/test_gpu_debug_bounds.py", "tests/test_gpu_block.py",
                 "tests/test_gpu_ring.py", "tests/test_gpu_backward.py",
                 "tests/test_gpu_nonfinite.py"]
        cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
               "-k", "not sampled and not 64k"] + files
        r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    summary = r.stdout.strip().splitlines()[-1]
    print("bounds-checked run:", summary)
    assert " passed" in summary
