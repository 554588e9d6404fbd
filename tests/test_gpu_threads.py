"""Host threads calling the library at once.

The library keeps per-device host state (the kernels' shared-memory
attribute, the device status word's address), set up the first time each
device reaches it.  These tests make that first call from two threads at
once, in a fresh process, and check that every result equals the serial
one; with two or more GPUs each thread drives its own device.
"""

import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, threading
import torch
sys.path.insert(0, {root!r})
import context_causal_attention_attn_gb300 as cp
from context_causal_attention_attn_gb300.inputs import make_dout, make_qkv

devices = {devices!r}
S, H, D, P = 2048, 8, 128, 4
data = {{}}
for i, d in enumerate(devices):
    dev = torch.device("cuda", d)
    q, k, v = make_qkv(S, H, D, dtype=torch.bfloat16, seed=70 + i, device=dev)
    do = make_dout(S, H, D, dtype=torch.bfloat16, seed=70 + i, device=dev)
    data[i] = (dev, q, k, v, do)
torch.cuda.synchronize()
results, errors = {{}}, []
barrier = threading.Barrier(len(devices))

def work(i):
    try:
        dev, q, k, v, do = data[i]
        torch.cuda.set_device(dev)
        s = torch.cuda.Stream(dev)
        with torch.cuda.stream(s):
            barrier.wait()   # first calls into the library at the same time
            out, lse = cp.cp_ring_forward(q, k, v, P, "zigzag", out_dtype=torch.bfloat16,
                                          stream=s)
            g = cp.cp_ring_backward(q, k, v, out, do, lse, P, "zigzag",
                                    grad_dtype=torch.float32, stream=s)
            s.synchronize()
            cp.cp_check_device_error(s)
        results[i] = [t.cpu() for t in (out, lse) + tuple(g)]
    except Exception as e:
        errors.append(repr(e))

threads = [threading.Thread(target=work, args=(i,)) for i in range(len(devices))]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
for i, d in enumerate(devices):
    dev, q, k, v, do = data[i]
    torch.cuda.set_device(dev)
    out, lse = cp.cp_ring_forward(q, k, v, P, "zigzag", out_dtype=torch.bfloat16)
    g = cp.cp_ring_backward(q, k, v, out, do, lse, P, "zigzag", grad_dtype=torch.float32)
    torch.cuda.synchronize()
    for a, b in zip(results[i], [t.cpu() for t in (out, lse) + tuple(g)]):
        assert torch.equal(a, b), "threaded result differs from the serial one"
print("threads ok")
"""


def _run(devices):
    from context_causal_attention_attn_gb300 import build
    build.build()
    code = SCRIPT.format(root=ROOT, devices=devices)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout + r.stderr


def test_two_threads_one_device_first_calls():
    _run([0, 0])


@pytest.mark.skipif(not torch.cuda.is_available() or torch.cuda.device_count() < 2,
                    reason="needs two GPUs")
def test_two_threads_two_devices_first_calls():
    _run([0, 1])
