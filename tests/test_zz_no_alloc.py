"""cp_ring_forward_noalloc: the ring forward for callers that may not allocate
device memory (a plugin inside a host framework's fixed memory budget, or a
latency-critical loop where cudaMalloc/cudaFree would synchronise the
device).  When the ring runs step by step its fp32 accumulator is a fixed
array inside the library instead of a caller workspace.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.  It passes alone in a fresh
process and after the rest of the suite.
"""

import pytest
import torch

import oracle
from context_causal_attention_attn_gb300.inputs import make_qkv, sample_rows
from gpu_common import ATOL_BF16_LSE, ATOL_BF16_OUT, ATOL_F32, compare, host


@pytest.fixture(scope="module")
def cp():
    from context_causal_attention_attn_gb300 import build
    build.build()
    import context_causal_attention_attn_gb300 as m
    return m


@pytest.mark.gpu
def test_noalloc_matches_workspace_version_twice(cp):
    """Two calls in a row through the C ABI on a ring that runs step by step
    (fp32 inputs, a bf16 output: the fp32 accumulator then lives in the
    library's scratch array, S*H*D exactly the scratch's limit) agree with
    cp_ring_forward (which takes a caller workspace) bit for bit, as both
    run the same launches, and the first call also with the oracle on 512
    seeded rows per head."""
    S, H, D, P = 16384, 8, 128, 8
    q, k, v = make_qkv(S, H, D, dtype=torch.float32, device="cuda", seed=3)
    assert not cp.ring_runs_fused(q, "striped")  # step by step: the scratch is used
    ref_out, ref_lse = cp.cp_ring_forward(q, k, v, P, "striped", out_dtype=torch.bfloat16)
    cp.cp_check_device_error()
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        cp.cp_ring_forward_noalloc(q, k, v, P, "striped", out=out, lse=lse)
        cp.cp_check_device_error()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), call
        if call == 0:
            # fp32 arithmetic; only the output is rounded to bf16
            rows = sample_rows(S, 512, seed=1, must=(0, S - 1))
            ro, rl = oracle.attention_monolithic(host(q), host(k), host(v), rows=rows)
            compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_F32, rows=rows)


@pytest.mark.gpu
@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_noalloc_one_launch_ring_uses_no_scratch(cp, layout):
    """A ring cp_ring_forward runs in one launch (bf16 inputs) keeps no
    accumulator: the call accepts sizes past the scratch's limit (S*H*D =
    33,554,432 here) and equals cp_ring_forward."""
    S, H, D, P = 8192, 32, 128, 4
    q, k, v = make_qkv(S, H, D, dtype=torch.bfloat16, device="cuda", seed=4)
    assert cp.ring_runs_fused(q, layout)
    ref_out, ref_lse = cp.cp_ring_forward(q, k, v, P, layout, out_dtype=torch.bfloat16)
    out, lse = cp.cp_ring_forward_noalloc(q, k, v, P, layout, out_dtype=torch.bfloat16)
    cp.cp_check_device_error()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


@pytest.mark.gpu
def test_noalloc_fp32_output_uses_no_scratch(cp):
    """With an fp32 output the output is the accumulator: no scratch is
    looked up and the call equals cp_ring_forward (the handbook's toy, fp32,
    atol 1e-5 against the oracle)."""
    q, k, v = (t.cuda() for t in make_qkv(32, 8, 16))
    ref_out, ref_lse = cp.cp_ring_forward(q, k, v, 4, "contiguous")
    for _ in range(2):
        out, lse = cp.cp_ring_forward_noalloc(q, k, v, 4, "contiguous")
        cp.cp_check_device_error()
        assert out.dtype == torch.float32
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
        ro, rl = oracle.attention(host(q), host(k), host(v))
        compare(out, lse, ro, rl, ATOL_F32, ATOL_F32)


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_the_scratch(cp):
    S, H, D, P = 16384, 16, 128, 8  # a step-by-step ring needing 128 MiB of accumulator
    q = torch.empty(S, H, D, dtype=torch.float32, device="cuda")
    with pytest.raises(cp.CpError) as e:
        cp.cp_ring_forward_noalloc(q, q, q, P, "striped", out_dtype=torch.bfloat16)
    assert "scratch" in str(e.value)
