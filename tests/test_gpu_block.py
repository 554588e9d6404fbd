"""GPU parity of cp_attn_block (fp32 CUDA-core and bf16 tensor-core paths)
against the fp64 oracle, every element, including ragged tails, offsets that
leave rows without keys, GQA and the non-causal case."""

import numpy as np
import pytest
import torch

import oracle
from context_causal_attention_attn_gb300.inputs import make_qkv
from gpu_common import ATOL_BF16_LSE, ATOL_BF16_OUT, ATOL_F32, compare, guarded, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    from context_causal_attention_attn_gb300 import build
    build.build()
    import context_causal_attention_attn_gb300 as m
    return m


def _qkv(Sq, Sk, H, Hkv, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(Sq, H, D, generator=g).to(dtype)
    k = torch.randn(Sk, Hkv, D, generator=g).to(dtype)
    v = torch.randn(Sk, Hkv, D, generator=g).to(dtype)
    return q, k, v


F32_CASES = [  # Sq, Sk, H, Hkv, D, causal, q_off, k_off
    (32, 32, 8, 8, 16, True, 0, 0),
    (37, 53, 4, 2, 16, True, 16, 0),
    (50, 20, 2, 2, 32, True, 0, 25),     # rows before every key: empty
    (64, 64, 4, 1, 64, False, 0, 0),
    (130, 70, 2, 2, 128, True, 100, 40),
]


@pytest.mark.parametrize("case", F32_CASES)
def test_block_fp32(cp, case):
    Sq, Sk, H, Hkv, D, causal, qo, ko = case
    q, k, v = _qkv(Sq, Sk, H, Hkv, D, torch.float32, 1)
    out, out_ok = guarded((Sq, H, D), torch.float32)
    lse, lse_ok = guarded((H, Sq), torch.float32)
    cp.cp_attn_block(q.cuda(), k.cuda(), v.cuda(), q_offset=qo, k_offset=ko, causal=causal,
                     out=out, lse=lse)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy(), causal=causal, q_offset=qo,
                              k_offset=ko)
    compare(out, lse, ro, rl, ATOL_F32, ATOL_F32)
    assert out_ok() and lse_ok(), "write outside out / lse"


BF16_CASES = [  # Sq, Sk, H, Hkv, D, causal, q_off, k_off
    (128, 128, 1, 1, 128, False, 0, 0),
    (128, 128, 1, 1, 128, True, 0, 0),
    (256, 256, 2, 2, 128, True, 0, 0),
    (300, 517, 2, 1, 128, True, 217, 0),   # ragged q and k tails, GQA
    (512, 384, 4, 2, 128, False, 0, 0),
    (129, 129, 2, 2, 128, True, 0, 0),
    (1, 1, 1, 1, 128, True, 0, 0),
    (200, 300, 2, 2, 128, True, 0, 50),    # the first 50 rows see no key
    (640, 1024, 4, 4, 128, True, 384, 0),  # several tiles, diagonal offset by 384
    (100, 900, 3, 1, 128, True, 5000, 0),  # every key visible (no masked tile)
]


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("case", BF16_CASES)
def test_block_bf16(cp, case, out_dtype):
    Sq, Sk, H, Hkv, D, causal, qo, ko = case
    q, k, v = _qkv(Sq, Sk, H, Hkv, D, torch.bfloat16, 2)
    out, out_ok = guarded((Sq, H, D), out_dtype)
    lse, lse_ok = guarded((H, Sq), torch.float32)
    cp.cp_attn_block(q.cuda(), k.cuda(), v.cuda(), q_offset=qo, k_offset=ko, causal=causal,
                     out=out, lse=lse)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(host(q), host(k), host(v), causal=causal, q_offset=qo, k_offset=ko)
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)
    assert out_ok() and lse_ok(), "write outside out / lse"


def test_block_bf16_large_logits(cp):
    """Scores far above 1 (q scaled by 8): exercises the lazy rescale of O."""
    q, k, v = _qkv(384, 640, 2, 2, 128, torch.bfloat16, 3)
    q = (q.float() * 8).to(torch.bfloat16)
    out, lse = cp.cp_attn_block(q.cuda(), k.cuda(), v.cuda(), q_offset=256, causal=True,
                                out_dtype=torch.float32)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(host(q), host(k), host(v), causal=True, q_offset=256)
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


def test_block_empty_keys(cp):
    q, _, _ = _qkv(40, 1, 2, 2, 128, torch.bfloat16, 4)
    k = torch.empty(0, 2, 128, dtype=torch.bfloat16)
    out, lse = cp.cp_attn_block(q.cuda(), k.cuda(), k.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_block_explicit_scale(cp):
    q, k, v = _qkv(256, 256, 2, 2, 128, torch.bfloat16, 5)
    out, lse = cp.cp_attn_block(q.cuda(), k.cuda(), v.cuda(), scale=0.05,
                                out_dtype=torch.float32)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(host(q), host(k), host(v), causal=True, scale=0.05)
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


def test_block_deterministic(cp):
    q, k, v = (t.cuda() for t in _qkv(512, 512, 4, 4, 128, torch.bfloat16, 6))
    a = cp.cp_attn_block(q, k, v, out_dtype=torch.float32)
    b = cp.cp_attn_block(q, k, v, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_timeout_selftest_reports_status(cp):
    """Failure detection: a bounded wait that expires is reported as a status,
    the context stays usable and the status clears after it is read."""
    cp.cp_selftest_wait_timeout(2000)
    with pytest.raises(cp.CpError) as e:
        cp.cp_check_device_error()
    assert e.value.code == cp.CP_ERR_TIMEOUT
    cp.cp_check_device_error()  # cleared
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0
