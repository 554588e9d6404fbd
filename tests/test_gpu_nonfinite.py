"""Non-finite inputs reach the outputs instead of being absorbed.

[CP-practice] section 8.3 lists a sanity check on the softmax's running max:
a NaN or Inf that enters the scores must not turn into a plausible-looking
result.  By the definition (scores -> mask -> logsumexp -> softmax . V) a
NaN in q[i], or in a key / value row that row i sees, makes row i's result
NaN, and rows that do not see it are unchanged.  These tests plant one
non-finite value at a time in q, k or v and check:

* the rows the definition makes NaN are NaN (out and lse; only the planted
  column of out for a NaN in v, whose lse is unaffected);
* every other entry is bit for bit the result of the same call on the clean
  inputs (the kernels are deterministic and rows are independent);
* no device-side wait expired (cp_check_device_error stays clean).

A NaN in a value row that a query does NOT see may still reach that query's
column when both share a 128-key tile (the tensor core multiplies the zero
weight by the NaN); those few entries are left unchecked.
"""

import numpy as np
import pytest
import torch

import oracle
from context_causal_attention_attn_gb300.inputs import make_qkv
from gpu_common import ATOL_BF16_LSE, ATOL_BF16_OUT, host, ring_by_steps

pytestmark = pytest.mark.gpu
NAN = float("nan")


@pytest.fixture(scope="module")
def cp():
    from context_causal_attention_attn_gb300 import build
    build.build()
    import context_causal_attention_attn_gb300 as m
    return m


def _expect(clean, dirty, nan_out, nan_lse, free_out=None):
    """nan_out [S,H,D] / nan_lse [H,S] boolean: entries that must be NaN;
    free_out: entries left unchecked; everything else equals the clean run."""
    o0, l0 = host(clean[0]), host(clean[1])
    o1, l1 = host(dirty[0]), host(dirty[1])
    assert np.all(np.isnan(o1[nan_out])), "a NaN input did not reach out"
    assert np.all(np.isnan(l1[nan_lse])), "a NaN input did not reach lse"
    keep = ~nan_out if free_out is None else ~(nan_out | free_out)
    assert np.array_equal(o1[keep], o0[keep], equal_nan=True), "unaffected out entries changed"
    assert np.array_equal(l1[~nan_lse], l0[~nan_lse], equal_nan=True), (
        "unaffected lse entries changed")


def _masks(S, H, D):
    return np.zeros((S, H, D), bool), np.zeros((H, S), bool)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_block_bf16_nan_in_q_k_v(cp, out_dtype):
    S, H, Hkv, D = 512, 4, 2, 128
    q, k, v = (t.cuda() for t in make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=61))
    run = lambda q_, k_, v_: cp.cp_attn_block(q_, k_, v_, out_dtype=out_dtype)
    clean = run(q, k, v)
    cp.cp_check_device_error()

    # q[100, head 1] -> row 100 of head 1
    qd = q.clone()
    qd[100, 1, 7] = NAN
    no, nl = _masks(S, H, D)
    no[100, 1, :] = True
    nl[1, 100] = True
    _expect(clean, run(qd, k, v), no, nl)

    # k[200, KV head 0] -> rows >= 200 of query heads 0 and 1
    kd = k.clone()
    kd[200, 0, 3] = NAN
    no, nl = _masks(S, H, D)
    no[200:, 0:2, :] = True
    nl[0:2, 200:] = True
    _expect(clean, run(q, kd, v), no, nl)

    # v[300, KV head 1, column 5] -> column 5 of rows >= 300 of heads 2, 3;
    # rows 256..299 share the key tile of row 300 and are left unchecked
    vd = v.clone()
    vd[300, 1, 5] = NAN
    no, nl = _masks(S, H, D)
    no[300:, 2:4, 5] = True
    free = np.zeros_like(no)
    free[256:300, 2:4, 5] = True
    _expect(clean, run(q, k, vd), no, nl, free)
    cp.cp_check_device_error()


def test_block_bf16_inf_in_k_against_oracle(cp):
    """+inf in one key: rows whose score with it is +inf become non-finite
    (the oracle, like the page's logsumexp, gives lse = +inf and out = NaN
    from inf - inf; the kernel gives NaN for both), rows whose score is -inf
    simply drop the key; the non-finite pattern and the finite values follow
    the fp64 oracle."""
    S, H, D = 384, 2, 128
    q, k, v = make_qkv(S, H, D, dtype=torch.bfloat16, seed=62)
    k[10, 1, 0] = float("inf")
    out, lse = cp.cp_attn_block(q.cuda(), k.cuda(), v.cuda(), out_dtype=torch.float32)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(host(q), host(k), host(v))
    o, l = host(out), host(lse)
    assert np.array_equal(np.isfinite(l), np.isfinite(rl)) and not np.isfinite(rl).all()
    assert np.array_equal(np.isfinite(o), np.isfinite(ro))
    fin = np.isfinite(ro)
    assert np.max(np.abs(o[fin] - ro[fin])) <= ATOL_BF16_OUT
    assert np.max(np.abs(l[np.isfinite(rl)] - rl[np.isfinite(rl)])) <= ATOL_BF16_LSE


@pytest.mark.parametrize("layout", ["zigzag", "striped", "contiguous"])
def test_ring_bf16_nan_in_k_reaches_every_later_row(cp, layout):
    """Through the ring's fused merges (striped items also merge blocks in
    which some rows see no key: an empty block must not wipe out a NaN
    accumulator)."""
    S, H, Hkv, D, P = 1024, 4, 2, 128, 4
    q, k, v = (t.cuda() for t in make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=63))
    # cp_ring_forward (one launch at this length, except striped) and the
    # per-step ring with its merges through the accumulator
    for run in (lambda k_: cp.cp_ring_forward(q, k_, v, P, layout, out_dtype=torch.bfloat16),
                lambda k_: ring_by_steps(cp, q, k_, v, P, layout, out_dtype=torch.bfloat16)):
        clean = run(k)
        for j0 in (5, 600):
            kd = k.clone()
            kd[j0, 1, 0] = NAN
            dirty = run(kd)
            cp.cp_check_device_error()
            no, nl = _masks(S, H, D)
            no[j0:, 2:4, :] = True
            nl[2:4, j0:] = True
            _expect(clean, dirty, no, nl)


def test_ring_fp32_toy_nan_in_q(cp):
    """The fp32 CUDA-core path (the handbook's toy through the ring)."""
    q, k, v = (t.cuda() for t in make_qkv(32, 8, 16))
    clean = cp.cp_ring_forward(q, k, v, 4, "contiguous")
    qd = q.clone()
    qd[13, 6, 2] = NAN
    dirty = cp.cp_ring_forward(qd, k, v, 4, "contiguous")
    cp.cp_check_device_error()
    no, nl = _masks(32, 8, 16)
    no[13, 6, :] = True
    nl[6, 13] = True
    _expect(clean, dirty, no, nl)
    kd = k.clone()
    kd[20, 0, 0] = NAN
    dirty = cp.cp_ring_forward(q, kd, v, 4, "zigzag")
    clean_z = cp.cp_ring_forward(q, k, v, 4, "zigzag")
    cp.cp_check_device_error()
    no, nl = _masks(32, 8, 16)
    no[20:, 0, :] = True
    nl[0, 20:] = True
    _expect(clean_z, dirty, no, nl)


def test_lse_merge_nan_sides(cp):
    """The stand-alone merge: a NaN side gives NaN, also when the other side
    is an empty block (lse = -inf)."""
    Sq, H, D = 8, 2, 16
    acc = torch.randn(Sq, H, D, device="cuda")
    lacc = torch.randn(H, Sq, device="cuda")
    blk = torch.randn(Sq, H, D, device="cuda")
    lblk = torch.randn(H, Sq, device="cuda")
    lacc[0, 1] = NAN               # NaN accumulator, regular block
    lacc[1, 2] = NAN               # NaN accumulator, empty block
    lblk[1, 2] = -float("inf")
    blk[2, 1] = 0.0
    lblk[0, 3] = NAN               # regular accumulator, NaN block
    lacc[1, 4] = -float("inf")     # empty accumulator, NaN block
    acc[4, 1] = 0.0
    lblk[1, 4] = NAN
    lacc[0, 5] = -float("inf")     # both empty stay empty
    lblk[0, 5] = -float("inf")
    acc[5, 0] = 0.0
    blk[5, 0] = 0.0
    cp.cp_lse_merge(acc, lacc, blk, lblk)
    cp.cp_check_device_error()
    l, o = host(lacc), host(acc)
    for h, i in ((0, 1), (1, 2), (0, 3), (1, 4)):
        assert np.isnan(l[h, i]) and np.all(np.isnan(o[i, h])), (h, i)
    assert l[0, 5] == -np.inf and np.all(o[5, 0] == 0)
    others = np.ones((H, Sq), bool)
    for h, i in ((0, 1), (1, 2), (0, 3), (1, 4), (0, 5)):
        others[h, i] = False
    assert np.all(np.isfinite(l[others]))
