"""GPU parity of the backward pass (block and ring) against the fp64 oracle.

Inputs to both sides: bf16 q, k, v, dO drawn by ``inputs``; the forward's
out (rounded to bf16) and lse (rounded to fp32) from the ORACLE's forward,
so no value the oracle reads comes from the CUDA path.  The expected
gradients are ``oracle.attention_backward`` of the whole sequence: the ring's
block gradients, computed with the whole-row lse, must add up to them.

Tolerance (derived from the arithmetic, not fitted to the kernel): the
kernels round P and dS to bf16 (relative 2^-9) before the gradient MMAs and
accumulate in fp32.  An fp32 emulation of exactly that rounding against the
fp64 gradients gives max|err| / max|ref| = 1.0e-3 to 2.2e-3 and
rms(err) / rms(ref) = 1.6e-3 for fp32 gradients (3.6e-3 and 2.3e-3 after a
bf16 cast of the gradients), at S = 1024 and 4096.  The bound is 4x that:
max|err| <= 1.5e-2 max|ref| and rms(err) <= 1e-2 rms(ref), per tensor.  A
dropped term, a wrong scale or a missed key tile moves whole rows by tens of
percent.
"""

import numpy as np
import pytest
import torch

import oracle
from context_causal_attention_attn_gb300.inputs import make_dout, make_qkv, sample_rows
from gpu_common import guarded, host

pytestmark = pytest.mark.gpu

MAX_REL = 1.5e-2
RMS_REL = 1e-2


@pytest.fixture(scope="module")
def cp():
    from context_causal_attention_attn_gb300 import build
    build.build()
    import context_causal_attention_attn_gb300 as m
    return m


def grads_close(got, ref, name, max_rel=MAX_REL, rms_rel=RMS_REL):
    g = host(got).astype(np.float64)
    assert np.all(np.isfinite(g)), f"{name}: non-finite gradient"
    scale_max = np.abs(ref).max()
    scale_rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(g - ref)
    if scale_max == 0:
        assert err.max() == 0, f"{name}: expected zeros, max {err.max():.3e}"
        return
    m = err.max() / scale_max
    r = np.sqrt(np.mean(err ** 2)) / scale_rms
    if not (m <= max_rel and r <= rms_rel):
        idx = np.unravel_index(np.argmax(err), err.shape)
        bad_rows = np.unique(np.argwhere(err > max_rel * scale_max)[:, 0])[:10]
        raise AssertionError(f"{name}: max|err|/max|ref| = {m:.3e} (tol {max_rel}), "
                             f"rms ratio {r:.3e} (tol {rms_rel}); worst at {idx}: got "
                             f"{g[idx]:.5f} want {ref[idx]:.5f}; rows {bad_rows}")


def forward_inputs(S, H, Hkv, seed, q_offset=0, k_offset=0, Sk=None, causal=True):
    """bf16 q, k, v, dO and the oracle's forward (out as bf16, lse as fp32)."""
    Sk = S if Sk is None else Sk
    q, _, _ = make_qkv(S, H, 128, Hkv=Hkv, dtype=torch.bfloat16, seed=seed)
    _, k, v = make_qkv(Sk, H, 128, Hkv=Hkv, dtype=torch.bfloat16, seed=seed)
    do = make_dout(S, H, 128, dtype=torch.bfloat16, seed=seed)
    q64, k64, v64 = (t.double().numpy() for t in (q, k, v))
    out, lse = oracle.attention(q64, k64, v64, causal=causal, q_offset=q_offset,
                                k_offset=k_offset)
    out_b = torch.from_numpy(out).to(torch.bfloat16)
    lse32 = torch.from_numpy(lse.astype(np.float32))
    return q, k, v, do, out_b, lse32


def oracle_grads(q, k, v, do, out_b, lse32, **kw):
    return oracle.attention_backward(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                     out_b.double().numpy(), lse32.double().numpy(),
                                     do.double().numpy(), **kw)


def dev(*ts):
    return [t.cuda().contiguous() for t in ts]


# ------------------------------------------------------------------ block
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("S,H,Hkv", [(128, 2, 2), (300, 4, 2), (700, 2, 1)])
def test_block_backward_causal(cp, S, H, Hkv, grad_dtype):
    """Whole causal block (one tile, ragged multi-tile, GQA 2:1 and 2:1 single
    KV head) on every element."""
    q, k, v, do, ob, l32 = forward_inputs(S, H, Hkv, seed=S)
    dq, dk, dv = cp.cp_attn_block_backward(*dev(q, k, v, ob, do, l32), grad_dtype=grad_dtype)
    cp.cp_check_device_error()
    rq, rk, rv = oracle_grads(q, k, v, do, ob, l32)
    grads_close(dq, rq, "dq")
    grads_close(dk, rk, "dk")
    grads_close(dv, rv, "dv")


@pytest.mark.parametrize("q_offset,k_offset,Sq,Sk", [
    (384, 0, 200, 384),    # queries after all keys: every pair visible
    (256, 128, 300, 400),  # diagonal crossing inside tiles, ragged both sides
    (0, 100, 260, 300),    # first 100 rows see no key (lse = -inf, zero gradients)
])
def test_block_backward_offsets(cp, q_offset, k_offset, Sq, Sk):
    H, Hkv = 2, 2
    q, _, _ = make_qkv(Sq, H, 128, Hkv=Hkv, dtype=torch.bfloat16, seed=7)
    _, k, v = make_qkv(Sk, H, 128, Hkv=Hkv, dtype=torch.bfloat16, seed=8)
    do = make_dout(Sq, H, 128, dtype=torch.bfloat16, seed=9)
    out, lse = oracle.attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                q_offset=q_offset, k_offset=k_offset)
    ob = torch.from_numpy(out).to(torch.bfloat16)
    l32 = torch.from_numpy(lse.astype(np.float32))
    dq, dk, dv = cp.cp_attn_block_backward(*dev(q, k, v, ob, do, l32), q_offset=q_offset,
                                           k_offset=k_offset, grad_dtype=torch.float32)
    cp.cp_check_device_error()
    rq, rk, rv = oracle_grads(q, k, v, do, ob, l32, q_offset=q_offset, k_offset=k_offset)
    grads_close(dq, rq, "dq")
    grads_close(dk, rk, "dk")
    grads_close(dv, rv, "dv")
    empty = ~np.isfinite(lse)
    if empty.any():
        assert np.all(host(dq)[np.where(empty.any(axis=0))[0]] == 0)


def test_block_backward_noncausal(cp):
    q, k, v, do, ob, l32 = forward_inputs(260, 2, 2, seed=21, causal=False)
    dq, dk, dv = cp.cp_attn_block_backward(*dev(q, k, v, ob, do, l32), causal=False,
                                           grad_dtype=torch.float32)
    cp.cp_check_device_error()
    rq, rk, rv = oracle_grads(q, k, v, do, ob, l32, causal=False)
    grads_close(dq, rq, "dq")
    grads_close(dk, rk, "dk")
    grads_close(dv, rv, "dv")


def test_block_backward_empty(cp):
    """Sk = 0: zero gradients written, no kernel work."""
    q, k, v, do, ob, l32 = forward_inputs(128, 2, 2, seed=5)
    dq = torch.full((128, 2, 128), 7.0, device="cuda")
    k0 = k[:0]
    dq, dk, dv = cp.cp_attn_block_backward(*dev(q, k0, k0, ob, do, l32), dq=dq,
                                           grad_dtype=torch.float32)
    cp.cp_check_device_error()
    assert torch.all(dq == 0)
    assert dk.numel() == 0 and dv.numel() == 0


# --------------------------------------------------------- fp32 (toy)
def _fp32_case(S, H, Hkv, D, seed, q_offset=0, k_offset=0, Sk=None):
    Sk = S if Sk is None else Sk
    q, _, _ = make_qkv(S, H, D, Hkv=Hkv, seed=seed)
    _, k, v = make_qkv(Sk, H, D, Hkv=Hkv, seed=seed + 1)
    do = make_dout(S, H, D, seed=seed)
    out, lse = oracle.attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                q_offset=q_offset, k_offset=k_offset)
    o32 = torch.from_numpy(out.astype(np.float32))
    l32 = torch.from_numpy(lse.astype(np.float32))
    ref = oracle.attention_backward(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                    o32.double().numpy(), l32.double().numpy(),
                                    do.double().numpy(), q_offset=q_offset, k_offset=k_offset)
    return (q, k, v, o32, do, l32), ref


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_toy_ring_backward_fp32(cp, layout):
    """The page's toy (S=32, H=8, D=16, fp32, P=4; q, k, v of one seed-0
    draw): ring gradients against the monolithic oracle at atol 1e-5 on
    every element (CUDA-core path)."""
    q, k, v = make_qkv(32, 8, 16)
    do = make_dout(32, 8, 16, seed=0)
    out, lse = oracle.attention(q.double().numpy(), k.double().numpy(), v.double().numpy())
    o = torch.from_numpy(out.astype(np.float32))
    l = torch.from_numpy(lse.astype(np.float32))
    ref = oracle.attention_backward(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                    o.double().numpy(), l.double().numpy(), do.double().numpy())
    got = cp.cp_ring_backward(*dev(q, k, v, o, do, l), 4, layout, grad_dtype=torch.float32)
    cp.cp_check_device_error()
    for g, want, name in zip(got, ref, ("dq", "dk", "dv")):
        err = np.abs(host(g).astype(np.float64) - want).max()
        assert err <= 1e-5, f"{name}: max|err| {err:.3e}"


@pytest.mark.parametrize("D", [32, 64, 128])
def test_block_backward_fp32_gqa_offsets(cp, D):
    """fp32 block with GQA 4:2, offsets that leave the first rows without a
    key, every D of the CUDA-core path; atol 1e-5."""
    (q, k, v, o, do, l), ref = _fp32_case(40, 4, 2, D, seed=D, q_offset=8, k_offset=16, Sk=36)
    got = cp.cp_attn_block_backward(*dev(q, k, v, o, do, l), q_offset=8, k_offset=16,
                                    grad_dtype=torch.float32)
    cp.cp_check_device_error()
    for g, want, name in zip(got, ref, ("dq", "dk", "dv")):
        err = np.abs(host(g).astype(np.float64) - want).max()
        assert err <= 1e-5, f"{name}: max|err| {err:.3e}"


# ------------------------------------------------------------------- ring
@pytest.fixture(scope="module")
def ring4k():
    """S=4096, H=4 (GQA 4:2), one draw shared by the layouts: inputs and the
    oracle's monolithic gradients."""
    q, k, v, do, ob, l32 = forward_inputs(4096, 4, 2, seed=4)
    return (q, k, v, do, ob, l32), oracle_grads(q, k, v, do, ob, l32)


@pytest.mark.parametrize("layout,P", [("zigzag", 4), ("contiguous", 4), ("striped", 4),
                                      ("zigzag", 8), ("zigzag", 1)])
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
def test_ring_backward_4k(cp, ring4k, layout, P, grad_dtype):
    """Ring backward over P virtual ranks equals monolithic gradients, every
    element (chunks of 512 rows = 4 tiles; P=8: 256-row chunks)."""
    (q, k, v, do, ob, l32), (rq, rk, rv) = ring4k
    dq, dk, dv = cp.cp_ring_backward(*dev(q, k, v, ob, do, l32), P, layout,
                                     grad_dtype=grad_dtype)
    cp.cp_check_device_error()
    grads_close(dq, rq, "dq")
    grads_close(dk, rk, "dk")
    grads_close(dv, rv, "dv")


@pytest.mark.parametrize("layout,S,P", [("zigzag", 1000, 3), ("contiguous", 1000, 3),
                                        ("zigzag", 2050, 4), ("striped", 1200, 6)])
def test_ring_backward_ragged(cp, layout, S, P):
    """Chunk counts that do not divide S (short / empty last chunks, partial
    tiles inside chunks) and a striped case with 200-row stripes."""
    q, k, v, do, ob, l32 = forward_inputs(S, 2, 1, seed=S + P)
    (dq, dq_ok), (dk, dk_ok), (dv, dv_ok) = (guarded(t.shape, torch.float32) for t in (q, k, v))
    cp.cp_ring_backward(*dev(q, k, v, ob, do, l32), P, layout, dq=dq, dk=dk, dv=dv)
    cp.cp_check_device_error()
    rq, rk, rv = oracle_grads(q, k, v, do, ob, l32)
    grads_close(dq, rq, "dq")
    grads_close(dk, rk, "dk")
    grads_close(dv, rv, "dv")
    assert dq_ok() and dk_ok() and dv_ok(), "write outside dq / dk / dv"


def test_ring_backward_matches_block_sum(cp):
    """The ring's gradients equal the sum of cp_attn_block_backward over the
    step schedule's blocks (the same kernels driven block by block)."""
    S, H, P = 1024, 2, 2
    q, k, v, do, ob, l32 = forward_inputs(S, H, H, seed=31)
    dq_r, dk_r, dv_r = cp.cp_ring_backward(*dev(q, k, v, ob, do, l32), P, "zigzag",
                                           grad_dtype=torch.float32)
    C = S // (2 * P)
    qd, kd, vd, obd, dod, ld = dev(q, k, v, ob, do, l32)
    dq = torch.zeros(S, H, 128, device="cuda")
    dk = torch.zeros(S, H, 128, device="cuda")
    dv = torch.zeros(S, H, 128, device="cuda")
    for t in range(P):
        for r, qc, kc, _ in cp.cp_ring_step_blocks(P, "zigzag", t):
            qs, ks = slice(qc * C, (qc + 1) * C), slice(kc * C, (kc + 1) * C)
            a, b, c = cp.cp_attn_block_backward(
                qd[qs].contiguous(), kd[ks].contiguous(), vd[ks].contiguous(),
                obd[qs].contiguous(), dod[qs].contiguous(), ld[:, qs].contiguous(),
                q_offset=qc * C, k_offset=kc * C, grad_dtype=torch.float32)
            dq[qs] += a
            dk[ks] += b
            dv[ks] += c
    cp.cp_check_device_error()
    for got, want, name in ((dq_r, dq, "dq"), (dk_r, dk, "dk"), (dv_r, dv, "dv")):
        diff = (got - want).abs().max().item()
        assert diff <= 1e-4 * want.abs().max().item(), f"{name}: ring vs block sum {diff:.3e}"


@pytest.mark.parametrize("layout", ["zigzag", "contiguous", "striped"])
def test_ring_backward_steps_equal_whole(cp, layout):
    """cp_ring_backward (bf16: two launches over every step) is
    cp_ring_backward_fused_step over launches -1, 0, 1, bit for bit; the
    per-step schedule (cp_ring_backward_step over -1 .. 2P-1) gives the same
    gradients within the derived tolerance and against the oracle."""
    S, H, P = 2048, 2, 4
    q, k, v, do, ob, l32 = forward_inputs(S, H, 1, seed=41)
    args = dev(q, k, v, ob, do, l32)
    a = cp.cp_ring_backward(*args, P, layout, grad_dtype=torch.bfloat16)
    ws = torch.empty(cp.cp_ring_backward_workspace_size(S, H, 1, 128, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    b = [torch.empty_like(t) for t in a]
    for launch in (-1, 0, 1):
        cp.cp_ring_backward_fused_step(*args, P, layout, launch, *b, ws)
    c = [torch.empty_like(t) for t in a]
    for launch in range(-1, 2 * P):
        cp.cp_ring_backward_step(*args, P, layout, launch, *c, ws)
    cp.cp_check_device_error()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    for got, want, name in zip(c, oracle_grads(q, k, v, do, ob, l32), ("dq", "dk", "dv")):
        grads_close(got, want, name + " (per step)")


@pytest.mark.parametrize("layout,S,P,Hkv", [("zigzag", 4096, 8, 2), ("zigzag", 4096, 16, 4),
                                            ("contiguous", 4096, 8, 4), ("zigzag", 1000, 3, 2),
                                            ("contiguous", 1500, 4, 1), ("zigzag", 300, 8, 4),
                                            ("zigzag", 2048, 1, 4), ("striped", 4096, 8, 2),
                                            ("striped", 1200, 6, 4), ("striped", 2048, 16, 1),
                                            ("striped", 96, 3, 2)])
def test_ring_backward_fused_against_oracle(cp, layout, S, P, Hkv):
    """The two-launch ring backward (every step inside one dK/dV and one dQ
    launch) against the oracle's monolithic gradients: degrees 1..16, GQA
    4:1 .. 4:4, chunks that are not multiples of the 128-row tile, a short
    last chunk, striped rings (200- and 32-row stripes among them); guard
    bands around the gradients."""
    q, k, v, do, ob, l32 = forward_inputs(S, 4, Hkv, seed=S + P + Hkv)
    (dq, dq_ok), (dk, dk_ok), (dv, dv_ok) = (guarded(t.shape, torch.float32) for t in (q, k, v))
    cp.cp_ring_backward(*dev(q, k, v, ob, do, l32), P, layout, dq=dq, dk=dk, dv=dv)
    cp.cp_check_device_error()
    rq, rk, rv = oracle_grads(q, k, v, do, ob, l32)
    grads_close(dq, rq, "dq")
    grads_close(dk, rk, "dk")
    grads_close(dv, rv, "dv")
    assert dq_ok() and dk_ok() and dv_ok(), "write outside dq / dk / dv"


# ------------------------------------------------- full size, sampled rows
@pytest.mark.slow
def test_ring_backward_128k_sampled(cp):
    """S=128K, H=32, D=128, P=8 zigzag (the long workload), forward and
    backward on the GPU.  dQ on 64 seeded rows per head (plus every chunk's
    first and last row) against the oracle computed one row at a time from
    the oracle's own forward of that row; dK, dV on the last 128 key rows
    (which only the last 128 queries see); and the identity
    sum_j dV_j = sum_i dO_i, which holds for every head at any size because
    each row of P sums to one."""
    S, H, D, P = 131072, 32, 128, 8
    q, k, v = make_qkv(S, H, D, dtype=torch.bfloat16, seed=0, device="cuda")
    do = make_dout(S, H, D, dtype=torch.bfloat16, seed=0, device="cuda")
    out, lse = cp.cp_ring_forward(q, k, v, P, "zigzag")
    dq, dk, dv = cp.cp_ring_backward(q, k, v, out, do, lse, P, "zigzag",
                                     grad_dtype=torch.float32)
    cp.cp_check_device_error()
    # identity on every head
    sum_dv = dv.double().sum(0)
    sum_do = do.double().sum(0)
    rel = ((sum_dv - sum_do).abs().max() / sum_do.abs().max()).item()
    assert rel < 1e-2, f"sum dV vs sum dO: {rel:.3e}"
    C = S // (2 * P)
    must = [c * C for c in range(2 * P)] + [c * C + C - 1 for c in range(2 * P)]
    rows = sample_rows(S, 64, seed=5, must=must)
    rows_d = torch.as_tensor(rows, device="cuda")
    for h in (0, 13, 31):
        # one head at a time on the host, as [S, 1, D] fp64
        qh, kh, vh, doh = (t[:, h:h + 1].float().cpu().double().numpy() for t in (q, k, v, do))
        # dq rows: the oracle's forward and backward of each sampled row
        ref = np.zeros((len(rows), D))
        for n, i in enumerate(rows):
            o_i, l_i = oracle.attention(qh[i:i + 1], kh[:i + 1], vh[:i + 1], q_offset=i)
            g = oracle.attention_backward(qh[i:i + 1], kh[:i + 1], vh[:i + 1], o_i, l_i,
                                          doh[i:i + 1], q_offset=i)
            ref[n] = g[0][0, 0]
        grads_close(dq[rows_d, h], ref, f"dq head {h}", rms_rel=2e-2)
        # the last 128 key rows: their gradients need only the last 128 queries
        tail = slice(S - 128, S)
        o_t, l_t = oracle.attention(qh[tail], kh, vh, q_offset=S - 128)
        g = oracle.attention_backward(qh[tail], kh[tail], vh[tail], o_t, l_t, doh[tail],
                                      q_offset=S - 128, k_offset=S - 128)
        grads_close(dk[tail, h], g[1][:, 0], f"dk tail head {h}", rms_rel=2e-2)
        grads_close(dv[tail, h], g[2][:, 0], f"dv tail head {h}", rms_rel=2e-2)


# ------------------------------------------------- host-buffer ring backward
@pytest.mark.parametrize("layout,H,Hkv,groups,grad_dtype,two_streams", [
    ("zigzag", 8, 4, 2, torch.bfloat16, True),
    ("contiguous", 8, 8, 4, torch.float32, True),
    ("striped", 8, 4, 4, torch.bfloat16, False),
    ("zigzag", 8, 2, 2, torch.bfloat16, True),   # one KV head per group
])
def test_ring_backward_host_equals_device(cp, layout, H, Hkv, groups, grad_dtype, two_streams):
    """cp_ring_backward_host (host buffers, heads in groups, copies on a second
    stream) gives cp_ring_backward's gradients bit for bit."""
    S, D, P = 2048, 128, 4
    q, k, v = make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=41)
    do = make_dout(S, H, D, dtype=torch.bfloat16, seed=41)
    out, lse = cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), P, layout,
                                  out_dtype=torch.bfloat16)
    ref = cp.cp_ring_backward(q.cuda(), k.cuda(), v.cuda(), out, do.cuda(), lse, P, layout,
                              grad_dtype=grad_dtype)
    host = [t.pin_memory() for t in (q, k, v, out.cpu(), do, lse.cpu())]
    side = torch.cuda.Stream() if two_streams else None
    (hdq, dq_ok), (hdk, dk_ok), (hdv, dv_ok) = (guarded(t.shape, grad_dtype, pin=True)
                                                for t in (q, k, v))
    got = cp.cp_ring_backward_host(*host, P, layout, hdq=hdq, hdk=hdk, hdv=hdv, groups=groups,
                                   copy_stream=side)
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    for g, r in zip(got, ref):
        assert torch.equal(g, r.cpu())
    assert dq_ok() and dk_ok() and dv_ok(), "write outside the host dq / dk / dv"


def test_ring_backward_host_fp32_toy(cp):
    """The fp32 path (CUDA cores) through host buffers equals the device call."""
    q, k, v = make_qkv(64, 8, 16)
    do = make_dout(64, 8, 16, dtype=torch.float32, seed=3)
    out, lse = cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), 4, "zigzag")
    ref = cp.cp_ring_backward(q.cuda(), k.cuda(), v.cuda(), out, do.cuda(), lse, 4, "zigzag",
                              grad_dtype=torch.float32)
    got = cp.cp_ring_backward_host(q, k, v, out.cpu(), do, lse.cpu(), 4, "zigzag",
                                   grad_dtype=torch.float32, groups=2,
                                   copy_stream=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    for g, r in zip(got, ref):
        assert torch.equal(g, r.cpu())
