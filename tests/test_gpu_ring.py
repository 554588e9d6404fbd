"""GPU parity of the ring schedule, the LSE merge, the Ulysses permutation and
the Ulysses forward against the fp64 oracle.

Small workloads are checked on every element; the long ones (32K, 64K,
128K) on 512 seeded query rows per head plus every chunk's first and last
row, computed by the oracle one row at a time against the full key set.
"""

import numpy as np
import pytest
import torch

import oracle
from context_causal_attention_attn_gb300.inputs import make_qkv, sample_rows
from gpu_common import (ATOL_BF16_LSE, ATOL_BF16_OUT, ATOL_F32, compare, guarded, host,
                        ring_by_steps)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    from context_causal_attention_attn_gb300 import build
    build.build()
    import context_causal_attention_attn_gb300 as m
    return m


# ------------------------------------------------------------------ toy
@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
def test_toy_ring_fp32(cp, layout):
    """The handbook's toy: S=32, H=8, D=16, fp32, P=4, against monolithic
    causal attention at atol 1e-5 on every element."""
    q, k, v = make_qkv(32, 8, 16)
    out, lse = cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), 4, layout)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    compare(out, lse, ro, rl, ATOL_F32, ATOL_F32)


def test_toy_ulysses_fp32(cp):
    q, k, v = make_qkv(32, 8, 16)
    out, lse = cp.cp_ulysses_forward(q.cuda(), k.cuda(), v.cuda(), 4)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    compare(out, lse, ro, rl, ATOL_F32, ATOL_F32)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("P", [1, 2, 3, 5])
def test_ring_fp32_other_degrees(cp, layout, P):
    S = 2 * P * 24
    q, k, v = make_qkv(S, 4, 32, Hkv=2, seed=P)
    out, lse = cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), P, layout)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    compare(out, lse, ro, rl, ATOL_F32, ATOL_F32)


# ------------------------------------------------------------ 4K, all rows
@pytest.fixture(scope="module")
def qkv4k():
    q, k, v = make_qkv(4096, 32, 128, dtype=torch.bfloat16)
    ro, rl = oracle.attention(host(q), host(k), host(v))
    return q, k, v, ro, rl


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("layout", ["zigzag", "contiguous", "striped"])
def test_ring_4k_all_rows(cp, qkv4k, layout, out_dtype):
    """S=4096, H=32, D=128, bf16, P=4: every row and head, through
    cp_ring_forward (all steps in one launch for bf16) and through the
    per-step ring."""
    q, k, v, ro, rl = qkv4k
    out, lse = cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), 4, layout, out_dtype=out_dtype)
    cp.cp_check_device_error()
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)
    fo, fl = cp.cp_ring_forward_fused(q.cuda(), k.cuda(), v.cuda(), 4, layout,
                                      out_dtype=out_dtype)
    assert torch.equal(fo, out) and torch.equal(fl, lse)
    so, sl = ring_by_steps(cp, q.cuda(), k.cuda(), v.cuda(), 4, layout, out_dtype=out_dtype)
    cp.cp_check_device_error()
    compare(so, sl, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


# ------------------------------------------------- the ring in one launch
@pytest.mark.parametrize("S,H,Hkv,P,layout", [(2048, 4, 2, 1, "zigzag"),
                                              (2048, 4, 2, 2, "contiguous"),
                                              (2048, 4, 4, 3, "zigzag"),
                                              (2048, 8, 2, 8, "zigzag"),
                                              (4096, 2, 2, 16, "zigzag"),
                                              (4096, 2, 1, 16, "contiguous"),
                                              (1000, 8, 4, 4, "zigzag"),    # 125-row chunks
                                              (1000, 8, 4, 3, "contiguous"),
                                              (300, 4, 2, 8, "zigzag"),     # 19-row chunks
                                              (5, 2, 1, 4, "zigzag"),       # empty chunks
                                              (129, 2, 2, 2, "contiguous"),
                                              (2048, 4, 2, 4, "striped"),
                                              (1024, 8, 2, 8, "striped"),
                                              (4096, 2, 1, 16, "striped"),
                                              (1000, 4, 4, 8, "striped"),   # 125-row stripes
                                              (96, 2, 2, 3, "striped"),     # 32-row stripes
                                              (7, 2, 1, 7, "striped")])     # 1-row stripes
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_ring_fused_against_oracle(cp, S, H, Hkv, P, layout, out_dtype):
    """cp_ring_forward_fused (every step of the ring inside one launch, the
    steps' blocks walked in ring order per query tile) against the oracle on
    every row: degrees 1..16, GQA, chunk lengths that are not multiples of
    the 128-key tile, a partial last chunk and empty chunks; guard bands
    around out and lse."""
    q, k, v = make_qkv(S, H, 128, Hkv=Hkv, dtype=torch.bfloat16, seed=S + P + H)
    out, out_ok = guarded((S, H, 128), out_dtype)
    lse, lse_ok = guarded((H, S), torch.float32)
    cp.cp_ring_forward_fused(q.cuda(), k.cuda(), v.cuda(), P, layout, out=out, lse=lse)
    cp.cp_check_device_error()
    ro, rl = oracle.ring_forward(host(q), host(k), host(v), P, layout)[:2]
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)
    assert out_ok() and lse_ok(), "write outside out / lse"


def test_ring_fused_32k_sampled(cp):
    """The one-launch ring at S=32768, P=8 zigzag (every query tile walks up
    to 256 KV tiles across the 8 steps), 512 seeded rows per head against the
    oracle."""
    S, H, P = 32768, 32, 8
    q, k, v = make_qkv(S, H, 128, dtype=torch.bfloat16, device="cuda")
    out, lse = cp.cp_ring_forward_fused(q, k, v, P, "zigzag")
    cp.cp_check_device_error()
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(lse).all())
    C = S // (2 * P)
    must = [c * C for c in range(2 * P)] + [c * C + C - 1 for c in range(2 * P)]
    rows = sample_rows(S, 512, seed=1, must=must)
    ro, rl = oracle.attention_monolithic(host(q), host(k), host(v), rows=rows)
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE, rows=rows)


def test_ring_fused_deterministic_and_close_to_steps(cp):
    """Repeated one-launch rings give the same bits; the per-step ring (other
    merge order of the same terms) agrees within the bf16 tolerances."""
    S, H, P = 4096, 8, 4
    q, k, v = make_qkv(S, H, 128, dtype=torch.bfloat16, seed=77, device="cuda")
    a = cp.cp_ring_forward_fused(q, k, v, P, "zigzag", out_dtype=torch.float32)
    b = cp.cp_ring_forward_fused(q, k, v, P, "zigzag", out_dtype=torch.float32)
    s = ring_by_steps(cp, q, k, v, P, "zigzag", out_dtype=torch.float32)
    cp.cp_check_device_error()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert (a[0] - s[0]).abs().max().item() <= ATOL_BF16_OUT
    assert (a[1] - s[1]).abs().max().item() <= ATOL_BF16_LSE


def test_ring_4k_block_equals_ring(cp, qkv4k):
    """The monolithic block call and the ring agree (both against the oracle)."""
    q, k, v, ro, rl = qkv4k
    out, lse = cp.cp_attn_block(q.cuda(), k.cuda(), v.cuda(), out_dtype=torch.float32)
    cp.cp_check_device_error()
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


def test_ring_steps_resume(cp, qkv4k):
    """Stopping after step t, saving (acc, lse), and resuming later gives the
    same bits as an uninterrupted ring."""
    q, k, v, _, _ = qkv4k
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    P, layout = 4, "zigzag"
    ref_out, ref_lse = ring_by_steps(cp, q, k, v, P, layout, out_dtype=torch.bfloat16)
    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    ws = torch.empty(cp.cp_ring_workspace_size(4096, 32, 128, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    for t in range(2):
        cp.cp_ring_step(q, k, v, P, layout, t, out, lse, ws)
    saved = (ws.clone(), lse.clone(), out.clone())
    ws.zero_()
    lse.zero_()
    ws.copy_(saved[0])
    lse.copy_(saved[1])
    out.copy_(saved[2])
    for t in range(2, P):
        cp.cp_ring_step(q, k, v, P, layout, t, out, lse, ws)
    cp.cp_check_device_error()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


@pytest.mark.parametrize("layout,out_dtype", [("zigzag", torch.bfloat16),
                                              ("contiguous", torch.float32),
                                              ("striped", torch.bfloat16)])
def test_ring_overlapped_steps_equal_separate_steps(cp, layout, out_dtype):
    """cp_ring_forward_steps launches steps 1..P-1 so that each overlaps the tail of
    the step before; the result is bit for bit that of the steps launched
    one at a time (cp_ring_step), at 32K where many CTAs of consecutive steps
    run together."""
    S, H, D, P = 32768, 8, 128, 8
    q, k, v = make_qkv(S, H, D, dtype=torch.bfloat16, seed=21, device="cuda")
    ref_out, ref_lse = cp.cp_ring_forward_steps(q, k, v, P, layout, out_dtype=out_dtype)
    out, lse = torch.empty_like(ref_out), torch.empty_like(ref_lse)
    n = cp.cp_ring_workspace_size(S, H, D, out_dtype)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    for t in range(P):
        cp.cp_ring_step(q, k, v, P, layout, t, out, lse, ws if n else None)
    cp.cp_check_device_error()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    again = cp.cp_ring_forward_steps(q, k, v, P, layout, out_dtype=out_dtype)
    assert torch.equal(again[0], ref_out) and torch.equal(again[1], ref_lse)


def test_ring_deterministic(cp, qkv4k):
    q, k, v, _, _ = qkv4k
    a = cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), 4, "zigzag")
    b = cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), 4, "zigzag")
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# -------------------------------------------------------- long, sampled rows
def _sampled_check(cp, S, H, Hkv, P, layout, n_rows=512, ulysses=False, usp_Pu=0):
    q, k, v = make_qkv(S, H, 128, Hkv=Hkv, dtype=torch.bfloat16, device="cuda")
    if ulysses:
        out, lse = cp.cp_ulysses_forward(q, k, v, P)
    elif usp_Pu:
        out, lse = cp.cp_usp_forward(q, k, v, usp_Pu, P, layout)
    else:
        out, lse = cp.cp_ring_forward(q, k, v, P, layout)
    cp.cp_check_device_error()
    # no NaN / Inf anywhere (every row of a causal sequence sees a key)
    assert bool(torch.isfinite(out).all()), "non-finite output"
    assert bool(torch.isfinite(lse).all()), "non-finite lse"
    nch = 2 * P if layout == "zigzag" else P
    C = S // nch
    must = [c * C for c in range(nch)] + [c * C + C - 1 for c in range(nch)]
    if layout == "striped":
        must = list(range(2 * P)) + list(range(S - 2 * P, S))
    rows = sample_rows(S, n_rows, seed=1, must=must)
    qh, kh, vh = host(q), host(k), host(v)
    ro, rl = oracle.attention_monolithic(qh, kh, vh, rows=rows)
    return compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE, rows=rows)


def test_ring_32k_zigzag_sampled(cp):
    _sampled_check(cp, 32768, 32, 32, 8, "zigzag")


@pytest.mark.parametrize("Hkv,P,layout", [(8, 16, "zigzag"), (32, 8, "contiguous"),
                                          (4, 4, "striped")])
def test_ring_32k_more_sampled(cp, Hkv, P, layout):
    """The one-launch ring at 32K in other shapes of its grid: GQA 32/8 with
    16 ranks (32 chunks of 1024 rows) and striped with GQA 32/4, whose K/V
    fits in L2 (the grid runs in the items' order across the heads), and
    contiguous chunks with 32 KV heads (head by head, shortest tiles last
    across the heads)."""
    _sampled_check(cp, 32768, 32, Hkv, P, layout)


@pytest.mark.parametrize("layout", ["zigzag", "contiguous", "striped"])
def test_ring_128k_sampled(cp, layout):
    _sampled_check(cp, 131072, 32, 32, 8, layout)


def test_ulysses_64k_gqa_sampled(cp):
    """S=65536, 32 query / 8 KV heads, P=8 (one KV head per virtual rank)."""
    _sampled_check(cp, 65536, 32, 8, 8, "contiguous", ulysses=True)


def test_usp_64k_gqa_sampled(cp):
    """S=65536, 32 query / 8 KV heads, Ulysses over 4 head groups x a zigzag
    ring of 2 in each: the four groups' rings share one launch, run head by
    head (the groups' K/V is more than half of L2)."""
    _sampled_check(cp, 65536, 32, 8, 2, "zigzag", usp_Pu=4)


# ------------------------------------------------------------ Ulysses small
@pytest.mark.parametrize("P,H,Hkv", [(2, 8, 2), (4, 8, 4), (8, 32, 8)])
def test_ulysses_bf16_all_rows(cp, P, H, Hkv):
    q, k, v = make_qkv(1024, H, 128, Hkv=Hkv, dtype=torch.bfloat16, seed=P)
    out, lse = cp.cp_ulysses_forward(q.cuda(), k.cuda(), v.cuda(), P, out_dtype=torch.float32)
    cp.cp_check_device_error()
    ro, rl = oracle.ulysses_forward(host(q), host(k), host(v), P)
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


# ---------------------------------------------------------------- permute
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("S,H,D,P", [(64, 8, 128, 4), (96, 6, 3, 3), (40, 4, 5, 2),
                                     (4096, 32, 128, 8), (256, 8, 128, 8)])
def test_permute_bit_exact(cp, dtype, S, H, D, P):
    x = torch.randn(S, H, D, generator=torch.Generator().manual_seed(S + H)).to(dtype)
    y = cp.cp_seq_to_head(x.cuda(), P)
    torch.cuda.synchronize()
    want = oracle.seq_to_head(x.view(torch.int16 if dtype == torch.bfloat16 else torch.int32)
                              .numpy(), P)
    got = y.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy()
    assert np.array_equal(got, want)
    back = cp.cp_head_to_seq(y)
    torch.cuda.synchronize()
    assert torch.equal(back.cpu(), x)


def test_permute_64k_bit_exact(cp):
    x = make_qkv(65536, 32, 128, dtype=torch.bfloat16, device="cuda")[0]
    y = cp.cp_seq_to_head(x, 8)
    torch.cuda.synchronize()
    want = x.view(65536, 8, 4 * 128).transpose(0, 1).contiguous().view(8, 65536, 4, 128)
    assert torch.equal(y, want)
    assert torch.equal(cp.cp_head_to_seq(y), x)


# ------------------------------------------------------------------ merge
def _partials(Sq, H, D, seed, empty_frac=0.1):
    rng = np.random.default_rng(seed)
    oa, ob = rng.standard_normal((Sq, H, D)), rng.standard_normal((Sq, H, D))
    la, lb = rng.standard_normal((H, Sq)) * 3, rng.standard_normal((H, Sq)) * 3
    la[rng.random((H, Sq)) < empty_frac] = -np.inf
    lb[rng.random((H, Sq)) < empty_frac] = -np.inf
    oa[~np.isfinite(la).T] = 0
    ob[~np.isfinite(lb).T] = 0
    return [x.astype(np.float32) for x in (oa, la, ob, lb)]


@pytest.mark.parametrize("Sq,H,D", [(300, 4, 128), (77, 8, 16), (64, 3, 64), (33, 2, 256)])
def test_lse_merge(cp, Sq, H, D):
    oa, la, ob, lb = _partials(Sq, H, D, Sq)
    acc, lacc = torch.from_numpy(oa).cuda(), torch.from_numpy(la).cuda()
    cp.cp_lse_merge(acc, lacc, torch.from_numpy(ob).cuda(), torch.from_numpy(lb).cuda())
    torch.cuda.synchronize()
    ro, rl = oracle.lse_merge(oa, la, ob, lb)
    compare(acc, lacc, ro, rl, ATOL_F32, ATOL_F32)


def test_lse_merge_matches_split_attention(cp):
    """merge(attn(K1), attn(K2)) on the GPU = attn(K1 u K2) from the oracle."""
    q, k, v = make_qkv(512, 4, 128, dtype=torch.bfloat16, seed=9)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    a, la = cp.cp_attn_block(qc, kc[:200].contiguous(), vc[:200].contiguous(),
                             out_dtype=torch.float32)
    b, lb = cp.cp_attn_block(qc, kc[200:].contiguous(), vc[200:].contiguous(), k_offset=200,
                             out_dtype=torch.float32)
    cp.cp_lse_merge(a, la, b, lb)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(host(q), host(k), host(v))
    compare(a, la, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


# ------------------------------------------- striped, ragged lengths, replicated KV
@pytest.mark.parametrize("S,P,layout", [(37, 4, "contiguous"), (37, 4, "zigzag"), (50, 3, "zigzag"),
                                        (5, 4, "zigzag"), (32, 4, "striped"), (60, 3, "striped")])
def test_ring_fp32_ragged_and_striped(cp, S, P, layout):
    q, k, v = make_qkv(S, 4, 16, Hkv=2, seed=S + P)
    out, out_ok = guarded((S, 4, 16), torch.float32)
    lse, lse_ok = guarded((4, S), torch.float32)
    cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), P, layout, out=out, lse=lse)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    compare(out, lse, ro, rl, ATOL_F32, ATOL_F32)
    assert out_ok() and lse_ok(), "write outside out / lse"


@pytest.mark.parametrize("S,P,layout", [(1000, 4, "zigzag"), (1000, 4, "contiguous"),
                                        (4096, 4, "striped"), (2048, 8, "striped"),
                                        (300, 8, "zigzag")])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_ring_bf16_ragged_and_striped(cp, S, P, layout, out_dtype):
    q, k, v = make_qkv(S, 8, 128, Hkv=4, dtype=torch.bfloat16, seed=S + P)
    out, out_ok = guarded((S, 8, 128), out_dtype)
    lse, lse_ok = guarded((8, S), torch.float32)
    cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), P, layout, out=out, lse=lse)
    cp.cp_check_device_error()
    ro, rl = oracle.ring_forward(host(q), host(k), host(v), P, layout)[:2]
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)
    assert out_ok() and lse_ok(), "write outside out / lse"


def test_ring_32k_striped_sampled(cp):
    _sampled_check(cp, 32768, 32, 32, 8, "striped")


@pytest.mark.parametrize("S,H,Hkv,P", [(1024, 32, 4, 8), (2048, 32, 8, 16), (512, 16, 2, 4)])
def test_ulysses_replicated_kv_bf16(cp, S, H, Hkv, P):
    """Degree above the KV head count: each KV head serves P/Hkv ranks."""
    q, k, v = make_qkv(S, H, 128, Hkv=Hkv, dtype=torch.bfloat16, seed=P)
    out, lse = cp.cp_ulysses_forward(q.cuda(), k.cuda(), v.cuda(), P, out_dtype=torch.float32)
    cp.cp_check_device_error()
    ro, rl = oracle.ulysses_forward(host(q), host(k), host(v), P)
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


def test_ulysses_replicated_kv_fp32(cp):
    q, k, v = make_qkv(64, 8, 16, Hkv=2, seed=11)
    out, lse = cp.cp_ulysses_forward(q.cuda(), k.cuda(), v.cuda(), 8)
    cp.cp_check_device_error()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    compare(out, lse, ro, rl, ATOL_F32, ATOL_F32)


# ------------------------------------------------------- copy-mode ring
@pytest.mark.parametrize("S,P,layout", [(4096, 4, "zigzag"), (4096, 4, "contiguous"),
                                        (4096, 4, "striped"), (1000, 4, "zigzag"),
                                        (1000, 3, "contiguous")])
def test_ring_copy_mode_equals_in_place(cp, S, P, layout):
    """KV passed rank to rank through double buffers on a second stream gives
    the same bits as the in-place ring, and matches the oracle."""
    q, k, v = make_qkv(S, 8, 128, Hkv=4, dtype=torch.bfloat16, seed=S + P, device="cuda")
    ref = ring_by_steps(cp, q, k, v, P, layout, out_dtype=torch.bfloat16)
    side = torch.cuda.Stream()
    out, lse = cp.cp_ring_forward_copy(q, k, v, P, layout, out_dtype=torch.bfloat16,
                                       copy_stream=side)
    cp.cp_check_device_error()
    torch.cuda.synchronize()
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])
    ro, rl = oracle.attention(host(q), host(k), host(v))
    compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


def test_ring_copy_mode_fp32_toy(cp):
    q, k, v = make_qkv(32, 8, 16)
    out, lse = cp.cp_ring_forward_copy(q.cuda(), k.cuda(), v.cuda(), 4, "contiguous",
                                       copy_stream=torch.cuda.Stream())
    cp.cp_check_device_error()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    compare(out, lse, ro, rl, ATOL_F32, ATOL_F32)


# ------------------------------------------------------------- USP hybrid
@pytest.mark.parametrize("S,H,Hkv,Pu,Pr,layout", [(1024, 32, 8, 4, 2, "zigzag"),
                                                  (1024, 16, 2, 4, 2, "striped"),
                                                  (1024, 16, 2, 4, 2, "zigzag"),
                                                  (1000, 8, 4, 2, 3, "contiguous"),
                                                  (2048, 32, 8, 8, 4, "zigzag")])
def test_usp_bf16(cp, S, H, Hkv, Pu, Pr, layout):
    """Ulysses over Pu head groups x ring of Pr ranks = monolithic attention."""
    q, k, v = make_qkv(S, H, 128, Hkv=Hkv, dtype=torch.bfloat16, seed=S + Pu + Pr)
    for out_dtype in (torch.bfloat16, torch.float32):
        out, lse = cp.cp_usp_forward(q.cuda(), k.cuda(), v.cuda(), Pu, Pr, layout,
                                     out_dtype=out_dtype)
        cp.cp_check_device_error()
        ro, rl = oracle.usp_forward(host(q), host(k), host(v), Pu, Pr, layout)
        compare(out, lse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


def test_usp_fp32_toy(cp):
    q, k, v = make_qkv(32, 8, 16)
    out, lse = cp.cp_usp_forward(q.cuda(), k.cuda(), v.cuda(), 2, 2, "zigzag")
    cp.cp_check_device_error()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    compare(out, lse, ro, rl, ATOL_F32, ATOL_F32)


# ------------------------------------------------------- host-buffer ring
@pytest.mark.parametrize("layout,groups,Hkv,pinned,two_streams", [
    ("zigzag", 1, 8, True, False),
    ("zigzag", 4, 8, True, True),
    ("contiguous", 2, 8, False, True),
    ("striped", 8, 8, True, True),
    ("zigzag", 2, 2, True, True),   # GQA 8 / 2: each group holds one KV head
])
def test_ring_host_equals_device_ring(cp, layout, groups, Hkv, pinned, two_streams):
    """cp_ring_forward_host (host buffers, heads in groups, copies on a
    second stream) gives the device ring's result bit for bit: heads are
    independent and each group runs the same launches on its heads."""
    S, H, D, P = 1536, 8, 128, 4
    q, k, v = make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=5)
    ref_out, ref_lse = cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), P, layout,
                                     out_dtype=torch.bfloat16)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    side = torch.cuda.Stream() if two_streams else None
    hout, hlse = cp.cp_ring_forward_host(q, k, v, P, layout, out_dtype=torch.bfloat16,
                                         groups=groups, copy_stream=side)
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    assert torch.equal(hout, ref_out.cpu())
    assert torch.equal(hlse, ref_lse.cpu())


def test_ring_host_against_oracle(cp):
    """The host-buffer ring at 4K (H=32, P=4 zigzag, 4 head groups) against
    the oracle on every row."""
    S, H, D, P = 4096, 32, 128, 4
    q, k, v = make_qkv(S, H, D, dtype=torch.bfloat16)
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    hout, hlse = cp.cp_ring_forward_host(q, k, v, P, "zigzag", out_dtype=torch.bfloat16,
                                         groups=4, copy_stream=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    ro, rl = oracle.attention(*(t.double().numpy() for t in (q, k, v)))
    compare(hout, hlse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


def test_ring_host_fp32_toy(cp):
    """The fp32 toy through host buffers (CUDA-core path), atol 1e-5."""
    q, k, v = make_qkv(32, 8, 16)
    hout, hlse = cp.cp_ring_forward_host(q, k, v, 4, "contiguous", groups=2,
                                         copy_stream=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    compare(hout, hlse, ro, rl, ATOL_F32, ATOL_F32)


def test_ring_host_back_to_back_calls(cp):
    """Consecutive calls on the same streams and workspace (the staging of
    call i+1 is overwritten only after call i has finished with it)."""
    S, H, D, P = 2048, 8, 128, 2
    dev = torch.device("cuda")
    ins = [tuple(t.pin_memory() for t in make_qkv(S, H, D, dtype=torch.bfloat16, seed=s))
           for s in (11, 12, 13)]
    side = torch.cuda.Stream()
    ws = torch.empty(cp.cp_ring_host_workspace_size(S, H, H, D, 4, torch.bfloat16,
                                                    torch.bfloat16), dtype=torch.uint8,
                     device=dev)
    outs = [cp.cp_ring_forward_host(*x, P, "zigzag", out_dtype=torch.bfloat16, groups=4,
                                    workspace=ws, copy_stream=side) for x in ins]
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    for (q, k, v), (hout, hlse) in zip(ins, outs):
        ro, rl = cp.cp_ring_forward(q.to(dev), k.to(dev), v.to(dev), P, "zigzag",
                               out_dtype=torch.bfloat16)
        assert torch.equal(hout, ro.cpu()) and torch.equal(hlse, rl.cpu())


# --------------------------------------------------- staged Ulysses / USP
@pytest.mark.parametrize("H,Hkv,P", [(8, 4, 4), (8, 2, 4)])
def test_ulysses_stages_equal_forward(cp, H, Hkv, P):
    """cp_ulysses_stage 0, 1, 2 in order is cp_ulysses_forward bit for bit
    (P dividing Hkv, and P a multiple of Hkv with replicated KV heads)."""
    S, D = 1024, 128
    q, k, v = (t.cuda() for t in make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=9))
    ref_out, ref_lse = cp.cp_ulysses_forward(q, k, v, P)
    out, lse = torch.empty_like(ref_out), torch.empty_like(ref_lse)
    ws = torch.empty(cp.cp_ulysses_workspace_size(S, H, Hkv, D, q.dtype, out.dtype),
                     dtype=torch.uint8, device=q.device)
    for st in range(3):
        cp.cp_ulysses_stage(q, k, v, P, st, out, lse, ws)
    cp.cp_check_device_error()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    with pytest.raises(cp.CpError):
        cp.cp_ulysses_stage(q, k, v, P, 3, out, lse, ws)


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_usp_stages_equal_forward(cp, layout):
    """cp_usp_stage 0 .. Pr+1 in order is cp_usp_forward bit for bit."""
    S, H, Hkv, D, Pu, Pr = 2048, 8, 4, 128, 2, 4
    q, k, v = (t.cuda() for t in make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=10))
    ref_out, ref_lse = cp.cp_usp_forward(q, k, v, Pu, Pr, layout, out_dtype=torch.bfloat16)
    out, lse = torch.empty_like(ref_out), torch.empty_like(ref_lse)
    ws = torch.empty(cp.cp_usp_workspace_size(S, H, Hkv, D, q.dtype, out.dtype),
                     dtype=torch.uint8, device=q.device)
    for st in range(Pr + 2):
        cp.cp_usp_stage(q, k, v, Pu, Pr, layout, st, out, lse, ws)
    cp.cp_check_device_error()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    with pytest.raises(cp.CpError):
        cp.cp_usp_stage(q, k, v, Pu, Pr, layout, Pr + 2, out, lse, ws)


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("entry", ["cp_ring_forward", "cp_ring_forward_steps"])
def test_ring_forward_in_cuda_graph(cp, layout, entry):
    """The ring captured into a CUDA graph (one launch; or one per step, those
    after the first carrying programmatic dependencies) replays to the eager
    result bit for bit; replaying is how a caller removes the host cost of
    small rings."""
    S, H, D, P = 4096, 32, 128, 4
    fn = getattr(cp, entry)
    q, k, v = make_qkv(S, H, D, dtype=torch.bfloat16, seed=31, device="cuda")
    out = torch.empty(S, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(H, S, dtype=torch.float32, device="cuda")
    ws = torch.empty(cp.cp_ring_workspace_size(S, H, D, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    ref = fn(q, k, v, P, layout, out_dtype=torch.bfloat16)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(q, k, v, P, layout, out=out, lse=lse, workspace=ws, stream=s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn(q, k, v, P, layout, out=out, lse=lse, workspace=ws, stream=s)
        out.zero_()
        lse.zero_()
        for _ in range(3):
            g.replay()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    cp.cp_check_device_error()
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])


@pytest.mark.parametrize("S,layout,out_dtype", [(1000, "zigzag", torch.float32),
                                                (1000, "contiguous", torch.bfloat16)])
def test_ring_host_ragged(cp, S, layout, out_dtype):
    """Host-buffer ring on a length the chunk count does not divide (short
    last chunks), with fp32 and bf16 output: equal to the device ring."""
    H, D, P = 8, 128, 4
    q, k, v = make_qkv(S, H, D, Hkv=4, dtype=torch.bfloat16, seed=17)
    ref_out, ref_lse = cp.cp_ring_forward(q.cuda(), k.cuda(), v.cuda(), P, layout,
                                     out_dtype=out_dtype)
    hout, out_ok = guarded((S, H, D), out_dtype, pin=True)
    hlse, lse_ok = guarded((H, S), torch.float32, pin=True)
    cp.cp_ring_forward_host(*(t.pin_memory() for t in (q, k, v)), P, layout, hout=hout,
                            hlse=hlse, groups=2, copy_stream=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    assert torch.equal(hout, ref_out.cpu()) and torch.equal(hlse, ref_lse.cpu())
    assert out_ok() and lse_ok(), "write outside the host out / lse"


# --------------------------------------------------------- host-buffer Ulysses
@pytest.mark.parametrize("H,Hkv,P,two_streams", [(8, 4, 4, True), (8, 2, 4, True),
                                                  (8, 8, 2, False)])
def test_ulysses_host_equals_device(cp, H, Hkv, P, two_streams):
    """cp_ulysses_forward_host (strided copies do the all-to-alls; P a divisor
    or a multiple of Hkv) equals cp_ulysses_forward bit for bit."""
    S, D = 1024, 128
    q, k, v = make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=23)
    ref_out, ref_lse = cp.cp_ulysses_forward(q.cuda(), k.cuda(), v.cuda(), P)
    side = torch.cuda.Stream() if two_streams else None
    hout, hlse = cp.cp_ulysses_forward_host(*(t.pin_memory() for t in (q, k, v)), P,
                                            copy_stream=side)
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    assert torch.equal(hout, ref_out.cpu()) and torch.equal(hlse, ref_lse.cpu())


@pytest.mark.parametrize("layout,Hkv", [("zigzag", 4), ("striped", 2)])
def test_usp_host_equals_device(cp, layout, Hkv):
    """cp_usp_forward_host (strided copies, a ring in every Ulysses group)
    equals cp_usp_forward bit for bit (Pu dividing Hkv, and a multiple of
    it)."""
    S, H, D, Pu, Pr = 2048, 8, 128, 4, 2
    q, k, v = make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=29)
    ref_out, ref_lse = cp.cp_usp_forward(q.cuda(), k.cuda(), v.cuda(), Pu, Pr, layout,
                                         out_dtype=torch.bfloat16)
    hout, hlse = cp.cp_usp_forward_host(*(t.pin_memory() for t in (q, k, v)), Pu, Pr, layout,
                                        out_dtype=torch.bfloat16, copy_stream=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    assert torch.equal(hout, ref_out.cpu()) and torch.equal(hlse, ref_lse.cpu())


@pytest.mark.parametrize("H,Hkv,P,out_dtype", [(8, 4, 4, torch.float32),
                                                (8, 2, 4, torch.bfloat16),
                                                (32, 8, 8, torch.bfloat16)])
def test_ulysses_host_against_oracle(cp, H, Hkv, P, out_dtype):
    """cp_ulysses_forward_host against the oracle's Ulysses forward on every
    row (P dividing Hkv, P a multiple of Hkv, and the 64K config's head
    shape at S=1024)."""
    S, D = 1024, 128
    q, k, v = make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=41 + P + Hkv)
    hout, hlse = cp.cp_ulysses_forward_host(*(t.pin_memory() for t in (q, k, v)), P,
                                            out_dtype=out_dtype,
                                            copy_stream=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    ro, rl = oracle.ulysses_forward(host(q), host(k), host(v), P)
    compare(hout, hlse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)


@pytest.mark.parametrize("layout,Hkv,Pu,Pr,out_dtype", [("zigzag", 4, 4, 2, torch.bfloat16),
                                                        ("striped", 2, 4, 2, torch.float32),
                                                        ("contiguous", 8, 2, 3, torch.bfloat16)])
def test_usp_host_against_oracle(cp, layout, Hkv, Pu, Pr, out_dtype):
    """cp_usp_forward_host against the oracle's USP forward on every row."""
    S, H, D = 1020 if layout == "contiguous" else 1024, 8, 128
    q, k, v = make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=51 + Pu + Pr)
    hout, hlse = cp.cp_usp_forward_host(*(t.pin_memory() for t in (q, k, v)), Pu, Pr, layout,
                                        out_dtype=out_dtype, copy_stream=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    cp.cp_check_device_error()
    ro, rl = oracle.usp_forward(host(q), host(k), host(v), Pu, Pr, layout)
    compare(hout, hlse, ro, rl, ATOL_BF16_OUT, ATOL_BF16_LSE)
