"""Pins of the fp64 oracle against things other than itself.

Each pin is a check function returning an error measure; the tests assert the
error is tiny, and ``test_planted_*`` plant a plausible mistake in the oracle
(on the CPU, via monkeypatch) and assert that at least one pin catches it.

Pins used:
  * brute force: pure-Python scalar loops of the softmax definition
    (e^s / sum e^s, no max shift) on tiny inputs;
  * library routine: torch's scaled_dot_product_attention in float64 (causal
    and non-causal, with GQA) for the cases that reduce to it;
  * closed forms: q = 0 gives uniform weights (out = prefix mean of v,
    lse = log(#visible)); a row seeing one key returns that key's v;
  * identities the pages state: merge(attn(K1), attn(K2)) = attn(K1 u K2),
    ring (contiguous, zigzag, striped, padded) over virtual ranks = monolithic
    causal attention, Ulysses (also with replicated KV heads) = monolithic,
    zigzag gives every rank equal work, striped nearly equal work per step;
  * page values: block counts of the contiguous ring, ``work`` values.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.blockattn as oatt
import oracle.ring as oring

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ----------------------------------------------------------------- brute force
def brute_attention(q, k, v, causal, q_off, k_off):
    """Scalar loops: w_ij = e^(s_ij) / sum_j e^(s_ij) over visible keys."""
    Sq, H, D = q.shape
    Sk, Hkv, _ = k.shape
    grp = H // Hkv
    out = [[[0.0] * D for _ in range(H)] for _ in range(Sq)]
    lse = [[-math.inf] * Sq for _ in range(H)]
    for h in range(H):
        hk = h // grp
        for i in range(Sq):
            e = []
            for j in range(Sk):
                if causal and (j + k_off) > (i + q_off):
                    continue
                s = sum(float(q[i, h, d]) * float(k[j, hk, d]) for d in range(D))
                e.append((j, math.exp(s / math.sqrt(D))))
            tot = sum(x for _, x in e)
            if not e:
                continue
            lse[h][i] = math.log(tot)
            for d in range(D):
                out[i][h][d] = sum(x * float(v[j, hk, d]) for j, x in e) / tot
    return np.array(out), np.array(lse)


def pin_brute_force():
    worst = 0.0
    cases = [  # Sq, Sk, H, Hkv, D, causal, q_off, k_off
        (5, 7, 2, 2, 4, True, 3, 0),
        (6, 6, 4, 2, 3, True, 0, 0),
        (4, 8, 2, 1, 5, False, 0, 0),
        (7, 5, 2, 2, 4, True, 2, 4),   # some rows fully masked
        (8, 3, 3, 3, 2, True, 10, 0),  # all keys visible
    ]
    for n, (Sq, Sk, H, Hkv, D, causal, qo, ko) in enumerate(cases):
        q = _rand((Sq, H, D), 10 + n)
        k = _rand((Sk, Hkv, D), 20 + n)
        v = _rand((Sk, Hkv, D), 30 + n)
        o, l = oracle.attention(q, k, v, causal=causal, q_offset=qo, k_offset=ko)
        bo, bl = brute_attention(q, k, v, causal, qo, ko)
        worst = max(worst, np.max(np.abs(o - bo)))
        fin = np.isfinite(bl)
        if not np.array_equal(fin, np.isfinite(l)):
            return np.inf
        worst = max(worst, np.max(np.abs(l[fin] - bl[fin]), initial=0.0))
    return worst


def test_brute_force():
    assert pin_brute_force() < 1e-12


# ------------------------------------------------------------ library routine
def _sdpa(q, k, v, causal):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).double().permute(1, 0, 2)[None]
    H, Hkv = q.shape[1], k.shape[1]
    o = torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k), t(v), is_causal=causal, enable_gqa=(H != Hkv))
    return o[0].permute(1, 0, 2).numpy()


def pin_sdpa():
    worst = 0.0
    for n, (S, H, Hkv, D) in enumerate([(33, 4, 4, 16), (40, 8, 2, 8), (17, 6, 3, 12)]):
        q, k, v = _rand((S, H, D), 40 + n), _rand((S, Hkv, D), 50 + n), _rand((S, Hkv, D), 60 + n)
        # causal, aligned offsets: standard causal attention
        o, _ = oracle.attention(q, k, v, causal=True, q_offset=5, k_offset=5)
        worst = max(worst, np.max(np.abs(o - _sdpa(q, k, v, True))))
        # causal but every key before every query: plain (non-causal) attention
        o, _ = oracle.attention(q, k, v, causal=True, q_offset=1000, k_offset=3)
        worst = max(worst, np.max(np.abs(o - _sdpa(q, k, v, False))))
        o, _ = oracle.attention(q, k, v, causal=False)
        worst = max(worst, np.max(np.abs(o - _sdpa(q, k, v, False))))
    return worst


def test_library_sdpa():
    assert pin_sdpa() < 1e-12


# --------------------------------------------------------------- closed forms
def pin_closed_forms():
    worst = 0.0
    S, H, D = 24, 3, 8
    k, v = _rand((S, H, D), 1), _rand((S, H, D), 2)
    o, l = oracle.attention(np.zeros((S, H, D)), k, v, causal=True)
    for i in range(S):
        worst = max(worst, np.max(np.abs(o[i] - v[:i + 1].mean(axis=0))))
        worst = max(worst, np.max(np.abs(l[:, i] - math.log(i + 1))))
    # query offset 2 ahead of the keys: row i sees i + 3 keys
    o, l = oracle.attention(np.zeros((S - 2, H, D)), k, v, causal=True, q_offset=2)
    for i in range(S - 2):
        worst = max(worst, np.max(np.abs(o[i] - v[:i + 3].mean(axis=0))))
        worst = max(worst, np.max(np.abs(l[:, i] - math.log(i + 3))))
    # row 0 sees exactly key 0
    q = _rand((S, H, D), 3)
    o, l = oracle.attention(q, k, v, causal=True)
    worst = max(worst, np.max(np.abs(o[0] - v[0])))
    worst = max(worst, np.max(np.abs(l[:, 0] - np.sum(q[0] * k[0], axis=1) / math.sqrt(D))))
    return worst


def test_closed_forms():
    assert pin_closed_forms() < 1e-12


# ------------------------------------------------------------ sampled rows
def pin_sampled_rows():
    """The sampled-row path every long GPU test relies on: rows given as
    positions (unsorted, first and last included), evaluated in small row
    blocks so each block truncates the keys at its own largest position.
    Checked against torch's float64 SDPA of the whole sequence (out) and the
    brute-force-pinned full oracle (lse) at those rows."""
    worst = 0.0
    S, H, Hkv, D = 300, 4, 2, 16
    q, k, v = _rand((S, H, D), 111), _rand((S, Hkv, D), 112), _rand((S, Hkv, D), 113)
    rng = np.random.default_rng(114)
    rows = np.concatenate([rng.choice(np.arange(1, S - 1), 40, replace=False), [S - 1, 0]])
    rng.shuffle(rows)
    ref_out = _sdpa(q, k, v, True)[rows]
    ref_lse = oracle.attention(q, k, v, causal=True)[1][:, rows]
    for got in (oracle.attention_monolithic(q, k, v, rows=rows),
                oracle.attention(q[rows], k, v, causal=True, q_positions=rows, row_block=7)):
        worst = max(worst, np.max(np.abs(got[0] - ref_out)), np.max(np.abs(got[1] - ref_lse)))
    return worst


def test_sampled_rows():
    assert pin_sampled_rows() < 1e-12


def test_fully_masked_rows():
    q, k, v = _rand((4, 2, 4), 5), _rand((6, 2, 4), 6), _rand((6, 2, 4), 7)
    o, l = oracle.attention(q, k, v, causal=True, q_offset=0, k_offset=2)
    # rows 0 and 1 see no key
    assert np.all(l[:, :2] == -np.inf) and np.all(o[:2] == 0)
    assert np.all(np.isfinite(l[:, 2:])) and np.all(np.isfinite(o))


def test_nonfinite_scores_follow_logsumexp():
    """A key row of +inf (scores +inf or -inf by the sign of q) and a NaN
    query: lse and out as the page's torch.logsumexp and exp(s - lse) @ v
    give them in float64, row by row (masked keys are -inf, not NaN)."""
    S, H, D = 6, 1, 4
    q, k, v = _rand((S, H, D), 13), _rand((S, H, D), 14), _rand((S, H, D), 15)
    k[2, 0, 1] = np.inf
    q[4, 0, 3] = np.nan
    o, l = oracle.attention(q, k, v, causal=True)
    qt, kt, vt = (torch.from_numpy(a[:, 0, :]) for a in (q, k, v))
    s = (qt @ kt.T) / math.sqrt(D)
    s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -math.inf)
    ref_l = torch.logsumexp(s, dim=-1)
    ref_o = torch.exp(s - ref_l[:, None]) @ vt
    assert np.array_equal(l[0], ref_l.numpy(), equal_nan=True)
    assert np.allclose(o[:, 0, :], ref_o.numpy(), rtol=0, atol=1e-12, equal_nan=True)
    assert np.isnan(l[0, 4]) and np.all(np.isnan(o[4, 0]))
    assert np.all(np.isfinite(l[0, :2])), "rows before the infinite key are unaffected"


def test_shift_invariance_of_offsets():
    q, k, v = _rand((9, 2, 4), 8), _rand((9, 2, 4), 9), _rand((9, 2, 4), 10)
    a = oracle.attention(q, k, v, q_offset=3, k_offset=1)
    b = oracle.attention(q, k, v, q_offset=103, k_offset=101)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------- LSE merge
def pin_merge_identity():
    worst = 0.0
    for n in range(4):
        S, H, Hkv, D = 19, 4, 2, 8
        q, k, v = _rand((S, H, D), 70 + n), _rand((S, Hkv, D), 80 + n), _rand((S, Hkv, D), 90 + n)
        cut = 3 + 4 * n
        full = oracle.attention(q, k, v, causal=True)
        a = oracle.attention(q, k[:cut], v[:cut], causal=True)
        b = oracle.attention(q, k[cut:], v[cut:], causal=True, k_offset=cut)
        m = oracle.lse_merge(*a, *b)
        m2 = oracle.lse_merge(*b, *a)  # commutativity
        worst = max(worst, np.max(np.abs(m[0] - full[0])), np.max(np.abs(m2[0] - full[0])))
        fin = np.isfinite(full[1])
        worst = max(worst, np.max(np.abs(m[1][fin] - full[1][fin])))
        # associativity over a three-way split
        c1, c2 = cut // 2 + 1, cut + 2
        p1 = oracle.attention(q, k[:c1], v[:c1], causal=True)
        p2 = oracle.attention(q, k[c1:c2], v[c1:c2], causal=True, k_offset=c1)
        p3 = oracle.attention(q, k[c2:], v[c2:], causal=True, k_offset=c2)
        left = oracle.lse_merge(*oracle.lse_merge(*p1, *p2), *p3)
        right = oracle.lse_merge(*p1, *oracle.lse_merge(*p2, *p3))
        worst = max(worst, np.max(np.abs(left[0] - full[0])), np.max(np.abs(right[0] - full[0])))
    return worst


def test_merge_identity():
    assert pin_merge_identity() < 1e-12


def test_merge_with_empty_block():
    o = _rand((3, 2, 4), 11)
    l = _rand((2, 3), 12)
    z, zl = np.zeros_like(o), np.full_like(l, -np.inf)
    mo, ml = oracle.lse_merge(o, l, z, zl)
    assert np.array_equal(ml, l) and np.max(np.abs(mo - o)) == 0
    mo, ml = oracle.lse_merge(z, zl, z, zl)
    assert np.all(ml == -np.inf) and np.all(mo == 0)


# ----------------------------------------------------------------- ring
def pin_ring_equals_monolithic():
    worst = 0.0
    for layout in ("contiguous", "zigzag"):
        for P in (1, 2, 3, 4):
            S = 2 * P * 5
            H, Hkv, D = 4, 2, 8
            q, k, v = _rand((S, H, D), P), _rand((S, Hkv, D), 10 + P), _rand((S, Hkv, D), 20 + P)
            ro, rl, _ = oracle.ring_forward(q, k, v, P, layout)
            mo, ml = oracle.attention(q, k, v, causal=True)
            worst = max(worst, np.max(np.abs(ro - mo)), np.max(np.abs(rl - ml)))
    return worst


def test_ring_equals_monolithic():
    assert pin_ring_equals_monolithic() < 1e-12


def test_ring_counts_page_values():
    with open(os.path.join(GOLDEN, "page_ring_counts.json")) as f:
        g = json.load(f)
    S, H, D = 32, 8, 16
    q, k, v = (t.numpy() for t in _page_toy(S, H, D))
    _, _, counts = oracle.ring_forward(q, k, v, g["P"], g["layout"])
    assert counts[0] == g["first_rank_blocks"]
    assert counts[-1] == g["last_rank_blocks"]
    assert counts == sorted(counts)


def test_contiguous_counts_follow_skip_rule():
    for P in (2, 3, 5, 8):
        sched = oracle.ring_schedule(P, "contiguous")
        counts = [sum(len(ks) for step in sched for qc, ks in step[r]["pairs"]) for r in range(P)]
        assert counts == list(range(1, P + 1))


def test_work_page_values():
    with open(os.path.join(GOLDEN, "page_zigzag_work.json")) as f:
        g = json.load(f)
    P = g["P"]
    got = [oracle.work(oracle.rank_chunks(P, r, "contiguous2")) for r in range(P)]
    assert got == g["contiguous"]
    assert [oracle.work(oracle.rank_chunks(P, r, "zigzag")) for r in range(P)] == g["zigzag"]


def pin_zigzag_balance(P):
    """Largest deviation from the page's equal-work claim, per rank and per step."""
    tot = [oracle.work(oracle.rank_chunks(P, r, "zigzag")) for r in range(P)]
    dev = max(abs(t - 2 * P) for t in tot)
    steps = oracle.per_step_work(P, "zigzag")
    dev = max(dev, max(abs(w - 2.0) for row in steps for w in row))
    # the ring's per-step work adds up to work() for every rank
    for r in range(P):
        dev = max(dev, abs(sum(steps[t][r] for t in range(P)) - tot[r]))
    return dev


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
def test_zigzag_equal_work(P):
    assert pin_zigzag_balance(P) == 0


def test_contiguous_work_matches_ring():
    for P in (2, 4, 8):
        steps = oracle.per_step_work(P, "contiguous")
        for r in range(P):
            # in units of (S/P)^2 blocks: r full blocks + one half diagonal
            assert sum(steps[t][r] for t in range(P)) == r + 0.5


def test_schedule_shapes():
    """Every (rank, step) evaluates at most 2 query chunks, each against at most
    2 KV chunks, in ascending order; every causal pair appears exactly once."""
    for P in (1, 2, 4, 8):
        seen = set()
        for step in oracle.ring_schedule(P, "zigzag"):
            for e in step:
                assert len(e["pairs"]) <= 2
                for qc, ks in e["pairs"]:
                    assert 1 <= len(ks) <= 2 and ks == sorted(ks)
                    for kc in ks:
                        assert (qc, kc) not in seen
                        seen.add((qc, kc))
        assert seen == {(a, b) for a in range(2 * P) for b in range(2 * P) if b <= a}


# ---------------------------------------------------------------- Ulysses
def pin_permute():
    S, H, D, P = 12, 8, 3, 4
    x = _rand((S, H, D), 13)
    y = oracle.seq_to_head(x, P)
    # library route: reshape/transpose view of the same permutation
    y2 = x.reshape(S, P, H // P, D).transpose(1, 0, 2, 3)
    err = np.max(np.abs(y - y2))
    err = max(err, np.max(np.abs(oracle.head_to_seq(y) - x)))
    return err


def test_permute():
    assert pin_permute() == 0


def pin_ulysses():
    worst = 0.0
    for P, (S, H, Hkv, D) in [(2, (16, 4, 2, 8)), (4, (24, 8, 4, 4)), (4, (16, 16, 4, 8))]:
        q = _rand((S, H, D), 100 + P)
        k = _rand((S, Hkv, D), 110 + P)
        v = _rand((S, Hkv, D), 120 + P)
        uo, ul = oracle.ulysses_forward(q, k, v, P)
        mo, ml = oracle.attention(q, k, v, causal=True)
        worst = max(worst, np.max(np.abs(uo - mo)), np.max(np.abs(ul - ml)))
    return worst


def test_ulysses_equals_monolithic():
    assert pin_ulysses() < 1e-12


def test_ulysses_degree_bound():
    """Degree above the KV head count that replication cannot serve (P not a
    multiple of Hkv) is rejected."""
    q = _rand((8, 12, 4), 1)
    k = _rand((8, 3, 4), 2)
    with pytest.raises(ValueError):
        oracle.ulysses_forward(q, k, k, 4)


# ---------------------------------------------------------------- page toy
def _page_toy(S=32, H=8, D=16):
    from context_causal_attention_attn_gb300.inputs import make_qkv
    return make_qkv(S, H, D)


def test_page_toy_ring_and_ulysses():
    """The page's own check: ring (P=4) and Ulysses (P=4) on make_qkv() agree
    with single-process causal attention (atol 1e-5 on the page; here 1e-12)."""
    q, k, v = (t.numpy() for t in _page_toy())
    mo, ml = oracle.attention(q, k, v)
    for layout in ("contiguous", "zigzag"):
        ro, rl, _ = oracle.ring_forward(q, k, v, 4, layout)
        assert np.max(np.abs(ro - mo)) < 1e-12 and np.max(np.abs(rl - ml)) < 1e-12
    uo, _ = oracle.ulysses_forward(q, k, v, 4)
    assert np.max(np.abs(uo - mo)) < 1e-12
    assert np.all(np.isfinite(mo)) and np.all(np.isfinite(ml))


def test_page_toy_recipe():
    """make_qkv follows the page's recipe: the global-generator draw after
    torch.manual_seed(0), q then k then v."""
    torch.manual_seed(0)
    a = [torch.randn(32, 8, 16) for _ in range(3)]
    b = _page_toy()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# ---------------------------------------------------------- planted mistakes
def _caught(*pins):
    for pin in pins:
        try:
            err = pin()
        except Exception:
            return True
        if not (err < 1e-9):
            return True
    return False


ALL_PINS = (pin_brute_force, pin_sdpa, pin_closed_forms, pin_sampled_rows, pin_merge_identity,
            pin_ring_equals_monolithic, pin_ulysses, pin_permute)


def test_pins_pass_unplanted():
    assert not _caught(*ALL_PINS)


def test_planted_strict_mask(monkeypatch):
    monkeypatch.setattr(oatt, "causal_visible",
                        lambda qp, kp: np.asarray(kp)[None, :] < np.asarray(qp)[:, None])
    assert _caught(pin_brute_force, pin_sdpa, pin_closed_forms)


def test_planted_future_key(monkeypatch):
    """Mask off by one the other way: each query also sees the next key."""
    real = oatt.causal_visible
    monkeypatch.setattr(oatt, "causal_visible", lambda qp, kp: real(np.asarray(qp) + 1, kp))
    assert _caught(pin_brute_force, pin_sdpa, pin_closed_forms)


def test_planted_gqa_modulo(monkeypatch):
    monkeypatch.setattr(oatt, "kv_head_of", lambda h, H, Hkv: h % Hkv)
    assert _caught(pin_brute_force, pin_sdpa)


def test_planted_merge_weights_swapped(monkeypatch):
    real = oatt.merge_weights

    def swapped(a, b):
        lse, wa, wb = real(a, b)
        return lse, wb, wa
    monkeypatch.setattr(oatt, "merge_weights", swapped)
    assert _caught(pin_merge_identity, pin_ring_equals_monolithic)


def test_planted_merge_dropped_log1p(monkeypatch):
    def wrong(a, b):
        lse = np.maximum(a, b)  # max instead of logaddexp
        return lse, np.exp(a - lse), np.exp(b - lse)
    monkeypatch.setattr(oatt, "merge_weights", wrong)
    assert _caught(pin_merge_identity)


def test_planted_zigzag_layout(monkeypatch):
    real = oring.rank_chunks

    def wrong(P, r, layout):
        if layout == "zigzag":
            return [r, (2 * P - 2 - r) % (2 * P)]
        return real(P, r, layout)
    monkeypatch.setattr(oring, "rank_chunks", wrong)
    assert _caught(pin_ring_equals_monolithic, lambda: pin_zigzag_balance(4))


def test_planted_ring_direction(monkeypatch):
    """Receiving from rank+1 instead of rank-1 breaks the causal skip rule's
    coverage: some pair is never evaluated."""
    real = oring.ring_schedule

    def wrong(P, layout):
        s = real(P, layout)
        for t, step in enumerate(s):
            for r, e in enumerate(step):
                src = (r + t) % P
                e["src"] = src
                held = oring.rank_chunks(P, src, layout)
                e["pairs"] = [(qc, sorted(kc for kc in held if kc <= qc))
                              for qc in oring.rank_chunks(P, r, layout)]
                e["pairs"] = [(qc, ks) for qc, ks in e["pairs"] if ks]
        return s
    monkeypatch.setattr(oring, "ring_schedule", wrong)
    # the same set of blocks is still covered (direction does not matter for
    # the result) -- the pin must NOT flag it: the page's result is unique.
    assert not _caught(pin_ring_equals_monolithic)


def test_planted_permute_transposed(monkeypatch):
    import oracle.ulysses as oul

    def wrong(x, P):
        x = np.asarray(x)
        S, H, D = x.shape
        return x.reshape(S, H // P, P, D).transpose(2, 0, 1, 3).copy()
    monkeypatch.setattr(oul, "seq_to_head", wrong)
    monkeypatch.setattr(oracle, "seq_to_head", wrong)
    assert _caught(pin_permute, pin_ulysses)


def test_planted_missing_scale(monkeypatch):
    real = oatt.attention

    def noscale(q, k, v, causal=True, q_offset=0, k_offset=0, scale=None, **kw):
        return real(q, k, v, causal, q_offset, k_offset, scale=1.0, **kw)
    monkeypatch.setattr(oracle, "attention", noscale)
    assert _caught(pin_brute_force, pin_sdpa)


# ------------------------------------------ striped layout, padding, replicated KV
def pin_striped():
    worst = 0.0
    for P in (1, 2, 3, 4):
        S = 4 * P * 3
        q, k, v = _rand((S, 4, 8), 200 + P), _rand((S, 2, 8), 210 + P), _rand((S, 2, 8), 220 + P)
        so, sl, counts = oracle.ring_forward(q, k, v, P, "striped")
        mo, ml = oracle.attention(q, k, v, causal=True)
        worst = max(worst, np.max(np.abs(so - mo)), np.max(np.abs(sl - ml)))
        if counts != [P] * P:
            return np.inf
    return worst


def test_striped_equals_monolithic():
    assert pin_striped() < 1e-12


def test_striped_balance():
    """Striped shards give every rank nearly the same number of visible
    (query, key) pairs at every step: at most one stripe length apart."""
    for P in (2, 4, 8):
        S = 64 * P
        C = S // P
        held = list(range(P))
        for t in range(P):
            counts = []
            for r in range(P):
                qt = oracle.striped_tokens(S, P, r)
                kt = oracle.striped_tokens(S, P, held[r])
                counts.append(int(np.sum(oracle.causal_visible(qt, kt))))
            assert max(counts) - min(counts) <= C
            held = [held[(r - 1) % P] for r in range(P)]


def pin_padded_ring():
    """[CP-practice] 7.1: a sequence the chunk count does not divide is padded
    at the end, run, and cut back; the real rows equal monolithic attention."""
    worst = 0.0
    for layout in ("contiguous", "zigzag"):
        for P, S in ((2, 13), (3, 20), (4, 37), (4, 5)):
            q = _rand((S, 4, 8), 300 + S)
            k = _rand((S, 2, 8), 310 + S)
            v = _rand((S, 2, 8), 320 + S)
            ro, rl, _ = oracle.ring_forward(q, k, v, P, layout)
            mo, ml = oracle.attention(q, k, v, causal=True)
            worst = max(worst, np.max(np.abs(ro - mo)), np.max(np.abs(rl - ml)))
    return worst


def test_padded_ring_equals_monolithic():
    assert pin_padded_ring() < 1e-12


def pin_ulysses_replicated():
    """Degree above the KV head count with each KV head copied to P/Hkv
    ranks ([CP-handbook] exercises, 16-way on 8 KV heads) = monolithic."""
    worst = 0.0
    for P, (S, H, Hkv) in ((4, (16, 8, 2)), (8, (24, 16, 4)), (16, (32, 32, 8))):
        q = _rand((S, H, 8), 400 + P)
        k = _rand((S, Hkv, 8), 410 + P)
        v = _rand((S, Hkv, 8), 420 + P)
        uo, ul = oracle.ulysses_forward(q, k, v, P)
        mo, ml = oracle.attention(q, k, v, causal=True)
        worst = max(worst, np.max(np.abs(uo - mo)), np.max(np.abs(ul - ml)))
    return worst


def test_ulysses_replicated_equals_monolithic():
    assert pin_ulysses_replicated() < 1e-12


def test_replicate_kv_layout():
    k = _rand((5, 2, 3), 9)
    r = oracle.replicate_kv(k, 8)
    for p in range(8):
        assert np.array_equal(r[:, p], k[:, p // 4])


def test_planted_striped_shift(monkeypatch):
    """A stripe that drops its last token leaves rows uncomputed."""
    real = oring.striped_tokens
    monkeypatch.setattr(oring, "striped_tokens", lambda S, P, r: real(S, P, r)[:-1])
    assert _caught(pin_striped)


def pin_usp():
    """Ulysses x Ring (USP) = monolithic, for every ring layout and with
    replicated KV heads."""
    worst = 0.0
    cases = ((2, 2, "zigzag", (16, 4, 2)), (2, 3, "contiguous", (18, 8, 4)),
             (4, 2, "striped", (16, 8, 2)), (2, 4, "zigzag", (22, 4, 2)))
    for Pu, Pr, layout, (S, H, Hkv) in cases:
        q = _rand((S, H, 8), 500 + S)
        k = _rand((S, Hkv, 8), 510 + S)
        v = _rand((S, Hkv, 8), 520 + S)
        uo, ul = oracle.usp_forward(q, k, v, Pu, Pr, layout)
        mo, ml = oracle.attention(q, k, v, causal=True)
        worst = max(worst, np.max(np.abs(uo - mo)), np.max(np.abs(ul - ml)))
    return worst


def test_usp_equals_monolithic():
    assert pin_usp() < 1e-12


# ------------------------------------------------------------------ backward
def _torch_grads(q, k, v, dout, causal):
    """Library route: autograd of torch SDPA in float64."""
    def t(a):
        x = torch.from_numpy(np.ascontiguousarray(a)).double()
        return x.permute(1, 0, 2)[None].requires_grad_(True)
    tq, tk, tv = t(q), t(k), t(v)
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, is_causal=causal, enable_gqa=(q.shape[1] != k.shape[1]))
    o.backward(torch.from_numpy(np.ascontiguousarray(dout)).double().permute(1, 0, 2)[None])
    g = lambda x: x.grad[0].permute(1, 0, 2).numpy()
    return g(tq), g(tk), g(tv)


def pin_backward_sdpa():
    worst = 0.0
    for n, (S, H, Hkv, D, causal) in enumerate([(17, 4, 4, 8, True), (24, 8, 2, 16, True),
                                                (13, 6, 3, 4, False)]):
        q = _rand((S, H, D), 600 + n)
        k = _rand((S, Hkv, D), 610 + n)
        v = _rand((S, Hkv, D), 620 + n)
        do = _rand((S, H, D), 630 + n)
        o, l = oracle.attention(q, k, v, causal=causal)
        got = oracle.attention_backward(q, k, v, o, l, do, causal=causal)
        want = _torch_grads(q, k, v, do, causal)
        worst = max(worst, *(np.max(np.abs(a - b)) for a, b in zip(got, want)))
    return worst


def test_backward_library_autograd():
    assert pin_backward_sdpa() < 1e-10


def test_backward_finite_differences():
    """Directional derivative of sum(out * dout) by central differences."""
    S, H, Hkv, D = 7, 2, 1, 4
    q, k, v = _rand((S, H, D), 640), _rand((S, Hkv, D), 641), _rand((S, Hkv, D), 642)
    do = _rand((S, H, D), 643)
    o, l = oracle.attention(q, k, v, q_offset=2, k_offset=1)
    dq, dk, dv = oracle.attention_backward(q, k, v, o, l, do, q_offset=2, k_offset=1)
    f = lambda qq, kk, vv: np.sum(oracle.attention(qq, kk, vv, q_offset=2, k_offset=1)[0] * do)
    eps = 1e-6
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        dirn = _rand(x.shape, 650 + which)
        args_p = [q, k, v]
        args_m = [q, k, v]
        args_p[which] = x + eps * dirn
        args_m[which] = x - eps * dirn
        fd = (f(*args_p) - f(*args_m)) / (2 * eps)
        assert abs(fd - np.sum(g * dirn)) < 1e-6 * max(1.0, abs(fd))


def pin_ring_backward():
    worst = 0.0
    for layout in ("contiguous", "zigzag", "striped"):
        for P in (1, 2, 3):
            S = 4 * P * 3
            q = _rand((S, 4, 8), 700 + P)
            k = _rand((S, 2, 8), 710 + P)
            v = _rand((S, 2, 8), 720 + P)
            do = _rand((S, 4, 8), 730 + P)
            o, l = oracle.attention(q, k, v)
            got = oracle.ring_backward(q, k, v, o, l, do, P, layout)
            want = oracle.attention_backward(q, k, v, o, l, do)
            worst = max(worst, *(np.max(np.abs(a - b)) for a, b in zip(got, want)))
    return worst


def test_ring_backward_equals_monolithic():
    assert pin_ring_backward() < 1e-12


def test_planted_backward_block_lse(monkeypatch):
    """Using each block's own lse instead of the whole row's breaks the ring
    backward (blocks no longer add up)."""
    import oracle.backward as obw
    real = obw.attention_backward

    def wrong(q, k, v, out, lse, dout, causal=True, q_offset=0, k_offset=0, scale=None,
              q_positions=None, k_positions=None):
        _, l_blk = oracle.attention(q, k, v, causal=causal, q_offset=q_offset, k_offset=k_offset,
                                    q_positions=q_positions, k_positions=k_positions)
        return real(q, k, v, out, l_blk, dout, causal, q_offset, k_offset, scale,
                    q_positions, k_positions)
    monkeypatch.setattr(obw, "attention_backward", wrong)
    assert _caught(pin_ring_backward)
