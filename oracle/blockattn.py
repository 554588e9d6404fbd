"""Block attention with global offsets and per-row LSE, and the LSE merge.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Definition followed ([CP-handbook], section "哪些运算可以直接切", the
``attention`` helper):

    scores[h, i, j] = q[i, h, :] . k[j, h, :] / sqrt(D)
    scores[h, i, j] = -inf   where  (j + k_offset) > (i + q_offset)   (causal)
    lse[h, i]       = log sum_j exp(scores[h, i, j])                  [H, Sq]
    out[i, h, :]    = sum_j exp(scores[h, i, j] - lse[h, i]) v[j, h, :]

Readings where the page is silent:

* GQA: the page's helper needs equal head counts.  Query head h reads KV head
  h // (H // Hkv) (contiguous groups of H/Hkv query heads share a KV head).
* A row with no visible key: lse = -inf and out = 0 (the page's expression
  would give NaN; its ring never evaluates such a row).  -inf is the identity
  of the merge, so this keeps merge(empty, x) = x.
* Scale: 1/sqrt(D) unless a positive scale is given.

Everything is computed in float64; inputs of any float dtype are upcast
exactly (bf16 and fp32 values are representable in fp64).
"""

import numpy as np

NEG_INF = -np.inf


def causal_visible(q_pos, k_pos):
    """Boolean [len(q_pos), len(k_pos)]: key visible to query iff k <= q.

    [CP-handbook] section "哪些运算可以直接切": positions are local index plus
    the block's global offset; entries with key position greater than query
    position are masked, so the diagonal is kept.
    """
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    return k_pos[None, :] <= q_pos[:, None]


def kv_head_of(h, H, Hkv):
    """KV head read by query head h under GQA (contiguous groups).

    Reading of [CP-handbook] section "练习" (32 query / 8 KV heads, degree
    bounded by the KV head count): each KV head serves H/Hkv consecutive
    query heads.
    """
    if H % Hkv != 0:
        raise ValueError("H must be a multiple of Hkv")
    return h // (H // Hkv)


def _row_lse_and_weights(s):
    """lse and softmax weights of each row of s (float64, -inf = masked).

    lse = m + log(sum exp(s - m)) with m the row max; rows whose entries are
    all -inf give lse = -inf and all-zero weights.  Non-finite scores follow
    the page's logsumexp / exp(s - lse): a NaN score makes the row NaN; a
    +inf score makes lse +inf and the weights exp(inf - inf) = NaN.
    """
    m = np.max(s, axis=1) if s.shape[1] > 0 else np.full(s.shape[0], NEG_INF)
    empty = m == NEG_INF
    pinf = m == np.inf
    m_safe = np.where(empty | pinf, 0.0, m)
    with np.errstate(invalid="ignore", over="ignore"):
        e = np.exp(s - m_safe[:, None])
        tot = np.sum(e, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(empty, NEG_INF, m_safe + np.log(np.where(empty, 1.0, tot)))
        lse = np.where(pinf, np.inf, lse)
        w = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, tot)[:, None])
    w = np.where(pinf[:, None], np.nan, w)
    return lse, w


def attention(q, k, v, causal=True, q_offset=0, k_offset=0, scale=None,
              q_positions=None, row_block=1024, k_positions=None):
    """Block attention of q [Sq,H,D] against k/v [Sk,Hkv,D] with offsets.

    Returns (out [Sq,H,D] float64, lse [H,Sq] float64).

    ``q_positions`` (optional, int array of length Sq) overrides the query
    positions ``q_offset + arange(Sq)``; it lets a caller evaluate an
    arbitrary subset of rows of a longer block (sampled parity checks).
    ``k_positions`` likewise overrides ``k_offset + arange(Sk)`` (strided
    token sets, e.g. a striped layout's shards).
    Rows are processed ``row_block`` at a time to bound memory; for a causal
    block only keys that some row of the block can see are read.
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    Sq, H, D = q.shape
    Sk, Hkv, Dk = k.shape
    if Dk != D or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k, v")
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(D)
    if q_positions is None:
        q_pos = q_offset + np.arange(Sq, dtype=np.int64)
    else:
        q_pos = np.asarray(q_positions, dtype=np.int64)
    if k_positions is None:
        k_pos = k_offset + np.arange(Sk, dtype=np.int64)
    else:
        k_pos = np.asarray(k_positions, dtype=np.int64)

    out = np.zeros((Sq, H, D), dtype=np.float64)
    lse = np.full((H, Sq), NEG_INF, dtype=np.float64)
    if Sq == 0:
        return out, lse
    for hk in range(Hkv):
        k64 = k[:, hk, :].astype(np.float64)
        v64 = v[:, hk, :].astype(np.float64)
        heads = [h for h in range(H) if kv_head_of(h, H, Hkv) == hk]
        for i0 in range(0, Sq, row_block):
            i1 = min(Sq, i0 + row_block)
            qp = q_pos[i0:i1]
            # keys that any row of this block can see (all keys if not causal)
            n_keys = Sk
            if causal and k_positions is None:
                n_keys = int(np.clip(np.max(qp) - k_offset + 1, 0, Sk))
            kb, vb = k64[:n_keys], v64[:n_keys]
            vis = causal_visible(qp, k_pos[:n_keys]) if causal else None
            for h in heads:
                s = (q[i0:i1, h, :].astype(np.float64) @ kb.T) * scale
                if causal:
                    s = np.where(vis, s, NEG_INF)
                l_blk, w = _row_lse_and_weights(s)
                lse[h, i0:i1] = l_blk
                out[i0:i1, h, :] = w @ vb
    return out, lse


def attention_monolithic(q, k, v, scale=None, rows=None):
    """Plain causal attention of the full sequence (offsets 0, Sq = Sk = S).

    ``rows`` optionally restricts the evaluation to a subset of query rows;
    the result then has one entry per requested row (out [R,H,D], lse [H,R]).
    """
    if rows is None:
        return attention(q, k, v, causal=True, scale=scale)
    rows = np.asarray(rows, dtype=np.int64)
    return attention(np.asarray(q)[rows], k, v, causal=True, scale=scale,
                     q_positions=rows)


def merge_weights(lse_a, lse_b):
    """(lse, w_a, w_b) of the LSE merge, with -inf handled.

    [CP-handbook] self-test answers and section "Ring Attention：KV 沿环传一圈":
    lse = log(e^lse_a + e^lse_b); w_a = e^(lse_a - lse); w_b = e^(lse_b - lse).
    Both -inf: lse = -inf and both weights 0 (the merge of two empty blocks
    is empty).  Computed as max + log1p(exp(-|a-b|)) to stay finite.
    """
    a = np.asarray(lse_a, dtype=np.float64)
    b = np.asarray(lse_b, dtype=np.float64)
    hi = np.maximum(a, b)
    both_empty = ~np.isfinite(hi)
    hi_safe = np.where(both_empty, 0.0, hi)
    with np.errstate(invalid="ignore"):
        diff = np.where(both_empty, 0.0, np.abs(a - b))
    diff = np.where(np.isnan(diff), np.inf, diff)
    lse = np.where(both_empty, NEG_INF, hi_safe + np.log1p(np.exp(-diff)))
    lse_safe = np.where(both_empty, 0.0, lse)
    w_a = np.where(both_empty, 0.0, np.exp(a - lse_safe))
    w_b = np.where(both_empty, 0.0, np.exp(b - lse_safe))
    return lse, w_a, w_b


def lse_merge(out_a, lse_a, out_b, lse_b):
    """Merge two partial attentions of the same query rows.

    out_* [Sq,H,D] (normalised block outputs), lse_* [H,Sq].
    Returns (out, lse) with out = out_a w_a + out_b w_b, weights broadcast from
    the transposed [Sq,H] view of lse exactly as the page's ring loop does.
    """
    lse, w_a, w_b = merge_weights(lse_a, lse_b)
    out = (np.asarray(out_a, dtype=np.float64) * w_a.T[..., None]
           + np.asarray(out_b, dtype=np.float64) * w_b.T[..., None])
    return out, lse
