"""Shared helpers of the GPU parity tests (comparison against the oracle)."""

import numpy as np
import torch

# Tolerances: fp32 CUDA-core path against fp64 (absolute, every element);
# bf16 inputs with fp32 accumulation (max-abs on out, on finite LSE).
ATOL_F32 = 1e-5
ATOL_BF16_OUT = 2e-2
ATOL_BF16_LSE = 1e-3


def host(t):
    return t.detach().to("cpu", torch.float32).numpy()


def compare(out, lse, ref_out, ref_lse, atol_out, atol_lse, rows=None):
    """Compare device (out [S,H,D], lse [H,S]) with oracle values.

    rows: evaluate only these rows of the device result (the oracle was
    computed on them).  Rows the oracle marks empty (lse = -inf) must be
    exactly -inf with out = 0.  Returns (max |d out|, max |d lse|).
    """
    o = host(out)
    l = host(lse)
    if rows is not None:
        o = o[rows]
        l = l[:, rows]
    assert np.all(np.isfinite(o)), "non-finite output"
    assert not np.any(np.isnan(l)), "NaN in lse"
    empty = ~np.isfinite(ref_lse)
    assert np.array_equal(empty, ~np.isfinite(l)), (
        f"empty-row pattern differs: {np.argwhere(empty != ~np.isfinite(l))[:5]}")
    d_out = float(np.max(np.abs(o - ref_out))) if o.size else 0.0
    d_lse = float(np.max(np.abs(l[~empty] - ref_lse[~empty]), initial=0.0))
    if not (d_out <= atol_out and d_lse <= atol_lse):
        err = np.abs(o - ref_out)
        idx = np.unravel_index(np.argmax(err), err.shape)
        raise AssertionError(
            f"max|dout|={d_out:.3e} (tol {atol_out}) at {idx}: got {o[idx]:.6f} want "
            f"{ref_out[idx]:.6f}; max|dlse|={d_lse:.3e} (tol {atol_lse}); rows with "
            f"|dout|>tol: {np.unique(np.argwhere(err > atol_out)[:, 0])[:10]}")
    return d_out, d_lse


# Guard bands: results written through a view into a larger buffer whose
# head and tail hold a sentinel; a kernel that writes past either end of its
# output (a ragged tail, a striped row stride, a host copy's pitch) changes
# a sentinel, which value comparisons inside the tensor would not see.
SENTINEL = -12288.0  # exact in bf16 and fp32, far outside any result


def guarded(shape, dtype, device="cuda", guard_rows=2, pin=False):
    """A tensor of ``shape`` inside a sentinel-filled buffer with at least
    ``guard_rows`` rows (of the last dimensions) before and after it, both
    bands a multiple of 64 elements (16-byte aligned views).  Returns (view,
    intact) where intact() tells whether both bands still hold the
    sentinel."""
    n = int(np.prod(shape))
    row = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    g = -(-max(guard_rows * row, 64) // 64) * 64
    kw = {"pin_memory": True} if pin else {"device": device}
    buf = torch.full((n + 2 * g,), SENTINEL, dtype=dtype, **kw)
    view = buf[g:g + n].view(shape)

    def intact():
        return bool((buf[:g] == SENTINEL).all()) and bool((buf[g + n:] == SENTINEL).all())
    return view, intact


def ring_by_steps(cp, q, k, v, P, layout, out_dtype=None, stream=None):
    """The per-step ring (cp_ring_step for t = 0 .. P-1 on one stream): the
    bitwise reference of every entry point that runs the ring step by step
    (copy mode, host buffers, sequences longer than the one-launch limit)."""
    S, H, D = q.shape
    out_dtype = out_dtype or q.dtype
    out = torch.empty(S, H, D, dtype=out_dtype, device=q.device)
    lse = torch.empty(H, S, dtype=torch.float32, device=q.device)
    n = cp.cp_ring_workspace_size(S, H, D, out_dtype)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device) if n else None
    for t in range(P):
        cp.cp_ring_step(q, k, v, P, layout, t, out, lse, ws, stream=stream)
    return out, lse
