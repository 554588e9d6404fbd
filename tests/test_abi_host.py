"""CPU-only checks of the C ABI: the library loads, exports every function the
header declares, and its host logic (argument validation, the ring
schedule) behaves as specified.  Nothing here launches a kernel."""

import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpattn.h")


@pytest.fixture(scope="module")
def cp():
    from context_causal_attention_attn_gb300 import build
    build.build()
    import context_causal_attention_attn_gb300 as m
    m.lib()
    return m


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int64_t|int)\s+(cp_\w+)\s*\(", text,
                                 re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("cp_attn_block", "cp_lse_merge", "cp_ring_forward", "cp_seq_to_head",
                 "cp_head_to_seq"):
        assert must in names


def test_library_exports_every_declared_symbol(cp):
    lib = ctypes.CDLL(cp.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version(cp):
    assert "sm_103a" in cp.cp_version()


def test_release_build_is_not_bounds_checked(cp):
    from context_causal_attention_attn_gb300 import build
    assert ctypes.CDLL(build.LIB).cp_debug_bounds() == 0


def test_bounds_checked_build_exports_every_declared_symbol():
    """The bounds-checked variant (sources compiled with CP_DEBUG_BOUNDS)
    compiles, links, exports the same boundary and reports that it checks."""
    from context_causal_attention_attn_gb300 import build
    path = build.build(debug=True)
    assert path == build.LIB_DEBUG != build.LIB
    lib = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert lib.cp_debug_bounds() == 1


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 16])
def test_ring_schedule_matches_oracle(cp, layout, P):
    sched = oracle.ring_schedule(P, layout)
    for t in range(P):
        got = sorted(cp.cp_ring_step_blocks(P, layout, t))
        want = sorted((r, qc, kc, int(kc == qc))
                      for r, e in enumerate(sched[t]) for qc, ks in e["pairs"] for kc in ks)
        assert got == want


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_striped_schedule(cp, P):
    """Striped: every rank evaluates exactly its held stripe at every step."""
    for t in range(P):
        got = sorted(cp.cp_ring_step_blocks(P, "striped", t))
        want = sorted((r, r, (r - t) % P, int((r - t) % P == r)) for r in range(P))
        assert got == want


def test_ring_schedule_rejects_bad_args(cp):
    L = cp.lib()
    assert L.cp_ring_step_blocks(0, 0, 0, None, 0) == -1
    assert L.cp_ring_step_blocks(17, 0, 0, None, 0) == -1
    assert L.cp_ring_step_blocks(4, 3, 0, None, 0) == -1
    assert L.cp_ring_step_blocks(4, 1, 4, None, 0) == -1
    assert "step" in cp.cp_last_error()


def test_validation_codes_without_gpu(cp):
    """Every check below fails before anything touches the device."""
    L = cp.lib()
    F32, BF16 = cp.CP_F32, cp.CP_BF16
    # bf16 needs D = 128
    assert L.cp_attn_block(None, None, None, BF16, 8, 8, 4, 4, 64, 0, 0, 1, 0.0, None, BF16,
                           None, None) == -2
    # fp32 D must be one of 16/32/64/128
    assert L.cp_attn_block(None, None, None, F32, 8, 8, 4, 4, 24, 0, 0, 1, 0.0, None, F32,
                           None, None) == -2
    # H % Hkv
    assert L.cp_attn_block(None, None, None, F32, 8, 8, 6, 4, 16, 0, 0, 1, 0.0, None, F32,
                           None, None) == -2
    # dtype
    assert L.cp_attn_block(None, None, None, 7, 8, 8, 4, 4, 16, 0, 0, 1, 0.0, None, F32,
                           None, None) == -3
    # null pointers with work to do
    assert L.cp_attn_block(None, None, None, F32, 8, 8, 4, 4, 16, 0, 0, 1, 0.0, None, F32,
                           None, None) == -1
    # Sq = 0 is a no-op even with null pointers
    assert L.cp_attn_block(None, None, None, F32, 0, 8, 4, 4, 16, 0, 0, 1, 0.0, None, F32,
                           None, None) == 0
    # misaligned pointer
    assert L.cp_attn_block(8, 16, 16, F32, 8, 8, 4, 4, 16, 0, 0, 1, 0.0, 16, F32, 16,
                           None) == -4
    # ring: striped with S not divisible by P, P out of range, bad layout,
    # bf16 out w/o workspace
    assert L.cp_ring_forward(16, 16, 16, BF16, 100, 4, 4, 128, 8, 2, 16, BF16, 16, None,
                             None) == -2
    assert L.cp_ring_forward(16, 16, 16, BF16, 128, 4, 4, 128, 17, 1, 16, BF16, 16, None,
                             None) == -1
    assert L.cp_ring_forward(16, 16, 16, BF16, 128, 4, 4, 128, 4, 5, 16, BF16, 16, None,
                             None) == -1
    # Ulysses: degree neither dividing nor a multiple of the KV head count
    assert L.cp_ulysses_forward(16, 16, 16, BF16, 64, 24, 3, 128, 4, 16, BF16, 16, 16,
                                None) == -2
    assert L.cp_ring_step(16, 16, 16, BF16, 128, 4, 4, 128, 4, 1, 0, 16, BF16, 16, None,
                          None) == -1
    assert "workspace" in cp.cp_last_error()
    # merge: D/4 must be a power of two (or a multiple of 32)
    assert L.cp_lse_merge(16, 16, 16, 16, 4, 2, 24, None) == -2
    # permute: H % P
    assert L.cp_seq_to_head(16, 16, F32, 8, 6, 4, 4, None) == -2
    # host-buffer ring: groups must divide Hkv; the ring's own checks; a
    # missing workspace; a misaligned workspace
    assert L.cp_ring_forward_host(16, 16, 16, BF16, 128, 8, 4, 128, 4, 1, 16, BF16, 16, 3, 16,
                                  None, None) == -2
    assert L.cp_ring_forward_host(16, 16, 16, BF16, 100, 8, 4, 128, 8, 2, 16, BF16, 16, 2, 16,
                                  None, None) == -2
    assert L.cp_ring_forward_host(16, 16, 16, BF16, 128, 8, 4, 128, 4, 1, 16, BF16, 16, 2,
                                  None, None, None) == -1
    assert L.cp_ring_forward_host(16, 16, 16, BF16, 128, 8, 4, 128, 4, 1, 16, BF16, 16, 2, 8,
                                  None, None) == -4
    assert L.cp_ring_host_workspace_size(128, 8, 4, 128, 0, BF16, BF16) == -2
    # host-buffer ring backward: groups must divide Hkv, null pointers,
    # misaligned workspace
    assert L.cp_ring_backward_host(16, 16, 16, 16, 16, 16, BF16, 128, 8, 4, 128, 4, 1, 16, 16,
                                   16, BF16, 3, 16, None, None) == -2
    assert L.cp_ring_backward_host(16, 16, 16, 16, 16, 16, BF16, 128, 8, 4, 128, 4, 1, 16, 16,
                                   16, BF16, 2, None, None, None) == -1
    assert L.cp_ring_backward_host(16, 16, 16, 16, 16, 16, BF16, 128, 8, 4, 128, 4, 1, 16, 16,
                                   16, BF16, 2, 8, None, None) == -4
    # host-buffer Ulysses: degree neither dividing nor a multiple of Hkv;
    # missing workspace
    assert L.cp_ulysses_forward_host(16, 16, 16, BF16, 64, 24, 3, 128, 4, 16, BF16, 16, 16,
                                     None, None) == -2
    assert L.cp_ulysses_forward_host(16, 16, 16, BF16, 64, 8, 4, 128, 4, 16, BF16, 16, None,
                                     None, None) == -1
    assert L.cp_ulysses_host_workspace_size(64, 24, 3, 128, 4, BF16, BF16) == -2
    assert L.cp_usp_forward_host(16, 16, 16, BF16, 64, 8, 4, 128, 2, 0, 1, 16, BF16, 16, 16,
                                 None, None) == -1
    assert L.cp_usp_host_workspace_size(64, 24, 3, 128, 4, BF16, BF16) == -2
    # staged Ulysses / USP: stage out of range
    assert L.cp_ulysses_stage(16, 16, 16, BF16, 64, 8, 4, 128, 4, 16, BF16, 16, 16, 3,
                              None) == -1
    assert L.cp_usp_stage(16, 16, 16, BF16, 64, 8, 4, 128, 2, 2, 1, 16, BF16, 16, 16, 4,
                          None) == -1
    assert L.cp_usp_stage(16, 16, 16, BF16, 64, 8, 4, 128, 2, 2, 1, 16, BF16, 16, 16, -1,
                          None) == -1



def test_backward_validation_codes_without_gpu(cp):
    """The backward entry points reject bad arguments before any device work."""
    L = cp.lib()
    F32, BF16 = cp.CP_F32, cp.CP_BF16
    # block: fp32 inputs with an unsupported D, bf16 with D != 128, H % Hkv,
    # unknown gradient dtype, null pointers, misaligned pointer
    args = lambda in_dt, D, H, Hkv, grad, ptr, ws: (ptr, ptr, ptr, ptr, ptr, ptr, in_dt, 8, 8, H,
                                                  Hkv, D, 0, 0, 1, 0.0, ptr, ptr, ptr, grad, ws,
                                                  None)
    assert L.cp_attn_block_backward(*args(F32, 24, 4, 4, F32, None, None)) == -2
    assert L.cp_attn_block_backward(*args(F32, 16, 4, 4, F32, None, None)) == -1
    assert L.cp_attn_block_backward(*args(BF16, 64, 4, 4, F32, None, None)) == -2
    assert L.cp_attn_block_backward(*args(BF16, 128, 6, 4, F32, None, None)) == -2
    assert L.cp_attn_block_backward(*args(BF16, 128, 4, 4, 9, None, None)) == -3
    assert L.cp_attn_block_backward(*args(BF16, 128, 4, 4, F32, None, None)) == -1
    assert L.cp_attn_block_backward(*args(BF16, 128, 4, 4, F32, 24, 32)) == -4
    # ring: layout, P, striped divisibility, missing workspace
    ring = lambda S, P, layout, ws: (16, 16, 16, 16, 16, 16, BF16, S, 4, 4, 128, P, layout, 16,
                                     16, 16, BF16, ws, None)
    assert L.cp_ring_backward(*ring(128, 4, 5, 16)) == -1
    assert L.cp_ring_backward(*ring(128, 17, 1, 16)) == -1
    assert L.cp_ring_backward(*ring(100, 8, 2, 16)) == -2
    assert L.cp_ring_backward(*ring(128, 4, 1, None)) == -1


def test_backward_workspace_sizes(cp):
    import torch
    assert cp.cp_attn_block_backward_workspace_size(1024, 4) == 16384
    assert cp.cp_attn_block_backward_workspace_size(1001, 4) == 16128  # 256-byte rounding
    S, H, Hkv, D = 4096, 32, 8, 128
    assert cp.cp_ring_backward_workspace_size(S, H, Hkv, D, torch.float32) == S * H * 4
    assert cp.cp_ring_backward_workspace_size(S, H, Hkv, D, torch.bfloat16) == (
        S * H * 4 + S * H * D * 4 + 2 * S * Hkv * D * 4)


def test_workspace_sizes(cp):
    import torch
    assert cp.cp_ring_workspace_size(4096, 32, 128, torch.float32) == 0
    assert cp.cp_ring_workspace_size(4096, 32, 128, torch.bfloat16) == 4096 * 32 * 128 * 4
    n = cp.cp_ulysses_workspace_size(1024, 32, 8, 128, torch.bfloat16, torch.bfloat16)
    assert n >= 1024 * (32 + 8 + 8 + 32) * 128 * 2
    # host-buffer ring staging: q, k, v, out, lse of all heads + one group's
    # fp32 accumulator (bf16 out only)
    S, H, Hkv, D = 1024, 32, 8, 128
    staged = S * (H + 2 * Hkv) * D * 2 + S * H * D * 2 + S * H * 4
    assert cp.cp_ring_host_workspace_size(S, H, Hkv, D, 4, torch.bfloat16,
                                          torch.bfloat16) == staged + S * (H // 4) * D * 4
    assert cp.cp_ring_host_workspace_size(S, H, Hkv, D, 2, torch.bfloat16, torch.float32) == (
        S * (H + 2 * Hkv) * D * 2 + S * H * D * 4 + S * H * 4)
    # backward: staged q, k, v, out, dout, lse and gradients, plus one group's
    # ring backward workspace (delta and fp32 accumulators)
    G = 4
    assert cp.cp_ring_backward_host_workspace_size(S, H, Hkv, D, G, torch.bfloat16,
                                                   torch.bfloat16) == (
        S * (3 * H + 2 * Hkv) * D * 2 + S * H * 4 + S * (H + 2 * Hkv) * D * 2 +
        cp.cp_ring_backward_workspace_size(S, H // G, Hkv // G, D, torch.bfloat16))


def test_product_does_not_import_oracle():
    """The library package and its build never reference the oracle."""
    pkg = os.path.join(ROOT, "context_causal_attention_attn_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_header_constants_match_the_binding(cp):
    text = open(HEADER).read()
    for name in ("CP_MAX_RANKS",):
        m = re.search(r"#define\s+" + name + r"\s+(\d+)", text)
        assert m and int(m.group(1)) == getattr(cp, name), name


def test_fused_ring_validation_without_gpu(cp):
    """The one-launch ring takes bf16 inputs (any layout, with the layout's
    own conditions); it rejects the rest before any device work."""
    L = cp.lib()
    F32, BF16 = cp.CP_F32, cp.CP_BF16
    ptr = ctypes.c_void_p(256)
    args = lambda in_dt, D, layout, P: (ptr, ptr, ptr, in_dt, 64, 4, 4, D, P, layout, ptr, BF16,
                                        ptr, None)
    assert L.cp_ring_forward_fused(*args(F32, 16, cp.CP_ZIGZAG, 2)) == -3
    assert "bf16" in cp.cp_last_error()
    assert L.cp_ring_forward_fused(*args(BF16, 128, cp.CP_STRIPED, 3)) == -2  # S % P != 0
    assert L.cp_ring_forward_fused(*args(BF16, 128, 7, 2)) == -1  # no such layout
    assert L.cp_ring_forward_fused(*args(BF16, 128, cp.CP_ZIGZAG, 17)) == -1
    assert L.cp_ring_forward_fused(*args(BF16, 64, cp.CP_ZIGZAG, 2)) == -2
    bad = ctypes.c_void_p(258)
    assert L.cp_ring_forward_fused(bad, ptr, ptr, BF16, 64, 4, 4, 128, 2, cp.CP_ZIGZAG, ptr,
                                   BF16, ptr, None) == -4


def test_fused_ring_backward_validation_without_gpu(cp):
    """The two-launch ring backward takes bf16 rings (any layout) and
    launches -1, 0, 1; anything else is rejected before any device work."""
    L = cp.lib()
    F32, BF16 = cp.CP_F32, cp.CP_BF16
    p = ctypes.c_void_p(256)

    def call(in_dt, D, layout, launch):
        return L.cp_ring_backward_fused_step(p, p, p, p, p, p, in_dt, 256, 4, 4, D, 2, layout,
                                             launch, p, p, p, BF16, p, None)
    assert call(F32, 16, cp.CP_ZIGZAG, 0) == -3
    assert call(BF16, 128, 9, 0) == -1  # no such layout
    assert call(BF16, 128, cp.CP_STRIPED, 2) == -1
    assert "launch" in cp.cp_last_error()
    assert call(BF16, 128, cp.CP_ZIGZAG, 2) == -1
    assert "launch" in cp.cp_last_error()
    assert call(BF16, 128, cp.CP_ZIGZAG, -2) == -1
