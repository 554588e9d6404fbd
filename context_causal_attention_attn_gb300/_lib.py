"""ctypes binding of libcpattn.so: argument marshalling only.

Every function takes torch tensors, checks dtypes / devices / contiguity,
passes raw pointers and the current CUDA stream to the C ABI of the same
name, and raises ``CpError`` on a non-zero status.  All arithmetic runs in the
library's CUDA kernels; there is no fallback: if the library is missing the
call fails.
"""

import ctypes
import os

import torch

from . import build as _build

CP_F32, CP_BF16 = 0, 1
CP_CONTIGUOUS, CP_ZIGZAG, CP_STRIPED = 0, 1, 2
CP_MAX_RANKS = 16
STATUS = {0: "CP_OK", -1: "CP_ERR_ARG", -2: "CP_ERR_SHAPE", -3: "CP_ERR_DTYPE",
          -4: "CP_ERR_ALIGN", -5: "CP_ERR_CUDA", -6: "CP_ERR_TIMEOUT", -7: "CP_ERR_BOUNDS"}
CP_ERR_TIMEOUT = -6
CP_ERR_BOUNDS = -7

_LIB = None


class CpError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


def debug_requested():
    """CPATTN_DEBUG=1 selects the bounds-checked library."""
    return os.environ.get("CPATTN_DEBUG", "0") not in ("", "0")


def library_path():
    return _build.lib_path(debug_requested())


def lib():
    """Load libcpattn.so (built in-tree by ``build.build()``), or with
    CPATTN_DEBUG=1 the bounds-checked libcpattn_debug.so
    (``build.build(debug=True)``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "context_causal_attention_attn_gb300.build.build(" +
                           ("debug=True)" if debug_requested() else ")"))
    L = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    sig = {
        "cp_attn_block": (i32, [vp, vp, vp, i32, i64, i64, i32, i32, i32, i64, i64, i32, f32,
                                vp, i32, vp, vp]),
        "cp_lse_merge": (i32, [vp, vp, vp, vp, i64, i32, i32, vp]),
        "cp_ring_workspace_size": (i64, [i64, i32, i32, i32]),
        "cp_ring_forward": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, vp, i32, vp,
                                  vp, vp]),
        "cp_ring_forward_noalloc": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, vp,
                                          i32, vp, vp]),
        "cp_ring_forward_fused": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, vp, i32,
                                        vp, vp]),
        "cp_ring_forward_steps": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, vp, i32,
                                        vp, vp, vp]),
        "cp_ring_copy_workspace_size": (i64, [i64, i32, i32, i32, i32, i32, i32, i32]),
        "cp_ring_forward_copy": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, vp, i32,
                                       vp, vp, vp, vp]),
        "cp_ring_step": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, i32, vp, i32, vp,
                               vp, vp]),
        "cp_ring_host_workspace_size": (i64, [i64, i32, i32, i32, i32, i32, i32]),
        "cp_ring_forward_host": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, vp, i32,
                                       vp, i32, vp, vp, vp]),
        "cp_ring_step_blocks": (i32, [i32, i32, i32, ctypes.POINTER(ctypes.c_int), i32]),
        "cp_seq_to_head": (i32, [vp, vp, i32, i64, i32, i32, i32, vp]),
        "cp_head_to_seq": (i32, [vp, vp, i32, i64, i32, i32, i32, vp]),
        "cp_ulysses_workspace_size": (i64, [i64, i32, i32, i32, i32, i32]),
        "cp_ulysses_forward": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, vp, i32, vp, vp,
                                     vp]),
        "cp_ulysses_host_workspace_size": (i64, [i64, i32, i32, i32, i32, i32, i32]),
        "cp_ulysses_forward_host": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, vp, i32, vp,
                                          vp, vp, vp]),
        "cp_usp_host_workspace_size": (i64, [i64, i32, i32, i32, i32, i32, i32]),
        "cp_usp_forward_host": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, i32, vp,
                                      i32, vp, vp, vp, vp]),
        "cp_ulysses_stage": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, vp, i32, vp, vp,
                                   i32, vp]),
        "cp_usp_stage": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, i32, vp, i32, vp,
                               vp, i32, vp]),
        "cp_usp_workspace_size": (i64, [i64, i32, i32, i32, i32, i32]),
        "cp_usp_forward": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, i32, vp, i32, vp,
                                 vp, vp]),
        "cp_attn_block_backward_workspace_size": (i64, [i64, i32]),
        "cp_attn_block_backward": (i32, [vp, vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32,
                                         i64, i64, i32, f32, vp, vp, vp, i32, vp, vp]),
        "cp_ring_backward_workspace_size": (i64, [i64, i32, i32, i32, i32]),
        "cp_ring_backward_host_workspace_size": (i64, [i64, i32, i32, i32, i32, i32, i32]),
        "cp_ring_backward_host": (i32, [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32,
                                        i32, vp, vp, vp, i32, i32, vp, vp, vp]),
        "cp_ring_backward": (i32, [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, i32,
                                   vp, vp, vp, i32, vp, vp]),
        "cp_ring_backward_step": (i32, [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32,
                                        i32, i32, vp, vp, vp, i32, vp, vp]),
        "cp_ring_backward_fused_step": (i32, [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                              i32, i32, i32, vp, vp, vp, i32, vp, vp]),
        "cp_check_device_error": (i32, [vp]),
        "cp_selftest_wait_timeout": (i32, [i32, vp]),
        "cp_debug_bounds": (i32, []),
        "cp_last_error": (ctypes.c_char_p, []),
        "cp_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = L
    return L


def cp_last_error():
    return lib().cp_last_error().decode()


def cp_version():
    return lib().cp_version().decode()


def _check(rc):
    if rc != 0:
        raise CpError(rc, cp_last_error())
    return rc


def _dt(t):
    if t.dtype == torch.float32:
        return CP_F32
    if t.dtype == torch.bfloat16:
        return CP_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _torch_dt(code):
    return torch.bfloat16 if code == CP_BF16 else torch.float32


def _dev(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _layout(layout):
    if layout in ("contiguous", CP_CONTIGUOUS):
        return CP_CONTIGUOUS
    if layout in ("zigzag", CP_ZIGZAG):
        return CP_ZIGZAG
    if layout in ("striped", CP_STRIPED):
        return CP_STRIPED
    raise ValueError(f"unknown layout {layout!r}")


def cp_attn_block(q, k, v, q_offset=0, k_offset=0, causal=True, scale=0.0, out=None,
                  out_dtype=None, lse=None, stream=None):
    """Block attention with global offsets -> (out [Sq,H,D], lse [H,Sq] fp32)."""
    Sq, H, D = q.shape
    Sk, Hkv, _ = k.shape
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    if out is None:
        out = torch.empty(Sq, H, D, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(H, Sq, dtype=torch.float32, device=q.device)
    _dev(q, k, v, out, lse)
    _check(lib().cp_attn_block(_ptr(q), _ptr(k), _ptr(v), _dt(q), Sq, Sk, H, Hkv, D,
                               int(q_offset), int(k_offset), 1 if causal else 0, float(scale),
                               _ptr(out), _dt(out), _ptr(lse), _stream(stream)))
    return out, lse


def cp_lse_merge(out_acc, lse_acc, out_blk, lse_blk, stream=None):
    """In place: (out_acc, lse_acc) <- merge with (out_blk, lse_blk)."""
    Sq, H, D = out_acc.shape
    _dev(out_acc, lse_acc, out_blk, lse_blk)
    for t in (out_acc, lse_acc, out_blk, lse_blk):
        if t.dtype != torch.float32:
            raise TypeError("merge operands are fp32")
    _check(lib().cp_lse_merge(_ptr(out_acc), _ptr(lse_acc), _ptr(out_blk), _ptr(lse_blk), Sq, H,
                              D, _stream(stream)))
    return out_acc, lse_acc


def cp_ring_workspace_size(S, H, D, out_dtype):
    n = lib().cp_ring_workspace_size(S, H, D, _dt(torch.empty(0, dtype=out_dtype)))
    if n < 0:
        raise CpError(int(n), cp_last_error())
    return int(n)


def _ring_buffers(q, out, out_dtype, lse, workspace):
    S, H, D = q.shape
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    if out is None:
        out = torch.empty(S, H, D, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(H, S, dtype=torch.float32, device=q.device)
    need = cp_ring_workspace_size(S, H, D, out.dtype)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    return out, lse, workspace


def ring_runs_fused(q, layout):
    """Whether cp_ring_forward runs the ring in one launch (bf16 inputs, any
    layout), which needs no workspace."""
    return q.dtype == torch.bfloat16 and layout in ("contiguous", "zigzag", "striped")


def ring_backward_runs_fused(q, layout):
    """Whether cp_ring_backward runs in two launches over all steps (bf16
    inputs, any layout)."""
    return q.dtype == torch.bfloat16 and layout in ("contiguous", "zigzag", "striped")


def cp_ring_forward(q, k, v, P, layout="zigzag", out=None, out_dtype=None, lse=None,
                    workspace=None, stream=None):
    """Ring attention of the whole sequence over P virtual ranks -> (out, lse)."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    if workspace is None and ring_runs_fused(q, layout):
        workspace = torch.empty(0, dtype=torch.uint8, device=q.device)  # unused
    out, lse, workspace = _ring_buffers(q, out, out_dtype, lse, workspace)
    _dev(q, k, v, out, lse, workspace)
    _check(lib().cp_ring_forward(_ptr(q), _ptr(k), _ptr(v), _dt(q), S, H, Hkv, D, int(P),
                                 _layout(layout), _ptr(out), _dt(out), _ptr(lse), _ptr(workspace),
                                 _stream(stream)))
    return out, lse


def cp_ring_forward_steps(q, k, v, P, layout="zigzag", out=None, out_dtype=None, lse=None,
                          workspace=None, stream=None):
    """The ring as one launch per step, merging through the fp32
    accumulator -> (out, lse)."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    out, lse, workspace = _ring_buffers(q, out, out_dtype, lse, workspace)
    _dev(q, k, v, out, lse, workspace)
    _check(lib().cp_ring_forward_steps(_ptr(q), _ptr(k), _ptr(v), _dt(q), S, H, Hkv, D, int(P),
                                       _layout(layout), _ptr(out), _dt(out), _ptr(lse),
                                       _ptr(workspace), _stream(stream)))
    return out, lse


def cp_ring_forward_fused(q, k, v, P, layout="zigzag", out=None, out_dtype=None, lse=None,
                          stream=None):
    """The ring with all P steps inside one launch (bf16 inputs, contiguous or
    zigzag) -> (out, lse); needs no workspace."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    if out is None:
        out = torch.empty(S, H, D, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(H, S, dtype=torch.float32, device=q.device)
    _dev(q, k, v, out, lse)
    _check(lib().cp_ring_forward_fused(_ptr(q), _ptr(k), _ptr(v), _dt(q), S, H, Hkv, D, int(P),
                                       _layout(layout), _ptr(out), _dt(out), _ptr(lse),
                                       _stream(stream)))
    return out, lse


def cp_ring_forward_noalloc(q, k, v, P, layout="zigzag", out=None, out_dtype=None, lse=None,
                            stream=None):
    """cp_ring_forward without a workspace: for callers that may not allocate
    device memory, the fp32 accumulator is a fixed 64 MiB array inside the
    library (S*H*D <= 16,777,216 for a bf16 output).  Pass ``out`` and ``lse``
    to avoid the allocations this wrapper would otherwise make for them."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    if out is None:
        out = torch.empty(S, H, D, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(H, S, dtype=torch.float32, device=q.device)
    _dev(q, k, v, out, lse)
    _check(lib().cp_ring_forward_noalloc(_ptr(q), _ptr(k), _ptr(v), _dt(q), S, H, Hkv, D, int(P),
                                         _layout(layout), _ptr(out), _dt(out), _ptr(lse),
                                         _stream(stream)))
    return out, lse


def cp_ring_host_workspace_size(S, H, Hkv, D, groups, in_dtype, out_dtype):
    n = lib().cp_ring_host_workspace_size(S, H, Hkv, D, int(groups),
                                          _dt(torch.empty(0, dtype=in_dtype)),
                                          _dt(torch.empty(0, dtype=out_dtype)))
    if n < 0:
        raise CpError(int(n), cp_last_error())
    return int(n)


def cp_ring_forward_host(hq, hk, hv, P, layout="zigzag", hout=None, out_dtype=None, hlse=None,
                         groups=1, workspace=None, stream=None, copy_stream=None, device=None):
    """cp_ring_forward on host tensors: q, k, v are copied in, out and lse
    copied back, in ``groups`` head groups whose copies (on ``copy_stream``)
    overlap the other groups' attention (on ``stream``).  Returns (hout, hlse)
    as host tensors (page-locked when this wrapper allocates them); they hold
    the result once ``stream`` has completed."""
    S, H, D = hq.shape
    Hkv = hk.shape[1]
    for t in (hq, hk, hv, hout, hlse):
        if t is None:
            continue
        if t.is_cuda:
            raise ValueError("cp_ring_forward_host takes host tensors")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    out_dtype = out_dtype or (hout.dtype if hout is not None else hq.dtype)
    if hout is None:
        hout = torch.empty(S, H, D, dtype=out_dtype, pin_memory=True)
    if hlse is None:
        hlse = torch.empty(H, S, dtype=torch.float32, pin_memory=True)
    if workspace is None:
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        workspace = torch.empty(cp_ring_host_workspace_size(S, H, Hkv, D, groups, hq.dtype,
                                                            hout.dtype),
                                dtype=torch.uint8, device=dev)
    _dev(workspace)
    cs = _stream(stream)
    xs = _stream(copy_stream) if copy_stream is not None else cs
    _check(lib().cp_ring_forward_host(_ptr(hq), _ptr(hk), _ptr(hv), _dt(hq), S, H, Hkv, D,
                                      int(P), _layout(layout), _ptr(hout), _dt(hout), _ptr(hlse),
                                      int(groups), _ptr(workspace), cs, xs))
    return hout, hlse


def cp_ring_copy_workspace_size(S, H, Hkv, D, P, layout, in_dtype, out_dtype):
    n = lib().cp_ring_copy_workspace_size(S, H, Hkv, D, int(P), _layout(layout),
                                          _dt(torch.empty(0, dtype=in_dtype)),
                                          _dt(torch.empty(0, dtype=out_dtype)))
    if n < 0:
        raise CpError(int(n), cp_last_error())
    return int(n)


def cp_ring_forward_copy(q, k, v, P, layout="zigzag", out=None, out_dtype=None, lse=None,
                         workspace=None, stream=None, copy_stream=None):
    """Ring with the KV physically passed rank to rank (double-buffered, the
    copies on ``copy_stream`` overlapping the attention on ``stream``)."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    if out is None:
        out = torch.empty(S, H, D, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(H, S, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(cp_ring_copy_workspace_size(S, H, Hkv, D, P, layout, q.dtype,
                                                            out.dtype),
                                dtype=torch.uint8, device=q.device)
    _dev(q, k, v, out, lse, workspace)
    _check(lib().cp_ring_forward_copy(_ptr(q), _ptr(k), _ptr(v), _dt(q), S, H, Hkv, D, int(P),
                                      _layout(layout), _ptr(out), _dt(out), _ptr(lse),
                                      _ptr(workspace), _stream(stream),
                                      ctypes.c_void_p(copy_stream.cuda_stream)
                                      if copy_stream is not None else _stream(stream)))
    return out, lse


def cp_ring_step(q, k, v, P, layout, step, out, lse, workspace=None, stream=None):
    """Step `step` of the ring (see cp_ring_forward); updates out/lse in place."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    _dev(q, k, v, out, lse, workspace)
    _check(lib().cp_ring_step(_ptr(q), _ptr(k), _ptr(v), _dt(q), S, H, Hkv, D, int(P),
                              _layout(layout), int(step), _ptr(out), _dt(out), _ptr(lse),
                              _ptr(workspace), _stream(stream)))
    return out, lse


def cp_ring_step_blocks(P, layout, step):
    """Host-only: list of (rank, q_chunk, kv_chunk, diagonal) the ring evaluates at `step`."""
    L = lib()
    n = L.cp_ring_step_blocks(int(P), _layout(layout), int(step), None, 0)
    if n < 0:
        raise CpError(n, cp_last_error())
    buf = (ctypes.c_int * (4 * max(n, 1)))()
    m = L.cp_ring_step_blocks(int(P), _layout(layout), int(step), buf, n)
    if m != n:
        raise CpError(-1, "block count changed")
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(n)]


def cp_seq_to_head(x, P, y=None, stream=None):
    """x [S,H,D] -> y [P,S,H/P,D]."""
    S, H, D = x.shape
    if y is None:
        y = torch.empty(P, S, H // P, D, dtype=x.dtype, device=x.device)
    _dev(x, y)
    _check(lib().cp_seq_to_head(_ptr(x), _ptr(y), _dt(x), S, H, D, int(P), _stream(stream)))
    return y


def cp_head_to_seq(y, x=None, stream=None):
    """y [P,S,H/P,D] -> x [S,H,D]."""
    P, S, G, D = y.shape
    if x is None:
        x = torch.empty(S, P * G, D, dtype=y.dtype, device=y.device)
    _dev(x, y)
    _check(lib().cp_head_to_seq(_ptr(y), _ptr(x), _dt(y), S, P * G, D, int(P), _stream(stream)))
    return x


def cp_ulysses_workspace_size(S, H, Hkv, D, in_dtype, out_dtype):
    n = lib().cp_ulysses_workspace_size(S, H, Hkv, D, _dt(torch.empty(0, dtype=in_dtype)),
                                        _dt(torch.empty(0, dtype=out_dtype)))
    if n < 0:
        raise CpError(int(n), cp_last_error())
    return int(n)


def cp_ulysses_forward(q, k, v, P, out=None, out_dtype=None, lse=None, workspace=None,
                       stream=None):
    """Ulysses attention with P virtual ranks -> (out [S,H,D], lse [H,S])."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    if out is None:
        out = torch.empty(S, H, D, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(H, S, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(cp_ulysses_workspace_size(S, H, Hkv, D, q.dtype, out.dtype),
                                dtype=torch.uint8, device=q.device)
    _dev(q, k, v, out, lse, workspace)
    _check(lib().cp_ulysses_forward(_ptr(q), _ptr(k), _ptr(v), _dt(q), S, H, Hkv, D, int(P),
                                    _ptr(out), _dt(out), _ptr(lse), _ptr(workspace),
                                    _stream(stream)))
    return out, lse


def cp_ulysses_host_workspace_size(S, H, Hkv, D, P, in_dtype, out_dtype):
    n = lib().cp_ulysses_host_workspace_size(S, H, Hkv, D, int(P),
                                             _dt(torch.empty(0, dtype=in_dtype)),
                                             _dt(torch.empty(0, dtype=out_dtype)))
    if n < 0:
        raise CpError(int(n), cp_last_error())
    return int(n)


def cp_ulysses_forward_host(hq, hk, hv, P, hout=None, out_dtype=None, hlse=None, workspace=None,
                            stream=None, copy_stream=None, device=None):
    """cp_ulysses_forward on host tensors, the all-to-alls done by strided
    copies; returns (hout, hlse), host tensors (page-locked when this wrapper
    allocates them) that hold the result once ``stream`` has completed."""
    S, H, D = hq.shape
    Hkv = hk.shape[1]
    for t in (hq, hk, hv, hout, hlse):
        if t is None:
            continue
        if t.is_cuda:
            raise ValueError("cp_ulysses_forward_host takes host tensors")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    out_dtype = out_dtype or (hout.dtype if hout is not None else hq.dtype)
    if hout is None:
        hout = torch.empty(S, H, D, dtype=out_dtype, pin_memory=True)
    if hlse is None:
        hlse = torch.empty(H, S, dtype=torch.float32, pin_memory=True)
    if workspace is None:
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        workspace = torch.empty(cp_ulysses_host_workspace_size(S, H, Hkv, D, P, hq.dtype,
                                                               hout.dtype),
                                dtype=torch.uint8, device=dev)
    _dev(workspace)
    cs = _stream(stream)
    xs = _stream(copy_stream) if copy_stream is not None else cs
    _check(lib().cp_ulysses_forward_host(_ptr(hq), _ptr(hk), _ptr(hv), _dt(hq), S, H, Hkv, D,
                                         int(P), _ptr(hout), _dt(hout), _ptr(hlse),
                                         _ptr(workspace), cs, xs))
    return hout, hlse


def cp_usp_host_workspace_size(S, H, Hkv, D, Pu, in_dtype, out_dtype):
    n = lib().cp_usp_host_workspace_size(S, H, Hkv, D, int(Pu),
                                         _dt(torch.empty(0, dtype=in_dtype)),
                                         _dt(torch.empty(0, dtype=out_dtype)))
    if n < 0:
        raise CpError(int(n), cp_last_error())
    return int(n)


def cp_usp_forward_host(hq, hk, hv, Pu, Pr, layout="zigzag", hout=None, out_dtype=None,
                        hlse=None, workspace=None, stream=None, copy_stream=None, device=None):
    """cp_usp_forward on host tensors (the Ulysses all-to-alls as strided
    copies, a ring of Pr ranks in each of the Pu groups); returns (hout, hlse),
    host tensors that hold the result once ``stream`` has completed."""
    S, H, D = hq.shape
    Hkv = hk.shape[1]
    for t in (hq, hk, hv, hout, hlse):
        if t is None:
            continue
        if t.is_cuda:
            raise ValueError("cp_usp_forward_host takes host tensors")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    out_dtype = out_dtype or (hout.dtype if hout is not None else hq.dtype)
    if hout is None:
        hout = torch.empty(S, H, D, dtype=out_dtype, pin_memory=True)
    if hlse is None:
        hlse = torch.empty(H, S, dtype=torch.float32, pin_memory=True)
    if workspace is None:
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        workspace = torch.empty(cp_usp_host_workspace_size(S, H, Hkv, D, Pu, hq.dtype,
                                                           hout.dtype),
                                dtype=torch.uint8, device=dev)
    _dev(workspace)
    cs = _stream(stream)
    xs = _stream(copy_stream) if copy_stream is not None else cs
    _check(lib().cp_usp_forward_host(_ptr(hq), _ptr(hk), _ptr(hv), _dt(hq), S, H, Hkv, D,
                                     int(Pu), int(Pr), _layout(layout), _ptr(hout), _dt(hout),
                                     _ptr(hlse), _ptr(workspace), cs, xs))
    return hout, hlse


def cp_ulysses_stage(q, k, v, P, stage, out, lse, workspace, stream=None):
    """One stage of cp_ulysses_forward (0 permute in, 1 attention, 2 permute
    out); out, lse and workspace carry the state between stages."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    _dev(q, k, v, out, lse, workspace)
    _check(lib().cp_ulysses_stage(_ptr(q), _ptr(k), _ptr(v), _dt(q), S, H, Hkv, D, int(P),
                                  _ptr(out), _dt(out), _ptr(lse), _ptr(workspace), int(stage),
                                  _stream(stream)))


def cp_usp_workspace_size(S, H, Hkv, D, in_dtype, out_dtype):
    n = lib().cp_usp_workspace_size(S, H, Hkv, D, _dt(torch.empty(0, dtype=in_dtype)),
                                    _dt(torch.empty(0, dtype=out_dtype)))
    if n < 0:
        raise CpError(int(n), cp_last_error())
    return int(n)


def cp_usp_forward(q, k, v, Pu, Pr, layout="zigzag", out=None, out_dtype=None, lse=None,
                   workspace=None, stream=None):
    """Ulysses over Pu head groups x ring of Pr ranks -> (out [S,H,D], lse [H,S])."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    if out is None:
        out = torch.empty(S, H, D, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(H, S, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(cp_usp_workspace_size(S, H, Hkv, D, q.dtype, out.dtype),
                                dtype=torch.uint8, device=q.device)
    _dev(q, k, v, out, lse, workspace)
    _check(lib().cp_usp_forward(_ptr(q), _ptr(k), _ptr(v), _dt(q), S, H, Hkv, D, int(Pu),
                                int(Pr), _layout(layout), _ptr(out), _dt(out), _ptr(lse),
                                _ptr(workspace), _stream(stream)))
    return out, lse


def cp_usp_stage(q, k, v, Pu, Pr, layout, stage, out, lse, workspace, stream=None):
    """One stage of cp_usp_forward (0 permute in, 1..Pr ring steps, Pr+1
    permute out); out, lse and workspace carry the state between stages."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    _dev(q, k, v, out, lse, workspace)
    _check(lib().cp_usp_stage(_ptr(q), _ptr(k), _ptr(v), _dt(q), S, H, Hkv, D, int(Pu), int(Pr),
                              _layout(layout), _ptr(out), _dt(out), _ptr(lse), _ptr(workspace),
                              int(stage), _stream(stream)))


def _grad_buffers(q, k, grad_dtype, dq, dk, dv):
    grad_dtype = grad_dtype or (dq.dtype if dq is not None else torch.float32)
    if dq is None:
        dq = torch.empty(q.shape, dtype=grad_dtype, device=q.device)
    if dk is None:
        dk = torch.empty(k.shape, dtype=grad_dtype, device=q.device)
    if dv is None:
        dv = torch.empty(k.shape, dtype=grad_dtype, device=q.device)
    if not (dq.dtype == dk.dtype == dv.dtype):
        raise ValueError("dq, dk and dv must share one dtype")
    return dq, dk, dv


def cp_attn_block_backward_workspace_size(Sq, H):
    n = lib().cp_attn_block_backward_workspace_size(Sq, H)
    if n < 0:
        raise CpError(int(n), cp_last_error())
    return int(n)


def cp_attn_block_backward(q, k, v, out, dout, lse, q_offset=0, k_offset=0, causal=True,
                           scale=0.0, grad_dtype=None, dq=None, dk=None, dv=None,
                           workspace=None, stream=None):
    """Gradients of one block given the whole-row out / lse -> (dq, dk, dv)."""
    Sq, H, D = q.shape
    Sk, Hkv, _ = k.shape
    dq, dk, dv = _grad_buffers(q, k, grad_dtype, dq, dk, dv)
    if workspace is None:
        workspace = torch.empty(max(cp_attn_block_backward_workspace_size(Sq, H), 16),
                                dtype=torch.uint8, device=q.device)
    _dev(q, k, v, out, dout, lse, dq, dk, dv, workspace)
    _check(lib().cp_attn_block_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _dt(q), Sq, Sk, H, Hkv, D,
        int(q_offset), int(k_offset), 1 if causal else 0, float(scale), _ptr(dq), _ptr(dk),
        _ptr(dv), _dt(dq), _ptr(workspace), _stream(stream)))
    return dq, dk, dv


def cp_ring_backward_workspace_size(S, H, Hkv, D, grad_dtype):
    n = lib().cp_ring_backward_workspace_size(S, H, Hkv, D,
                                              _dt(torch.empty(0, dtype=grad_dtype)))
    if n < 0:
        raise CpError(int(n), cp_last_error())
    return int(n)


def cp_ring_backward(q, k, v, out, dout, lse, P, layout="zigzag", grad_dtype=None, dq=None,
                     dk=None, dv=None, workspace=None, stream=None):
    """Gradients of cp_ring_forward by the same ring schedule -> (dq, dk, dv)."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    dq, dk, dv = _grad_buffers(q, k, grad_dtype, dq, dk, dv)
    if workspace is None:
        workspace = torch.empty(cp_ring_backward_workspace_size(S, H, Hkv, D, dq.dtype),
                                dtype=torch.uint8, device=q.device)
    _dev(q, k, v, out, dout, lse, dq, dk, dv, workspace)
    _check(lib().cp_ring_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _dt(q), S, H, Hkv, D,
        int(P), _layout(layout), _ptr(dq), _ptr(dk), _ptr(dv), _dt(dq), _ptr(workspace),
        _stream(stream)))
    return dq, dk, dv


def cp_ring_backward_host_workspace_size(S, H, Hkv, D, groups, in_dtype, grad_dtype):
    n = lib().cp_ring_backward_host_workspace_size(S, H, Hkv, D, int(groups),
                                                   _dt(torch.empty(0, dtype=in_dtype)),
                                                   _dt(torch.empty(0, dtype=grad_dtype)))
    if n < 0:
        raise CpError(int(n), cp_last_error())
    return int(n)


def cp_ring_backward_host(hq, hk, hv, hout, hdout, hlse, P, layout="zigzag", grad_dtype=None,
                          hdq=None, hdk=None, hdv=None, groups=1, workspace=None, stream=None,
                          copy_stream=None, device=None):
    """cp_ring_backward on host tensors (the counterpart of
    cp_ring_forward_host): returns (hdq, hdk, hdv), host tensors (page-locked
    when this wrapper allocates them) that hold the gradients once ``stream``
    has completed."""
    S, H, D = hq.shape
    Hkv = hk.shape[1]
    for t in (hq, hk, hv, hout, hdout, hlse, hdq, hdk, hdv):
        if t is None:
            continue
        if t.is_cuda:
            raise ValueError("cp_ring_backward_host takes host tensors")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    grad_dtype = grad_dtype or (hdq.dtype if hdq is not None else torch.float32)
    if hdq is None:
        hdq = torch.empty(S, H, D, dtype=grad_dtype, pin_memory=True)
    if hdk is None:
        hdk = torch.empty(S, Hkv, D, dtype=grad_dtype, pin_memory=True)
    if hdv is None:
        hdv = torch.empty(S, Hkv, D, dtype=grad_dtype, pin_memory=True)
    if workspace is None:
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        workspace = torch.empty(cp_ring_backward_host_workspace_size(S, H, Hkv, D, groups,
                                                                     hq.dtype, grad_dtype),
                                dtype=torch.uint8, device=dev)
    _dev(workspace)
    cs = _stream(stream)
    xs = _stream(copy_stream) if copy_stream is not None else cs
    _check(lib().cp_ring_backward_host(
        _ptr(hq), _ptr(hk), _ptr(hv), _ptr(hout), _ptr(hdout), _ptr(hlse), _dt(hq), S, H, Hkv, D,
        int(P), _layout(layout), _ptr(hdq), _ptr(hdk), _ptr(hdv), _dt(hdq), int(groups),
        _ptr(workspace), cs, xs))
    return hdq, hdk, hdv


def cp_ring_backward_step(q, k, v, out, dout, lse, P, layout, launch, dq, dk, dv, workspace,
                          stream=None):
    """One launch of the per-step ring backward: -1 delta, 2t dK/dV of step t,
    2t+1 dQ of step t."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    _dev(q, k, v, out, dout, lse, dq, dk, dv, workspace)
    _check(lib().cp_ring_backward_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _dt(q), S, H, Hkv, D,
        int(P), _layout(layout), int(launch), _ptr(dq), _ptr(dk), _ptr(dv), _dt(dq),
        _ptr(workspace), _stream(stream)))


def cp_ring_backward_fused_step(q, k, v, out, dout, lse, P, layout, launch, dq, dk, dv,
                                workspace, stream=None):
    """One launch of the two-launch ring backward (bf16 inputs):
    -1 delta, 0 dK/dV over every step, 1 dQ over every step."""
    S, H, D = q.shape
    Hkv = k.shape[1]
    _dev(q, k, v, out, dout, lse, dq, dk, dv, workspace)
    _check(lib().cp_ring_backward_fused_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _dt(q), S, H, Hkv, D,
        int(P), _layout(layout), int(launch), _ptr(dq), _ptr(dk), _ptr(dv), _dt(dq),
        _ptr(workspace), _stream(stream)))


def cp_check_device_error(stream=None):
    """Synchronise the stream; raise CpError(CP_ERR_TIMEOUT) if a kernel's
    bounded wait expired since the last check (CP_ERR_BOUNDS: a bounds check
    of the bounds-checked library failed)."""
    return _check(lib().cp_check_device_error(_stream(stream)))


def cp_debug_bounds():
    """True when the loaded library is the bounds-checked build."""
    return bool(lib().cp_debug_bounds())


def cp_selftest_wait_timeout(timeout_us=2000, stream=None):
    return _check(lib().cp_selftest_wait_timeout(int(timeout_us), _stream(stream)))
