"""Python binding of the GB300 tile-centric communication-overlapped GEMM library.

Argument marshalling only: every step of the path runs in the CUDA kernels of
``_lib/libtlgb300.so`` (built from ``csrc/`` by ``_build.build()``), reached
through the C ABI declared in ``include/tl.h``.  PyTorch supplies device memory
and streams.  There is no fallback: if the library is missing or the device is
not sm_103, the calls raise.

Entry points (same names as the C ABI): ``tl_ag_gemm``, ``tl_gemm_rs``,
``tl_mlp2``, ``tl_moe_combine`` and their ``*_workspace_bytes`` sizes, plus
``Context`` (tl_ctx_create / tl_ctx_check / tl_ctx_destroy / tl_ctx_set_trace),
the host-side tile maps ``tl_ag_tile_order`` / ``tl_rs_tile_order`` and
``tl_trace_bytes`` (the trace buffer is read by ``.trace``).
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = [
    "TL_OK", "TL_ERR_INVALID", "TL_ERR_UNSUPPORTED", "TL_ERR_CUDA", "TL_ERR_TIMEOUT", "TL_ERR_WORKSPACE",
    "TLError", "Config", "Context", "lib", "library_path", "build",
    "tl_ag_gemm", "tl_ag_gemm_ll_capable", "tl_allgather", "tl_gemm_rs", "tl_reduce_scatter", "tl_mlp2",
    "tl_moe_combine",
    "tl_ag_gemm_workspace_bytes", "tl_gemm_rs_workspace_bytes", "tl_gemm_rs_ring_workspace_bytes",
    "tl_mlp2_workspace_bytes", "tl_rs_ring_tile_order", "tl_moe_tile_order", "tl_moe_combine_order",
    "tl_moe_workspace_bytes", "tl_ag_tile_order", "tl_rs_tile_order", "tl_trace_bytes", "tl_ag_attention",
    "tl_ag_attention_workspace_bytes", "EXPORTED_SYMBOLS",
]

TL_OK = 0
TL_ERR_INVALID = -1
TL_ERR_UNSUPPORTED = -2
TL_ERR_CUDA = -3
TL_ERR_TIMEOUT = -4
TL_ERR_WORKSPACE = -5

library_path = _build.LIB
build = _build.build

_c_size = ctypes.c_size_t
_vp = ctypes.c_void_p
_i = ctypes.c_int


class Config(ctypes.Structure):
    """Mirror of ``tl_config`` (include/tl.h)."""
    _fields_ = [
        ("mover_warps", _i),
        ("chunks_per_slab", _i),
        ("swizzle", _i),
        ("grid_ctas", _i),
        ("combine_ctas", _i),
        ("debug_skip_chunk", _i),
        ("timeout_ns", ctypes.c_ulonglong),
        ("pair_ctas", _i),
        ("moe_renorm", _i),
        ("rs_ring", _i),
        ("ag_push", _i),
        ("mover_kparts", _i),
        ("ag_ll", _i),
        ("mover_tma", _i),
    ]


# name -> (restype, argtypes); the full exported C ABI.
_SIGS = {
    "tl_version": (_i, []),
    "tl_config_default": (_i, [ctypes.POINTER(Config)]),
    "tl_ctx_create": (_i, [ctypes.POINTER(_vp), _i, ctypes.POINTER(Config)]),
    "tl_ctx_destroy": (None, [_vp]),
    "tl_ctx_check": (_i, [_vp]),
    "tl_ctx_num_ctas": (_i, [_vp]),
    "tl_trace_bytes": (_c_size, [_i, _i]),
    "tl_ctx_set_trace": (_i, [_vp, _vp, _c_size, _i]),
    "tl_strerror": (ctypes.c_char_p, [_i]),
    "tl_ag_gemm_workspace_bytes": (_c_size, [_i, _i, _i, _i]),
    "tl_ag_gemm": (_i, [_vp, _i, _i, ctypes.POINTER(_vp), _vp, _vp, _vp, _c_size, _i, _i, _i, _vp]),
    "tl_ag_gemm_ll_capable": (_i, [_vp, _i, _i, _i, _i]),
    "tl_allgather": (_i, [_vp, _i, _i, ctypes.POINTER(_vp), _vp, _c_size, _i, _i, _vp]),
    "tl_gemm_rs_workspace_bytes": (_c_size, [_i, _i, _i, _i]),
    "tl_gemm_rs_ring_workspace_bytes": (_c_size, [_i, _i, _i, _i]),
    "tl_gemm_rs": (_i, [_vp, _i, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp, _c_size,
                        _i, _i, _i, _vp]),
    "tl_mlp2_workspace_bytes": (_c_size, [_i, _i, _i, _i]),
    "tl_mlp2": (_i, [_vp, _i, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                     _vp, _c_size, _i, _i, _i, _vp]),
    "tl_moe_workspace_bytes": (_c_size, [_i, _i, _i, _i, _i]),
    "tl_moe_combine": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_size, _i, _i, _i, _i, _vp]),
    "tl_reduce_scatter": (_i, [_vp, _i, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i, _i, _vp]),
    "tl_ag_gemm_static_scratch": (_i, [_vp, _i, _i, ctypes.POINTER(_vp), _vp, _vp, _i, _i, _i, _vp]),
    "tl_ag_attention_workspace_bytes": (_c_size, [_i, _i, _i, _i]),
    "tl_ag_attention": (_i, [_vp, _i, _i, _vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp, _vp, _c_size, _i, _i,
                             _i, _vp]),
    "tl_ag_tile_order": (_i, [_i, _i, _i, _i, _i, _vp, _vp, _vp, _i]),
    "tl_rs_tile_order": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _i]),
    "tl_rs_ring_tile_order": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i]),
    "tl_moe_tile_order": (_i, [_i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _i]),
    "tl_moe_combine_order": (_i, [_i, _i, _i, _i, _i, _i, _vp, _vp, _i]),
}
EXPORTED_SYMBOLS = tuple(_SIGS)

_lib = None


class TLError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {code} ({_strerror(code)})")


def lib():
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"CUDA library not built: {library_path} is missing (call build())")
        L = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _strerror(code: int) -> str:
    try:
        return lib().tl_strerror(code).decode()
    except Exception:
        return "?"


def _check(rc: int, what: str) -> None:
    if rc != TL_OK:
        raise TLError(rc, what)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _ptrs(ts):
    arr = (_vp * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _ptr(t)
    return arr


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _need(t, dtype_name: str, what: str):
    import torch
    dt = {"bf16": torch.bfloat16, "f32": torch.float32, "i32": torch.int32, "u8": torch.uint8}[dtype_name]
    if t is None:
        raise ValueError(f"{what} is required")
    if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CUDA {dtype_name} tensor (got {t.dtype}, {t.device})")


class Context:
    """A library context (``tl_ctx``) on one device."""

    def __init__(self, device: int = 0, **cfg):
        L = lib()
        c = Config()
        _check(L.tl_config_default(ctypes.byref(c)), "tl_config_default")
        for k, v in cfg.items():
            if not hasattr(c, k):
                raise ValueError(f"unknown config field {k!r}")
            setattr(c, k, v)
        h = _vp()
        _check(L.tl_ctx_create(ctypes.byref(h), device, ctypes.byref(c)), "tl_ctx_create")
        self.handle = h
        self.config = c
        self.device = device

    @property
    def num_ctas(self) -> int:
        return lib().tl_ctx_num_ctas(self.handle)

    def set_trace(self, buf, spans_per_warp: int) -> None:
        """tl_ctx_set_trace: record the persistent kernels' spans into ``buf`` (a CUDA uint8
        tensor of at least ``tl_trace_bytes(1, spans_per_warp)`` bytes), or stop with None."""
        if buf is None:
            _check(lib().tl_ctx_set_trace(self.handle, None, 0, spans_per_warp), "tl_ctx_set_trace")
            self._trace_buf = None
            return
        _need(buf, "u8", "trace buffer")
        _check(lib().tl_ctx_set_trace(self.handle, _ptr(buf), buf.numel(), spans_per_warp), "tl_ctx_set_trace")
        self._trace_buf = buf  # the library keeps the pointer: keep the memory alive

    def check(self) -> int:
        """tl_ctx_check: synchronise, read and clear the device status word (returns the code)."""
        return lib().tl_ctx_check(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            lib().tl_ctx_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------- workspace sizes
def tl_ag_gemm_workspace_bytes(W, m_per_rank, n, k) -> int:
    return lib().tl_ag_gemm_workspace_bytes(W, m_per_rank, n, k)


def tl_ag_gemm_ll_capable(ctx: Context, W, m_per_rank, n, k) -> bool:
    """Whether tl_ag_gemm on ctx with ag_ll=1 takes the low-latency gather for this shape."""
    return lib().tl_ag_gemm_ll_capable(ctx.handle, W, m_per_rank, n, k) == 1


def tl_gemm_rs_workspace_bytes(W, m, n, k_r) -> int:
    return lib().tl_gemm_rs_workspace_bytes(W, m, n, k_r)


def tl_gemm_rs_ring_workspace_bytes(W, m, n, k_r) -> int:
    return lib().tl_gemm_rs_ring_workspace_bytes(W, m, n, k_r)


def tl_mlp2_workspace_bytes(W, tokens, hidden, f_r) -> int:
    return lib().tl_mlp2_workspace_bytes(W, tokens, hidden, f_r)


def tl_moe_workspace_bytes(T, H, E, F, topk) -> int:
    return lib().tl_moe_workspace_bytes(T, H, E, F, topk)


def tl_ag_attention_workspace_bytes(W, heads, l_r, d) -> int:
    return lib().tl_ag_attention_workspace_bytes(W, heads, l_r, d)


def tl_ag_attention(ctx: Context, q, k_shards, v_shards, out, workspace, rank: int = 0, stream=None) -> None:
    """out[h] = softmax(q[h] K[h]^T / sqrt(d)) V[h] over the rank-order gather of the K/V
    shards (bf16 [heads, l_r, d] each); the kernel's mover warps gather them, overlapped."""
    W = len(k_shards)
    _need(q, "bf16", "q"); _need(out, "bf16", "out"); _need(workspace, "u8", "workspace")
    for i in range(W):
        _need(k_shards[i], "bf16", f"k_shards[{i}]"); _need(v_shards[i], "bf16", f"v_shards[{i}]")
    heads, l_r, d = q.shape
    if len(v_shards) != W or any(tuple(t.shape) != (heads, l_r, d) for t in list(k_shards) + list(v_shards) + [out]):
        raise ValueError("inconsistent shapes")
    rc = lib().tl_ag_attention(ctx.handle, W, rank, _ptr(q), _ptrs(k_shards), _ptrs(v_shards), _ptr(out),
                               _ptr(workspace), workspace.numel(), heads, l_r, d, _stream(stream))
    _check(rc, "tl_ag_attention")


def tl_trace_bytes(ctas, spans_per_warp) -> int:
    return lib().tl_trace_bytes(ctas, spans_per_warp)


# ---------------------------------------------------------------- operators
def tl_ag_gemm(ctx: Context, a_shards, b, c, workspace, rank: int = 0, stream=None) -> None:
    """C = [A_0; ...; A_{W-1}] . B  (bf16, fp32 accumulate).  Shapes from the tensors."""
    W = len(a_shards)
    for i, a in enumerate(a_shards):
        _need(a, "bf16", f"a_shards[{i}]")
    _need(b, "bf16", "b"); _need(c, "bf16", "c"); _need(workspace, "u8", "workspace")
    m_per_rank, k = a_shards[0].shape
    n = b.shape[1]
    if b.shape[0] != k or tuple(c.shape) != (W * m_per_rank, n) or any(tuple(a.shape) != (m_per_rank, k) for a in a_shards):
        raise ValueError("inconsistent shapes")
    rc = lib().tl_ag_gemm(ctx.handle, W, rank, _ptrs(a_shards), _ptr(b), _ptr(c), _ptr(workspace),
                          workspace.numel(), m_per_rank, n, k, _stream(stream))
    _check(rc, "tl_ag_gemm")


def tl_allgather(ctx: Context, a_shards, workspace, rank: int = 0, stream=None) -> None:
    """Pull-mode AllGather alone: the gathered [A_0; ...; A_{W-1}] lands at the start of workspace."""
    W = len(a_shards)
    for i, a in enumerate(a_shards):
        _need(a, "bf16", f"a_shards[{i}]")
    _need(workspace, "u8", "workspace")
    m_per_rank, k = a_shards[0].shape
    rc = lib().tl_allgather(ctx.handle, W, rank, _ptrs(a_shards), _ptr(workspace), workspace.numel(),
                            m_per_rank, k, _stream(stream))
    _check(rc, "tl_allgather")


def tl_gemm_rs(ctx: Context, a, b, out, workspace, stream=None) -> None:
    """out_o = rows_o(sum_p A_p . B_p) for every owner o (bf16)."""
    W = len(a)
    for i in range(W):
        _need(a[i], "bf16", f"a[{i}]"); _need(b[i], "bf16", f"b[{i}]"); _need(out[i], "bf16", f"out[{i}]")
    _need(workspace, "u8", "workspace")
    m, k_r = a[0].shape
    n = b[0].shape[1]
    if len(b) != W or len(out) != W or any(tuple(x.shape) != (m, k_r) for x in a) or \
            any(tuple(x.shape) != (k_r, n) for x in b) or any(tuple(x.shape) != (m // W, n) for x in out):
        raise ValueError("inconsistent shapes")
    rc = lib().tl_gemm_rs(ctx.handle, W, _ptrs(a), _ptrs(b), _ptrs(out), _ptr(workspace), workspace.numel(),
                          m, n, k_r, _stream(stream))
    _check(rc, "tl_gemm_rs")


def tl_reduce_scatter(ctx: Context, partials, out, stream=None) -> None:
    """ReduceScatter alone: out_o = rows_o(P_0 + ... + P_{W-1}) (fp32 partials, summed in order
    p = 0..W-1, bf16 out)."""
    W = len(partials)
    m, n = partials[0].shape
    if len(out) != W or any(tuple(x.shape) != (m, n) for x in partials) or \
            any(tuple(x.shape) != (m // W, n) for x in out) or m % W:
        raise ValueError("inconsistent shapes")
    for i in range(W):
        _need(partials[i], "f32", f"partials[{i}]"); _need(out[i], "bf16", f"out[{i}]")
    rc = lib().tl_reduce_scatter(ctx.handle, W, _ptrs(partials), _ptrs(out), m, n, _stream(stream))
    _check(rc, "tl_reduce_scatter")


def tl_mlp2(ctx: Context, x_shards, w1, w2, out, workspace, stream=None) -> None:
    """out_o = rows_o(sum_r GELU(AG(X) . W1_r) . W2_r) (bf16)."""
    W = len(x_shards)
    for i in range(W):
        _need(x_shards[i], "bf16", f"x_shards[{i}]"); _need(w1[i], "bf16", f"w1[{i}]")
        _need(w2[i], "bf16", f"w2[{i}]"); _need(out[i], "bf16", f"out[{i}]")
    _need(workspace, "u8", "workspace")
    tr, h = x_shards[0].shape
    f = w1[0].shape[1]
    if any(tuple(x.shape) != (tr, h) for x in x_shards) or any(tuple(x.shape) != (h, f) for x in w1) or \
            any(tuple(x.shape) != (f, h) for x in w2) or any(tuple(x.shape) != (tr, h) for x in out):
        raise ValueError("inconsistent shapes")
    rc = lib().tl_mlp2(ctx.handle, W, _ptrs(x_shards), _ptrs(w1), _ptrs(w2), _ptrs(out), _ptr(workspace),
                       workspace.numel(), tr * W, h, f, _stream(stream))
    _check(rc, "tl_mlp2")


def tl_moe_combine(ctx: Context, x, logits, topk: int, w_gate, w_up, w_down, out, workspace,
                   perm_out=None, counts_out=None, stream=None) -> None:
    """out[t] = sum_j gate_tj * (SiLU(x_t Wg_e) * (x_t Wu_e)) Wd_e (fp32 out)."""
    _need(x, "bf16", "x"); _need(logits, "f32", "logits"); _need(w_gate, "bf16", "w_gate")
    _need(w_up, "bf16", "w_up"); _need(w_down, "bf16", "w_down"); _need(out, "f32", "out")
    _need(workspace, "u8", "workspace")
    if perm_out is not None:
        _need(perm_out, "i32", "perm_out")
    if counts_out is not None:
        _need(counts_out, "i32", "counts_out")
    T, H = x.shape
    E, _, F = w_gate.shape
    if tuple(logits.shape) != (T, E) or tuple(w_up.shape) != (E, H, F) or tuple(w_down.shape) != (E, F, H) or \
            tuple(out.shape) != (T, H):
        raise ValueError("inconsistent shapes")
    rc = lib().tl_moe_combine(ctx.handle, _ptr(x), _ptr(logits), topk, _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                              _ptr(out), _ptr(perm_out), _ptr(counts_out), _ptr(workspace), workspace.numel(),
                              T, H, E, F, _stream(stream))
    _check(rc, "tl_moe_combine")


# ---------------------------------------------------------------- host-side tile maps
def tl_ag_tile_order(W, rank, m_per_rank, n, swizzle):
    import numpy as np
    L = lib()
    cnt = L.tl_ag_tile_order(W, rank, m_per_rank, n, swizzle, None, None, None, 0)
    if cnt < 0:
        raise TLError(cnt, "tl_ag_tile_order")
    out = [np.zeros(cnt, dtype=np.int32) for _ in range(3)]
    rc = L.tl_ag_tile_order(W, rank, m_per_rank, n, swizzle, *[o.ctypes.data for o in out], cnt)
    if rc < 0:
        raise TLError(rc, "tl_ag_tile_order")
    return tuple(out)


def tl_rs_tile_order(W, m, n, swizzle):
    import numpy as np
    L = lib()
    cnt = L.tl_rs_tile_order(W, m, n, swizzle, None, None, None, None, 0)
    if cnt < 0:
        raise TLError(cnt, "tl_rs_tile_order")
    out = [np.zeros(cnt, dtype=np.int32) for _ in range(4)]
    rc = L.tl_rs_tile_order(W, m, n, swizzle, *[o.ctypes.data for o in out], cnt)
    if rc < 0:
        raise TLError(rc, "tl_rs_tile_order")
    return tuple(out)


def tl_rs_ring_tile_order(W, m, n):
    import numpy as np
    L = lib()
    cnt = L.tl_rs_ring_tile_order(W, m, n, None, None, None, None, None, 0)
    if cnt < 0:
        raise TLError(cnt, "tl_rs_ring_tile_order")
    out = [np.zeros(cnt, dtype=np.int32) for _ in range(5)]
    rc = L.tl_rs_ring_tile_order(W, m, n, *[o.ctypes.data for o in out], cnt)
    if rc < 0:
        raise TLError(rc, "tl_rs_ring_tile_order")
    return tuple(out)


def tl_moe_tile_order(T, H, E, F, topk, m_tiles):
    import numpy as np
    L = lib()
    cnt = L.tl_moe_tile_order(T, H, E, F, topk, m_tiles, None, None, None, 0)
    if cnt < 0:
        raise TLError(cnt, "tl_moe_tile_order")
    out = [np.zeros(cnt, dtype=np.int32) for _ in range(3)]
    rc = L.tl_moe_tile_order(T, H, E, F, topk, m_tiles, *[o.ctypes.data for o in out], cnt)
    if rc < 0:
        raise TLError(rc, "tl_moe_tile_order")
    return tuple(out)


def tl_moe_combine_order(T, H, E, F, topk, m_tiles):
    import numpy as np
    L = lib()
    cnt = L.tl_moe_combine_order(T, H, E, F, topk, m_tiles, None, None, 0)
    if cnt < 0:
        raise TLError(cnt, "tl_moe_combine_order")
    out = [np.zeros(cnt, dtype=np.int32) for _ in range(2)]
    rc = L.tl_moe_combine_order(T, H, E, F, topk, m_tiles, *[o.ctypes.data for o in out], cnt)
    if rc < 0:
        raise TLError(rc, "tl_moe_combine_order")
    return tuple(out)


# ---------------------------------------------------------------- AllGather + GEMM without allocation
TL_AG_GEMM_STATIC_SCRATCH_BYTES = 16 << 20


def tl_ag_gemm_static_scratch(ctx: Context, a_shards, b, c, rank: int = 0, stream=None) -> None:
    """tl_ag_gemm for callers that cannot allocate device memory (stream capture, plug-ins
    without an allocator, allocation-free real-time paths): the scratch is the library's
    fixed 16 MiB device array, so problems needing more raise TLError(TL_ERR_WORKSPACE),
    and calls whose GPU work overlaps race on that array."""
    W = len(a_shards)
    m_per_rank, k = a_shards[0].shape
    n = b.shape[1]
    if b.shape[0] != k or tuple(c.shape) != (W * m_per_rank, n) or any(tuple(a.shape) != (m_per_rank, k) for a in a_shards):
        raise ValueError("inconsistent shapes")
    for i, a in enumerate(a_shards):
        _need(a, "bf16", f"a_shards[{i}]")
    _need(b, "bf16", "b"); _need(c, "bf16", "c")
    rc = lib().tl_ag_gemm_static_scratch(ctx.handle, W, rank, _ptrs(a_shards), _ptr(b), _ptr(c), m_per_rank, n, k,
                                         _stream(stream))
    _check(rc, "tl_ag_gemm_static_scratch")
