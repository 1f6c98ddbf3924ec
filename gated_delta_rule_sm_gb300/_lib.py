"""Thin Python binding of the KDA C ABI (``include/kda.h``).

Argument marshalling only: torch provides device memory and the current CUDA
stream, every step of the computation runs in the library's CUDA kernels.
There is no fallback: if ``libkda_gb300.so`` is missing or CUDA is not
available the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda_gb300.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT, KDA_ERR_WORKSPACE = range(6)
KDA_BF16, KDA_FP32 = 0, 1

# Every symbol include/kda.h declares.
EXPORTS = ("kda_fwd_workspace_size", "kda_bwd_workspace_size", "kda_fwd", "kda_fwd_simt", "kda_bwd",
           "kda_status_string", "kda_device_status", "kda_version", "kda_timing_begin", "kda_timing_end",
           "kda_kernel_name", "kda_fwd_noalloc", "kda_saved_size", "kda_fwd_save", "kda_bwd_saved",
           "kda_short_conv_fwd", "kda_short_conv_bwd_workspace_size", "kda_short_conv_bwd",
           "kda_fwd_segmented_workspace_size", "kda_fwd_segmented", "kda_bwd_segmented_workspace_size",
           "kda_bwd_segmented", "kda_selftest_wait_timeout",
           "kda_gated_norm_fwd", "kda_gated_norm_bwd_workspace_size", "kda_gated_norm_bwd")
NOALLOC_SCRATCH_BYTES = 32 << 20
GATES = {"lower_bounded": 0, "softplus": 1}   # kda_gate


class KdaDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int), ("K", ctypes.c_int),
                ("V", ctypes.c_int), ("dtype", ctypes.c_int), ("num_seqs", ctypes.c_int), ("Hk", ctypes.c_int),
                ("gate", ctypes.c_int)]


class KdaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} (status {code})")
        self.code = code


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (build it first with ``gated_delta_rule_sm_gb300.build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"KDA CUDA library not built: {path} is missing "
                              "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        lib = ctypes.CDLL(path)
        dims_p = ctypes.POINTER(KdaDims)
        lib.kda_fwd_workspace_size.restype = ctypes.c_size_t
        lib.kda_fwd_workspace_size.argtypes = [dims_p, ctypes.c_int]
        lib.kda_bwd_workspace_size.restype = ctypes.c_size_t
        lib.kda_bwd_workspace_size.argtypes = [dims_p, ctypes.c_int]
        # ... chunk_size, cu_seqlens, cu_seqlens_host, initial_state, out, final_state, workspace, bytes, stream
        fwd_args = [dims_p] + [_vp] * 7 + [ctypes.c_float, ctypes.c_float, ctypes.c_int] + [_vp] * 5 + \
            [_vp, ctypes.c_size_t, _vp]
        for name in ("kda_fwd", "kda_fwd_simt"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = fwd_args
        lib.kda_fwd_segmented_workspace_size.restype = ctypes.c_size_t
        lib.kda_fwd_segmented_workspace_size.argtypes = [dims_p, ctypes.c_int, ctypes.c_int]
        lib.kda_fwd_segmented.restype = ctypes.c_int
        # ... chunk_size, segments, cu_seqlens, cu_seqlens_host, initial_state, out, final_state, ws, bytes, stream
        lib.kda_fwd_segmented.argtypes = [dims_p] + [_vp] * 7 + [ctypes.c_float, ctypes.c_float, ctypes.c_int,
                                                                  ctypes.c_int] + [_vp] * 5 + [_vp, ctypes.c_size_t, _vp]
        gn = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, ctypes.c_float]
        lib.kda_gated_norm_fwd.restype = ctypes.c_int
        lib.kda_gated_norm_fwd.argtypes = gn + [_vp, _vp]
        lib.kda_gated_norm_bwd_workspace_size.restype = ctypes.c_size_t
        lib.kda_gated_norm_bwd_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int]
        lib.kda_gated_norm_bwd.restype = ctypes.c_int
        lib.kda_gated_norm_bwd.argtypes = gn + [_vp] * 4 + [_vp, ctypes.c_size_t, _vp]
        lib.kda_selftest_wait_timeout.restype = ctypes.c_int
        lib.kda_selftest_wait_timeout.argtypes = [_vp]
        lib.kda_fwd_noalloc.restype = ctypes.c_int
        lib.kda_fwd_noalloc.argtypes = [dims_p] + [_vp] * 7 + [ctypes.c_float, ctypes.c_float, ctypes.c_int] + \
            [_vp] * 5 + [_vp]
        lib.kda_bwd.restype = ctypes.c_int
        lib.kda_bwd.argtypes = [dims_p] + [_vp] * 7 + [ctypes.c_float, ctypes.c_float, ctypes.c_int] + \
            [_vp] * 3 + [_vp] * 2 + [_vp] * 8 + [_vp, ctypes.c_size_t, _vp]
        lib.kda_bwd_segmented_workspace_size.restype = ctypes.c_size_t
        lib.kda_bwd_segmented_workspace_size.argtypes = [dims_p, ctypes.c_int, ctypes.c_int]
        lib.kda_bwd_segmented.restype = ctypes.c_int
        lib.kda_bwd_segmented.argtypes = [dims_p] + [_vp] * 7 + [ctypes.c_float, ctypes.c_float, ctypes.c_int,
                                                                  ctypes.c_int] + [_vp] * 3 + [_vp] * 2 + [_vp] * 8 + \
            [_vp, ctypes.c_size_t, _vp]
        lib.kda_saved_size.restype = ctypes.c_size_t
        lib.kda_saved_size.argtypes = [dims_p, ctypes.c_int]
        lib.kda_fwd_save.restype = ctypes.c_int
        lib.kda_fwd_save.argtypes = fwd_args[:-3] + [_vp, ctypes.c_size_t] + fwd_args[-3:]
        lib.kda_bwd_saved.restype = ctypes.c_int
        lib.kda_bwd_saved.argtypes = lib.kda_bwd.argtypes[:-3] + [_vp, ctypes.c_size_t] + lib.kda_bwd.argtypes[-3:]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_device_status.restype = ctypes.c_int
        lib.kda_device_status.argtypes = [ctypes.c_int]
        lib.kda_version.restype = ctypes.c_int
        lib.kda_version.argtypes = []
        lib.kda_timing_begin.restype = ctypes.c_int
        lib.kda_timing_begin.argtypes = [ctypes.c_int]
        lib.kda_timing_end.restype = ctypes.c_int
        lib.kda_timing_end.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int), ctypes.c_int]
        lib.kda_kernel_name.restype = ctypes.c_char_p
        lib.kda_kernel_name.argtypes = [ctypes.c_int]
        conv = [ctypes.c_int] * 5 + [_vp] * 4 + [ctypes.c_int]
        lib.kda_short_conv_fwd.restype = ctypes.c_int
        lib.kda_short_conv_fwd.argtypes = conv + [_vp, _vp]
        lib.kda_short_conv_bwd_workspace_size.restype = ctypes.c_size_t
        lib.kda_short_conv_bwd_workspace_size.argtypes = [ctypes.c_int] * 4
        lib.kda_short_conv_bwd.restype = ctypes.c_int
        lib.kda_short_conv_bwd.argtypes = conv + [_vp] * 5 + [ctypes.c_size_t, _vp]
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().kda_status_string(int(code)).decode()


def device_status(reset: bool = True) -> int:
    """The device status word (synchronises the device)."""
    return load().kda_device_status(1 if reset else 0)


def timing_begin(max_launches: int) -> None:
    """Start recording per-kernel CUDA events inside the library (see kda_timing_begin)."""
    _check(load().kda_timing_begin(int(max_launches)), "kda_timing_begin")


def timing_end(cap: int = 1 << 16) -> list[tuple[str, float]]:
    """Stop recording; returns [(kernel name, milliseconds)] in launch order."""
    lib = load()
    ms = (ctypes.c_float * cap)()
    ids = (ctypes.c_int * cap)()
    n = lib.kda_timing_end(ms, ids, cap)
    if n < 0:
        raise KdaError(KDA_ERR_CUDA, "kda_timing_end")
    return [(lib.kda_kernel_name(ids[i]).decode(), float(ms[i])) for i in range(n)]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def host_offsets(cu_seqlens_host, n_expected: Optional[int] = None):
    """A host copy of packed-document offsets as a ctypes int32 array (None stays None).

    Accepts a CPU tensor or any sequence of ints.  ``n_expected``: the entry count the call needs
    (num_seqs + 1); a copy of another length is refused here, since the library reads exactly that
    many entries."""
    if cu_seqlens_host is None:
        return None
    if isinstance(cu_seqlens_host, torch.Tensor):
        if cu_seqlens_host.is_cuda:
            raise ValueError("cu_seqlens_host must live in host memory")
        vals = [int(x) for x in cu_seqlens_host.reshape(-1).tolist()]
    else:
        vals = [int(x) for x in cu_seqlens_host]
    if n_expected is not None and len(vals) != n_expected:
        raise ValueError(f"cu_seqlens_host has {len(vals)} entries, the call needs {n_expected}")
    return (ctypes.c_int32 * len(vals))(*vals)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_FP32
    raise TypeError(f"unsupported activation dtype {t.dtype} (bf16 or fp32)")


def _gate_code(gate: str) -> int:
    if gate not in GATES:
        raise ValueError(f"gate must be one of {sorted(GATES)}, got {gate!r}")
    return GATES[gate]


def make_dims(q: torch.Tensor, v: torch.Tensor, cu_seqlens: Optional[torch.Tensor],
              gate: str = "lower_bounded") -> KdaDims:
    """Shape of a call: q [B, T, Hk, K] (key heads), v [B, T, H, V] (value heads)."""
    B, T, Hk, K = q.shape
    H, V = v.shape[2], v.shape[-1]
    n = int(cu_seqlens.numel() - 1) if cu_seqlens is not None else 0
    return KdaDims(B, T, H, K, V, _dtype_code(q), n, Hk, _gate_code(gate))


def _check_shapes(q, k, v, g_raw, beta_raw, a_log, dt_bias):
    B, T, Hk, K = q.shape
    if k.shape != q.shape or v.dim() != 4 or tuple(v.shape[:2]) != (B, T):
        raise ValueError("q, k must share [B, T, Hk, K] and v must be [B, T, H, V]")
    H = v.shape[2]
    if H % Hk:
        raise ValueError(f"value heads ({H}) must be a multiple of key heads ({Hk})")
    if tuple(g_raw.shape) != (B, T, H, K) or tuple(beta_raw.shape) != (B, T, H):
        raise ValueError("g_raw must be [B, T, H, K] and beta_raw [B, T, H] (value heads)")
    if a_log.numel() != H or dt_bias.numel() != H * K:
        raise ValueError("a_log must hold H values and dt_bias H * K (value heads)")


class _Workspace:
    """Caches one device workspace per (device, kind); grows on demand."""

    def __init__(self):
        self.buf: dict = {}

    def get(self, device: torch.device, kind: str, nbytes: int) -> torch.Tensor:
        key = (device.index, kind)
        b = self.buf.get(key)
        if b is None or b.numel() < nbytes:
            b = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
            self.buf[key] = b
        return b

    def clear(self):
        self.buf.clear()


workspace_cache = _Workspace()


def _check(code: int, what: str):
    if code != KDA_OK:
        raise KdaError(code, what)


def _contig(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("KDA inputs must be contiguous CUDA tensors")


def forward(q, k, v, g_raw, beta_raw, a_log, dt_bias, *, scale: float, lower_bound: float = -5.0,
            gate: str = "lower_bounded", chunk_size: int = 64, cu_seqlens=None, cu_seqlens_host=None,
            initial_state=None, output_final_state: bool = False, out=None, final_state=None, simt: bool = False,
            saved: Optional[torch.Tensor] = None, segments: int = 0, stream: Optional[torch.cuda.Stream] = None):
    """KDA forward through ``kda_fwd`` (or ``kda_fwd_simt``).  Returns (out, final_state or None).

    ``gate``: "lower_bounded" (g = lower_bound * sigmoid(exp(a_log) * (g_raw + dt_bias))) or
    "softplus" (g = -exp(a_log) * softplus(g_raw + dt_bias), unbounded below).
    ``saved``: a device byte buffer of ``saved_size(...)`` bytes; the forward then runs
    ``kda_fwd_save`` and keeps the per-chunk quantities there for ``backward(..., saved=...)``.
    ``segments`` > 0: run ``kda_fwd_segmented``, the chain cut into pieces of about 1 / segments of a
    row (of the longest possible document with ``cu_seqlens``); for long rows with few rows x heads.
    ``cu_seqlens_host``: optional host copy of ``cu_seqlens`` (CPU tensor or sequence); the library then
    checks the offsets before it launches anything and a bad one raises ``KdaError`` (invalid argument).
    """
    lib = load()
    _contig(q, k, v, g_raw, beta_raw, a_log, dt_bias, cu_seqlens, initial_state)
    _check_shapes(q, k, v, g_raw, beta_raw, a_log, dt_bias)
    dims = make_dims(q, v, cu_seqlens, gate)
    B, T, _, K = q.shape
    H, V = v.shape[2], v.shape[-1]
    N = dims.num_seqs if cu_seqlens is not None else B
    if out is None:
        out = torch.empty((B, T, H, V), dtype=q.dtype, device=q.device)
    if output_final_state and final_state is None:
        final_state = torch.empty((N, H, K, V), dtype=torch.float32, device=q.device)
    if not output_final_state:
        final_state = None
    st = stream if stream is not None else torch.cuda.current_stream(q.device)
    cu_h = host_offsets(cu_seqlens_host, N + 1 if cu_seqlens is not None else None)
    if segments:
        if saved is not None or simt:
            raise ValueError("segments= runs without saved= or simt=")
        ws_bytes = lib.kda_fwd_segmented_workspace_size(ctypes.byref(dims), int(chunk_size), int(segments))
        ws = workspace_cache.get(q.device, "fwd", ws_bytes)
        code = lib.kda_fwd_segmented(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
                                     _ptr(a_log), _ptr(dt_bias), float(scale), float(lower_bound), int(chunk_size),
                                     int(segments), _ptr(cu_seqlens), cu_h, _ptr(initial_state), _ptr(out),
                                     _ptr(final_state), _ptr(ws), ctypes.c_size_t(ws.numel()),
                                     ctypes.c_void_p(st.cuda_stream))
        _check(code, "kda_fwd_segmented")
        return out, final_state
    ws_bytes = lib.kda_fwd_workspace_size(ctypes.byref(dims), chunk_size)
    ws = workspace_cache.get(q.device, "fwd", ws_bytes)
    head = (ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw), _ptr(a_log),
            _ptr(dt_bias), float(scale), float(lower_bound), int(chunk_size), _ptr(cu_seqlens), cu_h,
            _ptr(initial_state), _ptr(out), _ptr(final_state))
    tail = (_ptr(ws), ctypes.c_size_t(ws.numel()), ctypes.c_void_p(st.cuda_stream))
    if saved is not None:
        if simt:
            raise ValueError("saved= needs the tensor-core forward")
        code = lib.kda_fwd_save(*head, _ptr(saved), ctypes.c_size_t(saved.numel() * saved.element_size()), *tail)
        _check(code, "kda_fwd_save")
        return out, final_state
    fn = lib.kda_fwd_simt if simt else lib.kda_fwd
    code = fn(*head, *tail)
    _check(code, "kda_fwd_simt" if simt else "kda_fwd")
    return out, final_state


def saved_size(q, v, cu_seqlens=None, chunk_size: int = 64, gate: str = "lower_bounded") -> int:
    """Bytes of the buffer ``forward(..., saved=...)`` fills (0: the shape has no saved path)."""
    lib = load()
    dims = make_dims(q, v, cu_seqlens, gate)
    return int(lib.kda_saved_size(ctypes.byref(dims), int(chunk_size)))


def backward(q, k, v, g_raw, beta_raw, a_log, dt_bias, dout, *, scale: float, lower_bound: float = -5.0,
             gate: str = "lower_bounded", chunk_size: int = 64, cu_seqlens=None, cu_seqlens_host=None,
             initial_state=None, dfinal_state=None,
             want_dinitial_state: bool = True, grads: Optional[dict] = None,
             saved: Optional[torch.Tensor] = None, segments: int = 0,
             stream: Optional[torch.cuda.Stream] = None) -> dict:
    """KDA backward through ``kda_bwd``.  Returns a dict of fp32 gradients.

    ``saved``: the buffer a ``forward(..., saved=...)`` on the same inputs filled; the backward then
    runs ``kda_bwd_saved`` and skips rebuilding the per-chunk quantities.
    ``segments`` > 0: run ``kda_bwd_segmented``, both state chains cut into the pieces of
    ``forward(..., segments=...)``.
    """
    lib = load()
    _contig(q, k, v, g_raw, beta_raw, a_log, dt_bias, dout, cu_seqlens, initial_state, dfinal_state)
    _check_shapes(q, k, v, g_raw, beta_raw, a_log, dt_bias)
    dims = make_dims(q, v, cu_seqlens, gate)
    B, T, Hk, K = q.shape
    H, V = v.shape[2], v.shape[-1]
    N = dims.num_seqs if cu_seqlens is not None else B
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    if grads is None:
        grads = dict(dq=torch.empty((B, T, Hk, K), **f32), dk=torch.empty((B, T, Hk, K), **f32),
                     dv=torch.empty((B, T, H, V), **f32), dg_raw=torch.empty((B, T, H, K), **f32),
                     dbeta_raw=torch.empty((B, T, H), **f32), da_log=torch.empty((H,), **f32),
                     ddt_bias=torch.empty((H * K,), **f32),
                     dinitial_state=torch.empty((N, H, K, V), **f32) if want_dinitial_state else None)
    if segments and saved is not None:
        raise ValueError("segments= runs without saved=")
    ws_bytes = (lib.kda_bwd_segmented_workspace_size(ctypes.byref(dims), int(chunk_size), int(segments))
                if segments else lib.kda_bwd_workspace_size(ctypes.byref(dims), chunk_size))
    ws = workspace_cache.get(dev, "bwd", ws_bytes)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    cu_h = host_offsets(cu_seqlens_host, N + 1 if cu_seqlens is not None else None)
    head = (ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw), _ptr(a_log),
            _ptr(dt_bias), float(scale), float(lower_bound), int(chunk_size), _ptr(cu_seqlens), cu_h,
            _ptr(initial_state), _ptr(dout), _ptr(dfinal_state), _ptr(grads["dq"]), _ptr(grads["dk"]),
            _ptr(grads["dv"]), _ptr(grads["dg_raw"]), _ptr(grads["dbeta_raw"]), _ptr(grads["da_log"]),
            _ptr(grads["ddt_bias"]), _ptr(grads.get("dinitial_state")))
    tail = (_ptr(ws), ctypes.c_size_t(ws.numel()), ctypes.c_void_p(st.cuda_stream))
    if saved is not None:
        code = lib.kda_bwd_saved(*head, _ptr(saved), ctypes.c_size_t(saved.numel() * saved.element_size()), *tail)
        _check(code, "kda_bwd_saved")
        return grads
    if segments:
        # kda_bwd_segmented takes `segments` right after chunk_size
        code = lib.kda_bwd_segmented(*head[:11], int(segments), *head[11:], *tail)
        _check(code, "kda_bwd_segmented")
        return grads
    code = lib.kda_bwd(*head, *tail)
    _check(code, "kda_bwd")
    return grads


def short_conv(x, weight, bias=None, *, cu_seqlens=None, out=None, stream: Optional[torch.cuda.Stream] = None):
    """Causal depthwise short convolution + SiLU through ``kda_short_conv_fwd``.

    x: [B, T, C] (bf16 or fp32); weight: [C, W] fp32; bias: [C] fp32 or None.  Returns y like x.
    """
    lib = load()
    _contig(x, weight, bias, cu_seqlens)
    B, T, C = x.shape
    W = weight.shape[-1]
    if weight.numel() != C * W or (bias is not None and bias.numel() != C):
        raise ValueError("weight must be [C, W] and bias [C]")
    if out is None:
        out = torch.empty_like(x)
    st = stream if stream is not None else torch.cuda.current_stream(x.device)
    n = int(cu_seqlens.numel() - 1) if cu_seqlens is not None else 0
    code = lib.kda_short_conv_fwd(B, T, C, W, _dtype_code(x), _ptr(x), _ptr(weight), _ptr(bias), _ptr(cu_seqlens),
                                  n, _ptr(out), ctypes.c_void_p(st.cuda_stream))
    _check(code, "kda_short_conv_fwd")
    return out


def short_conv_backward(x, weight, bias, dy, *, cu_seqlens=None, stream: Optional[torch.cuda.Stream] = None) -> dict:
    """Reverse mode of :func:`short_conv`: dict(dx [B, T, C], dweight [C, W], dbias [C] or None), fp32."""
    lib = load()
    _contig(x, weight, bias, dy, cu_seqlens)
    B, T, C = x.shape
    W = weight.shape[-1]
    dev = x.device
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(dx=torch.empty((B, T, C), **f32), dweight=torch.empty((C, W), **f32),
             dbias=torch.empty((C,), **f32) if bias is not None else None)
    ws = workspace_cache.get(dev, "conv", int(lib.kda_short_conv_bwd_workspace_size(B, T, C, W)))
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    n = int(cu_seqlens.numel() - 1) if cu_seqlens is not None else 0
    code = lib.kda_short_conv_bwd(B, T, C, W, _dtype_code(x), _ptr(x), _ptr(weight), _ptr(bias), _ptr(cu_seqlens), n,
                                  _ptr(dy), _ptr(g["dx"]), _ptr(g["dweight"]), _ptr(g["dbias"]), _ptr(ws),
                                  ctypes.c_size_t(ws.numel()), ctypes.c_void_p(st.cuda_stream))
    _check(code, "kda_short_conv_bwd")
    return g


def _norm_types(o, *others):
    """The norm kernels read every activation with o's element size and the weight as fp32: refuse
    anything else before it reaches them (a bf16 weight, or a bf16 gate beside fp32 o, would be read
    past its end).  ``others``: gate, weight[, dy]."""
    gate, weight = others[0], others[1]
    acts = [gate] + list(others[2:])
    if any(t.dtype != o.dtype for t in acts):
        raise ValueError(f"gate and dy must have o's dtype ({o.dtype})")
    if weight.dtype != torch.float32:
        raise ValueError(f"weight must be float32, got {weight.dtype}")
    if any(t.device != o.device for t in others):
        raise ValueError("o, gate, weight and dy must be on one device")


def gated_norm(o, gate, weight, *, eps: float = 1e-6, out=None, stream: Optional[torch.cuda.Stream] = None):
    """The output epilogue through ``kda_gated_norm_fwd``: o / sqrt(mean(o^2) + eps) * weight * sigmoid(gate)
    over the last axis.  o, gate: [..., V] (bf16 or fp32, same dtype); weight: [V] fp32.  Returns y like o."""
    lib = load()
    _contig(o, gate, weight)
    if gate.shape != o.shape or weight.numel() != o.shape[-1]:
        raise ValueError("gate must match o, and weight must hold o.shape[-1] values")
    _norm_types(o, gate, weight)
    V = o.shape[-1]
    if out is None:
        out = torch.empty_like(o)
    st = stream if stream is not None else torch.cuda.current_stream(o.device)
    _check(lib.kda_gated_norm_fwd(o.numel() // V, V, _dtype_code(o), _ptr(o), _ptr(gate), _ptr(weight), float(eps),
                                  _ptr(out), ctypes.c_void_p(st.cuda_stream)), "kda_gated_norm_fwd")
    return out


def gated_norm_backward(o, gate, weight, dy, *, eps: float = 1e-6, stream: Optional[torch.cuda.Stream] = None) -> dict:
    """Reverse mode through ``kda_gated_norm_bwd``: dict(do, dgate [..., V], dweight [V]), all fp32."""
    lib = load()
    _contig(o, gate, weight, dy)
    if gate.shape != o.shape or dy.shape != o.shape or weight.numel() != o.shape[-1]:
        raise ValueError("gate and dy must match o, and weight must hold o.shape[-1] values")
    _norm_types(o, gate, weight, dy)
    V = o.shape[-1]
    rows = o.numel() // V
    f32 = dict(dtype=torch.float32, device=o.device)
    g = dict(do=torch.empty(o.shape, **f32), dgate=torch.empty(o.shape, **f32), dweight=torch.empty((V,), **f32))
    nb = lib.kda_gated_norm_bwd_workspace_size(rows, V)
    ws = workspace_cache.get(o.device, "norm", nb)
    st = stream if stream is not None else torch.cuda.current_stream(o.device)
    _check(lib.kda_gated_norm_bwd(rows, V, _dtype_code(o), _ptr(o), _ptr(gate), _ptr(weight), float(eps), _ptr(dy),
                                  _ptr(g["do"]), _ptr(g["dgate"]), _ptr(g["dweight"]), _ptr(ws),
                                  ctypes.c_size_t(ws.numel()), ctypes.c_void_p(st.cuda_stream)), "kda_gated_norm_bwd")
    return g
