"""Host-side checks of the C ABI (no GPU needed): the library loads, exports what include/kda.h
declares, and rejects bad arguments before it touches the device."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import __graft_entry__
from gated_delta_rule_sm_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return _lib.load()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert declared == set(_lib.EXPORTS), declared ^ set(_lib.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(6):
        assert _lib.status_string(code)
    assert lib.kda_version() >= 100


def _dims(**kw):
    d = dict(B=1, T=256, H=2, K=64, V=64, dtype=_lib.KDA_BF16, num_seqs=0)
    d.update(kw)
    return _lib.KdaDims(**d)


def _fwd(lib, dims, chunk=64, lb=-5.0, scale=0.125, ptr=1, ws=None, ws_bytes=0, cu=None, cu_host=None):
    p = ctypes.c_void_p(ptr) if ptr else None
    return lib.kda_fwd(ctypes.byref(dims), p, p, p, p, p, p, p, scale, lb, chunk, cu, cu_host, None, p, None, ws,
                       ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("bad,code", [
    (dict(B=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(T=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(K=8), _lib.KDA_ERR_INVALID_ARG),          # head dims below 16 are rejected
    (dict(V=12), _lib.KDA_ERR_INVALID_ARG),
    (dict(K=256), _lib.KDA_ERR_UNSUPPORTED),
    (dict(V=72), _lib.KDA_ERR_UNSUPPORTED),
    (dict(dtype=7), _lib.KDA_ERR_INVALID_ARG),
])
def test_shape_validation(lib, bad, code):
    assert _fwd(lib, _dims(**bad)) == code


def test_scalar_validation(lib):
    assert _fwd(lib, _dims(), chunk=0) == _lib.KDA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(), chunk=48) == _lib.KDA_ERR_UNSUPPORTED
    assert _fwd(lib, _dims(), chunk=128) == _lib.KDA_ERR_UNSUPPORTED
    for c in (16, 32, 64):   # accepted: validation passes and stops at the missing workspace
        assert _fwd(lib, _dims(), chunk=c) == _lib.KDA_ERR_WORKSPACE
    s = lambda c: lib.kda_fwd_workspace_size(ctypes.byref(_dims()), c)
    assert s(16) == s(32) == s(64) > 0
    assert _fwd(lib, _dims(), lb=0.0) == _lib.KDA_ERR_INVALID_ARG      # the gate needs a negative bound
    assert _fwd(lib, _dims(), lb=1.0) == _lib.KDA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(), lb=float("nan")) == _lib.KDA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(), scale=float("inf")) == _lib.KDA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(), ptr=0) == _lib.KDA_ERR_INVALID_ARG


def test_varlen_validation(lib):
    cu = ctypes.c_void_p(16)
    assert _fwd(lib, _dims(B=2, num_seqs=3), cu=cu) == _lib.KDA_ERR_INVALID_ARG   # packed needs B == 1
    assert _fwd(lib, _dims(num_seqs=0), cu=cu) == _lib.KDA_ERR_INVALID_ARG


def _bwd(lib, dims, cu=None, cu_host=None, ptr=16):
    p = ctypes.c_void_p(ptr)
    return lib.kda_bwd(ctypes.byref(dims), p, p, p, p, p, p, p, 0.125, -5.0, 64, cu, cu_host, None, p, None,
                       p, p, p, p, p, p, p, None, None, ctypes.c_size_t(0), None)


@pytest.mark.parametrize("offsets,ok", [
    ([0, 100, 256], True),
    ([0, 0, 100, 100, 256], True),      # empty segments pass their state through
    ([0, 256], True),
    ([1, 100, 256], False),             # does not start at 0
    ([0, 100, 255], False),             # does not end at T
    ([0, 100, 300], False),             # ends past T
    ([0, 150, 100, 256], False),        # decreasing
    ([0, -4, 256], False),
])
def test_host_offsets_validation(lib, offsets, ok):
    """A host copy of cu_seqlens is checked before anything is enqueued (packed-document contract:
    N + 1 entries from 0, never decreasing, ending at T).  Valid copies get past validation and stop at
    the missing workspace; the device pointer is never dereferenced here."""
    n = len(offsets) - 1
    host = _lib.host_offsets(offsets, n + 1)
    cu = ctypes.c_void_p(4096)          # stands for the device copy; not read on the host
    want = _lib.KDA_ERR_WORKSPACE if ok else _lib.KDA_ERR_INVALID_ARG
    d = _dims(num_seqs=n)
    assert _fwd(lib, d, cu=cu, cu_host=host, ptr=16) == want
    assert _bwd(lib, d, cu=cu, cu_host=host) == want
    p = ctypes.c_void_p(16)
    assert lib.kda_fwd_simt(ctypes.byref(d), p, p, p, p, p, p, p, 0.125, -5.0, 64, cu, host, None, p, None, None,
                            ctypes.c_size_t(0), None) == want
    d128 = _dims(num_seqs=n, K=128, V=128)
    want_save = _lib.KDA_ERR_WORKSPACE if ok else _lib.KDA_ERR_INVALID_ARG   # saved buffer missing
    assert lib.kda_fwd_save(ctypes.byref(d128), p, p, p, p, p, p, p, 0.125, -5.0, 64, cu, host, None, p, None,
                            None, ctypes.c_size_t(0), None, ctypes.c_size_t(0), None) == want_save
    assert lib.kda_bwd_saved(ctypes.byref(d128), p, p, p, p, p, p, p, 0.125, -5.0, 64, cu, host, None, p, None,
                             p, p, p, p, p, p, p, None, None, ctypes.c_size_t(0), None, ctypes.c_size_t(0),
                             None) == want_save


def test_host_offsets_without_device_offsets(lib):
    host = _lib.host_offsets([0, 256], 2)
    assert _fwd(lib, _dims(), cu=None, cu_host=host, ptr=16) == _lib.KDA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        _lib.host_offsets([0, 100, 256], 2)        # wrong entry count for the call


def test_workspace_validation(lib):
    d = _dims()
    need = lib.kda_fwd_workspace_size(ctypes.byref(d), 64)
    assert need > 0
    assert _fwd(lib, d, ws=None, ws_bytes=0) == _lib.KDA_ERR_WORKSPACE
    assert _fwd(lib, d, ws=ctypes.c_void_p(4096 + 8), ws_bytes=need) == _lib.KDA_ERR_WORKSPACE  # misaligned


def test_workspace_sizes_grow_with_problem(lib):
    s = lambda **kw: lib.kda_fwd_workspace_size(ctypes.byref(_dims(**kw)), 64)
    b = lambda **kw: lib.kda_bwd_workspace_size(ctypes.byref(_dims(**kw)), 64)
    assert s(T=512) > s(T=256) > 0
    assert s(H=4) > s(H=2)
    assert b(T=256) > s(T=256)
    assert s(num_seqs=5) >= s()            # packed sizing covers the fixed-length layout
    assert lib.kda_fwd_workspace_size(ctypes.byref(_dims(K=8)), 64) == 0
    assert lib.kda_fwd_workspace_size(None, 64) == 0


def _fwd_save(lib, dims, saved=None, saved_bytes=0, ptr=16, lb=-5.0):
    p = ctypes.c_void_p(ptr)
    return lib.kda_fwd_save(ctypes.byref(dims), p, p, p, p, p, p, p, 0.125, lb, 64, None, None, None, p, None,
                            saved, ctypes.c_size_t(saved_bytes), None, ctypes.c_size_t(0), None)


def _bwd_saved(lib, dims, saved=None, saved_bytes=0, ptr=16):
    p = ctypes.c_void_p(ptr)
    return lib.kda_bwd_saved(ctypes.byref(dims), p, p, p, p, p, p, p, 0.125, -5.0, 64, None, None, None, p, None,
                             p, p, p, p, p, p, p, None, saved, ctypes.c_size_t(saved_bytes), None,
                             ctypes.c_size_t(0), None)


def test_saved_context_sizes(lib):
    sz = lambda **kw: lib.kda_saved_size(ctypes.byref(_dims(**kw)), 64)
    assert sz(K=128, V=128, dtype=_lib.KDA_FP32) == 0       # fp32: no tensor-core path, nothing to keep
    assert sz(K=64, V=128) == 0 and sz(K=64, V=64, gate=_lib.GATES["softplus"]) == 0
    one = sz(K=128, V=128)
    assert sz() == one                                      # K = V = 64 heads keep the padded 128-channel record
    assert one > 0 and one % 256 == 0
    assert sz(K=128, V=128, T=512) == 2 * one               # one record per (chunk, head)
    assert sz(K=128, V=128, H=4) == 2 * one
    assert lib.kda_saved_size(None, 64) == 0


def test_saved_context_validation(lib):
    d64, d128 = _dims(K=64, V=128), _dims(K=128, V=128)
    need = lib.kda_saved_size(ctypes.byref(d128), 64)
    # shapes off the tensor-core path are refused, not silently recomputed
    assert _fwd_save(lib, d64) == _lib.KDA_ERR_UNSUPPORTED
    assert _bwd_saved(lib, d64) == _lib.KDA_ERR_UNSUPPORTED
    assert _fwd_save(lib, _dims(dtype=_lib.KDA_FP32)) == _lib.KDA_ERR_UNSUPPORTED
    assert _fwd_save(lib, d128, lb=-6.0) == _lib.KDA_ERR_UNSUPPORTED
    assert _fwd_save(lib, d128, ptr=24) == _lib.KDA_ERR_UNSUPPORTED          # unaligned activations
    # the saved buffer: missing, too small, misaligned
    assert _fwd_save(lib, d128) == _lib.KDA_ERR_WORKSPACE
    assert _fwd_save(lib, d128, saved=ctypes.c_void_p(4096), saved_bytes=need - 256) == _lib.KDA_ERR_WORKSPACE
    assert _fwd_save(lib, d128, saved=ctypes.c_void_p(4096 + 16), saved_bytes=need) == _lib.KDA_ERR_WORKSPACE
    assert _bwd_saved(lib, d128) == _lib.KDA_ERR_WORKSPACE
    assert _bwd_saved(lib, d128, saved=ctypes.c_void_p(4096), saved_bytes=need - 256) == _lib.KDA_ERR_WORKSPACE


def test_grouped_key_heads_validation(lib):
    """H value heads on Hk key heads: H must be a multiple of Hk; Hk = 0 means Hk = H."""
    assert _fwd(lib, _dims(H=3, Hk=2)) == _lib.KDA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(H=4, Hk=-1)) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_fwd_workspace_size(ctypes.byref(_dims(H=3, Hk=2)), 64) == 0
    f = lambda **kw: lib.kda_fwd_workspace_size(ctypes.byref(_dims(**kw)), 64)
    b = lambda **kw: lib.kda_bwd_workspace_size(ctypes.byref(_dims(**kw)), 64)
    assert f(H=4, Hk=2) == f(H=4) == f(H=4, Hk=4)           # the forward keeps nothing per key head
    assert b(H=4, Hk=2) > b(H=4, Hk=4) == b(H=4)             # dq, dk per value head before the group sum
    assert _fwd(lib, _dims(H=4, Hk=2), ws=None, ws_bytes=0) == _lib.KDA_ERR_WORKSPACE   # valid shape


def test_gate_selection_validation(lib):
    """kda_dims.gate: 0 (lower-bounded, the zero-initialised default) or 1 (softplus); else invalid."""
    SP = _lib.GATES["softplus"]
    assert _fwd(lib, _dims(gate=2)) == _lib.KDA_ERR_INVALID_ARG
    assert _fwd(lib, _dims(gate=-1)) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_fwd_workspace_size(ctypes.byref(_dims(gate=2)), 64) == 0
    assert _fwd(lib, _dims(gate=SP)) == _lib.KDA_ERR_WORKSPACE               # valid: stops at the workspace
    assert _fwd(lib, _dims(gate=SP), lb=0.0) == _lib.KDA_ERR_INVALID_ARG     # lower_bound checked under either gate
    f = lambda **kw: lib.kda_fwd_workspace_size(ctypes.byref(_dims(**kw)), 64)
    # K = V = 64: the lower-bounded gate's forward runs on the tensor-core path (records in the
    # workspace), the unbounded one on the SIMT path
    assert 0 < f(gate=SP) < f()
    # the unbounded gate takes the tensor-core path in both directions: the same saved context as the
    # lower-bounded gate, and the saved pair stops at the missing buffer; its backward workspace adds
    # the diagonal sub-blocks of the record pass
    d128, b128 = _dims(K=128, V=128, gate=SP), _dims(K=128, V=128)
    assert lib.kda_saved_size(ctypes.byref(d128), 64) == lib.kda_saved_size(ctypes.byref(b128), 64) > 0
    assert _fwd_save(lib, d128) == _lib.KDA_ERR_WORKSPACE
    assert _bwd_saved(lib, d128) == _lib.KDA_ERR_WORKSPACE
    assert _fwd_save(lib, d128, lb=-50.0) == _lib.KDA_ERR_WORKSPACE           # lower_bound not used by this gate
    bw = lambda d: lib.kda_bwd_workspace_size(ctypes.byref(d), 64)
    assert bw(d128) > bw(b128) > 0


def _conv_fwd(lib, B=1, T=64, C=64, W=4, dtype=_lib.KDA_BF16, ptr=16, cu=None, n=0, y=16):
    p = ctypes.c_void_p(ptr) if ptr else None
    yp = ctypes.c_void_p(y) if y else None
    return lib.kda_short_conv_fwd(B, T, C, W, dtype, p, p, None, cu, n, yp, None)


def test_short_conv_validation(lib):
    assert _conv_fwd(lib, B=0) == _lib.KDA_ERR_INVALID_ARG
    assert _conv_fwd(lib, W=0) == _lib.KDA_ERR_INVALID_ARG
    assert _conv_fwd(lib, dtype=5) == _lib.KDA_ERR_INVALID_ARG
    assert _conv_fwd(lib, ptr=0) == _lib.KDA_ERR_INVALID_ARG
    assert _conv_fwd(lib, y=0) == _lib.KDA_ERR_INVALID_ARG
    assert _conv_fwd(lib, B=2, cu=ctypes.c_void_p(16), n=2) == _lib.KDA_ERR_INVALID_ARG   # packed needs B == 1
    assert _conv_fwd(lib, W=9) == _lib.KDA_ERR_UNSUPPORTED        # at most 8 taps
    assert _conv_fwd(lib, C=12) == _lib.KDA_ERR_UNSUPPORTED       # 8-channel vectors
    assert _conv_fwd(lib, ptr=24) == _lib.KDA_ERR_UNSUPPORTED     # 16-byte aligned data
    ws = lambda **kw: lib.kda_short_conv_bwd_workspace_size(kw.get("B", 1), kw.get("T", 64), kw.get("C", 64),
                                                            kw.get("W", 4))
    assert ws() > 0 and ws() % 256 == 0
    assert ws(T=128) == 2 * ws()          # one partial row per 64-token tile
    assert ws(W=9) == 0 and ws(C=0) == 0


def _fwd_seg(lib, dims, segments=4, ws=None, ws_bytes=0, ptr=16, cu=None, cu_host=None):
    p = ctypes.c_void_p(ptr)
    return lib.kda_fwd_segmented(ctypes.byref(dims), p, p, p, p, p, p, p, 0.125, -5.0, 64, segments, cu, cu_host,
                                 None, p, None, ws, ctypes.c_size_t(ws_bytes), None)


def _bwd_seg(lib, dims, segments=4, ws=None, ws_bytes=0, ptr=16, cu=None, cu_host=None):
    p = ctypes.c_void_p(ptr)
    return lib.kda_bwd_segmented(ctypes.byref(dims), p, p, p, p, p, p, p, 0.125, -5.0, 64, segments, cu, cu_host,
                                 None, p, None, p, p, p, p, p, p, p, None, ws, ctypes.c_size_t(ws_bytes), None)


def test_segmented_forward_validation(lib):
    """kda_fwd_segmented: tensor-core shapes only, segments >= 1, its own workspace size."""
    d128 = _dims(K=128, V=128, T=4096)
    sz = lambda d, n: lib.kda_fwd_segmented_workspace_size(ctypes.byref(d), 64, n)
    assert _fwd_seg(lib, d128, segments=0) == _lib.KDA_ERR_INVALID_ARG
    assert _fwd_seg(lib, _dims(), segments=4) == _lib.KDA_ERR_UNSUPPORTED              # K = V = 64
    assert _fwd_seg(lib, _dims(K=128, V=128, dtype=_lib.KDA_FP32)) == _lib.KDA_ERR_UNSUPPORTED
    assert _fwd_seg(lib, d128, ptr=24) == _lib.KDA_ERR_UNSUPPORTED                     # unaligned activations
    assert _fwd_seg(lib, d128) == _lib.KDA_ERR_WORKSPACE                               # valid: needs its workspace
    assert sz(_dims(), 4) == 0 and sz(d128, 0) == 0
    # three fp32 states (64 KiB) per piece and head on top of the tensor-core forward's buffers
    assert sz(d128, 1) > 3 * 1 * 2 * 65536
    assert sz(d128, 8) - sz(d128, 4) >= 3 * 4 * 2 * 65536
    assert sz(d128, 8) > sz(d128, 4) > sz(d128, 1)
    assert sz(d128, 64) == sz(d128, 1000)            # never more pieces than chunks


def test_segmented_backward_validation(lib):
    """kda_bwd_segmented: the forward's shape rules, segments >= 1, a workspace of its own that holds
    the backward's buffers for the pieces plus three states per piece and head."""
    d128 = _dims(K=128, V=128, T=4096)
    sz = lambda d, n: lib.kda_bwd_segmented_workspace_size(ctypes.byref(d), 64, n)
    assert _bwd_seg(lib, d128, segments=0) == _lib.KDA_ERR_INVALID_ARG
    assert _bwd_seg(lib, _dims(), segments=4) == _lib.KDA_ERR_UNSUPPORTED              # K = V = 64
    assert _bwd_seg(lib, _dims(K=128, V=128, dtype=_lib.KDA_FP32)) == _lib.KDA_ERR_UNSUPPORTED
    assert _bwd_seg(lib, d128, ptr=24) == _lib.KDA_ERR_UNSUPPORTED                     # unaligned activations
    assert _bwd_seg(lib, d128) == _lib.KDA_ERR_WORKSPACE
    assert sz(_dims(), 4) == 0 and sz(d128, 0) == 0
    plain = lib.kda_bwd_workspace_size(ctypes.byref(d128), 64)
    assert sz(d128, 1) > plain + 3 * 1 * 2 * 65536
    assert sz(d128, 8) - sz(d128, 4) >= 3 * 4 * 2 * 65536
    assert sz(d128, 64) == sz(d128, 1000)


def test_segmented_packed_documents_host_checks(lib):
    """With packed documents both segmented entries check a host copy of the offsets before any
    launch, and size their workspace for one piece more per document."""
    lens = [100, 0, 300, 5]
    cu = (ctypes.c_int32 * 5)(0, 100, 100, 400, 405)
    bad = (ctypes.c_int32 * 5)(0, 100, 90, 400, 405)      # decreasing
    dev = ctypes.c_void_p(64)                              # device copy (never read on the host)
    d = _dims(K=128, V=128, B=1, T=sum(lens), num_seqs=len(lens))
    for f in (_fwd_seg, _bwd_seg):
        assert f(lib, d, cu=dev, cu_host=bad) == _lib.KDA_ERR_INVALID_ARG
        assert f(lib, d, cu=dev, cu_host=cu) == _lib.KDA_ERR_WORKSPACE
    rows = _dims(K=128, V=128, B=1, T=sum(lens))
    for f in (lib.kda_fwd_segmented_workspace_size, lib.kda_bwd_segmented_workspace_size):
        assert f(ctypes.byref(d), 64, 4) > f(ctypes.byref(rows), 64, 4) > 0


def test_gated_norm_validation(lib):
    p = ctypes.c_void_p(16)
    fwd = lambda rows=10, V=128, dtype=_lib.KDA_BF16, eps=1e-6, o=p, y=p: lib.kda_gated_norm_fwd(
        rows, V, dtype, o, p, p, eps, y, None)
    assert fwd(rows=0) == _lib.KDA_ERR_INVALID_ARG
    assert fwd(V=0) == _lib.KDA_ERR_INVALID_ARG
    assert fwd(dtype=3) == _lib.KDA_ERR_INVALID_ARG
    assert fwd(eps=-1.0) == _lib.KDA_ERR_INVALID_ARG
    assert fwd(eps=0.0) == _lib.KDA_ERR_INVALID_ARG      # an all-zero row would turn into NaN
    assert fwd(eps=float("nan")) == _lib.KDA_ERR_INVALID_ARG
    assert fwd(o=None) == _lib.KDA_ERR_INVALID_ARG
    assert fwd(y=None) == _lib.KDA_ERR_INVALID_ARG
    assert fwd(V=257) == _lib.KDA_ERR_UNSUPPORTED
    ws = lambda rows, V: lib.kda_gated_norm_bwd_workspace_size(rows, V)
    assert ws(10, 128) > 0 and ws(10, 128) % 256 == 0 and ws(10, 128) == ws(10 ** 6, 128)   # per-CTA partials
    assert ws(0, 128) == 0 and ws(10, 257) == 0
    bwd = lambda w=None, nbytes=0: lib.kda_gated_norm_bwd(10, 128, _lib.KDA_BF16, p, p, p, 1e-6, p, p, p, p, w,
                                                          ctypes.c_size_t(nbytes), None)
    assert bwd() == _lib.KDA_ERR_WORKSPACE
    assert bwd(ctypes.c_void_p(4096 + 16), ws(10, 128)) == _lib.KDA_ERR_WORKSPACE       # misaligned


def test_gated_norm_binding_refuses_mixed_types():
    """The norm kernels read every activation with o's element size and the weight as fp32; the
    binding refuses other combinations before anything reaches the library."""
    import torch
    o = torch.zeros(4, 128, dtype=torch.bfloat16)
    w = torch.ones(128)
    _lib._norm_types(o, o.clone(), w)                                    # accepted
    _lib._norm_types(o, o.clone(), w, o.clone())
    with pytest.raises(ValueError):
        _lib._norm_types(o, o.clone(), w.to(torch.bfloat16))             # bf16 weight
    with pytest.raises(ValueError):
        _lib._norm_types(o, o.float(), w)                                # fp32 gate beside bf16 o
    with pytest.raises(ValueError):
        _lib._norm_types(o.float(), o.float(), w, o)                     # bf16 dy beside fp32 o
