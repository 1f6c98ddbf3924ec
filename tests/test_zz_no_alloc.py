"""kda_fwd_noalloc: the forward for callers that cannot allocate device memory.

Plugin hosts that own every device allocation, or latency-critical loops that must not call
cudaMalloc (it can synchronise the device), cannot hand the library a workspace.  The entry point
under test takes its scratch from a fixed-size array built into the library instead.  Here it is
called through the C ABI twice in a row and compared with kda_fwd (which takes a caller-provided
workspace): the same kernels run on the same inputs with only the scratch address changed, so the
results must be bit-identical; a shape too large for the built-in scratch must be rejected with
KDA_ERR_WORKSPACE.  This file is collected last so that a failure here leaves every
other test already run.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gated_delta_rule_sm_gb300 import _lib  # noqa: E402
from gated_delta_rule_sm_gb300.inputs import Workload, make_inputs  # noqa: E402
from kda_cases import ACT, gpu_fwd  # noqa: E402

DEV = "cuda:0"


def _noalloc(x, out, fs):
    lib = _lib.load()
    dims = _lib.make_dims(x["q"], x["v"], x.get("cu_seqlens"))
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return lib.kda_fwd_noalloc(ctypes.byref(dims), *[ptr(x[n]) for n in ACT], float(x["scale"]),
                               float(x["lower_bound"]), 64, ptr(x.get("cu_seqlens")), None, ptr(x.get("initial_state")),
                               ptr(out), ptr(fs), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("w", [
    Workload("noalloc_tc", B=2, T=200, H=2, K=128, V=128, dtype="bf16", initial_state=True, seed=21),
    Workload("noalloc_simt", B=1, T=256, H=2, K=64, V=64, dtype="fp32", initial_state=True, seed=22),
], ids=lambda w: w.name)
def test_noalloc_matches_kda_fwd_twice(w):
    x = make_inputs(w, device=DEV)
    ref_out, ref_fs = gpu_fwd(x, final=True)
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        fs = torch.full_like(ref_fs, float("nan"))
        assert _noalloc(x, out, fs) == _lib.KDA_OK
        torch.cuda.synchronize()
        assert _lib.device_status() == 0
        assert torch.equal(out, ref_out)
        assert torch.equal(fs, ref_fs)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    w = Workload("noalloc_big", B=1, T=65536, H=8, K=128, V=128, dtype="bf16")
    dims = _lib.KdaDims(w.B, w.T, w.H, w.K, w.V, _lib.KDA_BF16, 0)
    lib = _lib.load()
    assert lib.kda_fwd_workspace_size(ctypes.byref(dims), 64) > _lib.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(16, device=DEV)
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = lib.kda_fwd_noalloc(ctypes.byref(dims), p, p, p, p, p, p, p, 0.1, -5.0, 64, None, None, None, p, None,
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.KDA_ERR_WORKSPACE
