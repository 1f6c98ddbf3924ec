"""Failure detection on the GPU, without a fault or a hang.

Every device-side wait in the library is bounded; one that gives up records KDA_ERR_TIMEOUT in the
device status word and its kernel returns.  ``kda_selftest_wait_timeout`` runs that path on purpose:
one CTA waits on an mbarrier nothing arrives on, gives up after a fixed number of polls and records
the timeout.  The host reads the status, and the same context then runs a forward that matches the
oracle.  This file is collected last so that a failure here leaves every other test already run.
"""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gated_delta_rule_sm_gb300 import _lib, device_status  # noqa: E402
from gated_delta_rule_sm_gb300.inputs import Workload, make_inputs  # noqa: E402
from kda_cases import gpu_fwd, oracle_fwd, rel_err, tol  # noqa: E402


def test_bounded_wait_reports_timeout_and_the_context_survives():
    lib = _lib.load()
    device_status(reset=True)
    assert lib.kda_selftest_wait_timeout(None) == _lib.KDA_OK
    assert device_status(reset=True) == _lib.KDA_ERR_TIMEOUT
    assert device_status(reset=True) == 0
    x = make_inputs(Workload("t", B=1, T=130, H=2, K=128, V=128, initial_state=True, seed=80), device="cuda:0")
    out, fs = gpu_fwd(x)
    torch.cuda.synchronize()
    assert device_status() == 0
    r_out, r_fs = oracle_fwd(x)
    assert rel_err(out, r_out, "bf16") <= tol("bf16")
    assert rel_err(fs, r_fs, "bf16") <= tol("bf16")
