"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle, element by element."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from kda_cases import f64, gpu_bwd, gpu_fwd, head_slice, oracle_bwd, oracle_fwd, rel_err, tol

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gated_delta_rule_sm_gb300 import device_status  # noqa: E402
from gated_delta_rule_sm_gb300.inputs import WORKLOADS, Workload, make_inputs  # noqa: E402

DEV = "cuda:0"


def _check_fwd(x, dtype, simt=False, final=True):
    out, fs = gpu_fwd(x, simt=simt, final=final)
    torch.cuda.synchronize()
    assert device_status() == 0
    r_out, r_fs = oracle_fwd(x)
    e = rel_err(out, r_out, dtype)
    assert e <= tol(dtype), ("out", e)
    if final:
        e2 = rel_err(fs, r_fs, dtype)
        assert e2 <= tol(dtype), ("final_state", e2)
    return out, fs


GRADS = ("dq", "dk", "dv", "dg_raw", "dbeta_raw", "da_log", "ddt_bias", "dinitial_state")


def _check_bwd(x, dtype, dfinal=None, segments=0):
    g = gpu_bwd(x, dfinal=dfinal, segments=segments)
    torch.cuda.synchronize()
    assert device_status() == 0
    r = oracle_bwd(x, dfinal=dfinal)
    errs = {n: rel_err(g[n], r[n], dtype) for n in GRADS}
    bad = {n: e for n, e in errs.items() if not e <= tol(dtype)}
    assert not bad, bad
    return g


# ------------------------------------------------------------------ the fp32 workload, exact config

@pytest.mark.parametrize("simt", [False, True])
def test_fwd_fp32_T256_H2_D64(simt):
    x = make_inputs(WORKLOADS["fwd_fp32_T256_H2_D64"], device=DEV)
    _check_fwd(x, "fp32", simt=simt)


# ------------------------------------------------------------------ small bf16 / fp32 cases

@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
@pytest.mark.parametrize("D", [64, 128])
def test_fwd_bf16_ragged(T, D):
    w = Workload("t", B=2, T=T, H=2, K=D, V=D, initial_state=True, seed=T)
    _check_fwd(make_inputs(w, device=DEV), "bf16")


@pytest.mark.parametrize("K,V", [(64, 128), (128, 48), (16, 16), (32, 96)])
def test_fwd_uneven_heads(K, V):
    w = Workload("t", B=1, T=130, H=3, K=K, V=V, initial_state=True, seed=K + V)
    _check_fwd(make_inputs(w, device=DEV), "bf16")


def test_fwd_mild_gate_long_memory():
    """g_raw ~ N(-4, 1) gives alpha close to 1, so early tokens and S0 still matter at the end."""
    w = Workload("t", B=1, T=700, H=2, K=128, V=128, initial_state=True, g_mean=-4.0, seed=5)
    _check_fwd(make_inputs(w, device=DEV), "bf16")


def test_fwd_fp32_mild_gate():
    w = Workload("t", B=2, T=300, H=2, K=64, V=64, dtype="fp32", initial_state=True, g_mean=-4.0, seed=6)
    _check_fwd(make_inputs(w, device=DEV), "fp32")


def test_fwd_varlen_with_empty_and_tiny_documents():
    lens = [5, 0, 64, 130, 1, 63, 65]
    w = Workload("t", B=1, T=sum(lens), H=2, K=128, V=128, varlen=True, initial_state=True, seed=7)
    x = make_inputs(w, device=DEV, lengths=lens)
    _check_fwd(x, "bf16")


def test_fwd_varlen_with_host_offsets():
    """The host copy of cu_seqlens: a valid copy changes nothing; a bad one is refused before launch."""
    import gated_delta_rule_sm_gb300 as kda
    from gated_delta_rule_sm_gb300 import KdaError
    lens = [5, 0, 64, 130, 1, 63, 65]
    w = Workload("t", B=1, T=sum(lens), H=2, K=128, V=128, varlen=True, initial_state=True, seed=7)
    x = make_inputs(w, device=DEV, lengths=lens)
    ref, ref_fs = gpu_fwd(x)
    host = x["cu_seqlens"].cpu()
    args = [x[n] for n in ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")]
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], cu_seqlens=x["cu_seqlens"],
              initial_state=x["initial_state"], output_final_state=True)
    out, fs = kda.forward(*args, cu_seqlens_host=host, **kw)
    torch.cuda.synchronize()
    assert device_status() == 0
    assert torch.equal(out, ref) and torch.equal(fs, ref_fs)
    bad = [int(v) for v in host.tolist()]
    bad[2], bad[3] = bad[3], bad[2]                      # decreasing (5, 69, 5, ...)
    assert bad[3] < bad[2]
    with pytest.raises(KdaError) as ei:
        kda.forward(*args, cu_seqlens_host=bad, **kw)
    assert ei.value.code == 1                            # KDA_ERR_INVALID_ARG, nothing enqueued


@pytest.mark.parametrize("bad", [[0, 150, 100, 256], [8, 100, 256], [0, 100, 200]],
                         ids=["decreasing", "nonzero_start", "short_end"])
@pytest.mark.parametrize("path", ["tc", "simt", "bwd"])
def test_bad_device_offsets_reported_in_status_word(bad, path):
    """Device-only cu_seqlens that break the packed-document contract (every value inside [0, T]): the
    call returns OK, the first kernel records KDA_ERR_INVALID_ARG in the status word and empties the
    chunk table, so no later kernel touches a token (out and dv keep their NaN fill) and the context
    stays usable for the next call."""
    import gated_delta_rule_sm_gb300 as kda
    D = 64 if path == "simt" else 128
    w = Workload("t", B=1, T=256, H=2, K=D, V=D, varlen=True, initial_state=True, backward=(path == "bwd"), seed=40)
    x = make_inputs(w, device=DEV, lengths=[100, 156])
    x["cu_seqlens"] = torch.tensor(bad, dtype=torch.int32, device=DEV)
    args = [x[n] for n in ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")]
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], cu_seqlens=x["cu_seqlens"])
    device_status()                                       # start from a clear word
    if path == "bwd":
        N = len(bad) - 1
        f32 = dict(dtype=torch.float32, device=DEV)
        K = x["q"].shape[-1]
        grads = dict(dq=torch.full((1, 256, 2, K), float("nan"), **f32), dk=torch.full((1, 256, 2, K), float("nan"), **f32),
                     dv=torch.full((1, 256, 2, K), float("nan"), **f32), dg_raw=torch.full((1, 256, 2, K), float("nan"), **f32),
                     dbeta_raw=torch.full((1, 256, 2), float("nan"), **f32), da_log=torch.empty(2, **f32),
                     ddt_bias=torch.empty(2 * K, **f32), dinitial_state=torch.empty((N, 2, K, K), **f32))
        kw["initial_state"] = torch.zeros((N, 2, K, K), **f32)
        kda.backward(*args, x["dout"], grads=grads, **kw)
        assert kda.device_status() == 1                  # KDA_ERR_INVALID_ARG
        assert torch.isnan(grads["dv"]).all() and torch.isnan(grads["dg_raw"]).all()
    else:
        N = len(bad) - 1
        kw["initial_state"] = torch.zeros((N, 2, D, D), dtype=torch.float32, device=DEV)
        out = torch.full_like(x["v"], float("nan"))
        kda.forward(*args, out=out, simt=(path == "simt"), **kw)
        assert kda.device_status() == 1
        assert torch.isnan(out.float()).all()
    # the context is still usable: a valid call right after runs clean and matches the oracle
    y = make_inputs(Workload("t", B=1, T=130, H=2, K=D, V=D, seed=41), device=DEV)
    _check_fwd(y, "bf16", simt=(path == "simt"))


def test_fwd_no_final_state_and_simt_agree():
    w = Workload("t", B=1, T=257, H=2, K=128, V=128, seed=8)
    x = make_inputs(w, device=DEV)
    o1, _ = gpu_fwd(x, final=False)
    o2, _ = gpu_fwd(x, simt=True, final=False)
    r, _ = oracle_fwd(x)
    assert rel_err(o1, r, "bf16") <= 2e-2 and rel_err(o2, r, "bf16") <= 2e-2


def test_fwd_is_deterministic():
    w = Workload("t", B=2, T=300, H=4, K=128, V=128, initial_state=True, seed=9)
    x = make_inputs(w, device=DEV)
    a, fa = gpu_fwd(x)
    b, fb = gpu_fwd(x)
    assert torch.equal(a, b) and torch.equal(fa, fb)


# ------------------------------------------------------------------ backward

@pytest.mark.parametrize("T", [1, 64, 150])
def test_bwd_bf16_small(T):
    w = Workload("t", B=2, T=T, H=2, K=64, V=64, initial_state=True, backward=True, seed=10 + T)
    x = make_inputs(w, device=DEV)
    dfinal = 0.1 * torch.randn((2, 2, 64, 64), generator=torch.Generator().manual_seed(T)).to(DEV)
    _check_bwd(x, "bf16", dfinal=dfinal)


def test_bwd_fp32():
    w = Workload("t", B=1, T=256, H=2, K=64, V=64, dtype="fp32", initial_state=True, backward=True,
                 g_mean=-2.0, seed=11)
    _check_bwd(make_inputs(w, device=DEV), "fp32")


def test_bwd_bf16_d128_varlen():
    lens = [70, 0, 1, 129]
    w = Workload("t", B=1, T=sum(lens), H=2, K=128, V=128, varlen=True, initial_state=True, backward=True,
                 seed=12)
    _check_bwd(make_inputs(w, device=DEV, lengths=lens), "bf16")


@pytest.mark.parametrize("B,H,T", [(1, 2, 150), (1, 64, 130), (2, 64, 130)])
def test_bwd_tc_reverse_chain_widths(B, H, T):
    """2, 64 and 128 (segment, head) chains: the reverse chain runs 32, 64 and 128 value columns
    per CTA on a 152-SM GB300 (the split is chosen from the SM count)."""
    w = Workload("t", B=B, T=T, H=H, K=128, V=128, initial_state=True, backward=True, seed=20 + H + B)
    x = make_inputs(w, device=DEV)
    dfinal = 0.05 * torch.randn((B, H, 128, 128), generator=torch.Generator().manual_seed(H)).to(DEV)
    _check_bwd(x, "bf16", dfinal=dfinal)


def test_bwd_tc_mild_gate_long_memory():
    """g_raw ~ N(-4, 1): per-token decay ~0.9, so state errors persist across chunks."""
    w = Workload("t", B=1, T=300, H=2, K=128, V=128, initial_state=True, backward=True, g_mean=-4.0, seed=14)
    x = make_inputs(w, device=DEV)
    dfinal = 0.05 * torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(7)).to(DEV)
    _check_bwd(x, "bf16", dfinal=dfinal)


def test_bwd_is_deterministic():
    w = Workload("t", B=1, T=200, H=2, K=128, V=128, backward=True, seed=13)
    x = make_inputs(w, device=DEV)
    a = gpu_bwd(x)
    b = gpu_bwd(x)
    for n in ("dq", "da_log", "ddt_bias"):
        assert torch.equal(a[n], b[n])


# ------------------------------------------------------------------ the quoted workloads at full size

def test_full_fwd_bf16_B2_T2048_H16_D128():
    x = make_inputs(WORKLOADS["fwd_bf16_B2_T2048_H16_D128"], device=DEV)
    _check_fwd(x, "bf16", final=False)


def test_full_varlen_fwd_bf16_T16384_H32_sampled_heads():
    x = make_inputs(WORKLOADS["varlen_fwd_bf16_T16384_H32_D128"], device=DEV)
    out, fs = gpu_fwd(x, final=True)
    torch.cuda.synchronize()
    assert device_status() == 0
    heads = [0, 5, 9, 13, 18, 22, 27, 31]
    xs = head_slice(x, heads)
    r_out, r_fs = oracle_fwd(xs)
    assert rel_err(out[:, :, heads], r_out, "bf16") <= 2e-2
    assert rel_err(fs[:, heads], r_fs, "bf16") <= 2e-2


def test_full_long_fwd_bf16_T65536_H32_sampled_heads():
    x = make_inputs(WORKLOADS["long_fwd_bf16_T65536_H32_D128"], device=DEV)
    out, fs = gpu_fwd(x, final=True)
    torch.cuda.synchronize()
    assert device_status() == 0
    heads = [0, 3, 8, 14, 19, 24, 30, 31]   # one oracle thread per head: eight run side by side
    xs = head_slice(x, heads)
    r_out, r_fs = oracle_fwd(xs)
    assert rel_err(out[:, :, heads], r_out, "bf16") <= 2e-2
    assert rel_err(fs[:, heads], r_fs, "bf16") <= 2e-2


def test_full_fwdbwd_bf16_B4_T4096_H32_sampled():
    """The training step as the benchmark runs it: the forward that keeps the per-chunk record, then the
    backward that reads it, at full size; every batch row of four heads against the oracle."""
    import gated_delta_rule_sm_gb300 as kda
    x = make_inputs(WORKLOADS["fwdbwd_bf16_B4_T4096_H32_D128"], device=DEV)
    names = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], chunk_size=64, cu_seqlens=x["cu_seqlens"],
              initial_state=x["initial_state"])
    saved = torch.empty(kda.saved_size(x["q"], x["v"], x["cu_seqlens"]), dtype=torch.uint8, device=DEV)
    out, _ = kda.forward(*[x[n] for n in names], saved=saved, **kw)
    g = kda.backward(*[x[n] for n in names], x["dout"], saved=saved, **kw)
    torch.cuda.synchronize()
    assert device_status() == 0
    heads = [1, 12, 17, 30]
    xs = head_slice(x, heads)
    r_out, _ = oracle_fwd(xs)
    assert rel_err(out[:, :, heads], r_out, "bf16") <= 2e-2
    r = oracle_bwd(xs)
    for n in ("dq", "dk", "dv", "dg_raw", "dbeta_raw"):
        assert rel_err(g[n][:, :, heads], r[n], "bf16") <= 2e-2, n
    if x.get("initial_state") is not None:
        assert rel_err(g["dinitial_state"][:, heads], r["dinitial_state"], "bf16") <= 2e-2
    # the parameter gradients sum over every row and token of their head
    assert rel_err(g["da_log"][heads], r["da_log"], "bf16") <= 2e-2
    K = x["q"].shape[-1]
    assert rel_err(g["ddt_bias"].view(-1, K)[heads], r["ddt_bias"].reshape(len(heads), K), "bf16") <= 2e-2


# ------------------------------------------------------------------ training pair (forward keeps, backward reuses)

def test_saved_pair_matches_plain_calls():
    import gated_delta_rule_sm_gb300 as kda
    lens = [70, 0, 129, 1, 64]
    w = Workload("t", B=1, T=sum(lens), H=3, K=128, V=128, varlen=True, initial_state=True, backward=True, seed=31)
    x = make_inputs(w, device=DEV, lengths=lens)
    names = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], chunk_size=64, cu_seqlens=x["cu_seqlens"],
              initial_state=x["initial_state"])
    nbytes = kda.saved_size(x["q"], x["v"], x["cu_seqlens"])
    assert nbytes > 0
    saved = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o1, f1 = kda.forward(*[x[n] for n in names], output_final_state=True, **kw)
    o2, f2 = kda.forward(*[x[n] for n in names], output_final_state=True, saved=saved, **kw)
    dfinal = 0.05 * torch.randn((len(lens), 3, 128, 128), generator=torch.Generator().manual_seed(3)).to(DEV)
    g1 = kda.backward(*[x[n] for n in names], x["dout"], dfinal_state=dfinal, **kw)
    g2 = kda.backward(*[x[n] for n in names], x["dout"], dfinal_state=dfinal, saved=saved, **kw)
    torch.cuda.synchronize()
    assert device_status() == 0
    # the forward-only pass forms the intra-chunk products its own way (tf32 decayed forms): both forwards
    # must meet the bound against the oracle; the backward is the same computation either way
    r_out, r_fs = oracle_fwd(x)
    for o, f in ((o1, f1), (o2, f2)):
        assert rel_err(o, r_out, "bf16") <= tol("bf16") and rel_err(f, r_fs, "bf16") <= tol("bf16")
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n


# ------------------------------------------------------------------ grouped key heads

@pytest.mark.parametrize("K,H,Hk", [(128, 4, 2), (128, 4, 1), (64, 4, 2)])
def test_grouped_heads_fwd_bwd(K, H, Hk):
    """H value heads on Hk key heads (value head h reads key head h // (H // Hk)); both head sizes
    take the tensor-core path (K = 64 zero-padded to 128 channels inside the kernels); dq, dk are
    summed over each group."""
    w = Workload("t", B=2, T=150, H=H, Hk=Hk, K=K, V=K, initial_state=True, backward=True, seed=31 + H + Hk)
    x = make_inputs(w, device=DEV)
    assert tuple(x["q"].shape) == (2, 150, Hk, K)
    _check_fwd(x, "bf16")
    dfinal = 0.1 * torch.randn((2, H, K, K), generator=torch.Generator().manual_seed(5)).to(DEV)
    names = _launched(lambda: _check_bwd(x, "bf16", dfinal=dfinal))
    assert {"kda_grad_tc", "kda_chain_bwd_tc", "kda_intra_tc"} <= names and "kda_grad_simt" not in names, names


def test_grouped_heads_varlen_and_saved_pair():
    lens = [5, 70, 130, 1]
    w = Workload("t", B=1, T=sum(lens), H=4, Hk=2, K=128, V=128, varlen=True, initial_state=True,
                 backward=True, seed=37)
    x = make_inputs(w, device=DEV, lengths=lens)
    _check_fwd(x, "bf16")
    _check_bwd(x, "bf16")
    import gated_delta_rule_sm_gb300 as kda
    names = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], cu_seqlens=x["cu_seqlens"],
              initial_state=x["initial_state"])
    buf = torch.empty(kda.saved_size(x["q"], x["v"], x["cu_seqlens"]), dtype=torch.uint8, device=DEV)
    o1, _ = kda.forward(*[x[n] for n in names], saved=buf, **kw)
    g1 = kda.backward(*[x[n] for n in names], x["dout"], saved=buf, **kw)
    o2, _ = kda.forward(*[x[n] for n in names], **kw)
    g2 = kda.backward(*[x[n] for n in names], x["dout"], **kw)
    torch.cuda.synchronize()
    r_out, _ = oracle_fwd(x)
    assert rel_err(o1, r_out, "bf16") <= tol("bf16") and rel_err(o2, r_out, "bf16") <= tol("bf16")
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n


# ------------------------------------------------------------------ short convolution + SiLU prologue

def _conv_case(B, T, C, W, dtype, bias=True, seed=0):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = torch.randn((B, T, C), generator=g).to(dt)
    w = (0.5 * torch.randn((C, W), generator=g)).float()
    b = (0.1 * torch.randn((C,), generator=g)).float() if bias else None
    dy = torch.randn((B, T, C), generator=g).to(dt)
    return x, w, b, dy


@pytest.mark.parametrize("B,T,C,W,dtype,bias", [(2, 150, 256, 4, "bf16", True), (1, 300, 64, 3, "fp32", False),
                                                (1, 97, 1024, 1, "bf16", True), (2, 70, 128, 8, "bf16", True),
                                                (4, 1024, 4096, 4, "bf16", True)])
def test_short_conv_fwd_bwd(B, T, C, W, dtype, bias):
    import gated_delta_rule_sm_gb300 as kda
    import oracle
    x, w, b, dy = _conv_case(B, T, C, W, dtype, bias, seed=T + C + W)
    d = lambda t: t.to(DEV) if t is not None else None
    y = kda.short_conv(d(x), d(w), d(b))
    g = kda.short_conv_backward(d(x), d(w), d(b), d(dy))
    torch.cuda.synchronize()
    ry = oracle.short_conv_fwd(f64(x), f64(w), f64(b) if b is not None else None)
    rg = oracle.short_conv_bwd(f64(x), f64(w), f64(b) if b is not None else None, f64(dy))
    assert rel_err(y, ry, "bf16" if dtype == "bf16" else "fp32") <= tol(dtype)
    # the gradients are fp32 computations on exact inputs: the fp32 bound applies to both dtypes
    for n in ("dx", "dweight") + (("dbias",) if bias else ()):
        assert rel_err(g[n], rg[n], "fp32") <= tol("fp32"), n


def test_short_conv_packed_documents():
    import gated_delta_rule_sm_gb300 as kda
    import oracle
    lens = [5, 70, 1, 130, 1]
    x, w, b, dy = _conv_case(1, sum(lens), 256, 4, "bf16", True, seed=7)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    y = kda.short_conv(x.to(DEV), w.to(DEV), b.to(DEV), cu_seqlens=cu.to(DEV))
    g = kda.short_conv_backward(x.to(DEV), w.to(DEV), b.to(DEV), dy.to(DEV), cu_seqlens=cu.to(DEV))
    torch.cuda.synchronize()
    ry = oracle.short_conv_fwd(f64(x), f64(w), f64(b), cu_seqlens=cu.numpy())
    rg = oracle.short_conv_bwd(f64(x), f64(w), f64(b), f64(dy), cu_seqlens=cu.numpy())
    assert rel_err(y, ry, "bf16") <= tol("bf16")
    for n in ("dx", "dweight", "dbias"):
        assert rel_err(g[n], rg[n], "fp32") <= tol("fp32"), n


@pytest.mark.parametrize("chunk", [16, 32])
def test_smaller_chunk_sizes_match_the_oracle(chunk):
    """The result does not depend on the chunk size; 16 and 32 are accepted and run the same kernels."""
    w = Workload("t", B=1, T=200, H=2, K=128, V=128, initial_state=True, backward=True, seed=50 + chunk,
                 chunk_size=chunk)
    x = make_inputs(w, device=DEV)
    assert x["chunk_size"] == chunk
    _check_fwd(x, "bf16")
    _check_bwd(x, "bf16")


# ------------------------------------------------------------------ the unbounded (softplus) gate

def _softplus_case(lengths=None, **kw):
    x = make_inputs(Workload("t", **kw), device=DEV, lengths=lengths)
    x["gate"] = "softplus"
    return x


def test_softplus_gate_fp32_fwd_bwd():
    x = _softplus_case(B=2, T=200, H=2, K=64, V=64, dtype="fp32", initial_state=True, backward=True, seed=60)
    _check_fwd(x, "fp32")
    _check_bwd(x, "fp32")


def _launched(fn):
    """Names of the library kernels fn() launches."""
    from gated_delta_rule_sm_gb300 import _lib
    _lib.timing_begin(4096)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        names = {n for n, _ in _lib.timing_end()}
    return names


def test_softplus_gate_bf16_d128_varlen_fwd_bwd():
    """bf16 K = V = 128 with the unbounded gate: both directions on the tensor-core path (the diagonal
    sub-blocks from the pre-pass in the record pass, summed pair by pair in the gradient kernel), and the
    training pair keeps the record for it too."""
    import gated_delta_rule_sm_gb300 as kda
    x = _softplus_case(B=1, T=400, H=2, K=128, V=128, varlen=True, initial_state=True, backward=True, seed=61,
                       lengths=[90, 1, 64, 200, 45])
    _check_fwd(x, "bf16")
    names = _launched(lambda: _check_bwd(x, "bf16"))
    assert {"kda_diag_tc", "kda_intra_tc", "kda_grad_tc", "kda_chain_bwd_tc"} <= names, names
    assert "kda_grad_simt" not in names, names
    args = [x[n] for n in ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")]
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], gate="softplus", cu_seqlens=x["cu_seqlens"],
              initial_state=x["initial_state"])
    nbytes = kda.saved_size(x["q"], x["v"], x["cu_seqlens"], gate="softplus")
    assert nbytes > 0
    buf = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o1, _ = kda.forward(*args, saved=buf, **kw)
    g1 = kda.backward(*args, x["dout"], saved=buf, **kw)
    g2 = kda.backward(*args, x["dout"], **kw)
    torch.cuda.synchronize()
    assert device_status() == 0
    r_out, _ = oracle_fwd(x)
    assert rel_err(o1, r_out, "bf16") <= tol("bf16")
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n


@pytest.mark.parametrize("case", ["rows", "packed", "grouped"])
def test_fwd_bf16_k64_tensor_core(case):
    """bf16 K = V = 64 heads take the tensor-core forward: the intra pass loads 128-channel tiles whose
    upper half the TMA fills with zeros, and the chain runs the two value slices that exist."""
    if case == "packed":
        lens = [1, 63, 64, 65, 130, 0, 17]
        x = make_inputs(Workload("t", B=1, T=sum(lens), H=3, K=64, V=64, varlen=True, initial_state=True, seed=71),
                        device=DEV, lengths=lens)
    else:
        x = make_inputs(Workload("t", B=2, T=300, H=4, Hk=2 if case == "grouped" else 0, K=64, V=64,
                                 initial_state=True, seed=70), device=DEV)
    names = _launched(lambda: _check_fwd(x, "bf16"))
    assert {"kda_intra_tc", "kda_chain_fwd_tc"} <= names and "kda_intra_simt" not in names, names


@pytest.mark.parametrize("case", ["rows", "packed", "mild"])
def test_bwd_bf16_k64_tensor_core(case):
    """bf16 K = V = 64 heads take the tensor-core backward: the record pass loads 128-channel tiles
    whose upper half is zero, the chains carry 128 x 128 states padded from the caller's 64 x 64 ones
    (initial state and final-state gradient in, initial-state gradient out), and the gradient kernel
    writes only the real channels."""
    if case == "packed":
        lens = [1, 63, 64, 65, 130, 0, 17]
        x = make_inputs(Workload("t", B=1, T=sum(lens), H=3, K=64, V=64, varlen=True, initial_state=True,
                                 backward=True, seed=86), device=DEV, lengths=lens)
        n = len(lens)
    else:
        x = make_inputs(Workload("t", B=2, T=300, H=3, K=64, V=64, initial_state=True, backward=True,
                                 g_mean=-4.0 if case == "mild" else 0.0, seed=87), device=DEV)
        n = 2
    dfinal = 0.1 * torch.randn((n, 3, 64, 64), generator=torch.Generator().manual_seed(9)).to(DEV)
    names = _launched(lambda: _check_bwd(x, "bf16", dfinal=dfinal))
    assert {"kda_intra_tc", "kda_bwd_pre", "kda_chain_rec_tc", "kda_chain_bwd_tc", "kda_grad_tc"} <= names, names
    assert "kda_grad_simt" not in names and "kda_intra_simt" not in names, names


def test_k64_saved_pair_matches_plain_calls():
    """The training pair takes K = V = 64 heads too (the record in its 128-channel layout): the
    gradients equal kda_bwd's bit for bit, and the forward stays within the bound of the oracle."""
    import gated_delta_rule_sm_gb300 as kda
    lens = [70, 0, 129, 1, 64]
    x = make_inputs(Workload("t", B=1, T=sum(lens), H=2, K=64, V=64, varlen=True, initial_state=True,
                             backward=True, seed=88), device=DEV, lengths=lens)
    names = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], chunk_size=64, cu_seqlens=x["cu_seqlens"],
              initial_state=x["initial_state"])
    nbytes = kda.saved_size(x["q"], x["v"], x["cu_seqlens"])
    assert nbytes > 0
    saved = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o2, f2 = kda.forward(*[x[n] for n in names], output_final_state=True, saved=saved, **kw)
    dfinal = 0.05 * torch.randn((len(lens), 2, 64, 64), generator=torch.Generator().manual_seed(4)).to(DEV)
    g1 = kda.backward(*[x[n] for n in names], x["dout"], dfinal_state=dfinal, **kw)
    g2 = kda.backward(*[x[n] for n in names], x["dout"], dfinal_state=dfinal, saved=saved, **kw)
    torch.cuda.synchronize()
    assert device_status() == 0
    r_out, r_fs = oracle_fwd(x)
    assert rel_err(o2, r_out, "bf16") <= 2e-2 and rel_err(f2, r_fs, "bf16") <= 2e-2
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n


@pytest.mark.parametrize("g_mean,Hk", [(0.0, 0), (4.0, 0), (-6.0, 0), (0.0, 1)])
def test_softplus_gate_tensor_core_backward(g_mean, Hk):
    """The tcgen05 backward under the unbounded gate: typical, steep (g near -64 per token: exp(Gamma)
    underflows inside a chunk) and mild decays, and grouped key heads, with a final-state gradient."""
    x = _softplus_case(B=2, T=300, H=2, K=128, V=128, initial_state=True, backward=True, g_mean=g_mean, Hk=Hk,
                       seed=66)
    dfinal = 0.1 * torch.randn((2, 2, 128, 128), generator=torch.Generator().manual_seed(7)).to(DEV)
    names = _launched(lambda: _check_bwd(x, "bf16", dfinal=dfinal))
    assert "kda_grad_tc" in names and "kda_grad_simt" not in names, names


def test_softplus_gate_mild_long_memory():
    """g_raw ~ N(-6, 1): softplus ~ 2.5e-3, so the state keeps its memory over hundreds of tokens."""
    x = _softplus_case(B=1, T=700, H=2, K=128, V=128, initial_state=True, backward=True, g_mean=-6.0, seed=62)
    _check_fwd(x, "bf16")
    _check_bwd(x, "bf16")


def test_softplus_gate_steep_decay_underflows_cleanly():
    """g_raw ~ N(4, 1) with a_log up to ln 16: g near -64 per token, so exp(Gamma) underflows to 0
    within a chunk; every decay is formed as exp(Gamma_t - Gamma_s) <= 1 and stays finite."""
    x = _softplus_case(B=1, T=300, H=2, K=64, V=64, dtype="fp32", initial_state=True, backward=True, g_mean=4.0,
                       seed=63)
    out, fs = _check_fwd(x, "fp32")
    assert torch.isfinite(out).all() and torch.isfinite(fs).all()
    _check_bwd(x, "fp32")


@pytest.mark.parametrize("g_mean,Hk", [(0.0, 0), (4.0, 0), (-6.0, 0), (0.0, 1)])
def test_softplus_gate_tensor_core_forward(g_mean, Hk):
    """bf16 K = V = 128: the forward takes the tcgen05 path with the diagonal sub-blocks from the pre-pass.
    Typical, steep (g near -64 per token) and mild decays, and grouped key heads; the SIMT forward
    agrees as well."""
    x = _softplus_case(B=2, T=300, H=2, K=128, V=128, initial_state=True, g_mean=g_mean, Hk=Hk, seed=64)
    out, fs = _check_fwd(x, "bf16")
    assert torch.isfinite(out.float()).all() and torch.isfinite(fs).all()
    _check_fwd(x, "bf16", simt=True)


def test_softplus_gate_tensor_core_forward_packed_documents():
    x = _softplus_case(B=1, T=333, H=3, K=128, V=128, varlen=True, initial_state=True, seed=65,
                       lengths=[1, 15, 16, 17, 0, 64, 200, 20])
    _check_fwd(x, "bf16")


# ------------------------------------------------------------------ segment-parallel forward

def _check_segmented(x, segments, dtype="bf16"):
    import gated_delta_rule_sm_gb300 as kda
    names = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")
    out, fs = kda.forward(*[x[n] for n in names], scale=x["scale"], lower_bound=x["lower_bound"],
                          gate=x.get("gate", "lower_bounded"), initial_state=x.get("initial_state"),
                          cu_seqlens=x.get("cu_seqlens"), output_final_state=True, segments=segments)
    torch.cuda.synchronize()
    assert device_status() == 0
    r_out, r_fs = oracle_fwd(x)
    e, e2 = rel_err(out, r_out, dtype), rel_err(fs, r_fs, dtype)
    assert e <= tol(dtype) and e2 <= tol(dtype), (segments, e, e2)
    return out, fs


@pytest.mark.parametrize("segments", [1, 3, 16, 100])
def test_segmented_forward_matches_the_oracle(segments):
    """Mild gates (g_raw ~ N(-4, 1)) so the entering states carry across many pieces; T = 1000 leaves a
    40-token tail; 100 segments ask for more pieces than the 16 chunks."""
    w = Workload("t", B=1, T=1000, H=2, K=128, V=128, initial_state=True, g_mean=-4.0, seed=70)
    _check_segmented(make_inputs(w, device=DEV), segments)


def test_segmented_forward_rows_heads_and_plain_agree():
    w = Workload("t", B=2, T=333, H=3, K=128, V=128, initial_state=True, g_mean=-3.0, seed=71)
    x = make_inputs(w, device=DEV)
    out, fs = _check_segmented(x, 4)
    o2, f2 = gpu_fwd(x)
    assert rel_err(out, f64(o2), "bf16") <= 2e-2 and rel_err(fs, f64(f2), "bf16") <= 2e-2


def test_segmented_forward_softplus_gate():
    x = _softplus_case(B=1, T=700, H=2, K=128, V=128, initial_state=True, g_mean=-6.0, seed=72)
    _check_segmented(x, 5)


def test_segmented_forward_packed_documents():
    """Documents of 0 to 700 tokens, each with its own initial state: a document gets as many pieces
    as its length needs (none when empty), and states never cross a document boundary."""
    lens = [700, 0, 1, 64, 65, 300, 17]
    w = Workload("t", B=1, T=sum(lens), H=2, K=128, V=128, varlen=True, initial_state=True, g_mean=-4.0,
                 seed=74)
    x = make_inputs(w, device=DEV, lengths=lens)
    for segments in (2, 5, 100):
        _check_segmented(x, segments)


def test_segmented_forward_long_row_few_heads():
    """The case the schedule is for: one 65536-token row on two heads (the long-context workload's
    distributions), 16 pieces; and a mild-gate row of 8192 tokens cut into 64-token pieces."""
    w = Workload("t", B=1, T=65536, H=2, K=128, V=128, initial_state=True, seed=73)
    _check_segmented(make_inputs(w, device=DEV), 16)
    w = Workload("t", B=1, T=8192, H=2, K=128, V=128, initial_state=True, g_mean=-4.0, seed=73)
    _check_segmented(make_inputs(w, device=DEV), 128)


# ------------------------------------------------------------------ segment-parallel backward

@pytest.mark.parametrize("segments", [1, 3, 16])
def test_segmented_backward_matches_the_oracle(segments):
    """Both state chains of the backward cut into pieces: mild gates so that the states and their
    gradients carry across pieces, an initial state and a final-state gradient, a 60-token tail."""
    w = Workload("t", B=1, T=700, H=2, K=128, V=128, initial_state=True, backward=True, g_mean=-4.0, seed=80)
    x = make_inputs(w, device=DEV)
    dfinal = 0.05 * torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(80)).to(DEV)
    _check_bwd(x, "bf16", dfinal=dfinal, segments=segments)


def test_segmented_backward_rows_and_plain_agree():
    """Two rows, three heads: every gradient agrees with the oracle and with kda_bwd."""
    w = Workload("t", B=2, T=333, H=3, K=128, V=128, initial_state=True, backward=True, g_mean=-3.0, seed=81)
    x = make_inputs(w, device=DEV)
    dfinal = 0.05 * torch.randn((2, 3, 128, 128), generator=torch.Generator().manual_seed(81)).to(DEV)
    g = _check_bwd(x, "bf16", dfinal=dfinal, segments=4)
    g0 = gpu_bwd(x, dfinal=dfinal)
    torch.cuda.synchronize()
    for n in GRADS:
        assert rel_err(g[n], f64(g0[n]), "bf16") <= 2e-2, n


def test_segmented_backward_packed_documents():
    lens = [300, 0, 1, 64, 200, 17]
    w = Workload("t", B=1, T=sum(lens), H=2, K=128, V=128, varlen=True, initial_state=True, backward=True,
                 g_mean=-4.0, seed=82)
    x = make_inputs(w, device=DEV, lengths=lens)
    dfinal = 0.05 * torch.randn((len(lens), 2, 128, 128), generator=torch.Generator().manual_seed(82)).to(DEV)
    for segments in (3, 40):
        _check_bwd(x, "bf16", dfinal=dfinal, segments=segments)


def test_segmented_backward_softplus_gate():
    x = _softplus_case(B=1, T=500, H=2, K=128, V=128, initial_state=True, g_mean=-6.0, seed=83, backward=True)
    _check_bwd(x, "bf16", segments=4)


def test_segmented_backward_long_row_few_heads():
    """One 8192-token row on two heads cut into 16 pieces (the backward workload's distributions),
    against the oracle on one head."""
    w = Workload("t", B=1, T=8192, H=2, K=128, V=128, initial_state=True, backward=True, seed=84)
    x = make_inputs(w, device=DEV)
    dfinal = 0.05 * torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(84)).to(DEV)
    g = gpu_bwd(x, dfinal=dfinal, segments=16)
    torch.cuda.synchronize()
    assert device_status() == 0
    heads = [1]
    r = oracle_bwd(head_slice(x, heads), dfinal=dfinal[:, heads])
    for n in ("dq", "dk", "dv", "dg_raw", "dbeta_raw"):
        assert rel_err(g[n][:, :, heads], r[n], "bf16") <= 2e-2, n
    assert rel_err(g["dinitial_state"][:, heads], r["dinitial_state"], "bf16") <= 2e-2
    assert rel_err(g["da_log"][heads], r["da_log"], "bf16") <= 2e-2


def test_unaligned_state_buffers_take_the_simt_path():
    """fp32 states at an address that is not a multiple of 16 bytes: the tensor-core path moves states
    16 bytes at a time, so kda_fwd / kda_bwd run such calls on the SIMT path, still against the
    oracle, and the segmented entry refuses them."""
    import gated_delta_rule_sm_gb300 as kda
    from gated_delta_rule_sm_gb300._lib import KdaError
    w = Workload("t", B=1, T=150, H=2, K=128, V=128, initial_state=True, backward=True, seed=85)
    x = make_inputs(w, device=DEV)
    n = x["initial_state"].numel()
    buf = torch.empty(n + 1, dtype=torch.float32, device=DEV)
    buf[1:].copy_(x["initial_state"].reshape(-1))
    x["initial_state"] = buf[1:].view_as(x["initial_state"])      # 4 bytes past a 16-byte boundary
    assert x["initial_state"].data_ptr() % 16 == 4
    names = _launched(lambda: _check_fwd(x, "bf16"))
    assert "kda_intra_tc" not in names and "kda_chain_fwd_simt" in names, names
    names = _launched(lambda: _check_bwd(x, "bf16"))
    assert "kda_grad_tc" not in names and "kda_grad_simt" in names, names
    with pytest.raises(KdaError):
        gpu_fwd(x, segments=2)


@pytest.mark.parametrize("case", ["k64", "segmented"])
def test_backward_without_states(case):
    """No initial state, no final-state gradient and no initial-state gradient requested: the K = 64
    tensor-core backward pads nothing, and the segmented backward's combines start from zero and
    write no row result."""
    import gated_delta_rule_sm_gb300 as kda
    D = 64 if case == "k64" else 128
    x = make_inputs(Workload("t", B=2, T=260, H=2, K=D, V=D, backward=True, seed=89), device=DEV)
    names = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")
    g = kda.backward(*[x[n] for n in names], x["dout"], scale=x["scale"], lower_bound=x["lower_bound"],
                     want_dinitial_state=False, segments=3 if case == "segmented" else 0)
    torch.cuda.synchronize()
    assert device_status() == 0
    assert g["dinitial_state"] is None
    r = oracle_bwd(x)
    for n in ("dq", "dk", "dv", "dg_raw", "dbeta_raw", "da_log", "ddt_bias"):
        assert rel_err(g[n], r[n], "bf16") <= tol("bf16"), n
