"""The e4m3 Q/K path (fa_fwd_qk8): S = Q K^T as an e4m3 product on the
tensor cores, P V in bf16.  The oracle takes Q and K as the exact e4m3
values times their descale factors, so the tolerances are those of the
bf16 path: max |dO| <= 2e-2, mean |dO| <= 2e-3, max |dLSE| <= 1e-3."""

import math

import pytest
import torch

import oracle
from exact_io_aware_fa2_gb300 import build as fabuild
from exact_io_aware_fa2_gb300 import fa
from exact_io_aware_fa2_gb300.workloads import (WORKLOADS, make_inputs,
                                                make_qk8_inputs, quantize_e4m3)

MAX_DO, MEAN_DO, MAX_DLSE = 2e-2, 2e-3, 1e-3
P = 1 << 20  # a 16-byte-aligned stand-in address; never dereferenced


@pytest.fixture(scope="module")
def lib():
    import os
    if not os.path.exists(fabuild.LIB_PATH):
        fabuild.build()
    return fa.load()


def _raw(**kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, Hq=2, Hkv=1, Nq=128, Nkv=128,
             D=128, scale=0.125, qd=0.01, kd=0.02, causal=0, stream=0)
    a.update(kw)
    return fa.fwd_qk8_raw(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"],
                          a["Hq"], a["Hkv"], a["Nq"], a["Nkv"], a["D"],
                          a["scale"], a["qd"], a["kd"], a["causal"],
                          a["stream"])


@pytest.mark.parametrize("kw", [dict(qd=0.0), dict(kd=-1.0),
                                dict(qd=float("nan")), dict(kd=float("inf")),
                                dict(q=0), dict(Nkv=0)])
def test_qk8_invalid_values_rejected(lib, kw):
    assert _raw(**kw) == 1  # FA_ERR_INVALID_VALUE


@pytest.mark.parametrize("D", [64, 192, 256])
def test_qk8_other_head_dims_unsupported(lib, D):
    assert _raw(D=D) == 2  # FA_ERR_UNSUPPORTED


def test_e4m3_oracle_inputs_are_exact():
    # the oracle's view of the inputs: e4m3 values are exact in float64
    q8, k8, v, qd, kd = make_qk8_inputs(1, 1, 1, 64, 64, 128, seed=1)
    x = q8.to(torch.float64)
    assert torch.equal(x.to(torch.float8_e4m3fn).to(torch.float64), x)
    assert 0 < qd and 0 < kd and x.abs().max() <= 448


def _compare(shape, causal, seed, q_std=1.0):
    B, Hq, Hkv, Nq, Nkv, D = shape
    q8, k8, v, qd, kd = make_qk8_inputs(B, Hq, Hkv, Nq, Nkv, D, seed=seed,
                                        q_std=q_std)
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.fwd_qk8(q8.cuda(), k8.cuda(), v.cuda(), scale=scale,
                        q_descale=qd, k_descale=kd, causal=causal)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    O, L = oracle.attention_fp64(q8.to(torch.float64) * qd,
                                 k8.to(torch.float64) * kd, v, scale, causal)
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    dO = (o.double() - O).abs()
    dL = (lse.double() - L).abs()
    msg = (f"{shape} c{causal}: max|dO|={dO.max():.3e} "
           f"mean|dO|={dO.mean():.3e} max|dLSE|={dL.max():.3e}")
    assert dO.max() <= MAX_DO, msg
    assert dO.mean() <= MEAN_DO, msg
    assert dL.max() <= MAX_DLSE, msg
    return msg


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 1, 128),
                                   (1, 2, 1, 384, 640, 128),
                                   (1, 2, 2, 129, 1000, 128),
                                   (2, 8, 2, 333, 1000, 128),
                                   (1, 4, 2, 100, 5000, 128)])
def test_qk8_parity(shape, causal):
    print(_compare(shape, causal, seed=sum(shape)))


@pytest.mark.gpu
def test_qk8_large_logits():
    print(_compare((1, 4, 4, 500, 3000, 128), True, seed=9, q_std=3.0))


@pytest.mark.gpu
@pytest.mark.parametrize("name", [n for n in WORKLOADS if WORKLOADS[n].qk8])
def test_qk8_workload_full_size_sampled(name):
    """The e4m3 workloads at full size, on sampled rows of every head."""
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    (q8, qd), (k8, kd) = quantize_e4m3(q), quantize_e4m3(k)
    o, lse = fa.fwd_qk8(q8.cuda(), k8.cuda(), v.cuda(), scale=w.scale,
                        q_descale=qd, k_descale=kd, causal=w.causal)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    q64, k64 = q8.to(torch.float64) * qd, k8.to(torch.float64) * kd
    gen = torch.Generator().manual_seed(0)
    for b in range(w.B):
        for h in range(w.Hq):
            rows = sorted({0, 127, 128, w.Nq - 1} |
                          set(torch.randint(0, w.Nq, (12,),
                                            generator=gen).tolist()))
            O, L = oracle.attention_rows_fp64(q64, k64, v, w.scale, w.causal,
                                              b, h, rows)
            dO = (o[b, h, rows].double() - O).abs()
            dL = (lse[b, h, rows].double() - L).abs()
            assert dO.max() <= MAX_DO and dO.mean() <= MEAN_DO
            assert dL.max() <= MAX_DLSE
