"""The MXFP8 path (fa_fwd_mxfp8): e4m3 Q and K with one power-of-two scale
per 32 head-dim elements, S = Q K^T as a block-scaled tensor-core product.

The oracle takes the exact values the MXFP8 inputs stand for (e4m3 value
times 2^(scale - 127), exact in float64), so the bf16 path's tolerances
apply unchanged: max |dO| <= 2e-2, mean |dO| <= 2e-3, max |dLSE| <= 1e-3.
The quantisation error itself (against the oracle on the bf16 inputs the
MXFP8 ones were made from) is printed, not asserted: it is the input
format's, not the kernel's.
"""

import math

import pytest
import torch

import oracle
from exact_io_aware_fa2_gb300 import fa
from exact_io_aware_fa2_gb300.workloads import (WORKLOADS, dequantize_mxfp8,
                                                make_inputs, make_mxfp8_inputs,
                                                quantize_mxfp8)

MAX_DO, MEAN_DO, MAX_DLSE = 2e-2, 2e-3, 1e-3


def _check(o, lse, O, L, what):
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all(), what
    dO = (o.double() - O).abs()
    dL = (lse.double() - L).abs()
    msg = (f"{what}: max|dO|={dO.max():.3e} mean|dO|={dO.mean():.3e} "
           f"max|dLSE|={dL.max():.3e}")
    assert dO.max() <= MAX_DO, msg
    assert dO.mean() <= MEAN_DO, msg
    assert dL.max() <= MAX_DLSE, msg
    return msg


def _run(q8, k8, v, qs, ks, scale, causal):
    args = [t.cuda() for t in (q8, k8, v, qs, ks)]
    o, lse = fa.fwd_mxfp8(*args, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    return o.cpu(), lse.cpu()


@pytest.mark.gpu
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,causal", [
    (1, 1, 1, 128, 128, False),
    (1, 2, 1, 300, 1000, False),
    (1, 2, 1, 1000, 300, True),
    (1, 2, 2, 127, 129, True),
    (2, 8, 2, 333, 333, True),        # GQA, ragged, batch
    (2, 8, 2, 333, 333, False),
    (1, 2, 1, 1, 700, False),         # one query row
    (1, 2, 1, 257, 1, False),         # one key
])
def test_mxfp8_parity(B, Hq, Hkv, Nq, Nkv, causal):
    q8, k8, v, qs, ks = make_mxfp8_inputs(B, Hq, Hkv, Nq, Nkv, 128,
                                          seed=Nq + 3 * Nkv)
    scale = 1.0 / math.sqrt(128)
    o, lse = _run(q8, k8, v, qs, ks, scale, causal)
    O, L = oracle.attention_fp64(dequantize_mxfp8(q8, qs),
                                 dequantize_mxfp8(k8, ks), v, scale, causal)
    print(_check(o, lse, O, L, f"mx {B}x{Hq}/{Hkv} {Nq}x{Nkv} c{causal}"))


@pytest.mark.gpu
@pytest.mark.parametrize("scale", [0.0, -0.2])
def test_mxfp8_zero_and_negative_scale(scale):
    q8, k8, v, qs, ks = make_mxfp8_inputs(1, 2, 2, 256, 384, 128, seed=5)
    o, lse = _run(q8, k8, v, qs, ks, scale, True)
    O, L = oracle.attention_fp64(dequantize_mxfp8(q8, qs),
                                 dequantize_mxfp8(k8, ks), v, scale, True)
    print(_check(o, lse, O, L, f"mx scale {scale}"))


@pytest.mark.gpu
def test_mxfp8_large_logits_and_varied_block_scales():
    """Rows whose 32-element blocks have very different magnitudes (so the
    four scale bytes of a row differ) and large logits."""
    q8, k8, v, qs, ks = make_mxfp8_inputs(1, 4, 2, 500, 1200, 128, seed=7,
                                          q_std=3.0)
    q = dequantize_mxfp8(q8, qs)
    k = dequantize_mxfp8(k8, ks)
    q[..., 32:64] *= 16.0
    k[..., 96:128] *= 1 / 64.0
    k[:, :, ::97] *= 8.0
    q8, qs = quantize_mxfp8(q)
    k8, ks = quantize_mxfp8(k)
    assert (qs[..., 1].int() - qs[..., 0].int()).abs().float().mean() >= 3
    scale = 1.0 / math.sqrt(128)
    for causal in (False, True):
        o, lse = _run(q8, k8, v, qs, ks, scale, causal)
        O, L = oracle.attention_fp64(dequantize_mxfp8(q8, qs),
                                     dequantize_mxfp8(k8, ks), v, scale,
                                     causal)
        print(_check(o, lse, O, L, f"mx varied scales c{causal}"))


@pytest.mark.gpu
def test_mxfp8_headline_shape_sampled_and_quantisation_error():
    """The pages' 4096 x 8192 shape with MXFP8 Q and K: sampled rows of every
    head against the oracle on the dequantised inputs, and the separate
    error of the MXFP8 inputs against the bf16 ones they came from."""
    w = WORKLOADS["mxfp8_b1_h8_q4096_kv8192_d128"]
    q, k, v = make_inputs(w)
    q8, qs = quantize_mxfp8(q)
    k8, ks = quantize_mxfp8(k)
    o, lse = _run(q8, k8, v, qs, ks, w.scale, w.causal)
    qd, kd = dequantize_mxfp8(q8, qs), dequantize_mxfp8(k8, ks)
    gen = torch.Generator().manual_seed(0)
    for h in range(w.Hq):
        rows = sorted({0, 1, 127, 128, 2047, 4095} |
                      set(torch.randint(0, w.Nq, (10,), generator=gen)
                          .tolist()))
        O, L = oracle.attention_rows_fp64(qd, kd, v, w.scale, False, 0, h,
                                          rows)
        msg = _check(o[0, h, rows], lse[0, h, rows], O, L, f"mx head {h}")
        Ob, Lb = oracle.attention_rows_fp64(q, k, v, w.scale, False, 0, h,
                                            rows)
        if h == 0:
            print(msg)
            print(f"quantisation error vs bf16 inputs: max|dO|="
                  f"{(o[0, h, rows].double() - Ob).abs().max():.3e} "
                  f"max|dLSE|={(lse[0, h, rows].double() - Lb).abs().max():.3e}")


# ------------------------------------------------------------ input recipe

def test_quantizer_picks_the_smallest_power_of_two_scale():
    """Every 32-element block gets the smallest 2^e with amax / 2^e <= 448,
    the e4m3 values stay within 448, and an all-zero block gets byte 0."""
    g = torch.Generator().manual_seed(3)
    x = torch.randn(3, 5, 128, generator=g) * torch.exp2(
        torch.randint(-20, 20, (3, 5, 128), generator=g).float() / 4)
    x[0, 0, :32] = 0
    q8, s = quantize_mxfp8(x)
    assert q8.dtype == torch.float8_e4m3fn and s.dtype == torch.uint8
    assert s.shape == (3, 5, 4)
    e = s.double() - 127
    amax = x.double().reshape(3, 5, 4, 32).abs().amax(-1)
    nz = amax > 0
    assert (amax[nz] / torch.exp2(e[nz]) <= 448).all()
    assert (amax[nz] / torch.exp2(e[nz] - 1) > 448).all()     # smallest
    assert s[0, 0, 0] == 0 and (q8[0, 0, :32].float() == 0).all()
    assert q8.float().abs().max() <= 448


def test_dequantize_reproduces_representable_values_exactly():
    """Values that are e4m3 numbers times a power of two come back exactly:
    here each block holds a multiple of 2^k of {+-1, +-1.5, ..., +-448}."""
    g = torch.Generator().manual_seed(4)
    base = torch.tensor([1.0, -1.5, 1.75, -2.5, 448.0, -0.015625, 3.0, 0.0])
    idx = torch.randint(0, len(base), (2, 3, 64), generator=g)
    x = base[idx] * torch.exp2(torch.tensor([-8.0, 3.0]).repeat(1, 1, 1)
                               .repeat_interleave(32, -1))
    q8, s = quantize_mxfp8(x)
    assert torch.equal(dequantize_mxfp8(q8, s), x.double())


def test_quantize_then_dequantize_is_within_e4m3_rounding():
    """Round to nearest e4m3 (3 mantissa bits): relative error at most
    2^-4 for values at least 2^-6 of their block's scale (the normal range),
    absolute error at most 2^-10 of the scale below it."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn(4, 256, generator=g).to(torch.bfloat16).float()
    q8, s = quantize_mxfp8(x)
    d = dequantize_mxfp8(q8, s)
    scale = torch.exp2(s.double() - 127).repeat_interleave(32, -1)
    err = (d - x.double()).abs()
    normal = x.double().abs() >= scale * 2 ** -6
    assert (err[normal] <= x.double().abs()[normal] * 2 ** -4).all()
    assert (err[~normal] <= scale[~normal] * 2 ** -10).all()
