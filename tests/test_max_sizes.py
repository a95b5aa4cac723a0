"""GPU parity at the size limits of the boundary: grid dimensions at 65535,
a million keys (split-KV and the wide-head kernel), and tensors of 2^29 and
2^31 elements (64-bit indexing).  Outputs are compared with the fp64 oracle
on sampled (batch, head, row) triples, on host copies of the same inputs.
Tolerances as in test_parity: max |dO| <= 2e-2, mean |dO| <= 2e-3,
max |dLSE| <= 1e-3."""

import math

import pytest
import torch

import oracle
from exact_io_aware_fa2_gb300 import fa
from exact_io_aware_fa2_gb300.workloads import make_custom_on_device

pytestmark = pytest.mark.gpu

MAX_DO, MEAN_DO, MAX_DLSE = 2e-2, 2e-3, 1e-3


def _check_sampled(q, k, v, o, lse, scale, causal, heads, rows):
    B, Hq, Nq, D = q.shape
    Hkv = k.shape[1]
    for b, h in heads:
        hk = h // (Hq // Hkv)
        qs = q[b:b + 1, h:h + 1].cpu()
        ks = k[b:b + 1, hk:hk + 1].cpu()
        vs = v[b:b + 1, hk:hk + 1].cpu()
        O, L = oracle.attention_rows_fp64(qs, ks, vs, scale, causal, 0, 0,
                                          rows)
        got = o[b, h, rows].cpu().double()
        gl = lse[b, h, rows].cpu().double()
        dO = (got - O).abs()
        dL = (gl - L).abs()
        msg = (f"b{b} h{h}: max|dO|={dO.max():.3e} mean|dO|={dO.mean():.3e} "
               f"max|dLSE|={dL.max():.3e}")
        assert dO.max() <= MAX_DO, msg
        assert dO.mean() <= MEAN_DO, msg
        assert dL.max() <= MAX_DLSE, msg
    return msg


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,causal", [
    (65535, 1, 1, 1, 3, 64, False),            # grid z at its limit
    (1, 65535, 1, 2, 5, 64, True),             # grid y at its limit
    (1, 65535, 1, 2, 5, 64, False),            # the same heads packed (GQA)
    (1, 8, 1, 1, 1 << 20, 128, False),         # a million keys: split-KV
    (1, 2, 1, 3, 1 << 20, 256, False),         # a million keys: wide kernel
    (1, 16, 16, 1 << 18, 1 << 18, 128, True),  # 2^29-element tensors
    (1, 16, 16, 1 << 20, 1 << 20, 128, True),  # 2^31 elements: 64-bit offsets
])
def test_maximum_sizes_sampled(B, Hq, Hkv, Nq, Nkv, D, causal):
    q, k, v = make_custom_on_device(B, Hq, Hkv, Nq, Nkv, D,
                                    seed=Nq + 7 * Nkv + D)
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.fwd(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    assert torch.isfinite(lse).all()
    gen = torch.Generator().manual_seed(1)
    heads = sorted({(0, 0), (B - 1, Hq - 1), (B // 2, Hq // 2)})
    rows = sorted({0, Nq - 1, Nq // 2} |
                  set(torch.randint(0, Nq, (5,), generator=gen).tolist()))
    print(_check_sampled(q, k, v, o, lse, scale, causal, heads, rows))
    # every output row is finite (checked on the device, chunked by batch)
    for b0 in range(0, B, 4096):
        assert torch.isfinite(o[b0:b0 + 4096].float()).all()


def test_host_path_with_more_groups_than_four_chunks_of_the_grid_limit():
    """fa_fwd_host cuts the job into chunks of (batch, kv head) groups and
    runs each chunk with B = its group count; with 65535 x 8 groups four
    chunks would pass the grid's 65535 limit, so it uses more.  With one key
    per head every output row is that key's value row exactly, and the LSE
    is scale * q . k (closed forms of softmax over one key)."""
    B, H, D = 65535, 8, 64
    gen = torch.Generator().manual_seed(5)
    q = torch.randn(B, H, 1, D, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, H, 1, D, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, H, 1, D, generator=gen).to(torch.bfloat16)
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    o, lse = fa.fwd_host(qp, kp, vp, scale=0.125, causal=False)
    assert torch.equal(o, v)
    ref = (q.double() * k.double()).sum(-1) * 0.125
    assert (lse.double() - ref).abs().max() <= 1e-3
