"""fa_fwd_noalloc (the forward that allocates nothing) against fa_fwd.

The entry point keeps its split-KV partials in one fixed device array that
every call shares, so the test makes calls in a row on shapes that need that
scratch, and checks each result against fa_fwd (scratch from the library's
pool) within the parity tolerances: max |dO| <= 2e-2, mean |dO| <= 2e-3,
max |dLSE| <= 1e-3.  Collected last, so it runs both alone and after every
other GPU test in one process.
"""

import pytest
import torch

from exact_io_aware_fa2_gb300 import fa
from exact_io_aware_fa2_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu

MAX_DO, MEAN_DO, MAX_DLSE = 2e-2, 2e-3, 1e-3


def _outputs(q):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    return o, lse


def _run(entry, q, k, v, Hkv, scale, causal):
    B, Hq, Nq, D = q.shape
    Nkv = k.shape[2]
    o, lse = _outputs(q)
    st = entry(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
               lse.data_ptr(), B, Hq, Hkv, Nq, Nkv, D, scale, causal,
               torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0, fa.status_string(st)
    assert fa.last_device_error() == 0
    return o, lse


def _compare(shape, seed, causal):
    B, Hq, Hkv, Nq, Nkv, D = shape
    q, k, v = (t.cuda() for t in make_custom(B, Hq, Hkv, Nq, Nkv, D,
                                             seed=seed))
    scale = D ** -0.5
    o_ref, l_ref = _run(fa.fwd_raw, q, k, v, Hkv, scale, causal)
    o, lse = _run(fa.fwd_noalloc_raw, q, k, v, Hkv, scale, causal)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    dO = (o.float() - o_ref.float()).abs()
    dL = (lse - l_ref).abs()
    msg = (f"{shape} causal={causal}: max|dO|={dO.max():.3e} "
           f"mean|dO|={dO.mean():.3e} max|dLSE|={dL.max():.3e}")
    assert dO.max() <= MAX_DO, msg
    assert dO.mean() <= MEAN_DO, msg
    assert dL.max() <= MAX_DLSE, msg
    return msg


# Shapes whose query blocks fill few SMs, so the forward splits the keys and
# uses scratch; each call in a row has a different layout of partials.
SPLIT_SHAPES = [
    ((1, 4, 2, 100, 5000, 128), 31, False),
    ((1, 2, 1, 1100, 1500, 64), 32, True),
    ((1, 4, 2, 100, 5000, 128), 33, False),
]


def test_split_shapes_need_scratch_within_the_limit():
    for (B, Hq, Hkv, Nq, Nkv, D), _, causal in SPLIT_SHAPES:
        need = fa.workspace_size(B, Hq, Hkv, Nq, Nkv, D, causal)
        assert 0 < need <= fa.NOALLOC_SCRATCH_BYTES


def test_calls_in_a_row_match_fa_fwd():
    for shape, seed, causal in SPLIT_SHAPES:
        print(_compare(shape, seed, causal))


def test_calls_leave_device_memory_unchanged():
    """The property the entry point exists for: a call on a shape that needs
    scratch takes no device memory.  After one call of each kind (modules
    loaded, torch's and the pool's memory in place), the free device memory
    reported by the driver is the same before and after two more no-alloc
    calls of split shapes."""
    shape, seed, causal = SPLIT_SHAPES[0]
    B, Hq, Hkv, Nq, Nkv, D = shape
    q, k, v = (t.cuda() for t in make_custom(B, Hq, Hkv, Nq, Nkv, D,
                                             seed=seed))
    o, lse = _outputs(q)
    s = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            lse.data_ptr(), B, Hq, Hkv, Nq, Nkv, D, D ** -0.5, causal, s)
    assert fa.fwd_raw(*args) == 0
    assert fa.fwd_noalloc_raw(*args) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        assert fa.fwd_noalloc_raw(*args) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert fa.last_device_error() == 0
    assert free1 == free0, (free0, free1)


def test_shape_without_scratch_matches_fa_fwd():
    assert fa.workspace_size(1, 8, 8, 4096, 1024, 128, False) == 0
    print(_compare((1, 8, 8, 4096, 1024, 128), 34, False))


def test_invalid_arguments_rejected():
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    p = q.data_ptr()
    assert fa.fwd_noalloc_raw(p, p, p, p, 0, 1, 2, 1, 8, 8, 0, 0.125, False,
                              s) == 1
    assert fa.fwd_noalloc_raw(p, p, p, p, 0, 1, 2, 1, 8, 8, 80, 0.125, False,
                              s) == 2
