"""GPU parity of the stream schedule (fa_fwd_stream.cuh) against the fp64
oracle, and its hand-off of partials between CTAs.

In the stream schedule every CTA takes an equal contiguous run of all
(tile pair, K/V block) items; a pair cut between CTAs is finished by the CTA
holding its last block, which combines the others' fp32 partials.  The
parity tests force the schedule (fa_set_schedule) so that small shapes run
it; on the 152-SM GB300 the shapes below exercise pairs cut into three
pieces (two partials per merger) and into 24 (23 partials), CTAs with four
segments (writer, whole pairs, merger), ragged query rows and keys, packed
grouped-query heads with pairs whose second tile is absent, pairs that never
have one (their softmax warps idle through every segment), and both head
dims of the two-tile kernel.  Each case checks that the call really runs
the stream schedule, then compares the whole output element by element with
the oracle (same tolerances as test_parity.py).  The automatic choice between
the schedules is checked on the CPU (test_schedule.py).
"""

import math

import pytest
import torch

import oracle
from exact_io_aware_fa2_gb300 import fa
from exact_io_aware_fa2_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu

MAX_DO, MEAN_DO, MAX_DLSE = 2e-2, 2e-3, 1e-3

# (B, Hq, Hkv, Nq, Nkv, D, what it exercises)
CASES = [
    (1, 100, 100, 200, 1300, 128, "3-piece pairs, ragged rows and keys"),
    (1, 100, 100, 200, 1300, 64, "3-piece pairs at D64"),
    (5, 100, 100, 256, 200, 64, "four segments per CTA"),
    (2, 48, 6, 300, 3000, 128, "packed GQA, pairs without a second tile"),
    (1, 300, 300, 256, 100, 128, "one block per pair: whole pairs only"),
    (500, 1, 1, 100, 300, 64, "no second tile in any pair, cut pairs"),
    (1, 2, 2, 256, 3000, 128, "24 pieces per pair, one block per CTA"),
]


def _needs_gb300_sm_count():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip(f"schedules chosen for 152 SMs, device has {sms}")


@pytest.fixture
def forced_stream():
    fa.set_schedule("stream")
    try:
        yield
    finally:
        fa.set_schedule("auto")


def _check(o, lse, O, L, what):
    assert torch.isfinite(o.float()).all(), f"{what}: non-finite O"
    assert torch.isfinite(lse).all(), f"{what}: non-finite LSE"
    dO = (o.double() - O).abs()
    dL = (lse.double() - L).abs()
    msg = (f"{what}: max|dO|={dO.max():.3e} mean|dO|={dO.mean():.3e} "
           f"max|dLSE|={dL.max():.3e}")
    assert dO.max() <= MAX_DO, msg
    assert dO.mean() <= MEAN_DO, msg
    assert dL.max() <= MAX_DLSE, msg
    return msg


@pytest.mark.parametrize("case", CASES, ids=[c[-1] for c in CASES])
def test_stream_schedule_parity(case, forced_stream):
    B, Hq, Hkv, Nq, Nkv, D, what = case
    _needs_gb300_sm_count()
    sch = fa.schedule(B, Hq, Hkv, Nq, Nkv, D, False)
    assert sch["kind"] == "stream", sch
    q, k, v = make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=Nq + Nkv + D)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.fwd(qd, kd, vd, scale=scale, causal=False)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    O, L = oracle.attention_fp64(q, k, v, scale, False)
    print(_check(o.cpu(), lse.cpu(), O, L, f"{what} {sch}"))


@pytest.mark.parametrize("boost", ["early keys", "late keys"])
@pytest.mark.parametrize("scale", [0.088, -0.2])
def test_stream_pieces_with_far_apart_maxima(boost, scale, forced_stream):
    """Pieces of a pair whose reference maxima differ by far more than the
    lazy-rescale threshold: the keys of the first five blocks (held by
    writers) or of the rest (mostly the mergers') are scaled by 4, so the
    merge weights 2^(m_k - M) are far from 1 in both directions.  V is
    scaled by 1/4 so that |O| stays where bf16 rounding of the output is
    well inside the tolerance (both scalings are exact in bf16)."""
    _needs_gb300_sm_count()
    B, Hq, Hkv, Nq, Nkv, D = 1, 100, 100, 200, 1300, 128
    assert fa.schedule(B, Hq, Hkv, Nq, Nkv, D, False)["kind"] == "stream"
    q, k, v = make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=31)
    if boost == "early keys":
        k[:, :, :640] *= 4
    else:
        k[:, :, 640:] *= 4
    v *= 0.25
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.fwd(qd, kd, vd, scale=scale, causal=False)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    O, L = oracle.attention_fp64(q, k, v, scale, False)
    print(_check(o.cpu(), lse.cpu(), O, L, f"{boost} scale {scale}"))


def test_stream_repeatable_and_noalloc_identical(forced_stream):
    """Two calls (different epochs) and the no-alloc entry point give
    bit-identical O and LSE: the result does not depend on which launch's
    flags or scratch a merger sees."""
    _needs_gb300_sm_count()
    B, Hq, Hkv, Nq, Nkv, D = 2, 48, 6, 300, 3000, 128
    q, k, v = (t.cuda() for t in make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=3))
    o1, l1 = fa.fwd(q, k, v, scale=0.088, causal=False)
    o2, l2 = fa.fwd(q, k, v, scale=0.088, causal=False)
    o3 = torch.empty_like(o1)
    l3 = torch.empty_like(l1)
    st = fa.fwd_noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                            o3.data_ptr(), l3.data_ptr(), B, Hq, Hkv, Nq,
                            Nkv, D, 0.088, False,
                            torch.cuda.current_stream().cuda_stream)
    assert st == 0, fa.status_string(st)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_stream_workspace_size(forced_stream):
    """One fp32 slot of 256 x (D + 3) words (O, m, and two row sums) and
    eight 8-byte flags per CTA."""
    _needs_gb300_sm_count()
    for B, Hq, Hkv, Nq, Nkv, D, _ in CASES:
        sch = fa.schedule(B, Hq, Hkv, Nq, Nkv, D, False)
        want = sch["ctas"] * (256 * (D + 3) * 4 + 8 * 8)
        assert fa.workspace_size(B, Hq, Hkv, Nq, Nkv, D, False) == want


def test_stream_graph_replay_with_new_inputs(forced_stream):
    """A launch captured once (one epoch) and replayed: each replay's
    mergers wait for that replay's writers, because each merger clears the
    flags it consumed.  Inputs change between replays; every replay must
    match an eager call on the same inputs bit for bit."""
    _needs_gb300_sm_count()
    B, Hq, Hkv, Nq, Nkv, D = 1, 100, 100, 200, 1300, 128
    assert fa.schedule(B, Hq, Hkv, Nq, Nkv, D, False)["kind"] == "stream"
    scale = 1.0 / math.sqrt(D)
    q, k, v = (t.cuda() for t in make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=1))
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, Nq, device="cuda", dtype=torch.float32)
    ws_bytes = fa.workspace_size(B, Hq, Hkv, Nq, Nkv, D, False)
    ws = torch.empty(ws_bytes, device="cuda", dtype=torch.uint8)

    def call(stream):
        return fa.fwd_ws_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                             o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Nq,
                             Nkv, D, scale, False, ws.data_ptr(), ws_bytes,
                             stream)

    assert call(torch.cuda.current_stream().cuda_stream) == 0   # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            st = call(side.cuda_stream)
    assert st == 0, fa.status_string(st)
    for seed in (11, 12, 13):
        nq, nk, nv = make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=seed)
        q.copy_(nq)
        k.copy_(nk)
        v.copy_(nv)
        g.replay()
        torch.cuda.synchronize()
        assert fa.last_device_error() == 0
        o_graph, l_graph = o.clone(), lse.clone()
        o_eager, l_eager = fa.fwd(q, k, v, scale=scale, causal=False)
        torch.cuda.synchronize()
        assert torch.equal(o_graph, o_eager), f"replay seed {seed}"
        assert torch.equal(l_graph, l_eager), f"replay seed {seed}"


def test_forced_plain_disables_split_and_stream():
    fa.set_schedule("plain")
    try:
        assert fa.schedule(1, 8, 8, 128, 32768, 128, False)["kind"] == "plain"
        assert fa.workspace_size(1, 8, 8, 128, 32768, 128, False) == 0
        q, k, v = (t.cuda() for t in make_custom(1, 4, 2, 100, 700, 64, seed=2))
        o, lse = fa.fwd(q, k, v, scale=0.125, causal=False)
        torch.cuda.synchronize()
        O, L = oracle.attention_fp64(q.cpu(), k.cpu(), v.cpu(), 0.125, False)
        print(_check(o.cpu(), lse.cpu(), O, L, "forced plain"))
    finally:
        fa.set_schedule("auto")


@pytest.mark.parametrize("shape", [(2, 32, 8, 256, 16384, 128),
                                   (2, 16, 4, 512, 16384, 64)])
def test_auto_stream_in_place_of_multiwave_split(shape):
    """Grouped-query shapes with few tile pairs whose split-KV pieces would
    need more than one wave run the stream schedule by themselves (no forced
    setting): packed GQA heads, 54 blocks per CTA; sampled heads against the
    oracle."""
    _needs_gb300_sm_count()
    B, Hq, Hkv, Nq, Nkv, D = shape
    assert fa.schedule(B, Hq, Hkv, Nq, Nkv, D, False)["kind"] == "stream"
    q, k, v = make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=Nq + Hq)
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=False,
                    check=True)
    o, lse = o.cpu(), lse.cpu()
    g = Hq // Hkv
    for b, h in {(0, 0), (0, g), (B - 1, Hq - 1)}:
        O, L = oracle.attention_fp64(q[b:b + 1, h:h + 1],
                                     k[b:b + 1, h // g:h // g + 1],
                                     v[b:b + 1, h // g:h // g + 1], scale,
                                     False)
        print(_check(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], O, L,
                     f"auto stream {shape} b{b} h{h}"))
