"""GPU parity: the sm_103a kernel through the C ABI against the fp64 oracle.

Tolerances (from the specification of this library): max |dO| <= 2e-2,
mean |dO| <= 2e-3 (absolute, against the fp64 O, not a bf16-rounded one)
and max |dLSE| <= 1e-3; any NaN/Inf fails.  Small and medium shapes are
compared element by element over the whole output; the full-size workloads
are compared on sampled rows of every (batch, head) — rows the oracle
computes one by one — plus properties that hold at any size.
"""

import math

import pytest
import torch

import oracle
from exact_io_aware_fa2_gb300 import fa
from exact_io_aware_fa2_gb300.workloads import (WORKLOADS, Workload,
                                                make_custom, make_inputs)

pytestmark = pytest.mark.gpu

MAX_DO, MEAN_DO, MAX_DLSE = 2e-2, 2e-3, 1e-3


def run_gpu(q, k, v, scale, causal):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.fwd(qd, kd, vd, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    return o.cpu(), lse.cpu()


def check(o, lse, O, L, what=""):
    assert torch.isfinite(o.float()).all(), f"{what}: non-finite O"
    assert torch.isfinite(lse).all(), f"{what}: non-finite LSE"
    dO = (o.double() - O).abs()
    dL = (lse.double() - L).abs()
    # the part no bf16 output can avoid: the oracle's own O rounded to bf16
    floor = (O.to(torch.bfloat16).double() - O).abs().max()
    msg = (f"{what}: max|dO|={dO.max():.3e} mean|dO|={dO.mean():.3e} "
           f"max|dLSE|={dL.max():.3e} (oracle O rounded to bf16: max "
           f"{floor:.3e})")
    assert dO.max() <= MAX_DO, msg
    assert dO.mean() <= MEAN_DO, msg
    assert dL.max() <= MAX_DLSE, msg
    return msg


def full_compare(q, k, v, scale, causal, what=""):
    o, lse = run_gpu(q, k, v, scale, causal)
    O, L = oracle.attention_fp64(q, k, v, scale, causal)
    return check(o, lse, O, L, what)


# ------------------------------------------------------------ small / exact

def test_tiny_workload_full():
    w = WORKLOADS["tiny_128_d64"]
    print(full_compare(*make_inputs(w), w.scale, w.causal, w.name))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nkv", [(128, 128), (384, 640), (640, 384),
                                    (1, 1), (1, 300), (127, 129), (129, 127),
                                    (257, 257), (1000, 1000)])
def test_shapes_full(D, causal, Nq, Nkv):
    q, k, v = make_custom(1, 2, 1, Nq, Nkv, D, seed=Nq * 7 + Nkv)
    scale = 1.0 / math.sqrt(D)
    print(full_compare(q, k, v, scale, causal, f"D{D} c{causal} {Nq}x{Nkv}"))


@pytest.mark.parametrize("causal", [False, True])
def test_batched_gqa_ragged(causal):
    q, k, v = make_custom(3, 8, 2, 333, 333, 128, seed=5)
    print(full_compare(q, k, v, 0.0883883, causal, "B3 Hq8 Hkv2 N333"))


def test_mqa_single_kv_head():
    q, k, v = make_custom(2, 6, 1, 200, 700, 64, seed=6)
    print(full_compare(q, k, v, 0.125, False, "MQA Hkv=1"))


@pytest.mark.parametrize("causal", [False, True])
def test_scale_zero_gives_mean_of_visible_v(causal):
    q, k, v = make_custom(1, 2, 2, 300, 300, 64, seed=7)
    o, lse = run_gpu(q, k, v, 0.0, causal)
    O, L = oracle.attention_fp64(q, k, v, 0.0, causal)
    check(o, lse, O, L, "scale 0")
    n = torch.arange(1, 301, dtype=torch.float64) if causal else \
        torch.full((300,), 300.0, dtype=torch.float64)
    assert torch.allclose(lse[0, 0].double(), n.log(), atol=1e-4)


def test_negative_scale():
    q, k, v = make_custom(1, 2, 2, 256, 384, 64, seed=8)
    print(full_compare(q, k, v, -0.2, True, "negative scale"))


def test_identical_keys_and_constant_values():
    q, k, v = make_custom(1, 2, 2, 256, 256, 128, seed=9)
    k = k[:, :, :1].expand_as(k).contiguous()
    o, lse = run_gpu(q, k, v, 0.088, True)
    O, L = oracle.attention_fp64(q, k, v, 0.088, True)
    check(o, lse, O, L, "identical keys")
    vc = v[:, :, :1].expand_as(v).contiguous()
    o2, _ = run_gpu(q, make_custom(1, 2, 2, 256, 256, 128, seed=10)[1], vc,
                    0.088, False)
    # a convex combination of one repeated row returns that row (to bf16)
    ref = vc[:, :, :1].expand_as(o2).float()
    assert (o2.float() - ref).abs().max() <= 1e-2


def test_causal_row0_is_v0():
    q, k, v = make_custom(2, 4, 4, 512, 512, 128, seed=11, q_std=3.0)
    o, lse = run_gpu(q, k, v, 0.0883883, True)
    assert torch.equal(o[:, :, 0], v[:, :, 0])
    ref = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1) * \
        float(torch.tensor(0.0883883, dtype=torch.float32))
    assert (lse[:, :, 0].double() - ref).abs().max() <= 1e-3


def test_deterministic():
    q, k, v = make_custom(1, 4, 4, 1024, 1024, 128, seed=12)
    a = run_gpu(q, k, v, 0.0883883, True)
    b = run_gpu(q, k, v, 0.0883883, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_lse_optional():
    q, k, v = (t.cuda() for t in make_custom(1, 2, 2, 256, 256, 64, seed=13))
    o_ref, _ = fa.fwd(q, k, v, causal=True)
    o, lse = fa.fwd(q, k, v, causal=True, want_lse=False)
    torch.cuda.synchronize()
    assert lse is None and torch.equal(o, o_ref)


def test_host_buffers_path():
    q, k, v = make_custom(1, 2, 2, 300, 500, 128, seed=14)
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    o, lse = fa.fwd_host(qp, kp, vp, scale=0.0883883, causal=False)
    O, L = oracle.attention_fp64(q, k, v, 0.0883883, False)
    check(o.clone(), lse.clone(), O, L, "host buffers")


@pytest.mark.parametrize("causal", [False, True])
def test_host_path_chunks_of_groups(causal):
    """fa_fwd_host cuts the job into at most 4 chunks of (batch, kv head)
    groups (here 12 groups of 3 query heads: chunks of three groups),
    copying each chunk in and out around its own forward; every row must
    land in its place, for GQA, a batch, ragged sizes and the causal mask."""
    q, k, v = make_custom(3, 12, 4, 333, 457, 64, seed=15)
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    o, lse = fa.fwd_host(qp, kp, vp, scale=0.125, causal=causal)
    O, L = oracle.attention_fp64(q, k, v, 0.125, causal)
    print(check(o.clone(), lse.clone(), O, L, f"host chunks causal={causal}"))


def test_host_path_reuses_buffers_and_accepts_pageable_memory():
    bufs = None
    for seed, pin in ((16, True), (17, False)):
        q, k, v = make_custom(2, 8, 2, 256, 700, 128, seed=seed)
        if pin:
            q, k, v = (t.pin_memory() for t in (q, k, v))
        if bufs is None:
            bufs = fa.host_buffers(q, k, v)
        o, lse = fa.fwd_host(q, k, v, scale=0.0883883, causal=False,
                             bufs=bufs)
        O, L = oracle.attention_fp64(q, k, v, 0.0883883, False)
        check(o.clone(), lse.clone(), O, L, f"host reuse seed {seed}")


# ------------------------------------------------------------- full-size

def _sample_rows(Nq, gen, extra=16):
    fixed = {0, 1, 63, 64, 127, 128, 129, Nq // 2, Nq - 129, Nq - 128,
             Nq - 2, Nq - 1}
    rnd = torch.randint(0, Nq, (extra,), generator=gen).tolist()
    return sorted(r for r in fixed.union(rnd) if 0 <= r < Nq)


@pytest.mark.parametrize("name", [n for n in WORKLOADS
                                  if n != "tiny_128_d64"
                                  and not WORKLOADS[n].qk8])
def test_workload_full_size_sampled(name):
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    o, lse = run_gpu(q, k, v, w.scale, w.causal)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    # convexity: every output lies within the range of the value rows
    assert o.float().abs().max() <= v.float().abs().max() + 1e-2
    gen = torch.Generator().manual_seed(0)
    worst = []
    for b in range(w.B):
        for h in range(w.Hq):
            rows = _sample_rows(w.Nq, gen)
            O, L = oracle.attention_rows_fp64(q, k, v, w.scale, w.causal, b, h,
                                              rows)
            worst.append(check(o[b, h, rows], lse[b, h, rows], O, L,
                               f"{name} b{b} h{h}"))
    print(worst[0])


@pytest.mark.parametrize("name", ["pages_b1_h8_q4096_kv8192_d128",
                                  "causal_b4_h16_n2048_d64",
                                  "causal_gqa_b2_hq32_hkv8_n8192_d128",
                                  "causal_b1_h16_n32768_d128_large_logits",
                                  "wide_b1_h8_q4096_kv8192_d256",
                                  "stream_b1_h5_q4096_kv8192_d128"])
def test_workload_full_compare_some_heads(name):
    """Whole heads (the first and the last query head) of the headline,
    causal D=64, causal GQA, long causal large-logit (32768 x 32768, where
    the mean |dO| headroom is smallest), D=256 and stream-schedule
    workloads, element by element against the oracle."""
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    o, lse = run_gpu(q, k, v, w.scale, w.causal)
    group = w.Hq // w.Hkv
    for h in (0, w.Hq - 1):
        hk = h // group
        O, L = oracle.attention_fp64(q[:1, h:h + 1], k[:1, hk:hk + 1],
                                     v[:1, hk:hk + 1], w.scale, w.causal)
        print(check(o[:1, h:h + 1], lse[:1, h:h + 1], O, L, f"{name} h{h}"))


# ------------------------------------------------------ bounded-wait path

def test_bounded_wait_expires_into_status_and_context_survives():
    assert fa.last_device_error() == 0
    assert fa.probe_bounded_wait(2_000_000) == 0    # 2 ms limit
    torch.cuda.synchronize()
    assert fa.last_device_error() == 5              # FA_ERR_TIMEOUT
    assert fa.last_device_error() == 0              # cleared by the read
    # the context is still usable
    w = WORKLOADS["tiny_128_d64"]
    full_compare(*make_inputs(w), w.scale, False, "after probe")


def test_flag_wait_expires_into_status_and_context_survives():
    """The stream schedule's wait for another CTA's partial (acquire loads of
    a global flag) gives up at its limit with FA_ERR_TIMEOUT, like the
    mbarrier waits; nothing faults and the context stays usable."""
    assert fa.last_device_error() == 0
    assert fa.probe_flag_wait(2_000_000) == 0       # 2 ms limit
    torch.cuda.synchronize()
    assert fa.last_device_error() == 5              # FA_ERR_TIMEOUT
    assert fa.last_device_error() == 0
    w = WORKLOADS["tiny_128_d64"]
    full_compare(*make_inputs(w), w.scale, False, "after flag probe")


# ------------------------------------------------ split-KV (few query blocks)

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Nq,Nkv", [(1, 4096), (64, 3000), (200, 2500),
                                    (300, 8192), (128, 640)])
def test_split_kv_full(D, causal, Nq, Nkv):
    """Shapes whose query blocks fill few SMs run split-KV (partials in
    scratch plus a merge kernel); they must match the oracle everywhere."""
    q, k, v = make_custom(1, 2, 1, Nq, Nkv, D, seed=Nq + 3 * Nkv)
    print(full_compare(q, k, v, 1.0 / math.sqrt(D), causal,
                       f"split D{D} c{causal} {Nq}x{Nkv}"))


def test_split_kv_is_used_for_decode_shapes():
    def kind(*shape):
        return fa.schedule(*shape)["kind"]
    assert kind(1, 8, 8, 128, 32768, 128, False) == "split_kv"
    assert kind(1, 2, 1, 1, 4096, 64, False) == "split_kv"
    assert fa.workspace_size(1, 8, 8, 128, 32768, 128, False) > 0
    # causal query row 0 sees one key: nothing worth splitting (the causal
    # shape runs the persistent schedule, which needs no scratch)
    assert kind(1, 2, 1, 1, 4096, 64, True) == "persist"
    assert fa.workspace_size(1, 2, 1, 1, 4096, 64, True) == 0
    w = WORKLOADS["pages_b1_h8_q4096_kv8192_d128"]
    assert kind(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D, w.causal) != "split_kv"


def test_split_kv_large_logits_and_gqa():
    q, k, v = make_custom(2, 8, 2, 150, 6000, 128, seed=21, q_std=3.0)
    k[:, :, ::97] *= 8
    print(full_compare(q, k, v, 0.0883883, True, "split large logits GQA"))


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D", [
    (1, 8, 1, 1, 2000, 128),       # one decode row per head, MQA
    (3, 16, 2, 5, 3000, 128),      # batched GQA, few rows: packed and split
    (2, 12, 4, 130, 700, 64),      # a packed query tile spans two heads
])
def test_gqa_heads_packed_non_causal(B, Hq, Hkv, Nq, Nkv, D):
    """Non-causal GQA runs each group of query heads as one long head; O
    and LSE must land in every head's own rows."""
    q, k, v = make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=Hq * Nq + Nkv)
    print(full_compare(q, k, v, 1.0 / math.sqrt(D), False,
                       f"packed GQA {B}x{Hq}/{Hkv} {Nq}x{Nkv} D{D}"))


# ------------------------------------------------------------ wide heads

@pytest.mark.parametrize("D", [192, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nkv", [(128, 128), (64, 64), (300, 200),
                                    (200, 300), (1, 513), (640, 640)])
def test_wide_heads_full(D, causal, Nq, Nkv):
    """Head dims 192 and 256 run the one-tile kernel with 64-key blocks and
    two score buffers; ragged tails of both sequences included."""
    q, k, v = make_custom(1, 2, 1, Nq, Nkv, D, seed=D + Nq * 3 + Nkv)
    print(full_compare(q, k, v, 1.0 / math.sqrt(D), causal,
                       f"wide D{D} c{causal} {Nq}x{Nkv}"))


@pytest.mark.parametrize("D", [192, 256])
def test_wide_heads_gqa_batched_large_logits(D):
    q, k, v = make_custom(2, 6, 2, 333, 1100, D, seed=D, q_std=3.0)
    k[:, :, ::53] *= 8
    print(full_compare(q, k, v, 1.0 / math.sqrt(D), True,
                       f"wide D{D} GQA large logits causal"))
    print(full_compare(q, k, v, 1.0 / math.sqrt(D), False,
                       f"wide D{D} GQA large logits"))


def test_wide_heads_split_kv_for_few_tiles():
    # few 128-row tiles over long keys: split-KV
    assert fa.workspace_size(1, 8, 8, 128, 32768, 256, False) > 0
    assert fa.workspace_size(1, 8, 2, 1, 4096, 192, False) > 0
    # enough tiles to fill the GPU: no split
    assert fa.workspace_size(1, 8, 8, 4096, 8192, 256, False) == 0


@pytest.mark.parametrize("D", [192, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv", [(1, 2, 1, 64, 5000),
                                              (1, 2, 1, 600, 3000),
                                              (2, 4, 2, 1, 4097)])
def test_wide_heads_split_kv_full(D, causal, B, Hq, Hkv, Nq, Nkv):
    """Wide heads with few query tiles split the keys: partials per K/V
    range, then the merge; compared with the oracle everywhere."""
    q, k, v = make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=D + Nq + Nkv)
    print(full_compare(q, k, v, 1.0 / math.sqrt(D), causal,
                       f"wide split D{D} c{causal} {B}x{Hq}/{Hkv} "
                       f"{Nq}x{Nkv}"))


def test_wide_heads_split_kv_large_logits():
    q, k, v = make_custom(1, 8, 2, 100, 6000, 256, seed=41, q_std=3.0)
    k[:, :, ::97] *= 8
    print(full_compare(q, k, v, 1.0 / 16.0, False, "wide split large logits"))
    print(full_compare(q, k, v, 1.0 / 16.0, True,
                       "wide split large logits causal"))


def test_pool_scratch_and_caller_workspace_agree():
    """fa_fwd (scratch from the library's pool) and fa_fwd_ws (caller's
    workspace) run the same schedule and give identical bits."""
    q, k, v = (t.cuda() for t in make_custom(1, 4, 2, 100, 5000, 128,
                                             seed=15))
    assert fa.workspace_size(1, 4, 2, 100, 5000, 128, False) > 0
    o1, l1 = fa.fwd(q, k, v, scale=0.0883883, causal=False)
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    st = fa.fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(),
                    l2.data_ptr(), 1, 4, 2, 100, 5000, 128, 0.0883883, False,
                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0 and fa.last_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_workspace_missing_or_small_is_rejected():
    q, k, v = (t.cuda() for t in make_custom(1, 2, 2, 64, 3000, 64, seed=16))
    need = fa.workspace_size(1, 2, 2, 64, 3000, 64, False)
    assert need > 0
    ws = torch.empty(need + 16, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    s = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), 0,
            1, 2, 2, 64, 3000, 64, 0.125, False)
    assert fa.fwd_ws_raw(*args, ws.data_ptr(), need - 16, s) == 1
    assert fa.fwd_ws_raw(*args, 0, 0, s) == 1
    assert fa.fwd_ws_raw(*args, ws.data_ptr() + 4, need, s) == 3
    assert fa.fwd_ws_raw(*args, ws.data_ptr(), need, s) == 0
    torch.cuda.synchronize()


# ------------------------------------------------------- tensor-map cache

def test_tensor_maps_are_cached_per_pointer_and_shape():
    """The four TMA maps of a call (Q, K, V, O) are encoded once per
    (pointer, shape): a repeat call on the same buffers encodes nothing, a
    new output buffer encodes one map, and results stay identical."""
    q, k, v = (t.cuda() for t in make_custom(1, 3, 1, 777, 555, 128,
                                             seed=77))
    o1 = torch.empty_like(q)
    lse = torch.empty(1, 3, 777, dtype=torch.float32, device="cuda")
    n0 = fa.tensor_map_encodes()
    fa.fwd(q, k, v, out=o1, lse=lse)
    n1 = fa.tensor_map_encodes()
    fa.fwd(q, k, v, out=o1, lse=lse)
    n2 = fa.tensor_map_encodes()
    o2 = torch.empty_like(q)
    fa.fwd(q, k, v, out=o2, lse=lse)
    n3 = fa.tensor_map_encodes()
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    # a shape used nowhere else: the first call encodes all four maps
    assert n1 - n0 == 4 and n2 == n1 and n3 - n2 == 1
    assert torch.equal(o1, o2)
    O, L = oracle.attention_fp64(q.cpu(), k.cpu(), v.cpu(), 128 ** -0.5,
                                 False)
    check(o2.cpu(), lse.cpu(), O, L, "cached maps")


def test_check_option_reads_the_device_status():
    """fwd(check=True) synchronises and raises on a bounded-wait timeout
    recorded by any kernel of the library; with none recorded it returns
    normally."""
    q, k, v = (t.cuda() for t in make_custom(1, 2, 2, 256, 256, 64, seed=78))
    o, _ = fa.fwd(q, k, v, check=True)
    assert fa.probe_bounded_wait(2_000_000) == 0    # records FA_ERR_TIMEOUT
    with pytest.raises(fa.FAError):
        fa.fwd(q, k, v, check=True)
    assert fa.last_device_error() == 0              # read and cleared
    o2, _ = fa.fwd(q, k, v, check=True)
    assert torch.equal(o, o2)


# ------------------------------------------------------ persistent schedule

def test_persistent_d64_rescales_in_late_blocks():
    """The persistent causal schedule at head dim 64 when a late block moves
    a row's reference max, so O (in TMEM, with the previous P*V's result)
    is rescaled mid-row: keys from 700 on are scaled by 6, so rows past 700
    move their reference in a late block; whole heads against the
    oracle."""
    B, Hq, Hkv, N, D = 2, 48, 8, 1536, 64
    q, k, v = make_custom(B, Hq, Hkv, N, N, D, seed=77, q_std=2.0)
    k[:, :, 700:] *= 6.0
    q, k, v = (t.cuda() for t in (q, k, v))
    scale = 1.0 / math.sqrt(D)
    assert fa.schedule(B, Hq, Hkv, N, N, D, True)["kind"] == "persist"
    o, lse = fa.fwd(q, k, v, scale=scale, causal=True, check=True)
    g = Hq // Hkv
    for b, h in {(0, 0), (1, 17), (B - 1, Hq - 1)}:
        O, L = oracle.attention_fp64(q[b:b + 1, h:h + 1].cpu(),
                                     k[b:b + 1, h // g:h // g + 1].cpu(),
                                     v[b:b + 1, h // g:h // g + 1].cpu(),
                                     scale, True)
        print(check(o[b:b + 1, h:h + 1].cpu(), lse[b:b + 1, h:h + 1].cpu(),
                    O, L, f"persist rescale b{b} h{h}"))


@pytest.mark.parametrize("B,Hq,Hkv,N,D", [
    (4, 16, 16, 2048, 64),      # 512 pairs: 3-4 pairs per CTA
    (2, 12, 4, 1000, 128),      # ragged tail tile, GQA
    (1, 3, 1, 300, 64),         # fewer pairs than SMs, tile B ragged
    (3, 50, 50, 640, 128),      # 450 pairs, pairs without a second tile
    (2, 24, 6, 1100, 64),       # GQA; each head's last pair has no tile B
])
def test_persistent_schedule_matches_one_cta_per_pair(B, Hq, Hkv, N, D):
    """Causal shapes run persistent CTAs over longest-first lists of tile
    pairs; the per-pair arithmetic is the two-tile kernel's, so the result
    equals, bit for bit, the same kernel run one pair per CTA, and matches
    the oracle on whole heads."""
    q, k, v = (t.cuda() for t in make_custom(B, Hq, Hkv, N, N, D,
                                             seed=B * Hq + N))
    scale = 1.0 / math.sqrt(D)
    assert fa.schedule(B, Hq, Hkv, N, N, D, True)["kind"] == "persist"
    o1, l1 = fa.fwd(q, k, v, scale=scale, causal=True)
    try:
        fa.set_schedule("plain")
        o2, l2 = fa.fwd(q, k, v, scale=scale, causal=True)
    finally:
        fa.set_schedule("auto")
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    if D == 128:      # the plain schedule runs the same two-tile kernel
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g = Hq // Hkv
    for b, h in {(0, 0), (B - 1, Hq - 1)}:
        O, L = oracle.attention_fp64(q[b:b + 1, h:h + 1].cpu(),
                                     k[b:b + 1, h // g:h // g + 1].cpu(),
                                     v[b:b + 1, h // g:h // g + 1].cpu(),
                                     scale, True)
        print(check(o1[b:b + 1, h:h + 1].cpu(), l1[b:b + 1, h:h + 1].cpu(),
                    O, L, f"persist B{B} H{Hq}/{Hkv} N{N} D{D} b{b} h{h}"))


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,scale", [
    (2, 8, 2, 1000, 700, 128, None),     # rows past the keys: end-of-keys tail
    (1, 4, 4, 640, 1300, 128, None),     # more keys than rows
    (2, 6, 3, 777, 777, 128, -0.09),     # negative scale: +inf hides a key
    (2, 10, 5, 1000, 1100, 64, 1.7),     # large scale at head dim 64
])
def test_persistent_hidden_keys_match_masked_path(B, Hq, Hkv, Nq, Nkv, D,
                                                  scale):
    """The persistent kernel hides a tile's masked keys by overwriting their
    scores in TMEM with the row extreme's identity and then runs the
    unmasked block code; the one-pair-per-CTA kernel masks key by key.  At
    head dim 128 both are the two-tile kernel's arithmetic, so the results
    agree bit for bit; at 64 (whose plain schedule is the one-tile kernel)
    both match the oracle on whole heads."""
    q, k, v = (t.cuda() for t in make_custom(B, Hq, Hkv, Nq, Nkv, D,
                                             seed=Nq * 7 + Nkv))
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    assert fa.schedule(B, Hq, Hkv, Nq, Nkv, D, True)["kind"] == "persist"
    o1, l1 = fa.fwd(q, k, v, scale=scale, causal=True)
    try:
        fa.set_schedule("plain")
        o2, l2 = fa.fwd(q, k, v, scale=scale, causal=True)
    finally:
        fa.set_schedule("auto")
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    if D == 128:
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g = Hq // Hkv
    for b, h in {(0, 0), (B - 1, Hq - 1)}:
        O, L = oracle.attention_fp64(q[b:b + 1, h:h + 1].cpu(),
                                     k[b:b + 1, h // g:h // g + 1].cpu(),
                                     v[b:b + 1, h // g:h // g + 1].cpu(),
                                     scale, True)
        print(check(o1[b:b + 1, h:h + 1].cpu(), l1[b:b + 1, h:h + 1].cpu(),
                    O, L, f"hidden keys B{B} H{Hq}/{Hkv} {Nq}x{Nkv} D{D}"))


def test_zero_scale_on_a_persistent_shape():
    """A zero scale leaves no score whose weight is 0, so a shape planned
    for the persistent kernel runs the one-pair-per-CTA kernel instead:
    every visible key gets weight 1, O is the mean of the visible V rows,
    and the result equals the plain schedule's bit for bit."""
    q, k, v = (t.cuda() for t in make_custom(2, 4, 2, 512, 512, 128, seed=9))
    assert fa.schedule(2, 4, 2, 512, 512, 128, True)["kind"] == "persist"
    o1, l1 = fa.fwd(q, k, v, scale=0.0, causal=True, check=True)
    try:
        fa.set_schedule("plain")
        o2, l2 = fa.fwd(q, k, v, scale=0.0, causal=True, check=True)
    finally:
        fa.set_schedule("auto")
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    n = torch.arange(1, 513, dtype=torch.float64)
    assert torch.allclose(l1[1, 3].double().cpu(), n.log(), atol=1e-4)
    O, L = oracle.attention_fp64(q[1:2, 3:4].cpu(), k[1:2, 1:2].cpu(),
                                 v[1:2, 1:2].cpu(), 0.0, True)
    print(check(o1[1:2, 3:4].cpu(), l1[1:2, 3:4].cpu(), O, L, "scale 0"))


@pytest.mark.parametrize("B,Hq,Hkv,N,D", [
    (1, 11, 11, 20000, 128),    # two-tile kernel: head groups 3, 3, 3, 2
    (1, 7, 7, 12000, 256),      # one-tile kernel: head groups 3, 3, 1
    (3, 4, 2, 12000, 192),      # one-tile kernel, GQA: a group spans batches
])
def test_causal_grid_order_covers_every_tile(B, Hq, Hkv, N, D):
    """Causal grids of one-unit CTAs run their units by head groups, longest
    first with the group's heads interleaved (a permutation of the grid):
    every row of every head is written exactly once (O starts as NaN), and
    sampled rows of the first, a middle and the last head match the
    oracle."""
    q, k, v = make_custom(B, Hq, Hkv, N, N, D, seed=N + D)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    assert fa.schedule(B, Hq, Hkv, N, N, D, True)["kind"] == "plain"
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq, N), float("nan"), device="cuda")
    scale = 1.0 / math.sqrt(D)
    fa.fwd(qd, kd, vd, scale=scale, causal=True, out=o, lse=lse, check=True)
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    gen = torch.Generator().manual_seed(1)
    for b, h in {(0, 0), (B - 1, Hq // 2), (B - 1, Hq - 1)}:
        rows = _sample_rows(N, gen)
        O, L = oracle.attention_rows_fp64(q, k, v, scale, True, b, h, rows)
        print(check(o[b, h, rows], lse[b, h, rows], O, L,
                    f"grid order B{B} H{Hq}/{Hkv} N{N} D{D} b{b} h{h}"))
