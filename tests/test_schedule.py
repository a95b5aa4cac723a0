"""The work schedule the host plans for a shape (fa_fwd_schedule_for: no GPU
needed).  Checks the choices measured on GB300 (152 SMs), the split-KV and
stream shapes and their scratch sizes, the forced settings, and invariants
of every schedule over a grid of shapes and SM counts."""

import itertools
import math

import pytest

from exact_io_aware_fa2_gb300 import fa

SLOT = {64: 256 * 67 * 4, 128: 256 * 131 * 4}   # stream / two-tile split slot:
# O [256][D], m, l (exact sums), w (bf16-weight sums), fp32


@pytest.fixture(autouse=True)
def auto_schedule():
    fa.set_schedule("auto")
    yield
    fa.set_schedule("auto")


def sched(B, Hq, Hkv, Nq, Nkv, D, causal=False, sms=152):
    return fa.schedule_for(B, Hq, Hkv, Nq, Nkv, D, causal, sms)


@pytest.mark.parametrize("shape,kind", [
    ((1, 8, 8, 4096, 8192, 128), "stream"),    # 128 pairs: 84% of a wave
    ((1, 9, 9, 4096, 8192, 128), "plain"),     # 144 pairs
    ((1, 16, 16, 4096, 8192, 128), "stream"),  # 256 pairs: 1.7 waves
    ((1, 8, 8, 4096, 4096, 128), "plain"),     # 128 pairs, 4096 keys
    ((1, 5, 5, 4096, 8192, 128), "stream"),    # 80 pairs: 53% of a wave
    ((1, 7, 7, 4096, 8192, 128), "stream"),    # 112 pairs
    ((1, 25, 25, 2048, 8192, 128), "stream"),  # 200 pairs: 1.3 waves
    ((1, 5, 5, 4096, 4096, 128), "stream"),    # 80 pairs, 4096 keys
    ((1, 5, 5, 4096, 2048, 128), "plain"),     # short rows: overhead wins
    ((1, 5, 5, 4096, 8192, 64), "stream"),
    ((1, 8, 8, 4096, 8192, 64), "stream"),     # 128 pairs at D = 64
    ((1, 16, 16, 4096, 4096, 64), "stream"),   # 256 pairs, 4096 keys
    ((1, 9, 9, 4096, 8192, 64), "plain"),      # 144 pairs
    # few pairs: split-KV while its pieces fit one wave, else stream
    ((1, 4, 4, 2048, 16384, 128), "split_kv"),   # 16 pairs x 4 pieces
    ((4, 8, 8, 512, 8192, 128), "split_kv"),     # 64 pairs x 2 pieces
    ((2, 16, 16, 512, 16384, 128), "stream"),    # would be 7 x 64 CTAs
    ((1, 16, 16, 1024, 16384, 64), "stream"),
    ((2, 8, 8, 1024, 32768, 128), "stream"),
])
def test_choices_measured_on_gb300(shape, kind):
    """The estimate picks the schedule measured faster on GB300 (stream
    against plain: 71 vs 98 us at 80 pairs, 87 vs 98 at 112, 96 vs 98 at
    128, 177 vs 193 at 256, 144 vs 191 at 200 pairs of 2048 rows, 47 vs 55
    with 4096 keys; plain: 100 vs 107 at 144 pairs, 55 vs 59 at 128 pairs
    of 4096 keys, 33 vs 38 on 2048-key rows; split against stream: 66 vs
    72 us for 16 pairs of 16384 keys, 68 vs 71 for 64 pairs of 8192; stream
    against a split of more than one wave: 112 vs 136 us for 64 pairs of
    16384 keys, 89 vs 101 at D = 64, 194 vs 209 for 32 pairs of 32768; at
    D = 64 stream 84 vs 90 us at 128 pairs and 86 vs 93 at 256 pairs of
    4096 keys, plain 90 vs 92 at 144 pairs)."""
    assert sched(*shape)["kind"] == kind


def test_headline_runs_the_stream_schedule():
    # 128 pairs x 64 blocks over 152 CTAs: 54 blocks each, one partial slot
    # and eight flags per CTA
    s = sched(1, 8, 8, 4096, 8192, 128)
    assert s == {"kind": "stream", "ctas": 152, "pieces": 1,
                 "blocks_per_cta": 54, "workspace": 152 * (SLOT[128] + 64)}


def test_decode_shape_splits_packed_gqa():
    # 32 query heads over 8 kv heads, 128 rows each: packed into 8 heads of
    # 512 rows = 2 pairs each; 256 K/V blocks cut into 9 pieces.
    s = sched(1, 32, 8, 128, 32768, 128)
    assert s["kind"] == "split_kv" and s["pieces"] == 9
    assert s["ctas"] == 2 * 8 * 9
    assert s["workspace"] == s["ctas"] * SLOT[128]


def test_causal_and_wide_shapes_never_stream():
    for shape in [(1, 5, 5, 4096, 8192, 128, True),
                  (1, 5, 5, 4096, 8192, 256, False),
                  (1, 5, 5, 4096, 8192, 192, False),
                  (4, 16, 16, 2048, 2048, 64, True)]:
        assert sched(*shape)["kind"] != "stream"
        fa.set_schedule("stream")
        assert sched(*shape)["kind"] != "stream"
        fa.set_schedule("auto")


@pytest.mark.parametrize("shape,ctas", [
    ((4, 16, 16, 2048, 2048, 64, True), 152),      # 512 pairs, 32 MiB K/V
    ((2, 32, 8, 8192, 8192, 128, True), 152),      # 2048 pairs, 64 MiB K/V
    ((1, 2, 2, 512, 512, 128, True), 4),           # fewer pairs than SMs
])
def test_causal_shapes_run_persistent(shape, ctas):
    """Causal shapes at head dims 64 and 128 that do not split, and whose K
    and V fit in 96 MiB, run the persistent schedule: at most one CTA per
    SM, no scratch; forcing the plain schedule turns it off."""
    s = sched(*shape)
    assert s == {"kind": "persist", "ctas": ctas, "pieces": 1,
                 "blocks_per_cta": 0, "workspace": 0}
    fa.set_schedule("plain")
    assert sched(*shape)["kind"] == "plain"


def test_causal_shapes_with_large_kv_run_one_pair_per_cta():
    """Past 96 MiB of K and V (here 256 MiB: 16 heads of 32768 keys) the
    longest-first list would keep every head's K/V in use at once and
    re-read it from DRAM; such shapes run one CTA per pair, whose grid
    walks the heads in order."""
    s = sched(1, 16, 16, 32768, 32768, 128, True)
    assert s["kind"] == "plain" and s["ctas"] == 16 * 128


def test_forced_settings():
    fa.set_schedule("plain")
    s = sched(1, 8, 8, 128, 32768, 128)
    assert s["kind"] == "plain" and s["workspace"] == 0
    fa.set_schedule("stream")
    # one block per CTA when there are fewer blocks than SMs: 2 pairs of 24
    s = sched(1, 2, 2, 256, 3000, 128)
    assert s["kind"] == "stream" and s["blocks_per_cta"] == 1
    assert s["ctas"] == 48 and s["workspace"] == 48 * (SLOT[128] + 64)
    fa.set_schedule("auto")
    assert sched(1, 2, 2, 256, 3000, 128)["kind"] != "stream"


def test_rejects_bad_arguments():
    with pytest.raises(fa.FAError):
        sched(1, 8, 8, 4096, 8192, 128, sms=0)
    with pytest.raises(fa.FAError):
        sched(1, 8, 3, 4096, 8192, 128)          # Hq % Hkv != 0
    with pytest.raises(fa.FAError):
        sched(1, 8, 8, 4096, 8192, 96)           # unsupported head dim


SHAPES = list(itertools.product(
    [1, 3], [1, 8, 24], [1, 4096], [1, 700, 8192], [64, 128, 256],
    [False, True]))


@pytest.mark.parametrize("sms", [8, 76, 152, 160])
def test_invariants(sms):
    for B, Hq, Nq, Nkv, D, causal in SHAPES:
        for Hkv in sorted({1, Hq}):
            s = sched(B, Hq, Hkv, Nq, Nkv, D, causal, sms)
            packed = not causal and Hq != Hkv
            H, N = (Hkv, (Hq // Hkv) * Nq) if packed else (Hq, Nq)
            one_tile = D in (192, 256) or (D == 64 and causal)
            rows = 128 if one_tile else 256
            units = math.ceil(N / rows) * H * B
            what = (B, Hq, Hkv, Nq, Nkv, D, causal, sms, s)
            if s["kind"] == "plain":
                assert s["ctas"] == units and s["pieces"] == 1, what
                assert s["workspace"] == 0, what
            elif s["kind"] == "persist":
                pairs = math.ceil(N / 256) * H * B
                assert causal and D in (64, 128), what
                assert s["ctas"] == min(pairs, sms), what
                assert s["pieces"] == 1 and s["workspace"] == 0, what
                assert 4 * B * Hkv * Nkv * D <= 96 << 20, what
                assert pairs * 2 > sms or sched(B, Hq, Hkv, Nq, Nkv, D,
                                                causal, sms)["kind"] == \
                    "persist", what
            elif s["kind"] == "split_kv":
                keys = 64 if one_tile else 128
                longest = math.ceil((min(N, Nkv) if causal else Nkv) / keys)
                assert 2 <= s["pieces"] <= 64, what
                assert s["pieces"] <= max(1, longest // 4), what
                assert s["ctas"] == units * s["pieces"], what
                assert units * 2 <= sms, what
                # without a mask at head dims 64 and 128 a split takes at
                # most one wave (else the stream schedule runs)
                assert causal or D not in (64, 128) or s["ctas"] <= sms, what
                slot = (rows * (D + 3)) * 4
                assert s["workspace"] == units * s["pieces"] * slot, what
            else:
                assert not causal and D in (64, 128), what
                nbp = math.ceil(Nkv / 128)
                total = units * nbp
                L = s["blocks_per_cta"]
                assert L == math.ceil(total / sms), what
                assert s["ctas"] == math.ceil(total / L) <= sms, what
                # at least half a pair per CTA, unless the shape would
                # otherwise split into more than one wave
                assert 2 * L >= nbp or units * 2 <= sms, what
                assert s["workspace"] == s["ctas"] * (SLOT[D] + 64), what
