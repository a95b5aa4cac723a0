"""The C-ABI library: builds, loads, exports every declared symbol, and
rejects bad arguments on the host before touching the GPU (CPU only)."""

import ctypes
import os
import re

import pytest

from exact_io_aware_fa2_gb300 import build as fabuild
from exact_io_aware_fa2_gb300 import fa

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include",
                      "fa.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fabuild.LIB_PATH):
        fabuild.build()
    return fa.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(fa_\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_expected_entry_points():
    assert _declared_functions() == sorted(fa.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    # and they are real exported C symbols (not C++-mangled)
    raw = ctypes.CDLL(fabuild.LIB_PATH)
    for name in _declared_functions():
        getattr(raw, name)


def test_status_strings(lib):
    for code, name in fa.STATUS_NAMES.items():
        assert fa.status_string(code) == name
    assert fa.status_string(99) == "FA_ERR_UNKNOWN"
    assert lib.fa_version() == 100


P = 1 << 20  # a 16-byte-aligned stand-in address; never dereferenced


def _call(**kw):
    args = dict(q=P, k=P, v=P, o=P, lse=P, B=1, Hq=2, Hkv=1, Nq=128, Nkv=128,
                D=64, scale=0.125, causal=0, stream=0)
    args.update(kw)
    return fa.fwd_raw(args["q"], args["k"], args["v"], args["o"], args["lse"],
                      args["B"], args["Hq"], args["Hkv"], args["Nq"],
                      args["Nkv"], args["D"], args["scale"], args["causal"],
                      args["stream"])


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(k=0), dict(v=0), dict(o=0),
    dict(B=0), dict(Hq=0), dict(Hkv=0), dict(Nq=0), dict(Nkv=0), dict(D=0),
    dict(B=-1), dict(Nkv=-5),
    dict(Hq=3, Hkv=2), dict(Hq=2, Hkv=4),
    dict(scale=float("nan")), dict(scale=float("inf")),
    dict(B=70000), dict(Hq=70000, Hkv=1),
])
def test_invalid_values_rejected_before_launch(lib, kw):
    assert _call(**kw) == 1  # FA_ERR_INVALID_VALUE


@pytest.mark.parametrize("D", [1, 16, 32, 80, 96, 160, 224, 320, 512])
def test_unsupported_head_dims(lib, D):
    assert _call(D=D) == 2  # FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw", [dict(q=P + 2), dict(k=P + 8), dict(v=P + 4),
                                dict(o=P + 1), dict(lse=P + 2)])
def test_misaligned_pointers_rejected(lib, kw):
    assert _call(**kw) == 3  # FA_ERR_MISALIGNED


def test_lse_may_be_null_for_validation(lib):
    # a null lse is legal; with everything else invalid the error is still
    # the validation one
    assert _call(lse=0, q=0) == 1


def test_probe_rejects_bad_limits(lib):
    assert lib.fa_probe_bounded_wait(0, None) == 1
    assert lib.fa_probe_bounded_wait(2_000_000_000, None) == 1
    assert lib.fa_probe_flag_wait(0, None) == 1
    assert lib.fa_probe_flag_wait(2_000_000_000, None) == 1


def test_binding_rejects_bad_tensors():
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.float32)
    with pytest.raises(TypeError):
        fa._check(q, q, q)
    qb = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa._check(qb, qb[:, :, :4], qb)
    with pytest.raises(ValueError):
        fa._check(qb.transpose(2, 3), qb, qb)


def test_host_binding_rejects_bad_tensors_before_any_device_work():
    """fa.fwd_host takes CPU bf16 [B, H, N, D] tensors; anything else is
    rejected on the host before buffers are allocated or the library is
    called."""
    import torch
    qf = torch.zeros(1, 2, 8, 64, dtype=torch.float32)
    with pytest.raises(TypeError):
        fa.fwd_host(qf, qf, qf)
    qb = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    kb = torch.zeros(1, 2, 5, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd_host(qb, kb, qb)                  # k and v shapes differ
    with pytest.raises(ValueError):
        fa.fwd_host(qb[0], qb[0], qb[0])         # not 4-D


def test_noalloc_limit_matches_header():
    text = open(HEADER).read()
    m = re.search(r"#define\s+FA_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)",
                  text)
    assert m is not None
    assert int(m.group(1)) << int(m.group(2)) == fa.NOALLOC_SCRATCH_BYTES


def test_set_schedule_validates_its_argument(lib):
    """fa_set_schedule takes FA_SCHEDULE_AUTO (-1), PLAIN (0) or STREAM (2)
    and rejects anything else without touching the device."""
    for bad in (-2, 1, 3, 99):
        assert lib.fa_set_schedule(bad) == 1          # FA_ERR_INVALID_VALUE
    for good in (2, 0, -1):                           # ends on AUTO
        assert lib.fa_set_schedule(good) == 0


def test_host_entry_point_checks_host_pointers_first(lib):
    """fa_fwd_host rejects a NULL host pointer, or lse_host and lse_dev not
    both NULL or both set, before touching the device."""
    dev = [ctypes.c_void_p(256)] * 5
    host = [ctypes.c_void_p(512)] * 5
    args = (1, 1, 1, 128, 128, 128, ctypes.c_float(0.1), 0, None)
    for i in range(4):
        bad = list(host)
        bad[i] = None
        assert lib.fa_fwd_host(*bad, *dev, *args) == 1
    assert lib.fa_fwd_host(*host[:4], None, *dev, *args) == 1
    assert lib.fa_fwd_host(*host, *dev[:4], None, *args) == 1


def test_host_binding_checks_every_buffer_before_any_device_work():
    """fa.fwd_host checks the caller's buffer set (device q, k, v, o, lse and
    host o_h, lse_h) against the inputs' shapes, dtypes, layout and device
    before calling the library, which copies whole tensors of those sizes:
    a buffer from a smaller shape would be overrun."""
    import torch
    q = torch.zeros(2, 4, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(2, 2, 16, 64, dtype=torch.bfloat16)

    def bufs(**over):
        b = {"q": torch.empty(q.shape, dtype=q.dtype, device="meta"),
             "k": torch.empty(k.shape, dtype=k.dtype, device="meta"),
             "v": torch.empty(k.shape, dtype=k.dtype, device="meta"),
             "o": torch.empty(q.shape, dtype=q.dtype, device="meta"),
             "lse": torch.empty(2, 4, 8, dtype=torch.float32, device="meta"),
             "o_h": torch.empty(q.shape, dtype=q.dtype),
             "lse_h": torch.empty(2, 4, 8, dtype=torch.float32)}
        b.update(over)
        return {n: t for n, t in b.items() if t is not None}

    small_o = torch.empty(2, 4, 4, 64, dtype=torch.bfloat16)
    cases = [
        (ValueError, dict(o=None)),                              # missing
        (ValueError, dict(o_h=small_o)),                         # smaller
        (ValueError, dict(lse_h=torch.empty(2, 4, 4))),          # smaller
        (TypeError, dict(lse_h=torch.empty(2, 4, 8,
                                           dtype=torch.float64))),
        (TypeError, dict(o_h=torch.empty(q.shape, dtype=torch.float32))),
        (ValueError, dict(o_h=torch.empty(2, 4, 64, 8, dtype=torch.bfloat16
                                          ).transpose(2, 3))),    # strided
        (ValueError, dict(k=torch.empty(2, 2, 8, 64, dtype=torch.bfloat16,
                                        device="meta"))),        # wrong N
    ]
    for exc, over in cases:
        with pytest.raises(exc):
            fa.fwd_host(q, k, k, bufs=bufs(**over))
    # correct shapes, but the "device" buffers are not CUDA tensors
    with pytest.raises(ValueError):
        fa.fwd_host(q, k, k, bufs=bufs())
    # host outputs on a non-CPU device are refused too
    with pytest.raises(ValueError):
        fa.fwd_host(q, k, k, bufs=bufs(
            o_h=torch.empty(q.shape, dtype=q.dtype, device="meta")))


def test_tensor_map_counter_needs_no_device(lib):
    """fa_tensor_map_encodes reads a host counter: callable without a GPU,
    and no failed call above encoded anything."""
    assert fa.tensor_map_encodes() == 0


def test_mxfp8_entry_validates_before_the_device(lib):
    """fa_fwd_mxfp8: a NULL scale pointer, a head dim other than 128 and a
    misaligned scale pointer are refused on the host."""
    vp = ctypes.c_void_p
    args = lambda qs, ks, D: (vp(P), vp(P), vp(P), vp(qs), vp(ks), vp(P),
                              vp(P), 1, 2, 1, 128, 128, D, ctypes.c_float(0.1),
                              0, None)
    assert lib.fa_fwd_mxfp8(*args(None, P, 128)) == 1
    assert lib.fa_fwd_mxfp8(*args(P, None, 128)) == 1
    assert lib.fa_fwd_mxfp8(*args(P, P, 64)) == 2
    assert lib.fa_fwd_mxfp8(*args(P + 2, P, 128)) == 3
