"""ctypes binding of the C ABI in ``include/fa.h`` (``libfa_gb300.so``).

Argument marshalling only: tensors become device pointers and sizes, the
current torch stream becomes the ``stream`` argument, and a nonzero status
becomes an exception.  Every step of the computation runs in the library's
kernels; there is no fallback of any kind — if the library is missing or the
device is not sm_103, calls raise.

    o, lse = fwd(q, k, v, scale=None, causal=False)

q: bf16 [B, Hq, Nq, D]; k, v: bf16 [B, Hkv, Nkv, D]; all CUDA, contiguous.
Returns o (bf16, like q) and lse (fp32 [B, Hq, Nq]).  ``fwd_host`` does the
same for pinned host tensors: it copies the inputs to the device, runs the
kernel and copies O and LSE back, all on the current stream.
"""

import contextlib
import ctypes
import math
import os
import threading

import torch

from .build import LIB_PATH

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_VALUE", 2: "FA_ERR_UNSUPPORTED",
                3: "FA_ERR_MISALIGNED", 4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT"}
# Every symbol the header declares.
SYMBOLS = ("fa_fwd", "fa_fwd_ws", "fa_fwd_workspace_size", "fa_fwd_noalloc",
           "fa_fwd_qk8", "fa_fwd_schedule", "fa_set_schedule", "fa_fwd_host",
           "fa_probe_flag_wait", "fa_fwd_schedule_for",
           "fa_status_string", "fa_last_device_error",
           "fa_probe_bounded_wait", "fa_version", "fa_tensor_map_encodes",
           "fa_fwd_mxfp8")

_lib = None
_lock = threading.Lock()


class FAError(RuntimeError):
    def __init__(self, status, what="fa_fwd"):
        self.status = status
        super().__init__(f"{what} failed: {STATUS_NAMES.get(status, status)}")


def library_path():
    return LIB_PATH


def load():
    """Load (once) and return the ctypes handle of the library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{os.path.basename(LIB_PATH)} is not built; run "
                "`python -c \"import __graft_entry__ as g; g.build()\"`")
        lib = ctypes.CDLL(LIB_PATH)
        vp, ci = ctypes.c_void_p, ctypes.c_int
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci,
                               ctypes.c_float, ci, vp]
        lib.fa_fwd.restype = ci
        lib.fa_fwd_ws.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci,
                                  ctypes.c_float, ci, vp, ctypes.c_size_t, vp]
        lib.fa_fwd_ws.restype = ci
        lib.fa_fwd_workspace_size.argtypes = [
            ci, ci, ci, ci, ci, ci, ci, ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_fwd_workspace_size.restype = ci
        lib.fa_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci,
                                       ci, ctypes.c_float, ci, vp]
        lib.fa_fwd_noalloc.restype = ci
        lib.fa_fwd_qk8.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci,
                                   ctypes.c_float, ctypes.c_float,
                                   ctypes.c_float, ci, vp]
        lib.fa_fwd_qk8.restype = ci
        lib.fa_status_string.argtypes = [ci]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_last_device_error.argtypes = []
        lib.fa_last_device_error.restype = ci
        lib.fa_probe_bounded_wait.argtypes = [ctypes.c_longlong, vp]
        lib.fa_probe_bounded_wait.restype = ci
        lib.fa_version.argtypes = []
        lib.fa_version.restype = ci
        pi = ctypes.POINTER(ci)
        lib.fa_fwd_schedule.argtypes = [ci, ci, ci, ci, ci, ci, ci, pi, pi,
                                        pi, pi]
        lib.fa_fwd_schedule.restype = ci
        lib.fa_set_schedule.argtypes = [ci]
        lib.fa_set_schedule.restype = ci
        lib.fa_fwd_host.argtypes = [vp] * 10 + [ci] * 6 + [ctypes.c_float,
                                                          ci, vp]
        lib.fa_fwd_host.restype = ci
        lib.fa_probe_flag_wait.argtypes = [ctypes.c_longlong, vp]
        lib.fa_probe_flag_wait.restype = ci
        lib.fa_fwd_schedule_for.argtypes = [ci] * 8 + [pi] * 4 + [
            ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_fwd_schedule_for.restype = ci
        lib.fa_fwd_mxfp8.argtypes = [vp] * 7 + [ci] * 6 + [ctypes.c_float,
                                                           ci, vp]
        lib.fa_fwd_mxfp8.restype = ci
        lib.fa_tensor_map_encodes.argtypes = []
        lib.fa_tensor_map_encodes.restype = ctypes.c_size_t
        _lib = lib
        return lib


def status_string(status):
    return load().fa_status_string(int(status)).decode()


def last_device_error():
    return int(load().fa_last_device_error())


def tensor_map_encodes():
    """TMA tensor maps encoded so far (``fa_tensor_map_encodes``); calls on
    buffers whose maps are cached add nothing."""
    return int(load().fa_tensor_map_encodes())


def probe_bounded_wait(timeout_ns, stream=None):
    st = stream if stream is not None else torch.cuda.current_stream()
    return int(load().fa_probe_bounded_wait(int(timeout_ns),
                                            ctypes.c_void_p(st.cuda_stream)))


def probe_flag_wait(timeout_ns, stream=None):
    st = stream if stream is not None else torch.cuda.current_stream()
    return int(load().fa_probe_flag_wait(int(timeout_ns),
                                         ctypes.c_void_p(st.cuda_stream)))


def _check(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, N, D]")
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, Hq, Nq, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k, v must be [B, Hkv, Nkv, D] matching q")
    return B, Hq, k.shape[1], Nq, k.shape[2], D


def _check_host(q, k, v):
    _check(q, k, v)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.device.type != "cpu":
            raise ValueError(f"{name} must be a host (CPU) tensor")


def fwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, Hq, Hkv, Nq, Nkv, D,
            scale, causal, stream_handle):
    """Direct call of ``fa_fwd`` with integer pointers; returns the status."""
    return int(load().fa_fwd(
        ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
        ctypes.c_void_p(o_ptr), ctypes.c_void_p(lse_ptr),
        B, Hq, Hkv, Nq, Nkv, D, ctypes.c_float(scale), 1 if causal else 0,
        ctypes.c_void_p(stream_handle)))


_ws_cache = {}


# Bytes of the fixed scratch array behind fa_fwd_noalloc.
NOALLOC_SCRATCH_BYTES = 32 << 20


def fwd_noalloc_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, Hq, Hkv, Nq, Nkv,
                    D, scale, causal, stream_handle):
    """Direct call of ``fa_fwd_noalloc`` (allocates nothing); returns the
    status."""
    return int(load().fa_fwd_noalloc(
        ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
        ctypes.c_void_p(o_ptr), ctypes.c_void_p(lse_ptr),
        B, Hq, Hkv, Nq, Nkv, D, ctypes.c_float(scale), 1 if causal else 0,
        ctypes.c_void_p(stream_handle)))


# Schedule names of fa_fwd_schedule's FA_SCHEDULE_* values.
SCHEDULES = {0: "plain", 1: "split_kv", 2: "stream", 3: "persist"}


def schedule(B, Hq, Hkv, Nq, Nkv, D, causal):
    """How the forward runs this shape on the current device:
    ``{"kind": "plain" | "split_kv" | "stream", "ctas", "pieces",
    "blocks_per_cta"}`` (``fa_fwd_schedule``)."""
    out = [ctypes.c_int(0) for _ in range(4)]
    st = int(load().fa_fwd_schedule(B, Hq, Hkv, Nq, Nkv, D,
                                    1 if causal else 0,
                                    *[ctypes.byref(o) for o in out]))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_schedule")
    kind, ctas, pieces, bpc = (int(o.value) for o in out)
    return {"kind": SCHEDULES[kind], "ctas": ctas, "pieces": pieces,
            "blocks_per_cta": bpc}


_SCHEDULE_CODES = {"auto": -1, "plain": 0, "stream": 2}


def set_schedule(kind):
    """Force the schedule of later calls process-wide: ``"auto"`` (the
    default), ``"plain"`` or ``"stream"`` (``fa_set_schedule``).  Clears the
    workspace-size cache, whose answers depend on it."""
    st = int(load().fa_set_schedule(_SCHEDULE_CODES[kind]))
    if st != FA_OK:
        raise FAError(st, "fa_set_schedule")
    _ws_cache.clear()


def schedule_for(B, Hq, Hkv, Nq, Nkv, D, causal, sms):
    """``schedule`` for a GPU with ``sms`` SMs, computed on the host without
    a device (``fa_fwd_schedule_for``); adds ``"workspace"``, the scratch
    bytes ``fa_fwd_ws`` would need there."""
    out = [ctypes.c_int(0) for _ in range(4)]
    ws = ctypes.c_size_t(0)
    st = int(load().fa_fwd_schedule_for(B, Hq, Hkv, Nq, Nkv, D,
                                        1 if causal else 0, sms,
                                        *[ctypes.byref(o) for o in out],
                                        ctypes.byref(ws)))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_schedule_for")
    kind, ctas, pieces, bpc = (int(o.value) for o in out)
    return {"kind": SCHEDULES[kind], "ctas": ctas, "pieces": pieces,
            "blocks_per_cta": bpc, "workspace": int(ws.value)}


def workspace_size(B, Hq, Hkv, Nq, Nkv, D, causal):
    """Scratch bytes ``fa_fwd_ws`` needs for this shape (current device);
    the answer depends only on the shape and the device, so it is cached."""
    key = (torch.cuda.current_device(), B, Hq, Hkv, Nq, Nkv, D, bool(causal))
    hit = _ws_cache.get(key)
    if hit is not None:
        return hit
    n = ctypes.c_size_t(0)
    st = int(load().fa_fwd_workspace_size(B, Hq, Hkv, Nq, Nkv, D,
                                          1 if causal else 0,
                                          ctypes.byref(n)))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_workspace_size")
    _ws_cache[key] = int(n.value)
    return int(n.value)


def fwd_ws_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, Hq, Hkv, Nq, Nkv, D,
               scale, causal, ws_ptr, ws_bytes, stream_handle):
    """Direct call of ``fa_fwd_ws`` with integer pointers; returns status."""
    return int(load().fa_fwd_ws(
        ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
        ctypes.c_void_p(o_ptr), ctypes.c_void_p(lse_ptr),
        B, Hq, Hkv, Nq, Nkv, D, ctypes.c_float(scale), 1 if causal else 0,
        ctypes.c_void_p(ws_ptr), ctypes.c_size_t(ws_bytes),
        ctypes.c_void_p(stream_handle)))


def fwd(q, k, v, scale=None, causal=False, out=None, lse=None,
        want_lse=True, workspace=None, check=False):
    """Attention forward through the C ABI on the current CUDA stream.

    Split-KV scratch (only for shapes that need it) comes from
    ``workspace`` (a uint8 CUDA tensor) or, if None, from torch's caching
    allocator for this call.

    The call returns without synchronising.  A kernel whose bounded wait
    ran out (``FA_ERR_TIMEOUT``, read by ``last_device_error`` after a
    synchronisation) leaves the rows it abandoned unwritten; with
    ``check=True`` the call synchronises the stream, reads that status and
    raises ``FAError`` if it is set."""
    B, Hq, Hkv, Nq, Nkv, D = _check(q, k, v)
    dev = q.device
    if dev.type != "cuda" or k.device != dev or v.device != dev:
        raise ValueError("q, k, v must be CUDA tensors on one device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if want_lse and lse is None:
        lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        need = workspace_size(B, Hq, Hkv, Nq, Nkv, D, causal)
        if need > 0 and (workspace is None or workspace.numel() < need):
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = fwd_ws_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                        out.data_ptr(),
                        lse.data_ptr() if lse is not None else 0,
                        B, Hq, Hkv, Nq, Nkv, D, scale, causal,
                        workspace.data_ptr() if need > 0 else 0, need, stream)
    if st != FA_OK:
        raise FAError(st)
    if check:
        _check_device_status(dev, "fa_fwd")
    return out, lse


def _check_device_status(dev, what):
    """Synchronise ``dev``'s current stream and raise if a kernel of the
    library gave up a bounded wait since the last query."""
    with torch.cuda.device(dev):
        torch.cuda.current_stream(dev).synchronize()
        st = last_device_error()
    if st != FA_OK:
        raise FAError(st, what)


def fwd_qk8_raw(q8_ptr, k8_ptr, v_ptr, o_ptr, lse_ptr, B, Hq, Hkv, Nq, Nkv,
                D, scale, q_descale, k_descale, causal, stream_handle):
    """Direct call of ``fa_fwd_qk8``; returns the status."""
    return int(load().fa_fwd_qk8(
        ctypes.c_void_p(q8_ptr), ctypes.c_void_p(k8_ptr),
        ctypes.c_void_p(v_ptr), ctypes.c_void_p(o_ptr),
        ctypes.c_void_p(lse_ptr), B, Hq, Hkv, Nq, Nkv, D,
        ctypes.c_float(scale), ctypes.c_float(q_descale),
        ctypes.c_float(k_descale), 1 if causal else 0,
        ctypes.c_void_p(stream_handle)))


def fwd_qk8(q8, k8, v, scale=None, q_descale=1.0, k_descale=1.0,
            causal=False, out=None, lse=None, check=False):
    """Forward with e4m3 Q and K (``torch.float8_e4m3fn``, with one descale
    factor each) and bf16 V, through ``fa_fwd_qk8``; D must be 128.
    ``check`` as for ``fwd``."""
    for name, t, dt in (("q8", q8, torch.float8_e4m3fn),
                        ("k8", k8, torch.float8_e4m3fn),
                        ("v", v, torch.bfloat16)):
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, N, D]")
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device != q8.device or t.device.type != "cuda":
            raise ValueError("q8, k8, v must be CUDA tensors on one device")
    B, Hq, Nq, D = q8.shape
    if k8.shape != v.shape or k8.shape[0] != B or k8.shape[3] != D:
        raise ValueError("k8, v must be [B, Hkv, Nkv, D] matching q8")
    Hkv, Nkv = k8.shape[1], k8.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = q8.device
    if out is None:
        out = torch.empty(B, Hq, Nq, D, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = fwd_qk8_raw(q8.data_ptr(), k8.data_ptr(), v.data_ptr(),
                         out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Nq, Nkv,
                         D, scale, q_descale, k_descale, causal,
                         torch.cuda.current_stream(dev).cuda_stream)
    if st != FA_OK:
        raise FAError(st)
    if check:
        _check_device_status(dev, "fa_fwd_qk8")
    return out, lse


def fwd_mxfp8_raw(q8_ptr, k8_ptr, v_ptr, qs_ptr, ks_ptr, o_ptr, lse_ptr, B,
                  Hq, Hkv, Nq, Nkv, D, scale, causal, stream_handle):
    """Direct call of ``fa_fwd_mxfp8``; returns the status."""
    return int(load().fa_fwd_mxfp8(
        *[ctypes.c_void_p(x) for x in (q8_ptr, k8_ptr, v_ptr, qs_ptr, ks_ptr,
                                       o_ptr, lse_ptr)],
        B, Hq, Hkv, Nq, Nkv, D, ctypes.c_float(scale), 1 if causal else 0,
        ctypes.c_void_p(stream_handle)))


def fwd_mxfp8(q8, k8, v, q_scale, k_scale, scale=None, causal=False,
              out=None, lse=None, check=False):
    """Forward with MXFP8 Q and K through ``fa_fwd_mxfp8``: e4m3 values
    (``torch.float8_e4m3fn`` [B, H, N, D]) with one ue8m0 scale byte per 32
    head-dim elements (``torch.uint8`` [B, H, N, D // 32]), and bf16 V; D
    must be 128.  ``check`` as for ``fwd``."""
    for name, t, dt in (("q8", q8, torch.float8_e4m3fn),
                        ("k8", k8, torch.float8_e4m3fn),
                        ("v", v, torch.bfloat16),
                        ("q_scale", q_scale, torch.uint8),
                        ("k_scale", k_scale, torch.uint8)):
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D")
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device != q8.device or t.device.type != "cuda":
            raise ValueError("all inputs must be CUDA tensors on one device")
    B, Hq, Nq, D = q8.shape
    if k8.shape != v.shape or k8.shape[0] != B or k8.shape[3] != D:
        raise ValueError("k8, v must be [B, Hkv, Nkv, D] matching q8")
    if D % 32 != 0 or q_scale.shape != (B, Hq, Nq, D // 32) or \
            k_scale.shape != (B, k8.shape[1], k8.shape[2], D // 32):
        raise ValueError("scales must be [B, H, N, D // 32] per operand")
    Hkv, Nkv = k8.shape[1], k8.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = q8.device
    if out is None:
        out = torch.empty(B, Hq, Nq, D, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = fwd_mxfp8_raw(q8.data_ptr(), k8.data_ptr(), v.data_ptr(),
                           q_scale.data_ptr(), k_scale.data_ptr(),
                           out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Nq,
                           Nkv, D, scale, causal,
                           torch.cuda.current_stream(dev).cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_mxfp8")
    if check:
        _check_device_status(dev, "fa_fwd_mxfp8")
    return out, lse


def _check_host_bufs(bufs, q, k, v):
    """Every buffer fa_fwd_host reads or writes, against the inputs' shapes:
    device q, k, v, o bf16 like the inputs and lse fp32 [B, Hq, Nq], all
    contiguous on one CUDA device; host o_h bf16 and lse_h fp32 of the same
    shapes, contiguous, on the CPU.  The library copies whole tensors of
    these sizes, so a smaller buffer would be overrun."""
    B, Hq, Nq, _ = q.shape
    want = {"q": (tuple(q.shape), torch.bfloat16, "cuda"),
            "k": (tuple(k.shape), torch.bfloat16, "cuda"),
            "v": (tuple(v.shape), torch.bfloat16, "cuda"),
            "o": (tuple(q.shape), torch.bfloat16, "cuda"),
            "lse": ((B, Hq, Nq), torch.float32, "cuda"),
            "o_h": (tuple(q.shape), torch.bfloat16, "cpu"),
            "lse_h": ((B, Hq, Nq), torch.float32, "cpu")}
    for name, (shape, dtype, kind) in want.items():
        t = bufs.get(name)
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"bufs[{name!r}] is missing")
        if tuple(t.shape) != shape:
            raise ValueError(f"bufs[{name!r}] must have shape {shape}, "
                             f"not {tuple(t.shape)}")
        if t.dtype != dtype:
            raise TypeError(f"bufs[{name!r}] must be {dtype}")
        if not t.is_contiguous():
            raise ValueError(f"bufs[{name!r}] must be contiguous")
    dev = None
    for name, (shape, dtype, kind) in want.items():
        t = bufs[name]
        if t.device.type != kind:
            raise ValueError(f"bufs[{name!r}] must be a {kind} tensor")
        if kind == "cuda":
            if dev is None:
                dev = t.device
            elif t.device != dev:
                raise ValueError("the device buffers must share one device")
    return dev


def fwd_host(q, k, v, scale=None, causal=False, device="cuda", bufs=None):
    """Forward on host tensors through ``fa_fwd_host``: the library copies
    Q, K, V in, runs the forward and copies O and LSE out, overlapping the
    copies with the computation chunk by chunk.

    ``q, k, v`` are CPU bf16 tensors (page-locked for the copies to
    overlap).  ``bufs`` may hold preallocated device buffers (q, k, v, o,
    lse) and pinned host outputs (o_h, lse_h) to reuse across calls
    (``host_buffers``).  Returns the host (o, lse); the call synchronises
    the current stream before returning.
    """
    _check_host(q, k, v)
    if bufs is None:
        bufs = host_buffers(q, k, v, device)
    dev = _check_host_bufs(bufs, q, k, v)
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    # the library works on the current device: make it the buffers' one
    # (entering the device context only when it differs: the call is
    # timed end to end, and the context costs microseconds)
    ctx = (contextlib.nullcontext() if torch.cuda.current_device() == dev.index
           else torch.cuda.device(dev))
    with ctx:
        stream = torch.cuda.current_stream(dev)
        st = int(load().fa_fwd_host(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), bufs["o_h"].data_ptr(),
            bufs["lse_h"].data_ptr(), bufs["q"].data_ptr(),
            bufs["k"].data_ptr(), bufs["v"].data_ptr(), bufs["o"].data_ptr(),
            bufs["lse"].data_ptr(), B, Hq, Hkv, Nq, Nkv, D, scale,
            1 if causal else 0, stream.cuda_stream))
        if st != FA_OK:
            raise FAError(st, "fa_fwd_host")
        stream.synchronize()
    return bufs["o_h"], bufs["lse_h"]


def host_buffers(q, k, v, device="cuda"):
    """Device inputs/outputs and pinned host outputs for ``fwd_host``."""
    B, Hq, Nq, D = q.shape
    return {
        "q": torch.empty(q.shape, dtype=q.dtype, device=device),
        "k": torch.empty(k.shape, dtype=k.dtype, device=device),
        "v": torch.empty(v.shape, dtype=v.dtype, device=device),
        "o": torch.empty(q.shape, dtype=q.dtype, device=device),
        "lse": torch.empty(B, Hq, Nq, dtype=torch.float32, device=device),
        "o_h": torch.empty(q.shape, dtype=q.dtype).pin_memory(),
        "lse_h": torch.empty(B, Hq, Nq, dtype=torch.float32).pin_memory(),
    }
