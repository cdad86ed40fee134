"""ctypes binding of the C ABI in include/attn.h (argument marshalling only).

Every step of the attention forward runs in the CUDA kernels of
libattn_gb300.so.  torch provides device memory and the current stream; there
is no CPU or library fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libattn_gb300.so"
_lib = None
_lock = threading.Lock()

ATTN_OK = 0
_ERRORS = {-1: "ATTN_ERR_ARG", -2: "ATTN_ERR_ALIGN", -3: "ATTN_ERR_ARCH", -4: "ATTN_ERR_LAUNCH",
           -5: "ATTN_ERR_TIMEOUT", -6: "ATTN_ERR_NOMEM", -7: "ATTN_ERR_DEVICE", -8: "ATTN_ERR_SCRATCH"}


class AttnPlan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("launches", ctypes.c_int), ("grid", ctypes.c_int),
                ("kv_splits", ctypes.c_int), ("d_slices", ctypes.c_int), ("workspace_bytes", ctypes.c_longlong)]


PATH_NAMES = {0: "none", 1: "nokeys", 2: "tc", 3: "tc_splitkv"}


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_ERRORS.get(code, code)}: {attn_strerror(code)}"
                         + (f" ({_last_cuda_error()})" if code == -4 else ""))


def library_path() -> str:
    return os.environ.get("ATTN_GB300_LIB", os.path.join(_PKG, _LIB_NAME))


def load_library() -> ctypes.CDLL:
    """Load libattn_gb300.so once; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it first with "
                              "`python -c 'import __graft_entry__ as g; g.build()'` "
                              "(there is no fallback implementation)")
        lib = ctypes.CDLL(path)
        vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp]
        lib.attn_fwd.restype = ci
        lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
        lib.attn_fwd_splitkv.restype = ci
        lib.attn_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
        lib.attn_fwd_splitkv_noalloc.restype = ci
        ll = ctypes.c_longlong
        lib.attn_fwd_masked.argtypes = [vp, vp, vp, vp, ll, ll, ll, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp]
        lib.attn_fwd_masked.restype = ci
        lib.attn_fp8_quantize.argtypes = [vp] * 9 + [ci] * 6 + [vp]
        lib.attn_fp8_quantize.restype = ci
        lib.attn_fwd_fp8.argtypes = [vp] * 8 + [ci] * 6 + [cf, ci, vp]
        lib.attn_fwd_fp8.restype = ci
        lib.attn_bwd.argtypes = [vp] * 9 + [ci] * 6 + [cf, ci, vp]
        lib.attn_bwd.restype = ci
        lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp]
        lib.attn_fwd_host.restype = ci
        lib.attn_set_debug.argtypes = [ci, ctypes.c_longlong]
        lib.attn_set_debug.restype = ci
        lib.attn_fwd_status.argtypes = [vp]
        lib.attn_fwd_status.restype = ci
        lib.attn_strerror.argtypes = [ci]
        lib.attn_strerror.restype = ctypes.c_char_p
        lib.attn_last_cuda_error.argtypes = []
        lib.attn_last_cuda_error.restype = ctypes.c_char_p
        lib.attn_fwd_plan.argtypes = [ci, ci, ci, ci, ci, ci, ci, ctypes.POINTER(AttnPlan)]
        lib.attn_fwd_plan.restype = ci
        lib.attn_version.argtypes = []
        lib.attn_version.restype = ci
        lib.attn_shutdown.argtypes = []
        lib.attn_shutdown.restype = ci
        _lib = lib
        return lib


def attn_strerror(code: int) -> str:
    return load_library().attn_strerror(int(code)).decode()


def _last_cuda_error() -> str:
    return load_library().attn_last_cuda_error().decode()


def attn_version() -> int:
    return int(load_library().attn_version())


def attn_shutdown() -> None:
    """Give back the device memory of the library's pools: see attn_shutdown in include/attn.h."""
    rc = load_library().attn_shutdown()
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_shutdown")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(t: torch.Tensor, name: str, dtype, ndim: int):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _mask_strides(mask: torch.Tensor, B: int, Hq: int, Nq: int, Nkv: int):
    """Element strides (batch, head, query row) of a bf16 CUDA mask that
    broadcasts to [B, Hq, Nq, Nkv] with contiguous keys; a broadcast or
    size-1 dimension gets stride 0."""
    if mask.dtype != torch.bfloat16:
        raise TypeError(f"mask must be bfloat16, got {mask.dtype}")
    if not mask.is_cuda:
        raise ValueError("mask must be a CUDA tensor")
    if mask.dim() > 4:
        raise ValueError(f"mask must have at most 4 dims, got shape {tuple(mask.shape)}")
    m = mask.reshape((1,) * (4 - mask.dim()) + tuple(mask.shape)).expand(B, Hq, Nq, Nkv)
    if Nkv > 1 and m.stride(3) != 1:
        raise ValueError("mask keys (last dim) must be contiguous")
    strides = [0 if m.shape[d] == 1 else m.stride(d) for d in range(3)]
    if any(st % 8 for st in strides) or m.data_ptr() % 16:
        raise ValueError(f"mask strides {strides} must be multiples of 8 elements and its base 16-byte aligned "
                         "(pad the key dimension to a multiple of 8)")
    return m, strides


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
             causal: bool = False, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
             stream=None, kv_splits: int | None = None, mask: torch.Tensor | None = None):
    """O, LSE = attention forward of bf16 q [B,Hq,Nq,D], k and v [B,Hkv,Nkv,D].

    O is bf16 [B,Hq,Nq,D]; LSE is fp32 [B,Hq,Nq] (natural log).  Runs
    asynchronously on ``stream`` (default: torch's current stream).
    ``kv_splits`` (None/0 = automatic) forces the number of key-range splits
    (attn_fwd_splitkv).  ``mask`` (bf16, broadcastable to [B,Hq,Nq,Nkv],
    keys contiguous) is an additive mask (attn_fwd_masked); it does not
    combine with a forced ``kv_splits``.
    """
    lib = load_library()
    _check(q, "q", torch.bfloat16, 4)
    _check(k, "k", torch.bfloat16, 4)
    _check(v, "v", torch.bfloat16, 4)
    B, Hq, Nq, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError(f"k {tuple(k.shape)} / v {tuple(v.shape)} do not match q {tuple(q.shape)}")
    Hkv, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    _check(out, "out", torch.bfloat16, 4)
    _check(lse, "lse", torch.float32, 3)
    if tuple(out.shape) != (B, Hq, Nq, D) or tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("out / lse shape mismatch")
    with torch.cuda.device(q.device):
        if mask is not None:
            if kv_splits:
                raise ValueError("mask and kv_splits do not combine (attn_fwd_masked splits automatically)")
            m, (sb, sh, sq) = _mask_strides(mask, B, Hq, Nq, Nkv)
            rc = lib.attn_fwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), m.data_ptr(), sb, sh, sq,
                                     out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Nq, Nkv, D, float(scale),
                                     int(bool(causal)), _stream_handle(stream))
        elif kv_splits:
            rc = lib.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                      B, Hq, Hkv, Nq, Nkv, D, float(scale), int(bool(causal)), int(kv_splits),
                                      _stream_handle(stream))
        else:
            rc = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                              B, Hq, Hkv, Nq, Nkv, D, float(scale), int(bool(causal)), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return out, lse


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
             dout: torch.Tensor, scale: float | None = None, causal: bool = False, stream=None,
             dq: torch.Tensor | None = None, dk: torch.Tensor | None = None, dv: torch.Tensor | None = None):
    """dq, dk, dv = gradients of attention forward (attn_bwd of the C ABI).

    q, k, v, o, dout bf16 and lse fp32 as attn_fwd takes and returns them;
    head dim 64 or 128.  Runs asynchronously on ``stream``.
    """
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _check(t, n, torch.bfloat16, 4)
    _check(lse, "lse", torch.float32, 3)
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError(f"k {tuple(k.shape)} / v {tuple(v.shape)} do not match q {tuple(q.shape)}")
    if o.shape != q.shape or dout.shape != q.shape or tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("o / dout / lse shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n, ref in ((dq, "dq", q), (dk, "dk", k), (dv, "dv", v)):
        _check(t, n, torch.bfloat16, 4)
        if t.shape != ref.shape:
            raise ValueError(f"{n} shape mismatch")
    with torch.cuda.device(q.device):
        rc = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Nq, Nkv, D, float(scale),
                          int(bool(causal)), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv


def attn_fp8_quantize(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, stream=None) -> dict:
    """FP8 operands of bf16 q, k, v (head dim 128): attn_fp8_quantize of the
    C ABI.  Returns a dict of q8, k8, vt8 (uint8) and sq, sk, sv (fp32)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, 4)
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError(f"k {tuple(k.shape)} / v {tuple(v.shape)} do not match q {tuple(q.shape)}")
    dev = q.device
    nkb = (Nkv + 127) // 128
    out = {
        "q8": torch.empty((B, Hq, Nq, D), dtype=torch.uint8, device=dev),
        "k8": torch.empty((B, Hkv, Nkv, D), dtype=torch.uint8, device=dev),
        "vt8": torch.empty((B, Hkv, D, nkb * 128), dtype=torch.uint8, device=dev),
        "sq": torch.empty((B, Hq, (Nq + 127) // 128), dtype=torch.float32, device=dev),
        "sk": torch.empty((B, Hkv, nkb), dtype=torch.float32, device=dev),
        "sv": torch.empty((B, Hkv), dtype=torch.float32, device=dev),
    }
    with torch.cuda.device(dev):
        rc = lib.attn_fp8_quantize(q.data_ptr(), k.data_ptr(), v.data_ptr(), out["q8"].data_ptr(),
                                   out["k8"].data_ptr(), out["vt8"].data_ptr(), out["sq"].data_ptr(),
                                   out["sk"].data_ptr(), out["sv"].data_ptr(), B, Hq, Hkv, Nq, Nkv, D,
                                   _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fp8_quantize")
    return out


def attn_fwd_fp8(qz: dict, scale: float | None = None, causal: bool = False, out: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None, stream=None):
    """O, LSE of the FP8 path from attn_fp8_quantize's operands."""
    lib = load_library()
    B, Hq, Nq, D = qz["q8"].shape
    Hkv, Nkv = qz["k8"].shape[1], qz["k8"].shape[2]
    dev = qz["q8"].device
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    _check(out, "out", torch.bfloat16, 4)
    _check(lse, "lse", torch.float32, 3)
    with torch.cuda.device(dev):
        rc = lib.attn_fwd_fp8(qz["q8"].data_ptr(), qz["k8"].data_ptr(), qz["vt8"].data_ptr(), qz["sq"].data_ptr(),
                              qz["sk"].data_ptr(), qz["sv"].data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv,
                              Nq, Nkv, D, float(scale), int(bool(causal)), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp8")
    return out, lse


def _check_host(t: torch.Tensor, name: str, dtype, ndim: int) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def attn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
                  causal: bool = False, device=None, out: torch.Tensor | None = None,
                  lse: torch.Tensor | None = None, stream=None):
    """attn_fwd_host of the C ABI: q, k, v, out and lse are CPU tensors (pin
    them for the copies to overlap the kernels); runs on ``device`` (default:
    the current CUDA device) and returns (O, LSE) on the CPU once they are there."""
    lib = load_library()
    _check_host(q, "q", torch.bfloat16, 4)
    _check_host(k, "k", torch.bfloat16, 4)
    _check_host(v, "v", torch.bfloat16, 4)
    B, Hq, Nq, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError(f"k {tuple(k.shape)} / v {tuple(v.shape)} do not match q {tuple(q.shape)}")
    Hkv, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, pin_memory=q.is_pinned())
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, pin_memory=q.is_pinned())
    _check_host(out, "out", torch.bfloat16, 4)
    _check_host(lse, "lse", torch.float32, 3)
    if tuple(out.shape) != (B, Hq, Nq, D) or tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("out / lse shape mismatch")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        rc = lib.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               B, Hq, Hkv, Nq, Nkv, D, float(scale), int(bool(causal)), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host")
    return out, lse


def attn_fwd_plan(B: int, Hq: int, Hkv: int, Nq: int, Nkv: int, D: int, causal: bool) -> dict:
    """The kernels attn_fwd would launch for these sizes on the current device."""
    plan = AttnPlan()
    rc = load_library().attn_fwd_plan(B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), ctypes.byref(plan))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_plan")
    d = {f: getattr(plan, f) for f, _ in AttnPlan._fields_}
    d["path_name"] = PATH_NAMES.get(plan.path, str(plan.path))
    return d


def attn_set_debug(flags: int = 0, wait_limit_ns: int = 0) -> None:
    """Test support: see attn_set_debug in include/attn.h."""
    rc = load_library().attn_set_debug(int(flags), int(wait_limit_ns))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_set_debug")


def attn_fwd_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(load_library().attn_fwd_status(_stream_handle(stream)))
