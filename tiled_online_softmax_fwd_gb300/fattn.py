"""ctypes binding of libfattn's C ABI (include/fattn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch supplies device memory and streams.  The checks mirror the
wrapper of "Triton programming template" (device, shape, dtype, contiguity)
so that misuse raises in Python before the C layer sees it; the C layer
checks again and is the authority.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libfattn.so")

FATTN_OK = 0
STATUS_NAMES = {0: "FATTN_OK", 1: "FATTN_ERR_INVALID_ARG", 2: "FATTN_ERR_UNSUPPORTED",
                3: "FATTN_ERR_CUDA", 4: "FATTN_ERR_TIMEOUT", 5: "FATTN_ERR_RANGE"}
EXPORTED = ["attn_bwd", "attn_bwd_workspace_size", "attn_fwd", "attn_fwd_fp16", "attn_fwd_host",
            "attn_fwd_kv", "attn_fwd_kv_workspace_size", "attn_fwd_simt", "attn_fwd_strided",
            "attn_fwd_split",
            "attn_fwd_split_count", "attn_fwd_split_noalloc", "attn_fwd_split_workspace_size",
            "fattn_status_string",
            "fattn_last_cuda_error", "fattn_get_device_status", "fattn_row_sum",
            "fattn_selftest_wait_timeout", "fattn_set_v_conversion", "fattn_softmax_rows",
            "fattn_trim_scratch", "fattn_v_conversion_route", "fattn_version"]
V_CONVERT = {"auto": 0, "on_chip": 1, "prepass": 2}

_lib = None
_lock = threading.Lock()


class FattnError(RuntimeError):
    """A libfattn call returned a status other than FATTN_OK."""

    def __init__(self, status: int, what: str, cuda_error: int = 0):
        name = STATUS_NAMES.get(status, "status %d" % status)
        msg = "%s: %s" % (what, name)
        if cuda_error:
            msg += " (CUDA error %d)" % cuda_error
        super().__init__(msg)
        self.status = status
        self.cuda_error = cuda_error


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libfattn.so (raises if it has not been built: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                "libfattn.so is not built (%s); run `python -m tiled_online_softmax_fwd_gb300.build`"
                % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        vp, ip, fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fwd_args = [vp, vp, vp, vp, vp, ip, ip, ip, ip, fp, ip, vp]
        for name in ("attn_fwd", "attn_fwd_fp16", "attn_fwd_simt"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = fwd_args
        lib.attn_fwd_split.restype = ctypes.c_int
        lib.attn_fwd_split.argtypes = fwd_args[:-1] + [ip, vp, ctypes.c_size_t, vp]
        lib.attn_fwd_split_noalloc.restype = ctypes.c_int
        lib.attn_fwd_split_noalloc.argtypes = fwd_args[:-1] + [ip, vp]
        lib.attn_fwd_split_count.restype = ctypes.c_int
        lib.attn_fwd_split_count.argtypes = [ip, ip, ip, ip, ip]
        lib.attn_fwd_split_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_split_workspace_size.argtypes = [ip, ip, ip, ip, ip]
        lib.attn_fwd_kv.restype = ctypes.c_int
        lib.attn_fwd_kv.argtypes = [vp] * 5 + [ip] * 5 + [fp, ip, ip, vp, ctypes.c_size_t, vp]
        i64p = ctypes.POINTER(ctypes.c_longlong)
        lib.attn_fwd_strided.restype = ctypes.c_int
        lib.attn_fwd_strided.argtypes = [vp] * 5 + [ip] * 5 + [i64p] * 4 + [
            fp, ip, ip, vp, ctypes.c_size_t, ip, vp]
        lib.attn_fwd_kv_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_kv_workspace_size.argtypes = [ip] * 7
        lib.attn_bwd.restype = ctypes.c_int
        lib.attn_bwd.argtypes = [vp] * 9 + [ip, ip, ip, ip, fp, ip, vp, ctypes.c_size_t, vp]
        lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.attn_bwd_workspace_size.argtypes = [ip, ip, ip, ip]
        lib.attn_fwd_host.restype = ctypes.c_int
        lib.attn_fwd_host.argtypes = [vp] * 10 + [ip, ip, ip, ip, fp, ip, vp]
        lib.fattn_status_string.restype = ctypes.c_char_p
        lib.fattn_status_string.argtypes = [ctypes.c_int]
        lib.fattn_last_cuda_error.restype = ctypes.c_int
        lib.fattn_last_cuda_error.argtypes = []
        lib.fattn_get_device_status.restype = ctypes.c_int
        lib.fattn_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), vp]
        lib.fattn_selftest_wait_timeout.restype = ctypes.c_int
        lib.fattn_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
        for name in ("fattn_softmax_rows", "fattn_row_sum"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [vp, vp, ip, ip, ip, vp]
        lib.fattn_version.restype = ctypes.c_char_p
        lib.fattn_version.argtypes = []
        lib.fattn_set_v_conversion.restype = ctypes.c_int
        lib.fattn_set_v_conversion.argtypes = [ip]
        lib.fattn_trim_scratch.restype = ctypes.c_int
        lib.fattn_trim_scratch.argtypes = []
        lib.fattn_v_conversion_route.restype = ctypes.c_int
        lib.fattn_v_conversion_route.argtypes = [ip, ip, ip]
        _lib = lib
        return lib


def _check(status: int, what: str):
    if status != FATTN_OK:
        cuda_err = load().fattn_last_cuda_error() if status == 3 else 0
        raise FattnError(status, what, cuda_err)


def default_scale(d: int) -> float:
    """1/sqrt(d) rounded to the fp32 value the kernel receives."""
    return float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _validate(q, k, v, dtype=torch.bfloat16):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a torch.Tensor" % name)
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
        if t.dtype != dtype:
            raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
        if t.dim() != 4:
            raise ValueError("%s must be [B, H, N, d]" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v shapes differ: %s %s %s" % (q.shape, k.shape, v.shape))
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v are on different devices")
    if q.shape[-1] not in (64, 96, 128, 256):
        raise ValueError("head dimension must be 64, 96, 128 or 256, got %d" % q.shape[-1])


def _forward(entry: str, q, k, v, causal, scale, out, lse, stream):
    dtype = torch.float16 if entry == "attn_fwd_fp16" else torch.bfloat16
    _validate(q, k, v, dtype)
    B, H, N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != dtype or not out.is_contiguous() \
            or out.device != q.device:
        raise ValueError("out must be a contiguous tensor of q's type and shape on q's device")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous() \
            or lse.device != q.device:
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor on q's device")
    lib = load()
    with torch.cuda.device(q.device):
        st = getattr(lib, entry)(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 lse.data_ptr(), B, H, N, d, float(scale), 1 if causal else 0,
                                 _stream_handle(stream, q.device))
    _check(st, entry)
    return out, lse


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
             stream=None):
    """O, lse = attention forward of bf16 [B, H, N, d] CUDA tensors (libfattn attn_fwd).

    scale defaults to 1/sqrt(d).  ``out`` / ``lse`` may be preallocated.  The
    kernel is enqueued on ``stream`` (default: the current stream)."""
    return _forward("attn_fwd", q, k, v, causal, scale, out, lse, stream)


def split_count(B: int, H: int, N: int, d: int, causal: bool, device=None) -> int:
    """Key-range splits the library would use for this shape on the device."""
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        n = lib.attn_fwd_split_count(B, H, N, d, 1 if causal else 0)
    if n < 1:
        raise FattnError(1, "attn_fwd_split_count")
    return n


def split_workspace_size(B: int, H: int, N: int, d: int, num_splits: int) -> int:
    return int(load().attn_fwd_split_workspace_size(B, H, N, d, num_splits))


def attn_fwd_split(q, k, v, causal: bool = False, scale: float | None = None,
                   num_splits: int | None = None, workspace=None, out=None, lse=None,
                   stream=None):
    """attn_fwd with the keys of every Q-tile pair split over num_splits CTAs
    (default: the library's choice for the device) and merged by a combine
    kernel.  ``workspace`` is a CUDA uint8 tensor of at least
    split_workspace_size(...) bytes; when omitted, one is allocated here with
    torch (the library itself takes only the V pre-pass scratch, see
    set_v_conversion)."""
    _validate(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    if num_splits is None:
        num_splits = split_count(B, H, N, d, causal, q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    need = split_workspace_size(B, H, N, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if need > 0 else 0
    lib = load()
    with torch.cuda.device(q.device):
        st = lib.attn_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, H, N, d, float(scale), 1 if causal else 0,
                                int(num_splits), ws_ptr, workspace.numel(),
                                _stream_handle(stream, q.device))
    _check(st, "attn_fwd_split")
    return out, lse


def kv_workspace_size(B: int, H: int, Nq: int, Nk: int, d: int, causal: bool,
                      num_splits: int = 0) -> int:
    """Scratch bytes attn_fwd_kv needs (num_splits 0: the library's schedule
    on the current device)."""
    return int(load().attn_fwd_kv_workspace_size(B, H, Nq, Nk, d, 1 if causal else 0,
                                                 num_splits))


def attn_fwd_kv(q, k, v, causal: bool = False, scale: float | None = None,
                num_splits: int = 0, workspace=None, out=None, lse=None, stream=None):
    """Queries q [B, H, Nq, d] against keys and values k, v [B, H, Nk, d]
    (libfattn attn_fwd_kv).  Under the causal mask the queries are the last Nq
    key positions.  num_splits 0 lets the library choose the key-range split;
    the scratch is allocated here with torch when not given."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 \
                or t.dim() != 4 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous 4-D bf16 CUDA tensor" % name)
    if k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B,H,Nq,d] and k, v [B,H,Nk,d] do not match: %s %s %s"
                         % (q.shape, k.shape, v.shape))
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v are on different devices")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = default_scale(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        need = kv_workspace_size(B, H, Nq, Nk, d, causal, num_splits)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        st = load().attn_fwd_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, H, Nq, Nk, d, float(scale), 1 if causal else 0,
                                int(num_splits), workspace.data_ptr() if need > 0 else 0,
                                workspace.numel(), _stream_handle(stream, q.device))
    _check(st, "attn_fwd_kv")
    return out, lse


def attn_fwd_strided(q, k, v, causal: bool = False, scale: float | None = None,
                     num_splits: int = 0, workspace=None, out=None, lse=None, stream=None,
                     bf16_p: bool = False):
    """attn_fwd_kv on 4-D bf16 or fp16 views [B, H, Nq|Nk, d] with any
    strides whose last dimension is contiguous (libfattn attn_fwd_strided):
    e.g. q, k, v sliced from one packed projection output.  ``out`` may be a
    strided view too; by default a contiguous one is allocated.  ``bf16_p``
    (bf16 only) rounds P to bf16 instead of fp16, for V of any bf16
    magnitude (dtype 2)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dim() != 4 \
                or t.dtype not in (torch.bfloat16, torch.float16) or t.stride(3) != 1 \
                or t.dtype != q.dtype:
            raise ValueError("%s must be a 4-D bf16 or fp16 CUDA tensor (all of one type) with "
                             "a contiguous last dimension" % name)
    if k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B,H,Nq,d] and k, v [B,H,Nk,d] do not match: %s %s %s"
                         % (q.shape, k.shape, v.shape))
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = default_scale(d)
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=q.dtype, device=q.device)
    if out.shape != q.shape or out.dtype != q.dtype or out.stride(3) != 1:
        raise ValueError("out must be a [B, H, Nq, d] view of q's type with a contiguous last "
                         "dimension")
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)

    def strides(t):
        return (ctypes.c_longlong * 3)(*t.stride()[:3])
    with torch.cuda.device(q.device):
        need = kv_workspace_size(B, H, Nq, Nk, d, causal, num_splits)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        st = load().attn_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                     lse.data_ptr(), B, H, Nq, Nk, d, strides(q), strides(k),
                                     strides(v), strides(out), float(scale),
                                     1 if causal else 0, int(num_splits),
                                     workspace.data_ptr() if need > 0 else 0, workspace.numel(),
                                     1 if q.dtype == torch.float16 else (2 if bf16_p else 0),
                                     _stream_handle(stream, q.device))
    _check(st, "attn_fwd_strided")
    return out, lse


def attn_bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
             workspace=None, dq=None, dk=None, dv=None, stream=None):
    """Gradients (dq, dk, dv) of attn_fwd for the upstream gradient dout, from
    the forward's inputs and saved outputs o, lse (libfattn attn_bwd).  The
    scratch for D = rowsum(dO * O) is allocated here with torch when not
    given (the library itself never allocates)."""
    _validate(q, k, v)
    B, H, N, d = q.shape
    if d not in (64, 128):
        raise ValueError("the backward takes head dimension 64 or 128, got %d" % d)
    for name, t in (("o", o), ("dout", dout)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous() \
                or t.device != q.device:
            raise ValueError("%s must be a contiguous bf16 tensor shaped like q" % name)
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    if scale is None:
        scale = default_scale(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = int(load().attn_bwd_workspace_size(B, H, N, d))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        st = load().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                             dv.data_ptr(), B, H, N, d, float(scale), 1 if causal else 0,
                             workspace.data_ptr(), workspace.numel(),
                             _stream_handle(stream, q.device))
    _check(st, "attn_bwd")
    return dq, dk, dv


def attn_fwd_fp16(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                  stream=None):
    """attn_fwd for fp16 [B, H, N, d] CUDA tensors (libfattn attn_fwd_fp16)."""
    return _forward("attn_fwd_fp16", q, k, v, causal, scale, out, lse, stream)


def attn_fwd_simt(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                  stream=None):
    """Same as attn_fwd through the plain SIMT cross-check kernel."""
    return _forward("attn_fwd_simt", q, k, v, causal, scale, out, lse, stream)


def attn_fwd_host(q_host, k_host, v_host, o_host, lse_host, dq, dk, dv, do, dlse,
                  causal: bool = False, scale: float | None = None, stream=None):
    """End-to-end call on host tensors through libfattn attn_fwd_host: copy in,
    compute, copy out, synchronise.  Host tensors should be pinned; the device
    tensors are the caller's buffers of matching shape."""
    B, H, N, d = q_host.shape
    for t in (q_host, k_host, v_host, o_host, lse_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors")
    for t in (q_host, k_host, v_host, o_host):
        if t.dtype != torch.bfloat16 or t.shape != (B, H, N, d):
            raise ValueError("host q/k/v/o must be bf16 [B, H, N, d]")
    if lse_host.dtype != torch.float32 or lse_host.shape != (B, H, N):
        raise ValueError("host lse must be fp32 [B, H, N]")
    _validate(dq, dk, dv)
    if scale is None:
        scale = default_scale(d)
    lib = load()
    with torch.cuda.device(dq.device):
        st = lib.attn_fwd_host(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(),
                               o_host.data_ptr(), lse_host.data_ptr(), dq.data_ptr(),
                               dk.data_ptr(), dv.data_ptr(), do.data_ptr(), dlse.data_ptr(),
                               B, H, N, d, float(scale), 1 if causal else 0,
                               _stream_handle(stream, dq.device))
    _check(st, "attn_fwd_host")
    return o_host, lse_host


def device_status(stream=None, device=None) -> int:
    """Read and clear the device status word (0 = no kernel reported a problem)."""
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    word = ctypes.c_int(0)
    with torch.cuda.device(dev):
        st = lib.fattn_get_device_status(ctypes.byref(word), _stream_handle(stream, dev))
    if st not in (FATTN_OK, 4, 5):
        _check(st, "fattn_get_device_status")
    return word.value


def selftest_wait_timeout(limit_us: int = 20000, stream=None, device=None):
    """Launch the failure-path self-test (a wait nothing satisfies, bounded by
    limit_us); read the result with device_status() after it completes."""
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        st = lib.fattn_selftest_wait_timeout(int(limit_us), _stream_handle(stream, dev))
    _check(st, "fattn_selftest_wait_timeout")


_DTYPES = {torch.float32: 0, torch.bfloat16: 1}


def _rowop_input(x):
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [M, N] tensor")
    if x.dtype not in _DTYPES:
        raise ValueError("x must be float32 or bfloat16")
    return x.shape[0], x.shape[1], _DTYPES[x.dtype]


def softmax_rows(x, out=None, stream=None):
    """Row softmax of a contiguous [M, N] fp32/bf16 CUDA tensor (out may be x)."""
    M, N, dt = _rowop_input(x)
    if out is None:
        out = torch.empty_like(x)
    if out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must match x")
    with torch.cuda.device(x.device):
        st = load().fattn_softmax_rows(x.data_ptr(), out.data_ptr(), M, N, dt,
                                       _stream_handle(stream, x.device))
    _check(st, "fattn_softmax_rows")
    return out


def row_sum(x, out=None, stream=None):
    """fp32 sums of the rows of a contiguous [M, N] fp32/bf16 CUDA tensor."""
    M, N, dt = _rowop_input(x)
    if out is None:
        out = torch.empty(M, dtype=torch.float32, device=x.device)
    if out.shape != (M,) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous fp32 [M] tensor")
    with torch.cuda.device(x.device):
        st = load().fattn_row_sum(x.data_ptr(), out.data_ptr(), M, N, dt,
                                  _stream_handle(stream, x.device))
    _check(st, "fattn_row_sum")
    return out


def version() -> str:
    return load().fattn_version().decode()


def set_v_conversion(mode: str) -> str:
    """Where bf16 calls with fp16 P round V to fp16: "auto", "on_chip" or
    "prepass" (fattn_set_v_conversion).  Returns the previous setting."""
    if mode not in V_CONVERT:
        raise ValueError("mode must be one of %s" % sorted(V_CONVERT))
    prev = load().fattn_set_v_conversion(V_CONVERT[mode])
    return {v: k for k, v in V_CONVERT.items()}[prev]


def v_conversion_route(N: int, d: int, causal: bool) -> str:
    """Where a bf16 call with N queries per head, head dimension d and the
    given mask rounds V under the current setting: "on_chip" or "prepass"
    (fattn_v_conversion_route)."""
    r = load().fattn_v_conversion_route(N, d, 1 if causal else 0)
    if r < 0:
        raise ValueError("unsupported N=%d, d=%d" % (N, d))
    return {v: k for k, v in V_CONVERT.items()}[r]


class v_conversion:
    """Context manager: set_v_conversion(mode) inside, the previous setting after."""

    def __init__(self, mode: str):
        self.mode = mode

    def __enter__(self):
        self.prev = set_v_conversion(self.mode)
        return self

    def __exit__(self, *exc):
        set_v_conversion(self.prev)


def trim_scratch():
    """Give the V pre-pass pool's unused device memory back (fattn_trim_scratch)."""
    _check(load().fattn_trim_scratch(), "fattn_trim_scratch")


def raw_call(entry: str, *args) -> int:
    """Call a C entry point with raw integer/float arguments and return its
    status (used by the boundary tests to probe argument checking)."""
    return getattr(load(), entry)(*args)
