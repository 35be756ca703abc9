"""ctypes binding of liblla.so: the C-ABI entry points under the same names.

Every function here only checks and marshals arguments (device pointers, sizes, the current
torch stream) and calls the library; all arithmetic runs in liblla's CUDA kernels. There is no
fallback: if the library is missing or the tensors are not on a CUDA device the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "LlaError", "library_path", "lla_forward", "lla_forward_ws", "lla_workspace_size",
    "lla_forward_host", "lla_moments", "lla_stream_status", "lla_status_string", "lla_version",
    "launch_count", "profile_enable", "profile_collect", "EXPORTED_SYMBOLS", "DTYPE_CODES",
    "lla_forward_noalloc", "NOALLOC_SCRATCH_BYTES", "PATH_AUTO", "PATH_CUDA_CORE",
    "PATH_TENSOR_CORE", "PATH_CG", "lla_parallax_forward", "lla_decode", "lla_parallax_decode",
    "FORM_CENTRED", "FORM_PAGE", "FAULT_WITHHOLD_KEYS", "lla_parallax_backward", "Options",
]

LLA_OK = 0
DTYPE_CODES = {torch.float32: 0, torch.bfloat16: 1}
NUM_STAGES = 5
STAGE_NAMES = ("prep", "weights", "moments", "solve", "readout")

# Every function include/lla.h declares.
EXPORTED_SYMBOLS = (
    "lla_forward", "lla_workspace_size", "lla_forward_ws", "lla_forward_host", "lla_moments",
    "lla_stream_status", "lla_status_string", "lla_version", "lla_launch_count",
    "lla_profile_enable", "lla_profile_collect", "lla_forward_noalloc", "lla_decode",
    "lla_parallax_decode", "lla_parallax_forward", "lla_parallax_backward", "lla_forward_ex",
    "lla_parallax_forward_ex", "lla_decode_ex", "lla_parallax_decode_ex",
    "lla_parallax_backward_ex",
)

# LLA_NOALLOC_SCRATCH_BYTES in include/lla.h: the fixed scratch of lla_forward_noalloc.
NOALLOC_SCRATCH_BYTES = 64 << 20

_lib = None

PATH_AUTO, PATH_CUDA_CORE, PATH_TENSOR_CORE, PATH_CG = 0, 1, 2, 3
FORM_CENTRED, FORM_PAGE = 0, 1
FAULT_WITHHOLD_KEYS = 1


class Options(ctypes.Structure):
    """lla_options: per-call choices of the *_ex entry points (all zero = the defaults)."""
    _fields_ = [("path", ctypes.c_int), ("form", ctypes.c_int), ("cg_max_iters", ctypes.c_int),
                ("cg_rel_tol", ctypes.c_float), ("test_fault", ctypes.c_int),
                ("reserved", ctypes.c_int * 3)]


def _options(path=0, form=0, cg=None, test_fault=0):
    """An Options struct, or None when every choice is the default (the plain entry point)."""
    if not path and not form and cg is None and not test_fault:
        return None
    o = Options()
    o.path, o.form, o.test_fault = int(path), int(form), int(test_fault)
    if cg is not None:
        o.cg_max_iters, o.cg_rel_tol = int(cg[0]), float(cg[1])
    return o


class LlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lla_status_string(status)} (status {status})")


def library_path() -> str:
    return os.environ.get("LLA_LIBRARY",
                          os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblla.so"))


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"liblla.so not found at {path}; build it with "
                          "`python -m local_linear_attention_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fp = ctypes.POINTER(ctypes.c_float)
    op = ctypes.POINTER(Options)
    sig = {
        "lla_forward": (i, [vp, vp, vp, vp, i, i, i, i, i, f, f, i, vp]),
        "lla_workspace_size": (sz, [i, i, i, i, i, i]),
        "lla_forward_ws": (i, [vp, vp, vp, vp, i, i, i, i, i, f, f, i, vp, sz, vp]),
        "lla_forward_host": (i, [vp, vp, vp, vp, i, i, i, i, i, f, f, i, vp]),
        "lla_moments": (i, [vp, vp, vp, vp, i, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]),
        "lla_stream_status": (i, [vp]),
        "lla_status_string": (ctypes.c_char_p, [i]),
        "lla_version": (i, []),
        "lla_launch_count": (ctypes.c_ulonglong, []),
        "lla_profile_enable": (i, [i]),
        "lla_profile_collect": (i, [fp, i, ctypes.POINTER(ctypes.c_int)]),
        "lla_forward_noalloc": (i, [vp, vp, vp, vp, i, i, i, i, i, f, f, i, vp]),
        "lla_parallax_forward": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]),
        "lla_decode": (i, [vp, vp, vp, vp, i, i, i, i, i, f, f, i, vp]),
        "lla_parallax_decode": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]),
        "lla_parallax_backward": (i, [vp] * 9 + [i, i, i, i, i, f, i, vp]),
        "lla_forward_ex": (i, [vp, vp, vp, vp, i, i, i, i, i, f, f, i, op, vp, sz, vp]),
        "lla_parallax_forward_ex": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, op, vp]),
        "lla_decode_ex": (i, [vp, vp, vp, vp, i, i, i, i, i, f, f, i, op, vp]),
        "lla_parallax_decode_ex": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, op, vp]),
        "lla_parallax_backward_ex": (i, [vp] * 9 + [i, i, i, i, i, f, i, op, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def lla_status_string(status: int) -> str:
    return _load().lla_status_string(int(status)).decode()


def lla_version() -> int:
    return _load().lla_version()


def launch_count() -> int:
    return int(_load().lla_launch_count())


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(st: int, where: str):
    if st != LLA_OK:
        raise LlaError(st, where)


def _shapes(q, k, v):
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("expected q, k [B,H,T,d] and v [B,H,T,dv]")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in DTYPE_CODES:
        raise ValueError("q, k, v must share one dtype: float32 or bfloat16")
    B, H, T, d = q.shape
    return B, H, T, d, v.shape[3], DTYPE_CODES[q.dtype]


def _device_inputs(q, k, v):
    for t in (q, k, v):
        if not t.is_cuda:
            raise ValueError("liblla runs on CUDA tensors only")
        if not t.is_contiguous():
            raise ValueError("inputs must be contiguous")
    return _shapes(q, k, v)


def _check_out(out, shape, like):
    if (tuple(out.shape) != tuple(shape) or out.dtype != like.dtype or out.device != like.device
            or not out.is_contiguous()):
        raise ValueError(f"out must be a contiguous tensor of shape {tuple(shape)}, dtype "
                         f"{like.dtype} on {like.device}")


def lla_forward(q, k, v, h: float, lam: float, out=None, stream=None, *, path=0, form=0, cg=None,
                test_fault=0, workspace=None):
    """Causal LLA forward on device tensors; returns `out` ([B,H,T,dv], dtype of the inputs).

    path / form / cg=(max_iters, rel_tol) / test_fault are this call's lla_options (defaults:
    automatic path, centred form); with any of them, or a workspace tensor, the call goes through
    lla_forward_ex, otherwise through lla_forward."""
    B, H, T, d, dv, code = _device_inputs(q, k, v)
    if out is None:
        out = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device)
    _check_out(out, (B, H, T, dv), q)
    opts = _options(path, form, cg, test_fault)
    if opts is None and workspace is None:
        st = _load().lla_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H,
                                 T, d, dv, float(h), float(lam), code, _stream_ptr(stream))
        _check(st, "lla_forward")
        return out
    wp, wb = (None, 0) if workspace is None else (
        workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = _load().lla_forward_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, T,
                                d, dv, float(h), float(lam), code,
                                ctypes.byref(opts) if opts is not None else None, wp, wb,
                                _stream_ptr(stream))
    _check(st, "lla_forward_ex")
    return out


def lla_parallax_forward(q, k, v, r, h: float, out=None, stream=None, *, path=0):
    """Causal Parallax forward with probe r ([B,H,T,d], like q); returns `out` ([B,H,T,dv]).
    path=PATH_CUDA_CORE forces the CUDA-core kernel (lla_parallax_forward_ex)."""
    B, H, T, d, dv, code = _device_inputs(q, k, v)
    if r.shape != q.shape or r.dtype != q.dtype or not r.is_cuda or not r.is_contiguous():
        raise ValueError("r must be a contiguous CUDA tensor shaped and typed like q")
    if out is None:
        out = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device)
    _check_out(out, (B, H, T, dv), q)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), r.data_ptr(), out.data_ptr(), B, H, T, d,
            dv, float(h), code)
    opts = _options(path)
    if opts is None:
        st = _load().lla_parallax_forward(*args, _stream_ptr(stream))
    else:
        st = _load().lla_parallax_forward_ex(*args, ctypes.byref(opts), _stream_ptr(stream))
    _check(st, "lla_parallax_forward")
    return out


def _decode_inputs(q, k, v):
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    if q.dim() != 3 or k.dim() != 4 or v.dim() != 4 or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("decode expects q [B,H,d], k [B,H,L,d], v [B,H,L,dv] of one dtype")
    B, H, d = q.shape
    if k.shape[:2] != (B, H) or k.shape[3] != d or v.shape[:3] != k.shape[:3]:
        raise ValueError("inconsistent decode shapes")
    if q.dtype not in DTYPE_CODES:
        raise ValueError("dtype must be float32 or bfloat16")
    return B, H, k.shape[2], d, v.shape[3], DTYPE_CODES[q.dtype]


def lla_decode(q, k, v, h: float, lam: float, out=None, stream=None, *, path=0):
    """LLA decode: q [B,H,d] against the cache k [B,H,L,d], v [B,H,L,dv]; returns [B,H,dv].
    path=PATH_CUDA_CORE forces the CUDA-core split kernel (lla_decode_ex)."""
    B, H, L, d, dv, code = _decode_inputs(q, k, v)
    if out is None:
        out = torch.empty(B, H, dv, dtype=q.dtype, device=q.device)
    _check_out(out, (B, H, dv), q)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, L, d, dv, float(h),
            float(lam), code)
    opts = _options(path)
    if opts is None:
        st = _load().lla_decode(*args, _stream_ptr(stream))
    else:
        st = _load().lla_decode_ex(*args, ctypes.byref(opts), _stream_ptr(stream))
    _check(st, "lla_decode")
    return out


def lla_parallax_decode(q, k, v, r, h: float, out=None, stream=None, *, path=0):
    """Parallax decode with probe r [B,H,d] (like q); returns [B,H,dv]."""
    B, H, L, d, dv, code = _decode_inputs(q, k, v)
    if r.shape != q.shape or r.dtype != q.dtype or not r.is_cuda or not r.is_contiguous():
        raise ValueError("r must be a contiguous CUDA tensor shaped and typed like q")
    if out is None:
        out = torch.empty(B, H, dv, dtype=q.dtype, device=q.device)
    _check_out(out, (B, H, dv), q)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), r.data_ptr(), out.data_ptr(), B, H, L, d,
            dv, float(h), code)
    opts = _options(path)
    if opts is None:
        st = _load().lla_parallax_decode(*args, _stream_ptr(stream))
    else:
        st = _load().lla_parallax_decode_ex(*args, ctypes.byref(opts), _stream_ptr(stream))
    _check(st, "lla_parallax_decode")
    return out


def lla_parallax_backward(q, k, v, r, dout, h: float, stream=None, *, path=0):
    """Gradients (dq, dk, dv, dr) of the causal Parallax forward for the upstream gradient dout
    ([B,H,T,dv], like the forward's output); each is shaped and typed like q, k, v, r."""
    B, H, T, d, dv, code = _device_inputs(q, k, v)
    for name, x, like in (("r", r, q), ("dout", dout, None)):
        shape = q.shape if like is not None else (B, H, T, dv)
        if tuple(x.shape) != tuple(shape) or x.dtype != q.dtype or not x.is_cuda \
                or not x.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor of shape {tuple(shape)} "
                             f"and dtype {q.dtype}")
    dq, dk, dvv, dr = (torch.empty_like(x) for x in (q, k, v, r))
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), r.data_ptr(), dout.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dvv.data_ptr(), dr.data_ptr(), B, H, T, d, dv, float(h),
            code)
    opts = _options(path)
    if opts is None:
        st = _load().lla_parallax_backward(*args, _stream_ptr(stream))
    else:
        st = _load().lla_parallax_backward_ex(*args, ctypes.byref(opts), _stream_ptr(stream))
    _check(st, "lla_parallax_backward")
    return dq, dk, dvv, dr


def lla_forward_noalloc(q, k, v, h: float, lam: float, out, stream=None):
    """lla_forward for callers that must not allocate device memory: the library's fixed scratch
    array is used, and `out` (a preallocated contiguous [B,H,T,dv] tensor of q's dtype on q's
    device) is required. The call runs with q's device current, so that the scratch array of
    that device is the one used."""
    B, H, T, d, dv, code = _device_inputs(q, k, v)
    if not (k.device == q.device and v.device == q.device):
        raise ValueError("q, k, v must be on one device")
    _check_out(out, (B, H, T, dv), q)
    with torch.cuda.device(q.device):
        st = _load().lla_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                         B, H, T, d, dv, float(h), float(lam), code,
                                         _stream_ptr(stream))
    _check(st, "lla_forward_noalloc")
    return out


def lla_workspace_size(B, H, T, d, dv, dtype) -> int:
    code = DTYPE_CODES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(_load().lla_workspace_size(B, H, T, d, dv, code))


def lla_forward_ws(q, k, v, h: float, lam: float, workspace, out=None, stream=None):
    """lla_forward with a caller-owned device workspace (a uint8 CUDA tensor)."""
    B, H, T, d, dv, code = _device_inputs(q, k, v)
    if out is None:
        out = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device)
    _check_out(out, (B, H, T, dv), q)
    st = _load().lla_forward_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, T,
                                d, dv, float(h), float(lam), code, workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(st, "lla_forward_ws")
    return out


def lla_forward_host(q, k, v, h: float, lam: float, out=None, stream=None):
    """End-to-end forward on HOST tensors (copies in, computes, copies out, synchronises)."""
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("lla_forward_host takes contiguous CPU tensors")
    B, H, T, d, dv, code = _shapes(q, k, v)
    if out is None:
        out = torch.empty(B, H, T, dv, dtype=q.dtype, pin_memory=q.is_pinned())
    st = _load().lla_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H,
                                  T, d, dv, float(h), float(lam), code, _stream_ptr(stream))
    _check(st, "lla_forward_host")
    return out


def lla_moments(q, k, v, idx, h: float, stream=None):
    """Debug entry: raw max-shifted moments of the queries at flat indices idx (int64 CUDA)."""
    B, H, T, d, dv, code = _device_inputs(q, k, v)
    idx = idx.to(device=q.device, dtype=torch.int64).contiguous()
    n = idx.numel()
    f = dict(dtype=torch.float32, device=q.device)
    res = {"m": torch.empty(n, **f), "omega": torch.empty(n, **f), "sk": torch.empty(n, d, **f),
           "sv": torch.empty(n, dv, **f), "Skk": torch.empty(n, d, d, **f),
           "Svk": torch.empty(n, dv, d, **f)}
    st = _load().lla_moments(q.data_ptr(), k.data_ptr(), v.data_ptr(), idx.data_ptr(), n,
                             *(res[x].data_ptr() for x in ("m", "omega", "sk", "sv", "Skk", "Svk")),
                             B, H, T, d, dv, float(h), code, _stream_ptr(stream))
    _check(st, "lla_moments")
    return res


def lla_stream_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(_load().lla_stream_status(_stream_ptr(stream)))


def profile_enable(on: bool = True):
    _check(_load().lla_profile_enable(1 if on else 0), "lla_profile_enable")


def profile_collect():
    """(summed ms per stage as a dict, number of recorded lla_forward calls)."""
    buf = (ctypes.c_float * NUM_STAGES)()
    n = ctypes.c_int(0)
    _check(_load().lla_profile_collect(buf, NUM_STAGES, ctypes.byref(n)), "lla_profile_collect")
    return dict(zip(STAGE_NAMES, list(buf))), n.value
