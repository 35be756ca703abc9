"""The C-ABI library loads, exports every function include/lla.h declares, and validates its
arguments on the host (CPU only: nothing here enqueues GPU work)."""
import ctypes
import os
import re

import pytest

from local_linear_attention_gb300 import build as lla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lla.h")


@pytest.fixture(scope="module")
def lib():
    path = lla_build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lla_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("lla_forward", "lla_moments", "lla_stream_status", "lla_status_string",
                     "lla_version"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from local_linear_attention_gb300.binding import EXPORTED_SYMBOLS
    names = declared_functions()
    assert sorted(EXPORTED_SYMBOLS) == names
    for name in names:
        assert hasattr(lib, name), name


def test_version_and_strings(lib):
    lib.lla_version.restype = ctypes.c_int
    assert lib.lla_version() == 200
    lib.lla_status_string.restype = ctypes.c_char_p
    for st in range(6):
        assert lib.lla_status_string(st).decode().startswith("LLA_")
    assert lib.lla_status_string(99) is not None


def _fwd(lib, q=1, k=1, v=1, out=1, B=1, H=1, T=4, d=16, dv=16, h=4.0, lam=0.01, dtype=0):
    vp = ctypes.c_void_p
    f = lib.lla_forward
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, vp, vp] + [ctypes.c_int] * 5 + [ctypes.c_float] * 2 + [ctypes.c_int, vp]
    p = lambda x: None if x is None else ctypes.c_void_p(16 * x)  # noqa: E731 (aligned, never dereferenced)
    return f(p(q), p(k), p(v), p(out), B, H, T, d, dv, h, lam, dtype, None)


def test_host_validation_codes(lib):
    INVALID, UNSUPPORTED = 1, 2
    assert _fwd(lib, q=None) == INVALID
    assert _fwd(lib, out=None) == INVALID
    assert _fwd(lib, d=48) == UNSUPPORTED
    assert _fwd(lib, dv=128) == UNSUPPORTED
    assert _fwd(lib, h=0.0) == INVALID
    assert _fwd(lib, h=float("nan")) == INVALID
    assert _fwd(lib, lam=-1.0) == INVALID
    assert _fwd(lib, lam=float("inf")) == INVALID
    assert _fwd(lib, dtype=7) == INVALID
    assert _fwd(lib, T=-1) == INVALID
    assert _fwd(lib, B=1 << 16, H=1 << 16, T=1) == UNSUPPORTED
    # empty problems are a no-op that succeeds without touching any pointer or device
    assert _fwd(lib, q=None, k=None, v=None, out=None, T=0) == 0
    assert _fwd(lib, q=None, k=None, v=None, out=None, B=0) == 0


def test_misaligned_pointer_rejected(lib):
    vp = ctypes.c_void_p
    f = lib.lla_forward
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, vp, vp] + [ctypes.c_int] * 5 + [ctypes.c_float] * 2 + [ctypes.c_int, vp]
    assert f(vp(16), vp(18), vp(32), vp(48), 1, 1, 4, 16, 16, 4.0, 0.01, 0, None) == 1


def test_workspace_size_is_host_only(lib):
    f = lib.lla_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 6
    assert f(1, 1, 0, 16, 16, 0) == 0
    assert f(1, 1, 4, 48, 16, 0) == 0
    small = f(1, 1, 128, 16, 16, 0)
    assert small > 0 and small % 256 == 0
    # bf16 with d < 64 runs on the d = dv = 64 tensor-core path with zero-padded copies of q, k,
    # v and out ahead of that path's scratch
    pad = 4 * ((128 * 64 * 2 + 255) // 256 * 256)
    for d, dv in ((16, 16), (32, 32), (32, 16), (16, 64)):
        assert f(1, 1, 128, d, dv, 1) == f(1, 1, 128, 64, 64, 1) + pad
    assert f(4, 8, 4096, 64, 64, 1) > 1 << 30         # headline shape: > 1 GiB of moments


def test_host_entry_and_moments_validation(lib):
    vp = ctypes.c_void_p
    fh = lib.lla_forward_host
    fh.restype = ctypes.c_int
    fh.argtypes = [vp, vp, vp, vp] + [ctypes.c_int] * 5 + [ctypes.c_float] * 2 + [ctypes.c_int, vp]
    assert fh(None, vp(16), vp(16), vp(16), 1, 1, 4, 16, 16, 4.0, 0.01, 0, None) == 1
    fm = lib.lla_moments
    fm.restype = ctypes.c_int
    fm.argtypes = [vp, vp, vp, vp, ctypes.c_int] + [vp] * 6 + [ctypes.c_int] * 5 + \
        [ctypes.c_float, ctypes.c_int, vp]
    assert fm(vp(16), vp(16), vp(16), None, 3, *([None] * 6), 1, 1, 4, 16, 16, 4.0, 0, None) == 1
    assert fm(vp(16), vp(16), vp(16), vp(16), -1, *([None] * 6), 1, 1, 4, 16, 16, 4.0, 0, None) == 1
    assert fm(None, None, None, None, 0, *([None] * 6), 1, 1, 4, 16, 16, 4.0, 0, None) == 0


def test_launch_counter_starts_at_zero(lib):
    lib.lla_launch_count.restype = ctypes.c_ulonglong
    assert lib.lla_launch_count() == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib
    import local_linear_attention_gb300.binding as b
    monkeypatch.setenv("LLA_LIBRARY", str(tmp_path / "missing.so"))
    monkeypatch.setattr(b, "_lib", None)
    with pytest.raises(ImportError):
        b.lla_version()
    importlib.reload(b)


def _fwd_ex(lib, opts, T=4, d=16, dtype=0):
    from local_linear_attention_gb300.binding import Options
    vp = ctypes.c_void_p
    f = lib.lla_forward_ex
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, vp, vp] + [ctypes.c_int] * 5 + [ctypes.c_float] * 2 + \
        [ctypes.c_int, ctypes.POINTER(Options), vp, ctypes.c_size_t, vp]
    p = ctypes.c_void_p(16)
    return f(p, p, p, p, 1, 1, T, d, d, 4.0, 0.01, dtype,
             ctypes.byref(opts) if opts is not None else None, None, 0, None)


def test_options_struct_layout():
    from local_linear_attention_gb300.binding import Options
    assert ctypes.sizeof(Options) == 32  # 5 fields + 3 reserved ints, as lla_options


def test_invalid_options_rejected_on_the_host(lib):
    """Options are validated before any device work (these calls would otherwise need a GPU)."""
    from local_linear_attention_gb300.binding import Options
    INVALID = 1

    def opts(**kw):
        o = Options()
        for key, val in kw.items():
            setattr(o, key, val)
        return o
    assert _fwd_ex(lib, opts(path=4)) == INVALID
    assert _fwd_ex(lib, opts(path=-1)) == INVALID
    assert _fwd_ex(lib, opts(form=2)) == INVALID
    assert _fwd_ex(lib, opts(cg_max_iters=1025)) == INVALID
    assert _fwd_ex(lib, opts(cg_rel_tol=1.0)) == INVALID
    assert _fwd_ex(lib, opts(cg_rel_tol=float("nan"))) == INVALID
    assert _fwd_ex(lib, opts(test_fault=2)) == INVALID
    o = opts()
    o.reserved[1] = 5
    assert _fwd_ex(lib, o) == INVALID
    # empty problems with valid options stay a no-op
    assert _fwd_ex(lib, opts(path=1), T=0) == 0
    assert _fwd_ex(lib, None, T=0) == 0
    # the other operations accept a path only
    vp = ctypes.c_void_p
    f = lib.lla_parallax_forward_ex
    f.restype = ctypes.c_int
    f.argtypes = [vp] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int,
                                                    ctypes.POINTER(Options), vp]
    p = vp(16)
    assert f(p, p, p, p, p, 1, 1, 4, 16, 16, 4.0, 0, ctypes.byref(opts(form=1)), None) == INVALID
    assert f(p, p, p, p, p, 1, 1, 4, 16, 16, 4.0, 0, ctypes.byref(opts(path=3)), None) == INVALID
    g = lib.lla_decode_ex
    g.restype = ctypes.c_int
    g.argtypes = [vp] * 4 + [ctypes.c_int] * 5 + [ctypes.c_float] * 2 + [
        ctypes.c_int, ctypes.POINTER(Options), vp]
    assert g(p, p, p, p, 1, 1, 4, 16, 16, 4.0, 0.01, 0, ctypes.byref(opts(test_fault=1)),
             None) == INVALID


def test_noalloc_size_limits_match_the_documented_ones(lib):
    """lla_forward_noalloc's documented limits (bf16 d = dv = 64: T <= 4343 at B*H = 1,
    T <= 704 at B*H = 8) follow from lla_workspace_size and the fixed scratch size, and the
    entry point refuses the next size up before touching any device."""
    from local_linear_attention_gb300.binding import NOALLOC_SCRATCH_BYTES
    ws = lib.lla_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [ctypes.c_int] * 6
    with open(os.path.join(ROOT, "include", "lla.h")) as fh:
        header = fh.read()
    assert "#define LLA_NOALLOC_SCRATCH_BYTES (64ull << 20)" in header
    assert NOALLOC_SCRATCH_BYTES == 64 << 20
    for BH, tmax in ((1, 4343), (8, 704)):
        assert ws(1, BH, tmax, 64, 64, 1) <= NOALLOC_SCRATCH_BYTES < ws(1, BH, tmax + 1, 64, 64, 1)
    vp = ctypes.c_void_p
    f = lib.lla_forward_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [vp] * 4 + [ctypes.c_int] * 5 + [ctypes.c_float] * 2 + [ctypes.c_int, vp]
    p = vp(16)
    assert f(p, p, p, p, 1, 1, 4344, 64, 64, 8.0, 0.01, 1, None) == 2   # LLA_ERR_UNSUPPORTED
    assert f(p, p, p, p, 1, 8, 705, 64, 64, 8.0, 0.01, 1, None) == 2
