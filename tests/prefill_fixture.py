"""The synthetic prefill fixture of the tests and the benchmark (tests/fixture/kvx_fixture.cu): a
bounded integer chain per layer on the caller's main stream, standing in for a layer's forward
compute, that records the layer's ready event. It is its own library, libkvx_fixture.so, built with
nvcc for sm_103a; the kvx library and its C-ABI do not contain it."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import tempfile

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_PKG = os.path.join(_ROOT, "disaggregated_prefill_decode_gb300")
_DIR = os.path.join(_HERE, "fixture")
_SRC = os.path.join(_DIR, "kvx_fixture.cu")
_HDR = os.path.join(_DIR, "kvx_fixture.h")
LIB_PATH = os.path.join(_DIR, "_build", "libkvx_fixture.so")


def build(force: bool = False) -> str:
    """Compile libkvx_fixture.so (one -gencode for sm_103a; it links libkvx.so, which must be built)
    unless it is newer than its sources."""
    newest = max(os.path.getmtime(p) for p in (_SRC, _HDR, __file__, os.path.join(_ROOT, "include", "kvx.h")))
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    os.makedirs(os.path.dirname(LIB_PATH), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(LIB_PATH))
    os.close(fd)
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo", "-Xcompiler",
           "-fPIC", "-shared", "-cudart", "static", "-I", _DIR, "-I", os.path.join(_ROOT, "include"), _SRC,
           "-o", tmp, "-L", _PKG, "-lkvx", "-Xlinker", f"-rpath,{_PKG}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        os.unlink(tmp)
        raise RuntimeError(f"nvcc failed on kvx_fixture.cu:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None


def lib():
    """The loaded fixture library (built on first use)."""
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build())
        l.kvx_fixture_prefill.restype = ctypes.c_int
        l.kvx_fixture_prefill.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
        l.kvx_fixture_launch_count.restype = ctypes.c_int64
        l.kvx_fixture_launch_count.argtypes = []
        l.kvx_fixture_last_error.restype = ctypes.c_char_p
        l.kvx_fixture_last_error.argtypes = []
        P = ctypes.c_void_p
        l.kvx_fixture_run_steps.restype = ctypes.c_int
        l.kvx_fixture_run_steps.argtypes = [P, P, P, ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int64, P, P, P, P, P, P, ctypes.c_int64, P, P, P,
                                            ctypes.c_int32]
        _lib = l
    return _lib


def _handle(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    for attr in ("cuda_stream", "cuda_event"):
        if hasattr(x, attr):
            return int(getattr(x, attr))
    return int(x.data_ptr())


def prefill(ctas: int, iters: int, buf=None, n_bytes: int = 0, seed: int = 0, stream=None, done=None) -> None:
    """One fixture launch on `stream` (torch stream or raw handle); `done` recorded after it."""
    if lib().kvx_fixture_prefill(ctas, iters, _handle(buf), n_bytes, seed & (2**64 - 1), _handle(stream),
                                 _handle(done)):
        raise RuntimeError(f"kvx_fixture_prefill: {lib().kvx_fixture_last_error().decode()}")


def launch_count() -> int:
    return int(lib().kvx_fixture_launch_count())
