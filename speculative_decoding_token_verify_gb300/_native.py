"""Build and load ``libspecverify.so``, the CUDA library behind the C ABI in
``include/spec_verify.h``.

The library is compiled in-tree for sm_103a with nvcc. Loading never falls
back to anything: if the library is missing or cannot be loaded, ``lib()``
raises, so no code path can run without the CUDA kernels.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_CSRC = os.path.join(_PKG, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
LIB_PATH = os.path.join(_PKG, "libspecverify.so")
# the same library with the kernels' index checks compiled in (SPEC_CHECKED);
# for tests
CHECKED_LIB_PATH = os.path.join(_PKG, "libspecverify_checked.so")
SOURCES = ("spec_verify.cu", "spec_nucleus.cu", "spec_estimator.cu", "spec_irls.cu", "spec_av.cu", "spec_ngram.cu")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]

_lock = threading.Lock()
_lib = None


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: cannot build libspecverify.so")


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = True) -> str:
    """Compile the CUDA sources (in parallel, one object each) and link the
    shared library next to this file; with `checked`, the checked variant
    (SPEC_CHECKED) as well, from the same nvcc run. Returns the library's
    path."""
    srcs = [os.path.join(_CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(_CSRC, "spec_device.cuh"), os.path.join(_CSRC, "spec_nucleus.cuh"),
            os.path.join(_INCLUDE, "spec_verify.h")]
    targets = [(LIB_PATH, [])] + ([(CHECKED_LIB_PATH, ["-DSPEC_CHECKED"])] if checked else [])
    newest = max(os.path.getmtime(d) for d in deps)
    targets = [(path, flags) for path, flags in targets
               if force or not os.path.exists(path) or os.path.getmtime(path) < newest]
    if not targets:
        return LIB_PATH
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", *ARCH_FLAGS, "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=default", f"-I{_INCLUDE}", f"-I{_CSRC}", *extra_flags]
    if verbose:
        common += ["-Xptxas", "-v"]
    tag = f"{os.getpid()}"
    jobs = []   # (target, objects)
    procs = []
    for k, (path, flags) in enumerate(targets):
        objs = []
        for s in srcs:
            o = os.path.join(_CSRC, os.path.basename(s) + f".{tag}.{k}.o")
            objs.append(o)
            procs.append(subprocess.Popen([nvcc, *common, *flags, "-c", s, "-o", o],
                                          stdout=subprocess.PIPE, stderr=subprocess.STDOUT))
        jobs.append((path, objs))
    logs = []
    ok = True
    for p in procs:
        out, _ = p.communicate()
        logs.append(out.decode(errors="replace"))
        ok &= p.returncode == 0
    try:
        if not ok:
            raise RuntimeError("nvcc failed:\n" + "\n".join(logs))
        for path, objs in jobs:
            tmp = path + f".{tag}.tmp"
            subprocess.check_call([nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs])
            os.replace(tmp, path)
    finally:
        for _, objs in jobs:
            for o in objs:
                if os.path.exists(o):
                    os.remove(o)
    if verbose:
        print("\n".join(logs))
    return LIB_PATH


class VerifyParams(ctypes.Structure):
    """Mirror of ``spec_verify_params``."""
    _fields_ = [
        ("B", ctypes.c_int32),
        ("K", ctypes.c_int32),
        ("V", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("mode", ctypes.c_int32),
        ("fly_window", ctypes.c_int32),
        ("fly_theta", ctypes.c_float),
        ("reserved", ctypes.c_int32),
        ("t_row_stride", ctypes.c_int64),
        ("d_row_stride", ctypes.c_int64),
    ]


# (name, restype, argtypes) of every symbol include/spec_verify.h declares
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
SIGNATURES = {
    "spec_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(VerifyParams)]),
    "spec_verify": (ctypes.c_int, [ctypes.POINTER(VerifyParams), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P, ctypes.c_size_t, _P]),
    "spec_verify_static": (ctypes.c_int, [ctypes.POINTER(VerifyParams), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          _P]),
    "spec_confidence_workspace_size": (ctypes.c_size_t, [_I32, _I32, _I32, _I32]),
    "spec_confidence": (ctypes.c_int, [_I32, _I32, _I32, _I32, _P, ctypes.c_int64, _P, _P, _P, _P,
                                       ctypes.c_size_t, _P]),
    "spec_estimator_update": (ctypes.c_int, [_I32, _I32, _P, _P, _P, ctypes.c_float, _P, _P, _P]),
    "spec_verify_ragged": (ctypes.c_int, [ctypes.POINTER(VerifyParams), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          _P, _P, ctypes.c_size_t, _P]),
    "spec_verify_temperature": (ctypes.c_int, [ctypes.POINTER(VerifyParams), _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                               _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "spec_verify_top_p": (ctypes.c_int, [ctypes.POINTER(VerifyParams), _P, _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                         _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "spec_estimator_update_ragged": (ctypes.c_int, [_I32, _I32, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P]),
    "spec_irls_accumulate_ragged": (ctypes.c_int, [_I32, _I32, _P, _P, _P, _P, _P, _P]),
    "spec_av_budget": (ctypes.c_int, [_I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P]),
    "spec_ngram_draft": (ctypes.c_int, [_I32, _I32, _P, _P, _I32, _I32, _I32, _P, _P, _P]),
    "spec_irls_state_size": (ctypes.c_size_t, [_I32]),
    "spec_irls_reset": (ctypes.c_int, [_I32, _P, _P]),
    "spec_irls_accumulate": (ctypes.c_int, [_I32, _I32, _P, _P, _P, _P, _P]),
    "spec_irls_refit": (ctypes.c_int, [_I32, _P, _P, ctypes.c_double, _P, _P]),
    "spec_get_device_status": (ctypes.c_int, [_P, ctypes.POINTER(_I32)]),
    "spec_static_device_status": (ctypes.c_int, [ctypes.POINTER(_I32)]),
    "spec_debug_set_wait_limit": (ctypes.c_uint32, [ctypes.c_uint32]),
    "spec_last_error": (ctypes.c_char_p, []),
    "spec_version": (ctypes.c_char_p, []),
}


def lib() -> ctypes.CDLL:
    """The loaded library. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        _lib = _load(LIB_PATH)
    return _lib


def _load(path):
    L = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


_checked = None


def lib_checked() -> ctypes.CDLL:
    """The checked variant (index checks in the kernels), for tests. Raises if
    it has not been built."""
    global _checked
    with _lock:
        if _checked is None:
            if not os.path.exists(CHECKED_LIB_PATH):
                raise RuntimeError(f"{CHECKED_LIB_PATH} is missing: build it first")
            _checked = _load(CHECKED_LIB_PATH)
    return _checked


def last_error() -> str:
    return (lib().spec_last_error() or b"").decode()
