"""Python binding of the gdnbeam C ABI (large-beam Gated DeltaNet decoding).

Argument marshalling only: every stage of the decode path runs in the CUDA
kernels of libgdnbeam.so. The functions keep the C names; tensors are passed
as device pointers (torch tensors are accepted and their data_ptr() taken),
streams as torch.cuda.Stream or raw handles.

Loading fails loudly if the library has not been built; there is no CPU or
library fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

from . import _build

__all__ = [
    "lib", "load", "Config", "Weights", "Dumps", "Footprint", "Records", "GdnbeamError",
    "F32", "BF16", "check", "ptr", "stream_handle",
]

F32, BF16 = 0, 1
MAX_T = 8
STAGES = ("ancestry", "embed", "project", "replay", "logits", "select", "prefill")

OK, EINVAL, EUNSUPPORTED, EWORKSPACE, ESTATE, ECUDA, EDEVICE, ENOMEM = 0, -1, -2, -3, -4, -5, -6, -7
# device error word bits (gdnbeam_device_status)
DERR_TOKEN, DERR_PARENT, DERR_SLOT, DERR_NONFINITE, DERR_TIMEOUT, DERR_SELECT = 1, 2, 4, 8, 16, 32
DERR = {"token": 1, "parent": 2, "slot": 4, "nonfinite": 8, "timeout": 16, "select": 32}


class Config(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("R", "layers", "H", "d_k", "d_v", "d_model", "V", "T",
                                       "W_max", "L_max", "dtype", "residual", "state_path",
                                       "H_k")]


class Weights(C.Structure):
    _fields_ = [("E", C.c_void_p), ("W_proj", C.c_void_p), ("W_o", C.c_void_p)]


class Dumps(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("q", "k", "v", "alpha", "beta", "delta", "o", "logits")]


class Footprint(C.Structure):
    _fields_ = [(n, C.c_size_t) for n in ("sctx_bytes", "record_elements", "records_bytes",
                                          "ancestry_bytes", "fullstate_bytes", "workspace_bytes")]


class Records(C.Structure):
    _fields_ = [("k", C.c_void_p), ("delta", C.c_void_p), ("alpha", C.c_void_p), ("W_j", C.c_int)]


class GdnbeamError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} ({status})" if what else strerror(status))


_P = C.c_void_p
_I = C.c_int
_SZ = C.c_size_t
_LL = C.c_longlong
_S = C.c_void_p  # stream

_SIGS = {
    "gdnbeam_footprint_of": (_I, [C.POINTER(Config), C.POINTER(Footprint)]),
    "gdnbeam_create": (_I, [C.POINTER(Config), C.POINTER(Weights), _P, _SZ, C.POINTER(_P)]),
    "gdnbeam_destroy": (None, [_P]),
    "gdnbeam_prefill_state": (_I, [_P, _P, _I, _P, _P, _S]),
    "gdnbeam_step": (_I, [_P, _I, _I, _P, _P, _P, _P, C.POINTER(Dumps), _S]),
    "gdnbeam_select": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _S]),
    "gdnbeam_get_paths": (_I, [_P, _I, _P, _P, _P, _S]),
    "gdnbeam_read_sctx": (_I, [_P, _P, _S]),
    "gdnbeam_reset": (_I, [_P, _P]),
    "gdnbeam_prefill_requests": (_I, [_P, _P, _I, _P, _I, _P, _P, _S]),
    "gdnbeam_status": (_I, [_P, _S]),
    "gdnbeam_device_status": (_I, [_I]),
    "gdnbeam_variant": (C.c_char_p, [_P]),
    "gdnbeam_strerror": (C.c_char_p, [_I]),
    "gdnbeam_timing": (_I, [_P, _I]),
    "gdnbeam_stage_times": (_I, [_P, C.POINTER(C.c_float), C.POINTER(C.c_int)]),
    "gdnbeam_launches": (C.c_longlong, [_I]),
    "gdnbeam_project_scratch_bytes": (_SZ, [C.POINTER(Config), _I]),
    "gdnbeam_project": (_I, [C.POINTER(Config), _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                             C.POINTER(Dumps), _S]),
    "gdnbeam_replay": (_I, [C.POINTER(Config), _I, _I, _P, _LL, _P, _P, _P, _P, _P,
                            C.POINTER(Records), _P, _I, _P, _P, _P, C.POINTER(Dumps), _S]),
    "gdnbeam_logits_scratch_bytes": (_SZ, [C.POINTER(Config), _I]),
    "gdnbeam_logits": (_I, [C.POINTER(Config), _I, _P, _P, _P, _P, _P, _SZ, C.POINTER(Dumps), _S]),
    "gdnbeam_select_scratch_bytes": (_SZ, [_I, _I, _I, _I]),
    "gdnbeam_select_topw": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _S]),
    "gdnbeam_select_noalloc_max_bytes": (_SZ, []),
    "gdnbeam_select_topw_noalloc": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _S]),
    "gdnbeam_ancestry": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _S]),
    "gdnbeam_prefill_scan_scratch_bytes": (_SZ, [C.POINTER(Config), _I, _I]),
    "gdnbeam_prefill_scan": (_I, [C.POINTER(Config), _I, _P, _P, _P, _P, _P, _P, _LL, _P, _P, _P, _SZ,
                                  _S]),
    "gdnbeam_fullstate_step": (_I, [C.POINTER(Config), _I, _I, _I, _P, _LL, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _P, _P, _S]),
    "gdnbeam_replayssm_step": (_I, [C.POINTER(Config), _I, _I, _P, _LL, _P, _P, _P, _P, _P,
                                    C.POINTER(Records), _P, _I, _P, _P, _S]),
}

_lib: Optional[C.CDLL] = None


def load(build: bool = True) -> C.CDLL:
    """Loads libgdnbeam.so (building it first if sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build else _build.LIB
    if not os.path.exists(path):
        raise OSError(f"libgdnbeam.so not built at {path}")
    lib_ = C.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib_, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib_
    return lib_


def lib() -> C.CDLL:
    return load()


def strerror(status: int) -> str:
    try:
        return load(build=False).gdnbeam_strerror(status).decode()
    except OSError:
        return f"status {status}"


def check(status: int, what: str = "") -> int:
    if status != OK:
        raise GdnbeamError(status, what)
    return status


def ptr(x) -> Optional[int]:
    """Device (or host) address of a tensor / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def stream_handle(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def dumps(**kw) -> Dumps:
    d = Dumps()
    for k, v in kw.items():
        setattr(d, k, ptr(v))
    return d


def __getattr__(name):
    # gdnbeam_* functions resolve to the loaded library's symbols
    if name.startswith("gdnbeam_"):
        return getattr(load(), name)
    raise AttributeError(name)
