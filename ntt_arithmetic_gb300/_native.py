"""ctypes binding of libfhe_ntt.so (include/fhe_ntt.h).

Argument marshalling only: every step of every call runs in the library's
CUDA kernels.  There is no CPU fallback; if the library is missing or fails
to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfhe_ntt.so")

FHE_OK = 0
FHE_EINVAL = -1
FHE_EALIAS = -2
FHE_ECUDA = -3
FHE_ESPACE = -4
FHE_EDEVICE = -5
FHE_DOMAIN_COEFF = 0
FHE_DOMAIN_NTT = 1
FHE_ROUND_TRUNCATE = 0
FHE_ROUND_NEAREST = 1
FHE_STATUS_TC_TIMEOUT = 1
FHE_MODUP_EXACT = 0
FHE_MODUP_APPROX = 1
FHE_BCONV_EXACT = 0
FHE_BCONV_APPROX = 1

_u64 = ctypes.c_uint64
_u64p = ctypes.POINTER(ctypes.c_uint64)
_int = ctypes.c_int
_vp = ctypes.c_void_p
_size = ctypes.c_size_t


class NttTables(ctypes.Structure):
    """Mirror of struct fhe_ntt_tables."""
    _fields_ = [
        ("log_n", ctypes.c_int32),
        ("L", ctypes.c_int32),
        ("q", _vp),
        ("consts", _vp),
        ("fwd", _vp),
        ("inv", _vp),
        ("twist", _vp),
        ("blob", _vp),
        ("bytes", _size),
    ]


# name -> (restype, argtypes); the exported C ABI, one entry per declaration
SIGNATURES = {
    "fhe_version": (_int, []),
    "fhe_status_str": (ctypes.c_char_p, [_int]),
    "fhe_launch_count": (_u64, []),
    "fhe_selftest_host": (_int, [_u64, _int]),
    "fhe_find_primes": (_int, [_int, _int, _int, _u64, _u64p]),
    "fhe_root_of_unity": (_int, [_u64, _int, _u64p]),
    "fhe_ntt_tables_bytes": (_int, [_int, _int, ctypes.POINTER(_size)]),
    "fhe_ntt_tables_build_host": (_int, [_int, _int, _u64p, _vp, _size]),
    "fhe_ntt_tables_bind": (_int, [_vp, _size, _int, _int, ctypes.POINTER(NttTables)]),
    "fhe_ntt_fwd_table_slot": (_int, [_int, ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32)]),
    "fhe_ntt_fwd": (_int, [_vp, _int, _int, _int, ctypes.POINTER(NttTables), _vp]),
    "fhe_ntt_inv": (_int, [_vp, _int, _int, _int, ctypes.POINTER(NttTables), _vp]),
    "fhe_mul_ntt": (_int, [_vp, _vp, _vp, _int, _int, _int, ctypes.POINTER(NttTables), _vp]),
    "fhe_tensor": (_int, [_vp, _vp, _vp, _int, _int, _int, ctypes.POINTER(NttTables), _vp]),
    "fhe_automorph": (_int, [_vp, _vp, _int, _int, _int, _u64, _int, ctypes.POINTER(NttTables), _vp]),
    "fhe_modup_tables_bytes": (_int, [_int, _int, _int, ctypes.POINTER(_size)]),
    "fhe_modup_tables_build_host": (_int, [_int, _int, _int, _u64p, _vp, _size]),
    "fhe_keyswitch_workspace_bytes": (_int, [_int, _int, _int, _int, _int, ctypes.POINTER(_size)]),
    "fhe_keyswitch_ip": (_int, [_vp, _vp, _size, _vp, _int, _int, _int, _int, _int, ctypes.POINTER(NttTables),
                                _vp, _vp, _size, _vp]),
    "fhe_keyswitch_ip_ex": (_int, [_vp, _vp, _size, _vp, _int, _int, _int, _int, _int, _int,
                                   ctypes.POINTER(NttTables), _vp, _vp, _size, _vp]),
    "fhe_keyswitch_hoisted": (_int, [_vp, _vp, _size, _vp, ctypes.POINTER(ctypes.c_uint32), _int, _int, _int, _int,
                                     _int, _int, _int, ctypes.POINTER(NttTables), _vp, _vp, _size, _vp]),
    "fhe_keyswitch_decompose": (_int, [_vp, _vp, _size, _int, _int, _int, _int, _int, _int,
                                       ctypes.POINTER(NttTables), _vp, _vp]),
    "fhe_keyswitch_apply": (_int, [_vp, _vp, _vp, ctypes.POINTER(ctypes.c_uint32), _int, _int, _int, _int, _int, _int,
                                   ctypes.POINTER(NttTables), _vp]),
    "fhe_bconv_tables_bytes": (_int, [_int, _int, ctypes.POINTER(_size)]),
    "fhe_bconv_tables_build_host": (_int, [_int, _u64p, _int, _u64p, _vp, _size]),
    "fhe_bconv": (_int, [_vp, _vp, _int, _int, _int, _int, _int, _vp, _vp]),
    "fhe_moddown_tables_bytes": (_int, [_int, _int, ctypes.POINTER(_size)]),
    "fhe_moddown_tables_build_host": (_int, [_int, _int, _u64p, _vp, _size]),
    "fhe_moddown_workspace_bytes": (_int, [_int, _int, _int, _int, ctypes.POINTER(_size)]),
    "fhe_moddown": (_int, [_vp, _vp, _int, _int, _int, _int, _int, _int, ctypes.POINTER(NttTables), _vp, _vp,
                           _size, _vp]),
    "fhe_rescale": (_int, [_vp, _vp, _int, _int, _int, _int, _int, ctypes.POINTER(NttTables), _vp, _vp, _size,
                           _vp]),
    "fhe_keyswitch_ip_noalloc": (_int, [_vp, _vp, _size, _vp, _int, _int, _int, _int, _int,
                                        ctypes.POINTER(NttTables), _vp, _vp]),
    "fhe_keyswitch_noalloc_max_bytes": (_size, []),
    "fhe_butterfly_probe": (_int, [_vp, _int, _int, ctypes.POINTER(NttTables), _vp]),
    "fhe_device_status": (_int, [ctypes.POINTER(_int), _int]),
}

_lib = None


class FheError(RuntimeError):
    def __init__(self, func: str, status: int):
        msg = lib().fhe_status_str(status).decode() if _lib is not None else str(status)
        super().__init__(f"{func} failed with status {status}: {msg}")
        self.status = status


def lib():
    """Load the library (once).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                           "(or ntt_arithmetic_gb300.build.build()); the CUDA path has no fallback")
    handle = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(handle, name)
        f.restype = res
        f.argtypes = args
    _lib = handle
    return handle


def check(func: str, status: int) -> None:
    if status != FHE_OK:
        raise FheError(func, status)


def call(func: str, *args) -> None:
    check(func, getattr(lib(), func)(*args))
