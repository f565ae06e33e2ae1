"""CPU oracle for the batched RNS negacyclic NTT and its NTT-domain kernels.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use this package; the library under
``ntt_arithmetic_gb300`` never does.  It is a thin ctypes wrapper over
``oracle.c`` (plain C11, ``unsigned __int128`` and ``%``), which shares no
code with the CUDA path.  See the header of ``oracle.c`` for the pages each
function follows and the readings taken where the pages are silent.

Every function here is pinned by ``tests/test_oracle_*.py`` against
definitions, closed forms, brute force and independent library routines.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None

_u64p = ctypes.POINTER(ctypes.c_uint64)
_u64 = ctypes.c_uint64
_int = ctypes.c_int


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = _build.library_path()
    if not os.path.exists(path) or _build.stale():
        _build.build()
    lib = ctypes.CDLL(path)
    sig = {
        "oracle_mulmod": (_u64, [_u64, _u64, _u64]),
        "oracle_powmod": (_u64, [_u64, _u64, _u64]),
        "oracle_is_prime": (_int, [_u64]),
        "oracle_primes": (_int, [_u64, _int, _int, _u64, _u64p]),
        "oracle_psi": (_u64, [_u64, _u64]),
        "oracle_brv": (_u64, [_u64, _int]),
        "oracle_ntt_direct": (None, [_u64p, _u64p, _int, _u64, _u64]),
        "oracle_intt_direct": (None, [_u64p, _u64p, _int, _u64, _u64]),
        "oracle_ntt": (None, [_u64p, _int, _u64, _u64]),
        "oracle_intt": (None, [_u64p, _int, _u64, _u64]),
        "oracle_negacyclic_mul": (None, [_u64p, _u64p, _u64p, _int, _u64]),
        "oracle_automorph_coeff": (None, [_u64p, _u64p, _int, _u64, _u64]),
        "oracle_automorph_ntt": (None, [_u64p, _u64p, _int, _u64, _u64, _u64]),
        "oracle_modup_coeff": (None, [_u64p, _u64p, _int, _u64p, _int, _u64p]),
        "oracle_ntt_batch": (None, [_u64p, _int, _int, _int, _u64p, _u64p, _int, _int]),
        "oracle_mul_batch": (None, [_u64p, _u64p, _u64p, _int, _int, _int, _u64p]),
        "oracle_tensor_batch": (None, [_u64p, _u64p, _u64p, _int, _int, _int, _u64p]),
        "oracle_automorph_batch": (None, [_u64p, _u64p, _int, _int, _int, _u64p, _u64p, _u64, _int, _int]),
        "oracle_modup_batch": (None, [_u64p, _u64p, _u64p, _int, _int, _int, _int, _int, _int]),
        "oracle_keyswitch_batch": (None, [_u64p, _u64p, _u64p, _u64p, _u64p, _int, _int, _int, _int, _int, _int]),
        "oracle_moddown_batch": (None, [_u64p, _u64p, _u64p, _int, _int, _int, _int, _int]),
        "oracle_bconv_coeff": (None, [_u64p, _u64p, _int, _u64p, _int, _int, _u64p]),
        "oracle_bconv_batch": (None, [_u64p, _u64p, _u64p, _int, _u64p, _int, _int, _int, _int, _int]),
        "oracle_modup_batch_ex": (None, [_u64p, _u64p, _u64p, _int, _int, _int, _int, _int, _int, _int]),
        "oracle_keyswitch_batch_ex": (None, [_u64p, _u64p, _u64p, _u64p, _u64p, _int, _int, _int, _int, _int,
                                             _int, _int]),
        "oracle_keyswitch_hoisted_batch": (None, [_u64p, _u64p, _u64p, _int, _u64p, _u64p, _u64p, _int, _int,
                                                  _int, _int, _int, _int, _int]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _arr(x, copy=False) -> np.ndarray:
    a = np.array(x, dtype=np.uint64, copy=True) if copy else np.ascontiguousarray(x, dtype=np.uint64)
    return a


def _p(a: np.ndarray):
    assert a.dtype == np.uint64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_u64p)


def _log2(n: int) -> int:
    if n < 1 or n & (n - 1):
        raise ValueError(f"n={n} is not a power of two")
    return n.bit_length() - 1


# ----------------------------------------------------------------------------
# scalars
# ----------------------------------------------------------------------------

def mulmod(a: int, b: int, q: int) -> int:
    return int(_load().oracle_mulmod(a, b, q))


def powmod(b: int, e: int, q: int) -> int:
    return int(_load().oracle_powmod(b, e, q))


def is_prime(n: int) -> bool:
    return bool(_load().oracle_is_prime(n))


def primes(m: int, count: int, bits: int = 50, below: int = 0) -> np.ndarray:
    """The ``count`` largest primes q < min(2^bits, below) with q = 1 mod m,
    in descending order."""
    out = np.zeros(count, dtype=np.uint64)
    got = _load().oracle_primes(m, bits, count, below, _p(out))
    if got != count:
        raise ValueError(f"only {got} primes = 1 mod {m} below 2^{bits}")
    return out


def psi(q: int, m: int) -> int:
    """Smallest primitive m-th root of unity mod q (m = 2n)."""
    return int(_load().oracle_psi(q, m))


def brv(x: int, bits: int) -> int:
    return int(_load().oracle_brv(x, bits))


# ----------------------------------------------------------------------------
# single polynomials
# ----------------------------------------------------------------------------

def ntt_direct(a, q: int, psi_: int) -> np.ndarray:
    a = _arr(a)
    out = np.zeros_like(a)
    _load().oracle_ntt_direct(_p(a), _p(out), _log2(a.size), q, psi_)
    return out


def intt_direct(a, q: int, psi_: int) -> np.ndarray:
    a = _arr(a)
    out = np.zeros_like(a)
    _load().oracle_intt_direct(_p(a), _p(out), _log2(a.size), q, psi_)
    return out


def ntt(a, q: int, psi_: int) -> np.ndarray:
    a = _arr(a, copy=True)
    _load().oracle_ntt(_p(a), _log2(a.size), q, psi_)
    return a


def intt(a, q: int, psi_: int) -> np.ndarray:
    a = _arr(a, copy=True)
    _load().oracle_intt(_p(a), _log2(a.size), q, psi_)
    return a


def negacyclic_mul(a, b, q: int) -> np.ndarray:
    a, b = _arr(a), _arr(b)
    out = np.zeros_like(a)
    _load().oracle_negacyclic_mul(_p(a), _p(b), _p(out), _log2(a.size), q)
    return out


def automorph_coeff(a, q: int, k: int) -> np.ndarray:
    a = _arr(a)
    out = np.zeros_like(a)
    _load().oracle_automorph_coeff(_p(a), _p(out), _log2(a.size), q, k)
    return out


def automorph_ntt(a, q: int, psi_: int, k: int) -> np.ndarray:
    a = _arr(a)
    out = np.zeros_like(a)
    _load().oracle_automorph_ntt(_p(a), _p(out), _log2(a.size), q, psi_, k)
    return out


def modup_coeff(x, digit_primes, targets) -> np.ndarray:
    x, d, t = _arr(x), _arr(digit_primes), _arr(targets)
    assert x.size == d.size <= 64 and t.size <= 256
    out = np.zeros(t.size, dtype=np.uint64)
    _load().oracle_modup_coeff(_p(x), _p(d), int(d.size), _p(t), int(t.size), _p(out))
    return out


# ----------------------------------------------------------------------------
# batched [batch][L][n] drivers
# ----------------------------------------------------------------------------

def psis(qs, n: int) -> np.ndarray:
    return np.array([psi(int(q), 2 * n) for q in qs], dtype=np.uint64)


def ntt_batch(a, qs, psi_list, inverse: bool = False, threads: int | None = None) -> np.ndarray:
    """Forward (or inverse) NTT of every row of a[batch][L][n]; returns a copy."""
    a = _arr(a, copy=True)
    L, n = a.shape[-2], a.shape[-1]
    batch = a.size // (L * n)
    qs, ps = _arr(qs), _arr(psi_list)
    _load().oracle_ntt_batch(_p(a), _log2(n), L, batch, _p(qs), _p(ps), int(inverse),
                             threads or default_threads())
    return a


def mul_batch(a, b, qs) -> np.ndarray:
    a, b, qs = _arr(a), _arr(b), _arr(qs)
    L, n = a.shape[-2], a.shape[-1]
    out = np.zeros_like(a)
    _load().oracle_mul_batch(_p(a), _p(b), _p(out), _log2(n), L, a.size // (L * n), _p(qs))
    return out


def tensor_batch(a, b, qs) -> np.ndarray:
    """a, b: [batch][2][L][n] -> d: [batch][3][L][n]."""
    a, b, qs = _arr(a), _arr(b), _arr(qs)
    L, n = a.shape[-2], a.shape[-1]
    batch = a.size // (2 * L * n)
    out = np.zeros((batch, 3, L, n), dtype=np.uint64)
    _load().oracle_tensor_batch(_p(a), _p(b), _p(out), _log2(n), L, batch, _p(qs))
    return out.reshape(a.shape[:-3] + (3, L, n))


def automorph_batch(a, qs, psi_list, k: int, ntt_domain: bool, threads: int | None = None) -> np.ndarray:
    a, qs, ps = _arr(a), _arr(qs), _arr(psi_list)
    L, n = a.shape[-2], a.shape[-1]
    out = np.zeros_like(a)
    _load().oracle_automorph_batch(_p(a), _p(out), _log2(n), L, a.size // (L * n), _p(qs), _p(ps),
                                   k, int(ntt_domain), threads or default_threads())
    return out


def modup_batch(a, qp, L: int, K: int, dnum: int, threads: int | None = None, approx: bool = False) -> np.ndarray:
    """a: [batch][L][n] -> [batch][dnum][L+K][n] (coefficient domain); exact
    Garner extension, or the approximate basis conversion if ``approx``."""
    a, qp = _arr(a), _arr(qp)
    n = a.shape[-1]
    batch = a.size // (L * n)
    out = np.zeros((batch, dnum, L + K, n), dtype=np.uint64)
    if approx:
        _load().oracle_modup_batch_ex(_p(a), _p(out), _p(qp), _log2(n), L, K, dnum, batch, 1,
                                      threads or default_threads())
    else:
        _load().oracle_modup_batch(_p(a), _p(out), _p(qp), _log2(n), L, K, dnum, batch,
                                   threads or default_threads())
    return out


def keyswitch_batch(a, keys, qp, psi_qp, L: int, K: int, dnum: int, threads: int | None = None,
                    approx: bool = False) -> np.ndarray:
    """a: [batch][L][n] coeff; keys: [dnum][2][L+K][n] NTT -> [batch][2][L+K][n] NTT."""
    a, keys, qp, ps = _arr(a), _arr(keys), _arr(qp), _arr(psi_qp)
    n = a.shape[-1]
    batch = a.size // (L * n)
    out = np.zeros((batch, 2, L + K, n), dtype=np.uint64)
    if approx:
        _load().oracle_keyswitch_batch_ex(_p(a), _p(keys), _p(out), _p(qp), _p(ps), _log2(n), L, K, dnum,
                                          batch, 1, threads or default_threads())
    else:
        _load().oracle_keyswitch_batch(_p(a), _p(keys), _p(out), _p(qp), _p(ps), _log2(n), L, K, dnum,
                                       batch, threads or default_threads())
    return out


def keyswitch_hoisted_batch(a, keys, ks, qp, psi_qp, L: int, K: int, dnum: int, threads: int | None = None,
                            approx: bool = False) -> np.ndarray:
    """Hoisted key switch for Galois elements ks[R]: a [batch][L][n] coeff;
    keys [R][dnum][2][L+K][n] NTT -> [R][batch][2][L+K][n] NTT."""
    a, keys, qp, ps = _arr(a), _arr(keys), _arr(qp), _arr(psi_qp)
    ks = _arr([int(k) for k in ks])
    n = a.shape[-1]
    R = int(ks.size)
    batch = a.size // (L * n)
    assert keys.size == R * dnum * 2 * (L + K) * n
    out = np.zeros((R, batch, 2, L + K, n), dtype=np.uint64)
    _load().oracle_keyswitch_hoisted_batch(_p(a), _p(keys), _p(ks), R, _p(out), _p(qp), _p(ps), _log2(n), L, K,
                                           dnum, batch, int(approx), threads or default_threads())
    return out


def bconv_coeff(x, src, dst, approx: bool) -> np.ndarray:
    """One coefficient from basis ``src`` to ``dst``: exact (X in [0, Q)) or
    approximate (X + e Q, 0 <= e < len(src))."""
    x, s, d = _arr(x), _arr(src), _arr(dst)
    assert x.size == s.size <= 64
    out = np.zeros(d.size, dtype=np.uint64)
    _load().oracle_bconv_coeff(_p(x), _p(s), int(s.size), _p(d), int(d.size), int(approx), _p(out))
    return out


def bconv_batch(a, src, dst, approx: bool = False, threads: int | None = None) -> np.ndarray:
    """a: [batch][S][n] over ``src`` -> [batch][T][n] over ``dst`` (coefficient
    domain).  Modraise is the exact case with ``src`` = the first S primes of
    the chain and ``dst`` = the whole chain."""
    a, s, d = _arr(a), _arr(src), _arr(dst)
    S, T, n = int(s.size), int(d.size), a.shape[-1]
    assert a.shape[-2] == S and S <= 64 and T <= 8192
    batch = a.size // (S * n)
    out = np.zeros((batch, T, n), dtype=np.uint64)
    _load().oracle_bconv_batch(_p(a), _p(out), _p(s), S, _p(d), T, _log2(n), batch, int(approx),
                               threads or default_threads())
    return out


def moddown_batch(a, qp, L: int, K: int, nearest: bool) -> np.ndarray:
    """a: [batch][L+K][n] coefficient domain over (q_0..q_{L-1}, p_0..p_{K-1})
    -> [batch][L][n]: floor((X + h) / P) mod q_l, h = (P-1)/2 if nearest else 0.
    Rescale is the case K = 1 with P = the last prime."""
    a, qp = _arr(a), _arr(qp)
    n = a.shape[-1]
    batch = a.size // ((L + K) * n)
    out = np.zeros((batch, L, n), dtype=np.uint64)
    _load().oracle_moddown_batch(_p(a), _p(out), _p(qp), _log2(n), L, K, batch, int(nearest))
    return out


def moddown_ntt_batch(a, qp, psi_qp, L: int, K: int, nearest: bool, threads: int | None = None) -> np.ndarray:
    """The same in the NTT domain, by definition: NTT_Q(moddown(INTT_QP(a)))."""
    a = _arr(a)
    n = a.shape[-1]
    coeff = ntt_batch(a, qp, psi_qp, inverse=True, threads=threads)
    md = moddown_batch(coeff, qp, L, K, nearest)
    return ntt_batch(md, _arr(qp)[:L], _arr(psi_qp)[:L], threads=threads)
