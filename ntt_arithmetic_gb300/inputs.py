"""Seeded synthetic inputs: uniform residues in [0, q) for [..., L, n] tensors.

This module is the one piece shared by the CUDA path's tests/bench and the CPU
oracle.  It holds none of the transform's arithmetic -- only a counter-based
random generator and rejection sampling -- and imports nothing from either
side.

Generator: each element draws candidates from the SplitMix64 output function
(Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014), applied to a counter formed from (seed, buffer, row, index,
attempt).  A candidate is masked to bit_length(q) bits and accepted when it is
below q; otherwise the next attempt is drawn.  This makes every value exactly
uniform on [0, q), independent of array shape and of any other element, and
reproducible bit for bit on any machine.
"""
from __future__ import annotations

import hashlib

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function, elementwise on uint64 (wrapping)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _keys(seed: int, buffer: int, rows: np.ndarray) -> np.ndarray:
    """Per-row stream keys from (seed, buffer, row), vectorized over rows."""
    k = np.full(rows.shape, np.uint64(0x5EED0000), dtype=np.uint64)
    with np.errstate(over="ignore"):
        for part in (np.uint64(seed & 0xFFFFFFFFFFFFFFFF), np.uint64(buffer & 0xFFFFFFFFFFFFFFFF), rows):
            k = _mix(k ^ part) + _GOLDEN
    return k


def _sample(qrow: np.ndarray, keys: np.ndarray, n: int) -> np.ndarray:
    """rows x n uniform residues; row r is uniform in [0, qrow[r])."""
    rows = keys.size
    bits = np.array([int(q).bit_length() for q in qrow], dtype=np.uint64)
    masks = (np.uint64(1) << bits) - np.uint64(1)
    i2 = np.arange(n, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    with np.errstate(over="ignore"):
        # attempt 0, dense
        out = _mix(keys[:, None] + i2[None, :] * _GOLDEN) & masks[:, None]
        bad_r, bad_i = np.nonzero(out >= qrow[:, None])
        attempt = 1
        while bad_r.size:          # rare: redraw only the rejected elements
            ctr = keys[bad_r] + (i2[bad_i] + np.uint64(attempt) * np.uint64(2 * n)) * _GOLDEN
            cand = _mix(ctr) & masks[bad_r]
            ok = cand < qrow[bad_r]
            out[bad_r[ok], bad_i[ok]] = cand[ok]
            bad_r, bad_i = bad_r[~ok], bad_i[~ok]
            attempt += 1
    return out


def uniform_row(q: int, n: int, seed: int, buffer: int, row: int) -> np.ndarray:
    """n values uniform in [0, q) for stream (seed, buffer, row)."""
    if int(q) < 2:
        raise ValueError("modulus must be >= 2")
    keys = _keys(seed, buffer, np.array([row], dtype=np.uint64))
    return _sample(np.array([int(q)], dtype=np.uint64), keys, n)[0]


def uniform_residues(shape, qs, seed: int, buffer: int = 0, threads: int = 1) -> np.ndarray:
    """Array of ``shape`` = (..., L, n) with row [..., l, :] uniform in [0, qs[l]).

    Rows are keyed by (seed, buffer, flat row index), so two buffers with
    different ``buffer`` ids are independent and regenerating any one row
    gives the same values (see ``uniform_row``).  ``threads`` > 1 fills
    chunks of rows concurrently (numpy releases the GIL in the array
    arithmetic); the values do not depend on it.
    """
    shape = tuple(int(s) for s in shape)
    L, n = shape[-2], shape[-1]
    if len(qs) != L:
        raise ValueError(f"{len(qs)} moduli for L={L}")
    qs = np.array([int(q) for q in qs], dtype=np.uint64)
    if (qs < 2).any():
        raise ValueError("modulus must be >= 2")
    rows = int(np.prod(shape[:-1]))
    out = np.empty((rows, n), dtype=np.uint64)
    chunk = max(1, (1 << 22) // max(n, 1))      # bound temporaries to ~4M elements

    def fill(r0: int) -> None:
        r = np.arange(r0, min(rows, r0 + chunk), dtype=np.uint64)
        out[r0:r0 + r.size] = _sample(qs[(r % np.uint64(L)).astype(np.int64)], _keys(seed, buffer, r), n)

    starts = range(0, rows, chunk)
    if threads > 1 and rows > chunk:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fill, starts))
    else:
        for r0 in starts:
            fill(r0)
    return out.reshape(shape)


def digest(a: np.ndarray) -> str:
    """SHA-256 of the little-endian bytes, logged with generated inputs."""
    return hashlib.sha256(np.ascontiguousarray(a, dtype="<u8").tobytes()).hexdigest()
