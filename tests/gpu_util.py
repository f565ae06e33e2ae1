"""Helpers for the GPU parity tests (imported only by gpu-marked tests)."""
from __future__ import annotations

import functools

import numpy as np
import torch

from ntt_arithmetic_gb300 import build as B

B.build()
from ntt_arithmetic_gb300 import api  # noqa: E402


def dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint64)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


@functools.lru_cache(maxsize=64)
def primes(log_n: int, count: int) -> tuple:
    return tuple(api.find_primes(log_n, count))


@functools.lru_cache(maxsize=64)
def tables(log_n: int, prime_tuple: tuple) -> api.NttTables:
    return api.NttTables(log_n, list(prime_tuple))


def qp_basis(log_n: int, L: int, K: int) -> list[int]:
    q = api.find_primes(log_n, L)
    p = api.find_primes(log_n, K, below=q[-1]) if K else []
    return q + p


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Device-side exact comparison (int64 views carry the same 64 bits)."""
    return bool(torch.equal(a.view(torch.int64), b.view(torch.int64)))
