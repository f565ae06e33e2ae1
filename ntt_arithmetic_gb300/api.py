"""Python API over the C ABI (include/fhe_ntt.h), with PyTorch tensors as the
device memory and PyTorch's current CUDA stream as the launch stream.

Residue tensors are contiguous CUDA tensors of dtype torch.uint64 (or
torch.int64 holding the same bits) with shape [..., L, n].  Every function
here only marshals arguments; all arithmetic runs in libfhe_ntt.so kernels.
"""
from __future__ import annotations

import ctypes
from typing import Sequence

import numpy as np
import torch

from . import _native as N

_RESIDUE_DTYPES = (torch.uint64, torch.int64)


def _stream(device: torch.device, stream=None):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _residues(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or t.dtype not in _RESIDUE_DTYPES:
        raise TypeError(f"{name} must be a torch.uint64/int64 tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _log2(n: int) -> int:
    if n < 2 or n & (n - 1):
        raise ValueError(f"n = {n} is not a power of two >= 2")
    return n.bit_length() - 1


# ---------------------------------------------------------------- primes ---

def find_primes(log_n: int, count: int, bits: int = 50, below: int = 0) -> list[int]:
    """The `count` largest primes q < min(2^bits, below) with q = 1 mod 2n, descending."""
    out = (ctypes.c_uint64 * count)()
    N.call("fhe_find_primes", log_n, bits, count, below, out)
    return [int(v) for v in out]


def root_of_unity(q: int, log_n: int) -> int:
    """Smallest primitive 2n-th root of unity modulo q."""
    v = ctypes.c_uint64()
    N.call("fhe_root_of_unity", q, log_n, ctypes.byref(v))
    return int(v.value)


def launch_count() -> int:
    """Kernels enqueued by the library so far in this process."""
    return int(N.lib().fhe_launch_count())


def device_status(reset: bool = True) -> int:
    """The library's device status word (fhe_device_status): 0 unless a
    tensor-core kernel gave up a bounded wait (FHE_STATUS_TC_TIMEOUT).
    Synchronizes the device; clears the word when `reset`."""
    v = ctypes.c_int(0)
    N.call("fhe_device_status", ctypes.byref(v), 1 if reset else 0)
    return int(v.value)


def butterfly_probe(out: torch.Tensor, iters: int, tables: "NttTables", stream=None) -> int:
    """Launch the butterfly throughput probe (fhe_butterfly_probe) with one
    CTA of 256 threads per 256 words of `out`; returns the number of
    butterflies the launch performs."""
    _residues(out, "out")
    if out.numel() % 256:
        raise ValueError("out must hold a multiple of 256 words")
    ctas = out.numel() // 256
    N.call("fhe_butterfly_probe", _ptr(out), ctas, int(iters), tables.ref(), _stream(out.device, stream))
    return ctas * 256 * int(iters) * 80


# ---------------------------------------------------------------- tables ---

class NttTables:
    """Twiddle/constant tables for primes q[0..L) at degree n = 2^log_n,
    built on the host by the library and held in one device tensor."""

    def __init__(self, log_n: int, primes: Sequence[int], device="cuda"):
        self.log_n = int(log_n)
        self.primes = [int(q) for q in primes]
        self.L = len(self.primes)
        self.device = torch.device(device)
        nbytes = ctypes.c_size_t()
        N.call("fhe_ntt_tables_bytes", self.log_n, self.L, ctypes.byref(nbytes))
        host = np.zeros(nbytes.value, dtype=np.uint8)
        qs = (ctypes.c_uint64 * self.L)(*self.primes)
        N.call("fhe_ntt_tables_build_host", self.log_n, self.L, qs, host.ctypes.data_as(ctypes.c_void_p),
               nbytes.value)
        self.host_blob = host
        self.blob = torch.from_numpy(host).to(self.device)
        self.struct = N.NttTables()
        N.call("fhe_ntt_tables_bind", _ptr(self.blob), nbytes.value, self.log_n, self.L,
               ctypes.byref(self.struct))

    @property
    def n(self) -> int:
        return 1 << self.log_n

    def ref(self):
        return ctypes.byref(self.struct)


class ModupTables:
    """Garner / mixed-radix constants of the key-switch basis extension for
    basis qp = (q_0..q_{L-1}, p_0..p_{K-1}) split into dnum digits."""

    def __init__(self, L: int, K: int, dnum: int, qp: Sequence[int], device="cuda"):
        self.L, self.K, self.dnum = int(L), int(K), int(dnum)
        if len(qp) != self.L + self.K:
            raise ValueError("qp must list L + K primes")
        nbytes = ctypes.c_size_t()
        N.call("fhe_modup_tables_bytes", self.L, self.K, self.dnum, ctypes.byref(nbytes))
        host = np.zeros(nbytes.value, dtype=np.uint8)
        arr = (ctypes.c_uint64 * len(qp))(*[int(v) for v in qp])
        N.call("fhe_modup_tables_build_host", self.L, self.K, self.dnum, arr,
               host.ctypes.data_as(ctypes.c_void_p), nbytes.value)
        self.blob = torch.from_numpy(host).to(torch.device(device))


def _shape(x: torch.Tensor, tables: NttTables):
    if x.dim() < 2:
        raise ValueError("residue tensor needs shape [..., L, n]")
    L, n = x.shape[-2], x.shape[-1]
    log_n = _log2(n)
    if log_n != tables.log_n:
        raise ValueError(f"n = {n} does not match the tables (n = {tables.n})")
    batch = x.numel() // (L * n)
    return log_n, L, batch


# ------------------------------------------------------------ transforms ---

def ntt_fwd(x: torch.Tensor, tables: NttTables, stream=None) -> torch.Tensor:
    """In-place forward negacyclic NTT of every [.., l, :] row; returns x."""
    _residues(x, "x")
    log_n, L, batch = _shape(x, tables)
    N.call("fhe_ntt_fwd", _ptr(x), log_n, L, batch, tables.ref(), _stream(x.device, stream))
    return x


def ntt_inv(x: torch.Tensor, tables: NttTables, stream=None) -> torch.Tensor:
    """In-place inverse NTT (with 1/n); returns x."""
    _residues(x, "x")
    log_n, L, batch = _shape(x, tables)
    N.call("fhe_ntt_inv", _ptr(x), log_n, L, batch, tables.ref(), _stream(x.device, stream))
    return x


def mul_ntt(out: torch.Tensor, a: torch.Tensor, b: torch.Tensor, tables: NttTables, stream=None) -> torch.Tensor:
    """out = a * b (mod q_l) elementwise; out may be a or b."""
    for t, nm in ((out, "out"), (a, "a"), (b, "b")):
        _residues(t, nm)
    if a.shape != b.shape or out.shape != a.shape:
        raise ValueError("a, b and out must have one shape")
    log_n, L, batch = _shape(a, tables)
    N.call("fhe_mul_ntt", _ptr(out), _ptr(a), _ptr(b), log_n, L, batch, tables.ref(), _stream(a.device, stream))
    return out


def tensor(d: torch.Tensor, a: torch.Tensor, b: torch.Tensor, tables: NttTables, stream=None) -> torch.Tensor:
    """Ciphertext tensor product: a, b [batch, 2, L, n] -> d [batch, 3, L, n]."""
    for t, nm in ((d, "d"), (a, "a"), (b, "b")):
        _residues(t, nm)
    if a.shape != b.shape or a.dim() < 3 or a.shape[-3] != 2:
        raise ValueError("a and b must have shape [..., 2, L, n]")
    if tuple(d.shape) != tuple(a.shape[:-3]) + (3,) + tuple(a.shape[-2:]):
        raise ValueError("d must have shape [..., 3, L, n]")
    log_n, L, batch2 = _shape(a, tables)
    N.call("fhe_tensor", _ptr(d), _ptr(a), _ptr(b), log_n, L, batch2 // 2, tables.ref(), _stream(a.device, stream))
    return d


def automorph(out: torch.Tensor, x: torch.Tensor, k: int, tables: NttTables, domain: str = "ntt",
              stream=None) -> torch.Tensor:
    """out = sigma_k(x) (a(X) -> a(X^k)); domain 'ntt' or 'coeff'."""
    _residues(out, "out")
    _residues(x, "x")
    if out.shape != x.shape:
        raise ValueError("out and x must have one shape")
    dom = {"ntt": N.FHE_DOMAIN_NTT, "coeff": N.FHE_DOMAIN_COEFF}[domain]
    log_n, L, batch = _shape(x, tables)
    N.call("fhe_automorph", _ptr(out), _ptr(x), log_n, L, batch, int(k), dom, tables.ref(),
           _stream(x.device, stream))
    return out


def keyswitch_workspace_bytes(log_n: int, L: int, K: int, dnum: int, batch: int) -> int:
    v = ctypes.c_size_t()
    N.call("fhe_keyswitch_workspace_bytes", log_n, L, K, dnum, batch, ctypes.byref(v))
    return int(v.value)


def _ks_input(x: torch.Tensor, L: int, n: int, in_offset: int, in_stride: int, batch: int | None) -> int:
    item = L * n
    if batch is None:
        if x.shape[-2:] != (L, n) or in_offset or in_stride:
            raise ValueError("x must be [..., L, n] (or pass batch with in_offset/in_stride)")
        batch = x.numel() // item
    stride = in_stride or item
    if in_offset < 0 or stride < item or in_offset + (batch - 1) * stride + item > x.numel():
        raise ValueError("in_offset/in_stride/batch reach outside x")
    return batch


def keyswitch_ip(out: torch.Tensor, x: torch.Tensor, keys: torch.Tensor, L: int, K: int, dnum: int,
                 tables_qp: NttTables, modup: ModupTables, workspace: torch.Tensor | None = None,
                 stream=None, in_offset: int = 0, in_stride: int = 0, batch: int | None = None,
                 approx: bool = False) -> torch.Tensor:
    """Hybrid key-switch inner product (before ModDown).

    x: coefficient-domain input, [batch, L, n] contiguous, or -- with
    in_offset/in_stride (elements) and batch -- `batch` items of [L, n] at
    x.flatten()[in_offset + b * in_stride:] (e.g. component d2 of a
    [batch, 3, L, n] tensor product);  keys: [dnum, 2, L+K, n] NTT domain;
    out: [batch, 2, L+K, n] NTT domain.  approx: approximate ModUp (the CRT
    sum without its e D_j correction) instead of the exact Garner extension."""
    for t, nm in ((out, "out"), (x, "x"), (keys, "keys")):
        _residues(t, nm)
    n = keys.shape[-1]
    log_n = _log2(n)
    if tuple(keys.shape) != (dnum, 2, L + K, n):
        raise ValueError("keys must be [dnum, 2, L+K, n]")
    batch = _ks_input(x, L, n, in_offset, in_stride, batch)
    if tuple(out.shape[-3:]) != (2, L + K, n) or out.numel() != batch * 2 * (L + K) * n:
        raise ValueError("out must be [batch, 2, L+K, n]")
    need = keyswitch_workspace_bytes(log_n, L, K, dnum, batch)
    if workspace is None:
        workspace = torch.empty(need // 8, dtype=torch.uint64, device=x.device)
    src = ctypes.c_void_p(x.data_ptr() + 8 * in_offset)
    ws = (_ptr(workspace), workspace.numel() * workspace.element_size(), _stream(x.device, stream))
    if approx:
        N.call("fhe_keyswitch_ip_ex", _ptr(out), src, in_stride, _ptr(keys), log_n, L, K, dnum, batch,
               N.FHE_MODUP_APPROX, tables_qp.ref(), _ptr(modup.blob), *ws)
    else:
        N.call("fhe_keyswitch_ip", _ptr(out), src, in_stride, _ptr(keys), log_n, L, K, dnum, batch, tables_qp.ref(),
               _ptr(modup.blob), *ws)
    return out


def keyswitch_hoisted(out: torch.Tensor, x: torch.Tensor, keys: torch.Tensor, galois: Sequence[int], L: int, K: int,
                      dnum: int, tables_qp: NttTables, modup: ModupTables, workspace: torch.Tensor | None = None,
                      stream=None, in_offset: int = 0, in_stride: int = 0, batch: int | None = None,
                      approx: bool = False) -> torch.Tensor:
    """Hoisted key switch for R = len(galois) rotations of the same input:
    one ModUp + NTT of the digits, then per Galois element the automorphism
    fused into the inner product.  keys: [R, dnum, 2, L+K, n] NTT domain;
    out: [R, batch, 2, L+K, n] NTT domain; x as in keyswitch_ip."""
    for t, nm in ((out, "out"), (x, "x"), (keys, "keys")):
        _residues(t, nm)
    R = len(galois)
    n = keys.shape[-1]
    log_n = _log2(n)
    if tuple(keys.shape) != (R, dnum, 2, L + K, n):
        raise ValueError("keys must be [R, dnum, 2, L+K, n]")
    batch = _ks_input(x, L, n, in_offset, in_stride, batch)
    if tuple(out.shape[-3:]) != (2, L + K, n) or out.numel() != R * batch * 2 * (L + K) * n:
        raise ValueError("out must be [R, batch, 2, L+K, n]")
    need = keyswitch_workspace_bytes(log_n, L, K, dnum, batch)
    if workspace is None:
        workspace = torch.empty(need // 8, dtype=torch.uint64, device=x.device)
    gal = (ctypes.c_uint32 * max(R, 1))(*[int(k) for k in galois])
    src = ctypes.c_void_p(x.data_ptr() + 8 * in_offset)
    N.call("fhe_keyswitch_hoisted", _ptr(out), src, in_stride, _ptr(keys), gal, R, log_n, L, K, dnum, batch,
           N.FHE_MODUP_APPROX if approx else N.FHE_MODUP_EXACT, tables_qp.ref(), _ptr(modup.blob), _ptr(workspace),
           workspace.numel() * workspace.element_size(), _stream(x.device, stream))
    return out


def keyswitch_ip_noalloc(out: torch.Tensor, x: torch.Tensor, keys: torch.Tensor, L: int, K: int, dnum: int,
                         tables_qp: NttTables, modup: ModupTables, stream=None) -> torch.Tensor:
    """keyswitch_ip without a workspace argument and without any device
    allocation: the library uses its fixed 16 MiB device array instead (for
    callers that cannot allocate; see fhe_keyswitch_ip_noalloc in the C
    header for the size limit and the rule that overlapping calls race).
    x: [batch, L, n] contiguous; keys: [dnum, 2, L+K, n]; out: [batch, 2, L+K, n]."""
    for t, nm in ((out, "out"), (x, "x"), (keys, "keys")):
        _residues(t, nm)
    n = keys.shape[-1]
    log_n = _log2(n)
    if tuple(keys.shape) != (dnum, 2, L + K, n) or x.shape[-2:] != (L, n):
        raise ValueError("x must be [..., L, n] and keys [dnum, 2, L+K, n]")
    batch = x.numel() // (L * n)
    if out.numel() != batch * 2 * (L + K) * n:
        raise ValueError("out must be [batch, 2, L+K, n]")
    N.call("fhe_keyswitch_ip_noalloc", _ptr(out), _ptr(x), 0, _ptr(keys), log_n, L, K, dnum, batch,
           tables_qp.ref(), _ptr(modup.blob), _stream(x.device, stream))
    return out


# ------------------------------------------------------------ ModDown ------

class ModdownTables:
    """Constants of the division by P = p_0..p_{K-1} for basis
    qp = (q_0..q_{L-1}, p_0..p_{K-1}).  Rescale uses (L-1, 1) over the chain."""

    def __init__(self, L: int, K: int, qp: Sequence[int], device="cuda"):
        self.L, self.K = int(L), int(K)
        if len(qp) != self.L + self.K:
            raise ValueError("qp must list L + K primes")
        nbytes = ctypes.c_size_t()
        N.call("fhe_moddown_tables_bytes", self.L, self.K, ctypes.byref(nbytes))
        host = np.zeros(nbytes.value, dtype=np.uint8)
        arr = (ctypes.c_uint64 * len(qp))(*[int(v) for v in qp])
        N.call("fhe_moddown_tables_build_host", self.L, self.K, arr, host.ctypes.data_as(ctypes.c_void_p),
               nbytes.value)
        self.blob = torch.from_numpy(host).to(torch.device(device))


def moddown_workspace_bytes(log_n: int, L: int, K: int, batch: int) -> int:
    v = ctypes.c_size_t()
    N.call("fhe_moddown_workspace_bytes", log_n, L, K, batch, ctypes.byref(v))
    return int(v.value)


def moddown(out: torch.Tensor, x: torch.Tensor, L: int, K: int, tables_qp: NttTables, md: ModdownTables,
            domain: str = "ntt", nearest: bool = True, workspace: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """out = floor((X + h) / P) mod q_l: x [batch, L+K, n] -> out [batch, L, n]."""
    _residues(out, "out")
    _residues(x, "x")
    n = x.shape[-1]
    log_n = _log2(n)
    if x.shape[-2] != L + K or out.shape[-2] != L or out.numel() * (L + K) != x.numel() * L:
        raise ValueError("x must be [batch, L+K, n] and out [batch, L, n]")
    batch = x.numel() // ((L + K) * n)
    dom = {"ntt": N.FHE_DOMAIN_NTT, "coeff": N.FHE_DOMAIN_COEFF}[domain]
    need = moddown_workspace_bytes(log_n, L, K, batch)
    if workspace is None:
        workspace = torch.empty(need // 8, dtype=torch.uint64, device=x.device)
    N.call("fhe_moddown", _ptr(out), _ptr(x), log_n, L, K, batch, dom,
           N.FHE_ROUND_NEAREST if nearest else N.FHE_ROUND_TRUNCATE, tables_qp.ref(), _ptr(md.blob),
           _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(x.device, stream))
    return out


def rescale(out: torch.Tensor, x: torch.Tensor, tables_q: NttTables, rs: ModdownTables, domain: str = "ntt",
            nearest: bool = True, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Drop the last prime: x [batch, L, n] -> out [batch, L-1, n], dividing by it with rounding."""
    L = x.shape[-2]
    return moddown(out, x, L - 1, 1, tables_q, rs, domain=domain, nearest=nearest, workspace=workspace,
                   stream=stream)


def keyswitch_decompose(digits: torch.Tensor, x: torch.Tensor, L: int, K: int, dnum: int, tables_qp: NttTables,
                        modup: ModupTables, stream=None, in_offset: int = 0, in_stride: int = 0,
                        batch: int | None = None, approx: bool = False) -> torch.Tensor:
    """digits [batch, dnum, L+K, n] (NTT domain) = NTT of every extended digit
    of x (x as in keyswitch_ip)."""
    _residues(digits, "digits")
    _residues(x, "x")
    n = digits.shape[-1]
    log_n = _log2(n)
    batch = _ks_input(x, L, n, in_offset, in_stride, batch)
    if tuple(digits.shape[-3:]) != (dnum, L + K, n) or digits.numel() != batch * dnum * (L + K) * n:
        raise ValueError("digits must be [batch, dnum, L+K, n]")
    src = ctypes.c_void_p(x.data_ptr() + 8 * in_offset)
    N.call("fhe_keyswitch_decompose", _ptr(digits), src, in_stride, log_n, L, K, dnum, batch,
           N.FHE_MODUP_APPROX if approx else N.FHE_MODUP_EXACT, tables_qp.ref(), _ptr(modup.blob),
           _stream(x.device, stream))
    return digits


def keyswitch_apply(out: torch.Tensor, digits: torch.Tensor, keys: torch.Tensor, L: int, K: int, dnum: int,
                    tables_qp: NttTables, galois: Sequence[int] | None = None, stream=None) -> torch.Tensor:
    """Inner product of precomputed digits with keys; with `galois`, one
    rotation per element, the automorphism fused into the read."""
    for t, nm in ((out, "out"), (digits, "digits"), (keys, "keys")):
        _residues(t, nm)
    n = digits.shape[-1]
    log_n = _log2(n)
    batch = digits.numel() // (dnum * (L + K) * n)
    R = 1 if galois is None else len(galois)
    kshape = (dnum, 2, L + K, n) if galois is None else (R, dnum, 2, L + K, n)
    if tuple(keys.shape) != kshape or out.numel() != R * batch * 2 * (L + K) * n:
        raise ValueError("keys/out shapes do not match")
    gal = None if galois is None else (ctypes.c_uint32 * max(R, 1))(*[int(k) for k in galois])
    N.call("fhe_keyswitch_apply", _ptr(out), _ptr(digits), _ptr(keys), gal, R, log_n, L, K, dnum, batch,
           tables_qp.ref(), _stream(digits.device, stream))
    return out


# ------------------------------------------------------ basis conversion ---

class BconvTables:
    """Constants of the conversion from primes ``src`` to primes ``dst``."""

    def __init__(self, src: Sequence[int], dst: Sequence[int], device="cuda"):
        self.src = [int(v) for v in src]
        self.dst = [int(v) for v in dst]
        S, T = len(self.src), len(self.dst)
        nbytes = ctypes.c_size_t()
        N.call("fhe_bconv_tables_bytes", S, T, ctypes.byref(nbytes))
        host = np.zeros(nbytes.value, dtype=np.uint8)
        a = (ctypes.c_uint64 * S)(*self.src)
        b = (ctypes.c_uint64 * T)(*self.dst)
        N.call("fhe_bconv_tables_build_host", S, a, T, b, host.ctypes.data_as(ctypes.c_void_p), nbytes.value)
        self.blob = torch.from_numpy(host).to(torch.device(device))


def bconv(out: torch.Tensor, x: torch.Tensor, tables: BconvTables, approx: bool = False, stream=None) -> torch.Tensor:
    """x [batch, S, n] over tables.src -> out [batch, T, n] over tables.dst
    (coefficient domain); exact (X in [0, Q)) or approximate (X + e Q)."""
    _residues(out, "out")
    _residues(x, "x")
    S, T = len(tables.src), len(tables.dst)
    n = x.shape[-1]
    log_n = _log2(n)
    if x.shape[-2] != S or out.shape[-2] != T or out.shape[-1] != n or x.numel() * T != out.numel() * S:
        raise ValueError("x must be [batch, S, n] and out [batch, T, n]")
    batch = x.numel() // (S * n)
    N.call("fhe_bconv", _ptr(out), _ptr(x), log_n, S, T, batch, N.FHE_BCONV_APPROX if approx else N.FHE_BCONV_EXACT,
           _ptr(tables.blob), _stream(x.device, stream))
    return out


def modraise(out: torch.Tensor, x: torch.Tensor, tables: BconvTables, stream=None) -> torch.Tensor:
    """Lift x [batch, S, n] over the first S primes of a chain to out
    [batch, T, n] over the whole chain (exact Garner extension; tables built
    with src = chain[:S], dst = chain)."""
    return bconv(out, x, tables, approx=False, stream=stream)
