"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, its host-side prime/root/table builders agree with the
oracle, its arithmetic self-test passes, and invalid calls fail on the host
with a status code before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from ntt_arithmetic_gb300 import _native as N
from ntt_arithmetic_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fhe_ntt.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fhe_\w+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for required in ["fhe_ntt_fwd", "fhe_ntt_inv", "fhe_mul_ntt", "fhe_tensor", "fhe_keyswitch_ip", "fhe_automorph"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in N.SIGNATURES, f"binding lacks {name}"


def test_version_and_status_strings(lib):
    assert lib.fhe_version() == 100
    for s in [0, -1, -2, -3, -4, -5, 7]:
        assert isinstance(lib.fhe_status_str(s), bytes) and lib.fhe_status_str(s)


def test_host_arithmetic_selftest(lib):
    assert lib.fhe_selftest_host(12345, 20000) == 0
    assert lib.fhe_selftest_host(0, 20000) == 0


@pytest.mark.parametrize("log_n,count", [(11, 112), (16, 32), (17, 64), (1, 4), (12, 8)])
def test_primes_match_oracle(lib, log_n, count):
    out = (ctypes.c_uint64 * count)()
    assert lib.fhe_find_primes(log_n, 50, count, 0, out) == 0
    assert [int(v) for v in out] == [int(v) for v in oracle.primes(2 << log_n, count)]


def test_special_primes_follow_the_chain(lib):
    # key switch: Q = 24 largest, P = the next 8 in the same descending scan
    q = (ctypes.c_uint64 * 24)()
    p = (ctypes.c_uint64 * 8)()
    assert lib.fhe_find_primes(16, 50, 24, 0, q) == 0
    assert lib.fhe_find_primes(16, 50, 8, q[23], p) == 0
    assert list(q) + list(p) == [int(v) for v in oracle.primes(1 << 17, 32)]


@pytest.mark.parametrize("log_n", [1, 2, 5, 11, 16, 17])
def test_root_of_unity_matches_oracle(lib, log_n):
    qs = oracle.primes(2 << log_n, 3)
    for q in qs:
        v = ctypes.c_uint64()
        assert lib.fhe_root_of_unity(int(q), log_n, ctypes.byref(v)) == 0
        assert v.value == oracle.psi(int(q), 2 << log_n)


def test_tables_contents(lib):
    """Spot-check the table blob against the definitions: fwd[k] = psi^brv(k)
    (merged forward), inv[h + j] = psi^(-j n / h) for h = 2^e (cyclic inverse
    twiddles omega_2h^-j), twist[j] = n^-1 psi^-j, each with its Shoup
    companion floor(w 2^64 / q)."""
    log_n, L = 6, 3
    n = 1 << log_n
    qs = [int(v) for v in oracle.primes(2 * n, L)]
    nb = ctypes.c_size_t()
    assert lib.fhe_ntt_tables_bytes(log_n, L, ctypes.byref(nb)) == 0
    blob = np.zeros(nb.value, dtype=np.uint8)
    arr = (ctypes.c_uint64 * L)(*qs)
    assert lib.fhe_ntt_tables_build_host(log_n, L, arr, blob.ctypes.data_as(ctypes.c_void_p), nb.value) == 0
    t = N.NttTables()
    base = blob.ctypes.data
    assert lib.fhe_ntt_tables_bind(ctypes.c_void_p(base), nb.value, log_n, L, ctypes.byref(t)) == 0
    words = lambda ptr, cnt: np.frombuffer(blob, dtype=np.uint64, count=cnt, offset=ptr - base)  # noqa: E731
    assert list(words(t.q, L)) == qs
    fwd = words(t.fwd, L * n * 2).reshape(L, n, 2)
    inv = words(t.inv, L * n * 2).reshape(L, n, 2)
    twi = words(t.twist, L * n * 2).reshape(L, n, 2)
    for l, q in enumerate(qs):
        psi = oracle.psi(q, 2 * n)
        for k in range(1, n):
            w = pow(psi, oracle.brv(k, log_n), q)
            slot = ctypes.c_uint32()
            assert lib.fhe_ntt_fwd_table_slot(log_n, k, ctypes.byref(slot)) == 0
            assert int(fwd[l, slot.value, 0]) == w and int(fwd[l, slot.value, 1]) == (w << 64) // q
            h = 1 << (k.bit_length() - 1)
            wi = pow(psi, -(k - h) * (n // h), q)
            assert int(inv[l, k, 0]) == wi and int(inv[l, k, 1]) == (wi << 64) // q
        for j in range(n):
            tj = pow(n, -1, q) * pow(psi, -j, q) % q
            assert int(twi[l, j, 0]) == tj and int(twi[l, j, 1]) == (tj << 64) // q


@pytest.mark.parametrize("log_n", list(range(1, 18)))
def test_fwd_table_slots_are_a_permutation_within_each_stage(lib, log_n):
    """The stored order of the forward twiddles is a permutation of each
    stage's block [2^s, 2^(s+1)), the identity outside the last pass."""
    n = 1 << log_n
    slot = ctypes.c_uint32()
    slots = []
    for k in range(n):
        assert lib.fhe_ntt_fwd_table_slot(log_n, k, ctypes.byref(slot)) == 0
        slots.append(slot.value)
    assert sorted(slots) == list(range(n))
    for k, s_ in enumerate(slots):
        if k >= 2:
            assert s_.bit_length() == k.bit_length()
    assert lib.fhe_ntt_fwd_table_slot(log_n, n, ctypes.byref(slot)) == N.FHE_EINVAL


def test_table_builder_rejects_bad_moduli(lib):
    nb = ctypes.c_size_t()
    lib.fhe_ntt_tables_bytes(4, 1, ctypes.byref(nb))
    blob = np.zeros(nb.value, dtype=np.uint8)
    ptr = blob.ctypes.data_as(ctypes.c_void_p)
    good = int(oracle.primes(32, 1)[0])
    for bad in [good + 32,            # = 1 mod 32 but composite
                97,                   # prime, too small
                int(oracle.primes(32, 1, bits=62)[0]),   # prime, too large
                good - 2]:            # not = 1 mod 2n
        assert lib.fhe_ntt_tables_build_host(4, 1, (ctypes.c_uint64 * 1)(bad), ptr, nb.value) == N.FHE_EINVAL
    assert lib.fhe_ntt_tables_build_host(4, 1, (ctypes.c_uint64 * 1)(good), ptr, nb.value - 1) == N.FHE_ESPACE
    assert lib.fhe_ntt_tables_build_host(4, 1, (ctypes.c_uint64 * 1)(good), ptr, nb.value) == N.FHE_OK


def test_invalid_calls_fail_before_launch(lib):
    """Host-side validation: bad sizes, k, tables and host pointers return a
    status code; nothing is launched (the launch counter does not move)."""
    before = lib.fhe_launch_count()
    t = N.NttTables()
    host = np.zeros(64, dtype=np.uint64)
    hp = ctypes.c_void_p(host.ctypes.data)
    assert lib.fhe_ntt_fwd(hp, 0, 1, 1, ctypes.byref(t), None) == N.FHE_EINVAL        # log_n = 0
    assert lib.fhe_ntt_fwd(hp, 18, 1, 1, ctypes.byref(t), None) == N.FHE_EINVAL       # log_n too big
    assert lib.fhe_ntt_fwd(hp, 5, 0, 1, ctypes.byref(t), None) == N.FHE_EINVAL        # L = 0
    assert lib.fhe_ntt_fwd(hp, 5, 1, 0, ctypes.byref(t), None) == N.FHE_EINVAL        # batch = 0
    assert lib.fhe_ntt_fwd(hp, 5, 1, 1, None, None) == N.FHE_EINVAL                   # no tables
    # a bound table struct whose blob is host memory: rejected as a host pointer
    nb = ctypes.c_size_t()
    lib.fhe_ntt_tables_bytes(5, 1, ctypes.byref(nb))
    blob = np.zeros(nb.value, dtype=np.uint8)
    q = int(oracle.primes(64, 1)[0])
    lib.fhe_ntt_tables_build_host(5, 1, (ctypes.c_uint64 * 1)(q), blob.ctypes.data_as(ctypes.c_void_p), nb.value)
    assert lib.fhe_ntt_tables_bind(ctypes.c_void_p(blob.ctypes.data), nb.value, 5, 1, ctypes.byref(t)) == 0
    assert lib.fhe_ntt_fwd(hp, 5, 1, 1, ctypes.byref(t), None) == N.FHE_EDEVICE
    assert lib.fhe_ntt_fwd(hp, 5, 2, 1, ctypes.byref(t), None) == N.FHE_EINVAL       # L > tables.L
    assert lib.fhe_ntt_fwd(hp, 6, 1, 1, ctypes.byref(t), None) == N.FHE_EINVAL       # n != tables n
    assert lib.fhe_automorph(hp, hp, 5, 1, 1, 4, 1, ctypes.byref(t), None) == N.FHE_EINVAL   # even k
    assert lib.fhe_automorph(hp, hp, 5, 1, 1, 65, 1, ctypes.byref(t), None) == N.FHE_EINVAL  # k >= 2n
    assert lib.fhe_automorph(hp, hp, 5, 1, 1, 3, 7, ctypes.byref(t), None) == N.FHE_EINVAL   # bad domain
    odd = ctypes.c_void_p(host.ctypes.data + 8)
    assert lib.fhe_mul_ntt(odd, hp, hp, 5, 1, 1, ctypes.byref(t), None) == N.FHE_EINVAL  # misaligned
    ws = ctypes.c_size_t()
    assert lib.fhe_keyswitch_workspace_bytes(16, 24, 8, 3, 1, ctypes.byref(ws)) == 0
    assert ws.value == 3 * 32 * 65536 * 8
    assert lib.fhe_keyswitch_workspace_bytes(16, 24, 8, 25, 1, ctypes.byref(ws)) == N.FHE_EINVAL  # dnum > L
    assert lib.fhe_keyswitch_workspace_bytes(16, 40, 30, 2, 1, ctypes.byref(ws)) == N.FHE_EINVAL  # L+K > 64
    assert lib.fhe_launch_count() == before


def test_modup_table_shapes(lib):
    nb = ctypes.c_size_t()
    assert lib.fhe_modup_tables_bytes(24, 8, 3, ctypes.byref(nb)) == 0
    assert lib.fhe_modup_tables_bytes(7, 3, 3, ctypes.byref(nb)) == 0        # ragged digits 3,3,1
    assert lib.fhe_modup_tables_bytes(40, 8, 2, ctypes.byref(nb)) == N.FHE_EINVAL   # alpha = 20 > 16
    assert lib.fhe_modup_tables_bytes(4, 1, 3, ctypes.byref(nb)) == N.FHE_EINVAL    # digit 2 would be empty


def test_butterfly_probe_validates_on_the_host(lib):
    t = N.NttTables()
    fake = ctypes.c_void_p(1 << 20)            # never dereferenced: validation fails first
    assert lib.fhe_butterfly_probe(None, 1, 1, ctypes.byref(t), None) == N.FHE_EINVAL
    assert lib.fhe_butterfly_probe(fake, 0, 1, ctypes.byref(t), None) == N.FHE_EINVAL
    assert lib.fhe_butterfly_probe(fake, 1, 0, ctypes.byref(t), None) == N.FHE_EINVAL
    assert lib.fhe_butterfly_probe(fake, 1, 129, ctypes.byref(t), None) == N.FHE_EINVAL
    assert lib.fhe_butterfly_probe(fake, 1, 1, None, None) == N.FHE_EINVAL
    t.log_n = 10                                # the probe reads 2048 table entries
    assert lib.fhe_butterfly_probe(fake, 1, 1, ctypes.byref(t), None) == N.FHE_EINVAL


def test_tampered_table_struct_fails_before_launch(lib):
    """A table struct whose array pointers are not where fhe_ntt_tables_bind
    put them (another buffer, host memory, a shifted offset) or whose size or
    shape fields were edited is refused with FHE_EINVAL before anything is
    launched, so no kernel reads twiddles from outside the caller's blob."""
    log_n, L = 5, 2
    nb = ctypes.c_size_t()
    lib.fhe_ntt_tables_bytes(log_n, L, ctypes.byref(nb))
    blob = np.zeros(nb.value, dtype=np.uint8)
    qs = [int(v) for v in oracle.primes(2 << log_n, L)]
    lib.fhe_ntt_tables_build_host(log_n, L, (ctypes.c_uint64 * L)(*qs), blob.ctypes.data_as(ctypes.c_void_p), nb.value)
    other = np.zeros(nb.value, dtype=np.uint8)
    host = np.zeros(4 << log_n, dtype=np.uint64)
    hp = ctypes.c_void_p(host.ctypes.data)
    fields = ["q", "consts", "fwd", "inv", "twist"]
    before = lib.fhe_launch_count()
    for field in fields + ["bytes", "L", "log_n", "blob"]:
        for how in ("other", "shift"):
            t = N.NttTables()
            assert lib.fhe_ntt_tables_bind(ctypes.c_void_p(blob.ctypes.data), nb.value, log_n, L, ctypes.byref(t)) == 0
            if field in fields:
                v = getattr(t, field)
                setattr(t, field, other.ctypes.data + (v - blob.ctypes.data) if how == "other" else v + 16)
            elif field == "bytes":
                t.bytes = t.bytes + 256 if how == "other" else t.bytes - 16
            elif field == "L":
                t.L = L + 1 if how == "other" else 0
            elif field == "log_n":
                t.log_n = 0 if how == "other" else 18
            else:
                t.blob = other.ctypes.data if how == "other" else t.blob + 8
            ref = ctypes.byref(t)
            assert lib.fhe_ntt_fwd(hp, log_n, 1, 1, ref, None) == N.FHE_EINVAL, (field, how)
            assert lib.fhe_ntt_inv(hp, log_n, 1, 1, ref, None) == N.FHE_EINVAL, (field, how)
            assert lib.fhe_mul_ntt(hp, hp, hp, log_n, 1, 1, ref, None) == N.FHE_EINVAL, (field, how)
            assert lib.fhe_tensor(hp, hp, hp, log_n, 1, 1, ref, None) == N.FHE_EINVAL, (field, how)
            assert lib.fhe_automorph(hp, hp, log_n, 1, 1, 3, 1, ref, None) == N.FHE_EINVAL, (field, how)
            assert lib.fhe_butterfly_probe(hp, 1, 1, ref, None) == N.FHE_EINVAL, (field, how)
    # the untouched struct passes the table check and stops only at the device check (host memory)
    t = N.NttTables()
    assert lib.fhe_ntt_tables_bind(ctypes.c_void_p(blob.ctypes.data), nb.value, log_n, L, ctypes.byref(t)) == 0
    assert lib.fhe_ntt_fwd(hp, log_n, 1, 1, ctypes.byref(t), None) == N.FHE_EDEVICE
    assert lib.fhe_launch_count() == before
