"""The allocation-free key switch (fhe_keyswitch_ip_noalloc), for callers of
this library that cannot allocate device memory.

Called through the C ABI, twice in a row on different inputs, it must give
exactly the output of fhe_keyswitch_ip with a caller-owned workspace (the
tests' tolerance for this integer path is bit-exact).  Oversized problems
must be refused before any launch.  This file is collected last, and passes
both alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest

from ntt_arithmetic_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import gpu_util
    return gpu_util


def _call_noalloc(g, out, x, keys, log_n, L, K, dnum, batch, t, mt):
    lib = g.api.N.lib()
    return lib.fhe_keyswitch_ip_noalloc(ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(x.data_ptr()), 0,
                                        ctypes.c_void_p(keys.data_ptr()), log_n, L, K, dnum, batch, t.ref(),
                                        ctypes.c_void_p(mt.blob.data_ptr()), None)


def test_noalloc_keyswitch_matches_allocating_entry_point_twice(g):
    import torch
    log_n, L, K, dnum, batch = 13, 24, 8, 3, 1          # 6 MiB of workspace: fits the 16 MiB array
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    lib = g.api.N.lib()
    assert lib.fhe_keyswitch_noalloc_max_bytes() == 16 << 20
    keys = g.dev(inputs.uniform_residues((dnum, 2, L + K, n), qp, 31, buffer=1))
    for call in range(2):
        x = g.dev(inputs.uniform_residues((batch, L, n), qp[:L], 31 + call, buffer=0))
        ref = torch.empty((batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
        g.api.keyswitch_ip(ref, x, keys, L, K, dnum, t, mt)
        out = torch.full((batch, 2, L + K, n), 7, dtype=torch.uint64, device="cuda")
        torch.cuda.synchronize()
        assert _call_noalloc(g, out, x, keys, log_n, L, K, dnum, batch, t, mt) == 0
        torch.cuda.synchronize()
        assert np.array_equal(g.host(out), g.host(ref)), f"call {call}"


def test_noalloc_keyswitch_refuses_oversized_problems(g):
    import torch
    log_n, L, K, dnum, batch = 16, 24, 8, 3, 1          # 48 MiB of workspace: beyond the array
    n = 1 << log_n
    qp = g.qp_basis(log_n, L, K)
    t = g.tables(log_n, tuple(qp))
    mt = g.api.ModupTables(L, K, dnum, qp)
    x = torch.zeros((batch, L, n), dtype=torch.uint64, device="cuda")
    keys = torch.zeros((dnum, 2, L + K, n), dtype=torch.uint64, device="cuda")
    out = torch.zeros((batch, 2, L + K, n), dtype=torch.uint64, device="cuda")
    before = g.api.launch_count()
    assert _call_noalloc(g, out, x, keys, log_n, L, K, dnum, batch, t, mt) == g.api.N.FHE_ESPACE
    assert g.api.launch_count() == before
