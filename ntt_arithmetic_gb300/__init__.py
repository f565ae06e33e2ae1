"""ntt_arithmetic_gb300: batched RNS negacyclic NTT and NTT-domain kernels of
RNS-CKKS (pointwise product, ciphertext tensor product, hybrid key-switch
inner product, Galois automorphism) as hand-written sm_103a CUDA kernels
behind a C ABI (include/fhe_ntt.h, libfhe_ntt.so).

The public Python API lives in ``ntt_arithmetic_gb300.api`` (PyTorch only
for device memory and streams); ``inputs`` holds the seeded input generator.
Attributes of ``api`` are also reachable from the package (loaded lazily so
that importing ``inputs`` does not import torch).
"""

__version__ = "0.1.0"


_SUBMODULES = {"api", "inputs", "build", "_native"}


def __getattr__(name):
    if name.startswith("_") or name in _SUBMODULES:
        raise AttributeError(name)      # let the import system load submodules
    from . import api
    try:
        return getattr(api, name)
    except AttributeError:
        raise AttributeError(f"module 'ntt_arithmetic_gb300' has no attribute '{name}'") from None
