"""GB300-native parallel sum reduction (sm_103a).

The product is the C-ABI library ``librdx.so`` (header ``include/rdx.h``),
built in-tree by ``reduction_rdx_sum_gb300.build``.  ``abi`` binds its entry
points under the same names; importing the package opens nothing on the GPU,
the library is loaded on the first call.  ``inputs`` draws the seeded
synthetic workloads.
"""
import importlib

from . import inputs  # noqa: F401


def __getattr__(name):
    if name.startswith("rdx_") or name in ("abi", "RdxError"):
        abi = importlib.import_module(__name__ + ".abi")
        return abi if name == "abi" else getattr(abi, name)
    raise AttributeError(name)
