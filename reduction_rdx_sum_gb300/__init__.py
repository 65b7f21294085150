"""GB300-native parallel sum reduction (sm_103a).

Importing the package loads nothing on the GPU; the CUDA library is opened on
the first call of an entry point (``reduction_rdx_sum_gb300.abi``).
"""
from . import inputs  # noqa: F401
