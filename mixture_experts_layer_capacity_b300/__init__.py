"""B300-native forward pass of one mixture-of-experts FFN layer.

The compute path is the CUDA library ``libmoe.so`` (C ABI in
``include/moe.h``); :mod:`.binding` marshals arguments to it.  Importing this
package does not load the library; the first call does, and fails loudly if
it is missing.
"""
from .workloads import WORKLOADS, Workload, make_inputs  # noqa: F401
