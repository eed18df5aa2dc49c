"""SmoothQuant W8A8 INT8 linear block for GB300 (sm_103a).

The compute runs in the C-ABI library ``libsq_gb300.so`` (hand-written CUDA);
this package is a thin ctypes binding with the same entry-point names, plus the
seeded workload generator and the roofline arithmetic.  The library is loaded
on first use; if it is missing, that call raises.
"""
from . import roofline, workloads  # noqa: F401


def __getattr__(name):
    # the ctypes binding loads the CUDA library; defer it to first use
    from . import binding
    if hasattr(binding, name):
        return getattr(binding, name)
    raise AttributeError(name)
