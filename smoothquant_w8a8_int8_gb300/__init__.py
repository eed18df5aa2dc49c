"""SmoothQuant W8A8 INT8 linear block for GB300 (sm_103a).

The compute runs in the C-ABI library ``libsq_gb300.so`` (hand-written CUDA);
``binding`` is a thin ctypes layer with the same entry-point names.
``workloads`` draws the seeded synthetic inputs and ``roofline`` holds the
metric arithmetic; ``pipeline`` streams host-resident activations through the
block and ``alpha_sweep`` calibrates the migration strength on synthetic data.
The library is loaded on first use; if it is missing, that call raises.
"""
import importlib

from . import roofline, workloads  # noqa: F401

_SUBMODULES = ("alpha_sweep", "binding", "build", "pipeline", "replicas", "roofline", "workloads")


def __getattr__(name):
    if name in _SUBMODULES:
        return importlib.import_module(f"{__name__}.{name}")
    if name.startswith("_"):
        raise AttributeError(name)
    binding = importlib.import_module(f"{__name__}.binding")
    try:
        return getattr(binding, name)
    except AttributeError:
        raise AttributeError(name) from None
