"""GB300-native (sm_103a) dense attention forward.

``fwd(q, k, v, scale=None) -> (o, lse)`` runs the CUDA library behind the C-ABI
entry point ``attn_fwd`` (see ``include/attn_fwd.h``).  The library is loaded on
first use; a missing or unbuilt library raises instead of falling back.
"""
from .workloads import Workload  # noqa: F401  (no CUDA needed)


def __getattr__(name):
    if name in ("fwd", "fwd_into", "library", "AttnError", "plan", "status_string", "lib_path",
                "device_status"):
        from . import attn
        return getattr(attn, name)
    raise AttributeError(name)
