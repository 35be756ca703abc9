"""liblla: causal Local Linear Attention forward for GB300 (sm_103a).

The compute path is the C-ABI shared library ``liblla.so`` (built from ``csrc/``); the Python
module ``binding`` marshals torch tensors into its entry points. Importing this package does not
load the library: the binding is loaded on first use and raises if the library is missing.
"""
from . import workloads  # noqa: F401

_BINDING = {
    "lla_forward", "lla_forward_ws", "lla_workspace_size", "lla_moments", "lla_forward_host",
    "lla_stream_status", "lla_status_string", "lla_version", "LlaError", "library_path",
    "launch_count", "profile_enable", "profile_collect", "lla_forward_noalloc",
    "lla_parallax_forward", "lla_decode", "lla_parallax_decode", "lla_parallax_backward",
    "Options",
}


def __getattr__(name):
    if name in _BINDING:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
