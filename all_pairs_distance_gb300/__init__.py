"""GB300-native DBSCAN hot path: eps-neighbour counting over all point pairs,
core detection, union-find cluster merging and border assignment, in
hand-written sm_103a CUDA kernels behind a C ABI (``include/dbscan.h``).

The Python names mirror the C entry points; they only marshal arguments
(see ``binding.py``).  Importing this package does not load the library; the
first call does, and raises if it has not been built.
"""
__all__ = [
    "dbscan_fit", "dbscan_fit_ex", "dbscan_fit_host", "dbscan_neighbor_counts",
    "dbscan_workspace_size", "dbscan_workspace_status", "dbscan_strerror",
    "dbscan_workspace_info", "dbscan_profile_begin", "dbscan_profile_end",
]

_BINDING_NAMES = set(__all__) | {"DbscanError", "Status", "library_path", "load", "workspace_for"}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
