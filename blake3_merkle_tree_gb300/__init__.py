"""GB300-native BLAKE3 digest (keyed, or the default unkeyed mode) of one buffer resident in
device memory.

The work runs in hand-written sm_103a CUDA kernels behind the C ABI declared in
``include/blake3_gb300.h`` (``libb3g.so``).  ``binding`` is a thin ctypes layer
with the same function names that only marshals torch tensors and streams into
that ABI.  ``workloads`` makes the seeded synthetic inputs.

The binding is imported lazily so that ``workloads`` can be used on machines
where the CUDA library has not been built; any call into the binding without
the library raises.
"""

from __future__ import annotations

_BINDING_NAMES = (
    "blake3_keyed_hash",
    "blake3_keyed_hash_ws",
    "blake3_keyed_hash_noalloc",
    "blake3_keyed_hash_xof",
    "blake3_keyed_hash_host",
    "blake3_hash",
    "blake3_hash_ws",
    "blake3_hash_xof",
    "blake3_hash_host",
    "Hasher",
    "blake3_workspace_size",
    "blake3_keyed_chunk_cvs",
    "blake3_keyed_subtree_root",
    "blake3_keyed_tile_roots",
    "blake3_keyed_reduce_cvs",
    "blake3_reduce_workspace_size",
    "blake3_device_status",
    "blake3_selftest_bounded_wait",
    "blake3_tile_count",
    "blake3_strerror",
    "blake3_set_option",
    "B3GError",
    "library",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
