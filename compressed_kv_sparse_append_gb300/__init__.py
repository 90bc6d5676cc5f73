"""Compressed-KV decode attention for GB300 (sm_103a).

The compute path is ``libckv.so`` (hand-written CUDA behind a C ABI, declared
in ``include/ckv.h``); ``binding`` marshals torch tensors into its calls.
Importing an entry point loads the library and raises if it was not built.
``workloads`` (seeded synthetic inputs) imports without it.
"""

_BINDING_NAMES = (
    "kv_append_quant", "csa_index_topk", "csa_sparse_attn", "hca_attn",
    "csa2_group_decode", "workspace_bytes", "read_device_status", "Plane", "lib",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
