"""Paged KV decode attention for NVIDIA GB300 (sm_103a).

The compute path is libpkv.so (hand-written CUDA behind the C ABI in
include/pkv.h); ``paged_kv_decode_04_gb300.binding`` marshals torch tensors
into it.  The binding is loaded lazily so that the seeded workload generator
(``paged_kv_decode_04_gb300.synth``) can be used without a GPU.
"""
__version__ = "0.1.0"

_BINDING_NAMES = {
    "kv_append", "paged_decode_attention", "decode_step", "kv_write_prefill", "workspace_bytes", "plan_splits", "strerror",
    "abi_version", "PkvError",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
