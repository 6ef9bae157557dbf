"""GB300-native DeltaNet recurrent-state path: verify block, greedy accept, commit, prefill checkpoints.

The compute lives in ``libdn.so`` (hand-written sm_103a CUDA kernels behind a
C ABI, declared in ``include/dn.h``). ``binding`` is the thin ctypes layer that
marshals torch tensors into those calls; it raises if the library is missing.
"""

_API = (
    "dn_verify_block", "dn_accept_greedy", "dn_commit", "dn_prefill_checkpoint",
    "dn_accept_workspace_bytes", "dn_status_string", "DnError", "load_library",
)


def __getattr__(name):
    if name in _API:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
