"""GB300-native DeltaNet recurrent-state path: verify block, greedy accept, commit, prefill checkpoints.

The compute lives in ``libdn.so`` (hand-written sm_103a CUDA kernels behind a
C ABI, declared in ``include/dn.h``). ``binding`` is the thin ctypes layer that
marshals torch tensors into those calls; it raises if the library is missing.
"""

_API = (
    # the scope's four entry points and their helpers
    "dn_verify_block", "dn_accept_greedy", "dn_commit", "dn_prefill_checkpoint",
    "dn_accept_workspace_bytes", "accept_workspace",
    # recompute on commit
    "dn_verify_block_deltas", "dn_commit_deltas",
    # accept without a caller workspace
    "dn_accept_greedy_noalloc",
    # drafts from the request's own context; prefix-cache index
    "dn_context_drafts", "PrefixCache",
    # bounded-wait diagnostics
    "dn_prefill_wait_timeouts", "dn_wait_selftest",
    # errors and loading
    "dn_status_string", "DnError", "load_library",
)


def __getattr__(name):
    if name in _API:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
