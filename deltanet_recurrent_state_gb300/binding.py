"""Thin ctypes binding of libdn.so (include/dn.h) for torch tensors.

Argument marshalling only: shapes, dtypes and devices are checked, raw device
pointers and the current CUDA stream are passed to the C ABI, and a non-OK
status raises ``DnError``. Every step of the computation runs in the library's
CUDA kernels; there is no other implementation to fall back to, so a missing
library raises at load time.
"""

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdn.so")

DN_OK, DN_ERR_INVALID_ARG, DN_ERR_UNSUPPORTED, DN_ERR_CUDA = 0, 1, 2, 3
DN_F16, DN_F32 = 0, 1
MAX_BLOCK = 16
PREFILL_CHUNK = 64

_DT = {torch.float16: DN_F16, torch.float32: DN_F32}

# Every exported symbol of include/dn.h with its ctypes signature.
_P, _I, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "dn_verify_block": (_I, [_I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dn_accept_workspace_bytes": (_S, [_I, _I, _I]),
    "dn_accept_greedy": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _S, _P]),
    "dn_commit": (_I, [_I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "dn_prefill_checkpoint": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _P, _P]),
    "dn_prefill_checkpoint_tc": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                      _P, _P, _P]),
    "dn_status_string": (ctypes.c_char_p, [_I]),
    "dn_accept_greedy_noalloc": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "dn_prefill_wait_timeouts": (ctypes.c_uint, []),
    "dn_wait_selftest": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "dn_verify_block_deltas": (_I, [_I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dn_commit_deltas": (_I, [_I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "dn_prefix_cache_create": (_P, [_I, _I]),
    "dn_prefix_cache_destroy": (None, [_P]),
    "dn_prefix_cache_insert": (_I, [_P, _P, _I, ctypes.c_int32, _P]),
    "dn_prefix_cache_lookup": (_I, [_P, _P, _I, _P, _P]),
    "dn_prefix_cache_size": (_I, [_P]),
    "dn_context_drafts": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
}


class DnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = load_library().dn_status_string(status).decode()
        super().__init__("%s failed: %s" % (fn, msg))


_lib = None


def load_library(path=None):
    """Load libdn.so (once) and declare the C signatures. Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            "libdn.so is not built (%s); build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`" % p)
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(name, status):
    if status != DN_OK:
        raise DnError(name, status)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _require(cond, what):
    """Argument check that survives python -O: the C ABI receives raw pointers and cannot
    see a tensor's size, so a wrong shape must stop here."""
    if not cond:
        raise ValueError(what)


def _dev(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("all tensors must be CUDA tensors")
            if not t.is_contiguous():
                raise ValueError("all tensors must be contiguous")


def dn_verify_block(q, k, v, beta, g, state_in, out=None, ckpt=None, stream=None):
    """q, k [N,T,H,dk]; v [N,T,H,dv]; beta, g [N,T,H] fp32; state_in [N,H,dv,dk].

    Returns (out [N,T,H,dv], ckpt [N,T,H,dv,dk]); allocates them with torch if not given.
    """
    N, T, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((N, T, H, dv), dtype=q.dtype, device=q.device)
    if ckpt is None:
        ckpt = torch.empty((N, T, H, dv, dk), dtype=state_in.dtype, device=q.device)
    _dev(q, k, v, beta, g, state_in, out, ckpt)
    _require(k.shape == q.shape and v.shape == (N, T, H, dv), "k like q, v [N,T,H,dv]")
    _require(beta.shape == (N, T, H) and g.shape == (N, T, H), "beta, g [N,T,H]")
    _require(beta.dtype == torch.float32 and g.dtype == torch.float32, "beta, g fp32")
    _require(state_in.shape == (N, H, dv, dk) and ckpt.shape == (N, T, H, dv, dk),
             "state_in [N,H,dv,dk], ckpt [N,T,H,dv,dk]")
    _require(out.shape == (N, T, H, dv) and out.dtype == q.dtype and ckpt.dtype == state_in.dtype,
             "out [N,T,H,dv] in q's dtype, ckpt in the state's")
    st = load_library().dn_verify_block(
        N, H, T, dk, dv, _DT[q.dtype], _DT[state_in.dtype], _ptr(q), _ptr(k), _ptr(v),
        _ptr(beta), _ptr(g), _ptr(state_in), _ptr(out), _ptr(ckpt), _stream(stream))
    _check("dn_verify_block", st)
    return out, ckpt


def dn_verify_block_deltas(q, k, v, beta, g, state_in, out=None, delta=None, stream=None):
    """As dn_verify_block, but writes delta [N,T,H,dv] fp32 instead of checkpoints."""
    N, T, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((N, T, H, dv), dtype=q.dtype, device=q.device)
    if delta is None:
        delta = torch.empty((N, T, H, dv), dtype=torch.float32, device=q.device)
    _dev(q, k, v, beta, g, state_in, out, delta)
    _require(k.shape == q.shape and v.shape == (N, T, H, dv) and state_in.shape == (N, H, dv, dk),
             "k like q, v [N,T,H,dv], state_in [N,H,dv,dk]")
    _require(delta.shape == (N, T, H, dv) and delta.dtype == torch.float32, "delta [N,T,H,dv] fp32")
    st = load_library().dn_verify_block_deltas(
        N, H, T, dk, dv, _DT[q.dtype], _DT[state_in.dtype], _ptr(q), _ptr(k), _ptr(v),
        _ptr(beta), _ptr(g), _ptr(state_in), _ptr(out), _ptr(delta), _stream(stream))
    _check("dn_verify_block_deltas", st)
    return out, delta


def dn_commit_deltas(k, g, delta, accepted_len, state, stream=None):
    """Rebuild the accepted state in place from delta [N,T,H,dv], k [N,T,H,dk], g [N,T,H]."""
    N, H, dv, dk = state.shape
    T = k.shape[1]
    B = accepted_len.shape[0]
    _dev(k, g, delta, accepted_len, state)
    _require(k.shape == (N, T, H, dk) and g.shape == (N, T, H) and delta.shape == (N, T, H, dv),
             "k [N,T,H,dk], g [N,T,H], delta [N,T,H,dv]")
    st = load_library().dn_commit_deltas(N, B, H, T, dk, dv, _DT[state.dtype], _ptr(k), _ptr(g),
                                         _ptr(delta), _ptr(accepted_len), _ptr(state),
                                         _stream(stream))
    _check("dn_commit_deltas", st)
    return state


def dn_accept_workspace_bytes(B, T, V):
    return int(load_library().dn_accept_workspace_bytes(B, T, V))


def accept_workspace(B, T, V, device):
    """A zeroed workspace of dn_accept_workspace_bytes(B, T, V) bytes."""
    n = dn_accept_workspace_bytes(B, T, V)
    return torch.zeros((max(n, 16),), dtype=torch.uint8, device=device)


def dn_accept_greedy(logits, draft_ids, target_ids=None, accepted_len=None, workspace=None,
                     stream=None):
    """logits [B,T,V] fp16/fp32, draft_ids [B,T] int32 -> (target_ids [B,T], accepted_len [B])."""
    B, T, V = logits.shape
    dev = logits.device
    if target_ids is None:
        target_ids = torch.empty((B, T), dtype=torch.int32, device=dev)
    if accepted_len is None:
        accepted_len = torch.empty((B,), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = accept_workspace(B, T, V, dev)
    _dev(logits, draft_ids, target_ids, accepted_len, workspace)
    _require(draft_ids.shape == (B, T) and draft_ids.dtype == torch.int32, "draft_ids [B,T] int32")
    _require(target_ids.shape == (B, T) and accepted_len.shape == (B,), "target_ids [B,T], accepted_len [B]")
    st = load_library().dn_accept_greedy(
        B, T, V, _DT[logits.dtype], _ptr(logits), _ptr(draft_ids), _ptr(target_ids),
        _ptr(accepted_len), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check("dn_accept_greedy", st)
    return target_ids, accepted_len


def dn_accept_greedy_noalloc(logits, draft_ids, target_ids, accepted_len, stream=None):
    """dn_accept_greedy with its scratch in the library's fixed device array (no workspace).

    For callers that cannot allocate device memory where they verify; the outputs must
    be passed in. Calls that overlap on one GPU race on the shared array.
    """
    B, T, V = logits.shape
    _dev(logits, draft_ids, target_ids, accepted_len)
    _require(draft_ids.shape == (B, T) and draft_ids.dtype == torch.int32, "draft_ids [B,T] int32")
    _require(target_ids.shape == (B, T) and target_ids.dtype == torch.int32, "target_ids [B,T] int32")
    _require(accepted_len.shape == (B,) and accepted_len.dtype == torch.int32, "accepted_len [B] int32")
    st = load_library().dn_accept_greedy_noalloc(
        B, T, V, _DT[logits.dtype], _ptr(logits), _ptr(draft_ids), _ptr(target_ids),
        _ptr(accepted_len), _stream(stream))
    _check("dn_accept_greedy_noalloc", st)
    return target_ids, accepted_len


def dn_commit(ckpt, accepted_len, state, stream=None):
    """ckpt [N,T,H,dv,dk], accepted_len [B] int32 (device), state [N,H,dv,dk] updated in place."""
    N, H, dv, dk = state.shape
    T = ckpt.shape[1]
    B = accepted_len.shape[0]
    _dev(ckpt, accepted_len, state)
    _require(ckpt.shape == (N, T, H, dv, dk) and ckpt.dtype == state.dtype, "ckpt [N,T,H,dv,dk] in the state's dtype")
    _require(accepted_len.dtype == torch.int32, "accepted_len int32")
    st = load_library().dn_commit(N, B, H, T, dk, dv, _DT[state.dtype], _ptr(ckpt),
                                  _ptr(accepted_len), _ptr(state), _stream(stream))
    _check("dn_commit", st)
    return state


def dn_prefill_checkpoint(q, k, v, beta, g, state_in=None, out=None, ckpt=None, state_out=None,
                          chunk=PREFILL_CHUNK, state_dtype=None, stream=None, engine="mma"):
    """q, k [N,P,H,dk]; v [N,P,H,dv]; beta, g [N,P,H]; state_in [N,H,dv,dk] or None.

    Returns (out [N,P,H,dv], ckpt [N,P//chunk,H,dv,dk], state_out [N,H,dv,dk]).
    engine "mma" calls dn_prefill_checkpoint, "tc" dn_prefill_checkpoint_tc (fp16, 128 x 128).
    """
    N, P, H, dk = q.shape
    dv = v.shape[-1]
    sdt = state_in.dtype if state_in is not None else (state_dtype or q.dtype)
    dev = q.device
    if out is None:
        out = torch.empty((N, P, H, dv), dtype=q.dtype, device=dev)
    if ckpt is None:
        ckpt = torch.empty((N, P // chunk, H, dv, dk), dtype=sdt, device=dev)
    if state_out is None:
        state_out = torch.empty((N, H, dv, dk), dtype=sdt, device=dev)
    _dev(q, k, v, beta, g, state_in, out, ckpt, state_out)
    _require(k.shape == q.shape and v.shape == (N, P, H, dv) and beta.shape == (N, P, H),
             "k like q, v [N,P,H,dv], beta [N,P,H]")
    _require(g.shape == (N, P, H) and out.shape == (N, P, H, dv), "g [N,P,H], out [N,P,H,dv]")
    _require(beta.dtype == torch.float32 and g.dtype == torch.float32, "beta and g are fp32")
    _require(ckpt.shape == (N, P // chunk, H, dv, dk) and state_out.shape == (N, H, dv, dk),
             "ckpt [N,P/chunk,H,dv,dk], state_out [N,H,dv,dk]")
    name = {"mma": "dn_prefill_checkpoint", "tc": "dn_prefill_checkpoint_tc"}[engine]
    st = getattr(load_library(), name)(
        N, H, P, chunk, dk, dv, _DT[q.dtype], _DT[sdt], _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
        _ptr(g), _ptr(state_in), _ptr(out), _ptr(ckpt) if ckpt.numel() else None,
        _ptr(state_out), _stream(stream))
    _check(name, st)
    return out, ckpt, state_out


def dn_prefill_wait_timeouts():
    return int(load_library().dn_prefill_wait_timeouts())


def dn_wait_selftest(budget_us, device=None, stream=None):
    """Runs the bounded-wait self-test; returns (gave_up, returned, drained, failures_counted)."""
    result = torch.tensor([11, 22, 33, 44], dtype=torch.int32, device=device or "cuda")
    _check("dn_wait_selftest", load_library().dn_wait_selftest(int(budget_us), result.data_ptr(), _stream(stream)))
    torch.cuda.synchronize(result.device)
    return tuple(int(x) for x in result.cpu())


def dn_context_drafts(context, lengths, n_max=4, n_min=1, K=8, drafts=None, count=None,
                      match_len=None, stream=None):
    """Drafts copied from each request's context: context [N, stride] int32, lengths [N] int32.

    Returns (drafts [N, K] int32 padded with -1, count [N] int32, match_len [N] int32).
    """
    N, stride = context.shape
    dev = context.device
    if drafts is None:
        drafts = torch.empty((N, K), dtype=torch.int32, device=dev)
    if count is None:
        count = torch.empty((N,), dtype=torch.int32, device=dev)
    if match_len is None:
        match_len = torch.empty((N,), dtype=torch.int32, device=dev)
    _dev(context, lengths, drafts, count, match_len)
    _require(context.dtype == lengths.dtype == drafts.dtype == count.dtype == torch.int32,
             "context, lengths, drafts, count int32")
    _require(lengths.shape == (N,) and drafts.shape == (N, K) and count.shape == (N,),
             "lengths [N], drafts [N,K], count [N]")
    st = load_library().dn_context_drafts(N, stride, n_max, n_min, K, _ptr(context), _ptr(lengths),
                                          _ptr(drafts), _ptr(count), _ptr(match_len),
                                          _stream(stream))
    _check("dn_context_drafts", st)
    return drafts, count, match_len


class PrefixCache:
    """Host-side prefix index of state checkpoints (dn_prefix_cache_* in include/dn.h)."""

    def __init__(self, capacity, chunk=PREFILL_CHUNK):
        self._lib = load_library()
        self._h = self._lib.dn_prefix_cache_create(chunk, capacity)
        if not self._h:
            raise ValueError("dn_prefix_cache_create failed")
        self.chunk = chunk

    @staticmethod
    def _tokens(tokens):
        import numpy as np
        a = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        return a, a.ctypes.data_as(ctypes.c_void_p)

    def insert(self, tokens, position, slot):
        """Record that the state after tokens[:position] is in `slot`; returns an evicted slot or -1."""
        a, p = self._tokens(tokens)
        if position > a.shape[0]:
            raise ValueError("position beyond the tokens")
        ev = ctypes.c_int32(-1)
        _check("dn_prefix_cache_insert",
               self._lib.dn_prefix_cache_insert(self._h, p, int(position), int(slot), ctypes.byref(ev)))
        return ev.value

    def lookup(self, tokens):
        """(position, slot) of the longest cached prefix of `tokens`, (0, -1) if none."""
        a, p = self._tokens(tokens)
        pos, slot = ctypes.c_int(0), ctypes.c_int32(-1)
        _check("dn_prefix_cache_lookup",
               self._lib.dn_prefix_cache_lookup(self._h, p, int(a.shape[0]), ctypes.byref(pos),
                                                ctypes.byref(slot)))
        return pos.value, slot.value

    def __len__(self):
        return int(self._lib.dn_prefix_cache_size(self._h))

    def close(self):
        if self._h:
            self._lib.dn_prefix_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dn_status_string(status):
    return load_library().dn_status_string(int(status)).decode()
