"""The C ABI: libdn.so loads, exports every symbol include/dn.h declares, and
rejects malformed arguments on the host before anything is enqueued (no GPU).

Invalid-argument cases pass buffers that are real device allocations when a GPU
is present (so nothing could touch a bad address even if a check were missing)
and aligned placeholder addresses otherwise; each case carries exactly one defect.
"""

import ctypes
import os
import re

import pytest
import torch

from deltanet_recurrent_state_gb300 import binding
from deltanet_recurrent_state_gb300 import build as dnbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dn.h")

OK, INVALID, UNSUPPORTED = binding.DN_OK, binding.DN_ERR_INVALID_ARG, binding.DN_ERR_UNSUPPORTED
F16, F32 = binding.DN_F16, binding.DN_F32


@pytest.fixture(scope="module")
def lib():
    dnbuild.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_four_operations():
    names = declared_functions()
    for n in ("dn_verify_block", "dn_accept_greedy", "dn_commit", "dn_prefill_checkpoint",
              "dn_accept_workspace_bytes", "dn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(binding.SIGNATURES)


def test_status_strings(lib):
    for s in range(4):
        assert lib.dn_status_string(s).decode().startswith(
            ["DN_OK", "DN_ERR_INVALID_ARG", "DN_ERR_UNSUPPORTED", "DN_ERR_CUDA"][s])
    assert b"unknown" in lib.dn_status_string(99)


def test_workspace_size(lib):
    assert lib.dn_accept_workspace_bytes(0, 4, 10) == 0
    assert lib.dn_accept_workspace_bytes(1, 0, 10) == 0
    n1 = lib.dn_accept_workspace_bytes(1, 16, 151936)
    n2 = lib.dn_accept_workspace_bytes(64, 4, 151936)
    assert n1 > 0 and n2 > n1 and n1 % 16 == 0
    # one 8-byte key per (row, 8192-entry chunk) plus two counter arrays
    assert n1 >= 16 * 19 * 8


class Bufs:
    """Addresses for argument checks: device allocations when CUDA exists."""

    def __init__(self):
        self.keep = []

    def __call__(self, nbytes=4096, offset=0):
        if torch.cuda.is_available():
            t = torch.zeros(nbytes + 64, dtype=torch.uint8, device="cuda")
            self.keep.append(t)
            return t.data_ptr() + offset
        return 0x100000 + 0x10000 * len(self.keep.append(None) or self.keep) + offset


def _verify_args(buf, **over):
    a = dict(N=1, H=1, T=2, dk=64, dv=64, io=F32, st=F32, q=buf(), k=buf(), v=buf(), beta=buf(),
             g=buf(), s=buf(64 * 64 * 4), out=buf(), ckpt=buf(2 * 64 * 64 * 4))
    a.update(over)
    return (a["N"], a["H"], a["T"], a["dk"], a["dv"], a["io"], a["st"], a["q"], a["k"], a["v"],
            a["beta"], a["g"], a["s"], a["out"], a["ckpt"], None)


@pytest.mark.parametrize("over,want", [
    (dict(T=0), INVALID), (dict(T=17), INVALID), (dict(N=-1), INVALID), (dict(H=0), INVALID),
    (dict(dk=96), UNSUPPORTED), (dict(dv=32), UNSUPPORTED), (dict(io=F16), UNSUPPORTED),
    (dict(io=7), INVALID), (dict(q=None), INVALID), (dict(ckpt=None), INVALID),
    (dict(beta=None), INVALID), ("misaligned_q", INVALID), ("misaligned_beta", INVALID),
])
def test_verify_rejects(lib, over, want):
    buf = Bufs()
    if over == "misaligned_q":
        over = dict(q=buf(offset=8))
    elif over == "misaligned_beta":
        over = dict(beta=buf(offset=2))
    assert lib.dn_verify_block(*_verify_args(buf, **over)) == want


def test_verify_empty_is_ok(lib):
    buf = Bufs()
    assert lib.dn_verify_block(*_verify_args(buf, N=0)) == OK


def _accept_args(buf, **over):
    a = dict(B=1, T=4, V=100, dt=F32, logits=buf(), draft=buf(), tgt=buf(), acc=buf(), ws=buf(),
             wsb=4096)
    a.update(over)
    return (a["B"], a["T"], a["V"], a["dt"], a["logits"], a["draft"], a["tgt"], a["acc"], a["ws"],
            a["wsb"], None)


@pytest.mark.parametrize("over", [
    dict(T=0), dict(V=0), dict(B=-1), dict(dt=5), dict(logits=None), dict(ws=None), dict(wsb=8),
    dict(B=300_000_000, T=8, V=151936), "misaligned_logits", "misaligned_draft",
])
def test_accept_rejects(lib, over):
    buf = Bufs()
    if over == "misaligned_logits":
        over = dict(logits=buf(offset=4))
    elif over == "misaligned_draft":
        over = dict(draft=buf(offset=2))
    assert lib.dn_accept_greedy(*_accept_args(buf, **over)) == INVALID


def _commit_args(buf, **over):
    a = dict(N=2, B=1, H=1, T=2, dk=64, dv=64, st=F16, ckpt=buf(4 * 64 * 64 * 2), acc=buf(),
             s=buf(2 * 64 * 64 * 2))
    a.update(over)
    return (a["N"], a["B"], a["H"], a["T"], a["dk"], a["dv"], a["st"], a["ckpt"], a["acc"], a["s"],
            None)


@pytest.mark.parametrize("over,want", [
    (dict(B=0), INVALID), (dict(N=3, B=2), INVALID), (dict(T=17), INVALID),
    (dict(dk=100), UNSUPPORTED), (dict(s=None), INVALID), (dict(acc=None), INVALID),
    ("misaligned_state", INVALID), (dict(N=50_000_000, B=1, H=48, dk=128, dv=128), INVALID),
])
def test_commit_rejects(lib, over, want):
    buf = Bufs()
    if over == "misaligned_state":
        over = dict(s=buf(offset=8))
    assert lib.dn_commit(*_commit_args(buf, **over)) == want


def _commit_deltas_args(buf, **over):
    a = dict(N=2, B=1, H=1, T=2, dk=64, dv=64, st=F16, k=buf(2 * 2 * 64 * 2), g=buf(),
             delta=buf(2 * 2 * 64 * 4), acc=buf(), s=buf(2 * 64 * 64 * 2))
    a.update(over)
    return (a["N"], a["B"], a["H"], a["T"], a["dk"], a["dv"], a["st"], a["k"], a["g"], a["delta"], a["acc"],
            a["s"], None)


@pytest.mark.parametrize("over,want", [
    (dict(B=0), INVALID), (dict(N=3, B=2), INVALID), (dict(T=17), INVALID), (dict(st=F32), UNSUPPORTED),
    (dict(dk=100), UNSUPPORTED), (dict(delta=None), INVALID), (dict(k=None), INVALID),
    ("misaligned_delta", INVALID), ("misaligned_state", INVALID),
])
def test_commit_deltas_rejects(lib, over, want):
    buf = Bufs()
    if over == "misaligned_delta":  # the deltas go in by 16-byte copies
        over = dict(delta=buf(offset=4))
    elif over == "misaligned_state":
        over = dict(s=buf(offset=8))
    assert lib.dn_commit_deltas(*_commit_deltas_args(buf, **over)) == want


def _prefill_args(buf, **over):
    a = dict(N=1, H=1, P=70, chunk=64, dk=64, dv=64, io=F32, st=F32, q=buf(70 * 256),
             k=buf(70 * 256), v=buf(70 * 256), beta=buf(), g=buf(), s_in=None, out=buf(70 * 256),
             ckpt=buf(64 * 64 * 4), s_out=buf(64 * 64 * 4))
    a.update(over)
    return (a["N"], a["H"], a["P"], a["chunk"], a["dk"], a["dv"], a["io"], a["st"], a["q"], a["k"],
            a["v"], a["beta"], a["g"], a["s_in"], a["out"], a["ckpt"], a["s_out"], None)


@pytest.mark.parametrize("over,want", [
    (dict(chunk=32), UNSUPPORTED), (dict(P=-1), INVALID), (dict(H=0), INVALID),
    (dict(ckpt=None), INVALID), (dict(s_out=None), INVALID), (dict(q=None), INVALID),
    (dict(dk=256), UNSUPPORTED), (dict(st=F16), UNSUPPORTED), ("misaligned_out", INVALID),
])
def test_prefill_rejects(lib, over, want):
    buf = Bufs()
    if over == "misaligned_out":
        over = dict(out=buf(offset=4))
    assert lib.dn_prefill_checkpoint(*_prefill_args(buf, **over)) == want


def test_binding_raises_dnerror_on_bad_status(lib):
    with pytest.raises(binding.DnError) as e:
        binding._check("dn_verify_block", INVALID)
    assert "DN_ERR_INVALID_ARG" in str(e.value)


def test_binding_refuses_missing_library(tmp_path):
    with pytest.raises(RuntimeError):
        binding.load_library(str(tmp_path / "missing.so"))


def _context_args(buf, **over):
    a = dict(N=2, stride=100, n_max=4, n_min=1, K=8, ctx=buf(800), lens=buf(), drafts=buf(64),
             count=buf(), match=None)
    a.update(over)
    return (a["N"], a["stride"], a["n_max"], a["n_min"], a["K"], a["ctx"], a["lens"], a["drafts"],
            a["count"], a["match"], None)


@pytest.mark.parametrize("over", [
    dict(N=-1), dict(stride=-1), dict(stride=1 << 27), dict(n_min=0), dict(n_min=5),
    dict(n_max=17, n_min=1), dict(K=0), dict(K=17), dict(ctx=None), dict(lens=None),
    dict(drafts=None), dict(count=None), "misaligned_ctx", "misaligned_match",
])
def test_context_drafts_rejects(lib, over):
    buf = Bufs()
    if over == "misaligned_ctx":
        over = dict(ctx=buf(offset=2))
    elif over == "misaligned_match":
        over = dict(match=buf(offset=1))
    assert lib.dn_context_drafts(*_context_args(buf, **over)) == INVALID


def test_context_drafts_empty_is_ok(lib):
    buf = Bufs()
    assert lib.dn_context_drafts(*_context_args(buf, N=0, ctx=None, lens=None, drafts=None,
                                                count=None)) == OK


@pytest.mark.parametrize("over,want", [
    (dict(dk=64), UNSUPPORTED), (dict(io=F32, st=F32), UNSUPPORTED), (dict(P=-1), INVALID),
    (dict(s_out=None), INVALID), ("misaligned_out", INVALID),
])
def test_prefill_tc_rejects(lib, over, want):
    buf = Bufs()
    base = dict(dk=128, dv=128, io=F16, st=F16, q=buf(70 * 256), k=buf(70 * 256), v=buf(70 * 256),
                out=buf(70 * 256), ckpt=buf(128 * 128 * 2), s_out=buf(128 * 128 * 2))
    if over == "misaligned_out":
        over = dict(out=buf(offset=4))
    base.update(over)
    assert lib.dn_prefill_checkpoint_tc(*_prefill_args(buf, **base)) == want


def test_package_exports_every_binding_entry_point():
    # every name the package advertises resolves, and every public binding function is advertised
    import inspect
    import deltanet_recurrent_state_gb300 as pkg
    from deltanet_recurrent_state_gb300 import binding
    for name in pkg._API:
        assert getattr(pkg, name) is getattr(binding, name), name
    public = {n for n, f in vars(binding).items()
              if (inspect.isfunction(f) or inspect.isclass(f)) and not n.startswith("_")
              and f.__module__ == binding.__name__}
    assert public <= set(pkg._API), public - set(pkg._API)
