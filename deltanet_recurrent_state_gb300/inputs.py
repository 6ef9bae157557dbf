"""Seeded synthetic inputs for the DeltaNet verify / accept / commit / prefill path.

This module is shared by the tests (which feed the same tensors to the CPU
oracle and to the CUDA path), by ``bench.py`` and by ``smoke()``. It holds none
of the method's arithmetic: it only draws random tensors with the stated
distributions and plants known answers (the argmax position and the accepted
length) by construction, so that no expected value has to be computed to build
an input.

Recipe (every draw from one ``torch.Generator`` seeded per workload):

* q, k ~ N(0, 1), each head vector L2-normalised in fp32, then cast to the io dtype;
* v ~ N(0, 1);  beta = sigmoid(N(0, 1));  g = exp(-softplus(N(0, 1)))  (fp32);
* initial state ~ N(0, 0.1^2) (standard deviation 0.1), cast to the state dtype;
* logits ~ N(0, std^2), clipped to +-6 std, with one planted entry of value
  8 std per row at a uniformly drawn target id, so the row's unique maximum is
  known without computing it. The clip is 6 standard deviations; the chance
  that a 151,936-wide row holds any clipped entry is about 3e-4;
* draft ids equal the planted target for the first ``a`` positions, a different
  uniformly drawn id at position ``a`` (when a < T), uniform ids after it.
"""

import math

import torch

_CHUNK_SETS = 256  # state sets generated per batch, bounds fp32 temporaries


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _dt(name):
    return {"f16": torch.float16, "f32": torch.float32}[name]


def _unit(x):
    return x / x.norm(dim=-1, keepdim=True)


def recurrence_inputs(N, T, H, dk, dv, io="f16", state="f16", seed=0, device="cpu",
                      s0_std=0.1, with_state=True):
    """q, k [N, T, H, dk]; v [N, T, H, dv]; beta, g [N, T, H] fp32; state [N, H, dv, dk].

    T is the verify-block width, or the prompt length P for prefill inputs.
    Returns a dict of tensors on ``device``.
    """
    gen = _gen(seed, device)
    iot, st = _dt(io), _dt(state)
    q = torch.empty((N, T, H, dk), dtype=iot, device=device)
    k = torch.empty((N, T, H, dk), dtype=iot, device=device)
    v = torch.empty((N, T, H, dv), dtype=iot, device=device)
    beta = torch.empty((N, T, H), dtype=torch.float32, device=device)
    g = torch.empty((N, T, H), dtype=torch.float32, device=device)
    s0 = torch.empty((N, H, dv, dk), dtype=st, device=device) if with_state else None
    for n0 in range(0, N, _CHUNK_SETS):
        n1 = min(N, n0 + _CHUNK_SETS)
        m = n1 - n0
        f32 = dict(dtype=torch.float32, device=device, generator=gen)
        q[n0:n1] = _unit(torch.randn((m, T, H, dk), **f32)).to(iot)
        k[n0:n1] = _unit(torch.randn((m, T, H, dk), **f32)).to(iot)
        v[n0:n1] = torch.randn((m, T, H, dv), **f32).to(iot)
        beta[n0:n1] = torch.sigmoid(torch.randn((m, T, H), **f32))
        g[n0:n1] = torch.exp(-torch.nn.functional.softplus(torch.randn((m, T, H), **f32)))
        if with_state:
            s0[n0:n1] = (s0_std * torch.randn((m, H, dv, dk), **f32)).to(st)
    return dict(q=q, k=k, v=v, beta=beta, g=g, state=s0)


def accepted_lengths(B, T, kind, seed=0, value=None, p=0.2):
    """Planted accepted lengths [B] int32 (CPU).

    kind: "uniform" -> U{0..T}; "fixed" -> ``value``; "geometric" -> geometric on
    {0, 1, ...} with success probability p (untruncated mean (1-p)/p = 4 at
    p = 0.2), clamped at T.
    """
    gen = _gen(seed, "cpu")
    if kind == "uniform":
        return torch.randint(0, T + 1, (B,), generator=gen, dtype=torch.int32)
    if kind == "fixed":
        assert value is not None and 0 <= value <= T
        return torch.full((B,), int(value), dtype=torch.int32)
    if kind == "geometric":
        u = torch.rand((B,), generator=gen, dtype=torch.float64).clamp_min(1e-300)
        a = torch.floor(torch.log(u) / math.log(1.0 - p))
        return a.clamp(max=T).to(torch.int32)
    raise ValueError(kind)


def logits_inputs(B, T, V, dtype="f16", std=2.0, seed=0, device="cpu"):
    """logits [B, T, V] with a planted unique maximum; returns (logits, target [B, T] int32)."""
    gen = _gen(seed, device)
    lt = _dt(dtype)
    logits = torch.empty((B, T, V), dtype=lt, device=device)
    for b in range(B):
        x = torch.randn((T, V), dtype=torch.float32, device=device, generator=gen) * std
        logits[b] = x.clamp(-6.0 * std, 6.0 * std).to(lt)
    target = torch.randint(0, V, (B, T), generator=gen, device=device, dtype=torch.int64)
    logits.scatter_(2, target[:, :, None], torch.full((B, T, 1), 8.0 * std, dtype=lt, device=device))
    return logits, target.to(torch.int32)


def draft_ids(target, accepted, V, seed=0):
    """Draft ids [B, T] int32 whose matching prefix against ``target`` is exactly ``accepted``.

    target [B, T] int32 (any device), accepted [B] int32 (CPU). Returned on target's device.
    """
    gen = _gen(seed, "cpu")
    tgt = target.detach().to("cpu", torch.int64)
    B, T = tgt.shape
    d = torch.randint(0, V, (B, T), generator=gen, dtype=torch.int64)
    for b in range(B):
        a = int(accepted[b])
        d[b, :a] = tgt[b, :a]
        if a < T:
            assert V > 1, "a rejected position needs a vocabulary of at least 2"
            off = int(torch.randint(1, V, (1,), generator=gen))
            d[b, a] = (tgt[b, a] + off) % V
    return d.to(torch.int32).to(target.device)


def context_inputs(N, prompt_len, gen_len, vocab, quote=True, ragged=False, seed=0, device="cpu"):
    """Token contexts for drafting from the request's own context.

    Each row is a prompt of ``prompt_len`` tokens followed by ``gen_len`` generated
    tokens. Prompt tokens are log-uniform over the vocabulary (P(t) proportional to
    1/(t+1), a Zipf-like spread, so short repeats are common). With ``quote`` the
    generated tokens are a verbatim copy of a uniformly placed passage of the prompt
    (the document-reproduction case); otherwise they are fresh log-uniform tokens.
    ``ragged`` draws each row's length uniformly from 0..prompt_len+gen_len; otherwise
    every row is full. Returns (context [N, prompt_len + gen_len] int32, lengths [N] int32).
    """
    g = _gen(seed, "cpu")
    Lmax = prompt_len + gen_len

    def loguniform(shape):
        u = torch.rand(shape, generator=g, dtype=torch.float64)
        return (torch.exp(u * math.log(vocab + 1)).floor() - 1).clamp_(0, vocab - 1).to(torch.int32)

    prompt = loguniform((N, prompt_len))
    if quote and gen_len > 0:
        if gen_len > prompt_len:
            raise ValueError("a quoted passage cannot be longer than the prompt")
        start = torch.randint(0, prompt_len - gen_len + 1, (N, 1), generator=g)
        gen = torch.gather(prompt, 1, start + torch.arange(gen_len)[None, :])
    else:
        gen = loguniform((N, gen_len))
    ctx = torch.cat([prompt, gen], dim=1).contiguous()
    if ragged:
        lengths = torch.randint(0, Lmax + 1, (N,), generator=g, dtype=torch.int32)
    else:
        lengths = torch.full((N,), Lmax, dtype=torch.int32)
    return ctx.to(device), lengths.to(device)
