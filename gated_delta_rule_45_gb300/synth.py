"""Seeded synthetic inputs for the KDA recurrence.

This module is shared by the tests, the bench and the oracle harness.  It
holds the input recipe only -- random draws, L2 normalisation of q and k,
sigmoids that map logits into (0, 1) for alpha and beta, rounding to the
storage dtype -- and none of the recurrence's arithmetic.  It imports nothing
from the rest of the package.

Recipe (one ``torch.Generator`` on the CPU, seeded once; draws in this order):

1. varlen only: sequence lengths, integers uniform in [len_lo, len_hi]
2. q ~ N(0, 1)   -- L2-normalised per token and head when ``q_norm``
3. k ~ N(0, 1)   -- always L2-normalised per token and head
4. v ~ N(0, 1)
5. beta  = sigmoid(N(0, 1))          fp32, one per token and head
6. alpha = sigmoid(N(alpha_mu, 1))   fp32, one per token, head and value channel
7. S0 ~ N(0, s0_std^2) fp32, skipped (zeros / None) when s0_std == 0

Normalisation happens in fp32, then q, k, v are rounded (round-to-nearest-even)
to the storage dtype; the rounded values are what every consumer sees.
"""
from __future__ import annotations

import dataclasses

import torch

_DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}


@dataclasses.dataclass(frozen=True)
class PrefillSpec:
    """A packed (varlen) prefill problem.  Fixed length when len_lo == len_hi."""
    num_seqs: int
    len_lo: int
    len_hi: int
    H: int
    d_k: int
    d_v: int
    dtype: str = "bf16"
    chunk: int = 64
    alpha_mu: float = 3.0
    s0_std: float = 0.0
    q_norm: bool = True
    seed: int = 0


@dataclasses.dataclass(frozen=True)
class DecodeSpec:
    """One decode step over B sequences (one token each), state updated in place."""
    B: int
    H: int
    d_k: int
    d_v: int
    dtype: str = "bf16"
    alpha_mu: float = 4.0
    s0_std: float = 0.1
    q_norm: bool = True
    seed: int = 0


# The five workloads: sizes, dtypes and distributions as the configuration list states them.
TINY = PrefillSpec(num_seqs=1, len_lo=64, len_hi=64, H=2, d_k=32, d_v=32, dtype="fp32",
                   chunk=16, alpha_mu=3.0, s0_std=0.0, q_norm=False)
DECODE = DecodeSpec(B=256, H=32, d_k=128, d_v=128, alpha_mu=4.0, s0_std=0.1)
PREFILL = PrefillSpec(num_seqs=8, len_lo=4096, len_hi=4096, H=32, d_k=128, d_v=128,
                      chunk=64, alpha_mu=3.0, s0_std=0.0)
LONG = PrefillSpec(num_seqs=1, len_lo=131072, len_hi=131072, H=32, d_k=128, d_v=128,
                   chunk=64, alpha_mu=5.0, s0_std=0.1)
VARLEN = PrefillSpec(num_seqs=64, len_lo=128, len_hi=8192, H=16, d_k=128, d_v=256,
                     chunk=64, alpha_mu=3.0, s0_std=0.1)
VARLEN_DECODE_STEPS = 32

# Contraction-phase case: 152 independent (sequence, head) chains of 6 chunks,
# ~110 MB of inputs and states, so that back-to-back launches are served from L2.
L2_RESIDENT = PrefillSpec(num_seqs=152, len_lo=384, len_hi=384, H=1, d_k=128, d_v=128,
                          chunk=64, s0_std=0.1)
# The long workload at a quarter of the length (32768 tokens), small enough for
# multi-pass profiler captures of the sequence-axis split's kernels.
LONG_SMALL = PrefillSpec(num_seqs=1, len_lo=32768, len_hi=32768, H=32, d_k=128, d_v=128,
                         chunk=64, alpha_mu=5.0, s0_std=0.1)
WORKLOADS = {"tiny": TINY, "decode": DECODE, "prefill": PREFILL, "long": LONG, "varlen": VARLEN,
             "l2_resident": L2_RESIDENT, "long_small": LONG_SMALL}


def _normal(gen: torch.Generator, shape, mean: float = 0.0, std: float = 1.0) -> torch.Tensor:
    x = torch.empty(shape, dtype=torch.float32, device=gen.device)
    x.normal_(mean=mean, std=std, generator=gen)
    return x


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    """Scale every last-axis vector to unit Euclidean length (fp32)."""
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def _draw_token_inputs(gen, T, H, d_k, d_v, dtype, alpha_mu, q_norm):
    store = _DTYPES[dtype]
    q = _normal(gen, (T, H, d_k))
    if q_norm:
        q = _unit_rows(q)
    q = q.to(store)
    k = _unit_rows(_normal(gen, (T, H, d_k))).to(store)
    v = _normal(gen, (T, H, d_v)).to(store)
    beta = torch.sigmoid(_normal(gen, (T, H)))
    alpha = _normal(gen, (T, H, d_v), mean=alpha_mu)
    torch.sigmoid_(alpha)
    return q, k, v, alpha, beta


def prefill_inputs(spec: PrefillSpec, generator: torch.Generator | None = None,
                   device: str = "cpu") -> dict:
    """Draw a prefill problem (on the CPU unless `device` says otherwise).

    Returns dict(q, k, v, alpha, beta, S0 (None when s0_std == 0), cu_seqlens
    int32 [N+1], lengths list, spec, generator).  The generator is returned so
    that follow-up draws (decode steps) continue the same stream.  The same
    recipe on another device draws other numbers from the same distributions
    (the oracle comparisons use the CPU draws; timing alone may draw on the
    GPU, which is much faster at full size).
    """
    gen = generator or torch.Generator(device=device).manual_seed(spec.seed)
    if spec.len_lo == spec.len_hi:
        lengths = [spec.len_lo] * spec.num_seqs
    else:
        lengths = torch.randint(spec.len_lo, spec.len_hi + 1, (spec.num_seqs,),
                                generator=gen, device=gen.device).tolist()
    cu = torch.zeros(spec.num_seqs + 1, dtype=torch.int32, device=gen.device)
    if spec.num_seqs:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu[-1])
    q, k, v, alpha, beta = _draw_token_inputs(gen, T, spec.H, spec.d_k, spec.d_v, spec.dtype,
                                              spec.alpha_mu, spec.q_norm)
    S0 = None
    if spec.s0_std > 0:
        S0 = _normal(gen, (spec.num_seqs, spec.H, spec.d_v, spec.d_k), std=spec.s0_std)
    return dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0, cu_seqlens=cu,
                lengths=lengths, spec=spec, generator=gen)


def backward_cotangents(d: dict, dS_T_std: float = 0.1) -> tuple:
    """Draw the incoming gradients of a backward pass for the prefill problem `d`
    (continuing its generator): dL/do ~ N(0, 1) in the storage dtype, and dL/dS_T
    ~ N(0, dS_T_std^2) fp32, or None when dS_T_std == 0."""
    spec, gen = d["spec"], d["generator"]
    T = int(d["cu_seqlens"][-1])
    dO = _normal(gen, (T, spec.H, spec.d_v)).to(_DTYPES[spec.dtype])
    dS_T = None
    if dS_T_std > 0:
        dS_T = _normal(gen, (spec.num_seqs, spec.H, spec.d_v, spec.d_k), std=dS_T_std)
    return dO, dS_T


@dataclasses.dataclass(frozen=True)
class AttnResSpec:
    """A network of Blocked Attention Residuals: T tokens of width d, layers in
    blocks of the given sizes (the network input is block 0)."""
    T: int
    d: int
    block_sizes: tuple
    dtype: str = "bf16"
    seed: int = 0


# 64 layers in 8 blocks of 8 (blocks of sqrt(L) layers), 16384 tokens of width 2048
ATTNRES = AttnResSpec(T=16384, d=2048, block_sizes=(8,) * 8)


def attnres_inputs(spec: AttnResSpec, device="cpu") -> dict:
    """Draw a network's inputs: h0 [T, d] and every layer's output [L, T, d]
    ~ N(0, 1) in the storage dtype (stand-ins for the layers, which are outside
    the library), queries [L, d] ~ N(0, 1) fp32."""
    gen = torch.Generator(device=device).manual_seed(spec.seed)
    L = sum(spec.block_sizes)
    store = _DTYPES[spec.dtype]
    def normal(shape):
        x = torch.empty(shape, dtype=torch.float32, device=device)
        x.normal_(generator=gen)
        return x
    h0 = normal((spec.T, spec.d)).to(store)
    outs = normal((L, spec.T, spec.d)).to(store)
    queries = normal((L, spec.d))
    return dict(h0=h0, outs=outs, queries=queries, spec=spec)


def decode_inputs(spec: DecodeSpec, generator: torch.Generator | None = None,
                  with_state: bool = True, device: str = "cpu") -> dict:
    """Draw one decode step (on the CPU unless `device` says otherwise):
    q, k [B,H,d_k]; v, alpha [B,H,d_v]; beta [B,H]; S."""
    gen = generator or torch.Generator(device=device).manual_seed(spec.seed)
    q, k, v, alpha, beta = _draw_token_inputs(gen, spec.B, spec.H, spec.d_k, spec.d_v,
                                              spec.dtype, spec.alpha_mu, spec.q_norm)
    S = None
    if with_state:
        S = _normal(gen, (spec.B, spec.H, spec.d_v, spec.d_k), std=spec.s0_std)
    return dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S=S, spec=spec, generator=gen)


def decode_sequence_inputs(steps: int, B: int, H: int, d_k: int, d_v: int, dtype: str,
                           alpha_mu: float, generator: torch.Generator,
                           q_norm: bool = True) -> list[dict]:
    """Per-step token inputs for `steps` decode steps that continue a prefill."""
    out = []
    for _ in range(steps):
        q, k, v, alpha, beta = _draw_token_inputs(generator, B, H, d_k, d_v, dtype, alpha_mu,
                                                  q_norm)
        out.append(dict(q=q, k=k, v=v, alpha=alpha, beta=beta))
    return out


def bf16_bits(x: torch.Tensor):
    """numpy uint16 view of a bf16 tensor's bit patterns (or float32 numpy for fp32)."""
    if x.dtype == torch.bfloat16:
        return x.contiguous().view(torch.int16).numpy().view("uint16")
    return x.contiguous().numpy()
