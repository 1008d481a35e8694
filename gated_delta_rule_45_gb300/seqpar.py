"""The sequence axis split across processes (one GPU each): every rank holds
one contiguous segment of the same batch of sequences.

Over a segment the recurrence is affine in the state it starts from ("Kimi
(AI)", section "Kimi Delta Attention (KDA)": forget gating and memory updating
composed over the segment's tokens):

    S_end = diag(g) S_start P + R

with g the product of alpha over the segment (per value channel), P the
product of its (I - beta_t k_t k_t^T) factors and R the state it reaches from
zero.  Each rank

1. computes its segment's map (g, P, R) with three prefills of special inputs
   (R: S0 = 0; P: v = 0, alpha = 1, S0 = I; g: k = 0, S0 = all ones);
2. gathers every rank's map (one all-gather per part, the only exchange);
3. scans the maps of the ranks before it, from the batch's S0 (rank 0's), into
   its own initial state: S_{r+1} = diag(g_r) S_r P_r + R_r;
4. prefills its segment from that state: its o is final, and the last rank's
   final state is the batch's S_T, broadcast to every rank.

Every step of the arithmetic runs in the library's kernels (``kda.prefill``,
``kda.segment_combine``); this module only arranges the calls and the
exchange.  The steps are taken through a ``backend`` object so that the
exchange and the scan can be checked on CPU ranks against a reference.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


class LibraryBackend:
    """The segment steps on the GPU, through libkda."""

    def __init__(self, chunk: int = 64, kernel: str = "auto"):
        from gated_delta_rule_45_gb300 import kda
        self.kda = kda
        self.chunk = chunk
        self.kernel = kernel

    def prefill(self, q, k, v, alpha, beta, S0, cu_seqlens):
        return self.kda.prefill(q, k, v, alpha, beta, S0, cu_seqlens, chunk=self.chunk,
                                kernel=self.kernel, check_device_status=True)

    def combine(self, S, g, P, R):
        return self.kda.segment_combine(S, g, P, R)


def segment_map(backend, q, k, v, alpha, beta, cu_seqlens):
    """(g [N, H, d_v], P [N, H, d_k, d_k], R [N, H, d_v, d_k]) of this rank's
    segment, from three prefills of special inputs."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    dev = q.device
    # R: the state reached from zero
    _, R = backend.prefill(q, k, v, alpha, beta, None, cu_seqlens)
    # P: the state reached from the identity with no decay and no values
    eye = torch.eye(d_k, device=dev, dtype=torch.float32).expand(N, H, d_k, d_k).contiguous()
    _, P = backend.prefill(q, k, torch.zeros(T, H, d_k, dtype=v.dtype, device=dev),
                           torch.ones(T, H, d_k, dtype=torch.float32, device=dev), beta, eye,
                           cu_seqlens)
    # g: with k = 0 the state only decays, so all ones become prod alpha
    dk_g = 16
    zq = torch.zeros(T, H, dk_g, dtype=q.dtype, device=dev)
    ones = torch.ones(N, H, d_v, dk_g, dtype=torch.float32, device=dev)
    _, G = backend.prefill(zq, zq, torch.zeros_like(v), alpha, beta, ones, cu_seqlens)
    g = G[..., 0].contiguous()
    return g, P, R


def prefill_sequence_parallel(q, k, v, alpha, beta, S0, cu_seqlens, *, group=None,
                              backend=None):
    """Prefill this rank's segment of every sequence with the state the
    segments before it leave, exchanged as affine maps.

    q, k, v, alpha, beta, cu_seqlens: this rank's tokens (rank r holds the
    r-th contiguous segment of each of the N sequences; a segment may be
    empty).  S0 [N, H, d_v, d_k] fp32: the batch's initial state, read on
    rank 0 (None: zeros).  Returns (o of this segment, S_T of the batch).
    """
    backend = backend or LibraryBackend()
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    dev = q.device

    g, P, R = segment_map(backend, q, k, v, alpha, beta, cu_seqlens)
    parts = []
    for x in (g, P, R):
        bufs = [torch.empty_like(x) for _ in range(world)]
        dist.all_gather(bufs, x.contiguous(), group=group)
        parts.append(bufs)
    gs, Ps, Rs = parts

    # the batch's initial state, from rank 0
    S = S0.contiguous() if (rank == 0 and S0 is not None) else \
        torch.zeros(N, H, d_v, d_k, dtype=torch.float32, device=dev)
    dist.broadcast(S, src=dist.get_global_rank(group, 0) if group is not None else 0, group=group)
    for j in range(rank):   # the segments before this one, in order
        S = backend.combine(S, gs[j], Ps[j], Rs[j])

    o, S_end = backend.prefill(q, k, v, alpha, beta, S, cu_seqlens)
    last = world - 1
    S_T = S_end.contiguous() if rank == last else torch.empty_like(S_end)
    dist.broadcast(S_T, src=dist.get_global_rank(group, last) if group is not None else last,
                   group=group)
    return o, S_T
