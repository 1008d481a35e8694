"""The steps of the cross-process sequence split taken by the oracle (fp64,
CPU), so that the exchange and the scan of gated_delta_rule_45_gb300.seqpar
can be checked on CPU ranks: prefill is the oracle's recurrence, combine is
diag(g) S P + R written out in numpy."""
import numpy as np
import torch

import oracle
from gated_delta_rule_45_gb300 import synth


def _np(x):
    return synth.bf16_bits(x) if x.dtype == torch.bfloat16 else x.double().numpy()


class OracleBackend:
    def prefill(self, q, k, v, alpha, beta, S0, cu_seqlens):
        s0 = None if S0 is None else S0.double().numpy()
        o, S_T = oracle.prefill(_np(q), _np(k), _np(v), alpha.float().numpy(),
                                beta.float().numpy(), s0, cu_seqlens.numpy().astype(np.int32),
                                nthreads=1)
        return torch.from_numpy(o), torch.from_numpy(S_T)

    def combine(self, S, g, P, R):
        S, g, P, R = (x.double().numpy() for x in (S, g, P, R))
        return torch.from_numpy(g[..., None] * np.einsum("nhvk,nhkl->nhvl", S, P) + R)


def split_batch(d, world):
    """Cut every sequence of the problem d into `world` contiguous segments of
    near-equal length; returns each rank's (q, k, v, alpha, beta, cu_seqlens)."""
    cu = d["cu_seqlens"].numpy()
    N = len(cu) - 1
    out = []
    for r in range(world):
        idx, lens = [], []
        for n in range(N):
            a, b = int(cu[n]), int(cu[n + 1])
            L = b - a
            s0, s1 = a + r * L // world, a + (r + 1) * L // world
            idx.extend(range(s0, s1))
            lens.append(s1 - s0)
        idx = torch.tensor(idx, dtype=torch.long)
        cur = torch.zeros(N + 1, dtype=torch.int32)
        cur[1:] = torch.cumsum(torch.tensor(lens), 0).to(torch.int32)
        out.append({key: d[key][idx].contiguous() for key in ("q", "k", "v", "alpha", "beta")}
                   | {"cu_seqlens": cur, "idx": idx})
    return out
