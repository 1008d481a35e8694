"""kda_backward against the oracle's reverse mode (GPU).

Every gradient (dq, dk, dv, dalpha, dbeta, dS0) is compared slice by slice,
one slice per (sequence, head), with the relative Frobenius error
||g - g_ref|| / ||g_ref|| against the fp64 oracle on the same bf16 inputs.
Gate: 2e-3, the bar the forward pass is held to; the kernel computes in fp32,
so the measured errors sit orders of magnitude below it.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from gated_delta_rule_45_gb300 import kda, synth

pytestmark = pytest.mark.gpu

TOL = 2e-3
NAMES = ("dq", "dk", "dv", "dalpha", "dbeta", "dS0")


def _oracle(d, dO, dS_T, pairs):
    """Oracle gradients for the listed (n, h) pairs, each run as its own sequence."""
    cu = d["cu_seqlens"].numpy()
    S0 = None if d["S0"] is None else d["S0"].double().numpy()
    sl = lambda x, a, b, h: x[a:b, h:h + 1]
    parts = {key: [] for key in ("q", "k", "v", "alpha", "beta", "dO")}
    s0s, dsts, lens = [], [], []
    for n, h in pairs:
        a, b = int(cu[n]), int(cu[n + 1])
        for key in ("q", "k", "v", "alpha", "beta"):
            parts[key].append(sl(d[key], a, b, h))
        parts["dO"].append(sl(dO, a, b, h))
        lens.append(b - a)
        s0s.append(np.zeros((d["spec"].d_v, d["spec"].d_k)) if S0 is None else S0[n, h])
        dsts.append(np.zeros_like(s0s[-1]) if dS_T is None else dS_T[n, h].double().numpy())
    cat = lambda key: torch.cat(parts[key])
    pcu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    g = oracle.backward(synth.bf16_bits(cat("q")), synth.bf16_bits(cat("k")),
                        synth.bf16_bits(cat("v")), cat("alpha").numpy(), cat("beta").numpy(),
                        np.stack(s0s)[:, None], pcu, cat("dO").double().numpy(),
                        np.stack(dsts)[:, None])
    out = {}
    for i, (n, h) in enumerate(pairs):
        a, b = pcu[i], pcu[i + 1]
        out[(n, h)] = {name: (g[name][a:b, 0] if name != "dS0" else g[name][i, 0])
                       for name in NAMES}
    return out


def _compare(d, got, ref):
    cu = d["cu_seqlens"].numpy()
    worst = {name: 0.0 for name in NAMES}
    cpu = {name: got[name].cpu().numpy() for name in NAMES if got.get(name) is not None}
    for (n, h), r in ref.items():
        a, b = int(cu[n]), int(cu[n + 1])
        for name in cpu:
            x = cpu[name][n, h] if name == "dS0" else cpu[name][a:b, h]
            if name != "dS0" and b == a:
                continue
            worst[name] = max(worst[name], parity.rel(x, r[name]))
    return worst


def _run(spec, dS_T_std=0.1, pairs=None, extra_tokens=0):
    d = synth.prefill_inputs(spec)
    dO, dS_T = synth.backward_cotangents(d, dS_T_std)
    dev = parity.to_device(d)
    T = dO.shape[0]
    q, k, v, al, be = (dev[x] for x in ("q", "k", "v", "alpha", "beta"))
    dO_dev = dO.cuda()
    if extra_tokens:   # tokens past the last sequence: not read, gradients not written
        pad = lambda x: torch.cat([x, torch.ones_like(x[:extra_tokens])])
        q, k, v, al, be, dO_dev = (pad(x) for x in (q, k, v, al, be, dO_dev))
    g = kda.backward(q, k, v, al, be, dev["S0"], dev["cu_seqlens"], dO_dev,
                     None if dS_T is None else dS_T.cuda(), check_device_status=True)
    torch.cuda.synchronize()
    if extra_tokens:
        for name in ("dq", "dk", "dv", "dalpha", "dbeta"):
            assert torch.count_nonzero(g[name][T:]) == 0, name
    if pairs is None:
        pairs = [(n, h) for n in range(spec.num_seqs) for h in range(spec.H)]
    ref = _oracle(d, dO, dS_T, pairs)
    worst = _compare(d, g, ref)
    assert all(e <= TOL for e in worst.values()), worst
    return g, worst


CASES = [
    # ragged lengths, several chunks, nonzero S0 and dS_T
    synth.PrefillSpec(num_seqs=4, len_lo=1, len_hi=400, H=2, d_k=128, d_v=128, s0_std=0.1,
                      seed=11),
    # d_v = 256: four row blocks summed for dq, dk, dbeta
    synth.PrefillSpec(num_seqs=3, len_lo=60, len_hi=300, H=2, d_k=128, d_v=256, s0_std=0.1,
                      seed=12),
    # d_v = 64: one row block; whole chunks only; zero S0
    synth.PrefillSpec(num_seqs=3, len_lo=128, len_hi=128, H=3, d_k=128, d_v=64, s0_std=0.0,
                      seed=13),
    # long memory (alpha near 1) and unnormalised q
    synth.PrefillSpec(num_seqs=2, len_lo=200, len_hi=330, H=2, d_k=128, d_v=128, alpha_mu=5.0,
                      s0_std=0.1, q_norm=False, seed=14),
    # fast decay: products of alpha over a chunk down to ~1e-12
    synth.PrefillSpec(num_seqs=2, len_lo=150, len_hi=200, H=2, d_k=128, d_v=128, alpha_mu=1.0,
                      s0_std=0.1, seed=15),
    # d_v = 192: three row blocks, and the kernel's own forward sweep (no
    # tensor-core checkpoints for a width that is not a multiple of 128)
    synth.PrefillSpec(num_seqs=3, len_lo=30, len_hi=220, H=2, d_k=128, d_v=192, s0_std=0.1,
                      seed=22),
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_backward_matches_oracle(idx):
    _run(CASES[idx])


def test_backward_without_state_gradient_and_past_the_end():
    """dS_T = None (zeros), tokens past cu_seqlens[-1], one-token sequences."""
    spec = synth.PrefillSpec(num_seqs=5, len_lo=1, len_hi=3, H=2, d_k=128, d_v=128,
                             s0_std=0.1, seed=16)
    _run(spec, dS_T_std=0.0, extra_tokens=5)


def test_backward_empty_sequences():
    """Zero-length sequences pass dS_T straight through to dS0."""
    d = synth.prefill_inputs(synth.PrefillSpec(num_seqs=3, len_lo=70, len_hi=70, H=2, d_k=128,
                                               d_v=128, s0_std=0.1, seed=17))
    cu = torch.tensor([0, 70, 70, 140, 140, 210], dtype=torch.int32)
    dev = parity.to_device(d)
    S0 = torch.randn(5, 2, 128, 128, device="cuda") * 0.1
    dO = torch.randn(210, 2, 128, device="cuda").to(torch.bfloat16)
    dS_T = torch.randn(5, 2, 128, 128, device="cuda")
    g = kda.backward(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], S0, cu.cuda(), dO,
                     dS_T, check_device_status=True)
    torch.cuda.synchronize()
    for n in (1, 3):
        assert torch.equal(g["dS0"][n], dS_T[n])


def test_backward_is_deterministic():
    spec = synth.PrefillSpec(num_seqs=3, len_lo=100, len_hi=300, H=2, d_k=128, d_v=256,
                             s0_std=0.1, seed=18)
    d = synth.prefill_inputs(spec)
    dO, dS_T = synth.backward_cotangents(d)
    dev = parity.to_device(d)
    args = (dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
            dev["cu_seqlens"], dO.cuda(), dS_T.cuda())
    a = kda.backward(*args)
    b = kda.backward(*args)
    torch.cuda.synchronize()
    for name in NAMES:
        assert torch.equal(a[name], b[name]), name


def test_backward_rejects_bad_cu_seqlens_on_device():
    spec = synth.PrefillSpec(num_seqs=2, len_lo=64, len_hi=64, H=1, d_k=128, d_v=128, seed=19)
    d = synth.prefill_inputs(spec)
    dev = parity.to_device(d)
    dO = torch.zeros(128, 1, 128, device="cuda", dtype=torch.bfloat16)
    bad = torch.tensor([0, 100, 90], dtype=torch.int32, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.backward(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], None, bad, dO,
                     check_device_status=True)
    assert e.value.status == kda.ERR_DEVICE_INPUT


def test_backward_prefill_workload_sampled():
    """The 8 x 4096-token, 32-head prefill workload at full size; the oracle
    checks three sampled (sequence, head) pairs over all 4096 tokens."""
    _run(synth.PREFILL, pairs=[(0, 0), (3, 17), (7, 31)])


@pytest.mark.parametrize("gate", ["head", "log_bf16"])
def test_backward_gate_layouts(gate):
    """kda_backward_gates: the gate expanded per channel for the oracle, whose
    per-channel gradient is reduced to the gate's layout (sum over the head's
    channels; alpha times it for log alpha)."""
    spec = synth.PrefillSpec(num_seqs=3, len_lo=40, len_hi=260, H=2, d_k=128, d_v=128,
                             s0_std=0.1, seed=21)
    d = synth.prefill_inputs(spec)
    dO, dS_T = synth.backward_cotangents(d)
    T, H, d_v = d["v"].shape
    if gate == "head":
        g_in = d["alpha"][:, :, 0].contiguous()
        a_full = g_in[:, :, None].expand(T, H, d_v).contiguous()
    else:
        g_in = torch.log(d["alpha"]).to(torch.bfloat16)
        a_full = torch.exp(g_in.double()).float()
    d_exp = dict(d, alpha=a_full)
    dev = parity.to_device(d)
    g = kda.backward_gates(dev["q"], dev["k"], dev["v"], g_in.cuda(), dev["beta"], dev["S0"],
                           dev["cu_seqlens"], dO.cuda(), dS_T.cuda(), gate=gate,
                           check_device_status=True)
    torch.cuda.synchronize()
    pairs = [(n, hh) for n in range(spec.num_seqs) for hh in range(H)]
    ref = _oracle(d_exp, dO, dS_T, pairs)
    for key in ref:
        da = ref[key]["dalpha"]
        n, hh = key
        a0, a1 = int(d["cu_seqlens"][n]), int(d["cu_seqlens"][n + 1])
        ref[key]["dalpha"] = da.sum(axis=1) if gate == "head" else \
            da * a_full[a0:a1, hh].double().numpy()
    g["dalpha"] = g.pop("dgate")
    worst = _compare(d, g, ref)
    assert all(e <= TOL for e in worst.values()), worst
