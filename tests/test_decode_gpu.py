"""kda_decode_step against the oracle (GPU)."""
import pytest
import torch

import oracle
import parity
from gated_delta_rule_45_gb300 import kda, synth

pytestmark = pytest.mark.gpu


def _run(spec):
    d = synth.decode_inputs(spec)
    dev = parity.to_device(d)
    S = dev["S"].clone()
    o = kda.decode_step(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], S)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.decode_step(*(parity._np(d[x]) for x in ("q", "k", "v")),
                                      d["alpha"].numpy(), d["beta"].numpy(),
                                      d["S"].double().numpy())
    o_g = o.float().cpu().numpy()
    S_g = S.cpu().numpy()
    store = torch.bfloat16 if spec.dtype == "bf16" else torch.float32
    # one token per (b, h): a short slice, gated against the correctly rounded value;
    # the whole step's o is also held to the exact value
    worst_o = max(parity.rel_gate(o_g[b, h], o_ref[b, h], store)
                  for b in range(spec.B) for h in range(spec.H))
    worst_o = max(worst_o, parity.rel(o_g, o_ref))
    worst_s = max(parity.rel(S_g[b, h], S_ref[b, h]) for b in range(spec.B) for h in range(spec.H))
    return worst_o, worst_s


@pytest.mark.parametrize("B,H,d_k,d_v,dtype", [
    (3, 2, 16, 48, "bf16"),
    (5, 3, 32, 32, "fp32"),
    (4, 2, 64, 80, "bf16"),
    (2, 2, 128, 128, "bf16"),
    (3, 1, 128, 200, "fp32"),
    (2, 2, 256, 96, "bf16"),
    (7, 3, 128, 256, "bf16"),
    (1, 1, 128, 1, "fp32"),
])
def test_decode_small(B, H, d_k, d_v, dtype):
    spec = synth.DecodeSpec(B=B, H=H, d_k=d_k, d_v=d_v, dtype=dtype, seed=B * 100 + d_k)
    wo, ws = _run(spec)
    tol = parity.TOL_BF16 if dtype == "bf16" else parity.TOL_FP32
    assert wo <= tol and ws <= tol, (wo, ws)


def test_decode_workload_full():
    """B = 256 sequences, H = 32, d_k = d_v = 128, bf16 (the decode-step workload), all slices."""
    wo, ws = _run(synth.DECODE)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)


def test_decode_state_only_in_place():
    """The kernel touches exactly S[b][h] and o[b][h]: guard bands around both stay intact."""
    spec = synth.DecodeSpec(B=3, H=2, d_k=64, d_v=32, seed=5)
    d = parity.to_device(synth.decode_inputs(spec))
    n_s = d["S"].numel()
    buf = torch.full((n_s + 2048,), 7.0, device="cuda")
    S = buf[1024:1024 + n_s].view_as(d["S"])
    S.copy_(d["S"])
    obuf = torch.full((3 * 2 * 32 + 256,), 3.0, device="cuda", dtype=torch.bfloat16)
    o = obuf[128:128 + 3 * 2 * 32].view(3, 2, 32)
    kda.decode_step(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S, o)
    torch.cuda.synchronize()
    assert torch.all(buf[:1024] == 7.0) and torch.all(buf[1024 + n_s:] == 7.0)
    assert torch.all(obuf[:128] == 3.0) and torch.all(obuf[128 + 192:] == 3.0)


@pytest.mark.parametrize("gate,d_k,d_v", [("head", 128, 128), ("log_bf16", 128, 256),
                                          ("head", 64, 80)])
def test_decode_gate_layouts(gate, d_k, d_v):
    """kda_decode_step_gates against the oracle with the gates expanded to
    alpha[b][h][r] (exp taken in float64)."""
    spec = synth.DecodeSpec(B=5, H=3, d_k=d_k, d_v=d_v, seed=41)
    d = synth.decode_inputs(spec)
    gen = torch.Generator().manual_seed(42)
    if gate == "head":
        g_in = torch.sigmoid(torch.randn(spec.B, spec.H, generator=gen) + 4.0)
        alpha = g_in[:, :, None].expand(spec.B, spec.H, d_v).contiguous()
    else:
        g_in = torch.log(torch.sigmoid(torch.randn(spec.B, spec.H, d_v, generator=gen) + 4.0))
        g_in = g_in.to(torch.bfloat16)
        alpha = torch.exp(g_in.double()).float()
    dev = parity.to_device(d)
    S = dev["S"].clone()
    o = kda.decode_step_gates(dev["q"], dev["k"], dev["v"], g_in.cuda(), dev["beta"], S,
                              gate=gate)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.decode_step(*(parity._np(d[x]) for x in ("q", "k", "v")),
                                      alpha.numpy(), d["beta"].numpy(), d["S"].double().numpy())
    o_g, S_g = o.float().cpu().numpy(), S.cpu().numpy()
    worst_o = max(max(parity.rel_gate(o_g[b, h], o_ref[b, h], torch.bfloat16)
                      for b in range(spec.B) for h in range(spec.H)), parity.rel(o_g, o_ref))
    worst_s = max(parity.rel(S_g[b, h], S_ref[b, h]) for b in range(spec.B) for h in range(spec.H))
    assert worst_o <= parity.TOL_BF16 and worst_s <= parity.TOL_BF16, (worst_o, worst_s)


def test_decode_additive_update():
    """kda_decode_step_additive against the oracle's additive recurrence."""
    spec = synth.DecodeSpec(B=8, H=4, d_k=128, d_v=96, seed=5)
    d = synth.decode_inputs(spec)
    S = d["S"].cuda()
    o = kda.decode_step_additive(*(d[k].cuda() for k in ("q", "k", "v", "alpha", "beta")), S)
    torch.cuda.synchronize()
    bits = synth.bf16_bits
    o_ref, S_ref = oracle.decode_step(bits(d["q"]), bits(d["k"]), bits(d["v"]),
                                      d["alpha"].numpy(), d["beta"].numpy(),
                                      d["S"].double().numpy(), additive=True)
    assert parity.rel(o.float().cpu().numpy(), parity.round_to(o_ref[:, :, :], torch.bfloat16)) <= 2e-3
    assert parity.rel(S.cpu().numpy(), S_ref) <= 2e-5


@pytest.mark.parametrize("mu", [1.0, 0.0, -1.0])
def test_decode_fast_decay(mu):
    """A decode step multiplies by alpha and divides by nothing: gates far from
    1 are exact as well (alpha = sigmoid(N(mu, 1)))."""
    spec = synth.DecodeSpec(B=16, H=4, d_k=128, d_v=128, alpha_mu=mu, seed=71)
    wo, ws = _run(spec)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)
