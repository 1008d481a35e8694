"""The Python binding rejects wrongly typed or placed tensors before it calls
into the library: the C ABI reads alpha, beta, states and gradients as fp32
and cu_seqlens as int32, so a tensor of another type would be misread, not
refused.  CPU only: nothing here reaches the C ABI."""
import pytest
import torch

from gated_delta_rule_45_gb300 import kda

T, H, DK, DV, N = 8, 2, 16, 16, 2
BF16, F32 = torch.bfloat16, torch.float32


def _prefill_args(**over):
    a = dict(q=torch.zeros(T, H, DK, dtype=BF16), k=torch.zeros(T, H, DK, dtype=BF16),
             v=torch.zeros(T, H, DV, dtype=BF16), alpha=torch.ones(T, H, DV),
             beta=torch.zeros(T, H), S0=torch.zeros(N, H, DV, DK),
             cu_seqlens=torch.tensor([0, 4, T], dtype=torch.int32),
             o=torch.zeros(T, H, DV, dtype=BF16), S_T=torch.zeros(N, H, DV, DK))
    a.update(over)
    return a


BAD_PREFILL = {
    "alpha_bf16": dict(alpha=torch.ones(T, H, DV, dtype=BF16)),
    "beta_f64": dict(beta=torch.zeros(T, H, dtype=torch.float64)),
    "S0_bf16": dict(S0=torch.zeros(N, H, DV, DK, dtype=BF16)),
    "S_T_f64": dict(S_T=torch.zeros(N, H, DV, DK, dtype=torch.float64)),
    "cu_int64": dict(cu_seqlens=torch.tensor([0, 4, T])),
    "k_f32": dict(k=torch.zeros(T, H, DK)),
    "o_f32": dict(o=torch.zeros(T, H, DV)),
    "q_f16": dict(q=torch.zeros(T, H, DK, dtype=torch.float16)),
}

_ORDER = ("q", "k", "v", "alpha", "beta", "S0", "cu_seqlens", "o", "S_T")
WS = torch.zeros(1024, dtype=torch.uint8)


def _call_prefill(fn, a):
    args = [a[n] for n in _ORDER]
    if fn == "prefill_noalloc_into":
        return kda.prefill_noalloc_into(*args)
    return getattr(kda, fn)(*args, WS)


@pytest.mark.parametrize("fn", ["prefill_into", "prefill_additive_into", "prefill_noalloc_into"])
@pytest.mark.parametrize("bad", sorted(BAD_PREFILL))
def test_prefill_rejects_types(fn, bad):
    with pytest.raises(TypeError):
        _call_prefill(fn, _prefill_args(**BAD_PREFILL[bad]))


@pytest.mark.parametrize("fn", ["prefill_into", "prefill_additive_into", "prefill_noalloc_into"])
def test_prefill_rejects_host_tensors(fn):
    with pytest.raises(ValueError, match="CUDA"):
        _call_prefill(fn, _prefill_args())


@pytest.mark.parametrize("gate,alpha", [
    ("channel", torch.ones(T, H, DV, dtype=BF16)),
    ("head", torch.ones(T, H, DV)),              # the head layout is rank 2
    ("log_bf16", torch.zeros(T, H, DV)),         # log alpha is stored in bf16
])
def test_prefill_gates_rejects_gate_types(gate, alpha):
    a = _prefill_args(alpha=alpha)
    with pytest.raises(TypeError):
        kda.prefill_gates_into(*[a[n] for n in _ORDER], WS, gate=gate)


def test_prefill_gates_rejects_state_and_placement():
    a = _prefill_args(S0=torch.zeros(N, H, DV, DK, dtype=BF16))
    with pytest.raises(TypeError):
        kda.prefill_gates_into(*[a[n] for n in _ORDER], WS)
    a = _prefill_args()
    with pytest.raises(ValueError, match="CUDA"):
        kda.prefill_gates_into(*[a[n] for n in _ORDER], WS)


def _decode_args(**over):
    B = 3
    a = dict(q=torch.zeros(B, H, DK, dtype=BF16), k=torch.zeros(B, H, DK, dtype=BF16),
             v=torch.zeros(B, H, DV, dtype=BF16), alpha=torch.ones(B, H, DV),
             beta=torch.zeros(B, H), S=torch.zeros(B, H, DV, DK))
    a.update(over)
    return a


BAD_DECODE = {
    "S_bf16": dict(S=torch.zeros(3, H, DV, DK, dtype=BF16)),
    "alpha_f64": dict(alpha=torch.ones(3, H, DV, dtype=torch.float64)),
    "beta_bf16": dict(beta=torch.zeros(3, H, dtype=BF16)),
    "v_f32": dict(v=torch.zeros(3, H, DV)),
}


@pytest.mark.parametrize("fn", ["decode_step", "decode_step_additive"])
@pytest.mark.parametrize("bad", sorted(BAD_DECODE))
def test_decode_rejects_types(fn, bad):
    a = _decode_args(**BAD_DECODE[bad])
    with pytest.raises(TypeError):
        getattr(kda, fn)(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S"])


@pytest.mark.parametrize("fn", ["decode_step", "decode_step_additive"])
def test_decode_rejects_host_tensors(fn):
    a = _decode_args()
    with pytest.raises(ValueError, match="CUDA"):
        getattr(kda, fn)(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S"])


def test_decode_gates_rejects_types():
    a = _decode_args()
    with pytest.raises(TypeError):    # the head layout wants [B, H]
        kda.decode_step_gates(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S"],
                              gate="head")
    a = _decode_args(S=torch.zeros(3, H, DV, DK, dtype=BF16))
    with pytest.raises(TypeError):
        kda.decode_step_gates(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S"])


def _grads(**over):
    g = dict(dq=torch.zeros(T, H, DK), dk=torch.zeros(T, H, DK), dv=torch.zeros(T, H, DV),
             dalpha=torch.zeros(T, H, DV), dbeta=torch.zeros(T, H),
             dS0=torch.zeros(N, H, DV, DK))
    g.update(over)
    return g


@pytest.mark.parametrize("bad", ["dO_f32", "dS_T_bf16", "dq_bf16", "dS0_f64", "cu_int64"])
def test_backward_rejects_types(bad):
    a = _prefill_args(cu_seqlens=torch.tensor([0, 4, T]) if bad == "cu_int64" else None)
    if a["cu_seqlens"] is None:
        a["cu_seqlens"] = torch.tensor([0, 4, T], dtype=torch.int32)
    dO = torch.zeros(T, H, DV, dtype=F32 if bad == "dO_f32" else BF16)
    dS_T = torch.zeros(N, H, DV, DK, dtype=BF16 if bad == "dS_T_bf16" else F32)
    over = {"dq_bf16": dict(dq=torch.zeros(T, H, DK, dtype=BF16)),
            "dS0_f64": dict(dS0=torch.zeros(N, H, DV, DK, dtype=torch.float64))}.get(bad, {})
    with pytest.raises(TypeError):
        kda.backward_into(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S0"],
                          a["cu_seqlens"], dO, dS_T, _grads(**over), WS)


def test_backward_rejects_host_tensors():
    a = _prefill_args()
    with pytest.raises(ValueError, match="CUDA"):
        kda.backward_into(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S0"],
                          a["cu_seqlens"], torch.zeros(T, H, DV, dtype=BF16), None, _grads(), WS)


def test_backward_gates_rejects_types_and_placement():
    a = _prefill_args()
    dO = torch.zeros(T, H, DV, dtype=BF16)
    with pytest.raises(TypeError):    # dS_T must be fp32
        kda.backward_gates(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S0"],
                           a["cu_seqlens"], dO, torch.zeros(N, H, DV, DK, dtype=BF16))
    with pytest.raises(TypeError):    # the head layout wants [T, H]
        kda.backward_gates(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S0"],
                           a["cu_seqlens"], dO, gate="head")
    with pytest.raises(ValueError, match="CUDA"):
        kda.backward_gates(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["S0"],
                           a["cu_seqlens"], dO)


@pytest.mark.parametrize("bad", ["q_bf16", "partial_bf16", "h_last_f32", "blocks_f16"])
def test_attnres_rejects_types(bad):
    d = 64
    blocks = torch.zeros(2, T, d, dtype=torch.float16 if bad == "blocks_f16" else BF16)
    q = torch.zeros(d, dtype=BF16 if bad == "q_bf16" else F32)
    partial = torch.zeros(T, d, dtype=BF16 if bad == "partial_bf16" else F32)
    h_last = torch.zeros(T, d, dtype=F32 if bad == "h_last_f32" else BF16)
    with pytest.raises(TypeError):
        kda.attnres_layer(blocks, q, partial=partial, h_last=h_last)


def test_attnres_rejects_host_tensors():
    with pytest.raises(ValueError, match="CUDA"):
        kda.attnres_layer(torch.zeros(2, T, 64, dtype=BF16), torch.zeros(64))
