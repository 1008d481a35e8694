"""kda_prefill against the oracle on small and ragged problems (GPU).

Sizes are chosen so the oracle finishes in seconds while still spanning
several chunks, several value-channel blocks and partial last chunks.
Both kernels run where the shape allows it.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from gated_delta_rule_45_gb300 import kda, synth

pytestmark = pytest.mark.gpu


def _kernels_for(spec):
    ks = ["simt"]
    dt = torch.bfloat16 if spec.dtype == "bf16" else torch.float32
    if kda.supported("tc", spec.H, spec.d_k, spec.d_v, dt, spec.chunk):
        ks.append("tc")
    return ks


def _check(spec, kernel, S0_override="keep", tol=None):
    d = synth.prefill_inputs(spec)
    if S0_override is None:
        d["S0"] = None
    dev = parity.to_device(d)
    o, S_T = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], chunk=spec.chunk, kernel=kernel,
                         check_device_status=True)
    torch.cuda.synchronize()
    pairs = [(n, h) for n in range(spec.num_seqs) for h in range(spec.H)]
    ref = parity.oracle_pairs(d, pairs)
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    if tol is None:
        tol = parity.TOL_BF16 if spec.dtype == "bf16" else parity.TOL_FP32
    assert wo <= tol and ws <= tol, (kernel, wo, ws)
    return o, S_T, d


SMALL = [
    synth.PrefillSpec(num_seqs=3, len_lo=1, len_hi=200, H=2, d_k=32, d_v=48, dtype="bf16",
                      chunk=16, s0_std=0.1, seed=1),
    synth.PrefillSpec(num_seqs=2, len_lo=100, len_hi=300, H=3, d_k=64, d_v=64, dtype="fp32",
                      chunk=32, s0_std=0.1, seed=2),
    synth.PrefillSpec(num_seqs=4, len_lo=1, len_hi=400, H=2, d_k=128, d_v=128, dtype="bf16",
                      chunk=64, s0_std=0.1, seed=3),
    synth.PrefillSpec(num_seqs=3, len_lo=60, len_hi=300, H=2, d_k=128, d_v=256, dtype="bf16",
                      chunk=64, s0_std=0.1, seed=4),
    synth.PrefillSpec(num_seqs=2, len_lo=129, len_hi=129, H=1, d_k=16, d_v=208, dtype="bf16",
                      chunk=64, s0_std=0.0, seed=5),
    synth.PrefillSpec(num_seqs=5, len_lo=64, len_hi=64, H=2, d_k=128, d_v=128, dtype="bf16",
                      chunk=64, alpha_mu=5.0, s0_std=0.1, seed=6),
]


@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_prefill_small(idx):
    spec = SMALL[idx]
    for kernel in _kernels_for(spec):
        _check(spec, kernel)


def test_tiny_workload_fp32_chunk16():
    """B = 1, H = 2, T = 64, d = 32, fp32, chunk 16 (the tiny oracle workload)."""
    _check(synth.TINY, "auto")


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_chunk_size_invariance(chunk):
    """The chunk size is an implementation choice: every chunk gives the oracle's answer."""
    spec = synth.PrefillSpec(num_seqs=2, len_lo=150, len_hi=250, H=2, d_k=64, d_v=64,
                             dtype="fp32", chunk=chunk, s0_std=0.2, seed=7)
    _check(spec, "simt")


def test_without_initial_state():
    spec = synth.PrefillSpec(num_seqs=3, len_lo=10, len_hi=200, H=2, d_k=128, d_v=128,
                             s0_std=0.1, seed=8)
    for kernel in _kernels_for(spec):
        _check(spec, kernel, S0_override=None)


def test_in_place_state_and_zero_length():
    """S_T may alias S0; zero-length sequences return S0 unchanged."""
    spec = synth.PrefillSpec(num_seqs=4, len_lo=50, len_hi=150, H=2, d_k=128, d_v=128,
                             s0_std=0.1, seed=9)
    d = synth.prefill_inputs(spec)
    # make sequences 1 and 3 empty
    lengths = [d["lengths"][0], 0, d["lengths"][2], 0]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    T = int(cu[-1])
    for key in ("q", "k", "v", "alpha", "beta"):
        d[key] = d[key][:T].contiguous()
    d["cu_seqlens"] = cu
    dev = parity.to_device(d)
    for kernel in _kernels_for(spec):
        S = dev["S0"].clone()
        o = torch.empty((T, spec.H, spec.d_v), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(kda.workspace_size(4), dtype=torch.uint8, device="cuda")
        kda.prefill_into(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], S,
                         dev["cu_seqlens"], o, S, ws, kernel=kernel)
        kda.device_status(ws)
        ref = parity.oracle_pairs(d, [(n, h) for n in range(4) for h in range(spec.H)])
        wo, wsr = parity.compare_pairs(d, o, S, ref)
        assert wo <= parity.TOL_BF16 and wsr <= parity.TOL_BF16, (kernel, wo, wsr)
        assert torch.equal(S[1], dev["S0"][1]) and torch.equal(S[3], dev["S0"][3])


def test_empty_batch_and_all_empty_sequences():
    H, d_k, d_v = 2, 128, 128
    z = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt, device="cuda")
    # all sequences empty: S_T = S0
    S0 = torch.randn(3, H, d_v, d_k, device="cuda")
    S_T = torch.empty_like(S0)
    cu = torch.zeros(4, dtype=torch.int32, device="cuda")
    ws = torch.empty(kda.workspace_size(3), dtype=torch.uint8, device="cuda")
    kda.prefill_into(z(0, H, d_k), z(0, H, d_k), z(0, H, d_v), z(0, H, d_v, dt=torch.float32),
                     z(0, H, dt=torch.float32), S0, cu, z(0, H, d_v), S_T, ws)
    kda.device_status(ws)
    assert torch.equal(S_T, S0)
    # no sequences at all
    cu0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.prefill_into(z(0, H, d_k), z(0, H, d_k), z(0, H, d_v), z(0, H, d_v, dt=torch.float32),
                     z(0, H, dt=torch.float32), None, cu0, z(0, H, d_v),
                     torch.empty(0, H, d_v, d_k, device="cuda"), ws)
    kda.device_status(ws)


@pytest.mark.parametrize("bad", [[1, 5, 9], [0, 6, 4], [0, 4, 12]])
def test_bad_cu_seqlens_reported_and_nothing_written(bad):
    """A malformed cu_seqlens is caught on the device: status reported, outputs untouched."""
    H, d_k, d_v, T = 2, 128, 128, 9
    g = torch.Generator(device="cpu").manual_seed(0)
    q = torch.randn(T, H, d_k, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(T, H, d_v, generator=g).to(torch.bfloat16).cuda()
    al = torch.full((T, H, d_v), 0.9, device="cuda")
    be = torch.full((T, H), 0.5, device="cuda")
    cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
    o = torch.full((T, H, d_v), 5.0, dtype=torch.bfloat16, device="cuda")
    S_T = torch.full((2, H, d_v, d_k), 5.0, device="cuda")
    ws = torch.empty(kda.workspace_size(2), dtype=torch.uint8, device="cuda")
    for kernel in ("simt", "tc"):
        try:
            kda.prefill_into(q, q, v, al, be, None, cu, o, S_T, ws, kernel=kernel)
        except kda.KdaError as e:
            assert e.status == kda.ERR_UNSUPPORTED and kernel == "tc"
            continue
        with pytest.raises(kda.KdaError) as ei:
            kda.device_status(ws)
        assert ei.value.status == kda.ERR_DEVICE_INPUT
        assert torch.all(o == 5.0) and torch.all(S_T == 5.0)


def _split_case(lengths, H, d_v, s0_std, seed, alpha_mu=3.0):
    spec = synth.PrefillSpec(num_seqs=len(lengths), len_lo=1, len_hi=1, H=H, d_k=128, d_v=d_v,
                             chunk=64, s0_std=s0_std, alpha_mu=alpha_mu, seed=seed)
    d = synth.prefill_inputs(spec)
    # replace the drawn lengths with the given ones (inputs are per token, so
    # a longer draw is cut to size)
    T = int(sum(lengths))
    big = synth.PrefillSpec(num_seqs=1, len_lo=T, len_hi=T, H=H, d_k=128, d_v=d_v, chunk=64,
                            s0_std=0.0, alpha_mu=alpha_mu, seed=seed)
    db = synth.prefill_inputs(big)
    for key in ("q", "k", "v", "alpha", "beta"):
        d[key] = db[key]
    d["cu_seqlens"] = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    d["lengths"] = list(lengths)
    return spec, d


@pytest.mark.parametrize("lengths,H,d_v,s0_std,alpha_mu", [
    ([1000, 60, 2500], 2, 128, 0.1, 3.0),   # one single-chunk sequence: mostly empty segments
    ([4096, 0, 3000], 1, 256, 0.1, 3.0),    # an empty sequence, two value blocks
    ([5000], 3, 128, 0.0, 3.0),             # no initial state
    ([6000, 3000], 2, 128, 0.5, 7.0),       # long memory: every chunk takes a correction
    ([4000, 130], 2, 256, 0.5, 1.0),        # quick decay: corrections die out in a few chunks
    ([3000], 48, 128, 0.5, 5.0),            # 48 chains: the rule takes two segments
])
def test_sequence_split_matches_oracle(lengths, H, d_v, s0_std, alpha_mu):
    """The split form (one pass: segment 0 from S0, every other segment from
    zero and as a transition from the identity; the scan of the segment maps;
    each later segment's output corrected by its initial state's share)
    against the oracle, on every (sequence, head)."""
    spec, d = _split_case(lengths, H, d_v, s0_std, seed=11, alpha_mu=alpha_mu)
    if not kda.supported("tc_split", H, 128, d_v, torch.bfloat16, 64):
        pytest.skip("tensor-core kernel not available for this shape")
    dev = parity.to_device(d)
    N = len(lengths)
    T = int(sum(lengths))
    ws_bytes = kda.workspace_size(N, H, 128, d_v, 64, T)
    assert ws_bytes > kda.workspace_size(N, H, 128, d_v, 64)   # room for the segments
    o, S_T = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], chunk=64, kernel="tc_split",
                         check_device_status=True)
    ref = parity.oracle_pairs(d, [(n, h) for n in range(N) for h in range(H)])
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)
    # the unsplit kernel on the same inputs agrees to rounding
    o2, S2 = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], chunk=64, kernel="tc", check_device_status=True)
    assert parity.rel(S_T.cpu().numpy(), S2.cpu().numpy()) < 1e-4
    assert parity.rel(o.float().cpu().numpy(), o2.float().cpu().numpy()) < 3e-3


def test_sequence_split_in_place_state():
    """S_T may alias S0 under the split form too."""
    spec, d = _split_case([3000, 2000], 2, 128, 0.1, seed=12)
    dev = parity.to_device(d)
    S = dev["S0"].clone()
    T = int(d["cu_seqlens"][-1])
    o = torch.empty((T, 2, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(kda.workspace_size(2, 2, 128, 128, 64, T), dtype=torch.uint8, device="cuda")
    kda.prefill_into(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], S,
                     dev["cu_seqlens"], o, S, ws, kernel="tc_split")
    kda.device_status(ws)
    ref = parity.oracle_pairs(d, [(n, h) for n in range(2) for h in range(2)])
    wo, wsr = parity.compare_pairs(d, o, S, ref)
    assert wo <= parity.TOL_BF16 and wsr <= parity.TOL_BF16, (wo, wsr)


@pytest.mark.parametrize("gate,d_v", [("head", 256), ("log_bf16", 128), ("channel", 128)])
def test_gate_layouts_match_oracle(gate, d_v):
    """kda_prefill_gates: one gate per (token, head) broadcast over the value
    channels (Gated DeltaNet's scalar gate), and log alpha in bf16; the oracle
    gets the same gates as alpha[t][h][r] (exp taken in float64)."""
    spec = synth.PrefillSpec(num_seqs=3, len_lo=60, len_hi=500, H=2, d_k=128, d_v=d_v,
                             s0_std=0.1, seed=31)
    d = synth.prefill_inputs(spec)
    T = int(d["cu_seqlens"][-1])
    gen = torch.Generator().manual_seed(32)
    if gate == "head":
        g_in = torch.sigmoid(torch.randn(T, spec.H, generator=gen) + 3.0)
        d["alpha"] = g_in[:, :, None].expand(T, spec.H, d_v).contiguous()
    elif gate == "log_bf16":
        g_in = torch.log(torch.sigmoid(torch.randn(T, spec.H, d_v, generator=gen) + 3.0))
        g_in = g_in.to(torch.bfloat16)
        d["alpha"] = torch.exp(g_in.double()).float()
    else:
        g_in = d["alpha"]
    dev = parity.to_device(d)
    o, S_T = kda.prefill_gates(dev["q"], dev["k"], dev["v"], g_in.cuda(), dev["beta"], dev["S0"],
                               dev["cu_seqlens"], gate=gate, check_device_status=True)
    ref = parity.oracle_pairs(d, [(n, h) for n in range(spec.num_seqs) for h in range(spec.H)])
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (gate, wo, ws)


@pytest.mark.parametrize("gate", ["head", "log_bf16"])
def test_gate_layouts_on_the_portable_kernel(gate):
    """The gate layouts on the fp32 CUDA-core kernel (d_k = 64, fp32 storage, chunk 32)."""
    spec = synth.PrefillSpec(num_seqs=2, len_lo=40, len_hi=200, H=2, d_k=64, d_v=48,
                             dtype="fp32", chunk=32, s0_std=0.1, seed=33)
    d = synth.prefill_inputs(spec)
    T = int(d["cu_seqlens"][-1])
    gen = torch.Generator().manual_seed(34)
    if gate == "head":
        g_in = torch.sigmoid(torch.randn(T, spec.H, generator=gen) + 3.0)
        d["alpha"] = g_in[:, :, None].expand(T, spec.H, spec.d_v).contiguous()
    else:
        g_in = torch.log(torch.sigmoid(torch.randn(T, spec.H, spec.d_v, generator=gen) + 3.0))
        g_in = g_in.to(torch.bfloat16)
        d["alpha"] = torch.exp(g_in.double()).float()
    dev = parity.to_device(d)
    o, S_T = kda.prefill_gates(dev["q"], dev["k"], dev["v"], g_in.cuda(), dev["beta"], dev["S0"],
                               dev["cu_seqlens"], gate=gate, chunk=32, kernel="simt",
                               check_device_status=True)
    ref = parity.oracle_pairs(d, [(n, h) for n in range(spec.num_seqs) for h in range(spec.H)])
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    assert wo <= 1e-4 and ws <= 1e-4, (gate, wo, ws)


@pytest.mark.parametrize("spec", [
    synth.PrefillSpec(num_seqs=4, len_lo=1, len_hi=300, H=2, d_k=128, d_v=128, s0_std=0.1,
                      seed=31),
    synth.PrefillSpec(num_seqs=2, len_lo=50, len_hi=200, H=3, d_k=64, d_v=48, dtype="fp32",
                      chunk=32, s0_std=0.1, seed=32),
])
def test_additive_update_matches_oracle(spec):
    """kda_prefill_additive (the update of linear attention without the
    prediction term) against the oracle's additive recurrence."""
    d = synth.prefill_inputs(spec)
    dev = parity.to_device(d)
    f = (lambda x: synth.bf16_bits(x)) if spec.dtype == "bf16" else (lambda x: x.numpy())
    o_ref, S_ref = oracle.prefill(f(d["q"]), f(d["k"]), f(d["v"]), d["alpha"].numpy(),
                                  d["beta"].numpy(),
                                  None if d["S0"] is None else d["S0"].double().numpy(),
                                  d["cu_seqlens"].numpy(), additive=True)
    cu = d["cu_seqlens"].numpy()
    tol = parity.TOL_BF16 if spec.dtype == "bf16" else parity.TOL_FP32
    dt = torch.bfloat16 if spec.dtype == "bf16" else torch.float32
    kernels = ["simt"] + (["tc"] if kda.supported("tc", spec.H, spec.d_k, spec.d_v, dt,
                                                  spec.chunk) else [])
    for kernel in kernels:
        o, S_T = kda.prefill_additive(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"],
                                      dev["S0"], dev["cu_seqlens"], chunk=spec.chunk,
                                      kernel=kernel, check_device_status=True)
        torch.cuda.synchronize()
        for n in range(spec.num_seqs):
            a, b = int(cu[n]), int(cu[n + 1])
            for h in range(spec.H):
                if b > a:
                    assert parity.rel_gate(o[a:b, h].float().cpu().numpy(), o_ref[a:b, h],
                                           o.dtype) <= tol, kernel
                assert parity.rel(S_T[n, h].cpu().numpy(), S_ref[n, h]) <= tol, kernel
    with pytest.raises(kda.KdaError):   # no sequence-axis split for the additive update
        kda.prefill_additive(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"],
                             dev["S0"], dev["cu_seqlens"], chunk=spec.chunk, kernel="tc_split")


# Fast decay: per-channel gates far from 1 ("Kimi (AI)", section "Kimi Delta
# Attention (KDA)", the forget gating line: alpha_t in (0, 1) per value
# channel).  At alpha = sigmoid(N(-1, 1)) the product over a 64-token chunk is
# about e^-96, beyond what the chunk form can divide by; such chunks run in
# passes of 16 tokens.
FAST_MU = [1.0, 0.0, -1.0]


@pytest.mark.parametrize("mu", FAST_MU)
def test_fast_decay_tensor_core_kernel(mu):
    spec = synth.PrefillSpec(num_seqs=4, len_lo=1, len_hi=400, H=2, d_k=128, d_v=256,
                             alpha_mu=mu, s0_std=0.1, seed=41)
    d = synth.prefill_inputs(spec)
    if not kda.supported("tc", spec.H, spec.d_k, spec.d_v, torch.bfloat16, 64):
        pytest.skip("tensor-core kernel not available for this shape")
    o, S_T, _ = _check(spec, "tc")
    assert torch.isfinite(o.float()).all() and torch.isfinite(S_T).all()


@pytest.mark.parametrize("mu", FAST_MU)
@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_fast_decay_portable_kernel(mu, chunk):
    spec = synth.PrefillSpec(num_seqs=3, len_lo=1, len_hi=300, H=2, d_k=64, d_v=48,
                             dtype="fp32", chunk=chunk, alpha_mu=mu, s0_std=0.1, seed=42)
    _check(spec, "simt")


@pytest.mark.parametrize("mu", FAST_MU)
def test_fast_decay_additive_update(mu):
    spec = synth.PrefillSpec(num_seqs=3, len_lo=1, len_hi=300, H=2, d_k=128, d_v=128,
                             alpha_mu=mu, s0_std=0.1, seed=43)
    d = synth.prefill_inputs(spec)
    dev = parity.to_device(d)
    o_ref, S_ref = oracle.prefill(synth.bf16_bits(d["q"]), synth.bf16_bits(d["k"]),
                                  synth.bf16_bits(d["v"]), d["alpha"].numpy(), d["beta"].numpy(),
                                  d["S0"].double().numpy(), d["cu_seqlens"].numpy(),
                                  additive=True)
    cu = d["cu_seqlens"].numpy()
    for kernel in ("simt", "tc"):
        o, S_T = kda.prefill_additive(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"],
                                      dev["S0"], dev["cu_seqlens"], kernel=kernel,
                                      check_device_status=True)
        torch.cuda.synchronize()
        for n in range(spec.num_seqs):
            a, b = int(cu[n]), int(cu[n + 1])
            for h in range(spec.H):
                if b > a:
                    assert parity.rel_gate(o[a:b, h].float().cpu().numpy(), o_ref[a:b, h],
                                           o.dtype) <= parity.TOL_BF16, (kernel, n, h)
                assert parity.rel(S_T[n, h].cpu().numpy(), S_ref[n, h]) <= parity.TOL_BF16


@pytest.mark.parametrize("kernel", ["simt", "tc"])
def test_decay_beyond_the_chunk_forms_range_is_reported(kernel):
    """A channel whose alpha multiplies to 1e-40 over 16 tokens: even one pass
    of 16 cannot divide by that, and the device reports KDA_ERR_DEVICE_RANGE
    (an input error, found on the device; nothing faults).  Sequences and heads
    that stay in range are still right."""
    spec = synth.PrefillSpec(num_seqs=2, len_lo=64, len_hi=200, H=2, d_k=128, d_v=128,
                             s0_std=0.1, seed=44)
    d = synth.prefill_inputs(spec)
    a = int(d["cu_seqlens"][1])
    d["alpha"][a:a + 16, 1, 5] = 10.0 ** -2.5     # sequence 1, head 1, channel 5
    dev = parity.to_device(d)
    with pytest.raises(kda.KdaError) as e:
        kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                    dev["cu_seqlens"], kernel=kernel, check_device_status=True)
    assert e.value.status == kda.ERR_DEVICE_RANGE
    o, S_T = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], kernel=kernel)
    torch.cuda.synchronize()
    ref = parity.oracle_pairs(d, [(0, 0), (0, 1), (1, 0)])
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)


def _lengths_case(lengths, H, d, seed, dtype="bf16"):
    """A batch with the given sequence lengths (inputs drawn for the total)."""
    T = int(sum(lengths))
    big = synth.PrefillSpec(num_seqs=1, len_lo=max(T, 1), len_hi=max(T, 1), H=H, d_k=d, d_v=d,
                            chunk=64, dtype=dtype, s0_std=0.0, seed=seed)
    d_ = synth.prefill_inputs(big)
    spec = synth.PrefillSpec(num_seqs=len(lengths), len_lo=1, len_hi=1, H=H, d_k=d, d_v=d,
                             chunk=64, dtype=dtype, s0_std=0.1, seed=seed)
    d_["S0"] = synth.prefill_inputs(spec)["S0"]
    d_["spec"] = spec
    for key in ("q", "k", "v", "alpha", "beta"):
        d_[key] = d_[key][:T]
    d_["cu_seqlens"] = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    d_["lengths"] = list(lengths)
    return d_


@pytest.mark.parametrize("N", [1, 7, 1024, 1025, 3000, 5000])
def test_planner_order_is_longest_first(N):
    """The planner's order (in the workspace after a prefill) is exactly the
    sequences sorted by (-length, index): one sorted run up to 1024
    sequences, several runs merged by rank beyond; lengths with many ties."""
    rng = np.random.default_rng(N)
    lengths = rng.integers(0, 40, size=N).tolist()
    d = _lengths_case(lengths, 1, 16, seed=N, dtype="fp32")
    dev = parity.to_device(d)
    T = int(sum(lengths))
    o = torch.empty((T, 1, 16), dtype=torch.float32, device="cuda")
    S_T = torch.empty((N, 1, 16, 16), dtype=torch.float32, device="cuda")
    ws = torch.empty(kda.workspace_size(N, 1, 16, 16, 16, T), dtype=torch.uint8, device="cuda")
    kda.prefill_into(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                     dev["cu_seqlens"], o, S_T, ws, chunk=16)
    kda.device_status(ws)
    order = ws[16:16 + 4 * N].cpu().view(torch.int32).tolist()
    assert order == sorted(range(N), key=lambda i: (-lengths[i], i))


def test_many_short_sequences_tensor_core():
    """1500 sequences (several planner runs) through the tensor-core kernel:
    sampled (sequence, head) pairs against the oracle, and every final state
    against the portable kernel."""
    rng = np.random.default_rng(77)
    lengths = rng.integers(1, 150, size=1500).tolist()
    d = _lengths_case(lengths, 1, 128, seed=77)
    if not kda.supported("tc", 1, 128, 128, torch.bfloat16, 64):
        pytest.skip("tensor-core kernel not available for this shape")
    dev = parity.to_device(d)
    o, S_T = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], chunk=64, kernel="tc", check_device_status=True)
    pairs = [(int(n), 0) for n in rng.choice(1500, size=40, replace=False)]
    pairs += [(int(np.argmax(lengths)), 0), (int(np.argmin(lengths)), 0)]
    ref = parity.oracle_pairs(d, sorted(set(pairs)))
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)
    o2, S2 = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], chunk=64, kernel="simt", check_device_status=True)
    assert parity.rel(S_T.cpu().numpy(), S2.cpu().numpy()) < 1e-3


def test_split_reports_decay_beyond_the_chunk_forms_range():
    """Under the sequence-axis split a chunk whose alpha product falls below the
    chunk form's range is reported (KDA_ERR_DEVICE_RANGE), not handed to the
    portable kernel; here it lies inside a later segment of one channel.  The
    other (sequence, head) pairs are still right: rows of the state, and so
    the segment maps' rows, do not mix."""
    spec, d = _split_case([2000, 1500], 2, 128, 0.1, seed=45)
    if not kda.supported("tc_split", 2, 128, 128, torch.bfloat16, 64):
        pytest.skip("tensor-core kernel not available for this shape")
    a = int(d["cu_seqlens"][1]) + 800
    d["alpha"][a:a + 16, 1, 5] = 10.0 ** -2.5     # sequence 1, head 1, channel 5
    dev = parity.to_device(d)
    with pytest.raises(kda.KdaError) as e:
        kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                    dev["cu_seqlens"], chunk=64, kernel="tc_split", check_device_status=True)
    assert e.value.status == kda.ERR_DEVICE_RANGE
    o, S_T = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], chunk=64, kernel="tc_split")
    torch.cuda.synchronize()
    ref = parity.oracle_pairs(d, [(0, 0), (0, 1), (1, 0)])
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)
