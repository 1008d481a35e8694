"""The C ABI without a GPU: the library loads, exports every symbol that
include/kda.h declares, and rejects bad arguments on the host before any
CUDA call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", n) for n in sorted(os.listdir(os.path.join(ROOT, "include")))
           if n.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_45_gb300 import build, kda
    build.build()
    return kda.load()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b((?:kda|attnres)_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("kda_prefill", "kda_decode_step", "kda_prefill_workspace_size",
                     "kda_status_string", "kda_prefill_device_status"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in kda.h but not exported"


def test_status_strings_and_version(lib):
    from gated_delta_rule_45_gb300 import kda
    for code in range(7):
        assert isinstance(kda.status_string(code), str)
    assert kda.status_string(0) == "ok"
    assert lib.kda_version() >> 16 == 1


def test_workspace_size(lib):
    from gated_delta_rule_45_gb300 import kda
    assert kda.workspace_size(0) >= 16
    assert kda.workspace_size(1000) >= 16 + 4 * 1000
    assert kda.workspace_size(1000) % 256 == 0
    assert lib.kda_prefill_workspace_size(-1, 1, 128, 128, 64) == 0
    # with the token count: never less than without it (the split's buffers,
    # where the device would take the split, replace the hand-back bitmap)
    for N, T, H, dv in ((1, 131072, 32, 128), (8, 32768, 32, 128), (64, 4096, 16, 256)):
        plain = kda.workspace_size(N, H, 128, dv, 64)
        tok = kda.workspace_size(N, H, 128, dv, 64, T)
        assert tok >= plain and tok % 256 == 0
    assert lib.kda_prefill_workspace_size_tokens(-1, 64, 1, 128, 128, 64) == 0
    assert lib.kda_prefill_workspace_size_tokens(1, -1, 1, 128, 128, 64) == 0


P = ctypes.c_void_p


def _fake(addr):
    # never dereferenced: each call below must return before any CUDA work
    return P(addr)


def _prefill(lib, **kw):
    args = dict(q=_fake(0x10000), k=_fake(0x20000), v=_fake(0x30000), alpha=_fake(0x40000),
                beta=_fake(0x50000), S0=None, cu=_fake(0x60000), N=2, T=64, H=2, d_k=64,
                d_v=64, dtype=0, chunk=64, o=_fake(0x70000), S_T=_fake(0x80000),
                ws=_fake(0x90000), ws_bytes=4096, kernel=0)
    args.update(kw)
    return lib.kda_prefill_ex(args["q"], args["k"], args["v"], args["alpha"], args["beta"],
                              args["S0"], args["cu"], args["N"], args["T"], args["H"],
                              args["d_k"], args["d_v"], args["dtype"], args["chunk"], args["o"],
                              args["S_T"], args["ws"], args["ws_bytes"], args["kernel"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(chunk=48), 2),
    (dict(chunk=128), 2),
    (dict(d_k=130), 2),
    (dict(d_k=256), 2),
    (dict(d_v=2048), 2),
    (dict(d_v=40), 2),
    (dict(H=0), 1),
    (dict(N=-1), 1),
    (dict(T=-5), 1),
    (dict(dtype=7), 1),
    (dict(kernel=9), 1),
    (dict(cu=None), 1),
    (dict(S_T=None), 1),
    (dict(ws=None), 1),
    (dict(q=None), 1),
    (dict(ws_bytes=8), 1),
    (dict(q=_fake(0x10004)), 1),            # misaligned
    (dict(o=_fake(0x10000)), 1),            # o overlaps q
    (dict(S0=_fake(0x80000 + 64)), 1),      # S_T partially overlaps S0
    (dict(kernel=2, d_k=64), 2),            # tensor-core kernel needs d_k == 128
])
def test_prefill_rejects_on_host(lib, kw, expect):
    assert _prefill(lib, **kw) == expect


def _decode(lib, **kw):
    args = dict(q=_fake(0x10000), k=_fake(0x20000), v=_fake(0x30000), alpha=_fake(0x40000),
                beta=_fake(0x50000), S=_fake(0x100000), B=2, H=2, d_k=128, d_v=128, dtype=0,
                o=_fake(0x90000))
    args.update(kw)
    return lib.kda_decode_step(args["q"], args["k"], args["v"], args["alpha"], args["beta"],
                               args["S"], args["B"], args["H"], args["d_k"], args["d_v"],
                               args["dtype"], args["o"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(d_k=96), 2),
    (dict(d_k=512), 2),
    (dict(d_v=5000), 2),
    (dict(H=0), 1),
    (dict(B=-1), 1),
    (dict(dtype=3), 1),
    (dict(S=None), 1),
    (dict(o=None), 1),
    (dict(v=_fake(0x30002)), 1),
    (dict(o=_fake(0x100000)), 1),           # o overlaps S
])
def test_decode_rejects_on_host(lib, kw, expect):
    assert _decode(lib, **kw) == expect


def test_supported_query(lib):
    from gated_delta_rule_45_gb300 import kda
    import torch
    assert kda.supported("simt", 2, 64, 64, torch.float32, 16)
    assert kda.supported("auto", 2, 128, 256, torch.bfloat16, 64)
    assert not kda.supported("simt", 2, 130, 64, torch.float32, 16)
    assert not kda.supported("tc", 2, 64, 128, torch.bfloat16, 64)
    assert not kda.supported("tc", 2, 128, 128, torch.float32, 64)
    assert lib.kda_prefill_supported(7, 1, 128, 128, 0, 64) == 1


def test_decode_empty_batch_is_noop(lib):
    assert _decode(lib, B=0, q=None, k=None, v=None, alpha=None, beta=None, S=None, o=None) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    from gated_delta_rule_45_gb300 import kda
    with pytest.raises(RuntimeError, match="libkda.so not found"):
        kda.load(str(tmp_path / "missing.so"))


def _prefill_gates(lib, **kw):
    args = dict(q=_fake(0x10000), k=_fake(0x20000), v=_fake(0x30000), alpha=_fake(0x40000),
                gate=1, beta=_fake(0x50000), S0=None, cu=_fake(0x60000), N=2, T=64, H=2,
                d_k=128, d_v=128, dtype=0, chunk=64, o=_fake(0x700000), S_T=_fake(0x800000),
                ws=_fake(0x900000), ws_bytes=4096, kernel=0)
    args.update(kw)
    return lib.kda_prefill_gates(args["q"], args["k"], args["v"], args["alpha"], args["gate"],
                                 args["beta"], args["S0"], args["cu"], args["N"], args["T"],
                                 args["H"], args["d_k"], args["d_v"], args["dtype"],
                                 args["chunk"], args["o"], args["S_T"], args["ws"],
                                 args["ws_bytes"], args["kernel"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(gate=7), 1),                      # unknown gate layout
    (dict(gate=1, kernel=3), 2),            # the other layouts never split
    (dict(gate=2, kernel=3), 2),
    (dict(gate=1, d_k=130), 2),             # not a supported shape at all
    (dict(gate=1, alpha=None), 1),
    (dict(gate=2, alpha=_fake(0x10002)), 1),   # misaligned
    # o may not overlap the gate, whose size depends on its layout
    (dict(gate=2, o=_fake(0x40000 + 16384)), 1),
    (dict(gate=1, o=_fake(0x40000 + 256)), 1),
])
def test_prefill_gates_rejects_on_host(lib, kw, expect):
    assert _prefill_gates(lib, **kw) == expect


def test_prefill_ex_split_needs_a_tensor_core_shape(lib):
    assert _prefill(lib, kernel=3, d_k=64) == 2


def test_decode_gates_rejects_on_host(lib):
    def call(gate, alpha=_fake(0x40000), o=_fake(0x900000)):
        return lib.kda_decode_step_gates(_fake(0x10000), _fake(0x20000), _fake(0x30000), alpha,
                                         gate, _fake(0x50000), _fake(0x100000), 2, 2, 128, 128,
                                         0, o, None)
    assert call(9) == 1                          # unknown layout
    assert call(1, alpha=None) == 1
    assert call(2, alpha=_fake(0x40008)) == 1    # misaligned
    assert call(1, o=_fake(0x40000)) == 1        # o overlaps the [B][H] gate


def _backward(lib, **kw):
    M = 0x1000000   # 16 MB apart: no two fake buffers of this shape overlap
    args = dict(q=_fake(1 * M), k=_fake(2 * M), v=_fake(3 * M), alpha=_fake(4 * M),
                beta=_fake(5 * M), S0=None, cu=_fake(6 * M), N=2, T=64, H=2, d_k=128, d_v=128,
                dtype=0, chunk=64, dO=_fake(7 * M), dS_T=None, dq=_fake(8 * M), dk=_fake(9 * M),
                dv=_fake(10 * M), dalpha=_fake(11 * M), dbeta=_fake(12 * M), dS0=None,
                ws=_fake(13 * M), ws_bytes=None)
    args.update(kw)
    if args["ws_bytes"] is None:
        args["ws_bytes"] = lib.kda_backward_workspace_size(args["N"], args["T"], args["H"],
                                                           128, 128, 64)
    return lib.kda_backward(args["q"], args["k"], args["v"], args["alpha"], args["beta"],
                            args["S0"], args["cu"], args["N"], args["T"], args["H"], args["d_k"],
                            args["d_v"], args["dtype"], args["chunk"], args["dO"], args["dS_T"],
                            args["dq"], args["dk"], args["dv"], args["dalpha"], args["dbeta"],
                            args["dS0"], args["ws"], args["ws_bytes"], None)


def test_backward_workspace_size(lib):
    f = lib.kda_backward_workspace_size
    assert f(2, 64, 2, 128, 128, 64) > 0
    # chunk-start states: (T / 64 + N) slots of H d_v d_k fp32, plus 2 partial sums per block
    assert f(8, 32768, 32, 128, 128, 64) >= (512 + 8) * 32 * 128 * 128 * 4 + \
        2 * 2 * 32768 * 32 * 128 * 4
    for bad in [(2, 64, 2, 64, 128, 64), (2, 64, 2, 128, 96, 64), (2, 64, 2, 128, 128, 32),
                (-1, 64, 2, 128, 128, 64), (2, 64, 0, 128, 128, 64)]:
        assert f(*bad) == 0


@pytest.mark.parametrize("kw,expect", [
    (dict(dtype=1), 2),                           # fp32 inputs: not implemented
    (dict(d_k=64), 2),
    (dict(d_v=96), 2),
    (dict(chunk=32), 2),
    (dict(dtype=5), 1),
    (dict(ws_bytes=1024), 1),                     # workspace too small
    (dict(dO=None), 1),
    (dict(dq=None), 1),
    (dict(dq=_fake(0x1000008)), 1),               # misaligned (and inside q)
    (dict(dk=_fake(8 * 0x1000000 + 4096)), 1),    # dk overlaps dq
    (dict(dv=_fake(3 * 0x1000000)), 1),           # dv is v
    (dict(dS0=_fake(4 * 0x1000000 + 256)), 1),    # dS0 overlaps alpha
    (dict(dalpha=_fake(13 * 0x1000000)), 1),      # dalpha inside the workspace
])
def test_backward_rejects_on_host(lib, kw, expect):
    assert _backward(lib, **kw) == expect


def _attnres(lib, **kw):
    M = 0x1000000
    args = dict(blocks=_fake(1 * M), nb=3, partial=None, h_last=None, partial_out=None,
                block_out=None, q=_fake(2 * M), scale=0.1, T=64, d=256, dtype=0, h=_fake(3 * M))
    args.update(kw)
    return lib.attnres_layer(args["blocks"], args["nb"], args["partial"], args["h_last"],
                             args["partial_out"], args["block_out"], args["q"], args["scale"],
                             args["T"], args["d"], args["dtype"], args["h"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(d=12), 2),                                   # d not a multiple of 8
    (dict(nb=65), 2),                                  # more than 64 sources
    (dict(nb=64, h_last=_fake(4 * 0x1000000)), 2),     # 64 blocks + the running sum
    (dict(nb=0), 1),                                   # no source at all
    (dict(nb=-1), 1),
    (dict(dtype=7), 1),
    (dict(partial_out=_fake(5 * 0x1000000)), 1),       # running sum out without one in
    (dict(q=None), 1),
    (dict(h=_fake(3 * 0x1000000 + 8)), 1),             # misaligned
    (dict(h=_fake(1 * 0x1000000 + 4096)), 1),          # h inside blocks
    (dict(h_last=_fake(4 * 0x1000000), block_out=_fake(4 * 0x1000000)), 1),   # block_out is h_last
])
def test_attnres_rejects_on_host(lib, kw, expect):
    assert _attnres(lib, **kw) == expect


def test_attnres_empty_is_a_no_op(lib):
    # T == 0 returns before any CUDA call
    assert _attnres(lib, T=0) == 0


def test_prefill_additive_rejects_on_host(lib):
    def call(**kw):
        args = dict(q=_fake(0x10000), k=_fake(0x20000), v=_fake(0x30000), alpha=_fake(0x40000),
                    beta=_fake(0x50000), S0=None, cu=_fake(0x60000), N=2, T=64, H=2, d_k=128,
                    d_v=128, dtype=0, chunk=64, o=_fake(0x70000), S_T=_fake(0x80000),
                    ws=_fake(0x90000), ws_bytes=4096, kernel=0)
        args.update(kw)
        return lib.kda_prefill_additive(args["q"], args["k"], args["v"], args["alpha"],
                                        args["beta"], args["S0"], args["cu"], args["N"],
                                        args["T"], args["H"], args["d_k"], args["d_v"],
                                        args["dtype"], args["chunk"], args["o"], args["S_T"],
                                        args["ws"], args["ws_bytes"], args["kernel"], None)
    assert call(kernel=3) == 2          # no sequence-axis split for the additive update
    assert call(kernel=9) == 1
    assert call(chunk=48) == 2
    assert call(o=None) == 1
    assert call(o=_fake(0x70008)) == 1  # misaligned


def test_decode_additive_rejects_on_host(lib):
    def call(**kw):
        args = dict(d_k=128, o=_fake(0x900000), S=_fake(0x100000))
        args.update(kw)
        return lib.kda_decode_step_additive(_fake(0x10000), _fake(0x20000), _fake(0x30000),
                                            _fake(0x40000), _fake(0x50000), args["S"], 2, 2,
                                            args["d_k"], 128, 0, args["o"], None)
    assert call(d_k=96) == 2
    assert call(o=None) == 1
    assert call(o=_fake(0x40000)) == 1  # o overlaps alpha


def test_backward_gates_host_checks(lib):
    f = lib.kda_backward_gates_workspace_size
    base = lib.kda_backward_workspace_size(2, 64, 2, 128, 128, 64)
    assert f(2, 64, 2, 128, 128, 64, 0) == base
    # the other layouts add the gate per channel and its gradient, fp32 each
    for gate in (1, 2):
        assert f(2, 64, 2, 128, 128, 64, gate) >= base + 2 * 64 * 2 * 128 * 4
    assert f(2, 64, 2, 128, 128, 64, 7) == 0
    M = 0x1000000

    def call(gate, ws_bytes=None, dgate=_fake(11 * M)):
        if ws_bytes is None:
            ws_bytes = f(2, 64, 2, 128, 128, 64, gate if gate in (0, 1, 2) else 0)
        return lib.kda_backward_gates(_fake(1 * M), _fake(2 * M), _fake(3 * M), _fake(4 * M),
                                      gate, _fake(5 * M), None, _fake(6 * M), 2, 64, 2, 128,
                                      128, 0, 64, _fake(7 * M), None, _fake(8 * M),
                                      _fake(9 * M), _fake(10 * M), dgate, _fake(12 * M), None,
                                      _fake(13 * M), ws_bytes, None)
    assert call(7) == 1                                  # unknown layout
    assert call(1, ws_bytes=base) == 1                   # too small for the expanded gate
    assert call(2, dgate=_fake(4 * M + 1024)) == 1       # d/d log alpha overlaps the gate
