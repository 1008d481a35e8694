"""The stored small case in ``tests/golden/kda_small.json``.

Its outputs were written by ``tests/golden/make_golden.py`` from the oracle
alone (the fp64 recurrence of "Kimi (AI)", section "Kimi Delta Attention
(KDA)").  Here, on the CPU, it anchors the oracle's arithmetic: a later
change that moves any output fails.  The GPU side (the fp32 CUDA-core chunk
kernel against the stored values) is in ``test_workloads_gpu.py``.
"""
import ast
import json
import os

import numpy as np

import oracle
import parity

HERE = os.path.dirname(os.path.abspath(__file__))
FIXTURE = os.path.join(HERE, "golden", "kda_small.json")
GENERATOR = os.path.join(HERE, "golden", "make_golden.py")


def load_fixture():
    with open(FIXTURE) as f:
        doc = json.load(f)
    x = {k: np.asarray(v, dtype=np.int32 if k == "cu_seqlens" else np.float64)
         for k, v in doc["inputs"].items()}
    y = {k: np.asarray(v, dtype=np.float64) for k, v in doc["outputs"].items()}
    return doc, x, y


def test_fixture_shapes_and_fp32_inputs():
    doc, x, y = load_fixture()
    sh = doc["shape"]
    T, N = sum(sh["lengths"]), len(sh["lengths"])
    H, d_k, d_v = sh["H"], sh["d_k"], sh["d_v"]
    assert x["q"].shape == x["k"].shape == (T, H, d_k)
    assert x["v"].shape == x["alpha"].shape == (T, H, d_v)
    assert x["beta"].shape == (T, H) and x["S0"].shape == (N, H, d_v, d_k)
    assert x["cu_seqlens"].tolist() == [0] + np.cumsum(sh["lengths"]).tolist()
    assert y["o"].shape == (T, H, d_v) and y["S_T"].shape == (N, H, d_v, d_k)
    for name in ("q", "k", "v", "alpha", "beta", "S0"):
        assert np.array_equal(x[name], x[name].astype(np.float32).astype(np.float64)), name


def test_generator_uses_only_the_oracle():
    """Stored expected values may come from the oracle alone."""
    tree = ast.parse(open(GENERATOR).read())
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            mods.add((node.module or "").split(".")[0])
    assert mods <= {"__future__", "json", "os", "sys", "numpy", "oracle"}, mods


def test_oracle_reproduces_the_fixture():
    _, x, y = load_fixture()
    o, S_T = oracle.prefill(x["q"].astype(np.float32), x["k"].astype(np.float32),
                            x["v"].astype(np.float32), x["alpha"].astype(np.float32),
                            x["beta"].astype(np.float32), x["S0"], x["cu_seqlens"])
    assert parity.rel(o, y["o"]) <= 1e-14
    assert parity.rel(S_T, y["S_T"]) <= 1e-14
