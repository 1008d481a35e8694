"""The Attention Residuals oracle against its pins, and planted mistakes
against the pins (CPU only)."""
import importlib.util

import numpy as np
import pytest

import oracle_attnres_pins as pins
from oracle import attnres

SRC = attnres.__file__

MUTANTS = {
    # normalised over tokens instead of over the sources
    "softmax_axis": ("w = w / w.sum(axis=1, keepdims=True)", "w = w / w.sum(axis=0, keepdims=True)"),
    # the scale dropped
    "no_scale": ("logits = scale * np.einsum", "logits = np.einsum"),
    # a block represented by its last output instead of its sum
    "block_last_not_sum": ("summaries = [sum(outs[j] for j in blk) for blk in blocks]",
                           "summaries = [outs[blk[-1]] for blk in blocks]"),
    # the current block's partial sum joined one layer late
    "partial_late": ("            if i >= 1:\n", "            if i >= 2:\n"),
    # the previous layer's output left out of the running sum
    "drop_last_output": ("P = P + np.asarray(h_last, dtype=np.float64)", "P = P + 0.0"),
    # values weighted by the logits instead of the softmax weights
    "weights_unnormalised": ("w = np.exp(logits)", "w = np.exp(logits) * 0 + logits"),
}


def _load(path):
    spec = importlib.util.spec_from_file_location("attnres_copy", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(pins.PINS))
def test_pin(name):
    fn, tol = pins.PINS[name]
    err = fn(attnres)
    assert np.isfinite(err) and err <= tol, f"{name}: {err:.3e} > {tol:.1e}"


# a planted mistake may well produce non-finite values on the way
@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / "attnres_mutant.py"
    path.write_text(src.replace(old, new))
    failing = pins.failing_pins(_load(str(path)))
    assert len(failing) >= 2, f"mutant {name} tripped only {failing}"


def test_unmutated_copy_passes(tmp_path):
    path = tmp_path / "attnres_copy.py"
    path.write_text(open(SRC).read())
    assert pins.failing_pins(_load(str(path))) == []
