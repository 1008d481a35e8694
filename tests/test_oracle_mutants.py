"""Plant plausible mistakes in a copy of the oracle; each must trip a pin.

Each mutant is a text substitution applied to a temporary copy of
``oracle/kda_oracle.c``, compiled with the oracle's own flags into a scratch
directory.  The committed oracle is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

MUTANTS = {
    # forget gate applied to the key side (columns) instead of value channels (rows)
    "alpha_on_columns": ("row[c] = a * row[c];",
                         "row[c] = (double)alpha[th * d_v + (c % d_v)] * row[c];"),
    # predict from the undecayed state S_{t-1} instead of S~_t
    "predict_before_decay": ("vpred[r] = acc;",
                             "vpred[r] = acc / (double)alpha[th * d_v + r];"),
    # wrong sign of the correction
    "update_sign": ("row[c] = row[c] + b * err * kt[c];",
                    "row[c] = row[c] - b * err * kt[c];"),
    # beta dropped from memory updating
    "drop_beta": ("row[c] = row[c] + b * err * kt[c];",
                  "row[c] = row[c] + err * kt[c];"),
    # prediction term dropped: plain decayed linear attention
    "drop_prediction": ("- vpred[r];", "- 0.0 * vpred[r];"),
    # output read with the key instead of the query
    "output_uses_key": ("acc += row[c] * qt[c];", "acc += row[c] * kt[c];"),
    # outer product with q instead of k in the write
    "write_with_query": ("row[c] = row[c] + b * err * kt[c];",
                         "row[c] = row[c] + b * err * qt[c];"),
    # off-by-one: beta read from the previous token
    "beta_index": ("const double b = (double)beta[th];",
                   "const double b = (double)beta[th > H ? th - H : th];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in the oracle"
    mutant_src = tmp_path / "kda_oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib_path = oracle.build(str(mutant_src), str(tmp_path / "libmutant.so"),
                            extra_flags=("-Wno-unused-variable",))
    lib = oracle.load(lib_path)
    failing = oracle_pins.failing_pins(lib)
    assert failing, f"mutant {name} passed every pin"


def test_unmutated_copy_passes_all(tmp_path):
    mutant_src = tmp_path / "kda_oracle_copy.c"
    mutant_src.write_text(open(SRC).read())
    lib = oracle.load(oracle.build(str(mutant_src), str(tmp_path / "libcopy.so"),
                                   extra_flags=("-Wno-unused-variable",)))
    assert oracle_pins.failing_pins(lib) == []
