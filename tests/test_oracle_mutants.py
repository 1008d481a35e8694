"""Plant plausible mistakes in a copy of the oracle; each must trip a pin.

Each mutant is a text substitution applied to a temporary copy of
``oracle/kda_oracle.c``, compiled with the oracle's own flags into a scratch
directory.  The committed oracle is never modified.
"""
import os

import pytest

import numpy as np

import oracle
import oracle_backward_pins
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
    # the additive update keeps the prediction term
    "additive_predicts": ("for (int32_t r = 0; r < d_v && !additive; ++r) {",
                          "for (int32_t r = 0; r < d_v; ++r) {"),
}


# Mistakes in the reverse mode (kda_oracle_backward); each must trip a
# reverse-mode pin.
BACKWARD_MUTANTS = {
    # wrong sign of the S~^T g term of dk
    "dk_sign": ("dk[th * d_k + c] = b * (du - sg);", "dk[th * d_k + c] = b * (du + sg);"),
    # dalpha against the state after the update instead of S_{t-1}
    "dalpha_wrong_state": ("da += Dr[c] * Pr[c];", "da += Dr[c] * S_t[(int64_t)r * d_k + c];"),
    # state gradient not decayed on its way back
    "no_decay_of_gradient": ("for (int32_t c = 0; c < d_k; ++c) Dr[c] = w->at[r] * Dr[c];",
                             "for (int32_t c = 0; c < d_k; ++c) Dr[c] = 1.0 * Dr[c];"),
    # dq read from S_{t-1} instead of S_t
    "dq_wrong_state": ("acc += S_t[(int64_t)r * d_k + c] * w->dot[r];",
                       "acc += S_prev[(int64_t)r * d_k + c] * w->dot[r];"),
    # dbeta with v in place of the prediction error
    "dbeta_uses_v": ("db += w->u[r] * acc;", "db += w->vt[r] * acc;"),
    # dv without beta
    "dv_no_beta": ("dv[th * d_v + r] = b * acc;", "dv[th * d_v + r] = acc;"),
    # the output's gradient added with k instead of q
    "output_gradient_with_key": ("Dr[c] += w->dot[r] * w->qt[c];",
                                 "Dr[c] += w->dot[r] * w->kt[c];"),
    # wrong sign of the projector term of dS~
    "projector_sign": ("Dr[c] = Dr[c] - b * w->g[r] * w->kt[c];",
                       "Dr[c] = Dr[c] + b * w->g[r] * w->kt[c];"),
}


def _build_mutant(tmp_path, old, new, name):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in the oracle"
    mutant_src = tmp_path / "kda_oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib_path = oracle.build(str(mutant_src), str(tmp_path / "libmutant.so"),
                            extra_flags=("-Wno-unused-variable",))
    return oracle.load(lib_path)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, old, new, name)
    failing = oracle_pins.failing_pins(lib)
    # two independent pins per mistake, so that no single pin carries one alone
    assert len(failing) >= 2, f"mutant {name} tripped only {failing}"


@pytest.mark.parametrize("name", sorted(BACKWARD_MUTANTS))
def test_backward_mutant_is_caught(tmp_path, name):
    old, new = BACKWARD_MUTANTS[name]
    lib = _build_mutant(tmp_path, old, new, name)
    failing = oracle_backward_pins.failing_pins(lib)
    assert len(failing) >= 2, f"backward mutant {name} tripped only {failing}"


def test_backward_tape_segment_does_not_change_results(tmp_path):
    """The tape keeps every OR_SEG-th state and re-runs the same fp64 step in
    between: a different segment length must give the same bits."""
    lib = _build_mutant(tmp_path, "#define OR_SEG 64", "#define OR_SEG 5", "segment")
    rng = np.random.default_rng(31)
    q, k, v, alpha, beta, S0, cu = oracle_pins._random_problem(rng, [70, 3, 0, 12], 2, 8, 4)
    dO = rng.standard_normal((q.shape[0], 2, 4))
    a = oracle.backward(q, k, v, alpha, beta, S0, cu, dO, None)
    b = oracle.backward(q, k, v, alpha, beta, S0, cu, dO, None, lib=lib)
    for name in a:
        assert np.array_equal(a[name], b[name]), name


def test_unmutated_copy_passes_all(tmp_path):
    mutant_src = tmp_path / "kda_oracle_copy.c"
    mutant_src.write_text(open(SRC).read())
    lib = oracle.load(oracle.build(str(mutant_src), str(tmp_path / "libcopy.so"),
                                   extra_flags=("-Wno-unused-variable",)))
    assert oracle_pins.failing_pins(lib) == []
    assert oracle_backward_pins.failing_pins(lib) == []
