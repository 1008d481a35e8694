"""The oracle against what the page and mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
import oracle_backward_pins
import oracle_pins


@pytest.mark.parametrize("name", sorted(oracle_pins.PINS))
def test_pin(oracle_lib, name):
    fn, tol = oracle_pins.PINS[name]
    err = fn(oracle_lib)
    assert np.isfinite(err) and err <= tol, f"{name}: error {err:.3e} > {tol:.1e}"


def test_bf16_widening_matches_torch():
    import torch
    x = torch.randn(1000, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), x.double().numpy())


def test_rejects_bad_cu_seqlens(oracle_lib):
    q = np.zeros((4, 1, 2), np.float32)
    v = np.zeros((4, 1, 2), np.float32)
    a = np.ones((4, 1, 2), np.float32)
    b = np.zeros((4, 1), np.float32)
    for cu in ([1, 4], [0, 3, 2], [0, 5]):
        with pytest.raises(ValueError):
            oracle.prefill(q, q, v, a, b, None, np.array(cu, np.int32), lib=oracle_lib)


def test_thread_count_does_not_change_results(oracle_lib):
    rng = np.random.default_rng(11)
    q, k, v, alpha, beta, S0, cu = oracle_pins._random_problem(rng, [30, 17, 22], 3, 8, 8)
    o1, s1 = oracle.prefill(q, k, v, alpha, beta, S0, cu, nthreads=1, lib=oracle_lib)
    o4, s4 = oracle.prefill(q, k, v, alpha, beta, S0, cu, nthreads=4, lib=oracle_lib)
    assert np.array_equal(o1, o4) and np.array_equal(s1, s4)


@pytest.mark.parametrize("name", sorted(oracle_backward_pins.PINS))
def test_backward_pin(oracle_lib, name):
    fn, tol = oracle_backward_pins.PINS[name]
    err = fn(oracle_lib)
    assert np.isfinite(err) and err <= tol, f"{name}: error {err:.3e} > {tol:.1e}"


def test_backward_thread_count_does_not_change_results(oracle_lib):
    rng = np.random.default_rng(12)
    q, k, v, alpha, beta, S0, cu = oracle_pins._random_problem(rng, [30, 0, 22], 3, 8, 4)
    dO = rng.standard_normal((q.shape[0], 3, 4))
    a = oracle.backward(q, k, v, alpha, beta, S0, cu, dO, None, nthreads=1, lib=oracle_lib)
    b = oracle.backward(q, k, v, alpha, beta, S0, cu, dO, None, nthreads=4, lib=oracle_lib)
    for name in a:
        assert np.array_equal(a[name], b[name]), name


def test_backward_rejects_bad_cu_seqlens(oracle_lib):
    q = np.zeros((4, 1, 2), np.float32)
    a = np.ones((4, 1, 2), np.float32)
    b = np.zeros((4, 1), np.float32)
    dO = np.zeros((4, 1, 2))
    for cu in ([1, 4], [0, 3, 2], [0, 5]):
        with pytest.raises(ValueError):
            oracle.backward(q, q, q, a, b, None, np.array(cu, np.int32), dO, lib=oracle_lib)
