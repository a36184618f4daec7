"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
from _pins import ALL_PINS, rand_inputs, rel


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.prefill)


def test_decode_is_one_token_prefill():
    # a decode step is the recurrence applied to a single token per sequence
    rng = np.random.default_rng(8)
    q, k, v, g, b = rand_inputs(rng, 5, 3, 4, 4)
    S = rng.standard_normal((5, 3, 4, 4))
    o, Sn = oracle.decode(q, k, v, g, b, S)
    for n in range(5):
        On, Sfn = oracle.prefill(q[n:n + 1], k[n:n + 1], v[n:n + 1], g[n:n + 1], b[n:n + 1],
                                 S0=S[n:n + 1])
        assert np.array_equal(o[n], On[0])
        assert np.array_equal(Sn[n], Sfn[0])


def test_head_subset_matches_full_run():
    rng = np.random.default_rng(9)
    q, k, v, g, b = rand_inputs(rng, 20, 4, 6, 5)
    S0 = rng.standard_normal((2, 4, 6, 5))
    cu = [0, 8, 20]
    O, Sf = oracle.prefill(q, k, v, g, b, cu_seqlens=cu, S0=S0)
    Os, Sfs = oracle.prefill(q, k, v, g, b, cu_seqlens=cu, S0=S0, heads=(1, 3))
    assert np.array_equal(Os, O[:, 1:3])
    assert np.array_equal(Sfs, Sf[:, 1:3])


def test_threads_do_not_change_results():
    rng = np.random.default_rng(10)
    q, k, v, g, b = rand_inputs(rng, 40, 6, 8, 8)
    O1, S1 = oracle.prefill(q, k, v, g, b, n_threads=1)
    O4, S4 = oracle.prefill(q, k, v, g, b, n_threads=4)
    assert np.array_equal(O1, O4) and np.array_equal(S1, S4)


def test_bad_arguments_are_rejected():
    rng = np.random.default_rng(11)
    q, k, v, g, b = rand_inputs(rng, 4, 1, 2, 2)
    with pytest.raises(ValueError):
        oracle.prefill(q, k, v, g, b, cu_seqlens=[0, 3, 2])


def test_chunk_form_flags_wrong_masks():
    """The chunk-form cross-check is itself sensitive: an exclusive M_qk mask
    (o_t read before the write) or an exclusive cumsum moves it off the token
    loop by far more than rounding."""
    import scipy.linalg
    rng = np.random.default_rng(12)
    q, k, v, g, b = rand_inputs(rng, 8, 1, 4, 3)
    O, _ = oracle.prefill(q, k, v, g, b)
    Q, K, V, G, B = q[:, 0], k[:, 0], v[:, 0], g[:, 0], b[:, 0]
    a = np.exp(np.cumsum(G, axis=0))
    Kd, Qd, Ki = a * K, a * Q, K / a
    L = np.tril(B[:, None] * (Kd @ Ki.T), -1)
    INV = scipy.linalg.solve_triangular(np.eye(8) + L, np.eye(8), lower=True)
    U = INV @ (B[:, None] * V)
    good = np.tril(Qd @ Ki.T) @ U
    bad = np.tril(Qd @ Ki.T, -1) @ U
    assert rel(good, O[:, 0]) < 1e-12
    assert rel(bad, O[:, 0]) > 1e-2
