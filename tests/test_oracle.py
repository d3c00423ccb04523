"""The fp64 oracle against its pins (CPU only).

See ``oracle_pins.py`` for what each pin checks and why it is independent of
the oracle's own code.
"""

import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_oracle_empty_and_bad_args(oracle_lib):
    import numpy as np
    import oracle

    z = np.zeros((1, 1, 0, 4))
    out = oracle.attention_forward_backward(z, z, z, z, True, 0.5, lib=oracle_lib)
    assert out["O"].shape == (1, 1, 0, 4) and out["L"].shape == (1, 1, 0)
    with pytest.raises(ValueError):
        oracle.attention_forward(np.zeros((1, 1, 2, 4)), np.zeros((1, 1, 3, 4)),
                                 np.zeros((1, 1, 2, 4)), False, 1.0, lib=oracle_lib)


def test_oracle_thread_count_independent(oracle_lib):
    """Each output element is written by one thread: results are bitwise equal
    for 1 thread and for all threads."""
    import numpy as np
    import oracle

    rng = np.random.default_rng(3)
    q, k, v, do = (rng.standard_normal((2, 3, 70, 16)) for _ in range(4))
    a = oracle.attention_forward_backward(q, k, v, do, True, 0.25, threads=1, lib=oracle_lib)
    b = oracle.attention_forward_backward(q, k, v, do, True, 0.25, threads=0, lib=oracle_lib)
    for name in a:
        assert np.array_equal(a[name], b[name]), name
