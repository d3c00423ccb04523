"""The fp64 Mamba-2 (SSD) oracle against its pins, and mutants of it that
the pins must catch (CPU only).  See ``ssd_pins.py`` for the pins."""

import os

import numpy as np
import pytest

import ssd_pins
from oracle import ssd

SRC = os.path.join(os.path.dirname(ssd.__file__), "ssd_oracle.c")


@pytest.fixture(scope="module")
def lib():
    return ssd.load()


@pytest.mark.parametrize("pin", ssd_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_ssd_oracle_pin(pin, lib):
    pin(lib)


def test_ssd_oracle_thread_count_independent(lib):
    rng = np.random.default_rng(7)
    case, dy = ssd_pins.make_case(rng, Bt=3, T=20, H=4, G=2, N=5, P=3)
    args = [case[n] for n in ssd_pins.NAMES]
    a = ssd.ssd_forward_backward(*args, dy, threads=1, lib=lib)
    b = ssd.ssd_forward_backward(*args, dy, threads=0, lib=lib)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_ssd_oracle_shapes_and_empty(lib):
    z4 = np.zeros((1, 0, 2, 3))
    o = ssd.ssd_forward_backward(z4, np.zeros((1, 0, 2)), -np.ones(2), np.zeros((1, 0, 1, 4)),
                                 np.zeros((1, 0, 1, 4)), np.ones(2), z4, lib=lib)
    assert o["y"].shape == (1, 0, 2, 3) and np.all(o["dA"] == 0) and np.all(o["dD"] == 0)
    with pytest.raises(ValueError):  # 3 heads do not split into 2 groups
        ssd.ssd_forward(np.zeros((1, 2, 3, 2)), np.zeros((1, 2, 3)), -np.ones(3),
                        np.zeros((1, 2, 2, 4)), np.zeros((1, 2, 2, 4)), np.ones(3), lib=lib)


MUTANTS = {
    "carry_without_decay": ("+ a_next * gs[n * P + p];", "+ gs[n * P + p];"),
    "dx_missing_dt": ("dxt[p] = d * acc + Dh * dyt[p];", "dxt[p] = acc + Dh * dyt[p];"),
    "dx_missing_skip": ("dxt[p] = d * acc + Dh * dyt[p];", "dxt[p] = d * acc;"),
    "db_missing_dt": ("dBt[n] = d * accb;", "dBt[n] = accb;"),
    "dc_uses_previous_state": ("accc += ht[n * P + p] * dyt[p];",
                               "accc += (hp ? hp[n * P + p] : 0.0) * dyt[p];"),
    "ddt_drops_decay_term": ("dd += gs[n * P + p] * (Ah * a * prev + Bt_[n] * xt[p]);",
                             "dd += gs[n * P + p] * (Bt_[n] * xt[p]);"),
    "da_sign_flip": ("sumA += da;", "sumA -= da;"),
    "forward_decay_off_by_one": ("const double a = exp(d * A);", "const double a = exp(A);"),
    "group_index_wrong": ("scan_forward(x, dt, A[h], Bm, Cm, D[h], b, h, h / hpg,",
                          "scan_forward(x, dt, A[h], Bm, Cm, D[h], b, h, 0,"),
    "groups_not_summed": ("for (long h = g * hpg; h < (g + 1) * hpg; ++h) {\n            sb",
                          "for (long h = g * hpg; h < g * hpg + 1; ++h) {\n            sb"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_ssd_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation anchor not found exactly once: %r" % old
    src = tmp_path / ("ssd_mutant_%s.c" % name)
    src.write_text(text.replace(old, new))
    lib = ssd.load(ssd.build(force=True, src=str(src), out=str(tmp_path / "libssdmut.so")))
    failures = []
    for pin in ssd_pins.ALL_PINS:
        if pin is ssd_pins.pin_finite_differences:
            continue  # the cheaper pins already see these mutants
        try:
            pin(lib)
        except (AssertionError, FloatingPointError) as e:
            failures.append("%s: %s" % (pin.__name__, e))
    assert failures, "mutant %s passed every pin" % name
