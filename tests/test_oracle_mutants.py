"""Every pin set must catch plausible mistakes planted in a copy of the oracle.

Each mutant is the oracle's C source with one textual change (a dropped term,
a flipped sign, a wrong index or mask), compiled on the CPU into a temporary
library.  The committed oracle is never modified.  A mutant that passes every
pin would mean the pins cannot see that class of mistake.
"""

import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "dq_missing_scale": ("for (long c = 0; c < d; ++c) dQi[c] *= scale;", ""),
    "dk_missing_scale": ("for (long c = 0; c < d; ++c) dKj[c] *= scale;", ""),
    "ds_sign_flip_in_dq": ("double ds = p * (dp - Di);", "double ds = p * (dp + Di);"),
    "ds_drops_D_in_dkdv": ("double ds = p * (dp - Dh[i]);", "double ds = p * dp;"),
    "lse_without_log_sum": ("double Li = m + log(l);", "double Li = m;"),
    "dv_uses_ds": ("dVj[c] += p * dOi[c];", "dVj[c] += ds * dOi[c];"),
    "dkdv_ignores_causal": ("long i0 = causal ? j : 0;", "long i0 = 0;"),
    "causal_excludes_diagonal": ("return causal ? i + 1 : N;", "return causal ? (i > 0 ? i : 1) : N;"),
    "dk_uses_k_not_q": ("dKj[c] += ds * qi[c];", "dKj[c] += ds * kj[c];"),
    "window_one_key_too_many": ("? i - window + 1 : 0;", "? i - window : 0;"),
    "doc_start_one_early": ("if (mk->causal && mk->doc && mk->doc[i] > lo) lo = mk->doc[i];",
                            "if (mk->causal && mk->doc && mk->doc[i] - 1 > lo) lo = mk->doc[i] - 1;"),
    "dkdv_ignores_documents": ("if (row_start(i, mk) > j) continue;", ""),
    "sampler_ignores_documents": ("const Mask mk = {causal, window, doc};",
                                  "const Mask mk = {causal, window, NULL};"),
    "sampler_ignores_window": ("const Mask mk = {causal, window, doc};",
                               "const Mask mk = {causal, 0, doc};"),
    "budget_vk_uses_k": ("vKj[c] += dsv * dsv * qrow[c] * qrow[c];",
                         "vKj[c] += dsv * dsv * krow[c] * krow[c];"),
    "budget_vp_not_squared": ("vPj[c] += prob * prob * dorow[c] * dorow[c];",
                              "vPj[c] += prob * dorow[c] * dorow[c];"),
    "D_uses_wrong_row": ("if (dOh && Di_out) *Di_out = dot(dOh + i * d, Oi, d);",
                         "if (dOh && Di_out) *Di_out = dot(dOh + (N - 1 - i) * d, Oi, d);"),
}


def _pins_pass(lib):
    failures = []
    for pin in oracle_pins.ALL_PINS:
        if pin is oracle_pins.pin_finite_differences:
            continue  # costly and the cheaper pins already see these mutants
        try:
            pin(lib)
        except (AssertionError, FloatingPointError) as e:
            failures.append("%s: %s" % (pin.__name__, e))
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation anchor not found exactly once: %r" % old
    src = tmp_path / ("mutant_%s.c" % name)
    src.write_text(text.replace(old, new))
    lib_path = oracle.build(force=True, src=str(src), out=str(tmp_path / "libmut.so"))
    lib = oracle.load(lib_path)
    failures = _pins_pass(lib)
    assert failures, "mutant %s passed every pin" % name
