"""Gate the gate: every gate input makes some plausible variant of the rules
fail, and the oracle follows the rules on it.

"Verification -- why you can trust the numbers", section "Layer 1": the B2B
chain gate hunts for inputs where the old and new quantize specs disagree and
requires the new one.  The GPU side of these cases is in
``test_gpu_parity.py``.
"""
import numpy as np
import pytest

import gate_cases as G


@pytest.mark.parametrize("case", G.row_cases(), ids=lambda c: c.name)
def test_row_case_is_not_vacuous_and_oracle_follows_spec(orc, case):
    var_q, var_scale = G.variant_of(case)
    assert (var_q, var_scale) != (case.spec_q, case.spec_scale), case.name
    Q, sc, iv, st = orc.quantize_rows(case.row[None, :])
    assert st == 0
    assert list(Q[0].astype(int)) == case.spec_q
    assert G.f2b(sc[0]) == case.spec_scale


@pytest.mark.parametrize("case", G.epi_cases(), ids=lambda c: c.name)
def test_epi_case_is_not_vacuous_and_oracle_follows_spec(orc, case):
    assert case.spec != case.variant
    c = orc.epi(case.s, float(G.b2f(case.a)), float(G.b2f(case.b)))
    assert G.f2b(np.float32(c)) == case.spec
