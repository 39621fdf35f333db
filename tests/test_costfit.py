"""Host-side checks of the InfiniPipe Eq. (1) cost model (no GPU): the model's
terms of a call, the fitting grid, the non-negative relative least squares
that turns call times into (alpha1, alpha2, beta1), and the committed fit."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import chunked_causal_attention_gb300 as cca  # noqa: E402
from chunked_causal_attention_gb300 import costfit  # noqa: E402


def test_model_terms_by_hand():
    # a slice of 100 tokens after 50 of context: (150^2 - 50^2) = 20000 pairs-term, 100 tokens;
    # a short sequence of 10 tokens with no context: 100 and 10
    assert costfit.model_terms([(50, 150, 0, 0), (200, 210, 200, 0)]) == (20000 + 100, 110)
    assert costfit.model_terms([]) == (0, 0)


def test_fit_grid_is_valid_for_the_streamed_calls():
    """Every call of the grid lies in the packed buffer and is accepted by the
    library's chunk-streamed backward (disjoint key ranges) and forward."""
    shape = cca.make_shape(1, costfit.H, costfit.T_BUF, costfit.D, costfit.T_BUF * costfit.H * costfit.D,
                           costfit.H * costfit.D, costfit.D, costfit.D ** -0.5)
    calls = costfit.fit_calls()
    assert len(calls) >= 20
    for c in calls:
        assert all(0 <= cb <= qb < qe <= costfit.T_BUF for qb, qe, cb, _ in c)
        assert cca.attn_workspace_size(shape, c, cca.PASS_BWD_CHUNK) > 0
        assert cca.attn_workspace_size(shape, c, cca.PASS_FWD) > 0
    # the grid spans both terms: long contexts (quadratic) and many short sequences (linear, per call)
    terms = [costfit.model_terms(c) for c in calls]
    assert max(q / l for q, l in terms) > 100 * min(q / l for q, l in terms)


def test_fit_recovers_exact_constants():
    """Times that follow the model exactly give back its constants."""
    a1, a2, b1 = 3.1e-10, 2.0e-5, 0.05
    rows = [[q, l, 1.0] for q, l in (costfit.model_terms(c) for c in costfit.fit_calls())]
    ms = [a1 * q + a2 * l + b1 for q, l, _ in rows]
    f1, f2, f3, rel = costfit.fit_constants(rows, ms)
    assert f1 == pytest.approx(a1, rel=1e-6) and f2 == pytest.approx(a2, rel=1e-6)
    assert f3 == pytest.approx(b1, rel=1e-5)
    assert float(rel.max()) < 1e-6


def test_fit_keeps_constants_non_negative():
    """A launch overhead that the data contradict is fitted as 0, not negative."""
    a1 = 3.0e-10
    rows = [[q, l, 1.0] for q, l in (costfit.model_terms(c) for c in costfit.fit_calls())]
    ms = [a1 * q - 1e-3 * (q > 0) + 1e-6 * l for q, l, _ in rows]
    ms = [max(m, 1e-4) for m in ms]
    f1, f2, f3, _ = costfit.fit_constants(rows, ms)
    assert min(f1, f2, f3) >= 0.0 and f1 > 0


def test_committed_fit():
    """The committed GB300 fit has positive quadratic and per-call terms and
    describes its own points within the error it records."""
    import json
    with open(costfit.COST_PATH) as f:
        c = json.load(f)
    a1, a2, b1 = costfit.load_cost()
    assert a1 > 0 and a2 >= 0 and b1 >= 0
    rows = [[p["quad"], p["tokens"], 1.0] for p in c["points"]]
    ms = [p["fwd_ms"] + p["bwd_ms"] for p in c["points"]]
    pred = [a1 * q + a2 * l + b1 for q, l, _ in rows]
    rel = [abs(p - m) / m for p, m in zip(pred, ms)]
    assert max(rel) == pytest.approx(c["max_rel_err"], rel=1e-6)
    # and the fit of its own points gives back the committed constants
    f1, f2, f3, _ = costfit.fit_constants(rows, ms)
    assert (f1, f2, f3) == pytest.approx((a1, a2, b1), rel=1e-9, abs=1e-15)
