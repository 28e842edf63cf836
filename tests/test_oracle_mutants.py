"""The pins must reject planted mistakes (CPU only).

Each mutant (tests/mutants.py) re-implements the recurrence with one plausible mistake. A pin
suite that let any of them through would not be pinning the oracle; this test fails in that case.
The unmodified numpy re-implementation must pass every pin, so the mutants fail for their
mistake and not for their plumbing.
"""
import pytest

import oracle
from tests import mutants, pins


def _fails_some_pin(run):
    failed = []
    for name, pin in pins.ALL_PINS.items():
        err = pin(run)
        if not (err <= max(pins.PIN_TOL[name], 1e-9)):
            failed.append(name)
    return failed


def test_clean_reimplementation_passes_all_pins():
    run = lambda *a: mutants.recurrence(*a, mistake=None)
    assert _fails_some_pin(run) == []


@pytest.mark.parametrize("mistake", mutants.RECURRENT_MISTAKES)
def test_recurrent_mistake_is_caught(mistake):
    run = lambda *a: mutants.recurrence(*a, mistake=mistake)
    assert _fails_some_pin(run), f"no pin rejects the planted mistake {mistake!r}"


@pytest.mark.parametrize("mistake", mutants.CHUNKED_MISTAKES)
def test_chunked_mistake_is_caught(mistake):
    """A chunked form with a planted mistake disagrees with the pinned recurrent oracle."""
    q, k, v, g, b, w, S0 = pins.rand_problem(31, B=1, T=13, Hk=1, Hv=2, dk=5, dv=4)
    o_ref, s_ref = oracle.run(q, k, v, g, b, w, S0, form="recurrent")
    o, s = mutants.chunked(q, k, v, g, b, w, S0, C=4, mistake=mistake)
    assert max(pins.rel(o, o_ref), pins.rel(s, s_ref)) > 1e-6
    o, s = mutants.chunked(q, k, v, g, b, w, S0, C=4, mistake=None)
    assert max(pins.rel(o, o_ref), pins.rel(s, s_ref)) < 1e-12
