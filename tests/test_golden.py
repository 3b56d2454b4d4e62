"""Closed-form cases (``tests/golden/closed_forms.json``): the fixture is what its script
writes, and the oracle reproduces every hand-derived output (CPU)."""
import dataclasses

import numpy as np
import pytest

import oracle
from tests.golden import PATH, load_cases
from tests.golden import make_golden

CASES = load_cases()


def test_fixture_is_what_the_script_writes():
    with open(PATH) as f:
        assert f.read() == make_golden.render()


def test_cases_cover_both_paths_and_dtypes():
    kinds = {(c["kind"], c["fp8"]) for _, _, _, _, c in CASES}
    assert kinds == {("prefill", False), ("prefill", True), ("decode", False), ("decode", True)}


@pytest.mark.parametrize("name,inp,O,L", [(n, i, o, l) for n, i, o, l, _ in CASES], ids=[c[0] for c in CASES])
def test_oracle_reproduces_closed_form(name, inp, O, L):
    run = oracle.mla_prefill if hasattr(inp, "S") else oracle.mla_decode
    O_ref, L_ref = run(inp)
    assert O_ref.shape == O.shape and L_ref.shape == L.shape
    tol = 1e-12 * np.maximum(1.0, np.abs(O))
    assert (np.abs(O_ref - O) <= tol).all(), np.argwhere(np.abs(O_ref - O) > tol)[:5]
    assert (np.isneginf(L_ref) == np.isneginf(L)).all()
    fin = np.isfinite(L)
    assert np.abs(L_ref[fin] - L[fin]).max() <= 1e-12


def test_a_dropped_rope_term_changes_the_dominant_case():
    # the dominant key's score is 150 from the nope part and 50 from the rope part: without
    # the rope keys the oracle must give LSE 150 for the rows that see it, not 200
    name, inp, O, L, _ = next(c for c in CASES if c[0] == "prefill_dominant_key")
    _, L_ref = oracle.mla_prefill(dataclasses.replace(inp, k_rope=np.zeros_like(inp.k_rope)))
    assert np.allclose(L_ref[0, 0, 3:], 150.0) and not np.allclose(L_ref[0, 0, 3:], L[0, 0, 3:])
