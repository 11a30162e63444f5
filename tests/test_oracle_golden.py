"""The oracle against its golden fixture, tests/golden/oracle_tiny_varlen.txt
(written from the oracle itself by tests/golden/make_golden.py; the pages
print no worked example of this computation).  A regression pin: the oracle's
independent pins are the finite-difference, closed-form and invariant tests;
this one makes any later change to its arithmetic a deliberate one, made
with a regenerated fixture.  The tolerance allows for fp64 contraction
differences between compilers and machines only."""
import importlib.util
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _make_golden():
    spec = importlib.util.spec_from_file_location(
        "make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_oracle_matches_golden_fixture():
    mg = _make_golden()
    oracle.build()
    got = mg.oracle_grads(mg.case())
    ref = mg.read_fixture()
    assert set(ref) == set(mg.KEYS)
    for k in mg.KEYS:
        assert got[k].shape == ref[k].shape, k
        np.testing.assert_allclose(got[k], ref[k], rtol=1e-10, atol=1e-13, err_msg=k)


def test_fixture_holds_the_empty_sequence_pass_through():
    # the middle sequence has no tokens: its dh0 is its dh_T, exactly
    mg = _make_golden()
    x = mg.case()
    ref = mg.read_fixture()
    np.testing.assert_array_equal(ref["dh0"][1], x["dhT"][1].double().numpy())
