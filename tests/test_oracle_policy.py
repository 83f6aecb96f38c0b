"""Pins of the oracle's step policy against the traces the pages print."""

import pytest

import oracle as O
from conftest import golden_lines


def _expand(tokens):
    out = []
    for t in tokens:
        mode, n = t.split("x")
        out += [mode] * int(n)
    return out


def test_published_traces():
    pol = O.StepPolicy()
    for row in golden_lines("step_traces.txt"):
        n = int(row[0])
        assert [O.step_mode(pol, s, n) for s in range(n)] == _expand(row[1:])


def test_first_a8_step_of_8_is_step_3():
    pol = O.StepPolicy()
    modes = [O.step_mode(pol, s, 8) for s in range(8)]
    assert modes.index("A8") == 3


def test_no_policy_runs_fully_quantized():
    for n in (1, 4, 8, 35):
        assert all(O.step_mode(None, s, n) == "A8" for s in range(n))
        assert all(O.step_mode(O.StepPolicy(enabled=False), s, n) == "A8" for s in range(n))


def test_pure_function_of_step_index():
    pol = O.StepPolicy()
    a = [O.step_mode(pol, s, 35) for s in range(35)]
    b = [O.step_mode(pol, s, 35) for s in reversed(range(35))][::-1]
    assert a == b          # cond / uncond branches query in any order


@pytest.mark.parametrize("kw,step,n", [
    (dict(schema_version=2), 0, 8),
    (dict(first_steps=-1), 0, 8),
    (dict(last_steps=-2), 0, 8),
    ({}, 8, 8),
    ({}, -1, 8),
    ({}, 0, 0),
])
def test_refusals(kw, step, n):
    with pytest.raises(O.PolicyError):
        O.step_mode(O.StepPolicy(**kw), step, n)


def test_zero_windows_all_a8():
    pol = O.StepPolicy(first_steps=0, last_steps=0)
    assert all(O.step_mode(pol, s, 8) == "A8" for s in range(8))
