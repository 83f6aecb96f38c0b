"""The C ABI's fail-closed diffusion_step_policy parser against the oracle's
independent parser (Python's json module plus the same refusal rules), on the
published policy and on every way of getting it wrong that the pages list."""

import itertools
import json

import pytest

import oracle as O


@pytest.fixture(scope="module")
def B():
    from w8a16_linear_gb300 import build as bld
    bld.build()
    from w8a16_linear_gb300 import binding
    return binding


PUBLISHED = {"schema_version": 1, "type": "first_last_n", "index_space": "scheduler_step",
             "default_mode": "w8a8", "overlap": "w8a16", "first_steps": 3, "last_steps": 3,
             "reasoner": "a16"}


def _both(B, text):
    """(ok, policy tuple, reasoner) from the C parser and from the oracle."""
    try:
        pol, rs = B.step_policy_parse(text)
        c = (True, (pol.enabled, pol.first_steps, pol.last_steps) if pol.enabled else (0,),
             {None: None, B.MODE_A16: "A16", B.MODE_A8: "A8"}[rs])
    except B.W8Error as e:
        assert e.status == 7, e
        c = (False, None, None)
    try:
        opol, ors = O.parse_policy(text)
        o = (True, (1, opol.first_steps, opol.last_steps) if opol.enabled else (0,), ors)
    except O.PolicyError:
        o = (False, None, None)
    return c, o


def _variants():
    yield json.dumps(PUBLISHED), True
    yield "null", True
    yield "  null \n", True
    yield json.dumps(dict(PUBLISHED, first_steps=0, last_steps=0, reasoner="a8")), True
    yield json.dumps(dict(PUBLISHED, first_steps=7, last_steps=1)), True
    for k in PUBLISHED:                                          # missing field
        d = dict(PUBLISHED)
        del d[k]
        yield json.dumps(d), False
    yield json.dumps(dict(PUBLISHED, extra=1)), False            # unknown field
    for k, bad in [("schema_version", 2), ("schema_version", 0), ("type", "every_n"),
                   ("index_space", "sigma"), ("default_mode", "w8a16"), ("overlap", "w8a8"),
                   ("reasoner", "a4"), ("first_steps", -1), ("last_steps", -3),
                   ("first_steps", 1.5), ("first_steps", "3"), ("schema_version", True),
                   ("type", None), ("first_steps", [3]), ("overlap", {"a": 1}),
                   ("last_steps", 2 ** 31), ("schema_version", 1.0)]:
        yield json.dumps(dict(PUBLISHED, **{k: bad})), False
    base = json.dumps(PUBLISHED)
    yield base[:-1] + ', "first_steps": 3}', False               # duplicate key
    yield base + " x", False                                     # trailing text
    yield "[" + base + "]", False
    yield "", False
    yield "{}", False
    yield base.replace('"first_last_n"', '"first_last\\u005fn"'), False   # escapes refused
    yield base.replace(": 3,", ": 03,", 1), False                # leading zero
    yield base.replace(": 3,", ": 3e0,", 1), False               # not an integer
    yield "nul", False
    yield "NaN", False


def test_c_parser_matches_oracle(B):
    n = 0
    for text, accept in _variants():
        c, o = _both(B, text)
        assert c == o, (text, c, o)
        assert c[0] == accept, (text, c)
        n += 1
    assert n > 40


def test_published_policy_gives_published_traces(B):
    pol, reasoner = B.step_policy_parse(json.dumps(PUBLISHED))
    assert reasoner == B.MODE_A16
    modes = [B.step_policy_dispatch(pol, s, 8) for s in range(8)]
    assert modes == [1, 1, 1, 0, 0, 1, 1, 1]
    pol0, r0 = B.step_policy_parse("null")
    assert r0 is None and all(B.step_policy_dispatch(pol0, s, 8) == 0 for s in range(8))


def test_key_order_is_free(B):
    for perm in itertools.islice(itertools.permutations(PUBLISHED), 0, 40, 7):
        text = json.dumps({k: PUBLISHED[k] for k in perm})
        pol, _ = B.step_policy_parse(text)
        assert (pol.enabled, pol.first_steps, pol.last_steps) == (1, 3, 3)
