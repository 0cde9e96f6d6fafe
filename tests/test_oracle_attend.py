"""Pins of the oracle's sparse attention (reading R13: absorbed latent attention over the
selected rows; "Layerwise and Sparse KV Cache Offloading Design", section 4, Decode step 7).

The pins come from outside the oracle: hand-derived cases (tests/golden/attend_cases.txt),
special cases with a closed form (one row, equal rows, zero scale = the plain mean, a dominant
score = that row), and invariances (order of the list, pads, a common shift of every score).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "attend_cases.txt")


def bf16_bits(x):
    """float -> bf16 bits, round to nearest even (the test's own conversion)."""
    a = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((a + 0x7FFF + ((a >> 16) & 1)) >> 16) & 0xFFFF
    return r.astype(np.uint16)


def bf16_vals(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _num(tok):
    tok = tok.strip()
    if tok.startswith("ln"):
        arg = tok[2:]
        if "/" in arg:
            a, b = arg.split("/")
            return math.log(float(a)) / float(b)
        return math.log(float(arg))
    return float(Fraction(tok))


def _vec(spec, n):
    v = np.zeros(n)
    for item in spec:
        i, x = item.split(":")
        v[int(i)] = _num(x)
    return v


def _cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "case":
            cur = {"name": rest[0], "rows": []}
            cases.append(cur)
        elif key == "scale":
            cur["scale"] = _num(rest[0])
        elif key == "query":
            cur["q"] = _vec(rest, 576)
        elif key == "row":
            cur["rows"].append(_vec(rest, 576))
        elif key == "expect_out":
            cur["out"] = _vec(rest, 512)
        elif key == "expect_lse":
            cur["lse"] = _num(rest[0])
    return cases


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_golden_cases(case):
    rows = bf16_bits(np.stack(case["rows"]))
    q = bf16_bits(case["q"][None, :])
    out, lse = oracle.attend_rows(rows, np.arange(len(case["rows"])), q, case["scale"])
    np.testing.assert_allclose(out[0], case["out"], rtol=0, atol=1e-12)
    assert abs(lse[0] - case["lse"]) < 1e-12


def _rand(rng, shape, scale=1.0):
    return bf16_bits(rng.standard_normal(shape) * scale)


def test_single_token_is_its_row():
    rng = np.random.default_rng(1)
    rows = _rand(rng, (10, 576))
    q = _rand(rng, (3, 576))
    tok = np.array([-1, 4, -1, -1], dtype=np.int32)
    out, lse = oracle.attend_rows(rows, tok, q, 0.07)
    for h in range(3):
        np.testing.assert_array_equal(out[h], bf16_vals(rows[4, :512]))
        dot = float(np.dot(bf16_vals(q[h]), bf16_vals(rows[4])))
        assert abs(lse[h] - 0.07 * dot) < 1e-9


def test_no_token_gives_zero_and_minus_inf():
    rng = np.random.default_rng(2)
    rows = _rand(rng, (5, 576))
    out, lse = oracle.attend_rows(rows, np.array([-1, -1], np.int32), _rand(rng, (2, 576)), 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    out, lse = oracle.attend_rows(rows, np.zeros(0, np.int32), _rand(rng, (1, 576)), 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_zero_scale_is_the_mean():
    rng = np.random.default_rng(3)
    rows = _rand(rng, (40, 576))
    tok = rng.choice(40, size=17, replace=False).astype(np.int32)
    out, lse = oracle.attend_rows(rows, tok, _rand(rng, (2, 576)), 0.0)
    mean = bf16_vals(rows[tok, :512]).mean(axis=0)
    np.testing.assert_allclose(out[0], mean, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[1], mean, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, math.log(17), rtol=0, atol=1e-12)


def test_equal_rows_give_that_row():
    rng = np.random.default_rng(4)
    base = _rand(rng, (576,))
    rows = np.tile(base, (12, 1))
    out, _ = oracle.attend_rows(rows, np.arange(12, dtype=np.int32), _rand(rng, (4, 576)), 0.3)
    for h in range(4):
        np.testing.assert_allclose(out[h], bf16_vals(base[:512]), rtol=0, atol=1e-12)


def test_dominant_score_selects_its_row():
    # integer-valued bf16 rows and a one-hot query: score gaps >= 1, scale 1000
    rng = np.random.default_rng(5)
    rows = bf16_bits(rng.integers(-3, 4, size=(20, 576)).astype(np.float64))
    rows[:, 3] = bf16_bits(np.arange(20, dtype=np.float64))  # distinct scores via element 3
    q = np.zeros((1, 576), np.uint16)
    q[0, 3] = bf16_bits(1.0)
    tok = np.array([2, 11, 7, 19, 5], dtype=np.int32)
    out, lse = oracle.attend_rows(rows, tok, q, 1000.0)
    np.testing.assert_array_equal(out[0], bf16_vals(rows[19, :512]))
    assert abs(lse[0] - 1000.0 * 19) < 1e-9


def test_order_and_pads_do_not_matter():
    rng = np.random.default_rng(6)
    rows = _rand(rng, (64, 576))
    q = _rand(rng, (3, 576), 0.2)
    tok = rng.choice(64, size=23, replace=False).astype(np.int32)
    a, la = oracle.attend_rows(rows, tok, q, 0.1)
    perm = np.concatenate([rng.permutation(tok), np.full(5, -1, np.int32)])
    perm = rng.permutation(perm)
    b, lb = oracle.attend_rows(rows, perm, q, 0.1)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    np.testing.assert_allclose(la, lb, rtol=0, atol=1e-12)


def test_common_score_shift_changes_only_lse():
    # every row holds c at element 575 (rope part): raising q[575] by d adds scale*c*d to
    # every score, which leaves the weights alone and moves lse by that amount
    rng = np.random.default_rng(7)
    rows = _rand(rng, (30, 576))
    c = 2.0
    rows[:, 575] = bf16_bits(c)
    q = _rand(rng, (2, 576), 0.3)
    q2 = q.copy()
    d = 1.5
    q2[:, 575] = bf16_bits(bf16_vals(q[:, 575]) + d)
    dd = bf16_vals(q2[:, 575]) - bf16_vals(q[:, 575])
    tok = np.arange(30, dtype=np.int32)
    a, la = oracle.attend_rows(rows, tok, q, 0.25)
    b, lb = oracle.attend_rows(rows, tok, q2, 0.25)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lb - la, 0.25 * c * dd, rtol=0, atol=1e-9)


def test_rope_part_scores_but_is_not_a_value():
    rng = np.random.default_rng(8)
    rows = _rand(rng, (16, 576))
    q = np.zeros((1, 576), np.uint16)  # only the latent part of the query is zero
    q[0, 512:] = _rand(rng, (64,))
    tok = np.arange(16, dtype=np.int32)
    a, _ = oracle.attend_rows(rows, tok, q, 0.5)
    rows2 = rows.copy()
    rows2[:, 512:] = rows[::-1, 512:]  # swap which row carries which rope key
    b, _ = oracle.attend_rows(rows2, tok, q, 0.5)
    assert np.abs(a - b).max() > 1e-3  # the rope part moves the weights
    rows3 = rows.copy()
    rows3[:, 512:] = 0
    q3 = np.zeros((1, 576), np.uint16)
    c, _ = oracle.attend_rows(rows3, tok, q3, 0.5)
    np.testing.assert_allclose(c[0], bf16_vals(rows[:, :512]).mean(axis=0), rtol=0, atol=1e-12)


def test_unit_attend_reads_its_history():
    rng = np.random.default_rng(9)
    u = oracle.OracleUnit(64, topk=8, capacity=16, n_pos=1)
    keys = _rand(rng, (40, 128))
    rows = _rand(rng, (40, 576))
    u.append(keys, rows)
    tok = np.array([3, 39, 17, -1], np.int32)
    q = _rand(rng, (2, 576), 0.1)
    a, la = u.attend(tok, q, 0.3)
    b, lb = oracle.attend_rows(rows, tok, q, 0.3)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
    # a token past the unit's length is not part of its history: treated as a pad
    c, lc = u.attend(np.array([3, 39, 17, 45], np.int32), q, 0.3)
    np.testing.assert_array_equal(a, c)
    np.testing.assert_array_equal(la, lc)
