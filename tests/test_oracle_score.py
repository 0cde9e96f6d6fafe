"""Pins of the oracle's indexer score (reading R1) against facts outside it.

- closed forms: one-hot queries return the key element exactly; small-integer
  inputs return the exact integer dot product;
- hand-derived values that only the chosen summation order produces
  (tests/golden/score_order_cases.txt);
- the fp32 error bound of an 11-deep summation against the exact value.
"""
import math
import os

import numpy as np
import pytest

import oracle
import workload as W
from tests.helpers import int_bf16, rand_int_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "score_order_cases.txt")


def _load_cases():
    cases = []
    cur = None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "case":
                cur = (parts[1], float(parts[2]), [])
            elif parts[0] == "end":
                cases.append(cur)
                cur = None
            else:
                cur[2].append((int(parts[0]), float(parts[1]), float(parts[2])))
    return cases


@pytest.mark.parametrize("case", _load_cases(), ids=lambda c: c[0])
def test_score_order_golden(case):
    name, expected, entries = case
    q = np.zeros(128, np.float32)
    k = np.zeros(128, np.float32)
    for d, qv, kv in entries:
        q[d], k[d] = qv, kv
    qb = (q.view(np.uint32) >> 16).astype(np.uint16)
    kb = (k.view(np.uint32) >> 16).astype(np.uint16)
    s = oracle.score(qb, kb)
    assert float(s) == expected, name
    assert not np.signbit(s) or expected < 0


def test_one_hot_query_returns_key_element():
    rng = np.random.default_rng(7)
    k = W.normal_bf16(11, W.KIND_KEYS, 0, 0, 0, 0, 128)
    kf = W.bf16_to_f32(k)
    for d in range(128):
        q = np.zeros(128, np.float32)
        q[d] = 1.0
        assert oracle.score(int_bf16(q), k) == kf[d]
        scale = float(2.0 ** rng.integers(-8, 8))
        q[d] = -scale
        assert oracle.score(int_bf16(q), k) == np.float32(-scale * kf[d])


def test_small_integers_give_exact_dot():
    rng = np.random.default_rng(3)
    for _ in range(200):
        qi, qb = rand_int_bf16(rng, 128, -7, 7)
        ki, kb = rand_int_bf16(rng, 128, -7, 7)
        assert float(oracle.score(qb, kb)) == float(np.dot(qi, ki))


def test_error_bound_against_exact_sum():
    # Every product of two bf16 values is exact in fp64 and in fp32; the sum
    # sees at most 7 chain roundings and 4 tree roundings.
    keys = W.normal_bf16(21, W.KIND_KEYS, 0, 0, 0, 0, 128 * 400).reshape(400, 128)
    qs = W.normal_bf16(21, W.KIND_QINIT, 0, 0, 0, 0, 128 * 4).reshape(4, 128)
    u = 2.0 ** -24
    gamma = 11 * u / (1 - 11 * u)
    worst = 0.0
    for q in qs:
        qf = W.bf16_to_f32(q).astype(np.float64)
        for k in keys:
            kf = W.bf16_to_f32(k).astype(np.float64)
            prods = qf * kf
            exact = math.fsum(prods.tolist())
            bound = gamma * float(np.abs(prods).sum())
            s = float(oracle.score(q, k))
            assert abs(s - exact) <= bound
            if bound > 0:
                worst = max(worst, abs(s - exact) / bound)
    assert worst < 1.0


def test_score_is_linear_in_sign():
    keys = W.normal_bf16(5, W.KIND_KEYS, 0, 0, 0, 0, 128 * 50).reshape(50, 128)
    q = W.normal_bf16(5, W.KIND_QINIT, 0, 0, 0, 0, 128)
    qneg = q ^ np.uint16(0x8000)
    for k in keys:
        assert oracle.score(qneg, k) == -oracle.score(q, k)
