"""Pins of the oracle's int8 indexer (reading R12: Hadamard rotation, fp16 scale, int8 codes).

Each check compares the oracle with something other than itself: numpy's fp16
conversion, the closed form of the Walsh-Hadamard matrix, hand-derived cases
(tests/golden/int8_quant_cases.txt), a quantization error bound against the
bf16 score, and brute-force selection on small units.
"""
import os

import numpy as np
import pytest

import oracle
from tests.helpers import int_bf16

HERE = os.path.dirname(os.path.abspath(__file__))


def hadamard128():
    r = np.arange(128)[:, None] & np.arange(128)[None, :]
    bits = np.zeros_like(r)
    for b in range(7):
        bits += (r >> b) & 1
    return np.where(bits % 2 == 0, 1.0, -1.0)


def test_f16_matches_numpy():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(3.0),
        rng.standard_normal(2000).astype(np.float32) * np.float32(1e-5),   # fp16 subnormals
        rng.standard_normal(1000).astype(np.float32) * np.float32(3e4),    # near overflow
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, np.inf, -np.inf], np.float32),
    ])
    # exact ties between fp16 neighbours (normal and subnormal): round to even
    h = np.arange(1, 0x7bff, 37, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float32)
    hi = (h + 1).view(np.float16).astype(np.float32)
    vals = np.concatenate([vals, (lo.astype(np.float64) / 2 + hi.astype(np.float64) / 2).astype(np.float32)])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    for v, r in zip(vals, ref):
        assert oracle.f32_to_f16(v) == int(r), v


def test_f16_to_f32_every_pattern():
    for b in range(0, 1 << 16, 7):
        ref = np.uint16(b).view(np.float16).astype(np.float32)
        got = oracle.f16_to_f32(b)
        if np.isnan(ref):
            assert np.isnan(got)
        else:
            assert got.view(np.uint32) == ref.view(np.uint32), hex(b)


def test_fwht_closed_form_and_involution():
    H = hadamard128()
    rng = np.random.default_rng(11)
    for _ in range(20):
        x = rng.integers(-50, 51, 128).astype(np.float32)    # every partial sum exact in fp32
        y = oracle.fwht128(x)
        assert np.array_equal(y, (H @ x.astype(np.float64)).astype(np.float32))
        assert np.array_equal(oracle.fwht128(y), np.float32(128) * x)
    # unit vectors give the columns of H
    for i in (0, 1, 77, 127):
        e = np.zeros(128, np.float32)
        e[i] = 1
        assert np.array_equal(oracle.fwht128(e), H[:, i].astype(np.float32))
    # general bf16 input: within the rounding bound of 7 fp32 stages
    for _ in range(20):
        x = int_bf16(rng.standard_normal(128)).view(np.uint16)
        xf = (x.astype(np.uint32) << 16).view(np.float32)
        y = oracle.fwht128(xf).astype(np.float64)
        ref = H @ xf.astype(np.float64)
        assert np.all(np.abs(y - ref) <= 8 * 2.0 ** -24 * np.abs(xf).sum())


def _golden():
    cases = []
    with open(os.path.join(HERE, "golden", "int8_quant_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, ins, sc, codes = [c.strip() for c in line.split("|")]
            y = np.zeros(128, np.float32)
            for tok in ins.split():
                i, v = tok.split(":")
                y[int(i)] = np.float32(float(v))
            want = np.zeros(128, np.int8)
            for tok in codes.split():
                i, v = tok.split(":")
                want[int(i)] = int(v)
            cases.append((name, y, int(sc, 16), want))
    return cases


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c[0])
def test_quantization_hand_cases(case):
    name, y, scale, want = case
    code, s = oracle.quant_rotated(y)
    assert s == scale, (name, hex(s))
    assert np.array_equal(code, want), name


def test_quant128_of_constant_vector():
    # x = v everywhere -> H x = (128 v, 0, ..., 0): code +-127 at 0, scale fp16(128 |v| / 127)
    for v in (1.0, -0.375, 3.0):
        x = int_bf16(np.full(128, v)).view(np.uint16)
        code, s = oracle.quant128(x)
        want = np.zeros(128, np.int8)
        want[0] = 127 if v > 0 else -127
        assert np.array_equal(code, want)
        assert s == int(np.float32(np.float32(128 * abs(v)) / np.float32(127)).astype(np.float16).view(np.uint16))


def test_score_i8_hand_cases():
    e0 = np.zeros(128, np.int8)
    e0[0] = 127
    one = 0x3c00
    # 127 * 127 / 128 = 126.0078125 exactly
    assert oracle.score_i8(e0, one, e0, one) == np.float32(126.0078125)
    neg = e0.copy()
    neg[0] = -127
    assert oracle.score_i8(e0, one, neg, one) == np.float32(-126.0078125)
    two = 0x4000
    assert oracle.score_i8(e0, two, e0, one) == np.float32(252.015625)
    z = np.zeros(128, np.int8)
    s = oracle.score_i8(z, one, e0, one)
    assert s == 0 and np.signbit(s) == False  # noqa: E712  (+0)


def test_int8_score_tracks_bf16_score_within_quantization_bound():
    H = hadamard128()
    rng = np.random.default_rng(5)
    for _ in range(200):
        q = int_bf16(rng.standard_normal(128)).view(np.uint16)
        k = int_bf16(rng.standard_normal(128)).view(np.uint16)
        qc, qs = oracle.quant128(q)
        kc, ks = oracle.quant128(k)
        s8 = float(oracle.score_i8(qc, qs, kc, ks))
        qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        kf = (k.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        exact = float(qf @ kf)
        sq, sk = float(oracle.f16_to_f32(qs)), float(oracle.f16_to_f32(ks))
        yq, yk_hat = H @ qf, kc.astype(np.float64) * sk
        # |y_q . y_k - yq_hat . yk_hat| <= sum|y_q| sk/2 + sum|yk_hat| sq/2, then / 128
        bound = (np.abs(yq).sum() * sk / 2 + np.abs(yk_hat).sum() * sq / 2) / 128
        assert abs(s8 - exact) <= bound * 1.001 + 1e-6 * abs(exact) + 1e-6, (s8, exact, bound)


def test_unit_int8_keys_and_brute_force_selection():
    rng = np.random.default_rng(9)
    L, P, K = 300, 3, 40
    keys = int_bf16(rng.standard_normal((L, 128))).view(np.uint16)
    # integer-valued keys produce many equal int8 scores: ties by token
    keys[::3] = int_bf16(np.clip(np.rint(rng.standard_normal((100, 128))), -1, 1)).view(np.uint16)
    u = oracle.OracleUnit(L, K, 4 * K, P, row_elems=8, keep_rows=False, idx_int8=True)
    assert u.append(keys) == oracle.OK
    kc, ks = u.key_codes()
    for t in (0, 1, 150, 299):
        c, s = oracle.quant128(keys[t])
        assert np.array_equal(kc[t], c) and ks[t] == s
    q = int_bf16(rng.standard_normal((P, 128))).view(np.uint16)
    r = u.step(q)
    for p in range(P):
        vis = L - (P - 1 - p)
        qc, qs = oracle.quant128(q[p])
        sc = np.array([oracle.score_i8(qc, qs, kc[t], ks[t]) for t in range(vis)], np.float32)
        order = sorted(range(vis), key=lambda t: (-sc[t], t))[:K]
        assert r.tok[p].tolist() == order
        assert np.array_equal(r.score[p], sc[order])
